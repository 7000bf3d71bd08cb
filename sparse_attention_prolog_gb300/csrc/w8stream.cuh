// Weight-stream int8 products for decode-size batches:
//
//   s[t, n] = sum_k a[t, k] b[n, k]      (exact int32, dp4a)
//
// for a few rows of a (t < M <= 32) against every row n of a large
// row-major int8 matrix b [N, K] that is read once from HBM.  Used by the
// int8 GEMM at decode sizes ([V4-TileLang §Int8 General Matrix
// Multiplication]) and by the MLA Prolog's q_lora . w_uq^T
// ([V3.2-PyPTO §Deepseek Indexer Attention], its first part).
//
// Layout of the work:
//   - one CTA per SM, each owning a contiguous range of b's rows, so that
//     its share of the stream is one contiguous block of bytes and every SM
//     streams the same amount (no second wave of CTAs);
//   - a producer warp pulls the block through a ring of stages, each stage
//     `sr` whole rows taken by one bulk copy;
//   - eight consumer warps compute.  The lanes of a warp split K into
//     16-byte chunks; when the rows of a would not fit in registers the
//     warps split K as well (`wk` groups of warps, the other 8 / wk groups
//     take alternate rows of a stage).  Each lane keeps its chunks of a's
//     rows in registers for the whole stream, so a weight chunk costs one
//     shared-memory load and 4 MT dp4a;
//   - a row's MT partial sums are reduced across the lanes by a transposing
//     butterfly (each exchange halves the values a lane keeps, 31 shuffles
//     for 32 tokens, 9 for 8), after which each lane holds one token's sum;
//     with wk > 1 the warps' sums of a row meet in shared memory (integer
//     atomics, exact in any order).
#pragma once
#include <cstdint>
#include "dsa_ptx.cuh"

namespace dsa {

constexpr int kW8Consumers = 8;                      // consumer warps
constexpr int kW8Threads = 32 * (kW8Consumers + 1);  // + the producer warp
constexpr uint32_t kW8RingBytes = 168 * 1024;        // stage ring in shared memory
constexpr uint32_t kW8StageTarget = 32 * 1024;       // bytes per stage, about
constexpr int kW8MaxStages = 8;
constexpr int kW8MaxStageRows = 64;

struct W8Plan {
  int wk;                // warps splitting K: 1, 2, 4 or 8
  int kw;                // 16-byte chunks of K per lane (0: K too large for the registers)
  int sr;                // rows per stage
  int ns;                // stages in the ring
  uint32_t stage_bytes;  // sr * K
};

// Host: the split for a product of MT (8, 16 or 32) rows of a with K
// columns, with a stage ring of at most ring_bytes.  a's chunks of a lane
// take kw * MT * 4 <= a_regs registers.
inline W8Plan w8_plan(int K, int MT, int a_regs, uint32_t ring_bytes = kW8RingBytes) {
  W8Plan p{};
  const int nck = K / 16, kwmax = a_regs / (4 * MT);
  for (p.wk = 1; p.wk <= 8; p.wk *= 2) {
    p.kw = (nck + 32 * p.wk - 1) / (32 * p.wk);
    if (p.kw <= kwmax) break;
  }
  if (p.wk > 8) {
    p.kw = 0;
    return p;
  }
  const int rg = kW8Consumers / p.wk;  // row groups
  int sr = static_cast<int>(kW8StageTarget / static_cast<uint32_t>(K));
  if (sr > kW8MaxStageRows) sr = kW8MaxStageRows;
  sr = sr / rg * rg;
  if (sr < rg) sr = rg;
  p.sr = sr;
  p.stage_bytes = static_cast<uint32_t>(sr) * static_cast<uint32_t>(K);
  p.ns = static_cast<int>(ring_bytes / p.stage_bytes);
  if (p.ns > kW8MaxStages) p.ns = kW8MaxStages;
  if (p.ns < 2) p.kw = 0;  // no room for a ring
  return p;
}

// Shared memory of a weight-stream kernel beyond its own: the ring, the
// cross-warp sums (2 x sr x MT int32) and 1 KB of alignment slack.
inline size_t w8_smem(const W8Plan& p, int MT) {
  return 1024 + static_cast<size_t>(p.ns) * p.stage_bytes + 2 * static_cast<size_t>(p.sr) * MT * 4;
}

// One lane's share of a warp sum of v[0..N) (N a power of two <= 32): after
// the exchanges, the return value is the sum over all 32 lanes of v[tok].
template <int N>
__device__ __forceinline__ int warp_transpose_sum(int (&v)[N], int lane, int& tok) {
  tok = 0;
#pragma unroll
  for (int w = N / 2, b = 16; w >= 1; w >>= 1, b >>= 1) {
    const bool up = (lane & b) != 0;  // the upper lane of the pair keeps v[w .. 2w)
#pragma unroll
    for (int i = 0; i < w; ++i) {
      const int send = up ? v[i] : v[i + w];
      const int keep = up ? v[i + w] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, b);
    }
    if (up) tok += w;
  }
#pragma unroll
  for (int b = 16 / N; b >= 1; b >>= 1) v[0] += __shfl_xor_sync(0xffffffffu, v[0], b);
  return v[0];
}

// The rows of b that CTA g of G owns: [r0, r1), balanced to within one row.
__device__ __forceinline__ void w8_rows(int N, int g, int G, int& r0, int& r1) {
  r0 = static_cast<int>(static_cast<long long>(N) * g / G);
  r1 = static_cast<int>(static_cast<long long>(N) * (g + 1) / G);
}

struct W8Ring {
  uint8_t* smem;   // ns stages of stage_bytes
  uint64_t* full;  // [ns] the stage's bytes have landed
  uint64_t* empty; // [ns] the consumer warps are done with the stage (count kW8Consumers)
  int* red;        // [2][sr][MT] cross-warp sums, zero on entry (wk > 1)
};

// Producer (one thread): rows [r0, r1) of b (row-major, K bytes per row) in
// stages of p.sr rows.  If a wait gives up, the stages still in flight land
// before it returns.
__device__ __forceinline__ void w8_produce(const W8Plan& p, const W8Ring& R, const int8_t* b, int K, int r0, int r1,
                                           uint32_t* err, volatile int* abort_flag) {
  const int n_st = (r1 - r0 + p.sr - 1) / p.sr;
  int issued = 0;
  for (int i = 0; i < n_st; ++i) {
    const int s = i % p.ns;
    if (i >= p.ns && !mbar_wait(&R.empty[s], ((i / p.ns) - 1) & 1, err, abort_flag)) break;
    const int row0 = r0 + i * p.sr;
    const int rows = min(p.sr, r1 - row0);
    const uint32_t bytes = static_cast<uint32_t>(rows) * static_cast<uint32_t>(K);
    mbar_arrive_expect_tx(&R.full[s], bytes);
    bulk_g2s(R.smem + static_cast<size_t>(s) * p.stage_bytes, b + static_cast<size_t>(row0) * K, bytes, &R.full[s]);
    issued = i + 1;
  }
  for (int i = issued > p.ns ? issued - p.ns : 0; i < issued; ++i) mbar_drain(&R.full[i % p.ns], (i / p.ns) & 1);
}

// Loads a lane's chunks of the rows of a (t < M; the other MT - M rows are
// zero): chunk j is column block c0 + lane + 32 j of the warp's K slice
// [c0, c1).  `a` may point to global or shared memory (lda bytes per row).
template <int MT, int KW>
__device__ __forceinline__ void w8_load_a(int4 (&areg)[KW][MT], const int8_t* a, int lda, int M, int c0, int c1,
                                          int lane) {
#pragma unroll
  for (int j = 0; j < KW; ++j) {
    const int c = c0 + lane + 32 * j;
#pragma unroll
    for (int t = 0; t < MT; ++t)
      areg[j][t] = (c < c1 && t < M) ? *reinterpret_cast<const int4*>(a + static_cast<size_t>(t) * lda + c * 16)
                                     : make_int4(0, 0, 0, 0);
  }
}

// Consumer warps (warp < kW8Consumers, all 256 threads call it): the stage
// loop.  epi(t, n, s) receives every finished sum once (t < M).  With
// p.wk > 1 the 256 consumer threads synchronise on named barrier 1 once per
// stage and take the abort decision together.
template <int MT, int KW, int RPW, class Epi>
__device__ __forceinline__ void w8_consume(const W8Plan& p, const W8Ring& R, const int4 (&areg)[KW][MT], int K, int M,
                                           int r0, int r1, int c0, int c1, Epi epi, uint32_t* err,
                                           volatile int* abort_flag) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rg = warp / p.wk, n_rg = kW8Consumers / p.wk;
  const int n_st = (r1 - r0 + p.sr - 1) / p.sr;
  for (int i = 0; i < n_st; ++i) {
    const int s = i % p.ns;
    bool ok = mbar_wait(&R.full[s], (i / p.ns) & 1, err, abort_flag);
    if (p.wk > 1) {
      uint32_t all;
      asm volatile("{\n.reg .pred p, q;\nsetp.ne.b32 p, %1, 0;\nbar.red.and.pred q, 1, 256, p;\nselp.u32 %0, 1, 0, q;\n}"
                   : "=r"(all) : "r"(ok ? 1u : 0u) : "memory");
      ok = all != 0;
    }
    if (!ok) break;
    const uint8_t* stage = R.smem + static_cast<size_t>(s) * p.stage_bytes;
    const int row0 = r0 + i * p.sr;
    const int rows = min(p.sr, r1 - row0);
    int* red = R.red + (i & 1) * p.sr * MT;
    // RPW rows of the stage at once per warp (RPW x MT <= 32): independent
    // dp4a chains, and one transposing reduction of their RPW x MT sums
    static_assert(RPW * MT <= 32, "one transposing reduction holds at most 32 sums");
    for (int r = rg * RPW; r < rows; r += n_rg * RPW) {
      int acc[RPW * MT];
#pragma unroll
      for (int i = 0; i < RPW * MT; ++i) acc[i] = 0;
#pragma unroll
      for (int j = 0; j < KW; ++j) {
        const int c = c0 + lane + 32 * j;
        if (c < c1) {
          int4 w[RPW];
#pragma unroll
          for (int q = 0; q < RPW; ++q)
            w[q] = r + q < rows ? *reinterpret_cast<const int4*>(stage + static_cast<size_t>(r + q) * K + c * 16)
                                : make_int4(0, 0, 0, 0);
          // component-major order: consecutive dp4a feed different sums
#pragma unroll
          for (int q = 0; q < RPW; ++q)
#pragma unroll
            for (int t = 0; t < MT; ++t) acc[q * MT + t] = __dp4a(w[q].x, areg[j][t].x, acc[q * MT + t]);
#pragma unroll
          for (int q = 0; q < RPW; ++q)
#pragma unroll
            for (int t = 0; t < MT; ++t) acc[q * MT + t] = __dp4a(w[q].y, areg[j][t].y, acc[q * MT + t]);
#pragma unroll
          for (int q = 0; q < RPW; ++q)
#pragma unroll
            for (int t = 0; t < MT; ++t) acc[q * MT + t] = __dp4a(w[q].z, areg[j][t].z, acc[q * MT + t]);
#pragma unroll
          for (int q = 0; q < RPW; ++q)
#pragma unroll
            for (int t = 0; t < MT; ++t) acc[q * MT + t] = __dp4a(w[q].w, areg[j][t].w, acc[q * MT + t]);
        }
      }
      int tok;
      const int v = warp_transpose_sum<RPW * MT>(acc, lane, tok);
      const int rr = r + tok / MT, t = tok % MT;
      if ((lane & (32 / (RPW * MT) - 1)) == 0 && t < M && rr < rows) {
        if (p.wk == 1) epi(t, row0 + rr, v);
        else atomicAdd(red + rr * MT + t, v);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&R.empty[s]);  // this warp has read the stage
    if (p.wk > 1) {
      asm volatile("bar.sync 1, 256;" ::: "memory");  // every warp's sums of the stage are in red
      for (int idx = tid; idx < rows * M; idx += 32 * kW8Consumers) {
        const int t = idx / rows, r = idx % rows;  // adjacent threads: adjacent rows n
        int* q = red + r * MT + t;
        epi(t, row0 + r, *q);
        *q = 0;  // ready for stage i + 2 (the next barrier separates them)
      }
    }
  }
}

}  // namespace dsa

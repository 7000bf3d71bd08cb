// Weight-stream int8 products on the tensor cores:
//
//   s[t, n] = sum_k a[t, k] b[n, k]      (exact int32)
//
// for up to NT (16 or 32) rows of a (decode tokens) against every row n of
// a row-major int8 matrix b [N, K] that is read once from HBM.  Used by the
// int8 GEMM at decode sizes ([V4-TileLang §Int8 General Matrix
// Multiplication]) and by the MLA Prolog's q_lora . w_uq^T
// ([V3.2-PyPTO §Deepseek Indexer Attention], its first part).
//
// The weight rows are the MMA's M dimension (128 per block) and the tokens
// its N, so a few tokens cost one M = 128, N = NT MMA per 16 columns of K
// instead of 4 NT dp4a per 16 weight bytes.  Both operands are converted
// to f16, exact for int8; a product is at most 2^14 in magnitude, so the
// fp32 sum of up to 1024 of them is an exact integer below 2^24: the MMAs
// switch accumulators every 1024 K and the epilogue adds the chunks in
// int32.  The sums equal the int32 product bit for bit.
//
// Work: one CTA per SM over a contiguous range of b's rows, in units of 16
// rows (ranges differ by at most one unit), walked in blocks of 128 rows;
// the last block may be partial.  Warp roles (448 threads):
//   warp 0     producer: 2-D TMA loads (128-byte swizzle) of 128-column
//              tiles of the block's rows (one 128-row box, or 16-row boxes
//              for a partial block) and, unless the tokens are resident in
//              shared memory, of the tokens' 128-column tile; a ring of up
//              to 12 stages (as many as the launch's shared memory holds)
//   warps 2-9  converters, two per TMEM lane quarter: thread r of the
//              first four converts columns 0-63 of weight row r of a tile
//              to f16 into tensor memory (the A operand), of the other four
//              columns 64-127; each thread also converts one 16-byte chunk
//              of the tokens' tile into shared memory (the B operand,
//              K-major, 128-byte swizzle); 3 stages of each
//   warp 1     one thread issues the MMAs (M = 128, N = NT, K = 16; A from
//              TMEM, B from shared memory) into one of two accumulators,
//              switching at every 1024-K chunk
//   warps 10-13 epilogue: thread = TMEM lane = weight row; adds each chunk
//              into int32 registers and hands the finished row to the job
//              (coalesced across the lanes of a warp).
// With resident tokens the eight converter warps first run the job's
// prologue, which writes the tokens into shared memory (the weight copies
// are in flight meanwhile).
#pragma once
#include <cstdint>
#include <cuda.h>
#include "dsa_ptx.cuh"

namespace dsa {

constexpr int kWtThreads = 448;
constexpr int kWtConv = 8;                        // converter warps (2..9)
constexpr int kWtEpi0 = 2 + kWtConv;              // first epilogue warp
constexpr int kWtRows = 128;                      // weight rows per block (the MMA's M)
constexpr int kWtK = 128;                         // K columns per stage
constexpr int kWtUnit = 16;                       // rows: unit of a CTA's range, height of a partial-block box
constexpr int kWtS8Max = 12, kWtS16 = 3;          // raw stages (at most; the launch picks), converted stages
constexpr int kWtChunk = 1024 / kWtK;             // stages per exact 1024-K chunk
constexpr uint32_t kWtRawW = kWtRows * kWtK;      // 16 KB: one raw weight tile
constexpr uint32_t kWtBoxUnit = kWtUnit * kWtK;   // 2 KB: a 16-row box
constexpr uint32_t kWtACol0 = 64;                 // TMEM: accumulators at [0, 2 NT), A stages from here
constexpr uint32_t kWtACols = kWtK / 2;           // one f16 A stage: 64 columns
constexpr uint32_t kWtTmemCols = 256;

struct WtMaps {
  CUtensorMap w128;  // b [N, K] int8, box {128 columns, 128 rows}
  CUtensorMap w16;   // b [N, K] int8, box {128 columns, 16 rows}
  CUtensorMap tok;   // a [M, K] int8, box {128 columns, NT rows} (streamed tokens)
};

struct __align__(8) WtBars {
  uint64_t full8[kWtS8Max], empty8[kWtS8Max], full16[kWtS16], empty16[kWtS16], tfull[2], tempty[2];
  uint64_t mdrain;    // the MMA thread's last commit
  uint64_t tokready;  // resident tokens are in shared memory
};

template <int NT, bool kResident>
struct WtLayout {
  static constexpr uint32_t kRawTok = kResident ? 0u : static_cast<uint32_t>(NT * kWtK);
  static constexpr uint32_t kStage8 = kWtRawW + kRawTok;
  static constexpr uint32_t kAtomB = NT * 128;  // 64 f16 columns of the tokens
  static constexpr uint32_t kTileB = 2 * kAtomB;
  // dynamic shared memory: alignment slack, raw ring of ns8 stages,
  // converted token tiles, resident tokens [NT][K]
  static size_t smem(int K, int ns8) {
    return 1024 + ns8 * static_cast<size_t>(kStage8) + kWtS16 * static_cast<size_t>(kTileB) +
           (kResident ? static_cast<size_t>(NT) * K : 0);
  }
  // the most raw stages (2 .. kWtS8Max) that fit in `budget` bytes
  static int stages(int K, size_t budget) {
    int n = kWtS8Max;
    while (n > 2 && smem(K, n) > budget) --n;
    return n;
  }
};

// The rows [r0, r1) of b that CTA g of G owns: whole 16-row units, balanced.
__device__ __forceinline__ void wt_rows(int N, int g, int G, int& r0, int& r1) {
  const long long U = (N + kWtUnit - 1) / kWtUnit;
  r0 = static_cast<int>(U * g / G) * kWtUnit;
  r1 = min(N, static_cast<int>(U * (g + 1) / G) * kWtUnit);
}

// Job interface (a struct passed by value):
//   int M, N, K                        tokens, weight rows, columns
//   float tok_scale(int t)             (called after the prologue)
//   float row_scale(int n)
//   void put(int t, int n, int s, float st, float sn)   one finished sum
//   void prologue(int w, int lane, int8_t* tok)  (resident: converter warp w
//       of 8 writes tokens into tok [NT][K]; rows >= M are zeroed here)
//   void tail(int warp, int lane)      after the stream, every warp
template <int NT, bool kResident, class Job>
__global__ void __launch_bounds__(kWtThreads, 1) wt_kernel(const __grid_constant__ WtMaps maps, const Job job,
                                                            const int ns8) {
  using L = WtLayout<NT, kResident>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* s8 = smem;                                   // [ns8][weights 16 KB | tokens], int8, swizzled
  uint8_t* sB = smem + ns8 * L::kStage8;                // [kWtS16][2 atoms], f16 tokens, swizzled
  int8_t* sTok = reinterpret_cast<int8_t*>(sB + kWtS16 * L::kTileB);  // resident tokens [NT][K]
  __shared__ WtBars bars;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int M = job.M, N = job.N, K = job.K;
  uint32_t* err = job.err;
  int r0, r1;
  wt_rows(N, blockIdx.x, gridDim.x, r0, r1);
  const int nst = (K + kWtK - 1) / kWtK;                 // stages per block
  const int cpb = (nst + kWtChunk - 1) / kWtChunk;       // exact chunks per block
  const int nb = r1 > r0 ? (r1 - r0 + kWtRows - 1) / kWtRows : 0;
  const int total = nb * nst;

  if (tid == 0) {
    for (int i = 0; i < ns8; ++i) { mbar_init(&bars.full8[i], 1); mbar_init(&bars.empty8[i], kWtConv); }
    for (int i = 0; i < kWtS16; ++i) { mbar_init(&bars.full16[i], kWtConv); mbar_init(&bars.empty16[i], 1); }
    for (int i = 0; i < 2; ++i) { mbar_init(&bars.tfull[i], 1); mbar_init(&bars.tempty[i], 4); }
    mbar_init(&bars.mdrain, 1);
    mbar_init(&bars.tokready, kWtConv);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(&tmem_base, kWtTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;
  volatile int* abort_v = &abort_flag;
  griddep_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // The weights are inputs of this call: their copies go out at once.
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&maps.w128)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&maps.w16)) : "memory");
      if (!kResident) griddep_wait();  // streamed tokens may come from the previous kernel
      int s = 0;
      bool ok = true;
      for (int bi = 0; bi < nb && ok; ++bi) {
        const int row_b = r0 + bi * kWtRows;
        const int rows_b = min(kWtRows, r1 - row_b);
        const int nbox = rows_b == kWtRows ? 1 : (rows_b + kWtUnit - 1) / kWtUnit;
        const uint32_t wbytes = rows_b == kWtRows ? kWtRawW : nbox * kWtBoxUnit;
        for (int k = 0; k < nst; ++k, ++s) {
          const int st = s % ns8;
          if (s >= ns8 && !mbar_wait(&bars.empty8[st], ((s / ns8) - 1) & 1, err, abort_v)) { ok = false; break; }
          uint8_t* dst = s8 + st * L::kStage8;
          mbar_arrive_expect_tx(&bars.full8[st], wbytes + L::kRawTok);  // columns past K, rows past N: zero fill
          if (rows_b == kWtRows) {
            tma_load_2d(dst, &maps.w128, k * kWtK, row_b, &bars.full8[st]);
          } else {
            for (int j = 0; j < nbox; ++j)
              tma_load_2d(dst + j * kWtBoxUnit, &maps.w16, k * kWtK, row_b + j * kWtUnit, &bars.full8[st]);
          }
          if (!kResident) tma_load_2d(dst + kWtRawW, &maps.tok, k * kWtK, 0, &bars.full8[st]);
        }
      }
      // if a wait gave up, the last stages' copies land before the CTA leaves
      for (int i = s > ns8 ? s - ns8 : 0; i < s; ++i) mbar_drain(&bars.full8[i % ns8], (i / ns8) & 1);
    }
  } else if (warp == 1) {
    // --------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_f16(kWtRows, NT, kFmtF16, 0, 0);
      int s = 0, gc = 0;
      bool ok = true;
      for (int bi = 0; bi < nb && ok; ++bi) {
        for (int k = 0; k < nst; ++k, ++s) {
          const int st = s % kWtS16, buf = gc & 1;
          const bool first_of_chunk = (k % kWtChunk) == 0;
          // the accumulator is free once the epilogue has read its previous chunk
          if (first_of_chunk && gc >= 2 && !mbar_wait(&bars.tempty[buf], ((gc / 2) - 1) & 1, err, abort_v)) {
            ok = false;
            break;
          }
          if (!mbar_wait(&bars.full16[st], (s / kWtS16) & 1, err, abort_v)) { ok = false; break; }
          tc_fence_after();
          const uint32_t b_base = smem_u32(sB + st * L::kTileB);
          const uint32_t a_tmem = tmem + kWtACol0 + st * kWtACols;
#pragma unroll
          for (int kk = 0; kk < kWtK / 16; ++kk) {
            const uint64_t bd = smem_desc(b_base + (kk / 4) * L::kAtomB + (kk % 4) * 32, 16, 1024, kSwizzle128B);
            mma_ts(tmem + buf * NT, a_tmem + kk * 8, bd, idesc, (!first_of_chunk || kk > 0) ? 1u : 0u);
          }
          mma_commit(&bars.empty16[st]);
          if ((k % kWtChunk) == kWtChunk - 1 || k == nst - 1) {
            mma_commit(&bars.tfull[buf]);
            ++gc;
          }
        }
      }
      // every MMA issued has completed before the tensor memory is freed
      mma_commit(&bars.mdrain);
      mbar_drain(&bars.mdrain, 0);
    }
  } else if (warp < kWtEpi0) {
    // ---------------------------------------------------------- converters
    // Thread = row r of the weight tile; a warp reaches the TMEM lanes of
    // its quarter (warp % 4), so r = 32 (warp % 4) + lane; converter warps
    // 2-5 take the tile's columns 0-63 (half 0), warps 6-9 columns 64-127.
    const int r = (warp & 3) * 32 + lane;
    const int half = (warp - 2) / 4;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16) + kWtACol0;
    // this thread's chunk of the tokens' tile: row tr, 16-byte chunk tq
    const int titem = (warp - 2) * 32 + lane, tr = titem >> 3, tq = titem & 7;
    bool ok = true;
    if (kResident) {
      job.prologue(warp - 2, lane, sTok);
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.tokready);  // release: this warp's tokens are written
      ok = mbar_wait(&bars.tokready, 0, err, abort_v);
    }
    for (int s = 0; s < total && ok; ++s) {
      const int st8 = s % ns8, st16 = s % kWtS16, k = s % nst;
      if (!mbar_wait(&bars.full8[st8], (s / ns8) & 1, err, abort_v)) break;
      if (s >= kWtS16 && !mbar_wait(&bars.empty16[st16], ((s / kWtS16) - 1) & 1, err, abort_v)) break;
      tc_fence_after();
      const uint8_t* src = s8 + st8 * L::kStage8;
      // weight row r, columns 64 half .. 64 half + 63 -> f16 pairs -> TMEM:
      // 16-byte chunk q of the row sits at q ^ (r & 7) (128-byte swizzle), so
      // a quarter warp reads 8 distinct bank groups.  Rows past a partial
      // block convert whatever the tile holds (their sums are never read).
      {
        uint4 va[4];
#pragma unroll
        for (int q = 0; q < 4; ++q)
          va[q] = *reinterpret_cast<const uint4*>(src + r * 128 + (((4 * half + q) ^ (r & 7)) << 4));
        uint32_t fa[32];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          i8x4_to_f16x4(va[q].x, fa[8 * q + 0], fa[8 * q + 1]);
          i8x4_to_f16x4(va[q].y, fa[8 * q + 2], fa[8 * q + 3]);
          i8x4_to_f16x4(va[q].z, fa[8 * q + 4], fa[8 * q + 5]);
          i8x4_to_f16x4(va[q].w, fa[8 * q + 6], fa[8 * q + 7]);
        }
        tmem_st32(lane_base + st16 * kWtACols + half * 32, fa);
      }
      // chunk tq of token row tr -> f16, K-major with the 128-byte swizzle
      // the MMA reads: columns 64h .. 64h + 63 are atom h
      if (tr < NT) {
        uint4 v;
        if (kResident) {
          const int col = k * kWtK + tq * 16;
          v = col < K ? *reinterpret_cast<const uint4*>(sTok + static_cast<size_t>(tr) * K + col)
                      : make_uint4(0u, 0u, 0u, 0u);
        } else {
          v = *reinterpret_cast<const uint4*>(src + kWtRawW + tr * 128 + ((tq ^ (tr & 7)) << 4));
        }
        uint32_t f[8];
        i8x4_to_f16x4(v.x, f[0], f[1]);
        i8x4_to_f16x4(v.y, f[2], f[3]);
        i8x4_to_f16x4(v.z, f[4], f[5]);
        i8x4_to_f16x4(v.w, f[6], f[7]);
        uint8_t* drow = sB + st16 * L::kTileB + (tq / 4) * L::kAtomB;
        *reinterpret_cast<uint4*>(drow + sw128_off(tr, 2 * (tq % 4))) = make_uint4(f[0], f[1], f[2], f[3]);
        *reinterpret_cast<uint4*>(drow + sw128_off(tr, 2 * (tq % 4) + 1)) = make_uint4(f[4], f[5], f[6], f[7]);
      }
      tmem_st_wait();
      fence_proxy_async_smem();  // generic stores -> tensor core reads
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&bars.full16[st16]);
        mbar_arrive(&bars.empty8[st8]);
      }
    }
  } else {
    // ----------------------------------------------------------- epilogue
    const int q4 = warp & 3;  // TMEM lane quarter of this warp
    const int row = q4 * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(q4 * 32) << 16);
    bool ok_tok = true;
    if (kResident && !mbar_wait(&bars.tokready, 0, err, abort_v)) ok_tok = false;  // the tokens' scales
    float st[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) st[t] = t < M ? job.tok_scale(t) : 0.f;
    int gc = 0;
    bool ok = ok_tok;
    for (int bi = 0; bi < nb && ok; ++bi) {
      const int row_b = r0 + bi * kWtRows;
      const int rows_b = min(kWtRows, r1 - row_b);
      const int n = row_b + row;
      const float sn = row < rows_b ? job.row_scale(n) : 0.f;
      int tot[NT];
#pragma unroll
      for (int t = 0; t < NT; ++t) tot[t] = 0;
      for (int ch = 0; ch < cpb; ++ch, ++gc) {
        const int buf = gc & 1;
        if (!mbar_wait(&bars.tfull[buf], (gc / 2) & 1, err, abort_v)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int c0 = 0; c0 < NT; c0 += 16) {
          uint32_t v[16];
          tmem_ld16(lane_base + buf * NT + c0, v);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j) tot[c0 + j] += __float2int_rn(__uint_as_float(v[j]));  // exact integers
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.tempty[buf]);
      }
      if (!ok) break;
      if (row < rows_b) {
#pragma unroll
        for (int t = 0; t < NT; ++t)
          if (t < M) job.put(t, n, tot[t], st[t], sn);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  job.tail(warp, lane);
  if (warp == 0) tmem_dealloc(tmem, kWtTmemCols);
}

}  // namespace dsa

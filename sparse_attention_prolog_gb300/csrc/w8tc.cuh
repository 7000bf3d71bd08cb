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
// The weight rows are the MMA's M dimension (128 per MMA block) and the
// tokens its N, so a few tokens cost one M = 128, N = NT MMA per 16 columns
// of K instead of 4 NT dp4a per 16 weight bytes.  Both operands are
// converted to f16, exact for int8; a product is at most 2^14 in magnitude,
// so the fp32 sum of up to 1024 of them is an exact integer below 2^24: the
// MMAs switch accumulators every 1024 K and the epilogue adds the chunks in
// int32.  The sums equal the int32 product bit for bit.
//
// Work: one CTA per SM over a contiguous range of b's rows, in units of 16
// rows (ranges differ by at most one unit), walked in super-blocks of up to
// 256 rows (two MMA blocks).  A stage is one TMA box as high as the
// super-block (16 to 256 rows) by 128 columns, so every copy moves up to
// 32 KB of the SM's range at once: at the decode shapes a CTA's 160-176
// rows are one super-block (separate boxes for the rows past 128 moved 4-6
// KB each and ran at about half the bytes per second).  Warp roles (448
// threads):
//   warp 0     producer: the 2-D TMA loads (128-byte swizzle) of the
//              super-block's tile and, unless the tokens are resident in
//              shared memory, of the tokens' 128-column tile; a ring of up
//              to 8 stages (as many as the launch's shared memory holds)
//   warps 2-9  converters, two per TMEM lane quarter: thread r of the
//              first four converts columns 0-63 of rows r and 128 + r of a
//              tile to f16 into tensor memory (the A operands of the two
//              blocks), of the other four columns 64-127; each thread also
//              converts one 16-byte chunk of the tokens' tile into shared
//              memory (the B operand, K-major, 128-byte swizzle); 3 stages
//   warp 1     allocates tensor memory; one thread issues the MMAs (M = 128,
//              N = NT, K = 16; A from TMEM, B from shared memory) into one
//              of two accumulator pairs, switching at every 1024-K chunk
//   warps 10-13 epilogue: thread = TMEM lane = weight row of each block;
//              adds each chunk into int32 registers and hands the finished
//              rows to the job (coalesced across the lanes of a warp)
// With resident tokens the eight converter warps first run the job's
// prologue, which writes the tokens into shared memory.  The producer needs
// neither the prologue nor the tensor memory, so the weight copies are in
// flight meanwhile.
#pragma once
#include <cstdint>
#include <cuda.h>
#include "dsa_ptx.cuh"

namespace dsa {

constexpr int kWtThreads = 448;
constexpr int kWtConv = 8;                          // converter warps (2..9)
constexpr int kWtEpi0 = 2 + kWtConv;                // first epilogue warp
constexpr int kWtRows = 128;                        // weight rows per MMA block (the MMA's M)
constexpr int kWtSuper = 2 * kWtRows;               // rows per super-block (one stage's box)
constexpr int kWtK = 128;                           // K columns per stage
constexpr int kWtUnit = 16;                         // rows: unit of a CTA's range and of a box's height
constexpr int kWtS8Max = 8, kWtS16 = 3;             // raw stages (at most; the launch picks), converted stages
constexpr int kWtChunk = 1024 / kWtK;               // stages per exact 1024-K chunk
constexpr uint32_t kWtRawW = kWtSuper * kWtK;       // 32 KB: the largest raw weight tile
constexpr uint32_t kWtBoxUnit = kWtUnit * kWtK;     // 2 KB: 16 rows of a tile
constexpr uint32_t kWtACols = kWtK / 2;             // one f16 A operand of a block: 64 columns
constexpr uint32_t kWtTmemCols = 512;

struct WtMaps {
  CUtensorMap w[kWtSuper / kWtUnit];  // b [N, K] int8, box {128 columns, 16 (i + 1) rows}
  CUtensorMap tok;                    // a [M, K] int8, box {128 columns, NT rows} (streamed tokens)
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
  // TMEM columns: the accumulators [buffer][block] of NT columns each, then
  // the A operands [stage][block] of 64 columns (4 NT + 384 <= 512)
  static constexpr uint32_t kACol0 = 4 * NT;
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

// Host: the weight maps over b [N, K] int8 (128-byte swizzle), one per box
// height 16, 32, .., 256 rows.  Needs dsa_internal.h.
inline bool wt_encode_weights(WtMaps& maps, const void* b, int N, int K) {
  const uint64_t st[1] = {static_cast<uint64_t>(K)};
  const uint64_t dims[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(N)};
  for (int i = 0; i < kWtSuper / kWtUnit; ++i) {
    const uint32_t box[2] = {static_cast<uint32_t>(kWtK), static_cast<uint32_t>((i + 1) * kWtUnit)};
    if (!encode_tmap(&maps.w[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, b, dims, st, box, 128)) return false;
  }
  return true;
}

// The rows [r0, r1) of b that CTA g of G owns: whole 16-row units, balanced.
__device__ __forceinline__ void wt_rows(int N, int g, int G, int& r0, int& r1) {
  const long long U = (N + kWtUnit - 1) / kWtUnit;
  r0 = static_cast<int>(U * g / G) * kWtUnit;
  r1 = min(N, static_cast<int>(U * (g + 1) / G) * kWtUnit);
}

// Job interface (a struct passed by value):
//   int M, N, K; uint32_t* err         tokens, weight rows, columns, error word
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
  uint8_t* s8 = smem;                                   // [ns8][weights | tokens], int8, swizzled
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
  const int nst = (K + kWtK - 1) / kWtK;                 // stages per super-block
  const int cpb = (nst + kWtChunk - 1) / kWtChunk;       // exact chunks per super-block
  const int nsb = r1 > r0 ? (r1 - r0 + kWtSuper - 1) / kWtSuper : 0;
  const int total = nsb * nst;
  // rows of super-block bi, and whether it has a second MMA block
  auto sb_rows = [&](int bi) { return min(kWtSuper, r1 - (r0 + bi * kWtSuper)); };

  if (tid == 0) {
    for (int i = 0; i < ns8; ++i) { mbar_init(&bars.full8[i], 1); mbar_init(&bars.empty8[i], kWtConv); }
    for (int i = 0; i < kWtS16; ++i) { mbar_init(&bars.full16[i], kWtConv); mbar_init(&bars.empty16[i], 1); }
    for (int i = 0; i < 2; ++i) { mbar_init(&bars.tfull[i], 1); mbar_init(&bars.tempty[i], 4); }
    mbar_init(&bars.mdrain, 1);
    mbar_init(&bars.tokready, kWtConv);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  volatile int* abort_v = &abort_flag;
  griddep_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // The weights are inputs of this call: their copies go out at once.
    if (lane == 0) {
      if (!kResident) griddep_wait();  // streamed tokens may come from the previous kernel
      int s = 0;
      bool ok = true;
      for (int bi = 0; bi < nsb && ok; ++bi) {
        const int row_b = r0 + bi * kWtSuper;
        const int units = (sb_rows(bi) + kWtUnit - 1) / kWtUnit;  // rows past N read as zero
        const CUtensorMap* wmap = &maps.w[units - 1];
        const uint32_t bytes = units * kWtBoxUnit + L::kRawTok;
        for (int k = 0; k < nst; ++k, ++s) {
          const int st = s % ns8;
          if (s >= ns8 && !mbar_wait(&bars.empty8[st], ((s / ns8) - 1) & 1, err, abort_v)) { ok = false; break; }
          uint8_t* dst = s8 + st * L::kStage8;
          mbar_arrive_expect_tx(&bars.full8[st], bytes);  // columns past K: zero fill
          tma_load_2d(dst, wmap, k * kWtK, row_b, &bars.full8[st]);
          if (!kResident) tma_load_2d(dst + kWtRawW, &maps.tok, k * kWtK, 0, &bars.full8[st]);
        }
      }
      // if a wait gave up, the last stages' copies land before the CTA leaves
      for (int i = s > ns8 ? s - ns8 : 0; i < s; ++i) mbar_drain(&bars.full8[i % ns8], (i / ns8) & 1);
    }
  } else {
    // Warps 1-13 wait for the tensor memory (the producer goes on without it).
    if (warp == 1) tmem_alloc(&tmem_base, kWtTmemCols);
    tc_fence_before();
    asm volatile("bar.sync 2, 416;" ::: "memory");
    tc_fence_after();
    const uint32_t tmem = tmem_base;
    if (warp == 1) {
      // ------------------------------------------------------- MMA issuer
      if (lane == 0) {
        const uint32_t idesc = idesc_f16(kWtRows, NT, kFmtF16, 0, 0);
        int s = 0, gc = 0;
        bool ok = true;
        for (int bi = 0; bi < nsb && ok; ++bi) {
          const int nmb = sb_rows(bi) > kWtRows ? 2 : 1;  // MMA blocks of the super-block
          for (int k = 0; k < nst; ++k, ++s) {
            const int st = s % kWtS16, buf = gc & 1;
            const bool first_of_chunk = (k % kWtChunk) == 0;
            // the accumulators are free once the epilogue has read their previous chunk
            if (first_of_chunk && gc >= 2 && !mbar_wait(&bars.tempty[buf], ((gc / 2) - 1) & 1, err, abort_v)) {
              ok = false;
              break;
            }
            if (!mbar_wait(&bars.full16[st], (s / kWtS16) & 1, err, abort_v)) { ok = false; break; }
            tc_fence_after();
            const uint32_t b_base = smem_u32(sB + st * L::kTileB);
            for (int mb = 0; mb < nmb; ++mb) {
              const uint32_t a_tmem = tmem + L::kACol0 + (st * 2 + mb) * kWtACols;
              const uint32_t d_tmem = tmem + (buf * 2 + mb) * NT;
#pragma unroll
              for (int kk = 0; kk < kWtK / 16; ++kk) {
                const uint64_t bd = smem_desc(b_base + (kk / 4) * L::kAtomB + (kk % 4) * 32, 16, 1024, kSwizzle128B);
                mma_ts(d_tmem, a_tmem + kk * 8, bd, idesc, (!first_of_chunk || kk > 0) ? 1u : 0u);
              }
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
      // -------------------------------------------------------- converters
      // Thread = rows r and 128 + r of the tile; a warp reaches the TMEM
      // lanes of its quarter (warp % 4), so r = 32 (warp % 4) + lane;
      // converter warps 2-5 take the tile's columns 0-63 (half 0), warps
      // 6-9 columns 64-127.
      const int r = (warp & 3) * 32 + lane;
      const int half = (warp - 2) / 4;
      const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16) + L::kACol0;
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
        const int nmb = sb_rows(s / nst) > kWtRows ? 2 : 1;
        if (!mbar_wait(&bars.full8[st8], (s / ns8) & 1, err, abort_v)) break;
        if (s >= kWtS16 && !mbar_wait(&bars.empty16[st16], ((s / kWtS16) - 1) & 1, err, abort_v)) break;
        tc_fence_after();
        const uint8_t* src = s8 + st8 * L::kStage8;
        // rows r and 128 + r, columns 64 half .. 64 half + 63 -> f16 pairs ->
        // TMEM: 16-byte chunk q of row x sits at q ^ (x & 7) (128-byte
        // swizzle), so a quarter warp reads 8 distinct bank groups.  Rows
        // past the CTA's range convert whatever the tile holds (their sums
        // are never read).
        for (int mb = 0; mb < nmb; ++mb) {
          const int x = mb * kWtRows + r;
          uint4 va[4];
#pragma unroll
          for (int q = 0; q < 4; ++q)
            va[q] = *reinterpret_cast<const uint4*>(src + x * 128 + (((4 * half + q) ^ (x & 7)) << 4));
          uint32_t fa[32];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            i8x4_to_f16x4(va[q].x, fa[8 * q + 0], fa[8 * q + 1]);
            i8x4_to_f16x4(va[q].y, fa[8 * q + 2], fa[8 * q + 3]);
            i8x4_to_f16x4(va[q].z, fa[8 * q + 4], fa[8 * q + 5]);
            i8x4_to_f16x4(va[q].w, fa[8 * q + 6], fa[8 * q + 7]);
          }
          tmem_st32(lane_base + (st16 * 2 + mb) * kWtACols + half * 32, fa);
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
      // --------------------------------------------------------- epilogue
      const int q4 = warp & 3;  // TMEM lane quarter of this warp
      const int row = q4 * 32 + lane;
      const uint32_t lane_base = tmem + (static_cast<uint32_t>(q4 * 32) << 16);
      bool ok = true;
      if (kResident && !mbar_wait(&bars.tokready, 0, err, abort_v)) ok = false;  // the tokens' scales
      float st[NT];
#pragma unroll
      for (int t = 0; t < NT; ++t) st[t] = t < M ? job.tok_scale(t) : 0.f;
      int gc = 0;
      for (int bi = 0; bi < nsb && ok; ++bi) {
        const int row_b = r0 + bi * kWtSuper;
        const int rows_b = sb_rows(bi);
        const bool two = rows_b > kWtRows;
        const float sn0 = row < rows_b ? job.row_scale(row_b + row) : 0.f;
        const float sn1 = kWtRows + row < rows_b ? job.row_scale(row_b + kWtRows + row) : 0.f;
        int tot0[NT], tot1[NT];
#pragma unroll
        for (int t = 0; t < NT; ++t) tot0[t] = tot1[t] = 0;
        for (int ch = 0; ch < cpb; ++ch, ++gc) {
          const int buf = gc & 1;
          if (!mbar_wait(&bars.tfull[buf], (gc / 2) & 1, err, abort_v)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int c0 = 0; c0 < NT; c0 += 16) {
            uint32_t v[16];
            tmem_ld16(lane_base + (buf * 2) * NT + c0, v);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 16; ++j) tot0[c0 + j] += __float2int_rn(__uint_as_float(v[j]));  // exact integers
            if (two) {
              tmem_ld16(lane_base + (buf * 2 + 1) * NT + c0, v);
              tmem_ld_wait();
#pragma unroll
              for (int j = 0; j < 16; ++j) tot1[c0 + j] += __float2int_rn(__uint_as_float(v[j]));
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars.tempty[buf]);
        }
        if (!ok) break;
        if (row < rows_b) {
#pragma unroll
          for (int t = 0; t < NT; ++t)
            if (t < M) job.put(t, row_b + row, tot0[t], st[t], sn0);
        }
        if (kWtRows + row < rows_b) {
#pragma unroll
          for (int t = 0; t < NT; ++t)
            if (t < M) job.put(t, row_b + kWtRows + row, tot1[t], st[t], sn1);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  job.tail(warp, lane);
  if (warp == 1) tmem_dealloc(tmem_base, kWtTmemCols);
}

}  // namespace dsa

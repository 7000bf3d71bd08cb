// Int8 GEMM with dequantisation on tcgen05 tensor cores, for activation
// blocks of more than 32 rows (prefill, batched decode).
//
//   c[m,n] = fp16( (sum_k a[m,k] * b[n,k]) * a_scale[m] * b_scale[n] )
//
// [V4-TileLang §Int8 General Matrix Multiplication] steps 1-4: an int32
// accumulation of int8 products, an fp32 dequantisation by the per-row
// scales, a cast to fp16.  sm_103a has no int8 tensor-core kind, so both
// operands are converted to f16 (exact for int8) and multiplied with
// kind::f16 MMAs accumulating in fp32.  A product is at most 2^14 in
// magnitude, so a sum of up to 1024 of them is an integer below 2^24 and
// every fp32 partial sum of it is exact; longer K is split into chunks of
// 1024 whose exact sums the epilogue adds in int32.  The result equals the
// int32 GEMM bit for bit.
//
// A persistent CTA per SM walks 128 x 128 output tiles (M rows of a, N
// rows of b):
//   warp 0     producer: 2-D TMA loads of the int8 tiles a[128 x 128] and
//              b[128 x 128] (128-byte swizzle, 16 KB boxes) into a 3-deep
//              ring
//   warps 2-5  converters: thread r converts row r of both tiles to f16:
//              the a row into tensor memory (the A operand of the MMA, so
//              shared memory carries only b's f16 tile), the b row K-major
//              with the 128-byte swizzle the MMA reads; 3 stages of each
//   warp 1     one thread issues the MMAs (M = N = 128, K = 16; A from
//              TMEM, B from shared memory) into one of two TMEM
//              accumulators, switching at every 1024-K chunk and every tile
//   warps 6-9  epilogue: thread = TMEM lane = output row; adds each
//              finished chunk into int32 registers, then dequantises and
//              stores the row's 128 fp16 values while the MMAs of the next
//              tile run
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include "dsa_internal.h"
#include "dsa_ptx.cuh"

namespace dsa {
namespace {

constexpr int kTcThreads = 320;
constexpr int kBM = 128, kBN = 128, kBK = 128;
constexpr int kS8 = 3, kS16 = 3;
constexpr int kChunkStages = 1024 / kBK;              // stages per exact 1024-K chunk
constexpr uint32_t kTile8 = kBM * kBK;                // 16 KB: one int8 operand tile (one TMA box)
constexpr uint32_t kStage8 = 2 * kTile8;              // a and b
constexpr uint32_t kAtomB = kBN * 128;                // 16 KB: 64 f16 columns of b (one 128-byte swizzle atom)
constexpr uint32_t kTileB16 = kBN * kBK * 2;          // 32 KB: b's f16 tile (a goes to TMEM)
constexpr size_t kTcSmem = 1024 + kS8 * kStage8 + kS16 * kTileB16;
constexpr uint32_t kAccCols = kBN;                    // one fp32 accumulator: 128 columns
constexpr uint32_t kACols = kBK / 2;                  // one f16 A stage in TMEM: 64 columns
constexpr uint32_t kTmemCols = 512;                   // 2 accumulators + 3 A stages = 448

struct __align__(8) TcBars {
  uint64_t full8[kS8], empty8[kS8], full16[kS16], empty16[kS16], tfull[2], tempty[2];
  uint64_t mdrain;  // the MMA thread's last commit
};

__global__ void __launch_bounds__(kTcThreads, 1)
    i8gemm_tc_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                     const float* __restrict__ a_scale, const float* __restrict__ b_scale, __half* __restrict__ c,
                     int M, int N, int K, uint32_t* err) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* s8 = smem;                     // [kS8][a 16 KB | b 16 KB], int8, 128-byte swizzle
  uint8_t* sB = smem + kS8 * kStage8;     // [kS16][2 atoms of 16 KB], f16, 128-byte swizzle
  __shared__ TcBars bars;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  __shared__ float sb_s[kBN];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tiles_n = (N + kBN - 1) / kBN, tiles_m = (M + kBM - 1) / kBM;
  const int n_tiles = tiles_n * tiles_m;
  const int nst = (K + kBK - 1) / kBK;                          // k stages per tile
  const int cpt = (nst + kChunkStages - 1) / kChunkStages;       // chunks per tile
  // this CTA's tiles: blockIdx.x, + gridDim.x, ... (consecutive CTAs take
  // neighbouring tiles, so the a and b tiles they share stay in L2)
  const int my_tiles = blockIdx.x < n_tiles ? (n_tiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  auto tile_mn = [&](int i, int& m0, int& n0) {
    const int t = blockIdx.x + i * gridDim.x;
    m0 = (t / tiles_n) * kBM;
    n0 = (t % tiles_n) * kBN;
  };

  if (tid == 0) {
    for (int i = 0; i < kS8; ++i) { mbar_init(&bars.full8[i], 1); mbar_init(&bars.empty8[i], 4); }
    for (int i = 0; i < kS16; ++i) { mbar_init(&bars.full16[i], 4); mbar_init(&bars.empty16[i], 1); }
    for (int i = 0; i < 2; ++i) { mbar_init(&bars.tfull[i], 1); mbar_init(&bars.tempty[i], 4); }
    mbar_init(&bars.mdrain, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(&tmem_base, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;
  const uint32_t a_col0 = 2 * kAccCols;
  volatile int* abort_v = &abort_flag;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_a)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_b)) : "memory");
      int s = 0;
      bool ok = true;
      for (int i = 0; i < my_tiles && ok; ++i) {
        int m0, n0;
        tile_mn(i, m0, n0);
        for (int k = 0; k < nst; ++k, ++s) {
          const int st = s % kS8;
          if (s >= kS8 && !mbar_wait(&bars.empty8[st], ((s / kS8) - 1) & 1, err, abort_v)) { ok = false; break; }
          uint8_t* dst = s8 + st * kStage8;
          mbar_arrive_expect_tx(&bars.full8[st], kStage8);  // columns past K, rows past M / N: zero fill
          tma_load_2d(dst, &tm_a, k * kBK, m0, &bars.full8[st]);
          tma_load_2d(dst + kTile8, &tm_b, k * kBK, n0, &bars.full8[st]);
        }
      }
      // if a wait gave up, the last stages' copies land before the CTA leaves
      for (int i = s > kS8 ? s - kS8 : 0; i < s; ++i) mbar_drain(&bars.full8[i % kS8], (i / kS8) & 1);
    }
  } else if (warp == 1) {
    // --------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_f16(kBM, kBN, kFmtF16, 0, 0);
      int s = 0, gc = 0;  // stage and chunk counters over all of this CTA's tiles
      bool ok = true;
      for (int i = 0; i < my_tiles && ok; ++i) {
        for (int k = 0; k < nst; ++k, ++s) {
          const int st = s % kS16, buf = gc & 1;
          const bool first_of_chunk = (k % kChunkStages) == 0;
          // the accumulator is free once the epilogue has drained its previous chunk
          if (first_of_chunk && gc >= 2 && !mbar_wait(&bars.tempty[buf], ((gc / 2) - 1) & 1, err, abort_v)) {
            ok = false;
            break;
          }
          if (!mbar_wait(&bars.full16[st], (s / kS16) & 1, err, abort_v)) { ok = false; break; }
          tc_fence_after();
          const uint32_t b_base = smem_u32(sB + st * kTileB16);
          const uint32_t a_tmem = tmem + a_col0 + st * kACols;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            const uint64_t bd = smem_desc(b_base + (kk / 4) * kAtomB + (kk % 4) * 32, 16, 1024, kSwizzle128B);
            mma_ts(tmem + buf * kAccCols, a_tmem + kk * 8, bd, idesc, (!first_of_chunk || kk > 0) ? 1u : 0u);
          }
          mma_commit(&bars.empty16[st]);
          if ((k % kChunkStages) == kChunkStages - 1 || k == nst - 1) {
            mma_commit(&bars.tfull[buf]);
            ++gc;
          }
        }
      }
      // every MMA issued has completed before the tensor memory is freed
      mma_commit(&bars.mdrain);
      mbar_drain(&bars.mdrain, 0);
    }
  } else if (warp < 6) {
    // ---------------------------------------------------------- converters
    // Thread = row r of both tiles; a warp reaches the TMEM lanes of its
    // quarter (warp % 4), so r = 32 (warp % 4) + lane.
    const int r = (warp & 3) * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16) + a_col0;
    const int total = my_tiles * nst;
    for (int s = 0; s < total; ++s) {
      const int st8 = s % kS8, st16 = s % kS16;
      if (!mbar_wait(&bars.full8[st8], (s / kS8) & 1, err, abort_v)) break;
      if (s >= kS16 && !mbar_wait(&bars.empty16[st16], ((s / kS16) - 1) & 1, err, abort_v)) break;
      tc_fence_after();
      const uint8_t* src = s8 + st8 * kStage8;
      // row r of an int8 tile: 16-byte chunk q at q ^ (r & 7) (128-byte
      // swizzle), so a quarter warp reads 8 distinct bank groups; four
      // chunks (64 columns) at a time
      const uint32_t a_st = lane_base + st16 * kACols;
      uint8_t* dB = sB + st16 * kTileB16;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint4 va[4], vb[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint32_t off = static_cast<uint32_t>(r * 128) + (((4 * h + q) ^ (r & 7)) << 4);
          va[q] = *reinterpret_cast<const uint4*>(src + off);
          vb[q] = *reinterpret_cast<const uint4*>(src + kTile8 + off);
        }
        // a row -> f16 pairs -> TMEM (A operand of the TS MMA)
        uint32_t fa[32];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          i8x4_to_f16x4(va[q].x, fa[8 * q + 0], fa[8 * q + 1]);
          i8x4_to_f16x4(va[q].y, fa[8 * q + 2], fa[8 * q + 3]);
          i8x4_to_f16x4(va[q].z, fa[8 * q + 4], fa[8 * q + 5]);
          i8x4_to_f16x4(va[q].w, fa[8 * q + 6], fa[8 * q + 7]);
        }
        tmem_st32(a_st + h * 32, fa);
        // b row -> f16, K-major with the 128-byte swizzle the MMA reads:
        // columns 64h .. 64h + 63 are atom h
        uint8_t* drow = dB + h * kAtomB;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t f[8];
          i8x4_to_f16x4(vb[q].x, f[0], f[1]);
          i8x4_to_f16x4(vb[q].y, f[2], f[3]);
          i8x4_to_f16x4(vb[q].z, f[4], f[5]);
          i8x4_to_f16x4(vb[q].w, f[6], f[7]);
          *reinterpret_cast<uint4*>(drow + sw128_off(r, 2 * q)) = make_uint4(f[0], f[1], f[2], f[3]);
          *reinterpret_cast<uint4*>(drow + sw128_off(r, 2 * q + 1)) = make_uint4(f[4], f[5], f[6], f[7]);
        }
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
    int gc = 0;
    bool ok = true;
    for (int i = 0; i < my_tiles && ok; ++i) {
      int m0, n0;
      tile_mn(i, m0, n0);
      const int m = m0 + row;
      asm volatile("bar.sync 1, 128;" ::: "memory");  // the previous tile's scales are read
      for (int j = tid - 192; j < kBN; j += 128) sb_s[j] = (n0 + j < N) ? __ldg(b_scale + n0 + j) : 0.f;
      asm volatile("bar.sync 1, 128;" ::: "memory");
      int tot[kBN];
#pragma unroll
      for (int j = 0; j < kBN; ++j) tot[j] = 0;
      for (int ch = 0; ch < cpt; ++ch, ++gc) {
        const int buf = gc & 1;
        if (!mbar_wait(&bars.tfull[buf], (gc / 2) & 1, err, abort_v)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int c0 = 0; c0 < kBN; c0 += 32) {
          uint32_t v[32];
          tmem_ld32(lane_base + buf * kAccCols + c0, v);
          tmem_ld_wait();
#pragma unroll
          for (int k = 0; k < 32; ++k) tot[c0 + k] += __float2int_rn(__uint_as_float(v[k]));  // exact integers
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.tempty[buf]);
      }
      // the four epilogue warps leave together (a warp that gave up must not
      // leave the others waiting at the named barrier of the next tile)
      uint32_t all_ok;
      asm volatile("{\n.reg .pred p, q;\nsetp.ne.b32 p, %1, 0;\nbar.red.and.pred q, 1, 128, p;\nselp.u32 %0, 1, 0, q;\n}"
                   : "=r"(all_ok) : "r"(static_cast<uint32_t>(ok && !*abort_v)) : "memory");
      if (!all_ok) break;
      if (m < M) {
        const float sa = __ldg(a_scale + m);
        __half* crow = c + static_cast<size_t>(m) * N + n0;
        const bool vec = (n0 + kBN <= N) && (N % 8 == 0);
#pragma unroll
        for (int j0 = 0; j0 < kBN; j0 += 8) {
          __half h[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) h[k] = __float2half_rn(static_cast<float>(tot[j0 + k]) * sa * sb_s[j0 + k]);
          if (vec) {
            *reinterpret_cast<uint4*>(crow + j0) = *reinterpret_cast<const uint4*>(h);
          } else {
#pragma unroll
            for (int k = 0; k < 8; ++k)
              if (n0 + j0 + k < N) crow[j0 + k] = h[k];
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

int launch_int8_gemm_tc(const dsa_int8_gemm_args& a, cudaStream_t s) {
  uint32_t* err = error_word();
  if (!err) return DSA_ERR_CUDA;
  // int8 [rows, K] tiles of 128 columns x 128 rows, 128-byte swizzle
  alignas(64) CUtensorMap tm_a, tm_b;
  const uint64_t st[1] = {static_cast<uint64_t>(a.K)};
  const uint64_t da[2] = {static_cast<uint64_t>(a.K), static_cast<uint64_t>(a.M)};
  const uint64_t db[2] = {static_cast<uint64_t>(a.K), static_cast<uint64_t>(a.N)};
  const uint32_t box_a[2] = {kBK, kBM}, box_b[2] = {kBK, kBN};
  if (!encode_tmap(&tm_a, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, a.a, da, st, box_a, 128) ||
      !encode_tmap(&tm_b, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, a.b, db, st, box_b, 128))
    return DSA_ERR_CUDA;
  cudaError_t e = cudaFuncSetAttribute(i8gemm_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kTcSmem));
  if (e != cudaSuccess) return DSA_ERR_CUDA;
  const long long tiles = static_cast<long long>((a.N + kBN - 1) / kBN) * ((a.M + kBM - 1) / kBM);
  if (tiles > 0x7fffffffLL) return DSA_ERR_UNSUPPORTED;
  const int grid = static_cast<int>(tiles < sm_count() ? tiles : sm_count());  // persistent: one CTA per SM
  i8gemm_tc_kernel<<<grid, kTcThreads, kTcSmem, s>>>(tm_a, tm_b, a.a_scale, a.b_scale,
                                                      reinterpret_cast<__half*>(a.c), a.M, a.N, a.K, err);
  return cuda_status(cudaGetLastError());
}

}  // namespace dsa

// Lightning Indexer scores on tcgen05 tensor cores.
//
//   I[t,s] = ks[s] * sum_h (w[t,h] * qs[t,h]) * ReLU(q[t,h,:] . K[s,:])
//
// [V3.2-PyPTO §Lightning Indexer] scores the int8 indexer q against the C8
// key cache (4 batch x 64K keys = 2048 key blocks of 128 on the NPU) and
// keeps only the per-query TopK.  Here one work item is a tile of 128 keys
// of one sequence against a group of G query tokens of that sequence
// (N = G * H_I query rows, padded to a multiple of 16):
//
//   D[128 keys, N rows] = K_tile[128, d_I] . Q[N, d_I]^T
//
// with the keys as the MMA's M dimension, so that the head reduction of the
// score is a per-thread loop over TMEM columns (thread = key) instead of a
// cross-lane reduction.  sm_103a has no int8 tensor-core kind, so both
// operands are converted to f16, which is exact for int8 and keeps every
// fp32 partial sum an exact integer (|sum| <= 128 * 127 * 128 < 2^24): the
// dots equal the int32 ones bit for bit.
//
// Warp roles of the persistent CTA (one per SM):
//   warp 8     producer: cp.async.bulk of the raw int8 key tile (16 KB)
//   warps 4-7  converters: int8 -> f16 into the 128B-swizzled K-major
//              layout the MMA reads; also stage Q for each new group
//   warp 9     one thread issues tcgen05.mma into a double-buffered TMEM
//              accumulator and commits to mbarriers
//   warps 0-3  epilogue: tcgen05.ld of the accumulator row of its key,
//              ReLU + head-weighted sum per token, times ks[s], causal mask,
//              and the fp32 score row store (coalesced over keys)
// The per-head scores [T, H_I, L] never leave the SM; only I[t, s] (fp32,
// [T, max_L]) is written, for the top-k pass.
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include "dsa_internal.h"
#include "dsa_ptx.cuh"

namespace dsa {
namespace {

constexpr int kTileKeys = 128;
constexpr int kStages8 = 4;   // raw int8 key tiles in flight
constexpr int kStages16 = 2;  // converted f16 tiles
constexpr int kThreads = 320;
constexpr int kMaxG = 32;     // tokens per group
constexpr int kCoef = 256;    // max query rows (N) of a group

struct IdxParams {
  int T, n_q, H_I, d_I, G, N, groups_per_seq, n_groups, n_tiles, max_L;
  const int8_t* q;
  const __half* q_scale;
  const float* w;
  const int8_t* k_cache;
  const __half* k_scale;
  const int32_t* block_table;
  int block_size, max_blocks;
  const int32_t* pos;
  float* scores;
  int64_t ld;
  uint32_t* err;
};

struct Group {
  int b, t0, ntok, maxpos;
};

__device__ __forceinline__ Group group_of(const IdxParams& P, int g) {
  Group G;
  G.b = g / P.groups_per_seq;
  const int gj = g % P.groups_per_seq;
  G.t0 = G.b * P.n_q + gj * P.G;
  G.ntok = min(P.G, P.n_q - gj * P.G);
  int m = -1;
  for (int i = 0; i < G.ntok; ++i) m = max(m, __ldg(P.pos + G.t0 + i));
  G.maxpos = min(m, P.max_L - 1);
  return G;
}

// Next active item (a tile that holds at least one visible key) of this
// CTA at or after item i; returns n_items when none is left.
__device__ __forceinline__ int next_item(const IdxParams& P, int i, int& g_cache, int& maxpos_cache) {
  const int n_items = P.n_groups * P.n_tiles;
  for (; i < n_items; i += gridDim.x) {
    const int g = i / P.n_tiles, j = i % P.n_tiles;
    if (g != g_cache) {
      g_cache = g;
      maxpos_cache = group_of(P, g).maxpos;
    }
    if (j * kTileKeys <= maxpos_cache) return i;
  }
  return n_items;
}

__device__ __forceinline__ int64_t key_row(const IdxParams& P, int b, int s) {
  if (P.block_table == nullptr) return static_cast<int64_t>(b) * P.max_L + s;
  const int blk = __ldg(P.block_table + static_cast<size_t>(b) * P.max_blocks + s / P.block_size);
  return static_cast<int64_t>(blk) * P.block_size + s % P.block_size;
}

struct __align__(8) Bars {
  uint64_t full8[kStages8], empty8[kStages8];
  uint64_t full16[kStages16], empty16[kStages16];
  uint64_t qfull, qempty;
  uint64_t tfull[2], tempty[2];
};

template <int HI>
__global__ void __launch_bounds__(kThreads, 1) indexer_kernel(const IdxParams P) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int d_I = P.d_I;
  const int N = P.N;
  const uint32_t tile8_bytes = kTileKeys * d_I;        // int8 tile
  const uint32_t tile16_bytes = kTileKeys * d_I * 2;   // f16 swizzled tile
  uint8_t* s8 = smem;                                  // [kStages8][tile8]
  uint8_t* s16 = s8 + kStages8 * tile8_bytes;          // [kStages16][tile16]
  uint8_t* sQ = s16 + kStages16 * tile16_bytes;        // [d_I/64 atoms][N rows][128 B]
  __shared__ Bars bars;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  __shared__ float coef[kCoef];
  __shared__ int tok_pos[kMaxG];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // Accumulator buffers start on 32-column boundaries so that every 32-column
  // load stays inside its own buffer.
  const int acc_stride = (N + 31) & ~31;
  const uint32_t tmem_cols = (2 * acc_stride <= 64) ? 64 : (2 * acc_stride <= 128) ? 128 : (2 * acc_stride <= 256) ? 256 : 512;

  if (tid == 0) {
    for (int i = 0; i < kStages8; ++i) { mbar_init(&bars.full8[i], 1); mbar_init(&bars.empty8[i], 4); }
    for (int i = 0; i < kStages16; ++i) { mbar_init(&bars.full16[i], 4); mbar_init(&bars.empty16[i], 1); }
    mbar_init(&bars.qfull, 4);
    mbar_init(&bars.qempty, 1);
    for (int i = 0; i < 2; ++i) { mbar_init(&bars.tfull[i], 1); mbar_init(&bars.tempty[i], 4); }
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(&tmem_base, tmem_cols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  griddep_launch_dependents();
  griddep_wait();  // q, w, qs and the new cache rows come from the prolog
  const uint32_t tmem = tmem_base;
  volatile int* abort_v = &abort_flag;

  int g_cache = -1, maxpos_cache = -1;
  if (warp == 8) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int st = 0;
      uint32_t ph = 0;
      for (int i = next_item(P, blockIdx.x, g_cache, maxpos_cache); i < P.n_groups * P.n_tiles;
           i = next_item(P, i + gridDim.x, g_cache, maxpos_cache)) {
        const int g = i / P.n_tiles, j = i % P.n_tiles;
        const int b = g / P.groups_per_seq;
        if (!mbar_wait(&bars.empty8[st], ph ^ 1, P.err, abort_v)) break;
        uint8_t* dst = s8 + st * tile8_bytes;
        const int s0 = j * kTileKeys;
        if (P.block_table == nullptr) {
          mbar_arrive_expect_tx(&bars.full8[st], tile8_bytes);
          bulk_g2s(dst, P.k_cache + (static_cast<int64_t>(b) * P.max_L + s0) * d_I, tile8_bytes, &bars.full8[st]);
        } else {
          const int bs = P.block_size;
          const int span = bs < kTileKeys ? bs : kTileKeys;  // keys per copy
          int64_t rows[kTileKeys / 8];
          uint32_t bytes = 0;
          int n_copies = 0;
          for (int k = 0; k < kTileKeys && s0 + k <= maxpos_cache; k += span) {
            const int64_t row = key_row(P, b, s0 + k);
            rows[n_copies++] = row;
            if (row >= 0) bytes += span * d_I;
            else atomicOr(P.err, kErrBadIndex);
          }
          mbar_arrive_expect_tx(&bars.full8[st], bytes);
          for (int c = 0; c < n_copies; ++c)
            if (rows[c] >= 0) bulk_g2s(dst + c * span * d_I, P.k_cache + rows[c] * d_I, span * d_I, &bars.full8[st]);
        }
        if (++st == kStages8) { st = 0; ph ^= 1; }
      }
    }
  } else if (warp >= 4 && warp < 8) {
    // ---------------------------------------------------------- converters
    const int ct = tid - 128;  // 0..127
    int st8 = 0, st16 = 0;
    uint32_t ph8 = 0, ph16 = 0, qph = 0;
    int cur_g = -1;
    bool first_group = true;
    const int chunks = d_I / 16;  // 16-byte int8 chunks per row
    for (int i = next_item(P, blockIdx.x, g_cache, maxpos_cache); i < P.n_groups * P.n_tiles;
         i = next_item(P, i + gridDim.x, g_cache, maxpos_cache)) {
      const int g = i / P.n_tiles;
      if (g != cur_g) {
        cur_g = g;
        if (!first_group && !mbar_wait(&bars.qempty, qph, P.err, abort_v)) break;
        if (!first_group) qph ^= 1;
        first_group = false;
        const Group G = group_of(P, g);
        const int rows_real = G.ntok * P.H_I;
        for (int task = ct; task < N * chunks; task += 128) {
          const int n = task / chunks, c = task % chunks;
          uint4 v = make_uint4(0, 0, 0, 0);
          if (n < rows_real) {
            const int8_t* src = P.q + (static_cast<size_t>(G.t0) * P.H_I + n) * d_I + c * 16;
            v = __ldg(reinterpret_cast<const uint4*>(src));
          }
          uint32_t f[8];
          i8x4_to_f16x4(v.x, f[0], f[1]);
          i8x4_to_f16x4(v.y, f[2], f[3]);
          i8x4_to_f16x4(v.z, f[4], f[5]);
          i8x4_to_f16x4(v.w, f[6], f[7]);
          uint8_t* atom = sQ + (c / 4) * (N * 128);
          const int cc = (c % 4) * 2;
          *reinterpret_cast<uint4*>(atom + sw128_off(n, cc)) = make_uint4(f[0], f[1], f[2], f[3]);
          *reinterpret_cast<uint4*>(atom + sw128_off(n, cc + 1)) = make_uint4(f[4], f[5], f[6], f[7]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.qfull);
      }
      if (!mbar_wait(&bars.full8[st8], ph8, P.err, abort_v)) break;
      if (!mbar_wait(&bars.empty16[st16], ph16 ^ 1, P.err, abort_v)) break;
      const uint8_t* src = s8 + st8 * tile8_bytes;
      uint8_t* dst = s16 + st16 * tile16_bytes;
      for (int task = ct; task < kTileKeys * chunks; task += 128) {
        const int r = task / chunks, c = task % chunks;
        const uint4 v = *reinterpret_cast<const uint4*>(src + r * d_I + c * 16);
        uint32_t f[8];
        i8x4_to_f16x4(v.x, f[0], f[1]);
        i8x4_to_f16x4(v.y, f[2], f[3]);
        i8x4_to_f16x4(v.z, f[4], f[5]);
        i8x4_to_f16x4(v.w, f[6], f[7]);
        uint8_t* atom = dst + (c / 4) * (kTileKeys * 128);
        const int cc = (c % 4) * 2;
        *reinterpret_cast<uint4*>(atom + sw128_off(r, cc)) = make_uint4(f[0], f[1], f[2], f[3]);
        *reinterpret_cast<uint4*>(atom + sw128_off(r, cc + 1)) = make_uint4(f[4], f[5], f[6], f[7]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&bars.full16[st16]);
        mbar_arrive(&bars.empty8[st8]);
      }
      if (++st8 == kStages8) { st8 = 0; ph8 ^= 1; }
      if (++st16 == kStages16) { st16 = 0; ph16 ^= 1; }
    }
  } else if (warp == 9) {
    // -------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_f16(128, N, kFmtF16, 0, 0);
      int st16 = 0, acc = 0;
      uint32_t ph16 = 0, qph = 0, aph = 0;
      int cur_g = -1;
      const int n_items = P.n_groups * P.n_tiles;
      int i = next_item(P, blockIdx.x, g_cache, maxpos_cache);
      while (i < n_items) {
        const int g = i / P.n_tiles;
        const int nxt = next_item(P, i + gridDim.x, g_cache, maxpos_cache);
        if (g != cur_g) {
          cur_g = g;
          if (!mbar_wait(&bars.qfull, qph, P.err, abort_v)) break;
          qph ^= 1;
        }
        if (!mbar_wait(&bars.full16[st16], ph16, P.err, abort_v)) break;
        if (!mbar_wait(&bars.tempty[acc], aph ^ 1, P.err, abort_v)) break;
        tc_fence_after();
        const uint32_t a_base = smem_u32(s16 + st16 * tile16_bytes);
        const uint32_t b_base = smem_u32(sQ);
        const uint32_t d_tmem = tmem + acc * acc_stride;
        for (int kk = 0; kk < d_I / 16; ++kk) {
          const uint64_t ad = smem_desc(a_base + (kk / 4) * (kTileKeys * 128) + (kk % 4) * 32, 16, 1024, kSwizzle128B);
          const uint64_t bd = smem_desc(b_base + (kk / 4) * (N * 128) + (kk % 4) * 32, 16, 1024, kSwizzle128B);
          mma_ss(d_tmem, ad, bd, idesc, kk > 0 ? 1u : 0u);
        }
        mma_commit(&bars.empty16[st16]);
        mma_commit(&bars.tfull[acc]);
        const bool group_ends = (nxt >= n_items) || (nxt / P.n_tiles != g);
        if (group_ends) mma_commit(&bars.qempty);
        if (++st16 == kStages16) { st16 = 0; ph16 ^= 1; }
        if (++acc == 2) { acc = 0; aph ^= 1; }
        i = nxt;
      }
    }
  } else if (warp < 4) {
    // ---------------------------------------------------------- epilogue
    int acc = 0;
    uint32_t aph = 0;
    int cur_g = -1;
    Group G{};
    const int r = warp * 32 + lane;  // key within the tile = TMEM lane
    for (int i = next_item(P, blockIdx.x, g_cache, maxpos_cache); i < P.n_groups * P.n_tiles;
         i = next_item(P, i + gridDim.x, g_cache, maxpos_cache)) {
      const int g = i / P.n_tiles, j = i % P.n_tiles;
      if (g != cur_g) {
        cur_g = g;
        G = group_of(P, g);
        asm volatile("bar.sync 1, 128;" ::: "memory");
        for (int n = tid; n < kCoef; n += 128) {
          const int gi = n / HI, h = n % HI;
          float c = 0.f;
          if (gi < G.ntok && h < P.H_I) {
            const int t = G.t0 + gi;
            c = __ldg(P.w + static_cast<size_t>(t) * P.H_I + h) *
                __half2float(__ldg(P.q_scale + static_cast<size_t>(t) * P.H_I + h));
          }
          coef[n] = c;
        }
        for (int gi = tid; gi < kMaxG; gi += 128) tok_pos[gi] = (gi < G.ntok) ? __ldg(P.pos + G.t0 + gi) : -1;
        asm volatile("bar.sync 1, 128;" ::: "memory");
      }
      if (!mbar_wait(&bars.tfull[acc], aph, P.err, abort_v)) break;
      tc_fence_after();
      const int s = j * kTileKeys + r;
      float ks = 0.f;
      if (s <= G.maxpos) {
        const int64_t row = key_row(P, G.b, s);
        if (row >= 0) ks = __half2float(__ldg(P.k_scale + row));
      }
      const uint32_t lane_addr = tmem + (static_cast<uint32_t>(warp * 32) << 16) + acc * acc_stride;
      const float ninf = -__int_as_float(0x7f800000);
      // Column n = gi * HI + h of the accumulator is token gi, head h.
      if (HI >= 32) {
        for (int gi = 0; gi < G.ntok; ++gi) {
          float sacc = 0.f;
#pragma unroll
          for (int c = 0; c < HI / 32; ++c) {
            uint32_t v[32];
            tmem_ld32(lane_addr + gi * HI + c * 32, v);
            tmem_ld_wait();
            const float* cf = coef + gi * HI + c * 32;
#pragma unroll
            for (int k = 0; k < 32; ++k) sacc = fmaf(cf[k], fmaxf(__uint_as_float(v[k]), 0.f), sacc);
          }
          P.scores[static_cast<size_t>(G.t0 + gi) * P.ld + s] = (s <= tok_pos[gi]) ? sacc * ks : ninf;
        }
      } else {
        constexpr int kTokPerChunk = HI >= 32 ? 1 : 32 / HI;
        const int n_chunks = (G.ntok * HI + 31) / 32;
        for (int cc = 0; cc < n_chunks; ++cc) {
          uint32_t v[32];
          tmem_ld32(lane_addr + cc * 32, v);
          tmem_ld_wait();
#pragma unroll
          for (int u = 0; u < kTokPerChunk; ++u) {
            const int gi = cc * kTokPerChunk + u;
            float sacc = 0.f;
#pragma unroll
            for (int k = 0; k < HI; ++k)
              sacc = fmaf(coef[cc * 32 + u * HI + k], fmaxf(__uint_as_float(v[u * HI + k]), 0.f), sacc);
            if (gi < G.ntok)
              P.scores[static_cast<size_t>(G.t0 + gi) * P.ld + s] = (s <= tok_pos[gi]) ? sacc * ks : ninf;
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.tempty[acc]);
      if (++acc == 2) { acc = 0; aph ^= 1; }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, tmem_cols);
}

// Plain SIMT int32 dots for bit-exact checks of the contraction.
__global__ void dots_kernel(const IdxParams P, int32_t* dots) {
  const int t = blockIdx.y;
  const int s = blockIdx.x * blockDim.x + threadIdx.x;
  if (s >= P.max_L) return;
  const int b = t / P.n_q;
  const int64_t row = key_row(P, b, s);
  if (row < 0) return;
  const int8_t* k = P.k_cache + row * P.d_I;
  for (int h = 0; h < P.H_I; ++h) {
    const int8_t* q = P.q + (static_cast<size_t>(t) * P.H_I + h) * P.d_I;
    int acc = 0;
    for (int d = 0; d < P.d_I; d += 4)
      acc = __dp4a(*reinterpret_cast<const int*>(k + d), *reinterpret_cast<const int*>(q + d), acc);
    dots[(static_cast<size_t>(t) * P.H_I + h) * P.max_L + s] = acc;
  }
}

IdxParams make_params(const dsa_topk_args& a, float* scores, int64_t ld) {
  IdxParams P{};
  P.T = a.T; P.n_q = a.n_q; P.H_I = a.H_I; P.d_I = a.d_I; P.max_L = a.max_L;
  P.G = a.H_I >= 128 ? 1 : (128 / a.H_I < a.n_q ? 128 / a.H_I : a.n_q);
  if (P.G > kMaxG) P.G = kMaxG;
  P.N = static_cast<int>(round_up(static_cast<size_t>(P.G) * a.H_I, 16));
  P.groups_per_seq = (a.n_q + P.G - 1) / P.G;
  P.n_groups = a.B * P.groups_per_seq;
  P.n_tiles = a.max_L / kTileKeys;
  P.q = a.q; P.q_scale = reinterpret_cast<const __half*>(a.q_scale); P.w = a.w;
  P.k_cache = a.k_cache; P.k_scale = reinterpret_cast<const __half*>(a.k_scale);
  P.block_table = a.block_table; P.block_size = a.block_size; P.max_blocks = a.max_blocks;
  P.pos = a.pos; P.scores = scores; P.ld = ld;
  P.err = error_word();
  return P;
}

template <int HI>
cudaError_t launch_hi(const IdxParams& P, cudaStream_t s) {
  const size_t smem = 1024 + static_cast<size_t>(kStages8) * kTileKeys * P.d_I +
                      static_cast<size_t>(kStages16) * kTileKeys * P.d_I * 2 + static_cast<size_t>(P.N) * P.d_I * 2;
  cudaError_t e = cudaFuncSetAttribute(indexer_kernel<HI>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const long long items = static_cast<long long>(P.n_groups) * P.n_tiles;
  const int grid = static_cast<int>(items < sm_count() ? items : sm_count());
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, indexer_kernel<HI>, P);
}

}  // namespace

int launch_indexer(const dsa_topk_args& a, float* scores, cudaStream_t s) {
  const IdxParams P = make_params(a, scores, a.max_L);
  if (!P.err) return DSA_ERR_CUDA;
  cudaError_t e;
  switch (a.H_I) {
    case 4: e = launch_hi<4>(P, s); break;
    case 8: e = launch_hi<8>(P, s); break;
    case 16: e = launch_hi<16>(P, s); break;
    case 32: e = launch_hi<32>(P, s); break;
    case 64: e = launch_hi<64>(P, s); break;
    case 128: e = launch_hi<128>(P, s); break;
    default: return DSA_ERR_UNSUPPORTED;
  }
  return cuda_status(e);
}

int launch_indexer_dots(const dsa_topk_args& a, int32_t* dots, cudaStream_t s) {
  const IdxParams P = make_params(a, nullptr, a.max_L);
  dim3 grid((a.max_L + 127) / 128, a.T);
  dots_kernel<<<grid, 128, 0, s>>>(P, dots);
  return cuda_status(cudaGetLastError());
}

}  // namespace dsa

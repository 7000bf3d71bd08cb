// MLA Prolog: the query latent and the latent KV row of each token, the
// quantised query latent, and the attention query with W_UK absorbed.
//
// [V3.2-PyPTO §Deepseek Indexer Attention] names the MLA Prolog as the first
// of the operator's four parts: it hands q_lora (int8, one fp16 scale per
// token) to the Indexer Prolog and q [T, H, 576] plus the latent KV rows
// [576] to the sparse attention.  At decode sizes (T <= 32 tokens) each of
// its three products is a weight stream, so each kernel is laid out for
// weight bandwidth:
//
//   mla_down    x . [w_dq; w_dkv]^T, split over D_x.  A CTA owns one
//               128-channel row block and a slice of D_x, pulls 64-column
//               atoms of the weights and of x through a 4-stage TMA ring
//               (128-byte swizzle), multiplies on the tensor core (bf16,
//               M = 128 channels, N = tokens padded to 16 or 32, fp32 in
//               tensor memory) and adds its partial sums into the fp32
//               workspace.
//   mla_up      q_lora . w_uq^T as exact int32 sums on the tensor-core
//               weight stream (w8tc.cuh): one CTA per SM over a contiguous
//               range of w_uq's rows.  Each CTA normalises the query latent
//               (RMSNorm) and quantises it per token from the sums (CTA 0
//               also writes q_lora), dequantises its rows' sums into the
//               workspace, and writes the latent-cache rows of some tokens
//               (RMSNorm of the KV latent, rotated rotary part).
//   mla_absorb  q[:, h, c] = sum_n u_nope[:, h, n] w_uk[h, n, c]: one CTA per
//               (head, half of the 512 latent dims), whose 64 KB of w_uk
//               arrive by bulk copies issued before it waits for mla_up; the
//               second half also rotates the head's rotary dims into
//               q[:, h, 512:576]; the CTAs clear mla_down's sums for the
//               next call.
// mla_up and mla_absorb start early (programmatic dependent launch) and
// fetch their weights while the kernel before them finishes.
#include <algorithm>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include "dsa_internal.h"
#include "dsa_ptx.cuh"
#include "w8tc.cuh"

namespace dsa {
namespace {

constexpr int kDc = 512, kDn = 128, kDr = 64;  // latent, no-position, rotary dims
constexpr int kDkv = kDc + kDr;                // latent KV row (576)
constexpr int kDh = kDn + kDr;                 // up-projected dims per head (192)

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// ------------------------------------------------------------------ down
constexpr int kDownThreads = 128;
constexpr int kDownStages = 4;
constexpr uint32_t kDownAtomW = 128 * 128;  // [128 rows][64 bf16]

struct DownParams {
  int T, K_q, D_x, n_rb_q, n_rb, per;
  float* sums;  // workspace: [T, K_q + 576] fp32, zero on entry
  uint32_t* err;
};

template <int NX>
__global__ void __launch_bounds__(kDownThreads, 1)
    mla_down_kernel(const __grid_constant__ DownParams P, const __grid_constant__ CUtensorMap tm_wdq,
                    const __grid_constant__ CUtensorMap tm_wdkv, const __grid_constant__ CUtensorMap tm_x) {
  constexpr uint32_t kStage = kDownAtomW + NX * 128;  // weight atom + x atom (multiple of 1024)
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t full[kDownStages], empty[kDownStages], mdone;
  __shared__ int abort_flag;
  __shared__ uint32_t tmem_base;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rb = blockIdx.x % P.n_rb, split = blockIdx.x / P.n_rb;
  const int a0 = split * P.per;
  const int na = min(P.per, P.D_x / 64 - a0);  // >= 1: the grid has no empty split
  const bool is_q = rb < P.n_rb_q;
  const CUtensorMap* tw = is_q ? &tm_wdq : &tm_wdkv;
  const int wrow = (is_q ? rb : rb - P.n_rb_q) * 128;  // first row of the block in its weight
  const int nrows = is_q ? 128 : min(128, kDkv - wrow);
  const int C = P.K_q + kDkv;
  if (tid == 0) {
    for (int s = 0; s < kDownStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(&mdone, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(&tmem_base, 32);  // D: 128 lanes x NX (<= 32) fp32 columns
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;
  griddep_launch_dependents();
  griddep_wait();
  if (tid == 0) {
    // producer: atom i of this slice into stage i % kDownStages, once the
    // MMAs that read the stage's previous atom have completed
    int issued = 0;
    for (int i = 0; i < na; ++i) {
      const int s = i % kDownStages;
      if (i >= kDownStages && !mbar_wait(&empty[s], ((i / kDownStages) - 1) & 1, P.err, &abort_flag)) break;
      uint8_t* st = smem + s * kStage;
      const int xc = (a0 + i) * 64;
      mbar_arrive_expect_tx(&full[s], kStage);
      tma_load_2d(st, tw, xc, wrow, &full[s]);  // rows past the weight read as zero
      tma_load_2d(st + kDownAtomW, &tm_x, xc, 0, &full[s]);  // tokens past T read as zero
      issued = i + 1;
    }
    // if a wait gave up, the last stages' copies land before the CTA leaves
    for (int i = issued > kDownStages ? issued - kDownStages : 0; i < issued; ++i)
      mbar_drain(&full[i % kDownStages], (i / kDownStages) & 1);
  } else if (tid == 32) {
    // MMA issuer: D (+)= W_atom [128 x 64] . X_atom^T [64 x NX], K = 16 per MMA
    const uint32_t idesc = idesc_f16(128, NX, kFmtBF16, 0, 0);
    for (int i = 0; i < na; ++i) {
      const int s = i % kDownStages;
      if (!mbar_wait(&full[s], (i / kDownStages) & 1, P.err, &abort_flag)) break;
      tc_fence_after();
      const uint32_t a = smem_u32(smem + s * kStage), b = a + kDownAtomW;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        mma_ss(tmem, smem_desc(a + kk * 32, 16, 1024, kSwizzle128B), smem_desc(b + kk * 32, 16, 1024, kSwizzle128B),
               idesc, (i > 0 || kk > 0) ? 1u : 0u);
      mma_commit(&empty[s]);
    }
    mma_commit(&mdone);
  }
  __syncwarp();
  // a CTA whose tiles never arrived adds nothing (its error is recorded); a
  // wait that gave up still lets the MMAs finish before TMEM is read or freed
  bool ok = mbar_wait(&mdone, 0, P.err, &abort_flag);
  if (!ok) mbar_drain(&mdone, 0);
  ok = ok && !*static_cast<volatile int*>(&abort_flag);
  __syncwarp();
  tc_fence_after();
  uint32_t v[32];
  tmem_ld32(tmem + (static_cast<uint32_t>(warp * 32) << 16), v);
  tmem_ld_wait();
  const int r = warp * 32 + lane;  // TMEM lane = row of the block = channel
  if (ok && r < nrows) {
    float* dst = P.sums + rb * 128 + r;
#pragma unroll
    for (int t = 0; t < NX; ++t)
      if (t < P.T) atomicAdd(dst + static_cast<size_t>(t) * C, __uint_as_float(v[t]));
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 32);
}

// -------------------------------------------------------------------- up
constexpr int kMaxQv = 2048 / 128;  // float4 per lane of a query-latent row

struct UpParams {
  int T, H, K_q, max_pos;
  int interleaved;
  float eps;
  const float* sums;  // workspace: [T, K_q + 576] from mla_down
  const float* gamma_q;
  const float* gamma_kv;
  const int8_t* w_uq;  // [H * 192, K_q]
  const __half* w_uq_scale;
  const int32_t* pos;
  const float* rope_cos;
  const float* rope_sin;
  int8_t* q_lora;
  __half* q_lora_scale;
  float* up;  // workspace: [T, H * 192] dequantised q_lora . w_uq^T
  __nv_bfloat16* kv_cache;
  const int64_t* slot;
  int64_t cache_rows;
  uint32_t* err;
};

// One warp, token t: c_q = RMSNorm(sums[t, :K_q]) * gamma_q, quantised per
// token.  The codes go to sA (row t, K_q bytes) and, in CTA 0, to q_lora;
// returns the fp16 scale as fp32.  Every CTA computes the same codes: the
// arithmetic is the same sequence of fp32 operations on the same sums.
__device__ __forceinline__ float quant_latent(const UpParams& P, int t, int lane, int8_t* sA, bool write_out) {
  const float* row = P.sums + static_cast<size_t>(t) * (P.K_q + kDkv);
  const int nj = P.K_q / 128;
  float4 v[kMaxQv];
  float ss = 0.f;
#pragma unroll
  for (int j = 0; j < kMaxQv; ++j) {
    if (j < nj) {
      v[j] = __ldcg(reinterpret_cast<const float4*>(row + 128 * j + 4 * lane));
      ss += v[j].x * v[j].x + v[j].y * v[j].y + v[j].z * v[j].z + v[j].w * v[j].w;
    }
  }
  const float rq = 1.0f / sqrtf(warp_sum(ss) / static_cast<float>(P.K_q) + P.eps);
  float amax = 0.f;
#pragma unroll
  for (int j = 0; j < kMaxQv; ++j) {
    if (j < nj) {
      const float4 g = __ldg(reinterpret_cast<const float4*>(P.gamma_q + 128 * j + 4 * lane));
      v[j] = make_float4(v[j].x * rq * g.x, v[j].y * rq * g.y, v[j].z * rq * g.z, v[j].w * rq * g.w);
      amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v[j].x), fabsf(v[j].y)), fmaxf(fabsf(v[j].z), fabsf(v[j].w))));
    }
  }
  amax = warp_max(amax);
  const __half s16 = __float2half_rn(amax / 127.0f);
  const float sdiv = __half2float(s16);
  auto code = [&](float y) -> uint32_t {
    const int c = sdiv > 0.f ? __float2int_rn(fminf(fmaxf(y / sdiv, -127.0f), 127.0f)) : 0;
    return static_cast<uint32_t>(c) & 0xffu;
  };
#pragma unroll
  for (int j = 0; j < kMaxQv; ++j) {
    if (j < nj) {
      const uint32_t w4 = code(v[j].x) | (code(v[j].y) << 8) | (code(v[j].z) << 16) | (code(v[j].w) << 24);
      *reinterpret_cast<uint32_t*>(sA + static_cast<size_t>(t) * P.K_q + 128 * j + 4 * lane) = w4;
      if (write_out) *reinterpret_cast<uint32_t*>(P.q_lora + static_cast<size_t>(t) * P.K_q + 128 * j + 4 * lane) = w4;
    }
  }
  if (write_out && lane == 0) P.q_lora_scale[t] = s16;
  return sdiv;
}

// One warp, token t: the latent KV row, RMSNorm(sums[t, K_q : K_q + 512]) *
// gamma_kv and the rotated last 64 dims, to kv_cache[slot[t]].
__device__ __forceinline__ void kv_row(const UpParams& P, int t, int lane) {
  const int64_t dst = __ldg(P.slot + t);
  const int p = __ldg(P.pos + t);
  if (dst >= P.cache_rows || p < 0 || p >= P.max_pos) {
    if (lane == 0) atomicOr(P.err, kErrBadIndex);
    return;
  }
  if (dst < 0) return;
  const float* kv = P.sums + static_cast<size_t>(t) * (P.K_q + kDkv) + P.K_q;
  float4 v[kDc / 128];
  float ss = 0.f;
#pragma unroll
  for (int j = 0; j < kDc / 128; ++j) {
    v[j] = __ldcg(reinterpret_cast<const float4*>(kv + 128 * j + 4 * lane));
    ss += v[j].x * v[j].x + v[j].y * v[j].y + v[j].z * v[j].z + v[j].w * v[j].w;
  }
  const int ia = P.interleaved ? 2 * lane : lane, ib = P.interleaved ? 2 * lane + 1 : lane + kDr / 2;
  const float a = __ldcg(kv + kDc + ia), b = __ldcg(kv + kDc + ib);
  const float cs = __ldg(P.rope_cos + static_cast<size_t>(p) * (kDr / 2) + lane);
  const float sn = __ldg(P.rope_sin + static_cast<size_t>(p) * (kDr / 2) + lane);
  const float rk = 1.0f / sqrtf(warp_sum(ss) / static_cast<float>(kDc) + P.eps);
  __nv_bfloat16* out = P.kv_cache + dst * kDkv;
#pragma unroll
  for (int j = 0; j < kDc / 128; ++j) {
    const float4 g = __ldg(reinterpret_cast<const float4*>(P.gamma_kv + 128 * j + 4 * lane));
    const __nv_bfloat162 lo = __floats2bfloat162_rn(v[j].x * rk * g.x, v[j].y * rk * g.y);
    const __nv_bfloat162 hi = __floats2bfloat162_rn(v[j].z * rk * g.z, v[j].w * rk * g.w);
    uint2 pk;
    pk.x = *reinterpret_cast<const uint32_t*>(&lo);
    pk.y = *reinterpret_cast<const uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(out + 128 * j + 4 * lane) = pk;
  }
  out[kDc + ia] = __float2bfloat16_rn(a * cs - b * sn);
  out[kDc + ib] = __float2bfloat16_rn(b * cs + a * sn);
}

// q_lora . w_uq^T on the tensor-core weight stream (w8tc.cuh): one CTA per
// SM over a contiguous range of w_uq's H * 192 rows, whose copies start at
// the kernel's start (the weights do not depend on mla_down).  The
// converter warps first wait for mla_down's sums and quantise the query
// latent of every token into the CTA's resident token tile (CTA 0 also
// writes q_lora); the epilogue dequantises the sums of its rows into `up`:
// up[t, n] = s * sa[t] * w_uq_scale[n], the product in that order.  After
// the stream, warp 0 of CTA t (mod the grid) writes token t's latent row.
__device__ __forceinline__ float* up_token_scales() {
  __shared__ float sa[32];
  return sa;
}

struct UpWtJob {
  int M, N, K;
  uint32_t* err;
  UpParams P;
  __device__ __forceinline__ void prologue(int w, int lane, int8_t* tok) const {
    griddep_wait();  // the sums come from mla_down
    float* sa = up_token_scales();
    for (int t = w; t < P.T; t += 8) {
      const float sdiv = quant_latent(P, t, lane, tok, blockIdx.x == 0);
      if (lane == 0) sa[t] = sdiv;
    }
    // token rows past T are zero (the tile holds 16 or 32 rows)
    const int nt = P.T <= 16 ? 16 : 32;
    uint4* z = reinterpret_cast<uint4*>(tok + static_cast<size_t>(P.T) * P.K_q);
    const int nz = (nt - P.T) * P.K_q / 16;
    for (int i = w * 32 + lane; i < nz; i += 256) z[i] = make_uint4(0u, 0u, 0u, 0u);
  }
  __device__ __forceinline__ float tok_scale(int t) const { return up_token_scales()[t]; }
  __device__ __forceinline__ float row_scale(int n) const { return __half2float(__ldg(P.w_uq_scale + n)); }
  __device__ __forceinline__ void put(int t, int n, int s, float st, float sn) const {
    P.up[static_cast<size_t>(t) * N + n] = static_cast<float>(s) * st * sn;
  }
  __device__ __forceinline__ void tail(int warp, int lane) const {
    if (warp == 0) {
      griddep_wait();  // the latent sums come from mla_down
      for (int t = blockIdx.x; t < P.T; t += gridDim.x) kv_row(P, t, lane);
    }
  }
};

// ---------------------------------------------------------------- absorb
constexpr int kAbsThreads = 256;
constexpr uint32_t kAbsW = kDn * (kDc / 2) * 2;  // [128 n][256 c] bf16 = 64 KB

struct AbsParams {
  int T, H, n_sums, max_pos, interleaved;
  const __nv_bfloat16* w_uk;  // [H, 128, 512]
  const float* up;            // workspace: [T, H, 192] from mla_up
  float* sums;                // workspace: mla_down's sums, cleared here for the next call
  const int32_t* pos;
  const float* rope_cos;
  const float* rope_sin;
  __nv_bfloat16* q;           // [T, H, 576]
  uint32_t* err;
};

template <int TM>
__global__ void __launch_bounds__(kAbsThreads, TM <= 16 ? 2 : 1) mla_absorb_kernel(const __grid_constant__ AbsParams P) {
  extern __shared__ __align__(16) uint8_t smem[];
  __nv_bfloat16* sW = reinterpret_cast<__nv_bfloat16*>(smem);                 // [128][256]
  float* sQ = reinterpret_cast<float*>(smem + kAbsW);                          // [TM][128]
  float* sPart = sQ + TM * kDn;                                                 // [TM][256]
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.x >> 1, half = blockIdx.x & 1;
  if (tid == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  griddep_launch_dependents();
  if (warp == 0) {
    if (lane == 0) mbar_arrive_expect_tx(&bar, kAbsW);
    __syncwarp();
    const __nv_bfloat16* src = P.w_uk + static_cast<size_t>(h) * kDn * kDc + half * (kDc / 2);
    constexpr uint32_t kRowBytes = (kDc / 2) * sizeof(__nv_bfloat16);  // 512 bytes of row r
    for (int r = lane; r < kDn; r += 32) bulk_g2s(sW + r * (kDc / 2), src + static_cast<size_t>(r) * kDc, kRowBytes, &bar);
  }
  griddep_wait();  // the no-position dims come from mla_up, which has read every sum
  for (int i = blockIdx.x * kAbsThreads + tid; i < P.n_sums; i += gridDim.x * kAbsThreads) P.sums[i] = 0.f;
  for (int i = tid; i < TM * kDn; i += kAbsThreads) {
    const int t = i / kDn;
    sQ[i] = t < P.T ? __ldcg(P.up + (static_cast<size_t>(t) * P.H + h) * kDh + i % kDn) : 0.f;
  }
  if (half == 1) {
    // the head's rotary dims: q[:, h, 512:576] = RoPE(up[:, h, 128:192])
    for (int idx = tid; idx < P.T * (kDr / 2); idx += kAbsThreads) {
      const int t = idx / (kDr / 2), l = idx % (kDr / 2);
      const int p = __ldg(P.pos + t);
      if (p < 0 || p >= P.max_pos) {
        if (h == 0) atomicOr(P.err, kErrBadIndex);
        continue;
      }
      const int ia = P.interleaved ? 2 * l : l, ib = P.interleaved ? 2 * l + 1 : l + kDr / 2;
      const float cs = __ldg(P.rope_cos + static_cast<size_t>(p) * (kDr / 2) + l);
      const float sn = __ldg(P.rope_sin + static_cast<size_t>(p) * (kDr / 2) + l);
      const float* r = P.up + (static_cast<size_t>(t) * P.H + h) * kDh + kDn;
      const float a = __ldcg(r + ia), b = __ldcg(r + ib);
      __nv_bfloat16* out = P.q + (static_cast<size_t>(t) * P.H + h) * kDkv + kDc;
      out[ia] = __float2bfloat16_rn(a * cs - b * sn);
      out[ib] = __float2bfloat16_rn(b * cs + a * sn);
    }
  }
  bool ok = mbar_wait(&bar, 0, P.err, &abort_flag);
  if (!ok) mbar_drain(&bar, 0);  // the slab's copies land before it is read or the CTA leaves
  __syncthreads();
  // thread: column pair cp of this half, no-position dims [64 nh, 64 nh + 64)
  const int cp = tid & 127, nh = tid >> 7;
  float acc[TM][2];
#pragma unroll
  for (int t = 0; t < TM; ++t) acc[t][0] = acc[t][1] = 0.f;
  if (ok) {
#pragma unroll 4
    for (int n = nh * 64; n < nh * 64 + 64; ++n) {
      const float2 w = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(sW + n * (kDc / 2) + 2 * cp));
#pragma unroll
      for (int t = 0; t < TM; ++t) {
        const float qv = sQ[t * kDn + n];
        acc[t][0] = fmaf(qv, w.x, acc[t][0]);
        acc[t][1] = fmaf(qv, w.y, acc[t][1]);
      }
    }
  }
  if (nh == 1) {
#pragma unroll
    for (int t = 0; t < TM; ++t) *reinterpret_cast<float2*>(sPart + t * (kDc / 2) + 2 * cp) = make_float2(acc[t][0], acc[t][1]);
  }
  __syncthreads();
  if (nh == 1 || !ok) return;
#pragma unroll
  for (int t = 0; t < TM; ++t) {
    if (t < P.T) {
      const float2 o = *reinterpret_cast<const float2*>(sPart + t * (kDc / 2) + 2 * cp);
      *reinterpret_cast<__nv_bfloat162*>(P.q + (static_cast<size_t>(t) * P.H + h) * kDkv + half * (kDc / 2) + 2 * cp) =
          __floats2bfloat162_rn(acc[t][0] + o.x, acc[t][1] + o.y);
    }
  }
}

size_t down_sums_bytes(const dsa_mla_prolog_args& a) {
  return round_up(static_cast<size_t>(a.T) * (a.K_q + kDkv) * sizeof(float), 256);
}

}  // namespace

// Workspace: [T, K_q + 576] fp32 sums of mla_down (zero between calls), then
// [T, H, 192] fp32 up-projected query dims of mla_up.
size_t mla_workspace(const dsa_mla_prolog_args& a) {
  return down_sums_bytes(a) + round_up(static_cast<size_t>(a.T) * a.H * kDh * sizeof(float), 256);
}

int launch_mla(const dsa_mla_prolog_args& a, void* ws, cudaStream_t stream) {
  uint32_t* err = error_word();
  if (!err) return DSA_ERR_CUDA;
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  float* sums = reinterpret_cast<float*>(wsb);
  float* up = reinterpret_cast<float*>(wsb + down_sums_bytes(a));

  // ---- down: row blocks x slices of D_x, as many slices as fill the SMs
  DownParams D{};
  D.T = a.T; D.K_q = a.K_q; D.D_x = a.D_x;
  D.n_rb_q = a.K_q / 128;
  D.n_rb = D.n_rb_q + (kDkv + 127) / 128;
  const int atoms = a.D_x / 64;
  int n_split = sm_count() / D.n_rb;
  if (n_split < 1) n_split = 1;
  if (n_split > atoms) n_split = atoms;
  D.per = (atoms + n_split - 1) / n_split;
  n_split = (atoms + D.per - 1) / D.per;
  D.sums = sums;
  D.err = err;
  const int nx = a.T <= 16 ? 16 : 32;
  alignas(64) CUtensorMap tm_wdq, tm_wdkv, tm_x;
  {
    const uint64_t st[1] = {static_cast<uint64_t>(a.D_x) * 2};
    const uint64_t dq[2] = {static_cast<uint64_t>(a.D_x), static_cast<uint64_t>(a.K_q)};
    const uint64_t dk[2] = {static_cast<uint64_t>(a.D_x), static_cast<uint64_t>(kDkv)};
    const uint64_t dx[2] = {static_cast<uint64_t>(a.D_x), static_cast<uint64_t>(a.T)};
    const uint32_t bw[2] = {64, 128}, bx[2] = {64, static_cast<uint32_t>(nx)};
    if (!encode_tmap(&tm_wdq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.w_dq, dq, st, bw, 128) ||
        !encode_tmap(&tm_wdkv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.w_dkv, dk, st, bw, 128) ||
        !encode_tmap(&tm_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.x, dx, st, bx, 128))
      return DSA_ERR_CUDA;
  }
  const size_t smem_down = 1024 + kDownStages * (kDownAtomW + static_cast<size_t>(nx) * 128);
  auto go_down = [&](auto kern) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem_down));
    // the SM keeps its full shared memory, so an mla_up CTA fits beside
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    kern<<<D.n_rb * n_split, kDownThreads, smem_down, stream>>>(D, tm_wdq, tm_wdkv, tm_x);
    return cudaGetLastError();
  };
  cudaError_t e = nx == 16 ? go_down(mla_down_kernel<16>) : go_down(mla_down_kernel<32>);
  if (e != cudaSuccess) return DSA_ERR_CUDA;

  // ---- up and absorb: programmatic dependent launches
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  const int tm = a.T <= 8 ? 8 : (a.T <= 16 ? 16 : 32);

  UpParams U{};
  U.T = a.T; U.H = a.H; U.K_q = a.K_q; U.interleaved = a.rope_interleaved; U.max_pos = a.rope_max_pos;
  U.eps = a.rms_eps;
  U.sums = sums; U.gamma_q = a.gamma_q; U.gamma_kv = a.gamma_kv;
  U.w_uq = a.w_uq;
  U.w_uq_scale = reinterpret_cast<const __half*>(a.w_uq_scale);
  U.pos = a.pos; U.rope_cos = a.rope_cos; U.rope_sin = a.rope_sin;
  U.q_lora = a.q_lora; U.q_lora_scale = reinterpret_cast<__half*>(a.q_lora_scale);
  U.up = up;
  U.kv_cache = reinterpret_cast<__nv_bfloat16*>(a.kv_cache); U.slot = a.slot; U.cache_rows = a.cache_rows;
  U.err = err;
  const int nt = a.T <= 16 ? 16 : 32;
  alignas(64) WtMaps maps;
  {
    if (!wt_encode_weights(maps, a.w_uq, a.H * kDh, a.K_q)) return DSA_ERR_CUDA;
    maps.tok = maps.w[0];  // unused: the tokens are resident
  }
  const UpWtJob job{a.T, a.H * kDh, a.K_q, err, U};
  const long long units = (static_cast<long long>(a.H) * kDh + kWtUnit - 1) / kWtUnit;
  cudaLaunchConfig_t cu = {};
  cu.gridDim = dim3(static_cast<unsigned>(std::min<long long>(units, sm_count())));
  cu.blockDim = dim3(kWtThreads);
  cu.stream = stream;
  cu.attrs = pdl;
  cu.numAttrs = 1;
  // A ring small enough that an mla_up CTA fits beside an mla_down CTA on
  // one SM: the up-projection's weights stream while mla_down runs.
  const size_t budget = 228 * 1024 - 2048 - smem_down - 4096;
  auto go_up = [&](auto kern, auto layout) {
    using L = decltype(layout);
    const int ns8 = L::stages(a.K_q, budget);
    cu.dynamicSmemBytes = L::smem(a.K_q, ns8);
    cudaError_t r = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(cu.dynamicSmemBytes));
    if (r == cudaSuccess)
      r = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    return r == cudaSuccess ? cudaLaunchKernelEx(&cu, kern, maps, job, ns8) : r;
  };
  e = nt == 16 ? go_up(wt_kernel<16, true, UpWtJob>, WtLayout<16, true>{})
               : go_up(wt_kernel<32, true, UpWtJob>, WtLayout<32, true>{});
  if (e != cudaSuccess) return DSA_ERR_CUDA;

  AbsParams A{};
  A.T = a.T; A.H = a.H; A.n_sums = a.T * (a.K_q + kDkv);
  A.w_uk = reinterpret_cast<const __nv_bfloat16*>(a.w_uk); A.up = up; A.sums = sums;
  A.pos = a.pos; A.rope_cos = a.rope_cos; A.rope_sin = a.rope_sin;
  A.max_pos = a.rope_max_pos; A.interleaved = a.rope_interleaved;
  A.q = reinterpret_cast<__nv_bfloat16*>(a.q); A.err = err;
  const size_t smem_abs = kAbsW + static_cast<size_t>(tm) * (kDn + kDc / 2) * sizeof(float);
  cudaLaunchConfig_t ca = cu;
  ca.gridDim = dim3(2 * a.H);
  ca.blockDim = dim3(kAbsThreads);
  ca.dynamicSmemBytes = smem_abs;
  auto go_abs = [&](auto kern) {
    cudaError_t r = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem_abs));
    if (r == cudaSuccess)
      r = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    return r == cudaSuccess ? cudaLaunchKernelEx(&ca, kern, A) : r;
  };
  e = tm == 8 ? go_abs(mla_absorb_kernel<8>) : (tm == 16 ? go_abs(mla_absorb_kernel<16>) : go_abs(mla_absorb_kernel<32>));
  return cuda_status(e);
}

}  // namespace dsa

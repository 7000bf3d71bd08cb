// Indexer Prolog: the q stream (int8 GEMM + dequant, RoPE, Hadamard,
// DynamicQuant), the k stream (bf16 GEMM, LayerNorm, RoPE, Hadamard,
// DynamicQuant, cache scatter) and the optional weight stream, in one launch.
//
// [V3.2-PyPTO §Indexer Prolog] gives the three formulas and observes that
// the q stream (an (8,1536)x(1536,8192) int8 GEMM) dominates and is bound by
// weight traffic.  At T <= 32 tokens every output channel is a K_q-long dot
// against <= 32 activation rows: the work is a weight stream, not a GEMM
// that tensor cores would shorten, so it runs as dp4a over shared-memory
// slabs filled by bulk async copies, one CTA per SM, in a single wave:
//
//   * q stream: a cluster of 2 CTAs per head splits K_q in two; each CTA
//     streams its [d_I x K_q/2] weight slab (96 KB at the decode shape) with
//     cp.async.bulk, computes int32 partial dots, and the pair sums its
//     partials through distributed shared memory.  Each CTA then finishes
//     the tokens t = rank (mod 2): dequant -> RoPE -> Hadamard (warp
//     butterfly over shuffles) -> int8 quantisation.
//   * k / weight streams: split over D_x.  Each CTA takes a slice of
//     64-column atoms of w_k, w_proj and x (TMA tiles, 128-byte swizzle)
//     and forms its partial [channels x tokens] product on the tensor core
//     (bf16 operands, fp32 accumulation in tensor memory), so a CTA reads
//     its weight slice and only its slice of x.  The partial sums are added
//     into the fp32 workspace; the last CTA to finish (atomic ticket) runs
//     LayerNorm -> RoPE -> Hadamard -> quantisation, writes the key-cache
//     rows and the weights, and clears the workspace for the next call.
// Every scale, RoPE row, gamma/beta and position an epilogue needs is
// prefetched into shared memory while the weight slabs are in flight.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include "dsa_internal.h"
#include "dsa_ptx.cuh"

namespace dsa {
namespace {

constexpr int kThreads = 256;
constexpr int kQSplit = 2;       // cluster size and K_q split of the q stream
constexpr int kKwMaxAtoms = 6;   // 64-column atoms of D_x per k/weight CTA (shared memory)
constexpr uint32_t kKwAtom = 128 * 128;  // [128 rows][64 bf16] operand atom
constexpr int kMaxT = 32;
constexpr int kMaxRope = 64;     // max d_rope / 2 entries per RoPE row

struct PrologParams {
  int T, H_I, d_I, d_rope, K_q, D_x, interleaved, n_q_ctas, n_kw_ctas, n_kw_channels, kw_atoms, rope_max_pos;
  const int8_t* q_lora;
  const __half* q_lora_scale;
  const int8_t* w_qb;
  const __half* w_qb_scale;
  const __nv_bfloat16* x;
  const __nv_bfloat16* w_k;
  const float* ln_gamma;
  const float* ln_beta;
  float ln_eps;
  const __nv_bfloat16* w_proj;
  float w_scale;
  const int32_t* pos;
  const float* rope_cos;
  const float* rope_sin;
  int8_t* q_out;
  __half* q_scale_out;
  int8_t* k_cache;
  __half* k_scale_cache;
  const int64_t* slot;
  int64_t cache_rows;
  float* w_out;
  uint32_t* ticket;  // workspace: last-CTA ticket (left at 0)
  float* kw;         // workspace: [T, n_kw_channels] fp32 sums (left at 0)
  uint32_t* err;
};

// Small per-CTA tables filled before the big wait.
struct Pre {
  float cos_t[kMaxT][kMaxRope];
  float sin_t[kMaxT][kMaxRope];
  float sa[kMaxT];
  float sb[128];
  float gamma[128];
  float beta[128];
  int64_t slot[kMaxT];
  int pos_ok[kMaxT];  // pos[t] lies in [0, rope_max_pos)
};

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

// RoPE rows of the tokens (d_rope/2 cos and sin each) into shared memory.
// A position outside [0, rope_max_pos) reads no table row: the token is
// marked (its q and key rows are then not written) and the error recorded.
__device__ __forceinline__ void prefetch_rope(const PrologParams& P, Pre& pre, int tid) {
  const int half = P.d_rope / 2;
  if (tid < P.T) {
    const int p = __ldg(P.pos + tid);
    const bool ok = p >= 0 && p < P.rope_max_pos;
    pre.pos_ok[tid] = ok;
    if (!ok && blockIdx.x == 0) atomicOr(P.err, kErrBadIndex);
  }
  for (int i = tid; i < P.T * half; i += kThreads) {
    const int t = i / half, c = i % half;
    const int p = __ldg(P.pos + t);
    const bool ok = p >= 0 && p < P.rope_max_pos;
    const size_t off = static_cast<size_t>(ok ? p : 0) * half + c;
    pre.cos_t[t][c] = ok ? __ldg(P.rope_cos + off) : 0.f;
    pre.sin_t[t][c] = ok ? __ldg(P.rope_sin + off) : 0.f;
  }
}

// One warp holds one d_I = 32*DPL row, lane l owning dims l*DPL .. l*DPL+DPL-1.
// Applies RoPE (the token's cos/sin rows), the scaled Sylvester Hadamard
// transform and the int8 quantisation; returns the codes and the fp16 scale.
template <int DPL>
__device__ __forceinline__ void rope_hadamard_quant(float (&v)[DPL], int lane, const float* crow,
                                                    const float* srow, int d_rope, int interleaved,
                                                    int (&c)[DPL], __half& scale16) {
  const int half = d_rope / 2;
  if (interleaved) {
#pragma unroll
    for (int j = 0; j < DPL; j += 2) {
      const int d = lane * DPL + j;
      if (d < d_rope) {
        const float cs = crow[d / 2], sn = srow[d / 2];
        const float a = v[j], b = v[j + 1];
        v[j] = a * cs - b * sn;
        v[j + 1] = b * cs + a * sn;
      }
    }
  } else {
    const int off = half / DPL;  // partner lane distance
    const int d0 = lane * DPL;
    int src = lane;
    if (d0 < half) src = lane + off;
    else if (d0 < d_rope) src = lane - off;
#pragma unroll
    for (int j = 0; j < DPL; ++j) {
      const float partner = __shfl_sync(0xffffffffu, v[j], src);
      const int d = d0 + j;
      if (d < half) {
        v[j] = v[j] * crow[d] - partner * srow[d];
      } else if (d < d_rope) {
        v[j] = v[j] * crow[d - half] + partner * srow[d - half];
      }
    }
  }
  // Hadamard: in-thread butterflies, then across lanes.
#pragma unroll
  for (int s = 1; s < DPL; s <<= 1) {
#pragma unroll
    for (int j = 0; j < DPL; ++j) {
      if ((j & s) == 0) {
        const float a = v[j], b = v[j + s];
        v[j] = a + b;
        v[j + s] = a - b;
      }
    }
  }
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    const bool upper = (lane & m) != 0;
#pragma unroll
    for (int j = 0; j < DPL; ++j) {
      const float o = __shfl_xor_sync(0xffffffffu, v[j], m);
      v[j] = upper ? (o - v[j]) : (v[j] + o);
    }
  }
  const float norm = (DPL == 4) ? 0.08838834764831845f : 0.125f;  // (32*DPL)^-1/2
  float amax = 0.f;
#pragma unroll
  for (int j = 0; j < DPL; ++j) {
    v[j] *= norm;
    amax = fmaxf(amax, fabsf(v[j]));
  }
  amax = warp_max(amax);
  scale16 = __float2half_rn(amax / 127.0f);
  const float sdiv = __half2float(scale16);
#pragma unroll
  for (int j = 0; j < DPL; ++j) {
    if (sdiv > 0.f) {
      const float y = fminf(fmaxf(v[j] / sdiv, -127.0f), 127.0f);
      c[j] = __float2int_rn(y);
    } else {
      c[j] = 0;
    }
  }
}

template <int DPL>
__device__ __forceinline__ void store_codes(int8_t* dst, const int (&c)[DPL]) {
  if (DPL == 4) {
    const uint32_t w = (uint32_t)(c[0] & 0xff) | ((uint32_t)(c[1] & 0xff) << 8) |
                       ((uint32_t)(c[2] & 0xff) << 16) | ((uint32_t)(c[3] & 0xff) << 24);
    *reinterpret_cast<uint32_t*>(dst) = w;
  } else {
    const uint16_t w = (uint16_t)((c[0] & 0xff) | ((c[1] & 0xff) << 8));
    *reinterpret_cast<uint16_t*>(dst) = w;
  }
}

// ---------------------------------------------------------------- q stream
template <int DPL, int TM>
__device__ void q_stream(const PrologParams& P, uint8_t* smem, Pre& pre) {
  constexpr int D = 32 * DPL;           // d_I
  constexpr int TG = kThreads / D;      // token groups per channel
  constexpr int TPT = TM / TG;          // tokens per thread (rows >= T are zero)
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int head = blockIdx.x / kQSplit;
  const uint32_t rank = cluster_ctarank();
  const int kchunk = P.K_q / kQSplit;
  const int wstride = kchunk + 16;  // padded rows: conflict-free 16-byte reads
  const int T = P.T;

  uint8_t* sW = smem;                                   // [D][wstride]
  uint8_t* sQ = sW + D * wstride;                       // [T][kchunk]
  int32_t* sPart = reinterpret_cast<int32_t*>(sQ + kMaxT * kchunk);  // [T][D]
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;

  if (tid == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  griddep_launch_dependents();
  // The weight slab is never written by the previous kernel: its copies go
  // out before the wait for that kernel (programmatic launch), the
  // activation rows after it.
  if (warp == 0) {
    const uint32_t bytes = static_cast<uint32_t>((D + T) * kchunk);
    if (lane == 0) mbar_arrive_expect_tx(&bar, bytes);
    __syncwarp();
    const int8_t* wsrc = P.w_qb + static_cast<size_t>(head) * D * P.K_q + rank * kchunk;
    for (int r = lane; r < D; r += 32) bulk_g2s(sW + r * wstride, wsrc + static_cast<size_t>(r) * P.K_q, kchunk, &bar);
  }
  griddep_wait();  // q_lora and its scales may come from the previous kernel
  if (warp == 0) {
    const int8_t* qsrc = P.q_lora + rank * kchunk;
    for (int t = lane; t < T; t += 32) bulk_g2s(sQ + t * kchunk, qsrc + static_cast<size_t>(t) * P.K_q, kchunk, &bar);
  }
  // rows T..TM-1 of the activation slab are zero so that the dot loop
  // below runs without per-token branches
  for (int i = tid; i < (TM - T) * kchunk / 16; i += kThreads)
    reinterpret_cast<int4*>(sQ + T * kchunk)[i] = make_int4(0, 0, 0, 0);
  // epilogue inputs, while the slabs are in flight
  if (tid < D) pre.sb[tid] = __half2float(__ldg(P.w_qb_scale + head * D + tid));
  if (tid >= D && tid - D < T) pre.sa[tid - D] = __half2float(__ldg(P.q_lora_scale + (tid - D)));
  prefetch_rope(P, pre, tid);
  // a wait that gave up still lets every copy land before the slabs are read
  // (or the CTA leaves): the copies write this CTA's shared memory
  if (!mbar_wait(&bar, 0, P.err, &abort_flag)) mbar_drain(&bar, 0);
  __syncthreads();  // zero rows and prefetched tables written by other threads

  // int32 partial dots over this CTA's K_q slice.
  const int n = tid % D, tg = tid / D;
  int acc[TPT];
#pragma unroll
  for (int i = 0; i < TPT; ++i) acc[i] = 0;
  const uint8_t* wrow = sW + n * wstride;
  const uint8_t* qcol = sQ + tg * kchunk;
#pragma unroll 2
  for (int k = 0; k < kchunk; k += 16) {
    const int4 w = *reinterpret_cast<const int4*>(wrow + k);
    int4 q[TPT];
#pragma unroll
    for (int i = 0; i < TPT; ++i) q[i] = *reinterpret_cast<const int4*>(qcol + i * TG * kchunk + k);
#pragma unroll
    for (int i = 0; i < TPT; ++i) {
      acc[i] = __dp4a(w.x, q[i].x, acc[i]);
      acc[i] = __dp4a(w.y, q[i].y, acc[i]);
      acc[i] = __dp4a(w.z, q[i].z, acc[i]);
      acc[i] = __dp4a(w.w, q[i].w, acc[i]);
    }
  }
#pragma unroll
  for (int i = 0; i < TPT; ++i) {
    const int t = tg + i * TG;
    if (t < T) sPart[t * D + n] = acc[i];
  }
  cluster_sync();

  // Tokens t = rank (mod kQSplit): sum the pair's partials, then the
  // dequant -> RoPE -> Hadamard -> quant epilogue, one warp per token.
  for (int t = rank + kQSplit * warp; t < T; t += kQSplit * (kThreads / 32)) {
    if (!pre.pos_ok[t]) continue;  // warp-uniform: the whole warp skips the token
    float v[DPL];
    const float sa = pre.sa[t];
    uint32_t pv[kQSplit][DPL];
#pragma unroll
    for (int r = 0; r < kQSplit; ++r)
#pragma unroll
      for (int j = 0; j < DPL; ++j) pv[r][j] = ld_cluster_u32(mapa(smem_u32(&sPart[t * D + lane * DPL + j]), r));
#pragma unroll
    for (int j = 0; j < DPL; ++j) {
      int s = 0;
#pragma unroll
      for (int r = 0; r < kQSplit; ++r) s += static_cast<int>(pv[r][j]);
      v[j] = (static_cast<float>(s) * sa) * pre.sb[lane * DPL + j];
    }
    int c[DPL];
    __half s16;
    rope_hadamard_quant<DPL>(v, lane, pre.cos_t[t], pre.sin_t[t], P.d_rope, P.interleaved, c, s16);
    store_codes<DPL>(P.q_out + (static_cast<size_t>(t) * P.H_I + head) * D + lane * DPL, c);
    if (lane == 0) P.q_scale_out[t * P.H_I + head] = s16;
  }
  cluster_sync();  // the peer may still read this CTA's partials
}

// ------------------------------------------------------- k / weight stream
// CTA c owns the 64-column atoms [c*kw_atoms, (c+1)*kw_atoms) of D_x.  Its
// partial products D0 = w_k[:, slice] . x[:, slice]^T (channels x tokens)
// and D1 = w_proj[:, slice] . x[:, slice]^T come from M=128, N=NX bf16 MMAs
// (rows past d_I / H_I and tokens past T are zero fill of the tiles).
template <int DPL, int NX>
__device__ void kw_stream(const PrologParams& P, const CUtensorMap* tm_wk, const CUtensorMap* tm_wp,
                          const CUtensorMap* tm_x, uint8_t* smem_raw, Pre& pre) {
  constexpr int D = 32 * DPL;
  constexpr uint32_t kAtomX = NX * 128;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int cta = blockIdx.x - P.n_q_ctas;
  if (cta >= P.n_kw_ctas) {  // padding CTA of the last cluster
    griddep_launch_dependents();
    return;
  }
  const int T = P.T;
  const int nb = P.kw_atoms;
  const int x0 = cta * nb * 64;
  const bool has_w = P.w_proj != nullptr;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA0 = smem;                // w_k atoms    [nb][128 rows][128 B]
  uint8_t* sA1 = sA0 + nb * kKwAtom;  // w_proj atoms [nb][128 rows][128 B]
  uint8_t* sB = sA1 + nb * kKwAtom;   // x atoms      [nb][NX rows][128 B]
  __shared__ bool is_last;
  __shared__ __align__(8) uint64_t bar, mdone;
  __shared__ int abort_flag;
  __shared__ uint32_t tmem_base;
  if (tid == 0) {
    mbar_init(&bar, 1);
    mbar_init(&mdone, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(&tmem_base, 64);  // D0 in columns [0, NX), D1 in [32, 32 + NX)
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;
  griddep_launch_dependents();
  // the weight tiles before the wait for the previous kernel, x after it
  if (tid == 0) {
    mbar_arrive_expect_tx(&bar, static_cast<uint32_t>(nb) * ((has_w ? 2u : 1u) * kKwAtom + kAtomX));
    for (int a = 0; a < nb; ++a) {
      const int xc = x0 + a * 64;  // atoms past D_x read as zero
      tma_load_2d(sA0 + a * kKwAtom, tm_wk, xc, 0, &bar);
      if (has_w) tma_load_2d(sA1 + a * kKwAtom, tm_wp, xc, 0, &bar);
    }
  }
  griddep_wait();
  if (tid == 0)
    for (int a = 0; a < nb; ++a) tma_load_2d(sB + a * kAtomX, tm_x, x0 + a * 64, 0, &bar);
  // inputs of the last CTA's epilogue
  if (tid < D) {
    pre.gamma[tid] = __ldg(P.ln_gamma + tid);
    pre.beta[tid] = __ldg(P.ln_beta + tid);
  }
  if (tid >= D && tid - D < T) pre.slot[tid - D] = __ldg(P.slot + (tid - D));
  prefetch_rope(P, pre, tid);

  if (tid == 0) {
    const bool loaded = mbar_wait(&bar, 0, P.err, &abort_flag);
    if (loaded) {
      tc_fence_after();
      const uint32_t idesc = idesc_f16(128, NX, kFmtBF16, 0, 0);
      for (int a = 0; a < nb; ++a) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {  // K = 16 per MMA, 32 bytes into the swizzled atom
          const uint32_t acc = (a > 0 || kk > 0) ? 1u : 0u;
          const uint64_t bd = smem_desc(smem_u32(sB + a * kAtomX) + kk * 32, 16, 1024, kSwizzle128B);
          mma_ss(tmem, smem_desc(smem_u32(sA0 + a * kKwAtom) + kk * 32, 16, 1024, kSwizzle128B), bd, idesc, acc);
          if (has_w)
            mma_ss(tmem + 32, smem_desc(smem_u32(sA1 + a * kKwAtom) + kk * 32, 16, 1024, kSwizzle128B), bd, idesc,
                   acc);
        }
      }
    }
    mma_commit(&mdone);
    if (!loaded) mbar_drain(&bar, 0);  // the tiles land before the CTA leaves
  }
  if (warp < 4) {
    // Row r of D0 / D1 (TMEM lane r) is channel r / d_I + r; column t is token t.
    // a CTA whose weight tiles never arrived adds nothing (its error is
    // recorded); a wait on the MMAs that gave up still lets them finish
    // before the tensor memory is read or released
    bool ok = mbar_wait(&mdone, 0, P.err, &abort_flag);
    if (!ok) mbar_drain(&mdone, 0);
    ok = ok && !*static_cast<volatile int*>(&abort_flag);
    tc_fence_after();
    const int r = warp * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    uint32_t v[32];
    tmem_ld32(lane_base, v);
    tmem_ld_wait();
    if (ok && r < D) {
#pragma unroll
      for (int t = 0; t < NX; ++t)
        if (t < T) atomicAdd(P.kw + static_cast<size_t>(t) * P.n_kw_channels + r, __uint_as_float(v[t]));
    }
    if (has_w) {
      tmem_ld32(lane_base + 32, v);
      tmem_ld_wait();
      if (ok && r < P.H_I) {
#pragma unroll
        for (int t = 0; t < NX; ++t)
          if (t < T) atomicAdd(P.kw + static_cast<size_t>(t) * P.n_kw_channels + D + r, __uint_as_float(v[t]));
      }
    }
  }
  tc_fence_before();
  __threadfence();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 64);
  if (tid == 0) is_last = (atomicAdd(P.ticket, 1u) == static_cast<uint32_t>(P.n_kw_ctas - 1));
  __syncthreads();
  if (!is_last) return;
  __threadfence();

  // Last CTA: LayerNorm -> RoPE -> Hadamard -> quant for every token's key.
  for (int t = warp; t < T; t += kThreads / 32) {
    if (!pre.pos_ok[t]) continue;  // warp-uniform
    float v[DPL];
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < DPL; ++j) {
      v[j] = __ldcg(P.kw + static_cast<size_t>(t) * P.n_kw_channels + lane * DPL + j);
      s += v[j];
    }
    const float mean = warp_sum(s) / static_cast<float>(D);
    float q = 0.f;
#pragma unroll
    for (int j = 0; j < DPL; ++j) {
      const float dlt = v[j] - mean;
      q += dlt * dlt;
    }
    const float var = warp_sum(q) / static_cast<float>(D);
    const float rstd = 1.0f / sqrtf(var + P.ln_eps);
#pragma unroll
    for (int j = 0; j < DPL; ++j) {
      const int d = lane * DPL + j;
      v[j] = (v[j] - mean) * rstd * pre.gamma[d] + pre.beta[d];
    }
    int c[DPL];
    __half s16;
    rope_hadamard_quant<DPL>(v, lane, pre.cos_t[t], pre.sin_t[t], P.d_rope, P.interleaved, c, s16);
    const int64_t row = pre.slot[t];
    if (row >= 0 && row < P.cache_rows) {
      store_codes<DPL>(P.k_cache + row * D + lane * DPL, c);
      if (lane == 0) P.k_scale_cache[row] = s16;
    } else if (row >= P.cache_rows && lane == 0) {
      atomicOr(P.err, kErrBadIndex);
    }
  }
  if (P.w_out != nullptr) {
    for (int i = tid; i < T * P.H_I; i += kThreads) {
      const int t = i / P.H_I, h = i % P.H_I;
      P.w_out[i] = __ldcg(P.kw + static_cast<size_t>(t) * P.n_kw_channels + D + h) * P.w_scale;
    }
  }
  __syncthreads();  // every sum is read: clear them for the next call
  for (int i = tid; i < T * P.n_kw_channels; i += kThreads) P.kw[i] = 0.f;
  if (tid == 0) *P.ticket = 0u;  // ready for the next call
}

template <int DPL, int TM>
__global__ void __launch_bounds__(kThreads, 1)
    prolog_kernel(const __grid_constant__ PrologParams P, const __grid_constant__ CUtensorMap tm_wk,
                  const __grid_constant__ CUtensorMap tm_wp, const __grid_constant__ CUtensorMap tm_x) {
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ Pre pre;
  if (static_cast<int>(blockIdx.x) < P.n_q_ctas) {
    q_stream<DPL, TM>(P, smem, pre);
  } else {
    kw_stream<DPL, (TM < 16 ? 16 : TM)>(P, &tm_wk, &tm_wp, &tm_x, smem, pre);
  }
}

}  // namespace

size_t prolog_workspace(const dsa_prolog_args& a) {
  const int nch = a.d_I + (a.w_proj ? a.H_I : 0);
  return 256 + round_up(static_cast<size_t>(a.T) * nch * sizeof(float), 256);
}

int launch_prolog(const dsa_prolog_args& a, void* ws, cudaStream_t stream) {
  PrologParams P{};
  P.T = a.T; P.H_I = a.H_I; P.d_I = a.d_I; P.d_rope = a.d_rope; P.K_q = a.K_q; P.D_x = a.D_x;
  P.interleaved = a.rope_interleaved;
  P.n_q_ctas = a.H_I * kQSplit;
  P.n_kw_channels = a.d_I + (a.w_proj ? a.H_I : 0);
  // The k / weight CTAs split D_x into 64-column atoms, as few per CTA as
  // the SMs left over by the q stream allow (at most kKwMaxAtoms, and at
  // most what fits in shared memory beside the kernel's static tables).
  const int tm = a.T <= 8 ? 8 : (a.T <= 16 ? 16 : 32);
  const int nx = tm < 16 ? 16 : tm;  // MMA N: tokens padded with zero rows
  const void* kern = a.d_I == 128 ? (tm == 8 ? (const void*)prolog_kernel<4, 8>
                                             : tm == 16 ? (const void*)prolog_kernel<4, 16>
                                                        : (const void*)prolog_kernel<4, 32>)
                                  : (tm == 8 ? (const void*)prolog_kernel<2, 8>
                                             : tm == 16 ? (const void*)prolog_kernel<2, 16>
                                                        : (const void*)prolog_kernel<2, 32>);
  cudaFuncAttributes fa{};
  if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess) return DSA_ERR_CUDA;
  constexpr size_t kSmemPerBlock = 232448;  // 227 KB opt-in limit of sm_103a
  const size_t per_atom = 2 * kKwAtom + static_cast<size_t>(nx) * 128;
  const int fit_atoms = static_cast<int>((kSmemPerBlock - fa.sharedSizeBytes - 1024) / per_atom);
  const int atoms = a.D_x / 64;
  const int spare = sm_count() - P.n_q_ctas;
  const int want = spare >= 8 ? spare : 8;
  P.kw_atoms = (atoms + want - 1) / want;
  if (P.kw_atoms > kKwMaxAtoms) P.kw_atoms = kKwMaxAtoms;
  if (P.kw_atoms > fit_atoms) P.kw_atoms = fit_atoms;
  P.n_kw_ctas = (atoms + P.kw_atoms - 1) / P.kw_atoms;
  P.q_lora = a.q_lora; P.q_lora_scale = reinterpret_cast<const __half*>(a.q_lora_scale);
  P.w_qb = a.w_qb; P.w_qb_scale = reinterpret_cast<const __half*>(a.w_qb_scale);
  P.x = reinterpret_cast<const __nv_bfloat16*>(a.x);
  P.w_k = reinterpret_cast<const __nv_bfloat16*>(a.w_k);
  P.ln_gamma = a.ln_gamma; P.ln_beta = a.ln_beta; P.ln_eps = a.ln_eps;
  P.w_proj = reinterpret_cast<const __nv_bfloat16*>(a.w_proj); P.w_scale = a.w_scale;
  P.pos = a.pos; P.rope_cos = a.rope_cos; P.rope_sin = a.rope_sin; P.rope_max_pos = a.rope_max_pos;
  P.q_out = a.q_out; P.q_scale_out = reinterpret_cast<__half*>(a.q_scale_out);
  P.k_cache = a.k_cache; P.k_scale_cache = reinterpret_cast<__half*>(a.k_scale_cache);
  P.slot = a.slot; P.cache_rows = a.cache_rows; P.w_out = a.w_out;
  P.ticket = static_cast<uint32_t*>(ws);
  P.kw = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + 256);
  P.err = error_word();
  if (!P.err) return DSA_ERR_CUDA;

  const int kchunk = a.K_q / kQSplit;
  const size_t smem_q = static_cast<size_t>(a.d_I) * (kchunk + 16) + static_cast<size_t>(kMaxT) * kchunk +
                        static_cast<size_t>(kMaxT) * a.d_I * 4;
  const size_t smem_kw = 1024 + static_cast<size_t>(P.kw_atoms) * (2 * kKwAtom + nx * 128);
  const size_t smem = smem_q > smem_kw ? smem_q : smem_kw;
  // bf16 tiles of 64 columns x rows; rows past the tensor (channels past
  // d_I or H_I, tokens past T) and columns past D_x read as zero.
  alignas(64) CUtensorMap tm_wk, tm_wp, tm_x;
  {
    const uint64_t strides[1] = {static_cast<uint64_t>(a.D_x) * 2};
    const uint64_t dk[2] = {static_cast<uint64_t>(a.D_x), static_cast<uint64_t>(a.d_I)};
    const uint64_t dx[2] = {static_cast<uint64_t>(a.D_x), static_cast<uint64_t>(a.T)};
    const uint32_t box_w[2] = {64, 128}, box_x[2] = {64, static_cast<uint32_t>(nx)};
    if (!encode_tmap(&tm_wk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.w_k, dk, strides, box_w, 128) ||
        !encode_tmap(&tm_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.x, dx, strides, box_x, 128))
      return DSA_ERR_CUDA;
    tm_wp = tm_wk;
    if (a.w_proj) {
      const uint64_t dp[2] = {static_cast<uint64_t>(a.D_x), static_cast<uint64_t>(a.H_I)};
      if (!encode_tmap(&tm_wp, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.w_proj, dp, strides, box_w, 128))
        return DSA_ERR_CUDA;
    }
  }
  const int grid = P.n_q_ctas + static_cast<int>(round_up(P.n_kw_ctas, kQSplit));
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kQSplit;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cudaError_t e;
  auto go = [&](auto kern) {
    cudaError_t r = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    return r == cudaSuccess ? cudaLaunchKernelEx(&cfg, kern, P, tm_wk, tm_wp, tm_x) : r;
  };
  if (a.d_I == 128) {
    e = tm == 8 ? go(prolog_kernel<4, 8>) : (tm == 16 ? go(prolog_kernel<4, 16>) : go(prolog_kernel<4, 32>));
  } else {
    e = tm == 8 ? go(prolog_kernel<2, 8>) : (tm == 16 ? go(prolog_kernel<2, 16>) : go(prolog_kernel<2, 32>));
  }
  return cuda_status(e);
}

}  // namespace dsa

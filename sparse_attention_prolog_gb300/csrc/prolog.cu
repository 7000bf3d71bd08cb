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
//   * k / weight streams: CTAs of 8 output channels over the full D_x (the
//     8 weight rows are bulk-copied into shared memory); fp32 results go to
//     the workspace and the last CTA to finish (atomic ticket) runs
//     LayerNorm -> RoPE -> Hadamard -> quantisation, writes the key-cache
//     rows and the weights.
// Every scale, RoPE row, gamma/beta and position an epilogue needs is
// prefetched into shared memory while the weight slabs are in flight.
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include "dsa_internal.h"
#include "dsa_ptx.cuh"

namespace dsa {
namespace {

constexpr int kThreads = 256;
constexpr int kQSplit = 2;       // cluster size and K_q split of the q stream
constexpr int kKwChannels = 8;   // output channels per k/weight CTA
constexpr int kMaxT = 32;
constexpr int kMaxRope = 64;     // max d_rope / 2 entries per RoPE row

struct PrologParams {
  int T, H_I, d_I, d_rope, K_q, D_x, interleaved, n_q_ctas, n_kw_ctas, n_kw_channels;
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
  float* kw;         // workspace: [T, n_kw_channels]
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
__device__ __forceinline__ void prefetch_rope(const PrologParams& P, Pre& pre, int tid) {
  const int half = P.d_rope / 2;
  for (int i = tid; i < P.T * half; i += kThreads) {
    const int t = i / half, c = i % half;
    const size_t off = static_cast<size_t>(__ldg(P.pos + t)) * half + c;
    pre.cos_t[t][c] = __ldg(P.rope_cos + off);
    pre.sin_t[t][c] = __ldg(P.rope_sin + off);
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
  griddep_wait();
  if (warp == 0) {
    const uint32_t bytes = static_cast<uint32_t>((D + T) * kchunk);
    if (lane == 0) mbar_arrive_expect_tx(&bar, bytes);
    __syncwarp();
    const int8_t* wsrc = P.w_qb + static_cast<size_t>(head) * D * P.K_q + rank * kchunk;
    for (int r = lane; r < D; r += 32) bulk_g2s(sW + r * wstride, wsrc + static_cast<size_t>(r) * P.K_q, kchunk, &bar);
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
  mbar_wait(&bar, 0, P.err, &abort_flag);
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
template <int DPL>
__device__ void kw_stream(const PrologParams& P, uint8_t* smem, Pre& pre) {
  constexpr int D = 32 * DPL;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int cta = blockIdx.x - P.n_q_ctas;
  if (cta >= P.n_kw_ctas) {  // padding CTA of the last cluster
    griddep_launch_dependents();
    return;
  }
  const int T = P.T;
  const int c0 = cta * kKwChannels;
  const int nch = min(kKwChannels, P.n_kw_channels - c0);
  const size_t row_bytes = static_cast<size_t>(P.D_x) * 2;
  __nv_bfloat16* sWk = reinterpret_cast<__nv_bfloat16*>(smem);  // [nch][D_x]
  __shared__ float red[kThreads / 32][8 * kKwChannels];
  __shared__ bool is_last;
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (tid == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  griddep_launch_dependents();
  griddep_wait();
  if (warp == 0) {
    if (lane == 0) mbar_arrive_expect_tx(&bar, static_cast<uint32_t>(nch * row_bytes));
    __syncwarp();
    for (int c = lane; c < nch; c += 32) {
      const int ch = c0 + c;
      const __nv_bfloat16* src = (ch < D) ? P.w_k + static_cast<size_t>(ch) * P.D_x
                                          : P.w_proj + static_cast<size_t>(ch - D) * P.D_x;
      bulk_g2s(sWk + static_cast<size_t>(c) * P.D_x, src, static_cast<uint32_t>(row_bytes), &bar);
    }
  }
  // inputs of the last CTA's epilogue
  if (tid < D) {
    pre.gamma[tid] = __ldg(P.ln_gamma + tid);
    pre.beta[tid] = __ldg(P.ln_beta + tid);
  }
  if (tid >= D && tid - D < T) pre.slot[tid - D] = __ldg(P.slot + (tid - D));
  prefetch_rope(P, pre, tid);

  mbar_wait(&bar, 0, P.err, &abort_flag);
  // Tokens in blocks of 8: each thread owns 16-byte column chunks of the
  // weight rows (read once per block from shared memory) and streams the
  // matching x chunks of the block's tokens from L2.
  constexpr int kTB = 8;
  for (int tb = 0; tb < T; tb += kTB) {
    float acc[kTB][kKwChannels];
#pragma unroll
    for (int t = 0; t < kTB; ++t)
#pragma unroll
      for (int c = 0; c < kKwChannels; ++c) acc[t][c] = 0.f;
    // x chunks of the block's tokens, one iteration ahead (rows past T repeat
    // the last row; their sums are discarded)
    auto load_x = [&](int k, uint4 (&xv)[kTB]) {
#pragma unroll
      for (int t = 0; t < kTB; ++t)
        xv[t] = __ldg(reinterpret_cast<const uint4*>(P.x + static_cast<size_t>(min(tb + t, T - 1)) * P.D_x + k));
    };
    uint4 xnext[kTB];
    if (tid * 8 < P.D_x) load_x(tid * 8, xnext);
    for (int k = tid * 8; k < P.D_x; k += kThreads * 8) {
      uint4 xv[kTB];
#pragma unroll
      for (int t = 0; t < kTB; ++t) xv[t] = xnext[t];
      if (k + kThreads * 8 < P.D_x) load_x(k + kThreads * 8, xnext);
      float wf[kKwChannels][8];
#pragma unroll
      for (int c = 0; c < kKwChannels; ++c) {
        uint4 wv = make_uint4(0, 0, 0, 0);
        if (c < nch) wv = *reinterpret_cast<const uint4*>(sWk + static_cast<size_t>(c) * P.D_x + k);
        const __nv_bfloat162* w2 = reinterpret_cast<const __nv_bfloat162*>(&wv);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 f = __bfloat1622float2(w2[j]);
          wf[c][2 * j] = f.x;
          wf[c][2 * j + 1] = f.y;
        }
      }
#pragma unroll
      for (int t = 0; t < kTB; ++t) {
        const __nv_bfloat162* x2 = reinterpret_cast<const __nv_bfloat162*>(&xv[t]);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 f = __bfloat1622float2(x2[j]);
#pragma unroll
          for (int c = 0; c < kKwChannels; ++c) {
            acc[t][c] = fmaf(f.x, wf[c][2 * j], acc[t][c]);
            acc[t][c] = fmaf(f.y, wf[c][2 * j + 1], acc[t][c]);
          }
        }
      }
    }
    // Block reduction of every (token, channel) sum of this token block.
#pragma unroll
    for (int t = 0; t < kTB; ++t) {
      if (tb + t < T) {
#pragma unroll
        for (int c = 0; c < kKwChannels; ++c) {
          const float sum = warp_sum(acc[t][c]);
          if (lane == 0) red[warp][t * kKwChannels + c] = sum;
        }
      }
    }
    __syncthreads();
    for (int i = tid; i < kTB * kKwChannels; i += kThreads) {
      const int t = i / kKwChannels, c = i % kKwChannels;
      if (tb + t < T && c < nch) {
        float sum = 0.f;
#pragma unroll
        for (int w = 0; w < kThreads / 32; ++w) sum += red[w][i];
        P.kw[static_cast<size_t>(tb + t) * P.n_kw_channels + c0 + c] = sum;
      }
    }
    __syncthreads();
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) is_last = (atomicAdd(P.ticket, 1u) == static_cast<uint32_t>(P.n_kw_ctas - 1));
  __syncthreads();
  if (!is_last) return;
  __threadfence();

  // Last CTA: LayerNorm -> RoPE -> Hadamard -> quant for every token's key.
  for (int t = warp; t < T; t += kThreads / 32) {
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
  if (tid == 0) *P.ticket = 0u;  // ready for the next call
}

template <int DPL, int TM>
__global__ void __launch_bounds__(kThreads, 1) prolog_kernel(const PrologParams P) {
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ Pre pre;
  if (static_cast<int>(blockIdx.x) < P.n_q_ctas) {
    q_stream<DPL, TM>(P, smem, pre);
  } else {
    kw_stream<DPL>(P, smem, pre);
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
  P.n_kw_ctas = (P.n_kw_channels + kKwChannels - 1) / kKwChannels;
  P.q_lora = a.q_lora; P.q_lora_scale = reinterpret_cast<const __half*>(a.q_lora_scale);
  P.w_qb = a.w_qb; P.w_qb_scale = reinterpret_cast<const __half*>(a.w_qb_scale);
  P.x = reinterpret_cast<const __nv_bfloat16*>(a.x);
  P.w_k = reinterpret_cast<const __nv_bfloat16*>(a.w_k);
  P.ln_gamma = a.ln_gamma; P.ln_beta = a.ln_beta; P.ln_eps = a.ln_eps;
  P.w_proj = reinterpret_cast<const __nv_bfloat16*>(a.w_proj); P.w_scale = a.w_scale;
  P.pos = a.pos; P.rope_cos = a.rope_cos; P.rope_sin = a.rope_sin;
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
  const size_t smem_kw = static_cast<size_t>(kKwChannels) * a.D_x * 2;
  const size_t smem = smem_q > smem_kw ? smem_q : smem_kw;
  const int grid = P.n_q_ctas + static_cast<int>(round_up(P.n_kw_ctas, kQSplit));
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kQSplit;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e;
  auto go = [&](auto kern) {
    cudaError_t r = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    return r == cudaSuccess ? cudaLaunchKernelEx(&cfg, kern, P) : r;
  };
  const int tm = a.T <= 8 ? 8 : (a.T <= 16 ? 16 : 32);
  if (a.d_I == 128) {
    e = tm == 8 ? go(prolog_kernel<4, 8>) : (tm == 16 ? go(prolog_kernel<4, 16>) : go(prolog_kernel<4, 32>));
  } else {
    e = tm == 8 ? go(prolog_kernel<2, 8>) : (tm == 16 ? go(prolog_kernel<2, 16>) : go(prolog_kernel<2, 32>));
  }
  return cuda_status(e);
}

}  // namespace dsa

// Indexer Prolog: the q stream (int8 GEMM + dequant, RoPE, Hadamard,
// DynamicQuant), the k stream (bf16 GEMM, LayerNorm, RoPE, Hadamard,
// DynamicQuant, cache scatter) and the optional weight stream, in one launch.
//
// [V3.2-PyPTO §Indexer Prolog] gives the three formulas and observes that
// the q stream (an (8,1536)x(1536,8192) int8 GEMM) dominates and is bound by
// weight traffic.  At T <= 32 tokens every output channel is a 1536-long dot
// against <= 32 activation rows: the work is a weight stream, not a GEMM
// that tensor cores would speed up, so it runs as dp4a over shared-memory
// tiles filled by bulk async copies, spread over every SM:
//
//   * q stream: a cluster of 4 CTAs per head splits K_q in 4; each CTA
//     streams its [d_I x K_q/4] weight slab into shared memory with
//     cp.async.bulk, computes int32 partial dots, and the cluster sums the
//     4 partials through distributed shared memory.  Each CTA then finishes
//     the tokens t = rank (mod 4): dequant -> RoPE -> 128-point Hadamard
//     (warp butterfly over shuffles) -> int8 quantisation.
//   * k / weight streams: 2 output channels per CTA over the full D_x; the
//     fp32 results go to the workspace and the last CTA to finish (atomic
//     ticket) runs LayerNorm -> RoPE -> Hadamard -> quantisation and writes
//     the key-cache rows and the weights.
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include "dsa_internal.h"
#include "dsa_ptx.cuh"

namespace dsa {
namespace {

constexpr int kThreads = 256;
constexpr int kQSplit = 4;  // cluster size and K_q split of the q stream
constexpr int kKwChannels = 2;
constexpr int kMaxT = 32;

struct PrologParams {
  int T, H_I, d_I, d_rope, K_q, D_x, rope_max_pos, interleaved, n_q_ctas, n_kw_ctas, n_kw_channels;
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

// One warp holds one d_I = 32*DPL row, lane l owning dims l*DPL .. l*DPL+DPL-1.
// Applies RoPE (table row `p`), the scaled Sylvester Hadamard transform and
// the int8 quantisation; returns the codes in c[] and the fp16 scale.
template <int DPL>
__device__ __forceinline__ void rope_hadamard_quant(float (&v)[DPL], int lane, int p, const float* cos_t,
                                                    const float* sin_t, int d_rope, int interleaved,
                                                    int (&c)[DPL], __half& scale16) {
  const int half = d_rope / 2;
  const float* crow = cos_t + static_cast<size_t>(p) * half;
  const float* srow = sin_t + static_cast<size_t>(p) * half;
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
template <int DPL>
__device__ void q_stream(const PrologParams& P, uint8_t* smem) {
  constexpr int D = 32 * DPL;           // d_I
  constexpr int TG = kThreads / D;      // token groups per channel
  constexpr int TPT = kMaxT / TG;       // max tokens per thread
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int head = blockIdx.x / kQSplit;
  const uint32_t rank = cluster_ctarank();
  const int kchunk = P.K_q / kQSplit;
  const int wstride = kchunk + 16;
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
  mbar_wait(&bar, 0, P.err, &abort_flag);

  // int32 partial dots over this CTA's K_q slice.
  const int n = tid % D, tg = tid / D;
  int acc[TPT];
#pragma unroll
  for (int i = 0; i < TPT; ++i) acc[i] = 0;
  const uint8_t* wrow = sW + n * wstride;
  for (int k = 0; k < kchunk; k += 16) {
    const int4 w = *reinterpret_cast<const int4*>(wrow + k);
#pragma unroll
    for (int i = 0; i < TPT; ++i) {
      const int t = tg + i * TG;
      if (t < T) {
        const int4 q = *reinterpret_cast<const int4*>(sQ + t * kchunk + k);
        acc[i] = __dp4a(w.x, q.x, acc[i]);
        acc[i] = __dp4a(w.y, q.y, acc[i]);
        acc[i] = __dp4a(w.z, q.z, acc[i]);
        acc[i] = __dp4a(w.w, q.w, acc[i]);
      }
    }
  }
#pragma unroll
  for (int i = 0; i < TPT; ++i) {
    const int t = tg + i * TG;
    if (t < T) sPart[t * D + n] = acc[i];
  }
  cluster_sync();

  // Tokens t = rank (mod kQSplit): sum the cluster's partials, then the
  // dequant -> RoPE -> Hadamard -> quant epilogue, one warp per token.
  for (int t = rank + kQSplit * warp; t < T; t += kQSplit * (kThreads / 32)) {
    float v[DPL];
    const float sa = __half2float(P.q_lora_scale[t]);
#pragma unroll
    for (int j = 0; j < DPL; ++j) {
      const int d = lane * DPL + j;
      const uint32_t local = smem_u32(&sPart[t * D + d]);
      int s = 0;
#pragma unroll
      for (int r = 0; r < kQSplit; ++r) s += static_cast<int>(ld_cluster_u32(mapa(local, r)));
      const float sb = __half2float(P.w_qb_scale[head * D + d]);
      v[j] = (static_cast<float>(s) * sa) * sb;
    }
    int c[DPL];
    __half s16;
    rope_hadamard_quant<DPL>(v, lane, P.pos[t], P.rope_cos, P.rope_sin, P.d_rope, P.interleaved, c, s16);
    store_codes<DPL>(P.q_out + (static_cast<size_t>(t) * P.H_I + head) * D + lane * DPL, c);
    if (lane == 0) P.q_scale_out[t * P.H_I + head] = s16;
  }
  cluster_sync();  // peers may still read this CTA's partials
}

// ------------------------------------------------------- k / weight stream
template <int DPL>
__device__ void kw_stream(const PrologParams& P) {
  constexpr int D = 32 * DPL;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int cta = blockIdx.x - P.n_q_ctas;
  if (cta >= P.n_kw_ctas) return;
  const int T = P.T;
  const int c0 = cta * kKwChannels;
  __shared__ float red[kThreads / 32][kMaxT * kKwChannels];
  __shared__ bool is_last;
  griddep_wait();

  float acc[kMaxT][kKwChannels];
#pragma unroll
  for (int t = 0; t < kMaxT; ++t)
#pragma unroll
    for (int c = 0; c < kKwChannels; ++c) acc[t][c] = 0.f;

  const __nv_bfloat16* wrow[kKwChannels];
  bool cvalid[kKwChannels];
#pragma unroll
  for (int c = 0; c < kKwChannels; ++c) {
    const int ch = c0 + c;
    cvalid[c] = ch < P.n_kw_channels;
    const int chc = cvalid[c] ? ch : 0;
    wrow[c] = (chc < D) ? P.w_k + static_cast<size_t>(chc) * P.D_x
                        : P.w_proj + static_cast<size_t>(chc - D) * P.D_x;
  }
  for (int k = tid * 8; k < P.D_x; k += kThreads * 8) {
    float wf[kKwChannels][8];
#pragma unroll
    for (int c = 0; c < kKwChannels; ++c) {
      const uint4 wv = __ldg(reinterpret_cast<const uint4*>(wrow[c] + k));
      const __nv_bfloat162* w2 = reinterpret_cast<const __nv_bfloat162*>(&wv);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 f = __bfloat1622float2(w2[j]);
        wf[c][2 * j] = f.x;
        wf[c][2 * j + 1] = f.y;
      }
    }
#pragma unroll
    for (int t = 0; t < kMaxT; ++t) {
      if (t < T) {
        const uint4 xv = __ldg(reinterpret_cast<const uint4*>(P.x + static_cast<size_t>(t) * P.D_x + k));
        const __nv_bfloat162* x2 = reinterpret_cast<const __nv_bfloat162*>(&xv);
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
  }
  // Block reduction of every (token, channel) sum.
#pragma unroll
  for (int t = 0; t < kMaxT; ++t) {
    if (t < T) {
#pragma unroll
      for (int c = 0; c < kKwChannels; ++c) {
        const float s = warp_sum(acc[t][c]);
        if (lane == 0) red[warp][t * kKwChannels + c] = s;
      }
    }
  }
  __syncthreads();
  for (int i = tid; i < T * kKwChannels; i += kThreads) {
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) s += red[w][i];
    const int t = i / kKwChannels, c = i % kKwChannels;
    if (c0 + c < P.n_kw_channels) P.kw[static_cast<size_t>(t) * P.n_kw_channels + c0 + c] = s;
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
      v[j] = (v[j] - mean) * rstd * P.ln_gamma[d] + P.ln_beta[d];
    }
    int c[DPL];
    __half s16;
    rope_hadamard_quant<DPL>(v, lane, P.pos[t], P.rope_cos, P.rope_sin, P.d_rope, P.interleaved, c, s16);
    const int64_t row = P.slot[t];
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

template <int DPL>
__global__ void __launch_bounds__(kThreads) prolog_kernel(const PrologParams P) {
  extern __shared__ __align__(16) uint8_t smem[];
  if (static_cast<int>(blockIdx.x) < P.n_q_ctas) {
    q_stream<DPL>(P, smem);
  } else {
    kw_stream<DPL>(P);
  }
  griddep_launch_dependents();
}

}  // namespace

size_t prolog_workspace(const dsa_prolog_args& a) {
  const int nch = a.d_I + (a.w_proj ? a.H_I : 0);
  return 256 + round_up(static_cast<size_t>(a.T) * nch * sizeof(float), 256);
}

int launch_prolog(const dsa_prolog_args& a, void* ws, cudaStream_t stream) {
  PrologParams P{};
  P.T = a.T; P.H_I = a.H_I; P.d_I = a.d_I; P.d_rope = a.d_rope; P.K_q = a.K_q; P.D_x = a.D_x;
  P.rope_max_pos = a.rope_max_pos; P.interleaved = a.rope_interleaved;
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
  const size_t smem = static_cast<size_t>(a.d_I) * (kchunk + 16) + static_cast<size_t>(kMaxT) * kchunk +
                      static_cast<size_t>(kMaxT) * a.d_I * 4;
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
  if (a.d_I == 128) {
    e = cudaFuncSetAttribute(prolog_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess) e = cudaLaunchKernelEx(&cfg, prolog_kernel<4>, P);
  } else {
    e = cudaFuncSetAttribute(prolog_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess) e = cudaLaunchKernelEx(&cfg, prolog_kernel<2>, P);
  }
  return cuda_status(e);
}

}  // namespace dsa

// Activation Quantization, the standalone operator of [V4-TileLang
// §Activation Quantization] steps 1-4: per row of x (bf16 [M, N]) the
// maximum of |x| in fp32, scale = max / 127 (with round_scale the power of
// two at or above it), y = rint(clamp(x / scale, -127, 127)) as int8, and
// the fp32 scale written back.
//
// One CTA per row: the row is read from HBM once into shared memory (the
// first pass reduces its maximum while it lands), and quantised from there,
// so the kernel moves 2 bytes in and 1 byte out per element.  The quotient
// is an IEEE fp32 division and the power of two comes from frexp/ldexp
// (both exact), so the codes equal a host fp32 computation bit for bit.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include "dsa_internal.h"
#include "dsa_ptx.cuh"
#include "w8tc.cuh"

namespace dsa {
namespace {

constexpr int kQThreads = 256;

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// The code of v: rint of the IEEE fp32 quotient v / s, clamped.  (Products
// with 1/s, even with an exact division near ties, measured slower.)
__device__ __forceinline__ uint32_t quant4(float a, float b, float c, float d, float s) {
  auto q = [s](float v) -> uint32_t {
    const float t = fminf(fmaxf(v / s, -127.f), 127.f);
    return static_cast<uint32_t>(__float2int_rn(t)) & 0xffu;
  };
  if (!(s > 0.f)) return 0u;
  return q(a) | (q(b) << 8) | (q(c) << 16) | (q(d) << 24);
}

__global__ void __launch_bounds__(kQThreads) act_quant_kernel(const uint16_t* __restrict__ x, int8_t* __restrict__ y,
                                                              float* __restrict__ scale, int N, int round_scale) {
  extern __shared__ uint4 srow[];  // the row: N / 8 chunks of 8 bf16
  __shared__ float wmax[kQThreads / 32];
  const int row = blockIdx.x;
  const int nv = N / 8;
  const uint4* xr = reinterpret_cast<const uint4*>(x + static_cast<size_t>(row) * N);
  float amax = 0.f;
  for (int i = threadIdx.x; i < nv; i += kQThreads) {
    const uint4 v = __ldcs(xr + i);  // read once: streaming
    srow[i] = v;
    amax = fmaxf(amax, fmaxf(fmaxf(fabsf(bf16_lo(v.x)), fabsf(bf16_hi(v.x))), fmaxf(fabsf(bf16_lo(v.y)), fabsf(bf16_hi(v.y)))));
    amax = fmaxf(amax, fmaxf(fmaxf(fabsf(bf16_lo(v.z)), fabsf(bf16_hi(v.z))), fmaxf(fabsf(bf16_lo(v.w)), fabsf(bf16_hi(v.w)))));
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = wmax[0];
#pragma unroll
  for (int w = 1; w < kQThreads / 32; ++w) amax = fmaxf(amax, wmax[w]);
  float s = amax / 127.f;
  if (round_scale && s > 0.f) {
    int e;
    const float m = frexpf(s, &e);  // s = m * 2^e, m in [0.5, 1)
    s = ldexpf(1.f, m == 0.5f ? e - 1 : e);
  }
  if (threadIdx.x == 0) scale[row] = s;
  uint2* yr = reinterpret_cast<uint2*>(y + static_cast<size_t>(row) * N);
  for (int i = threadIdx.x; i < nv; i += kQThreads) {
    const uint4 v = srow[i];
    uint2 o;
    o.x = quant4(bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y), s);
    o.y = quant4(bf16_lo(v.z), bf16_hi(v.z), bf16_lo(v.w), bf16_hi(v.w), s);
    __stcs(yr + i, o);
  }
}

// ---------------------------------------------------------------------- mHC
// [V4-TileLang §Manifold-Constrained Hyper-Connections] steps 1-5 for hc
// streams: per token, mixes [hc (2 + hc)] -> pre [hc], post [hc], comb
// [hc, hc] (row-major).  One thread per token, everything in registers in
// fp32: scale + base, the sigmoids, the row softmax + eps, then the column /
// row / column Sinkhorn-Knopp normalisations.  The 20-round normalisation
// makes the kernel issue-bound, so the memory side is kept to the fewest
// instructions: each thread moves its own rows with 16-byte accesses (a row
// is a whole number of float4) and L1 absorbs the 96- / 320-byte stride
// between the lanes of a warp.
constexpr int kMhcTokens = 128;

// The hardware reciprocal (one multi-function-unit instruction, relative
// error below 2^-22) for the Sinkhorn normalisations: each pass divides by
// a row or column sum, and the correctly rounded reciprocal costs several
// instructions more per division in a kernel bound by instruction issue.
__device__ __forceinline__ float rcp_fast(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int HC>
__global__ void __launch_bounds__(kMhcTokens) mhc_kernel(const float* __restrict__ mixes, const float* __restrict__ hc_scale,
                                                         const float* __restrict__ hc_base, float* __restrict__ pre,
                                                         float* __restrict__ post, float* __restrict__ comb, int n,
                                                         int iters, float eps) {
  constexpr int W = HC * (2 + HC);
  static_assert(W % 4 == 0 && HC % 4 == 0, "rows must be whole float4");
  const int t = blockIdx.x * kMhcTokens + threadIdx.x;
  if (t >= n) return;
  float z[W];
  const float4* src = reinterpret_cast<const float4*>(mixes + static_cast<size_t>(t) * W);
#pragma unroll
  for (int v = 0; v < W / 4; ++v) {
    const float4 q = __ldg(src + v);
    z[4 * v] = q.x;
    z[4 * v + 1] = q.y;
    z[4 * v + 2] = q.z;
    z[4 * v + 3] = q.w;
  }
  const float s0 = __ldg(hc_scale), s1 = __ldg(hc_scale + 1), s2 = __ldg(hc_scale + 2);
  float pr[HC], po[HC], c[HC][HC];
#pragma unroll
  for (int i = 0; i < HC; ++i) {
    const float zp = z[i] * s0 + __ldg(hc_base + i);
    const float zq = z[HC + i] * s1 + __ldg(hc_base + HC + i);
    pr[i] = 1.f / (1.f + expf(-zp)) + eps;
    po[i] = 2.f / (1.f + expf(-zq));
  }
#pragma unroll
  for (int i = 0; i < HC; ++i) {
    float m = -3.402823466e38f;
#pragma unroll
    for (int j = 0; j < HC; ++j) {
      c[i][j] = z[2 * HC + i * HC + j] * s2 + __ldg(hc_base + 2 * HC + i * HC + j);
      m = fmaxf(m, c[i][j]);
    }
    float sum = 0.f;
#pragma unroll
    for (int j = 0; j < HC; ++j) {
      c[i][j] = expf(c[i][j] - m);
      sum += c[i][j];
    }
    const float inv = 1.f / sum;
#pragma unroll
    for (int j = 0; j < HC; ++j) c[i][j] = c[i][j] * inv + eps;
  }
  auto col_norm = [&]() {
#pragma unroll
    for (int j = 0; j < HC; ++j) {
      float sum = 0.f;
#pragma unroll
      for (int i = 0; i < HC; ++i) sum += c[i][j];
      const float inv = rcp_fast(sum + eps);
#pragma unroll
      for (int i = 0; i < HC; ++i) c[i][j] *= inv;
    }
  };
  col_norm();
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int i = 0; i < HC; ++i) {
      float sum = 0.f;
#pragma unroll
      for (int j = 0; j < HC; ++j) sum += c[i][j];
      const float inv = rcp_fast(sum + eps);
#pragma unroll
      for (int j = 0; j < HC; ++j) c[i][j] *= inv;
    }
    col_norm();
  }
  float4* dpre = reinterpret_cast<float4*>(pre + static_cast<size_t>(t) * HC);
  float4* dpost = reinterpret_cast<float4*>(post + static_cast<size_t>(t) * HC);
  float4* dcomb = reinterpret_cast<float4*>(comb + static_cast<size_t>(t) * HC * HC);
#pragma unroll
  for (int v = 0; v < HC / 4; ++v) {
    dpre[v] = make_float4(pr[4 * v], pr[4 * v + 1], pr[4 * v + 2], pr[4 * v + 3]);
    dpost[v] = make_float4(po[4 * v], po[4 * v + 1], po[4 * v + 2], po[4 * v + 3]);
  }
#pragma unroll
  for (int i = 0; i < HC; ++i)
#pragma unroll
    for (int v = 0; v < HC / 4; ++v)
      dcomb[i * (HC / 4) + v] = make_float4(c[i][4 * v], c[i][4 * v + 1], c[i][4 * v + 2], c[i][4 * v + 3]);
}

}  // namespace

int launch_mhc(const dsa_mhc_args& a, cudaStream_t s) {
  const dim3 grid((a.n + kMhcTokens - 1) / kMhcTokens);
  if (a.hc == 4)
    mhc_kernel<4><<<grid, kMhcTokens, 0, s>>>(a.mixes, a.hc_scale, a.hc_base, a.pre, a.post, a.comb, a.n, a.iters,
                                              a.eps);
  else
    mhc_kernel<8><<<grid, kMhcTokens, 0, s>>>(a.mixes, a.hc_scale, a.hc_base, a.pre, a.post, a.comb, a.n, a.iters,
                                              a.eps);
  return cuda_status(cudaGetLastError());
}

// ---------------------------------------------------------------- int8 GEMM
// [V4-TileLang §Int8 General Matrix Multiplication] steps 1-4 for the
// decode regime (M <= 32 activation rows): c[m, n] = fp16(sum_k a[m,k]
// b[n,k] * a_scale[m] * b_scale[n]).  With so few rows every weight byte is
// used at most 32 times, so the product is a weight stream, run on the
// tensor cores with the weights as the MMA's M dimension (w8tc.cuh).

// c[t, n] = fp16(s * a_scale[t] * b_scale[n]), the product in that order.
struct GemmWtJob {
  int M, N, K;
  uint32_t* err;
  const float* a_scale;
  const float* b_scale;
  __half* c;
  __device__ __forceinline__ float tok_scale(int t) const { return __ldg(a_scale + t); }
  __device__ __forceinline__ float row_scale(int n) const { return __ldg(b_scale + n); }
  __device__ __forceinline__ void put(int t, int n, int s, float st, float sn) const {
    c[static_cast<size_t>(t) * N + n] = __float2half_rn(static_cast<float>(s) * st * sn);
  }
  __device__ __forceinline__ void prologue(int, int, int8_t*) const {}
  __device__ __forceinline__ void tail(int, int) const {}
};

// Shared memory the weight-stream GEMM's ring may fill (it runs alone).
constexpr size_t kWtSmemBudget = 220 * 1024;

int launch_int8_gemm_wt(const dsa_int8_gemm_args& a, cudaStream_t s) {
  uint32_t* err = error_word();
  if (!err) return DSA_ERR_CUDA;
  if (a.M > 32) return DSA_ERR_UNSUPPORTED;
  const int NT = a.M <= 16 ? 16 : 32;
  alignas(64) WtMaps maps;
  const uint64_t st[1] = {static_cast<uint64_t>(a.K)};
  const uint64_t da[2] = {static_cast<uint64_t>(a.K), static_cast<uint64_t>(a.M)};
  const uint32_t bt[2] = {kWtK, static_cast<uint32_t>(NT)};
  if (!wt_encode_weights(maps, a.b, a.N, a.K) || !encode_tmap(&maps.tok, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, a.a, da, st, bt, 128))
    return DSA_ERR_CUDA;
  const GemmWtJob job{a.M, a.N, a.K, err, a.a_scale, a.b_scale, reinterpret_cast<__half*>(a.c)};
  const long long units = (static_cast<long long>(a.N) + kWtUnit - 1) / kWtUnit;
  const int grid = static_cast<int>(units < sm_count() ? units : sm_count());
  auto go = [&](auto kern, auto layout) {
    using L = decltype(layout);
    const int ns8 = L::stages(a.K, kWtSmemBudget);
    const size_t smem = L::smem(a.K, ns8);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    kern<<<grid, kWtThreads, smem, s>>>(maps, job, ns8);
    return cudaGetLastError();
  };
  const cudaError_t e = NT == 16 ? go(wt_kernel<16, false, GemmWtJob>, WtLayout<16, false>{})
                                 : go(wt_kernel<32, false, GemmWtJob>, WtLayout<32, false>{});
  return cuda_status(e);
}

int launch_act_quant(const dsa_act_quant_args& a, cudaStream_t s) {
  const size_t smem = static_cast<size_t>(a.N) * 2;
  cudaError_t e = cudaSuccess;
  if (smem > 48 * 1024)
    e = cudaFuncSetAttribute(act_quant_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return cuda_status(e);
  act_quant_kernel<<<a.M, kQThreads, smem, s>>>(a.x, a.y, a.scale, a.N, a.round_scale);
  return cuda_status(cudaGetLastError());
}

}  // namespace dsa

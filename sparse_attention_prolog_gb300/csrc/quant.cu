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
#include <cuda_runtime.h>
#include "dsa_internal.h"

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

}  // namespace

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

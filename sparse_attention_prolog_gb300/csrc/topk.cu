// Per-row top-k of the Lightning Indexer scores by radix select.
//
// [V3.2-PyPTO §Lightning Indexer] reports the final TopK as a single-core
// sort-and-merge with a long tail and proposes to sort earlier and only
// merge at the end.  A GPU has no such tail problem per row if the row is
// selected, not sorted: an exact radix select over the order-preserving
// 32-bit image of the fp32 scores finds the k-th largest key in three
// digit passes (11, 11, 10 bits) with shared-memory histograms, then one
// pass emits every key above the threshold and as many threshold-equal keys
// as are still missing.  The output is the set (order unspecified), -1
// padded when the row has fewer than k visible keys.
//
// A row is split over a cluster of CTAs (up to 8) whose histograms are
// summed through distributed shared memory, so long rows (64K-128K keys)
// use several SMs while short rows (prefill) use one CTA each.
#include <cuda_runtime.h>
#include "dsa_internal.h"
#include "dsa_ptx.cuh"

namespace dsa {
namespace {

constexpr int kThreads = 1024;
constexpr int kBins = 2048;

__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

struct TopkParams {
  const float* scores;
  int64_t ld;
  const int32_t* pos;
  int max_L, topk;
  int32_t* out;
};

// Block-wide search from the top bin: finds the bin b at which the running
// count (from the highest bin down) first reaches `need`; returns b and the
// count strictly above it.
__device__ __forceinline__ void find_bin(const uint32_t* hist, uint32_t need, int& bin, uint32_t& above,
                                         uint32_t* scratch /*[kThreads/32 + 2]*/) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int per = kBins / kThreads;  // 2 bins per thread, thread 0 = highest
  uint32_t mine[per];
  uint32_t s = 0;
#pragma unroll
  for (int i = 0; i < per; ++i) {
    mine[i] = hist[kBins - 1 - (tid * per + i)];
    s += mine[i];
  }
  // inclusive warp scan
  uint32_t incl = s;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) scratch[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    uint32_t w = (lane < kThreads / 32) ? scratch[lane] : 0;
    uint32_t wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t n = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += n;
    }
    if (lane < kThreads / 32) scratch[lane] = wi - w;  // exclusive warp offsets
  }
  __syncthreads();
  uint32_t before = scratch[warp] + incl - s;
#pragma unroll
  for (int i = 0; i < per; ++i) {
    if (before < need && before + mine[i] >= need) {
      scratch[kThreads / 32] = kBins - 1 - (tid * per + i);
      scratch[kThreads / 32 + 1] = before;
    }
    before += mine[i];
  }
  __syncthreads();
  bin = static_cast<int>(scratch[kThreads / 32]);
  above = scratch[kThreads / 32 + 1];
  __syncthreads();
}

// Cluster of CS CTAs per row; CTA r of the cluster owns the contiguous
// slice [r*chunk, (r+1)*chunk) of the row's visible keys.
template <int CS>
__global__ void __launch_bounds__(kThreads) topk_kernel(const TopkParams P) {
  __shared__ uint32_t hist[kBins];
  __shared__ uint32_t total[kBins];
  __shared__ uint32_t scratch[kThreads / 32 + 2];
  __shared__ uint32_t cnt_gt, cnt_eq, base_gt, base_eq;
  const int tid = threadIdx.x;
  const int row = blockIdx.x / CS;
  const uint32_t rank = (CS > 1) ? cluster_ctarank() : 0;
  griddep_wait();
  const int n_valid = min(P.pos[row] + 1, P.max_L);
  const int k = P.topk;
  int32_t* out = P.out + static_cast<size_t>(row) * k;
  const float* src = P.scores + static_cast<size_t>(row) * P.ld;

  if (n_valid <= k) {  // the whole visible row is the answer
    if (rank == 0) {
      for (int i = tid; i < k; i += kThreads) out[i] = (i < n_valid) ? i : -1;
    }
    return;  // uniform across the cluster: no cluster barrier is pending
  }
  const int chunk = (n_valid + CS - 1) / CS;
  const int lo = rank * chunk, hi = min(n_valid, lo + chunk);

  uint32_t prefix = 0, prefix_mask = 0;
  uint32_t need = static_cast<uint32_t>(k);
  const int shifts[3] = {21, 10, 0};
  const int widths[3] = {11, 11, 10};
  for (int pass = 0; pass < 3; ++pass) {
    const int sh = shifts[pass];
    const uint32_t dmask = (1u << widths[pass]) - 1u;
    for (int i = tid; i < kBins; i += kThreads) hist[i] = 0;
    __syncthreads();
    for (int i = lo + tid; i < hi; i += kThreads) {
      const uint32_t key = order_key(src[i]);
      if ((key & prefix_mask) == prefix) atomicAdd(&hist[(key >> sh) & dmask], 1u);
    }
    __syncthreads();
    if (CS > 1) {
      cluster_sync();
      for (int i = tid; i < kBins; i += kThreads) {
        const uint32_t a = smem_u32(&hist[i]);
        uint32_t s = 0;
#pragma unroll
        for (int r = 0; r < CS; ++r) s += ld_cluster_u32(mapa(a, r));
        total[i] = s;
      }
      cluster_sync();
    } else {
      for (int i = tid; i < kBins; i += kThreads) total[i] = hist[i];
      __syncthreads();
    }
    int bin;
    uint32_t above;
    find_bin(total, need, bin, above, scratch);
    need -= above;
    prefix |= static_cast<uint32_t>(bin) << sh;
    prefix_mask |= dmask << sh;
  }
  // prefix is now the exact k-th largest key; `need` keys equal to it are
  // taken, all keys above it are taken.
  const uint32_t thr = prefix;
  const uint32_t n_gt = static_cast<uint32_t>(k) - need;
  if (tid == 0) { cnt_gt = 0; cnt_eq = 0; }
  __syncthreads();
  for (int i = lo + tid; i < hi; i += kThreads) {
    const uint32_t key = order_key(src[i]);
    if (key > thr) atomicAdd(&cnt_gt, 1u);
    else if (key == thr) atomicAdd(&cnt_eq, 1u);
  }
  __syncthreads();
  // Exclusive offsets of this CTA among the cluster (ranks below it).
  if (CS > 1) {
    cluster_sync();
    if (tid == 0) {
      uint32_t g = 0, e = 0;
      for (uint32_t r = 0; r < rank; ++r) {
        g += ld_cluster_u32(mapa(smem_u32(&cnt_gt), r));
        e += ld_cluster_u32(mapa(smem_u32(&cnt_eq), r));
      }
      base_gt = g;
      base_eq = e;
    }
    cluster_sync();
  } else {
    if (tid == 0) { base_gt = 0; base_eq = 0; }
  }
  __syncthreads();
  if (tid == 0) { cnt_gt = 0; cnt_eq = 0; }
  __syncthreads();
  for (int i = lo + tid; i < hi; i += kThreads) {
    const uint32_t key = order_key(src[i]);
    if (key > thr) {
      const uint32_t p = base_gt + atomicAdd(&cnt_gt, 1u);
      out[p] = i;
    } else if (key == thr) {
      const uint32_t e = base_eq + atomicAdd(&cnt_eq, 1u);
      if (e < need) out[n_gt + e] = i;
    }
  }
  if (CS > 1) cluster_sync();  // keep counters alive for the peers' reads
}

template <int CS>
cudaError_t launch_cs(const TopkParams& P, int T, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (CS > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = CS;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[na].val.programmaticStreamSerializationAllowed = 1;
  ++na;
  cfg.gridDim = dim3(T * CS);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, topk_kernel<CS>, P);
}

}  // namespace

int launch_topk(const dsa_topk_args& a, const float* scores, int64_t ld, cudaStream_t s) {
  TopkParams P{scores, ld, a.pos, a.max_L, a.topk, a.topk_idx};
  // Split long rows over a cluster so that each CTA scans <= ~8K keys.
  cudaError_t e;
  if (a.max_L > 32768) e = launch_cs<8>(P, a.T, s);
  else if (a.max_L > 16384) e = launch_cs<4>(P, a.T, s);
  else if (a.max_L > 8192) e = launch_cs<2>(P, a.T, s);
  else e = launch_cs<1>(P, a.T, s);
  return cuda_status(e);
}

}  // namespace dsa

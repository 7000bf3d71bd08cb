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

// Warp-aggregated slot reservation: returns base + rank of this lane among
// the lanes with `pred`.
__device__ __forceinline__ uint32_t warp_reserve(uint32_t* counter, bool pred) {
  const uint32_t m = __ballot_sync(0xffffffffu, pred);
  const int lane = threadIdx.x & 31;
  uint32_t base = 0;
  if (m != 0) {
    const int leader = __ffs(m) - 1;
    if (lane == leader) base = atomicAdd(counter, static_cast<uint32_t>(__popc(m)));
    base = __shfl_sync(0xffffffffu, base, leader);
  }
  return base + static_cast<uint32_t>(__popc(m & ((1u << lane) - 1u)));
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
// slice [r*chunk, (r+1)*chunk) of the row's visible keys.  A slice of up to
// kThreads * kPer keys stays in registers for all passes (one L2 read);
// longer slices are re-read for each pass.
constexpr int kPer = 16;

template <int CS>
__global__ void __launch_bounds__(kThreads) topk_kernel(const TopkParams P) {
  __shared__ uint32_t hist[kBins];
  __shared__ uint32_t total[kBins];
  __shared__ uint32_t scratch[kThreads / 32 + 2];
  __shared__ uint32_t cnt_gt, cnt_eq, base_gt, base_eq;
  const int tid = threadIdx.x;
  const int row = blockIdx.x / CS;
  const uint32_t rank = (CS > 1) ? cluster_ctarank() : 0;
  griddep_launch_dependents();
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
  const bool in_regs = (hi - lo) <= kThreads * kPer;
  uint32_t keys[kPer];
  if (in_regs) {
#pragma unroll
    for (int e = 0; e < kPer; ++e) {
      const int i = lo + tid + e * kThreads;
      keys[e] = (i < hi) ? order_key(src[i]) : 0u;
    }
  }

  uint32_t prefix = 0, prefix_mask = 0;
  uint32_t need = static_cast<uint32_t>(k);
#pragma unroll 1
  for (int pass = 0; pass < 3; ++pass) {
    const int sh = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
    const uint32_t dmask = pass == 2 ? 0x3FFu : 0x7FFu;
    for (int i = tid; i < kBins; i += kThreads) hist[i] = 0;
    __syncthreads();
    if (in_regs) {
#pragma unroll
      for (int e = 0; e < kPer; ++e) {
        const int i = lo + tid + e * kThreads;
        if (i < hi && (keys[e] & prefix_mask) == prefix) atomicAdd(&hist[(keys[e] >> sh) & dmask], 1u);
      }
    } else {
      for (int i0 = lo; i0 < hi; i0 += kThreads) {  // warp-uniform trip count
        const int i = i0 + tid;
        const uint32_t key = i < hi ? order_key(src[i]) : 0u;
        if (i < hi && (key & prefix_mask) == prefix) atomicAdd(&hist[(key >> sh) & dmask], 1u);
      }
    }
    __syncthreads();
    if (CS > 1) {
      // CTA r owns bins [r*kBins/CS, (r+1)*kBins/CS): it sums them over the
      // cluster; then every CTA reads the totals from their owners.
      cluster_sync();
      constexpr int kSlice = kBins / CS;
      for (int i = tid; i < kSlice; i += kThreads) {
        const int bin = static_cast<int>(rank) * kSlice + i;
        const uint32_t a = smem_u32(&hist[bin]);
        uint32_t v[CS];
#pragma unroll
        for (int r = 0; r < CS; ++r) v[r] = ld_cluster_u32(mapa(a, r));
        uint32_t sum = 0;
#pragma unroll
        for (int r = 0; r < CS; ++r) sum += v[r];
        total[bin] = sum;
      }
      cluster_sync();
      for (int i = tid; i < kBins; i += kThreads) {
        const uint32_t owner = static_cast<uint32_t>(i / kSlice);
        if (owner != rank) hist[i] = ld_cluster_u32(mapa(smem_u32(&total[i]), owner));
        else hist[i] = total[i];
      }
      cluster_sync();  // owners' totals may be overwritten next pass only now
      int bin;
      uint32_t above;
      find_bin(hist, need, bin, above, scratch);
      need -= above;
      prefix |= static_cast<uint32_t>(bin) << sh;
      prefix_mask |= dmask << sh;
    } else {
      int bin;
      uint32_t above;
      find_bin(hist, need, bin, above, scratch);
      need -= above;
      prefix |= static_cast<uint32_t>(bin) << sh;
      prefix_mask |= dmask << sh;
    }
  }
  // prefix is now the exact k-th largest key; `need` keys equal to it are
  // taken, all keys above it are taken.
  const uint32_t thr = prefix;
  const uint32_t n_gt = static_cast<uint32_t>(k) - need;
  if (tid == 0) { cnt_gt = 0; cnt_eq = 0; }
  __syncthreads();
  uint32_t my_gt = 0, my_eq = 0;
  if (in_regs) {
#pragma unroll
    for (int e = 0; e < kPer; ++e) {
      const int i = lo + tid + e * kThreads;
      if (i < hi) { my_gt += keys[e] > thr; my_eq += keys[e] == thr; }
    }
  } else {
    for (int i = lo + tid; i < hi; i += kThreads) {
      const uint32_t key = order_key(src[i]);
      my_gt += key > thr;
      my_eq += key == thr;
    }
  }
  if (my_gt) atomicAdd(&cnt_gt, my_gt);
  if (my_eq) atomicAdd(&cnt_eq, my_eq);
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
  // Output slots by warp-aggregated reservations.
  auto emit = [&](uint32_t key, int i, bool valid) {
    const bool gt = valid && key > thr;
    const bool eq = valid && key == thr;
    const uint32_t pg = warp_reserve(&cnt_gt, gt);
    const uint32_t pe = warp_reserve(&cnt_eq, eq);
    if (gt) out[base_gt + pg] = i;
    if (eq && base_eq + pe < need) out[n_gt + base_eq + pe] = i;
  };
  if (in_regs) {
#pragma unroll
    for (int e = 0; e < kPer; ++e) {
      const int i = lo + tid + e * kThreads;
      emit(keys[e], i, i < hi);
    }
  } else {
    for (int i0 = lo; i0 < hi; i0 += kThreads) {
      const int i = i0 + tid;
      emit(i < hi ? order_key(src[i]) : 0u, i, i < hi);
    }
  }
  if (CS > 1) cluster_sync();  // keep counters alive for the peers' reads
}


// ---------------------------------------------------------------------------
// Top-k with the leading digit known in advance.  The indexer has counted
// every row's visible scores by the leading 12 bits of their order key, so
// the k-th largest key's leading digit B and the number of keys above it
// follow from the histogram alone.  S CTAs share a row (<= 8192 keys each,
// held in registers): keys above B go straight to the output, keys inside B
// become candidates; the last CTA of the row (atomic ticket) selects the
// remaining ones among the candidates by the low 20 bits, then clears the
// row's histogram and counters for the next call.
constexpr int kHB = kTopkHistBins;

struct TopkHistParams {
  const float* scores;
  int64_t ld;
  const int32_t* pos;
  int max_L, topk, slices;
  int32_t* out;
  uint32_t* hist;  // [T][kHB]
  uint32_t* ctr;   // [T][4]: keys above B emitted, candidates, CTAs done
  uint2* cand;     // [T][kTopkCandCap]: (key, index)
  uint32_t* err;
};

// Exclusive block scan of (a, b) pairs; returns totals through ta, tb.
__device__ __forceinline__ void block_scan2(uint32_t a, uint32_t b, uint32_t& ea, uint32_t& eb, uint32_t& ta,
                                            uint32_t& tb, uint32_t* sh /*[2 * 33]*/) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t ia = a, ib = b;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t na = __shfl_up_sync(0xffffffffu, ia, o);
    const uint32_t nb = __shfl_up_sync(0xffffffffu, ib, o);
    if (lane >= o) { ia += na; ib += nb; }
  }
  if (lane == 31) { sh[warp] = ia; sh[33 + warp] = ib; }
  __syncthreads();
  if (warp == 0) {
    uint32_t wa = sh[lane], wb = sh[33 + lane];
    uint32_t xa = wa, xb = wb;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t na = __shfl_up_sync(0xffffffffu, xa, o);
      const uint32_t nb = __shfl_up_sync(0xffffffffu, xb, o);
      if (lane >= o) { xa += na; xb += nb; }
    }
    sh[lane] = xa - wa;
    sh[33 + lane] = xb - wb;
    if (lane == 31) { sh[32] = xa; sh[65] = xb; }
  }
  __syncthreads();
  ea = sh[warp] + ia - a;
  eb = sh[33 + warp] + ib - b;
  ta = sh[32];
  tb = sh[65];
  __syncthreads();
}

// Finds, scanning bins from the top, the bin where the running count
// reaches `need`; per = bins per thread (nbins = per * kThreads).
template <int PER>
__device__ __forceinline__ void find_from_top(const uint32_t* hist, uint32_t need, int& bin, uint32_t& above,
                                              uint32_t* sh) {
  constexpr int nbins = PER * kThreads;
  const int tid = threadIdx.x;
  uint32_t mine[PER];
  uint32_t s = 0;
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    mine[i] = hist[nbins - 1 - (tid * PER + i)];
    s += mine[i];
  }
  uint32_t ex, dummy, tot, t2;
  block_scan2(s, 0u, ex, dummy, tot, t2, sh);
  uint32_t before = ex;
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    if (before < need && before + mine[i] >= need) {
      sh[66] = nbins - 1 - (tid * PER + i);
      sh[67] = before;
    }
    before += mine[i];
  }
  __syncthreads();
  bin = static_cast<int>(sh[66]);
  above = sh[67];
  __syncthreads();
}

__global__ void __launch_bounds__(kThreads) topk_hist_kernel(const TopkHistParams P) {
  __shared__ uint32_t sh[80];
  __shared__ uint32_t lh[1024];
  __shared__ uint32_t base[2];
  const int tid = threadIdx.x;
  const int row = blockIdx.x / P.slices, sl = blockIdx.x % P.slices;
  griddep_launch_dependents();
  griddep_wait();
  const int n_valid = min(P.pos[row] + 1, P.max_L);
  const int k = P.topk;
  int32_t* out = P.out + static_cast<size_t>(row) * k;
  uint32_t* hist = P.hist + static_cast<size_t>(row) * kHB;
  uint32_t* ctr = P.ctr + static_cast<size_t>(row) * 4;
  uint2* cand = P.cand + static_cast<size_t>(row) * kTopkCandCap;
  if (n_valid <= k) {
    if (sl == 0) {
      for (int i = tid; i < k; i += kThreads) out[i] = (i < n_valid) ? i : -1;
      for (int i = tid; i < kHB; i += kThreads) hist[i] = 0;
    }
    return;
  }
  // Leading digit of the k-th largest key, keys above it, keys in it.
  int B;
  uint32_t c_above;
  find_from_top<kHB / kThreads>(hist, static_cast<uint32_t>(k), B, c_above, sh);
  const uint32_t c_bin = hist[B];
  const uint32_t need = static_cast<uint32_t>(k) - c_above;

  // This CTA's slice of the row, in registers.
  const int chunk = (n_valid + P.slices - 1) / P.slices;
  const int lo = sl * chunk, hi = min(n_valid, lo + chunk);
  const float* src = P.scores + static_cast<size_t>(row) * P.ld;
  uint32_t keys[kPer];
  uint32_t n_gt = 0, n_eq = 0;
#pragma unroll
  for (int e = 0; e < kPer; ++e) {
    const int i = lo + tid + e * kThreads;
    keys[e] = (i < hi) ? order_key(src[i]) : 0u;
    if (i < hi) {
      n_gt += (keys[e] >> 20) > static_cast<uint32_t>(B);
      n_eq += (keys[e] >> 20) == static_cast<uint32_t>(B);
    }
  }
  uint32_t off_gt, off_eq, tot_gt, tot_eq;
  block_scan2(n_gt, n_eq, off_gt, off_eq, tot_gt, tot_eq, sh);
  if (tid == 0) {
    base[0] = tot_gt ? atomicAdd(&ctr[0], tot_gt) : 0u;
    base[1] = tot_eq ? atomicAdd(&ctr[1], tot_eq) : 0u;
  }
  __syncthreads();
  uint32_t pg = base[0] + off_gt, pe = base[1] + off_eq;
#pragma unroll
  for (int e = 0; e < kPer; ++e) {
    const int i = lo + tid + e * kThreads;
    if (i < hi) {
      const uint32_t d = keys[e] >> 20;
      if (d > static_cast<uint32_t>(B)) {
        if (pg < c_above) out[pg] = i;
        ++pg;
      } else if (d == static_cast<uint32_t>(B)) {
        if (pe < kTopkCandCap) cand[pe] = make_uint2(keys[e], static_cast<uint32_t>(i));
        ++pe;
      }
    }
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) sh[70] = (atomicAdd(&ctr[2], 1u) == static_cast<uint32_t>(P.slices - 1));
  __syncthreads();
  if (!sh[70]) return;
  __threadfence();

  // Last CTA of the row: the `need` largest candidates by the low 20 bits.
  if (c_bin > static_cast<uint32_t>(kTopkCandCap)) {
    if (tid == 0) atomicOr(P.err, kErrBadIndex);  // leading digit too crowded
  } else {
    constexpr int kC = kTopkCandCap / kThreads;
    uint32_t ck[kC], ci[kC];
#pragma unroll
    for (int e = 0; e < kC; ++e) {
      const int i = tid + e * kThreads;
      if (i < static_cast<int>(c_bin)) {
        const uint2 v = __ldcg(cand + i);
        ck[e] = v.x;
        ci[e] = v.y;
      } else {
        ck[e] = 0u;
        ci[e] = 0xffffffffu;
      }
    }
    uint32_t prefix = static_cast<uint32_t>(B) << 20, mask = 0xFFF00000u, nd = need;
#pragma unroll 1
    for (int pass = 0; pass < 2; ++pass) {
      const int sh_ = pass == 0 ? 10 : 0;
      lh[tid] = 0;
      __syncthreads();
#pragma unroll
      for (int e = 0; e < kC; ++e)
        if (ci[e] != 0xffffffffu && (ck[e] & mask) == prefix) atomicAdd(&lh[(ck[e] >> sh_) & 1023u], 1u);
      __syncthreads();
      int bn;
      uint32_t ab;
      find_from_top<1>(lh, nd, bn, ab, sh);
      nd -= ab;
      prefix |= static_cast<uint32_t>(bn) << sh_;
      mask |= 1023u << sh_;
    }
    const uint32_t thr = prefix;  // the k-th largest key; nd of its copies are taken
    if (tid == 0) { base[0] = 0; base[1] = 0; }
    __syncthreads();
    const uint32_t n_gt_c = need - nd;
#pragma unroll
    for (int e = 0; e < kC; ++e) {
      if (ci[e] == 0xffffffffu) continue;
      if (ck[e] > thr) {
        out[c_above + atomicAdd(&base[0], 1u)] = static_cast<int32_t>(ci[e]);
      } else if (ck[e] == thr) {
        const uint32_t q = atomicAdd(&base[1], 1u);
        if (q < nd) out[c_above + n_gt_c + q] = static_cast<int32_t>(ci[e]);
      }
    }
  }
  // Leave the row's histogram and counters zeroed for the next call.
  for (int i = tid; i < kHB; i += kThreads) hist[i] = 0;
  if (tid < 3) ctr[tid] = 0;
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

bool topk_hist_eligible(const dsa_topk_args& a) {
  // groups of at most two tokens (the indexer's histogram), and a bounded
  // candidate workspace
  const int G = a.H_I >= 128 ? 1 : (128 / a.H_I < a.n_q ? 128 / a.H_I : a.n_q);
  return G <= 2 && a.H_I >= 64 && a.T <= 512 && a.max_L <= kThreads * kPer * 64;
}

size_t topk_hist_workspace(const dsa_topk_args& a) {
  return round_up(static_cast<size_t>(a.T) * kTopkHistBins * 4, 256) + round_up(static_cast<size_t>(a.T) * 16, 256) +
         round_up(static_cast<size_t>(a.T) * kTopkCandCap * 8, 256);
}

int launch_topk_hist(const dsa_topk_args& a, const float* scores, int64_t ld, void* ws, cudaStream_t s) {
  TopkHistParams P{};
  P.scores = scores; P.ld = ld; P.pos = a.pos; P.max_L = a.max_L; P.topk = a.topk; P.out = a.topk_idx;
  P.slices = (a.max_L + kThreads * 8 - 1) / (kThreads * 8);
  uint8_t* w = static_cast<uint8_t*>(ws);
  P.hist = reinterpret_cast<uint32_t*>(w);
  w += round_up(static_cast<size_t>(a.T) * kTopkHistBins * 4, 256);
  P.ctr = reinterpret_cast<uint32_t*>(w);
  w += round_up(static_cast<size_t>(a.T) * 16, 256);
  P.cand = reinterpret_cast<uint2*>(w);
  P.err = error_word();
  if (!P.err) return DSA_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(a.T * P.slices);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cuda_status(cudaLaunchKernelEx(&cfg, topk_hist_kernel, P));
}

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

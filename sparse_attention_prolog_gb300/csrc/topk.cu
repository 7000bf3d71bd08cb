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
// follow from that histogram alone.  One cluster of CS CTAs (<= 8) takes a
// row; CTA r holds keys [r * kThreads * PER, (r + 1) * kThreads * PER) in
// registers (one read of the row).  Keys above B go straight to the output
// (slots reserved with one cluster atomic per warp on CTA 0).  The missing
// `need` keys are the largest of bin B, found by a radix select on the low
// 20 bits (two 10-bit passes):
//   - bin B holds at most kCandMax keys (the usual case): every CTA stores
//     its bin-B keys into CTA 0's shared memory, the other CTAs leave after
//     one cluster barrier, and CTA 0 selects among the candidates alone;
//   - otherwise (heavy ties) the passes run over the registers of every CTA,
//     with per-CTA histograms summed in CTA 0 by cluster atomics.
// The row's histogram is left zeroed for the next call.
constexpr int kHB = kTopkHistBins;
constexpr int kLowBins = 1024;  // 10-bit digits of the second and third pass
constexpr int kCandMax = 8192;  // bin-B keys CTA 0 can hold (dynamic shared memory)

struct TopkHistParams {
  const float* scores;
  int64_t ld;
  const int32_t* pos;
  int max_L, topk;
  int32_t* out;
  uint32_t* hist;  // [T][kHB]
  uint32_t* err;
};

__device__ __forceinline__ uint32_t atom_add_cluster(uint32_t addr, uint32_t v) {
  uint32_t old;
  asm volatile("atom.shared::cluster.add.u32 %0, [%1], %2;" : "=r"(old) : "r"(addr), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ void red_add_cluster(uint32_t addr, uint32_t v) {
  asm volatile("red.shared::cluster.add.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// Reserves n consecutive output slots for this thread from the counter at
// cluster address `ctr` (one atomic per warp); returns the first slot.
__device__ __forceinline__ uint32_t warp_reserve_n(uint32_t ctr, uint32_t n) {
  const int lane = threadIdx.x & 31;
  uint32_t incl = n;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  const uint32_t total = __shfl_sync(0xffffffffu, incl, 31);
  uint32_t base = 0;
  if (lane == 31 && total) base = atom_add_cluster(ctr, total);
  base = __shfl_sync(0xffffffffu, base, 31);
  return base + incl - n;
}

// Block-wide search from the top bin: thread tid holds the counts of bins
// nbins-1-(tid*PER+i); returns the bin where the running count (from the
// top) first reaches `need`, the count strictly above it, and its own count.
// bin = -1 if the counts never reach `need`.
template <int PER>
__device__ __forceinline__ void find_from_top(const uint32_t (&mine)[PER], uint32_t need, int& bin,
                                              uint32_t& above, uint32_t& count, uint32_t* sh /*[36]*/) {
  constexpr int nbins = PER * kThreads;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t s = 0;
#pragma unroll
  for (int i = 0; i < PER; ++i) s += mine[i];
  uint32_t incl = s;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) sh[warp] = incl;
  if (tid == 0) sh[32] = 0xffffffffu;
  __syncthreads();
  // exclusive offset of this warp: a shuffle scan of the warp totals
  uint32_t wt = lane < kThreads / 32 ? sh[lane] : 0u, wincl = wt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t v = __shfl_up_sync(0xffffffffu, wincl, o);
    if (lane >= o) wincl += v;
  }
  uint32_t before = incl - s + __shfl_sync(0xffffffffu, wincl - wt, warp);
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    if (before < need && before + mine[i] >= need) {
      sh[32] = nbins - 1 - (tid * PER + i);
      sh[33] = before;
      sh[34] = mine[i];
    }
    before += mine[i];
  }
  __syncthreads();
  bin = sh[32] == 0xffffffffu ? -1 : static_cast<int>(sh[32]);
  above = sh[33];
  count = sh[34];
  __syncthreads();
}

// Reserves n_a slots from the 32-bit counter at cluster address ctr and n_b
// from the one after it, with one 64-bit atomic per warp; returns each
// thread's first slot of both.
__device__ __forceinline__ void warp_reserve_pair(uint32_t ctr, uint32_t n_a, uint32_t n_b, uint32_t& p_a,
                                                  uint32_t& p_b) {
  const int lane = threadIdx.x & 31;
  uint32_t ia = n_a, ib = n_b;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t va = __shfl_up_sync(0xffffffffu, ia, o);
    const uint32_t vb = __shfl_up_sync(0xffffffffu, ib, o);
    if (lane >= o) { ia += va; ib += vb; }
  }
  const uint32_t ta = __shfl_sync(0xffffffffu, ia, 31), tb = __shfl_sync(0xffffffffu, ib, 31);
  unsigned long long base = 0;
  if (lane == 31 && (ta | tb)) {
    const unsigned long long add = static_cast<unsigned long long>(ta) | (static_cast<unsigned long long>(tb) << 32);
    asm volatile("atom.shared::cluster.add.u64 %0, [%1], %2;" : "=l"(base) : "r"(ctr), "l"(add) : "memory");
  }
  base = __shfl_sync(0xffffffffu, base, 31);
  p_a = static_cast<uint32_t>(base) + ia - n_a;
  p_b = static_cast<uint32_t>(base >> 32) + ib - n_b;
}

__device__ __forceinline__ void st_cluster_v2(uint32_t addr, uint32_t a, uint32_t b) {
  asm volatile("st.shared::cluster.v2.u32 [%0], {%1, %2};" ::"r"(addr), "r"(a), "r"(b) : "memory");
}
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

template <int PER>
__global__ void __launch_bounds__(kThreads, 1) topk_hist_kernel(const TopkHistParams P) {
  extern __shared__ __align__(16) uint2 cand[];  // CTA 0: [kCandMax] (key, index) of bin B
  __shared__ uint32_t sh[40];
  __shared__ uint32_t lh[2][kLowBins];  // this CTA's counts, passes 1 and 2
  __shared__ uint32_t gh[2][kLowBins];  // CTA 0: the cluster's counts (tie path)
  __shared__ __align__(8) uint32_t cnt[4];  // CTA 0: slots above B, candidates (one u64), emission
  __shared__ uint2 grp_s[32];               // CTA 0: the k-th key's group when it is small
  __shared__ uint32_t grp_n;
  const int tid = threadIdx.x;
  const uint32_t rank = cluster_ctarank();
  uint32_t ncta;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(ncta));
  const int row = blockIdx.x / static_cast<int>(ncta);
  for (int i = tid; i < kLowBins; i += kThreads) {
    lh[0][i] = 0; lh[1][i] = 0; gh[0][i] = 0; gh[1][i] = 0;
  }
  if (tid < 4) cnt[tid] = 0;
  if (tid == 0) grp_n = 0;
  // CTA 0's counters are zero before any peer's atomics: the arrive is here,
  // the matching wait just before the first remote access, so the barrier
  // overlaps the loads below.
  cluster_arrive();
  griddep_launch_dependents();
  griddep_wait();  // scores and histogram come from the indexer

  // Issue every global load at once: the row's histogram, this CTA's keys
  // (up to max_L; masked by the row's causal limit once pos arrives).
  const float* src = P.scores + static_cast<size_t>(row) * P.ld;
  uint32_t* hist = P.hist + static_cast<size_t>(row) * kHB;
  const int lo = static_cast<int>(rank) * kThreads * PER;
  constexpr int kHPer = kHB / kThreads;
  uint32_t hv[kHPer];
#pragma unroll
  for (int i = 0; i < kHPer; ++i) hv[i] = __ldcg(hist + kHB - 1 - (tid * kHPer + i));
  uint32_t keys[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) {
    const int i = lo + tid + e * kThreads;
    keys[e] = i < P.max_L ? order_key(__ldcg(src + i)) : 0u;
  }
  const int n_valid = min(__ldg(P.pos + row) + 1, P.max_L);
  const int k = P.topk;
  int32_t* out = P.out + static_cast<size_t>(row) * k;
  if (n_valid <= k) {  // every visible key, then -1 (same branch in every CTA)
    if (rank == 0) {
      for (int i = tid; i < k; i += kThreads) out[i] = (i < n_valid) ? i : -1;
      for (int i = tid; i < kHB; i += kThreads) hist[i] = 0;
    }
    return;
  }
  auto valid = [&](int e) { return lo + tid + e * kThreads < n_valid; };

  // Leading digit B of the k-th largest key and the keys above it.
  int B;
  uint32_t c_above, c_bin;
  find_from_top<kHPer>(hv, static_cast<uint32_t>(k), B, c_above, c_bin, sh);
  if (B < 0) {  // histogram and row disagree: the workspace was not zeroed
    if (tid == 0) atomicOr(P.err, kErrBadIndex);
    return;
  }
  const uint32_t ub = static_cast<uint32_t>(B);
  const uint32_t cnt0 = mapa(smem_u32(cnt), 0);
  // Once every CTA has read the histogram: the CTAs other than CTA 0 clear
  // it (CTA 0 goes on with the candidates), CTA 0 alone when it has no peer.
  auto zero_hist_slice = [&]() {
    const int nz = ncta > 1 ? static_cast<int>(ncta) - 1 : 1;
    const int z = ncta > 1 ? static_cast<int>(rank) - 1 : 0;
    if (z < 0) return;
    const int h0 = z * kHB / nz, h1 = (z + 1) * kHB / nz;
    for (int i = h0 + tid; i < h1; i += kThreads) hist[i] = 0;
  };
  cluster_wait();

  // Keys above the leading digit take output slots [0, c_above); keys of
  // bin B become candidates in CTA 0 (fast path).  One 64-bit cluster
  // atomic per warp reserves both kinds (cnt[0] counts the first, cnt[1]
  // the second).
  const bool fast = c_bin <= static_cast<uint32_t>(kCandMax);
  uint32_t p_above, p_cand;
  {
    uint32_t n_a = 0, n_c = 0;
#pragma unroll
    for (int e = 0; e < PER; ++e) {
      n_a += (valid(e) && (keys[e] >> 20) > ub) ? 1u : 0u;
      n_c += (fast && valid(e) && (keys[e] >> 20) == ub) ? 1u : 0u;
    }
    warp_reserve_pair(cnt0, n_a, n_c, p_above, p_cand);
  }
#pragma unroll
  for (int e = 0; e < PER; ++e)
    if (valid(e) && (keys[e] >> 20) > ub) {
      if (p_above < c_above) out[p_above] = lo + tid + e * kThreads;
      ++p_above;
    }
  uint32_t need = static_cast<uint32_t>(k) - c_above;

  if (fast) {
    // ---------------- bin B to CTA 0, which selects among the candidates
    {
      const uint32_t cand0 = mapa(smem_u32(cand), 0);
#pragma unroll
      for (int e = 0; e < PER; ++e)
        if (valid(e) && (keys[e] >> 20) == ub) {
          if (p_cand < static_cast<uint32_t>(kCandMax))
            st_cluster_v2(cand0 + p_cand * 8, keys[e], static_cast<uint32_t>(lo + tid + e * kThreads));
          ++p_cand;
        }
    }
    cluster_arrive();  // candidates stored; every CTA has read the histogram
    cluster_wait();
    zero_hist_slice();
    if (rank != 0) return;
    const uint32_t n_cand = min(cnt[1], static_cast<uint32_t>(kCandMax));
    if (tid == 0 && n_cand != c_bin) atomicOr(P.err, kErrBadIndex);
    uint32_t prefix = ub << 20, mask = 0xFFF00000u;
    bool whole_bin = false;  // the k-th key's digit group is taken entirely
    bool small = false;      // or it holds at most 32 keys: one warp ranks them, no second pass
#pragma unroll 1
    for (int pass = 0; pass < 2 && !whole_bin && !small; ++pass) {
      const int shift = pass == 0 ? 10 : 0;
      for (uint32_t i = tid; i < n_cand; i += kThreads) {
        const uint32_t key = cand[i].x;
        if ((key & mask) == prefix) atomicAdd(&lh[pass][(key >> shift) & (kLowBins - 1)], 1u);
      }
      __syncthreads();
      uint32_t g1[1] = {lh[pass][kLowBins - 1 - tid]};
      int bn;
      uint32_t ab, cb;
      find_from_top<1>(g1, need, bn, ab, cb, sh);
      if (bn < 0) {  // cannot happen when the histogram matches the row
        if (tid == 0) atomicOr(P.err, kErrBadIndex);
        bn = 0;
      }
      need -= ab;
      prefix |= static_cast<uint32_t>(bn) << shift;
      mask |= static_cast<uint32_t>(kLowBins - 1) << shift;
      // every key of the found group is needed: the lower bits do not matter
      whole_bin = (cb == need);
      small = !whole_bin && cb <= 32u;
    }
    // Keys of bin B above the group `prefix/mask` come first; then `need`
    // keys of the group itself (all of it when whole_bin, else the copies of
    // the k-th key `prefix`).
    const uint32_t base_eq = static_cast<uint32_t>(k) - need;
    for (uint32_t i = tid; i < n_cand; i += kThreads) {
      const uint2 c = cand[i];
      const uint32_t g = c.x & mask;
      if (g > prefix) {
        const uint32_t q = atomicAdd(&cnt[2], 1u);
        if (c_above + q < base_eq) out[c_above + q] = static_cast<int32_t>(c.y);
      } else if (g == prefix) {
        if (small) {
          const uint32_t q = atomicAdd(&grp_n, 1u);
          if (q < 32u) grp_s[q] = c;
        } else {
          const uint32_t q = atomicAdd(&cnt[3], 1u);
          if (q < need) out[base_eq + q] = static_cast<int32_t>(c.y);
        }
      }
    }
    if (small) {  // the `need` largest keys of the group (equal keys in list order)
      __syncthreads();
      if (tid < 32) {
        const uint32_t n = min(grp_n, 32u);
        const uint2 me = tid < static_cast<int>(n) ? grp_s[tid] : make_uint2(0u, 0u);
        uint32_t rank = 0;
        for (uint32_t m = 0; m < n; ++m) {
          const uint2 o = grp_s[m];
          rank += (o.x > me.x || (o.x == me.x && m < static_cast<uint32_t>(tid))) ? 1u : 0u;
        }
        if (tid < static_cast<int>(n) && rank < need) out[base_eq + rank] = static_cast<int32_t>(me.y);
      }
    }
    return;
  }

  // ---------------- heavy ties: radix passes over every CTA's registers
  uint32_t prefix = ub << 20, mask = 0xFFF00000u;
#pragma unroll 1
  for (int pass = 0; pass < 2; ++pass) {
    const int shift = pass == 0 ? 10 : 0;
#pragma unroll
    for (int e = 0; e < PER; ++e)
      if (valid(e) && (keys[e] & mask) == prefix) atomicAdd(&lh[pass][(keys[e] >> shift) & (kLowBins - 1)], 1u);
    __syncthreads();
    {
      const uint32_t v = lh[pass][tid];
      if (v) red_add_cluster(mapa(smem_u32(&gh[pass][tid]), 0), v);
    }
    cluster_sync();
    if (pass == 0) zero_hist_slice();
    uint32_t g1[1] = {ld_cluster_u32(mapa(smem_u32(&gh[pass][kLowBins - 1 - tid]), 0))};
    int bn;
    uint32_t ab, cb;
    find_from_top<1>(g1, need, bn, ab, cb, sh);
    if (bn < 0) {  // cannot happen when the histogram matches the row
      if (tid == 0) atomicOr(P.err, kErrBadIndex);
      bn = 0;
    }
    need -= ab;
    prefix |= static_cast<uint32_t>(bn) << shift;
    mask |= static_cast<uint32_t>(kLowBins - 1) << shift;
  }
  // prefix is now the k-th largest key; `need` of its copies are taken after
  // the (k - c_above - need) keys of bin B above it.
  const uint32_t thr = prefix;
  const uint32_t base_gt = c_above, base_eq = static_cast<uint32_t>(k) - need;
  {
    uint32_t n_gt = 0, n_eq = 0;
#pragma unroll
    for (int e = 0; e < PER; ++e) {
      const bool inb = valid(e) && (keys[e] >> 20) == ub;
      n_gt += (inb && keys[e] > thr) ? 1u : 0u;
      n_eq += (inb && keys[e] == thr) ? 1u : 0u;
    }
    uint32_t pg = base_gt + warp_reserve_n(cnt0 + 8, n_gt);
    uint32_t pe = warp_reserve_n(cnt0 + 12, n_eq);
#pragma unroll
    for (int e = 0; e < PER; ++e) {
      const bool inb = valid(e) && (keys[e] >> 20) == ub;
      if (inb && keys[e] > thr) {
        if (pg < base_eq) out[pg] = lo + tid + e * kThreads;
        ++pg;
      } else if (inb && keys[e] == thr) {
        if (pe < need) out[base_eq + pe] = lo + tid + e * kThreads;
        ++pe;
      }
    }
  }
  cluster_sync();  // CTA 0's shared memory stays alive until every atomic is done
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
  // groups of at most two tokens (the indexer's histogram); a row fits one
  // cluster of at most 8 CTAs with 16 keys per thread
  return indexer_group_tokens(a) <= 2 && a.H_I >= 64 && a.T <= 512 && a.max_L <= kThreads * 16 * 8;
}

size_t topk_hist_workspace(const dsa_topk_args& a) {
  return round_up(static_cast<size_t>(a.T) * kTopkHistBins * 4, 256);
}

int launch_topk_hist(const dsa_topk_args& a, const float* scores, int64_t ld, void* ws, cudaStream_t s) {
  TopkHistParams P{};
  P.scores = scores; P.ld = ld; P.pos = a.pos; P.max_L = a.max_L; P.topk = a.topk; P.out = a.topk_idx;
  P.hist = static_cast<uint32_t*>(ws);
  P.err = error_word();
  if (!P.err) return DSA_ERR_CUDA;
  const int per = a.max_L <= kThreads * 8 * 8 ? 8 : 16;
  const int cs = (a.max_L + kThreads * per - 1) / (kThreads * per);
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = cs;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.gridDim = dim3(a.T * cs);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kCandMax * sizeof(uint2);
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cudaError_t e = cudaFuncSetAttribute(per == 8 ? topk_hist_kernel<8> : topk_hist_kernel<16>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kCandMax * (int)sizeof(uint2));
  if (e != cudaSuccess) return DSA_ERR_CUDA;
  e = per == 8 ? cudaLaunchKernelEx(&cfg, topk_hist_kernel<8>, P) : cudaLaunchKernelEx(&cfg, topk_hist_kernel<16>, P);
  return cuda_status(e);
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

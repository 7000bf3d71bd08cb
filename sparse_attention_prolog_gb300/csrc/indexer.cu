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
//   warp 12    producer: 2-D TMA loads (128B swizzle) of the raw int8 key
//              tile into an 8-deep shared-memory ring
//   warps 4-7  converters: one thread per key row reads its 128 bytes
//              (bank-conflict free thanks to the swizzle), converts them to
//              f16 and stores the row into TMEM, where it is the A operand
//              of the MMA; they also stage Q (the B operand, shared memory)
//              for each new group
//   warp 13    one thread issues tcgen05.mma (A from TMEM, B from shared
//              memory) into two or three rotating TMEM accumulators
// Keeping the keys out of shared memory after the TMA halves the shared
// memory traffic per tile, which otherwise bounds the kernel.
//   warps 0-3, 8-11  epilogue, two groups of four warps over the same TMEM
//              lanes (warp w reads lanes 32 (w % 4) ..): group e takes the
//              tokens e, e + 2, ... of the tile.  tcgen05.ld of the
//              accumulator row of its key, ReLU + head-weighted sum per
//              token, times ks[s], causal mask, and the fp32 score row store
//              (coalesced over keys)
// Each role waits for the previous kernel (programmatic launch) only before
// its first read of that kernel's outputs (q, w, qs, new cache rows), so the
// work list is built while the producing kernel is still finishing.
// The per-head scores [T, H_I, L] never leave the SM; only I[t, s] (fp32,
// [T, max_L]) is written, for the top-k pass.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include "dsa_internal.h"
#include "dsa_ptx.cuh"

namespace dsa {
namespace {

constexpr int kTileKeys = 128;
constexpr int kStages8 = 8;   // raw int8 key tiles in flight
constexpr int kStages16 = 3;  // converted f16 key tiles (in TMEM)
constexpr int kThreads = 448;  // 14 warps, see the role map above
constexpr int kMaxG = 32;     // tokens per group
constexpr int kCoef = 256;    // max query rows (N) of a group
// Cost of a group change, in tiles, in the split of the work over CTAs: the
// group's queries are staged and its head weights loaded while no tile is
// scored (measured on a causal prefill: a group's first tile takes about
// two tiles' time longer than the others).
constexpr int kGroupCost = 2;
constexpr int kGroupCostMinGroups = 64;
constexpr int kHistBins = 4096;  // leading 12 bits of the score's order key

struct IdxParams {
  // n_groups: the group count of a uniform batch (seq == null), else the
  // most groups the token map may form (the size of the group table).
  int T, B, n_q, H_I, d_I, G, N, groups_per_seq, n_groups, n_tiles, max_L;
  const int32_t* seq;  // [T] sequence of each token, or null (token t in sequence t / n_q)
  const int8_t* q;
  const __half* q_scale;
  const float* w;
  const int8_t* k_cache;
  const __half* k_scale;
  const int32_t* block_table;
  int block_size, max_blocks, box_rows;
  const int32_t* pos;
  float* scores;
  int64_t ld;
  uint32_t* hist;  // [T][kHistBins] leading-digit counts of the scores, or null
  uint32_t* err;
};

struct Group {
  int b, t0, ntok, maxpos;
};

// Group g of a batch given by its token map: tokens [grp[g], grp[g + 1])
// (a run of adjacent tokens of one sequence, at most G long; built on the
// device by build_groups).  Of a uniform batch: the G-token slices of each
// sequence's n_q tokens.

// max(x, 0) of two floats packed into one 64-bit register (fma_f32x2 operand).
__device__ __forceinline__ uint64_t relu_pair(uint32_t x, uint32_t y) {
  return pack_f32x2(fmaxf(__uint_as_float(x), 0.f), fmaxf(__uint_as_float(y), 0.f));
}

__device__ __forceinline__ Group group_of(const IdxParams& P, const uint16_t* grp, int g) {
  Group G;
  if (grp != nullptr) {
    G.t0 = grp[g];
    G.ntok = grp[g + 1] - G.t0;
    const int b = __ldg(P.seq + G.t0);
    G.b = (b >= 0 && b < P.B) ? b : 0;  // out of range: recorded by build_groups
  } else {
    G.b = g / P.groups_per_seq;
    const int gj = g % P.groups_per_seq;
    G.t0 = G.b * P.n_q + gj * P.G;
    G.ntok = min(P.G, P.n_q - gj * P.G);
  }
  int m = -1;
  for (int i = 0; i < G.ntok; ++i) m = max(m, __ldg(P.pos + G.t0 + i));
  G.maxpos = min(m, P.max_L - 1);
  return G;
}

// Work list: the active tiles (tiles holding at least one visible key) of
// all groups in group-major order.  Every CTA computes the per-group tile
// counts and their prefix sum, then walks its own contiguous, equal share of
// the list, so a decode CTA stays in one group and a prefill CTA gets an
// equal number of tiles however causal masking thins the groups.

struct Walker {
  int g, j, left;  // current group, tile within the group, items left
};

__device__ __forceinline__ int group_tiles(const IdxParams& P, const uint16_t* grp, int g) {
  const Group G = group_of(P, grp, g);
  return G.maxpos < 0 ? 0 : min(P.n_tiles, G.maxpos / kTileKeys + 1);
}

// Advances to the next tile of the walk (skips groups without tiles).
__device__ __forceinline__ bool walk_next(const int* tiles_prefix, int n_groups, Walker& w) {
  if (w.left <= 0) return false;
  --w.left;
  if (w.left == 0) return false;
  ++w.j;
  while (w.g < n_groups && w.j >= tiles_prefix[w.g + 1] - tiles_prefix[w.g]) {
    ++w.g;
    w.j = 0;
  }
  return true;
}

// Exclusive block-wide scan (sum, or max when kMax) of one value per thread
// of a kThreads-thread block; `tmp` holds one int per warp.  Every thread
// must call it; returns the exclusive prefix and sets `total`.
template <bool kMax, int kNT>
__device__ __forceinline__ int block_scan_excl(int v, int* tmp, int& total, int identity) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl = kMax ? max(incl, n) : incl + n;
  }
  if (lane == 31) tmp[warp] = incl;
  __syncthreads();
  int woff = identity, all = identity;
  for (int w2 = 0; w2 < kNT / 32; ++w2) {
    if (w2 < warp) woff = kMax ? max(woff, tmp[w2]) : woff + tmp[w2];
    all = kMax ? max(all, tmp[w2]) : all + tmp[w2];
  }
  __syncthreads();  // tmp may be reused by the next scan
  const int excl_in_warp = __shfl_up_sync(0xffffffffu, incl, 1);
  const int excl = lane == 0 ? woff : (kMax ? max(woff, excl_in_warp) : woff + excl_in_warp);
  total = all;
  return excl;
}

// Group table of a batch given by its token map: a group starts at every
// token whose sequence differs from the previous token's and then every G
// tokens within such a run.  grp[0..n) receives the first token of each
// group and grp[n] = T; returns n (the same in every thread).  Out-of-range
// sequence ids, and more groups than the table holds (the tokens of a
// sequence not adjacent), are recorded in the error word; groups past the
// table are dropped.
template <int kNT>
__device__ int build_groups(const IdxParams& P, uint16_t* grp, int* tmp) {
  const int T = P.T;
  const int per = (T + kNT - 1) / kNT;
  const int c0 = min(T, static_cast<int>(threadIdx.x) * per), c1 = min(T, c0 + per);
  int last = -1;
  bool bad = false;
  for (int t = c0; t < c1; ++t) {
    const int b = __ldg(P.seq + t);
    bad |= (b < 0 || b >= P.B);
    if (t == 0 || b != __ldg(P.seq + t - 1)) last = t;
  }
  if (bad) atomicOr(P.err, kErrBadIndex);
  int unused;
  const int rs0 = block_scan_excl<true, kNT>(last, tmp, unused, -1);  // start of the run entering the chunk
  int rs = rs0, cnt = 0;
  for (int t = c0; t < c1; ++t) {
    if (t == 0 || __ldg(P.seq + t) != __ldg(P.seq + t - 1)) rs = t;
    cnt += ((t - rs) % P.G) == 0;
  }
  int n = 0;
  int off = block_scan_excl<false, kNT>(cnt, tmp, n, 0);
  rs = rs0;
  for (int t = c0; t < c1; ++t) {
    if (t == 0 || __ldg(P.seq + t) != __ldg(P.seq + t - 1)) rs = t;
    if (((t - rs) % P.G) == 0) {
      // entry n_groups of a full table is the start of the first dropped
      // group, so the last kept group still ends where it should
      if (off <= P.n_groups) grp[off] = static_cast<uint16_t>(t);
      ++off;
    }
  }
  if (n > P.n_groups) {
    if (threadIdx.x == 0) atomicOr(P.err, kErrBadIndex);
    n = P.n_groups;
  } else if (threadIdx.x == 0) {
    grp[n] = static_cast<uint16_t>(T);
  }
  __syncthreads();
  return n;
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
  uint64_t tfull[3], tempty[3];
  uint64_t epsync;  // barrier of the 8 epilogue warps (bounded wait)
  uint64_t mdrain;  // the MMA thread's last commit: every MMA done before TMEM is freed
};

template <int HI, int DI>
__global__ void __launch_bounds__(kThreads, 1)
    indexer_kernel(const __grid_constant__ IdxParams P, const __grid_constant__ CUtensorMap tmap) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr int d_I = DI;
  const int N = P.N;
  constexpr uint32_t tile8_bytes = kTileKeys * DI;     // int8 tile (TMA-swizzled)
  uint8_t* s8 = smem;                                  // [kStages8][tile8]
  uint8_t* sQ = s8 + kStages8 * tile8_bytes;           // [d_I/64 atoms][N rows][128 B]
  // [n_groups + 1] tile prefix, then (token map only) the group table
  int* tiles_prefix = reinterpret_cast<int*>(sQ + static_cast<size_t>(N) * DI * 2);
  uint16_t* grp = P.seq != nullptr ? reinterpret_cast<uint16_t*>(tiles_prefix + P.n_groups + 1) : nullptr;
  // [n_groups + 1] prefix of the work's cost: scratch in the key ring, which
  // no copy writes before the setup below is done
  int* cost_prefix = reinterpret_cast<int*>(smem);
  __shared__ Bars bars;
  // fp16 key scales of each ring stage, copied with its key tile.
  __shared__ __align__(16) unsigned short ks_s[kStages8][kTileKeys];
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  __shared__ __align__(16) float coef[kCoef];
  __shared__ int tok_pos[kMaxG];
  __shared__ int scan_tmp[kThreads / 32], scan_tmp2[kThreads / 32];
  // Per-token histogram of each visible score's leading 12 key bits (groups
  // of at most two tokens, H_I >= 64); flushed to global memory at every
  // group change so the top-k pass can find its threshold digit at once.
  constexpr bool kHist = HI >= 64;
  __shared__ uint32_t hist_s[kHist ? 2 * kHistBins : 1];
  if (kHist)
    for (int i = threadIdx.x; i < 2 * kHistBins; i += kThreads) hist_s[i] = 0;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // Accumulator buffers start on 32-column boundaries so that every 32-column
  // load stays inside its own buffer.
  // TMEM: n_acc fp32 accumulators (three when they fit in the 512 columns),
  // then three f16 key tiles (DI/2 columns each), so that the converters
  // can run two tiles ahead of the MMA.
  const int acc_stride = (N + 31) & ~31;
  // Three accumulators let the MMA of a tile run while the epilogue still
  // reads the two before it; they take precedence over a third key stage.
  const int n16 = 3 * acc_stride + kStages16 * DI / 2 <= 512 ? kStages16 : 2;
  const int n_acc = 3 * acc_stride + n16 * DI / 2 <= 512 ? 3 : 2;
  const uint32_t a_col0 = n_acc * acc_stride;
  const int need_cols = n_acc * acc_stride + n16 * DI / 2;
  const uint32_t tmem_cols = need_cols <= 64 ? 64 : need_cols <= 128 ? 128 : need_cols <= 256 ? 256 : 512;

  if (tid == 0) {
    // A ring stage is free once the 4 converter warps have read its keys
    // and the 8 epilogue warps its key scales.
    for (int i = 0; i < kStages8; ++i) { mbar_init(&bars.full8[i], 1); mbar_init(&bars.empty8[i], 12); }
    for (int i = 0; i < kStages16; ++i) { mbar_init(&bars.full16[i], 4); mbar_init(&bars.empty16[i], 1); }
    mbar_init(&bars.qfull, 4);
    mbar_init(&bars.qempty, 1);
    for (int i = 0; i < 3; ++i) { mbar_init(&bars.tfull[i], 1); mbar_init(&bars.tempty[i], 8); }
    mbar_init(&bars.epsync, 256);
    mbar_init(&bars.mdrain, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(&tmem_base, tmem_cols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  griddep_launch_dependents();
  const uint32_t tmem = tmem_base;
  volatile int* abort_v = &abort_flag;

  // The group table of a token map (uniform batches need none), then the
  // per-group tile counts and their exclusive prefix (block-wide scan).
  const int ngroups = grp != nullptr ? build_groups<kThreads>(P, grp, scan_tmp) : P.n_groups;
  // Group changes weigh in the split only when groups are many and short
  // (a prefill); a decode's few long groups split by tiles alone.
  const int group_cost = ngroups > kGroupCostMinGroups ? kGroupCost : 0;
  {
    const int ng = ngroups;
    const int per = (ng + kThreads - 1) / kThreads;
    const int g0 = min(ng, tid * per), g1 = min(ng, g0 + per);
    int local = 0, lcost = 0;
    for (int g = g0; g < g1; ++g) {
      const int tg = group_tiles(P, grp, g);
      local += tg;
      lcost += tg > 0 ? tg + group_cost : 0;
    }
    int incl = local, cincl = lcost;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, incl, o);
      const int c = __shfl_up_sync(0xffffffffu, cincl, o);
      if (lane >= o) { incl += n; cincl += c; }
    }
    if (lane == 31) { scan_tmp[warp] = incl; scan_tmp2[warp] = cincl; }
    __syncthreads();
    int woff = 0, cwoff = 0;
    for (int w2 = 0; w2 < warp; ++w2) { woff += scan_tmp[w2]; cwoff += scan_tmp2[w2]; }
    int run = woff + incl - local, crun = cwoff + cincl - lcost;
    for (int g = g0; g < g1; ++g) {
      tiles_prefix[g] = run;
      if (group_cost > 0) cost_prefix[g] = crun;
      const int tg = group_tiles(P, grp, g);
      run += tg;
      crun += tg > 0 ? tg + group_cost : 0;
    }
    if (tid == kThreads - 1) {
      tiles_prefix[ng] = run;
      if (group_cost > 0) cost_prefix[ng] = crun;
    }
    __syncthreads();
  }
  // Equal shares of the work's cost, as tile ranges: tile j of group g sits
  // at cost position cost_prefix[g] + group_cost + j, and a CTA takes the
  // tiles whose positions fall in its share.
  auto tiles_below = [&](long long u) -> int {  // tiles at positions below u
    int lo = 0, hi = ngroups;  // largest g with cost_prefix[g] <= u
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (cost_prefix[mid] <= u) lo = mid; else hi = mid;
    }
    const long long in_g = u - cost_prefix[lo] - group_cost;
    const int tg = tiles_prefix[lo + 1] - tiles_prefix[lo];
    return tiles_prefix[lo] + static_cast<int>(in_g < 0 ? 0 : (in_g > tg ? tg : in_g));
  };
  const long long total_cost = group_cost > 0 ? cost_prefix[ngroups] : tiles_prefix[ngroups];
  const long long u_lo = total_cost * blockIdx.x / gridDim.x, u_hi = total_cost * (blockIdx.x + 1) / gridDim.x;
  const int item_lo = group_cost > 0 ? tiles_below(u_lo) : static_cast<int>(u_lo);
  const int item_hi = group_cost > 0 ? tiles_below(u_hi) : static_cast<int>(u_hi);
  // First (group, tile) of this CTA's share: binary search in the prefix.
  Walker w0{0, 0, item_hi - item_lo};
  {
    int lo = 0, hi = ngroups;  // largest g with tiles_prefix[g] <= item_lo
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (tiles_prefix[mid] <= item_lo) lo = mid; else hi = mid;
    }
    while (lo < ngroups && tiles_prefix[lo + 1] <= item_lo) ++lo;
    w0.g = lo;
    w0.j = item_lo - tiles_prefix[lo];
  }

  if (warp == 12) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap)) : "memory");
      int st = 0;
      uint32_t ph = 0;
      // Per-group values are set at each group change; a contiguous cache
      // loads a tile as one box at row b * max_L + s0, without the per-box
      // arithmetic of the paged layout (this thread's loop is on the
      // critical path of every tile).
      const bool contiguous = P.block_table == nullptr;
      int cur_g = -1, maxpos_cache = -1, b = 0;
      int64_t row0 = 0;
      auto set_group = [&](int g) {
        const Group G = group_of(P, grp, g);
        cur_g = g;
        maxpos_cache = G.maxpos;
        b = G.b;
        row0 = static_cast<int64_t>(b) * P.max_L;
      };
      if (w0.left > 0) set_group(w0.g);
      griddep_wait();  // the key cache holds rows the previous kernel wrote
      int issued = 0;  // stages loaded, in order
      Walker w = w0;
      for (bool more = w.left > 0; more; more = walk_next(tiles_prefix, ngroups, w)) {
        const int g = w.g, j = w.j;
        if (g != cur_g) set_group(g);
        if (!mbar_wait(&bars.empty8[st], ph ^ 1, P.err, abort_v)) break;
        uint8_t* dst = s8 + st * tile8_bytes;
        const int s0 = j * kTileKeys;
        if (contiguous) {
          const int64_t row = row0 + s0;
          mbar_arrive_expect_tx(&bars.full8[st], static_cast<uint32_t>(kTileKeys * (DI + 2)));
          tma_load_2d(dst, &tmap, 0, static_cast<int>(row), &bars.full8[st]);
          bulk_g2s(&ks_s[st][0], P.k_scale + row, static_cast<uint32_t>(kTileKeys * 2), &bars.full8[st]);
          ++issued;
          if (++st == kStages8) { st = 0; ph ^= 1; }
          continue;
        }
        const int bh = P.box_rows;  // 128 (contiguous) or the page size (< 128)
        // Boxes of bh rows that cover the tile's visible keys (>= 1: the
        // walk only visits tiles with a visible key).
        const int n_loads = min(kTileKeys / bh, (maxpos_cache - s0) / bh + 1);
        mbar_arrive_expect_tx(&bars.full8[st], static_cast<uint32_t>(n_loads * bh * (DI + 2)));
        for (int c = 0; c < n_loads; ++c) {
          int64_t row = key_row(P, b, s0 + c * bh);
          if (row < 0) {  // unmapped page: flag it and load row 0 so the stage still completes
            atomicOr(P.err, kErrBadIndex);
            row = 0;
          }
          tma_load_2d(dst + c * bh * DI, &tmap, 0, static_cast<int>(row), &bars.full8[st]);
          // The box's key scales: bh * 2 bytes, 16-byte aligned (rows of a
          // box start at a multiple of 8, k_scale is 16-byte aligned).
          bulk_g2s(&ks_s[st][c * bh], P.k_scale + row, static_cast<uint32_t>(bh * 2), &bars.full8[st]);
        }
        ++issued;
        if (++st == kStages8) { st = 0; ph ^= 1; }
      }
      // If a wait gave up, the last stages' copies may still be in flight:
      // let them land before the CTA leaves (stage i % 8, phase i / 8; a
      // stage consumed already has completed that phase).
      for (int i = issued > kStages8 ? issued - kStages8 : 0; i < issued; ++i)
        mbar_drain(&bars.full8[i % kStages8], (i / kStages8) & 1);
    }
  } else if (warp >= 4 && warp < 8) {
    // ---------------------------------------------------------- converters
    griddep_wait();  // q comes from the previous kernel
    const int ct = tid - 128;  // 0..127
    int st8 = 0, st16 = 0;
    uint32_t ph8 = 0, ph16 = 0, qph = 0;
    int cur_g = -1;
    bool first_group = true;
    const int chunks = d_I / 16;  // 16-byte int8 chunks per row
    Walker w = w0;
    for (bool more = w.left > 0; more; more = walk_next(tiles_prefix, ngroups, w)) {
      const int g = w.g;
      if (g != cur_g) {
        cur_g = g;
        if (!first_group && !mbar_wait(&bars.qempty, qph, P.err, abort_v)) break;
        if (!first_group) qph ^= 1;
        first_group = false;
        const Group G = group_of(P, grp, g);
        const int rows_real = G.ntok * P.H_I;
        // in batches of 8 chunks per thread, every load of a batch issued
        // before any is used
        constexpr int kQBatch = 8;
        for (int b0 = ct; b0 < N * chunks; b0 += 128 * kQBatch) {
          uint4 qv[kQBatch];
#pragma unroll
          for (int i = 0; i < kQBatch; ++i) {
            const int task = b0 + i * 128;
            const int n = task / chunks, c = task % chunks;
            qv[i] = make_uint4(0, 0, 0, 0);
            if (task < N * chunks && n < rows_real)
              qv[i] = __ldg(reinterpret_cast<const uint4*>(P.q + (static_cast<size_t>(G.t0) * P.H_I + n) * d_I + c * 16));
          }
#pragma unroll
          for (int i = 0; i < kQBatch; ++i) {
            const int task = b0 + i * 128;
            if (task >= N * chunks) break;
            const int n = task / chunks, c = task % chunks;
            uint32_t f[8];
            i8x4_to_f16x4(qv[i].x, f[0], f[1]);
            i8x4_to_f16x4(qv[i].y, f[2], f[3]);
            i8x4_to_f16x4(qv[i].z, f[4], f[5]);
            i8x4_to_f16x4(qv[i].w, f[6], f[7]);
            uint8_t* atom = sQ + (c / 4) * (N * 128);
            const int cc = (c % 4) * 2;
            *reinterpret_cast<uint4*>(atom + sw128_off(n, cc)) = make_uint4(f[0], f[1], f[2], f[3]);
            *reinterpret_cast<uint4*>(atom + sw128_off(n, cc + 1)) = make_uint4(f[4], f[5], f[6], f[7]);
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.qfull);
      }
      if (!mbar_wait(&bars.full8[st8], ph8, P.err, abort_v)) break;
      if (!mbar_wait(&bars.empty16[st16], ph16 ^ 1, P.err, abort_v)) break;
      tc_fence_after();
      {
        // This thread's key row: TMA swizzle (16-byte chunk c of row r sits
        // at chunk c ^ (r & 7) for 128-byte rows, c ^ ((r >> 1) & 3) for
        // 64-byte rows), so a quarter warp reads 8 distinct bank groups.
        const int r = ct;
        const uint8_t* tile = s8 + st8 * tile8_bytes;
        constexpr uint32_t kSwMask = DI == 128 ? 7u : 3u;
        uint32_t f[DI / 2];
#pragma unroll
        for (int c = 0; c < DI / 16; ++c) {
          uint32_t off = static_cast<uint32_t>(r * DI + c * 16);
          off ^= ((off >> 7) & kSwMask) << 4;
          const uint4 v = *reinterpret_cast<const uint4*>(tile + off);
          i8x4_to_f16x4(v.x, f[8 * c + 0], f[8 * c + 1]);
          i8x4_to_f16x4(v.y, f[8 * c + 2], f[8 * c + 3]);
          i8x4_to_f16x4(v.z, f[8 * c + 4], f[8 * c + 5]);
          i8x4_to_f16x4(v.w, f[8 * c + 6], f[8 * c + 7]);
        }
        const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16) + a_col0 + st16 * (DI / 2);
#pragma unroll
        for (int c0 = 0; c0 < DI / 2; c0 += 32) {
          uint32_t rr[32];
#pragma unroll
          for (int k = 0; k < 32; ++k) rr[k] = f[c0 + k];
          tmem_st32(lane_base + c0, rr);
        }
        tmem_st_wait();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&bars.full16[st16]);
        mbar_arrive(&bars.empty8[st8]);
      }
      if (++st8 == kStages8) { st8 = 0; ph8 ^= 1; }
      if (++st16 == n16) { st16 = 0; ph16 ^= 1; }
    }
  } else if (warp == 13) {
    // -------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_f16(128, N, kFmtF16, 0, 0);
      int st16 = 0, acc = 0;
      uint32_t ph16 = 0, qph = 0, aph = 0;
      int cur_g = -1;
      Walker w = w0;
      for (bool more = w.left > 0; more;) {
        const int g = w.g;
        more = walk_next(tiles_prefix, ngroups, w);
        if (g != cur_g) {
          cur_g = g;
          if (!mbar_wait(&bars.qfull, qph, P.err, abort_v)) break;
          qph ^= 1;
        }
        if (!mbar_wait(&bars.full16[st16], ph16, P.err, abort_v)) break;
        if (!mbar_wait(&bars.tempty[acc], aph ^ 1, P.err, abort_v)) break;
        tc_fence_after();
        const uint32_t a_tmem = tmem + a_col0 + st16 * (DI / 2);
        const uint32_t b_base = smem_u32(sQ);
        const uint32_t d_tmem = tmem + acc * acc_stride;
#pragma unroll
        for (int kk = 0; kk < DI / 16; ++kk) {
          const uint64_t bd = smem_desc(b_base + (kk / 4) * (N * 128) + (kk % 4) * 32, 16, 1024, kSwizzle128B);
          mma_ts(d_tmem, a_tmem + kk * 8, bd, idesc, kk > 0 ? 1u : 0u);
        }
        mma_commit(&bars.empty16[st16]);
        mma_commit(&bars.tfull[acc]);
        const bool group_ends = !more || w.g != g;
        if (group_ends) mma_commit(&bars.qempty);
        if (++st16 == n16) { st16 = 0; ph16 ^= 1; }
        if (++acc == n_acc) { acc = 0; aph ^= 1; }
      }
      // every MMA issued has completed before the tensor memory is freed
      mma_commit(&bars.mdrain);
      mbar_drain(&bars.mdrain, 0);
    }
  } else if (warp < 4 || (warp >= 8 && warp < 12)) {
    // ---------------------------------------------------------- epilogue
    const int eg = warp >= 8 ? 1 : 0;  // token parity this group scores
    const int q4 = warp & 3;           // TMEM lane quarter
    const int et = eg * 128 + q4 * 32 + lane;  // 0..255 over both groups
    const int r = q4 * 32 + lane;      // key within the tile = TMEM lane
    // Barrier of the 256 epilogue threads on an mbarrier, so that a thread
    // that gave up (abort) makes the others time out instead of hanging.
    uint32_t ep_ph = 0;
    auto ep_sync = [&]() -> bool {
      mbar_arrive(&bars.epsync);
      const bool ok = mbar_wait(&bars.epsync, ep_ph, P.err, abort_v);
      ep_ph ^= 1;
      return ok;
    };
    int acc = 0;
    uint32_t aph = 0;
    int cur_g = -1;
    Group G{};
    const float ninf = -__int_as_float(0x7f800000);
    int st8 = 0;  // ring stage of the current item (same order as the producer)
    uint32_t ph8 = 0;
    const bool do_hist = kHist && P.hist != nullptr;
    auto flush_hist = [&]() -> bool {  // G is the group whose counts are flushed
      if (!ep_sync()) return false;
      for (int gi = 0; gi < G.ntok && gi < 2; ++gi)
        for (int bin = et; bin < kHistBins; bin += 256) {
          const uint32_t v = hist_s[gi * kHistBins + bin];
          if (v) {
            atomicAdd(P.hist + static_cast<size_t>(G.t0 + gi) * kHistBins + bin, v);
            hist_s[gi * kHistBins + bin] = 0;
          }
        }
      return ep_sync();
    };
    auto release = [&]() {  // this warp has read the accumulator
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.tempty[acc]);
    };
    // Scores one item; false if a wait gave up.
    auto score_item = [&](const Walker& it) -> bool {
      const int g = it.g, j = it.j;
      if (g != cur_g) {
        if (do_hist && cur_g >= 0 && !flush_hist()) return false;
        cur_g = g;
        G = group_of(P, grp, g);
        if (!ep_sync()) return false;
        for (int n = et; n < kCoef; n += 256) {
          const int gi = n / HI, h = n % HI;
          float c = 0.f;
          if (gi < G.ntok && h < P.H_I) {
            const int t = G.t0 + gi;
            c = __ldg(P.w + static_cast<size_t>(t) * P.H_I + h) *
                __half2float(__ldg(P.q_scale + static_cast<size_t>(t) * P.H_I + h));
          }
          coef[n] = c;
        }
        for (int gi = et; gi < kMaxG; gi += 256) tok_pos[gi] = (gi < G.ntok) ? __ldg(P.pos + G.t0 + gi) : -1;
        if (!ep_sync()) return false;
      }
      if (!mbar_wait(&bars.tfull[acc], aph, P.err, abort_v)) return false;
      tc_fence_after();
      // This key's scale from the ring stage (complete long ago: the
      // converters consumed it before the MMA); then free the stage.
      if (!mbar_wait(&bars.full8[st8], ph8, P.err, abort_v)) return false;
      const float ks = __half2float(__ushort_as_half(ks_s[st8][r]));
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.empty8[st8]);
      if (++st8 == kStages8) { st8 = 0; ph8 ^= 1; }
      const int s = j * kTileKeys + r;
      const uint32_t lane_addr = tmem + (static_cast<uint32_t>(q4 * 32) << 16) + acc * acc_stride;
      bool released = false;
      // Column n = gi * HI + h of the accumulator is token gi, head h.
      if (HI >= 32) {
        for (int gi = eg; gi < G.ntok; gi += 2) {
          // Head-weighted ReLU sum with packed fp32x2 FMAs over head pairs.
          uint64_t part[2] = {0ull, 0ull};
#pragma unroll
          for (int c = 0; c < HI / 32; c += 2) {
            uint32_t v0[32], v1[32];
            tmem_ld32(lane_addr + gi * HI + c * 32, v0);
            if (c + 1 < HI / 32) tmem_ld32(lane_addr + gi * HI + (c + 1) * 32, v1);
            tmem_ld_wait();
            if (gi + 2 >= G.ntok && c + 2 >= HI / 32) {  // last columns this warp reads
              release();
              released = true;
            }
            const uint64_t* cf = reinterpret_cast<const uint64_t*>(coef + gi * HI + c * 32);
#pragma unroll
            for (int k = 0; k < 16; ++k)
              part[k & 1] = fma_f32x2(cf[k], relu_pair(v0[2 * k], v0[2 * k + 1]), part[k & 1]);
            if (c + 1 < HI / 32) {
#pragma unroll
              for (int k = 0; k < 16; ++k)
                part[k & 1] = fma_f32x2(cf[16 + k], relu_pair(v1[2 * k], v1[2 * k + 1]), part[k & 1]);
            }
          }
          const float sacc = (lo_f32(part[0]) + hi_f32(part[0])) + (lo_f32(part[1]) + hi_f32(part[1]));
          const bool vis = s <= tok_pos[gi];
          const float val = vis ? sacc * ks : ninf;
          P.scores[static_cast<size_t>(G.t0 + gi) * P.ld + s] = val;
          if (kHist && do_hist && vis && gi < 2) atomicAdd(&hist_s[gi * kHistBins + (order_key(val) >> 20)], 1u);
        }
      } else {
        constexpr int kTokPerChunk = HI >= 32 ? 1 : 32 / HI;
        const int n_chunks = (G.ntok * HI + 31) / 32;
        for (int cc = eg; cc < n_chunks; cc += 2) {
          uint32_t v[32];
          tmem_ld32(lane_addr + cc * 32, v);
          tmem_ld_wait();
          if (cc + 2 >= n_chunks) {
            release();
            released = true;
          }
#pragma unroll
          for (int u = 0; u < kTokPerChunk; ++u) {
            const int gi = cc * kTokPerChunk + u;
            float part[2] = {0.f, 0.f};
#pragma unroll
            for (int k = 0; k < HI; ++k)
              part[k & 1] = fmaf(coef[cc * 32 + u * HI + k], fmaxf(__uint_as_float(v[u * HI + k]), 0.f), part[k & 1]);
            if (gi < G.ntok)
              P.scores[static_cast<size_t>(G.t0 + gi) * P.ld + s] =
                  (s <= tok_pos[gi]) ? (part[0] + part[1]) * ks : ninf;
          }
        }
      }
      if (!released) release();  // nothing of this tile for this group
      if (++acc == n_acc) { acc = 0; aph ^= 1; }
      return true;
    };

    griddep_wait();  // w and qs come from the previous kernel
    bool aborted = false;
    Walker w = w0;
    for (bool more = w.left > 0; more; more = walk_next(tiles_prefix, ngroups, w))
      if (!score_item(w)) { aborted = true; break; }
    if (do_hist && cur_g >= 0 && !aborted) flush_hist();
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
  int b = t / P.n_q;
  if (P.seq != nullptr) {
    b = __ldg(P.seq + t);
    if (b < 0 || b >= P.B) return;
  }
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

IdxParams make_params(const dsa_topk_args& a, float* scores, int64_t ld, uint32_t* hist) {
  IdxParams P{};
  P.T = a.T; P.B = a.B; P.n_q = a.n_q; P.H_I = a.H_I; P.d_I = a.d_I; P.max_L = a.max_L;
  P.seq = a.seq_of_token;
  P.G = indexer_group_tokens(a);
  P.N = static_cast<int>(round_up(static_cast<size_t>(P.G) * a.H_I, 16));
  if (P.seq != nullptr) {
    // runs of adjacent tokens of one sequence, each cut into G-token groups:
    // at most ceil(T / G) + B groups when every sequence's tokens are adjacent
    P.groups_per_seq = 0;
    const long long ub = (a.T + P.G - 1) / P.G + static_cast<long long>(a.B);
    P.n_groups = static_cast<int>(ub < a.T ? ub : a.T);
  } else {
    P.groups_per_seq = (a.n_q + P.G - 1) / P.G;
    P.n_groups = a.B * P.groups_per_seq;
  }
  P.n_tiles = a.max_L / kTileKeys;
  P.q = a.q; P.q_scale = reinterpret_cast<const __half*>(a.q_scale); P.w = a.w;
  P.k_cache = a.k_cache; P.k_scale = reinterpret_cast<const __half*>(a.k_scale);
  P.block_table = a.block_table; P.block_size = a.block_size; P.max_blocks = a.max_blocks;
  P.pos = a.pos; P.scores = scores; P.ld = ld; P.hist = hist;
  P.err = error_word();
  return P;
}

// Dynamic shared memory: alignment slack, the int8 ring, Q, the tile prefix
// and (token map) the group table.
size_t indexer_smem(const IdxParams& P, int DI) {
  size_t n = 1024 + static_cast<size_t>(kStages8) * kTileKeys * DI + static_cast<size_t>(P.N) * DI * 2;
  n += 4 * static_cast<size_t>(P.n_groups + 1);
  if (P.seq != nullptr) n += 2 * static_cast<size_t>(P.n_groups + 1);
  return n;
}

constexpr size_t kSmemPerBlock = 232448;  // 227 KB opt-in limit of sm_103a

template <int HI, int DI>
cudaError_t launch_hi(const IdxParams& P, const CUtensorMap& tmap, cudaStream_t s, bool& too_big) {
  const size_t smem = indexer_smem(P, DI);
  cudaFuncAttributes fa{};
  cudaError_t e = cudaFuncGetAttributes(&fa, indexer_kernel<HI, DI>);
  if (e != cudaSuccess) return e;
  too_big = smem + fa.sharedSizeBytes > kSmemPerBlock;
  if (too_big) return cudaSuccess;
  e = cudaFuncSetAttribute(indexer_kernel<HI, DI>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
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
  return cudaLaunchKernelEx(&cfg, indexer_kernel<HI, DI>, P, tmap);
}

template <int DI>
cudaError_t launch_di(int H_I, const IdxParams& P, const CUtensorMap& tmap, cudaStream_t s, bool& too_big) {
  switch (H_I) {
    case 4: return launch_hi<4, DI>(P, tmap, s, too_big);
    case 8: return launch_hi<8, DI>(P, tmap, s, too_big);
    case 16: return launch_hi<16, DI>(P, tmap, s, too_big);
    case 32: return launch_hi<32, DI>(P, tmap, s, too_big);
    case 64: return launch_hi<64, DI>(P, tmap, s, too_big);
    default: return launch_hi<128, DI>(P, tmap, s, too_big);
  }
}

}  // namespace

int indexer_group_tokens(const dsa_topk_args& a) {
  // 128 query rows (tokens x heads) per MMA; a uniform batch never groups
  // more tokens than one sequence has
  int G = a.H_I >= 128 ? 1 : 128 / a.H_I;
  if (a.seq_of_token == nullptr && a.n_q < G) G = a.n_q;
  return G < kMaxG ? G : kMaxG;
}

int launch_indexer(const dsa_topk_args& a, float* scores, uint32_t* hist, cudaStream_t s) {
  IdxParams P = make_params(a, scores, a.max_L, hist);
  if (!P.err) return DSA_ERR_CUDA;
  if (a.H_I != 4 && a.H_I != 8 && a.H_I != 16 && a.H_I != 32 && a.H_I != 64 && a.H_I != 128)
    return DSA_ERR_UNSUPPORTED;
  // One TMA box is a whole 128-key tile of a contiguous cache, or one page.
  P.box_rows = a.block_table ? (a.block_size < kTileKeys ? a.block_size : kTileKeys) : kTileKeys;
  const uint64_t rows = a.block_table ? (1ull << 31) - 1 : static_cast<uint64_t>(a.B) * a.max_L;
  alignas(64) CUtensorMap tmap;
  if (!encode_tmap_u8_2d(&tmap, a.k_cache, a.d_I, rows, a.d_I, P.box_rows, a.d_I == 128 ? 128 : 64))
    return DSA_ERR_CUDA;
  bool too_big = false;
  const cudaError_t e =
      a.d_I == 128 ? launch_di<128>(a.H_I, P, tmap, s, too_big) : launch_di<64>(a.H_I, P, tmap, s, too_big);
  if (e == cudaSuccess && too_big) return DSA_ERR_UNSUPPORTED;  // too many token groups
  return cuda_status(e);
}

int launch_indexer_dots(const dsa_topk_args& a, int32_t* dots, cudaStream_t s) {
  const IdxParams P = make_params(a, nullptr, a.max_L, nullptr);
  dim3 grid((a.max_L + 127) / 128, a.T);
  dots_kernel<<<grid, 128, 0, s>>>(P, dots);
  return cuda_status(cudaGetLastError());
}

}  // namespace dsa

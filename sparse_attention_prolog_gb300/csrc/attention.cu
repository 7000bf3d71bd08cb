// Sparse MLA flash attention over the top-k latent rows, on tcgen05.
//
// [V4-TileLang §Sparse Flash Attention] steps: (1) parallel over (b, m);
// (2) idx = topk_idxs[...] or -1 past topk, gather the kv rows and build the
// mask; (3) S = q . k^T, mask, scale; (4) online softmax with running max
// and sum; (5) P . V; (6) accumulate and rescale; (8) write back.
// [V3.2-PyPTO §Deepseek Indexer Attention] found the discrete gather to be
// over 70% of the fused operator and fixed it by gathering straight into the
// matrix unit's buffer.  On sm_103a the same idea is a cp.async row gather
// straight into the 128B-swizzled layout tcgen05 reads.
//
// One 2-CTA cluster per (token, head block of 128, chunk of R selected rows):
//
//   CTA 0  (QK + softmax): q [128 x 576] bf16 lives in TMEM (288 columns)
//          and is the A operand of S = q . K^T (M=128 heads, N=64 rows,
//          K=576); S is double-buffered in TMEM.  Four softmax warps (one
//          thread per head) apply the mask and scale, keep the running max
//          (rescaling only when it grows by more than 2^8) and the row sum,
//          and store P (bf16) and the per-row rescale factor straight into
//          CTA 1's shared memory with st.async.
//   CTA 1  (PV): O [128 x 512] fp32 fills its whole TMEM; P (shared memory,
//          K-major) times V (the first 512 dims of the gathered rows, read
//          MN-major from the same swizzled layout) accumulates into O.
//          Correction warps rescale O rows in the rare case the max grew;
//          at the end they and the MMA warpgroup normalise O and write it
//          (or a split-K partial) with TMA stores.
//
// Both CTAs gather the same rows (the second read is an L2 hit), each with
// 16 warps.  Chunks of one token are merged by attn_combine_kernel with
// their log-sum-exp.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include "dsa_internal.h"
#include "dsa_ptx.cuh"

namespace dsa {
namespace {

constexpr int kDqk = 576, kDv = 512;
constexpr int kRows = 64;                       // rows per tile
constexpr int kAtomsK = kDqk / 64;              // 9 swizzle atoms per full row
constexpr int kAtomsV = kDv / 64;               // 8
constexpr int kStageK = kAtomsK * kRows * 128;  // 73,728 B
constexpr int kStageV = kAtomsV * kRows * 128;  // 65,536 B
constexpr int kStagesK = 3, kStagesV = 2;
constexpr int kPSlot = 128 * 128;               // P tile [128 heads x 64 rows] bf16
// 24 warps in six warpgroups: 0 softmax / correction (and half of the
// epilogue), 1-4 gather, 5 MMA, relay and the other half of the epilogue.
// The gather warpgroups give registers to the other two (setmaxnreg): the
// launch grants 80 per thread, 768 x 80 = 128 x 168 + 512 x 40 + 128 x 152.
constexpr int kThreads = 768;
constexpr int kGatherWarps = 16, kRowsPerWarp = 64 / kGatherWarps;  // rows of a tile per gather warp
constexpr int kMmaWarp = 20, kRelayWarp = 21;
constexpr int kRegsLaunch = 80, kRegsSoftmax = 168, kRegsGather = 40, kRegsLast = 152;
static_assert(128 * kRegsSoftmax + 4 * 128 * kRegsGather + 128 * kRegsLast <= kThreads * kRegsLaunch,
              "register split exceeds the launch allocation");
constexpr int kOutAtom = 128 * 128;  // output staging atom [128 heads x 64 cols] bf16
constexpr uint32_t kPBytes = 128 * (8 * 16 + 4);  // P row + alpha, per tile
constexpr uint32_t kFinalBytes = 128 * 8;
constexpr uint32_t kTmemQ = 0, kTmemS = 288;    // CTA 0 column map
constexpr int kSmemA = kStagesK * kStageK;  // 221,184 B

struct AttnParams {
  int T, B, n_q, H, topk, max_L, n_chunks, chunk_rows, head_blocks;
  const int32_t* seq;  // [T] sequence of each token, or null (token t in sequence t / n_q)
  float scale_log2;
  const __nv_bfloat16* q;
  const __nv_bfloat16* kv;
  const int32_t* block_table;
  int block_size, max_blocks;
  const int32_t* idx;
  __nv_bfloat16* out;
  float* lse;
  const float* sink;      // [H] attention sink logits (natural-log units), or null
  __nv_bfloat16* part_o;  // [T][n_chunks][H][512], O_c / l_c, when n_chunks > 1
  float2* part_ml; // [T][n_chunks][H]: (max, sum) in log2 units
  uint32_t* err;
};

struct __align__(8) Bars {
  uint64_t kfull[kStagesK], kempty[kStagesK];   // CTA 0 gather ring
  uint64_t sfull[2], sempty[2];                 // CTA 0 S buffers
  uint64_t pfree[2];                            // CTA 0: P slot of CTA 1 free
  uint64_t vfull[kStagesV], vempty[kStagesV];   // CTA 1 gather ring
  uint64_t pfull[2], pcons[2];                  // CTA 1 P slots
  uint64_t ready[2], odone, ffull;              // CTA 1 correction / MMA
  uint64_t alldone;                             // CTA 1: every PV MMA complete
  uint64_t qready;                              // CTA 0: q is in TMEM
  uint64_t tiles;                               // the chunk's tile count is known (gather warps)
  uint64_t mdrain;                              // the MMA thread's last commit
};

__device__ __forceinline__ int64_t kv_row(const AttnParams& P, int b, int s) {
  if (P.block_table == nullptr) return static_cast<int64_t>(b) * P.max_L + s;
  const int blk = __ldg(P.block_table + static_cast<size_t>(b) * P.max_blocks + s / P.block_size);
  return blk < 0 ? -1 : static_cast<int64_t>(blk) * P.block_size + s % P.block_size;
}

// Physical row of the slot this lane looks up for tile slot0 of producer
// warp pw (lane l covers row pw*kRowsPerWarp + l%kRowsPerWarp); -1 for
// masked slots.
__device__ __forceinline__ long long gather_row(const AttnParams& P, const int32_t* idx_row, int b, int slot0,
                                                int pw, int lane) {
  const int slot = slot0 + pw * kRowsPerWarp + (lane % kRowsPerWarp);
  const int s = (slot < P.topk) ? __ldg(idx_row + slot) : -1;
  return (s >= 0 && s < P.max_L) ? kv_row(P, b, s) : -1;
}

// Gathers the 64 rows of one tile into a swizzled stage: `atoms` 64-dim
// atoms of every row, zero rows for masked slots.  Producer warp pw owns
// rows pw*kRowsPerWarp .. +kRowsPerWarp-1 whose physical addresses (one per
// lane, see gather_row, looked up a tile ahead) are broadcast by shuffle.
// Lanes copy consecutive 16-byte chunks of a row (coalesced) with cp.async.
// A random-row gather is bound by the memory requests an SM keeps in
// flight, so sixteen warps of every CTA gather.
__device__ __forceinline__ void gather_tile(const AttnParams& P, long long row, uint8_t* stage, int atoms, int pw,
                                            int lane) {
  const int chunks = atoms * 8;
  const uint32_t sbase = smem_u32(stage);
#pragma unroll 4
  for (int rr = 0; rr < kRowsPerWarp; ++rr) {
    const long long prow = __shfl_sync(0xffffffffu, row, rr);
    const int r = pw * kRowsPerWarp + rr;
    const __nv_bfloat16* rsrc = P.kv + (prow >= 0 ? prow : 0) * kDqk;
    const uint32_t bytes = prow >= 0 ? 16u : 0u;
    for (int c = lane; c < chunks; c += 32)
      cp_async16(sbase + (c >> 3) * (kRows * 128) + sw128_off(r, c & 7), rsrc + c * 8, bytes);
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    sparse_attn_kernel(const __grid_constant__ AttnParams P, const __grid_constant__ CUtensorMap tmap_o) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ Bars bars;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_ctarank();
  const int chunk = blockIdx.x >> 1, hb = blockIdx.y, t = blockIdx.z;
  int b = t / P.n_q;
  bool bad_seq = false;
  if (P.seq != nullptr) {  // a token outside [0, B) reads no row and gets out = 0
    b = __ldg(P.seq + t);
    bad_seq = b < 0 || b >= P.B;
    if (bad_seq) {
      if (tid == 0 && rank == 0 && chunk == 0 && hb == 0) atomicOr(P.err, kErrBadIndex);
      b = 0;
    }
  }
  const int slot_begin = chunk * P.chunk_rows;
  const int rows_here = bad_seq ? 0 : max(0, min(P.chunk_rows, P.topk - slot_begin));
  // The chunk's tiles end at its last valid index (slots past it are masked
  // and add nothing): the gather warps find it once the index rows are
  // there and publish the count; every other role waits for it.
  __shared__ int last_valid, n_tiles_sh;
  const int32_t* idx_row = P.idx + static_cast<size_t>(t) * P.topk;

  // CTA 1 layout: V stages, then P slots, alpha, final (m, l)
  uint8_t* sV = smem;
  uint8_t* sP = smem + kStagesV * kStageV;
  float* sAlpha = reinterpret_cast<float*>(sP + 2 * kPSlot);  // [2][128]
  float2* sFinal = reinterpret_cast<float2*>(sAlpha + 256);     // [128]
  uint8_t* sK = smem;                                           // CTA 0: K stages

  if (tid == 0) {
    for (int i = 0; i < kStagesK; ++i) { mbar_init(&bars.kfull[i], kGatherWarps * 32); mbar_init(&bars.kempty[i], 1); }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars.sfull[i], 1); mbar_init(&bars.sempty[i], 4); mbar_init(&bars.pfree[i], 1);
      mbar_init(&bars.pfull[i], 1); mbar_init(&bars.pcons[i], 1); mbar_init(&bars.ready[i], 4);
    }
    for (int i = 0; i < kStagesV; ++i) { mbar_init(&bars.vfull[i], kGatherWarps * 32); mbar_init(&bars.vempty[i], 1); }
    mbar_init(&bars.odone, 1);
    mbar_init(&bars.alldone, 1);
    mbar_init(&bars.ffull, 1);
    mbar_init(&bars.qready, 4);
    mbar_init(&bars.tiles, 1);
    last_valid = -1;
    mbar_init(&bars.mdrain, 1);
    abort_flag = 0;
    fence_mbar_init();
    if (rank == 1) {
      mbar_arrive_expect_tx(&bars.pfull[0], kPBytes);
      mbar_arrive_expect_tx(&bars.pfull[1], kPBytes);
      mbar_arrive_expect_tx(&bars.ffull, kFinalBytes);
    }
  }
  if (warp == 0) tmem_alloc(&tmem_base, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;
  volatile int* abort_v = &abort_flag;
  const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
  auto tile_count = [&]() -> int {  // roles other than the gather warps
    if (!mbar_wait_polling<false>(&bars.tiles, 0, P.err, abort_v)) return 0;
    return n_tiles_sh;
  };

  const int q_rows = max(0, min(128, P.H - hb * 128));  // real heads of this block
  cluster_sync();  // both CTAs' barriers are initialised before any remote use
  griddep_launch_dependents();
  // Roles wait for the previous kernel (griddep_wait) only before reading
  // what it wrote (topk_idx); q and the kv cache are this call's inputs, so
  // q is in TMEM before the top-k has finished.

  if (warp >= 4 && warp < 4 + kGatherWarps) {
    setmaxnreg_dec<kRegsGather>();
    griddep_wait();  // the index rows come from the previous kernel
    // the first tile's rows are looked up together with the chunk's last slot
    long long row_next = rows_here > 0 ? gather_row(P, idx_row, b, slot_begin, warp - 4, lane) : -1;
    int n_tiles;
    {
      // a valid last slot (every decode chunk) ends the chunk at once; else
      // the gather warps find the last valid slot together
      const int last = rows_here > 0 ? __ldg(idx_row + slot_begin + rows_here - 1) : -1;
      if (rows_here == 0 || (last >= 0 && last < P.max_L)) {
        n_tiles = (rows_here + kRows - 1) / kRows;
      } else {
        int mx = -1;
        for (int i = (warp - 4) * 32 + lane; i < rows_here; i += kGatherWarps * 32) {
          const int s = __ldg(idx_row + slot_begin + i);
          if (s >= 0 && s < P.max_L) mx = i;
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        if (lane == 0 && mx >= 0) atomicMax(&last_valid, mx);
        asm volatile("bar.sync 1, %0;" ::"n"(kGatherWarps * 32) : "memory");
        n_tiles = (last_valid + kRows) / kRows;
      }
      if (warp == 4 && lane == 0) {
        n_tiles_sh = n_tiles;
        mbar_arrive(&bars.tiles);
      }
    }
    if (rank == 0) {
      // ------------------------------------------------ gather K (CTA 0)
      int st = 0;
      uint32_t ph = 0;
      for (int j = 0; j < n_tiles; ++j) {
        const long long row = row_next;
        if (j + 1 < n_tiles) row_next = gather_row(P, idx_row, b, slot_begin + (j + 1) * kRows, warp - 4, lane);
        if (!mbar_wait_polling<false>(&bars.kempty[st], ph ^ 1, P.err, abort_v)) break;
        gather_tile(P, row, sK + st * kStageK, kAtomsK, warp - 4, lane);
        // the stage's barrier counts this thread once its copies have landed
        cp_async_mbar_arrive(&bars.kfull[st]);
        if (++st == kStagesK) { st = 0; ph ^= 1; }
      }
      asm volatile("cp.async.wait_all;" ::: "memory");
    } else {
      // ------------------------------------------------ gather V (CTA 1)
      int st = 0;
      uint32_t ph = 0;
      for (int j = 0; j < n_tiles; ++j) {
        const long long row = row_next;
        if (j + 1 < n_tiles) row_next = gather_row(P, idx_row, b, slot_begin + (j + 1) * kRows, warp - 4, lane);
        if (!mbar_wait_polling<false>(&bars.vempty[st], ph ^ 1, P.err, abort_v)) break;
        gather_tile(P, row, sV + st * kStageV, kAtomsV, warp - 4, lane);
        // the stage's barrier counts this thread once its copies have landed
        cp_async_mbar_arrive(&bars.vfull[st]);
        if (++st == kStagesV) { st = 0; ph ^= 1; }
      }
      asm volatile("cp.async.wait_all;" ::: "memory");
    }
  } else {
    bool ok = true;
    int n_tiles = -1;  // set by each role where it first needs it (tile_count)
    if (warp < 4) {
      setmaxnreg_inc<kRegsSoftmax>();
      if (rank == 0) {
        // ------------------------------------------------- softmax (CTA 0)
        const int hrow = warp * 32 + lane;
        const uint32_t remote_p = mapa(smem_u32(sP), 1);
        const uint32_t remote_alpha = mapa(smem_u32(sAlpha), 1);
        const uint32_t remote_final = mapa(smem_u32(sFinal), 1);
        const uint32_t remote_pfull[2] = {mapa(smem_u32(&bars.pfull[0]), 1), mapa(smem_u32(&bars.pfull[1]), 1)};
        const uint32_t remote_ffull = mapa(smem_u32(&bars.ffull), 1);
        // The pairs of the first half of the tokens start first (lowest block
        // indices); each pulls its slice of the query of token t + T/2 into
        // L2 for the pairs that may start only when SMs free up.
        if (P.n_chunks > 1 && t < P.T / 2 && hrow == 0) {
          const int t2 = t + P.T / 2;
          const int per = (q_rows + P.n_chunks - 1) / P.n_chunks;
          const int h0 = chunk * per, nh = min(per, q_rows - h0);
          if (nh > 0) prefetch_l2(P.q + (static_cast<size_t>(t2) * P.H + hb * 128 + h0) * kDqk, nh * kDqk * 2);
        }
        // q row of this thread's head: global -> registers -> TMEM columns
        // [0, 288), three atoms (24 independent 16-byte loads) per round.
        {
          const uint4* qrow = reinterpret_cast<const uint4*>(P.q + (static_cast<size_t>(t) * P.H + hb * 128 + hrow) * kDqk);
          const bool real = hrow < q_rows;
  #pragma unroll 1
          for (int a0 = 0; a0 < kAtomsK; a0 += 3) {
            uint4 v[24];
  #pragma unroll
            for (int i = 0; i < 24; ++i) v[i] = real ? __ldg(qrow + a0 * 8 + i) : make_uint4(0, 0, 0, 0);
  #pragma unroll
            for (int a = 0; a < 3; ++a) {
              uint32_t r[32];
  #pragma unroll
              for (int c = 0; c < 8; ++c) {
                r[4 * c] = v[a * 8 + c].x; r[4 * c + 1] = v[a * 8 + c].y;
                r[4 * c + 2] = v[a * 8 + c].z; r[4 * c + 3] = v[a * 8 + c].w;
              }
              tmem_st32(tmem + lane_off + kTmemQ + (a0 + a) * 32, r);
            }
          }
          tmem_st_wait();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.qready);
        griddep_wait();  // the index rows come from the previous kernel
        const float ninf = -__int_as_float(0x7f800000);
        float m_used = ninf, l_sum = 0.f;
        int sb = 0;
        uint32_t phs = 0;
        bool ok = true;
        // this lane's two index slots of a tile, loaded one tile ahead
        auto load_idx = [&](int jj, int& lo, int& hi) {
          const int slot0 = slot_begin + jj * kRows;
          lo = (slot0 + lane < P.topk) ? __ldg(idx_row + slot0 + lane) : -1;
          hi = (slot0 + 32 + lane < P.topk) ? __ldg(idx_row + slot0 + 32 + lane) : -1;
        };
        int nx_lo = -1, nx_hi = -1;
        if (rows_here > 0) load_idx(0, nx_lo, nx_hi);  // before the tile count: one round trip
        n_tiles = tile_count();
        for (int j = 0; j < n_tiles && ok; ++j) {
          const int s_lo = nx_lo, s_hi = nx_hi;
          if (j + 1 < n_tiles) load_idx(j + 1, nx_lo, nx_hi);
          if (!mbar_wait_polling<false>(&bars.sfull[sb], phs, P.err, abort_v)) { ok = false; break; }
          const uint32_t v_lo = __ballot_sync(0xffffffffu, s_lo >= 0 && s_lo < P.max_L);
          const uint32_t v_hi = __ballot_sync(0xffffffffu, s_hi >= 0 && s_hi < P.max_L);
          tc_fence_after();
          uint32_t s0[32], s1[32];
          tmem_ld32(tmem + lane_off + kTmemS + sb * kRows, s0);
          tmem_ld32(tmem + lane_off + kTmemS + sb * kRows + 32, s1);
          tmem_ld_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars.sempty[sb]);
          float x[64];
          float mt = ninf;
  #pragma unroll
          for (int k = 0; k < 32; ++k) {
            x[k] = ((v_lo >> k) & 1u) ? __uint_as_float(s0[k]) * P.scale_log2 : ninf;
            x[32 + k] = ((v_hi >> k) & 1u) ? __uint_as_float(s1[k]) * P.scale_log2 : ninf;
            mt = fmaxf(mt, fmaxf(x[k], x[32 + k]));
          }
          float alpha = 1.f;
          if (mt > m_used + 8.f) {  // also taken when m_used is -inf
            alpha = ex2_approx(m_used - mt);
            l_sum *= alpha;
            m_used = mt;
          }
          uint32_t pk[32];
          float lt = 0.f;
  #pragma unroll
          for (int k = 0; k < 32; ++k) {
            const float p0 = (x[2 * k] == ninf) ? 0.f : ex2_approx(x[2 * k] - m_used);
            const float p1 = (x[2 * k + 1] == ninf) ? 0.f : ex2_approx(x[2 * k + 1] - m_used);
            lt += p0 + p1;
            __nv_bfloat162 pb = __floats2bfloat162_rn(p0, p1);
            pk[k] = *reinterpret_cast<uint32_t*>(&pb);
          }
          l_sum += lt;
          const int ps = j & 1;
          if (!mbar_wait_polling<true>(&bars.pfree[ps], ((j >> 1) & 1) ^ 1, P.err, abort_v)) { ok = false; break; }
          const uint32_t prow = remote_p + ps * kPSlot;
  #pragma unroll
          for (int c = 0; c < 8; ++c)
            st_async_v4(prow + sw128_off(hrow, c), make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]),
                        remote_pfull[ps]);
          st_async_b32(remote_alpha + (ps * 128 + hrow) * 4, __float_as_uint(alpha), remote_pfull[ps]);
          if (++sb == 2) { sb = 0; phs ^= 1; }
        }
        st_async_v2(remote_final + hrow * 8, __float_as_uint(m_used), __float_as_uint(l_sum), remote_ffull);
      } else {
        // ----------------------------------------- correction (CTA 1)
        n_tiles = tile_count();
        const int hrow = warp * 32 + lane;
        int consumed = 0;  // odone phases observed
        for (int j = 0; j < n_tiles && ok; ++j) {
          const int ps = j & 1;
          if (!mbar_wait_polling<true>(&bars.pfull[ps], (j >> 1) & 1, P.err, abort_v)) { ok = false; break; }
          const float alpha = sAlpha[ps * 128 + hrow];
          const bool need = __any_sync(0xffffffffu, alpha != 1.f) && j > 0;
          if (need) {
            // O must hold PV of tile j-1 before it is rescaled.
            while (consumed < j) {
              if (!mbar_wait_polling<false>(&bars.odone, consumed & 1, P.err, abort_v)) { ok = false; break; }
              ++consumed;
            }
            if (!ok) break;
            tc_fence_after();
            for (int c0 = 0; c0 < kDv; c0 += 32) {
              uint32_t v[32];
              tmem_ld32(tmem + lane_off + c0, v);
              tmem_ld_wait();
  #pragma unroll
              for (int k = 0; k < 32; ++k) v[k] = __float_as_uint(__uint_as_float(v[k]) * alpha);
              tmem_st32(tmem + lane_off + c0, v);
            }
            tmem_st_wait();
            tc_fence_before();
          }
          fence_proxy_async_smem();  // P arrived through st.async; the MMA reads it
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars.ready[ps]);
          // keep at most one PV completion unobserved
          while (consumed < j) {
            if (!mbar_wait_polling<false>(&bars.odone, consumed & 1, P.err, abort_v)) { ok = false; break; }
            ++consumed;
          }
        }
      }
    } else {
      setmaxnreg_inc<kRegsLast>();
      if (warp == kMmaWarp && rank == 0) {
        // ---------------------------------------------- QK^T MMA (CTA 0)
        if (lane == 0) {
          n_tiles = tile_count();
          const uint32_t idesc = idesc_f16(128, kRows, kFmtBF16, 0, 0);
          int st = 0, sb = 0;
          uint32_t ph = 0, phs = 0;
          if (n_tiles > 0 && mbar_wait_polling<false>(&bars.qready, 0, P.err, abort_v)) tc_fence_after();
          for (int j = 0; j < n_tiles; ++j) {
            if (!mbar_wait_polling<false>(&bars.kfull[st], ph, P.err, abort_v)) break;
            if (!mbar_wait_polling<false>(&bars.sempty[sb], phs ^ 1, P.err, abort_v)) break;
            fence_proxy_async_smem();  // cp.async (generic proxy) data -> tensor core reads
            tc_fence_after();
            const uint32_t base = smem_u32(sK + st * kStageK);
            for (int kk = 0; kk < kDqk / 16; ++kk) {
              const uint64_t bd = smem_desc(base + (kk / 4) * (kRows * 128) + (kk % 4) * 32, 16, 1024, kSwizzle128B);
              mma_ts(tmem + kTmemS + sb * kRows, tmem + kTmemQ + kk * 8, bd, idesc, kk > 0 ? 1u : 0u);
            }
            mma_commit(&bars.kempty[st]);
            mma_commit(&bars.sfull[sb]);
            if (++st == kStagesK) { st = 0; ph ^= 1; }
            if (++sb == 2) { sb = 0; phs ^= 1; }
          }
          // every MMA issued has completed before the tensor memory is freed
          mma_commit(&bars.mdrain);
          mbar_drain(&bars.mdrain, 0);
        }
      } else if (warp == kMmaWarp) {
        // ------------------------------------------------- PV MMA (CTA 1)
        if (lane == 0) {
          n_tiles = tile_count();
          const uint32_t idesc = idesc_f16(128, 256, kFmtBF16, 0, 1);
          int st = 0;
          uint32_t ph = 0;
          for (int j = 0; j < n_tiles; ++j) {
            const int ps = j & 1;
            if (!mbar_wait_polling<false>(&bars.vfull[st], ph, P.err, abort_v)) break;
            if (!mbar_wait_polling<false>(&bars.ready[ps], (j >> 1) & 1, P.err, abort_v)) break;
            fence_proxy_async_smem();  // cp.async / st.async data -> tensor core reads
            tc_fence_after();
            const uint32_t pbase = smem_u32(sP + ps * kPSlot);
            const uint32_t vbase = smem_u32(sV + st * kStageV);
            for (int kk = 0; kk < kRows / 16; ++kk) {
              const uint64_t ad = smem_desc(pbase + kk * 32, 16, 1024, kSwizzle128B);
  #pragma unroll
              for (int nh = 0; nh < 2; ++nh) {
                const uint64_t bd = smem_desc(vbase + nh * 4 * (kRows * 128) + kk * 16 * 128, kRows * 128, 1024,
                                              kSwizzle128B);
                mma_ss(tmem + nh * 256, ad, bd, idesc, (j > 0 || kk > 0) ? 1u : 0u);
              }
            }
            mma_commit(&bars.vempty[st]);
            mma_commit(&bars.pcons[ps]);
            mma_commit(&bars.odone);
            if (++st == kStagesV) { st = 0; ph ^= 1; }
            if (j + 1 == n_tiles) mma_commit(&bars.alldone);
          }
          mma_commit(&bars.mdrain);
          mbar_drain(&bars.mdrain, 0);
        }
      } else if (warp == kRelayWarp && rank == 1) {
        // ----------------------------------- relay: P slot consumed -> CTA 0
        if (lane == 0) {
          n_tiles = tile_count();
          const uint32_t remote_pfree[2] = {mapa(smem_u32(&bars.pfree[0]), 0), mapa(smem_u32(&bars.pfree[1]), 0)};
          for (int j = 0; j + 2 < n_tiles; ++j) {
            const int ps = j & 1;
            if (!mbar_wait_polling<false>(&bars.pcons[ps], (j >> 1) & 1, P.err, abort_v)) break;
            mbar_arrive_expect_tx(&bars.pfull[ps], kPBytes);  // arm the slot's next use
            mbar_arrive_remote(remote_pfree[ps]);
          }
        }
      }
    }
    if (rank == 1) {
      // --------------------- epilogue (CTA 1, warpgroups 0 and 5: 8 warps)
      // Every PV product is in O (alldone) and (m, l) of each head has
      // arrived: normalise, convert to bf16 into a swizzled staging tile (the
      // free V stages) and write it with TMA stores, 64 columns x 128 heads
      // per box (heads past H are clipped by the tensor map).
      if (n_tiles < 0) n_tiles = tile_count();
      __syncwarp();
      if (ok && n_tiles > 0) ok = mbar_wait_polling<false>(&bars.alldone, 0, P.err, abort_v);
      if (ok) ok = mbar_wait_polling<true>(&bars.ffull, 0, P.err, abort_v);
      tc_fence_after();
      const int hrow = (warp & 3) * 32 + lane;
      const int half = warp < 4 ? 0 : 1;  // columns [256 half, 256 half + 256)
      const float2 ml = sFinal[hrow];
      const bool empty = !ok || (n_tiles == 0) || !(ml.y > 0.f);
      const int h = hb * 128 + hrow;
      float inv_l = empty ? 0.f : 1.f / ml.y;
      float lse2 = empty ? -__int_as_float(0x7f800000) : ml.x + log2f(ml.y);  // log2 units
      if (P.sink != nullptr && P.n_chunks == 1) {
        // The sink adds 2^s2 to the denominator; taken relative to
        // max(m, s2) so that neither term overflows.  (Split chunks get
        // it in attn_combine_kernel.)
        const float s2 = (h < P.H ? __ldg(P.sink + h) : -__int_as_float(0x7f800000)) * 1.4426950408889634f;
        if (!empty) {
          const float mx = fmaxf(ml.x, s2);
          const float den = ml.y * exp2f(ml.x - mx) + exp2f(s2 - mx);
          inv_l = exp2f(ml.x - mx) / den;
          lse2 = mx + log2f(den);
        } else {
          lse2 = s2;
        }
      }
#pragma unroll 1
      for (int c0 = half * 256; c0 < half * 256 + 256; c0 += 64) {  // one atom per round
        uint32_t v0[32], v1[32];
        tmem_ld32(tmem + lane_off + c0, v0);
        tmem_ld32(tmem + lane_off + c0 + 32, v1);
        tmem_ld_wait();
        uint32_t pk[32];
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          __nv_bfloat162 pa = __floats2bfloat162_rn(__uint_as_float(v0[2 * k]) * inv_l, __uint_as_float(v0[2 * k + 1]) * inv_l);
          __nv_bfloat162 pb = __floats2bfloat162_rn(__uint_as_float(v1[2 * k]) * inv_l, __uint_as_float(v1[2 * k + 1]) * inv_l);
          pk[k] = empty ? 0u : *reinterpret_cast<uint32_t*>(&pa);
          pk[16 + k] = empty ? 0u : *reinterpret_cast<uint32_t*>(&pb);
        }
        uint8_t* atom = sV + (c0 / 64) * kOutAtom;
#pragma unroll
        for (int k = 0; k < 8; ++k)
          *reinterpret_cast<uint4*>(atom + sw128_off(hrow, k)) =
              make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
        // the 4 warps of this half have written the atom: store it while
        // they convert the next one
        fence_proxy_async_smem();  // generic writes -> TMA store reads
        asm volatile("bar.sync %0, 128;" ::"r"(2 + half) : "memory");
        if ((warp & 3) == 0 && lane == 0) {
          const int z = P.n_chunks == 1 ? t : t * P.n_chunks + chunk;
          tma_store_3d(&tmap_o, atom, c0, hb * 128, z);
          bulk_commit_group();
        }
      }
      if ((warp & 3) == 0 && lane == 0) bulk_wait_group_read0();
      if (warp < 4 && h < P.H) {
        if (P.n_chunks == 1) {
          if (P.lse != nullptr) P.lse[static_cast<size_t>(t) * P.H + h] = lse2 * 0.69314718055994531f;
        } else {
          P.part_ml[(static_cast<size_t>(t) * P.n_chunks + chunk) * P.H + h] =
              empty ? make_float2(-__int_as_float(0x7f800000), 0.f) : make_float2(ml.x, ml.y);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no CTA leaves while its peer may still address it
  if (warp == 0) tmem_dealloc(tmem, 512);
}

// Merges the split chunks of every (token, head): out = sum_c w_c O_c /
// (sum_c w_c [+ 2^(sink - M)]) with w_c = l_c 2^(m_c - M) (O_c already
// divided by l_c); the optional attention sink is one more denominator term.
// One warp per (token, head, half of the 512 columns), 8 columns per lane.
// Chunks are taken kBatch at a time and every load of a batch (its (m, l)
// pairs and its partial rows) is issued before any of them is used, so a
// batch costs one memory round trip.  The running maximum is rescaled
// between batches like the online softmax.
constexpr int kCombineBatch = 8;

__global__ void __launch_bounds__(256) attn_combine_kernel(const AttnParams P) {
  griddep_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int item = blockIdx.x * 8 + warp;  // (token, head, column half)
  if (item >= P.T * P.H * 2) return;
  const int th = item >> 1, half = item & 1;
  const int t = th / P.H, h = th % P.H;
  const int col = half * 256 + lane * 8;  // this lane's 8 columns
  const float ninf = -__int_as_float(0x7f800000);
  float acc[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) acc[k] = 0.f;
  float M = ninf, wsum = 0.f;
  for (int c0 = 0; c0 < P.n_chunks; c0 += kCombineBatch) {
    float2 ml[kCombineBatch];
    uint4 raw[kCombineBatch];
#pragma unroll
    for (int i = 0; i < kCombineBatch; ++i) {
      const int c = c0 + i;
      const size_t row = (static_cast<size_t>(t) * P.n_chunks + c) * P.H + h;
      if (c < P.n_chunks) {
        ml[i] = __ldcg(P.part_ml + row);
        raw[i] = __ldcg(reinterpret_cast<const uint4*>(P.part_o + row * kDv + col));
      } else {
        ml[i] = make_float2(ninf, 0.f);
        raw[i] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    float Mb = M;
#pragma unroll
    for (int i = 0; i < kCombineBatch; ++i)
      if (ml[i].y > 0.f) Mb = fmaxf(Mb, ml[i].x);
    if (Mb == ninf) continue;  // nothing visible yet
    const float r = (M == ninf) ? 0.f : exp2f(M - Mb);
    wsum *= r;
#pragma unroll
    for (int k = 0; k < 8; ++k) acc[k] *= r;
    M = Mb;
#pragma unroll
    for (int i = 0; i < kCombineBatch; ++i) {
      const float wc = ml[i].y > 0.f ? ml[i].y * exp2f(ml[i].x - M) : 0.f;
      wsum += wc;
      const uint32_t wds[4] = {raw[i].x, raw[i].y, raw[i].z, raw[i].w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wds[k]));
        acc[2 * k] = fmaf(wc, f.x, acc[2 * k]);
        acc[2 * k + 1] = fmaf(wc, f.y, acc[2 * k + 1]);
      }
    }
  }
  if (P.sink != nullptr) {
    // one more term 2^s2 in the denominator (a zero-value key); -inf: none
    const float s2 = __ldg(P.sink + h) * 1.4426950408889634f;
    if (s2 != ninf) {
      if (wsum > 0.f) {
        const float mx = fmaxf(M, s2);
        const float r = exp2f(M - mx);
#pragma unroll
        for (int k = 0; k < 8; ++k) acc[k] *= r;
        wsum = wsum * r + exp2f(s2 - mx);
        M = mx;
      } else {  // nothing selected: out 0, lse = sink
        M = s2;
        wsum = 1.f;
      }
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  uint32_t pk[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    __nv_bfloat162 b2 = __floats2bfloat162_rn(acc[2 * k] * inv, acc[2 * k + 1] * inv);
    pk[k] = *reinterpret_cast<uint32_t*>(&b2);
  }
  *reinterpret_cast<uint4*>(P.out + (static_cast<size_t>(t) * P.H + h) * kDv + col) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
  if (half == 0 && lane == 0 && P.lse != nullptr)
    P.lse[static_cast<size_t>(t) * P.H + h] = wsum > 0.f ? (M + log2f(wsum)) * 0.69314718055994531f : ninf;
}

void plan(const dsa_attn_args& a, int& head_blocks, int& n_chunks, int& chunk_rows) {
  head_blocks = (a.H + 127) / 128;
  const int tiles = (a.topk + kRows - 1) / kRows;
  const long long pairs_per_chunk = static_cast<long long>(a.T) * head_blocks;
  long long target = sm_count() / (2 * pairs_per_chunk);
  if (target < 1) target = 1;
  const int tiles_per_chunk = static_cast<int>((tiles + target - 1) / target);
  chunk_rows = tiles_per_chunk * kRows;
  n_chunks = (tiles + tiles_per_chunk - 1) / tiles_per_chunk;
}

}  // namespace

size_t attn_workspace(const dsa_attn_args& a) {
  int hb, nc, cr;
  plan(a, hb, nc, cr);
  if (nc == 1) return 0;
  const size_t o = static_cast<size_t>(a.T) * nc * a.H * kDv * sizeof(__nv_bfloat16);
  const size_t ml = static_cast<size_t>(a.T) * nc * a.H * sizeof(float2);
  return round_up(o, 256) + round_up(ml, 256);
}

int launch_attn(const dsa_attn_args& a, void* ws, cudaStream_t s) {
  AttnParams P{};
  plan(a, P.head_blocks, P.n_chunks, P.chunk_rows);
  P.T = a.T; P.B = a.B; P.n_q = a.n_q; P.H = a.H; P.topk = a.topk; P.max_L = a.max_L;
  P.seq = a.seq_of_token;
  P.scale_log2 = a.scale * 1.4426950408889634f;
  P.q = reinterpret_cast<const __nv_bfloat16*>(a.q);
  P.kv = reinterpret_cast<const __nv_bfloat16*>(a.kv);
  P.block_table = a.block_table; P.block_size = a.block_size; P.max_blocks = a.max_blocks;
  P.idx = a.topk_idx;
  P.out = reinterpret_cast<__nv_bfloat16*>(a.out);
  P.lse = a.lse;
  P.sink = a.sink;
  if (P.n_chunks > 1) {
    P.part_o = static_cast<__nv_bfloat16*>(ws);
    P.part_ml = reinterpret_cast<float2*>(static_cast<uint8_t*>(ws) +
                                          round_up(static_cast<size_t>(a.T) * P.n_chunks * a.H * kDv * 2, 256));
  }
  P.err = error_word();
  if (!P.err) return DSA_ERR_CUDA;

  // output (or split-K partials): [Z, H, 512] bf16, stored as 64-column x
  // 128-head boxes; heads past H are clipped by the map.
  alignas(64) CUtensorMap tmap_o;
  {
    const uint64_t z = P.n_chunks == 1 ? static_cast<uint64_t>(a.T) : static_cast<uint64_t>(a.T) * P.n_chunks;
    const uint64_t dims[3] = {static_cast<uint64_t>(kDv), static_cast<uint64_t>(a.H), z};
    const uint64_t strides[2] = {static_cast<uint64_t>(kDv) * 2, static_cast<uint64_t>(a.H) * kDv * 2};
    const uint32_t box[3] = {64, 128, 1};
    void* base = P.n_chunks == 1 ? static_cast<void*>(P.out) : static_cast<void*>(P.part_o);
    if (!encode_tmap(&tmap_o, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, 128)) return DSA_ERR_CUDA;
  }
  const size_t smem = 1024 + static_cast<size_t>(kSmemA > kStagesV * kStageV + 2 * kPSlot + 2048
                                                    ? kSmemA
                                                    : kStagesV * kStageV + 2 * kPSlot + 2048);
  cudaError_t e = cudaFuncSetAttribute(sparse_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return DSA_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(P.n_chunks * 2, P.head_blocks, a.T);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  e = cudaLaunchKernelEx(&cfg, sparse_attn_kernel, P, tmap_o);
  if (e != cudaSuccess) return DSA_ERR_CUDA;
  if (P.n_chunks > 1) {
    cudaLaunchConfig_t c2 = {};
    c2.gridDim = dim3((a.T * a.H * 2 + 7) / 8);
    c2.blockDim = dim3(256);
    c2.dynamicSmemBytes = 0;
    c2.stream = s;
    c2.attrs = &attr[1];
    c2.numAttrs = 1;
    e = cudaLaunchKernelEx(&c2, attn_combine_kernel, P);
  }
  return cuda_status(e);
}

}  // namespace dsa

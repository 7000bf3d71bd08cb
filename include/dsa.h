/*
 * dsa.h - C ABI of the DeepSeek Sparse Attention (DSA) decode hot path on
 * GB300 (sm_103a):
 *
 *   dsa_indexer_prolog  : Indexer Prolog (q / k / weight streams)
 *   dsa_indexer_topk    : Lightning Indexer scores + per-query top-k
 *   dsa_sparse_attn     : Sparse (MLA) flash attention over the top-k rows
 *   dsa_act_quant       : standalone activation quantisation (int8, per row)
 *   dsa_int8_gemm       : standalone int8 GEMM + dequant to fp16
 *   dsa_mhc             : manifold-constrained hyper-connection mappings
 *   dsa_mla_prolog      : MLA Prolog (q_lora, absorbed query, latent KV rows)
 *
 * Page citations:
 *   [V3.2-PyPTO]  "NPU DeepSeek-V3.2-Exp PyPTO 融合算子开发优化实践",
 *                 sections Indexer Prolog, Deepseek Indexer Attention,
 *                 Lightning Indexer.
 *   [V4-TileLang] "NPU DeepSeek-V4 TileLang算子开发实践", sections Sparse
 *                 Flash Attention, Int8 General Matrix Multiplication,
 *                 Activation Quantization.
 *
 * Conventions shared by every entry point
 *   - Every pointer inside an args struct is a DEVICE pointer owned by the
 *     caller; the library never allocates or frees device memory on these
 *     paths.  Scratch memory is a caller-provided device workspace whose
 *     size the matching *_workspace() call returns.
 *   - fp16 / bf16 values are passed as their raw 16-bit patterns
 *     (uint16_t).  All arrays are dense, row-major, without padding.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Work is
 *     enqueued asynchronously; argument checks run on the host before any
 *     launch, and a rejected call enqueues nothing.
 *   - Return value: DSA_OK or an error status.  No C++ exception crosses
 *     this boundary.  A launch failure returns DSA_ERR_CUDA.  A kernel whose
 *     bounded wait expired, or that met invalid device-side data, records it
 *     in a device error word that dsa_get_device_error() reads
 *     (DSA_ERR_DEVICE_TIMEOUT, DSA_ERR_DEVICE_DATA).
 *   - T = 0 (no query tokens) is a no-op returning DSA_OK.
 *   - Kernels are launched with programmatic dependent launch: a call's
 *     kernel may start while the kernel enqueued just before it on the
 *     stream is still running, and waits for that kernel to complete before
 *     it reads anything the kernel may have written.  The exceptions are
 *     inputs that a decode step never produces in the kernel right before
 *     the call, which are read as soon as the kernel starts: the weights
 *     w_qb, w_k and w_proj of dsa_indexer_prolog, pos and seq_of_token of
 *     dsa_indexer_topk / dsa_indexer_scores, and q and seq_of_token of
 *     dsa_sparse_attn.  The
 *     kernel enqueued just before such a call must not write them (an event
 *     or a memcpy in between lifts the rule).
 */
#ifndef DSA_H_
#define DSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DSA_OK = 0,
  DSA_ERR_INVALID_ARG = 1,   /* null pointer, bad size or alignment        */
  DSA_ERR_UNSUPPORTED = 2,   /* valid but not implemented (e.g. d_I = 96)  */
  DSA_ERR_WORKSPACE = 3,     /* workspace missing or smaller than needed   */
  DSA_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed       */
  DSA_ERR_DEVICE_TIMEOUT = 5, /* a device-side bounded wait expired        */
  DSA_ERR_DEVICE_DATA = 6     /* a kernel met invalid device-side data: an
                                 out-of-range slot or position, an unmapped
                                 page, or a workspace not zero-filled; what
                                 depended on it was not written            */
} dsa_status_t;

/* Static description of a status code.  Never NULL. */
const char* dsa_status_string(int status);

/* ABI version of this header (major * 100 + minor). */
int dsa_abi_version(void);

/* Synchronises `stream`, then returns DSA_OK if no kernel of this library
 * has recorded a device-side error since the last call, else
 * DSA_ERR_DEVICE_TIMEOUT if a bounded wait expired, else
 * DSA_ERR_DEVICE_DATA; the error word is cleared.  DSA_ERR_CUDA if the
 * synchronisation itself fails. */
int dsa_get_device_error(void* stream);

/* Sets the time limit of every bounded device-side wait of this library's
 * kernels on the current device (nanoseconds; 0 restores the default of 4 s;
 * at most 60 s, else DSA_ERR_INVALID_ARG).  A wait that runs out records
 * DSA_ERR_DEVICE_TIMEOUT (see dsa_get_device_error) and its CTA leaves its
 * loops, after letting the bulk copies and tensor-core operations it issued
 * finish (each such drain bounded by 4 s).  After a timed-out call, zero the
 * call's workspace again before the next one.  Waits are timed on the
 * global timer, so a limit shorter than its tick (about 1 us) runs out at
 * the first tick; under a limit below 20 us a wait never blocks in the
 * hardware.  Synchronous: it takes effect for kernels launched after it
 * returns; call it while none of this library's kernels runs.  No
 * counterpart on the pages: a test hook. */
int dsa_set_wait_limit_ns(uint64_t ns);

/* ------------------------------------------------------------------------
 * Indexer Prolog  [V3.2-PyPTO §Indexer Prolog, the three formulas; the
 * quantisation paragraph: W8A8 q.w_qb, A8 indexer q, C8 key cache, FP16
 * dequant factors; V4-TileLang §Int8 GEMM steps 1-3 and §Activation
 * Quantization steps 1-3]
 *
 *   q, q_scale = DynamicQuant(Hadamard(RoPE(DeQuant(q_lora . w_qb))))
 *   k, k_scale = DynamicQuant(Hadamard(RoPE(LayerNorm(x . w_k))))
 *   w          = (x . w_proj) * w_scale                (optional)
 *
 * DeQuant: acc[t,n] = sum_c q_lora[t,c] * w_qb[n,c] (exact int32), times
 * q_lora_scale[t] * w_qb_scale[n] in fp32.  RoPE rotates dims [0, d_rope)
 * of each d_I-dim head by the fp32 tables rope_cos/rope_sin
 * [rope_max_pos, d_rope/2] at row pos[t]; pairs are (i, i + d_rope/2), or
 * (2i, 2i+1) if rope_interleaved.  Hadamard is the Sylvester transform of
 * order d_I scaled by d_I^-1/2.  DynamicQuant per (token, head) row:
 * scale = fp16(absmax / 127) (the division in fp32), code =
 * round_half_even(clamp(x / scale, -127, 127)), code 0 when scale is 0.
 * LayerNorm: biased variance, eps inside the square root, fp32 gamma/beta.
 *
 * Shapes: q_lora int8 [T, K_q]; q_lora_scale fp16 [T]; w_qb int8
 * [H_I*d_I, K_q] (K-major: row n is output channel n); w_qb_scale fp16
 * [H_I*d_I]; x bf16 [T, D_x]; w_k bf16 [d_I, D_x]; w_proj bf16 [H_I, D_x]
 * or NULL; pos int32 [T] (each in [0, rope_max_pos): a position outside
 * it is recorded as DSA_ERR_DEVICE_DATA and that token's q, q_scale and key
 * rows are not written; its w row is); q_out int8
 * [T, H_I, d_I]; q_scale_out fp16 [T, H_I]; k_cache int8 [cache_rows, d_I];
 * k_scale_cache fp16 [cache_rows]; slot int64 [T]: row of k_cache that
 * receives token t's key, -1 = none (slots must not repeat; a slot >=
 * cache_rows is recorded as DSA_ERR_DEVICE_DATA and that key row is not
 * written); w_out fp32 [T, H_I] (required iff w_proj != NULL).
 * Supported: 1 <= T <= 32, d_I in {64, 128}, 1 <= H_I <= 128, d_rope even
 * with d_rope <= d_I and (d_rope/2) a multiple of d_I/32, K_q <= 2048 and
 * D_x <= 12288, both multiples of 64; x, w_k and w_proj 16-byte aligned.
 * Workspace: dsa_indexer_prolog_workspace() bytes; it must be zero-filled
 * once before its first use (each call leaves it zeroed; after a call that
 * ended in DSA_ERR_DEVICE_TIMEOUT, zero it again).
 * ---------------------------------------------------------------------- */
typedef struct {
  int32_t T, H_I, d_I, d_rope, K_q, D_x;
  const int8_t* q_lora;
  const uint16_t* q_lora_scale;
  const int8_t* w_qb;
  const uint16_t* w_qb_scale;
  const uint16_t* x;
  const uint16_t* w_k;
  const float* ln_gamma;
  const float* ln_beta;
  float ln_eps;
  const uint16_t* w_proj;
  float w_scale;
  const int32_t* pos;
  const float* rope_cos;
  const float* rope_sin;
  int32_t rope_max_pos;
  int32_t rope_interleaved;
  int8_t* q_out;
  uint16_t* q_scale_out;
  int8_t* k_cache;
  uint16_t* k_scale_cache;
  const int64_t* slot;
  int64_t cache_rows;
  float* w_out;
} dsa_prolog_args;

size_t dsa_indexer_prolog_workspace(const dsa_prolog_args* args);
int dsa_indexer_prolog(const dsa_prolog_args* args, void* workspace, size_t workspace_bytes, void* stream);

/* dsa_indexer_prolog_noalloc: the Indexer Prolog for callers that cannot
 * allocate device memory.  The pages have no counterpart: this is an
 * interface convenience of this library, not part of the method.
 *
 * Some callers are handed only their input and output tensors and have no
 * device allocator (a plug-in inside a host framework that owns all device
 * memory), or run a loop that must never call cudaMalloc because it can
 * synchronise the device.  This entry point takes the same arguments and
 * gives the same results as dsa_indexer_prolog but needs no workspace: its
 * scratch is one 64 KiB array compiled into the library, held on every GPU
 * that loads the library until the process exits.  It allocates nothing.
 *
 *   - Requests whose workspace would exceed 64 KiB are rejected with
 *     DSA_ERR_WORKSPACE before anything is enqueued (every supported prolog
 *     shape, T <= 32 and d_I + H_I <= 256 channels, fits).
 *   - The first call on a device, with that device current, looks up the
 *     array's device address (cudaGetSymbolAddress) and caches it with the
 *     current context; make that first call before any stream capture.  A
 *     call made under another context (after cudaDeviceReset, or with a
 *     context the caller created) looks the address up again.
 *   - Every call shares the one array and clears the part that must start at
 *     zero itself; calls that may overlap on the GPU (other streams, other
 *     threads) race on it and must be serialised by the caller. */
int dsa_indexer_prolog_noalloc(const dsa_prolog_args* args, void* stream);

/* ------------------------------------------------------------------------
 * Lightning Indexer + top-k  [V3.2-PyPTO §Lightning Indexer: the int8 q
 * scored against the C8 key cache, then a per-query TopK; V4-TileLang
 * §Sparse Flash Attention step 2 for the -1 marker of unused slots]
 *
 *   I[t,s] = ks[s] * sum_h (w[t,h] * qs[t,h]) * ReLU(sum_d q[t,h,d] K[s,d])
 *
 * for keys 0 <= s <= pos[t] of token t's sequence; topk_idx[t] receives the
 * positions of the `topk` largest I[t,.] (as a set, in no particular order),
 * followed by -1 when fewer than `topk` keys are visible.  Equal scores at
 * the boundary are broken arbitrarily.
 *
 * Token layout: seq_of_token int32 [T] names each token's sequence (in
 * [0, B)); the tokens of one sequence must be adjacent in the token order
 * (the indexer scores up to G = min(128 / H_I, 32) adjacent tokens of a
 * sequence against each key tile together).  seq_of_token == NULL is the
 * uniform batch: T = B * n_q, token t in sequence t / n_q.  An id outside
 * [0, B), or a sequence whose tokens are split, is recorded as
 * DSA_ERR_DEVICE_DATA (that token's outputs are then unspecified).  With a
 * map, n_q is ignored and T <= 65535.
 * Shapes: q int8 [T, H_I, d_I]; q_scale fp16 [T, H_I]; w fp32 [T, H_I];
 * pos int32 [T] with 0 <= pos[t] < max_L; topk_idx int32 [T, topk];
 * scores_out fp32 [T, max_L] or NULL (when given it receives I, with -inf
 * for s > pos[t]; columns past the largest visible key are unspecified).
 * Key cache, contiguous (block_table == NULL): k_cache int8 [B, max_L, d_I],
 * k_scale fp16 [B, max_L].  Paged: k_cache int8 [n_rows, d_I], k_scale fp16
 * [n_rows], key s of sequence b at row block_table[b, s / block_size] *
 * block_size + s % block_size, block_table int32 [B, max_blocks],
 * max_L = max_blocks * block_size.  k_cache and k_scale are 16-byte
 * aligned (each tile's scales are copied with its keys in bulk).  Every
 * block_table entry that a visible key reaches must name a page of the
 * cache (0 <= id and (id + 1) * block_size <= n_rows): n_rows is not an
 * argument, so the upper bound is the caller's to keep.  A negative entry
 * is recorded as DSA_ERR_DEVICE_DATA (row 0 is read in its place; the
 * scores of that page are unspecified).
 * Supported: d_I in {64, 128}; H_I in {4, 8, 16, 32, 64, 128}; topk >= 1;
 * a token-group table that fits shared memory (B * ceil(n_q / G) <= 4096
 * groups for a uniform batch, G = min(n_q, 128 / H_I, 32); about
 * ceil(T / G) + B <= 4096 with a map; else DSA_ERR_UNSUPPORTED);
 * max_L a multiple of 128; block_size a multiple of 8 that divides 128 or
 * is a multiple of 128.  Workspace: dsa_indexer_topk_workspace() bytes (the
 * fp32 score rows live there when scores_out is NULL, and, for H_I >= 64
 * with at most 512 tokens and max_L <= 131072, per-token score histograms);
 * it must be zero-filled once before its first use (the library leaves it
 * zeroed; after a call that ended in DSA_ERR_DEVICE_TIMEOUT, zero it again).
 * ---------------------------------------------------------------------- */
typedef struct {
  int32_t T, B, n_q, H_I, d_I, topk, max_L;
  const int8_t* q;
  const uint16_t* q_scale;
  const float* w;
  const int8_t* k_cache;
  const uint16_t* k_scale;
  const int32_t* block_table;
  int32_t block_size, max_blocks;
  const int32_t* pos;
  int32_t* topk_idx;
  float* scores_out;
  const int32_t* seq_of_token;
} dsa_topk_args;

size_t dsa_indexer_topk_workspace(const dsa_topk_args* args);
int dsa_indexer_topk(const dsa_topk_args* args, void* workspace, size_t workspace_bytes, void* stream);

/* The two halves of dsa_indexer_topk as separate calls, for pipelines that
 * keep the score rows.  dsa_indexer_scores writes I into `scores` fp32
 * [T, max_L] (device; -inf for s > pos[t]; columns past the largest visible
 * key of a token's group are not written); args->topk_idx and
 * args->scores_out are ignored.  dsa_topk_from_scores selects, per token,
 * the args->topk largest of scores[t, 0..pos[t]] (rows `ld` floats apart,
 * ld >= max_L) into args->topk_idx, with the same output rules as above. */
int dsa_indexer_scores(const dsa_topk_args* args, float* scores, void* stream);
int dsa_topk_from_scores(const dsa_topk_args* args, const float* scores, int64_t ld, void* stream);

/* Exact int32 dot products dots[t, h, s] = sum_d q[t,h,d] K[b(t),s,d] for
 * s in [0, max_L), for checking the integer contraction bit by bit (test
 * use; a plain SIMT kernel, not the production path).  dots int32
 * [T, H_I, max_L]. */
int dsa_indexer_dots_debug(const dsa_topk_args* args, int32_t* dots, void* stream);

/* ------------------------------------------------------------------------
 * Sparse MLA attention  [V4-TileLang §Sparse Flash Attention steps 1-6 and
 * 8; V3.2-PyPTO §Deepseek Indexer Attention: the TopK rows are gathered
 * from the latent cache straight into on-chip memory]
 *
 *   out[t,h,:] = sum_j softmax_j(scale * q[t,h,:] . KV[r_j, :]) KV[r_j, :d_v]
 *
 * over the rows r_j of token t's sequence named by topk_idx[t, j] >= 0
 * (logical positions; -1 selects nothing).  lse[t,h] = natural log of
 * sum_j exp(scale * q . k_j); a token with no selected row gets out = 0 and
 * lse = -inf.
 *
 * sink: fp32 [H] or NULL.  The attention sink of step 7 (the page prints
 * its operator garbled), read as one more term exp(sink[h]) in head h's
 * softmax denominator - a key with logit sink[h] (natural-log units, like
 * scale * q . k) and a zero value:
 *   out[t,h,:] = sum_j e^{s_j} KV[r_j, :d_v] / (sum_j e^{s_j} + e^{sink[h]})
 *   lse[t,h]   = log(sum_j e^{s_j} + e^{sink[h]})
 * so a token with no selected row gets out = 0 and lse = sink[h].  Entries
 * are finite or -inf (-inf = no sink for that head).
 *
 * Token layout: seq_of_token int32 [T] (each in [0, B); any order) or NULL
 * for the uniform batch T = B * n_q, token t in sequence t / n_q.  A token
 * whose id lies outside [0, B) is recorded as DSA_ERR_DEVICE_DATA and gets
 * out = 0 (no row read).
 * Shapes: q bf16 [T, H, d_qk]; kv bf16 contiguous [B, max_L, d_qk] or paged
 * [n_rows, d_qk] through block_table int32 [B, max_blocks] as above;
 * topk_idx int32 [T, topk] with entries in [-1, max_L); out bf16
 * [T, H, d_v]; lse fp32 [T, H] or NULL.  A selected index must lie in a
 * page of the cache (as for dsa_indexer_topk, the upper bound is not
 * checked); one whose block_table entry is negative reads a zero row (a
 * logit of 0 with a zero value) and is not reported.
 * Supported: d_qk = 576, d_v = 512, 1 <= H <= 128, 1 <= topk <= 65536.
 * Workspace: dsa_sparse_attn_workspace() bytes.
 * ---------------------------------------------------------------------- */
typedef struct {
  int32_t T, B, n_q, H, d_qk, d_v, topk, max_L;
  float scale;
  const uint16_t* q;
  const uint16_t* kv;
  const int32_t* block_table;
  int32_t block_size, max_blocks;
  const int32_t* topk_idx;
  uint16_t* out;
  float* lse;
  const float* sink;
  const int32_t* seq_of_token;
} dsa_attn_args;

size_t dsa_sparse_attn_workspace(const dsa_attn_args* args);
int dsa_sparse_attn(const dsa_attn_args* args, void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * Activation Quantization  [V4-TileLang §Activation Quantization, steps
 * 1-4] - a standalone export of the quantiser (the prolog fuses its own).
 *
 *   scale[m] = max_n |x[m,n]| / 127           (fp32; round_scale != 0: the
 *                                               power of two at or above it)
 *   y[m,n]   = rint(clamp(x[m,n] / scale[m], -127, 127))   (int8)
 *
 * One scale per row of N values; the quotient is an fp32 division and ties
 * round to even; a row of zeros gets scale 0 and codes 0.
 * Shapes: x bf16 [M, N] (16-byte aligned); y int8 [M, N] (8-byte aligned);
 * scale fp32 [M].  Supported: 8 <= N <= 32768, N a multiple of 8.  No
 * workspace.  M = 0 is a no-op.
 * ---------------------------------------------------------------------- */
typedef struct {
  int32_t M, N;
  const uint16_t* x;
  int8_t* y;
  float* scale;
  int32_t round_scale;
} dsa_act_quant_args;

int dsa_act_quant(const dsa_act_quant_args* args, void* stream);

/* ------------------------------------------------------------------------
 * Int8 GEMM  [V4-TileLang §Int8 General Matrix Multiplication, steps 1-4]
 * - a standalone export.
 *
 *   c[m,n] = fp16( (sum_k a[m,k] * b[n,k]) * a_scale[m] * b_scale[n] )
 *
 * The int32 sum is exact; the dequantisation is fp32 (the product in the
 * order written), rounded once to fp16.  Both paths run on the tensor
 * cores (int8 converted exactly to f16, fp32 sums of at most 1024
 * products, added in int32) and give bit-identical results: up to 32 rows
 * (decode tokens) a weight stream with b's rows as the MMA's M dimension
 * and one CTA per SM over a contiguous range of them; more rows, tiles of
 * 128 x 128.
 * Shapes: a int8 [M, K]; b int8 [N, K] (K-major, row n = output column n);
 * a_scale fp32 [M]; b_scale fp32 [N]; c fp16 [M, N].  a and b 16-byte
 * aligned.  Supported: 1 <= M <= 8388608, N >= 1, K a multiple of 16 up to
 * 65536.  No workspace.  M = 0 or N = 0 is a no-op.
 * ---------------------------------------------------------------------- */
typedef struct {
  int32_t M, N, K;
  const int8_t* a;
  const float* a_scale;
  const int8_t* b;
  const float* b_scale;
  uint16_t* c;
} dsa_int8_gemm_args;

int dsa_int8_gemm(const dsa_int8_gemm_args* args, void* stream);

/* ------------------------------------------------------------------------
 * Manifold-Constrained Hyper-Connections  [V4-TileLang §Manifold-
 * Constrained Hyper-Connections, steps 1-5] - per token, hc streams:
 *
 *   z    = mixes * hc_scale[part] + hc_base      (parts: pre, post, comb)
 *   pre  = sigmoid(z_pre) + eps                  [n, hc]
 *   post = 2 sigmoid(z_post)                     [n, hc]
 *   comb = softmax_rows(z_comb) + eps, then / (column sums + eps), then
 *          `iters` times / (row sums + eps) and / (column sums + eps)
 *                                                [n, hc, hc]
 *
 * A row of mixes (fp32 [n, hc (2 + hc)]) holds z_pre (hc), z_post (hc) and
 * z_comb (hc x hc, row-major); hc_scale fp32 [3]; hc_base fp32
 * [hc (2 + hc)].  All fp32; mixes, pre, post and comb 16-byte aligned,
 * hc_scale and hc_base 4-byte aligned (else DSA_ERR_INVALID_ARG).
 * Supported: hc in {4, 8}, 0 <= iters <= 100.  n = 0 is a no-op.  No
 * workspace.
 * ---------------------------------------------------------------------- */
typedef struct {
  int32_t n, hc, iters;
  float eps;
  const float* mixes;
  const float* hc_scale;
  const float* hc_base;
  float* pre;
  float* post;
  float* comb;
} dsa_mhc_args;

int dsa_mhc(const dsa_mhc_args* args, void* stream);

/* ------------------------------------------------------------------------
 * MLA Prolog  [V3.2-PyPTO §Deepseek Indexer Attention: the first of its four
 * parts, feeding q_lora to the Indexer Prolog and q plus the latent KV rows
 * to the sparse attention; the pages give it no formula, so the operation
 * below is a reading of it]
 *
 *   c_q          = RMSNorm(x . w_dq^T) * gamma_q                 [T, K_q]
 *   q_lora, q_lora_scale = DynamicQuant(c_q)  (per token, as the Indexer
 *                  Prolog's quantiser: scale = fp16(absmax / 127), codes
 *                  round_half_even(clamp(c / scale, -127, 127)))
 *   u            = DeQuant(q_lora . w_uq^T)                    [T, H, 192]
 *                  (exact int32 sums times q_lora_scale[t] * w_uq_scale[n]
 *                  in fp32; per head 128 no-position dims, then 64 rotary)
 *   q[t, h]      = bf16([u[t,h,:128] . w_uk[h] | RoPE(u[t,h,128:])])
 *                                                              [T, H, 576]
 *   c            = x . w_dkv^T                                  [T, 576]
 *   kv_cache[slot[t]] = bf16([RMSNorm(c[:512]) * gamma_kv | RoPE(c[512:])])
 *
 * RMSNorm: x / sqrt(mean(x^2) + rms_eps).  RoPE rotates the 64 rotary dims
 * with the fp32 tables rope_cos / rope_sin [rope_max_pos, 32] at row pos[t];
 * pairs (i, i + 32), or (2i, 2i+1) if rope_interleaved.
 *
 * Shapes: x bf16 [T, D_x]; w_dq bf16 [K_q, D_x] (row n = output channel n);
 * gamma_q fp32 [K_q]; w_dkv bf16 [576, D_x] (512 latent rows, then 64
 * rotary rows); gamma_kv fp32 [512]; w_uq int8 [H*192, K_q]; w_uq_scale fp16
 * [H*192]; w_uk bf16 [H, 128, 512]; pos int32 [T]; q_lora int8 [T, K_q];
 * q_lora_scale fp16 [T]; q bf16 [T, H, 576]; kv_cache bf16
 * [cache_rows, 576]; slot int64 [T] (-1 = not written; slots must not
 * repeat).  A slot >= cache_rows or a pos outside [0, rope_max_pos) is
 * recorded in the device error word and that token's latent row is not
 * written.
 * Supported: 1 <= T <= 32, 1 <= H <= 128, K_q a multiple of 128 in
 * [128, 2048], D_x a multiple of 64 in [64, 16384], rms_eps >= 0.
 * x, w_dq, gamma_q, w_dkv, gamma_kv, w_uq, w_uk, q_lora, q and kv_cache
 * 16-byte aligned.
 * Workspace: dsa_mla_prolog_workspace() bytes, 256-byte aligned; it must
 * be zero-filled once before its first use (each call leaves its sums
 * zeroed; after a call that ended in DSA_ERR_DEVICE_TIMEOUT, zero it again).
 * ---------------------------------------------------------------------- */
typedef struct {
  int32_t T, H, K_q, D_x;
  float rms_eps;
  int32_t rope_max_pos;
  int32_t rope_interleaved;
  const uint16_t* x;
  const uint16_t* w_dq;
  const float* gamma_q;
  const uint16_t* w_dkv;
  const float* gamma_kv;
  const int8_t* w_uq;
  const uint16_t* w_uq_scale;
  const uint16_t* w_uk;
  const int32_t* pos;
  const float* rope_cos;
  const float* rope_sin;
  int8_t* q_lora;
  uint16_t* q_lora_scale;
  uint16_t* q;
  uint16_t* kv_cache;
  const int64_t* slot;
  int64_t cache_rows;
} dsa_mla_prolog_args;

size_t dsa_mla_prolog_workspace(const dsa_mla_prolog_args* args);
int dsa_mla_prolog(const dsa_mla_prolog_args* args, void* workspace, size_t workspace_bytes, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* DSA_H_ */

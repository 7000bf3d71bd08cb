// The C ABI: argument validation, workspace sizing, device error word.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <mutex>
#include "dsa_internal.h"
#include "dsa_ptx.cuh"

namespace dsa {

// Per device: the error word kernels OR their error bits into, and the time
// limit of their bounded waits (read through the same pointer, see
// wait_limit_ns() in dsa_ptx.cuh).
struct DeviceControl {
  uint32_t error_word;
  uint32_t reserved;
  uint64_t wait_limit_ns;
};
static_assert(offsetof(DeviceControl, wait_limit_ns) == kWaitLimitOffset, "wait limit offset");
static __device__ __align__(16) DeviceControl g_ctl = {0u, 0u, DSA_WAIT_NS};

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_mu;
// Device address of g_ctl per device, with the context it was
// resolved in: a different current context (a reset device, a context the
// caller created) resolves it again.
void* g_err_ctx[kMaxDevices] = {};
uint32_t* g_err_ptr[kMaxDevices] = {};
int g_sms[kMaxDevices] = {};

int current_device() {
  int d = -1;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) return -1;
  return d;
}
}  // namespace

void* current_context() {
  static PFN_cuCtxGetCurrent_v4000 fn = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!fn) {
      cudaDriverEntryPointQueryResult q;
      void* p = nullptr;
      if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) != cudaSuccess ||
          q != cudaDriverEntryPointSuccess || !p)
        return nullptr;
      fn = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    }
  }
  CUcontext c = nullptr;
  if (fn(&c) != CUDA_SUCCESS) return nullptr;
  return c;
}

uint32_t* error_word() {
  const int d = current_device();
  if (d < 0) return nullptr;
  // cudaGetDevice made the device's primary context current if none was.
  void* ctx = current_context();
  if (!ctx) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_err_ptr[d] || g_err_ctx[d] != ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_ctl) != cudaSuccess) return nullptr;
    g_err_ptr[d] = static_cast<uint32_t*>(p);
    g_err_ctx[d] = ctx;
  }
  return g_err_ptr[d];
}

int sm_count() {
  const int d = current_device();
  if (d < 0) return 1;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_sms[d]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d) != cudaSuccess || n <= 0) n = 1;
    g_sms[d] = n;
  }
  return g_sms[d];
}

bool encode_tmap(void* out, int dtype, int rank, const void* base, const uint64_t* dims, const uint64_t* strides,
                 const uint32_t* box, int swizzle_bytes) {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!fn) {
      cudaDriverEntryPointQueryResult q;
      void* p = nullptr;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
              cudaSuccess ||
          q != cudaDriverEntryPointSuccess || !p)
        return false;
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
  }
  if (rank < 1 || rank > 5) return false;
  cuuint64_t d[5], st[4];
  cuuint32_t bx[5], es[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
    if (i + 1 < rank) st[i] = strides[i];
  }
  const CUtensorMapSwizzle sw = swizzle_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                               : swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                     : CU_TENSOR_MAP_SWIZZLE_NONE;
  const CUresult r = fn(static_cast<CUtensorMap*>(out), static_cast<CUtensorMapDataType>(dtype),
                        static_cast<cuuint32_t>(rank), const_cast<void*>(base), d, st, bx, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool encode_tmap_u8_2d(void* out, const void* base, uint64_t inner, uint64_t rows, uint64_t row_stride,
                       uint32_t box_rows, int swizzle_bytes) {
  const uint64_t dims[2] = {inner, rows};
  const uint64_t strides[1] = {row_stride};
  const uint32_t box[2] = {static_cast<uint32_t>(inner), box_rows};
  return encode_tmap(out, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, dims, strides, box, swizzle_bytes);
}

}  // namespace dsa

using namespace dsa;

namespace {

bool bad_ptr(const void* p, size_t align) { return p == nullptr || !aligned(p, align); }

int check_prolog(const dsa_prolog_args* a) {
  if (!a) return DSA_ERR_INVALID_ARG;
  if (a->T < 0 || a->T > 32) return a->T < 0 ? DSA_ERR_INVALID_ARG : DSA_ERR_UNSUPPORTED;
  if (a->d_I != 64 && a->d_I != 128) return DSA_ERR_UNSUPPORTED;
  if (a->H_I < 1 || a->H_I > 128) return DSA_ERR_UNSUPPORTED;
  if (a->d_rope < 0 || a->d_rope > a->d_I || (a->d_rope % 2) != 0 || ((a->d_rope / 2) % (a->d_I / 32)) != 0)
    return DSA_ERR_UNSUPPORTED;
  if (a->K_q <= 0 || a->K_q % 64 != 0 || a->K_q > 2048) return DSA_ERR_UNSUPPORTED;
  if (a->D_x <= 0 || a->D_x % 64 != 0 || a->D_x > 12288) return DSA_ERR_UNSUPPORTED;
  if (a->rope_max_pos <= 0 || a->cache_rows < 0 || !(a->ln_eps >= 0.f)) return DSA_ERR_INVALID_ARG;
  if (a->T == 0) return DSA_OK;
  const size_t code_align = a->d_I == 128 ? 4 : 2;
  if (bad_ptr(a->q_lora, 16) || bad_ptr(a->q_lora_scale, 2) || bad_ptr(a->w_qb, 16) ||
      bad_ptr(a->w_qb_scale, 2) || bad_ptr(a->x, 16) || bad_ptr(a->w_k, 16) || bad_ptr(a->ln_gamma, 4) ||
      bad_ptr(a->ln_beta, 4) || bad_ptr(a->pos, 4) || bad_ptr(a->rope_cos, 4) || bad_ptr(a->rope_sin, 4) ||
      bad_ptr(a->q_out, code_align) || bad_ptr(a->q_scale_out, 2) || bad_ptr(a->k_cache, code_align) ||
      bad_ptr(a->k_scale_cache, 2) || bad_ptr(a->slot, 8))
    return DSA_ERR_INVALID_ARG;
  if ((a->w_proj == nullptr) != (a->w_out == nullptr)) return DSA_ERR_INVALID_ARG;
  if (a->w_proj && (bad_ptr(a->w_proj, 16) || bad_ptr(a->w_out, 4))) return DSA_ERR_INVALID_ARG;
  return DSA_OK;
}

// The token layout: a map (any T, B >= 1) or the uniform batch T = B * n_q.
int check_tokens(int T, int B, int n_q, const int32_t* seq) {
  if (T < 0) return DSA_ERR_INVALID_ARG;
  if (seq != nullptr) {
    if (B < 1 || !aligned(seq, 4)) return T == 0 ? DSA_OK : DSA_ERR_INVALID_ARG;
    return T > 65535 ? DSA_ERR_UNSUPPORTED : DSA_OK;
  }
  if (B < 1 || n_q < 1 || static_cast<long long>(B) * n_q != T) return T == 0 ? DSA_OK : DSA_ERR_INVALID_ARG;
  return DSA_OK;
}

int check_topk(const dsa_topk_args* a) {
  if (!a) return DSA_ERR_INVALID_ARG;
  {
    const int st = check_tokens(a->T, a->B, a->n_q, a->seq_of_token);
    if (st != DSA_OK || a->T == 0) return st;
  }
  if (a->d_I != 64 && a->d_I != 128) return DSA_ERR_UNSUPPORTED;
  switch (a->H_I) {
    case 4: case 8: case 16: case 32: case 64: case 128: break;
    default: return DSA_ERR_UNSUPPORTED;
  }
  if (a->topk < 1) return DSA_ERR_INVALID_ARG;
  if (a->max_L < 128 || a->max_L % 128 != 0) return DSA_ERR_UNSUPPORTED;
  if (bad_ptr(a->q, 16) || bad_ptr(a->q_scale, 2) || bad_ptr(a->w, 4) || bad_ptr(a->k_cache, 16) ||
      bad_ptr(a->k_scale, 16) || bad_ptr(a->pos, 4) || bad_ptr(a->topk_idx, 4))
    return DSA_ERR_INVALID_ARG;
  if (a->scores_out && !aligned(a->scores_out, 16)) return DSA_ERR_INVALID_ARG;
  if (a->block_table) {
    if (!aligned(a->block_table, 4) || a->block_size < 8 || a->block_size % 8 != 0) return DSA_ERR_INVALID_ARG;
    if (!(128 % a->block_size == 0 || a->block_size % 128 == 0)) return DSA_ERR_UNSUPPORTED;
    if (static_cast<long long>(a->max_blocks) * a->block_size != a->max_L) return DSA_ERR_INVALID_ARG;
  }
  return DSA_OK;
}

int check_attn(const dsa_attn_args* a) {
  if (!a) return DSA_ERR_INVALID_ARG;
  {
    const int st = check_tokens(a->T, a->B, a->n_q, a->seq_of_token);
    if (st != DSA_OK || a->T == 0) return st;
  }
  if (a->d_qk != 576 || a->d_v != 512) return DSA_ERR_UNSUPPORTED;
  if (a->H < 1 || a->topk < 1 || a->topk > 65536 || a->max_L < 1) return DSA_ERR_INVALID_ARG;
  if (!(a->scale > 0.f)) return DSA_ERR_INVALID_ARG;
  if (bad_ptr(a->q, 16) || bad_ptr(a->kv, 16) || bad_ptr(a->topk_idx, 4) || bad_ptr(a->out, 16))
    return DSA_ERR_INVALID_ARG;
  if (a->lse && !aligned(a->lse, 4)) return DSA_ERR_INVALID_ARG;
  if (a->sink && !aligned(a->sink, 4)) return DSA_ERR_INVALID_ARG;
  if (a->block_table) {
    if (!aligned(a->block_table, 4) || a->block_size < 1) return DSA_ERR_INVALID_ARG;
    if (static_cast<long long>(a->max_blocks) * a->block_size != a->max_L) return DSA_ERR_INVALID_ARG;
  }
  return DSA_OK;
}

size_t topk_scores_bytes(const dsa_topk_args* a) {
  return a->scores_out ? 0 : round_up(static_cast<size_t>(a->T) * a->max_L * sizeof(float), 256);
}

// Workspace of dsa_indexer_topk: score rows (unless scores_out is given),
// then, on the fused path, the per-token score histograms.
size_t topk_total_bytes(const dsa_topk_args* a) {
  return topk_scores_bytes(a) + (topk_hist_eligible(*a) ? topk_hist_workspace(*a) : 0);
}

}  // namespace

extern "C" {

const char* dsa_status_string(int status) {
  switch (status) {
    case DSA_OK: return "ok";
    case DSA_ERR_INVALID_ARG: return "invalid argument";
    case DSA_ERR_UNSUPPORTED: return "unsupported shape or option";
    case DSA_ERR_WORKSPACE: return "workspace missing or too small";
    case DSA_ERR_CUDA: return "CUDA error";
    case DSA_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
    case DSA_ERR_DEVICE_DATA: return "invalid device-side data (index, page or unzeroed workspace)";
    default: return "unknown status";
  }
}

int dsa_abi_version(void) { return 104; }

int dsa_set_wait_limit_ns(uint64_t ns) {
  if (ns > 60000000000ull) return DSA_ERR_INVALID_ARG;
  const uint64_t v = ns == 0 ? DSA_WAIT_NS : ns;
  if (!error_word()) return DSA_ERR_CUDA;
  return cudaMemcpyToSymbol(g_ctl, &v, sizeof(v), offsetof(DeviceControl, wait_limit_ns)) == cudaSuccess
             ? DSA_OK
             : DSA_ERR_CUDA;
}

int dsa_get_device_error(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return DSA_ERR_CUDA;
  uint32_t* p = error_word();
  if (!p) return DSA_ERR_CUDA;
  uint32_t v = 0;
  if (cudaMemcpy(&v, p, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return DSA_ERR_CUDA;
  if (v == 0) return DSA_OK;
  const uint32_t zero = 0;
  if (cudaMemcpy(p, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return DSA_ERR_CUDA;
  return (v & kErrTimeout) ? DSA_ERR_DEVICE_TIMEOUT : DSA_ERR_DEVICE_DATA;
}

size_t dsa_indexer_prolog_workspace(const dsa_prolog_args* a) {
  if (check_prolog(a) != DSA_OK) return 0;
  return prolog_workspace(*a);
}

int dsa_indexer_prolog(const dsa_prolog_args* a, void* ws, size_t ws_bytes, void* stream) {
  const int st = check_prolog(a);
  if (st != DSA_OK || a->T == 0) return st;
  if (ws == nullptr || !aligned(ws, 256) || ws_bytes < prolog_workspace(*a)) return DSA_ERR_WORKSPACE;
  return launch_prolog(*a, ws, static_cast<cudaStream_t>(stream));
}

size_t dsa_indexer_topk_workspace(const dsa_topk_args* a) {
  if (check_topk(a) != DSA_OK) return 0;
  return topk_total_bytes(a);
}

int dsa_indexer_topk(const dsa_topk_args* a, void* ws, size_t ws_bytes, void* stream) {
  const int st = check_topk(a);
  if (st != DSA_OK || a->T == 0) return st;
  const size_t need = topk_total_bytes(a);
  if (need > 0 && (ws == nullptr || !aligned(ws, 256) || ws_bytes < need)) return DSA_ERR_WORKSPACE;
  float* scores = a->scores_out ? a->scores_out : static_cast<float*>(ws);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (topk_hist_eligible(*a)) {
    void* hws = static_cast<uint8_t*>(ws) + topk_scores_bytes(a);
    int r = launch_indexer(*a, scores, static_cast<uint32_t*>(hws), s);
    if (r != DSA_OK) return r;
    return launch_topk_hist(*a, scores, a->max_L, hws, s);
  }
  int r = launch_indexer(*a, scores, nullptr, s);
  if (r != DSA_OK) return r;
  return launch_topk(*a, scores, a->max_L, s);
}

int dsa_indexer_scores(const dsa_topk_args* a, float* scores, void* stream) {
  const int st = check_topk(a);
  if (st != DSA_OK || a->T == 0) return st;
  if (bad_ptr(scores, 16)) return DSA_ERR_INVALID_ARG;
  return launch_indexer(*a, scores, nullptr, static_cast<cudaStream_t>(stream));
}

int dsa_topk_from_scores(const dsa_topk_args* a, const float* scores, int64_t ld, void* stream) {
  const int st = check_topk(a);
  if (st != DSA_OK || a->T == 0) return st;
  if (bad_ptr(scores, 4) || ld < a->max_L) return DSA_ERR_INVALID_ARG;
  return launch_topk(*a, scores, ld, static_cast<cudaStream_t>(stream));
}

int dsa_indexer_dots_debug(const dsa_topk_args* a, int32_t* dots, void* stream) {
  const int st = check_topk(a);
  if (st != DSA_OK || a->T == 0) return st;
  if (bad_ptr(dots, 4)) return DSA_ERR_INVALID_ARG;
  return launch_indexer_dots(*a, dots, static_cast<cudaStream_t>(stream));
}

size_t dsa_sparse_attn_workspace(const dsa_attn_args* a) {
  if (check_attn(a) != DSA_OK || a->T == 0) return 0;
  return attn_workspace(*a);
}

int dsa_sparse_attn(const dsa_attn_args* a, void* ws, size_t ws_bytes, void* stream) {
  const int st = check_attn(a);
  if (st != DSA_OK || a->T == 0) return st;
  const size_t need = attn_workspace(*a);
  if (need > 0 && (ws == nullptr || !aligned(ws, 256) || ws_bytes < need)) return DSA_ERR_WORKSPACE;
  return launch_attn(*a, ws, static_cast<cudaStream_t>(stream));
}

int dsa_act_quant(const dsa_act_quant_args* a, void* stream) {
  if (!a || a->M < 0) return DSA_ERR_INVALID_ARG;
  if (a->N < 8 || a->N % 8 != 0 || a->N > 32768) return DSA_ERR_UNSUPPORTED;
  if (a->M == 0) return DSA_OK;
  if (bad_ptr(a->x, 16) || bad_ptr(a->y, 8) || bad_ptr(a->scale, 4)) return DSA_ERR_INVALID_ARG;
  return launch_act_quant(*a, static_cast<cudaStream_t>(stream));
}

int dsa_int8_gemm(const dsa_int8_gemm_args* a, void* stream) {
  if (!a || a->M < 0 || a->N < 0 || a->K < 0) return DSA_ERR_INVALID_ARG;
  if (a->K < 16 || a->K % 16 != 0 || a->K > 65536 || a->M > 8388608) return DSA_ERR_UNSUPPORTED;
  if (a->M == 0 || a->N == 0) return DSA_OK;
  if (bad_ptr(a->a, 16) || bad_ptr(a->b, 16) || bad_ptr(a->a_scale, 4) || bad_ptr(a->b_scale, 4) ||
      bad_ptr(a->c, 2))
    return DSA_ERR_INVALID_ARG;
  // Up to 32 activation rows the GEMM is a weight stream on the tensor cores
  // (weights as the MMA's M, the rows of a as its N = 16 or 32); beyond, the
  // tiled tensor-core GEMM.  Measured, 1 to 16 rows: 15.0 us at N = 8192,
  // K = 1536 (tiled 19.1 us), 23.2 us at N = 24576, K = 1536 (tiled 29.3),
  // 70.3 us at N = 24576, K = 7168 (tiled 94.8); 24 rows 17.0 / 25.2 / 76.4.
  if (a->M <= 32) return launch_int8_gemm_wt(*a, static_cast<cudaStream_t>(stream));
  return launch_int8_gemm_tc(*a, static_cast<cudaStream_t>(stream));
}

int dsa_mhc(const dsa_mhc_args* a, void* stream) {
  if (!a || a->n < 0 || a->iters < 0 || !(a->eps >= 0.f)) return DSA_ERR_INVALID_ARG;
  if ((a->hc != 4 && a->hc != 8) || a->iters > 100) return DSA_ERR_UNSUPPORTED;
  if (a->n == 0) return DSA_OK;
  if (bad_ptr(a->mixes, 16) || bad_ptr(a->hc_scale, 4) || bad_ptr(a->hc_base, 4) || bad_ptr(a->pre, 16) ||
      bad_ptr(a->post, 16) || bad_ptr(a->comb, 16))
    return DSA_ERR_INVALID_ARG;
  return launch_mhc(*a, static_cast<cudaStream_t>(stream));
}

static int check_mla(const dsa_mla_prolog_args* a) {
  if (!a || a->T < 0 || a->H < 1 || !(a->rms_eps >= 0.f) || a->cache_rows < 0 || a->rope_max_pos < 1 ||
      (a->rope_interleaved != 0 && a->rope_interleaved != 1))
    return DSA_ERR_INVALID_ARG;
  if (a->T > 32 || a->H > 128 || a->K_q < 128 || a->K_q > 2048 || a->K_q % 128 != 0 || a->D_x < 64 ||
      a->D_x > 16384 || a->D_x % 64 != 0)
    return DSA_ERR_UNSUPPORTED;
  if (a->T == 0) return DSA_OK;
  if (bad_ptr(a->x, 16) || bad_ptr(a->w_dq, 16) || bad_ptr(a->gamma_q, 16) || bad_ptr(a->w_dkv, 16) ||
      bad_ptr(a->gamma_kv, 16) || bad_ptr(a->w_uq, 16) || bad_ptr(a->w_uq_scale, 2) || bad_ptr(a->w_uk, 16) ||
      bad_ptr(a->pos, 4) || bad_ptr(a->rope_cos, 4) || bad_ptr(a->rope_sin, 4) || bad_ptr(a->q_lora, 16) ||
      bad_ptr(a->q_lora_scale, 2) || bad_ptr(a->q, 16) || bad_ptr(a->kv_cache, 16) || bad_ptr(a->slot, 8))
    return DSA_ERR_INVALID_ARG;
  return DSA_OK;
}

size_t dsa_mla_prolog_workspace(const dsa_mla_prolog_args* a) {
  if (check_mla(a) != DSA_OK || a->T == 0) return 0;
  return mla_workspace(*a);
}

int dsa_mla_prolog(const dsa_mla_prolog_args* a, void* ws, size_t ws_bytes, void* stream) {
  const int st = check_mla(a);
  if (st != DSA_OK || a->T == 0) return st;
  if (ws == nullptr || !aligned(ws, 256) || ws_bytes < mla_workspace(*a)) return DSA_ERR_WORKSPACE;
  return launch_mla(*a, ws, static_cast<cudaStream_t>(stream));
}

}  // extern "C"

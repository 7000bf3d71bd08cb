// dsa_indexer_prolog_noalloc: the Indexer Prolog for callers that cannot
// allocate device memory.
//
// Who needs it: code that is handed only its input and output tensors and
// has no device allocator of its own (a plug-in inside a host framework that
// owns all device memory), or a latency-critical loop that must never call
// cudaMalloc, which can synchronise the whole device.  The regular entry
// point asks such a caller for a workspace it has no way to obtain.
//
// Instead of a caller workspace, this variant uses one fixed scratch array
// compiled into the library (kNoAllocScratchBytes = 64 KiB per device).  Every
// GPU that loads the library holds that array until the process exits.
#include <cuda_runtime.h>
#include <mutex>
#include "dsa_internal.h"

namespace dsa {
namespace {

constexpr size_t kNoAllocScratchBytes = 64 * 1024;

// The scratch lives in device memory of every GPU that loads the library.
// In host code `g_noalloc_scratch` is only a host-side stand-in for the
// symbol: its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};
void* g_scratch_ctx[kMaxDevices] = {};

// Device address of the scratch array on the current device.  Resolved on
// the first call made while that device is current, then cached together
// with the context it was resolved in: when another context is current (the
// device was reset, or the caller made its own context current) the
// address is resolved again.
int scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DSA_ERR_CUDA;
  void* ctx = current_context();
  if (ctx == nullptr) return DSA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_scratch_ptr[dev] == nullptr || g_scratch_ctx[dev] != ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return DSA_ERR_CUDA;
    g_scratch_ptr[dev] = p;
    g_scratch_ctx[dev] = ctx;
  }
  *out = g_scratch_ptr[dev];
  return DSA_OK;
}

}  // namespace
}  // namespace dsa

extern "C" int dsa_indexer_prolog_noalloc(const dsa_prolog_args* a, void* stream) {
  // Same argument rules and results as dsa_indexer_prolog.
  const size_t need = dsa_indexer_prolog_workspace(a);
  if (a == nullptr || need == 0) return dsa_indexer_prolog(a, nullptr, 0, stream);  // reports the arg error
  if (a->T == 0) return DSA_OK;
  // Every shape the prolog supports needs at most 33 KB (T <= 32 tokens of
  // d_I + H_I <= 256 fp32 sums, plus the 256-byte ticket): this check only
  // guards shapes a later version may add.
  if (need > dsa::kNoAllocScratchBytes) return DSA_ERR_WORKSPACE;
  void* scratch = nullptr;
  const int st = dsa::scratch_address(&scratch);
  if (st != DSA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The kernel's completion ticket and its k / weight sums must start at
  // zero; the array keeps whatever the previous call left there.
  if (cudaMemsetAsync(scratch, 0, need, s) != cudaSuccess) return DSA_ERR_CUDA;
  return dsa_indexer_prolog(a, scratch, dsa::kNoAllocScratchBytes, stream);
}

// Host-side helpers shared by the launchers of the C ABI (not exported).
#pragma once
#include <cuda_runtime.h>
#include <cstdint>
#include <cstddef>
#include "dsa.h"

namespace dsa {

// Bits of the per-library device error word: a bounded wait that timed out;
// invalid device-side data (an out-of-range slot or position, an unmapped
// page, a histogram that disagrees with its row because the workspace was
// not zero-filled).
constexpr uint32_t kErrTimeout = 1u;
constexpr uint32_t kErrBadIndex = 2u;
// Byte offset, from the error word, of the uint64 time limit (ns) of every
// bounded device wait (set by dsa_set_wait_limit_ns).
constexpr size_t kWaitLimitOffset = 8;

// Address of the library's device error word on the current device
// (resolved once per device and context).  nullptr if CUDA fails.
uint32_t* error_word();

// The calling thread's current CUDA context (a CUcontext), nullptr if none
// or if the driver entry point is unavailable.
void* current_context();

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Number of SMs of the current device (cached per device).
int sm_count();

// Encodes a tiled tensor map (rank <= 5) into `out` (128 bytes, 64-aligned):
// dtype is a CUtensorMapDataType, dims innermost first, strides in bytes of
// dims 1..rank-1, box in elements; OOB elements read as zero.  Returns false
// if the driver entry point is unavailable or rejects the map.
bool encode_tmap(void* out, int dtype, int rank, const void* base, const uint64_t* dims, const uint64_t* strides,
                 const uint32_t* box, int swizzle_bytes);

// Encodes a 2-D tiled tensor map of uint8 rows (inner extent `inner` bytes,
// `rows` rows, `row_stride` bytes apart) with box {inner, box_rows} and the
// given swizzle (0 none, 64 or 128 bytes) into `out` (128 bytes, 64-aligned).
// Returns false if the driver entry point is unavailable or rejects it.
bool encode_tmap_u8_2d(void* out, const void* base, uint64_t inner, uint64_t rows, uint64_t row_stride,
                       uint32_t box_rows, int swizzle_bytes);

inline int cuda_status(cudaError_t e) { return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA; }

// Launchers implemented by the kernel translation units.
int launch_prolog(const dsa_prolog_args& a, void* ws, cudaStream_t s);
size_t prolog_workspace(const dsa_prolog_args& a);

int launch_indexer(const dsa_topk_args& a, float* scores, uint32_t* hist, cudaStream_t s);
// Query tokens the indexer scores together against one key tile (a group).
int indexer_group_tokens(const dsa_topk_args& a);

// Fused top-k path: the indexer also counts each token's scores by their
// leading 12 key bits; the top-k pass then needs one read of the row.
constexpr int kTopkHistBins = 4096;
bool topk_hist_eligible(const dsa_topk_args& a);
size_t topk_hist_workspace(const dsa_topk_args& a);  // the per-token histograms
int launch_topk_hist(const dsa_topk_args& a, const float* scores, int64_t ld, void* ws, cudaStream_t s);
int launch_indexer_dots(const dsa_topk_args& a, int32_t* dots, cudaStream_t s);
int launch_topk(const dsa_topk_args& a, const float* scores, int64_t scores_ld, cudaStream_t s);

size_t attn_workspace(const dsa_attn_args& a);
int launch_attn(const dsa_attn_args& a, void* ws, cudaStream_t s);
int launch_act_quant(const dsa_act_quant_args& a, cudaStream_t s);
// The weight stream of the int8 GEMM on the tensor cores (M <= 32).
int launch_int8_gemm_wt(const dsa_int8_gemm_args& a, cudaStream_t s);
// The tensor-core path of the int8 GEMM (any M; exact int32 sums).
int launch_int8_gemm_tc(const dsa_int8_gemm_args& a, cudaStream_t s);
int launch_mhc(const dsa_mhc_args& a, cudaStream_t s);
size_t mla_workspace(const dsa_mla_prolog_args& a);
int launch_mla(const dsa_mla_prolog_args& a, void* ws, cudaStream_t s);

}  // namespace dsa

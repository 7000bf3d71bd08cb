// Host-side helpers shared by the launchers of the C ABI (not exported).
#pragma once
#include <cuda_runtime.h>
#include <cstdint>
#include <cstddef>
#include "dsa.h"

namespace dsa {

// Address of the library's device error word on the current device
// (resolved once per device).  nullptr if CUDA fails.
uint32_t* error_word();

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Number of SMs of the current device (cached per device).
int sm_count();

inline int cuda_status(cudaError_t e) { return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA; }

// Launchers implemented by the kernel translation units.
int launch_prolog(const dsa_prolog_args& a, void* ws, cudaStream_t s);
size_t prolog_workspace(const dsa_prolog_args& a);

int launch_indexer(const dsa_topk_args& a, float* scores, cudaStream_t s);
int launch_indexer_dots(const dsa_topk_args& a, int32_t* dots, cudaStream_t s);
int launch_topk(const dsa_topk_args& a, const float* scores, int64_t scores_ld, cudaStream_t s);

size_t attn_workspace(const dsa_attn_args& a);
int launch_attn(const dsa_attn_args& a, void* ws, cudaStream_t s);

}  // namespace dsa

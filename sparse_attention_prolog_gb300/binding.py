"""ctypes binding of libdsa.so: argument marshalling only.

Each wrapper takes torch CUDA tensors, fills the C argument struct with their
device pointers and calls the entry point of the same name; every step of
the computation runs in the library's kernels.  Loading fails loudly when the
library has not been built.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libdsa.so")

c_int = ctypes.c_int32
c_ptr = ctypes.c_void_p


class PrologArgs(ctypes.Structure):
    _fields_ = [
        ("T", c_int), ("H_I", c_int), ("d_I", c_int), ("d_rope", c_int), ("K_q", c_int), ("D_x", c_int),
        ("q_lora", c_ptr), ("q_lora_scale", c_ptr), ("w_qb", c_ptr), ("w_qb_scale", c_ptr),
        ("x", c_ptr), ("w_k", c_ptr), ("ln_gamma", c_ptr), ("ln_beta", c_ptr), ("ln_eps", ctypes.c_float),
        ("w_proj", c_ptr), ("w_scale", ctypes.c_float), ("pos", c_ptr), ("rope_cos", c_ptr), ("rope_sin", c_ptr),
        ("rope_max_pos", c_int), ("rope_interleaved", c_int), ("q_out", c_ptr), ("q_scale_out", c_ptr),
        ("k_cache", c_ptr), ("k_scale_cache", c_ptr), ("slot", c_ptr), ("cache_rows", ctypes.c_int64),
        ("w_out", c_ptr),
    ]


class TopkArgs(ctypes.Structure):
    _fields_ = [
        ("T", c_int), ("B", c_int), ("n_q", c_int), ("H_I", c_int), ("d_I", c_int), ("topk", c_int), ("max_L", c_int),
        ("q", c_ptr), ("q_scale", c_ptr), ("w", c_ptr), ("k_cache", c_ptr), ("k_scale", c_ptr),
        ("block_table", c_ptr), ("block_size", c_int), ("max_blocks", c_int), ("pos", c_ptr),
        ("topk_idx", c_ptr), ("scores_out", c_ptr), ("seq_of_token", c_ptr),
    ]


class AttnArgs(ctypes.Structure):
    _fields_ = [
        ("T", c_int), ("B", c_int), ("n_q", c_int), ("H", c_int), ("d_qk", c_int), ("d_v", c_int), ("topk", c_int),
        ("max_L", c_int), ("scale", ctypes.c_float), ("q", c_ptr), ("kv", c_ptr), ("block_table", c_ptr),
        ("block_size", c_int), ("max_blocks", c_int), ("topk_idx", c_ptr), ("out", c_ptr), ("lse", c_ptr),
        ("sink", c_ptr), ("seq_of_token", c_ptr),
    ]


class ActQuantArgs(ctypes.Structure):
    _fields_ = [("M", c_int), ("N", c_int), ("x", c_ptr), ("y", c_ptr), ("scale", c_ptr), ("round_scale", c_int)]


class Int8GemmArgs(ctypes.Structure):
    _fields_ = [("M", c_int), ("N", c_int), ("K", c_int), ("a", c_ptr), ("a_scale", c_ptr), ("b", c_ptr),
                ("b_scale", c_ptr), ("c", c_ptr)]


class MhcArgs(ctypes.Structure):
    _fields_ = [("n", c_int), ("hc", c_int), ("iters", c_int), ("eps", ctypes.c_float), ("mixes", c_ptr),
                ("hc_scale", c_ptr), ("hc_base", c_ptr), ("pre", c_ptr), ("post", c_ptr), ("comb", c_ptr)]


class MlaArgs(ctypes.Structure):
    _fields_ = [("T", c_int), ("H", c_int), ("K_q", c_int), ("D_x", c_int), ("rms_eps", ctypes.c_float),
                ("rope_max_pos", c_int), ("rope_interleaved", c_int), ("x", c_ptr), ("w_dq", c_ptr),
                ("gamma_q", c_ptr), ("w_dkv", c_ptr), ("gamma_kv", c_ptr), ("w_uq", c_ptr), ("w_uq_scale", c_ptr),
                ("w_uk", c_ptr), ("pos", c_ptr), ("rope_cos", c_ptr), ("rope_sin", c_ptr), ("q_lora", c_ptr),
                ("q_lora_scale", c_ptr), ("q", c_ptr), ("kv_cache", c_ptr), ("slot", c_ptr),
                ("cache_rows", ctypes.c_int64)]


EXPORTS = [
    "dsa_status_string", "dsa_abi_version", "dsa_get_device_error", "dsa_set_wait_limit_ns",
    "dsa_indexer_prolog_workspace", "dsa_indexer_prolog",
    "dsa_indexer_topk_workspace", "dsa_indexer_topk", "dsa_indexer_dots_debug",
    "dsa_indexer_scores", "dsa_topk_from_scores",
    "dsa_sparse_attn_workspace", "dsa_sparse_attn", "dsa_indexer_prolog_noalloc", "dsa_act_quant",
    "dsa_int8_gemm", "dsa_mhc", "dsa_mla_prolog_workspace", "dsa_mla_prolog",
]

_lib = None


class DSAError(RuntimeError):
    pass


def load(path: str = LIB_PATH):
    """Loads libdsa.so once; raises if it is missing (no fallback path)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise DSAError(f"{path} is missing: build it with sparse_attention_prolog_gb300.build.build()")
    lib = ctypes.CDLL(path)
    lib.dsa_status_string.restype = ctypes.c_char_p
    lib.dsa_status_string.argtypes = [c_int]
    lib.dsa_abi_version.restype = c_int
    lib.dsa_get_device_error.argtypes = [c_ptr]
    lib.dsa_get_device_error.restype = c_int
    lib.dsa_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
    lib.dsa_set_wait_limit_ns.restype = c_int
    for name, st in (("prolog", PrologArgs), ("topk", TopkArgs), ("attn", AttnArgs)):
        ws = {"prolog": "dsa_indexer_prolog_workspace", "topk": "dsa_indexer_topk_workspace",
              "attn": "dsa_sparse_attn_workspace"}[name]
        run = {"prolog": "dsa_indexer_prolog", "topk": "dsa_indexer_topk", "attn": "dsa_sparse_attn"}[name]
        getattr(lib, ws).argtypes = [ctypes.POINTER(st)]
        getattr(lib, ws).restype = ctypes.c_size_t
        getattr(lib, run).argtypes = [ctypes.POINTER(st), c_ptr, ctypes.c_size_t, c_ptr]
        getattr(lib, run).restype = c_int
    lib.dsa_indexer_prolog_noalloc.argtypes = [ctypes.POINTER(PrologArgs), c_ptr]
    lib.dsa_indexer_prolog_noalloc.restype = c_int
    lib.dsa_indexer_dots_debug.argtypes = [ctypes.POINTER(TopkArgs), c_ptr, c_ptr]
    lib.dsa_indexer_dots_debug.restype = c_int
    lib.dsa_indexer_scores.argtypes = [ctypes.POINTER(TopkArgs), c_ptr, c_ptr]
    lib.dsa_indexer_scores.restype = c_int
    lib.dsa_topk_from_scores.argtypes = [ctypes.POINTER(TopkArgs), c_ptr, ctypes.c_int64, c_ptr]
    lib.dsa_topk_from_scores.restype = c_int
    lib.dsa_act_quant.argtypes = [ctypes.POINTER(ActQuantArgs), c_ptr]
    lib.dsa_act_quant.restype = c_int
    lib.dsa_int8_gemm.argtypes = [ctypes.POINTER(Int8GemmArgs), c_ptr]
    lib.dsa_int8_gemm.restype = c_int
    lib.dsa_mhc.argtypes = [ctypes.POINTER(MhcArgs), c_ptr]
    lib.dsa_mhc.restype = c_int
    lib.dsa_mla_prolog_workspace.argtypes = [ctypes.POINTER(MlaArgs)]
    lib.dsa_mla_prolog_workspace.restype = ctypes.c_size_t
    lib.dsa_mla_prolog.argtypes = [ctypes.POINTER(MlaArgs), c_ptr, ctypes.c_size_t, c_ptr]
    lib.dsa_mla_prolog.restype = c_int
    _lib = lib
    return lib


def status_string(code: int) -> str:
    return load().dsa_status_string(code).decode()


def _check(code: int, what: str):
    if code != 0:
        raise DSAError(f"{what}: {status_string(code)} ({code})")


def _p(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ws(nbytes: int, device, ws: Optional[torch.Tensor]):
    if nbytes == 0:
        return None, 0
    if ws is not None:
        assert ws.numel() * ws.element_size() >= nbytes
        return ws, ws.numel() * ws.element_size()
    return torch.zeros(nbytes, dtype=torch.uint8, device=device), nbytes


# ---------------------------------------------------------------- prolog
def prolog_args(T, H_I, d_I, d_rope, q_lora, q_lora_scale, w_qb, w_qb_scale, x, w_k, ln_gamma, ln_beta,
                ln_eps, w_proj, w_scale, pos, rope_cos, rope_sin, rope_interleaved, q_out, q_scale_out,
                k_cache, k_scale_cache, slot, w_out) -> PrologArgs:
    return PrologArgs(
        T, H_I, d_I, d_rope, q_lora.shape[1] if T else 0, x.shape[1] if T else 0,
        _p(q_lora), _p(q_lora_scale), _p(w_qb), _p(w_qb_scale), _p(x), _p(w_k), _p(ln_gamma), _p(ln_beta),
        float(ln_eps), _p(w_proj), float(w_scale), _p(pos), _p(rope_cos), _p(rope_sin), rope_cos.shape[0],
        int(rope_interleaved), _p(q_out), _p(q_scale_out), _p(k_cache), _p(k_scale_cache), _p(slot),
        k_cache.shape[0], _p(w_out))


def dsa_indexer_prolog(args: PrologArgs, workspace: Optional[torch.Tensor] = None, stream=None,
                       device=None):
    lib = load()
    need = lib.dsa_indexer_prolog_workspace(ctypes.byref(args))
    ws, n = _ws(need, device or "cuda", workspace)
    _check(lib.dsa_indexer_prolog(ctypes.byref(args), _p(ws), n, _stream(stream)), "dsa_indexer_prolog")
    return ws


def dsa_indexer_prolog_noalloc(args: PrologArgs, stream=None):
    """The prolog without a workspace: its scratch is a fixed array inside the
    library, for callers that cannot allocate device memory."""
    _check(load().dsa_indexer_prolog_noalloc(ctypes.byref(args), _stream(stream)), "dsa_indexer_prolog_noalloc")


# ----------------------------------------------------------------- top-k
def topk_args(T, B, n_q, H_I, d_I, topk, max_L, q, q_scale, w, k_cache, k_scale, pos, topk_idx,
              block_table=None, block_size=0, scores_out=None, seq_of_token=None) -> TopkArgs:
    """seq_of_token: int32 [T] sequence of each token (then n_q is ignored), or
    None for the uniform batch T = B * n_q."""
    max_blocks = 0 if block_table is None else block_table.shape[1]
    return TopkArgs(T, B, n_q, H_I, d_I, topk, max_L, _p(q), _p(q_scale), _p(w), _p(k_cache), _p(k_scale),
                    _p(block_table), block_size, max_blocks, _p(pos), _p(topk_idx), _p(scores_out),
                    _p(seq_of_token))


def dsa_indexer_topk(args: TopkArgs, workspace: Optional[torch.Tensor] = None, stream=None, device=None):
    lib = load()
    need = lib.dsa_indexer_topk_workspace(ctypes.byref(args))
    ws, n = _ws(need, device or "cuda", workspace)
    _check(lib.dsa_indexer_topk(ctypes.byref(args), _p(ws), n, _stream(stream)), "dsa_indexer_topk")
    return ws


def dsa_indexer_dots_debug(args: TopkArgs, dots: torch.Tensor, stream=None):
    _check(load().dsa_indexer_dots_debug(ctypes.byref(args), _p(dots), _stream(stream)), "dsa_indexer_dots_debug")


def dsa_indexer_scores(args: TopkArgs, scores: torch.Tensor, stream=None):
    _check(load().dsa_indexer_scores(ctypes.byref(args), _p(scores), _stream(stream)), "dsa_indexer_scores")


def dsa_topk_from_scores(args: TopkArgs, scores: torch.Tensor, stream=None):
    _check(load().dsa_topk_from_scores(ctypes.byref(args), _p(scores), scores.stride(0), _stream(stream)),
           "dsa_topk_from_scores")


# -------------------------------------------------------------- attention
def attn_args(T, B, n_q, H, topk, max_L, scale, q, kv, topk_idx, out, lse=None, block_table=None,
              block_size=0, d_qk=576, d_v=512, sink=None, seq_of_token=None) -> AttnArgs:
    max_blocks = 0 if block_table is None else block_table.shape[1]
    return AttnArgs(T, B, n_q, H, d_qk, d_v, topk, max_L, float(scale), _p(q), _p(kv), _p(block_table),
                    block_size, max_blocks, _p(topk_idx), _p(out), _p(lse), _p(sink), _p(seq_of_token))


def dsa_sparse_attn(args: AttnArgs, workspace: Optional[torch.Tensor] = None, stream=None, device=None):
    lib = load()
    need = lib.dsa_sparse_attn_workspace(ctypes.byref(args))
    ws, n = _ws(need, device or "cuda", workspace)
    _check(lib.dsa_sparse_attn(ctypes.byref(args), _p(ws), n, _stream(stream)), "dsa_sparse_attn")
    return ws


def workspace_bytes(kind: str, args) -> int:
    lib = load()
    fn = {"prolog": lib.dsa_indexer_prolog_workspace, "topk": lib.dsa_indexer_topk_workspace,
          "attn": lib.dsa_sparse_attn_workspace, "mla": lib.dsa_mla_prolog_workspace}[kind]
    return int(fn(ctypes.byref(args)))


def device_error(stream=None) -> int:
    return int(load().dsa_get_device_error(_stream(stream)))


def set_wait_limit_ns(ns: int):
    """Time limit of the library's bounded device waits on the current device
    (0 restores the default)."""
    _check(load().dsa_set_wait_limit_ns(int(ns)), "dsa_set_wait_limit_ns")


def dsa_act_quant(x: torch.Tensor, y: torch.Tensor, scale: torch.Tensor, round_scale: bool = False, stream=None):
    """x bf16 [M, N] -> y int8 [M, N], scale fp32 [M] (see dsa.h)."""
    M, N = x.shape
    args = ActQuantArgs(M, N, _p(x), _p(y), _p(scale), int(bool(round_scale)))
    _check(load().dsa_act_quant(ctypes.byref(args), _stream(stream)), "dsa_act_quant")


def dsa_int8_gemm(a: torch.Tensor, a_scale: torch.Tensor, b: torch.Tensor, b_scale: torch.Tensor,
                  c: torch.Tensor, stream=None):
    """a int8 [M, K], b int8 [N, K], fp32 scales -> c fp16 [M, N] (see dsa.h)."""
    M, K = a.shape
    N = b.shape[0]
    args = Int8GemmArgs(M, N, K, _p(a), _p(a_scale), _p(b), _p(b_scale), _p(c))
    _check(load().dsa_int8_gemm(ctypes.byref(args), _stream(stream)), "dsa_int8_gemm")


def dsa_mhc(mixes: torch.Tensor, hc_scale: torch.Tensor, hc_base: torch.Tensor, hc: int, iters: int, eps: float,
            pre: torch.Tensor, post: torch.Tensor, comb: torch.Tensor, stream=None):
    """mixes fp32 [n, hc (2 + hc)] -> pre [n, hc], post [n, hc], comb [n, hc, hc] (see dsa.h)."""
    args = MhcArgs(mixes.shape[0], hc, iters, float(eps), _p(mixes), _p(hc_scale), _p(hc_base), _p(pre), _p(post),
                   _p(comb))
    _check(load().dsa_mhc(ctypes.byref(args), _stream(stream)), "dsa_mhc")


# ------------------------------------------------------------ MLA Prolog
def mla_args(x, w_dq, gamma_q, w_dkv, gamma_kv, rms_eps, w_uq, w_uq_scale, w_uk, pos, rope_cos, rope_sin,
             rope_interleaved, q_lora, q_lora_scale, q, kv_cache, slot) -> MlaArgs:
    """x bf16 [T, D_x], w_dq bf16 [K_q, D_x], w_dkv bf16 [576, D_x], w_uq int8 [H*192, K_q], w_uk bf16
    [H, 128, 512]; outputs q_lora int8 [T, K_q], q_lora_scale fp16 [T], q bf16 [T, H, 576] and the
    kv_cache bf16 [rows, 576] rows at slot (see dsa.h)."""
    T, D_x = x.shape
    return MlaArgs(T, w_uk.shape[0], w_dq.shape[0], D_x, float(rms_eps), rope_cos.shape[0], int(rope_interleaved),
                   _p(x), _p(w_dq), _p(gamma_q), _p(w_dkv), _p(gamma_kv), _p(w_uq), _p(w_uq_scale), _p(w_uk),
                   _p(pos), _p(rope_cos), _p(rope_sin), _p(q_lora), _p(q_lora_scale), _p(q), _p(kv_cache),
                   _p(slot), kv_cache.shape[0])


def dsa_mla_prolog(args: MlaArgs, workspace: Optional[torch.Tensor] = None, stream=None, device=None):
    """Runs the MLA Prolog; a new workspace is zero-filled, a given one must
    have been zero-filled before its first use.  Returns the workspace."""
    lib = load()
    need = lib.dsa_mla_prolog_workspace(ctypes.byref(args))
    ws, n = _ws(need, device or "cuda", workspace)
    _check(lib.dsa_mla_prolog(ctypes.byref(args), _p(ws), n, _stream(stream)), "dsa_mla_prolog")
    return ws

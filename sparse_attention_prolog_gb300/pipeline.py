"""Device-side buffers and the decode step chain (prolog -> indexer/top-k ->
sparse attention) over the C ABI.  PyTorch provides device memory and
streams only; the computation is the library's."""
from __future__ import annotations

import numpy as np
import torch

from . import binding as B

INT16_VIEW = {"fp16": torch.float16, "bf16": torch.bfloat16}


def to_dev(a: np.ndarray, device, kind: str = None) -> torch.Tensor:
    """Uploads a numpy array; uint16 arrays holding fp16/bf16 bits become
    fp16/bf16 tensors with the same bits."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        t = torch.from_numpy(a.view(np.int16)).to(device)
        return t.view(INT16_VIEW[kind or "bf16"])
    if a.dtype == np.float16:
        return torch.from_numpy(a).to(device)
    return torch.from_numpy(a).to(device)


class PrologBuffers:
    """Device copies of a workloads.PrologInputs plus its outputs.  q_lora,
    q_lora_scale and x may be given as device tensors (another kernel's
    outputs or inputs, e.g. the MLA Prolog's)."""

    def __init__(self, p, device, k_cache: torch.Tensor = None, k_scale_cache: torch.Tensor = None,
                 q_lora: torch.Tensor = None, q_lora_scale: torch.Tensor = None, x: torch.Tensor = None):
        self.p = p
        d = device
        self.q_lora = to_dev(p.q_lora, d) if q_lora is None else q_lora
        self.q_lora_scale = to_dev(p.q_lora_scale, d) if q_lora_scale is None else q_lora_scale
        self.w_qb = to_dev(p.w_qb, d)
        self.w_qb_scale = to_dev(p.w_qb_scale, d)
        self.x = to_dev(p.x, d, "bf16") if x is None else x
        self.w_k = to_dev(p.w_k, d, "bf16")
        self.ln_gamma = to_dev(p.ln_gamma, d)
        self.ln_beta = to_dev(p.ln_beta, d)
        self.w_proj = None if p.w_proj is None else to_dev(p.w_proj, d, "bf16")
        self.pos = to_dev(p.pos, d)
        self.rope_cos = to_dev(p.rope_cos, d)
        self.rope_sin = to_dev(p.rope_sin, d)
        self.slot = to_dev(p.slot, d)
        T, H, D = p.T, p.H_I, p.d_I
        self.q_out = torch.zeros(T, H, D, dtype=torch.int8, device=d)
        self.q_scale_out = torch.zeros(T, H, dtype=torch.float16, device=d)
        rows = int(max(p.slot.max() + 1, 1)) if k_cache is None else k_cache.shape[0]
        self.k_cache = k_cache if k_cache is not None else torch.zeros(rows, D, dtype=torch.int8, device=d)
        self.k_scale_cache = (k_scale_cache if k_scale_cache is not None
                              else torch.zeros(rows, dtype=torch.float16, device=d))
        self.w_out = None if p.w_proj is None else torch.zeros(T, H, dtype=torch.float32, device=d)
        self.args = B.prolog_args(T, H, D, p.d_rope, self.q_lora, self.q_lora_scale, self.w_qb, self.w_qb_scale,
                                  self.x, self.w_k, self.ln_gamma, self.ln_beta, p.ln_eps, self.w_proj, p.w_scale,
                                  self.pos, self.rope_cos, self.rope_sin, p.rope_interleaved, self.q_out,
                                  self.q_scale_out, self.k_cache, self.k_scale_cache, self.slot, self.w_out)
        self.ws = torch.zeros(max(B.workspace_bytes("prolog", self.args), 256), dtype=torch.uint8, device=d)

    def run(self, stream=None):
        B.dsa_indexer_prolog(self.args, self.ws, stream)


class MlaBuffers:
    """Device copies of a workloads.MlaInputs plus the MLA Prolog's outputs
    (q_lora, q_lora_scale, q) and a latent cache of ``cache_rows`` rows."""

    def __init__(self, p, device, cache_rows: int, kv_fill: float = 0.0, kv_cache: torch.Tensor = None):
        self.p = p
        d = device
        self.x = to_dev(p.x, d, "bf16")
        self.w_dq = to_dev(p.w_dq, d, "bf16")
        self.gamma_q = to_dev(p.gamma_q, d)
        self.w_dkv = to_dev(p.w_dkv, d, "bf16")
        self.gamma_kv = to_dev(p.gamma_kv, d)
        self.w_uq = to_dev(p.w_uq, d)
        self.w_uq_scale = to_dev(p.w_uq_scale, d)
        self.w_uk = to_dev(p.w_uk, d, "bf16")
        self.pos = to_dev(p.pos, d)
        self.rope_cos = to_dev(p.rope_cos, d)
        self.rope_sin = to_dev(p.rope_sin, d)
        self.slot = to_dev(p.slot, d)
        self.q_lora = torch.zeros(p.T, p.K_q, dtype=torch.int8, device=d)
        self.q_lora_scale = torch.zeros(p.T, dtype=torch.float16, device=d)
        self.q = torch.zeros(p.T, p.H, 576, dtype=torch.bfloat16, device=d)
        self.kv_cache = (torch.full((cache_rows, 576), kv_fill, dtype=torch.bfloat16, device=d) if kv_cache is None
                         else kv_cache)
        self.args = B.mla_args(self.x, self.w_dq, self.gamma_q, self.w_dkv, self.gamma_kv, p.rms_eps, self.w_uq,
                               self.w_uq_scale, self.w_uk, self.pos, self.rope_cos, self.rope_sin,
                               p.rope_interleaved, self.q_lora, self.q_lora_scale, self.q, self.kv_cache, self.slot)
        self.ws = torch.zeros(max(B.workspace_bytes("mla", self.args), 256), dtype=torch.uint8, device=d)

    def run(self, stream=None):
        B.dsa_mla_prolog(self.args, self.ws, stream)


def is_uniform(inp) -> bool:
    """True if token t of the batch belongs to sequence t // n_q, n_q = T / B."""
    if inp.T % inp.B:
        return False
    return bool(np.array_equal(inp.seq_of_token, np.repeat(np.arange(inp.B, dtype=np.int32), inp.T // inp.B)))


class DecodeBuffers:
    """Device copies of a workloads.DecodeInputs and the indexer/attention
    outputs.  ``q_idx``/``q_idx_scale``/``w_idx`` may be replaced by the
    prolog's outputs (then pass them in).  The calls get the token map
    (seq_of_token) when the batch is not uniform, or when ``seq_map``."""

    def __init__(self, inp, device, q_idx=None, q_idx_scale=None, w_idx=None, k_cache=None, k_scale=None,
                 with_attention=True, keep_scores=False, seq_map=False, q_attn=None, kv=None):
        self.inp = inp
        d = device
        self.q_idx = q_idx if q_idx is not None else to_dev(inp.q_idx, d)
        self.q_idx_scale = q_idx_scale if q_idx_scale is not None else to_dev(inp.q_idx_scale, d)
        self.w_idx = w_idx if w_idx is not None else to_dev(inp.w_idx, d)
        self.k_cache = k_cache if k_cache is not None else to_dev(inp.k_cache, d)
        self.k_scale = k_scale if k_scale is not None else to_dev(inp.k_scale, d)
        self.block_table = None if inp.block_table is None else to_dev(inp.block_table, d)
        self.pos = to_dev(inp.pos, d)
        T = inp.T
        self.seq = to_dev(inp.seq_of_token.astype(np.int32), d) if (seq_map or not is_uniform(inp)) else None
        n_q = max(T // inp.B, 1)
        self.topk_idx = torch.full((T, inp.topk), -7, dtype=torch.int32, device=d)
        self.scores = torch.empty(T, inp.max_L, dtype=torch.float32, device=d) if keep_scores else None
        self.targs = B.topk_args(T, inp.B, n_q, inp.H_I, inp.d_I, inp.topk, inp.max_L, self.q_idx,
                                 self.q_idx_scale, self.w_idx, self.k_cache, self.k_scale, self.pos, self.topk_idx,
                                 self.block_table, inp.block_size, self.scores, seq_of_token=self.seq)
        self.tws = torch.zeros(max(B.workspace_bytes("topk", self.targs), 256), dtype=torch.uint8, device=d)
        self.with_attention = with_attention
        if with_attention:
            self.q_attn = to_dev(inp.q_attn, d, "bf16") if q_attn is None else q_attn
            self.kv = to_dev(inp.kv_cache, d, "bf16") if kv is None else kv
            self.out = torch.zeros(T, inp.H, inp.d_v, dtype=torch.bfloat16, device=d)
            self.lse = torch.zeros(T, inp.H, dtype=torch.float32, device=d)
            self.aargs = B.attn_args(T, inp.B, n_q, inp.H, inp.topk, inp.max_L, inp.scale, self.q_attn,
                                     self.kv, self.topk_idx, self.out, self.lse, self.block_table, inp.block_size,
                                     seq_of_token=self.seq)
            self.aws = torch.zeros(max(B.workspace_bytes("attn", self.aargs), 256), dtype=torch.uint8, device=d)

    def run_topk(self, stream=None):
        B.dsa_indexer_topk(self.targs, self.tws, stream)

    def run_attn(self, stream=None):
        B.dsa_sparse_attn(self.aargs, self.aws, stream)

    def run(self, stream=None):
        self.run_topk(stream)
        if self.with_attention:
            self.run_attn(stream)


class DiaBuffers:
    """One decode step of DeepSeek Indexer Attention on the device: the MLA
    Prolog (query latent q_lora, attention query q, latent KV rows into the
    latent cache) -> the Indexer Prolog (fed the MLA Prolog's q_lora and the
    same hidden states x; new keys into the key cache) -> Lightning Indexer
    + top-k -> sparse attention (the MLA Prolog's q over the latent cache).
    `dia` is a workloads.DiaInputs."""

    def __init__(self, dia, device, keep_scores=False):
        d = device
        inp = dia.decode
        self.dia = dia
        self.k_cache = to_dev(inp.k_cache, d)
        self.k_scale = to_dev(inp.k_scale, d)
        self.kv = to_dev(inp.kv_cache, d, "bf16")
        self.mla = MlaBuffers(dia.mla, d, self.kv.shape[0], kv_cache=self.kv)
        self.pro = PrologBuffers(dia.prolog, d, self.k_cache, self.k_scale, q_lora=self.mla.q_lora,
                                 q_lora_scale=self.mla.q_lora_scale, x=self.mla.x)
        self.buf = DecodeBuffers(inp, d, q_idx=self.pro.q_out, q_idx_scale=self.pro.q_scale_out, w_idx=self.pro.w_out,
                                 k_cache=self.k_cache, k_scale=self.k_scale, keep_scores=keep_scores,
                                 q_attn=self.mla.q, kv=self.kv)

    def run(self, stream=None):
        self.mla.run(stream)
        self.pro.run(stream)
        self.buf.run(stream)

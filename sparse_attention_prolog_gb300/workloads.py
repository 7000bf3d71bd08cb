"""Seeded synthetic inputs for the DSA decode hot path.

This module only draws random numbers and lays them out; it holds none of
the method's arithmetic (no quantisation, no GEMM, no RoPE, no Hadamard, no
softmax).  Both the CUDA path's callers (tests, bench) and the CPU oracle's
callers take their inputs from here; the oracle never imports it.

Recipes (numpy PCG64, one seed per workload):

* int8 operands that the pages produce by dynamic per-row quantisation of
  N(0,1) data (indexer q, the C8 key cache, q_lora, w_qb) are drawn directly
  as codes ``clip(rint(N(0,1) * 127/4), -127, 127)`` with FP16 scales
  ``(4/127) * sigma * U(0.9, 1.1)``: the same shape and spread as quantised
  normals without running the quantiser.
* bf16 tensors (x, w_k, w_proj, attention q, latent KV) are N(0, sigma)
  rounded to bf16 (round to nearest even), stored as raw uint16 bits.
* RoPE cos/sin tables are built in float64 from theta_i = base^(-2i/d_rope)
  and rounded to fp32; they are inputs of the prolog, the same way a model
  precomputes its rotary cache.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

I8_CODE_STD = 127.0 / 4.0  # code spread of a quantised N(0,1) row


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest even) and return the uint16 bit pattern."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounding = ((b >> 16) & 1) + np.uint32(0x7FFF)
    return ((b + rounding) >> 16).astype(np.uint16)


def bf16_normal(rng, shape, sigma=1.0, mean=0.0) -> np.ndarray:
    x = rng.standard_normal(int(np.prod(shape)), dtype=np.float32)
    if sigma != 1.0:
        x *= np.float32(sigma)
    if mean != 0.0:
        x += np.float32(mean)
    return f32_to_bf16_bits(x).reshape(shape)


def int8_codes(rng, shape) -> np.ndarray:
    x = rng.standard_normal(int(np.prod(shape)), dtype=np.float32) * np.float32(I8_CODE_STD)
    return np.clip(np.rint(x), -127, 127).astype(np.int8).reshape(shape)


def fp16_scales(rng, shape, sigma=1.0) -> np.ndarray:
    u = rng.uniform(0.9, 1.1, size=shape)
    return (u * sigma * 4.0 / 127.0).astype(np.float16)


def rope_tables(max_pos: int, d_rope: int, base: float = 10000.0):
    """cos/sin [max_pos, d_rope/2] fp32, angle(p, i) = p * base^(-2i/d_rope)."""
    half = d_rope // 2
    inv = base ** (-(2.0 * np.arange(half, dtype=np.float64)) / d_rope)
    ang = np.arange(max_pos, dtype=np.float64)[:, None] * inv[None, :]
    return np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)


# ----------------------------------------------------------------------------
# Indexer Prolog inputs
# ----------------------------------------------------------------------------
@dataclasses.dataclass
class PrologInputs:
    T: int
    H_I: int
    d_I: int
    d_rope: int
    q_lora: np.ndarray        # int8 [T, K_q]
    q_lora_scale: np.ndarray  # fp16 [T]
    w_qb: np.ndarray          # int8 [H_I*d_I, K_q]  (K-major: row n holds w_qb[:, n])
    w_qb_scale: np.ndarray    # fp16 [H_I*d_I]
    x: np.ndarray             # bf16 bits [T, D_x]
    w_k: np.ndarray           # bf16 bits [d_I, D_x]
    ln_gamma: np.ndarray      # fp32 [d_I]
    ln_beta: np.ndarray       # fp32 [d_I]
    ln_eps: float
    w_proj: Optional[np.ndarray]  # bf16 bits [H_I, D_x] or None
    w_scale: float
    pos: np.ndarray           # int32 [T]
    rope_cos: np.ndarray      # fp32 [max_pos, d_rope/2]
    rope_sin: np.ndarray
    rope_interleaved: int
    slot: np.ndarray          # int64 [T] flat key-cache row, -1 = do not write


def make_prolog_inputs(T, pos, slot, seed, H_I=64, d_I=128, K_q=1536, D_x=7168,
                       d_rope=64, with_weights=True, max_pos=None,
                       rope_interleaved=0) -> PrologInputs:
    rng = _rng(seed)
    pos = np.asarray(pos, dtype=np.int32)
    if max_pos is None:
        max_pos = int(pos.max()) + 1
    cos, sin = rope_tables(max_pos, d_rope)
    N = H_I * d_I
    return PrologInputs(
        T=T, H_I=H_I, d_I=d_I, d_rope=d_rope,
        q_lora=int8_codes(rng, (T, K_q)),
        q_lora_scale=fp16_scales(rng, (T,), 1.0),
        w_qb=int8_codes(rng, (N, K_q)),
        w_qb_scale=fp16_scales(rng, (N,), 0.02),
        x=bf16_normal(rng, (T, D_x)),
        w_k=bf16_normal(rng, (d_I, D_x), sigma=0.02),
        ln_gamma=(1.0 + 0.1 * rng.standard_normal(d_I)).astype(np.float32),
        ln_beta=(0.1 * rng.standard_normal(d_I)).astype(np.float32),
        ln_eps=1e-6,
        w_proj=bf16_normal(rng, (H_I, D_x), sigma=1.0 / math.sqrt(D_x)) if with_weights else None,
        w_scale=1.0 / math.sqrt(H_I),
        pos=pos, rope_cos=cos, rope_sin=sin, rope_interleaved=rope_interleaved,
        slot=np.asarray(slot, dtype=np.int64),
    )


# ----------------------------------------------------------------------------
# MLA Prolog inputs
# ----------------------------------------------------------------------------
@dataclasses.dataclass
class MlaInputs:
    T: int
    H: int
    K_q: int
    D_x: int
    x: np.ndarray             # bf16 bits [T, D_x]
    w_dq: np.ndarray          # bf16 bits [K_q, D_x] (row n = output channel n)
    gamma_q: np.ndarray       # fp32 [K_q]
    w_dkv: np.ndarray         # bf16 bits [576, D_x]: 512 latent rows, then 64 rotary rows
    gamma_kv: np.ndarray      # fp32 [512]
    rms_eps: float
    w_uq: np.ndarray          # int8 [H*192, K_q]: per head 128 no-position rows, then 64 rotary rows
    w_uq_scale: np.ndarray    # fp16 [H*192]
    w_uk: np.ndarray          # bf16 bits [H, 128, 512]
    pos: np.ndarray           # int32 [T]
    rope_cos: np.ndarray      # fp32 [max_pos, 32]
    rope_sin: np.ndarray
    rope_interleaved: int
    slot: np.ndarray          # int64 [T] latent-cache row, -1 = do not write


def make_mla_inputs(T, pos, slot, seed, H=128, K_q=1536, D_x=7168, max_pos=None,
                    rope_interleaved=0) -> MlaInputs:
    """Projections scaled so that every intermediate is about N(0, 1):
    w_dq, w_dkv ~ N(0, 1/D_x); w_uq codes like a quantised normal with
    scales (4/127) K_q^-1/2 U(0.9, 1.1); w_uk ~ N(0, 1/128); gammas
    1 + 0.1 N(0, 1)."""
    rng = _rng(seed)
    pos = np.asarray(pos, dtype=np.int32)
    if max_pos is None:
        max_pos = int(pos.max()) + 1
    cos, sin = rope_tables(max_pos, 64)
    return MlaInputs(
        T=T, H=H, K_q=K_q, D_x=D_x,
        x=bf16_normal(rng, (T, D_x)),
        w_dq=bf16_normal(rng, (K_q, D_x), sigma=1.0 / math.sqrt(D_x)),
        gamma_q=(1.0 + 0.1 * rng.standard_normal(K_q)).astype(np.float32),
        w_dkv=bf16_normal(rng, (576, D_x), sigma=1.0 / math.sqrt(D_x)),
        gamma_kv=(1.0 + 0.1 * rng.standard_normal(512)).astype(np.float32),
        rms_eps=1e-6,
        w_uq=int8_codes(rng, (H * 192, K_q)),
        w_uq_scale=fp16_scales(rng, (H * 192,), 1.0 / math.sqrt(K_q)),
        w_uk=bf16_normal(rng, (H, 128, 512), sigma=1.0 / math.sqrt(128)),
        pos=pos, rope_cos=cos, rope_sin=sin, rope_interleaved=rope_interleaved,
        slot=np.asarray(slot, dtype=np.int64),
    )


# ----------------------------------------------------------------------------
# Indexer (+ top-k) and sparse attention inputs
# ----------------------------------------------------------------------------
@dataclasses.dataclass
class DecodeInputs:
    """One batch of query tokens over B sequences.

    Token t belongs to sequence ``seq_of_token[t]`` and may see keys
    ``s <= pos[t]``.  Caches are either contiguous ([B, max_L, .]) or paged
    (physical rows [n_blocks*block_size, .] addressed through
    ``block_table[b, s // block_size]``).
    """
    T: int
    B: int
    max_L: int
    H_I: int
    d_I: int
    topk: int
    seq_of_token: np.ndarray   # int32 [T]
    pos: np.ndarray            # int32 [T]
    seq_len: np.ndarray        # int32 [B]  (keys that exist per sequence)
    q_idx: np.ndarray          # int8 [T, H_I, d_I]
    q_idx_scale: np.ndarray    # fp16 [T, H_I]
    w_idx: np.ndarray          # fp32 [T, H_I]
    k_cache: np.ndarray        # int8 [rows, d_I]
    k_scale: np.ndarray        # fp16 [rows]
    block_table: Optional[np.ndarray]  # int32 [B, max_blocks] or None
    block_size: int
    # attention
    H: int
    d_qk: int
    d_v: int
    scale: float
    q_attn: np.ndarray         # bf16 bits [T, H, d_qk]
    kv_cache: np.ndarray       # bf16 bits [rows, d_qk]


def make_decode_inputs(B, n_q, seq_lens, H_I, d_I, topk, H, seed, max_L=None,
                       w_sigma=None, block_size=0, d_qk=576, d_v=512,
                       with_attention=True) -> DecodeInputs:
    """Decode/prefill batch.  n_q is the query-token count of every sequence
    (an int) or of each sequence (a list, e.g. mixed MTP depths); token j of
    sequence b sits at position seq_len[b] - n_q[b] + j (so a prefill of S
    tokens uses n_q = S), and the tokens of a sequence are adjacent."""
    rng = _rng(seed)
    seq_lens = np.asarray(seq_lens, dtype=np.int64)
    counts = np.full(B, n_q, dtype=np.int64) if np.isscalar(n_q) else np.asarray(n_q, dtype=np.int64)
    assert seq_lens.shape == (B,) and counts.shape == (B,) and (counts >= 1).all() and (seq_lens >= counts).all()
    T = int(counts.sum())
    if max_L is None:
        max_L = int(seq_lens.max())
    seq_of_token = np.repeat(np.arange(B, dtype=np.int32), counts)
    pos = np.concatenate([np.arange(int(L) - int(c), int(L)) for L, c in zip(seq_lens, counts)]).astype(np.int32)
    if w_sigma is None:
        w_sigma = 1.0 / math.sqrt(H_I)
    block_table = None
    if block_size:
        blocks_per_seq = [int(-(-int(L) // block_size)) for L in seq_lens]
        max_blocks = -(-max_L // block_size)
        n_blocks = int(sum(blocks_per_seq))
        perm = rng.permutation(n_blocks).astype(np.int32)
        block_table = np.full((B, max_blocks), -1, dtype=np.int32)
        o = 0
        for b, nb in enumerate(blocks_per_seq):
            block_table[b, :nb] = perm[o:o + nb]
            o += nb
        rows = n_blocks * block_size
    else:
        rows = B * max_L
    inp = DecodeInputs(
        T=T, B=B, max_L=max_L, H_I=H_I, d_I=d_I, topk=topk,
        seq_of_token=seq_of_token, pos=pos, seq_len=seq_lens.astype(np.int32),
        q_idx=int8_codes(rng, (T, H_I, d_I)),
        q_idx_scale=fp16_scales(rng, (T, H_I)),
        w_idx=(rng.standard_normal((T, H_I)) * w_sigma).astype(np.float32),
        k_cache=int8_codes(rng, (rows, d_I)),
        k_scale=fp16_scales(rng, (rows,)),
        block_table=block_table, block_size=block_size,
        H=H, d_qk=d_qk, d_v=d_v, scale=192.0 ** -0.5,
        q_attn=bf16_normal(rng, (T, H, d_qk)) if with_attention else np.zeros((T, H, d_qk), np.uint16),
        kv_cache=bf16_normal(rng, (rows, d_qk)) if with_attention else np.zeros((0, d_qk), np.uint16),
    )
    return inp


# ----------------------------------------------------------------------------
# The five workloads
# ----------------------------------------------------------------------------
def tiny_decode(seed=1001):
    """B=1, 2 query tokens at positions 254/255 over L=256; H_I=4 x d_I=64;
    top-k 32; 4 attention heads."""
    return make_decode_inputs(B=1, n_q=2, seq_lens=[256], H_I=4, d_I=64, topk=32,
                              H=4, seed=seed, w_sigma=0.5)


def decode_64k(seed=1002, with_attention=True):
    """B=4, MTP1 (2 tokens per sequence), L=65536; H_I=64 x d_I=128; top-k
    2048; 128 attention heads (the headline decode step)."""
    return make_decode_inputs(B=4, n_q=2, seq_lens=[65536] * 4, H_I=64, d_I=128,
                              topk=2048, H=128, seed=seed, w_sigma=1.0 / 8.0,
                              with_attention=with_attention)


def decode_64k_prolog(seed=2002):
    """Prolog inputs of the headline decode step: T=8 tokens whose new keys
    go to the last two rows of each of the four 64K sequences."""
    L = 65536
    pos = np.array([L - 2, L - 1] * 4, dtype=np.int32)
    slot = np.array([b * L + p for b in range(4) for p in (L - 2, L - 1)], dtype=np.int64)
    return make_prolog_inputs(T=8, pos=pos, slot=slot, seed=seed, max_pos=L)


def prolog_alone(seed=1003):
    """T=8 tokens at positions 0..7, no weight stream, cache of 8 rows."""
    return make_prolog_inputs(T=8, pos=np.arange(8), slot=np.arange(8), seed=seed,
                              with_weights=False)


def causal_prefill(seed=1004, S=8192, with_attention=True):
    """B=1, S query tokens over S keys, top-k 2048 among s <= t."""
    return make_decode_inputs(B=1, n_q=S, seq_lens=[S], H_I=64, d_I=128, topk=2048,
                              H=128, seed=seed, w_sigma=1.0 / 8.0,
                              with_attention=with_attention)


def ragged_paged_decode(seed=1005, B=32, lo=4096, hi=131072, block_size=64,
                        with_attention=True):
    """B sequences with lengths ~ U[lo, hi], one query token each, both caches
    paged in 64-token blocks through a shuffled block table."""
    rng = _rng(seed + 7919)
    lens = rng.integers(lo, hi + 1, size=B)
    return make_decode_inputs(B=B, n_q=1, seq_lens=lens, H_I=64, d_I=128, topk=2048,
                              H=128, seed=seed, w_sigma=1.0 / 8.0, block_size=block_size,
                              max_L=hi, with_attention=with_attention)


# ----------------------------------------------------------------------------
# One decode step of DeepSeek Indexer Attention (MLA Prolog + Indexer Prolog
# + Lightning Indexer + sparse attention)
# ----------------------------------------------------------------------------
@dataclasses.dataclass
class DiaInputs:
    """The decode batch and the two prologs' inputs of one DIA step.  The
    Indexer Prolog takes the MLA Prolog's hidden states x (prolog.x is
    mla.x) and, at run time, the MLA Prolog's q_lora / q_lora_scale (the
    prolog's own q_lora fields are placeholders of the right shape); the
    attention takes the MLA Prolog's query and the latent cache its KV rows
    go to (decode.q_attn is unused)."""
    decode: DecodeInputs
    mla: MlaInputs
    prolog: PrologInputs


def dia_decode(B=4, n_q=2, L=65536, seed=3002, H=128, K_q=1536, D_x=7168):
    """The DIA step at the headline decode shape: B=4 sequences of L keys,
    MTP1 (2 query tokens each at L-2, L-1), whose new keys and latent rows go
    to those two positions of each sequence."""
    inp = make_decode_inputs(B=B, n_q=n_q, seq_lens=[L] * B, H_I=64, d_I=128, topk=2048, H=H, seed=seed,
                             w_sigma=1.0 / 8.0)
    slot = (inp.seq_of_token.astype(np.int64) * inp.max_L + inp.pos).astype(np.int64)
    mla = make_mla_inputs(inp.T, inp.pos, slot, seed=seed + 1, H=H, K_q=K_q, D_x=D_x, max_pos=L)
    pro = make_prolog_inputs(T=inp.T, pos=inp.pos, slot=slot, seed=seed + 2, K_q=K_q, D_x=D_x, max_pos=L)
    pro.x = mla.x
    return DiaInputs(decode=inp, mla=mla, prolog=pro)

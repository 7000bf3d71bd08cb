"""Plain, slow CPU oracle of the DeepSeek Sparse Attention decode hot path.

TEST INFRASTRUCTURE ONLY: used by the tests, the smoke check and the CPU
baseline of the benchmark; the CUDA path never imports it.

Everything is float64 unless a page fixes a precision.  Page citations name
the page and its section:

* [V4-TileLang] "NPU DeepSeek-V4 TileLang算子开发实践" (TileLang-Ascend
  DeepSeek-V4 operators): sections Sparse Flash Attention (steps 1-8),
  Int8 General Matrix Multiplication (steps 1-4), Activation Quantization
  (steps 1-4).
* [V3.2-PyPTO] "NPU DeepSeek-V3.2-Exp PyPTO 融合算子开发优化实践" (PyPTO
  fused operators): sections Indexer Prolog (the Indexer Q, Indexer Cache
  and Indexer Weight formulas and the quantisation strategy paragraph),
  Deepseek Indexer Attention, Lightning Indexer.

Readings taken where the pages are silent or garbled are stated at each
function.  Pins: tests/test_oracle_pins.py.
"""
from __future__ import annotations

import numpy as np

F64 = np.float64

__all__ = [
    "bf16_bits_to_f64", "sylvester_hadamard", "hadamard_rows", "dynamic_quant",
    "int8_gemm_dequant", "int8_gemm", "act_quant", "rope", "layer_norm", "indexer_prolog",
    "indexer_dots", "indexer_scores_token", "topk_indices",
    "sparse_attention_token", "sparse_attention", "cache_rows", "logical_rows", "mhc",
    "rms_norm", "mla_q", "mla_kv", "mla_prolog",
]


def bf16_bits_to_f64(bits) -> np.ndarray:
    """Decode raw bf16 bit patterns (uint16) to float64 exactly."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(F64)


# ----------------------------------------------------------------------------
# Hadamard transform  [V3.2-PyPTO §Indexer Prolog: "the Hadamard transform is
# a right-multiplication by hadamard_q / hadamard_k"]
# ----------------------------------------------------------------------------
def sylvester_hadamard(n: int) -> np.ndarray:
    """Unscaled Sylvester Hadamard matrix of order n (a power of two):
    H_1 = [1], H_2m = [[H_m, H_m], [H_m, -H_m]] (natural order).
    Reading: the pages give no order or scale; Sylvester natural order with
    a 1/sqrt(n) scale (orthonormal) is used."""
    assert n >= 1 and n & (n - 1) == 0
    h = np.ones((1, 1), dtype=F64)
    while h.shape[0] < n:
        h = np.block([[h, h], [h, -h]])
    return h


def hadamard_rows(x: np.ndarray) -> np.ndarray:
    """x @ (H_n / sqrt(n)) over the last axis, as an explicit matrix product."""
    n = x.shape[-1]
    return np.asarray(x, dtype=F64) @ (sylvester_hadamard(n) / np.sqrt(n))


# ----------------------------------------------------------------------------
# DynamicQuant  [V4-TileLang §Activation Quantization steps 1-3;
# V3.2-PyPTO §Indexer Prolog: per-token-head int8, FP16 dequant factors]
# ----------------------------------------------------------------------------
def dynamic_quant(x: np.ndarray):
    """Symmetric int8 quantisation of each row (last axis).

    Steps as the Activation Quantization section orders them, in fp32 as it
    states: (1) take |x| in fp32 and its row maximum; (2) scale = max / 127
    (round_scale=False); (3) y = round(clamp(x / scale, -127, 127)).
    Readings: the scale is stored as FP16 (V3.2-PyPTO) and the division uses
    that stored FP16 value, so that code * scale is exactly the dequantised
    value a consumer sees; rounding is half-to-even; a row whose stored
    scale is 0 gets all-zero codes.
    Returns (codes int8, scale fp16)."""
    x32 = np.asarray(x, dtype=F64).astype(np.float32)
    amax = np.max(np.abs(x32), axis=-1)
    s32 = amax / np.float32(127.0)
    s16 = s32.astype(np.float16)
    sdiv = s16.astype(np.float32)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        y = x32 / sdiv
    y = np.clip(y, np.float32(-127.0), np.float32(127.0))
    codes = np.where(sdiv > 0, np.rint(y), np.float32(0.0))
    return codes.astype(np.int8), s16


def act_quant(x_bits: np.ndarray, round_scale: bool = False):
    """The standalone Activation Quantization operator of [V4-TileLang
    §Activation Quantization] steps 1-4, on bf16 input (raw bits [M, N]).

    (1) |x| in fp32 and its maximum per row (reading: "per column" in the
    text, but the scale is indexed by row; one scale per row of N values,
    as for the prolog's per-(token, head) rows); (2) scale = max / 127 in
    fp32, and with round_scale the power of two at or above it (reading:
    rounding up keeps |x / scale| <= 127); (3) y = round(clamp(x / scale,
    -127, 127)), half to even, the division in fp32 (the page's precision,
    and the one the quantiser's decision is taken in); the fp16 -> int8
    casts of the page are exact for these integers; (4) both written back,
    the scale as fp32.  A row of zeros gets scale 0 and codes 0.
    Returns (codes int8 [M, N], scale fp32 [M])."""
    x32 = bf16_bits_to_f64(x_bits).astype(np.float32)
    amax = np.max(np.abs(x32), axis=-1)
    s = amax / np.float32(127.0)
    if round_scale:
        m, e = np.frexp(s)  # s = m * 2^e, m in [0.5, 1) (s > 0)
        up = np.where(m == 0.5, e - 1, e).astype(np.int32)
        s = np.where(s > 0, np.ldexp(np.float32(1.0), up), np.float32(0.0)).astype(np.float32)
    sd = s[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        y = x32 / sd
    y = np.clip(y, np.float32(-127.0), np.float32(127.0))
    codes = np.where(sd > 0, np.rint(y), np.float32(0.0))
    return codes.astype(np.int8), s.astype(np.float32)


# ----------------------------------------------------------------------------
# Int8 GEMM + dequant  [V4-TileLang §Int8 GEMM steps 1-3]
# ----------------------------------------------------------------------------
def int8_gemm_dequant(a: np.ndarray, a_scale: np.ndarray, b: np.ndarray,
                      b_scale: np.ndarray) -> np.ndarray:
    """C[i, j] = (sum_k a[i,k] * b[j,k]) * a_scale[i] * b_scale[j].

    a int8 [M, K] with a_scale [M]; b int8 [N, K] (K-major, as the page's
    b_int8 [N, K]) with b_scale [N].  The integer sum is exact (a float64
    matmul of int8 values is exact: every partial sum is an integer far
    below 2^53); the dequant is float64 (reading: the fused prolog keeps full
    precision up to the quantiser, no fp16 output cast)."""
    acc = np.asarray(a, dtype=F64) @ np.asarray(b, dtype=F64).T
    return acc * np.asarray(a_scale, dtype=F64)[:, None] * np.asarray(b_scale, dtype=F64)[None, :]


def int8_gemm(a: np.ndarray, a_scale: np.ndarray, b: np.ndarray, b_scale: np.ndarray) -> np.ndarray:
    """The standalone Int8 GEMM operator of [V4-TileLang §Int8 General Matrix
    Multiplication] steps 1-4: the exact int32 product, dequantised by the
    row scale of a and of b, and cast to the target type (fp16, the page's
    example), rounding to nearest even.  Returns fp16 [M, N]."""
    return int8_gemm_dequant(a, a_scale, b, b_scale).astype(np.float16)


# ----------------------------------------------------------------------------
# RoPE  [V3.2-PyPTO §Indexer Prolog, Indexer Q and Indexer Cache formulas]
# ----------------------------------------------------------------------------
def rope(x: np.ndarray, pos: np.ndarray, cos_tab: np.ndarray, sin_tab: np.ndarray,
         d_rope: int, interleaved: bool = False) -> np.ndarray:
    """Rotate dims [0, d_rope) of x [T, ..., d] by angle(pos[t], i).

    Readings (the pages give none of these): the first d_rope dims rotate,
    the rest pass through; pairs are (i, i + d_rope/2) ("half split"), or
    (2i, 2i+1) when interleaved; cos/sin come from the given tables
    [max_pos, d_rope/2]; pair (a, b) maps to (a cos - b sin, b cos + a sin)."""
    x = np.asarray(x, dtype=F64)
    out = x.copy()
    half = d_rope // 2
    pos = np.asarray(pos, dtype=np.int64)
    extra = (1,) * (x.ndim - 2)
    c = np.asarray(cos_tab, dtype=F64)[pos].reshape((x.shape[0],) + extra + (half,))
    s = np.asarray(sin_tab, dtype=F64)[pos].reshape((x.shape[0],) + extra + (half,))
    i = np.arange(half)
    ia, ib = (2 * i, 2 * i + 1) if interleaved else (i, i + half)
    xa, xb = x[..., ia], x[..., ib]
    out[..., ia] = xa * c - xb * s
    out[..., ib] = xb * c + xa * s
    return out


def layer_norm(x: np.ndarray, gamma, beta, eps: float) -> np.ndarray:
    """LayerNorm over the last axis [V3.2-PyPTO §Indexer Prolog, Indexer Cache
    formula].  Reading: biased variance, eps inside the square root, affine
    gamma/beta."""
    x = np.asarray(x, dtype=F64)
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)
    return (x - mu) / np.sqrt(var + eps) * np.asarray(gamma, F64) + np.asarray(beta, F64)


# ----------------------------------------------------------------------------
# Indexer Prolog  [V3.2-PyPTO §Indexer Prolog, the three formulas]
# ----------------------------------------------------------------------------
def indexer_prolog(p, k_cache=None, k_scale_cache=None):
    """The three independent streams of the Indexer Prolog.

      q, q_scale = DynamicQuant(Hadamard(RoPE(DeQuant(q_lora . w_qb))))
      k, k_scale = DynamicQuant(Hadamard(RoPE(LayerNorm(x . w_k))))
      weight     = (x . w_proj) * w_scale

    ``p`` carries the fields of workloads.PrologInputs (plain arrays).  q is
    quantised per (token, head), k per token.  When caches are given, row
    slot[t] >= 0 receives k[t] / k_scale[t].  Returns a dict with q [T,H,D]
    int8, q_scale [T,H] fp16, k [T,D] int8, k_scale [T] fp16 and, if w_proj
    is given, w [T,H] fp32 (reading: fp32 output, not the page's FP16)."""
    T, H, D = p.T, p.H_I, p.d_I
    qf = int8_gemm_dequant(p.q_lora, p.q_lora_scale, p.w_qb, p.w_qb_scale).reshape(T, H, D)
    qr = rope(qf, p.pos, p.rope_cos, p.rope_sin, p.d_rope, bool(p.rope_interleaved))
    q, q_scale = dynamic_quant(hadamard_rows(qr))

    x = bf16_bits_to_f64(p.x)
    kf = x @ bf16_bits_to_f64(p.w_k).T
    kn = layer_norm(kf, p.ln_gamma, p.ln_beta, p.ln_eps)
    kr = rope(kn[:, None, :], p.pos, p.rope_cos, p.rope_sin, p.d_rope,
              bool(p.rope_interleaved))[:, 0, :]
    k, k_scale = dynamic_quant(hadamard_rows(kr))

    out = {"q": q, "q_scale": q_scale, "k": k, "k_scale": k_scale,
           "q_prequant": hadamard_rows(qr), "k_prequant": hadamard_rows(kr)}
    if p.w_proj is not None:
        out["w"] = ((x @ bf16_bits_to_f64(p.w_proj).T) * float(p.w_scale)).astype(np.float32)
    if k_cache is not None:
        for t in range(T):
            if p.slot[t] >= 0:
                k_cache[p.slot[t]] = k[t]
                k_scale_cache[p.slot[t]] = k_scale[t]
    return out


# ----------------------------------------------------------------------------
# Lightning Indexer  [V3.2-PyPTO §Lightning Indexer: int8 q against the C8
# key cache, then a per-query TopK; §Indexer Prolog for the scale types]
# ----------------------------------------------------------------------------
def cache_rows(inp, b: int, s) -> np.ndarray:
    """Physical cache rows of the keys at logical positions s of sequence b:
    b * max_L + s for a contiguous [B, max_L, .] cache, else block
    block_table[b, s // block_size], row s % block_size of that block
    (reading: the paged-cache addressing of the PagedAttention-style block
    table that the ragged workload uses; the pages give block sizes only)."""
    s = np.asarray(s, dtype=np.int64)
    if inp.block_table is None:
        return b * inp.max_L + s
    blk = np.asarray(inp.block_table)[b, s // inp.block_size].astype(np.int64)
    return blk * inp.block_size + s % inp.block_size


def logical_rows(inp, b: int, n: int) -> np.ndarray:
    """Physical cache rows of keys 0..n-1 of sequence b."""
    return cache_rows(inp, b, np.arange(n, dtype=np.int64))


def indexer_dots(q_tok: np.ndarray, keys: np.ndarray) -> np.ndarray:
    """Exact int64 dots [H, n] = q_tok[h] . keys[s] (int8 x int8)."""
    d = np.asarray(q_tok, dtype=F64) @ np.asarray(keys, dtype=F64).T
    return d.astype(np.int64)


def indexer_scores_token(q_tok, q_scale_tok, w_tok, keys, key_scale, pos_t: int):
    """I[s] = ks[s] * sum_h w[h] * qs[h] * ReLU(q[h] . K[s]) for s <= pos_t,
    -inf for s > pos_t.

    Reading: the score is sum_h w[h] * ReLU(q_h . k_s) on the dequantised
    operands; as both scales are non-negative, ReLU(qs*ks*dot) =
    qs*ks*ReLU(dot), which is the factorisation written here."""
    dots = indexer_dots(q_tok, keys).astype(F64)
    coef = np.asarray(w_tok, F64) * np.asarray(q_scale_tok, F64)
    I = np.asarray(key_scale, F64) * (coef[:, None] * np.maximum(dots, 0.0)).sum(axis=0)
    I[np.arange(keys.shape[0]) > pos_t] = -np.inf
    return I


def topk_indices(scores: np.ndarray, n_valid: int, k: int) -> np.ndarray:
    """Indices of the k largest scores among positions [0, n_valid), by a
    full sort (score descending, then index ascending); if fewer than k are
    valid, all valid positions then -1 (the unused-slot marker of
    [V4-TileLang §Sparse Flash Attention step 2])."""
    s = np.asarray(scores, dtype=F64)[:n_valid]
    order = np.lexsort((np.arange(n_valid), -s))
    sel = order[:k]
    out = np.full(k, -1, dtype=np.int64)
    out[:sel.size] = sel
    return out


# ----------------------------------------------------------------------------
# Sparse Flash Attention  [V4-TileLang §Sparse Flash Attention steps 2-6, 8]
# ----------------------------------------------------------------------------
def sparse_attention_token(q_tok: np.ndarray, rows: np.ndarray, scale: float, d_v: int, sink=None):
    """Softmax attention of q_tok [H, d_qk] over the selected latent rows
    [n, d_qk] (value = first d_v dims).  Returns (out [H, d_v], lse [H]),
    lse = natural log of sum_j exp(scale * q.k_j).  No rows: out 0, lse -inf.
    Reading: the online softmax of the page computes exactly this.

    sink [H] (natural-log units) or None: the attention sink of
    [V4-TileLang §Sparse Flash Attention] step 7, whose operator the page
    prints garbled.  Read as one extra term exp(sink[h]) in each head's
    softmax denominator, i.e. a virtual key with logit sink[h] and a zero
    value: out = sum_j e^{s_j} v_j / (sum_j e^{s_j} + e^{sink}), lse =
    log(sum_j e^{s_j} + e^{sink}); with no rows, out 0 and lse = sink."""
    q = np.asarray(q_tok, dtype=F64)
    H = q.shape[0]
    sk = None if sink is None else np.asarray(sink, dtype=F64).reshape(H)
    if rows.shape[0] == 0:
        return np.zeros((H, d_v)), (np.full(H, -np.inf) if sk is None else sk.copy())
    kv = np.asarray(rows, dtype=F64)
    S = scale * (q @ kv.T)
    m = S.max(axis=1, keepdims=True)
    if sk is not None:
        m = np.maximum(m, sk[:, None])
    p = np.exp(S - m)
    l = p.sum(axis=1, keepdims=True)
    if sk is not None:
        l = l + np.exp(sk[:, None] - m)
    out = (p @ kv[:, :d_v]) / l
    return out, (m + np.log(l))[:, 0]


def sparse_attention(inp, topk_idx: np.ndarray, tokens=None, sink=None):
    """Sparse attention for the given tokens of a workloads.DecodeInputs-like
    object; index -1 selects nothing; optional per-head sink [H] (see
    sparse_attention_token).  Returns (out [n_tok, H, d_v], lse)."""
    if tokens is None:
        tokens = range(inp.T)
    outs, lses = [], []
    for t in tokens:
        idx = np.asarray(topk_idx[t], dtype=np.int64)
        idx = idx[idx >= 0]
        b = int(inp.seq_of_token[t])
        phys = cache_rows(inp, b, idx) if idx.size else np.zeros(0, np.int64)
        rows = bf16_bits_to_f64(inp.kv_cache[phys])
        o, l = sparse_attention_token(bf16_bits_to_f64(inp.q_attn[t]), rows, inp.scale, inp.d_v, sink)
        outs.append(o)
        lses.append(l)
    return np.stack(outs), np.stack(lses)


# ----------------------------------------------------------------------------
# Manifold-Constrained Hyper-Connections  [V4-TileLang §Manifold-Constrained
# Hyper-Connections, steps 1-5]
# ----------------------------------------------------------------------------
def mhc(mixes: np.ndarray, hc_scale: np.ndarray, hc_base: np.ndarray, hc: int, iters: int, eps: float):
    """pre [n, hc], post [n, hc], comb [n, hc, hc] from mixes [n, hc*(2+hc)].

    Readings where the page is garbled or silent: a row of mixes holds the
    pre part (hc values), the post part (hc) and the comb matrix (hc x hc,
    row-major) - the only split that makes the page's row and column
    normalisations of comb meaningful (it prints comb as [n, hc]); hc_scale
    [3] scales the three parts in that order (step 1: mixes * scale +
    hc_base); pre = sigmoid(.) + eps and post = 2 sigmoid(.) (steps 2-3,
    whose printed operands are garbled); comb = softmax over each row + eps
    (step 4), then divided by its column sums + eps, then `iters` rounds of
    row sums + eps and column sums + eps (step 5, in the page's order)."""
    x = np.asarray(mixes, dtype=F64)
    n = x.shape[0]
    sc = np.concatenate([np.full(hc, hc_scale[0]), np.full(hc, hc_scale[1]), np.full(hc * hc, hc_scale[2])])
    z = x * sc + np.asarray(hc_base, dtype=F64)
    sig = lambda v: 1.0 / (1.0 + np.exp(-v))
    pre = sig(z[:, :hc]) + eps
    post = 2.0 * sig(z[:, hc:2 * hc])
    c = z[:, 2 * hc:].reshape(n, hc, hc)
    c = np.exp(c - c.max(axis=-1, keepdims=True))
    c = c / c.sum(axis=-1, keepdims=True) + eps
    c = c / (c.sum(axis=-2, keepdims=True) + eps)
    for _ in range(iters):
        c = c / (c.sum(axis=-1, keepdims=True) + eps)
        c = c / (c.sum(axis=-2, keepdims=True) + eps)
    return pre, post, c



# ----------------------------------------------------------------------------
# MLA Prolog  [V3.2-PyPTO §Deepseek Indexer Attention: the first of the four
# parts; it feeds q_lora to the Indexer Prolog (§Indexer Prolog, the Indexer
# Q formula) and q plus the latent KV rows to Sparse Flash Attention]
# ----------------------------------------------------------------------------
MLA_D_C, MLA_D_N, MLA_D_R = 512, 128, 64  # latent, no-position and rotary dims


def rms_norm(x: np.ndarray, gamma, eps: float) -> np.ndarray:
    """x / sqrt(mean(x^2) + eps) * gamma over the last axis (reading: the
    RMS normalisation of the MLA latents, eps inside the root)."""
    x = np.asarray(x, dtype=F64)
    return x / np.sqrt((x * x).mean(axis=-1, keepdims=True) + eps) * np.asarray(gamma, F64)


def mla_q(q_lora, q_lora_scale, w_uq, w_uq_scale, w_uk, H: int, pos, cos_tab, sin_tab,
          interleaved: bool = False) -> np.ndarray:
    """Query of the sparse MLA attention from the quantised query latent.

    u = DeQuant(q_lora . w_uq) [T, H, d_n + d_r] (the Indexer Q formula's
    int8 GEMM and dequant, the same q_lora feeding both); per head the
    first d_n = 128 dims are multiplied into the latent space by w_uk[h]
    [d_n, d_c] (q_abs = u_nope . w_uk[h], so that q_abs . c = u_nope .
    (w_uk[h] c) for a latent row c), the last d_r = 64 dims are rotated.
    Returns float64 [T, H, d_c + d_r] = [q_abs | RoPE(u_rope)]."""
    T = np.asarray(q_lora).shape[0]
    u = int8_gemm_dequant(q_lora, q_lora_scale, w_uq, w_uq_scale).reshape(T, H, MLA_D_N + MLA_D_R)
    q_abs = np.einsum("thn,hnc->thc", u[..., :MLA_D_N], np.asarray(w_uk, dtype=F64))
    q_pe = rope(u[..., MLA_D_N:], pos, cos_tab, sin_tab, MLA_D_R, interleaved)
    return np.concatenate([q_abs, q_pe], axis=-1)


def mla_kv(x, w_dkv, gamma_kv, eps: float, pos, cos_tab, sin_tab, interleaved: bool = False) -> np.ndarray:
    """Latent KV row of each token: c = x . w_dkv^T [T, d_c + d_r]; the first
    d_c = 512 dims RMS-normalised (gamma_kv), the last d_r = 64 rotated.
    Returns float64 [T, d_c + d_r]."""
    c = np.asarray(x, dtype=F64) @ np.asarray(w_dkv, dtype=F64).T
    lat = rms_norm(c[:, :MLA_D_C], gamma_kv, eps)
    pe = rope(c[:, None, MLA_D_C:], pos, cos_tab, sin_tab, MLA_D_R, interleaved)[:, 0, :]
    return np.concatenate([lat, pe], axis=-1)


def mla_prolog(p, kv_cache=None):
    """The MLA Prolog of one step of query tokens.

    The pages give it no formula.  Reading (the plainest one that its
    neighbours support): the query latent is c_q = RMSNorm(x . w_dq^T) *
    gamma_q [T, K_q]; its per-token DynamicQuant (the Indexer Prolog's
    quantiser, one fp16 scale per token) is the int8 q_lora with fp16 scale
    that the Indexer Q formula consumes; the same q_lora gives the
    attention query through `mla_q` (w_uq int8 with per-channel fp16
    scales, w_uk bf16 absorbed, 576 = 512 + 64 dims as the attention's
    latent rows); the latent KV row comes from `mla_kv` and goes to
    kv_cache[slot[t]] (slot -1: not written).  x, w_dq, w_dkv and w_uk are
    raw bf16 bits.  Returns a dict: c_q float64 [T, K_q], q_lora int8
    [T, K_q], q_lora_scale fp16 [T], q float64 [T, H, 576], kv float64
    [T, 576]."""
    x = bf16_bits_to_f64(p.x)
    c_q = rms_norm(x @ bf16_bits_to_f64(p.w_dq).T, p.gamma_q, p.rms_eps)
    q_lora, q_lora_scale = dynamic_quant(c_q)
    inter = bool(p.rope_interleaved)
    q = mla_q(q_lora, q_lora_scale, p.w_uq, p.w_uq_scale, bf16_bits_to_f64(p.w_uk), p.H, p.pos,
              p.rope_cos, p.rope_sin, inter)
    kv = mla_kv(x, bf16_bits_to_f64(p.w_dkv), p.gamma_kv, p.rms_eps, p.pos, p.rope_cos, p.rope_sin, inter)
    if kv_cache is not None:
        for t in range(p.T):
            if p.slot[t] >= 0:
                kv_cache[p.slot[t]] = kv[t]
    return {"c_q": c_q, "q_lora": q_lora, "q_lora_scale": q_lora_scale, "q": q, "kv": kv}

"""Pins of the CPU oracle to facts outside itself: closed forms, library
routines, brute force and a hand-worked case.  CPU only."""
import math
import os

import numpy as np
import pytest
import scipy.linalg
import scipy.special
import torch

import oracle as O
from sparse_attention_prolog_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(12345)


# ---------------------------------------------------------------- Hadamard
@pytest.mark.parametrize("n", [1, 2, 4, 8, 16, 64, 128, 256])
def test_hadamard_is_sylvester_and_orthogonal(n):
    H = O.sylvester_hadamard(n)
    np.testing.assert_array_equal(H, scipy.linalg.hadamard(n))  # Sylvester natural order
    np.testing.assert_array_equal(H @ H, n * np.eye(n))         # H.H = n.I (H symmetric)


def _fwht(v):
    """Independent recursive fast Walsh-Hadamard butterfly (natural order)."""
    v = list(v)
    if len(v) == 1:
        return v
    h = len(v) // 2
    a, b = _fwht(v[:h]), _fwht(v[h:])
    return [x + y for x, y in zip(a, b)] + [x - y for x, y in zip(a, b)]


def test_hadamard_rows_matches_butterfly_and_keeps_norm():
    x = rng.standard_normal((3, 128))
    y = O.hadamard_rows(x)
    ref = np.array([_fwht(r) for r in x]) / math.sqrt(128)
    np.testing.assert_allclose(y, ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(np.linalg.norm(y, axis=1), np.linalg.norm(x, axis=1), rtol=1e-12)
    e0 = np.zeros(128); e0[0] = 1
    np.testing.assert_allclose(O.hadamard_rows(e0), np.full(128, 1 / math.sqrt(128)), atol=1e-15)


# ---------------------------------------------------------- DynamicQuant
def test_quant_argmax_maps_to_127_and_error_bound():
    x = rng.standard_normal((50, 128)) * rng.uniform(0.01, 10, size=(50, 1))
    c, s = O.dynamic_quant(x)
    assert c.dtype == np.int8 and s.dtype == np.float16
    am = np.argmax(np.abs(x), axis=1)
    np.testing.assert_array_equal(np.abs(c[np.arange(50), am]), 127)
    np.testing.assert_array_equal(np.sign(c[np.arange(50), am]), np.sign(x[np.arange(50), am]))
    sf = s.astype(np.float64)[:, None]
    err = np.abs(c * sf - x)
    # half a step, plus the clamp of |x| <= amax against 127*fp16(amax/127)
    assert (err <= sf * 0.5 + np.abs(x).max(1, keepdims=True) * 2.0 ** -10).all()
    assert np.abs(c).max() <= 127


def test_quant_codes_are_nearest_on_the_stored_scale_grid():
    """Away from the clamp, code * scale is the point of the stored fp16
    scale's grid nearest to x, to within the fp32 rounding of x and of
    x / scale (1.5e-5 of a step at |code| <= 127): the division uses the
    stored scale, not absmax / 127 before its rounding to fp16."""
    x = rng.standard_normal((200, 128)) * rng.uniform(0.01, 10, size=(200, 1))
    c, s = O.dynamic_quant(x)
    sf = np.broadcast_to(s.astype(np.float64)[:, None], x.shape)
    inside = np.abs(x) <= 126.5 * sf
    err = np.abs(c * sf - x)
    assert (err[inside] <= sf[inside] * (0.5 + 3e-5)).all()


def test_quant_zero_row_and_exact_grid():
    c, s = O.dynamic_quant(np.zeros((2, 64)))
    assert (c == 0).all() and (s == 0).all()
    s16 = np.float16(0.0371)
    codes = rng.integers(-127, 128, size=128)
    codes[5] = -127
    x = codes.astype(np.float64) * float(s16)
    c, s = O.dynamic_quant(x[None])
    assert s[0] == s16
    np.testing.assert_array_equal(c[0], codes)


def test_quant_rounds_half_to_even():
    # scale 1.0 exactly (amax 127): x / scale lands on .5 ties
    x = np.array([127.0, 2.5, 3.5, -2.5, -3.5, 0.5, -0.5, 1.5] + [0.0] * 8)
    c, s = O.dynamic_quant(x[None])
    assert float(s[0]) == 1.0
    np.testing.assert_array_equal(c[0, :8], [127, 2, 4, -2, -4, 0, 0, 2])


# ------------------------------------------------------------ Int8 GEMM
def test_int8_gemm_brute_force_and_closed_form():
    a = rng.integers(-128, 128, size=(3, 7)).astype(np.int8)
    b = rng.integers(-128, 128, size=(5, 7)).astype(np.int8)
    sa = np.array([1.0, 0.5, 2.0], np.float16)
    sb = np.array([1.0, 0.25, 3.0, 0.125, 1.5], np.float16)
    got = O.int8_gemm_dequant(a, sa, b, sb)
    for i in range(3):
        for j in range(5):
            acc = sum(int(a[i, k]) * int(b[j, k]) for k in range(7))
            assert got[i, j] == acc * float(sa[i]) * float(sb[j])
    K = 1536
    full = O.int8_gemm_dequant(np.full((2, K), 127, np.int8), np.ones(2, np.float16),
                               np.full((3, K), 127, np.int8), np.ones(3, np.float16))
    assert (full == 16129 * K).all()
    neg = O.int8_gemm_dequant(np.full((1, K), -128, np.int8), np.ones(1, np.float16),
                              np.full((1, K), -128, np.int8), np.ones(1, np.float16))
    assert neg[0, 0] == 16384 * K


# ------------------------------------------------------------------ RoPE
def _tables(max_pos, d_rope, base=10000.0):
    from sparse_attention_prolog_gb300.workloads import rope_tables
    return rope_tables(max_pos, d_rope, base)


@pytest.mark.parametrize("interleaved", [False, True])
def test_rope_matches_complex_rotation(interleaved):
    T, H, d, dr = 5, 3, 128, 64
    cos, sin = _tables(70000, dr)
    pos = np.array([0, 1, 17, 4095, 65535])
    x = rng.standard_normal((T, H, d))
    y = O.rope(x, pos, cos, sin, dr, interleaved)
    half = dr // 2
    theta = 10000.0 ** (-(2.0 * np.arange(half)) / dr)
    ia = 2 * np.arange(half) if interleaved else np.arange(half)
    ib = ia + 1 if interleaved else ia + half
    z = (x[..., ia] + 1j * x[..., ib]) * np.exp(1j * pos[:, None, None] * theta)
    # tables are fp32-rounded: compare within fp32 angle rounding
    np.testing.assert_allclose(y[..., ia], z.real, atol=2e-6 * np.abs(x).max())
    np.testing.assert_allclose(y[..., ib], z.imag, atol=2e-6 * np.abs(x).max())
    np.testing.assert_array_equal(y[..., dr:], x[..., dr:])
    np.testing.assert_array_equal(y[0], x[0])  # pos 0 is the identity
    np.testing.assert_allclose(np.hypot(y[..., ia], y[..., ib]), np.hypot(x[..., ia], x[..., ib]),
                               rtol=1e-6)


def test_rope_conventions_agree_after_permutation():
    cos, sin = _tables(64, 64)
    x = rng.standard_normal((4, 2, 128))
    pos = np.array([3, 9, 27, 63])
    perm = np.concatenate([np.stack([np.arange(32), np.arange(32) + 32], 1).reshape(-1),
                           np.arange(64, 128)])  # half-split order -> interleaved order
    y_half = O.rope(x, pos, cos, sin, 64, False)
    y_int = O.rope(x[..., perm], pos, cos, sin, 64, True)
    np.testing.assert_allclose(y_int, y_half[..., perm], rtol=0, atol=1e-14)


# ------------------------------------------------------------- LayerNorm
def test_layer_norm_matches_torch_and_closed_form():
    x = rng.standard_normal((6, 128)) * 3 + 1
    g = rng.standard_normal(128)
    b = rng.standard_normal(128)
    ref = torch.nn.functional.layer_norm(torch.from_numpy(x), (128,), torch.from_numpy(g),
                                         torch.from_numpy(b), eps=1e-6).numpy()
    np.testing.assert_allclose(O.layer_norm(x, g, b, 1e-6), ref, rtol=1e-12, atol=1e-12)
    y = O.layer_norm(x, np.ones(128), np.zeros(128), 1e-6)
    v = x.var(axis=1)
    np.testing.assert_allclose(y.mean(1), 0, atol=1e-12)
    np.testing.assert_allclose(y.var(1), v / (v + 1e-6), rtol=1e-12)


# ---------------------------------------------------------- Indexer Prolog
def _prolog_fixture(T=1, H=2, D=128, Kq=16, Dx=32, pos=(0,)):
    from sparse_attention_prolog_gb300.workloads import PrologInputs, f32_to_bf16_bits
    cos, sin = _tables(max(pos) + 1, 64)
    return PrologInputs(
        T=T, H_I=H, d_I=D, d_rope=64,
        q_lora=np.zeros((T, Kq), np.int8), q_lora_scale=np.ones(T, np.float16),
        w_qb=np.zeros((H * D, Kq), np.int8), w_qb_scale=np.ones(H * D, np.float16),
        x=f32_to_bf16_bits(np.zeros((T, Dx), np.float32)),
        w_k=f32_to_bf16_bits(np.zeros((D, Dx), np.float32)),
        ln_gamma=np.ones(D, np.float32), ln_beta=np.zeros(D, np.float32), ln_eps=1e-6,
        w_proj=None, w_scale=1.0, pos=np.array(pos, np.int32), rope_cos=cos, rope_sin=sin,
        rope_interleaved=0, slot=np.full(T, -1, np.int64))


def test_prolog_q_one_hot_gives_hadamard_row_codes():
    """q_lora . w_qb = one-hot e_j per head -> Hadamard row j -> codes 127*H[j]."""
    from sparse_attention_prolog_gb300.workloads import f32_to_bf16_bits
    p = _prolog_fixture()
    p.q_lora[0, 3] = 5
    p.q_lora_scale[0] = np.float16(0.5)
    js = [70, 5]       # head 0: a pass-through dim; head 1: a rotated dim at pos 0
    for h, j in enumerate(js):
        p.w_qb[h * 128 + j, 3] = 2
        p.w_qb_scale[h * 128 + j] = np.float16(0.2)
    p.x = f32_to_bf16_bits(np.zeros((1, 32), np.float32))
    r = O.indexer_prolog(p)
    H = scipy.linalg.hadamard(128)
    amp = 5 * 2 * 0.5 * float(np.float16(0.2)) / math.sqrt(128)
    for h, j in enumerate(js):
        np.testing.assert_array_equal(r["q"][0, h], 127 * H[j])
        expect = np.float16(np.float32(amp) / np.float32(127))
        assert r["q_scale"][0, h] == expect


def test_prolog_k_alternating_gives_single_code():
    """x . w_k = alternating +-a -> LayerNorm -> +-1 -> Hadamard -> sqrt(128) e_1."""
    from sparse_attention_prolog_gb300.workloads import f32_to_bf16_bits
    p = _prolog_fixture(Dx=4)
    p.x = f32_to_bf16_bits(np.array([[3.0, 0, 0, 0]], np.float32))
    wk = np.zeros((128, 4), np.float32)
    wk[:, 0] = np.where(np.arange(128) % 2 == 0, 1.0, -1.0)
    p.w_k = f32_to_bf16_bits(wk)
    p.ln_eps = 0.0
    r = O.indexer_prolog(p)
    expect = np.zeros(128, np.int64); expect[1] = 127
    np.testing.assert_array_equal(r["k"][0], expect)
    assert r["k_scale"][0] == np.float16(np.float32(math.sqrt(128)) / np.float32(127))


def test_prolog_weight_stream_and_cache_write_brute_force():
    from sparse_attention_prolog_gb300.workloads import f32_to_bf16_bits
    p = _prolog_fixture(T=2, Dx=6, pos=(0, 1))
    xv = rng.standard_normal((2, 6)).astype(np.float32)
    wp = rng.standard_normal((2, 6)).astype(np.float32)
    p.x, p.w_proj, p.w_scale = f32_to_bf16_bits(xv), f32_to_bf16_bits(wp), 0.125
    p.slot = np.array([3, -1], np.int64)
    cache = np.full((5, 128), 9, np.int8)
    cs = np.full(5, 7, np.float16)
    r = O.indexer_prolog(p, cache, cs)
    xb = O.bf16_bits_to_f64(p.x)
    wb = O.bf16_bits_to_f64(p.w_proj)
    for t in range(2):
        for h in range(2):
            ref = sum(xb[t, c] * wb[h, c] for c in range(6)) * 0.125
            assert abs(float(r["w"][t, h]) - ref) <= 1e-6 * max(1.0, abs(ref))
    np.testing.assert_array_equal(cache[3], r["k"][0])
    assert cs[3] == r["k_scale"][0]
    assert (cache[[0, 1, 2, 4]] == 9).all() and (cs[[0, 1, 2, 4]] == 7).all()


def test_prolog_cache_rows_take_each_tokens_key():
    """Slots [3, -1, 1]: rows 3 and 1 receive the codes and the scale of
    tokens 0 and 2 (keys in different directions, so different scales);
    token 1 writes nothing."""
    from sparse_attention_prolog_gb300.workloads import f32_to_bf16_bits
    p = _prolog_fixture(T=3, Dx=8, pos=(0, 1, 2))
    r2 = np.random.default_rng(31)
    p.x = f32_to_bf16_bits(r2.standard_normal((3, 8)).astype(np.float32))
    p.w_k = f32_to_bf16_bits(r2.standard_normal((128, 8)).astype(np.float32))
    p.slot = np.array([3, -1, 1], np.int64)
    cache = np.full((5, 128), 9, np.int8)
    cs = np.full(5, 7, np.float16)
    r = O.indexer_prolog(p, cache, cs)
    assert r["k_scale"][0] != r["k_scale"][2]
    for row, t in ((3, 0), (1, 2)):
        np.testing.assert_array_equal(cache[row], r["k"][t])
        assert cs[row] == r["k_scale"][t]
    assert (cache[[0, 2, 4]] == 9).all() and (cs[[0, 2, 4]] == 7).all()


def test_prolog_q_and_k_rotary_relative_position():
    """The Hadamard transform is orthonormal, so the pre-quantisation q . k
    of two tokens is the dot of their rotated vectors: moving both positions
    by the same amount keeps it, moving only one changes it."""
    from sparse_attention_prolog_gb300.workloads import make_prolog_inputs

    def score(pos):
        p = make_prolog_inputs(T=2, pos=pos, slot=[-1, -1], seed=41, H_I=2, d_I=64, K_q=128, D_x=128,
                               with_weights=False, max_pos=64)
        r = O.indexer_prolog(p)
        return np.einsum("hd,d->h", r["q_prequant"][0], r["k_prequant"][1])

    a, b, c = score([5, 20]), score([17, 32]), score([17, 20])
    np.testing.assert_allclose(a, b, rtol=1e-5)
    assert not np.allclose(a, c, rtol=1e-3)


# ------------------------------------------------------- Lightning Indexer
def _read_golden():
    g = {}
    with open(os.path.join(GOLDEN, "indexer_hand_case.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split()
            key = parts[0] + ("_" + parts[1] if parts[0] in ("q", "k", "dots") else "")
            vals = parts[2:] if parts[0] in ("q", "k", "dots") else parts[1:]
            g[key] = [float(v) for v in vals]
    return g


def test_indexer_hand_worked_case():
    g = _read_golden()
    q = np.array([g["q_h0"], g["q_h1"]], np.int8)
    K = np.array([g["k_s0"], g["k_s1"]], np.int8)
    w = np.array(g["w"], np.float32)
    np.testing.assert_array_equal(O.indexer_dots(q, K), [g["dots_h0"], g["dots_h1"]])
    I = O.indexer_scores_token(q, np.ones(2, np.float16), w, K, np.ones(2, np.float16), pos_t=1)
    np.testing.assert_array_equal(I, g["scores"])
    np.testing.assert_array_equal(O.topk_indices(I, 2, 1), g["top1"])
    np.testing.assert_array_equal(O.topk_indices(I, 2, 2), g["top2"])
    I0 = O.indexer_scores_token(q, np.ones(2, np.float16), w, K, np.ones(2, np.float16), pos_t=0)
    np.testing.assert_array_equal(O.topk_indices(I0, 1, 2), g["top2_pos0"])


def _golden_value(tok):
    """A value of the attention golden file: "a/b", "log a/b" or "-inf"."""
    from fractions import Fraction
    if tok == "-inf":
        return -np.inf
    if tok.startswith("log "):
        return float(np.log(float(Fraction(tok[4:]))))
    return float(Fraction(tok))


def test_attention_hand_worked_case():
    g = {}
    with open(os.path.join(GOLDEN, "attention_hand_case.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, rest = line.split(None, 1)
            if key in ("q", "row"):
                name, vals = rest.split(None, 1)
                g.setdefault(key, []).append([float(v) for v in vals.split()])
            elif key == "scale":
                g[key] = _golden_value(rest)
            else:
                name, val = rest.split(None, 1)
                g.setdefault(key, []).append(_golden_value(val))
    q, rows = np.array(g["q"]), np.array(g["row"])
    out, lse = O.sparse_attention_token(q, rows, g["scale"], 1)
    np.testing.assert_allclose(out[:, 0], g["out"], rtol=1e-13)
    np.testing.assert_allclose(lse, g["lse"], rtol=1e-13)
    out, lse = O.sparse_attention_token(q, rows, g["scale"], 1, sink=np.array(g["sink"]))
    np.testing.assert_allclose(out[:, 0], g["out_sink"], rtol=1e-13)
    np.testing.assert_allclose(lse, g["lse_sink"], rtol=1e-13)
    out, lse = O.sparse_attention_token(q, rows[:0], g["scale"], 1, sink=np.array(g["sink"]))
    assert (out == 0).all()
    np.testing.assert_array_equal(lse, g["empty_lse_sink"])


def test_attention_sink_far_above_the_logits():
    """A sink 1000 above every logit takes the whole softmax: the output is
    0 to within e^-999 and lse equals the sink, without overflow (a
    softmax shifted by the logits' max alone would divide by infinity)."""
    q = np.array([[0.0, 1.0]])
    rows = np.array([[2.0, 0.0], [6.0, 1.0]])
    out, lse = O.sparse_attention_token(q, rows, 1.0, 1, sink=np.array([1000.0]))
    assert np.isfinite(out).all() and np.abs(out).max() < 1e-300
    np.testing.assert_allclose(lse, [1000.0], rtol=1e-15)


def test_indexer_scores_brute_force_loops():
    H, D, n = 3, 8, 11
    q = rng.integers(-127, 128, size=(H, D)).astype(np.int8)
    K = rng.integers(-127, 128, size=(n, D)).astype(np.int8)
    qs = rng.uniform(0.01, 0.05, H).astype(np.float16)
    ks = rng.uniform(0.01, 0.05, n).astype(np.float16)
    w = rng.standard_normal(H).astype(np.float32)
    I = O.indexer_scores_token(q, qs, w, K, ks, pos_t=7)
    for s in range(n):
        if s > 7:
            assert I[s] == -np.inf
            continue
        ref = 0.0
        for h in range(H):
            # dequantise both operands first, then ReLU of the real dot
            dot = sum(float(q[h, d]) * float(qs[h]) * float(K[s, d]) * float(ks[s]) for d in range(D))
            ref += float(w[h]) * max(dot, 0.0)
        assert abs(I[s] - ref) <= 1e-12 * max(1.0, abs(ref))
    assert O.indexer_dots(np.full((1, 128), 127, np.int8), np.full((1, 128), -127, np.int8))[0, 0] \
        == -16129 * 128


# ------------------------------------------------------------------ Top-k
def test_topk_against_library_selection():
    s = rng.standard_normal(5000)
    k = 300
    got = O.topk_indices(s, 4000, k)
    ref = np.argpartition(-s[:4000], k)[:k]
    assert set(got.tolist()) == set(ref.tolist())
    assert (np.diff(s[got]) <= 0).all()  # sorted by score, descending
    perm = rng.permutation(4000)
    got_p = O.topk_indices(s[:4000][perm], 4000, k)
    assert set(perm[got_p].tolist()) == set(got.tolist())


def test_topk_short_rows_and_ties():
    s = np.array([1.0, 5.0, 5.0, -2.0, 7.0])
    np.testing.assert_array_equal(O.topk_indices(s, 3, 5), [1, 2, 0, -1, -1])
    np.testing.assert_array_equal(O.topk_indices(s, 5, 2), [4, 1])   # tie 1/2 -> lower index
    np.testing.assert_array_equal(O.topk_indices(s, 0, 3), [-1, -1, -1])


# ------------------------------------------------------- Sparse attention
def _bf16(x):
    from sparse_attention_prolog_gb300.workloads import f32_to_bf16_bits
    return O.bf16_bits_to_f64(f32_to_bf16_bits(x.astype(np.float32)))


def test_attention_equals_dense_masked_sdpa():
    H, L, d, dv, scale = 4, 40, 576, 512, 192 ** -0.5
    q = _bf16(rng.standard_normal((H, d)))
    kv = _bf16(rng.standard_normal((L, d)))
    sel = np.array([3, 17, 0, 39, 22, 8])
    out, lse = O.sparse_attention_token(q, kv[sel], scale, dv)
    mask = torch.zeros(H, L, dtype=torch.bool)
    mask[:, torch.from_numpy(sel)] = True
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[None], torch.from_numpy(kv)[None], torch.from_numpy(kv[:, :dv])[None],
        attn_mask=mask[None], scale=scale)[0].numpy()
    np.testing.assert_allclose(out, ref, rtol=1e-10, atol=1e-12)
    full = scale * q @ kv.T
    np.testing.assert_allclose(lse, scipy.special.logsumexp(full[:, sel], axis=1), rtol=1e-12)


def test_attention_padding_selects_nothing():
    """Through the batched call, -1 entries of a token's index row select
    nothing: the result is torch's SDPA over the other rows only."""
    from types import SimpleNamespace
    r = np.random.default_rng(19)
    H, L, d, dv = 2, 16, 48, 32
    q = _bf16(r.standard_normal((1, H, d)))
    kv = _bf16(r.standard_normal((L, d)))
    from sparse_attention_prolog_gb300.workloads import f32_to_bf16_bits
    inp = SimpleNamespace(T=1, max_L=L, block_table=None, block_size=0, seq_of_token=np.zeros(1, np.int32),
                          q_attn=f32_to_bf16_bits(q.astype(np.float32)), kv_cache=f32_to_bf16_bits(kv.astype(np.float32)),
                          scale=0.3, d_v=dv)
    out, _ = O.sparse_attention(inp, np.array([[5, -1, 11, -1, -1]]))
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q), torch.from_numpy(kv[[5, 11]])[None], torch.from_numpy(kv[[5, 11], :dv])[None],
        scale=0.3)[0].numpy()
    np.testing.assert_allclose(out[0], ref, rtol=1e-10, atol=1e-12)


def test_attention_special_cases():
    H, d, dv = 3, 576, 512
    q = _bf16(rng.standard_normal((H, d)))
    rows = _bf16(rng.standard_normal((5, d)))
    out, _ = O.sparse_attention_token(q, rows[:1], 0.1, dv)      # one row -> its value
    np.testing.assert_allclose(out, np.repeat(rows[:1, :dv], H, 0), rtol=1e-14)
    # identical keys -> mean of the values: q is zero on the value dims and
    # all rows share dims >= dv, so every score is equal
    q2 = q.copy(); q2[:, :dv] = 0
    mix = rows[1:5].copy(); mix[:, dv:] = rows[0, dv:]
    out2, lse2 = O.sparse_attention_token(q2, mix, 0.1, dv)
    # (sums of O(1) terms in another order: equal to float64 rounding, so
    # entries that nearly cancel get an absolute bound at that scale)
    np.testing.assert_allclose(out2, np.repeat(mix[:, :dv].mean(0, keepdims=True), H, 0), rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(lse2, 0.1 * q2 @ rows[0] + math.log(4), rtol=1e-12)
    out3, lse3 = O.sparse_attention_token(q, rows[:0], 0.1, dv)
    assert (out3 == 0).all() and np.isneginf(lse3).all()
    # a duplicated index is counted twice
    o_dup, _ = O.sparse_attention_token(q, rows[[0, 0, 1]], 0.1, dv)
    w = np.exp(0.1 * q @ rows[[0, 1]].T)
    w[:, 0] *= 2
    ref = (w @ rows[[0, 1], :dv]) / w.sum(1, keepdims=True)
    np.testing.assert_allclose(o_dup, ref, rtol=1e-12, atol=1e-14)


def test_attention_sink_is_a_zero_value_key_with_logit_sink():
    """The sink reading, pinned by torch's SDPA: an extra key whose score is
    the sink (a zero key row plus an additive mask of sink[h]) and whose
    value row is zero."""
    H, L, d, dv, scale = 4, 30, 576, 512, 192 ** -0.5
    q = _bf16(rng.standard_normal((H, d)))
    kv = _bf16(rng.standard_normal((L, d)))
    sel = np.array([2, 9, 29, 14])
    sink = np.array([-1.5, 0.3, 4.0, -np.inf])
    out, lse = O.sparse_attention_token(q, kv[sel], scale, dv, sink)
    keys = np.concatenate([kv[sel], np.zeros((1, d))])
    vals = np.concatenate([kv[sel, :dv], np.zeros((1, dv))])
    bias = np.zeros((H, len(sel) + 1))
    bias[:, -1] = sink
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[:, None], torch.from_numpy(keys)[None].expand(H, -1, -1),
        torch.from_numpy(vals)[None].expand(H, -1, -1), attn_mask=torch.from_numpy(bias)[:, None],
        scale=scale)[:, 0].numpy()
    np.testing.assert_allclose(out, ref, rtol=1e-10, atol=1e-12)
    scores = np.concatenate([scale * q @ kv[sel].T, sink[:, None]], axis=1)
    np.testing.assert_allclose(lse, scipy.special.logsumexp(scores, axis=1), rtol=1e-12)
    # sink -inf is no sink; no rows leave out = 0 and lse = sink
    o0, l0 = O.sparse_attention_token(q, kv[sel], scale, dv)
    np.testing.assert_array_equal(out[3], o0[3])
    assert lse[3] == l0[3]
    oe, le = O.sparse_attention_token(q, kv[:0], scale, dv, sink)
    assert (oe == 0).all() and np.array_equal(le, sink)


def test_attention_all_causal_keys_is_causal_attention():
    H, L, d, dv, scale = 2, 16, 576, 512, 192 ** -0.5
    q = _bf16(rng.standard_normal((L, H, d)))
    kv = _bf16(rng.standard_normal((L, d)))
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q).transpose(0, 1), torch.from_numpy(kv)[None].expand(H, L, d),
        torch.from_numpy(kv[:, :dv])[None].expand(H, L, dv), is_causal=True,
        scale=scale).transpose(0, 1).numpy()
    for t in range(L):
        out, _ = O.sparse_attention_token(q[t], kv[: t + 1], scale, dv)
        np.testing.assert_allclose(out, ref[t], rtol=1e-10, atol=1e-12)


# ------------------------------------------------- Activation Quantization
def _bits(x):
    from sparse_attention_prolog_gb300.workloads import f32_to_bf16_bits
    return f32_to_bf16_bits(np.asarray(x, np.float32))


def test_act_quant_hand_worked_rows():
    """x = [1, -2.5, 0.5, 0]: scale 2.5/127, codes 51 -127 25 0 (1/s = 50.8,
    0.5/s = 25.4); with round_scale the scale is 2^-5 (2.5/127 = 0.0197 lies
    in (2^-6, 2^-5]) and the codes are 32 -80 16 0."""
    x = _bits([[1.0, -2.5, 0.5, 0.0]])
    y, s = O.act_quant(x)
    assert s[0] == np.float32(2.5) / np.float32(127.0)
    assert y.tolist() == [[51, -127, 25, 0]]
    y2, s2 = O.act_quant(x, round_scale=True)
    assert s2[0] == np.float32(2.0 ** -5)
    assert y2.tolist() == [[32, -80, 16, 0]]
    # The division is in fp32, as the page states: for max 0.5859375 the
    # fp32 scale is a little above max/127, so x = max/2 divided by it is
    # 63.4999982 exactly but 63.5 in fp32, a tie that goes to the even 64.
    y3, _ = O.act_quant(_bits([[0.5859375, 0.29296875, -0.29296875, 0.0]]))
    assert y3.tolist() == [[127, 64, -64, 0]]
    # max 1.984375 = 127/64: the scale is exactly 2^-6, already a power of
    # two, so round_scale keeps it (codes 127 and 64 for 1.0)
    y4, s4 = O.act_quant(_bits([[1.984375, 1.0, 0.0, 0.0]]), round_scale=True)
    assert s4[0] == np.float32(2.0 ** -6) and y4.tolist() == [[127, 64, 0, 0]]


def test_act_quant_properties():
    r = np.random.default_rng(7)
    x = r.standard_normal((64, 256)) * np.exp(r.uniform(-8, 8, (64, 1)))
    x[3] = 0.0
    xb = _bits(x)
    xf = O.bf16_bits_to_f64(xb)
    for rs in (False, True):
        y, s = O.act_quant(xb, round_scale=rs)
        amax = np.abs(xf).max(axis=1)
        assert s[3] == 0 and (y[3] == 0).all()                      # zero row
        nz = amax > 0
        if rs:
            m, _ = np.frexp(s[nz])
            assert (m == 0.5).all()                                 # powers of two
            assert (s[nz] >= amax[nz] / 127).all() and (s[nz] < 2 * amax[nz] / 127).all()
            big = np.abs(y[nz].astype(int)).max(axis=1)
            assert (big >= 63).all() and (big <= 127).all()
        else:
            assert (np.abs(y[nz].astype(int)).max(axis=1) == 127).all()  # the row max maps to +-127
        err = np.abs(y.astype(np.float64) * s[:, None].astype(np.float64) - xf)
        # half a step, plus the fp32 rounding of the quotient (<= 127 * 2^-24 steps)
        assert (err <= (0.5 + 1e-5) * s[:, None].astype(np.float64)).all()
    # where max/127 is exactly an fp16 value, the prolog's quantiser agrees
    row = np.linspace(-15.875, 15.875, 128)
    yp, sp = O.dynamic_quant(O.bf16_bits_to_f64(_bits(row))[None])
    ya, sa = O.act_quant(_bits(row)[None])
    assert float(sp[0]) == float(sa[0]) == 0.125
    assert np.array_equal(yp, ya)


def test_int8_gemm_fp16_output():
    """The standalone operator is the exact product, dequantised, rounded
    once to fp16: a hand-worked 1x1 case and the fp16 cast of the pinned
    dequantised product."""
    c = O.int8_gemm(np.array([[3, -2]], np.int8), np.array([0.5]), np.array([[4, 1]], np.int8), np.array([0.25]))
    assert c.dtype == np.float16 and float(c[0, 0]) == (3 * 4 - 2 * 1) * 0.5 * 0.25
    r = np.random.default_rng(11)
    a = r.integers(-128, 128, (5, 96)).astype(np.int8)
    b = r.integers(-128, 128, (7, 96)).astype(np.int8)
    sa, sb = r.uniform(0.001, 0.1, 5), r.uniform(0.001, 0.1, 7)
    exact = a.astype(np.int64) @ b.astype(np.int64).T
    assert np.array_equal(O.int8_gemm(a, sa, b, sb), (exact * sa[:, None] * sb[None, :]).astype(np.float16))


# ------------------------------------------- Manifold-constrained HC (mHC)
def test_mhc_pins():
    """Closed forms and the Sinkhorn fixed point: zero mixes and zero base
    give pre = 1/2 + eps, post = 1, comb = the uniform doubly stochastic
    matrix; with many iterations every comb is doubly stochastic (rows and
    columns sum to 1 within eps); a scaled-up comb block becomes a
    permutation when its rows pick distinct columns; softmax invariance to
    a per-row shift of the comb logits."""
    hc, eps = 4, 1e-6
    n = 6
    z0 = np.zeros((n, hc * (2 + hc)))
    pre, post, comb = O.mhc(z0, np.ones(3), np.zeros(hc * (2 + hc)), hc, 20, eps)
    np.testing.assert_allclose(pre, 0.5 + eps)
    np.testing.assert_allclose(post, 1.0)
    np.testing.assert_allclose(comb, np.full((n, hc, hc), 1.0 / hc), rtol=1e-5)
    r = np.random.default_rng(5)
    mixes = r.standard_normal((n, hc * (2 + hc)))
    base = r.standard_normal(hc * (2 + hc)) * 0.1
    _, _, c = O.mhc(mixes, np.array([1.0, 1.0, 1.0]), base, hc, 50, eps)
    np.testing.assert_allclose(c.sum(axis=-1), 1.0, atol=1e-4)
    np.testing.assert_allclose(c.sum(axis=-2), 1.0, atol=1e-4)
    perm = np.array([2, 0, 3, 1])
    logits = np.zeros((1, hc * (2 + hc)))
    logits[0, 2 * hc:] = (np.eye(hc)[perm] * 40.0).reshape(-1)
    _, _, cp = O.mhc(logits, np.ones(3), np.zeros(hc * (2 + hc)), hc, 5, 0.0)
    np.testing.assert_allclose(cp[0], np.eye(hc)[perm], atol=1e-9)
    shifted = mixes.copy()
    shifted[:, 2 * hc:] += np.repeat(r.standard_normal((n, hc)), hc, axis=1)  # + a constant per comb row
    _, _, c1 = O.mhc(mixes, np.ones(3), base, hc, 3, eps)
    _, _, c2 = O.mhc(shifted, np.ones(3), base, hc, 3, eps)
    np.testing.assert_allclose(c1, c2, rtol=1e-12)



def test_mhc_hand_worked_eps_placement():
    """hc = 2, zero inputs, eps = 0.1, worked by hand: the row softmax gives
    1/2 everywhere, + eps 0.6; divided by the column sums 1.2 + eps: 6/13.
    One more round: rows sum to 12/13 + 1/10 = 133/130, giving 60/133;
    columns sum to 120/133 + 1/10 = 1333/1330, giving 600/1333.  The gates:
    pre = 1/2 + eps, post = 2 * 1/2."""
    for iters, want in ((0, 6 / 13), (1, 600 / 1333)):
        pre, post, c = O.mhc(np.zeros((1, 8)), np.ones(3), np.zeros(8), 2, iters, 0.1)
        np.testing.assert_allclose(c, np.full((1, 2, 2), want), rtol=1e-14)
        np.testing.assert_allclose(pre, 0.6, rtol=1e-15)
        np.testing.assert_allclose(post, 1.0, rtol=1e-15)


def test_mhc_scale_order_and_sinkhorn_limit():
    """Independent of the step order written in the oracle: (1) the three
    parts take hc_scale[0], [1], [2] in that order and the gates are the
    logistic function, checked through its tanh form (1 + tanh(z/2)) / 2;
    (2) with eps = 0 the last step is a column normalisation, so every column
    sums to one and the rows in general do not; (3) a positive 2 x 2 matrix
    has the Sinkhorn limit [[p, 1 - p], [1 - p, p]] with
    p / (1 - p) = sqrt(c00 c11 / (c01 c10)), the cross ratio that row and
    column scalings leave unchanged; after a row softmax it equals
    exp(z00 + z11 - z01 - z10)."""
    hc = 4
    w = hc * (2 + hc)
    x = np.zeros((1, w))
    x[0, :hc] = [0.5, -1.0, 2.0, 0.0]
    x[0, hc:2 * hc] = [1.0, -0.25, 0.0, 3.0]
    scale = np.array([2.0, 3.0, 5.0])
    base = np.zeros(w)
    base[:2 * hc] = np.linspace(-0.3, 0.4, 2 * hc)
    pre, post, _ = O.mhc(x, scale, base, hc, 0, 1e-3)
    logistic = lambda v: 0.5 * (1.0 + np.tanh(0.5 * v))
    np.testing.assert_allclose(pre[0], logistic(2.0 * x[0, :hc] + base[:hc]) + 1e-3, rtol=1e-13)
    np.testing.assert_allclose(post[0], 2.0 * logistic(3.0 * x[0, hc:2 * hc] + base[hc:2 * hc]), rtol=1e-13)
    r = np.random.default_rng(11)
    mixes = r.standard_normal((8, w))
    for iters in (0, 3):
        _, _, c = O.mhc(mixes, np.ones(3), np.zeros(w), hc, iters, 0.0)
        np.testing.assert_allclose(c.sum(axis=-2), 1.0, rtol=1e-13)
        assert np.abs(c.sum(axis=-1) - 1.0).max() > 1e-6
    z = np.array([[0.7, -0.4], [0.2, 1.1]])
    m2 = np.zeros((1, 2 * 4))
    m2[0, 4:] = z.reshape(-1)
    # the comb logits take hc_scale[2] (0.3 z under scale 5: a cross ratio of
    # about e^3.9, within reach of 400 rounds)
    for sc, zz in ((np.ones(3), z), (np.array([2.0, 3.0, 5.0]), 0.3 * z)):
        m2[0, 4:] = zz.reshape(-1)
        _, _, c = O.mhc(m2, sc, np.zeros(8), 2, 400, 0.0)
        ratio = np.sqrt(np.exp(sc[2] * (zz[0, 0] + zz[1, 1] - zz[0, 1] - zz[1, 0])))
        p = ratio / (1.0 + ratio)
        np.testing.assert_allclose(c[0], [[p, 1.0 - p], [1.0 - p, p]], atol=1e-12)


# ------------------------------------------------------------- MLA Prolog
def test_rms_norm_pins():
    """[3, 4] has mean square 12.5; a constant row c maps to
    gamma c / sqrt(c^2 + eps); scale and sign equivariance at eps = 0; and
    torch's own rms_norm on random rows."""
    np.testing.assert_allclose(O.rms_norm(np.array([3.0, 4.0]), [1.0, 1.0], 0.0),
                               np.array([3.0, 4.0]) / math.sqrt(12.5), rtol=1e-15)
    g = np.array([0.5, 2.0, -1.0])
    np.testing.assert_allclose(O.rms_norm(np.full(3, 0.1), g, 1e-2), g * 0.1 / math.sqrt(0.01 + 1e-2), rtol=1e-14)
    r = np.random.default_rng(21)
    x = r.standard_normal((5, 64))
    gam = 1.0 + 0.1 * r.standard_normal(64)
    np.testing.assert_allclose(O.rms_norm(-3.5 * x, gam, 0.0), -O.rms_norm(x, gam, 0.0), rtol=1e-12)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(x), (64,), torch.from_numpy(gam), eps=1e-6).numpy()
    np.testing.assert_allclose(O.rms_norm(x, gam, 1e-6), ref, rtol=1e-12)


def _mla_small(T=3, H=2, K_q=128, D_x=128, pos=None, seed=31, interleaved=0):
    pos = np.arange(T, dtype=np.int32) + 5 if pos is None else np.asarray(pos, dtype=np.int32)
    return W.make_mla_inputs(T, pos, np.arange(T), seed, H=H, K_q=K_q, D_x=D_x, max_pos=64,
                             rope_interleaved=interleaved)


def test_mla_absorption_identity():
    """The absorbed query scores a latent row c exactly as the head's
    no-position query scores the up-projected key w_uk[h] c (both sides built
    here from int8_gemm_dequant, which has its own pins)."""
    p = _mla_small()
    r = np.random.default_rng(3)
    codes = W.int8_codes(r, (p.T, p.K_q))
    sa = np.array([0.02, 0.03, 0.05])
    wuk = O.bf16_bits_to_f64(p.w_uk)
    q = O.mla_q(codes, sa, p.w_uq, p.w_uq_scale, wuk, p.H, p.pos, p.rope_cos, p.rope_sin)
    u = O.int8_gemm_dequant(codes, sa, p.w_uq, p.w_uq_scale).reshape(p.T, p.H, 192)
    c = r.standard_normal(512)
    for h in range(p.H):
        np.testing.assert_allclose(q[:, h, :512] @ c, u[:, h, :128] @ (wuk[h] @ c), rtol=1e-10)


def test_mla_rope_relative_position():
    """Rotary property: the q . k score of the rotary dims depends on the two
    positions only through their difference (here both move by 11)."""
    for inter in (0, 1):
        a = _mla_small(pos=[3, 9, 20], interleaved=inter)
        b = _mla_small(pos=[14, 20, 31], interleaved=inter)
        ra, rb = O.mla_prolog(a), O.mla_prolog(b)
        sa = np.einsum("thd,td->th", ra["q"][..., 512:], ra["kv"][:, 512:])
        sb = np.einsum("thd,td->th", rb["q"][..., 512:], rb["kv"][:, 512:])
        np.testing.assert_allclose(sa, sb, rtol=1e-5, atol=1e-6)
        assert not np.allclose(ra["q"][..., 512:], rb["q"][..., 512:])


def test_mla_one_hot_layout():
    """One-hot inputs at position 0 (identity rotation) reduce every
    projection to indexing: the kv row is [RMSNorm(a w_dkv[:512, j]) |
    a w_dkv[512:, j]], token rows scaled by different a > 0 give the same
    normalised query latent (per-token normalisation), a one-hot q_lora
    selects column k of w_uq, whose rows per head are 128 no-position
    dims then 64 rotary dims."""
    T, j = 2, 7
    p = _mla_small(T=T, pos=[0, 0])
    x = np.zeros((T, p.D_x), np.float32)
    x[0, j], x[1, j] = 2.0, 0.5
    p.x = W.f32_to_bf16_bits(x)
    p.gamma_q[:] = 1.0
    p.gamma_kv[:] = 1.0
    p.rms_eps = 0.0  # exact scale invariance
    r = O.mla_prolog(p)
    np.testing.assert_allclose(r["c_q"][0], r["c_q"][1], rtol=1e-9)
    col = O.bf16_bits_to_f64(p.w_dkv)[:, j]
    for t, a in ((0, 2.0), (1, 0.5)):
        lat = a * col[:512]
        np.testing.assert_allclose(r["kv"][t, :512], lat / np.sqrt((lat ** 2).mean() + p.rms_eps), rtol=1e-12)
        np.testing.assert_allclose(r["kv"][t, 512:], a * col[512:], rtol=1e-12)
    k = 5
    codes = np.zeros((1, p.K_q), np.int8)
    codes[0, k] = 1
    q = O.mla_q(codes, np.ones(1), p.w_uq, np.ones(p.H * 192), O.bf16_bits_to_f64(p.w_uk), p.H,
                np.zeros(1, np.int32), p.rope_cos, p.rope_sin)
    wuk = O.bf16_bits_to_f64(p.w_uk)
    for h in range(p.H):
        rows = p.w_uq[h * 192:(h + 1) * 192, k].astype(np.float64)
        np.testing.assert_allclose(q[0, h, 512:], rows[128:], rtol=1e-15)
        np.testing.assert_allclose(q[0, h, :512], rows[:128] @ wuk[h], rtol=1e-12)


def test_mla_gammas_select_channels():
    """A one-hot gamma keeps one channel: gamma_q = e_j makes the query
    latent of every token a single code of magnitude 127 at j; gamma_kv =
    e_i leaves one nonzero latent dim i in every KV row (the rotary dims
    have no gamma)."""
    p = _mla_small()
    p.gamma_q[:] = 0.0
    p.gamma_q[9] = 1.5
    p.gamma_kv[:] = 0.0
    p.gamma_kv[100] = 0.7
    r = O.mla_prolog(p)
    assert (np.abs(r["q_lora"][:, 9]) == 127).all()
    assert (np.delete(r["q_lora"], 9, axis=1) == 0).all()
    assert (np.delete(r["kv"][:, :512], 100, axis=1) == 0).all()
    assert (r["kv"][:, 100] != 0).all() and (r["kv"][:, 512:] != 0).any()


def test_mla_cache_slots():
    """Rows go to kv_cache[slot[t]]; slot -1 writes nothing."""
    p = _mla_small()
    p.slot = np.array([4, -1, 1], dtype=np.int64)
    cache = np.full((6, 576), 7.0)
    r = O.mla_prolog(p, cache)
    np.testing.assert_array_equal(cache[4], r["kv"][0])
    np.testing.assert_array_equal(cache[1], r["kv"][2])
    assert np.all(cache[[0, 2, 3, 5]] == 7.0)


def test_paged_and_contiguous_caches_agree():
    """The same sequences stored contiguously and in shuffled 16-row blocks
    (the blocks scattered here, block by block, without the oracle's address
    function) give the same key rows and the same sparse attention; an
    identity block table reproduces the contiguous addresses."""
    from types import SimpleNamespace
    r = np.random.default_rng(77)
    B, max_L, bs, d_qk, d_v, H, T = 3, 64, 16, 40, 32, 2, 4
    nblk = max_L // bs
    contig = W.f32_to_bf16_bits(r.standard_normal((B * max_L, d_qk)).astype(np.float32))
    table = r.permutation(B * nblk).reshape(B, nblk).astype(np.int32)
    paged = np.zeros_like(contig)
    for b in range(B):
        for j in range(nblk):
            paged[table[b, j] * bs:(table[b, j] + 1) * bs] = contig[b * max_L + j * bs:b * max_L + (j + 1) * bs]
    q = W.f32_to_bf16_bits(r.standard_normal((T, H, d_qk)).astype(np.float32))
    seq = np.array([0, 2, 1, 2], np.int32)
    common = dict(T=T, max_L=max_L, block_size=bs, seq_of_token=seq, q_attn=q, scale=d_qk ** -0.5, d_v=d_v)
    a = SimpleNamespace(block_table=None, kv_cache=contig, **common)
    p = SimpleNamespace(block_table=table, kv_cache=paged, **common)
    for b in range(B):
        np.testing.assert_array_equal(paged[O.logical_rows(p, b, 50)], contig[b * max_L + np.arange(50)])
    ident = SimpleNamespace(block_table=np.arange(B * nblk, dtype=np.int32).reshape(B, nblk), block_size=bs, max_L=max_L)
    np.testing.assert_array_equal(O.cache_rows(ident, 2, [0, 17, 63]), 2 * max_L + np.array([0, 17, 63]))
    idx = np.stack([r.choice(max_L, 20, replace=False) for _ in range(T)])
    idx[1, 5:] = -1
    oa, la = O.sparse_attention(a, idx)
    op, lp = O.sparse_attention(p, idx)
    np.testing.assert_array_equal(oa, op)
    np.testing.assert_array_equal(la, lp)

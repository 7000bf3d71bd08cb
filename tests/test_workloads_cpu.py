"""The seeded input generators (CPU only): the shapes, positions, page
tables and value spreads that the input recipe states, and determinism.
The generators hold none of the method's arithmetic; these tests only check
that they produce the workloads they describe."""
import numpy as np
import torch

from sparse_attention_prolog_gb300 import workloads as W


def test_same_seed_same_inputs_other_seed_other_inputs():
    a, b, c = W.tiny_decode(), W.tiny_decode(), W.tiny_decode(seed=7)
    for f in ("q_idx", "q_idx_scale", "w_idx", "k_cache", "k_scale", "q_attn", "kv_cache"):
        assert np.array_equal(getattr(a, f), getattr(b, f)), f
    assert not np.array_equal(a.k_cache, c.k_cache)
    p, q = W.decode_64k_prolog(), W.decode_64k_prolog()
    assert np.array_equal(p.w_qb, q.w_qb) and np.array_equal(p.x, q.x)


def test_headline_decode_batch():
    """B=4 sequences of 65536 keys, two query tokens each at the last two
    positions, H_I=64 x d_I=128, top-2048, 128 heads; the prolog's new keys
    go to the last two rows of each sequence."""
    inp = W.decode_64k(with_attention=False)
    assert (inp.B, inp.T, inp.max_L, inp.H_I, inp.d_I, inp.topk, inp.H) == (4, 8, 65536, 64, 128, 2048, 128)
    assert inp.pos.tolist() == [65534, 65535] * 4
    assert inp.seq_of_token.tolist() == [0, 0, 1, 1, 2, 2, 3, 3]
    assert inp.k_cache.shape == (4 * 65536, 128) and inp.block_table is None
    p = W.decode_64k_prolog()
    assert (p.T, p.H_I, p.d_I, p.q_lora.shape[1], p.x.shape[1]) == (8, 64, 128, 1536, 7168)
    assert p.slot.tolist() == [b * 65536 + s for b in range(4) for s in (65534, 65535)]
    assert p.pos.tolist() == inp.pos.tolist()


def test_causal_prefill_positions():
    inp = W.causal_prefill(S=1024, with_attention=False)
    assert inp.B == 1 and inp.T == 1024 and inp.max_L == 1024
    assert np.array_equal(inp.pos, np.arange(1024)) and (inp.seq_of_token == 0).all()


def test_ragged_paged_recipe():
    """Lengths within [4096, 131072], one token per sequence at its last
    position, 64-token pages: every physical page belongs to exactly one
    sequence (a shuffled permutation), unused table entries are -1."""
    inp = W.ragged_paged_decode(B=6, with_attention=False)
    lens = inp.seq_len.astype(np.int64)
    assert ((lens >= 4096) & (lens <= 131072)).all()
    assert inp.max_L == 131072 and inp.block_size == 64
    assert np.array_equal(inp.pos, lens - 1)
    used = []
    for b in range(inp.B):
        nb = -(-int(lens[b]) // 64)
        assert (inp.block_table[b, :nb] >= 0).all() and (inp.block_table[b, nb:] == -1).all()
        used.extend(inp.block_table[b, :nb].tolist())
    assert sorted(used) == list(range(len(used)))
    assert used != sorted(used)  # shuffled
    assert inp.k_cache.shape == (len(used) * 64, 128)


def test_code_and_scale_spreads():
    """int8 codes are rounded N(0, (127/4)^2) clipped to +-127, the spread
    of a quantised N(0,1) row; fp16 scales are (4/127) sigma U(0.9, 1.1)."""
    rng = np.random.default_rng(5)
    c = W.int8_codes(rng, (1 << 20,))
    assert c.dtype == np.int8 and np.abs(c.astype(int)).max() <= 127
    assert abs(c.astype(np.float64).std() / (127 / 4) - 1) < 0.01
    s = W.fp16_scales(rng, (1 << 16,), sigma=2.0).astype(np.float64)
    lo, hi = 0.9 * 2 * 4 / 127, 1.1 * 2 * 4 / 127
    assert (s >= lo * (1 - 1e-3)).all() and (s <= hi * (1 + 1e-3)).all()


def test_bf16_rounding_matches_torch():
    """Round to nearest even, as torch's float32 -> bfloat16 conversion,
    including exact ties and values near the largest finite bf16."""
    rng = np.random.default_rng(6)
    x = (rng.standard_normal(1 << 16) * np.exp(rng.uniform(-30, 30, 1 << 16))).astype(np.float32)
    ties = (np.arange(1, 257, dtype=np.uint32) << 16 | 0x8000).view(np.float32)
    x = np.concatenate([x, ties, -ties, np.float32([0.0, -0.0, 3.3e38, -3.3e38])])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(W.f32_to_bf16_bits(x), ref)


def test_rope_tables_are_the_rotary_angles():
    """cos/sin of p * 10000^(-2i/d_rope): row 0 is (1, 0), cos^2 + sin^2 = 1,
    and a sampled entry equals its angle."""
    cos, sin = W.rope_tables(4096, 64)
    assert cos.shape == sin.shape == (4096, 32) and cos.dtype == np.float32
    assert (cos[0] == 1).all() and (sin[0] == 0).all()
    np.testing.assert_allclose(cos.astype(np.float64) ** 2 + sin.astype(np.float64) ** 2, 1.0, atol=1e-6)
    ang = 3000 * 10000.0 ** (-2 * 5 / 64)
    assert abs(cos[3000, 5] - np.cos(ang)) < 1e-6 and abs(sin[3000, 5] - np.sin(ang)) < 1e-6

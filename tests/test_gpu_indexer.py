"""Lightning Indexer + top-k: CUDA path vs oracle."""
import numpy as np
import pytest
import torch

import oracle as O
from parity_utils import check_topk_exact_on_scores, check_topk_set, oracle_scores_row
from sparse_attention_prolog_gb300 import binding as B
from sparse_attention_prolog_gb300 import workloads as W
from sparse_attention_prolog_gb300.pipeline import DecodeBuffers, to_dev

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _check_all(inp, buf, tokens=None):
    torch.cuda.synchronize()
    assert B.device_error() == 0
    idx = buf.topk_idx.cpu().numpy()
    sc = buf.scores.cpu().numpy()
    tokens = range(inp.T) if tokens is None else tokens
    for t in tokens:
        ref = oracle_scores_row(inp, t)
        n = int(inp.pos[t]) + 1
        g = sc[t, :n].astype(np.float64)
        scale = max(np.abs(ref).max(), 1e-30)
        assert np.abs(g - ref).max() <= 2e-6 * scale, f"t={t}: score err {np.abs(g - ref).max() / scale:.2e}"
        if n < inp.max_L:
            pass
        check_topk_set(idx[t], ref, n, inp.topk, f"t={t}")
        check_topk_exact_on_scores(idx[t], sc[t], n, inp.topk, f"t={t}")


def test_tiny_decode_indexer(cuda_lib):
    inp = W.tiny_decode()
    buf = DecodeBuffers(inp, DEV, with_attention=False, keep_scores=True)
    buf.run_topk()
    _check_all(inp, buf)


def test_ragged_mid_decode_indexer(cuda_lib):
    """Two sequences (3001 and 4096 keys), MTP1, H_I=64 x d_I=128, top-512:
    many key tiles, a ragged last tile, masked tail columns."""
    inp = W.make_decode_inputs(B=2, n_q=2, seq_lens=[3001, 4096], H_I=64, d_I=128, topk=512, H=8, seed=11,
                               with_attention=False)
    buf = DecodeBuffers(inp, DEV, with_attention=False, keep_scores=True)
    buf.run_topk()
    _check_all(inp, buf)


def test_paged_decode_indexer(cuda_lib):
    """Paged key cache, 64-token blocks, shuffled block table, n_q=1."""
    inp = W.make_decode_inputs(B=3, n_q=1, seq_lens=[700, 2048, 1500], H_I=64, d_I=128, topk=256, H=8, seed=12,
                               block_size=64, max_L=2048, with_attention=False)
    buf = DecodeBuffers(inp, DEV, with_attention=False, keep_scores=True)
    buf.run_topk()
    _check_all(inp, buf)


@pytest.mark.parametrize("block_size,d_I,H_I", [(8, 128, 64), (16, 64, 32), (32, 128, 16), (128, 128, 64),
                                                 (256, 64, 128)])
def test_paged_page_sizes(block_size, d_I, H_I, cuda_lib):
    """Every supported kind of page: pages smaller than a 128-key tile (8,
    16, 32 keys: one box per page, the last tile's boxes cut after the last
    visible key), a page of one tile and pages of two tiles; both key
    widths, and head counts on both top-k paths (histogram-seeded for
    H_I >= 64, the general kernel below)."""
    inp = W.make_decode_inputs(B=3, n_q=2, seq_lens=[700, 2048, 1501], H_I=H_I, d_I=d_I, topk=256, H=8,
                               seed=40 + block_size, block_size=block_size, max_L=2048, with_attention=False)
    buf = DecodeBuffers(inp, DEV, with_attention=False, keep_scores=True)
    buf.run_topk()
    _check_all(inp, buf)


@pytest.mark.parametrize("topk,H_I", [(1, 64), (7, 64), (4096, 64), (1, 32), (4096, 32)])
def test_topk_extreme_k(topk, H_I, cuda_lib):
    """k = 1 (the single largest key), a small odd k, and k = 4096 (twice the
    decode selection), on the histogram-seeded top-k (H_I = 64) and on the
    general kernel (H_I = 32); one sequence is shorter than 4096 keys, so
    that row is padded with -1 when k = 4096."""
    inp = W.make_decode_inputs(B=2, n_q=2, seq_lens=[3001, 20000], H_I=H_I, d_I=128, topk=topk, H=8,
                               seed=50 + topk, max_L=20096, with_attention=False)
    buf = DecodeBuffers(inp, DEV, with_attention=False, keep_scores=True)
    buf.run_topk()
    _check_all(inp, buf)


@pytest.mark.parametrize("H_I,d_I,n_q", [(8, 64, 16), (4, 128, 40), (16, 128, 3)])
def test_tokens_per_key_tile(H_I, d_I, n_q, cuda_lib):
    """The indexer scores G = min(n_q, 128 / H_I, 32) tokens of a sequence
    against each key tile: 16 tokens at H_I = 8, 32 + 8 at H_I = 4 (a
    group cut at the 32-token bound), and 3 of the possible 8 at H_I = 16."""
    inp = W.make_decode_inputs(B=2, n_q=n_q, seq_lens=[3000, 2100], H_I=H_I, d_I=d_I, topk=300, H=8,
                               seed=20 + n_q, max_L=3072, with_attention=False)
    buf = DecodeBuffers(inp, DEV, with_attention=False, keep_scores=True)
    buf.run_topk()
    _check_all(inp, buf)


def test_most_token_groups(cuda_lib):
    """4096 one-token sequences of 1 to 128 keys: the largest token-group
    table the indexer takes (4096 groups), on the general top-k kernel
    (T > 512); 128 sampled tokens, the first and last included."""
    L = np.random.default_rng(3).integers(1, 129, 4096)
    inp = W.make_decode_inputs(B=4096, n_q=1, seq_lens=L, H_I=64, d_I=128, topk=32, H=8, seed=33, max_L=128,
                               with_attention=False)
    buf = DecodeBuffers(inp, DEV, with_attention=False, keep_scores=True)
    buf.run_topk()
    tokens = sorted(set(np.random.default_rng(4).choice(4096, 126, replace=False).tolist()) | {0, 4095})
    _check_all(inp, buf, tokens=tokens)


@pytest.mark.parametrize("H_I,n_q", [(64, 2), (16, [3, 1])])
def test_scores_and_selection_as_two_calls(H_I, n_q, cuda_lib):
    """dsa_indexer_scores then dsa_topk_from_scores: the score rows (-inf
    past each token's causal limit within its group's columns) and the
    selection from a copy of them with a row pitch wider than max_L."""
    inp = W.make_decode_inputs(B=2, n_q=n_q, seq_lens=[3001, 4096], H_I=H_I, d_I=128, topk=512, H=8, seed=25,
                               with_attention=False)
    buf = DecodeBuffers(inp, DEV, with_attention=False)
    scores = torch.full((inp.T, inp.max_L), float("nan"), dtype=torch.float32, device=DEV)
    B.dsa_indexer_scores(buf.targs, scores)
    wide = torch.full((inp.T, inp.max_L + 96), float("nan"), dtype=torch.float32, device=DEV)
    wide[:, :inp.max_L] = scores
    B.dsa_topk_from_scores(buf.targs, wide)
    torch.cuda.synchronize()
    assert B.device_error() == 0
    sc = scores.cpu().numpy()
    idx = buf.topk_idx.cpu().numpy()
    for t in range(inp.T):
        ref = oracle_scores_row(inp, t)
        n = int(inp.pos[t]) + 1
        g = sc[t, :n].astype(np.float64)
        assert np.abs(g - ref).max() <= 2e-6 * max(np.abs(ref).max(), 1e-30), f"t={t}"
        last = int(inp.pos[inp.seq_of_token == inp.seq_of_token[t]].max())
        assert np.isneginf(sc[t, n:last + 1]).all(), f"t={t}: columns past pos not -inf"
        check_topk_set(idx[t], ref, n, inp.topk, f"t={t}")
        check_topk_exact_on_scores(idx[t], sc[t], n, inp.topk, f"t={t}")


def test_short_rows_pad_with_minus_one(cuda_lib):
    """Prefill-like causal rows where early tokens see fewer than k keys."""
    inp = W.make_decode_inputs(B=1, n_q=384, seq_lens=[384], H_I=64, d_I=128, topk=200, H=8, seed=13,
                               with_attention=False)
    buf = DecodeBuffers(inp, DEV, with_attention=False, keep_scores=True)
    buf.run_topk()
    _check_all(inp, buf, tokens=[0, 1, 63, 199, 200, 201, 255, 383])


@pytest.mark.parametrize("seq_lens,max_L", [([24576, 20000], 24576), ([98304, 70000], 98304)])
def test_fused_topk_row_splits(seq_lens, max_L, cuda_lib):
    """Rows of 24576 keys (a 3-CTA cluster of 8 keys per thread) and 98304
    keys (6 CTAs of 16 keys per thread) on the histogram top-k path."""
    inp = W.make_decode_inputs(B=2, n_q=2, seq_lens=seq_lens, H_I=64, d_I=128, topk=2048, H=8, seed=16,
                               max_L=max_L, with_attention=False)
    buf = DecodeBuffers(inp, DEV, with_attention=False, keep_scores=True)
    buf.run_topk()
    _check_all(inp, buf)


@pytest.mark.parametrize("L,H_I", [(131072, 64), (200064, 64), (12032, 32)])
def test_long_rows(L, H_I, cuda_lib):
    """A full row of 131072 keys, the longest the histogram-seeded top-k
    takes (8 CTAs of 16 keys per thread); 200064 keys, past it (the general
    kernel on 8-CTA clusters); 12032 keys on the general kernel's 2-CTA
    clusters.  The other sequence is short."""
    inp = W.make_decode_inputs(B=2, n_q=2, seq_lens=[L, 5000], H_I=H_I, d_I=128, topk=2048, H=8, seed=19,
                               with_attention=False)
    buf = DecodeBuffers(inp, DEV, with_attention=False, keep_scores=True)
    buf.run_topk()
    _check_all(inp, buf)


def test_fused_topk_all_scores_equal(cuda_lib):
    """Zero queries make every visible score 0: any k distinct visible keys
    are a correct answer."""
    inp = W.make_decode_inputs(B=2, n_q=2, seq_lens=[5000, 9000], H_I=64, d_I=128, topk=1024, H=8, seed=17, max_L=9088,
                               with_attention=False)
    inp.q_idx[:] = 0
    buf = DecodeBuffers(inp, DEV, with_attention=False, keep_scores=True)
    buf.run_topk()
    _check_all(inp, buf)


def test_fused_topk_many_ties_at_threshold(cuda_lib):
    """Keys of 0/1 bytes against all-ones queries with equal key scales give
    at most 129 distinct scores, so the k-th score is shared by many keys
    and only some of its copies may be taken."""
    inp = W.make_decode_inputs(B=2, n_q=2, seq_lens=[12000, 16384], H_I=64, d_I=128, topk=2048, H=8, seed=18,
                               with_attention=False)
    rng = np.random.default_rng(118)
    inp.k_cache[:] = (rng.random(inp.k_cache.shape) < 0.5).astype(np.int8)
    inp.k_scale[:] = np.float16(0.03125)
    inp.q_idx[:] = 1
    buf = DecodeBuffers(inp, DEV, with_attention=False, keep_scores=True)
    buf.run_topk()
    _check_all(inp, buf)
    sc = buf.scores.cpu().numpy()
    for t in range(inp.T):  # the tie case really occurs
        n = int(inp.pos[t]) + 1
        kth = np.sort(sc[t, :n])[::-1][inp.topk - 1]
        assert (sc[t, :n] == kth).sum() > 1


@pytest.mark.parametrize("sign", [1, -1])
def test_tensor_core_dots_bit_exact(sign, cuda_lib):
    """One-hot head weights with unit scales make I[t,s] = ReLU(dot[t,h0,s])
    an exact integer in fp32, exposing the tcgen05 contraction bit by bit
    (negated q exposes the negative dots)."""
    inp = W.make_decode_inputs(B=2, n_q=2, seq_lens=[1000, 1024], H_I=64, d_I=128, topk=64, H=8, seed=14,
                               with_attention=False)
    inp.q_idx[0, :, :4] = 127
    inp.k_cache[:8, :4] = -128  # extreme operands in the contraction
    q = (inp.q_idx.astype(np.int16) * sign).clip(-128, 127).astype(np.int8)
    ones = np.ones_like(inp.q_idx_scale)
    for h0 in (0, 17, 63):
        w = np.zeros_like(inp.w_idx)
        w[:, h0] = 1.0
        buf = DecodeBuffers(inp, DEV, q_idx=to_dev(q, DEV), q_idx_scale=to_dev(ones, DEV), w_idx=to_dev(w, DEV),
                            k_scale=to_dev(np.ones_like(inp.k_scale), DEV), with_attention=False, keep_scores=True)
        buf.run_topk()
        torch.cuda.synchronize()
        sc = buf.scores.cpu().numpy()
        for t in range(inp.T):
            n = int(inp.pos[t]) + 1
            rows = O.logical_rows(inp, int(inp.seq_of_token[t]), n)
            dots = O.indexer_dots(q[t, h0:h0 + 1], inp.k_cache[rows])[0]
            np.testing.assert_array_equal(sc[t, :n], np.maximum(dots, 0).astype(np.float32))


def test_debug_dots_kernel(cuda_lib):
    inp = W.make_decode_inputs(B=1, n_q=2, seq_lens=[256], H_I=4, d_I=64, topk=32, H=4, seed=15,
                               with_attention=False)
    buf = DecodeBuffers(inp, DEV, with_attention=False)
    dots = torch.zeros(inp.T, inp.H_I, inp.max_L, dtype=torch.int32, device=DEV)
    B.dsa_indexer_dots_debug(buf.targs, dots)
    torch.cuda.synchronize()
    for t in range(inp.T):
        ref = O.indexer_dots(inp.q_idx[t], inp.k_cache[O.logical_rows(inp, 0, inp.max_L)])
        np.testing.assert_array_equal(dots[t].cpu().numpy(), ref)


def test_workspace_scores_path(cuda_lib):
    """Without scores_out the score rows live in the caller's workspace."""
    inp = W.tiny_decode()
    buf = DecodeBuffers(inp, DEV, with_attention=False, keep_scores=False)
    assert B.workspace_bytes("topk", buf.targs) >= inp.T * inp.max_L * 4
    buf.run_topk()
    torch.cuda.synchronize()
    idx = buf.topk_idx.cpu().numpy()
    for t in range(inp.T):
        check_topk_set(idx[t], oracle_scores_row(inp, t), int(inp.pos[t]) + 1, inp.topk)

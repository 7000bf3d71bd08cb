"""Batches whose sequences carry different numbers of query tokens (mixed MTP
depths, a prefill chunk beside decode tokens), given to dsa_indexer_topk and
dsa_sparse_attn through the per-token map seq_of_token: CUDA path vs oracle,
with the same tolerances as the uniform batches."""
import numpy as np
import pytest
import torch

import oracle as O
from parity_utils import check_attention, check_topk_exact_on_scores, check_topk_set, oracle_scores_row
from sparse_attention_prolog_gb300 import binding as B
from sparse_attention_prolog_gb300 import workloads as W
from sparse_attention_prolog_gb300.pipeline import DecodeBuffers, is_uniform

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
DSA_ERR_DEVICE_DATA = 6


def _check_chain(inp, buf, tokens=None):
    """Scores and top-k sets of every token against the oracle, then the
    attention over the kernel's own selection."""
    torch.cuda.synchronize()
    assert B.device_error() == 0
    idx = buf.topk_idx.cpu().numpy()
    sc = buf.scores.cpu().numpy()
    tokens = list(range(inp.T)) if tokens is None else tokens
    for t in tokens:
        ref = oracle_scores_row(inp, t)
        n = int(inp.pos[t]) + 1
        g = sc[t, :n].astype(np.float64)
        scale = max(np.abs(ref).max(), 1e-30)
        assert np.abs(g - ref).max() <= 2e-6 * scale, f"t={t}: score err {np.abs(g - ref).max() / scale:.2e}"
        check_topk_set(idx[t], ref, n, inp.topk, f"t={t}")
        check_topk_exact_on_scores(idx[t], sc[t], n, inp.topk, f"t={t}")
    ref_o, ref_l = O.sparse_attention(inp, idx, tokens)
    check_attention(buf.out.float().cpu().numpy()[tokens], ref_o, buf.lse.cpu().numpy()[tokens], ref_l, "attn")


def test_uneven_tokens_per_sequence(cuda_lib):
    """3, 1 and 2 query tokens over three sequences (ragged last key tiles)."""
    inp = W.make_decode_inputs(B=3, n_q=[3, 1, 2], seq_lens=[3001, 4096, 2500], H_I=64, d_I=128, topk=512,
                               H=128, seed=61)
    assert not is_uniform(inp)
    buf = DecodeBuffers(inp, DEV, keep_scores=True)
    assert buf.seq is not None
    buf.run()
    _check_chain(inp, buf)


def test_uneven_paged(cuda_lib):
    """The token map with a paged cache of 64-token blocks."""
    inp = W.make_decode_inputs(B=3, n_q=[1, 3, 2], seq_lens=[700, 2048, 1500], H_I=64, d_I=128, topk=256, H=64,
                               seed=62, block_size=64, max_L=2048)
    buf = DecodeBuffers(inp, DEV, keep_scores=True)
    buf.run()
    _check_chain(inp, buf)


def test_runs_longer_than_a_group(cuda_lib):
    """H_I = 16 scores up to 8 tokens of a sequence together: runs of 5, 12
    and 1 tokens become groups of 5, 8 + 4 and 1."""
    inp = W.make_decode_inputs(B=3, n_q=[5, 12, 1], seq_lens=[1000, 1300, 640], H_I=16, d_I=64, topk=128, H=16,
                               seed=63, max_L=1408)
    buf = DecodeBuffers(inp, DEV, keep_scores=True)
    buf.run()
    _check_chain(inp, buf)


def test_prefill_chunk_beside_decode_tokens(cuda_lib):
    """A 300-token prefill chunk (causal rows shorter than k at its start)
    next to two one-token decode sequences."""
    inp = W.make_decode_inputs(B=3, n_q=[1, 300, 1], seq_lens=[5000, 300, 2100], H_I=64, d_I=128, topk=256,
                               H=32, seed=64, max_L=5120)
    buf = DecodeBuffers(inp, DEV, keep_scores=True)
    buf.run()
    _check_chain(inp, buf, tokens=[0, 1, 2, 150, 255, 256, 257, 300, 301])


def test_map_of_a_uniform_batch_matches_the_uniform_call(cuda_lib):
    """The same uniform batch with and without the map: equal scores, equal
    selections and equal attention outputs (the same kernels, grouped alike)."""
    inp = W.make_decode_inputs(B=2, n_q=2, seq_lens=[3001, 4096], H_I=64, d_I=128, topk=512, H=128, seed=65)
    a = DecodeBuffers(inp, DEV, keep_scores=True)
    b = DecodeBuffers(inp, DEV, keep_scores=True, seq_map=True)
    assert a.seq is None and b.seq is not None
    a.run()
    b.run()
    torch.cuda.synchronize()
    assert B.device_error() == 0
    for t in range(inp.T):
        n = int(inp.pos[t]) + 1
        np.testing.assert_array_equal(a.scores.cpu().numpy()[t, :n], b.scores.cpu().numpy()[t, :n])
        assert set(a.topk_idx.cpu().numpy()[t].tolist()) == set(b.topk_idx.cpu().numpy()[t].tolist())
    _check_chain(inp, b)


def test_out_of_range_sequence_id_is_reported(cuda_lib):
    """A token whose id lies outside [0, B): recorded as invalid device data;
    its attention output is zero, the other tokens are unaffected."""
    inp = W.make_decode_inputs(B=2, n_q=[2, 1], seq_lens=[900, 1200], H_I=64, d_I=128, topk=128, H=16, seed=66,
                               max_L=1280)
    buf = DecodeBuffers(inp, DEV, keep_scores=True)
    buf.run()
    torch.cuda.synchronize()
    assert B.device_error() == 0
    good = buf.out.float().cpu().numpy().copy()
    bad = inp.seq_of_token.copy()
    bad[2] = 7  # the third token names a sequence that does not exist
    buf.seq.copy_(torch.from_numpy(bad.astype(np.int32)))
    buf.run_attn()
    torch.cuda.synchronize()
    assert B.device_error() == DSA_ERR_DEVICE_DATA
    out = buf.out.float().cpu().numpy()
    assert (out[2] == 0).all()
    np.testing.assert_array_equal(out[:2], good[:2])
    buf.run_topk()
    torch.cuda.synchronize()
    assert B.device_error() == DSA_ERR_DEVICE_DATA
    assert B.device_error() == 0  # reading the word cleared it

"""Whole decode steps on the five workloads: each stage is checked against
the oracle fed with the CUDA path's own upstream outputs (stage isolation),
so that legitimate top-k ties do not spread into the attention check."""
import numpy as np
import pytest
import torch

import oracle as O
from parity_utils import check_attention, check_codes, check_topk_exact_on_scores, check_topk_set, \
    oracle_scores_row
from sparse_attention_prolog_gb300 import binding as B
from sparse_attention_prolog_gb300 import workloads as W
from sparse_attention_prolog_gb300.pipeline import DecodeBuffers, PrologBuffers

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _check_tokens(inp, buf, tokens, q=None, qs=None, w=None, kc=None, ks=None):
    idx = buf.topk_idx.cpu().numpy()
    sc = buf.scores.cpu().numpy() if buf.scores is not None else None
    for t in tokens:
        ref = oracle_scores_row(inp, t, q, qs, w, kc, ks)
        n = int(inp.pos[t]) + 1
        if sc is not None:
            scale = max(np.abs(ref).max(), 1e-30)
            assert np.abs(sc[t, :n] - ref).max() <= 2e-6 * scale, f"t={t} scores"
            check_topk_exact_on_scores(idx[t], sc[t], n, inp.topk, f"t={t}")
        check_topk_set(idx[t], ref, n, inp.topk, f"t={t}")
    if buf.with_attention:
        ref_o, ref_l = O.sparse_attention(inp, idx, tokens)
        check_attention(buf.out.float().cpu().numpy()[tokens], ref_o, buf.lse.cpu().numpy()[tokens], ref_l,
                        "attention")


def test_tiny_decode_chain(cuda_lib):
    inp = W.tiny_decode()
    buf = DecodeBuffers(inp, DEV, keep_scores=True)
    buf.run()
    torch.cuda.synchronize()
    assert B.device_error() == 0
    _check_tokens(inp, buf, range(inp.T))


def test_decode_64k_full_step(cuda_lib):
    """B=4, MTP1, 64K: prolog -> indexer/top-k -> attention, every token."""
    inp = W.decode_64k()
    p = W.decode_64k_prolog()
    kc = torch.from_numpy(inp.k_cache).to(DEV)
    ks = torch.from_numpy(inp.k_scale).to(DEV)
    pro = PrologBuffers(p, DEV, kc, ks)
    buf = DecodeBuffers(inp, DEV, q_idx=pro.q_out, q_idx_scale=pro.q_scale_out, w_idx=pro.w_out, k_cache=kc,
                        k_scale=ks, keep_scores=True)
    pro.run()
    buf.run()
    torch.cuda.synchronize()
    assert B.device_error() == 0
    # prolog stage
    ref_cache = inp.k_cache.copy()
    ref_cs = inp.k_scale.copy()
    ref = O.indexer_prolog(p, ref_cache, ref_cs)
    check_codes(pro.q_out.cpu().numpy(), pro.q_scale_out.cpu().numpy(), ref["q"], ref["q_scale"], "q")
    kc_h = kc.cpu().numpy()
    ks_h = ks.cpu().numpy()
    check_codes(kc_h[p.slot], ks_h[p.slot], ref_cache[p.slot], ref_cs[p.slot], "k")
    assert np.array_equal(np.delete(kc_h, p.slot, axis=0), np.delete(inp.k_cache, p.slot, axis=0))
    # indexer / top-k / attention stages on the prolog's device outputs
    q = pro.q_out.cpu().numpy()
    qs = pro.q_scale_out.cpu().numpy()
    w = pro.w_out.cpu().numpy()
    _check_tokens(inp, buf, list(range(inp.T)), q, qs, w, kc_h, ks_h)


@pytest.mark.slow
def test_causal_prefill_8192_sampled(cuda_lib):
    inp = W.causal_prefill()
    buf = DecodeBuffers(inp, DEV, keep_scores=True)
    buf.run()
    torch.cuda.synchronize()
    assert B.device_error() == 0
    _check_tokens(inp, buf, [0, 1, 2, 127, 1000, 2046, 2047, 2048, 2049, 4095, 6000, 8190, 8191])


@pytest.mark.slow
def test_ragged_paged_decode_sampled(cuda_lib):
    inp = W.ragged_paged_decode()
    buf = DecodeBuffers(inp, DEV, keep_scores=True)
    buf.run()
    torch.cuda.synchronize()
    assert B.device_error() == 0
    lens = inp.seq_len
    picks = sorted({int(np.argmin(lens)), int(np.argmax(lens)), 0, 7, 19, 31})
    _check_tokens(inp, buf, picks)

"""Whole decode steps on the five workloads: each stage is checked against
the oracle fed with the CUDA path's own upstream outputs (stage isolation),
so that legitimate top-k ties do not spread into the attention check."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle as O
from parity_utils import check_attention, check_codes, check_topk_exact_on_scores, check_topk_set, \
    oracle_scores_row
from sparse_attention_prolog_gb300 import binding as B
from sparse_attention_prolog_gb300 import workloads as W
from sparse_attention_prolog_gb300.pipeline import DecodeBuffers, DiaBuffers, PrologBuffers

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


def _bits(t: torch.Tensor) -> np.ndarray:
    """Raw bf16 bits of a device tensor (the oracle takes bf16 inputs as bits)."""
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _close_bf16(gpu, ref, what):
    """Within the bf16 output rounding: |gpu - ref| <= 8e-3 |ref| + 2e-3."""
    err = np.abs(gpu - ref) - (8e-3 * np.abs(ref) + 2e-3)
    assert err.max() <= 0, f"{what}: worst excess {err.max():.3e}"


def test_dia_decode_64k_full_step(cuda_lib):
    """One DeepSeek Indexer Attention step at B=4, MTP1, 64K: MLA Prolog ->
    Indexer Prolog (fed the MLA Prolog's q_lora and hidden states) ->
    Lightning Indexer + top-k -> sparse attention (the MLA Prolog's query
    over the latent cache holding its new rows).  Every stage is checked
    against the oracle fed the CUDA path's own upstream outputs."""
    dia = W.dia_decode()
    inp, mp, pp = dia.decode, dia.mla, dia.prolog
    st = DiaBuffers(dia, DEV, keep_scores=True)
    st.run()
    torch.cuda.synchronize()
    assert B.device_error() == 0
    # MLA Prolog
    ref_m = O.mla_prolog(mp)
    gl, gs = st.mla.q_lora.cpu().numpy(), st.mla.q_lora_scale.cpu().numpy()
    check_codes(gl, gs, ref_m["q_lora"], ref_m["q_lora_scale"], "q_lora")
    q_ref = O.mla_q(gl, gs, mp.w_uq, mp.w_uq_scale, O.bf16_bits_to_f64(mp.w_uk), mp.H, mp.pos, mp.rope_cos,
                    mp.rope_sin, bool(mp.rope_interleaved))
    _close_bf16(st.mla.q.float().cpu().numpy(), q_ref, "attention query")
    kv_bits = _bits(st.kv)
    kv_rows = O.bf16_bits_to_f64(kv_bits[mp.slot])
    _close_bf16(kv_rows, ref_m["kv"], "latent rows")
    others = np.ones(kv_bits.shape[0], bool)
    others[mp.slot] = False
    assert np.array_equal(kv_bits[others], inp.kv_cache[others]), "latent rows without a slot were written"
    # Indexer Prolog on the MLA Prolog's q_lora
    p2 = dataclasses.replace(pp, q_lora=gl, q_lora_scale=gs)
    ref_cache, ref_cs = inp.k_cache.copy(), inp.k_scale.copy()
    ref_p = O.indexer_prolog(p2, ref_cache, ref_cs)
    check_codes(st.pro.q_out.cpu().numpy(), st.pro.q_scale_out.cpu().numpy(), ref_p["q"], ref_p["q_scale"], "q")
    kc_h, ks_h = st.k_cache.cpu().numpy(), st.k_scale.cpu().numpy()
    check_codes(kc_h[pp.slot], ks_h[pp.slot], ref_cache[pp.slot], ref_cs[pp.slot], "k")
    w = st.pro.w_out.cpu().numpy()
    assert np.abs(w - ref_p["w"]).max() <= 1e-4 * max(1.0, np.abs(ref_p["w"]).max())
    # indexer, top-k and attention on the CUDA path's prolog outputs, query
    # and latent cache
    inp2 = dataclasses.replace(inp, q_attn=_bits(st.mla.q), kv_cache=kv_bits)
    _check_tokens(inp2, st.buf, list(range(inp.T)), st.pro.q_out.cpu().numpy(), st.pro.q_scale_out.cpu().numpy(),
                  w, kc_h, ks_h)

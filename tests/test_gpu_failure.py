"""Failure paths on the GPU, made without a fault: a bounded device wait that
runs out (a limit far shorter than the copies it waits for) and a position
outside the RoPE table.  Both are reported through the device error word and
leave the context usable; the next call passes parity."""
import numpy as np
import pytest
import torch

import oracle as O
from parity_utils import check_codes
from sparse_attention_prolog_gb300 import binding as B
from sparse_attention_prolog_gb300 import workloads as W
from sparse_attention_prolog_gb300.pipeline import PrologBuffers

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
DSA_ERR_DEVICE_TIMEOUT = 5
DSA_ERR_DEVICE_DATA = 6


def _prolog(rows=64, large=False):
    """The decode step's prolog (8 tokens), or with large=True one token
    against the largest weights (K_q = 2048, D_x = 12288): each CTA's weight
    copies take microseconds from a cold L2, while the work before its first
    wait (one token's RoPE row) is a single round trip."""
    if large:
        T = 1
        p = W.make_prolog_inputs(T=T, pos=np.arange(1000, 1000 + T), slot=np.arange(T), seed=71, K_q=2048,
                                 D_x=12288, max_pos=2048)
    else:
        p = W.decode_64k_prolog()
    p.slot = np.arange(p.T, dtype=np.int64) * 2  # distinct rows of a small cache
    kc = torch.full((rows, p.d_I), 99, dtype=torch.int8, device=DEV)
    ks = torch.full((rows,), 7.0, dtype=torch.float16, device=DEV)
    return p, PrologBuffers(p, DEV, kc, ks)


def _check_against_oracle(p, buf, tokens, rows=64):
    ref_cache = np.full((rows, p.d_I), 99, np.int8)
    ref_cs = np.full(rows, 7.0, np.float16)
    ref = O.indexer_prolog(p, ref_cache, ref_cs)
    tokens = np.asarray(tokens)
    check_codes(buf.q_out.cpu().numpy()[tokens], buf.q_scale_out.cpu().numpy()[tokens], ref["q"][tokens],
                ref["q_scale"][tokens], "q")
    sl = p.slot[tokens]
    check_codes(buf.k_cache.cpu().numpy()[sl], buf.k_scale_cache.cpu().numpy()[sl], ref_cache[sl], ref_cs[sl], "k")
    wg = buf.w_out.cpu().numpy().astype(np.float64)
    wr = ref["w"].astype(np.float64)
    assert np.abs(wg - wr).max() <= 1e-4 * max(1.0, np.abs(wr).max())


def test_wait_limit_runs_out_then_next_call_passes(cuda_lib):
    """With a 1 ns limit the prolog CTAs give up waiting for their weight
    copies (L2 is flushed first, so they come from HBM and take microseconds):
    the call reports a device timeout.  The CTAs let their copies and MMAs
    finish before leaving, so with the default limit restored the next call on
    the same buffers matches the oracle."""
    p, buf = _prolog(large=True)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=DEV)
    torch.cuda.synchronize()
    assert B.device_error() == 0
    B.set_wait_limit_ns(1)
    try:
        flush.zero_()  # evicts the weights the upload left in L2
        buf.run()
        torch.cuda.synchronize()
        assert B.device_error() == DSA_ERR_DEVICE_TIMEOUT
    finally:
        B.set_wait_limit_ns(0)
    buf.ws.zero_()  # as the header asks after a timed-out call
    buf.q_out.zero_()
    buf.run()
    torch.cuda.synchronize()
    assert B.device_error() == 0
    _check_against_oracle(p, buf, np.arange(p.T))


def test_wait_limit_argument_checks(cuda_lib):
    lib = B.load()
    assert lib.dsa_set_wait_limit_ns(61 * 10 ** 9) == 1  # beyond 60 s: invalid argument
    assert lib.dsa_set_wait_limit_ns(0) == 0


def test_prolog_position_outside_the_rope_table(cuda_lib):
    """pos = rope_max_pos and pos = -1: recorded as invalid device data, the
    two tokens' q and key rows are not written, every other token matches the
    oracle."""
    p, buf = _prolog()
    bad = p.pos.copy()
    bad[3] = p.rope_cos.shape[0]
    bad[5] = -1
    buf.pos.copy_(torch.from_numpy(bad))
    buf.q_out.fill_(0x55)
    buf.run()
    torch.cuda.synchronize()
    assert B.device_error() == DSA_ERR_DEVICE_DATA
    q = buf.q_out.cpu().numpy()
    assert (q[3] == 0x55).all() and (q[5] == 0x55).all()
    kc = buf.k_cache.cpu().numpy()
    assert (kc[p.slot[3]] == 99).all() and (kc[p.slot[5]] == 99).all()
    good = [t for t in range(p.T) if t not in (3, 5)]
    _check_against_oracle(p, buf, good)
    # the same buffers with valid positions again
    buf.pos.copy_(torch.from_numpy(p.pos))
    buf.run()
    torch.cuda.synchronize()
    assert B.device_error() == 0
    _check_against_oracle(p, buf, np.arange(p.T))


def test_wait_limit_runs_out_in_the_decode_step_then_next_step_passes(cuda_lib):
    """The decode step (prolog, indexer + top-k, attention + combine) with a
    1 ns limit after an L2 flush: the waits of the prolog, the indexer and
    the attention give up, each CTA lets its copies and MMAs finish before it
    leaves, and the step reports a device timeout.  With the default limit
    and zeroed workspaces the next step on the same buffers matches the
    oracle (stage by stage on its own upstream outputs)."""
    from parity_utils import check_attention, check_topk_set, oracle_scores_row
    from sparse_attention_prolog_gb300.pipeline import DecodeBuffers
    inp = W.make_decode_inputs(B=2, n_q=2, seq_lens=[8192, 6000], H_I=64, d_I=128, topk=512, H=128, seed=81)
    buf = DecodeBuffers(inp, DEV, keep_scores=True)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=DEV)
    torch.cuda.synchronize()
    assert B.device_error() == 0
    B.set_wait_limit_ns(1)
    try:
        flush.zero_()
        buf.run()
        torch.cuda.synchronize()
        assert B.device_error() == DSA_ERR_DEVICE_TIMEOUT
    finally:
        B.set_wait_limit_ns(0)
    buf.tws.zero_()
    buf.aws.zero_()
    buf.run()
    torch.cuda.synchronize()
    assert B.device_error() == 0
    idx = buf.topk_idx.cpu().numpy()
    sc = buf.scores.cpu().numpy()
    for t in range(inp.T):
        ref = oracle_scores_row(inp, t)
        n = int(inp.pos[t]) + 1
        assert np.abs(sc[t, :n] - ref).max() <= 2e-6 * max(np.abs(ref).max(), 1e-30)
        check_topk_set(idx[t], ref, n, inp.topk, f"t={t}")
    ref_o, ref_l = O.sparse_attention(inp, idx)
    check_attention(buf.out.float().cpu().numpy(), ref_o, buf.lse.cpu().numpy(), ref_l, "attention")


def test_wait_limit_runs_out_in_the_mla_prolog_and_the_int8_gemm(cuda_lib):
    """The MLA Prolog and both int8 GEMM paths (512 rows: tiled; 8 rows: the
    weight stream) with a 1 ns limit report a device timeout; with the
    default limit the next calls give the oracle's q_lora codes and the
    exact GEMMs."""
    from sparse_attention_prolog_gb300.pipeline import MlaBuffers
    T = 8
    p = W.make_mla_inputs(T, np.arange(T) * 5, np.arange(T, dtype=np.int64), seed=82, max_pos=64)
    mla = MlaBuffers(p, DEV, 16)
    M, N, K = 512, 2048, 3072
    r = np.random.default_rng(83)
    a = r.integers(-128, 128, (M, K)).astype(np.int8)
    b = r.integers(-128, 128, (N, K)).astype(np.int8)
    sa = np.full(M, 1.0 / 128, np.float32)
    sb = np.full(N, 1.0 / (128 * K ** 0.5), np.float32)
    ta, tb = torch.from_numpy(a).to(DEV), torch.from_numpy(b).to(DEV)
    tsa, tsb = torch.from_numpy(sa).to(DEV), torch.from_numpy(sb).to(DEV)
    c = torch.zeros((M, N), dtype=torch.float16, device=DEV)
    c8 = torch.zeros((8, N), dtype=torch.float16, device=DEV)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=DEV)
    torch.cuda.synchronize()
    assert B.device_error() == 0
    for run in (lambda: mla.run(), lambda: B.dsa_int8_gemm(ta, tsa, tb, tsb, c),
                lambda: B.dsa_int8_gemm(ta[:8], tsa[:8], tb, tsb, c8)):
        B.set_wait_limit_ns(1)
        try:
            flush.zero_()
            run()
            torch.cuda.synchronize()
            assert B.device_error() == DSA_ERR_DEVICE_TIMEOUT
        finally:
            B.set_wait_limit_ns(0)
    mla.ws.zero_()
    mla.run()
    B.dsa_int8_gemm(ta, tsa, tb, tsb, c)
    B.dsa_int8_gemm(ta[:8], tsa[:8], tb, tsb, c8)
    torch.cuda.synchronize()
    assert B.device_error() == 0
    ref = O.mla_prolog(p)
    check_codes(mla.q_lora.cpu().numpy(), mla.q_lora_scale.cpu().numpy(), ref["q_lora"], ref["q_lora_scale"], "q_lora")
    want = O.int8_gemm(a, sa.astype(np.float64), b, sb.astype(np.float64)).astype(np.float64)
    got = c.cpu().numpy().astype(np.float64)
    assert (np.abs(got - want) <= np.maximum(np.abs(want) * 2.0 ** -10, 2.0 ** -24)).all()
    np.testing.assert_array_equal(c8.cpu().numpy(), c.cpu().numpy()[:8])  # the two paths agree bit for bit


def test_prolog_slot_past_the_cache(cuda_lib):
    """A slot equal to cache_rows: recorded as invalid device data and that
    key row is not written; every other token matches the oracle, and the
    same buffers with valid slots pass again."""
    p, buf = _prolog()
    bad = p.slot.copy()
    bad[2] = 64  # the cache has 64 rows
    buf.slot.copy_(torch.from_numpy(bad))
    buf.run()
    torch.cuda.synchronize()
    assert B.device_error() == DSA_ERR_DEVICE_DATA
    assert (buf.k_cache.cpu().numpy()[p.slot[2]] == 99).all()
    _check_against_oracle(p, buf, [t for t in range(p.T) if t != 2])
    buf.slot.copy_(torch.from_numpy(p.slot))
    buf.run()
    torch.cuda.synchronize()
    assert B.device_error() == 0
    _check_against_oracle(p, buf, np.arange(p.T))


def test_mla_slot_past_the_cache(cuda_lib):
    """The MLA Prolog with a slot equal to cache_rows: recorded, that latent
    row not written, the other rows within the bf16 rounding; then a call
    with valid slots on the same workspace passes."""
    from sparse_attention_prolog_gb300.pipeline import MlaBuffers
    T, rows, fill = 4, 8, 5.0
    p = W.make_mla_inputs(T, np.arange(T) + 10, np.arange(T, dtype=np.int64) * 2, seed=811, H=8, K_q=256, D_x=512,
                          max_pos=64)
    buf = MlaBuffers(p, DEV, rows, fill)
    bad = p.slot.copy()
    bad[1] = rows
    buf.slot.copy_(torch.from_numpy(bad))
    buf.run()
    torch.cuda.synchronize()
    assert B.device_error() == DSA_ERR_DEVICE_DATA
    ref = O.mla_prolog(p)

    def close(tokens):
        kv = buf.kv_cache.float().cpu().numpy().astype(np.float64)
        for t in tokens:
            err = np.abs(kv[p.slot[t]] - ref["kv"][t]) - (8e-3 * np.abs(ref["kv"][t]) + 2e-3)
            assert err.max() <= 0, f"kv row of token {t}"

    assert (buf.kv_cache.float().cpu().numpy()[p.slot[1]] == fill).all()
    close([0, 2, 3])
    buf.slot.copy_(torch.from_numpy(p.slot))
    buf.run()
    torch.cuda.synchronize()
    assert B.device_error() == 0
    close(range(T))


def test_indexer_negative_page_entry(cuda_lib):
    """A visible page of sequence 0 unmapped (-1 in its block table):
    recorded as invalid device data; sequence 1's scores and selection are
    unaffected, and the restored table passes."""
    from parity_utils import check_topk_set, oracle_scores_row
    from sparse_attention_prolog_gb300.pipeline import DecodeBuffers
    inp = W.make_decode_inputs(B=2, n_q=1, seq_lens=[1000, 1500], H_I=64, d_I=128, topk=256, H=8, seed=45,
                               block_size=64, max_L=1536, with_attention=False)
    buf = DecodeBuffers(inp, DEV, with_attention=False, keep_scores=True)

    def check(tokens):
        sc = buf.scores.cpu().numpy()
        idx = buf.topk_idx.cpu().numpy()
        for t in tokens:
            ref = oracle_scores_row(inp, t)
            n = int(inp.pos[t]) + 1
            assert np.abs(sc[t, :n] - ref).max() <= 2e-6 * np.abs(ref).max(), f"t={t}"
            check_topk_set(idx[t], ref, n, inp.topk, f"t={t}")

    bt = inp.block_table.copy()
    bt[0, 3] = -1
    buf.block_table.copy_(torch.from_numpy(bt))
    buf.run_topk()
    torch.cuda.synchronize()
    assert B.device_error() == DSA_ERR_DEVICE_DATA
    check([1])
    buf.block_table.copy_(torch.from_numpy(inp.block_table))
    buf.run_topk()
    torch.cuda.synchronize()
    assert B.device_error() == 0
    check([0, 1])

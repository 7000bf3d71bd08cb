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
    """The decode step's prolog (8 tokens), or with large=True the largest
    supported one: 32 tokens, K_q = 2048, D_x = 12288 (each CTA's copies
    take longest)."""
    if large:
        T = 32
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
    """With a 1 ns limit every prolog CTA gives up waiting for its weight
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

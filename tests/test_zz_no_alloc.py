"""dsa_indexer_prolog_noalloc, for callers that cannot allocate device
memory (a plug-in handed only its tensors, or a loop that must not call
cudaMalloc): its scratch is a fixed array inside the library.  Its output
must match the regular dsa_indexer_prolog's, call after call, because every
call reuses the same array.

Kept in a file that pytest collects last, so that a stop at the first failure
has already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

from parity_utils import check_codes
from sparse_attention_prolog_gb300 import binding as B
from sparse_attention_prolog_gb300 import workloads as W
from sparse_attention_prolog_gb300.pipeline import PrologBuffers

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _outputs(buf):
    torch.cuda.synchronize()
    rows = buf.p.slot[buf.p.slot >= 0]
    return (buf.q_out.cpu().numpy().copy(), buf.q_scale_out.cpu().numpy().copy(),
            buf.k_cache.cpu().numpy()[rows].copy(), buf.k_scale_cache.cpu().numpy()[rows].copy(),
            buf.w_out.cpu().numpy().copy())


def _clear(buf):
    buf.q_out.zero_()
    buf.q_scale_out.zero_()
    buf.k_cache.zero_()
    buf.k_scale_cache.zero_()
    buf.w_out.zero_()


def test_noalloc_prolog_matches_regular_twice(cuda_lib):
    """q rows and scales bit for bit (the q stream sums its int32 partials in
    a fixed order); key rows within one code and weights within fp32
    rounding, because the k / weight stream adds its CTAs' fp32 partial sums
    with atomics in whatever order they finish (two regular calls differ the
    same way)."""
    p = W.decode_64k_prolog()
    p.slot = np.arange(8, dtype=np.int64) * 5  # a small cache: 8 distinct rows in 64
    buf = PrologBuffers(p, DEV, torch.zeros(64, p.d_I, dtype=torch.int8, device=DEV),
                        torch.zeros(64, dtype=torch.float16, device=DEV))
    buf.run()
    ref = _outputs(buf)
    lib = B.load()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        _clear(buf)
        rc = lib.dsa_indexer_prolog_noalloc(ctypes.byref(buf.args), stream)
        assert rc == 0, B.status_string(rc)
        got = _outputs(buf)
        np.testing.assert_array_equal(got[0], ref[0], err_msg=f"q codes (call {call})")
        np.testing.assert_array_equal(got[1], ref[1], err_msg=f"q scales (call {call})")
        check_codes(got[2], got[3], ref[2], ref[3], f"k (call {call})")
        np.testing.assert_allclose(got[4], ref[4], rtol=1e-6, atol=1e-6)
    assert B.device_error() == 0


def test_noalloc_prolog_passes_argument_errors_through(cuda_lib):
    """An unsupported shape (T = 33 tokens) gets the regular entry point's
    status, DSA_ERR_UNSUPPORTED, before anything is enqueued.  (No supported
    shape needs more than the 64 KiB array, so its own size check cannot be
    reached with a valid argument set.)"""
    p = W.decode_64k_prolog()
    p.slot = np.arange(8, dtype=np.int64) * 5
    buf = PrologBuffers(p, DEV, torch.zeros(64, p.d_I, dtype=torch.int8, device=DEV),
                        torch.zeros(64, dtype=torch.float16, device=DEV))
    need = B.workspace_bytes("prolog", buf.args)
    assert 0 < need <= 64 * 1024
    args = B.PrologArgs.from_buffer_copy(buf.args)
    args.T = 33
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert B.load().dsa_indexer_prolog_noalloc(ctypes.byref(args), stream) == 2

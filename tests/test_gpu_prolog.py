"""Indexer Prolog: CUDA path vs oracle (codes within 1 LSB, scales 1e-3)."""
import numpy as np
import pytest
import torch

import oracle as O
from parity_utils import check_codes
from sparse_attention_prolog_gb300 import workloads as W
from sparse_attention_prolog_gb300.pipeline import PrologBuffers

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _run_and_check(p, cuda_lib, cache_rows=None):
    rows = int(p.slot.max()) + 1 if cache_rows is None else cache_rows
    kc = torch.full((rows, p.d_I), 99, dtype=torch.int8, device=DEV)
    ks = torch.full((rows,), 7.0, dtype=torch.float16, device=DEV)
    buf = PrologBuffers(p, DEV, kc, ks)
    buf.run()
    torch.cuda.synchronize()
    from sparse_attention_prolog_gb300 import binding
    assert binding.device_error() == 0
    ref_cache = np.full((rows, p.d_I), 99, np.int8)
    ref_cs = np.full(rows, 7.0, np.float16)
    ref = O.indexer_prolog(p, ref_cache, ref_cs)
    fq = check_codes(buf.q_out.cpu().numpy(), buf.q_scale_out.cpu().numpy(), ref["q"], ref["q_scale"], "q")
    sl = p.slot[p.slot >= 0]
    fk = 0.0
    if sl.size:
        fk = check_codes(kc.cpu().numpy()[sl], ks.cpu().numpy()[sl], ref_cache[sl], ref_cs[sl], "k")
    untouched = np.setdiff1d(np.arange(rows), sl)
    assert (kc.cpu().numpy()[untouched] == 99).all(), "rows without a slot were written"
    if p.w_proj is not None:
        wg = buf.w_out.cpu().numpy().astype(np.float64)
        wr = ref["w"].astype(np.float64)
        assert np.abs(wg - wr).max() <= 1e-4 * max(1.0, np.abs(wr).max())
    return fq, fk


def test_prolog_alone_T8(cuda_lib):
    """T=8 at positions 0..7, H_I=64 x d_I=128, K_q=1536, D_x=7168, no weights."""
    _run_and_check(W.prolog_alone(), cuda_lib)


def test_prolog_decode_with_weights(cuda_lib):
    """The decode step's prolog: positions 65534/65535, cache slots at the
    end of four 64K sequences, weight stream on."""
    p = W.decode_64k_prolog()
    _run_and_check(p, cuda_lib, cache_rows=4 * 65536)


@pytest.mark.parametrize("T", [1, 5, 32])
def test_prolog_token_counts_and_skip_slots(T, cuda_lib):
    pos = (np.arange(T) * 37) % 4096
    slot = np.arange(T, dtype=np.int64) * 3
    slot[::4] = -1  # some tokens write no key
    p = W.make_prolog_inputs(T=T, pos=pos, slot=slot, seed=50 + T, max_pos=4096)
    _run_and_check(p, cuda_lib, cache_rows=3 * T + 1)


def test_prolog_small_heads_interleaved(cuda_lib):
    """d_I=64, H_I=4, interleaved RoPE pairs, smaller K_q / D_x."""
    p = W.make_prolog_inputs(T=6, pos=np.arange(6) * 11, slot=np.arange(6), seed=77, H_I=4, d_I=64,
                             K_q=512, D_x=1024, rope_interleaved=1, max_pos=64)
    _run_and_check(p, cuda_lib)


@pytest.mark.parametrize("d_I", [64, 128])
def test_prolog_128_heads_two_waves(d_I, cuda_lib):
    """H_I=128: 256 q CTAs (more than one wave), 256 k/weight channels, so the
    D_x slices per k/weight CTA hit their shared-memory cap."""
    p = W.make_prolog_inputs(T=3, pos=np.array([5, 900, 4000]), slot=np.array([0, 2, 1]), seed=91, H_I=128,
                             d_I=d_I, K_q=512, D_x=3072, max_pos=4096)
    _run_and_check(p, cuda_lib)


@pytest.mark.parametrize("H_I,d_I", [(64, 128), (128, 64)])
def test_prolog_largest_supported_shape(H_I, d_I, cuda_lib):
    """T = 32 tokens, K_q = 2048, D_x = 12288 (every bound of the header at
    once): the k / weight CTAs take as many D_x atoms as fit beside the
    kernel's static tables, so more of them run than there are spare SMs."""
    T = 32
    p = W.make_prolog_inputs(T=T, pos=np.arange(T) * 61, slot=np.arange(T) * 2, seed=93, H_I=H_I, d_I=d_I,
                             K_q=2048, D_x=12288, max_pos=2048)
    _run_and_check(p, cuda_lib, cache_rows=2 * T)


@pytest.mark.parametrize("H_I,d_I,d_rope,interleaved", [(1, 128, 64, 0), (3, 64, 32, 1), (17, 128, 8, 0),
                                                        (100, 128, 128, 1), (7, 64, 64, 0)])
def test_prolog_head_counts_and_rotary_widths(H_I, d_I, d_rope, interleaved, cuda_lib):
    """Head counts that are not powers of two (one q CTA pair, a few, and
    200 q CTAs in two waves with a weight tile cut at row 100) and rotary
    widths from 8 dims to the whole head, both pair layouts."""
    T = 5
    p = W.make_prolog_inputs(T=T, pos=np.array([0, 3, 77, 500, 1023]), slot=np.array([4, -1, 0, 2, 1]),
                             seed=95 + H_I, H_I=H_I, d_I=d_I, d_rope=d_rope, K_q=1024, D_x=2048,
                             max_pos=1024, rope_interleaved=interleaved)
    _run_and_check(p, cuda_lib, cache_rows=6)


def test_prolog_repeated_calls_share_the_workspace(cuda_lib):
    """The k / weight sums accumulate in the workspace and the call leaves
    it zeroed: three calls on one workspace give the same checked result."""
    p = W.decode_64k_prolog()
    rows = 4 * 65536
    kc = torch.full((rows, p.d_I), 99, dtype=torch.int8, device=DEV)
    ks = torch.full((rows,), 7.0, dtype=torch.float16, device=DEV)
    buf = PrologBuffers(p, DEV, kc, ks)
    ref_cache = np.full((rows, p.d_I), 99, np.int8)
    ref_cs = np.full(rows, 7.0, np.float16)
    ref = O.indexer_prolog(p, ref_cache, ref_cs)
    from sparse_attention_prolog_gb300 import binding
    for _ in range(3):
        buf.run()
        torch.cuda.synchronize()
        assert binding.device_error() == 0
        check_codes(kc.cpu().numpy()[p.slot], ks.cpu().numpy()[p.slot], ref_cache[p.slot], ref_cs[p.slot], "k")
        wg = buf.w_out.cpu().numpy().astype(np.float64)
        wr = ref["w"].astype(np.float64)
        assert np.abs(wg - wr).max() <= 1e-4 * max(1.0, np.abs(wr).max())
    assert (buf.ws == 0).all(), "workspace not left zeroed"


def test_prolog_zero_tokens_is_noop(cuda_lib):
    from sparse_attention_prolog_gb300 import binding as B
    p = W.prolog_alone()
    buf = PrologBuffers(p, DEV)
    buf.args.T = 0
    B.dsa_indexer_prolog(buf.args, buf.ws)
    torch.cuda.synchronize()
    assert (buf.q_out == 0).all()

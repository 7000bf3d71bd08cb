"""Sparse MLA attention: CUDA path vs oracle (max-abs 2e-2, rel-RMS 5e-3)."""
import numpy as np
import pytest
import torch

import oracle as O
from parity_utils import check_attention
from sparse_attention_prolog_gb300 import binding as B
from sparse_attention_prolog_gb300 import workloads as W
from sparse_attention_prolog_gb300.pipeline import DecodeBuffers, to_dev

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _attn_with_idx(inp, idx_np, tokens=None, sink=None):
    buf = DecodeBuffers(inp, DEV, with_attention=True)
    buf.topk_idx.copy_(torch.from_numpy(idx_np.astype(np.int32)))
    if sink is not None:
        sink_dev = torch.from_numpy(np.asarray(sink, np.float32)).to(DEV)
        buf.aargs.sink = sink_dev.data_ptr()
    buf.run_attn()
    torch.cuda.synchronize()
    assert B.device_error() == 0
    tokens = list(range(inp.T)) if tokens is None else tokens
    ref_o, ref_l = O.sparse_attention(inp, idx_np, tokens, sink)
    out = buf.out.float().cpu().numpy()[tokens]
    lse = buf.lse.cpu().numpy()[tokens]
    return check_attention(out, ref_o, lse, ref_l, "attn")


def _random_idx(rng, inp, frac_invalid=0.0):
    idx = np.empty((inp.T, inp.topk), np.int64)
    for t in range(inp.T):
        n = int(inp.pos[t]) + 1
        idx[t] = rng.choice(n, size=inp.topk, replace=n < inp.topk)
        if frac_invalid:
            idx[t, rng.random(inp.topk) < frac_invalid] = -1
    return idx


def test_tiny_heads_single_chunk(cuda_lib):
    inp = W.tiny_decode()
    rng = np.random.default_rng(1)
    _attn_with_idx(inp, _random_idx(rng, inp))


@pytest.mark.parametrize("topk", [64, 200, 1000])
def test_128_heads_chunks_and_ragged_tiles(topk, cuda_lib):
    """128 heads, several split chunks, a ragged last tile, masked slots."""
    inp = W.make_decode_inputs(B=2, n_q=2, seq_lens=[3001, 4096], H_I=4, d_I=64, topk=topk, H=128, seed=21)
    rng = np.random.default_rng(topk)
    _attn_with_idx(inp, _random_idx(rng, inp, frac_invalid=0.1))


def test_all_masked_and_duplicates(cuda_lib):
    inp = W.make_decode_inputs(B=1, n_q=4, seq_lens=[600], H_I=4, d_I=64, topk=96, H=128, seed=22)
    idx = np.full((4, 96), -1, np.int64)          # token 0: nothing selected
    idx[1, :1] = 5                                 # token 1: one row
    idx[2] = 7                                     # token 2: one row, 96 times
    idx[3] = np.random.default_rng(3).integers(0, 597, 96)
    _attn_with_idx(inp, idx)


def test_masked_tails_end_chunks_early(cuda_lib):
    """Chunks of four 64-row tiles (16 tokens, top-1024) whose index rows end
    in masked slots: the chunk stops at its last valid slot, found from the
    chunk's last slot when that is valid and by a scan of the chunk when it
    is not (valid slots after masked ones included)."""
    inp = W.make_decode_inputs(B=2, n_q=8, seq_lens=[3000, 2500], H_I=4, d_I=64, topk=1024, H=128, seed=26)
    rng = np.random.default_rng(26)
    idx = _random_idx(rng, inp)
    idx[0, 300:] = -1                  # a valid prefix: chunk 1 keeps one tile, chunks 2-3 none
    idx[1, 255::256] = -1              # every chunk's last slot masked, the one before valid
    idx[2] = -1
    idx[2, ::256] = 11                 # one valid slot at the start of each chunk
    idx[3] = -1
    idx[3, 190] = 40                   # one valid slot in chunk 0's third tile
    idx[4] = -1                        # nothing selected
    idx[5, rng.random(inp.topk) < 0.3] = -1
    idx[5, 700:] = -1                  # scattered holes, then a masked tail
    idx[6, 1000:1023] = -1             # a valid last slot after masked ones
    _attn_with_idx(inp, idx)


def test_large_scores_trigger_rescale(cuda_lib):
    """Scaled-up q and rope dims make later tiles exceed the running max by
    far more than 2^8, exercising the O rescale path; the value dims keep
    their N(0,1) scale."""
    inp = W.make_decode_inputs(B=1, n_q=2, seq_lens=[2048], H_I=4, d_I=64, topk=512, H=128, seed=23)
    q = O.bf16_bits_to_f64(inp.q_attn) * 6.0
    inp.q_attn = W.f32_to_bf16_bits(q.astype(np.float32))
    kv = O.bf16_bits_to_f64(inp.kv_cache)
    kv[1200:, 512:] *= 8.0                      # rows late in the selection dominate
    inp.kv_cache = W.f32_to_bf16_bits(kv.astype(np.float32))
    idx = np.tile(np.arange(1024, 1536), (2, 1))
    _attn_with_idx(inp, idx)


def test_paged_kv(cuda_lib):
    inp = W.make_decode_inputs(B=3, n_q=1, seq_lens=[700, 2048, 1500], H_I=4, d_I=64, topk=300, H=128,
                               seed=24, block_size=64, max_L=2048)
    rng = np.random.default_rng(5)
    _attn_with_idx(inp, _random_idx(rng, inp))


@pytest.mark.parametrize("block_size", [1, 3, 16, 256])
def test_paged_kv_page_sizes(block_size, cuda_lib):
    """Pages of one row, of an odd row count (max_L = 2049 = 683 pages of
    3), of 16 rows and of 256 rows: each selected row is looked up through
    its own page."""
    max_L = -(-2048 // block_size) * block_size
    inp = W.make_decode_inputs(B=3, n_q=1, seq_lens=[700, 2000, 1500], H_I=4, d_I=64, topk=300, H=128,
                               seed=60 + block_size, block_size=block_size, max_L=max_L)
    rng = np.random.default_rng(block_size)
    _attn_with_idx(inp, _random_idx(rng, inp, frac_invalid=0.05))


@pytest.mark.parametrize("topk", [1, 8192])
def test_extreme_selection_sizes(topk, cuda_lib):
    """One selected row per token, and 8192 rows per token (many split
    chunks merged by the combine), 128 heads."""
    inp = W.make_decode_inputs(B=1, n_q=2, seq_lens=[9000], H_I=4, d_I=64, topk=topk, H=128, seed=70 + topk)
    rng = np.random.default_rng(topk + 1)
    _attn_with_idx(inp, _random_idx(rng, inp))


@pytest.mark.parametrize("H", [1, 64, 100])
def test_head_counts_below_128(H, cuda_lib):
    """Head blocks only partly filled (1, 64 and 100 of 128 rows), over
    several split chunks, with a sink per head for H = 100."""
    inp = W.make_decode_inputs(B=2, n_q=2, seq_lens=[1500, 3000], H_I=4, d_I=64, topk=600, H=H, seed=80 + H)
    rng = np.random.default_rng(H + 3)
    _attn_with_idx(inp, _random_idx(rng, inp, frac_invalid=0.05), sink=_sinks(H, 90) if H == 100 else None)


@pytest.mark.parametrize("topk", [64, 1000])
def test_without_lse_output(topk, cuda_lib):
    """lse = NULL (the output alone), on one chunk per token and on split
    chunks merged by the combine."""
    inp = W.make_decode_inputs(B=2, n_q=2, seq_lens=[3001, 4096], H_I=4, d_I=64, topk=topk, H=128, seed=27)
    buf = DecodeBuffers(inp, DEV, with_attention=True)
    idx = _random_idx(np.random.default_rng(topk + 9), inp, frac_invalid=0.1)
    buf.topk_idx.copy_(torch.from_numpy(idx.astype(np.int32)))
    buf.aargs.lse = None
    buf.lse.fill_(7.0)
    buf.run_attn()
    torch.cuda.synchronize()
    assert B.device_error() == 0
    ref_o, _ = O.sparse_attention(inp, idx, list(range(inp.T)), None)
    check_attention(buf.out.float().cpu().numpy(), ref_o, what="attn without lse")
    assert (buf.lse.cpu().numpy() == 7.0).all()


def test_heads_above_128(cuda_lib):
    inp = W.make_decode_inputs(B=1, n_q=2, seq_lens=[512], H_I=4, d_I=64, topk=128, H=160, seed=25)
    rng = np.random.default_rng(6)
    _attn_with_idx(inp, _random_idx(rng, inp))


def _sinks(H, seed):
    """Per-head sinks around the score range, with a head switched off
    (-inf) and one that dominates its softmax."""
    r = np.random.default_rng(seed)
    sink = r.normal(0.0, 2.0, H)
    sink[0] = -np.inf
    sink[H - 1] = 40.0
    return sink


def test_attention_sink_single_chunk(cuda_lib):
    """The sink applied in the attention epilogue (one chunk per token), a
    token with nothing selected (out 0, lse = sink)."""
    inp = W.tiny_decode()
    rng = np.random.default_rng(31)
    idx = _random_idx(rng, inp)
    idx[1] = -1
    _attn_with_idx(inp, idx, sink=_sinks(inp.H, 32))


@pytest.mark.parametrize("topk", [200, 1000])
def test_attention_sink_split_chunks(topk, cuda_lib):
    """The sink applied once, in the merge of the split chunks."""
    inp = W.make_decode_inputs(B=2, n_q=2, seq_lens=[3001, 4096], H_I=4, d_I=64, topk=topk, H=128, seed=33)
    rng = np.random.default_rng(34 + topk)
    idx = _random_idx(rng, inp, frac_invalid=0.1)
    idx[2] = -1
    _attn_with_idx(inp, idx, sink=_sinks(inp.H, 35))


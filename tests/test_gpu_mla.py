"""MLA Prolog: CUDA path vs the float64 oracle, stage by stage.

q_lora codes within 1 LSB (at most 1 % off by one) and scales within 1e-3
of the oracle's quantisation of its own query latent; the latent-cache rows
and the query (the oracle's up-projection fed the CUDA path's own q_lora)
within the bf16 output rounding: |gpu - ref| <= 8e-3 |ref| + 2e-3 (half a
bf16 ulp is 2^-9 relative; the fp32 sums add ~1e-6)."""
import numpy as np
import pytest
import torch

import oracle as O
from parity_utils import check_codes
from sparse_attention_prolog_gb300 import binding as B
from sparse_attention_prolog_gb300 import workloads as W
from sparse_attention_prolog_gb300.pipeline import MlaBuffers

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
FILL = 5.0  # latent-cache rows without a slot keep this value


def _bf16(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def _close(gpu, ref, what):
    err = np.abs(gpu - ref) - (8e-3 * np.abs(ref) + 2e-3)
    assert err.max() <= 0, f"{what}: worst excess {err.max():.3e} at {np.unravel_index(err.argmax(), err.shape)}"


def _check(p, buf, rows):
    torch.cuda.synchronize()
    assert B.device_error() == 0
    ref = O.mla_prolog(p)
    check_codes(buf.q_lora.cpu().numpy(), buf.q_lora_scale.cpu().numpy(), ref["q_lora"], ref["q_lora_scale"],
                "q_lora")
    gl, gs = buf.q_lora.cpu().numpy(), buf.q_lora_scale.cpu().numpy()
    q_ref = O.mla_q(gl, gs, p.w_uq, p.w_uq_scale, O.bf16_bits_to_f64(p.w_uk), p.H, p.pos, p.rope_cos, p.rope_sin,
                    bool(p.rope_interleaved))
    _close(_bf16(buf.q), q_ref, "q")
    kv = _bf16(buf.kv_cache)
    written = p.slot[p.slot >= 0]
    for t in range(p.T):
        if p.slot[t] >= 0:
            _close(kv[p.slot[t]], ref["kv"][t], f"kv row of token {t}")
    untouched = np.setdiff1d(np.arange(rows), written)
    assert (kv[untouched] == FILL).all(), "rows without a slot were written"
    # the split-K sums are left zeroed for the next call
    sums = buf.ws[:p.T * (p.K_q + 576) * 4].view(torch.float32)
    assert int(torch.count_nonzero(sums)) == 0


@pytest.mark.parametrize("T,H,K_q,D_x,inter", [
    (3, 4, 256, 512, 0),      # every row block, one atom per slice
    (8, 128, 1536, 7168, 0),  # the decode step (B=4, MTP1)
    (17, 16, 2048, 1024, 1),  # 32-token tiles with a ragged tail, the largest K_q, interleaved pairs
    (32, 8, 128, 64, 0),      # the most tokens, one query row block, one atom in all
    (1, 1, 128, 64, 1),       # one token, one head: the smallest call
    (5, 100, 640, 3072, 0),   # a head count that is not a power of two, K_q of five 128-blocks
    (32, 128, 2048, 16384, 1),  # every bound of the header at once
])
def test_mla_matches_oracle(T, H, K_q, D_x, inter, cuda_lib):
    pos = (np.arange(T) * 97 + 11) % 8192
    slot = np.arange(T, dtype=np.int64) * 2 + 1
    slot[1::3] = -1  # some tokens write no latent row
    p = W.make_mla_inputs(T, pos, slot, seed=700 + T, H=H, K_q=K_q, D_x=D_x, max_pos=8192, rope_interleaved=inter)
    rows = 2 * T + 2
    buf = MlaBuffers(p, DEV, rows, FILL)
    buf.run()
    _check(p, buf, rows)


def test_mla_repeated_calls_share_workspace(cuda_lib):
    """Three calls on one workspace (the split-K sums must be cleared by
    each), the second and third with other tokens' inputs."""
    T, rows = 8, 20
    p = W.make_mla_inputs(T, np.arange(T) + 100, np.arange(T, dtype=np.int64), seed=801, H=16, K_q=512, D_x=2048,
                          max_pos=256)
    buf = MlaBuffers(p, DEV, rows, FILL)
    for seed in (801, 802, 803):
        q = W.make_mla_inputs(T, np.arange(T) + seed % 50, np.arange(T, dtype=np.int64), seed=seed, H=16, K_q=512,
                              D_x=2048, max_pos=256)
        q.w_dq, q.w_dkv, q.w_uq, q.w_uq_scale, q.w_uk = p.w_dq, p.w_dkv, p.w_uq, p.w_uq_scale, p.w_uk
        q.gamma_q, q.gamma_kv = p.gamma_q, p.gamma_kv
        buf.x.copy_(torch.from_numpy(q.x.view(np.int16)).view(torch.bfloat16))
        buf.pos.copy_(torch.from_numpy(q.pos))
        buf.run()
        _check(q, buf, rows)

"""Standalone Activation Quantization: CUDA path vs the oracle, bit for bit
(codes and fp32 scales), with and without power-of-two scales."""
import numpy as np
import pytest
import torch

import oracle as O
from sparse_attention_prolog_gb300 import binding as B
from sparse_attention_prolog_gb300.workloads import f32_to_bf16_bits

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _rows(M, N, seed):
    """Rows of standard normals times row magnitudes over many octaves,
    with a zero row, a row with one large outlier and a constant row."""
    r = np.random.default_rng(seed)
    x = r.standard_normal((M, N)) * np.exp(r.uniform(-20, 20, (M, 1)))
    x[0] = 0.0
    if M > 1:
        x[1, N // 2] = 1e4
    if M > 2:
        x[2] = -3.0
    return f32_to_bf16_bits(x.astype(np.float32))


@pytest.mark.parametrize("M,N", [(37, 7168), (5, 8), (3, 32768), (64, 1000), (130, 128)])
@pytest.mark.parametrize("round_scale", [False, True])
def test_act_quant_bit_exact(M, N, round_scale, cuda_lib):
    bits = _rows(M, N, seed=M * 7 + N)
    x = torch.from_numpy(bits.view(np.int16)).to(DEV).view(torch.bfloat16)
    y = torch.full((M, N), 99, dtype=torch.int8, device=DEV)
    s = torch.full((M,), -1.0, dtype=torch.float32, device=DEV)
    B.dsa_act_quant(x, y, s, round_scale)
    torch.cuda.synchronize()
    ry, rs = O.act_quant(bits, round_scale=round_scale)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), rs.view(np.uint32)), "scales differ"
    assert np.array_equal(y.cpu().numpy(), ry), "codes differ"

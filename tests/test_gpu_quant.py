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


@pytest.mark.parametrize("M,N,K", [
    (8, 8192, 1536),     # weight stream: 64 rows of 128 per SM (rows per SM differ by one 16-row unit)
    (1, 100, 16),        # weight stream: a partial block only, one 16-column stage, columns past K zero
    (5, 300, 1008),      # weight stream: K not a multiple of the 128-column stage
    (8, 2000, 8208),     # weight stream: 65 stages, a 1024-K chunk left partial
    (6, 24576, 7168),    # the decode-size GEMM: full and partial blocks per SM
    (3, 24576, 1536),    # the MLA up-projection's shape
    (12, 1000, 4096), (16, 999, 512),  # 16 token rows: all of the MMA's N used
    (8, 300, 65536),     # weight stream at the longest K: 64 exact 1024-K chunks
    (2, 40000, 256),     # weight stream: 256 or 272 rows per SM, a full super-block and a 16-row one
    (32, 256, 7168), (17, 129, 64),    # 32 token rows (N = 32)
    (33, 300, 1008),     # tensor cores: one ragged M tile, an N tail that is not a multiple of 8, K past a 64 stage
    (64, 8192, 1536),    # half an M tile, two 1024-K chunks
    (512, 8192, 1536),
    (4096, 8192, 1536),  # 2048 output tiles
    (130, 136, 4096),    # two M tiles, four chunks
    (64, 256, 65536),    # the longest K: 64 chunks through both accumulators
])
def test_int8_gemm_matches_oracle(M, N, K, cuda_lib):
    """Exact int32 sums, so the fp16 outputs agree to the last place up to
    the fp32 rounding of the dequantisation (at most one fp16 ulp)."""
    r = np.random.default_rng(M * 131 + N + K)
    a = r.integers(-128, 128, (M, K)).astype(np.int8)
    b = r.integers(-128, 128, (N, K)).astype(np.int8)
    sa = r.uniform(0.5, 2.0, M).astype(np.float32) * np.float32(1.0 / 128)
    sb = r.uniform(0.5, 2.0, N).astype(np.float32) / np.float32(128 * max(K, 64) ** 0.5)
    c = torch.full((M, N), float("nan"), dtype=torch.float16, device=DEV)
    B.dsa_int8_gemm(torch.from_numpy(a).to(DEV), torch.from_numpy(sa).to(DEV), torch.from_numpy(b).to(DEV),
                    torch.from_numpy(sb).to(DEV), c)
    torch.cuda.synchronize()
    assert B.device_error() == 0
    ref = O.int8_gemm(a, sa.astype(np.float64), b, sb.astype(np.float64)).astype(np.float64)
    got = c.cpu().numpy().astype(np.float64)
    ulp = np.maximum(np.abs(ref) * 2.0 ** -10, 2.0 ** -24)
    assert np.isfinite(got).all()
    assert (np.abs(got - ref) <= ulp).all(), f"max excess {np.max(np.abs(got - ref) / ulp):.2f} ulp"


@pytest.mark.parametrize("M", [8, 130])
def test_int8_gemm_sums_are_exact_past_fp32_precision(M, cuda_lib):
    """Rows of +-127 against b = 127 whose running sums pass 2^24 (where an
    fp32 accumulator can no longer add 16129 exactly) and end at small
    integers: with unit scales c is the int32 sum itself, so both paths must
    give it exactly (the tensor-core path adds exact 1024-product chunks)."""
    K, N = 4096, 136
    r = np.random.default_rng(M)
    a = np.empty((M, K), np.int8)
    for i in range(M):
        row = np.concatenate([np.full(K // 2, 127), np.full(K // 2, -127)]).astype(np.int64)
        row[-1 - (i % 7)] += 1 + i % 5  # a small remainder
        if i % 2:
            row = row[r.permutation(K)]
        a[i] = row.astype(np.int8)
    b = np.full((N, K), 127, np.int8)
    b[1::3, -1] = 126
    sa = np.ones(M, np.float32)
    sb = np.ones(N, np.float32)
    c = torch.full((M, N), float("nan"), dtype=torch.float16, device=DEV)
    B.dsa_int8_gemm(torch.from_numpy(a).to(DEV), torch.from_numpy(sa).to(DEV), torch.from_numpy(b).to(DEV),
                    torch.from_numpy(sb).to(DEV), c)
    torch.cuda.synchronize()
    assert B.device_error() == 0
    exact = a.astype(np.int64) @ b.astype(np.int64).T
    assert np.abs(exact).max() < 2048  # exactly representable in fp16
    assert (np.abs(np.cumsum(a[0].astype(np.int64) * 127)) > 2 ** 24).any()  # the running sum passes 2^24
    np.testing.assert_array_equal(c.cpu().numpy().astype(np.int64), exact)


def test_int8_gemm_random_shapes_and_paths_agree(cuda_lib):
    """Seeded random shapes on both paths (up to 32 rows the weight stream,
    above the tiled GEMM): exact sums against the oracle, and the first 32
    rows of a 33-row call (tiled) equal a 32-row call (weight stream) bit
    for bit."""
    r = np.random.default_rng(2024)
    for _ in range(12):
        M = int(r.integers(1, 41))
        N = int(r.integers(1, 3000))
        K = 16 * int(r.integers(1, 257))
        a = r.integers(-128, 128, (M, K)).astype(np.int8)
        b = r.integers(-128, 128, (N, K)).astype(np.int8)
        sa = r.uniform(0.5, 2.0, M).astype(np.float32) * np.float32(1.0 / 128)
        sb = r.uniform(0.5, 2.0, N).astype(np.float32) / np.float32(128 * max(K, 64) ** 0.5)
        c = torch.full((M, N), float("nan"), dtype=torch.float16, device=DEV)
        B.dsa_int8_gemm(torch.from_numpy(a).to(DEV), torch.from_numpy(sa).to(DEV), torch.from_numpy(b).to(DEV),
                        torch.from_numpy(sb).to(DEV), c)
        torch.cuda.synchronize()
        assert B.device_error() == 0
        ref = O.int8_gemm(a, sa.astype(np.float64), b, sb.astype(np.float64)).astype(np.float64)
        got = c.cpu().numpy().astype(np.float64)
        ulp = np.maximum(np.abs(ref) * 2.0 ** -10, 2.0 ** -24)
        assert (np.abs(got - ref) <= ulp).all(), f"M={M} N={N} K={K}"
    M, N, K = 33, 777, 1040
    a = r.integers(-128, 128, (M, K)).astype(np.int8)
    b = r.integers(-128, 128, (N, K)).astype(np.int8)
    sa = r.uniform(0.5, 2.0, M).astype(np.float32)
    sb = r.uniform(0.5, 2.0, N).astype(np.float32) / np.float32(128 * 128)
    ta, tb = torch.from_numpy(a).to(DEV), torch.from_numpy(b).to(DEV)
    tsa, tsb = torch.from_numpy(sa).to(DEV), torch.from_numpy(sb).to(DEV)
    c33 = torch.empty((33, N), dtype=torch.float16, device=DEV)
    c32 = torch.empty((32, N), dtype=torch.float16, device=DEV)
    B.dsa_int8_gemm(ta, tsa, tb, tsb, c33)
    B.dsa_int8_gemm(ta[:32].contiguous(), tsa[:32].contiguous(), tb, tsb, c32)
    torch.cuda.synchronize()
    assert B.device_error() == 0
    np.testing.assert_array_equal(c32.cpu().numpy(), c33.cpu().numpy()[:32])


def test_act_quant_at_the_benchmarked_size_sampled(cuda_lib):
    """[16384, 7168], the benchmarked size, in one launch; every row is
    quantised on its own, so 64 sampled rows are compared bit for bit (and
    no code is left at its fill value)."""
    M, N = 16384, 7168
    g = torch.Generator(device="cpu").manual_seed(11)
    x32 = torch.randn((M, N), generator=g) * torch.exp(torch.empty((M, 1)).uniform_(-20, 20, generator=g))
    x = x32.to(torch.bfloat16)
    y = torch.full((M, N), 99, dtype=torch.int8, device=DEV)
    s = torch.full((M,), -1.0, dtype=torch.float32, device=DEV)
    B.dsa_act_quant(x.to(DEV), y, s, False)
    torch.cuda.synchronize()
    rows = np.random.default_rng(12).choice(M, 64, replace=False)
    bits = x[rows].view(torch.int16).numpy().view(np.uint16)
    ry, rs = O.act_quant(bits, round_scale=False)
    assert np.array_equal(s.cpu().numpy()[rows].view(np.uint32), rs.view(np.uint32)), "scales differ"
    assert np.array_equal(y.cpu().numpy()[rows], ry), "codes differ"
    assert (s.cpu().numpy() > 0).all()

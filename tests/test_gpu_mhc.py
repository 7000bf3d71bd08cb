"""Manifold-constrained hyper-connection mappings: CUDA path (fp32) vs the
float64 oracle."""
import numpy as np
import pytest
import torch

import oracle as O
from sparse_attention_prolog_gb300 import binding as B

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.mark.parametrize("hc", [4, 8])
@pytest.mark.parametrize("iters", [0, 3, 20])
def test_mhc_matches_oracle(hc, iters, cuda_lib):
    n = 1000  # not a multiple of the 128-thread block
    r = np.random.default_rng(hc * 10 + iters)
    w = hc * (2 + hc)
    mixes = (r.standard_normal((n, w)) * 2.0).astype(np.float32)
    scale = np.array([0.8, 1.3, 1.7], np.float32)
    base = (r.standard_normal(w) * 0.5).astype(np.float32)
    eps = 1e-6
    d = lambda a: torch.from_numpy(a).to(DEV)
    pre = torch.empty((n, hc), device=DEV)
    post = torch.empty((n, hc), device=DEV)
    comb = torch.empty((n, hc, hc), device=DEV)
    B.dsa_mhc(d(mixes), d(scale), d(base), hc, iters, eps, pre, post, comb)
    torch.cuda.synchronize()
    rp, rq, rc = O.mhc(mixes.astype(np.float64), scale.astype(np.float64), base.astype(np.float64), hc, iters, eps)
    np.testing.assert_allclose(pre.cpu().numpy(), rp, rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(post.cpu().numpy(), rq, rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(comb.cpu().numpy(), rc, rtol=1e-4, atol=1e-6)


@pytest.mark.parametrize("n,iters,eps,mag", [(1, 100, 1e-6, 2.0), (129, 100, 0.0, 2.0), (300, 5, 1e-6, 40.0)])
def test_mhc_limits(n, iters, eps, mag, cuda_lib):
    """One token; the largest round count (100) with and without eps; and
    mixes of magnitude ~40, whose comb logits would overflow exp in fp32
    without the softmax's max shift and whose sigmoids saturate."""
    hc = 4
    r = np.random.default_rng(n + iters)
    w = hc * (2 + hc)
    mixes = (r.standard_normal((n, w)) * mag).astype(np.float32)
    scale = np.array([0.8, 1.3, 1.7], np.float32)
    base = (r.standard_normal(w) * 0.5).astype(np.float32)
    d = lambda a: torch.from_numpy(a).to(DEV)
    pre = torch.empty((n, hc), device=DEV)
    post = torch.empty((n, hc), device=DEV)
    comb = torch.empty((n, hc, hc), device=DEV)
    B.dsa_mhc(d(mixes), d(scale), d(base), hc, iters, eps, pre, post, comb)
    torch.cuda.synchronize()
    rp, rq, rc = O.mhc(mixes.astype(np.float64), scale.astype(np.float64), base.astype(np.float64), hc, iters, eps)
    assert np.isfinite(comb.cpu().numpy()).all()
    np.testing.assert_allclose(pre.cpu().numpy(), rp, rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(post.cpu().numpy(), rq, rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(comb.cpu().numpy(), rc, rtol=1e-4, atol=1e-6)


def test_mhc_at_the_benchmarked_size_sampled(cuda_lib):
    """2^20 tokens, 4 streams, 20 rounds (the benchmarked call) in one
    launch; tokens are independent, so 256 sampled tokens are compared."""
    n, hc, iters, eps = 1 << 20, 4, 20, 1e-6
    w = hc * (2 + hc)
    g = torch.Generator(device="cpu").manual_seed(13)
    mixes = torch.randn((n, w), generator=g) * 2.0
    scale = torch.tensor([0.8, 1.3, 1.7])
    base = torch.randn(w, generator=g) * 0.5
    pre = torch.empty((n, hc), device=DEV)
    post = torch.empty((n, hc), device=DEV)
    comb = torch.empty((n, hc, hc), device=DEV)
    B.dsa_mhc(mixes.to(DEV), scale.to(DEV), base.to(DEV), hc, iters, eps, pre, post, comb)
    torch.cuda.synchronize()
    rows = np.sort(np.random.default_rng(14).choice(n, 256, replace=False))
    rows[-1] = n - 1
    mx = mixes.numpy()[rows].astype(np.float64)
    rp, rq, rc = O.mhc(mx, scale.numpy().astype(np.float64), base.numpy().astype(np.float64), hc, iters, eps)
    np.testing.assert_allclose(pre.cpu().numpy()[rows], rp, rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(post.cpu().numpy()[rows], rq, rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(comb.cpu().numpy()[rows], rc, rtol=1e-4, atol=1e-6)

"""GPU parity of hc_split_sinkhorn (sa_hc_split_sinkhorn) against the CPU oracle.

The kernel computes in f32, as the page does; the oracle in f64 from the same f32 inputs.  Each
comb entry passes through about 2 * iters dependent normalisations of sums of positive terms
(~5 roundings each, no cancellation) after a 2-ulp expf, so its relative error stays near
40 * 5 * 2^-24 ~ 1.2e-5; the test allows |gpu - oracle| <= 1e-6 + 1e-4 * |oracle|."""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import sparse_latent_attention_gb300 as sa
from sparse_latent_attention_gb300 import build

pytestmark = pytest.mark.gpu
ATOL, RTOL = 1e-6, 1e-4


@pytest.fixture(scope="session")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    sa.load()
    return torch.device("cuda:0")


def _close(got, want, what):
    g = got.double().cpu().numpy()
    err = np.abs(g - want)
    bad = ~(err <= ATOL + RTOL * np.abs(want))
    assert not bad.any(), f"{what}: {bad.sum()} out of tolerance, max err {err.max():.3e}"


@pytest.mark.parametrize("shape,spread,iters,eps", [
    ((1,), 1.0, 20, 1e-6),           # one token
    ((1000,), 1.0, 20, 1e-6),        # three full blocks of 256 and a ragged one
    ((4, 8192), 2.0, 20, 1e-6),      # a prefill's tokens, wide logits
    ((300,), 1.0, 1, 1e-2),          # one round, a larger eps
    ((64, 1), 1.0, 7, 1e-6),         # decode tokens, another round count
])
def test_hc_split_sinkhorn_matches_oracle(dev, shape, spread, iters, eps):
    rng = np.random.default_rng(len(shape) * 100 + iters)
    m = (rng.standard_normal(shape + (24,)) * spread).astype(np.float32)
    sc = rng.uniform(0.5, 2.0, 3).astype(np.float32)
    base = (rng.standard_normal(24) * 0.5).astype(np.float32)
    pre, post, comb = sa.hc_split_sinkhorn(torch.from_numpy(m).to(dev), torch.from_numpy(sc).to(dev),
                                           torch.from_numpy(base).to(dev), 4, iters, eps)
    torch.cuda.synchronize()
    wp, wq, wc = oracle.hc_split_sinkhorn(m, sc, base, 4, iters, eps)
    assert pre.shape == shape + (4,) and comb.shape == shape + (4, 4)
    _close(pre, wp, "pre")
    _close(post, wq, "post")
    _close(comb, wc, "comb")


def test_hc_split_sinkhorn_saturated(dev):
    # logits of +-80: the sigmoids saturate (pre -> eps or 1 + eps, post -> 0 or 2) and the row
    # softmax is one-hot before eps; the normalisations still give the oracle's values
    rng = np.random.default_rng(7)
    m = (np.sign(rng.standard_normal((513, 24))) * 40).astype(np.float32)
    sc = np.full(3, 2.0, np.float32)
    base = np.zeros(24, np.float32)
    pre, post, comb = sa.hc_split_sinkhorn(torch.from_numpy(m).to(dev), torch.from_numpy(sc).to(dev),
                                           torch.from_numpy(base).to(dev))
    torch.cuda.synchronize()
    wp, wq, wc = oracle.hc_split_sinkhorn(m, sc, base)
    _close(pre, wp, "pre")
    _close(post, wq, "post")
    _close(comb, wc, "comb")

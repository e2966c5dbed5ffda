"""Backward pass of the shifted-window attention block (V1).

CPU (not gpu): the float64 torch restatement against the pinned forward
oracle, finite differences, and two identities of the gradients.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import backward as obw

RNG = np.random.default_rng(7077)


def _params(C, heads, M, scale=0.3):
    return dict(Wqkv=RNG.normal(size=(3 * C, C)) * scale, bqkv=RNG.normal(size=3 * C) * 0.1,
                table=RNG.normal(size=((2 * M - 1) ** 2, heads)) * 0.3, Wproj=RNG.normal(size=(C, C)) * scale,
                bproj=RNG.normal(size=C) * 0.1)


@pytest.mark.parametrize("B,H,W,C,heads,M,s", [(1, 14, 14, 32, 1, 7, 3), (2, 8, 16, 64, 2, 4, 2),
                                               (1, 6, 6, 32, 2, 3, 0)])
def test_torch_forward_equals_the_pinned_oracle(B, H, W, C, heads, M, s):
    x = RNG.normal(size=(B, H, W, C))
    p = _params(C, heads, M)
    ref = oracle.forward(x, p["Wqkv"], p["bqkv"], p["table"], None, p["Wproj"], p["bproj"], heads=heads, M=M,
                         shift=s, mode=oracle.V1)
    t = {k: torch.tensor(v) for k, v in p.items()}
    got = obw.block_v1(torch.tensor(x), t["Wqkv"], t["bqkv"], t["table"], t["Wproj"], t["bproj"], heads=heads, M=M,
                       shift=s).numpy()
    assert np.allclose(got, ref, rtol=0, atol=1e-12)


def test_gradients_match_finite_differences():
    B, H, W, C, heads, M, s = 1, 6, 6, 8, 2, 3, 1
    x = torch.tensor(RNG.normal(size=(B, H, W, C)), requires_grad=True)
    p = {k: torch.tensor(v, requires_grad=True) for k, v in _params(C, heads, M).items()}

    def f(x, Wqkv, bqkv, table, Wproj, bproj):
        return obw.block_v1(x, Wqkv, bqkv, table, Wproj, bproj, heads=heads, M=M, shift=s)

    assert torch.autograd.gradcheck(f, (x, p["Wqkv"], p["bqkv"], p["table"], p["Wproj"], p["bproj"]), eps=1e-6,
                                    atol=1e-7, rtol=1e-5)


@pytest.mark.parametrize("s", [0, 3])
def test_gradient_identities(s):
    """Each head's table-gradient column sums to zero (a softmax row's logit
    gradients sum to zero); the projection-bias gradient is the token sum of
    the output gradient."""
    B, H, W, C, heads, M = 2, 14, 14, 32, 2, 7
    x = RNG.normal(size=(B, H, W, C))
    dy = RNG.normal(size=(B, H, W, C))
    g = obw.gradients(x, **_params(C, heads, M), dy=dy, heads=heads, M=M, shift=s)
    assert np.allclose(g["dtable"].sum(axis=0), 0.0, atol=1e-9)
    assert np.allclose(g["dbproj"], dy.reshape(-1, C).sum(axis=0), atol=1e-9)
    assert g["dx"].shape == x.shape and g["dWqkv"].shape == (3 * C, C)

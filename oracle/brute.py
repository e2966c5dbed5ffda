"""Window-free NumPy statement of the shifted-window attention block.

TEST INFRASTRUCTURE ONLY (see the package docstring).  It forms no roll, no
partition and no mask.  Shifted windows connect tokens that lie in the same
M x M cell of the grid displaced by s ("Boosting Swin Transformer Speed",
Introduction: windowed attention with shifted windows); the cyclic shift
would also put tokens from opposite image edges into one cell, and the
shift-region mask removes exactly those pairs.  So in the original frame a
query p = (i1, j1) attends to a key q = (i2, j2) of the same image iff

    ((i1 - s) mod H) // M == ((i2 - s) mod H) // M      (same shifted cell)
    ((j1 - s) mod W) // M == ((j2 - s) mod W) // M
    |i1 - i2| < M  and  |j1 - j2| < M                    (no wrap-around)

and its relative position bias is read at the original displacement
(i1 - i2, j1 - j2).  This holds when H >= 2M and W >= 2M (a pair joined only
by the wrap is then at least M + 1 apart), or when s = 0.  Pure Python loops
over tokens: tiny grids only.
"""
from __future__ import annotations

import numpy as np


def allowed_keys(H, W, M, s):
    """Boolean [H*W, H*W] matrix: query p may attend to key q."""
    ii, jj = np.divmod(np.arange(H * W), W)
    cell_i = ((ii - s) % H) // M
    cell_j = ((jj - s) % W) // M
    same = (cell_i[:, None] == cell_i[None, :]) & (cell_j[:, None] == cell_j[None, :])
    near = (np.abs(ii[:, None] - ii[None, :]) < M) & (np.abs(jj[:, None] - jj[None, :]) < M)
    return same & near


def forward(x, Wqkv, bqkv, table, tau, Wproj, bproj, *, heads, M, shift, mode):
    """Same arguments and result as oracle.forward, for tiny grids."""
    x = np.asarray(x, dtype=np.float64)
    B, H, W, C = x.shape
    d = C // heads
    if shift > 0:
        assert H >= 2 * M and W >= 2 * M, "window-free statement needs H, W >= 2M when s > 0"
    Wqkv = np.asarray(Wqkv, np.float64)
    Wproj = np.asarray(Wproj, np.float64)
    bqkv = np.zeros(3 * C) if bqkv is None else np.asarray(bqkv, np.float64)
    bproj = np.zeros(C) if bproj is None else np.asarray(bproj, np.float64)
    table = np.asarray(table, np.float64)
    ok = allowed_keys(H, W, M, shift)
    ii, jj = np.divmod(np.arange(H * W), W)
    out = np.empty_like(x)
    for b in range(B):
        tokens = x[b].reshape(H * W, C)
        qkv = tokens @ Wqkv.T + bqkv
        o = np.zeros((H * W, C))
        for hd in range(heads):
            q = qkv[:, hd * d:(hd + 1) * d]
            k = qkv[:, C + hd * d:C + (hd + 1) * d]
            v = qkv[:, 2 * C + hd * d:2 * C + (hd + 1) * d]
            for p in range(H * W):
                keys = np.nonzero(ok[p])[0]
                logits = np.empty(len(keys))
                for n, key in enumerate(keys):
                    if mode == 1:
                        cos = q[p] @ k[key] / (max(np.sqrt(q[p] @ q[p]), 1e-12)
                                               * max(np.sqrt(k[key] @ k[key]), 1e-12))
                        logit = cos / max(float(tau[hd]), 0.01)
                    else:
                        logit = q[p] @ k[key] / np.sqrt(d)
                    dr, dc = ii[p] - ii[key], jj[p] - jj[key]
                    logits[n] = logit + table[(dr + M - 1) * (2 * M - 1) + (dc + M - 1), hd]
                w = np.exp(logits - logits.max())
                w /= w.sum()
                o[p, hd * d:(hd + 1) * d] = w @ v[keys]
        out[b] = (o @ Wproj.T + bproj).reshape(H, W, C)
    return out

"""Float64 CPU oracle of the backward pass of the shifted-window attention
block (V1: dot-product logits with a learned relative-bias table).

TEST INFRASTRUCTURE ONLY, under the same rule as the rest of this package.

The training result of "Boosting Swin Transformer Speed: Profiling, Mixed
Precision, and Kernel Fusion Secrets" (Training Optimization: the fused MHA
kernel and the index-mapping kernels of window partition, shift and
reverse) needs the gradients of the block.  This module restates the block
with plain PyTorch CPU operations in float64 -- torch.roll for the cyclic
shift, reshape / permute for the window partition and reverse, explicit
relative indices and region masks -- independently of ``swin_oracle.c``,
and takes the gradients with torch.autograd.

Pins in ``tests/test_backward.py``: its forward equals the pinned
``oracle.forward``; gradients match central finite differences
(torch.autograd.gradcheck) on a small grid; each head's column of the table
gradient sums to zero (every softmax row's logit gradients sum to zero);
the projection-bias gradient is the sum of the output gradient over tokens.
"""
from __future__ import annotations

import numpy as np
import torch


def _region_ids(H, W, M, s):
    """Shift region of every position of the shifted frame (0 everywhere
    without a shift): bands [0, n-M), [n-M, n-s), [n-s, n) per axis."""
    def band(n):
        b = torch.zeros(n, dtype=torch.int64)
        if s > 0:
            b[n - M:n - s] = 1
            b[n - s:] = 2
        return b
    return band(H)[:, None] * 3 + band(W)[None, :]


def _rel_index(M):
    """idx(i, j) = (ri - rj + M - 1) * (2M - 1) + (ci - cj + M - 1) for
    in-window tokens i, j (row-major)."""
    r = torch.arange(M).repeat_interleave(M)
    c = torch.arange(M).repeat(M)
    return (r[:, None] - r[None, :] + M - 1) * (2 * M - 1) + (c[:, None] - c[None, :] + M - 1)


def block_v1(x, Wqkv, bqkv, table, Wproj, bproj, *, heads, M, shift):
    """The V1 block in torch (differentiable).  x [B, H, W, C]."""
    B, H, W, C = x.shape
    d, N = C // heads, M * M
    nh, nw = H // M, W // M
    xs = torch.roll(x, shifts=(-shift, -shift), dims=(1, 2))
    win = xs.reshape(B, nh, M, nw, M, C).permute(0, 1, 3, 2, 4, 5).reshape(B * nh * nw, N, C)
    qkv = win @ Wqkv.T + bqkv                                    # [nW, N, 3C]
    q, k, v = (qkv[..., i * C:(i + 1) * C].reshape(-1, N, heads, d).transpose(1, 2) for i in range(3))
    logits = q @ k.transpose(-1, -2) / np.sqrt(d)                # [nW, h, N, N]
    bias = table[_rel_index(M)]                                  # [N, N, h]
    logits = logits + bias.permute(2, 0, 1)[None]
    if shift > 0:
        reg = _region_ids(H, W, M, shift).reshape(nh, M, nw, M).permute(0, 2, 1, 3).reshape(nh * nw, N)
        masked = reg[:, :, None] != reg[:, None, :]              # [nh*nw, N, N]
        masked = masked.repeat(B, 1, 1)[:, None]
        logits = logits.masked_fill(masked, float("-inf"))
    P = torch.softmax(logits, dim=-1)
    o = (P @ v).transpose(1, 2).reshape(-1, N, C)
    y = o @ Wproj.T + bproj
    y = y.reshape(B, nh, nw, M, M, C).permute(0, 1, 3, 2, 4, 5).reshape(B, H, W, C)
    return torch.roll(y, shifts=(shift, shift), dims=(1, 2))


def gradients(x, Wqkv, bqkv, table, Wproj, bproj, dy, *, heads, M, shift):
    """Gradients of sum(block(x) * dy) with respect to x and every parameter,
    as float64 numpy arrays: dict with dx, dWqkv, dbqkv, dtable, dWproj,
    dbproj."""
    t = {n: torch.tensor(np.asarray(a, dtype=np.float64), requires_grad=True)
         for n, a in dict(x=x, Wqkv=Wqkv, bqkv=bqkv, table=table, Wproj=Wproj, bproj=bproj).items()}
    y = block_v1(t["x"], t["Wqkv"], t["bqkv"], t["table"], t["Wproj"], t["bproj"], heads=heads, M=M, shift=shift)
    (y * torch.tensor(np.asarray(dy, dtype=np.float64))).sum().backward()
    return {"d" + n: v.grad.numpy() for n, v in t.items()}

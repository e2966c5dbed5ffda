"""Float64 CPU oracle of the backward pass of the shifted-window attention
block: V1 (dot-product logits with a learned relative-bias table) and V2
(scaled-cosine logits, the table from the meta-network G).

TEST INFRASTRUCTURE ONLY, under the same rule as the rest of this package.

The training result of "Boosting Swin Transformer Speed: Profiling, Mixed
Precision, and Kernel Fusion Secrets" (Training Optimization: the fused MHA
kernel and the index-mapping kernels of window partition, shift and
reverse) needs the gradients of the block.  This module restates the block
with plain PyTorch CPU operations in float64 -- torch.roll for the cyclic
shift, reshape / permute for the window partition and reverse, explicit
relative indices and region masks -- independently of ``swin_oracle.c``,
and takes the gradients with torch.autograd.

V2 ("Swin Transformer V2" (neura.market), How It Works: the logit is the
cosine of query and key divided by a learned per-head tau clipped at 0.01,
plus the bias that G maps from log-spaced relative coordinates): q and k
scaled to unit length (norm clamped at 1e-12), logit = cos / max(tau, 0.01)
+ G-table, no 1/sqrt(d); G(u) = W2 relu(W1 u + b1) over u = (sign(dr)
ln(1+|dr|), sign(dc) ln(1+|dc|)).

Pins in ``tests/test_backward.py``: the forward equals the pinned
``oracle.forward`` (both modes) and the G table the pinned
``oracle.cpb_table``; gradients match central finite differences
(torch.autograd.gradcheck) on small grids; each head's column of the table
gradient sums to zero (every softmax row's logit gradients sum to zero);
the projection-bias gradient is the sum of the output gradient over tokens;
V1's key-bias gradient vanishes; V2's tau gradient equals its closed form
-sum(dS cos) / tau^2, and vanishes below the 0.01 clip.
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
    return _block(x, Wqkv, bqkv, table, None, Wproj, bproj, heads=heads, M=M, shift=shift)


def block_v2(x, Wqkv, bqkv, table, tau, Wproj, bproj, *, heads, M, shift):
    """The V2 block in torch (differentiable); tau [heads]."""
    return _block(x, Wqkv, bqkv, table, tau, Wproj, bproj, heads=heads, M=M, shift=shift)


def cpb_table(W1, b1, W2, *, M):
    """G over the relative coordinates of an M x M window (differentiable):
    [(2M-1)^2, heads], row (dr+M-1)(2M-1) + (dc+M-1)."""
    d = torch.arange(-(M - 1), M, dtype=torch.float64)
    dr, dc = d.repeat_interleave(2 * M - 1), d.repeat(2 * M - 1)
    u = torch.stack([torch.sign(dr) * torch.log1p(dr.abs()), torch.sign(dc) * torch.log1p(dc.abs())], 1)
    return torch.relu(u @ W1.T + b1) @ W2.T


def _block(x, Wqkv, bqkv, table, tau, Wproj, bproj, *, heads, M, shift, aux=None):
    B, H, W, C = x.shape
    d, N = C // heads, M * M
    nh, nw = H // M, W // M
    xs = torch.roll(x, shifts=(-shift, -shift), dims=(1, 2))
    win = xs.reshape(B, nh, M, nw, M, C).permute(0, 1, 3, 2, 4, 5).reshape(B * nh * nw, N, C)
    qkv = win @ Wqkv.T + bqkv                                    # [nW, N, 3C]
    q, k, v = (qkv[..., i * C:(i + 1) * C].reshape(-1, N, heads, d).transpose(1, 2) for i in range(3))
    if tau is None:
        logits = q @ k.transpose(-1, -2) / np.sqrt(d)            # [nW, h, N, N]
    else:
        qn = q / q.norm(dim=-1, keepdim=True).clamp_min(1e-12)
        kn = k / k.norm(dim=-1, keepdim=True).clamp_min(1e-12)
        cos = qn @ kn.transpose(-1, -2)
        logits = cos / tau.clamp_min(0.01)[None, :, None, None]
        if aux is not None:
            aux["cos"] = cos
    bias = table[_rel_index(M)]                                  # [N, N, h]
    logits = logits + bias.permute(2, 0, 1)[None]
    if shift > 0:
        reg = _region_ids(H, W, M, shift).reshape(nh, M, nw, M).permute(0, 2, 1, 3).reshape(nh * nw, N)
        masked = reg[:, :, None] != reg[:, None, :]              # [nh*nw, N, N]
        masked = masked.repeat(B, 1, 1)[:, None]
        logits = logits.masked_fill(masked, float("-inf"))
    if aux is not None and logits.requires_grad:
        logits.retain_grad()
        aux["logits"] = logits
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


def gradients_v2(x, Wqkv, bqkv, tau, W1, b1, W2, Wproj, bproj, dy, *, heads, M, shift):
    """V2: gradients of sum(block(x) * dy) with respect to x, Wqkv, bqkv,
    tau, the table (as the block consumes it), G's W1, b1, W2, Wproj and
    bproj, as float64 numpy arrays (dict; the table gradient under
    "dtable")."""
    t = {n: torch.tensor(np.asarray(a, dtype=np.float64), requires_grad=True)
         for n, a in dict(x=x, Wqkv=Wqkv, bqkv=bqkv, tau=tau, W1=W1, b1=b1, W2=W2, Wproj=Wproj,
                          bproj=bproj).items()}
    table = cpb_table(t["W1"], t["b1"], t["W2"], M=M)
    table.retain_grad()
    aux = {}
    y = _block(t["x"], t["Wqkv"], t["bqkv"], table, t["tau"], t["Wproj"], t["bproj"], heads=heads, M=M,
               shift=shift, aux=aux)
    (y * torch.tensor(np.asarray(dy, dtype=np.float64))).sum().backward()
    out = {"d" + n: v.grad.numpy() for n, v in t.items()}
    out["dtable"] = table.grad.numpy()
    out["table"] = table.detach().numpy()
    # dtau = -sum(dS cos) / tau^2 is a sum with heavy cancellation (every row of
    # dS sums to zero): the size of its terms, sum |dS cos| / tau^2, bounds the
    # effect of rounding the terms
    tau = t["tau"].detach()
    dS = aux["logits"].grad                                  # gradient of the logits (0 where masked)
    terms = (dS * aux["cos"]).abs().sum(dim=(0, 2, 3)).detach()
    out["dtau_terms"] = torch.where(tau > 0.01, terms / tau ** 2, torch.zeros_like(terms)).numpy()
    return out

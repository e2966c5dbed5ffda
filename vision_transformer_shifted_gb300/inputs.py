"""Seeded synthetic inputs for the shifted-window attention block.

This module only draws numbers: it holds none of the block's arithmetic, so
both the GPU library's callers and the float64 oracle take their inputs from
here.  No dataset is used; the shapes stand in for Swin-T / Swin-B at 224^2
and SwinV2 at 1536^2 ("Boost Vision Transformer with GPU-Friendly Sparsity
and Quantization", Fig. 4 (model family); "Swin Transformer V2: Scaling Up
Capacity and Resolution", TLDR (1,536 x 1,536 inputs)).

Recipe (one CPU ``torch.Generator`` per workload, seed 1000 + workload
index): x ~ N(0,1); Wqkv, Wproj ~ N(0, 0.02); bqkv = bproj = 0 (or
N(0, 0.02) with ``nonzero_bias``); V1 relative-bias table ~ N(0, 0.02) of
shape [(2M-1)^2, heads]; V2: tau = 0.1 per head, meta-network weights
W1 [512, 2], W2 [heads, 512] ~ N(0, 0.02) and b1 = 0.  Everything is drawn in
fp32 and rounded once to the workload's dtype; the same rounded values feed
both sides.

The whole block (``generate_block``, the same generator continued, seed
2000 + workload index): LayerNorm gains 1 + N(0, 0.1) and shifts N(0, 0.1);
MLP weights W1 [rC, C] ~ N(0, 1/C), W2 [C, rC] ~ N(0, 1/(rC)) (so that the
MLP branch is of the same order as the main branch, not a vanishing
correction) and biases N(0, 0.02).
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import torch

V1, V2 = 0, 1
CPB_HIDDEN = 512


@dataclass(frozen=True)
class Workload:
    key: str
    name: str
    B: int
    H: int
    W: int
    C: int
    heads: int
    M: int
    shift: int
    mode: int          # V1 or V2
    dtype: str         # "bf16" or "fp32"
    seed: int

    @property
    def d(self):
        return self.C // self.heads

    @property
    def N(self):
        return self.M * self.M

    @property
    def tokens(self):
        return self.B * self.H * self.W

    @property
    def n_windows(self):
        return self.B * (self.H // self.M) * (self.W // self.M)

    @property
    def flops(self):
        """Algorithmic MMA FLOPs: 6TC^2 (QKV) + 4TNC (logits and P.V) + 2TC^2 (proj)."""
        T, C, N = self.tokens, self.C, self.N
        return 8 * T * C * C + 4 * T * N * C

    @property
    def elem_bytes(self):
        return 2 if self.dtype == "bf16" else 4

    @property
    def io_bytes(self):
        """Algorithmic HBM bytes: x read once, out written once, weights, biases
        and the bias table read once."""
        C, e = self.C, self.elem_bytes
        return 2 * self.tokens * C * e + (4 * C * C + 4 * C + (2 * self.M - 1) ** 2 * self.heads) * e

    def with_(self, **kw):
        return replace(self, **kw)


WORKLOADS = {
    "tiny": Workload("tiny", "tiny fp32 V1 block", 1, 14, 14, 32, 1, 7, 3, V1, "fp32", 1000),
    "swin_t_s1": Workload("swin_t_s1", "Swin-T stage-1 shifted block, bf16 V1", 64, 56, 56, 96, 3, 7, 3,
                          V1, "bf16", 1001),
    "swin_b_s1": Workload("swin_b_s1", "Swin-B stage-1 shifted block, bf16 V1", 64, 56, 56, 128, 4, 7, 3,
                          V1, "bf16", 1002),
    "swin_b_s3": Workload("swin_b_s3", "Swin-B stage-3 shifted block, bf16 V1", 64, 14, 14, 512, 16, 7, 3,
                          V1, "bf16", 1002),
    "swinv2_t_s1": Workload("swinv2_t_s1", "SwinV2-T stage-1 shifted block, bf16 V2 cosine", 32, 64, 64, 96,
                            3, 8, 4, V2, "bf16", 1003),
    "swinv2_l_w24": Workload("swinv2_l_w24", "SwinV2-L 1536^2 shifted block, window 24, bf16 V2 cosine", 4,
                             384, 384, 192, 6, 24, 12, V2, "bf16", 1004),
}


def torch_dtype(w: Workload):
    return torch.bfloat16 if w.dtype == "bf16" else torch.float32


def generate(w: Workload, nonzero_bias: bool = False, tau=0.1):
    """Seeded CPU tensors for workload ``w`` (already rounded to its dtype):
    x, Wqkv, bqkv, Wproj, bproj, and either ``table`` (V1) or the meta-network
    weights W1, b1, W2 (V2, the table is built from them) plus ``tau``
    (``tau``: one value for every head, or a sequence of one per head)."""
    g = torch.Generator().manual_seed(w.seed)
    dt = torch_dtype(w)
    C, h, M = w.C, w.heads, w.M

    def normal(shape, std):
        return (torch.randn(shape, generator=g, dtype=torch.float32) * std).to(dt)

    out = {}
    out["x"] = torch.randn((w.B, w.H, w.W, C), generator=g, dtype=torch.float32).to(dt)
    out["Wqkv"] = normal((3 * C, C), 0.02)
    out["bqkv"] = normal((3 * C,), 0.02) if nonzero_bias else torch.zeros(3 * C, dtype=dt)
    out["Wproj"] = normal((C, C), 0.02)
    out["bproj"] = normal((C,), 0.02) if nonzero_bias else torch.zeros(C, dtype=dt)
    if w.mode == V1:
        out["table"] = normal(((2 * M - 1) ** 2, h), 0.02)
        out["tau"] = None
    else:
        out["W1"] = torch.randn((CPB_HIDDEN, 2), generator=g, dtype=torch.float32) * 0.02
        out["b1"] = torch.zeros(CPB_HIDDEN, dtype=torch.float32)
        out["W2"] = torch.randn((h, CPB_HIDDEN), generator=g, dtype=torch.float32) * 0.02
        if isinstance(tau, (int, float)):
            out["tau"] = torch.full((h,), float(tau), dtype=torch.float32)
        else:
            assert len(tau) == h, "one tau per head"
            out["tau"] = torch.tensor([float(t) for t in tau], dtype=torch.float32)
    return out


def sample_windows(w: Workload, count: int, seed: int = 7):
    """Window numbers for sampled parity checks at full size: the four corner
    windows of the first and last image (where the shift mask and the
    wrap-around bite), plus ``count`` seeded random windows."""
    nh, nw = w.H // w.M, w.W // w.M
    per = nh * nw
    fixed = []
    for b in (0, w.B - 1):
        for wi in (0, nh - 1):
            for wj in (0, nw - 1):
                fixed.append(b * per + wi * nw + wj)
    g = torch.Generator().manual_seed(seed)
    rnd = torch.randint(0, w.n_windows, (count,), generator=g).tolist()
    return sorted(set(fixed + rnd))


def generate_block(w: Workload, ratio: int = 4, nonzero_bias: bool = True):
    """Seeded CPU tensors for the whole block of workload ``w`` (bf16): the
    attention inputs of ``generate`` plus ln1_gamma, ln1_beta, ln2_gamma,
    ln2_beta [C], mlp_W1 [rC, C], mlp_b1 [rC], mlp_W2 [C, rC], mlp_b2 [C]."""
    out = generate(w, nonzero_bias=nonzero_bias)
    g = torch.Generator().manual_seed(w.seed + 1000)
    dt = torch_dtype(w)
    C, R = w.C, ratio * w.C

    def normal(shape, std, mean=0.0):
        return (torch.randn(shape, generator=g, dtype=torch.float32) * std + mean).to(dt)

    out["ln1_gamma"] = normal((C,), 0.1, 1.0)
    out["ln1_beta"] = normal((C,), 0.1)
    out["ln2_gamma"] = normal((C,), 0.1, 1.0)
    out["ln2_beta"] = normal((C,), 0.1)
    out["mlp_W1"] = normal((R, C), C ** -0.5)
    out["mlp_b1"] = normal((R,), 0.02)
    out["mlp_W2"] = normal((C, R), R ** -0.5)
    out["mlp_b2"] = normal((C,), 0.02)
    return out

"""Float64 CPU oracle of the whole Swin Transformer block around the
shifted-window attention: LayerNorm, the residual connections and the MLP.

TEST INFRASTRUCTURE ONLY, under the same rule as the rest of this package:
the tests, ``__graft_entry__.smoke()`` and the CPU legs of ``bench.py`` use
it; the GPU library never does, and nothing here imports the library.

The attention sub-layer is ``oracle.forward`` (the float64 block the rest of
the package pins).  Around it ("Swin Transformer V2" (neura.market), How It
Works: the original Swin normalises before each sub-layer; V2 normalises the
output of each residual branch before adding it back to the main branch):

    V1 (pre-norm):           z = x + attn(LN1(x));  y = z + MLP(LN2(z))
    V2 (residual post-norm): z = x + LN1(attn(x));  y = z + LN2(MLP(z))

The pages give no formula for the sub-layers; the readings taken (the plain
transformer-block ones): LayerNorm over the C channels of a token with the
biased variance, eps = 1e-5, per-channel gain and shift; MLP(u) =
GELU(u W1^T + b1) W2^T + b2 with hidden width r*C; GELU the exact form
x * Phi(x), Phi the standard normal CDF.  The extra LayerNorm that V2
inserts every six blocks of its largest models is a stage-level detail and
is not part of one block.

Between stages of the hierarchy ("Boosting Swin Transformer Speed",
Introduction: a pyramid of stages; "Boost Vision Transformer with
GPU-Friendly Sparsity and Quantization", Fig. 4: the number of blocks per
stage) the pages give no formula for the merging step; the reading taken is
the usual one: each 2 x 2 neighbourhood is concatenated in the order (0,0),
(1,0), (0,1), (1,1) (row offset first), normalised over its 4C channels and
mapped to 2C channels by a linear layer without bias.  A stage is ``depth``
blocks with the shift alternating 0, M/2, 0, ... followed (optionally) by
that merging.

Pins in ``tests/test_block.py``: LayerNorm statistics and its affine part,
GELU's odd-part identity and the normal CDF at +-1, +-2 (textbook values),
the MLP against an explicit sum, and closed forms of the whole block when a
sub-layer is switched off.
"""
from __future__ import annotations

import math

import numpy as np

from . import V1, V2, forward

LN_EPS = 1e-5


def layer_norm(x, gamma, beta, eps=LN_EPS):
    """LayerNorm over the last axis: (x - mean) / sqrt(var + eps) * gamma +
    beta, var the biased (1/C) variance."""
    x = np.asarray(x, dtype=np.float64)
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)
    return (x - mu) / np.sqrt(var + eps) * np.asarray(gamma, np.float64) + np.asarray(beta, np.float64)


_erf = np.vectorize(math.erf, otypes=[np.float64])


def gelu(x):
    """Exact GELU: x * Phi(x) = x/2 * (1 + erf(x / sqrt 2))."""
    x = np.asarray(x, dtype=np.float64)
    return 0.5 * x * (1.0 + _erf(x / math.sqrt(2.0)))


def mlp(u, W1, b1, W2, b2):
    """GELU(u W1^T + b1) W2^T + b2 over the last axis of u; W1 [rC, C],
    W2 [C, rC]."""
    u = np.asarray(u, dtype=np.float64)
    h = gelu(u @ np.asarray(W1, np.float64).T + np.asarray(b1, np.float64))
    return h @ np.asarray(W2, np.float64).T + np.asarray(b2, np.float64)


def block(x, p, *, heads, M, shift, mode, attn_out=None):
    """The whole block in float64.  x [B,H,W,C]; ``p`` a dict with ln1_g, ln1_b,
    Wqkv, bqkv, table, tau, Wproj, bproj, ln2_g, ln2_b, W1, b1, W2, b2 (the
    attention entries as ``oracle.forward`` takes them).  ``attn_out``, if
    given, receives the attention sub-layer's output.  Returns (y, z): the
    block output and the main branch after the attention sub-layer."""
    x = np.asarray(x, dtype=np.float64)

    def attn(u):
        a = forward(u, p["Wqkv"], p["bqkv"], p["table"], p["tau"], p["Wproj"], p["bproj"], heads=heads, M=M,
                    shift=shift, mode=mode)
        if attn_out is not None:
            attn_out[...] = a
        return a

    if mode == V1:
        z = x + attn(layer_norm(x, p["ln1_g"], p["ln1_b"]))
        y = z + mlp(layer_norm(z, p["ln2_g"], p["ln2_b"]), p["W1"], p["b1"], p["W2"], p["b2"])
    elif mode == V2:
        z = x + layer_norm(attn(x), p["ln1_g"], p["ln1_b"])
        y = z + layer_norm(mlp(z, p["W1"], p["b1"], p["W2"], p["b2"]), p["ln2_g"], p["ln2_b"])
    else:
        raise ValueError("mode must be V1 or V2")
    return y, z


def merge_concat(x):
    """[B, H, W, C] -> [B, H/2, W/2, 4C]: the 2 x 2 neighbourhood of output
    (i, j) in the order (2i, 2j), (2i+1, 2j), (2i, 2j+1), (2i+1, 2j+1)."""
    x = np.asarray(x, dtype=np.float64)
    B, H, W, C = x.shape
    assert H % 2 == 0 and W % 2 == 0
    out = np.empty((B, H // 2, W // 2, 4 * C))
    for part, (di, dj) in enumerate(((0, 0), (1, 0), (0, 1), (1, 1))):
        out[..., part * C:(part + 1) * C] = x[:, di::2, dj::2, :]
    return out


def patch_merge(x, gamma, beta, Wm):
    """Merging step between stages: LN(merge_concat(x)) Wm^T, Wm [2C, 4C]."""
    return layer_norm(merge_concat(x), gamma, beta) @ np.asarray(Wm, np.float64).T


def stage(x, blocks, *, heads, M, mode, merge=None, extra_norm=None):
    """``len(blocks)`` blocks (parameter dicts as ``block`` takes them) with
    shifts 0, M/2, 0, M/2, ...; then ``patch_merge`` with merge = (gamma, beta,
    Wm) if given.

    extra_norm = (every, [(gamma, beta), ...]): the extra LayerNorm of V2's
    largest models ("Swin Transformer V2" (neura.market), How It Works: a
    layer normalisation inserted every six blocks).  Reading: applied to the
    main branch after blocks every, 2 every, ... (the k-th time with the k-th
    gain and shift), before the merging step."""
    y = np.asarray(x, dtype=np.float64)
    k = 0
    for i, p in enumerate(blocks):
        y, _ = block(y, p, heads=heads, M=M, shift=0 if i % 2 == 0 else M // 2, mode=mode)
        if extra_norm is not None and (i + 1) % extra_norm[0] == 0:
            g, b = extra_norm[1][k]
            y = layer_norm(y, g, b)
            k += 1
    if merge is not None:
        y = patch_merge(y, *merge)
    return y

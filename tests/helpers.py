"""Shared helpers of the GPU parity tests: inputs on the device, float64
oracle references, tolerances."""
import numpy as np
import torch

import oracle
from vision_transformer_shifted_gb300.inputs import V2

# Tolerances against the float64 oracle.  bf16 tensors: max-abs 1e-2 and
# mean-abs 1e-3 (the stated bar), plus a relative L2 bound that bf16
# rounding of q/k/v, P and the output stays well inside.  fp32: 1e-5 max-abs.
BF16_MAX_ABS, BF16_MEAN_ABS, BF16_REL_L2 = 1e-2, 1e-3, 3e-2
FP32_MAX_ABS = 1e-5


def to_f64(t):
    return None if t is None else t.double().cpu().numpy()


def device_inputs(g, dev="cuda"):
    return {k: (v.to(dev) if v is not None else None) for k, v in g.items()}


def oracle_table(w, g):
    """Bias table as the forward consumes it (same dtype as x): V1 draws it,
    V2 builds it with the oracle's G and rounds it once."""
    if w.mode != V2:
        return g["table"]
    t = oracle.cpb_table(to_f64(g["W1"]), to_f64(g["b1"]), to_f64(g["W2"]), M=w.M, heads=w.heads)
    return torch.from_numpy(t).to(g["x"].dtype)


def oracle_forward(w, g, table, windows=None, Wproj=None, bproj="same"):
    a = {k: to_f64(v) for k, v in g.items() if k in ("x", "Wqkv", "bqkv", "tau", "Wproj", "bproj")}
    Wp = a["Wproj"] if Wproj is None else Wproj
    bp = a["bproj"] if isinstance(bproj, str) else bproj
    return oracle.forward(a["x"], a["Wqkv"], a["bqkv"], to_f64(table), a.get("tau"), Wp, bp,
                          heads=w.heads, M=w.M, shift=w.shift, mode=w.mode, windows=windows)


def window_tokens(w, windows):
    """Flat token indices (b*H*W + i*W + j) of the listed windows, in window
    order, from the oracle's own roll and partition."""
    idx = np.arange(w.B * w.H * w.W, dtype=np.float64).reshape(w.B, w.H, w.W, 1)
    xw = oracle.partition(oracle.roll(idx, -w.shift), w.M)
    return xw[np.asarray(windows)].astype(np.int64).reshape(-1)


def compare(got, ref, dtype):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape
    assert np.isfinite(got).all(), "non-finite output"
    err = np.abs(got - ref)
    stats = dict(max_abs=float(err.max()), mean_abs=float(err.mean()),
                 rel_l2=float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)))
    if dtype == "fp32":
        assert stats["max_abs"] <= FP32_MAX_ABS, stats
    else:
        assert stats["max_abs"] <= BF16_MAX_ABS, stats
        assert stats["mean_abs"] <= BF16_MEAN_ABS, stats
        assert stats["rel_l2"] <= BF16_REL_L2, stats
    print("parity", stats)
    return stats

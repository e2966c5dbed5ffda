"""The whole Swin block around the attention (LayerNorm, residuals, MLP).

CPU (not gpu): the float64 block oracle against what the mathematics fixes
-- LayerNorm statistics, GELU's odd part and the normal CDF at a few
points, an MLP that reduces to the identity, closed forms of the block with
the attention switched off -- and the C ABI's argument checks.
GPU: the LayerNorm kernel and the whole block, through the C ABI, against
the oracle.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import block as ob
from vision_transformer_shifted_gb300 import binding as sw
from vision_transformer_shifted_gb300.inputs import V1, V2, WORKLOADS, generate_block

from helpers import oracle_table, to_f64

DEV = "cuda"
RNG = np.random.default_rng(20261202)

# ---- oracle pins (CPU) ---------------------------------------------------------


def test_layer_norm_statistics_and_affine_part():
    x = RNG.normal(size=(64, 96)) * 3.0 + 1.5
    y = ob.layer_norm(x, np.ones(96), np.zeros(96))
    var = x.var(axis=-1)                                  # biased
    assert np.allclose(y.mean(axis=-1), 0.0, atol=1e-12)
    # the normalised row has variance var / (var + eps): catches an unbiased
    # variance or eps taken outside the square root
    assert np.allclose(y.var(axis=-1), var / (var + ob.LN_EPS), rtol=1e-12)
    g, b = RNG.normal(size=96), RNG.normal(size=96)
    assert np.allclose(ob.layer_norm(x, g, b), y * g + b, rtol=0, atol=1e-12)
    # a constant row normalises to the shift
    assert np.allclose(ob.layer_norm(np.full((1, 8), 7.0), g[:8], b[:8]), b[:8], atol=1e-12)


def test_gelu_is_x_times_normal_cdf():
    x = RNG.normal(size=1000) * 4
    # odd part: GELU(x) - GELU(-x) = x (Phi(x) + Phi(-x) = 1)
    assert np.allclose(ob.gelu(x) - ob.gelu(-x), x, atol=1e-12)
    # standard normal CDF at 1 and 2 (textbook values); a tanh approximation
    # misses these by ~1e-4
    assert abs(ob.gelu(1.0) - 0.8413447460685429) < 1e-14
    assert abs(ob.gelu(-1.0) + 0.15865525393145707) < 1e-14
    assert abs(ob.gelu(2.0) - 2 * 0.9772498680518208) < 1e-13
    assert ob.gelu(0.0) == 0.0


def test_mlp_reduces_to_identity_through_gelus_odd_part():
    C = 8
    I = np.eye(C)
    W1, W2 = np.vstack([I, -I]), np.hstack([I, -I])       # [2C, C], [C, 2C]
    u = RNG.normal(size=(10, C)) * 2
    b2 = RNG.normal(size=C)
    assert np.allclose(ob.mlp(u, W1, np.zeros(2 * C), W2, b2), u + b2, atol=1e-12)
    # with a first-layer bias [c; -c] the pair sees u + c: the MLP is u + c
    # (a bias applied after the GELU would give u + 2c)
    c = RNG.normal(size=C)
    assert np.allclose(ob.mlp(u, W1, np.concatenate([c, -c]), W2, np.zeros(C)), u + c, atol=1e-12)
    # even part: GELU(u) + GELU(-u) = u erf(u / sqrt 2)
    even = ob.mlp(u, W1, np.zeros(2 * C), np.hstack([I, I]), np.zeros(C))
    erf = np.vectorize(math.erf)
    assert np.allclose(even, u * erf(u / math.sqrt(2.0)), atol=1e-12)


def _tiny_params(C, heads, M, mode, zero_attention):
    W1, W2 = np.vstack([np.eye(C), -np.eye(C)]), np.hstack([np.eye(C), -np.eye(C)])
    p = dict(ln1_g=1 + 0.1 * RNG.normal(size=C), ln1_b=0.1 * RNG.normal(size=C),
             ln2_g=1 + 0.1 * RNG.normal(size=C), ln2_b=0.1 * RNG.normal(size=C),
             Wqkv=RNG.normal(size=(3 * C, C)) * 0.2, bqkv=RNG.normal(size=3 * C) * 0.02,
             table=RNG.normal(size=((2 * M - 1) ** 2, heads)) * 0.1, tau=None if mode == V1 else np.full(heads, 0.3),
             Wproj=np.zeros((C, C)) if zero_attention else RNG.normal(size=(C, C)) * 0.2,
             bproj=np.zeros(C) if zero_attention else RNG.normal(size=C) * 0.02,
             W1=W1, b1=np.zeros(2 * C), W2=W2, b2=np.zeros(C))
    return p


@pytest.mark.parametrize("mode", [V1, V2])
def test_block_closed_forms_with_attention_off(mode):
    """Attention output 0 and an identity MLP: V1 y = x + LN2(x); V2 (LN of a
    zero vector is its shift) z = x + beta1, y = z + LN2(z)."""
    B, H, W, C, heads, M, s = 1, 14, 14, 32, 1, 7, 3
    x = RNG.normal(size=(B, H, W, C))
    p = _tiny_params(C, heads, M, mode, zero_attention=True)
    y, z = ob.block(x, p, heads=heads, M=M, shift=s, mode=mode)
    if mode == V1:
        assert np.allclose(z, x, atol=1e-12)
    else:
        assert np.allclose(z, x + p["ln1_b"], atol=1e-12)
    assert np.allclose(y, z + ob.layer_norm(z, p["ln2_g"], p["ln2_b"]), atol=1e-12)


@pytest.mark.parametrize("mode", [V1, V2])
def test_block_attention_branch_placement(mode):
    """V1 feeds LN1(x) to the attention and adds its output; V2 feeds x and
    adds LN1 of its output (so, with unit gain and zero shift, z - x is a
    normalised vector: mean 0 per token)."""
    B, H, W, C, heads, M, s = 1, 14, 14, 32, 1, 7, 3
    x = RNG.normal(size=(B, H, W, C))
    p = _tiny_params(C, heads, M, mode, zero_attention=False)
    if mode == V2:
        p["ln1_g"], p["ln1_b"] = np.ones(C), np.zeros(C)
        p["ln2_g"], p["ln2_b"] = np.ones(C), np.zeros(C)
        p["b2"] = RNG.normal(size=C)   # identity MLP plus a shift: MLP(z) = z + b2
    a = np.empty_like(x)
    y, z = ob.block(x, p, heads=heads, M=M, shift=s, mode=mode, attn_out=a)
    if mode == V1:
        ref = oracle.forward(ob.layer_norm(x, p["ln1_g"], p["ln1_b"]), p["Wqkv"], p["bqkv"], p["table"], p["tau"],
                             p["Wproj"], p["bproj"], heads=heads, M=M, shift=s, mode=mode)
        assert np.allclose(z - x, ref, atol=1e-12)
        # identity MLP: the second sub-layer adds LN2 of the main branch z (not of x)
        assert np.allclose(y - z, ob.layer_norm(z, p["ln2_g"], p["ln2_b"]), atol=1e-12)
    else:
        assert np.allclose((z - x).mean(axis=-1), 0.0, atol=1e-12)
        assert np.allclose(z - x, ob.layer_norm(a, np.ones(C), np.zeros(C)), atol=1e-12)
        # the second branch is normalised after the MLP: LN(z + b2), mean 0 per
        # token (an MLP after the LayerNorm would give LN(z) + b2)
        assert np.allclose((y - z).mean(axis=-1), 0.0, atol=1e-12)
        assert np.allclose(y - z, ob.layer_norm(z + p["b2"], np.ones(C), np.zeros(C)), atol=1e-12)


def test_merge_concat_matches_a_reshape_statement():
    """The 2 x 2 concatenation as a reshape: [B, H/2, 2, W/2, 2, C] with the
    column offset outer and the row offset inner in the channel dimension."""
    B, H, W, C = 2, 6, 8, 3
    x = RNG.normal(size=(B, H, W, C))
    ref = x.reshape(B, H // 2, 2, W // 2, 2, C).transpose(0, 1, 3, 4, 2, 5).reshape(B, H // 2, W // 2, 4 * C)
    assert np.array_equal(ob.merge_concat(x), ref)
    # every input element appears exactly once
    assert np.allclose(np.sort(ob.merge_concat(x).ravel()), np.sort(x.ravel()))


def test_patch_merge_selects_normalised_channels():
    """With unit gain, zero shift and Wm selecting channels, the output is those
    channels of the normalised concatenation (mean 0 over the 4C channels)."""
    B, H, W, C = 1, 4, 4, 8
    x = RNG.normal(size=(B, H, W, C)) * 2 + 1
    Wm = np.zeros((2 * C, 4 * C))
    Wm[np.arange(2 * C), np.arange(2 * C)] = 1.0
    out = ob.patch_merge(x, np.ones(4 * C), np.zeros(4 * C), Wm)
    u = ob.merge_concat(x)
    n = (u - u.mean(-1, keepdims=True)) / np.sqrt(u.var(-1, keepdims=True) + ob.LN_EPS)
    assert np.allclose(out, n[..., :2 * C], atol=1e-12)
    assert out.shape == (B, H // 2, W // 2, 2 * C)


def test_stage_alternates_shifts_starting_unshifted():
    B, H, W, C, heads, M = 1, 14, 14, 32, 1, 7
    x = RNG.normal(size=(B, H, W, C))
    p0 = _tiny_params(C, heads, M, V1, zero_attention=False)
    p1 = _tiny_params(C, heads, M, V1, zero_attention=False)
    y = ob.stage(x, [p0, p1], heads=heads, M=M, mode=V1)
    y0, _ = ob.block(x, p0, heads=heads, M=M, shift=0, mode=V1)
    y1, _ = ob.block(y0, p1, heads=heads, M=M, shift=M // 2, mode=V1)
    assert np.allclose(y, y1, atol=1e-12)
    y_wrong, _ = ob.block(ob.block(x, p0, heads=heads, M=M, shift=M // 2, mode=V1)[0], p1, heads=heads, M=M, shift=0,
                          mode=V1)
    assert not np.allclose(y, y_wrong, atol=1e-6)


def test_stage_extra_norm_every_six_blocks():
    """V2's extra LayerNorm: after block 6 of a stage, not before and not when
    the stage has fewer blocks; with gain 1 and shift 0 each output token then
    has mean 0 and variance var / (var + eps) exactly (a LayerNorm's output),
    which the stage without it does not."""
    B, H, W, C, heads, M = 1, 8, 8, 32, 1, 4
    x = RNG.normal(size=(B, H, W, C))
    blocks = [_tiny_params(C, heads, M, V2, zero_attention=False) for _ in range(7)]
    one, zero = np.ones(C), np.zeros(C)
    gam, bet = 1 + 0.1 * RNG.normal(size=C), 0.1 * RNG.normal(size=C)
    plain6 = ob.stage(x, blocks[:6], heads=heads, M=M, mode=V2)
    # placement: LN of the main branch after block 6
    y6 = ob.stage(x, blocks[:6], heads=heads, M=M, mode=V2, extra_norm=(6, [(gam, bet)]))
    assert np.allclose(y6, ob.layer_norm(plain6, gam, bet), atol=1e-12)
    # five blocks: nothing inserted
    y5 = ob.stage(x, blocks[:5], heads=heads, M=M, mode=V2, extra_norm=(6, [(gam, bet)]))
    assert np.array_equal(y5, ob.stage(x, blocks[:5], heads=heads, M=M, mode=V2))
    # block 7 runs on the normalised branch
    y7 = ob.stage(x, blocks, heads=heads, M=M, mode=V2, extra_norm=(6, [(gam, bet)]))
    assert np.allclose(y7, ob.block(y6, blocks[6], heads=heads, M=M, shift=0, mode=V2)[0], atol=1e-12)
    # the closed form of a LayerNorm's output rows
    yn = ob.stage(x, blocks[:6], heads=heads, M=M, mode=V2, extra_norm=(6, [(one, zero)]))
    var = plain6.var(axis=-1)
    assert np.allclose(yn.mean(axis=-1), 0.0, atol=1e-12)
    assert np.allclose(yn.var(axis=-1), var / (var + ob.LN_EPS), atol=1e-12)
    assert not np.allclose(plain6.mean(axis=-1), 0.0, atol=1e-3)


# ---- C ABI argument checks (CPU) ---------------------------------------------------


def test_block_create_rejects_bad_arguments():
    lib = sw.load()
    h = ctypes.c_void_p(123)
    assert lib.swin_block_create(ctypes.byref(h), 96, 3, 7, 3, sw.V1, 0) == sw.EINVAL      # mlp_ratio
    assert h.value is None
    assert lib.swin_block_create(ctypes.byref(h), 96, 3, 7, 3, sw.V1, 9) == sw.EINVAL
    assert lib.swin_block_create(ctypes.byref(h), 96, 3, 7, 3, sw.V1 | sw.FP32, 4) == sw.EUNSUPPORTED
    assert lib.swin_block_create(ctypes.byref(h), 100, 3, 7, 3, sw.V1, 4) == sw.EINVAL     # C % 16
    assert lib.swin_block_create(None, 96, 3, 7, 3, sw.V1, 4) == sw.EINVAL
    assert lib.swin_block_forward(None, None, 1, 7, 7, None, None, None) == sw.EINVAL
    assert lib.swin_block_destroy(None) == sw.OK


def test_merge_rejects_bad_arguments():
    lib = sw.load()
    h = ctypes.c_void_p(123)
    assert lib.swin_merge_create(ctypes.byref(h), 100) == sw.EINVAL      # C % 8
    assert h.value is None
    assert lib.swin_merge_create(ctypes.byref(h), 1024) == sw.EINVAL     # 4C > 2048
    assert lib.swin_merge_create(None, 96) == sw.EINVAL
    assert lib.swin_merge_forward(None, None, 1, 8, 8, None, None, None, None, None) == sw.EINVAL
    assert lib.swin_merge_destroy(None) == sw.OK


def test_stage_norm_rejects_bad_arguments():
    lib = sw.load()
    p16, p32 = ctypes.c_void_p(16), ctypes.c_void_p(32)
    assert lib.swin_stage_norm(p16, 4, 100, p16, p16, p16, None) == sw.EINVAL   # C % 8
    assert lib.swin_stage_norm(p16, -1, 96, p16, p16, p16, None) == sw.EINVAL   # rows
    assert lib.swin_stage_norm(None, 4, 96, p16, p16, p16, None) == sw.EINVAL
    assert lib.swin_stage_norm(ctypes.c_void_p(18), 4, 96, p16, p16, p32, None) == sw.EINVAL   # misaligned
    assert lib.swin_stage_norm(p16, 4, 96, p16, p16, p32, None) == sw.EINVAL   # partial overlap
    assert lib.swin_stage_norm(p16, 0, 96, p16, p16, p16, None) == sw.OK


def test_block_layernorm_hook_rejects_bad_arguments():
    lib = sw.load()
    p16 = ctypes.c_void_p(16)
    assert lib.swin_block_test_layernorm(p16, None, p16, p16, None, p16, 4, 100, 0, None) == sw.EINVAL  # C % 8
    assert lib.swin_block_test_layernorm(p16, None, p16, p16, None, p16, 4, 96, 3, None) == sw.EINVAL   # flags
    assert lib.swin_block_test_layernorm(p16, None, p16, p16, None, p16, 4, 96, 1, None) == sw.EINVAL   # b missing
    assert lib.swin_block_test_layernorm(ctypes.c_void_p(18), None, p16, p16, None, p16, 4, 96, 0,
                                         None) == sw.EINVAL                                              # alignment
    assert lib.swin_block_test_layernorm(p16, None, p16, p16, None, p16, 0, 96, 0, None) == sw.OK     # no rows


# ---- GPU parity ------------------------------------------------------------------------

def _bf16(a):
    return torch.from_numpy(np.asarray(a, dtype=np.float32)).to(torch.bfloat16)


def _block_compare(got, ref, mode=V1):
    """bf16 block output vs float64: the residual stream z, the LayerNorm
    outputs, the GELU activations and y are each rounded to bf16 once (2^-9
    relative each), so the bounds scale with |y|.  In V2 the LayerNorm after
    the attention rescales a small branch (std ~0.05) to unit variance, so the
    attention's own relative error (~0.4% rel-L2, bf16 q/k/v/P, the logits
    scaled by 1/tau = 10) reaches the main branch as ~4e-3 rms absolute:
    hence the mean bound 2^-8 mean|y| + 2e-3, and a per-element allowance of
    0.05 in V2 (about ten times that rms: the whole full-size output, 12.6 M
    elements, reaches 0.046) against 0.02 in V1."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert np.isfinite(got).all()
    err = np.abs(got - ref)
    stats = dict(max_abs=float(err.max()), mean_abs=float(err.mean()),
                 rel_l2=float(np.linalg.norm(got - ref) / np.linalg.norm(ref)))
    assert (err <= 2.0 ** -7 * np.abs(ref) + (5e-2 if mode == V2 else 2e-2)).all(), stats
    assert stats["mean_abs"] <= 2.0 ** -8 * float(np.abs(ref).mean()) + 2e-3, stats
    assert stats["rel_l2"] <= 1e-2, stats
    print("block parity", stats)


@pytest.mark.gpu
@pytest.mark.parametrize("C", [96, 128, 192, 512])
@pytest.mark.parametrize("flags", [0, 1, 2])
def test_layernorm_kernel(C, flags):
    rows = 1000
    a = _bf16(RNG.normal(size=(rows, C)) * 2 + 0.5)
    b = _bf16(RNG.normal(size=(rows, C)))
    g = _bf16(1 + 0.1 * RNG.normal(size=C))
    be = _bf16(0.1 * RNG.normal(size=C))
    out_sum = torch.empty(rows, C, dtype=torch.bfloat16, device=DEV)
    out_ln = torch.empty(rows, C, dtype=torch.bfloat16, device=DEV)
    sw.swin_block_test_layernorm(a.to(DEV), b.to(DEV), g.to(DEV), be.to(DEV), out_sum if flags == 1 else None,
                                 out_ln, flags)
    torch.cuda.synchronize()
    A, Bm, G, Be = (to_f64(t) for t in (a, b, g, be))
    if flags == 1:
        s = (a.float() + b.float()).to(torch.bfloat16)   # the sum is stored, and normalised, as bf16
        assert torch.equal(out_sum.cpu(), s)
        ref = ob.layer_norm(to_f64(s), G, Be)
    elif flags == 2:
        ref = Bm + ob.layer_norm(A, G, Be)
    else:
        ref = ob.layer_norm(A, G, Be)
    err = np.abs(to_f64(out_ln.cpu()) - ref)
    assert (err <= 2.0 ** -8 * np.abs(ref) + 2e-3).all(), float(err.max())


def _block_params_dev(g, table):
    return dict(ln1_gamma=g["ln1_gamma"], ln1_beta=g["ln1_beta"], Wqkv=g["Wqkv"], bqkv=g["bqkv"], bias_table=table,
                logit_scale=g["tau"], Wproj=g["Wproj"], bproj=g["bproj"], ln2_gamma=g["ln2_gamma"],
                ln2_beta=g["ln2_beta"], W1=g["mlp_W1"], b1=g["mlp_b1"], W2=g["mlp_W2"], b2=g["mlp_b2"])


def _oracle_params(g, table):
    return dict(ln1_g=to_f64(g["ln1_gamma"]), ln1_b=to_f64(g["ln1_beta"]), Wqkv=to_f64(g["Wqkv"]),
                bqkv=to_f64(g["bqkv"]), table=to_f64(table), tau=None if g["tau"] is None else to_f64(g["tau"]),
                Wproj=to_f64(g["Wproj"]), bproj=to_f64(g["bproj"]), ln2_g=to_f64(g["ln2_gamma"]),
                ln2_b=to_f64(g["ln2_beta"]), W1=to_f64(g["mlp_W1"]), b1=to_f64(g["mlp_b1"]), W2=to_f64(g["mlp_W2"]),
                b2=to_f64(g["mlp_b2"]))


def _run_block(w, g, table, ratio=4):
    dev = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in _block_params_dev(g, table).items()}
    x = g["x"].to(DEV)
    out = torch.empty_like(x)
    h = sw.swin_block_create(w.C, w.heads, w.M, w.shift, w.mode, ratio)
    try:
        sw.swin_block_forward(h, x, dev, out)
        sw.swin_block_sync_status(h)
    finally:
        sw.swin_block_destroy(h)
    return out.cpu()


@pytest.mark.gpu
@pytest.mark.parametrize("key,B,H,W", [("swin_t_s1", 2, 14, 21), ("swinv2_t_s1", 1, 16, 24), ("swin_t_s1", 1, 7, 7),
                                       ("swin_b_s1", 1, 14, 14), ("swin_b_s1", 8, 56, 56), ("swin_b_s3", 2, 14, 14),
                                       ("swinv2_b_s1", 2, 16, 24), ("swin_c64", 3, 14, 21), ("swinv2_c64", 2, 16, 16)])
def test_block_forward_small(key, B, H, W):
    """Grids of one to two tiles per CTA.  Where the attention is the fused
    kernel (C = 64, 96, 128 with windows of 7 or 8) the block folds LayerNorm 1
    and the first residual into it; V2 at C = 128 and the C = 512 stage take
    the separate LayerNorm kernel."""
    if key == "swinv2_b_s1":   # V2 at C = 128, four heads
        w = WORKLOADS["swinv2_t_s1"].with_(B=B, H=H, W=W, C=128, heads=4)
    elif key in ("swin_c64", "swinv2_c64"):   # C = 64, two heads (the fused MLP's second shape)
        w = WORKLOADS["swin_t_s1" if key == "swin_c64" else "swinv2_t_s1"].with_(B=B, H=H, W=W, C=64, heads=2)
    else:
        w = WORKLOADS[key].with_(B=B, H=H, W=W)
    g = generate_block(w)
    table = oracle_table(w, g)
    got = _run_block(w, g, table)
    ref, _ = ob.block(to_f64(g["x"]), _oracle_params(g, table), heads=w.heads, M=w.M, shift=w.shift, mode=w.mode)
    _block_compare(to_f64(got), ref, w.mode)


@pytest.mark.gpu
@pytest.mark.parametrize("key,C,heads,want", [("swin_t_s1", 96, 3, 2), ("swinv2_t_s1", 96, 3, 2),
                                              ("swin_t_s1", 64, 2, 2), ("swinv2_t_s1", 64, 2, 2),
                                              ("swin_b_s1", 128, 4, 4), ("swinv2_t_s1", 128, 4, 5),
                                              ("swin_b_s3", 512, 16, None)])
def test_block_launches_show_the_fusions(key, C, heads, want):
    """Where the attention is the fused kernel, LayerNorm 1 and the first
    residual are inside it; where the MLP's weights fit one SM (C = 64, 96) the
    MLP is one kernel with LayerNorm 2 and the second residual inside it: two
    launches in either mode.  C = 128: attention, LayerNorm 2, two GEMMs (V2
    without the fold: attention, LayerNorm, two GEMMs, LayerNorm); C = 512:
    the unfused sequence."""
    w = WORKLOADS[key].with_(B=1, H=2 * WORKLOADS[key].M, W=2 * WORKLOADS[key].M, C=C, heads=heads)
    g = generate_block(w)
    table = oracle_table(w, g)
    dev = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in _block_params_dev(g, table).items()}
    x = g["x"].to(DEV)
    out = torch.empty_like(x)
    h = sw.swin_block_create(w.C, w.heads, w.M, w.shift, w.mode, 4)
    try:
        assert sw.swin_block_last_launches(h) == 0
        sw.swin_block_forward(h, x, dev, out)
        sw.swin_block_sync_status(h)
        n = sw.swin_block_last_launches(h)
    finally:
        sw.swin_block_destroy(h)
    assert (n == want) if want else (n >= 7), n


@pytest.mark.gpu
@pytest.mark.parametrize("key", ["swin_t_s1", "swinv2_t_s1", "swin_b_s1"])
def test_overlapped_block_calls_give_the_same_bits(key):
    """SWIN_BLOCK_OPT_OVERLAP_CALLS lets each of the block's fused kernels start
    while the kernel before it finishes: three chained blocks on one stream
    (each block's x the previous block's output, so every kernel reads what
    the one before wrote) give the bits of the same blocks without it."""
    w = WORKLOADS[key].with_(B=4)
    g = generate_block(w)
    table = oracle_table(w, g)
    dev = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in _block_params_dev(g, table).items()}
    x = g["x"].to(DEV)

    def chain(overlap):
        h = sw.swin_block_create(w.C, w.heads, w.M, w.shift, w.mode, 4)
        try:
            sw.swin_block_set_option(h, sw.BLOCK_OPT_OVERLAP_CALLS, overlap)
            outs, cur = [], x
            for _ in range(3):
                o = torch.full_like(x, float("nan"))
                sw.swin_block_forward(h, cur, dev, o)
                outs.append(o)
                cur = o
            assert sw.swin_block_sync_status(h) == sw.OK
            return outs
        finally:
            sw.swin_block_destroy(h)

    plain, overlapped = chain(0), chain(1)
    for a, b in zip(plain, overlapped):
        assert torch.equal(a, b)


@pytest.mark.gpu
@pytest.mark.parametrize("key", ["swin_t_s1", "swinv2_t_s1"])
def test_block_forward_full_size(key):
    """Full-size grid, every output element against the block oracle."""
    w = WORKLOADS[key]
    g = generate_block(w)
    table = oracle_table(w, g)
    got = to_f64(_run_block(w, g, table))
    ref, _ = ob.block(to_f64(g["x"]), _oracle_params(g, table), heads=w.heads, M=w.M, shift=w.shift, mode=w.mode)
    _block_compare(got, ref, w.mode)


def _merge_inputs(C, seed):
    g = torch.Generator().manual_seed(seed)
    gam = (1 + 0.1 * torch.randn(4 * C, generator=g)).bfloat16()
    bet = (0.1 * torch.randn(4 * C, generator=g)).bfloat16()
    Wm = (torch.randn(2 * C, 4 * C, generator=g) * (4 * C) ** -0.5).bfloat16()
    return gam, bet, Wm


@pytest.mark.gpu
@pytest.mark.parametrize("B,H,W,C", [(2, 56, 56, 96), (1, 28, 42, 192), (3, 14, 14, 384), (1, 2, 2, 32)])
def test_merge_forward(B, H, W, C):
    x = torch.randn(B, H, W, C, generator=torch.Generator().manual_seed(B + H + C)).bfloat16()
    gam, bet, Wm = _merge_inputs(C, 5 + C)
    out = torch.empty(B, H // 2, W // 2, 2 * C, dtype=torch.bfloat16, device=DEV)
    h = sw.swin_merge_create(C)
    try:
        sw.swin_merge_forward(h, x.to(DEV), gam.to(DEV), bet.to(DEV), Wm.to(DEV), out)
        torch.cuda.synchronize()
    finally:
        sw.swin_merge_destroy(h)
    ref = ob.patch_merge(to_f64(x), to_f64(gam), to_f64(bet), to_f64(Wm))
    _block_compare(to_f64(out.cpu()), ref)


@pytest.mark.gpu
@pytest.mark.parametrize("mode", [V1, V2])
def test_stage_forward(mode):
    """A stage of depth 2 (unshifted block, shifted block) and the merging step,
    composed from the C ABI calls, against the oracle's stage."""
    key = "swin_t_s1" if mode == V1 else "swinv2_t_s1"
    w0 = WORKLOADS[key].with_(B=1, H=4 * WORKLOADS[key].M, W=2 * WORKLOADS[key].M)
    p_blocks, dev_blocks = [], []
    for i in range(2):
        wi = w0.with_(shift=0 if i == 0 else w0.M // 2, seed=w0.seed + 17 * i)
        g = generate_block(wi)
        table = oracle_table(wi, g)
        p_blocks.append(_oracle_params(g, table))
        dev_blocks.append((wi, {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v)
                               for k, v in _block_params_dev(g, table).items()}))
        if i == 0:
            x = g["x"]
    gam, bet, Wm = _merge_inputs(w0.C, 99)
    cur = x.to(DEV)
    for wi, params in dev_blocks:
        nxt = torch.empty_like(cur)
        h = sw.swin_block_create(wi.C, wi.heads, wi.M, wi.shift, wi.mode, 4)
        try:
            sw.swin_block_forward(h, cur, params, nxt)
            sw.swin_block_sync_status(h)
        finally:
            sw.swin_block_destroy(h)
        cur = nxt
    out = torch.empty(w0.B, w0.H // 2, w0.W // 2, 2 * w0.C, dtype=torch.bfloat16, device=DEV)
    hm = sw.swin_merge_create(w0.C)
    try:
        sw.swin_merge_forward(hm, cur, gam.to(DEV), bet.to(DEV), Wm.to(DEV), out)
        torch.cuda.synchronize()
    finally:
        sw.swin_merge_destroy(hm)
    ref = ob.stage(to_f64(x), p_blocks, heads=w0.heads, M=w0.M, mode=w0.mode,
                   merge=(to_f64(gam), to_f64(bet), to_f64(Wm)))
    _block_compare(to_f64(out.cpu()), ref)


@pytest.mark.gpu
def test_stage_with_extra_norm_forward():
    """A V2 stage of seven blocks with the extra LayerNorm after the sixth
    (swin_stage_norm in place on the main branch) and the merging step,
    against the oracle's stage."""
    key = "swinv2_t_s1"
    M = WORKLOADS[key].M
    w0 = WORKLOADS[key].with_(B=1, H=2 * M, W=2 * M)
    p_blocks, dev_blocks = [], []
    for i in range(7):
        wi = w0.with_(shift=0 if i % 2 == 0 else M // 2, seed=w0.seed + 31 * i)
        g = generate_block(wi)
        table = oracle_table(wi, g)
        p_blocks.append(_oracle_params(g, table))
        dev_blocks.append((wi, {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v)
                               for k, v in _block_params_dev(g, table).items()}))
        if i == 0:
            x = g["x"]
    gn = torch.Generator().manual_seed(123)
    gam = (1 + 0.1 * torch.randn(w0.C, generator=gn)).bfloat16()
    bet = (0.1 * torch.randn(w0.C, generator=gn)).bfloat16()
    mg, mb, mW = _merge_inputs(w0.C, 77)
    cur = x.to(DEV)
    for i, (wi, params) in enumerate(dev_blocks):
        nxt = torch.empty_like(cur)
        h = sw.swin_block_create(wi.C, wi.heads, wi.M, wi.shift, wi.mode, 4)
        try:
            sw.swin_block_forward(h, cur, params, nxt)
            sw.swin_block_sync_status(h)
        finally:
            sw.swin_block_destroy(h)
        cur = nxt
        if i == 5:
            sw.swin_stage_norm(cur, gam.to(DEV), bet.to(DEV), cur)
    out = torch.empty(w0.B, w0.H // 2, w0.W // 2, 2 * w0.C, dtype=torch.bfloat16, device=DEV)
    hm = sw.swin_merge_create(w0.C)
    try:
        sw.swin_merge_forward(hm, cur, mg.to(DEV), mb.to(DEV), mW.to(DEV), out)
        torch.cuda.synchronize()
    finally:
        sw.swin_merge_destroy(hm)
    ref = ob.stage(to_f64(x), p_blocks, heads=w0.heads, M=w0.M, mode=w0.mode,
                   merge=(to_f64(mg), to_f64(mb), to_f64(mW)), extra_norm=(6, [(to_f64(gam), to_f64(bet))]))
    _block_compare(to_f64(out.cpu()), ref, w0.mode)

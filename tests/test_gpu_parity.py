"""GPU parity: every kernel against the float64 oracle, through the C ABI.

Index maps are compared bit-exactly on integer-tagged tokens (through the
stage hooks, and through the whole forward with one-hot attention);
floating-point results within the tolerances in tests/helpers.py.  Small
cases span several 128-row tiles and a ragged tail; the full-size workloads
are compared on every output element.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from vision_transformer_shifted_gb300 import binding as sw
from vision_transformer_shifted_gb300.inputs import V1, V2, WORKLOADS, generate

from helpers import compare, device_inputs, oracle_forward, oracle_table, to_f64

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    sw.load()


def run_forward(w, t, table, path=sw.PATH_AUTO):
    h = sw.swin_wattn_create(w.C, w.heads, w.M, w.shift, w.mode | (sw.FP32 if w.dtype == "fp32" else 0))
    try:
        if path:
            sw.swin_wattn_set_option(h, sw.OPT_PATH, path)
        out = torch.full_like(t["x"], float("nan"))
        sw.swin_wattn_forward(h, t["x"], t["Wqkv"], t["bqkv"], table, t.get("tau"), t["Wproj"], t["bproj"], out)
        assert sw.swin_wattn_sync_status(h) == sw.OK
        return out
    finally:
        sw.swin_wattn_destroy(h)


# ---- the tensor-core GEMM building block ------------------------------------

@pytest.mark.parametrize("swizzle", [128, 64])
@pytest.mark.parametrize("rows,N,K", [(128, 64, 64), (300, 288, 96), (77, 16, 16), (1000, 1536, 512),
                                      (513, 576, 192), (256, 384, 128), (129, 96, 32)])
def test_gemm_block(rows, N, K, swizzle):
    g = torch.Generator().manual_seed(rows + N + K)
    A = torch.randn(rows, K, generator=g).bfloat16()
    Bw = (torch.randn(N, K, generator=g) * 0.1).bfloat16()
    bias = (torch.randn(N, generator=g) * 0.1).bfloat16()
    D = torch.empty(rows, N, dtype=torch.bfloat16, device=DEV)
    sw.swin_wattn_test_gemm(A.to(DEV), Bw.to(DEV), bias.to(DEV), D, swizzle)
    torch.cuda.synchronize()
    ref = A.double() @ Bw.double().T + bias.double()
    err = (D.double().cpu() - ref).abs()
    # one bf16 rounding of the fp32 result (relative 2^-9) plus fp32 accumulation
    assert (err <= ref.abs() * 2.0 ** -8 + 1e-4).all(), float(err.max())


@pytest.mark.parametrize("rows,N,K", [(128, 32, 32), (200, 32, 128), (77, 64, 64), (300, 64, 112)])
def test_gemm_b_mn_major(rows, N, K):
    """An N-major B operand (64-byte swizzle): B given as [K, N] row-major."""
    g = torch.Generator().manual_seed(11 * rows + N + K)
    A = torch.randn(rows, K, generator=g).bfloat16()
    Bkn = (torch.randn(K, N, generator=g) * 0.1).bfloat16()
    bias = (torch.randn(N, generator=g) * 0.1).bfloat16()
    D = torch.empty(rows, N, dtype=torch.bfloat16, device=DEV)
    # the hook reads N from Bw.shape[0]: pass a [N, K]-shaped view of the [K, N] data
    Ad, Bd, bd = A.to(DEV), Bkn.to(DEV), bias.to(DEV)
    rc = sw.load().swin_wattn_test_gemm(ctypes.c_void_p(Ad.data_ptr()), ctypes.c_void_p(Bd.data_ptr()),
                                        ctypes.c_void_p(bd.data_ptr()), ctypes.c_void_p(D.data_ptr()),
                                        rows, N, K, -64, None)
    assert rc == sw.OK
    torch.cuda.synchronize()
    ref = A.double() @ Bkn.double() + bias.double()
    err = (D.double().cpu() - ref).abs()
    assert (err <= ref.abs() * 2.0 ** -8 + 1e-4).all(), float(err.max())


@pytest.mark.parametrize("rows,N,K", [(128, 32, 32), (200, 128, 128), (77, 256, 64), (384, 96, 96)])
def test_gemm_a_from_tmem(rows, N, K):
    """The MMA form that reads A from tensor memory (two bf16 of K per column)."""
    g = torch.Generator().manual_seed(7 * rows + N + K)
    A = torch.randn(rows, K, generator=g).bfloat16()
    Bw = (torch.randn(N, K, generator=g) * 0.1).bfloat16()
    bias = (torch.randn(N, generator=g) * 0.1).bfloat16()
    D = torch.empty(rows, N, dtype=torch.bfloat16, device=DEV)
    sw.swin_wattn_test_gemm(A.to(DEV), Bw.to(DEV), bias.to(DEV), D, 0)
    torch.cuda.synchronize()
    ref = A.double() @ Bw.double().T + bias.double()
    err = (D.double().cpu() - ref).abs()
    assert (err <= ref.abs() * 2.0 ** -8 + 1e-4).all(), float(err.max())


@pytest.mark.parametrize("rows,N,K", [(128, 64, 32), (256, 64, 96), (200, 128, 128), (77, 32, 64)])
def test_gemm_lane_masked_pair(rows, N, K):
    """Two MMAs into the same accumulator columns with complementary lane masks:
    rows 0..63 of every 128-row block against one B, rows 64..127 against another
    (both MMA forms: A from shared memory and A from tensor memory)."""
    g = torch.Generator().manual_seed(13 * rows + N + K)
    A = torch.randn(rows, K, generator=g).bfloat16()
    B2 = (torch.randn(2 * N, K, generator=g) * 0.1).bfloat16()
    D = torch.empty(rows, 2 * N, dtype=torch.bfloat16, device=DEV)
    Ad, Bd = A.to(DEV), B2.to(DEV)
    rc = sw.load().swin_wattn_test_gemm(ctypes.c_void_p(Ad.data_ptr()), ctypes.c_void_p(Bd.data_ptr()), None,
                                        ctypes.c_void_p(D.data_ptr()), rows, N, K, 1, None)
    assert rc == sw.OK
    torch.cuda.synchronize()
    top = (torch.arange(rows) % 128) < 64
    ref = torch.where(top[:, None], A.double() @ B2[:N].double().T, A.double() @ B2[N:].double().T)
    got = D.double().cpu()
    for part in range(2):
        err = (got[:, part * N:(part + 1) * N] - ref).abs()
        assert (err <= ref.abs() * 2.0 ** -8 + 1e-4).all(), (part, float(err.max()))


# ---- index maps, bit-exact ----------------------------------------------------

def tagged(B, H, W, C):
    """Integer-valued tokens (exact in bf16): channels 0..2 carry b, i, j."""
    b, i, j, c = np.meshgrid(np.arange(B), np.arange(H), np.arange(W), np.arange(C), indexing="ij")
    x = ((b * 7 + i * 3 + j * 5 + c * 11) % 61 - 30).astype(np.float64)
    x[..., 0] = b[..., 0]
    x[..., 1] = i[..., 0] % 251
    x[..., 2] = j[..., 0] % 251 + 0.5 * (i[..., 0] // 251)
    return x


@pytest.mark.parametrize("B,H,W,C,M,s", [(2, 14, 21, 96, 7, 3), (1, 16, 24, 64, 8, 4), (2, 14, 14, 96, 7, 0),
                                         (1, 48, 48, 64, 24, 12)])
def test_qkv_gather_and_proj_scatter_bit_exact(B, H, W, C, M, s):
    heads = C // 32
    h = sw.swin_wattn_create(C, heads, M, s, V1)
    try:
        x = tagged(B, H, W, C)
        xt = torch.from_numpy(x).bfloat16().to(DEV)
        Wqkv = torch.zeros(3 * C, C, dtype=torch.bfloat16)
        Wqkv[:C] = torch.eye(C)
        qkv = torch.full((B * H * W, 3 * C), float("nan"), dtype=torch.bfloat16, device=DEV)
        sw.swin_wattn_test_qkv(h, xt, Wqkv.to(DEV), None, qkv)
        # projection with the identity on a window-ordered tagged tensor
        attn = torch.from_numpy(tagged(1, B * H * W, 1, C).reshape(B * H * W, C)).bfloat16().to(DEV)
        out = torch.full((B, H, W, C), float("nan"), dtype=torch.bfloat16, device=DEV)
        sw.swin_wattn_test_proj(h, attn, B, H, W, torch.eye(C).bfloat16().to(DEV), None, out)
        assert sw.swin_wattn_sync_status(h) == sw.OK
    finally:
        sw.swin_wattn_destroy(h)
    want_q = oracle.partition(oracle.roll(x, -s), M).reshape(B * H * W, C)
    got = qkv.double().cpu().numpy()
    assert np.array_equal(got[:, :C], want_q)
    assert np.array_equal(got[:, C:], np.zeros((B * H * W, 2 * C)))
    want_out = oracle.roll(oracle.reverse(attn.double().cpu().numpy().reshape(-1, M * M, C), B, H, W, M), s)
    assert np.array_equal(out.double().cpu().numpy(), want_out)


# ---- attention stage alone ------------------------------------------------------

@pytest.mark.parametrize("key,B,H,W", [("swin_t_s1", 2, 14, 21), ("swinv2_t_s1", 1, 16, 24),
                                       ("swinv2_l_w24", 1, 48, 72)])
def test_attention_stage(key, B, H, W):
    w = WORKLOADS[key].with_(B=B, H=H, W=W)
    g = generate(w, nonzero_bias=True)
    table = oracle_table(w, g)
    t = device_inputs(g)
    h = sw.swin_wattn_create(w.C, w.heads, w.M, w.shift, w.mode)
    try:
        qkv = torch.empty(w.tokens, 3 * w.C, dtype=torch.bfloat16, device=DEV)
        attn = torch.full((w.tokens, w.C), float("nan"), dtype=torch.bfloat16, device=DEV)
        sw.swin_wattn_test_qkv(h, t["x"], t["Wqkv"], t["bqkv"], qkv)
        sw.swin_wattn_test_attn(h, qkv, B, H, W, table.to(DEV), t.get("tau"), attn)
        assert sw.swin_wattn_sync_status(h) == sw.OK
    finally:
        sw.swin_wattn_destroy(h)
    # oracle o in window order: forward with Wproj = I, bproj = 0, then roll(-s) + partition
    o_img = oracle_forward(w, g, table, Wproj=np.eye(w.C), bproj=None)
    o_win = oracle.partition(oracle.roll(o_img, -w.shift), w.M).reshape(w.tokens, w.C)
    compare(attn.double().cpu().numpy(), o_win, "bf16")


# ---- whole block, small grids (several tiles, ragged tails) ----------------------

SMALL = [
    ("swin_t_s1", 2, 14, 21, False), ("swin_t_s1", 3, 7, 21, True),     # odd window count
    ("swin_b_s1", 2, 28, 28, True), ("swin_b_s1", 3, 21, 14, True),   # C = 128: one tile in flight
    ("swin_b_s3", 3, 14, 14, False),
    ("swinv2_t_s1", 2, 16, 24, True), ("swinv2_t_s1", 1, 8, 8, False),   # one window, mask everywhere
    ("swinv2_l_w24", 1, 48, 48, True),
]


PATHS = [sw.PATH_AUTO, sw.PATH_THREE_KERNELS]


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("key,B,H,W,bias", SMALL)
def test_forward_small(key, B, H, W, bias, path):
    w = WORKLOADS[key].with_(B=B, H=H, W=W)
    g = generate(w, nonzero_bias=bias)
    table = oracle_table(w, g)
    out = run_forward(w, device_inputs(g), table.to(DEV), path)
    compare(out.double().cpu().numpy(), oracle_forward(w, g, table), w.dtype)


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("key,B,H,W", [("swin_t_s1", 1, 7, 7), ("swin_t_s1", 1, 14, 7), ("swinv2_t_s1", 3, 8, 24),
                                       ("swin_t_s1", 5, 21, 14)])
def test_forward_ragged_tiles(key, B, H, W, path):
    """Window counts 1, 2, 9 and 30: a lone window in the last two-window
    tile, tiles per CTA > 1 on small grids, images that end mid-tile."""
    w = WORKLOADS[key].with_(B=B, H=H, W=W, shift=min(WORKLOADS[key].shift, 3) if H > 7 else 0)
    g = generate(w, nonzero_bias=True)
    table = oracle_table(w, g)
    out = run_forward(w, device_inputs(g), table.to(DEV), path)
    compare(out.double().cpu().numpy(), oracle_forward(w, g, table), w.dtype)


def test_fused_path_is_chosen_where_supported():
    for key, want in [("swin_t_s1", sw.PATH_FUSED), ("swinv2_t_s1", sw.PATH_FUSED), ("swin_b_s1", sw.PATH_FUSED),
                      ("swin_b_s3", 1), ("swinv2_l_w24", 1), ("tiny", sw.PATH_FP32)]:
        w = WORKLOADS[key]
        h = sw.swin_wattn_create(w.C, w.heads, w.M, w.shift, w.mode | (sw.FP32 if w.dtype == "fp32" else 0))
        try:
            assert sw.swin_wattn_path(h, w.B, w.H, w.W) == want, key
        finally:
            sw.swin_wattn_destroy(h)


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("M,B,H,W", [(8, 2, 16, 24), (7, 3, 21, 14)])
def test_forward_v2_four_heads(M, B, H, W, path):
    """V2 cosine attention with C = 128 (four heads): the fused kernel's
    one-tile-in-flight variant, whose q passes through TMEM."""
    w = WORKLOADS["swinv2_t_s1"].with_(B=B, H=H, W=W, C=128, heads=4, M=M, shift=M // 2)
    g = generate(w, nonzero_bias=True)
    table = oracle_table(w, g)
    out = run_forward(w, device_inputs(g), table.to(DEV), path)
    compare(out.double().cpu().numpy(), oracle_forward(w, g, table), w.dtype)


@pytest.mark.parametrize("path", PATHS)
def test_forward_global_window_no_shift(path):
    """M = H = W and s = 0: one window per image (plain attention with bias)."""
    w = WORKLOADS["swinv2_t_s1"].with_(B=3, H=8, W=8, shift=0)
    g = generate(w, nonzero_bias=True)
    table = oracle_table(w, g)
    out = run_forward(w, device_inputs(g), table.to(DEV), path)
    compare(out.double().cpu().numpy(), oracle_forward(w, g, table), w.dtype)


def test_tiny_fp32_workload():
    w = WORKLOADS["tiny"]
    for bias in (False, True):
        g = generate(w, nonzero_bias=bias)
        out = run_forward(w, device_inputs(g), g["table"].to(DEV))
        compare(out.double().cpu().numpy(), oracle_forward(w, g, g["table"]), "fp32")


def test_fp32_v2_small():
    w = WORKLOADS["swinv2_t_s1"].with_(B=2, H=16, W=16, dtype="fp32")
    g = generate(w, nonzero_bias=True)
    table = oracle_table(w, g)
    out = run_forward(w, device_inputs(g), table.to(DEV))
    compare(out.double().cpu().numpy(), oracle_forward(w, g, table), "fp32")


# ---- full-size workloads, every output element ------------------------------

# float64 oracle outputs of the full-size workloads, shared by the two paths
_FULL_REF = {}


def full_reference(key):
    w = WORKLOADS[key]
    if key not in _FULL_REF:
        g = generate(w)
        table = oracle_table(w, g)
        _FULL_REF.clear()   # one workload at a time (SwinV2-L window 24: 0.9 GB)
        _FULL_REF[key] = (g, table, oracle_forward(w, g, table))
    return _FULL_REF[key]


@pytest.mark.parametrize("key,path", [("swin_t_s1", sw.PATH_AUTO), ("swin_t_s1", sw.PATH_THREE_KERNELS),
                                      ("swin_b_s1", sw.PATH_AUTO), ("swin_b_s3", sw.PATH_AUTO),
                                      ("swinv2_t_s1", sw.PATH_AUTO), ("swinv2_t_s1", sw.PATH_THREE_KERNELS),
                                      ("swinv2_l_w24", sw.PATH_AUTO)])
def test_forward_full_size(key, path):
    """The whole output of every full-size workload against the oracle: every
    tile of every CTA, the persistent kernels' tile order and buffer / phase
    alternation (which only grids of more tiles than SMs reach), every edge
    window."""
    w = WORKLOADS[key]
    g, table, ref = full_reference(key)
    out = run_forward(w, device_inputs(g), table.to(DEV), path)
    compare(out.double().cpu().numpy(), ref, w.dtype)


# ---- V2 with a different tau per head, below the clip too ------------------------

# tau per head: above the clip, at it, below it (clipped to 0.01), ...
TAUS = {3: (0.3, 0.01, 0.004), 6: (0.3, 0.01, 0.004, 0.05, 1.0, 0.02)}


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("key,B,H,W", [("swinv2_t_s1", 2, 16, 24), ("swinv2_t_s1", 32, 64, 64),
                                       ("swinv2_l_w24", 1, 48, 72)])
def test_forward_v2_tau_per_head(key, B, H, W, path):
    """Distinct tau per head, one of them below the 0.01 clip: a wrong head
    index into tau, or a missing clip, changes the result.  The fused kernel
    (windows of 8 x 8), the three-kernel path and the large-window kernel
    (window 24) all take this case."""
    w = WORKLOADS[key].with_(B=B, H=H, W=W)
    if path == sw.PATH_AUTO and w.M > 8:
        pytest.skip("window 24 runs the three-kernel path either way")
    g = generate(w, nonzero_bias=True, tau=TAUS[w.heads])
    table = oracle_table(w, g)
    out = run_forward(w, device_inputs(g), table.to(DEV), path)
    compare(out.double().cpu().numpy(), oracle_forward(w, g, table), w.dtype)


@pytest.mark.parametrize("key,kw", [
    ("swin_t_s1", dict(B=1, H=24, W=36, M=12, shift=6)),                      # V1: 144-token windows (tiles 128, 16)
    ("swin_t_s1", dict(B=2, H=32, W=32, M=16, shift=8, C=64, heads=2)),       # window 16: two full query tiles
    ("swin_t_s1", dict(B=1, H=40, W=40, M=20, shift=10, C=64, heads=2)),      # window 20: 400 tokens
    ("swinv2_t_s1", dict(B=1, H=24, W=24, M=12, shift=6, C=768, heads=24)),   # more heads than the kernel's warps
])
def test_forward_large_windows(key, kw):
    """The large-window kernel (windows of more than 64 tokens) at every window
    size it is built for, V1 (online softmax) and V2 with 24 heads whose tau
    puts some on the fixed reference and some on the online softmax (each
    head's choice is made in the kernel's prologue, a warp per head).  At C =
    768, Wqkv and Wproj are halved (exact in bf16) so that v, and the output
    (a sum over 4x the channels of the C = 192 cases), keep the magnitude the
    absolute bounds are set for."""
    w = WORKLOADS[key].with_(**kw)
    g = generate(w, nonzero_bias=True, tau=TAUS[6] * 4 if w.heads == 24 else 0.1)
    if w.C == 768:
        g["Wqkv"], g["Wproj"] = g["Wqkv"] * 0.5, g["Wproj"] * 0.5
    table = oracle_table(w, g)
    out = run_forward(w, device_inputs(g), table.to(DEV), sw.PATH_AUTO)
    compare(out.double().cpu().numpy(), oracle_forward(w, g, table), w.dtype)


# ---- the index maps through the whole forward, bit-exact -----------------------

def one_hot_attention_inputs(w, x):
    """Weights under which the block returns x exactly: Wq = Wk = 0 (every
    logit is its bias), Wv = I, Wproj = I, zero biases, and a table that is 0
    at displacement (0, 0) and -1e4 elsewhere.  Each row's softmax is then
    exactly one-hot on the token itself (every other exp2 underflows to 0),
    so out = x bit for bit on bf16-exact x whatever the shift mask does."""
    C, L = w.C, 2 * w.M - 1
    Wqkv = torch.zeros(3 * C, C, dtype=torch.bfloat16)
    Wqkv[2 * C:] = torch.eye(C)
    table = torch.full((L * L, w.heads), -1e4, dtype=torch.bfloat16)
    table[(w.M - 1) * L + (w.M - 1)] = 0
    t = {"x": torch.from_numpy(x).bfloat16().to(DEV), "Wqkv": Wqkv.to(DEV), "bqkv": None,
         "Wproj": torch.eye(C, dtype=torch.bfloat16).to(DEV), "bproj": None}
    if w.mode == V2:
        t["tau"] = torch.full((w.heads,), 0.1, dtype=torch.float32, device=DEV)
    return t, table.to(DEV)


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("key,B,H,W", [("swin_t_s1", 64, 56, 56), ("swin_t_s1", 3, 21, 35),
                                       ("swinv2_t_s1", 32, 64, 64), ("swinv2_t_s1", 1, 24, 16),
                                       ("swin_b_s1", 5, 28, 28), ("swinv2_l_w24", 2, 48, 72)])
def test_index_maps_bit_exact_through_whole_forward(key, B, H, W, path):
    """S1 (roll by -s, partition) and S8 (reverse, roll by +s) compared bit
    for bit through the whole forward on integer-tagged tokens: with the
    one-hot weights above the block is the identity exactly when both maps
    are right.  The full-size grids run every tile of the persistent fused
    kernel (its TMA boxes for windows the shift does not wrap, cp.async and
    plain stores for those it does)."""
    w = WORKLOADS[key].with_(B=B, H=H, W=W)
    if path == sw.PATH_AUTO and w.M > 8:
        pytest.skip("window 24 runs the three-kernel path either way")
    t, table = one_hot_attention_inputs(w, tagged(B, H, W, w.C))
    out = run_forward(w, t, table, path)
    assert torch.equal(out, t["x"]), int((out != t["x"]).sum())


# ---- meta-network G table ---------------------------------------------------------

@pytest.mark.parametrize("key", ["swinv2_t_s1", "swinv2_l_w24"])
def test_cpb_table(key):
    w = WORKLOADS[key]
    g = generate(w)
    ref = oracle.cpb_table(to_f64(g["W1"]), to_f64(g["b1"]), to_f64(g["W2"]), M=w.M, heads=w.heads)
    for fp32 in (True, False):
        if fp32 and w.M * w.M > 64:
            # the fp32 block keeps a whole window in shared memory: 576-token windows are refused
            with pytest.raises(sw.SwinWAttnError) as ei:
                sw.swin_wattn_create(w.C, w.heads, w.M, w.shift, w.mode | sw.FP32)
            assert ei.value.code == sw.EUNSUPPORTED
            continue
        h = sw.swin_wattn_create(w.C, w.heads, w.M, w.shift, w.mode | (sw.FP32 if fp32 else 0))
        try:
            dt = torch.float32 if fp32 else torch.bfloat16
            tab = torch.full(((2 * w.M - 1) ** 2, w.heads), float("nan"), dtype=dt, device=DEV)
            sw.swin_wattn_cpb_table(h, g["W1"].to(DEV), g["b1"].to(DEV), g["W2"].to(DEV), tab)
            assert sw.swin_wattn_sync_status(h) == sw.OK
        finally:
            sw.swin_wattn_destroy(h)
        got = tab.double().cpu().numpy()
        if fp32:
            assert np.max(np.abs(got - ref)) <= 1e-6 * max(1.0, np.abs(ref).max())
        else:
            assert np.all(np.abs(got - ref) <= np.abs(ref) * 2.0 ** -8 + 1e-7)


# ---- host-buffer entry point, edge cases, argument errors, watchdog ---------------

@pytest.mark.parametrize("chunks", [None, 1, 3, 16])
def test_forward_host_matches_device_forward(chunks):
    w = WORKLOADS["swin_t_s1"].with_(B=5, H=14, W=14)
    g = generate(w, nonzero_bias=True)
    t = device_inputs(g)
    dev_out = run_forward(w, t, t["table"])
    h = sw.swin_wattn_create(w.C, w.heads, w.M, w.shift, w.mode)
    try:
        if chunks:   # (16 chunks of a 5-image batch: one image each)
            sw.swin_wattn_set_option(h, sw.OPT_HOST_CHUNKS, chunks)
        x_host = g["x"].pin_memory()
        out_host = torch.empty_like(x_host).pin_memory()
        sw.swin_wattn_forward_host(h, x_host, t["Wqkv"], t["bqkv"], t["table"], None, t["Wproj"], t["bproj"],
                                   out_host)
        assert sw.swin_wattn_sync_status(h) == sw.OK
        for bad in (0, 17):
            with pytest.raises(sw.SwinWAttnError):
                sw.swin_wattn_set_option(h, sw.OPT_HOST_CHUNKS, bad)
    finally:
        sw.swin_wattn_destroy(h)
    assert torch.equal(out_host, dev_out.cpu())


@pytest.mark.parametrize("path", [sw.PATH_AUTO, sw.PATH_THREE_KERNELS])
def test_forward_host_repeated_calls(path):
    """The host-buffer forward is pipelined in image chunks and replayed from a
    captured graph while its arguments stay the same: new contents in the same
    buffers, a different batch size and device forwards in between (which
    reallocate the workspace) must all give the device forward's result."""
    base = WORKLOADS["swin_t_s1"].with_(H=14, W=21)
    h = sw.swin_wattn_create(base.C, base.heads, base.M, base.shift, base.mode)
    try:
        if path:
            sw.swin_wattn_set_option(h, sw.OPT_PATH, path)
        bufs = {}
        for B, seed in ((9, 1), (9, 2), (9, 3), (3, 4), (9, 5), (17, 6), (9, 7)):
            w = base.with_(B=B, seed=base.seed + seed)
            g = generate(w, nonzero_bias=True)
            t = device_inputs(g)
            dev_out = run_forward(w, t, t["table"], path)
            if B not in bufs:
                bufs[B] = (g["x"].pin_memory(), torch.empty_like(g["x"]).pin_memory())
            x_host, out_host = bufs[B]
            x_host.copy_(g["x"])   # the same host buffers again, new contents
            out_host.fill_(float("nan"))
            sw.swin_wattn_forward_host(h, x_host, t["Wqkv"], t["bqkv"], t["table"], None, t["Wproj"], t["bproj"],
                                       out_host)
            assert sw.swin_wattn_sync_status(h) == sw.OK
            assert torch.equal(out_host, dev_out.cpu()), (B, seed)
            # a device forward on a larger grid with the same handle between
            # host calls (the three-kernel path grows its workspace)
            big = base.with_(B=B + 8)
            gb = device_inputs(generate(big))
            ob = torch.empty_like(gb["x"])
            sw.swin_wattn_forward(h, gb["x"], gb["Wqkv"], gb["bqkv"], gb["table"], None, gb["Wproj"], gb["bproj"], ob)
            assert sw.swin_wattn_sync_status(h) == sw.OK
    finally:
        sw.swin_wattn_destroy(h)


def test_empty_batch_is_a_no_op():
    w = WORKLOADS["swin_t_s1"]
    h = sw.swin_wattn_create(w.C, w.heads, w.M, w.shift, w.mode)
    try:
        buf = torch.zeros(3 * w.C * w.C, dtype=torch.bfloat16, device=DEV)
        out = torch.zeros(16, dtype=torch.bfloat16, device=DEV)
        p = ctypes.c_void_p(buf.data_ptr())
        rc = sw.load().swin_wattn_forward(h, p, 0, 14, 14, p, None, p, None, p, None,
                                          ctypes.c_void_p(out.data_ptr()), None)
        assert rc == sw.OK
        assert sw.swin_wattn_last_launches(h) == 0
        assert sw.swin_wattn_sync_status(h) == sw.OK
    finally:
        sw.swin_wattn_destroy(h)


def test_bad_forward_arguments_are_rejected():
    w = WORKLOADS["swin_t_s1"].with_(B=1, H=14, W=14)
    g = device_inputs(generate(w))
    h = sw.swin_wattn_create(w.C, w.heads, w.M, w.shift, w.mode)
    try:
        out = torch.empty_like(g["x"])

        def fwd(**kw):
            a = dict(x=g["x"], Wqkv=g["Wqkv"], bqkv=g["bqkv"], bias_table=g["table"], logit_scale=None,
                     Wproj=g["Wproj"], bproj=g["bproj"], out=out)
            a.update(kw)
            with pytest.raises(sw.SwinWAttnError) as ei:
                sw.swin_wattn_forward(h, **a)
            return ei.value.code

        assert fwd(x=torch.zeros(1, 15, 14, w.C, dtype=torch.bfloat16, device=DEV)) == sw.EINVAL  # H % M
        assert fwd(out=g["x"]) == sw.EINVAL                                                      # aliasing
        flat = torch.zeros(14 * 14 * w.C + 8, dtype=torch.bfloat16, device=DEV)
        assert fwd(out=flat[1:1 + 14 * 14 * w.C].view(1, 14, 14, w.C)) == sw.EINVAL               # misaligned
        assert fwd(bias_table=None) == sw.EINVAL
        assert sw.swin_wattn_last_launches(h) == 0
    finally:
        sw.swin_wattn_destroy(h)
    h2 = sw.swin_wattn_create(w.C, w.heads, w.M, w.shift, V2)
    try:
        with pytest.raises(sw.SwinWAttnError) as ei:   # V2 needs logit_scale
            sw.swin_wattn_forward(h2, g["x"], g["Wqkv"], g["bqkv"], g["table"], None, g["Wproj"], g["bproj"], out)
        assert ei.value.code == sw.EINVAL
    finally:
        sw.swin_wattn_destroy(h2)


def test_bounded_wait_reports_timeout_and_context_survives():
    w = WORKLOADS["swin_t_s1"].with_(B=1, H=14, W=14)
    h = sw.swin_wattn_create(w.C, w.heads, w.M, w.shift, w.mode)
    try:
        sw.swin_wattn_set_option(h, sw.OPT_WAIT_LIMIT_US, 20000)
        sw.swin_wattn_test_watchdog(h)
        assert sw.swin_wattn_sync_status(h) == sw.ETIMEOUT
        assert sw.swin_wattn_sync_status(h) == sw.OK   # cleared
    finally:
        sw.swin_wattn_destroy(h)
    g = generate(w, nonzero_bias=True)
    out = run_forward(w, device_inputs(g), g["table"].to(DEV))
    compare(out.double().cpu().numpy(), oracle_forward(w, g, g["table"]), "bf16")


# ---- the stored oracle outputs (tests/golden) --------------------------------

@pytest.mark.parametrize("key,path,B,H,W", [("swin_t_s1", 0, 8, 56, 56), ("swinv2_t_s1", 0, 8, 64, 64),
                                            ("swin_t_s1", 1, 8, 56, 56), ("swinv2_l_w24", 0, 1, 96, 96)])
def test_overlapped_calls_give_the_same_bits(key, path, B, H, W):
    """SWIN_WATTN_OPT_OVERLAP_CALLS lets a call's kernels start while the
    kernels before them finish (the fused kernel the previous call's; on the
    three-kernel path each kernel the one before it): three chained calls on
    one stream (each call's x the previous call's output) give the bits of the
    same calls without the option."""
    w = WORKLOADS[key].with_(B=B, H=H, W=W)
    g = generate(w, nonzero_bias=True, tau=(0.3, 0.01, 0.05, 0.1, 0.2, 0.02)[: w.heads] if w.mode == V2 else 0.1)
    t = device_inputs(g)
    table = oracle_table(w, g).to(DEV)

    def chain(overlap):
        h = sw.swin_wattn_create(w.C, w.heads, w.M, w.shift, w.mode)
        try:
            sw.swin_wattn_set_option(h, sw.OPT_OVERLAP_CALLS, overlap)
            if path:
                sw.swin_wattn_set_option(h, sw.OPT_PATH, path)
            outs, cur = [], t["x"]
            for _ in range(3):
                o = torch.full_like(t["x"], float("nan"))
                sw.swin_wattn_forward(h, cur, t["Wqkv"], t["bqkv"], table, t.get("tau"), t["Wproj"], t["bproj"], o)
                outs.append(o)
                cur = o
            assert sw.swin_wattn_sync_status(h) == sw.OK
            assert sw.swin_wattn_last_launches(h) == (3 if path == 1 or w.M > 8 else 1)
            return outs
        finally:
            sw.swin_wattn_destroy(h)

    plain, overlapped = chain(0), chain(1)
    for a, b in zip(plain, overlapped):
        assert torch.equal(a, b)
    with pytest.raises(sw.SwinWAttnError):
        h = sw.swin_wattn_create(w.C, w.heads, w.M, w.shift, w.mode)
        try:
            sw.swin_wattn_set_option(h, sw.OPT_OVERLAP_CALLS, 2)
        finally:
            sw.swin_wattn_destroy(h)



@pytest.mark.parametrize("name", ["v1", "v2"])
def test_stored_golden_case(name):
    """The tiny stored case (8 x 8 tokens, C = 32, one head, M = 4, shift 2)
    against the oracle output kept in tests/golden/ (no oracle run here); the
    inputs are bf16 values, so the kernel consumes exactly what the oracle did."""
    import os
    import sys
    sys.path.insert(0, os.path.join(os.path.dirname(__file__), "golden"))
    import make_golden as mg
    mode = mg.CASES[name]["mode"]
    p = mg.inputs()
    bf = lambda a: torch.tensor(a).bfloat16().to(DEV)  # noqa: E731
    h = sw.swin_wattn_create(mg.C, mg.HEADS, mg.M, mg.SHIFT, V2 if mode else V1)
    try:
        x = bf(p["x"])
        out = torch.full_like(x, float("nan"))
        tau = torch.tensor(p["tau"], dtype=torch.float32, device=DEV) if mode else None
        sw.swin_wattn_forward(h, x, bf(p["Wqkv"]), bf(p["bqkv"]), bf(p["table"]), tau, bf(p["Wproj"]),
                              bf(p["bproj"]), out)
        assert sw.swin_wattn_sync_status(h) == sw.OK
    finally:
        sw.swin_wattn_destroy(h)
    stored = np.loadtxt(mg.path(name)).reshape(mg.B, mg.H, mg.W, mg.C)
    compare(out.double().cpu().numpy(), stored, "bf16")

"""Pins of the float64 oracle to things other than itself (CPU only).

Each test names what holds the oracle: a library routine (numpy.roll, a
reshape, float64 scaled_dot_product_attention), a closed form, an invariant,
or the window-free brute force in oracle/brute.py, which shares no step with
the windowed statement.  Together they make a plausible slip in the oracle
(roll sign, index order, relative-bias sign, mask band, missing scale, tau
clip, the G coordinates) fail at least one test.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import brute
from vision_transformer_shifted_gb300.inputs import V1, V2, WORKLOADS


def rand_block(B, H, W, C, heads, M, mode, seed=0, bias=True, tau=0.1):
    r = np.random.default_rng(seed)
    p = dict(
        x=r.standard_normal((B, H, W, C)),
        Wqkv=r.standard_normal((3 * C, C)) * 0.3,
        bqkv=r.standard_normal(3 * C) * 0.1 if bias else None,
        table=r.standard_normal(((2 * M - 1) ** 2, heads)) * 0.5,
        tau=np.full(heads, tau) if mode == V2 else None,
        Wproj=r.standard_normal((C, C)) * 0.3,
        bproj=r.standard_normal(C) * 0.1 if bias else None,
    )
    return p


def run(p, **kw):
    return oracle.forward(p["x"], p["Wqkv"], p["bqkv"], p["table"], p["tau"], p["Wproj"], p["bproj"], **kw)


# ---- S1 / S8 index maps --------------------------------------------------

@pytest.mark.parametrize("s", [0, 1, 3, 5])
def test_roll_is_numpy_roll_and_inverts(s):
    x = np.arange(2 * 14 * 21 * 3, dtype=np.float64).reshape(2, 14, 21, 3)
    y = oracle.roll(x, -s)
    assert np.array_equal(y, np.roll(x, -s, axis=(1, 2)))
    # cyclic shift by -s: the element at (i+s, j+s) lands on (i, j)
    assert np.array_equal(y[1, 0, 0], x[1, s % 14, s % 21])
    assert np.array_equal(oracle.roll(y, s), x)


@pytest.mark.parametrize("M", [1, 4, 7])
def test_partition_is_reshape_and_reverse_inverts(M):
    B, H, W, C = 2, 14 if M != 4 else 12, 28, 5
    x = np.arange(B * H * W * C, dtype=np.float64).reshape(B, H, W, C)
    xw = oracle.partition(x, M)
    ref = x.reshape(B, H // M, M, W // M, M, C).transpose(0, 1, 3, 2, 4, 5).reshape(-1, M * M, C)
    assert np.array_equal(xw, ref)
    assert np.array_equal(oracle.reverse(xw, B, H, W, M), x)


# ---- whole block against the window-free statement ------------------------

CASES = [
    # B, H, W, C, heads, M, s, mode
    (2, 14, 14, 8, 2, 7, 3, V1),
    (1, 14, 21, 6, 3, 7, 2, V1),
    (1, 8, 12, 8, 2, 4, 1, V1),
    (2, 12, 12, 8, 1, 6, 0, V1),
    (1, 16, 16, 8, 2, 8, 4, V2),
    (2, 12, 18, 6, 2, 6, 5, V2),
]


@pytest.mark.parametrize("case", CASES)
def test_windowed_oracle_equals_window_free_brute_force(case):
    B, H, W, C, heads, M, s, mode = case
    p = rand_block(B, H, W, C, heads, M, mode, seed=hash(case) % 1000)
    got = run(p, heads=heads, M=M, shift=s, mode=mode)
    ref = brute.forward(p["x"], p["Wqkv"], p["bqkv"], p["table"], p["tau"], p["Wproj"], p["bproj"],
                        heads=heads, M=M, shift=s, mode=mode)
    assert np.max(np.abs(got - ref)) < 1e-12


def test_window_subset_matches_full():
    B, H, W, C, heads, M, s = 2, 14, 14, 8, 2, 7, 3
    p = rand_block(B, H, W, C, heads, M, V1, seed=3)
    full = run(p, heads=heads, M=M, shift=s, mode=V1)
    part = run(p, heads=heads, M=M, shift=s, mode=V1, windows=[1, 6])
    xs = oracle.roll(np.arange(B * H * W, dtype=np.float64).reshape(B, H, W, 1), -s)
    toks = oracle.partition(xs, M)[[1, 6]].astype(int).ravel()
    flat_p, flat_f = part.reshape(-1, C), full.reshape(-1, C)
    assert np.array_equal(flat_p[toks], flat_f[toks])
    rest = np.setdiff1d(np.arange(B * H * W), toks)
    assert np.all(np.isnan(flat_p[rest]))


def test_batch_permutation_equivariance():
    B, H, W, C, heads, M, s = 3, 8, 8, 8, 2, 4, 2
    p = rand_block(B, H, W, C, heads, M, V2, seed=5)
    out = run(p, heads=heads, M=M, shift=s, mode=V2)
    perm = [2, 0, 1]
    q = dict(p, x=p["x"][perm])
    assert np.array_equal(run(q, heads=heads, M=M, shift=s, mode=V2), out[perm])


# ---- softmax / mask / bias pins -------------------------------------------

def band_lengths(n, M, s):
    """Length of the band each shifted-frame coordinate falls in."""
    L = np.full(n, M)
    if s > 0:
        L[n - M:n - s] = M - s
        L[n - s:] = s
    return L


@pytest.mark.parametrize("mode", [V1, V2])
def test_probabilities_rows_mask_and_counts(mode):
    B, H, W, C, heads, M, s = 1, 14, 14, 8, 2, 7, 3
    p = rand_block(B, H, W, C, heads, M, mode, seed=11)
    nwin = (H // M) * (W // M)
    counts = set()
    for win in range(nwin):
        logits, probs, _ = oracle.window_attention(
            p["x"], p["Wqkv"], p["bqkv"], p["table"], p["tau"], p["Wproj"], p["bproj"],
            heads=heads, M=M, shift=s, mode=mode, win=win)
        assert np.all(np.abs(probs.sum(-1) - 1) < 1e-12)
        masked = np.isneginf(logits)
        assert np.all(probs[masked] == 0.0)
        assert np.all(probs[~masked] > 0.0)
        # allowed keys per query = product of its row and column band lengths
        wi, wj = divmod(win, W // M)
        ti, tj = np.divmod(np.arange(M * M), M)
        want = band_lengths(H, M, s)[wi * M + ti] * band_lengths(W, M, s)[wj * M + tj]
        got = (~masked[0]).sum(-1)
        assert np.array_equal(got, want)
        counts |= set(got.tolist())
        # diagonal always allowed
        assert not masked[:, np.arange(M * M), np.arange(M * M)].any()
    assert counts == {49, 28, 21, 16, 12, 9}


def test_shift_zero_has_no_mask():
    p = rand_block(1, 14, 14, 8, 2, 7, V1, seed=2)
    for win in range(4):
        logits, _, _ = oracle.window_attention(p["x"], p["Wqkv"], p["bqkv"], p["table"], None, p["Wproj"],
                                               p["bproj"], heads=2, M=7, shift=0, mode=V1, win=win)
        assert np.isfinite(logits).all()


def test_v2_logit_bound_and_tau_clip():
    B, H, W, C, heads, M, s = 1, 16, 16, 8, 2, 8, 4
    for tau in (0.1, 0.5, 0.01, 0.002):
        p = rand_block(B, H, W, C, heads, M, V2, seed=4, tau=tau)
        logits, _, _ = oracle.window_attention(p["x"], p["Wqkv"], p["bqkv"], p["table"], p["tau"], p["Wproj"],
                                               p["bproj"], heads=heads, M=M, shift=s, mode=V2, win=3)
        ti, tj = np.divmod(np.arange(M * M), M)
        idx = (ti[:, None] - ti[None, :] + M - 1) * (2 * M - 1) + (tj[:, None] - tj[None, :] + M - 1)
        for hd in range(heads):
            fin = np.isfinite(logits[hd])
            dev = np.abs(logits[hd] - p["table"][idx, hd])[fin]
            assert dev.max() <= 1.0 / max(tau, 0.01) * (1 + 1e-12)
        # the diagonal of cos is exactly 1 (q with itself is not the same as k,
        # so only the bound holds there; it must be attained up to the bound)
    # tau below the clip behaves as tau = 0.01
    p1 = rand_block(B, H, W, C, heads, M, V2, seed=4, tau=0.001)
    p2 = rand_block(B, H, W, C, heads, M, V2, seed=4, tau=0.01)
    p3 = rand_block(B, H, W, C, heads, M, V2, seed=4, tau=0.02)
    o1 = run(p1, heads=heads, M=M, shift=s, mode=V2)
    o2 = run(p2, heads=heads, M=M, shift=s, mode=V2)
    o3 = run(p3, heads=heads, M=M, shift=s, mode=V2)
    assert np.array_equal(o1, o2)
    assert np.max(np.abs(o3 - o2)) > 1e-6


def test_v2_cosine_attains_bound_with_identical_q_k():
    """With Wq = Wk the logit of a token with itself is exactly 1/tau + bias."""
    B, H, W, C, heads, M, s = 1, 8, 8, 4, 1, 4, 0
    p = rand_block(B, H, W, C, heads, M, V2, seed=9, tau=0.25)
    p["Wqkv"][C:2 * C] = p["Wqkv"][:C]
    p["bqkv"][C:2 * C] = p["bqkv"][:C]
    logits, _, _ = oracle.window_attention(p["x"], p["Wqkv"], p["bqkv"], p["table"], p["tau"], p["Wproj"],
                                           p["bproj"], heads=1, M=M, shift=0, mode=V2, win=2)
    diag = np.diagonal(logits[0])
    assert np.allclose(diag, 4.0 + p["table"][(M - 1) * (2 * M - 1) + (M - 1), 0], atol=1e-12)


def test_uniform_attention_closed_form():
    """Wq = Wk = 0 and a zero table: every allowed key gets the same weight,
    so out = proj(mean of the allowed keys' v); allowed counts from the band
    closed form, membership from the original-frame adjacency."""
    B, H, W, C, heads, M, s = 1, 14, 14, 6, 2, 7, 3
    p = rand_block(B, H, W, C, heads, M, V1, seed=21)
    p["Wqkv"][:2 * C] = 0.0
    p["bqkv"][:2 * C] = 0.0
    p["table"][:] = 0.0
    out = run(p, heads=heads, M=M, shift=s, mode=V1)
    tok = p["x"][0].reshape(-1, C)
    v = tok @ p["Wqkv"][2 * C:].T + p["bqkv"][2 * C:]
    ii, jj = np.divmod(np.arange(H * W), W)
    for q in range(H * W):
        # shifted-frame coordinates of q and of every key
        si, sj = (ii - s) % H, (jj - s) % W
        same = (si // M == si[q] // M) & (sj // M == sj[q] // M)
        near = (np.abs(ii - ii[q]) < M) & (np.abs(jj - jj[q]) < M)
        keys = np.nonzero(same & near)[0]
        assert len(keys) == band_lengths(H, M, s)[si[q]] * band_lengths(W, M, s)[sj[q]]
        want = v[keys].mean(0) @ p["Wproj"].T + p["bproj"]
        assert np.max(np.abs(out[0, ii[q], jj[q]] - want)) < 1e-12


@pytest.mark.parametrize("mode", [V1, V2])
def test_global_window_equals_sdpa(mode):
    """shift 0 and M = H = W: one window holding the whole image, i.e. textbook
    multi-head attention with an additive bias (float64 SDPA on the CPU)."""
    B, H, W, C, heads, M = 2, 6, 6, 8, 2, 6
    d = C // heads
    p = rand_block(B, H, W, C, heads, M, mode, seed=31, tau=0.3)
    out = run(p, heads=heads, M=M, shift=0, mode=mode)
    x = torch.from_numpy(p["x"]).reshape(B, H * W, C)
    qkv = x @ torch.from_numpy(p["Wqkv"]).T + torch.from_numpy(p["bqkv"])
    q, k, v = [qkv[..., i * C:(i + 1) * C].reshape(B, H * W, heads, d).transpose(1, 2) for i in range(3)]
    ti, tj = np.divmod(np.arange(H * W), W)
    idx = (ti[:, None] - ti[None, :] + M - 1) * (2 * M - 1) + (tj[:, None] - tj[None, :] + M - 1)
    bias = torch.from_numpy(p["table"][idx].transpose(2, 0, 1))  # [heads, N, N]
    if mode == V1:
        o = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=bias)
    else:
        qn = torch.nn.functional.normalize(q, dim=-1, eps=1e-12)
        kn = torch.nn.functional.normalize(k, dim=-1, eps=1e-12)
        o = torch.nn.functional.scaled_dot_product_attention(qn, kn, v, attn_mask=bias,
                                                             scale=1.0 / max(p["tau"][0], 0.01))
    o = o.transpose(1, 2).reshape(B, H * W, C)
    y = (o @ torch.from_numpy(p["Wproj"]).T + torch.from_numpy(p["bproj"])).reshape(B, H, W, C)
    assert np.max(np.abs(out - y.numpy())) < 1e-12


def test_relative_bias_sign_query_minus_key():
    """A table that is large only at displacement (+1, 0) (query one row below
    the key) makes each query look at the key straight above it."""
    B, H, W, C, heads, M, s = 1, 8, 8, 4, 1, 4, 0
    p = rand_block(B, H, W, C, heads, M, V1, seed=41)
    p["Wqkv"][:2 * C] = 0.0
    p["bqkv"][:2 * C] = 0.0
    p["table"][:] = 0.0
    p["table"][(1 + M - 1) * (2 * M - 1) + (0 + M - 1), 0] = 60.0
    _, probs, _ = oracle.window_attention(p["x"], p["Wqkv"], p["bqkv"], p["table"], None, p["Wproj"],
                                          p["bproj"], heads=1, M=M, shift=0, mode=V1, win=0)
    for t in range(M, M * M):
        assert probs[0, t, t - M] >= 1 - 1e-12
        others = np.delete(probs[0, t], t - M)
        assert others.max() < 1e-25


def test_v1_scale_is_inverse_sqrt_d():
    """Two keys, known dot products: the weight ratio is exp((a-b)/sqrt(d))."""
    B, H, W, C, heads, M = 1, 1, 2, 16, 1, 1
    # M = 1 windows hold one token: softmax over a single key gives weight 1
    # whatever the scale; use M = 2 on a 2x2 image instead.
    H, W, M = 2, 2, 2
    r = np.random.default_rng(0)
    x = r.standard_normal((1, H, W, C))
    Wqkv = np.zeros((3 * C, C))
    Wqkv[:C] = np.eye(C)
    Wqkv[C:2 * C] = np.eye(C)
    Wqkv[2 * C:] = np.eye(C)
    table = np.zeros(((2 * M - 1) ** 2, 1))
    _, probs, _ = oracle.window_attention(x, Wqkv, None, table, None, np.eye(C), None,
                                          heads=1, M=M, shift=0, mode=V1, win=0)
    tok = x[0].reshape(-1, C)
    a = tok @ tok.T / math.sqrt(C)
    want = np.exp(a - a.max(1, keepdims=True))
    want /= want.sum(1, keepdims=True)
    assert np.max(np.abs(probs[0] - want)) < 1e-14


# ---- meta-network G (log-spaced continuous position bias) -----------------

def test_cpb_table_closed_form():
    """G reduced to two hidden units that pass u_r and -u_c through the ReLU:
    table[idx(dr,dc)] = (relu(sign(dr) ln(1+|dr|)), relu(-sign(dc) ln(1+|dc|)))."""
    M, heads, hidden = 5, 2, 4
    W1 = np.zeros((hidden, 2))
    W1[0] = [1.0, 0.0]
    W1[1] = [0.0, -1.0]
    W2 = np.zeros((heads, hidden))
    W2[0, 0] = 1.0
    W2[1, 1] = 1.0
    t = oracle.cpb_table(W1, np.zeros(hidden), W2, M=M, heads=heads)
    L = 2 * M - 1
    for dr in range(-(M - 1), M):
        for dc in range(-(M - 1), M):
            idx = (dr + M - 1) * L + (dc + M - 1)
            ur = math.copysign(math.log1p(abs(dr)), dr) if dr else 0.0
            uc = math.copysign(math.log1p(abs(dc)), dc) if dc else 0.0
            assert t[idx, 0] == pytest.approx(max(ur, 0.0), abs=1e-15)
            assert t[idx, 1] == pytest.approx(max(-uc, 0.0), abs=1e-15)


def test_cpb_table_zero_row_and_shape():
    w = WORKLOADS["swinv2_t_s1"]
    r = np.random.default_rng(1)
    W1 = r.standard_normal((512, 2)) * 0.02
    W2 = r.standard_normal((w.heads, 512)) * 0.02
    t = oracle.cpb_table(W1, np.zeros(512), W2, M=w.M, heads=w.heads)
    assert t.shape == (225, 3)
    centre = (w.M - 1) * (2 * w.M - 1) + (w.M - 1)
    assert np.all(t[centre] == 0.0)
    # with a hidden bias the centre row is W2 relu(b1)
    b1 = r.standard_normal(512) * 0.1
    t2 = oracle.cpb_table(W1, b1, W2, M=w.M, heads=w.heads)
    assert np.allclose(t2[centre], W2 @ np.maximum(b1, 0), atol=1e-15)


# ---- the tiny workload through both formulations ---------------------------

def test_tiny_workload_both_formulations():
    from vision_transformer_shifted_gb300.inputs import generate
    w = WORKLOADS["tiny"]
    g = generate(w, nonzero_bias=True)
    a = {k: (v.double().numpy() if v is not None else None) for k, v in g.items()}
    out = oracle.forward(a["x"], a["Wqkv"], a["bqkv"], a["table"], None, a["Wproj"], a["bproj"],
                         heads=w.heads, M=w.M, shift=w.shift, mode=w.mode)
    ref = brute.forward(a["x"], a["Wqkv"], a["bqkv"], a["table"], None, a["Wproj"], a["bproj"],
                        heads=w.heads, M=w.M, shift=w.shift, mode=w.mode)
    assert np.max(np.abs(out - ref)) < 1e-12
    assert np.isfinite(out).all()


# ---- stored oracle outputs (tests/golden) ----------------------------------

@pytest.mark.parametrize("name", ["v1", "v2"])
def test_oracle_still_matches_its_stored_outputs(name):
    """The files under tests/golden/ were written by tests/golden/make_golden.py
    from this oracle; any later change to its arithmetic shows up here (and
    must then name the passage that justifies it)."""
    import os
    import sys
    sys.path.insert(0, os.path.join(os.path.dirname(__file__), "golden"))
    import make_golden as mg
    stored = np.loadtxt(mg.path(name)).reshape(mg.B, mg.H, mg.W, mg.C)
    _, out = mg.compute(mg.CASES[name]["mode"])
    assert np.allclose(out, stored, rtol=1e-12, atol=1e-13)

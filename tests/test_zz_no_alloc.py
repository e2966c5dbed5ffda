"""swin_wattn_forward_noalloc: the forward for callers that cannot allocate.

Some callers cannot call cudaMalloc: code running under an allocator it does
not own (a framework caching allocator that must account for every byte, an
embedded runtime with a fixed budget) or code that must not allocate once it
is serving (a cudaMalloc would synchronise the device).  The entry point
keeps its intermediates in a fixed array inside the library.  These tests
call it through the C ABI and check it on two calls in a row (the array
keeps the previous call's contents, so the second call must not depend on
them): against the float64 oracle within the bf16 tolerances, and bit for
bit against swin_wattn_forward (the entry point with a handle-owned
workspace) forced onto the same three kernels.  They also check that the
device's free memory does not move across calls, that a call too large for
the array is refused before any launch, and that a kernel's bounded-wait
timeout reaches the caller through swin_wattn_noalloc_sync_status, and
that a call can be captured into a CUDA graph in global capture mode.

This file is collected last on purpose, and it needs no state from the
other test files.
"""
import pytest
import torch

from vision_transformer_shifted_gb300 import binding as sw
from vision_transformer_shifted_gb300.inputs import V2, WORKLOADS, generate

from helpers import compare, device_inputs, oracle_forward, oracle_table

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    sw.load()


def forward_with_handle(w, t, table, path):
    h = sw.swin_wattn_create(w.C, w.heads, w.M, w.shift, w.mode)
    try:
        sw.swin_wattn_set_option(h, sw.OPT_PATH, path)
        out = torch.full_like(t["x"], float("nan"))
        sw.swin_wattn_forward(h, t["x"], t["Wqkv"], t["bqkv"], table, t.get("tau"), t["Wproj"], t["bproj"], out)
        assert sw.swin_wattn_sync_status(h) == sw.OK
        return out
    finally:
        sw.swin_wattn_destroy(h)


def noalloc(w, t, table, out):
    sw.swin_wattn_forward_noalloc(w.C, w.heads, w.M, w.shift, w.mode, t["x"], t["Wqkv"], t["bqkv"], table,
                                  t.get("tau"), t["Wproj"], t["bproj"], out)


@pytest.mark.parametrize("key,B,H,W", [("swin_t_s1", 4, 56, 56), ("swinv2_t_s1", 2, 64, 64),
                                       ("swinv2_l_w24", 1, 48, 96)])
def test_noalloc_matches_oracle_and_forward_on_two_calls_in_a_row(key, B, H, W):
    w = WORKLOADS[key].with_(B=B, H=H, W=W)
    assert 8 * w.tokens * w.C <= sw.NOALLOC_MAX_INTERMEDIATE_BYTES
    results = []
    for seed_shift in (0, 1):   # two different inputs, one call after the other
        g = generate(w.with_(seed=w.seed + 17 * seed_shift), nonzero_bias=True,
                     tau=(0.3, 0.01, 0.004, 0.05, 1.0, 0.02)[:w.heads] if w.mode == V2 else 0.1)
        t = device_inputs(g)
        table = oracle_table(w, g)
        td = table.to(DEV)
        out = torch.full_like(t["x"], float("nan"))
        torch.cuda.synchronize()
        noalloc(w, t, td, out)
        assert sw.swin_wattn_noalloc_sync_status() == sw.OK
        results.append((g, table, out, forward_with_handle(w, t, td, sw.PATH_THREE_KERNELS)))
    for g, table, got, same_kernels in results:
        compare(got.double().cpu().numpy(), oracle_forward(w, g, table), "bf16")
        # the same three kernels on the same inputs: the same bits
        assert torch.equal(got, same_kernels)
    assert not torch.equal(results[0][2], results[1][2])
    # a third call on the first inputs: no device memory taken or given back
    g, table, first, _ = results[0]
    t = device_inputs(g)
    td = table.to(DEV)
    out = torch.full_like(t["x"], float("nan"))
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    noalloc(w, t, td, out)
    assert sw.swin_wattn_noalloc_sync_status() == sw.OK
    assert torch.cuda.mem_get_info()[0] == free_before
    assert torch.equal(out, first)


def test_noalloc_call_captures_into_a_cuda_graph():
    """After one call, a second one on the same arguments is captured into a
    CUDA graph in global capture mode, which refuses cudaMalloc and every
    call that synchronises the device: the capture goes through, nothing runs
    until the replay, and the replay writes the first call's bits."""
    w = WORKLOADS["swin_t_s1"].with_(B=2)
    g = generate(w, nonzero_bias=True)
    t = device_inputs(g)
    table = t["table"]
    out = torch.full_like(t["x"], float("nan"))
    noalloc(w, t, table, out)
    assert sw.swin_wattn_noalloc_sync_status() == sw.OK
    first = out.clone()
    out.fill_(float("nan"))
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, capture_error_mode="global"):
        noalloc(w, t, table, out)
    torch.cuda.synchronize()
    assert bool(torch.isnan(out).all())   # captured, not run
    graph.replay()
    assert sw.swin_wattn_noalloc_sync_status() == sw.OK
    assert torch.equal(out, first)


def test_noalloc_refuses_calls_larger_than_its_scratch():
    w = WORKLOADS["swin_t_s1"]          # B = 64: 154 MB of intermediates
    assert 8 * w.tokens * w.C > sw.NOALLOC_MAX_INTERMEDIATE_BYTES
    t = device_inputs(generate(w.with_(B=1)))
    x = torch.zeros(w.B, w.H, w.W, w.C, dtype=torch.bfloat16, device=DEV)
    out = torch.full_like(x, 7.0)
    with pytest.raises(sw.SwinWAttnError) as ei:
        sw.swin_wattn_forward_noalloc(w.C, w.heads, w.M, w.shift, w.mode, x, t["Wqkv"], t["bqkv"], t["table"],
                                      None, t["Wproj"], t["bproj"], out)
    assert ei.value.code == sw.ESCRATCH
    assert "scratch" in sw.strerror(sw.ESCRATCH)
    torch.cuda.synchronize()
    assert bool((out == 7.0).all())     # nothing was launched


def test_noalloc_rejects_bad_arguments():
    w = WORKLOADS["swin_t_s1"].with_(B=1, H=14, W=14)
    t = device_inputs(generate(w))
    out = torch.empty_like(t["x"])
    args = (t["x"], t["Wqkv"], t["bqkv"], t["table"], None, t["Wproj"], t["bproj"], out)
    for params, code in [((96, 5, 7, 3, 0), sw.EINVAL), ((96, 3, 7, 7, 0), sw.EINVAL),
                         ((96, 3, 7, 3, sw.FP32), sw.EUNSUPPORTED), ((96, 3, 7, 3, V2), sw.EINVAL)]:
        with pytest.raises(sw.SwinWAttnError) as ei:
            sw.swin_wattn_forward_noalloc(*params, *args)
        assert ei.value.code == code


def test_noalloc_reports_a_bounded_wait_timeout():
    """A kernel that waits on a barrier nothing completes (20 ms limit)
    records the timeout in the fixed array's status word: the status call
    reports it once, clears it, and a normal call then succeeds."""
    sw.swin_wattn_test_noalloc_watchdog(20000)
    assert sw.swin_wattn_noalloc_sync_status() == sw.ETIMEOUT
    assert sw.swin_wattn_noalloc_sync_status() == sw.OK
    w = WORKLOADS["swin_t_s1"].with_(B=2, H=14, W=21)
    g = generate(w, nonzero_bias=True)
    t = device_inputs(g)
    out = torch.full_like(t["x"], float("nan"))
    noalloc(w, t, t["table"], out)
    assert sw.swin_wattn_noalloc_sync_status() == sw.OK
    compare(out.double().cpu().numpy(), oracle_forward(w, g, g["table"]), "bf16")

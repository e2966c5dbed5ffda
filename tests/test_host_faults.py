"""Faults made on the host, none of which faults, traps or hangs the GPU:

* a simulated allocation failure (SWIN_WATTN_FAIL_ALLOC): every workspace
  allocation of a handle fails as if the device were out of memory; the call
  returns ENOMEM before any launch, and the same handle works again once the
  switch is unset;
* guard bands (SWIN_WATTN_DEBUG): the workspaces get 4 KiB bands of a byte
  pattern on either side, read back after every call that used them; a
  normal call leaves them intact (no kernel writes outside its buffer), and a
  byte overwritten by the test hook is reported as ECORRUPT.
"""
import os

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


class env:
    def __init__(self, name, value):
        self.name, self.value = name, value

    def __enter__(self):
        self.old = os.environ.get(self.name)
        os.environ[self.name] = self.value

    def __exit__(self, *exc):
        if self.old is None:
            del os.environ[self.name]
        else:
            os.environ[self.name] = self.old


def test_simulated_allocation_failure_then_normal_call():
    w = WORKLOADS["swin_t_s1"].with_(B=2, H=14, W=21)
    g = generate(w, nonzero_bias=True)
    t = device_inputs(g)
    h = sw.swin_wattn_create(w.C, w.heads, w.M, w.shift, w.mode)
    try:
        sw.swin_wattn_set_option(h, sw.OPT_PATH, sw.PATH_THREE_KERNELS)
        out = torch.full_like(t["x"], 5.0)
        with env("SWIN_WATTN_FAIL_ALLOC", "1"):
            with pytest.raises(sw.SwinWAttnError) as ei:
                sw.swin_wattn_forward(h, t["x"], t["Wqkv"], t["bqkv"], t["table"], None, t["Wproj"], t["bproj"], out)
            assert ei.value.code == sw.ENOMEM
            assert sw.swin_wattn_last_launches(h) == 0
            # the backward's workspace too
            C, L = w.C, 2 * w.M - 1
            f32 = dict(device=DEV, dtype=torch.float32)
            with pytest.raises(sw.SwinWAttnError) as ei:
                sw.swin_wattn_backward(h, t["x"], t["Wqkv"], t["bqkv"], t["table"], t["Wproj"], t["bproj"],
                                       torch.zeros_like(t["x"]), torch.empty_like(t["x"]),
                                       torch.empty(3 * C, C, **f32), torch.empty(3 * C, **f32),
                                       torch.empty(L * L, w.heads, **f32), torch.empty(C, C, **f32),
                                       torch.empty(C, **f32))
            assert ei.value.code == sw.ENOMEM
        torch.cuda.synchronize()
        assert bool((out == 5.0).all())   # nothing ran
        sw.swin_wattn_forward(h, t["x"], t["Wqkv"], t["bqkv"], t["table"], None, t["Wproj"], t["bproj"], out)
        assert sw.swin_wattn_sync_status(h) == sw.OK
    finally:
        sw.swin_wattn_destroy(h)
    compare(out.double().cpu().numpy(), oracle_forward(w, g, g["table"]), "bf16")


def test_simulated_allocation_failure_of_the_whole_block():
    w = WORKLOADS["swin_t_s1"].with_(B=1, H=14, W=14)
    C = w.C
    h = sw.swin_block_create(C, w.heads, w.M, w.shift, w.mode, 4)
    try:
        x = torch.zeros(1, 14, 14, C, dtype=torch.bfloat16, device=DEV)
        z = lambda *s: torch.zeros(*s, dtype=torch.bfloat16, device=DEV)  # noqa: E731
        params = dict(ln1_gamma=z(C), ln1_beta=z(C), Wqkv=z(3 * C, C), bqkv=z(3 * C),
                      bias_table=z((2 * w.M - 1) ** 2, w.heads), Wproj=z(C, C), bproj=z(C), ln2_gamma=z(C),
                      ln2_beta=z(C), W1=z(4 * C, C), b1=z(4 * C), W2=z(C, 4 * C), b2=z(C))
        out = torch.empty_like(x)
        with env("SWIN_WATTN_FAIL_ALLOC", "1"):
            with pytest.raises(sw.SwinWAttnError) as ei:
                sw.swin_block_forward(h, x, params, out)
            assert ei.value.code == sw.ENOMEM
        sw.swin_block_forward(h, x, params, out)
        sw.swin_block_sync_status(h)
    finally:
        sw.swin_block_destroy(h)


@pytest.mark.parametrize("key", ["swin_t_s1", "swinv2_l_w24"])
def test_guard_bands_stay_intact_and_catch_an_overwrite(key):
    w = WORKLOADS[key].with_(B=1, H=2 * WORKLOADS[key].M, W=3 * WORKLOADS[key].M)
    g = generate(w, nonzero_bias=True)
    table = oracle_table(w, g)
    t = device_inputs(g)
    with env("SWIN_WATTN_DEBUG", "1"):
        h = sw.swin_wattn_create(w.C, w.heads, w.M, w.shift, w.mode)
        try:
            sw.swin_wattn_set_option(h, sw.OPT_PATH, sw.PATH_THREE_KERNELS)
            out = torch.full_like(t["x"], float("nan"))
            for _ in range(2):   # the bands are read back after each call
                sw.swin_wattn_forward(h, t["x"], t["Wqkv"], t["bqkv"], table.to(DEV), t.get("tau"), t["Wproj"],
                                      t["bproj"], out)
            assert sw.swin_wattn_sync_status(h) == sw.OK
            compare(out.double().cpu().numpy(), oracle_forward(w, g, table), "bf16")
            for side in (0, 1):
                sw.swin_wattn_test_corrupt_workspace(h, side)
                with pytest.raises(sw.SwinWAttnError) as ei:
                    sw.swin_wattn_forward(h, t["x"], t["Wqkv"], t["bqkv"], table.to(DEV), t.get("tau"),
                                          t["Wproj"], t["bproj"], out)
                assert ei.value.code == sw.ECORRUPT
        finally:
            sw.swin_wattn_destroy(h)


def test_corrupt_hook_refuses_an_unguarded_workspace():
    w = WORKLOADS["swin_t_s1"].with_(B=1, H=14, W=14)
    h = sw.swin_wattn_create(w.C, w.heads, w.M, w.shift, w.mode)
    try:
        with pytest.raises(sw.SwinWAttnError) as ei:
            sw.swin_wattn_test_corrupt_workspace(h, 0)
        assert ei.value.code == sw.EINVAL
    finally:
        sw.swin_wattn_destroy(h)

"""C-ABI boundary checks that need no GPU: the library builds and loads, it
exports every function the headers declare, and argument checks that come
before any device call return their status codes."""
import ctypes
import os
import re

import pytest

from vision_transformer_shifted_gb300 import binding as sw

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for hdr in os.listdir(os.path.join(ROOT, "include")):
        text = open(os.path.join(ROOT, "include", hdr)).read()
        names |= set(re.findall(r"^\s*(?:int|const char \*)\s*(swin_(?:wattn|block|merge|stage)_\w+)\s*\(", text, re.M))
    return names


def test_library_exports_every_declared_function():
    lib = sw.load()
    names = declared_functions()
    assert len(names) >= 15
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing
    assert names == set(sw.exported_symbols())


def test_strerror_covers_every_status():
    for code in (sw.OK, sw.EINVAL, sw.EUNSUPPORTED, sw.ECUDA, sw.ENOMEM, sw.ETIMEOUT, sw.ESCRATCH, sw.ECORRUPT):
        assert sw.strerror(code) != "unknown status"
    assert sw.strerror(12345) == "unknown status"


@pytest.mark.parametrize("args,code", [
    ((96, 5, 7, 3, sw.V1), sw.EINVAL),          # C % heads != 0
    ((96, 3, 7, 7, sw.V1), sw.EINVAL),          # shift >= M
    ((96, 3, 7, -1, sw.V1), sw.EINVAL),         # negative shift
    ((96, 3, 0, 0, sw.V1), sw.EINVAL),          # M = 0
    ((96, 3, 7, 3, 0x40), sw.EINVAL),           # unknown mode bit
    ((128, 2, 7, 3, sw.V1), sw.EUNSUPPORTED),   # bf16 kernels need d = 32
    ((48, 2, 7, 3, sw.V2), sw.EUNSUPPORTED),    # d = 24
    ((96, 3, 80, 3, sw.V1), sw.EUNSUPPORTED),   # window larger than the kernels take
])
def test_create_rejects_bad_arguments_before_any_device_call(args, code):
    lib = sw.load()
    h = ctypes.c_void_p(123)
    assert lib.swin_wattn_create(ctypes.byref(h), *args) == code
    assert h.value is None
    assert lib.swin_wattn_create(None, 96, 3, 7, 3, 0) == sw.EINVAL


def test_null_handle_calls():
    lib = sw.load()
    assert lib.swin_wattn_forward(None, None, 1, 7, 7, None, None, None, None, None, None, None, None) == sw.EINVAL
    assert lib.swin_wattn_destroy(None) == sw.OK
    assert lib.swin_wattn_set_option(None, 1, 0) == sw.EINVAL
    assert lib.swin_wattn_backward(None, None, 1, 7, 7, *([None] * 15)) == sw.EINVAL
    assert lib.swin_wattn_cpb_backward(None, None, None, None, 512, None, None, None, None, None) == sw.EINVAL
    assert lib.swin_wattn_backward_launches(None) == 0
    assert lib.swin_wattn_path(None, 1, 7, 7) == sw.EINVAL
    assert lib.swin_wattn_sync_status(None, None) == sw.EINVAL
    assert lib.swin_wattn_test_gemm(None, None, None, None, 1, 16, 16, 128, None) == sw.EINVAL
    assert lib.swin_wattn_test_gemm(ctypes.c_void_p(16), ctypes.c_void_p(16), None, ctypes.c_void_p(16),
                                    1, 24, 16, 128, None) == sw.EINVAL  # N % 16
    assert lib.swin_wattn_test_gemm(ctypes.c_void_p(16), ctypes.c_void_p(16), None, ctypes.c_void_p(16),
                                    1, 16, 16, 32, None) == sw.EINVAL  # swizzle
    assert lib.swin_wattn_test_gemm(ctypes.c_void_p(16), ctypes.c_void_p(16), None, ctypes.c_void_p(16),
                                    1, 16, 48, 1, None) == sw.EINVAL  # masked pair: K % 32
    assert lib.swin_wattn_test_gemm(ctypes.c_void_p(16), ctypes.c_void_p(16), None, ctypes.c_void_p(16),
                                    1, 144, 32, 1, None) == sw.EINVAL  # masked pair: N > 128


def header_enums():
    vals = {}
    for hdr in os.listdir(os.path.join(ROOT, "include")):
        text = open(os.path.join(ROOT, "include", hdr)).read()
        for name, v in re.findall(r"\b(SWIN_(?:WATTN|BLOCK)_[A-Z0-9_]+)\s*=\s*(-?(?:0x[0-9a-fA-F]+|\d+))\b", text):
            vals[name] = int(v, 0)
    return vals


def test_binding_constants_match_the_headers():
    """Every mode, status and option constant of the binding has the value the
    headers give it (SWIN_WATTN_X is the binding's X, SWIN_BLOCK_OPT_X its
    BLOCK_OPT_X), and every enumerator of the headers has its binding name."""
    vals = header_enums()
    assert len(vals) >= 16
    missing = []
    for name, v in vals.items():
        py = name[len("SWIN_WATTN_"):] if name.startswith("SWIN_WATTN_") else name[len("SWIN_"):]
        if not hasattr(sw, py):
            missing.append(name)
            continue
        assert getattr(sw, py) == v, (name, getattr(sw, py), v)
    assert not missing, missing

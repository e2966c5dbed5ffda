"""ctypes binding of libswin_wattn (include/swin_wattn.h, swin_wattn_test.h,
swin_block.h, swin_wattn_backward.h).

Argument marshalling only: every function here passes tensor pointers and
sizes to the C ABI of the same name and raises on a non-OK status.  torch is
used for device memory and streams; no step of the block runs in Python, and
there is no CPU fallback: if the library cannot be loaded every call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

V1, V2, FP32 = 0, 1, 0x10
OK, EINVAL, EUNSUPPORTED, ECUDA, ENOMEM, ETIMEOUT, ESCRATCH, ECORRUPT = 0, -1, -2, -3, -4, -5, -6, -7
NOALLOC_MAX_INTERMEDIATE_BYTES = (64 << 20) - 256
OPT_PATH, OPT_WAIT_LIMIT_US, OPT_HOST_CHUNKS, OPT_OVERLAP_CALLS = 1, 2, 3, 4
BLOCK_OPT_OVERLAP_CALLS = 1
PATH_AUTO, PATH_THREE_KERNELS, PATH_FUSED, PATH_FP32 = 0, 1, 2, 3

_lib = None


class SwinWAttnError(RuntimeError):
    def __init__(self, fn, code):
        self.code = code
        super().__init__("%s failed: %s (%d)" % (fn, strerror(code) if _lib else "?", code))


_SIGNATURES = {
    "swin_wattn_create": ["pp", "i", "i", "i", "i", "i"],
    "swin_wattn_destroy": ["p"],
    "swin_wattn_forward": ["p", "p", "i", "i", "i", "p", "p", "p", "p", "p", "p", "p", "p"],
    "swin_wattn_forward_host": ["p", "p", "i", "i", "i", "p", "p", "p", "p", "p", "p", "p", "p"],
    "swin_wattn_cpb_table": ["p", "p", "p", "p", "i", "p", "p"],
    "swin_wattn_sync_status": ["p", "p"],
    "swin_wattn_set_option": ["p", "i", "l"],
    "swin_wattn_path": ["p", "i", "i", "i"],
    "swin_wattn_last_launches": ["p"],
    "swin_wattn_test_qkv": ["p", "p", "i", "i", "i", "p", "p", "p", "p"],
    "swin_wattn_test_attn": ["p", "p", "i", "i", "i", "p", "p", "p", "p"],
    "swin_wattn_test_proj": ["p", "p", "i", "i", "i", "p", "p", "p", "p"],
    "swin_wattn_test_gemm": ["p", "p", "p", "p", "i", "i", "i", "i", "p"],
    "swin_wattn_test_watchdog": ["p", "p"],
    "swin_wattn_test_corrupt_workspace": ["p", "i"],
    "swin_wattn_forward_noalloc": ["i", "i", "i", "i", "i", "p", "i", "i", "i", "p", "p", "p", "p", "p", "p", "p",
                                   "p"],
    "swin_wattn_noalloc_sync_status": ["p"],
    "swin_wattn_test_noalloc_watchdog": ["l", "p"],
    "swin_block_create": ["pp", "i", "i", "i", "i", "i", "i"],
    "swin_block_forward": ["p", "p", "i", "i", "i", "p", "p", "p"],
    "swin_block_sync_status": ["p", "p"],
    "swin_block_destroy": ["p"],
    "swin_block_last_launches": ["p"],
    "swin_block_set_option": ["p", "i", "l"],
    "swin_block_test_layernorm": ["p", "p", "p", "p", "p", "p", "i", "i", "i", "p"],
    "swin_stage_norm": ["p", "i", "i", "p", "p", "p", "p"],
    "swin_merge_create": ["pp", "i"],
    "swin_merge_forward": ["p", "p", "i", "i", "i", "p", "p", "p", "p", "p"],
    "swin_merge_destroy": ["p"],
    "swin_wattn_backward": ["p", "p", "i", "i", "i", "p", "p", "p", "p", "p", "p", "p", "p", "p", "p", "p", "p",
                            "p", "p", "p"],
    "swin_wattn_cpb_backward": ["p", "p", "p", "p", "i", "p", "p", "p", "p", "p"],
    "swin_wattn_backward_launches": ["p"],
}

# swin_block_params (include/swin_block.h), field for field
BLOCK_PARAM_FIELDS = ("ln1_gamma", "ln1_beta", "Wqkv", "bqkv", "bias_table", "logit_scale", "Wproj", "bproj",
                      "ln2_gamma", "ln2_beta", "W1", "b1", "W2", "b2")


class BlockParams(ctypes.Structure):
    _fields_ = [(name, ctypes.c_void_p) for name in BLOCK_PARAM_FIELDS]
_CT = {"p": ctypes.c_void_p, "pp": ctypes.POINTER(ctypes.c_void_p), "i": ctypes.c_int, "l": ctypes.c_int64}


def load(build_if_missing: bool = True):
    """Loads libswin_wattn.so (building it first if it is missing)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB
    if not os.path.exists(path):
        if not build_if_missing:
            raise OSError("libswin_wattn.so is not built")
        _build.build()
    lib = ctypes.CDLL(path)
    for name, args in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.argtypes = [_CT[a] for a in args]
        fn.restype = ctypes.c_int
    lib.swin_wattn_strerror.argtypes = [ctypes.c_int]
    lib.swin_wattn_strerror.restype = ctypes.c_char_p
    lib.swin_wattn_last_cuda_error.argtypes = [ctypes.c_void_p]
    lib.swin_wattn_last_cuda_error.restype = ctypes.c_char_p
    _lib = lib
    return lib


def exported_symbols():
    """Names of the functions the C headers declare."""
    return sorted(list(_SIGNATURES) + ["swin_wattn_strerror", "swin_wattn_last_cuda_error"])


def strerror(code: int) -> str:
    return load().swin_wattn_strerror(int(code)).decode()


def _check(fn, rc):
    if rc != OK:
        raise SwinWAttnError(fn, rc)
    return rc


def _p(t):
    """Pointer of a tensor (None -> NULL)."""
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        if torch.cuda.is_available():
            return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        return None
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def swin_wattn_create(C, heads, M, shift, mode):
    h = ctypes.c_void_p()
    _check("swin_wattn_create", load().swin_wattn_create(ctypes.byref(h), C, heads, M, shift, mode))
    return h


def swin_wattn_destroy(h):
    return _check("swin_wattn_destroy", load().swin_wattn_destroy(h))


def swin_wattn_forward(h, x, Wqkv, bqkv, bias_table, logit_scale, Wproj, bproj, out, stream=None):
    B, H, W, _ = x.shape
    rc = load().swin_wattn_forward(
        h, _p(x), B, H, W, _p(Wqkv), _p(bqkv), _p(bias_table), _p(logit_scale), _p(Wproj), _p(bproj), _p(out),
        _stream(stream))
    if rc == ECUDA:
        raise SwinWAttnError("swin_wattn_forward (%s)" % swin_wattn_last_cuda_error(h), rc)
    return _check("swin_wattn_forward", rc)


def swin_wattn_backward(h, x, Wqkv, bqkv, bias_table, Wproj, bproj, dy, dx, dWqkv, dbqkv, dtable, dWproj, dbproj,
                        logit_scale=None, dlogit_scale=None, stream=None):
    B, H, W, _ = x.shape
    return _check("swin_wattn_backward", load().swin_wattn_backward(
        h, _p(x), B, H, W, _p(Wqkv), _p(bqkv), _p(bias_table), _p(logit_scale), _p(Wproj), _p(bproj), _p(dy), _p(dx),
        _p(dWqkv), _p(dbqkv), _p(dtable), _p(dlogit_scale), _p(dWproj), _p(dbproj), _stream(stream)))


def swin_wattn_cpb_backward(h, W1, b1, W2, dtable, dW1, db1, dW2, stream=None):
    return _check("swin_wattn_cpb_backward", load().swin_wattn_cpb_backward(
        h, _p(W1), _p(b1), _p(W2), W1.shape[0], _p(dtable), _p(dW1), _p(db1), _p(dW2), _stream(stream)))


def swin_wattn_backward_launches(h):
    return load().swin_wattn_backward_launches(h)


def swin_wattn_last_cuda_error(h):
    return load().swin_wattn_last_cuda_error(h).decode()


def swin_wattn_forward_host(h, x_host, Wqkv, bqkv, bias_table, logit_scale, Wproj, bproj, out_host, stream=None):
    B, H, W, _ = x_host.shape
    return _check("swin_wattn_forward_host", load().swin_wattn_forward_host(
        h, _p(x_host), B, H, W, _p(Wqkv), _p(bqkv), _p(bias_table), _p(logit_scale), _p(Wproj), _p(bproj),
        _p(out_host), _stream(stream)))


def swin_wattn_cpb_table(h, W1, b1, W2, table, stream=None):
    return _check("swin_wattn_cpb_table", load().swin_wattn_cpb_table(
        h, _p(W1), _p(b1), _p(W2), W1.shape[0], _p(table), _stream(stream)))


def swin_wattn_sync_status(h, stream=None):
    """Returns the status code (OK, ETIMEOUT or ECUDA) without raising."""
    return load().swin_wattn_sync_status(h, _stream(stream))


def swin_wattn_set_option(h, option, value):
    return _check("swin_wattn_set_option", load().swin_wattn_set_option(h, option, int(value)))


def swin_wattn_path(h, B, H, W):
    return load().swin_wattn_path(h, B, H, W)


def swin_wattn_last_launches(h):
    return load().swin_wattn_last_launches(h)


def swin_wattn_forward_noalloc(C, heads, M, shift, mode, x, Wqkv, bqkv, bias_table, logit_scale, Wproj, bproj,
                               out, stream=None):
    B, H, W, _ = x.shape
    return _check("swin_wattn_forward_noalloc", load().swin_wattn_forward_noalloc(
        C, heads, M, shift, mode, _p(x), B, H, W, _p(Wqkv), _p(bqkv), _p(bias_table), _p(logit_scale), _p(Wproj),
        _p(bproj), _p(out), _stream(stream)))


def swin_wattn_noalloc_sync_status(stream=None):
    """Status of the swin_wattn_forward_noalloc calls on the current device:
    the status code (OK, ETIMEOUT or ECUDA), without raising."""
    return load().swin_wattn_noalloc_sync_status(_stream(stream))


def swin_wattn_test_noalloc_watchdog(wait_limit_us, stream=None):
    return _check("swin_wattn_test_noalloc_watchdog",
                  load().swin_wattn_test_noalloc_watchdog(int(wait_limit_us), _stream(stream)))


def swin_wattn_test_qkv(h, x, Wqkv, bqkv, qkv, stream=None):
    B, H, W, _ = x.shape
    return _check("swin_wattn_test_qkv", load().swin_wattn_test_qkv(
        h, _p(x), B, H, W, _p(Wqkv), _p(bqkv), _p(qkv), _stream(stream)))


def swin_wattn_test_attn(h, qkv, B, H, W, bias_table, logit_scale, attn, stream=None):
    return _check("swin_wattn_test_attn", load().swin_wattn_test_attn(
        h, _p(qkv), B, H, W, _p(bias_table), _p(logit_scale), _p(attn), _stream(stream)))


def swin_wattn_test_proj(h, attn, B, H, W, Wproj, bproj, out, stream=None):
    return _check("swin_wattn_test_proj", load().swin_wattn_test_proj(
        h, _p(attn), B, H, W, _p(Wproj), _p(bproj), _p(out), _stream(stream)))


def swin_wattn_test_gemm(A, Bw, bias, D, swizzle_bytes=128, stream=None):
    rows, K = A.shape
    N = Bw.shape[0]
    return _check("swin_wattn_test_gemm", load().swin_wattn_test_gemm(
        _p(A), _p(Bw), _p(bias), _p(D), rows, N, K, swizzle_bytes, _stream(stream)))


def swin_wattn_test_corrupt_workspace(h, side):
    return _check("swin_wattn_test_corrupt_workspace", load().swin_wattn_test_corrupt_workspace(h, side))


def swin_wattn_test_watchdog(h, stream=None):
    return _check("swin_wattn_test_watchdog", load().swin_wattn_test_watchdog(h, _stream(stream)))


# ---- swin_block.h -------------------------------------------------------------

def swin_block_create(C, heads, M, shift, mode, mlp_ratio=4):
    h = ctypes.c_void_p()
    _check("swin_block_create", load().swin_block_create(ctypes.byref(h), C, heads, M, shift, mode, mlp_ratio))
    return h


def swin_block_destroy(h):
    return _check("swin_block_destroy", load().swin_block_destroy(h))


def swin_block_forward(h, x, params, out, stream=None):
    """params: dict with the swin_block_params fields (tensors or None)."""
    B, H, W, _ = x.shape
    bp = BlockParams(*[(_p(params.get(n)).value if params.get(n) is not None else None)
                       for n in BLOCK_PARAM_FIELDS])
    return _check("swin_block_forward", load().swin_block_forward(
        h, _p(x), B, H, W, ctypes.cast(ctypes.byref(bp), ctypes.c_void_p), _p(out), _stream(stream)))


def swin_block_last_launches(h):
    return load().swin_block_last_launches(h)


def swin_block_set_option(h, option, value):
    return _check("swin_block_set_option", load().swin_block_set_option(h, option, int(value)))


def swin_block_sync_status(h, stream=None):
    return _check("swin_block_sync_status", load().swin_block_sync_status(h, _stream(stream)))


def swin_block_test_layernorm(a, b, gamma, beta, out_sum, out_ln, flags, stream=None):
    rows, C = a.shape[0], a.shape[-1]
    return _check("swin_block_test_layernorm", load().swin_block_test_layernorm(
        _p(a), _p(b), _p(gamma), _p(beta), _p(out_sum), _p(out_ln), rows, C, flags, _stream(stream)))


def swin_stage_norm(x, gamma, beta, out, stream=None):
    """out = LN(x) over the last axis of x [..., C] (the extra LayerNorm of a V2
    stage); out may be x."""
    C = x.shape[-1]
    return _check("swin_stage_norm", load().swin_stage_norm(
        _p(x), x.numel() // C, C, _p(gamma), _p(beta), _p(out), _stream(stream)))


def swin_merge_create(C):
    h = ctypes.c_void_p()
    _check("swin_merge_create", load().swin_merge_create(ctypes.byref(h), C))
    return h


def swin_merge_destroy(h):
    return _check("swin_merge_destroy", load().swin_merge_destroy(h))


def swin_merge_forward(h, x, gamma, beta, Wm, out, stream=None):
    B, H, W, _ = x.shape
    return _check("swin_merge_forward", load().swin_merge_forward(
        h, _p(x), B, H, W, _p(gamma), _p(beta), _p(Wm), _p(out), _stream(stream)))

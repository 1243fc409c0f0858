"""Exact training attention (forward O, L and backward dQ, dK, dV) on one GB300.

Thin Python binding of the C-ABI library `libfa_gb300.so` (declared in include/fa_train.h).
This module only marshals arguments: PyTorch provides device memory and streams, and every
step of the computation runs in the library's sm_103a kernels. There is no fallback: if the
library is missing or was not built for this GPU, the calls raise.
"""
from __future__ import annotations

import ctypes
import os
import threading

from .build import LIB_PATH, build

__all__ = [
    "FaParams", "fa_train_fwd", "fa_train_bwd", "fa_device_status", "fa_error_string",
    "fa_version", "fa_profile_enable", "fa_profile_read", "attention_fwd", "attention_bwd", "load_library", "build", "LIB_PATH",
    "FA_OK", "FA_ERR_INVALID", "FA_ERR_CUDA", "FA_ERR_DEVICE_TIMEOUT", "FA_ERR_UNSUPPORTED",
    "FA_ERR_TOO_LARGE",
]

FA_OK = 0
FA_ERR_INVALID = 1
FA_ERR_CUDA = 2
FA_ERR_DEVICE_TIMEOUT = 3
FA_ERR_UNSUPPORTED = 4
FA_ERR_TOO_LARGE = 5


class FaParams(ctypes.Structure):
    """Mirror of `fa_params` in include/fa_train.h."""

    _fields_ = [
        ("batch", ctypes.c_int32),
        ("n_heads", ctypes.c_int32),
        ("n_kv_heads", ctypes.c_int32),
        ("ql", ctypes.c_int32),
        ("kl", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("scale", ctypes.c_float),
        ("causal", ctypes.c_int32),
    ]


_lib = None
_lock = threading.Lock()


class FaError(RuntimeError):
    def __init__(self, code, where):
        lib = load_library()
        text = lib.fa_error_string(code).decode()
        cuda = lib.fa_last_cuda_error().decode() if code == FA_ERR_CUDA else ""
        super().__init__(f"{where}: {text}" + (f" [{cuda}]" if cuda else ""))
        self.code = code


def load_library():
    """Load libfa_gb300.so (it must have been built: `flash_attention_gb300.build()`)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build the CUDA library first "
                    "(python -c 'import flash_attention_gb300 as f; f.build()')")
            lib = ctypes.CDLL(LIB_PATH)
            vp, fp = ctypes.c_void_p, ctypes.c_void_p
            pp = ctypes.POINTER(FaParams)
            lib.fa_train_fwd.argtypes = [vp, vp, vp, fp, vp, fp, pp, vp]
            lib.fa_train_fwd.restype = ctypes.c_int
            lib.fa_train_bwd.argtypes = [vp, vp, vp, vp, fp, vp, fp, vp, vp, vp, pp, vp]
            lib.fa_train_bwd.restype = ctypes.c_int
            lib.fa_device_status.argtypes = [ctypes.c_int]
            lib.fa_device_status.restype = ctypes.c_int
            lib.fa_error_string.argtypes = [ctypes.c_int]
            lib.fa_error_string.restype = ctypes.c_char_p
            lib.fa_last_cuda_error.restype = ctypes.c_char_p
            lib.fa_version.restype = ctypes.c_char_p
            lib.fa_profile_enable.argtypes = [ctypes.c_int]
            lib.fa_profile_enable.restype = ctypes.c_int
            lib.fa_profile_read.argtypes = [ctypes.POINTER(ctypes.c_double),
                                            ctypes.POINTER(ctypes.c_int64)]
            lib.fa_profile_read.restype = ctypes.c_int
            lib.fa_kernel_name.argtypes = [ctypes.c_int]
            lib.fa_kernel_name.restype = ctypes.c_char_p
            _lib = lib
    return _lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream):
    if stream is None:
        import torch

        stream = torch.cuda.current_stream()
    h = getattr(stream, "cuda_stream", stream)
    return ctypes.c_void_p(int(h))


def make_params(q, k, *, scale, causal) -> FaParams:
    B, H, ql, d = q.shape
    Bk, Hk, kl, dk = k.shape
    if B != Bk or d != dk:
        raise ValueError("q and k disagree on batch or head_dim")
    return FaParams(B, H, Hk, ql, kl, d, float(scale), int(bool(causal)))


def _check(t, dtype, name):
    import torch

    if t.dtype != dtype or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA {dtype} tensor")


def fa_train_fwd(q, k, v, mask, o, lse, params: FaParams, stream=None) -> None:
    """C call `fa_train_fwd` on torch tensors (q, k, v, o bf16; mask, lse f32)."""
    import torch

    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o")):
        _check(t, torch.bfloat16, n)
    _check(lse, torch.float32, "lse")
    if mask is not None:
        _check(mask, torch.float32, "mask")
    rc = load_library().fa_train_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(mask), _ptr(o), _ptr(lse),
                                     ctypes.byref(params), _stream_handle(stream))
    if rc:
        raise FaError(rc, "fa_train_fwd")


def fa_train_bwd(q, k, v, o, lse, dO, mask, dq, dk, dv, params: FaParams, stream=None) -> None:
    """C call `fa_train_bwd` on torch tensors."""
    import torch

    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (dO, "dO"), (dq, "dq"), (dk, "dk"),
                 (dv, "dv")):
        _check(t, torch.bfloat16, n)
    _check(lse, torch.float32, "lse")
    if mask is not None:
        _check(mask, torch.float32, "mask")
    rc = load_library().fa_train_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO),
                                     _ptr(mask), _ptr(dq), _ptr(dk), _ptr(dv),
                                     ctypes.byref(params), _stream_handle(stream))
    if rc:
        raise FaError(rc, "fa_train_bwd")


def fa_device_status(clear: bool = True) -> int:
    return load_library().fa_device_status(int(bool(clear)))


FA_NUM_KERNELS = 4


def fa_profile_enable(on: bool) -> None:
    load_library().fa_profile_enable(int(bool(on)))


def fa_profile_read():
    """{kernel name: (total device ms, launches)} since the last read (then cleared)."""
    lib = load_library()
    ms = (ctypes.c_double * FA_NUM_KERNELS)()
    n = (ctypes.c_int64 * FA_NUM_KERNELS)()
    rc = lib.fa_profile_read(ms, n)
    if rc:
        raise FaError(rc, "fa_profile_read")
    return {lib.fa_kernel_name(k).decode(): (ms[k], n[k]) for k in range(FA_NUM_KERNELS)}


def fa_error_string(code: int) -> str:
    return load_library().fa_error_string(int(code)).decode()


def fa_version() -> str:
    return load_library().fa_version().decode()


def attention_fwd(q, k, v, *, scale, causal, mask=None, stream=None):
    """Allocate O and L and run the forward: returns (o, lse)."""
    import torch

    B, H, ql, d = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, H, ql), dtype=torch.float32, device=q.device)
    fa_train_fwd(q, k, v, mask, o, lse, make_params(q, k, scale=scale, causal=causal), stream)
    return o, lse


def attention_bwd(q, k, v, o, lse, dO, *, scale, causal, mask=None, stream=None):
    """Allocate dQ, dK, dV and run the backward: returns (dq, dk, dv)."""
    import torch

    dq = torch.empty_like(q)
    dk = torch.empty_like(k)
    dv = torch.empty_like(v)
    fa_train_bwd(q, k, v, o, lse, dO, mask, dq, dk, dv,
                 make_params(q, k, scale=scale, causal=causal), stream)
    return dq, dk, dv

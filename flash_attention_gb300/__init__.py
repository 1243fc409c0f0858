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
    "FA_ERR_TOO_LARGE", "FA_ERR_BAD_INPUT", "FaOptions", "FaPagedParams", "paged_attention",
    "fa_paged_attention", "fa_paged_attention_bwd", "fa_train_fwd_ex", "fa_train_bwd_ex", "make_options",
    "FA_MASK_F32", "FA_MASK_BF16", "FA_MASK_BOOL",
]

FA_OK = 0
FA_ERR_INVALID = 1
FA_ERR_CUDA = 2
FA_ERR_DEVICE_TIMEOUT = 3
FA_ERR_UNSUPPORTED = 4
FA_ERR_TOO_LARGE = 5
FA_ERR_BAD_INPUT = 6


FA_MASK_F32 = 0
FA_MASK_BF16 = 1
FA_MASK_BOOL = 2
FA_LAYOUT_Q_BSHD = 1   # q, o, dO, dq as [batch, seq, heads, dim] in memory
FA_LAYOUT_KV_BSHD = 2  # k, v, dk, dv as [batch, seq, kv_heads, dim] in memory


class FaOptions(ctypes.Structure):
    """Mirror of `fa_options` in include/fa_train.h."""

    _fields_ = [
        ("window_left", ctypes.c_int32),
        ("window_right", ctypes.c_int32),
        ("mask_type", ctypes.c_int32),
        ("value_dim", ctypes.c_int32),
        ("mask_stride_b", ctypes.c_int64),
        ("mask_stride_h", ctypes.c_int64),
        ("mask_stride_q", ctypes.c_int64),
        ("sinks", ctypes.c_void_p),
        ("dsinks", ctypes.c_void_p),
        ("deterministic", ctypes.c_int32),
        ("layout", ctypes.c_int32),
        ("cu_seqlens_q", ctypes.c_void_p),
        ("cu_seqlens_k", ctypes.c_void_p),
        ("total_q", ctypes.c_int32),
        ("total_k", ctypes.c_int32),
    ]


class FaPagedParams(ctypes.Structure):
    """Mirror of `fa_paged_params` in include/fa_train.h."""

    _fields_ = [
        ("batch", ctypes.c_int32),
        ("n_heads", ctypes.c_int32),
        ("n_kv_heads", ctypes.c_int32),
        ("q_len", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("max_pages", ctypes.c_int32),
        ("num_pages", ctypes.c_int32),
        ("scale", ctypes.c_float),
        ("causal", ctypes.c_int32),
        ("num_splits", ctypes.c_int32),
        ("reserved", ctypes.c_int32),
    ]


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
            po = ctypes.POINTER(FaOptions)
            lib.fa_train_fwd_ex.argtypes = [vp, vp, vp, vp, vp, fp, pp, po, vp]
            lib.fa_train_fwd_ex.restype = ctypes.c_int
            lib.fa_train_bwd_ex.argtypes = [vp, vp, vp, vp, fp, vp, vp, vp, vp, vp, pp, po, vp]
            lib.fa_train_bwd_ex.restype = ctypes.c_int
            lib.fa_paged_attention.argtypes = [vp, vp, vp, vp, vp, vp, fp, vp, vp]
            lib.fa_paged_attention.restype = ctypes.c_int
            lib.fa_paged_attention_bwd.argtypes = [vp, vp, vp, vp, vp, vp, fp, vp, vp, vp, vp,
                                                   vp, vp]
            lib.fa_paged_attention_bwd.restype = ctypes.c_int
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
            lib.fa_train_bwd_noalloc.argtypes = [vp, vp, vp, vp, fp, vp, fp, vp, vp, vp, pp, vp]
            lib.fa_train_bwd_noalloc.restype = ctypes.c_int
            lib.fa_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
            lib.fa_set_wait_limit_ns.restype = ctypes.c_int
            lib.fa_get_wait_limit_ns.argtypes = []
            lib.fa_get_wait_limit_ns.restype = ctypes.c_uint64
            lib.fa_debug_ex2.argtypes = [vp, vp, vp, vp, ctypes.c_int64, vp]
            lib.fa_debug_ex2.restype = ctypes.c_int
            lib.fa_debug_wait_timeout.argtypes = [vp, vp]
            lib.fa_debug_wait_timeout.restype = ctypes.c_int
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


def _layout_bit(t) -> int:
    """0 if `t` ([..., heads, rows, dim]) is contiguous, 1 if it is the transposed view of a
    contiguous [..., rows, heads, dim] tensor (the memory layout the FA_LAYOUT_* flags name)."""
    if t.is_contiguous():
        return 0
    if t.transpose(-3, -2).is_contiguous():
        return 1
    raise ValueError("a [.., heads, rows, dim] tensor must be contiguous or a transposed view of "
                     "a contiguous [.., rows, heads, dim] tensor")


def _check_bf16(t, bshd, name):
    import torch

    if t.dtype != torch.bfloat16 or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA bfloat16 tensor")
    ok = t.transpose(-3, -2).is_contiguous() if bshd else t.is_contiguous()
    if not ok:
        raise ValueError(f"{name} must be laid out as " +
                         ("[.., rows, heads, dim]" if bshd else "[.., heads, rows, dim]"))


def _check_sides(options, q_side, kv_side):
    """Checks the q-side (q, o, dO, dq) and kv-side (k, v, dk, dv) tensors against the layout
    flags of `options`."""
    for t, n in q_side:
        _check_bf16(t, options.layout & FA_LAYOUT_Q_BSHD, n)
    for t, n in kv_side:
        _check_bf16(t, options.layout & FA_LAYOUT_KV_BSHD, n)


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


def make_options(q, k, mask=None, window=(-1, -1), v=None, sinks=None, dsinks=None,
                 deterministic=False) -> FaOptions:
    """fa_options for a mask tensor of any supported dtype (float32, bfloat16, bool) whose shape
    broadcasts to [B, H, ql, kl] with the keys contiguous, a (left, right) window, the value
    head dim of `v` (when it differs from q's), float32 [H] sinks / dsinks tensors, the
    deterministic backward, and the memory layouts of q and k (contiguous, or transposed views
    of [B, seq, heads, dim] tensors)."""
    import torch

    B, H, ql, d = q.shape
    kl = k.shape[2]
    wl, wr = window if window is not None else (-1, -1)
    layout = FA_LAYOUT_Q_BSHD * _layout_bit(q) | FA_LAYOUT_KV_BSHD * _layout_bit(k)
    opt = FaOptions(int(wl), int(wr), FA_MASK_F32, 0, 0, 0, 0, None, None,
                    1 if deterministic else 0, layout, None, None, 0, 0)
    if v is not None and v.shape[-1] != d:
        opt.value_dim = int(v.shape[-1])
    if mask is not None:
        types = {torch.float32: FA_MASK_F32, torch.bfloat16: FA_MASK_BF16, torch.bool: FA_MASK_BOOL,
                 torch.uint8: FA_MASK_BOOL}
        if mask.dtype not in types or not mask.is_cuda:
            raise ValueError("mask must be a CUDA float32, bfloat16 or bool tensor")
        e = mask.expand(B, H, ql, kl)
        sb, sh, sq, sk = e.stride()
        if kl > 1 and sk != 1:
            raise ValueError("the mask's key dimension must be contiguous")
        opt.mask_type = types[mask.dtype]
        opt.mask_stride_b, opt.mask_stride_h, opt.mask_stride_q = sb, sh, sq
    for name, t in (("sinks", sinks), ("dsinks", dsinks)):
        if t is None:
            continue
        if t.dtype != torch.float32 or not t.is_cuda or tuple(t.shape) != (H,) or \
                not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA float32 tensor of shape [{H}]")
        setattr(opt, name, t.data_ptr())
    return opt


def fa_train_fwd_ex(q, k, v, mask, o, lse, params: FaParams, options: FaOptions,
                    stream=None) -> None:
    """C call `fa_train_fwd_ex` (window, mask type and broadcast in `options`)."""
    import torch

    _check_sides(options, ((q, "q"), (o, "o")), ((k, "k"), (v, "v")))
    _check(lse, torch.float32, "lse")
    rc = load_library().fa_train_fwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(mask), _ptr(o), _ptr(lse),
                                        ctypes.byref(params), ctypes.byref(options),
                                        _stream_handle(stream))
    if rc:
        raise FaError(rc, "fa_train_fwd_ex")


def fa_train_bwd_ex(q, k, v, o, lse, dO, mask, dq, dk, dv, params: FaParams, options: FaOptions,
                    stream=None) -> None:
    """C call `fa_train_bwd_ex`."""
    import torch

    _check_sides(options, ((q, "q"), (o, "o"), (dO, "dO"), (dq, "dq")),
                 ((k, "k"), (v, "v"), (dk, "dk"), (dv, "dv")))
    _check(lse, torch.float32, "lse")
    rc = load_library().fa_train_bwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO),
                                        _ptr(mask), _ptr(dq), _ptr(dk), _ptr(dv),
                                        ctypes.byref(params), ctypes.byref(options),
                                        _stream_handle(stream))
    if rc:
        raise FaError(rc, "fa_train_bwd_ex")


def fa_device_status(clear: bool = True) -> int:
    return load_library().fa_device_status(int(bool(clear)))


FA_NUM_KERNELS = 10


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


def fa_train_bwd_noalloc(q, k, v, o, lse, dO, mask, dq, dk, dv, params: FaParams,
                         stream=None) -> None:
    """C call `fa_train_bwd_noalloc` (the backward with its scratch in the library's fixed
    device array; no allocation)."""
    import torch

    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (dO, "dO"), (dq, "dq"), (dk, "dk"),
                 (dv, "dv")):
        _check(t, torch.bfloat16, n)
    _check(lse, torch.float32, "lse")
    if mask is not None:
        _check(mask, torch.float32, "mask")
    rc = load_library().fa_train_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                             _ptr(dO), _ptr(mask), _ptr(dq), _ptr(dk), _ptr(dv),
                                             ctypes.byref(params), _stream_handle(stream))
    if rc:
        raise FaError(rc, "fa_train_bwd_noalloc")


def fa_set_wait_limit_ns(ns: int) -> None:
    """Limit of one barrier wait in the kernels launched from now on (0: the default 2 s)."""
    rc = load_library().fa_set_wait_limit_ns(int(ns))
    if rc:
        raise FaError(rc, "fa_set_wait_limit_ns")


def fa_get_wait_limit_ns() -> int:
    return int(load_library().fa_get_wait_limit_ns())


def fa_debug_ex2(x, stream=None):
    """The softmax's two exp2 forms and CUDA's exp2f on a CUDA float32 tensor:
    (polynomial, hardware approximation, exp2f)."""
    import torch

    _check(x, torch.float32, "x")
    outs = [torch.empty_like(x) for _ in range(3)]
    rc = load_library().fa_debug_ex2(_ptr(x), *(_ptr(t) for t in outs), x.numel(),
                                     _stream_handle(stream))
    if rc:
        raise FaError(rc, "fa_debug_ex2")
    return tuple(outs)


def fa_debug_wait_timeout(stream=None):
    """Launches the kernel that waits on a barrier nothing completes; returns a CUDA int64
    tensor that receives how long it waited (ns)."""
    import torch

    waited = torch.zeros(1, dtype=torch.int64, device="cuda")
    rc = load_library().fa_debug_wait_timeout(_ptr(waited), _stream_handle(stream))
    if rc:
        raise FaError(rc, "fa_debug_wait_timeout")
    return waited


def _plain_call(q, k, v, mask, window, sinks):
    """True when the base entry point covers the call (dense f32 mask or none, no window, no
    sinks, value head dim = head dim)."""
    import torch

    B, H, ql, d = q.shape
    dense = mask is None or (mask.dtype == torch.float32 and mask.dim() == 4
                             and mask.is_contiguous()
                             and tuple(mask.shape) == (B, H, ql, k.shape[2]))
    contiguous = q.is_contiguous() and k.is_contiguous() and v.is_contiguous()
    return dense and contiguous and window is None and sinks is None and v.shape[-1] == d


def attention_fwd(q, k, v, *, scale, causal, mask=None, window=None, sinks=None, stream=None):
    """Allocate O and L and run the forward: returns (o, lse). `mask`: None, or a float32 /
    bfloat16 additive or bool mask broadcastable to [B, H, ql, kl]; `window`: None or
    (left, right) with -1 for an unbounded side; `sinks`: None or float32 [H] logits. v may
    have its own head dim (o then has it too)."""
    import torch

    B, H, ql, d = q.shape
    if _layout_bit(q):  # o in q's layout
        o = torch.empty((B, ql, H, v.shape[-1]), dtype=q.dtype, device=q.device).transpose(1, 2)
    else:
        o = torch.empty((B, H, ql, v.shape[-1]), dtype=q.dtype, device=q.device)
    lse = torch.empty((B, H, ql), dtype=torch.float32, device=q.device)
    params = make_params(q, k, scale=scale, causal=causal)
    if _plain_call(q, k, v, mask, window, sinks):
        fa_train_fwd(q, k, v, mask, o, lse, params, stream)
    else:
        fa_train_fwd_ex(q, k, v, mask, o, lse, params,
                        make_options(q, k, mask, window, v=v, sinks=sinks), stream)
    return o, lse


def attention_bwd(q, k, v, o, lse, dO, *, scale, causal, mask=None, window=None, sinks=None,
                  deterministic=False, stream=None):
    """Allocate dQ, dK, dV and run the backward: returns (dq, dk, dv), or (dq, dk, dv, dsinks)
    when `sinks` is given. `mask`, `window` and `sinks` as given to attention_fwd;
    `deterministic` makes every output bitwise reproducible (dQ from its own kernel)."""
    import torch

    dq = torch.empty_like(q)
    dk = torch.empty_like(k)
    dv = torch.empty_like(v)
    params = make_params(q, k, scale=scale, causal=causal)
    if _plain_call(q, k, v, mask, window, sinks) and not deterministic:
        fa_train_bwd(q, k, v, o, lse, dO, mask, dq, dk, dv, params, stream)
        return dq, dk, dv
    dsinks = None if sinks is None else torch.empty_like(sinks)
    fa_train_bwd_ex(q, k, v, o, lse, dO, mask, dq, dk, dv, params,
                    make_options(q, k, mask, window, v=v, sinks=sinks, dsinks=dsinks,
                                 deterministic=deterministic), stream)
    return (dq, dk, dv) if sinks is None else (dq, dk, dv, dsinks)


def fa_paged_attention(q, k_cache, v_cache, block_table, lengths, o, lse, params: FaPagedParams,
                       stream=None) -> None:
    """C call `fa_paged_attention` (q, caches, o bf16; block_table, lengths int32; lse f32 or
    None)."""
    import torch

    for t, n in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache"), (o, "o")):
        _check(t, torch.bfloat16, n)
    _check(block_table, torch.int32, "block_table")
    _check(lengths, torch.int32, "lengths")
    if lse is not None:
        _check(lse, torch.float32, "lse")
    rc = load_library().fa_paged_attention(_ptr(q), _ptr(k_cache), _ptr(v_cache),
                                           _ptr(block_table), _ptr(lengths), _ptr(o), _ptr(lse),
                                           ctypes.byref(params), _stream_handle(stream))
    if rc:
        raise FaError(rc, "fa_paged_attention")


def paged_attention(q, k_cache, v_cache, block_table, lengths, *, scale, causal=True,
                    num_splits=0, stream=None):
    """Attention of q [B, H, q_len, d] over paged caches [num_pages, Hk, page_size, d] with a
    block table [B, max_pages] and lengths [B] (int32, on the device): returns (o, lse). The
    q_len queries are each sequence's last positions (causal: bottom-right per sequence)."""
    import torch

    B, H, lq, d = q.shape
    P, Hk, bs, _ = k_cache.shape
    params = FaPagedParams(B, H, Hk, lq, d, bs, block_table.shape[1], P, float(scale),
                           int(bool(causal)), int(num_splits), 0)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, lq), dtype=torch.float32, device=q.device)
    fa_paged_attention(q, k_cache, v_cache, block_table, lengths, o, lse, params, stream)
    return o, lse


def fa_paged_attention_bwd(q, k_cache, v_cache, block_table, lengths, o, lse, dO, dq, dk_cache,
                           dv_cache, params: FaPagedParams, stream=None) -> None:
    """C call `fa_paged_attention_bwd` (gradients for q and both caches)."""
    import torch

    for t, n in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache"), (o, "o"), (dO, "dO"),
                 (dq, "dq"), (dk_cache, "dk_cache"), (dv_cache, "dv_cache")):
        _check(t, torch.bfloat16, n)
    _check(block_table, torch.int32, "block_table")
    _check(lengths, torch.int32, "lengths")
    _check(lse, torch.float32, "lse")
    rc = load_library().fa_paged_attention_bwd(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(lengths), _ptr(o),
        _ptr(lse), _ptr(dO), _ptr(dq), _ptr(dk_cache), _ptr(dv_cache), ctypes.byref(params),
        _stream_handle(stream))
    if rc:
        raise FaError(rc, "fa_paged_attention_bwd")


def paged_attention_bwd(q, k_cache, v_cache, block_table, lengths, o, lse, dO, *, scale,
                        causal=True, stream=None):
    """Gradients of paged_attention: returns (dq, dk_cache, dv_cache), the cache gradients
    shaped like the caches (0 in every slot no sequence reads)."""
    import torch

    B, H, lq, d = q.shape
    P, Hk, bs, _ = k_cache.shape
    params = FaPagedParams(B, H, Hk, lq, d, bs, block_table.shape[1], P, float(scale),
                           int(bool(causal)), 0, 0)
    dq = torch.empty_like(q)
    dk = torch.empty_like(k_cache)
    dv = torch.empty_like(v_cache)
    fa_paged_attention_bwd(q, k_cache, v_cache, block_table, lengths, o, lse, dO, dq, dk, dv,
                           params, stream)
    return dq, dk, dv


def varlen_params_options(q, k, v, cu_q, cu_k, max_q, max_k, *, scale, causal, window=None,
                          sinks=None, dsinks=None, deterministic=False):
    """FaParams and FaOptions of a variable-length batch: q [H, total_q, d], k and v
    [Hk, total_k, d(v)], cu_q / cu_k int32 CUDA tensors of batch + 1 offsets, max_q / max_k the
    longest sequence."""
    import torch

    H, Tq, d = q.shape
    Hk, Tk, _ = k.shape
    for t, n in ((cu_q, "cu_q"), (cu_k, "cu_k")):
        _check(t, torch.int32, n)
    B = cu_q.numel() - 1
    params = FaParams(B, H, Hk, int(max_q), int(max_k), d, float(scale), int(bool(causal)))
    opt = make_options(q[None], k[None], None, window, v=v[None], sinks=sinks, dsinks=dsinks,
                       deterministic=deterministic)
    opt.cu_seqlens_q = cu_q.data_ptr()
    opt.cu_seqlens_k = cu_k.data_ptr()
    opt.total_q, opt.total_k = Tq, Tk
    return params, opt


def varlen_attention_fwd(q, k, v, cu_q, cu_k, max_q, max_k, *, scale, causal, window=None,
                         sinks=None, stream=None):
    """Forward of a variable-length batch (see varlen_params_options): returns (o, lse) with
    o [H, total_q, dv] and lse [H, total_q]."""
    import torch

    H, Tq, _ = q.shape
    if _layout_bit(q):  # o in q's layout: [total_q, H, dv] memory
        o = torch.empty((Tq, H, v.shape[2]), dtype=q.dtype, device=q.device).transpose(0, 1)
    else:
        o = torch.empty((H, Tq, v.shape[2]), dtype=q.dtype, device=q.device)
    lse = torch.empty((H, Tq), dtype=torch.float32, device=q.device)
    params, opt = varlen_params_options(q, k, v, cu_q, cu_k, max_q, max_k, scale=scale,
                                        causal=causal, window=window, sinks=sinks)
    fa_train_fwd_ex(q, k, v, None, o, lse, params, opt, stream)
    return o, lse


def varlen_attention_bwd(q, k, v, o, lse, dO, cu_q, cu_k, max_q, max_k, *, scale, causal,
                         window=None, sinks=None, deterministic=False, stream=None):
    """Backward of a variable-length batch: returns (dq, dk, dv) (+ dsinks with sinks)."""
    import torch

    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    dsinks = None if sinks is None else torch.empty_like(sinks)
    params, opt = varlen_params_options(q, k, v, cu_q, cu_k, max_q, max_k, scale=scale,
                                        causal=causal, window=window, sinks=sinks,
                                        dsinks=dsinks, deterministic=deterministic)
    fa_train_bwd_ex(q, k, v, o, lse, dO, None, dq, dk, dv, params, opt, stream)
    return (dq, dk, dv) if sinks is None else (dq, dk, dv, dsinks)

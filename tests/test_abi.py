"""The C-ABI library without a GPU: it loads, exports every symbol include/fa_train.h declares,
and rejects bad arguments with FA_ERR_INVALID before it touches the device or any pointer."""
import ctypes
import os
import re

import pytest

import flash_attention_gb300 as fa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa_train.h")


@pytest.fixture(scope="module")
def lib():
    fa.build()
    return fa.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("fa_train_fwd", "fa_train_bwd", "fa_error_string"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in include/fa_train.h but not exported"


def test_error_strings(lib):
    for code in range(7):
        assert fa.fa_error_string(code)
    names = [fa.load_library().fa_kernel_name(k).decode() for k in range(fa.FA_NUM_KERNELS)]
    assert len(set(names)) == fa.FA_NUM_KERNELS and "unknown" not in " ".join(names)
    assert {"bwd_dq_det_kernel", "paged_attn_kernel", "paged_combine_kernel"} <= set(names)
    assert "paged" in fa.fa_error_string(fa.FA_ERR_BAD_INPUT)
    assert "unknown" in fa.fa_error_string(99)
    assert "sm_103a" in fa.fa_version()


def test_params_struct_layout():
    assert ctypes.sizeof(fa.FaParams) == 32
    assert fa.FaParams.scale.offset == 24 and fa.FaParams.causal.offset == 28


GOOD = dict(batch=1, n_heads=4, n_kv_heads=2, ql=128, kl=128, head_dim=128, scale=0.125, causal=1)
FAKE = 0x100000  # a 16-byte aligned address that is never dereferenced: checks come first


def _fwd(lib, params, q=FAKE, k=FAKE, v=FAKE, mask=None, o=FAKE, lse=FAKE):
    p = fa.FaParams(**params)
    return lib.fa_train_fwd(q, k, v, mask, o, lse, ctypes.byref(p), None)


def _bwd(lib, params, ptrs=None, mask=None):
    p = fa.FaParams(**params)
    a = [FAKE] * 9 if ptrs is None else ptrs
    q, k, v, o, lse, dO, dq, dk, dv = a
    return lib.fa_train_bwd(q, k, v, o, lse, dO, mask, dq, dk, dv, ctypes.byref(p), None)


BAD_PARAMS = [
    ("batch", 0), ("n_heads", 0), ("n_kv_heads", 0), ("ql", 0), ("kl", -3), ("head_dim", 96),
    ("head_dim", 32), ("n_heads", 3), ("scale", 0.0), ("scale", -1.0), ("scale", float("inf")),
    ("scale", float("nan")), ("causal", 2), ("ql", (1 << 22) + 1), ("kl", 1 << 23),
]


@pytest.mark.parametrize("field,value", BAD_PARAMS)
def test_bad_params_rejected(lib, field, value):
    bad = dict(GOOD, **{field: value})
    assert _fwd(lib, bad) == fa.FA_ERR_INVALID
    assert _bwd(lib, bad) == fa.FA_ERR_INVALID


def test_null_params_rejected(lib):
    assert lib.fa_train_fwd(FAKE, FAKE, FAKE, None, FAKE, FAKE, None, None) == fa.FA_ERR_INVALID


@pytest.mark.parametrize("slot", range(5))
def test_null_or_misaligned_pointer_rejected_fwd(lib, slot):
    for bad in (None, FAKE + 2, FAKE + 8):
        ptrs = [FAKE] * 5
        ptrs[slot] = bad
        q, k, v, o, lse = ptrs
        assert _fwd(lib, GOOD, q, k, v, None, o, lse) == fa.FA_ERR_INVALID


@pytest.mark.parametrize("slot", range(9))
def test_null_or_misaligned_pointer_rejected_bwd(lib, slot):
    for bad in (None, FAKE + 2):
        ptrs = [FAKE] * 9
        ptrs[slot] = bad
        assert _bwd(lib, GOOD, ptrs) == fa.FA_ERR_INVALID


def test_misaligned_mask_rejected(lib):
    assert _fwd(lib, GOOD, mask=FAKE + 4) == fa.FA_ERR_INVALID
    assert _bwd(lib, GOOD, mask=FAKE + 4) == fa.FA_ERR_INVALID


def test_valid_call_without_gpu_fails_cleanly(lib):
    """With no usable device the call reports a CUDA or device error; it never crashes."""
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    rc = _fwd(lib, GOOD)
    assert rc in (fa.FA_ERR_CUDA, fa.FA_ERR_UNSUPPORTED)


def _fwd_ex(lib, params, opts, mask=None):
    p = fa.FaParams(**params)
    return lib.fa_train_fwd_ex(FAKE, FAKE, FAKE, mask, FAKE, FAKE, ctypes.byref(p),
                               ctypes.byref(opts) if opts is not None else None, None)


def _bwd_ex(lib, params, opts, mask=None):
    p = fa.FaParams(**params)
    return lib.fa_train_bwd_ex(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, mask, FAKE, FAKE, FAKE,
                               ctypes.byref(p), ctypes.byref(opts) if opts is not None else None,
                               None)


def _opts(**kw):
    base = dict(window_left=-1, window_right=-1, mask_type=0, value_dim=0, mask_stride_b=0,
                mask_stride_h=0, mask_stride_q=128, sinks=None, dsinks=None, deterministic=0,
                layout=0, cu_seqlens_q=None, cu_seqlens_k=None, total_q=0, total_k=0)
    base.update(kw)
    return fa.FaOptions(**base)


BAD_OPTIONS = [
    dict(window_left=-2), dict(window_right=-5), dict(mask_type=3), dict(mask_type=-1),
    dict(value_dim=-1), dict(mask_stride_b=-1), dict(mask_stride_h=-4),
    dict(mask_stride_q=-128), dict(sinks=FAKE + 2), dict(deterministic=2), dict(layout=4), dict(layout=-1),
    dict(cu_seqlens_q=FAKE), dict(cu_seqlens_q=FAKE, cu_seqlens_k=FAKE + 2, total_q=4, total_k=4),
    dict(cu_seqlens_q=FAKE, cu_seqlens_k=FAKE, total_q=0, total_k=4),
]


@pytest.mark.parametrize("kw", BAD_OPTIONS, ids=lambda kw: ",".join(f"{k}={v}" for k, v in kw.items()))
def test_bad_options_rejected(lib, kw):
    assert _fwd_ex(lib, GOOD, _opts(**kw), mask=FAKE) == fa.FA_ERR_INVALID
    assert _bwd_ex(lib, GOOD, _opts(**kw), mask=FAKE) == fa.FA_ERR_INVALID


def test_mask_alignment_follows_its_element_type(lib):
    # f32 needs 4-byte alignment, bf16 2, bool 1
    assert _fwd_ex(lib, GOOD, _opts(mask_type=0), mask=FAKE + 2) == fa.FA_ERR_INVALID
    assert _fwd_ex(lib, GOOD, _opts(mask_type=1), mask=FAKE + 1) == fa.FA_ERR_INVALID
    import torch

    if not torch.cuda.is_available():
        # checks pass, then the device check fails cleanly
        assert _fwd_ex(lib, GOOD, _opts(mask_type=2), mask=FAKE + 1) in (fa.FA_ERR_CUDA,
                                                                          fa.FA_ERR_UNSUPPORTED)
        assert _fwd_ex(lib, GOOD, _opts(window_left=0, window_right=0)) in (
            fa.FA_ERR_CUDA, fa.FA_ERR_UNSUPPORTED)


def test_dsinks_rules_in_the_backward(lib):
    # dsinks needs sinks, and 4-byte alignment; the forward ignores dsinks
    assert _bwd_ex(lib, GOOD, _opts(dsinks=FAKE)) == fa.FA_ERR_INVALID
    assert _bwd_ex(lib, GOOD, _opts(sinks=FAKE, dsinks=FAKE + 2)) == fa.FA_ERR_INVALID
    import torch

    if not torch.cuda.is_available():
        assert _fwd_ex(lib, GOOD, _opts(dsinks=FAKE)) in (fa.FA_ERR_CUDA, fa.FA_ERR_UNSUPPORTED)
        assert _bwd_ex(lib, GOOD, _opts(sinks=FAKE, dsinks=FAKE)) in (fa.FA_ERR_CUDA,
                                                                       fa.FA_ERR_UNSUPPORTED)


def test_value_dim_without_kernels_is_unsupported(lib):
    assert not lib.fa_value_dim_supported(128, 96)
    assert not lib.fa_value_dim_supported(64, 128)
    assert lib.fa_value_dim_supported(128, 128)
    assert lib.fa_value_dim_supported(128, 64)
    assert _fwd_ex(lib, GOOD, _opts(value_dim=96)) == fa.FA_ERR_UNSUPPORTED
    assert _bwd_ex(lib, GOOD, _opts(value_dim=96)) == fa.FA_ERR_UNSUPPORTED


def test_varlen_with_a_mask_is_unsupported(lib):
    o = _opts(cu_seqlens_q=FAKE, cu_seqlens_k=FAKE, total_q=8, total_k=8)
    assert _fwd_ex(lib, GOOD, o, mask=FAKE) == fa.FA_ERR_UNSUPPORTED


def test_options_struct_layout():
    assert ctypes.sizeof(fa.FaOptions) == 88
    assert fa.FaOptions.cu_seqlens_q.offset == 64 and fa.FaOptions.total_k.offset == 84
    assert fa.FaOptions.deterministic.offset == 56
    assert fa.FaOptions.mask_stride_b.offset == 16
    assert fa.FaOptions.sinks.offset == 40 and fa.FaOptions.dsinks.offset == 48


PAGED_GOOD = dict(batch=2, n_heads=8, n_kv_heads=2, q_len=1, head_dim=128, page_size=16,
                  max_pages=4, num_pages=10, scale=0.1, causal=1, num_splits=0, reserved=0)


def _paged(lib, params, table=FAKE, lens=FAKE, lse=None, q=FAKE):
    p = fa.FaPagedParams(**params)
    return lib.fa_paged_attention(q, FAKE, FAKE, table, lens, FAKE, lse, ctypes.byref(p), None)


BAD_PAGED = [
    ("batch", 0), ("n_heads", 7), ("q_len", 0), ("head_dim", 96), ("page_size", 12),
    ("page_size", 4), ("page_size", 512), ("max_pages", 0), ("num_pages", 0), ("scale", 0.0),
    ("causal", 3), ("num_splits", -1), ("reserved", 2), ("max_pages", 1 << 19),
]


@pytest.mark.parametrize("field,value", BAD_PAGED)
def test_paged_bad_params_rejected(lib, field, value):
    assert _paged(lib, dict(PAGED_GOOD, **{field: value})) == fa.FA_ERR_INVALID


def test_paged_bad_pointers_rejected(lib):
    assert lib.fa_paged_attention(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, None) == \
        fa.FA_ERR_INVALID
    assert _paged(lib, PAGED_GOOD, table=None) == fa.FA_ERR_INVALID
    assert _paged(lib, PAGED_GOOD, lens=FAKE + 2) == fa.FA_ERR_INVALID
    assert _paged(lib, PAGED_GOOD, lse=FAKE + 1) == fa.FA_ERR_INVALID
    assert _paged(lib, PAGED_GOOD, q=FAKE + 8) == fa.FA_ERR_INVALID


def _paged_bwd(lib, params, lse=FAKE, dk=FAKE, q=FAKE):
    p = fa.FaPagedParams(**params)
    return lib.fa_paged_attention_bwd(q, FAKE, FAKE, FAKE, FAKE, FAKE, lse, FAKE, FAKE, dk, FAKE,
                                      ctypes.byref(p), None)


@pytest.mark.parametrize("field,value", BAD_PAGED)
def test_paged_bwd_bad_params_rejected(lib, field, value):
    assert _paged_bwd(lib, dict(PAGED_GOOD, **{field: value})) == fa.FA_ERR_INVALID


def test_paged_bwd_bad_pointers_rejected(lib):
    assert _paged_bwd(lib, PAGED_GOOD, lse=None) == fa.FA_ERR_INVALID  # lse is required
    assert _paged_bwd(lib, PAGED_GOOD, lse=FAKE + 4) == fa.FA_ERR_INVALID
    assert _paged_bwd(lib, PAGED_GOOD, dk=FAKE + 2) == fa.FA_ERR_INVALID
    assert _paged_bwd(lib, PAGED_GOOD, q=None) == fa.FA_ERR_INVALID
    # more than 8 query rows per kv head take the packed path, whose batch * capacity rows
    # per kv head must stay within the tensor maps
    assert _paged_bwd(lib, dict(PAGED_GOOD, batch=600, n_heads=16, n_kv_heads=8, q_len=8,
                                max_pages=65536, num_pages=1000)) == fa.FA_ERR_INVALID


def test_paged_params_struct_layout():
    assert ctypes.sizeof(fa.FaPagedParams) == 48
    assert fa.FaPagedParams.scale.offset == 32

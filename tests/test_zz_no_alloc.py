"""The backward entry point that allocates no device memory (fa_train_bwd_noalloc).

It exists for callers that cannot let a library allocate on the GPU: a process whose device
memory belongs to a pool allocator that has already reserved it, or a step loop in which an
allocation is not allowed to block or fail. Those callers hand in every input and output, and
the library takes its scratch from a fixed array that is part of the library itself.

This test calls it through the C ABI and checks that, on two calls in a row, it gives what the
ordinary allocating entry point fa_train_bwd gives, within the gradient tolerance of the parity
tests (max |difference| <= 2e-2 * max |gradient|). It also checks that a problem too large for
the fixed array is refused before anything runs. It is self-contained, so it passes alone in a
fresh process as well as after the other tests; the file name makes pytest collect it last.
"""
import ctypes

import numpy as np
import pytest

import fa_inputs
from tests import parity

pytestmark = pytest.mark.gpu

SHAPES = [
    fa_inputs.Workload("noalloc_gqa_d128", 2, 8, 2, 1024, 1024, 128, 128 ** -0.5, True,
                       do_std=0.1),
    fa_inputs.Workload("noalloc_masked_d256", 1, 4, 2, 200, 330, 256, 1.0 / 16, False,
                       masked=True),
]


@pytest.fixture(scope="module")
def lib():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import flash_attention_gb300 as fa

    fa.build()
    lib = fa.load_library()
    vp = ctypes.c_void_p
    lib.fa_train_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                         ctypes.POINTER(fa.FaParams), vp]
    lib.fa_train_bwd_noalloc.restype = ctypes.c_int
    return lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


@pytest.mark.parametrize("w", SHAPES, ids=lambda w: w.name)
def test_noalloc_backward_matches_allocating_backward(lib, w):
    import torch

    import flash_attention_gb300 as fa

    inp = fa_inputs.make_inputs(w, index=11)
    d = parity.to_device(inp)
    q, k, v, do, mask = d["q"], d["k"], d["v"], d["do"], d["mask"]
    o, lse = fa.attention_fwd(q, k, v, scale=w.scale, causal=w.causal, mask=mask)
    dq_ref, dk_ref, dv_ref = fa.attention_bwd(q, k, v, o, lse, do, scale=w.scale,
                                              causal=w.causal, mask=mask)
    torch.cuda.synchronize()
    ref = {n: t.float().cpu().numpy() for n, t in (("dq", dq_ref), ("dk", dk_ref), ("dv", dv_ref))}
    params = fa.make_params(q, k, scale=w.scale, causal=w.causal)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        dq, dk, dv = torch.full_like(q, 7.0), torch.full_like(k, 7.0), torch.full_like(v, 7.0)
        rc = lib.fa_train_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do),
                                      _ptr(mask), _ptr(dq), _ptr(dk), _ptr(dv),
                                      ctypes.byref(params), stream)
        assert rc == fa.FA_OK, fa.fa_error_string(rc)
        torch.cuda.synchronize()
        for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
            got = t.float().cpu().numpy()
            assert not np.isnan(got).any()
            bound = parity.G_REL * float(np.abs(ref[name]).max())
            err = float(np.abs(got - ref[name]).max())
            assert err <= bound, f"call {call}: {name} differs by {err:.3e} > {bound:.3e}"


def test_noalloc_refuses_a_problem_beyond_its_scratch(lib):
    import flash_attention_gb300 as fa

    # 4 * 64 * 4096 * (128 + 2) bytes of scratch > 64 MiB; nothing is dereferenced or launched
    p = fa.FaParams(2, 32, 8, 4096, 4096, 128, 0.088, 1)
    fake = ctypes.c_void_p(0x100000)
    rc = lib.fa_train_bwd_noalloc(fake, fake, fake, fake, fake, fake, None, fake, fake, fake,
                                  ctypes.byref(p), None)
    assert rc == fa.FA_ERR_TOO_LARGE

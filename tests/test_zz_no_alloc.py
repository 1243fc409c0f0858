"""The backward entry point that allocates no device memory (fa_train_bwd_noalloc).

It exists for callers that cannot let a library allocate on the GPU: a process whose device
memory belongs to a pool allocator that has already reserved it, or a step loop in which an
allocation is not allowed to block or fail. Those callers hand in every input and output, and
the library takes its scratch from a fixed array that is part of the library itself.

The test calls it through the C ABI. For each shape it first runs a call of another shape, so
that the fixed array holds that call's leftovers, then makes two calls in a row and checks
both against the CPU oracle (the gradient tolerance of the parity tests: max |difference| <=
2e-2 * max |gradient| + 1e-4) and against the ordinary allocating entry point fa_train_bwd.
It also checks that a problem too large for the fixed array is refused before anything runs.
It is self-contained, so it passes alone in a fresh process as well as after the other tests;
the file name makes pytest collect it last.
"""
import ctypes

import numpy as np
import pytest

import fa_inputs
import oracle
from tests import parity

pytestmark = pytest.mark.gpu

SHAPES = [
    fa_inputs.Workload("noalloc_gqa_d128", 2, 8, 2, 1024, 1024, 128, 128 ** -0.5, True,
                       do_std=0.1),
    fa_inputs.Workload("noalloc_masked_d256", 1, 4, 2, 200, 330, 256, 1.0 / 16, False,
                       masked=True),
]
# runs first in each case: other head dim, other row counts, so the array holds its leftovers
POISON = {
    "noalloc_gqa_d128": fa_inputs.Workload("poison_d64", 1, 4, 4, 700, 900, 64, 0.125, False,
                                           masked=True),
    "noalloc_masked_d256": fa_inputs.Workload("poison_d128", 2, 4, 1, 300, 300, 128, 0.09,
                                              True),
}


@pytest.fixture(scope="module")
def lib():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import flash_attention_gb300 as fa

    fa.build()
    oracle.build()
    lib = fa.load_library()
    vp = ctypes.c_void_p
    lib.fa_train_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                         ctypes.POINTER(fa.FaParams), vp]
    lib.fa_train_bwd_noalloc.restype = ctypes.c_int
    return lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _noalloc(lib, w, d, o, lse):
    """One fa_train_bwd_noalloc call through the C ABI; outputs start as 7.0 everywhere."""
    import torch

    import flash_attention_gb300 as fa

    q, k, v, do, mask = d["q"], d["k"], d["v"], d["do"], d["mask"]
    params = fa.make_params(q, k, scale=w.scale, causal=w.causal)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    dq, dk, dv = torch.full_like(q, 7.0), torch.full_like(k, 7.0), torch.full_like(v, 7.0)
    rc = lib.fa_train_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do),
                                  _ptr(mask), _ptr(dq), _ptr(dk), _ptr(dv),
                                  ctypes.byref(params), stream)
    assert rc == fa.FA_OK, fa.fa_error_string(rc)
    torch.cuda.synchronize()
    return {n: t.float().cpu().numpy().astype(np.float64)
            for n, t in (("dq", dq), ("dk", dk), ("dv", dv))}


def _forward(w, index):
    import flash_attention_gb300 as fa

    inp = fa_inputs.make_inputs(w, index=index)
    d = parity.to_device(inp)
    o, lse = fa.attention_fwd(d["q"], d["k"], d["v"], scale=w.scale, causal=w.causal,
                              mask=d["mask"])
    return inp, d, o, lse


@pytest.mark.parametrize("w", SHAPES, ids=lambda w: w.name)
def test_noalloc_backward_matches_oracle_and_allocating_backward(lib, w):
    import torch

    import flash_attention_gb300 as fa

    pw = POISON[w.name]
    _, pd, po, plse = _forward(pw, 12)
    _noalloc(lib, pw, pd, po, plse)  # leaves this shape's rows in the fixed array

    inp, d, o, lse = _forward(w, 11)
    dq_a, dk_a, dv_a = fa.attention_bwd(d["q"], d["k"], d["v"], o, lse, d["do"], scale=w.scale,
                                        causal=w.causal, mask=d["mask"])
    torch.cuda.synchronize()
    alloc = {n: t.float().cpu().numpy().astype(np.float64)
             for n, t in (("dq", dq_a), ("dk", dk_a), ("dv", dv_a))}
    q, k, v, do = inp.widened()
    dq_r, dk_r, dv_r = oracle.bwd(q, k, v, inp.mask, do, scale=w.scale, causal=w.causal)
    ref = {"dq": dq_r, "dk": dk_r, "dv": dv_r}
    for call in range(2):
        got = _noalloc(lib, w, d, o, lse)
        for name in ("dq", "dk", "dv"):
            parity.check_grad(got[name], ref[name], name, f"{w.name} call {call} vs oracle")
            parity.check_grad(got[name], alloc[name], name,
                              f"{w.name} call {call} vs fa_train_bwd")
    assert fa.fa_device_status(True) == fa.FA_OK


def test_noalloc_refuses_a_problem_beyond_its_scratch(lib):
    import flash_attention_gb300 as fa

    # 4 * 64 * 4096 * (128 + 2) bytes of scratch > 64 MiB - 256; nothing is dereferenced or
    # launched
    p = fa.FaParams(2, 32, 8, 4096, 4096, 128, 0.088, 1)
    fake = ctypes.c_void_p(0x100000)
    rc = lib.fa_train_bwd_noalloc(fake, fake, fake, fake, fake, fake, None, fake, fake, fake,
                                  ctypes.byref(p), None)
    assert rc == fa.FA_ERR_TOO_LARGE

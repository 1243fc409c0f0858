"""Bounded waits on the GPU, tested without breaking any kernel.

Every mbarrier wait in the kernels gives up once it has lasted the wait limit (2 s by default,
settable with fa_set_wait_limit_ns); the CTA then winds down -- copies and MMAs it started are
let finish, TMEM is freed -- and the kernel records FA_ERR_DEVICE_TIMEOUT for fa_device_status.

  * a diagnostic kernel waits on a barrier that nothing ever completes, with a 1 ms limit: the
    wait must run out after about that long, the status must say so, and the device must stay
    usable;
  * the real forward and backward run on the 4k grouped-query shape with a 1 ns limit, so that
    ordinary pipeline waits run out: the status must report the timeout, and after the default
    limit is restored the same calls must again match the CPU oracle.
Nothing here faults, traps or hangs: the waits end by themselves.
"""
import numpy as np
import pytest

import fa_inputs
import oracle
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import flash_attention_gb300 as fa

    fa.build()
    oracle.build()
    fa.fa_device_status(True)
    yield
    fa.fa_set_wait_limit_ns(0)
    assert fa.fa_device_status(True) == fa.FA_OK


def _small_parity():
    """A small call after a timeout: must match the oracle element by element."""
    w = fa_inputs.Workload("after_timeout", 1, 4, 2, 200, 260, 128, 128 ** -0.5, True,
                           do_std=0.1)
    inp = fa_inputs.make_inputs(w, index=41)
    gpu = parity.run_gpu(w, inp)
    ref = parity.oracle_full(w, inp)
    return parity.compare_full(w, gpu, ref, w.name)


def test_wait_on_a_barrier_nothing_completes_runs_out():
    import torch

    import flash_attention_gb300 as fa

    limit = 1_000_000  # 1 ms
    fa.fa_set_wait_limit_ns(limit)
    try:
        waited = fa.fa_debug_wait_timeout()
        torch.cuda.synchronize()
    finally:
        fa.fa_set_wait_limit_ns(0)
    ns = int(waited.item())
    assert limit <= ns < 1_000_000_000, f"waited {ns} ns with a limit of {limit} ns"
    assert fa.fa_device_status(True) == fa.FA_ERR_DEVICE_TIMEOUT
    assert fa.fa_device_status(True) == fa.FA_OK  # cleared
    print("after the timeout:", _small_parity())


def test_real_kernels_wind_down_when_their_waits_run_out():
    import torch

    import flash_attention_gb300 as fa

    w = fa_inputs.BY_NAME["gqa_d128_4k"]
    inp = fa_inputs.make_inputs(w)
    d = parity.to_device(inp)
    fa.fa_set_wait_limit_ns(1)
    try:
        o, lse = fa.attention_fwd(d["q"], d["k"], d["v"], scale=w.scale, causal=w.causal)
        fa.attention_bwd(d["q"], d["k"], d["v"], o, lse, d["do"], scale=w.scale,
                         causal=w.causal)
        torch.cuda.synchronize()
    finally:
        fa.fa_set_wait_limit_ns(0)
    assert fa.fa_get_wait_limit_ns() == 2_000_000_000
    assert fa.fa_device_status(True) == fa.FA_ERR_DEVICE_TIMEOUT
    assert fa.fa_device_status(True) == fa.FA_OK
    # with the default limit the same shapes run normally again
    o, lse = fa.attention_fwd(d["q"], d["k"], d["v"], scale=w.scale, causal=w.causal)
    torch.cuda.synchronize()
    assert fa.fa_device_status(True) == fa.FA_OK
    assert torch.isfinite(lse).all()
    print("after the timeout:", _small_parity())


def test_no_allocation_backward_records_its_timeouts():
    """fa_train_bwd_noalloc keeps its status word in its fixed array; a timeout there must
    reach fa_device_status as well."""
    import torch

    import flash_attention_gb300 as fa

    w = fa_inputs.Workload("noalloc_timeout", 2, 8, 2, 4096, 4096, 128, 128 ** -0.5, True,
                           do_std=0.1)
    inp = fa_inputs.make_inputs(w, index=43)
    d = parity.to_device(inp)
    o, lse = fa.attention_fwd(d["q"], d["k"], d["v"], scale=w.scale, causal=w.causal)
    dq, dk, dv = (torch.empty_like(t) for t in (d["q"], d["k"], d["v"]))
    params = fa.make_params(d["q"], d["k"], scale=w.scale, causal=w.causal)
    torch.cuda.synchronize()
    assert fa.fa_device_status(True) == fa.FA_OK
    fa.fa_set_wait_limit_ns(1)
    try:
        fa.fa_train_bwd_noalloc(d["q"], d["k"], d["v"], o, lse, d["do"], None, dq, dk, dv,
                                params)
        torch.cuda.synchronize()
    finally:
        fa.fa_set_wait_limit_ns(0)
    assert fa.fa_device_status(True) == fa.FA_ERR_DEVICE_TIMEOUT
    assert fa.fa_device_status(True) == fa.FA_OK
    fa.fa_train_bwd_noalloc(d["q"], d["k"], d["v"], o, lse, d["do"], None, dq, dk, dv, params)
    torch.cuda.synchronize()
    assert fa.fa_device_status(True) == fa.FA_OK

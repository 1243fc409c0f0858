"""A value head dim different from the q/k head dim (head_dim 128, value_dim 64) on the GPU,
against the CPU oracle: O and dV have 64 columns, dQ and dK 128. Covers causal, rectangular,
GQA, a window, a mask and sinks. Tolerances as in tests/parity.py."""
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
    assert fa.fa_device_status(True) == fa.FA_OK


def W(name, B, H, Hk, ql, kl, causal, masked=False, wl=-1, wr=-1):
    return fa_inputs.Workload(name, B, H, Hk, ql, kl, 128, 128 ** -0.5, causal, masked,
                              window_left=wl, window_right=wr, value_dim=64)


CASES = [
    W("dv64_causal", 1, 4, 2, 256, 256, True),
    W("dv64_rect_ragged", 2, 4, 1, 77, 300, True),
    W("dv64_noncausal_masked", 1, 2, 2, 130, 190, False, masked=True),
    W("dv64_window", 1, 4, 4, 300, 300, True, wl=70),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_value_dim_elementwise(w):
    inp = fa_inputs.make_inputs(w, index=60 + CASES.index(w))
    gpu = parity.run_gpu(w, inp)
    assert gpu["o"].shape[-1] == 64 and gpu["dv"].shape[-1] == 64 and gpu["dq"].shape[-1] == 128
    ref = parity.oracle_full(w, inp)
    stats = parity.compare_full(w, gpu, ref, w.name)
    print(w.name, stats)


def test_value_dim_with_sinks():
    import torch

    import flash_attention_gb300 as fa

    w = W("dv64_sinks", 1, 4, 2, 200, 260, True)
    inp = fa_inputs.make_inputs(w, index=70)
    sinks = np.array([0.5, -1.0, 2.0, 0.0], np.float32)
    dev = parity.to_device(inp)
    s_t = torch.from_numpy(sinks).cuda()
    o, lse = fa.attention_fwd(dev["q"], dev["k"], dev["v"], scale=w.scale, causal=True,
                              sinks=s_t)
    dq, dk, dv, ds = fa.attention_bwd(dev["q"], dev["k"], dev["v"], o, lse, dev["do"],
                                      scale=w.scale, causal=True, sinks=s_t)
    torch.cuda.synchronize()
    assert fa.fa_device_status(True) == fa.FA_OK
    gpu = {n: t.float().cpu().numpy().astype(np.float64)
           for n, t in (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv))}
    q, k, v, do = inp.widened()
    with oracle.sinks(sinks):
        o_r, l_r = oracle.fwd(q, k, v, None, scale=w.scale, causal=True)
        dq_r, dk_r, dv_r = oracle.bwd(q, k, v, None, do, scale=w.scale, causal=True)
        ds_r = oracle.dsinks(q, k, v, None, do, scale=w.scale, causal=True)
    parity.compare_full(w, gpu, {"o": o_r, "lse": l_r, "dq": dq_r, "dk": dk_r, "dv": dv_r},
                        w.name)
    parity.check_grad(ds.cpu().numpy(), ds_r, "dsinks", w.name)

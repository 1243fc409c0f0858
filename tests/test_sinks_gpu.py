"""Attention sinks on the GPU against the CPU oracle: O, L, dQ, dK, dV and the sink gradient,
with causal / window / mask combinations, rows that see no key (O = 0, L = sink) and a sink of
-inf next to finite ones. Tolerances as in tests/parity.py (dsinks is held to the gradient
rule)."""
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


CASES = [
    # (B, H, Hk, ql, kl, d, causal, window, mask kind)
    (1, 4, 2, 200, 200, 64, True, None, None),
    (2, 4, 1, 130, 260, 128, False, None, "bool"),
    (1, 2, 2, 150, 330, 256, True, None, None),
    (1, 4, 4, 300, 120, 128, True, None, None),          # ql > kl: 180 rows see no key
    (1, 4, 2, 257, 257, 128, True, (60, -1), None),      # sliding window
    (2, 2, 1, 96, 160, 64, False, (30, 10), "additive"),
]


def _mask(kind, shape, rng):
    import torch

    if kind is None:
        return None, None
    if kind == "bool":
        m = rng.random(shape) > 0.2
        m[:, :, 3, :] = False  # a row hidden by the mask alone
        return m, torch.bool
    m = rng.uniform(-2.0, 0.5, size=shape).astype(np.float32)
    m[rng.random(shape) < 0.1] = -np.inf
    m[:, :, 5, :] = -np.inf
    return m, torch.float32


def _ids(c):
    w = "none" if c[7] is None else f"{c[7][0]}_{c[7][1]}"
    return f"d{c[5]}_q{c[3]}_k{c[4]}_causal{int(c[6])}_win{w}_mask_{c[8]}"


@pytest.mark.parametrize("idx", range(len(CASES)), ids=[_ids(c) for c in CASES])
def test_sinks_fwd_bwd(idx):
    import torch

    import flash_attention_gb300 as fa

    B, H, Hk, ql, kl, d, causal, window, mkind = CASES[idx]
    w = fa_inputs.Workload("sinks", B, H, Hk, ql, kl, d, d ** -0.5, causal)
    inp = fa_inputs.make_inputs(w, index=40 + idx)
    rng = np.random.default_rng(4000 + idx)
    sinks = fa_inputs.bf16_bits_to_f32(fa_inputs.f32_to_bf16_bits(
        (1.5 * rng.standard_normal(H) + 1.0).astype(np.float32)))
    sinks[-1] = -np.inf  # the last head has no sink
    m_np, m_dtype = _mask(mkind, (B, H, ql, kl), rng)
    dev = parity.to_device(inp)
    m_t = None if m_np is None else torch.from_numpy(m_np).to(m_dtype).cuda()
    s_t = torch.from_numpy(sinks).cuda()
    o, lse = fa.attention_fwd(dev["q"], dev["k"], dev["v"], scale=w.scale, causal=causal,
                              mask=m_t, window=window, sinks=s_t)
    dq, dk, dv, ds = fa.attention_bwd(dev["q"], dev["k"], dev["v"], o, lse, dev["do"],
                                      scale=w.scale, causal=causal, mask=m_t, window=window,
                                      sinks=s_t)
    # dsinks is summed in a fixed order: a second backward gives the same bits
    _, _, _, ds2 = fa.attention_bwd(dev["q"], dev["k"], dev["v"], o, lse, dev["do"],
                                    scale=w.scale, causal=causal, mask=m_t, window=window,
                                    sinks=s_t)
    torch.cuda.synchronize()
    assert fa.fa_device_status(True) == fa.FA_OK
    assert torch.equal(ds, ds2)
    gpu = {n: t.float().cpu().numpy().astype(np.float64)
           for n, t in (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv))}
    q, k, v, do = inp.widened()
    dm = oracle.dense_mask(m_np, (B, H, ql, kl))
    with oracle.window(*(window or (-1, -1))), oracle.sinks(sinks):
        o_r, l_r = oracle.fwd(q, k, v, dm, scale=w.scale, causal=causal)
        dq_r, dk_r, dv_r = oracle.bwd(q, k, v, dm, do, scale=w.scale, causal=causal)
        ds_r = oracle.dsinks(q, k, v, dm, do, scale=w.scale, causal=causal)
    ref = {"o": o_r, "lse": l_r, "dq": dq_r, "dk": dk_r, "dv": dv_r}
    stats = parity.compare_full(w, gpu, ref, _ids(CASES[idx]))
    stats.update(parity.check_grad(ds.cpu().numpy(), ds_r, "dsinks", _ids(CASES[idx])))
    # rows that see no key: O = 0 exactly, L = the head's sink (-inf for the sinkless head)
    dead = ~np.isfinite(l_r) | np.isclose(l_r, sinks[None, :, None].astype(np.float64) *
                                          np.ones_like(l_r), rtol=0, atol=0)
    if dead.any():
        assert (gpu["o"][dead] == 0).all()
    print(_ids(CASES[idx]), stats)


def test_sink_above_the_scores_keeps_single_key_rows_accurate():
    """Sinks larger than every score. Causal row 0 sees one key, so O_0 = w * v_0 with
    w = 1 / (1 + exp(sink - s_00)): the weight must be formed in f32, not by rounding the key's
    P to bf16 relative to the sink (an error of up to 2^-9 |O|). Row 0 is held to half a bf16
    ulp of the output plus 2e-4 relative; all rows to the usual O and L tolerances."""
    import torch

    import flash_attention_gb300 as fa

    w = fa_inputs.Workload("sink_high", 1, 4, 2, 256, 256, 128, 128 ** -0.5, True)
    inp = fa_inputs.make_inputs(w, index=50)
    sinks = np.array([3.0, 5.0, 8.0, 2.5], np.float32)
    dev = parity.to_device(inp)
    s_t = torch.from_numpy(sinks).cuda()
    o, lse = fa.attention_fwd(dev["q"], dev["k"], dev["v"], scale=w.scale, causal=True,
                              sinks=s_t)
    torch.cuda.synchronize()
    assert fa.fa_device_status(True) == fa.FA_OK
    q, k, v, _ = inp.widened()
    with oracle.sinks(sinks):
        o_r, l_r = oracle.fwd(q, k, v, None, scale=w.scale, causal=True)
    o_g = o.float().cpu().numpy().astype(np.float64)
    parity.check_o(o_g, o_r, "sink_high")
    parity.check_l(lse.float().cpu().numpy(), l_r, "sink_high")
    row0_err = np.abs(o_g[:, :, 0] - o_r[:, :, 0])
    bound = 0.5 * parity.bf16_ulp(o_r[:, :, 0]) + 2e-4 * np.maximum(1.0, np.abs(o_r[:, :, 0]))
    assert (row0_err <= bound).all(), f"single-key row: max error {row0_err.max():.3e}"

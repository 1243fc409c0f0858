"""Memory layouts on the GPU: q, o, dO, dQ and/or k, v, dK, dV given as transposed views of
[batch, seq, heads, dim] tensors ([total, heads, dim] for packed sequences). The page
"nuvec-core tests/fast.rs", `attention_kernels_match_the_fallback`, passes K and V as
transposed views.

Each case is compared with the CPU oracle at the parity tolerances of tests/parity.py. O, L, dK
and dV must also equal, bit for bit, the same call on contiguous tensors: the kernels do the
same arithmetic in the same order, and only the addresses differ. dQ is held to the tolerance
only, because its f32 accumulation order across CTAs is not fixed. In the deterministic mode it
is held to bit equality too.
"""
import numpy as np
import pytest

import fa_inputs
import oracle
from tests import parity

pytestmark = pytest.mark.gpu

Q_SIDE, KV_SIDE = 1, 2


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import flash_attention_gb300 as fa

    fa.build()
    fa.load_library()
    oracle.build()
    fa.fa_device_status(True)
    yield
    assert fa.fa_device_status(True) == fa.FA_OK


def W(name, B, H, Hk, ql, kl, d, causal, **kw):
    return fa_inputs.Workload(name, B, H, Hk, ql, kl, d, d ** -0.5, causal, **kw)


CASES = [
    (W("d64_q_side", 2, 4, 2, 200, 300, 64, True), Q_SIDE),
    (W("d128_kv_side_gqa", 2, 8, 2, 333, 257, 128, True), KV_SIDE),
    (W("d128_both_window", 1, 8, 2, 300, 300, 128, True, window_left=70), Q_SIDE | KV_SIDE),
    (W("d256_both_pairs", 1, 4, 2, 190, 330, 256, True), Q_SIDE | KV_SIDE),
    (W("d256_kv_side_masked", 1, 4, 1, 64, 192, 256, False, masked=True), KV_SIDE),
    (W("d128_dv64_both", 1, 4, 2, 140, 200, 128, True, value_dim=64), Q_SIDE | KV_SIDE),
    (W("d128_both_deterministic", 2, 4, 2, 150, 260, 128, True, deterministic=True),
     Q_SIDE | KV_SIDE),
    (W("d64_both_sinks", 1, 4, 4, 129, 129, 64, True, sinks=True), Q_SIDE | KV_SIDE),
]


def _bshd(t):
    """The same logical [B, H, L, D] tensor, stored as [B, L, H, D]."""
    return t.transpose(1, 2).contiguous().transpose(1, 2)


def _run(w, d, layout):
    import torch

    import flash_attention_gb300 as fa

    q, do = d["q"], d["do"]
    k, v = d["k"], d["v"]
    if layout & Q_SIDE:
        q, do = _bshd(q), _bshd(do)
    if layout & KV_SIDE:
        k, v = _bshd(k), _bshd(v)
    win = (w.window_left, w.window_right) if w.windowed else None
    o, lse = fa.attention_fwd(q, k, v, scale=w.scale, causal=w.causal, mask=d["mask"],
                              window=win, sinks=d["sinks"])
    g = fa.attention_bwd(q, k, v, o, lse, do, scale=w.scale, causal=w.causal, mask=d["mask"],
                         window=win, sinks=d["sinks"], deterministic=w.deterministic)
    torch.cuda.synchronize()
    assert fa.fa_device_status(True) == fa.FA_OK
    out = {"o": o, "lse": lse, "dq": g[0], "dk": g[1], "dv": g[2]}
    if d["sinks"] is not None:
        out["dsinks"] = g[3]
    # outputs come back in the layout of their inputs
    for name, like in (("o", q), ("dq", q), ("dk", k), ("dv", v)):
        assert out[name].is_contiguous() == like.is_contiguous(), name
    return out


@pytest.mark.parametrize("case", CASES, ids=[c[0].name for c in CASES])
def test_layout_matches_oracle_and_contiguous_call(case):
    import torch

    w, layout = case
    inp = fa_inputs.make_inputs(w, index=61)
    d = parity.to_device(inp)
    got = _run(w, d, layout)
    base = _run(w, d, 0)
    exact = ["o", "lse", "dk", "dv"] + (["dq"] if w.deterministic else []) + \
        (["dsinks"] if w.sinks else [])
    for name in exact:
        assert torch.equal(got[name], base[name]), f"{name} differs from the contiguous call"
    ref = parity.oracle_full(w, inp)
    gpu = {n: t.float().cpu().numpy().astype(np.float64) for n, t in got.items()}
    stats = parity.compare_full(w, gpu, ref, f"{w.name} layout {layout}")
    print(w.name, layout, stats)


def test_packed_sequences_in_token_major_layout():
    """A variable-length batch with q, k, v, dO as [total, heads, dim] tensors."""
    import torch

    import flash_attention_gb300 as fa

    w = fa_inputs.VarlenWorkload("tok_major", 8, 2, 128, (300, 17, 129, 640), (300, 40, 129, 700))
    x = fa_inputs.make_varlen_inputs(w, index=171)

    def bf(bits, token_major):
        t = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).cuda()
        return t.transpose(0, 1).contiguous().transpose(0, 1) if token_major else t

    cq, ck = torch.from_numpy(x.cu_q).cuda(), torch.from_numpy(x.cu_k).cuda()
    mq, mk = max(w.q_lens), max(w.k_lens)
    res = {}
    for tm in (True, False):
        q, k, v, do = (bf(t, tm) for t in (x.q, x.k, x.v, x.do))
        o, lse = fa.varlen_attention_fwd(q, k, v, cq, ck, mq, mk, scale=w.scale, causal=w.causal)
        dq, dk, dv = fa.varlen_attention_bwd(q, k, v, o, lse, do, cq, ck, mq, mk, scale=w.scale,
                                             causal=w.causal)
        torch.cuda.synchronize()
        assert fa.fa_device_status(True) == fa.FA_OK
        assert o.is_contiguous() != tm and dq.is_contiguous() != tm
        res[tm] = {"o": o, "lse": lse, "dq": dq, "dk": dk, "dv": dv}
    for name in ("o", "lse", "dk", "dv"):
        assert torch.equal(res[True][name], res[False][name]), name
    q64, k64, v64, do64 = x.widened()
    o_r, l_r = oracle.varlen_fwd(q64, k64, v64, x.cu_q, x.cu_k, scale=w.scale, causal=w.causal)
    dq_r, dk_r, dv_r = oracle.varlen_bwd(q64, k64, v64, do64, x.cu_q, x.cu_k, scale=w.scale,
                                         causal=w.causal)
    ref = {"o": o_r, "lse": l_r, "dq": dq_r, "dk": dk_r, "dv": dv_r}
    gpu = {n: t.float().cpu().numpy().astype(np.float64) for n, t in res[True].items()}
    print(w.name, parity.compare_full(w, gpu, ref, w.name))

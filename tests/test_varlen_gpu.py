"""Variable-length batches on the GPU: packed sequences (q [H, total_q, d], k, v
[Hk, total_k, d]) against the oracle's per-sequence composition, forward and backward, for head
dims 64 / 128 / 256 and value_dim 64, GQA, an empty query sequence, sequences with no keys,
ql > kl, windows, sinks and the deterministic mode. Tolerances as in tests/parity.py."""
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
    fa.fa_device_status(True)


def V(name, H, Hk, d, ql, kl, causal=True, wl=-1, wr=-1):
    return fa_inputs.VarlenWorkload(name, H, Hk, d, tuple(ql), tuple(kl), causal, wl, wr)


CASES = [
    (V("d128_gqa_ragged", 8, 2, 128, [300, 17, 129, 640], [300, 40, 129, 700]), {}),
    (V("d64_noncausal", 4, 4, 64, [100, 0, 257], [64, 90, 300], causal=False), {}),
    (V("d256_causal", 4, 2, 256, [190, 65], [190, 330]), {}),
    (V("no_keys_and_short_keys", 4, 1, 128, [50, 200, 33], [0, 120, 33]), {}),
    (V("window", 4, 2, 128, [400, 150], [400, 300], wl=70), {}),
    (V("sinks", 4, 2, 128, [130, 0, 260], [200, 10, 100]), {"sinks": True}),
    (V("deterministic", 4, 2, 128, [300, 77], [300, 500]), {"deterministic": True}),
    (V("dv64", 4, 2, 128, [140, 300], [140, 310]), {"dv": 64}),
]


def run(w, x, sinks=None, deterministic=False, dv=None):
    import torch

    import flash_attention_gb300 as fa

    def bf(bits):
        return torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).cuda()

    q, k, v, do = bf(x.q), bf(x.k), bf(x.v), bf(x.do)
    cq, ck = torch.from_numpy(x.cu_q).cuda(), torch.from_numpy(x.cu_k).cuda()
    win = (w.window_left, w.window_right) if w.windowed else None
    s_t = None if sinks is None else torch.from_numpy(sinks).cuda()
    mq, mk = max(max(w.q_lens), 1), max(max(w.k_lens), 1)
    o, lse = fa.varlen_attention_fwd(q, k, v, cq, ck, mq, mk, scale=w.scale, causal=w.causal,
                                     window=win, sinks=s_t)
    g = fa.varlen_attention_bwd(q, k, v, o, lse, do, cq, ck, mq, mk, scale=w.scale,
                                causal=w.causal, window=win, sinks=s_t,
                                deterministic=deterministic)
    torch.cuda.synchronize()
    assert fa.fa_device_status(True) == fa.FA_OK
    out = {"o": o, "lse": lse, "dq": g[0], "dk": g[1], "dv": g[2]}
    if sinks is not None:
        out["dsinks"] = g[3]
    return {n: t.float().cpu().numpy().astype(np.float64) for n, t in out.items()}, g


def reference(w, x, sinks=None):
    q, k, v, do = x.widened()
    with oracle.window(w.window_left, w.window_right), oracle.sinks(sinks):
        o, lse = oracle.varlen_fwd(q, k, v, x.cu_q, x.cu_k, scale=w.scale, causal=w.causal)
        dq, dk, dv = oracle.varlen_bwd(q, k, v, do, x.cu_q, x.cu_k, scale=w.scale,
                                       causal=w.causal)
        ref = {"o": o, "lse": lse, "dq": dq, "dk": dk, "dv": dv}
        if sinks is not None:
            ds = np.zeros(w.n_heads)
            for b in range(w.batch):
                qs, qe, ks, ke = x.cu_q[b], x.cu_q[b + 1], x.cu_k[b], x.cu_k[b + 1]
                if qe > qs and ke > ks:
                    ds += oracle.dsinks(q[None, :, qs:qe], k[None, :, ks:ke], v[None, :, ks:ke],
                                        None, do[None, :, qs:qe], scale=w.scale, causal=w.causal)
                elif qe > qs:  # no keys: L = sink, P_sink = 1, D = dO . 0 = 0
                    pass
            ref["dsinks"] = ds
    return ref


@pytest.mark.parametrize("idx", range(len(CASES)), ids=[c[0].name for c in CASES])
def test_varlen_matches_oracle(idx):
    import torch

    w, extra = CASES[idx]
    x = fa_inputs.make_varlen_inputs(w, index=150 + idx)
    if extra.get("dv"):
        dvd = extra["dv"]
        rng_v = fa_inputs.normal_bf16(777 + idx, (w.n_kv_heads, x.k.shape[1], dvd))
        rng_do = fa_inputs.normal_bf16(778 + idx, (w.n_heads, x.q.shape[1], dvd))
        x = fa_inputs.VarlenInputs(x.q, x.k, rng_v, rng_do, x.cu_q, x.cu_k)
    sinks = np.array([0.5, -1.0, 2.0, 1.0], np.float32) if extra.get("sinks") else None
    gpu, g1 = run(w, x, sinks, extra.get("deterministic", False))
    if extra.get("deterministic"):
        _, g2 = run(w, x, sinks, True)
        for a, b in zip(g1, g2):
            assert torch.equal(a, b)
    ref = reference(w, x, sinks)
    stats = parity.compare_full(w, gpu, ref, w.name)
    print(w.name, stats)

"""Helpers of the GPU parity tests: run the CUDA path through the C ABI and compare it with the
CPU oracle on the same seeded bf16 inputs.

Tolerances (written here, used by every parity test):
  * L:  |L_gpu - L_ref| <= 3e-3 (absolute), and L_gpu = -inf exactly where L_ref = -inf;
  * O:  |O_gpu - O_ref| <= 5e-3 + ulp_bf16(O_ref) / 2. The 5e-3 is the stated tolerance of the
        f32 result; O is stored in bf16, whose round-to-nearest adds at most half an ulp of the
        value (7.8e-3 already at |O| in [2, 4)), so that half ulp is added on top. The strict
        mlx-native rule (|O_gpu - bf16(O_ref)| <= 5e-3) is also evaluated and the number of
        elements that miss it by one bf16 ulp is reported, not hidden;
  * dQ, dK, dV: max |g_gpu - g_ref| <= 2e-2 * max |g_ref| + 1e-4 per tensor. The absolute
        1e-4 only matters where a gradient vanishes in exact arithmetic: a row whose only
        visible key is its own (window 0) has P = 1, O = V and dS = dP - D = 0, so the oracle's
        dQ is exactly 0 while the kernel's dP and D, two f32 dot products of length d, leave a
        cancellation residue of order d * 2^-24 * |dO| |V| (about 1e-6 at d = 64).
References are the oracle's unrounded f64 values.
"""
from __future__ import annotations

import numpy as np

import fa_inputs
import oracle

O_ATOL = 5e-3
L_ATOL = 3e-3
G_REL = 2e-2
G_ABS = 1e-4


def bf16_ulp(x):
    """Spacing of bf16 numbers at |x| (8 significant bits)."""
    ax = np.maximum(np.abs(np.asarray(x, np.float64)), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(ax)) - 7)


def round_bf16(x):
    return fa_inputs.bf16_bits_to_f32(fa_inputs.f32_to_bf16_bits(np.asarray(x, np.float32)))


def check_o(o_gpu, o_ref, label=""):
    """Returns a dict of statistics; raises AssertionError on a tolerance miss."""
    o_gpu = np.asarray(o_gpu, np.float64)
    o_ref = np.asarray(o_ref, np.float64)
    assert not np.isnan(o_gpu).any(), f"{label}: NaN in O"
    err = np.abs(o_gpu - o_ref)
    tol = O_ATOL + 0.5 * bf16_ulp(o_ref)
    bad = err > tol
    o_ref_bf = round_bf16(o_ref)
    strict = np.abs(o_gpu - o_ref_bf) > O_ATOL
    stats = {"o_max_err": float(err.max(initial=0.0)),
             "o_strict_misses": int(strict.sum()),
             "o_elements": int(o_ref.size)}
    if bad.any():
        i = np.unravel_index(np.argmax(np.where(bad, err - tol, -1)), err.shape)
        raise AssertionError(f"{label}: O error {err[i]:.3e} > {tol[i]:.3e} at {i} "
                             f"(gpu {o_gpu[i]!r}, ref {o_ref[i]!r}); {int(bad.sum())} bad")
    if strict.any():
        # every miss of the strict rule must be the neighbouring bf16 value of bf16(O_ref): a
        # rounding flip of a correct f32 result, nothing larger
        gb = fa_inputs.f32_to_bf16_bits(o_gpu[strict].astype(np.float32)).astype(np.int64)
        rb = fa_inputs.f32_to_bf16_bits(o_ref_bf[strict].astype(np.float32)).astype(np.int64)
        dist = np.abs(gb - rb)
        assert (dist == 1).all(), (f"{label}: {int((dist != 1).sum())} strict-rule misses are "
                                   f"not one bf16 ulp (largest distance {int(dist.max())} ulps)")
    return stats


def check_l(l_gpu, l_ref, label=""):
    l_gpu = np.asarray(l_gpu, np.float64)
    l_ref = np.asarray(l_ref, np.float64)
    assert not np.isnan(l_gpu).any(), f"{label}: NaN in L"
    ninf = np.isneginf(l_ref)
    assert np.array_equal(np.isneginf(l_gpu), ninf), f"{label}: -inf pattern of L differs"
    err = np.abs(np.where(ninf, 0.0, l_gpu - np.where(ninf, 0.0, l_ref)))
    mx = float(err.max(initial=0.0))
    assert mx <= L_ATOL, f"{label}: L max error {mx:.3e} > {L_ATOL}"
    return {"l_max_err": mx}


def check_grad(g_gpu, g_ref, name, label="", scale_ref=None):
    g_gpu = np.asarray(g_gpu, np.float64)
    g_ref = np.asarray(g_ref, np.float64)
    assert not np.isnan(g_gpu).any(), f"{label}: NaN in {name}"
    gmax = float(np.abs(g_ref).max(initial=0.0)) if scale_ref is None else scale_ref
    err = float(np.abs(g_gpu - g_ref).max(initial=0.0))
    bound = G_REL * gmax + G_ABS
    assert err <= bound, (
        f"{label}: {name} max error {err:.3e} > {G_REL} * max|{name}| + {G_ABS} = {bound:.3e}")
    return {f"{name}_max_err": err, f"{name}_max_abs": gmax}


# ---------------------------------------------------------------- running the CUDA path
def to_device(inp: fa_inputs.Inputs):
    import torch

    def bf(bits):
        return torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).cuda()

    dev = {"q": bf(inp.q), "k": bf(inp.k), "v": bf(inp.v), "do": bf(inp.do)}
    dev["mask"] = None if inp.mask is None else torch.from_numpy(inp.mask).cuda()
    dev["sinks"] = None if inp.sinks is None else torch.from_numpy(inp.sinks).cuda()
    return dev


def run_gpu(w: fa_inputs.Workload, inp: fa_inputs.Inputs, bwd=True):
    """fwd (+ bwd) on the GPU through the C ABI. Returns numpy f64 arrays."""
    import torch

    import flash_attention_gb300 as fa

    d = to_device(inp)
    win = (w.window_left, w.window_right) if w.windowed else None
    o, lse = fa.attention_fwd(d["q"], d["k"], d["v"], scale=w.scale, causal=w.causal,
                              mask=d["mask"], window=win, sinks=d["sinks"])
    out = {"o": o, "lse": lse}
    if bwd:
        g = fa.attention_bwd(d["q"], d["k"], d["v"], o, lse, d["do"], scale=w.scale,
                             causal=w.causal, mask=d["mask"], window=win, sinks=d["sinks"])
        out.update(dq=g[0], dk=g[1], dv=g[2])
        if d["sinks"] is not None:
            out["dsinks"] = g[3]
    torch.cuda.synchronize()
    assert fa.fa_device_status(True) == fa.FA_OK, "a kernel gave up a bounded wait"
    return {k: v.float().cpu().numpy().astype(np.float64) for k, v in out.items()}


def oracle_full(w: fa_inputs.Workload, inp: fa_inputs.Inputs, bwd=True):
    q, k, v, do = inp.widened()
    with oracle.window(w.window_left, w.window_right), oracle.sinks(inp.sinks):
        o, lse = oracle.fwd(q, k, v, inp.mask, scale=w.scale, causal=w.causal)
        res = {"o": o, "lse": lse}
        if bwd:
            dq, dk, dv = oracle.bwd(q, k, v, inp.mask, do, scale=w.scale, causal=w.causal)
            res.update(dq=dq, dk=dk, dv=dv)
            if inp.sinks is not None:
                res["dsinks"] = oracle.dsinks(q, k, v, inp.mask, do, scale=w.scale,
                                              causal=w.causal)
    return res


def compare_full(w, gpu, ref, label):
    stats = {}
    stats.update(check_o(gpu["o"], ref["o"], label))
    stats.update(check_l(gpu["lse"], ref["lse"], label))
    if "dq" in gpu:
        for n in ("dq", "dk", "dv"):
            stats.update(check_grad(gpu[n], ref[n], n, label))
    if "dsinks" in gpu:
        stats.update(check_grad(gpu["dsinks"], ref["dsinks"], "dsinks", label))
    return stats

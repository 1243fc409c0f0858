"""Pins of the CPU oracle: checks against things other than the oracle itself.

Each `pin_*` function returns a list of failure strings (empty = pass). They are called by
`test_oracle_pins.py` one by one, and all together by the planted-mistake test, which shows
that each mistake planted in the oracle fails at least one of them.

Sources of truth used here (none of them is the oracle's own formula retyped):
  * torch's CPU library kernels in f64: `_scaled_dot_product_flash_attention_for_cpu`
    (O and logsumexp) and autograd through `scaled_dot_product_attention` (dQ, dK, dV), with
    bottom-right causal taken from torch's own `causal_lower_right` bias;
  * f64 central finite differences (with Richardson extrapolation) of the oracle's forward;
  * closed forms and invariants of softmax attention (constant V, a single visible key, Q = 0,
    mask shifts, rows of P summing to one, zero column sums of dK, ...);
  * structural facts from the mlx-native training tests (page "mlx-native
    tests/test_flash_attn_train.rs": the causal sentinel-K test of section 6 and the GQA
    accumulation test of section 16) and the nuvec-core direct formula (page "nuvec-core
    tests/fast.rs", `attention_fallback_matches_a_direct_formula`: bottom-right causal).
"""
from __future__ import annotations

import numpy as np
import torch
import torch.nn.functional as F
from torch.nn.attention.bias import causal_lower_right

import oracle

TOL = 1e-10


def _rand(rng, shape, lo=None):
    return rng.standard_normal(shape).astype(np.float32)


def _bf16_exact(x):
    # values with at most 8 significant bits, like the bf16 inputs the oracle always receives
    from fa_inputs import bf16_bits_to_f32, f32_to_bf16_bits

    return bf16_bits_to_f32(f32_to_bf16_bits(x))


def _problem(seed, B, H, Hk, ql, kl, d, mask=False, neg_inf_frac=0.0):
    rng = np.random.default_rng(seed)
    q = _bf16_exact(_rand(rng, (B, H, ql, d)))
    k = _bf16_exact(_rand(rng, (B, Hk, kl, d)))
    v = _bf16_exact(_rand(rng, (B, Hk, kl, d)))
    do = _bf16_exact(_rand(rng, (B, H, ql, d)))
    m = None
    if mask:
        m = rng.uniform(-2, 0, size=(B, H, ql, kl)).astype(np.float32)
        if neg_inf_frac:
            m[rng.random(m.shape) < neg_inf_frac] = -np.inf
    return q, k, v, do, m


def _torch_bias(ql, kl, causal, mask, H, B, window=None):
    """Additive f64 bias [B,H,ql,kl] from torch's own lower-right causal bias, a local window
    band built with torch.tril / torch.triu around the same diagonal, and the mask."""
    bias = torch.zeros(B, H, ql, kl, dtype=torch.float64)
    if causal:
        allowed = causal_lower_right(ql, kl)._materialize(device="cpu")
        bias = bias.masked_fill(~allowed, float("-inf"))
    if window is not None:
        wl, wr = window
        band = torch.ones(ql, kl, dtype=torch.bool)
        off = kl - ql
        if wr >= 0:
            band = band.tril(diagonal=off + wr)
        if wl >= 0:
            band = band.triu(diagonal=off - wl)
        bias = bias.masked_fill(~band, float("-inf"))
    if mask is not None:
        bias = bias + torch.from_numpy(mask).double()
    return bias


def _torch_fwd(q, k, v, mask, scale, causal, window=None):
    B, H, ql, d = q.shape
    G = H // k.shape[1]
    kt = torch.from_numpy(k).double().repeat_interleave(G, dim=1)
    vt = torch.from_numpy(v).double().repeat_interleave(G, dim=1)
    qt = torch.from_numpy(q).double()
    bias = _torch_bias(ql, k.shape[2], causal, mask, H, B, window)
    o, lse = torch.ops.aten._scaled_dot_product_flash_attention_for_cpu(
        qt, kt, vt, 0.0, False, attn_mask=bias, scale=scale)
    return o.numpy(), lse.numpy()


def _torch_grads(q, k, v, mask, do, scale, causal, window=None):
    B, H, ql, d = q.shape
    qt = torch.from_numpy(q).double().requires_grad_()
    kt = torch.from_numpy(k).double().requires_grad_()
    vt = torch.from_numpy(v).double().requires_grad_()
    if causal and mask is None and window is None:
        bias = causal_lower_right(ql, k.shape[2])
    else:
        bias = _torch_bias(ql, k.shape[2], causal, mask, H, B, window)
    with torch.nn.attention.sdpa_kernel(torch.nn.attention.SDPBackend.MATH):
        o = F.scaled_dot_product_attention(qt, kt, vt, attn_mask=bias, scale=scale,
                                           enable_gqa=True)
    (o * torch.from_numpy(do).double()).sum().backward()
    return qt.grad.numpy(), kt.grad.numpy(), vt.grad.numpy()


def _cmp(name, got, want, tol=TOL, out=None):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    if got.shape != want.shape:
        out.append(f"{name}: shape {got.shape} vs {want.shape}")
        return
    same_inf = np.isinf(want) & (got == want)
    with np.errstate(invalid="ignore"):
        err = np.where(same_inf, 0.0, np.abs(got - want))
    scale = np.maximum(1.0, np.where(np.isfinite(want), np.abs(want), 1.0))
    bad = ~(err <= tol * scale)
    if bad.any():
        idx = np.unravel_index(np.argmax(np.where(bad, err, -1)), err.shape)
        out.append(f"{name}: {int(bad.sum())} bad, worst at {idx}: got {got[idx]!r} want {want[idx]!r}")


# Shapes for the library pins: (B, H, Hk, ql, kl, d, causal, mask)
LIB_CASES = [
    (1, 1, 1, 5, 7, 4, False, False),
    (2, 4, 2, 6, 6, 8, True, False),
    (1, 2, 1, 3, 9, 4, True, False),     # bottom-right rectangle, kl > ql
    (1, 2, 2, 4, 5, 8, False, True),     # additive mask
    (1, 4, 1, 5, 8, 4, True, True),      # causal + mask + GQA 4:1
]


def pin_fwd_vs_torch_cpu_flash():
    fails = []
    for n, (B, H, Hk, ql, kl, d, causal, mask) in enumerate(LIB_CASES):
        q, k, v, do, m = _problem(100 + n, B, H, Hk, ql, kl, d, mask)
        scale = 0.37
        o, lse = oracle.fwd(q, k, v, m, scale=scale, causal=causal)
        to, tl = _torch_fwd(q, k, v, m, scale, causal)
        _cmp(f"case{n} O", o, to, out=fails)
        _cmp(f"case{n} L", lse, tl, out=fails)
    return fails


def pin_bwd_vs_torch_autograd():
    fails = []
    for n, (B, H, Hk, ql, kl, d, causal, mask) in enumerate(LIB_CASES):
        q, k, v, do, m = _problem(200 + n, B, H, Hk, ql, kl, d, mask)
        scale = 0.41
        dq, dk, dv = oracle.bwd(q, k, v, m, do, scale=scale, causal=causal)
        tq, tk, tv = _torch_grads(q, k, v, m, do, scale, causal)
        _cmp(f"case{n} dQ", dq, tq, out=fails)
        _cmp(f"case{n} dK", dk, tk, out=fails)
        _cmp(f"case{n} dV", dv, tv, out=fails)
    return fails


def pin_bwd_vs_finite_differences():
    """loss = sum(O * dO); Richardson-extrapolated central differences with steps 2^-8, 2^-9,
    which are exact in f32 for bf16-valued inputs of magnitude < 8."""
    fails = []
    B, H, Hk, ql, kl, d = 1, 2, 1, 3, 5, 4
    q, k, v, do, m = _problem(300, B, H, Hk, ql, kl, d, mask=True, neg_inf_frac=0.15)
    scale, causal = 0.6, True
    dq, dk, dv = oracle.bwd(q, k, v, m, do, scale=scale, causal=causal)

    def loss(qq, kk, vv):
        o, _ = oracle.fwd(qq, kk, vv, m, scale=scale, causal=causal, nthreads=1)
        return float((o * do.astype(np.float64)).sum())

    for name, arr, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros(arr.shape)
        for idx in np.ndindex(arr.shape):
            ests = []
            for h in (2.0 ** -8, 2.0 ** -9):
                plus, minus = arr.copy(), arr.copy()
                plus[idx] += np.float32(h)
                minus[idx] -= np.float32(h)
                args_p = {"q": (plus, k, v), "k": (q, plus, v), "v": (q, k, plus)}[name]
                args_m = {"q": (minus, k, v), "k": (q, minus, v), "v": (q, k, minus)}[name]
                ests.append((loss(*args_p) - loss(*args_m)) / (2 * h))
            num[idx] = (4 * ests[1] - ests[0]) / 3
        _cmp(f"FD d{name}", grad, num, tol=2e-7, out=fails)
    return fails


def pin_closed_forms():
    fails = []
    rng = np.random.default_rng(7)
    B, H, Hk, ql, kl, d = 1, 2, 1, 4, 6, 8
    q, k, v, do, _ = _problem(400, B, H, Hk, ql, kl, d)
    scale = 0.5
    # constant V along keys -> O = that constant row (every row has a visible key)
    vc = np.broadcast_to(v[:, :, :1, :], v.shape).copy()
    o, _ = oracle.fwd(q, k, vc, None, scale=scale, causal=True)
    _cmp("constant V", o, np.broadcast_to(vc[:, :1, :1, :].repeat(H, 1), o.shape), out=fails)
    # Q = 0 -> uniform weights over the visible keys: O = mean of visible V, L = log(#visible)
    qz = np.zeros_like(q)
    o, lse = oracle.fwd(qz, k, v, None, scale=scale, causal=True)
    off = kl - ql
    for i in range(ql):
        n_vis = off + i + 1
        want = v[0, 0, :n_vis, :].astype(np.float64).mean(axis=0)
        for h in range(H):
            _cmp(f"Q=0 O row {i}", o[0, h, i], want, out=fails)
            _cmp(f"Q=0 L row {i}", lse[0, h, i], np.log(n_vis), out=fails)
    # a single key -> O = V_0 and L = s_00 = scale * <q, k_0>
    o, lse = oracle.fwd(q, k[:, :, :1], v[:, :, :1], None, scale=scale, causal=False)
    _cmp("single key O", o, np.broadcast_to(v[:, :, :1], o.shape), out=fails)
    want_l = scale * np.einsum("bhid,bd->bhi", q.astype(np.float64), k[:, 0, 0].astype(np.float64))
    _cmp("single key L", lse, want_l, out=fails)
    # square causal: row 0 sees only key 0
    o, lse = oracle.fwd(q, k[:, :, :ql], v[:, :, :ql], None, scale=scale, causal=True)
    _cmp("causal row 0 O", o[:, :, 0], np.broadcast_to(v[:, 0, 0], o[:, :, 0].shape), out=fails)
    # adding c to a whole mask row shifts L by c and leaves O unchanged
    m = _bf16_exact(rng.uniform(-1, 0, size=(B, H, ql, kl)).astype(np.float32))  # + 0.75 exact
    o1, l1 = oracle.fwd(q, k, v, m, scale=scale, causal=False)
    o2, l2 = oracle.fwd(q, k, v, m + np.float32(0.75), scale=scale, causal=False)
    _cmp("mask shift O", o2, o1, tol=1e-12, out=fails)
    _cmp("mask shift L", l2, l1 + 0.75, tol=1e-12, out=fails)
    # V = identity (d = kl) makes O = P: each row is a distribution, hidden keys get 0
    kk = k[:, :, :, :]
    eye = np.broadcast_to(np.eye(kl, dtype=np.float32), (B, Hk, kl, kl)).copy()
    qq = q[..., :kl] if d >= kl else np.concatenate([q, q], -1)[..., :kl]
    kk = kk[..., :kl] if d >= kl else np.concatenate([kk, kk], -1)[..., :kl]
    p, _ = oracle.fwd(np.ascontiguousarray(qq), np.ascontiguousarray(kk), eye, None, scale=scale,
                      causal=True)
    _cmp("P rows sum to 1", p.sum(-1), np.ones(p.shape[:-1]), out=fails)
    for i in range(ql):
        if (p[..., i, off + i + 1:] != 0).any():
            fails.append(f"P row {i} puts weight on a hidden key")
    return fails


def pin_causal_structure():
    fails = []
    # bottom-right rectangle == last ql rows of the square causal problem over kl queries
    B, H, Hk, ql, kl, d = 1, 2, 1, 3, 7, 4
    q, k, v, do, _ = _problem(500, B, H, Hk, ql, kl, d)
    rng = np.random.default_rng(501)
    top = _bf16_exact(_rand(rng, (B, H, kl - ql, d)))
    qs = np.concatenate([top, q], axis=2)
    dos = np.concatenate([np.zeros_like(top), do], axis=2)
    scale = 0.45
    o, lse = oracle.fwd(q, k, v, None, scale=scale, causal=True)
    os_, ls = oracle.fwd(qs, k, v, None, scale=scale, causal=True)
    _cmp("rect O = square tail", o, os_[:, :, kl - ql:], tol=1e-13, out=fails)
    _cmp("rect L = square tail", lse, ls[:, :, kl - ql:], tol=1e-13, out=fails)
    dq, dk, dv = oracle.bwd(q, k, v, None, do, scale=scale, causal=True)
    dqs, dks, dvs = oracle.bwd(qs, k, v, None, dos, scale=scale, causal=True)
    _cmp("rect dQ = square tail", dq, dqs[:, :, kl - ql:], tol=1e-13, out=fails)
    _cmp("rect dK = square (zero dO on top rows)", dk, dks, tol=1e-13, out=fails)
    _cmp("rect dV = square (zero dO on top rows)", dv, dvs, tol=1e-13, out=fails)
    # mlx-native sentinel test: K rows after the target set to 128 leave O[0..=target] unchanged
    ql = kl = 16
    target = 7
    q, k, v, do, _ = _problem(502, 1, 1, 1, ql, kl, 8)
    kp = k.copy()
    kp[:, :, target + 1:, :] = 128.0
    o1, _ = oracle.fwd(q, k, v, None, scale=0.35, causal=True)
    o2, _ = oracle.fwd(q, kp, v, None, scale=0.35, causal=True)
    _cmp("sentinel K prefix", o2[:, :, :target + 1], o1[:, :, :target + 1], tol=0, out=fails)
    if np.allclose(o2[:, :, target + 1:], o1[:, :, target + 1:]):
        fails.append("sentinel K did not change the rows that may see it")
    return fails


def pin_gqa_equals_repeated_mha():
    fails = []
    B, H, Hk, ql, kl, d = 2, 6, 2, 5, 5, 4
    q, k, v, do, m = _problem(600, B, H, Hk, ql, kl, d, mask=True)
    G = H // Hk
    kr, vr = np.repeat(k, G, axis=1), np.repeat(v, G, axis=1)
    scale = 0.3
    o, lse = oracle.fwd(q, k, v, m, scale=scale, causal=True)
    o2, l2 = oracle.fwd(q, kr, vr, m, scale=scale, causal=True)
    _cmp("GQA O", o, o2, tol=0, out=fails)
    _cmp("GQA L", lse, l2, tol=0, out=fails)
    dq, dk, dv = oracle.bwd(q, k, v, m, do, scale=scale, causal=True)
    dq2, dk2, dv2 = oracle.bwd(q, kr, vr, m, do, scale=scale, causal=True)
    _cmp("GQA dQ", dq, dq2, tol=1e-13, out=fails)
    _cmp("GQA dK = sum over repeats", dk, dk2.reshape(B, Hk, G, kl, d).sum(2), tol=1e-13, out=fails)
    _cmp("GQA dV = sum over repeats", dv, dv2.reshape(B, Hk, G, kl, d).sum(2), tol=1e-13, out=fails)
    return fails


def pin_bwd_invariants():
    fails = []
    B, H, Hk, ql, kl, d = 1, 4, 2, 6, 8, 4
    q, k, v, do, m = _problem(700, B, H, Hk, ql, kl, d, mask=True, neg_inf_frac=0.2)
    m[0, 1, 2, :] = -np.inf  # one fully masked row
    scale = 0.5
    o, lse = oracle.fwd(q, k, v, m, scale=scale, causal=True)
    dq, dk, dv = oracle.bwd(q, k, v, m, do, scale=scale, causal=True)
    # sum_j dS_ij = 0  =>  sum_j dK_j = 0 for every kv head
    _cmp("sum_j dK = 0", dk.sum(axis=2), np.zeros((B, Hk, d)), tol=1e-12, out=fails)
    # sum_j dV_j = sum of dO over the group's rows that see at least one key
    G = H // Hk
    live = np.isfinite(lse)
    want = (do.astype(np.float64) * live[..., None]).reshape(B, Hk, G, ql, d).sum(axis=(2, 3))
    _cmp("sum_j dV = sum dO of live rows", dv.sum(axis=2), want, tol=1e-12, out=fails)
    # the fully masked row: O = 0, L = -inf, dQ = 0 exactly, and nothing is NaN
    if not (o[0, 1, 2] == 0).all() or lse[0, 1, 2] != -np.inf or not (dq[0, 1, 2] == 0).all():
        fails.append("fully masked row is not O=0, L=-inf, dQ=0")
    for name, a in (("O", o), ("dQ", dq), ("dK", dk), ("dV", dv)):
        if np.isnan(a).any():
            fails.append(f"NaN in {name}")
    # all keys equal -> constant scores per row -> dQ = 0
    ke = np.broadcast_to(k[:, :, :1], k.shape).copy()
    dq0, _, _ = oracle.bwd(q, ke, v, None, do, scale=scale, causal=False)
    _cmp("equal keys -> dQ = 0", dq0, np.zeros_like(dq0), tol=1e-12, out=fails)
    return fails


def pin_base2_mode_agrees():
    fails = []
    q, k, v, do, m = _problem(800, 2, 4, 2, 9, 13, 16, mask=True, neg_inf_frac=0.1)
    m[1, 3, 4, :] = -np.inf
    for causal in (False, True):
        o1, l1 = oracle.fwd(q, k, v, m, scale=0.25, causal=causal)
        o2, l2 = oracle.fwd(q, k, v, m, scale=0.25, causal=causal, base2=True)
        _cmp(f"base2 O causal={causal}", o2, o1, tol=1e-12, out=fails)
        _cmp(f"base2 L causal={causal}", l2, l1, tol=1e-12, out=fails)
    return fails


def pin_sampled_entry_points_agree():
    fails = []
    B, H, Hk, ql, kl, d = 2, 4, 2, 7, 9, 8
    q, k, v, do, m = _problem(900, B, H, Hk, ql, kl, d, mask=True)
    scale = 0.3
    o, lse = oracle.fwd(q, k, v, m, scale=scale, causal=True)
    dq, dk, dv = oracle.bwd(q, k, v, m, do, scale=scale, causal=True)
    rows = np.array([0, 5, 13, 40, B * H * ql - 1])
    o_r, l_r = oracle.fwd_rows(q, k, v, m, scale=scale, causal=True, rows=rows)
    _cmp("fwd_rows O", o_r, o.reshape(-1, d)[rows], tol=0, out=fails)
    _cmp("fwd_rows L", l_r, lse.reshape(-1)[rows], tol=0, out=fails)
    dq_r = oracle.bwd_q_rows(q, k, v, m, do, scale=scale, causal=True, rows=rows)
    _cmp("bwd_q_rows", dq_r, dq.reshape(-1, d)[rows], tol=0, out=fails)
    js = [0, 4, 8]
    dk_r, dv_r = oracle.bwd_kv_rows(q, k, v, m, do, scale=scale, causal=True, b=1, kh=1, js=js)
    _cmp("bwd_kv_rows dK", dk_r, dk[1, 1, js], tol=1e-14, out=fails)
    _cmp("bwd_kv_rows dV", dv_r, dv[1, 1, js], tol=1e-14, out=fails)
    return fails


# Local-window cases: (B, H, Hk, ql, kl, d, causal, mask, (window_left, window_right))
WINDOW_CASES = [
    (1, 2, 1, 9, 9, 4, True, False, (3, -1)),
    (1, 2, 2, 6, 11, 8, False, False, (2, 1)),
    (2, 4, 2, 7, 7, 4, True, True, (0, -1)),
    (1, 2, 1, 5, 12, 4, False, True, (-1, 2)),
]


def pin_window_vs_torch():
    """The oracle's local window against torch's CPU kernels with a tril/triu band."""
    fails = []
    for n, (B, H, Hk, ql, kl, d, causal, mask, win) in enumerate(WINDOW_CASES):
        q, k, v, do, m = _problem(1000 + n, B, H, Hk, ql, kl, d, mask)
        scale = 0.43
        with oracle.window(*win):
            o, lse = oracle.fwd(q, k, v, m, scale=scale, causal=causal)
            dq, dk, dv = oracle.bwd(q, k, v, m, do, scale=scale, causal=causal)
        to, tl = _torch_fwd(q, k, v, m, scale, causal, win)
        live = np.isfinite(tl)
        _cmp(f"win{n} O", o[live], to[live], out=fails)
        _cmp(f"win{n} L", lse, tl, out=fails)
        if live.all():
            tq, tk, tv = _torch_grads(q, k, v, m, do, scale, causal, win)
            _cmp(f"win{n} dQ", dq, tq, out=fails)
            _cmp(f"win{n} dK", dk, tk, out=fails)
            _cmp(f"win{n} dV", dv, tv, out=fails)
    return fails


def pin_window_closed_forms():
    fails = []
    B, H, Hk, ql, kl, d = 1, 2, 1, 6, 10, 4
    q, k, v, do, _ = _problem(1100, B, H, Hk, ql, kl, d)
    off = kl - ql
    # causal with a zero-width left window: row i sees only key off + i, so O = V[off + i]
    with oracle.window(0, -1):
        o, lse = oracle.fwd(q, k, v, None, scale=0.5, causal=True)
    want = np.broadcast_to(v[:, :, off:off + ql, :], o.shape)
    _cmp("window 0: O = diagonal V", o, want, tol=0, out=fails)
    want_l = 0.5 * np.einsum("bhid,bhid->bhi", q.astype(np.float64),
                             np.broadcast_to(k[:, :, off:off + ql, :], q.shape).astype(np.float64))
    _cmp("window 0: L = diagonal score", lse, want_l, out=fails)
    # a window wider than the keys changes nothing
    o0, l0 = oracle.fwd(q, k, v, None, scale=0.5, causal=True)
    with oracle.window(kl + 5, kl + 5):
        o1, l1 = oracle.fwd(q, k, v, None, scale=0.5, causal=True)
    _cmp("wide window O", o1, o0, tol=0, out=fails)
    _cmp("wide window L", l1, l0, tol=0, out=fails)
    # the window equals the same band given as an additive -inf mask (the pages' SWA form)
    ii = np.arange(ql)[:, None] + off
    jj = np.arange(kl)[None, :]
    band = np.where((jj >= ii - 3) & (jj <= ii + 1), 0.0, -np.inf).astype(np.float32)
    mband = np.broadcast_to(band, (B, H, ql, kl)).copy()
    with oracle.window(3, 1):
        ow, lw = oracle.fwd(q, k, v, None, scale=0.5, causal=False)
        gw = oracle.bwd(q, k, v, None, do, scale=0.5, causal=False)
    om, lm = oracle.fwd(q, k, v, mband, scale=0.5, causal=False)
    gm = oracle.bwd(q, k, v, mband, do, scale=0.5, causal=False)
    _cmp("window = band mask O", ow, om, tol=0, out=fails)
    _cmp("window = band mask L", lw, lm, tol=0, out=fails)
    for a, b_, n in zip(gw, gm, ("dQ", "dK", "dV")):
        _cmp(f"window = band mask {n}", a, b_, tol=1e-15, out=fails)
    return fails


# ------------------------------------------------------------------ attention sinks
# A sink is one extra logit per query head that joins the softmax normaliser and carries no
# value. torch has no sink argument, so the pin builds the equivalent problem for torch: one
# extra key with k = 0 and v = 0 whose additive bias column is sink_h. torch's own kernels
# then compute O and L, and autograd through that bias column gives d(sinks).
SINK_CASES = [
    # (B, H, Hk, ql, kl, d, causal, mask, window)
    (1, 2, 1, 4, 6, 8, False, False, None),
    (2, 4, 2, 5, 5, 4, True, False, None),
    (1, 2, 2, 3, 7, 8, True, True, None),       # rectangle + mask
    (1, 4, 1, 6, 6, 4, True, False, (2, -1)),   # causal sliding window
]


def _sink_aug(k, v, sinks_t, bias, B, ql):
    """k, v with a zero key/value prepended, and the bias with the sink column in front."""
    Bk, Hk, kl, d = k.shape
    kz = np.concatenate([np.zeros((Bk, Hk, 1, d), np.float32), k], axis=2)
    vz = np.concatenate([np.zeros((Bk, Hk, 1, v.shape[3]), np.float32), v], axis=2)
    H = sinks_t.shape[0]
    col = sinks_t.view(1, H, 1, 1).expand(B, H, ql, 1)
    return kz, vz, torch.cat([col, bias], dim=-1)


def pin_sinks_vs_torch():
    fails = []
    for n, (B, H, Hk, ql, kl, d, causal, mask, win) in enumerate(SINK_CASES):
        q, k, v, do, m = _problem(800 + n, B, H, Hk, ql, kl, d, mask)
        if mask:  # one fully masked row: with a sink it has O = 0 and L = sink
            m[0, 0, 1, :] = -np.inf
        rng = np.random.default_rng(850 + n)
        sinks = _bf16_exact((2.0 * rng.standard_normal(H)).astype(np.float32))
        scale = 0.45
        with oracle.window(*(win or (-1, -1))), oracle.sinks(sinks):
            o, lse = oracle.fwd(q, k, v, m, scale=scale, causal=causal)
            dq, dk, dv = oracle.bwd(q, k, v, m, do, scale=scale, causal=causal)
            ds = oracle.dsinks(q, k, v, m, do, scale=scale, causal=causal)
        bias = _torch_bias(ql, kl, causal, m, H, B, win)
        # forward: torch's CPU flash kernel on the augmented problem
        st = torch.from_numpy(sinks).double()
        kz, vz, bz = _sink_aug(k, v, st, bias, B, ql)
        G = H // Hk
        to, tl = torch.ops.aten._scaled_dot_product_flash_attention_for_cpu(
            torch.from_numpy(q).double(), torch.from_numpy(kz).double().repeat_interleave(G, 1),
            torch.from_numpy(vz).double().repeat_interleave(G, 1), 0.0, False, attn_mask=bz,
            scale=scale)
        _cmp(f"sink case{n} O", o, to.numpy(), out=fails)
        _cmp(f"sink case{n} L", lse, tl.numpy(), out=fails)
        # backward: autograd through the math backend, sinks as a leaf
        st = torch.from_numpy(sinks).double().requires_grad_()
        qt = torch.from_numpy(q).double().requires_grad_()
        kt = torch.from_numpy(kz).double().requires_grad_()
        vt = torch.from_numpy(vz).double().requires_grad_()
        _, _, bz = _sink_aug(k, v, st, bias, B, ql)
        with torch.nn.attention.sdpa_kernel(torch.nn.attention.SDPBackend.MATH):
            ot = F.scaled_dot_product_attention(qt, kt, vt, attn_mask=bz, scale=scale,
                                                enable_gqa=True)
        (ot * torch.from_numpy(do).double()).sum().backward()
        _cmp(f"sink case{n} dQ", dq, qt.grad.numpy(), out=fails)
        _cmp(f"sink case{n} dK", dk, kt.grad.numpy()[:, :, 1:], out=fails)
        _cmp(f"sink case{n} dV", dv, vt.grad.numpy()[:, :, 1:], out=fails)
        _cmp(f"sink case{n} dsinks", ds, st.grad.numpy(), out=fails)
    return fails


def pin_sinks_closed_forms():
    """Q = 0 with no mask: every visible score is 0, so O = sum(v) / (n + e^sink) and
    L = log(n + e^sink); a row that sees nothing has O = 0, L = sink; a very negative sink is
    no sink; and d(sinks) against central differences of the oracle's forward."""
    fails = []
    B, H, Hk, ql, kl, d = 1, 2, 1, 3, 5, 4
    _, k, v, do, _ = _problem(870, B, H, Hk, ql, kl, d)
    q0 = np.zeros((B, H, ql, d), np.float32)
    sinks = np.array([0.5, -1.25], np.float32)
    with oracle.sinks(sinks):
        o, lse = oracle.fwd(q0, k, v, None, scale=0.5, causal=False)
    z = kl + np.exp(sinks.astype(np.float64))
    want_o = np.broadcast_to(v.astype(np.float64).sum(axis=2, keepdims=True), (B, Hk, 1, d))
    want_o = np.repeat(want_o, H // Hk, axis=1) / z[None, :, None, None]
    _cmp("sink Q=0 O", o, np.broadcast_to(want_o, o.shape), tol=1e-13, out=fails)
    _cmp("sink Q=0 L", lse, np.broadcast_to(np.log(z)[None, :, None], lse.shape), tol=1e-13,
         out=fails)
    # a fully masked row (causal with ql > kl: the first ql - kl rows see no key)
    q, k2, v2, do2, _ = _problem(871, 1, 2, 1, 6, 4, 4)
    with oracle.sinks(sinks):
        o, lse = oracle.fwd(q, k2, v2, None, scale=0.5, causal=True)
        dq, _, _ = oracle.bwd(q, k2, v2, None, do2, scale=0.5, causal=True)
    _cmp("sink dead row O", o[:, :, :2], np.zeros_like(o[:, :, :2]), tol=0, out=fails)
    _cmp("sink dead row L", lse[:, :, :2],
         np.broadcast_to(sinks.astype(np.float64)[None, :, None], (1, 2, 2)), tol=0, out=fails)
    _cmp("sink dead row dQ", dq[:, :, :2], np.zeros_like(dq[:, :, :2]), tol=0, out=fails)
    # a sink far below every score changes nothing
    q, k3, v3, do3, m3 = _problem(872, 1, 2, 2, 4, 5, 4, mask=True)
    o_ref, l_ref = oracle.fwd(q, k3, v3, m3, scale=0.5, causal=True)
    with oracle.sinks(np.full(2, -200.0, np.float32)):
        o_s, l_s = oracle.fwd(q, k3, v3, m3, scale=0.5, causal=True)
    _cmp("sink -200 O", o_s, o_ref, tol=1e-15, out=fails)
    _cmp("sink -200 L", l_s, l_ref, tol=1e-15, out=fails)
    # dsinks against central differences of sum(O * dO)
    q, k4, v4, do4, m4 = _problem(873, 1, 2, 1, 4, 6, 4, mask=True, neg_inf_frac=0.2)
    base = np.array([0.75, -0.5], np.float32)
    with oracle.sinks(base):
        ds = oracle.dsinks(q, k4, v4, m4, do4, scale=0.6, causal=True)
    num = np.zeros(2)
    for h in range(2):
        ests = []
        for step in (2.0 ** -8, 2.0 ** -9):
            vals = []
            for sgn in (1, -1):
                sk = base.copy()
                sk[h] += np.float32(sgn * step)
                with oracle.sinks(sk):
                    o4, _ = oracle.fwd(q, k4, v4, m4, scale=0.6, causal=True, nthreads=1)
                vals.append(float((o4 * do4.astype(np.float64)).sum()))
            ests.append((vals[0] - vals[1]) / (2 * step))
        num[h] = (4 * ests[1] - ests[0]) / 3
    _cmp("FD dsinks", ds, num, tol=2e-7, out=fails)
    return fails


# ------------------------------------------------------------------ value head dim != d
DV_CASES = [
    # (B, H, Hk, ql, kl, d, dv, causal, mask)
    (1, 2, 1, 4, 6, 8, 4, False, False),
    (2, 4, 2, 5, 5, 4, 8, True, False),
    (1, 2, 2, 3, 7, 8, 12, True, True),
]


def pin_value_dim_vs_torch():
    """dv != d: L does not depend on V, so torch's CPU flash kernel with a d-wide V gives it;
    O and the gradients come from torch's math backend, which takes any value width."""
    fails = []
    for n, (B, H, Hk, ql, kl, d, dvd, causal, mask) in enumerate(DV_CASES):
        q, k, v_d, do_d, m = _problem(900 + n, B, H, Hk, ql, kl, d, mask)
        rng = np.random.default_rng(950 + n)
        v = _bf16_exact(rng.standard_normal((B, Hk, kl, dvd)).astype(np.float32))
        do = _bf16_exact(rng.standard_normal((B, H, ql, dvd)).astype(np.float32))
        scale = 0.39
        o, lse = oracle.fwd(q, k, v, m, scale=scale, causal=causal)
        dq, dk, dv = oracle.bwd(q, k, v, m, do, scale=scale, causal=causal)
        _, tl = _torch_fwd(q, k, v_d, m, scale, causal)
        _cmp(f"dv case{n} L", lse, tl, out=fails)
        bias = _torch_bias(ql, kl, causal, m, H, B)
        qt = torch.from_numpy(q).double().requires_grad_()
        kt = torch.from_numpy(k).double().requires_grad_()
        vt = torch.from_numpy(v).double().requires_grad_()
        with torch.nn.attention.sdpa_kernel(torch.nn.attention.SDPBackend.MATH):
            ot = F.scaled_dot_product_attention(qt, kt, vt, attn_mask=bias, scale=scale,
                                                enable_gqa=True)
        (ot * torch.from_numpy(do).double()).sum().backward()
        _cmp(f"dv case{n} O", o, ot.detach().numpy(), out=fails)
        _cmp(f"dv case{n} dQ", dq, qt.grad.numpy(), out=fails)
        _cmp(f"dv case{n} dK", dk, kt.grad.numpy(), out=fails)
        _cmp(f"dv case{n} dV", dv, vt.grad.numpy(), out=fails)
    return fails


def pin_value_dim_identity():
    """dv = kl and V = I (per kv head): O is the P matrix itself, so each live row of O sums to
    one, hidden keys get exactly 0, and O_ij = exp(s_ij - L_i) with the scores from torch."""
    fails = []
    B, H, Hk, ql, kl, d = 1, 2, 1, 4, 6, 8
    q, k, _, _, _ = _problem(960, B, H, Hk, ql, kl, d)
    v = np.broadcast_to(np.eye(kl, dtype=np.float32), (B, Hk, kl, kl)).copy()
    o, lse = oracle.fwd(q, k, v, None, scale=0.3, causal=True)
    _cmp("V=I rows sum to 1", o.sum(axis=-1), np.ones((B, H, ql)), tol=1e-14, out=fails)
    allowed = causal_lower_right(ql, kl)._materialize(device="cpu").numpy()
    hidden = np.broadcast_to(~allowed, o.shape)
    _cmp("V=I hidden keys", np.where(hidden, o, 0.0), np.zeros_like(o), tol=0, out=fails)
    s = torch.from_numpy(q).double() @ torch.from_numpy(k).double().repeat_interleave(
        H // Hk, 1).transpose(-1, -2) * 0.3
    want = np.where(hidden, 0.0, np.exp(s.numpy() - lse[..., None]))
    _cmp("V=I O = P", o, want, tol=1e-13, out=fails)
    return fails


# ------------------------------------------------------------------ paged key/value cache
# (batch, query heads, kv heads, queries, head dim, page size, min len, max len, causal)
PAGED_CASES = [
    (1, 4, 4, 1, 16, 4, 9, 9, False),
    (3, 4, 2, 1, 8, 4, 1, 13, True),
    (2, 4, 1, 3, 8, 4, 3, 11, True),     # several queries: bottom-right causal per sequence
    (2, 2, 2, 4, 8, 8, 2, 17, True),     # lq > len for a short sequence: rows with no key
    (2, 4, 2, 2, 8, 4, 6, 10, False),
]


def _paged(n, case, poison=True):
    import fa_inputs

    B, H, Hk, lq, d, bs, lo, hi, causal = case
    w = fa_inputs.DecodeWorkload(f"pin{n}", B, H, Hk, lq, d, bs, lo, hi, causal)
    return w, fa_inputs.make_paged_inputs(w, index=100 + n, poison=poison)


def _gather(cache, table, b, length, bs):
    """Keys 0 .. length-1 of sequence b as [Hk, length, d] (numpy fancy indexing)."""
    j = np.arange(length)
    return cache[table[b, j // bs], :, j % bs, :].transpose(1, 0, 2)


def pin_paged_vs_torch():
    """Each sequence's keys gathered from the pages with numpy, then torch's CPU flash kernel
    with its own bottom-right causal bias (the sequence's queries are its last positions)."""
    fails = []
    for n, case in enumerate(PAGED_CASES):
        w, x = _paged(n, case)
        q, kc, vc = x.widened()
        o, lse = oracle.paged_fwd(q, kc, vc, x.block_table, x.lengths, scale=w.scale,
                                  causal=w.causal)
        G = w.n_heads // w.n_kv_heads
        for b in range(w.batch):
            L = int(x.lengths[b])
            if L == 0:
                continue
            kb = torch.from_numpy(_gather(kc, x.block_table, b, L, w.page_size)).double()
            vb = torch.from_numpy(_gather(vc, x.block_table, b, L, w.page_size)).double()
            qb = torch.from_numpy(q[b:b + 1]).double()
            bias = torch.zeros(1, w.n_heads, w.q_len, L, dtype=torch.float64)
            if w.causal:
                allowed = causal_lower_right(w.q_len, L)._materialize(device="cpu")
                bias = bias.masked_fill(~allowed, float("-inf"))
            to, tl = torch.ops.aten._scaled_dot_product_flash_attention_for_cpu(
                qb, kb[None].repeat_interleave(G, 1), vb[None].repeat_interleave(G, 1), 0.0,
                False, attn_mask=bias, scale=w.scale)
            dead = torch.isinf(tl) | torch.isnan(tl)  # rows that see no key
            to = torch.where(dead[..., None], torch.zeros_like(to), to)
            tl = torch.where(dead, torch.full_like(tl, float("-inf")), tl)
            _cmp(f"paged case{n} seq{b} O", o[b:b + 1], to.numpy(), out=fails)
            _cmp(f"paged case{n} seq{b} L", lse[b:b + 1], tl.numpy(), out=fails)
    return fails


def pin_paged_layout_invariance():
    """The physical placement of the pages is invisible: a different page order (table
    updated), and NaN instead of zeros in every slot that holds no key, give identical bits;
    and the result equals the contiguous oracle on each sequence's gathered keys."""
    fails = []
    for n, case in enumerate(PAGED_CASES):
        w, x = _paged(n, case, poison=True)
        _, xz = _paged(n, case, poison=False)
        q, kc, vc = x.widened()
        o1, l1 = oracle.paged_fwd(q, kc, vc, x.block_table, x.lengths, scale=w.scale,
                                  causal=w.causal)
        qz, kz, vz = xz.widened()
        o0, l0 = oracle.paged_fwd(qz, kz, vz, xz.block_table, xz.lengths, scale=w.scale,
                                  causal=w.causal)
        _cmp(f"paged case{n} NaN-free O", o1, o0, tol=0, out=fails)
        _cmp(f"paged case{n} NaN-free L", l1, l0, tol=0, out=fails)
        # move every page to a new place
        rng = np.random.default_rng(7 + n)
        perm = rng.permutation(kc.shape[0])
        inv = np.argsort(perm)
        o2, l2 = oracle.paged_fwd(q, kc[perm], vc[perm], inv[x.block_table].astype(np.int32),
                                  x.lengths, scale=w.scale, causal=w.causal)
        _cmp(f"paged case{n} moved pages O", o2, o1, tol=0, out=fails)
        _cmp(f"paged case{n} moved pages L", l2, l1, tol=0, out=fails)
        for b in range(w.batch):
            L = int(x.lengths[b])
            if L == 0:
                continue
            kb = _gather(kc, x.block_table, b, L, w.page_size)[None]
            vb = _gather(vc, x.block_table, b, L, w.page_size)[None]
            oc, lc = oracle.fwd(q[b:b + 1], kb, vb, None, scale=w.scale, causal=w.causal)
            _cmp(f"paged case{n} seq{b} = contiguous O", o1[b:b + 1], oc, tol=1e-15, out=fails)
            _cmp(f"paged case{n} seq{b} = contiguous L", l1[b:b + 1], lc, tol=1e-15, out=fails)
    return fails


def _torch_paged_loss(q, kc, vc, table, lens, do, scale, causal, G):
    """sum(O * dO) of the paged attention, composed from torch ops on the whole caches (the
    keys of each sequence gathered by advanced indexing), so that autograd differentiates the
    page lookup itself."""
    B, H, lq, d = q.shape
    bs = kc.shape[2]
    loss = q.new_zeros(())
    for b in range(B):
        n = int(lens[b])
        if n == 0:
            continue
        j = torch.arange(n)
        pages = torch.as_tensor(table[b], dtype=torch.long)[j // bs]
        kb = kc[pages, :, j % bs, :].permute(1, 0, 2).repeat_interleave(G, 0)  # [H, n, d]
        vb = vc[pages, :, j % bs, :].permute(1, 0, 2).repeat_interleave(G, 0)
        s_ = q[b] @ kb.transpose(1, 2) * scale  # [H, lq, n]
        if causal:
            i = torch.arange(lq)[:, None]
            hidden = j[None, :] > n - lq + i  # bottom-right: query i is position n - lq + i
        else:
            hidden = torch.zeros(lq, n, dtype=torch.bool)
        dead = hidden.all(dim=1)  # rows that see no key: O = 0
        s_ = s_.masked_fill(hidden[None], float("-inf"))
        s_ = torch.where(dead[None, :, None], torch.zeros_like(s_), s_)  # finite softmax input
        p_ = torch.softmax(s_, dim=-1)
        p_ = torch.where(dead[None, :, None], torch.zeros_like(p_), p_)
        loss = loss + ((p_ @ vb) * do[b]).sum()
    return loss


PAGED_BWD_CASES = [
    # (B, H, Hk, lq, d, page_size, lengths, causal, shared): shared names one page twice
    (2, 4, 2, 1, 8, 4, (6, 11), False, False),
    (2, 4, 1, 3, 8, 4, (9, 2), True, False),    # lq > len for the short sequence
    (3, 2, 2, 2, 4, 8, (17, 0, 8), True, False),  # an empty sequence
    (2, 4, 2, 2, 8, 4, (8, 8), True, True),     # a page read by both sequences
]


def pin_paged_bwd_vs_torch_autograd():
    """The paged gradients (dQ and both cache gradients) against torch autograd in f64 through
    a paged forward built from torch ops on the whole caches: unused slots and pages get
    exactly 0, and a page named by two sequences gets the sum of both."""
    import fa_inputs

    fails = []
    for n, (B, H, Hk, lq, d, bs, lens, causal, shared) in enumerate(PAGED_BWD_CASES):
        G = H // Hk
        per = max(-(-L // bs) for L in lens) if max(lens) else 1
        P = B * per + 3  # three pages nobody uses
        rng = np.random.default_rng(500 + n)
        order = rng.permutation(P)
        table = order[:B * per].reshape(B, per).astype(np.int32)
        if shared:
            table[1, 0] = table[0, 0]
        q = fa_inputs.bf16_bits_to_f32(fa_inputs.normal_bf16(900 + 4 * n, (B, H, lq, d)))
        kc = fa_inputs.bf16_bits_to_f32(fa_inputs.normal_bf16(901 + 4 * n, (P, Hk, bs, d)))
        vc = fa_inputs.bf16_bits_to_f32(fa_inputs.normal_bf16(902 + 4 * n, (P, Hk, bs, d)))
        do = fa_inputs.bf16_bits_to_f32(fa_inputs.normal_bf16(903 + 4 * n, (B, H, lq, d)))
        lens_a = np.asarray(lens, np.int32)
        dq, dk, dv = oracle.paged_bwd(q, kc, vc, table, lens_a, do, scale=0.35, causal=causal)
        tq, tk, tv = (torch.from_numpy(x).double().requires_grad_() for x in (q, kc, vc))
        _torch_paged_loss(tq, tk, tv, table, lens_a, torch.from_numpy(do).double(), 0.35,
                          causal, G).backward()
        _cmp(f"paged bwd case{n} dQ", dq, tq.grad.numpy(), out=fails)
        _cmp(f"paged bwd case{n} dK cache", dk, tk.grad.numpy(), out=fails)
        _cmp(f"paged bwd case{n} dV cache", dv, tv.grad.numpy(), out=fails)
        unused = np.setdiff1d(np.arange(P), table.ravel())
        if np.abs(dk[unused]).max(initial=0) != 0 or np.abs(dv[unused]).max(initial=0) != 0:
            fails.append(f"paged bwd case{n}: an unused page got a gradient")
    return fails


def pin_paged_bwd_vs_finite_differences():
    """The paged gradients against f64 central differences (Richardson-extrapolated, steps
    2^-8 and 2^-9, exact for bf16-valued inputs) of loss = sum(O * dO) through the oracle's
    paged forward, for every element of q and of both caches on a tiny causal multi-query
    problem with shuffled pages, a partly filled last page and a page nobody uses."""
    import fa_inputs

    fails = []
    B, H, Hk, lq, d, bs, lens = 2, 2, 1, 2, 4, 4, (5, 3)
    P = 2 * 2 + 1
    table = np.array([[3, 0], [4, 2]], np.int32)  # page 1 unused; sequence 1 uses one page
    q = fa_inputs.bf16_bits_to_f32(fa_inputs.normal_bf16(950, (B, H, lq, d)))
    kc = fa_inputs.bf16_bits_to_f32(fa_inputs.normal_bf16(951, (P, Hk, bs, d)))
    vc = fa_inputs.bf16_bits_to_f32(fa_inputs.normal_bf16(952, (P, Hk, bs, d)))
    do = fa_inputs.bf16_bits_to_f32(fa_inputs.normal_bf16(953, (B, H, lq, d)))
    lens_a = np.asarray(lens, np.int32)
    scale = 0.45
    dq, dk, dv = oracle.paged_bwd(q, kc, vc, table, lens_a, do, scale=scale, causal=True)

    def loss(qq, kk, vv):
        o, _ = oracle.paged_fwd(qq, kk, vv, table, lens_a, scale=scale, causal=True)
        return float((o * do.astype(np.float64)).sum())

    for name, arr, grad in (("q", q, dq), ("k cache", kc, dk), ("v cache", vc, dv)):
        num = np.zeros(arr.shape)
        for idx in np.ndindex(arr.shape):
            ests = []
            for h in (2.0 ** -8, 2.0 ** -9):
                plus, minus = arr.copy(), arr.copy()
                plus[idx] += np.float32(h)
                minus[idx] -= np.float32(h)
                args_p = {"q": (plus, kc, vc), "k cache": (q, plus, vc), "v cache": (q, kc, plus)}
                args_m = {"q": (minus, kc, vc), "k cache": (q, minus, vc),
                          "v cache": (q, kc, minus)}
                ests.append((loss(*args_p[name]) - loss(*args_m[name])) / (2 * h))
            num[idx] = (4 * ests[1] - ests[0]) / 3
        _cmp(f"paged FD d{name}", grad, num, tol=2e-7, out=fails)
    return fails


# ------------------------------------------------------------------ variable-length batches
VARLEN_CASES = [
    # (H, Hk, d, q_lens, k_lens, causal)
    (4, 2, 8, (3, 5, 1), (3, 7, 4), True),
    (2, 2, 4, (4, 0, 6), (9, 3, 2), False),     # an empty query sequence
    (4, 1, 8, (2, 5), (0, 5), True),            # a sequence with no keys
    (2, 1, 8, (6, 3, 4), (6, 2, 9), True),      # ql > kl: rows that see no key
]


def pin_varlen_vs_torch():
    """Each packed sequence against torch's CPU flash kernel (O, L) and autograd (dQ, dK, dV)
    on that sequence alone, with torch's bottom-right causal bias."""
    import fa_inputs

    fails = []
    for n, (H, Hk, d, ql, kl, causal) in enumerate(VARLEN_CASES):
        w = fa_inputs.VarlenWorkload(f"pin{n}", H, Hk, d, ql, kl, causal)
        x = fa_inputs.make_varlen_inputs(w, index=140 + n)
        q, k, v, do = x.widened()
        o, lse = oracle.varlen_fwd(q, k, v, x.cu_q, x.cu_k, scale=0.4, causal=causal)
        dq, dk, dv = oracle.varlen_bwd(q, k, v, do, x.cu_q, x.cu_k, scale=0.4, causal=causal)
        for b in range(w.batch):
            qs, qe, ks, ke = x.cu_q[b], x.cu_q[b + 1], x.cu_k[b], x.cu_k[b + 1]
            if qe == qs:
                continue
            tag = f"varlen case{n} seq{b}"
            if ke == ks:
                _cmp(tag + " O (no keys)", o[:, qs:qe], np.zeros_like(o[:, qs:qe]), tol=0, out=fails)
                _cmp(tag + " L (no keys)", lse[:, qs:qe], np.full_like(lse[:, qs:qe], -np.inf),
                     tol=0, out=fails)
                continue
            qb, kb, vb, dob = (t[None, :, a:e] for t, (a, e) in
                               ((q, (qs, qe)), (k, (ks, ke)), (v, (ks, ke)), (do, (qs, qe))))
            to, tl = _torch_fwd(qb, kb, vb, None, 0.4, causal)
            # rows that see no key (causal, query position before the first key): O = 0 and
            # L = -inf by the definition; torch reports another L there
            rows = np.arange(qe - qs)
            dead = np.broadcast_to(causal & ((ke - ks) - (qe - qs) + rows < 0), tl.shape)
            to = np.where(dead[..., None], 0.0, to)
            tl = np.where(dead, -np.inf, tl)
            _cmp(tag + " O", o[None, :, qs:qe], to, out=fails)
            _cmp(tag + " L", lse[None, :, qs:qe], tl, out=fails)
            tq, tk, tv = _torch_grads(qb, kb, vb, None, dob, 0.4, causal)
            tq = np.nan_to_num(tq)
            _cmp(tag + " dQ", dq[None, :, qs:qe], tq, out=fails)
            _cmp(tag + " dK", dk[None, :, ks:ke], np.nan_to_num(tk), out=fails)
            _cmp(tag + " dV", dv[None, :, ks:ke], np.nan_to_num(tv), out=fails)
        # keys and values of other sequences are untouched: their gradients stay 0 outside
        # every sequence's rows, and equal lengths give the batched problem
    return fails


def pin_mask_forms_vs_torch():
    """The mask forms the CUDA path accepts, through `oracle.dense_mask`, against torch given the
    same mask in its own form (page "nuvec-core tests/fast.rs",
    `attention_kernels_match_the_fallback`: bool [lq, lk] masks and additive [1, Hq, Lq, Lk]
    masks). torch's scaled_dot_product_attention reads a bool `attn_mask` as True = the key takes
    part, and broadcasts a mask of shape [ql, kl], [B, 1, ql, kl] or [1, H, ql, kl] itself; an
    additive bf16 mask is widened to f64 by torch. O, dQ, dK and dV come from torch's math kernel
    and autograd (f64); L from torch.logsumexp over torch's masked scores. A row that the mask
    hides entirely must give O = 0 (torch's math kernel returns zeros there), L = -inf and zero
    gradients."""
    out = []
    B, H, Hk, ql, kl, d = 2, 4, 2, 9, 13, 8
    q, k, v, do, _ = _problem(71, B, H, Hk, ql, kl, d)
    rng = np.random.default_rng(72)
    scale = 0.35
    m_2d = rng.random((ql, kl)) > 0.3
    m_2d[3, :] = False  # one row hidden entirely
    m_b1 = rng.random((B, 1, ql, kl)) > 0.3
    m_bf = rng.uniform(-2.0, 0.5, size=(1, H, ql, kl)).astype(np.float32)
    m_bf[rng.random(m_bf.shape) < 0.1] = -np.inf
    m_bf = _bf16_exact(m_bf)
    cases = [("bool [ql,kl]", m_2d, False), ("bool [B,1,ql,kl] causal", m_b1, True),
             ("bf16 [1,H,ql,kl]", m_bf, False)]
    G = H // Hk
    for name, m_np, causal in cases:
        dm = oracle.dense_mask(m_np, (B, H, ql, kl))
        o, lse = oracle.fwd(q, k, v, dm, scale=scale, causal=causal)
        dq, dk, dv = oracle.bwd(q, k, v, dm, do, scale=scale, causal=causal)
        if m_np.dtype == np.bool_:
            tm = torch.from_numpy(m_np)
            if causal:
                tm = tm & causal_lower_right(ql, kl)._materialize(device="cpu")
        else:  # (the additive case runs without causal)
            tm = torch.from_numpy(m_np).to(torch.bfloat16).double()
        qt = torch.from_numpy(q).double().requires_grad_()
        kt = torch.from_numpy(k).double().requires_grad_()
        vt = torch.from_numpy(v).double().requires_grad_()
        with torch.nn.attention.sdpa_kernel(torch.nn.attention.SDPBackend.MATH):
            ot = F.scaled_dot_product_attention(qt, kt, vt, attn_mask=tm, scale=scale,
                                                enable_gqa=True)
        (ot * torch.from_numpy(do).double()).sum().backward()
        _cmp(f"mask {name} O", o, ot.detach().numpy(), out=out)
        _cmp(f"mask {name} dQ", dq, qt.grad.numpy(), out=out)
        _cmp(f"mask {name} dK", dk, kt.grad.numpy(), out=out)
        _cmp(f"mask {name} dV", dv, vt.grad.numpy(), out=out)
        with torch.no_grad():
            s = scale * torch.from_numpy(q).double() @ torch.from_numpy(k).double() \
                .repeat_interleave(G, dim=1).transpose(-1, -2)
            if tm.dtype == torch.bool:
                s = s.masked_fill(~tm, float("-inf"))
            else:
                s = s + tm
            lt = torch.logsumexp(s, dim=-1).numpy()
        _cmp(f"mask {name} L", lse, lt, out=out)
    # the hidden row of the [ql, kl] bool mask: O = 0, L = -inf, dQ = 0 in every batch and head
    dm = oracle.dense_mask(m_2d, (B, H, ql, kl))
    o, lse = oracle.fwd(q, k, v, dm, scale=scale, causal=False)
    dq, _, _ = oracle.bwd(q, k, v, dm, do, scale=scale, causal=False)
    if not (np.all(o[:, :, 3] == 0) and np.all(np.isneginf(lse[:, :, 3])) and np.all(dq[:, :, 3] == 0)):
        out.append("mask: a row hidden by the bool mask must give O = 0, L = -inf, dQ = 0")
    return out


ALL_PINS = [
    pin_fwd_vs_torch_cpu_flash,
    pin_bwd_vs_torch_autograd,
    pin_bwd_vs_finite_differences,
    pin_closed_forms,
    pin_causal_structure,
    pin_gqa_equals_repeated_mha,
    pin_bwd_invariants,
    pin_base2_mode_agrees,
    pin_window_vs_torch,
    pin_window_closed_forms,
    pin_sinks_vs_torch,
    pin_sinks_closed_forms,
    pin_value_dim_vs_torch,
    pin_value_dim_identity,
    pin_paged_vs_torch,
    pin_paged_layout_invariance,
    pin_paged_bwd_vs_torch_autograd,
    pin_paged_bwd_vs_finite_differences,
    pin_varlen_vs_torch,
    pin_mask_forms_vs_torch,
]

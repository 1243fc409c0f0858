"""Guard bands around every output: the kernels must write exactly their outputs.

Each output (O, L, dQ, dK, dV, dsinks; the packed tensors of a variable-length batch; the
paged attention's O and L and its gradients dQ, dK cache, dV cache) is placed in the middle of
a larger device buffer whose two guard bands of 4096 elements hold a sentinel bit pattern.
After ragged tiles, ql > kl, windows, masks, sinks, a value head dim below the q/k one, the
deterministic backward, packed sequences, outputs written as transposed views and paged
calls, the guard bands must hold the sentinel bit for bit (nothing was
written outside an output), and no sentinel may be left inside (every output element was
written). The guarded results must also equal the same calls on plain allocations: bit for bit
for O, L, dK, dV (their order of operations is fixed) and within the gradient tolerance for dQ,
whose f32 accumulation order varies.
"""
import zlib

import numpy as np
import pytest

import fa_inputs
from tests import parity

pytestmark = pytest.mark.gpu

GUARD = 4096
PAT16 = 0x5A5A          # bf16 ~1.5e16: not a value any output here can take
PAT32 = 0x5A5A5A5A      # f32 ~1.5e16


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import flash_attention_gb300 as fa

    fa.build()
    fa.fa_device_status(True)
    yield
    assert fa.fa_device_status(True) == fa.FA_OK


class Guarded:
    """An output tensor of `shape` inside a sentinel-filled buffer (guard bands on both sides)."""

    def __init__(self, shape, dtype):
        import torch

        self.n = int(np.prod(shape))
        self.dtype = dtype
        self.buf = torch.empty(self.n + 2 * GUARD, dtype=dtype, device="cuda")
        self.bits().fill_(self.pat())
        self.t = self.buf[GUARD:GUARD + self.n].view(shape)

    def pat(self):
        import torch

        return PAT16 if self.dtype == torch.bfloat16 else PAT32

    def bits(self):
        import torch

        return self.buf.view(torch.int16 if self.dtype == torch.bfloat16 else torch.int32)

    def check(self, name):
        b = self.bits().cpu().numpy()
        pat = np.array(self.pat()).astype(b.dtype)
        lo, mid, hi = b[:GUARD], b[GUARD:GUARD + self.n], b[GUARD + self.n:]
        assert (lo == pat).all(), f"{name}: written before the output ({int((lo != pat).sum())})"
        assert (hi == pat).all(), f"{name}: written after the output ({int((hi != pat).sum())})"
        assert not (mid == pat).any(), f"{name}: {int((mid == pat).sum())} elements not written"


def _grad_close(a, b, name):
    a = a.float().cpu().numpy().astype(np.float64)
    b = b.float().cpu().numpy().astype(np.float64)
    parity.check_grad(a, b, name, "guarded vs plain")


CASES = [
    # (B, H, Hk, ql, kl, d, dv, causal, window, mask form, sinks, deterministic)
    (1, 4, 2, 77, 330, 128, 128, True, None, None, False, False),
    (2, 2, 2, 200, 77, 128, 128, True, None, None, False, False),
    (1, 2, 1, 100, 77, 64, 64, False, None, "f32", False, False),
    (1, 2, 1, 65, 330, 256, 256, True, None, None, False, False),
    (1, 4, 2, 150, 190, 128, 128, True, (40, -1), "bf16_h1", True, False),
    (1, 4, 2, 300, 250, 128, 128, True, None, None, True, True),
    (1, 4, 2, 130, 170, 128, 64, False, (30, 20), "bool_2d", False, False),
    (2, 4, 4, 129, 129, 64, 64, True, None, None, False, True),
]


def _ids(c):
    return (f"d{c[5]}v{c[6]}_{c[3]}x{c[4]}_causal{int(c[7])}_win{c[8]}_mask{c[9]}"
            f"_sinks{int(c[10])}_det{int(c[11])}")


@pytest.mark.parametrize("case", CASES, ids=_ids)
def test_outputs_stay_inside_their_buffers(case):
    import torch

    import flash_attention_gb300 as fa

    B, H, Hk, ql, kl, d, dv, causal, window, mform, with_sinks, det = case
    g = torch.Generator(device="cpu").manual_seed(zlib.crc32(repr(case).encode()))

    def rnd(*shape, std=1.0):
        return (torch.randn(*shape, generator=g) * std).to(torch.bfloat16).cuda()

    q, k, v = rnd(B, H, ql, d), rnd(B, Hk, kl, d), rnd(B, Hk, kl, dv)
    do = rnd(B, H, ql, dv, std=0.1)
    mask = None
    if mform == "f32":
        mask = (torch.rand(B, H, ql, kl, generator=g) * -2).cuda()
    elif mform == "bf16_h1":
        mask = (torch.rand(B, 1, ql, kl, generator=g) * -2).to(torch.bfloat16).cuda()
    elif mform == "bool_2d":
        mask = (torch.rand(ql, kl, generator=g) > 0.2).cuda()
    sinks = torch.randn(H, generator=g).cuda() if with_sinks else None
    scale = d ** -0.5
    params = fa.make_params(q, k, scale=scale, causal=causal)

    o, lse = Guarded((B, H, ql, dv), torch.bfloat16), Guarded((B, H, ql), torch.float32)
    dq, dk, dvg = (Guarded(tuple(t.shape), torch.bfloat16) for t in (q, k, v))
    dsinks = Guarded((H,), torch.float32) if with_sinks else None
    fa.fa_train_fwd_ex(q, k, v, mask, o.t, lse.t, params,
                       fa.make_options(q, k, mask, window, v=v, sinks=sinks))
    fa.fa_train_bwd_ex(q, k, v, o.t, lse.t, do, mask, dq.t, dk.t, dvg.t, params,
                       fa.make_options(q, k, mask, window, v=v, sinks=sinks,
                                       dsinks=None if dsinks is None else dsinks.t,
                                       deterministic=det))
    torch.cuda.synchronize()
    assert fa.fa_device_status(True) == fa.FA_OK
    for name, gd in (("O", o), ("L", lse), ("dQ", dq), ("dK", dk), ("dV", dvg)):
        gd.check(name)
    if dsinks is not None:
        dsinks.check("dsinks")

    o2, lse2 = fa.attention_fwd(q, k, v, scale=scale, causal=causal, mask=mask, window=window,
                                sinks=sinks)
    g2 = fa.attention_bwd(q, k, v, o2, lse2, do, scale=scale, causal=causal, mask=mask,
                          window=window, sinks=sinks, deterministic=det)
    torch.cuda.synchronize()
    assert torch.equal(o.t, o2) and torch.equal(lse.t, lse2)
    assert torch.equal(dk.t, g2[1]) and torch.equal(dvg.t, g2[2])
    if det:
        assert torch.equal(dq.t, g2[0])
    else:
        _grad_close(dq.t, g2[0], "dq")
    if dsinks is not None:
        assert torch.equal(dsinks.t, g2[3])


@pytest.mark.parametrize("d", [64, 128])
def test_packed_sequences_stay_inside_their_buffers(d):
    import torch

    import flash_attention_gb300 as fa

    w = fa_inputs.VarlenWorkload("canary_varlen", 4, 2, d, (5, 130, 0, 77), (9, 130, 40, 200),
                                 True, do_std=0.1)
    x = fa_inputs.make_varlen_inputs(w, index=61)

    def bf(bits):
        return torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).cuda()

    q, k, v, do = bf(x.q), bf(x.k), bf(x.v), bf(x.do)
    cu_q, cu_k = torch.from_numpy(x.cu_q).cuda(), torch.from_numpy(x.cu_k).cuda()
    mq, mk = max(w.q_lens), max(w.k_lens)
    params, opt = fa.varlen_params_options(q, k, v, cu_q, cu_k, mq, mk, scale=w.scale,
                                           causal=True)
    o, lse = Guarded(tuple(q.shape), torch.bfloat16), Guarded(tuple(q.shape[:2]), torch.float32)
    dq, dk, dv = (Guarded(tuple(t.shape), torch.bfloat16) for t in (q, k, v))
    fa.fa_train_fwd_ex(q, k, v, None, o.t, lse.t, params, opt)
    fa.fa_train_bwd_ex(q, k, v, o.t, lse.t, do, None, dq.t, dk.t, dv.t, params, opt)
    torch.cuda.synchronize()
    assert fa.fa_device_status(True) == fa.FA_OK
    for name, gd in (("O", o), ("L", lse), ("dQ", dq), ("dK", dk), ("dV", dv)):
        gd.check(name)
    o2, lse2 = fa.varlen_attention_fwd(q, k, v, cu_q, cu_k, mq, mk, scale=w.scale, causal=True)
    g2 = fa.varlen_attention_bwd(q, k, v, o2, lse2, do, cu_q, cu_k, mq, mk, scale=w.scale,
                                 causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o.t, o2) and torch.equal(lse.t, lse2)
    assert torch.equal(dk.t, g2[1]) and torch.equal(dv.t, g2[2])
    _grad_close(dq.t, g2[0], "dq")


@pytest.mark.parametrize("q_len,splits", [(1, 0), (4, 3)])
def test_paged_outputs_stay_inside_their_buffers(q_len, splits):
    import torch

    import flash_attention_gb300 as fa

    w = fa_inputs.DecodeWorkload("canary_paged", 3, 8, 2, q_len, 128, 16, 1, 300,
                                 lengths=(1, 77, 300))
    x = fa_inputs.make_paged_inputs(w, index=62)

    def bf(bits):
        return torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).cuda()

    q, kc, vc = bf(x.q), bf(x.k_cache), bf(x.v_cache)
    table = torch.from_numpy(x.block_table).cuda()
    lens = torch.from_numpy(x.lengths).cuda()
    B, H, lq, d = q.shape
    P, Hk, bs, _ = kc.shape
    params = fa.FaPagedParams(B, H, Hk, lq, d, bs, table.shape[1], P, d ** -0.5, 1, splits, 0)
    o, lse = Guarded(tuple(q.shape), torch.bfloat16), Guarded((B, H, lq), torch.float32)
    fa.fa_paged_attention(q, kc, vc, table, lens, o.t, lse.t, params)
    torch.cuda.synchronize()
    assert fa.fa_device_status(True) == fa.FA_OK
    o.check("O")
    lse.check("L")
    o2, lse2 = fa.paged_attention(q, kc, vc, table, lens, scale=d ** -0.5, causal=True,
                                  num_splits=splits)
    torch.cuda.synchronize()
    assert torch.equal(o.t, o2) and torch.equal(lse.t, lse2)
    # the gradients through the cache: dQ and both cache gradients
    do = bf(fa_inputs.normal_bf16(4000 + q_len, tuple(q.shape)))
    dq = Guarded(tuple(q.shape), torch.bfloat16)
    dkc, dvc = Guarded(tuple(kc.shape), torch.bfloat16), Guarded(tuple(vc.shape), torch.bfloat16)
    fa.fa_paged_attention_bwd(q, kc, vc, table, lens, o.t, lse.t, do, dq.t, dkc.t, dvc.t, params)
    torch.cuda.synchronize()
    assert fa.fa_device_status(True) == fa.FA_OK
    for name, gd in (("dQ", dq), ("dK cache", dkc), ("dV cache", dvc)):
        gd.check(name)
    g2 = fa.paged_attention_bwd(q, kc, vc, table, lens, o2, lse2, do, scale=d ** -0.5,
                                causal=True)
    torch.cuda.synchronize()
    assert torch.equal(dkc.t, g2[1]) and torch.equal(dvc.t, g2[2])
    _grad_close(dq.t, g2[0], "dq")


@pytest.mark.parametrize("layout", [1, 2, 3], ids=["q_side", "kv_side", "both"])
def test_transposed_views_stay_inside_their_buffers(layout):
    """Outputs written as [B, seq, heads, dim] memory (transposed views) stay in their buffers."""
    import torch

    import flash_attention_gb300 as fa

    B, H, Hk, ql, kl, d = 2, 4, 2, 130, 190, 128
    g = torch.Generator(device="cpu").manual_seed(77 + layout)

    def rnd(*shape, bshd, std=1.0):  # logical [B, heads, rows, d]
        t = (torch.randn(*shape, generator=g) * std).to(torch.bfloat16).cuda()
        return t.transpose(1, 2).contiguous().transpose(1, 2) if bshd else t

    qs, ks = bool(layout & 1), bool(layout & 2)
    q, do = rnd(B, H, ql, d, bshd=qs), rnd(B, H, ql, d, bshd=qs, std=0.1)
    k, v = rnd(B, Hk, kl, d, bshd=ks), rnd(B, Hk, kl, d, bshd=ks)

    def out(shape, bshd):  # a guarded output with the layout of its side
        if not bshd:
            return Guarded(shape, torch.bfloat16), lambda gd: gd.t
        b_, h_, r_, d_ = shape
        return Guarded((b_, r_, h_, d_), torch.bfloat16), lambda gd: gd.t.transpose(1, 2)

    params = fa.make_params(q, k, scale=d ** -0.5, causal=True)
    (o, ov), lse = out((B, H, ql, d), qs), Guarded((B, H, ql), torch.float32)
    (dq, dqv), (dk, dkv), (dv, dvv) = out((B, H, ql, d), qs), out((B, Hk, kl, d), ks), \
        out((B, Hk, kl, d), ks)
    opt = fa.make_options(q, k, v=v)
    fa.fa_train_fwd_ex(q, k, v, None, ov(o), lse.t, params, opt)
    fa.fa_train_bwd_ex(q, k, v, ov(o), lse.t, do, None, dqv(dq), dkv(dk), dvv(dv), params, opt)
    torch.cuda.synchronize()
    assert fa.fa_device_status(True) == fa.FA_OK
    for name, gd in (("O", o), ("L", lse), ("dQ", dq), ("dK", dk), ("dV", dv)):
        gd.check(name)

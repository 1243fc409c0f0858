"""Gradients through the paged cache on the GPU (fa_paged_attention_bwd) against the CPU oracle
(oracle.paged_bwd), for the shapes of page "nuvec-core tests/fast.rs",
`paged_attention_equals_contiguous_attention` ("paged grads"): decode and causal multi-query
steps, GQA, head dims 64 / 128 / 256, page sizes 8 to 64, short and long (two-pass) caches,
a non-causal multi-query step and 8 query heads per kv head.

The caches hold the keys in shuffled pages with three pages nobody uses. Every slot that holds
no key is NaN, so a read outside the keys would show. dQ and both cache gradients are compared
element by element at the gradient tolerance of tests/parity.py. Slots that no sequence reads
must come back exactly 0. A page named by two sequences must be reported as FA_ERR_BAD_INPUT.
"""
import numpy as np
import pytest

import fa_inputs
import oracle
from tests import parity

pytestmark = pytest.mark.gpu

# (batch, query heads, kv heads, queries, head dim, page size, lengths)
CASES = [
    (1, 4, 4, 1, 128, 16, (37,)),
    (3, 8, 2, 1, 128, 32, (1, 64, 300)),
    (2, 4, 1, 4, 64, 16, (4, 77)),
    (2, 2, 2, 1, 256, 8, (9, 513)),
    (2, 8, 2, 1, 128, 32, (1500, 3000)),
    (1, 8, 2, 4, 128, 64, (2100,)),
    (1, 4, 2, 1, 256, 16, (1100,)),
    (3, 4, 2, 3, 128, 16, (0, 2, 40)),  # an empty sequence and one shorter than q_len
    (2, 4, 2, 3, 128, 16, (30, 77), False),  # no causal rule: the query heads packed as rows
    (2, 16, 2, 1, 64, 8, (104, 64)),  # 8 query heads per kv head; a sequence at capacity
    (2, 8, 2, 2, 256, 16, (40, 900)),  # 8 rows per kv head at head dim 256 (causal, 2 queries)
    (2, 4, 1, 1, 64, 16, (700, 33)),   # 4 rows per kv head at head dim 64, several key blocks
]


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


def _problem(n, case, shared=False):
    B, H, Hk, lq, d, bs, lens = case[:7]
    causal = case[7] if len(case) > 7 else lq > 1
    per = max(1, max(-(-L // bs) for L in lens))
    P = B * per + 3
    rng = np.random.default_rng(2100 + n)
    table = rng.permutation(P)[:B * per].reshape(B, per).astype(np.int32)
    if shared:
        table[1, 0] = table[0, 0]
    base = 3000 + 8 * n
    q = fa_inputs.normal_bf16(base, (B, H, lq, d))
    kc = fa_inputs.normal_bf16(base + 1, (P, Hk, bs, d))
    vc = fa_inputs.normal_bf16(base + 2, (P, Hk, bs, d))
    do = fa_inputs.normal_bf16(base + 3, (B, H, lq, d))
    nan = np.array([0x7FC0], np.uint16)[0]  # bf16 NaN
    used = np.zeros((P, bs), bool)
    for b, L in enumerate(lens):
        j = np.arange(L)
        used[table[b, j // bs], j % bs] = True
    for c in (kc, vc):
        c.transpose(0, 2, 1, 3)[~used] = nan  # [P, bs, Hk, d] view: every head of the slot
    return dict(B=B, H=H, Hk=Hk, lq=lq, d=d, bs=bs, P=P, lens=np.asarray(lens, np.int32),
                table=table, q=q, kc=kc, vc=vc, do=do, used=used, causal=causal,
                scale=d ** -0.5)


def _run(x):
    import torch

    import flash_attention_gb300 as fa

    def bf(bits):
        return torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).cuda()

    q, kc, vc, do = bf(x["q"]), bf(x["kc"]), bf(x["vc"]), bf(x["do"])
    table = torch.from_numpy(x["table"]).cuda()
    lens = torch.from_numpy(x["lens"]).cuda()
    o, lse = fa.paged_attention(q, kc, vc, table, lens, scale=x["scale"], causal=x["causal"])
    dq, dk, dv = fa.paged_attention_bwd(q, kc, vc, table, lens, o, lse, do, scale=x["scale"],
                                        causal=x["causal"])
    torch.cuda.synchronize()
    return dq, dk, dv


@pytest.mark.parametrize("n", range(len(CASES)), ids=[str(c[:6] + (c[6][:2],) + c[7:]) for c in CASES])
def test_paged_gradients_match_oracle(n):
    import flash_attention_gb300 as fa

    x = _problem(n, CASES[n])
    dq, dk, dv = _run(x)
    assert fa.fa_device_status(True) == fa.FA_OK
    w = fa_inputs.bf16_bits_to_f32
    ref = oracle.paged_bwd(w(x["q"]), np.nan_to_num(w(x["kc"])), np.nan_to_num(w(x["vc"])),
                           x["table"], x["lens"], w(x["do"]), scale=x["scale"],
                           causal=x["causal"])
    got = [t.float().cpu().numpy().astype(np.float64) for t in (dq, dk, dv)]
    stats = {}
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        assert np.isfinite(g).all(), f"{name} has non-finite values"
        stats.update(parity.check_grad(g, r, name, f"paged case {n}"))
    # slots no sequence reads: exactly zero
    for name, g in (("dk", got[1]), ("dv", got[2])):
        assert (g[~x["used"][:, None, :].repeat(x["Hk"], 1)] == 0).all(), \
            f"{name}: a slot nobody reads got a gradient"
    print(CASES[n], stats)


def test_shared_page_is_reported():
    import flash_attention_gb300 as fa

    x = _problem(90, (2, 4, 2, 1, 128, 16, (40, 40)), shared=True)
    _run(x)
    assert fa.fa_device_status(True) == fa.FA_ERR_BAD_INPUT


@pytest.mark.parametrize("lq", [1, 4], ids=["decode_path", "packed_path"])
def test_table_entry_outside_the_cache_is_reported(lq):
    """A used table entry past the cache reads as zero keys in both passes, writes no gradient
    outside the caches and makes fa_device_status return FA_ERR_BAD_INPUT; the outputs stay
    finite."""
    import torch

    import flash_attention_gb300 as fa

    x = _problem(91, (2, 8, 2, lq, 128, 16, (40, 40)))
    x["table"][1, 1] = x["P"] + 5  # (slot 1 holds keys 16 .. 31 of sequence 1)
    dq, dk, dv = _run(x)
    assert fa.fa_device_status(True) == fa.FA_ERR_BAD_INPUT
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        assert torch.isfinite(t.float()).all(), name

"""Paged key/value cache attention on the GPU against the CPU oracle: the case list of the
nuvec-core paged-attention test (decode and several queries, page sizes 8 to 64, one and two
passes), forced split counts, unused cache slots holding NaN, and lengths or table entries out
of range (clamped or read as zeros, and reported by fa_device_status, never a fault).
Tolerances: O and L as in tests/parity.py."""
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


def D(name, B, H, Hk, lq, d, bs, lengths, causal=True):
    return fa_inputs.DecodeWorkload(name, B, H, Hk, lq, d, bs, min(lengths), max(lengths),
                                    causal, lengths=tuple(lengths))


CASES = [
    D("b1_h4_d128_bs16", 1, 4, 4, 1, 128, 16, [37]),
    D("b3_gqa4_d128_bs32", 3, 8, 2, 1, 128, 32, [1, 64, 300]),
    D("b2_lq4_d64_bs16", 2, 4, 1, 4, 64, 16, [4, 77]),
    D("b2_d256_bs8", 2, 2, 2, 1, 256, 8, [9, 513]),
    D("long_two_pass", 2, 8, 2, 1, 128, 32, [1500, 3000]),
    D("long_lq4_bs64", 1, 8, 2, 4, 128, 64, [2100]),
    D("long_d256_bs16", 1, 4, 2, 1, 256, 16, [1100]),
    D("noncausal_lq3", 2, 4, 2, 3, 128, 16, [40, 200], causal=False),
    D("lq_gt_len", 2, 4, 2, 6, 64, 8, [3, 50]),           # queries that see no key
    D("empty_sequence", 2, 4, 2, 1, 128, 16, [0, 90]),
    D("bs128", 1, 8, 1, 2, 128, 128, [700]),
]


def to_dev(x):
    import torch

    def bf(bits):
        return torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).cuda()

    return (bf(x.q), bf(x.k_cache), bf(x.v_cache), torch.from_numpy(x.block_table).cuda(),
            torch.from_numpy(x.lengths).cuda())


def run(w, x, num_splits=0):
    import torch

    import flash_attention_gb300 as fa

    q, kc, vc, tb, ln = to_dev(x)
    o, lse = fa.paged_attention(q, kc, vc, tb, ln, scale=w.scale, causal=w.causal,
                                num_splits=num_splits)
    torch.cuda.synchronize()
    return o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


def reference(w, x):
    q, kc, vc = x.widened()
    return oracle.paged_fwd(q, kc, vc, x.block_table, x.lengths, scale=w.scale, causal=w.causal)


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_paged_matches_oracle(w):
    import flash_attention_gb300 as fa

    x = fa_inputs.make_paged_inputs(w, index=90 + CASES.index(w))
    o, lse = run(w, x)
    assert fa.fa_device_status(True) == fa.FA_OK
    o_r, l_r = reference(w, x)
    stats = {}
    stats.update(parity.check_o(o, o_r, w.name))
    stats.update(parity.check_l(lse, l_r, w.name))
    dead = np.isneginf(l_r)
    assert (o[dead] == 0).all()
    print(w.name, stats)


@pytest.mark.parametrize("splits", [1, 2, 3, 7, 40])
def test_paged_forced_splits(splits):
    import flash_attention_gb300 as fa

    w = D("splits", 2, 8, 2, 2, 128, 16, [900, 2500])
    x = fa_inputs.make_paged_inputs(w, index=120)
    o, lse = run(w, x, num_splits=splits)
    assert fa.fa_device_status(True) == fa.FA_OK
    o_r, l_r = reference(w, x)
    parity.check_o(o, o_r, f"splits={splits}")
    parity.check_l(lse, l_r, f"splits={splits}")


def test_paged_out_of_range_inputs_are_flagged_not_faulted():
    import torch

    import flash_attention_gb300 as fa

    w = D("bad", 2, 4, 2, 1, 128, 16, [50, 100])
    x = fa_inputs.make_paged_inputs(w, index=121)
    q, kc, vc, tb, ln = to_dev(x)
    # a length past the table's capacity is clamped to it
    ln_bad = ln.clone()
    ln_bad[0] = w.max_pages * w.page_size + 500
    fa.paged_attention(q, kc, vc, tb, ln_bad, scale=w.scale, causal=True)
    assert fa.fa_device_status(True) == fa.FA_ERR_BAD_INPUT
    # a table entry outside the cache reads as zero keys and values
    tb_bad = tb.clone()
    tb_bad[1, 0] = kc.shape[0] + 7
    tb_bad[1, 1] = -3
    o, _ = fa.paged_attention(q, kc, vc, tb_bad, ln, scale=w.scale, causal=True)
    torch.cuda.synchronize()
    assert fa.fa_device_status(True) == fa.FA_ERR_BAD_INPUT
    assert torch.isfinite(o.float()).all()
    # and a clean call afterwards is clean again
    fa.paged_attention(q, kc, vc, tb, ln, scale=w.scale, causal=True)
    assert fa.fa_device_status(True) == fa.FA_OK


def test_paged_decode_full_size_sampled():
    """The benchmark's decode workload at full size, checked on a sample of sequences."""
    import flash_attention_gb300 as fa

    w = fa_inputs.DECODE_BY_NAME["paged_decode_d128"]
    x = fa_inputs.make_paged_inputs(w)
    o, lse = run(w, x)
    assert fa.fa_device_status(True) == fa.FA_OK
    q, kc, vc = x.widened()
    for b in (0, w.batch // 2, w.batch - 1):
        sub = fa_inputs.PagedInputs(x.q[b:b + 1], x.k_cache, x.v_cache, x.block_table[b:b + 1],
                                    x.lengths[b:b + 1])
        o_r, l_r = oracle.paged_fwd(q[b:b + 1], kc, vc, sub.block_table, sub.lengths,
                                    scale=w.scale, causal=w.causal)
        parity.check_o(o[b:b + 1], o_r, f"{w.name} seq {b}")
        parity.check_l(lse[b:b + 1], l_r, f"{w.name} seq {b}")

"""Host-side workload bookkeeping: visible (query, key) pair counts and the FLOP rule."""
import itertools

import pytest

import fa_inputs


def brute_visible(w):
    off = w.kl - w.ql
    n = 0
    for i, j in itertools.product(range(w.ql), range(w.kl)):
        qa = off + i
        if w.causal and j > qa:
            continue
        if w.window_left >= 0 and j < qa - w.window_left:
            continue
        if w.window_right >= 0 and j > qa + w.window_right:
            continue
        n += 1
    return n


SHAPES = [(17, 17), (9, 30), (30, 9), (1, 40), (40, 1)]
WINDOWS = [(-1, -1), (0, -1), (3, -1), (-1, 0), (-1, 4), (2, 5), (0, 0), (100, 100)]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("ql,kl", SHAPES)
@pytest.mark.parametrize("wl,wr", WINDOWS)
def test_visible_pairs_brute_force(causal, ql, kl, wl, wr):
    w = fa_inputs.Workload("t", 1, 1, 1, ql, kl, 64, 0.125, causal, window_left=wl,
                           window_right=wr)
    assert w.visible_pairs() == brute_visible(w)


def test_flop_rule():
    w = fa_inputs.BY_NAME["gqa_d128_4k"]
    base = w.batch * w.n_heads * w.ql * w.kl * w.head_dim
    assert w.flops() == (4.0 * base * 0.5, 10.0 * base * 0.5)  # causal counted as half
    s = fa_inputs.BY_NAME["swa_d128_16k"]
    # a window has no halving rule: the exact visible fraction is counted
    assert s.flops() == s.flops(exact=True)
    rows_full = s.kl - s.window_left  # rows that see a full 4096-key window
    pairs = rows_full * (s.window_left + 1) + sum(range(1, s.window_left + 1))
    assert s.visible_pairs() == pairs


def test_existing_seeds_unchanged():
    # appending workloads must not move the seeds of the existing ones
    names = [w.name for w in fa_inputs.WORKLOADS[:5]]
    assert names == ["tiny_gqa_d64", "masked_d256", "train_d64", "gqa_d128_4k", "rect_d256"]


def test_exp2_bound_binds_the_d64_forward_only():
    """The secondary (exp2 on MUFU) bound: at head_dim 64 the forward's exponentials outweigh its
    tensor work, at 128 the tensor work dominates, and the backward (2.5x the forward's FLOPs
    for the same exponentials) stays tensor-bound."""
    import bench

    peak, n_sm, mhz = 1945.3, 152, 2070.0
    d64 = bench.kernel_bounds(fa_inputs.BY_NAME["train_d64"], peak, n_sm, mhz)["kernels"]
    d128 = bench.kernel_bounds(fa_inputs.BY_NAME["gqa_d128_4k"], peak, n_sm, mhz)["kernels"]
    assert d64["fwd_kernel"]["binds"] == "exp2"
    assert d64["bwd_main_kernel"]["binds"] == "tensor"
    assert d128["fwd_kernel"]["binds"] == "tensor" and d128["bwd_main_kernel"]["binds"] == "tensor"
    # one exponential per visible pair: B*H*ql*kl/2 for causal
    w = fa_inputs.BY_NAME["gqa_d128_4k"]
    assert bench.kernel_exps(w)["fwd_kernel"] == w.batch * w.n_heads * w.ql * w.kl * 0.5
    exp_us = d128["fwd_kernel"]["exp2_mufu_us"]
    assert abs(exp_us - w.batch * w.n_heads * w.ql * w.kl * 0.5 / (16 * n_sm * mhz * 1e6) * 1e6) < 1e-6


def test_source_hash_ignores_comments_only():
    """A recorded capture stays valid across comment edits and is voided by code edits."""
    import bench

    code = "int f(int x) {  // doubles\n  /* the\n  body */ return 2 * x;\n}\n"
    assert bench.code_only(code) == bench.code_only(code.replace("doubles", "twice x"))
    assert bench.code_only(code) == bench.code_only(code + "\n\n// trailing note\n")
    assert bench.code_only(code) != bench.code_only(code.replace("2 * x", "3 * x"))


def test_reference_arm_json_line():
    """`bench.py --impl reference` (the CPU oracle arm, runnable without a GPU) prints one JSON
    line with the contract's keys."""
    import json
    import os
    import subprocess
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0", "--workload", "tiny_gqa_d64"],
                       capture_output=True, text=True, timeout=300, cwd=root)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["config"]["workload"] == "tiny_gqa_d64"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


def test_paged_grad_bytes_and_oracle_sample():
    """The paged-gradient bench counts: brute-force byte counts on a small cache, and the
    oracle sample (forward + gradients per sequence on its own pages) covers whole sequences
    and matches the oracle on the full cache for the first one."""
    import os
    import sys

    import numpy as np

    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    import oracle

    w = fa_inputs.DecodeWorkload("tiny_paged_grad", 3, 4, 2, 1, 64, 8, 5, 30)
    x = fa_inputs.make_paged_inputs(w, index=7)
    step, per = bench.paged_grad_bytes(w, x)
    el = 64 * 2
    used_keys = sum(int(n) for n in x.lengths)
    qb = 3 * 4 * 1 * el
    cache = x.k_cache.size * 2
    # 2 query rows per kv head: the decode path
    assert per["paged_decode_bwd_kernel"] == 4 * used_keys * 2 * el + 3 * qb
    assert per["paged_scatter_kernel"] == 2 * (cache - used_keys * 2 * el) + 3 * qb
    assert step == bench.paged_bytes(w, x) + 4 * qb + 2 * used_keys * 2 * el + 2 * cache
    wide = fa_inputs.DecodeWorkload("tiny_paged_grad_wide", 3, 8, 2, 3, 64, 8, 5, 30)
    xw = fa_inputs.make_paged_inputs(wide, index=8)
    _, perw = bench.paged_grad_bytes(wide, xw)
    used_w = sum(int(n) for n in xw.lengths) * 2 * el
    qw = 3 * 8 * 3 * el
    assert perw["bwd_main_kernel"] == 4 * used_w + 2 * qw
    assert perw["paged_scatter_kernel"] == 2 * used_w + 2 * xw.k_cache.size * 2 + 2 * qw

    do = fa_inputs.normal_bf16(5, tuple(x.q.shape), 0.1)
    b_, s_, n_ = bench.paged_grad_oracle_sample(w, x, do, step, budget_s=1e-9)
    assert n_ == 1 and 0 < b_ < step and s_ > 0
    # the per-sequence copy of its own pages gives the full cache's gradients
    q, kc, vc = x.widened()
    dof = fa_inputs.bf16_bits_to_f32(do)
    L = int(x.lengths[0])
    pages = x.block_table[0, :-(-L // 8)]
    sub = oracle.paged_bwd(q[:1], kc[pages], vc[pages], np.arange(len(pages))[None],
                           x.lengths[:1], dof[:1], scale=w.scale, causal=True)
    full = oracle.paged_bwd(q[:1], np.nan_to_num(kc), np.nan_to_num(vc), x.block_table[:1],
                            x.lengths[:1], dof[:1], scale=w.scale, causal=True)
    np.testing.assert_allclose(sub[0], full[0], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(np.nan_to_num(sub[1]), full[1][pages], rtol=1e-12, atol=1e-14)

"""The FMA-pipe exp2 that takes a share of the softmax's exponentials (`ex2_poly` in
flash_attention_gb300/csrc/fa_common.cuh): Cody-Waite reduction x = n + f with n = round(x),
f in [-0.5, 0.5], a degree-3 polynomial for 2^f, and 2^n added to the exponent field.

CPU: the committed coefficients, read from the source, against 2^f in f64 on [-0.5, 0.5], and
the whole function emulated step by step in f32 over the arguments the softmax can produce
(base-2 scores minus a running maximum that may lag the true one by up to 8: [-126, 8]); the
stated bound is a relative error of 7.5e-5 wherever the result is a normal float (x >= -125),
far below the 2^-9 half-ulp of the bf16 P it feeds; on [-126, -125) the result may fall into
the denormal encoding, where only an absolute error below 2^-138 is claimed (such a p is added
to a row sum of at least 1, and rounds to 0 in bf16).
GPU: the device function itself, through the test entry point fa_debug_ex2, against CUDA's
exp2f on a dense grid over the same range.
"""
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "flash_attention_gb300", "csrc", "fa_common.cuh")
BOUND = 7.5e-5


def _coefficients():
    text = open(SRC).read()
    body = text[text.index("float ex2_poly(float x)"):]
    m = re.search(r"c0 = ([0-9.eE+-]+)f, c1 = ([0-9.eE+-]+)f, c2 = ([0-9.eE+-]+)f, "
                  r"c3 = ([0-9.eE+-]+)f;", body)
    assert m, "coefficients of ex2_poly not found"
    return [np.float32(float(c)) for c in m.groups()]


def _emulate(x):
    """ex2_poly step by step in f32 (numpy); the FMAs are evaluated in f64 and rounded once."""
    c0, c1, c2, c3 = _coefficients()
    x = np.asarray(x, np.float32)
    magic = np.float32(12582912.0)
    xc = np.maximum(x, np.float32(-126.0))
    t = (xc + magic).astype(np.float32)
    n = (t - magic).astype(np.float32)
    f = (xc - n).astype(np.float32)

    def fma(a, b, c):
        return (a.astype(np.float64) * b.astype(np.float64) + np.float64(c)).astype(np.float32)

    p = fma(fma(fma(np.full_like(f, c3), f, c2), f, c1), f, c0)
    e = (t.view(np.int32).astype(np.int64) << 23).astype(np.int64) & 0xFFFFFFFF
    r = ((p.view(np.int32).astype(np.int64) + e) & 0xFFFFFFFF).astype(np.uint32).view(np.float32)
    return np.where(x < np.float32(-126.0), np.float32(0.0), r)


def test_polynomial_meets_its_stated_bound():
    c0, c1, c2, c3 = (np.float64(c) for c in _coefficients())
    f = np.linspace(-0.5, 0.5, 200001)
    p = ((c3 * f + c2) * f + c1) * f + c0
    rel = np.abs(p / np.exp2(f) - 1.0)
    assert rel.max() <= BOUND, rel.max()
    # and it is a real minimax-quality fit, not a loose one: the bound is nearly attained
    assert rel.max() > 0.5 * BOUND


def test_whole_function_in_f32_over_the_softmax_range():
    x = np.concatenate([np.linspace(-126.0, 8.0, 400001, dtype=np.float32),
                        np.float32([-126.0, -125.5, -0.5, 0.5, 0.0, 8.0, -1e-7, 1e-7])])
    y = _emulate(x).astype(np.float64)
    ref = np.exp2(x.astype(np.float64))
    normal = x >= -125.0
    rel = np.abs(y[normal] / ref[normal] - 1.0)
    assert rel.max() <= BOUND + 2.0 ** -22, rel.max()
    assert np.abs(y[~normal] - ref[~normal]).max() <= 2.0 ** -138
    assert _emulate(np.float32([-127.0, -200.0, -np.inf])).tolist() == [0.0, 0.0, 0.0]


@pytest.mark.gpu
def test_device_ex2_poly_against_exp2f():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import flash_attention_gb300 as fa

    fa.build()
    x = torch.cat([torch.linspace(-126.0, 8.0, 1 << 22, dtype=torch.float32),
                   torch.tensor([-126.0, -125.5, -0.5, 0.5, 0.0, 8.0, -1e-7, 1e-7, -127.0,
                                 -1000.0, float("-inf")])]).cuda()
    y_poly, y_mufu, y_ref = (t.double().cpu().numpy() for t in fa.fa_debug_ex2(x))
    torch.cuda.synchronize()
    xs = x.double().cpu().numpy()
    live = xs >= -126.0
    normal = xs >= -125.0
    rel_poly = np.abs(y_poly[normal] / y_ref[normal] - 1.0)
    rel_mufu = np.abs(y_mufu[normal] / y_ref[normal] - 1.0)
    print(f"max relative error vs exp2f: polynomial {rel_poly.max():.3e}, "
          f"hardware approximation {rel_mufu.max():.3e}")
    assert rel_poly.max() <= BOUND + 2.0 ** -22
    assert np.abs(y_poly[live & ~normal] - y_ref[live & ~normal]).max() <= 2.0 ** -138
    assert (y_poly[~live] == 0.0).all()
    # the device function is the emulated one (FMA rounding may differ in the last bit)
    emu = _emulate(xs.astype(np.float32)).astype(np.float64)
    assert np.abs(y_poly[normal] / emu[normal] - 1.0).max() <= 2.0 ** -21

"""Local (sliding-window) attention and the extended mask forms (bool, bf16, broadcast) on the
GPU, against the CPU oracle (which sees the window through `oracle.window` and every mask as
its dense f32 additive form). Tolerances as in tests/parity.py."""
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


def _mask(kind, shape, rng):
    """A mask of the given kind for a [B, H, ql, kl] problem: (numpy array, torch dtype)."""
    import torch

    B, H, ql, kl = shape
    if kind is None:
        return None, None
    form, dtype = kind
    full = {"dense": (B, H, ql, kl), "b1": (1, H, ql, kl), "h1": (B, 1, ql, kl),
            "2d": (ql, kl)}[form]
    if dtype == "bool":
        m = rng.random(full) > 0.25
        return m, torch.bool
    m = rng.uniform(-2.0, 0.5, size=full).astype(np.float32)
    m[rng.random(full) < 0.1] = -np.inf
    if dtype == "bf16":
        m = fa_inputs.bf16_bits_to_f32(fa_inputs.f32_to_bf16_bits(m))
        return m, torch.bfloat16
    return m, torch.float32


def run_case(B, H, Hk, ql, kl, d, causal, window, mask_kind, seed):
    import torch

    import flash_attention_gb300 as fa

    w = fa_inputs.Workload("case", B, H, Hk, ql, kl, d, d ** -0.5, causal)
    inp = fa_inputs.make_inputs(w, index=20 + seed)
    rng = np.random.default_rng(seed)
    m_np, m_dtype = _mask(mask_kind, (B, H, ql, kl), rng)
    dev = parity.to_device(inp)
    m_t = None if m_np is None else torch.from_numpy(m_np).to(m_dtype).cuda()
    o, lse = fa.attention_fwd(dev["q"], dev["k"], dev["v"], scale=w.scale, causal=causal,
                              mask=m_t, window=window)
    dq, dk, dv = fa.attention_bwd(dev["q"], dev["k"], dev["v"], o, lse, dev["do"], scale=w.scale,
                                  causal=causal, mask=m_t, window=window)
    torch.cuda.synchronize()
    assert fa.fa_device_status(True) == fa.FA_OK
    gpu = {n: t.float().cpu().numpy().astype(np.float64)
           for n, t in (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv))}
    q, k, v, do = inp.widened()
    dm = oracle.dense_mask(m_np, (B, H, ql, kl))
    with oracle.window(*(window or (-1, -1))):
        o_r, l_r = oracle.fwd(q, k, v, dm, scale=w.scale, causal=causal)
        dq_r, dk_r, dv_r = oracle.bwd(q, k, v, dm, do, scale=w.scale, causal=causal)
    ref = {"o": o_r, "lse": l_r, "dq": dq_r, "dk": dk_r, "dv": dv_r}
    stats = parity.compare_full(w, gpu, ref, f"d{d} w{window} m{mask_kind}")
    dead = np.isneginf(l_r)
    if dead.any():
        assert (gpu["o"][dead] == 0).all() and (gpu["dq"][dead] == 0).all()
    return stats


CASES = [
    # (B, H, Hk, ql, kl, d, causal, window, mask)
    (1, 4, 2, 300, 300, 128, True, (100, -1), None),          # causal sliding window
    (1, 2, 1, 257, 390, 64, False, (50, 30), None),            # two-sided window, ragged
    (1, 4, 1, 200, 500, 256, True, (64, -1), None),            # rectangle, d256
    (2, 2, 2, 160, 96, 128, True, (40, -1), None),             # ql > kl: rows with no key
    (1, 2, 1, 190, 190, 64, True, (0, -1), None),              # window 0: the diagonal only
    (1, 4, 2, 200, 200, 128, False, None, ("dense", "bool")),  # bool mask
    (2, 4, 2, 130, 170, 128, True, None, ("b1", "bf16")),      # bf16 mask, shared by batches
    (2, 2, 1, 150, 150, 64, False, None, ("2d", "f32")),       # one [ql, kl] mask for all
    (2, 4, 4, 140, 260, 256, False, (90, 20), ("h1", "f32")),  # window + mask shared by heads
    (1, 2, 2, 256, 384, 128, True, (128, -1), ("dense", "bool")),
]


def _case_id(c):
    w = "none" if c[7] is None else f"{c[7][0]}_{c[7][1]}"
    m = "none" if c[8] is None else "_".join(c[8])
    return f"d{c[5]}_causal{int(c[6])}_win{w}_mask_{m}"


@pytest.mark.parametrize("idx", range(len(CASES)), ids=[_case_id(c) for c in CASES])
def test_window_and_mask_forms(idx):
    case = CASES[idx]
    stats = run_case(*case, seed=idx)
    print(case, {k: round(v, 5) if isinstance(v, float) else v for k, v in stats.items()})

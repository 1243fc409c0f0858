"""Host-side logic of the library that needs no GPU: the per-device once-only setup (kernel
attributes are per device context, so a process driving several GPUs sets them on each, from
any thread) and the bounded-wait limit the kernels receive."""
import os
import shutil
import subprocess

import pytest

import flash_attention_gb300 as fa

HERE = os.path.dirname(os.path.abspath(__file__))


def test_once_per_device_setup_logic(tmp_path):
    """fa_once.h under 16 threads and 70 keys: each key's step succeeds exactly once, a failing
    step is retried, keys outside the range run every time (tests/native/once_test.cpp)."""
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no C++ compiler")
    exe = tmp_path / "once_test"
    subprocess.run([cxx, "-O2", "-std=c++17", "-pthread", "-o", str(exe),
                    os.path.join(HERE, "native", "once_test.cpp")], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr


def test_wait_limit_setting():
    fa.build()
    default = fa.fa_get_wait_limit_ns()
    assert default == 2_000_000_000
    try:
        fa.fa_set_wait_limit_ns(5000)
        assert fa.fa_get_wait_limit_ns() == 5000
        fa.fa_set_wait_limit_ns(0)  # back to the default
        assert fa.fa_get_wait_limit_ns() == default
        with pytest.raises(fa.FaError):
            fa.fa_set_wait_limit_ns(61 * 10**9)
        assert fa.fa_get_wait_limit_ns() == default
    finally:
        fa.fa_set_wait_limit_ns(0)


def test_debug_entry_points_check_arguments():
    lib = fa.load_library()
    fake = 0x100000
    assert lib.fa_debug_ex2(fake, fake, fake, fake, -1, None) == fa.FA_ERR_INVALID
    assert lib.fa_debug_ex2(fake + 2, fake, fake, fake, 8, None) == fa.FA_ERR_INVALID
    assert lib.fa_debug_ex2(None, fake, fake, fake, 8, None) == fa.FA_ERR_INVALID
    assert lib.fa_debug_wait_timeout(fake + 4, None) == fa.FA_ERR_INVALID


def test_layout_detection_of_the_binding():
    """The binding names a tensor's memory layout for the FA_LAYOUT_* flags: contiguous
    [B, H, L, D] is 0, a transposed view of a contiguous [B, L, H, D] tensor is 1, anything else
    is refused rather than copied."""
    torch = pytest.importorskip("torch")
    t = torch.zeros(2, 4, 8, 64)
    assert fa._layout_bit(t) == 0
    assert fa._layout_bit(torch.zeros(2, 8, 4, 64).transpose(1, 2)) == 1
    assert fa._layout_bit(torch.zeros(8, 4, 64).transpose(0, 1)) == 1  # packed [total, H, D]
    with pytest.raises(ValueError):
        fa._layout_bit(t[..., ::2])  # dim not contiguous
    with pytest.raises(ValueError):
        fa._layout_bit(t.transpose(0, 1))  # [H, B, L, D] memory
    opt = fa.make_options(torch.zeros(2, 8, 4, 64).transpose(1, 2), t)
    assert opt.layout == fa.FA_LAYOUT_Q_BSHD
    opt = fa.make_options(t, torch.zeros(2, 8, 4, 64).transpose(1, 2))
    assert opt.layout == fa.FA_LAYOUT_KV_BSHD

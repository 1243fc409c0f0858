"""CPU oracle for exact training attention -- TEST INFRASTRUCTURE.

Only `tests/`, `__graft_entry__.smoke()` and the benchmark's CPU-baseline leg may import this
package. The product path (`flash_attention_gb300`) never imports, links or calls it, and the
oracle imports nothing from the product.

The arithmetic lives in `fa_oracle.c` (plain C, f64). This module compiles it with gcc and
marshals numpy arrays through ctypes. Inputs are f32 arrays that hold exact bf16 values
(`fa_inputs.bf16_bits_to_f32`); outputs are f64.

What each function computes, and the passages it follows, is written at the top of
`fa_oracle.c`.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libfa_oracle.so")
_lib = None
_lock = threading.Lock()
_active_sinks = None  # the values of the enclosing sinks(...) block

# Planted-mistake codes understood by fa_oracle_set_mutation (tests only).
MUTATIONS = {
    "no_scale": 1,
    "top_left_causal": 2,
    "gqa_modulo": 3,
    "no_normalise": 4,
    "mask_sign": 5,
    "lse_no_max": 6,
    "ds_no_d": 7,
    "dk_uses_k": 8,
    "dv_uses_ds": 9,
    "causal_off_by_one": 10,
    "dq_no_scale": 11,
    "d_from_do_only": 12,
    "window_off_by_one": 13,
    "sink_scaled": 14,
    "dsink_sign": 15,
    "v_stride_d": 16,
    "table_stride": 17,
    "decode_top_left": 18,
    "bool_mask_inverted": 19,
    "paged_grad_slot": 20,
}
# Codes above handled here in Python (the mask-form conversion, the paged gradient's slot
# mapping), not in fa_oracle.c.
_PY_MUTATION_BOOL_INVERTED = 19
_PY_MUTATION_PAGED_SLOT = 20
_py_mutation = 0


def build(force: bool = False) -> str:
    """Compile fa_oracle.c into libfa_oracle.so next to it (gcc, no fast-math, no FMA
    contraction, so that x86 and Arm give the same bits)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-ffp-contract=off",
           "-fno-fast-math", "-Wall", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            f = ctypes.c_void_p
            i = ctypes.c_int
            d = ctypes.c_double
            lib.fa_oracle_fwd_rows.argtypes = [f, f, f, f, i, i, i, i, i, i, i, d, i, f,
                                               ctypes.c_long, i, f, f, i]
            lib.fa_oracle_bwd_q_rows.argtypes = [f, f, f, f, f, i, i, i, i, i, i, i, d, i, f,
                                                 ctypes.c_long, f, i]
            lib.fa_oracle_bwd_kv_rows.argtypes = [f, f, f, f, f, i, i, i, i, i, i, i, d, i, i,
                                                  i, f, i, f, f, i]
            lib.fa_oracle_bwd.argtypes = [f, f, f, f, f, i, i, i, i, i, i, i, d, i, f, f, f, i]
            lib.fa_oracle_dsinks.argtypes = [f, f, f, f, f, i, i, i, i, i, i, i, d, i, f, i]
            lib.fa_oracle_paged_fwd.argtypes = [f, f, f, f, f, i, i, i, i, i, i, i, i, d, i, f, f,
                                                i]
            lib.fa_oracle_paged_fwd.restype = i
            lib.fa_oracle_set_mutation.argtypes = [i]
            lib.fa_oracle_set_window.argtypes = [i, i]
            lib.fa_oracle_set_sinks.argtypes = [f]
            lib.fa_oracle_get_mutation.restype = i
            for fn in (lib.fa_oracle_fwd_rows, lib.fa_oracle_bwd_q_rows,
                       lib.fa_oracle_bwd_kv_rows, lib.fa_oracle_bwd, lib.fa_oracle_dsinks):
                fn.restype = i
            _lib = lib
    return _lib


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def _f32(x):
    a = np.ascontiguousarray(x, dtype=np.float32)
    return a


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _shape(q, k, v):
    """(B, H, Hk, ql, kl, d, dv): d from q/k, dv (the value head dim) from v."""
    B, H, ql, d = q.shape
    Bk, Hk, kl, dk = k.shape
    if B != Bk or d != dk:
        raise ValueError("q and k disagree on batch or head_dim")
    if tuple(v.shape[:3]) != (B, Hk, kl):
        raise ValueError("v must be [B, Hk, kl, dv]")
    if H % Hk:
        raise ValueError("n_heads must be a multiple of n_kv_heads")
    return B, H, Hk, ql, kl, d, int(v.shape[3])


class window:
    """Context manager: local attention window (left, right) for the oracle calls inside it;
    -1 leaves a side unbounded. Key j is hidden when j < q_abs - left or j > q_abs + right,
    with q_abs = kl - ql + i."""

    def __init__(self, left=-1, right=-1):
        self.left, self.right = int(left), int(right)

    def __enter__(self):
        _load().fa_oracle_set_window(self.left, self.right)
        return self

    def __exit__(self, *exc):
        _load().fa_oracle_set_window(-1, -1)
        return False


class sinks:
    """Context manager: per-head sink logits (natural-log units, shape [H]) for the oracle calls
    inside it; None means no sinks. The row normaliser gains exp(sink_h); the sink carries no
    value."""

    def __init__(self, values):
        self.values = None if values is None else np.ascontiguousarray(values, np.float32)

    def __enter__(self):
        global _active_sinks
        _load().fa_oracle_set_sinks(_ptr(self.values))
        _active_sinks = self.values
        return self

    def __exit__(self, *exc):
        global _active_sinks
        _load().fa_oracle_set_sinks(None)
        _active_sinks = None
        return False


def dense_mask(mask, shape):
    """Any mask form the CUDA path accepts, as the oracle's dense f32 additive mask [B,H,ql,kl]:
    bool masks (True = visible) become 0 / -inf, bf16 and f32 masks their f32 values, and
    broadcast shapes ([ql,kl], [1,H,ql,kl], [B,1,ql,kl], ...) are expanded."""
    if mask is None:
        return None
    m = np.asarray(mask)
    if m.dtype == np.bool_ or m.dtype == np.uint8:
        visible = m != 0
        if _py_mutation == _PY_MUTATION_BOOL_INVERTED:
            visible = ~visible
        m = np.where(visible, np.float32(0.0), np.float32(-np.inf))
    m = np.broadcast_to(m.astype(np.float32), shape)
    return np.ascontiguousarray(m)


def set_mutation(name_or_code) -> None:
    """Plant one known mistake in the oracle (tests only); 0 or None removes it."""
    global _py_mutation
    code = MUTATIONS.get(name_or_code, name_or_code) if name_or_code else 0
    _py_mutation = int(code)
    _load().fa_oracle_set_mutation(int(code))


def fwd(q, k, v, mask=None, *, scale, causal, base2=False, nthreads=None):
    """Full forward: (O [B,H,ql,d] f64, L [B,H,ql] f64)."""
    return fwd_rows(q, k, v, mask, scale=scale, causal=causal, rows=None, base2=base2,
                    nthreads=nthreads)


def fwd_rows(q, k, v, mask=None, *, scale, causal, rows=None, base2=False, nthreads=None):
    """O and L of the flat rows (b*H + h)*ql + i listed in `rows` (None: every row, returned
    in [B,H,ql,(d)] shape)."""
    q, k, v = _f32(q), _f32(k), _f32(v)
    mask = None if mask is None else _f32(mask)
    B, H, Hk, ql, kl, d, dv = _shape(q, k, v)
    full = rows is None
    r = None if full else np.ascontiguousarray(rows, dtype=np.int64)
    n = B * H * ql if full else len(r)
    o = np.empty((n, dv), np.float64)
    lse = np.empty((n,), np.float64)
    rc = _load().fa_oracle_fwd_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(mask), B, H, Hk, ql, kl, d,
                                    dv, float(scale), int(bool(causal)), _ptr(r), n,
                                    int(bool(base2)), _ptr(o), _ptr(lse),
                                    nthreads or default_threads())
    if rc:
        raise ValueError(f"oracle fwd failed ({rc})")
    if full:
        return o.reshape(B, H, ql, dv), lse.reshape(B, H, ql)
    return o, lse


def bwd_q_rows(q, k, v, mask, do, *, scale, causal, rows=None, nthreads=None):
    """dQ of the listed flat query rows (None: all rows, shaped [B,H,ql,d])."""
    q, k, v, do = _f32(q), _f32(k), _f32(v), _f32(do)
    mask = None if mask is None else _f32(mask)
    B, H, Hk, ql, kl, d, dv = _shape(q, k, v)
    full = rows is None
    r = None if full else np.ascontiguousarray(rows, dtype=np.int64)
    n = B * H * ql if full else len(r)
    dq = np.empty((n, d), np.float64)
    rc = _load().fa_oracle_bwd_q_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(mask), _ptr(do), B, H, Hk,
                                      ql, kl, d, dv, float(scale), int(bool(causal)), _ptr(r), n,
                                      _ptr(dq), nthreads or default_threads())
    if rc:
        raise ValueError(f"oracle bwd_q_rows failed ({rc})")
    return dq.reshape(B, H, ql, d) if full else dq


def bwd_kv_rows(q, k, v, mask, do, *, scale, causal, b, kh, js, nthreads=None):
    """dK and dV rows js of kv head kh in batch b: arrays [len(js), d] and [len(js), dv]."""
    q, k, v, do = _f32(q), _f32(k), _f32(v), _f32(do)
    mask = None if mask is None else _f32(mask)
    B, H, Hk, ql, kl, d, dvd = _shape(q, k, v)
    jarr = np.ascontiguousarray(js, dtype=np.int32)
    dk = np.empty((len(jarr), d), np.float64)
    dv = np.empty((len(jarr), dvd), np.float64)
    rc = _load().fa_oracle_bwd_kv_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(mask), _ptr(do), B, H,
                                       Hk, ql, kl, d, dvd, float(scale), int(bool(causal)),
                                       int(b), int(kh), _ptr(jarr), len(jarr), _ptr(dk),
                                       _ptr(dv), nthreads or default_threads())
    if rc:
        raise ValueError(f"oracle bwd_kv_rows failed ({rc})")
    return dk, dv


def bwd(q, k, v, mask, do, *, scale, causal, nthreads=None):
    """Full backward: (dQ [B,H,ql,d], dK [B,Hk,kl,d], dV [B,Hk,kl,dv]) in f64."""
    q, k, v, do = _f32(q), _f32(k), _f32(v), _f32(do)
    mask = None if mask is None else _f32(mask)
    B, H, Hk, ql, kl, d, dvd = _shape(q, k, v)
    dq = np.empty((B, H, ql, d), np.float64)
    dk = np.empty((B, Hk, kl, d), np.float64)
    dv = np.empty((B, Hk, kl, dvd), np.float64)
    rc = _load().fa_oracle_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(mask), _ptr(do), B, H, Hk, ql, kl,
                               d, dvd, float(scale), int(bool(causal)), _ptr(dq), _ptr(dk),
                               _ptr(dv), nthreads or default_threads())
    if rc:
        raise ValueError(f"oracle bwd failed ({rc})")
    return dq, dk, dv


def dsinks(q, k, v, mask, do, *, scale, causal, nthreads=None):
    """Gradient of sum(O * dO) with respect to the sink logits of the enclosing `sinks(...)`
    block: [H] f64, dsink_h = -sum over batch and rows of exp(sink_h - L) * D."""
    q, k, v, do = _f32(q), _f32(k), _f32(v), _f32(do)
    mask = None if mask is None else _f32(mask)
    B, H, Hk, ql, kl, d, dvd = _shape(q, k, v)
    out = np.empty((H,), np.float64)
    rc = _load().fa_oracle_dsinks(_ptr(q), _ptr(k), _ptr(v), _ptr(mask), _ptr(do), B, H, Hk, ql,
                                  kl, d, dvd, float(scale), int(bool(causal)), _ptr(out),
                                  nthreads or default_threads())
    if rc:
        raise ValueError(f"oracle dsinks failed ({rc}); is a sinks(...) block active?")
    return out


def paged_fwd(q, k_cache, v_cache, block_table, lengths, *, scale, causal, nthreads=None):
    """Attention of q [B, H, lq, d] over paged caches [num_pages, Hk, page_size, d] with block
    table [B, max_pages] (int32) and lengths [B] (int32): (O [B, H, lq, d], L [B, H, lq]) in
    f64. The lq queries are each sequence's last lq positions (bottom-right causal)."""
    q, kc, vc = _f32(q), _f32(k_cache), _f32(v_cache)
    table = np.ascontiguousarray(block_table, dtype=np.int32)
    lens = np.ascontiguousarray(lengths, dtype=np.int32)
    B, H, lq, d = q.shape
    P, Hk, bs, dk = kc.shape
    if dk != d or vc.shape != kc.shape or table.shape[0] != B or lens.shape != (B,):
        raise ValueError("paged_fwd: inconsistent shapes")
    o = np.empty((B, H, lq, d), np.float64)
    lse = np.empty((B, H, lq), np.float64)
    rc = _load().fa_oracle_paged_fwd(_ptr(q), _ptr(kc), _ptr(vc), _ptr(table), _ptr(lens), B, H,
                                     Hk, lq, d, bs, table.shape[1], P, float(scale),
                                     int(bool(causal)), _ptr(o), _ptr(lse),
                                     nthreads or default_threads())
    if rc:
        raise ValueError(f"oracle paged_fwd failed ({rc})")
    return o, lse


def paged_bwd(q, k_cache, v_cache, block_table, lengths, do, *, scale, causal, nthreads=None):
    """Gradients of sum(O * dO) for `paged_fwd` with respect to q [B, H, lq, d] and to both
    caches [num_pages, Hk, page_size, d], in f64: (dQ, dK_cache, dV_cache).

    Page "nuvec-core tests/fast.rs", `paged_attention_equals_contiguous_attention`, takes the
    gradients of the paged attention for q and the caches ("paged grads"). Each sequence is the
    fixed-length problem on the keys its table names (logical key j in page
    block_table[b, j // page_size], slot j % page_size), so its gradients are `bwd` on those
    gathered keys. A cache slot's gradient is the sum over every (sequence, key) that reads it
    (a page named by two sequences gets both contributions); slots no sequence reads get 0."""
    q, kc, vc, do = _f32(q), _f32(k_cache), _f32(v_cache), _f32(do)
    table = np.asarray(block_table, np.int64)
    lens = np.asarray(lengths, np.int64)
    B, H, lq, d = q.shape
    _, Hk, bs, _ = kc.shape
    dq = np.zeros(q.shape, np.float64)
    dkc = np.zeros(kc.shape, np.float64)
    dvc = np.zeros(vc.shape, np.float64)
    for b in range(B):
        n = int(lens[b])
        if n == 0:
            continue
        j = np.arange(n)
        pages = table[b, j // bs]
        slots = (j + 1) % bs if _py_mutation == _PY_MUTATION_PAGED_SLOT else j % bs
        kb = kc[pages, :, slots, :].transpose(1, 0, 2)[None]  # [1, Hk, n, d]
        vb = vc[pages, :, slots, :].transpose(1, 0, 2)[None]
        g = bwd(q[b:b + 1], kb, vb, None, do[b:b + 1], scale=scale, causal=causal,
                nthreads=nthreads)
        dq[b] = g[0][0]
        np.add.at(dkc, (pages, slice(None), slots, slice(None)), g[1][0].transpose(1, 0, 2))
        np.add.at(dvc, (pages, slice(None), slots, slice(None)), g[2][0].transpose(1, 0, 2))
    return dq, dkc, dvc


# ------------------------------------------------------------------ variable-length batches
def _seq_bounds(cu, b):
    return int(cu[b]), int(cu[b + 1])


def varlen_fwd(q, k, v, cu_q, cu_k, *, scale, causal, nthreads=None):
    """A batch of independent sequences packed without padding: q [H, total_q, d], k and v
    [Hk, total_k, d(v)], sequence b owning rows cu_q[b] .. cu_q[b+1] of q and cu_k[b] ..
    cu_k[b+1] of k, v. Each sequence is the fixed-length problem on its own rows (causal
    bottom-right within the sequence). Returns (O [H, total_q, dv], L [H, total_q]) in f64;
    a query of a sequence with no keys gets O = 0 and L = -inf. Window and sinks come from the
    enclosing `window(...)` / `sinks(...)` blocks."""
    H, Tq, d = q.shape
    dvd = v.shape[2]
    o = np.zeros((H, Tq, dvd), np.float64)
    lse = np.full((H, Tq), -np.inf, np.float64)
    for b in range(len(cu_q) - 1):
        qs, qe = _seq_bounds(cu_q, b)
        ks, ke = _seq_bounds(cu_k, b)
        if qe == qs:
            continue
        if ke == ks:  # no keys: O = 0; L = -inf, or the head's sink where sinks are set
            if _active_sinks is not None:
                lse[:, qs:qe] = np.asarray(_active_sinks, np.float64)[:, None]
            continue
        ob, lb = fwd(q[None, :, qs:qe], k[None, :, ks:ke], v[None, :, ks:ke], None,
                     scale=scale, causal=causal, nthreads=nthreads)
        o[:, qs:qe] = ob[0]
        lse[:, qs:qe] = lb[0]
    return o, lse


def varlen_bwd(q, k, v, do, cu_q, cu_k, *, scale, causal, nthreads=None):
    """dQ [H, total_q, d], dK [Hk, total_k, d], dV [Hk, total_k, dv] of `varlen_fwd` (f64)."""
    dq = np.zeros(q.shape, np.float64)
    dk = np.zeros(k.shape, np.float64)
    dv = np.zeros(v.shape, np.float64)
    for b in range(len(cu_q) - 1):
        qs, qe = _seq_bounds(cu_q, b)
        ks, ke = _seq_bounds(cu_k, b)
        if qe == qs or ke == ks:
            continue
        g = bwd(q[None, :, qs:qe], k[None, :, ks:ke], v[None, :, ks:ke], None,
                do[None, :, qs:qe], scale=scale, causal=causal, nthreads=nthreads)
        dq[:, qs:qe] = g[0][0]
        dk[:, ks:ke] = g[1][0]
        dv[:, ks:ke] = g[2][0]
    return dq, dk, dv

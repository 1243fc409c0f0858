"""Seeded synthetic inputs for exact training attention.

This module is shared by the parity tests, the benchmark and the CPU oracle runs. It holds no
attention arithmetic: only random draws, the round-to-nearest-even narrowing of those draws to
bf16, and the shapes of the five workloads. Both the CUDA path and the oracle receive the very
same bf16 bit patterns from here.

Conventions taken from the mlx-native training tests (page "mlx-native
tests/test_flash_attn_train.rs", section "Test helpers" and `oracle_for_bf16`):

* inputs are drawn in f32 and rounded once to bf16; the oracle widens those bf16 values exactly;
* the seed constant 0x5452_4149_4E30_3031 ("TRAIN001") is the base of every seed.

The draws themselves are N(0, 1) from NumPy's PCG64 generator, as the workload list asks; the
page's own LCG is not reused (it yields only negative values).
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

SEED_BASE = 0x5452_4149_4E30_3031

# tensor_idx part of a seed: seed = SEED_BASE + 16 * workload_index + tensor_idx
T_Q, T_K, T_V, T_DO, T_MASK, T_SINK = 0, 1, 2, 3, 4, 5


@dataclass(frozen=True)
class Workload:
    """One attention problem: sizes, scale, causal flag and how its inputs are drawn."""

    name: str
    batch: int
    n_heads: int
    n_kv_heads: int
    ql: int
    kl: int
    head_dim: int
    scale: float
    causal: bool
    masked: bool = False  # additive f32 mask [batch, n_heads, ql, kl]
    do_std: float = 1.0  # dO ~ N(0, 1) * do_std
    # local attention window: key j is hidden from row i when j < q_abs - window_left or
    # j > q_abs + window_right (q_abs = kl - ql + i); -1 leaves that side unbounded
    window_left: int = -1
    window_right: int = -1
    value_dim: int = 0  # head dim of v, O, dO (0 = head_dim)
    sinks: bool = False  # one sink logit per query head, N(0, 1) in natural-log units
    deterministic: bool = False  # the backward's bitwise-reproducible mode

    @property
    def windowed(self) -> bool:
        return self.window_left >= 0 or self.window_right >= 0

    @property
    def group(self) -> int:
        return self.n_heads // self.n_kv_heads

    def q_shape(self):
        return (self.batch, self.n_heads, self.ql, self.head_dim)

    def kv_shape(self):
        return (self.batch, self.n_kv_heads, self.kl, self.head_dim)

    @property
    def dv(self) -> int:
        return self.value_dim or self.head_dim

    def v_shape(self):
        return (self.batch, self.n_kv_heads, self.kl, self.dv)

    def o_shape(self):
        return (self.batch, self.n_heads, self.ql, self.dv)

    def lse_shape(self):
        return (self.batch, self.n_heads, self.ql)

    def mask_shape(self):
        return (self.batch, self.n_heads, self.ql, self.kl)

    def visible_pairs(self) -> int:
        """Number of (query, key) pairs the causal bottom-right mask and the window leave
        visible (per b, h); the additive mask is not counted."""
        q_abs = np.arange(self.ql, dtype=np.int64) + (self.kl - self.ql)
        lo = np.zeros_like(q_abs)
        hi = np.full_like(q_abs, self.kl - 1)
        if self.window_left >= 0:
            lo = np.maximum(lo, q_abs - self.window_left)
        if self.causal:
            hi = np.minimum(hi, q_abs)
        if self.window_right >= 0:
            hi = np.minimum(hi, q_abs + self.window_right)
        return int(np.maximum(0, hi - lo + 1).sum())

    def flops(self, exact: bool = False):
        """(fwd, bwd) FLOPs: 4*B*H*ql*kl*d*f and 10*B*H*ql*kl*d*f, or with a value head dim
        dv != d: 2*(d + dv) (QK^T, PV) and 2*(3d + 2dv) (S, dP, dV, dK, dQ) per pair.

        f = 0.5 for causal (the headline counting rule), 1 otherwise; with exact=True, or with a
        window (which has no such rule), f is the visible fraction of (query, key) pairs.
        """
        if exact or self.windowed:
            f = self.visible_pairs() / (self.ql * self.kl)
        else:
            f = 0.5 if self.causal else 1.0
        pairs = self.batch * self.n_heads * self.ql * self.kl * f
        d, dv = self.head_dim, self.dv
        return 2.0 * (d + dv) * pairs, 2.0 * (3 * d + 2 * dv) * pairs


# The workloads, in order (index = workload_index in the seed formula; new ones go last).
WORKLOADS = [
    Workload("tiny_gqa_d64", 1, 2, 1, 64, 64, 64, 1.0 / 8.0, True),
    Workload("masked_d256", 2, 4, 2, 128, 128, 256, 1.0 / 16.0, False, masked=True),
    Workload("train_d64", 4, 16, 16, 2048, 2048, 64, 1.0 / 8.0, True, do_std=0.1),
    Workload("gqa_d128_4k", 2, 32, 8, 4096, 4096, 128, 1.0 / math.sqrt(128.0), True, do_std=0.1),
    Workload("rect_d256", 1, 16, 4, 1024, 8192, 256, 1.0 / 16.0, True, do_std=0.1),
    # sliding-window causal attention: every row sees its last 4096 keys (itself included)
    Workload("swa_d128_16k", 1, 32, 8, 16384, 16384, 128, 1.0 / math.sqrt(128.0), True,
             do_std=0.1, window_left=4095),
    # the headline shape with a sink logit per query head
    Workload("gqa_d128_4k_sinks", 2, 32, 8, 4096, 4096, 128, 1.0 / math.sqrt(128.0), True,
             do_std=0.1, sinks=True),
    # the headline shape with a value head dim of 64 (q, k keep 128)
    Workload("gqa_d128_dv64_4k", 2, 32, 8, 4096, 4096, 128, 1.0 / math.sqrt(128.0), True,
             do_std=0.1, value_dim=64),
    # the headline shape with the deterministic backward
    Workload("gqa_d128_4k_det", 2, 32, 8, 4096, 4096, 128, 1.0 / math.sqrt(128.0), True,
             do_std=0.1, deterministic=True),
]
BY_NAME = {w.name: w for w in WORKLOADS}


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round f32 values to bf16 bit patterns, round-to-nearest-even (NaN-free inputs only).

    Same bit trick as the page "tang src/compute/cuda.rs", `f32_to_bf16`.
    """
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (b >> np.uint64(16)) & np.uint64(1)
    return ((b + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to f32 exactly."""
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(
        np.float32
    )


def normal_bf16(seed: int, shape, std: float = 1.0) -> np.ndarray:
    """N(0,1)*std drawn in f32 from PCG64(seed), rounded to bf16; returned as bf16 bits."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x = x * np.float32(std)
    return f32_to_bf16_bits(x)


def additive_mask(seed: int, shape, p_neg_inf: float = 0.1, full_rows: int = 2) -> np.ndarray:
    """f32 natural-log additive mask: U[-2, 0], then each entry -inf with probability p_neg_inf,
    then `full_rows` distinct rows per (b, h) set entirely to -inf."""
    rng = np.random.default_rng(seed)
    m = rng.uniform(-2.0, 0.0, size=shape).astype(np.float32)
    m[rng.random(size=shape) < p_neg_inf] = -np.inf
    b_, h_, ql, _ = shape
    for b in range(b_):
        for h in range(h_):
            rows = rng.choice(ql, size=min(full_rows, ql), replace=False)
            m[b, h, rows, :] = -np.inf
    return m


@dataclass
class Inputs:
    """bf16 bit patterns of q, k, v, dO (uint16) and an optional f32 mask."""

    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    do: np.ndarray
    mask: np.ndarray | None
    sinks: np.ndarray | None = None  # f32 [H] holding exact bf16 values

    def widened(self):
        """(q, k, v, dO) as f32 arrays holding the exact bf16 values."""
        return tuple(bf16_bits_to_f32(t) for t in (self.q, self.k, self.v, self.do))


def make_inputs(w: Workload, index: int | None = None, seed_base: int | None = None) -> Inputs:
    """Seeded inputs of workload `w` (index = its position in WORKLOADS unless given)."""
    if index is None:
        index = WORKLOADS.index(w) if w in WORKLOADS else 15
    base = (SEED_BASE if seed_base is None else seed_base) + 16 * index
    q = normal_bf16(base + T_Q, w.q_shape())
    k = normal_bf16(base + T_K, w.kv_shape())
    v = normal_bf16(base + T_V, w.v_shape())
    do = normal_bf16(base + T_DO, w.o_shape(), w.do_std)
    mask = additive_mask(base + T_MASK, w.mask_shape()) if w.masked else None
    sinks = bf16_bits_to_f32(normal_bf16(base + T_SINK, (w.n_heads,))) if w.sinks else None
    return Inputs(q, k, v, do, mask, sinks)


# ------------------------------------------------------------------ paged KV-cache inputs
@dataclass(frozen=True)
class DecodeWorkload:
    """Queries over a paged key/value cache: `q_len` new positions per sequence (1 = decode),
    sequence lengths drawn in [min_len, max_len] (the last sequence gets max_len), caches in
    pages of `page_size` positions placed in a shuffled order with `spare_pages` unused."""

    name: str
    batch: int
    n_heads: int
    n_kv_heads: int
    q_len: int
    head_dim: int
    page_size: int
    min_len: int
    max_len: int
    causal: bool = True
    spare_pages: int = 3
    lengths: tuple = ()  # fixed lengths instead of drawn ones

    @property
    def scale(self) -> float:
        return self.head_dim ** -0.5

    @property
    def max_pages(self) -> int:
        return (self.max_len + self.page_size - 1) // self.page_size


@dataclass
class PagedInputs:
    q: np.ndarray            # bf16 bits [B, H, lq, d]
    k_cache: np.ndarray      # bf16 bits [num_pages, Hk, page_size, d]
    v_cache: np.ndarray      # bf16 bits [num_pages, Hk, page_size, d]
    block_table: np.ndarray  # int32 [B, max_pages]
    lengths: np.ndarray      # int32 [B]

    def widened(self):
        """(q, k_cache, v_cache) as f32 arrays (NaN where the cache holds no key)."""
        return tuple(bf16_bits_to_f32(t) for t in (self.q, self.k_cache, self.v_cache))


BF16_NAN_BITS = 0x7FC0


def make_paged_inputs(w: DecodeWorkload, index: int | None = None,
                      seed_base: int | None = None, poison: bool = True) -> PagedInputs:
    """Seeded paged inputs. Every cache slot that holds no key of its sequence (past its
    length, and the spare pages) is set to NaN when `poison` is on, so that a kernel that reads
    past a sequence's end shows it."""
    if index is None:
        index = 40 + DECODE_WORKLOADS.index(w) if w in DECODE_WORKLOADS else 31
    base = (SEED_BASE if seed_base is None else seed_base) + 16 * index
    rng = np.random.default_rng(base + T_MASK)
    B, Hk, bs, d = w.batch, w.n_kv_heads, w.page_size, w.head_dim
    if w.lengths:
        lens = np.array(w.lengths, np.int32)
    else:
        lens = rng.integers(w.min_len, w.max_len + 1, size=B).astype(np.int32)
        lens[-1] = w.max_len
    per = w.max_pages
    n_pages = B * per + w.spare_pages
    order = rng.permutation(n_pages).astype(np.int32)
    table = order[:B * per].reshape(B, per).copy()
    q = normal_bf16(base + T_Q, (B, w.n_heads, w.q_len, d))
    caches = []
    for tix in (T_K, T_V):
        logical = normal_bf16(base + tix, (B, Hk, per * bs, d))  # position-major per sequence
        if poison:
            pos = np.arange(per * bs)[None, :] >= lens[:, None]      # [B, positions]
            logical[np.broadcast_to(pos[:, None, :, None], logical.shape)] = BF16_NAN_BITS
        cache = np.full((n_pages, Hk, bs, d), BF16_NAN_BITS if poison else 0, np.uint16)
        # page p of sequence b holds positions p*bs .. p*bs + bs - 1
        blocks = logical.reshape(B, Hk, per, bs, d).transpose(0, 2, 1, 3, 4)  # [B, per, Hk, bs, d]
        cache[table.reshape(-1)] = blocks.reshape(B * per, Hk, bs, d)
        caches.append(cache)
    return PagedInputs(q, caches[0], caches[1], table, lens)


# Paged-cache workloads of the benchmark (index = position + 40 in the seed formula).
DECODE_WORKLOADS = [
    # single-query decode: 16 sequences of 2k-16k keys, GQA 32:8, pages of 16 positions
    DecodeWorkload("paged_decode_d128", 16, 32, 8, 1, 128, 16, 2048, 16384),
    # four new positions per sequence (causal) against the same kind of cache
    DecodeWorkload("paged_prefill4_d128", 16, 32, 8, 4, 128, 16, 2048, 16384),
]
DECODE_BY_NAME = {w.name: w for w in DECODE_WORKLOADS}


# ------------------------------------------------------------------ variable-length batches
@dataclass(frozen=True)
class VarlenWorkload:
    """Independent sequences packed without padding, head-major: q [H, total_q, d], k and v
    [Hk, total_k, d]; sequence b has q_lens[b] queries and k_lens[b] keys."""

    name: str
    n_heads: int
    n_kv_heads: int
    head_dim: int
    q_lens: tuple
    k_lens: tuple
    causal: bool = True
    window_left: int = -1
    window_right: int = -1
    do_std: float = 1.0

    @property
    def scale(self) -> float:
        return self.head_dim ** -0.5

    @property
    def batch(self) -> int:
        return len(self.q_lens)

    def cu(self, lens):
        return np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)

    @property
    def windowed(self) -> bool:
        return self.window_left >= 0 or self.window_right >= 0

    def flops(self):
        """(fwd, bwd) FLOPs over the visible pairs of every sequence (4d and 10d per pair)."""
        pairs = 0
        for ql, kl in zip(self.q_lens, self.k_lens):
            w = Workload("s", 1, 1, 1, max(ql, 1), max(kl, 1), self.head_dim, 1.0, self.causal,
                         window_left=self.window_left, window_right=self.window_right)
            pairs += w.visible_pairs() if ql > 0 and kl > 0 else 0
        return 4.0 * self.head_dim * pairs * self.n_heads, 10.0 * self.head_dim * pairs * self.n_heads


@dataclass
class VarlenInputs:
    q: np.ndarray    # bf16 bits [H, total_q, d]
    k: np.ndarray    # bf16 bits [Hk, total_k, d]
    v: np.ndarray
    do: np.ndarray   # bf16 bits [H, total_q, d]
    cu_q: np.ndarray  # int32 [B + 1]
    cu_k: np.ndarray

    def widened(self):
        return tuple(bf16_bits_to_f32(t) for t in (self.q, self.k, self.v, self.do))


def make_varlen_inputs(w: VarlenWorkload, index: int = 33, seed_base: int | None = None):
    base = (SEED_BASE if seed_base is None else seed_base) + 16 * index
    cu_q, cu_k = w.cu(w.q_lens), w.cu(w.k_lens)
    tq, tk = max(int(cu_q[-1]), 1), max(int(cu_k[-1]), 1)
    q = normal_bf16(base + T_Q, (w.n_heads, tq, w.head_dim))
    k = normal_bf16(base + T_K, (w.n_kv_heads, tk, w.head_dim))
    v = normal_bf16(base + T_V, (w.n_kv_heads, tk, w.head_dim))
    do = normal_bf16(base + T_DO, (w.n_heads, tq, w.head_dim), w.do_std)
    return VarlenInputs(q, k, v, do, cu_q, cu_k)


# Variable-length workloads of the benchmark (index = position + 50 in the seed formula).
_MIX = (8192, 512, 3000, 1024, 6000, 256, 4096, 2048, 7000, 768, 1500, 5000, 300, 2500, 3500,
        4500)
VARLEN_WORKLOADS = [
    # 16 causal sequences of 256 to 8192 tokens packed together, GQA 32:8, head_dim 128
    VarlenWorkload("varlen_d128_mix", 32, 8, 128, _MIX, _MIX, True, do_std=0.1),
]
VARLEN_BY_NAME = {w.name: w for w in VARLEN_WORKLOADS}

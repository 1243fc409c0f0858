"""Benchmark: exact training attention, forward + backward, bf16, on GB300.

One step = one pass of the whole path over one batch of synthetic inputs: the forward
(O, L) and the backward (dQ, dK, dV) through the C ABI on the current stream.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--no-cpu-baseline]

Prints ONE JSON line (rank 0). `value` is whole-job fwd+bwd TFLOP/s with inputs resident in
HBM (device CUDA events, max over ranks; causal FLOPs counted as half: fwd 4*B*H*ql*kl*d*f,
bwd 10*B*H*ql*kl*d*f, f = 0.5). `e2e` repeats the measurement through the same C calls with
the step's inputs copied from pinned host memory and the gradients read back inside the timed
region, pipelined over two buffer sets (copies of neighbouring steps overlap a step's kernels);
`e2e.serial` is the same with copy-in, compute and copy-out one after another. `roofline` is for the kernel with the largest device time, timed live with CUDA events
on its launch stream by the library's timing facility. `cpu_baseline` times the CPU oracle on a
bounded sample of the same workload (rank 0, N = 1 only).

--impl reference times the CPU oracle (the only reference implementation this project has) on
the host cores, on the same workload, metric and unit, each step a bounded sample.

Several GPUs (torchrun, one process per GPU): every rank runs the full workload on its own GPU
(independent problems, no collective on the data path): "scaling": "weak".
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import fa_inputs  # noqa: E402

METRIC = "attention fwd+bwd TFLOP/s (bf16, causal) at 1 GB300; % of dense bf16 tensor peak"
DEFAULT_WORKLOAD = "gqa_d128_4k"
KERNEL_SOURCES = {
    "fwd_kernel": ["flash_attention_gb300/csrc/fa_fwd.cu", "flash_attention_gb300/csrc/fa_common.cuh",
                   "flash_attention_gb300/csrc/fa_band.cuh"],
    "bwd_main_kernel": ["flash_attention_gb300/csrc/fa_bwd_main.cuh",
                        "flash_attention_gb300/csrc/fa_bwd_common.cuh",
                        "flash_attention_gb300/csrc/fa_common.cuh"],
    "bwd_dq_det_kernel": ["flash_attention_gb300/csrc/fa_bwd_dq.cu",
                          "flash_attention_gb300/csrc/fa_common.cuh",
                          "flash_attention_gb300/csrc/fa_band.cuh"],
    "paged_attn_kernel": ["flash_attention_gb300/csrc/fa_paged.cu",
                          "flash_attention_gb300/csrc/fa_common.cuh"],
    "paged_decode_bwd_kernel": ["flash_attention_gb300/csrc/fa_paged_bwd.cu",
                                "flash_attention_gb300/csrc/fa_common.cuh"],
}
# at head_dim 256 the backward main pass is the CTA-pair kernel (timed under the same name)
PAIR_SOURCES = ["flash_attention_gb300/csrc/fa_bwd_pair.cu",
                "flash_attention_gb300/csrc/fa_bwd_common.cuh",
                "flash_attention_gb300/csrc/fa_common.cuh"]


def kernel_sources(kernel, workload):
    """Source files whose hash dates a traffic figure of `kernel` on `workload`."""
    w = fa_inputs.BY_NAME.get(workload)
    if kernel == "bwd_main_kernel" and w is not None and w.head_dim == 256:
        return PAIR_SOURCES
    return KERNEL_SOURCES.get(kernel, [])


def kernel_flops(w):
    """Algorithmic FLOPs of one launch of each tensor-core kernel, by the workload's counting
    rule: the forward 2(d + dv) per pair; the backward main pass 2(3d + 2dv) (S, dP, dV, dK,
    dQ), or 2(2d + 2dv) in deterministic mode, where the dQ kernel does 2(2d + dv) (S, dP, dQ)."""
    fwd_f, bwd_f = w.flops()
    d, dv = w.head_dim, w.dv
    pairs = bwd_f / (2.0 * (3 * d + 2 * dv))
    out = {"fwd_kernel": fwd_f, "bwd_main_kernel": bwd_f}
    if w.deterministic:
        out["bwd_main_kernel"] = pairs * 2.0 * (2 * d + 2 * dv)
        out["bwd_dq_det_kernel"] = pairs * 2.0 * (2 * d + dv)
    return out


# exp2 rate of the special-function (MUFU) unit of an sm_100-family SM: 4 per clock in each of
# its four sub-partitions.
MUFU_EX2_PER_SM_CLK = 16


def kernel_exps(w):
    """exp2 evaluations of one launch by the counting rule: one per (query, key) pair in the
    forward (P) and again in the backward main pass (P recomputed from L); the deterministic dQ
    kernel recomputes P once more."""
    fwd_f, _ = w.flops()
    pairs = fwd_f / (2.0 * (w.head_dim + w.dv))
    out = {"fwd_kernel": pairs, "bwd_main_kernel": pairs}
    if w.deterministic:
        out["bwd_dq_det_kernel"] = pairs
    return out


def kernel_bounds(w, tensor_tflops, n_sm, sm_mhz):
    """Two lower bounds on each tensor-core kernel's time: its FLOPs at the tensor peak, and
    its exp2 count at the MUFU rate (every exponential on MUFU; the forward moves a share of
    them to an FMA-pipe polynomial, so its own ceiling there is higher). The larger binds."""
    fl, ex = kernel_flops(w), kernel_exps(w)
    mufu = MUFU_EX2_PER_SM_CLK * n_sm * sm_mhz * 1e6
    out = {}
    for k in fl:
        t_tc = fl[k] / (tensor_tflops * 1e12) * 1e6
        t_ex = ex.get(k, 0.0) / mufu * 1e6
        out[k] = {"tensor_us": t_tc, "exp2_mufu_us": t_ex,
                  "binds": "tensor" if t_tc >= t_ex else "exp2"}
    return {"exp2_per_s": mufu, "n_sm": n_sm, "sm_mhz": sm_mhz, "kernels": out}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    choices=sorted(fa_inputs.BY_NAME) + sorted(fa_inputs.DECODE_BY_NAME)
                    + sorted(PAGED_GRAD)
                    + sorted(fa_inputs.VARLEN_BY_NAME))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--ncu", action="store_true",
                    help="profiling mode: run exactly warmup + steps fwd+bwd steps, no timing, "
                         "no e2e, no CPU baseline, no JSON line (for ncu captures)")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def shard_inputs(w, rank):
    """Inputs of this rank's shard: every rank draws its own batches (seed offset by rank),
    so N ranks process N independent copies of the workload's shape (weak scaling)."""
    base = fa_inputs.SEED_BASE + 1_000_003 * rank
    return fa_inputs.make_inputs(w, seed_base=base)


def reduce_max(x, world, device=None):
    """Max of a float over ranks (identity for one rank). Timing only: no data-path traffic."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            pk = json.load(f)
        return {"bf16_tflops": float(pk["bf16_tflops"]),
                "bf16_tflops_sustained": float(pk.get("bf16_tflops_sustained", pk["bf16_tflops"])),
                "hbm_gbs": float(pk["hbm_gbs"]), "source": "measured"}
    return {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0,
            "source": "fallback"}


def code_only(text):
    """Source text without its comments and blank lines: what the compiler sees of a kernel,
    so that a comment edit does not void a recorded capture."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    out = []
    for line in text.splitlines():
        i = line.find("//")
        if i >= 0:
            line = line[:i]
        line = line.rstrip()
        if line:
            out.append(line)
    return "\n".join(out)


def source_hash(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), encoding="utf-8") as fh:
            h.update(code_only(fh.read()).encode("utf-8"))
    return h.hexdigest()[:16]


def recorded_traffic(kernel, workload):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on the current
    source of that kernel (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    e = rec.get(kernel, {}).get(workload)
    if not e or e.get("source_hash") != source_hash(kernel_sources(kernel, workload)):
        return None
    return e.get("dram_bytes_per_launch")


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.proc = None
        self.path = os.path.join("/tmp", f"fa_bench_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 7:
                    continue
                try:
                    sm.append(float(parts[0]))
                    mx = max(mx, float(parts[1]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[3:7]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm), "window": "warm-up and timed steps, 20 ms sampling"}


# ------------------------------------------------------------------ CPU oracle sample
def oracle_head_sample(w, inp, heads, nthreads=None):
    """Full forward + backward of single query heads (with their kv head) by the CPU oracle:
    each is 1/(B*H) of the workload's units. Returns (flops counted by the rule, seconds)."""
    import numpy as np

    import oracle

    q, k, v, do = inp.widened()
    G = w.n_heads // w.n_kv_heads
    fwd_f, bwd_f = w.flops()
    per_head = (fwd_f + bwd_f) / (w.batch * w.n_heads)
    t0 = time.perf_counter()
    win = oracle.window(w.window_left, w.window_right)
    win.__enter__()
    for (b, h) in heads:
        sk = oracle.sinks(None if inp.sinks is None else inp.sinks[h:h + 1])
        sk.__enter__()
        kh = h // G
        qs = np.ascontiguousarray(q[b:b + 1, h:h + 1])
        ks = np.ascontiguousarray(k[b:b + 1, kh:kh + 1])
        vs = np.ascontiguousarray(v[b:b + 1, kh:kh + 1])
        dos = np.ascontiguousarray(do[b:b + 1, h:h + 1])
        ms = None if inp.mask is None else np.ascontiguousarray(inp.mask[b:b + 1, h:h + 1])
        oracle.fwd(qs, ks, vs, ms, scale=w.scale, causal=w.causal, nthreads=nthreads)
        oracle.bwd(qs, ks, vs, ms, dos, scale=w.scale, causal=w.causal, nthreads=nthreads)
        if inp.sinks is not None:
            oracle.dsinks(qs, ks, vs, ms, dos, scale=w.scale, causal=w.causal, nthreads=nthreads)
        sk.__exit__(None, None, None)
    win.__exit__(None, None, None)
    dt = time.perf_counter() - t0
    return per_head * len(heads), dt


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ------------------------------------------------------------------ reference arm
def run_reference(args, w):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle

    oracle.build()
    inp = fa_inputs.make_inputs(w)
    cores = cpu_cores()
    B, H = w.batch, w.n_heads
    order = [(b, h) for b in range(B) for h in range(H)]
    for s in range(args.warmup):
        oracle_head_sample(w, inp, [order[s % len(order)]], nthreads=cores)
    times, flops = [], []
    for s in range(args.steps):
        f, dt = oracle_head_sample(w, inp, [order[(args.warmup + s) % len(order)]], nthreads=cores)
        times.append(dt)
        flops.append(f)
    tot_t = sum(times)
    value = sum(flops) / tot_t / 1e12
    out = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": tot_t / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(w, args.gpus),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": f"per step: full fwd+bwd of one query head (1/{B * H} of the "
                                   f"workload) on the CPU oracle, heads taken in turn"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


# ------------------------------------------------------------------ paged key/value cache
PAGED_METRIC = "paged attention: key/value bytes read per second (bf16 cache) at 1 GB300"
PAGED_GRAD_METRIC = ("paged attention forward + gradients for q and the caches: bytes moved per "
                     "second (bf16 cache) at 1 GB300")
# Gradient workloads: the forward and fa_paged_attention_bwd on a decode workload's caches.
PAGED_GRAD = {"paged_decode_d128_grad": "paged_decode_d128",
              "paged_prefill4_d128_grad": "paged_prefill4_d128"}


def paged_grad_bytes(w, x):
    """Algorithmic bytes of one forward + gradient step, and of each gradient kernel.
    The step: the forward's, then the gradients' least traffic (q, O, dO in and dq out; the
    keys and values each sequence reads; both cache gradients written whole, since slots no
    sequence reads get 0). Per kernel, what its own interface makes it move. With G * q_len
    <= 8 query rows per kv head (the decode path): the gradient kernel (used keys and values
    in, their dK, dV rows out; q, O, dO in) and the fill (every other cache-gradient row out,
    dq in f32 and out). Otherwise (the packed path): the gather (used keys and values in and
    out, packed; q, O, dO in and out, packed), the backward main pass on the packed problem
    (K, V in and dK, dV out; q and dO in) and the scatter (packed dK, dV in; both cache
    gradients out; dq in and out)."""
    el = w.head_dim * 2
    lens = x.lengths.astype(np.int64)
    used = int(lens.sum()) * w.n_kv_heads * el
    cache = x.k_cache.shape[0] * w.n_kv_heads * w.page_size * el
    qbytes = w.batch * w.n_heads * w.q_len * el
    step = paged_bytes(w, x) + 4 * qbytes + 2 * used + 2 * cache
    if (w.n_heads // w.n_kv_heads) * w.q_len <= 8:
        per = {"paged_decode_bwd_kernel": 4 * used + 3 * qbytes,
               "paged_scatter_kernel": 2 * (cache - used) + 3 * qbytes}
    else:
        per = {"paged_gather_kernel": 4 * used + 6 * qbytes,
               "bwd_main_kernel": 4 * used + 2 * qbytes,
               "paged_scatter_kernel": 2 * used + 2 * cache + 2 * qbytes}
    return step, per


def paged_bytes(w, x):
    """Algorithmic bytes of one call: every key and value of every sequence once, q, o, lse,
    the used block-table entries and the lengths."""
    kv = int(x.lengths.astype(np.int64).sum()) * w.n_kv_heads * w.head_dim * 2 * 2
    qo = 2 * w.batch * w.n_heads * w.q_len * w.head_dim * 2 + w.batch * w.n_heads * w.q_len * 4
    pages = int(((x.lengths.astype(np.int64) + w.page_size - 1) // w.page_size).sum())
    return kv + qo + 4 * pages + 4 * w.batch


def paged_config(w, n):
    return {"workload": w.name, "batch": w.batch, "n_heads": w.n_heads,
            "n_kv_heads": w.n_kv_heads, "q_len": w.q_len, "head_dim": w.head_dim,
            "page_size": w.page_size, "lengths": f"uniform in [{w.min_len}, {w.max_len}]",
            "causal": w.causal, "pages": "shuffled, unused slots NaN",
            "l2": "inputs larger than L2 (no flush)",
            "parallelism": "replicas" if n == 1 else f"{n} independent replicas"}


def paged_oracle_sample(w, x, budget_s=10.0, cores=None):
    """The CPU oracle on whole sequences, taken in turn until ~budget_s: (bytes, seconds, n)."""
    import oracle

    q, kc, vc = x.widened()
    spent, nbytes, n = 0.0, 0, 0
    while spent < budget_s and n < w.batch:
        t0 = time.perf_counter()
        oracle.paged_fwd(q[n:n + 1], kc, vc, x.block_table[n:n + 1], x.lengths[n:n + 1],
                         scale=w.scale, causal=w.causal, nthreads=cores)
        spent += time.perf_counter() - t0
        nbytes += int(x.lengths[n]) * w.n_kv_heads * w.head_dim * 4
        n += 1
    return nbytes, spent, n


def paged_grad_oracle_sample(w, x, do_bits, total_bytes, budget_s=10.0, cores=None):
    """The CPU oracle's paged forward and gradients on whole sequences, taken in turn until
    ~budget_s. Each sequence runs on a cache of just its own pages (copied outside the timed
    part). Returns (bytes, seconds, n): the sequences' share of the step's algorithmic bytes,
    by key count."""
    import oracle

    q, kc, vc = x.widened()
    do = fa_inputs.bf16_bits_to_f32(do_bits)
    bs = w.page_size
    total_keys = max(int(x.lengths.astype(np.int64).sum()), 1)
    spent, nbytes, n = 0.0, 0, 0
    while spent < budget_s and n < w.batch:
        L = int(x.lengths[n])
        pages = x.block_table[n, :-(-L // bs)]
        sub_k, sub_v = kc[pages], vc[pages]
        table = np.arange(len(pages), dtype=np.int32)[None]
        lens = x.lengths[n:n + 1]
        t0 = time.perf_counter()
        o = oracle.paged_fwd(q[n:n + 1], sub_k, sub_v, table, lens, scale=w.scale,
                             causal=w.causal, nthreads=cores)
        oracle.paged_bwd(q[n:n + 1], sub_k, sub_v, table, lens, do[n:n + 1], scale=w.scale,
                         causal=w.causal, nthreads=cores)
        spent += time.perf_counter() - t0
        del o
        nbytes += total_bytes * L // total_keys
        n += 1
    return nbytes, spent, n


def run_paged_reference(args, w, grad=False):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle

    oracle.build()
    x = fa_inputs.make_paged_inputs(w)
    cores = cpu_cores()
    per_step = max(1.0, 120.0 / max(args.steps + args.warmup, 1))
    if grad:
        do_bits = fa_inputs.normal_bf16(fa_inputs.SEED_BASE + 77, tuple(x.q.shape), 0.1)
        step_bytes = paged_grad_bytes(w, x)[0]

        def sample(budget):
            return paged_grad_oracle_sample(w, x, do_bits, step_bytes, budget, cores)
    else:
        def sample(budget):
            return paged_oracle_sample(w, x, budget, cores)
    for _ in range(args.warmup):
        sample(min(per_step, 2.0))
    tot_b, tot_s = 0, 0.0
    for _ in range(args.steps):
        b_, s_, _ = sample(per_step)
        tot_b += b_
        tot_s += s_
    value = tot_b / tot_s / 1e9
    cfg = paged_config(w, args.gpus)
    if grad:
        cfg["workload"] = w.name + "_grad"
    out = {"impl": "reference", "metric": PAGED_GRAD_METRIC if grad else PAGED_METRIC,
           "value": value, "unit": "GB/s",
           "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": tot_s / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": cfg,
           "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle",
                            "sample": "per step: whole sequences in turn for ~"
                                      f"{per_step:.0f} s of the CPU oracle"
                                      + (" (forward + gradients)" if grad else "")},
           "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def run_paged(args, w, grad=False):
    import torch

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import flash_attention_gb300 as fa

    fa.build()
    fa.load_library()
    x = fa_inputs.make_paged_inputs(w, seed_base=fa_inputs.SEED_BASE + 1_000_003 * rank)

    def bf(bits):
        return torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16)

    h_q = bf(x.q).pin_memory()
    h_tb = torch.from_numpy(x.block_table).pin_memory()
    h_ln = torch.from_numpy(x.lengths).pin_memory()
    q, tb, ln = h_q.to(dev), h_tb.to(dev), h_ln.to(dev)
    kc, vc = bf(x.k_cache).to(dev), bf(x.v_cache).to(dev)  # the cache stays on the GPU
    o = torch.empty_like(q)
    lse = torch.empty((w.batch, w.n_heads, w.q_len), dtype=torch.float32, device=dev)
    params = fa.FaPagedParams(w.batch, w.n_heads, w.n_kv_heads, w.q_len, w.head_dim,
                              w.page_size, x.block_table.shape[1], x.k_cache.shape[0],
                              w.scale, int(w.causal), 0, 0)
    stream = torch.cuda.current_stream(dev)
    if grad:
        h_do = bf(fa_inputs.normal_bf16(fa_inputs.SEED_BASE + 77 + rank, tuple(x.q.shape),
                                        0.1)).pin_memory()
        do = h_do.to(dev)
        dq, dkc, dvc = torch.empty_like(q), torch.empty_like(kc), torch.empty_like(vc)

    def step():
        fa.fa_paged_attention(q, kc, vc, tb, ln, o, lse, params, stream)
        if grad:
            fa.fa_paged_attention_bwd(q, kc, vc, tb, ln, o, lse, do, dq, dkc, dvc, params,
                                      stream)

    def barrier():
        if world > 1:
            import torch.distributed as dist

            dist.barrier()

    if args.ncu:
        for _ in range(args.warmup + args.steps):
            step()
        torch.cuda.synchronize()
        rc = fa.fa_device_status(True)
        print(f"ncu mode: {args.warmup + args.steps} steps of {w.name}, status {rc}", flush=True)
        if rc != fa.FA_OK:
            raise RuntimeError("paged kernel reported an error")
        return

    clocks = ClockSampler(local)
    clocks.start()
    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    if fa.fa_device_status(True) != fa.FA_OK:
        clocks.stop()
        raise RuntimeError("paged kernel reported an error during warm-up")
    barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    fa.fa_profile_enable(True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    fa.fa_profile_enable(False)
    barrier()
    prof = fa.fa_profile_read()
    if fa.fa_device_status(True) != fa.FA_OK:
        clocks.stop()
        raise RuntimeError("paged kernel reported an error during the timed steps")
    # The same K steps again (without the per-kernel events) until the timed regions add up to
    # about 300 ms, so that the clock samples cover the measurement; `value` is the median.
    rep_ms = [reduce_max(e0.elapsed_time(e1) / args.steps, world, dev)]
    n_rep = min(99, max(0, math.ceil(300.0 / (rep_ms[0] * args.steps)) - 1))
    for _ in range(n_rep):
        barrier()
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        rep_ms.append(reduce_max(e0.elapsed_time(e1) / args.steps, world, dev))
    clk = clocks.stop()
    if fa.fa_device_status(True) != fa.FA_OK:
        raise RuntimeError("paged kernel reported an error during the repeated steps")
    tot_ms = statistics.median(rep_ms)
    repeats = {"regions": len(rep_ms), "steps_each": args.steps,
               "spread_pct": 100.0 * (max(rep_ms) - min(rep_ms)) / tot_ms}
    nbytes = paged_bytes(w, x)
    kern_bytes = {"paged_attn_kernel": nbytes}
    if grad:
        nbytes, per = paged_grad_bytes(w, x)
        kern_bytes.update(per)
    value = world * nbytes / (tot_ms * 1e-3) / 1e9
    peaks = load_peaks()
    hbm = peaks["hbm_gbs"]
    # the dominant kernel by device time, against the bytes it must move
    dom = max(kern_bytes, key=lambda k: prof[k][0])
    ms, n = prof[dom]
    kern_ms = ms / max(n, 1)
    roofline = {"bound": "hbm", "kernel": dom,
                "achieved": kern_bytes[dom] / (kern_ms * 1e-3) / 1e9, "peak": hbm, "unit": "GB/s",
                "frac": kern_bytes[dom] / (kern_ms * 1e-3) / 1e9 / hbm,
                "traffic": recorded_traffic(dom, w.name + ("_grad" if grad else "")),
                "peak_source": f"hbm_gbs, {peaks['source']}",
                "per_kernel_ms": {k: (t / max(c, 1)) for k, (t, c) in prof.items() if c}}
    launches = sum(c for _, c in prof.values())
    if grad and prof.get("paged_decode_bwd_kernel", (0, 0))[1]:
        launches += prof["paged_scatter_kernel"][1]  # (fill and dq convert in one region)
    elif grad:  # timed regions of several launches: gather (index, gather, tail, q side), scatter
        launches += 3 * prof["paged_gather_kernel"][1] + prof["paged_scatter_kernel"][1]

    e2e = None
    if not args.no_e2e:
        h_o = torch.empty(o.shape, dtype=o.dtype).pin_memory()
        h_dq = torch.empty(q.shape, dtype=q.dtype).pin_memory() if grad else None

        def e2e_step():  # new queries, table and lengths in; the attention output back
            q.copy_(h_q, non_blocking=True)
            tb.copy_(h_tb, non_blocking=True)
            ln.copy_(h_ln, non_blocking=True)
            if grad:
                do.copy_(h_do, non_blocking=True)
            step()
            h_o.copy_(o, non_blocking=True)
            if grad:
                h_dq.copy_(dq, non_blocking=True)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        barrier()
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        f0.record(stream)
        for _ in range(args.steps):
            e2e_step()
        f1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = reduce_max(f0.elapsed_time(f1) / args.steps, world, dev)
        h2d = sum(t.numel() * t.element_size() for t in (h_q, h_tb, h_ln) + ((h_do,) if grad else ()))
        e2e = {"value": world * nbytes / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
               "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": sum(t.numel() * t.element_size()
                                         for t in (h_o,) + ((h_dq,) if grad else ())),
               "note": "the key/value cache stays resident on the GPU, as in serving"
                       + ("; its gradients stay on the GPU, dq comes back" if grad else "")}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cores = cpu_cores()
        if grad:
            b_, s_, n_ = paged_grad_oracle_sample(w, x, h_do.view(torch.int16).numpy()
                                                  .view(np.uint16), nbytes, 10.0, cores)
            what = "forward + gradients"
        else:
            b_, s_, n_ = paged_oracle_sample(w, x, 10.0, cores)
            what = "forward"
        cpu = {"value": b_ / s_ / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
               "sample": f"{what} of {n_} whole sequence(s) of {w.batch}, f64, {s_:.1f} s"}

    if rank == 0:
        cfg = paged_config(w, world)
        if grad:
            cfg["workload"] = w.name + "_grad"
            cfg["step"] = "fa_paged_attention + fa_paged_attention_bwd (dO ~ N(0, 0.01))"
        out = {"metric": PAGED_GRAD_METRIC if grad else PAGED_METRIC, "value": value,
               "unit": "GB/s", "n_gpus": world,
               "steps": args.steps, "warmup": args.warmup, "ms_per_step": tot_ms,
               "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
               "dtype": "bf16", "data": "synthetic", "config": cfg,
               "bytes_per_step": nbytes, "roofline": roofline, "cpu_baseline": cpu,
               "e2e": e2e, "gpu_launches": int(launches), "clocks": clk, "repeats": repeats}
        print(json.dumps(out), flush=True)


# ------------------------------------------------------------------ variable-length batches
def varlen_config(w, n):
    return {"workload": w.name, "n_heads": w.n_heads, "n_kv_heads": w.n_kv_heads,
            "head_dim": w.head_dim, "sequences": w.batch, "lengths": list(w.q_lens),
            "total_tokens": int(sum(w.q_lens)), "causal": w.causal,
            "flop_rule": "fwd 4d, bwd 10d per visible (query, key) pair of each sequence",
            "l2": "inputs larger than L2 (no flush)",
            "parallelism": "replicas" if n == 1 else f"{n} independent replicas"}


def varlen_oracle_sample(w, x, budget_s, cores):
    """The CPU oracle (fwd + bwd) on whole sequences, shortest first, for ~budget_s:
    (FLOPs, seconds, sequences)."""
    import oracle

    q, k, v, do = x.widened()
    order = sorted(range(w.batch), key=lambda b: w.q_lens[b])
    spent, fl, n = 0.0, 0.0, 0
    for b in order:
        if spent >= budget_s:
            break
        qs, qe, ks, ke = x.cu_q[b], x.cu_q[b + 1], x.cu_k[b], x.cu_k[b + 1]
        sub = fa_inputs.VarlenWorkload("s", w.n_heads, w.n_kv_heads, w.head_dim, (qe - qs,),
                                       (ke - ks,), w.causal)
        t0 = time.perf_counter()
        oracle.fwd(q[None, :, qs:qe], k[None, :, ks:ke], v[None, :, ks:ke], None, scale=w.scale,
                   causal=w.causal, nthreads=cores)
        oracle.bwd(q[None, :, qs:qe], k[None, :, ks:ke], v[None, :, ks:ke], None,
                   do[None, :, qs:qe], scale=w.scale, causal=w.causal, nthreads=cores)
        spent += time.perf_counter() - t0
        fl += sum(sub.flops())
        n += 1
    return fl, spent, n


def run_varlen_reference(args, w):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle

    oracle.build()
    x = fa_inputs.make_varlen_inputs(w, index=50 + fa_inputs.VARLEN_WORKLOADS.index(w))
    cores = cpu_cores()
    per_step = max(1.0, 120.0 / max(args.steps + args.warmup, 1))
    for _ in range(args.warmup):
        varlen_oracle_sample(w, x, min(per_step, 2.0), cores)
    fl, sec = 0.0, 0.0
    for _ in range(args.steps):
        f_, s_, _ = varlen_oracle_sample(w, x, per_step, cores)
        fl += f_
        sec += s_
    value = fl / sec / 1e12
    out = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
           "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": sec / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": varlen_config(w, args.gpus),
           "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                            "sample": f"per step: whole sequences, shortest first, ~{per_step:.0f} s"},
           "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def run_varlen(args, w):
    import torch

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import flash_attention_gb300 as fa

    fa.build()
    fa.load_library()
    x = fa_inputs.make_varlen_inputs(w, index=50 + fa_inputs.VARLEN_WORKLOADS.index(w),
                                     seed_base=fa_inputs.SEED_BASE + 1_000_003 * rank)

    def bf(bits):
        return torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16)

    h_q, h_k, h_v, h_do = (bf(t).pin_memory() for t in (x.q, x.k, x.v, x.do))
    q, k, v, do = (t.to(dev) for t in (h_q, h_k, h_v, h_do))
    cq, ck = torch.from_numpy(x.cu_q).to(dev), torch.from_numpy(x.cu_k).to(dev)
    mq, mk = max(w.q_lens), max(w.k_lens)
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    params, opts = fa.varlen_params_options(q, k, v, cq, ck, mq, mk, scale=w.scale,
                                            causal=w.causal)
    stream = torch.cuda.current_stream(dev)

    def step():
        fa.fa_train_fwd_ex(q, k, v, None, o, lse, params, opts, stream)
        fa.fa_train_bwd_ex(q, k, v, o, lse, do, None, dq, dk, dv, params, opts, stream)

    def barrier():
        if world > 1:
            import torch.distributed as dist

            dist.barrier()

    if args.ncu:
        for _ in range(args.warmup + args.steps):
            step()
        torch.cuda.synchronize()
        print(f"ncu mode: {w.name}, status {fa.fa_device_status(True)}", flush=True)
        return

    clocks = ClockSampler(local)
    clocks.start()
    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    if fa.fa_device_status(True) != fa.FA_OK:
        clocks.stop()
        raise RuntimeError("a kernel reported an error during warm-up")
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    fa.fa_profile_enable(True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    fa.fa_profile_enable(False)
    clk = clocks.stop()
    barrier()
    prof = fa.fa_profile_read()
    if fa.fa_device_status(True) != fa.FA_OK:
        raise RuntimeError("a kernel reported an error during the timed steps")
    tot_ms = reduce_max(e0.elapsed_time(e1) / args.steps, world, dev)
    fwd_f, bwd_f = w.flops()
    value = world * (fwd_f + bwd_f) / (tot_ms * 1e-3) / 1e12
    peaks = load_peaks()
    dom_name, (dom_ms, dom_n) = max(prof.items(), key=lambda kv: kv[1][0])
    algo = {"fwd_kernel": fwd_f, "bwd_main_kernel": bwd_f}.get(dom_name, 0.0)
    achieved = algo / (dom_ms / max(dom_n, 1) * 1e-3) / 1e12
    roofline = {"bound": "tensor", "kernel": dom_name, "achieved": achieved,
                "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": achieved / peaks["bf16_tflops"],
                "traffic": recorded_traffic(dom_name, w.name),
                "peak_source": f"bf16_tflops burst, {peaks['source']}",
                "per_kernel_ms": {n: (t / max(c, 1)) for n, (t, c) in prof.items() if c}}
    e2e = None
    if not args.no_e2e:
        h_dq, h_dk, h_dv = (torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in (dq, dk, dv))

        def e2e_step():
            for d_, h_ in ((q, h_q), (k, h_k), (v, h_v), (do, h_do)):
                d_.copy_(h_, non_blocking=True)
            step()
            for d_, h_ in ((dq, h_dq), (dk, h_dk), (dv, h_dv)):
                h_.copy_(d_, non_blocking=True)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        f0.record(stream)
        for _ in range(args.steps):
            e2e_step()
        f1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = reduce_max(f0.elapsed_time(f1) / args.steps, world, dev)
        e2e = {"value": world * (fwd_f + bwd_f) / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
               "ms_per_step": e2e_ms,
               "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in (h_q, h_k, h_v, h_do)),
               "d2h_bytes_per_step": sum(t.numel() * t.element_size() for t in (h_dq, h_dk, h_dv))}
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cores = cpu_cores()
        f_, s_, n_ = varlen_oracle_sample(w, x, 10.0, cores)
        cpu = {"value": f_ / s_ / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
               "sample": f"fwd+bwd of the {n_} shortest sequence(s), f64, {s_:.1f} s"}
    if rank == 0:
        out = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
               "steps": args.steps, "warmup": args.warmup, "ms_per_step": tot_ms,
               "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
               "dtype": "bf16", "data": "synthetic", "config": varlen_config(w, world),
               "pct_of_peak": 100.0 * value / (world * peaks["bf16_tflops"]),
               "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
               "gpu_launches": int(sum(c for _, c in prof.values())), "clocks": clk}
        print(json.dumps(out), flush=True)


def config_of(w, n):
    return {"workload": w.name, "batch": w.batch, "n_heads": w.n_heads,
            "n_kv_heads": w.n_kv_heads, "ql": w.ql, "kl": w.kl, "head_dim": w.head_dim,
            "scale": w.scale, "causal": w.causal, "mask": w.masked,
            **({"window": [w.window_left, w.window_right]} if w.windowed else {}),
            **({"value_dim": w.dv} if w.dv != w.head_dim else {}),
            **({"sinks": True} if w.sinks else {}),
            **({"deterministic": True} if w.deterministic else {}),
            "flop_rule": "fwd 4*B*H*ql*kl*d*f, bwd 10*B*H*ql*kl*d*f, "
                         + ("f = visible fraction of (query, key) pairs under the window"
                            if w.windowed else "f=0.5 causal"),
            "l2": "inputs larger than L2 (no flush): a step touches "
                  f"{step_bytes(w) / 1e6:.0f} MB",
            "parallelism": "replicas" if n == 1 else f"{n} independent replicas"}


def step_bytes(w):
    qb = w.batch * w.n_heads * w.ql * w.head_dim * 2
    ob = w.batch * w.n_heads * w.ql * w.dv * 2
    kb = w.batch * w.n_kv_heads * w.kl * w.head_dim * 2
    vb = w.batch * w.n_kv_heads * w.kl * w.dv * 2
    # q, dq, o (twice), dO + k, dk + v, dv + the f32 dQ accumulator (read and written)
    return 2 * qb + 3 * ob + 2 * kb + 2 * vb + 4 * qb


# ------------------------------------------------------------------ our arm
def run_ours(args, w):
    import numpy as np
    import torch

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import flash_attention_gb300 as fa

    fa.build()
    fa.load_library()

    inp = shard_inputs(w, rank)

    def bf(bits):
        return torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16)

    h_q, h_k, h_v, h_do = (bf(t).pin_memory() for t in (inp.q, inp.k, inp.v, inp.do))
    q, k, v, do = (t.to(dev) for t in (h_q, h_k, h_v, h_do))
    mask = None if inp.mask is None else torch.from_numpy(inp.mask).to(dev)
    o = torch.empty(w.o_shape(), dtype=q.dtype, device=dev)
    lse = torch.empty(w.lse_shape(), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    params = fa.FaParams(w.batch, w.n_heads, w.n_kv_heads, w.ql, w.kl, w.head_dim, w.scale,
                         int(w.causal))
    sinks = None if inp.sinks is None else torch.from_numpy(inp.sinks).to(dev)
    dsinks = None if sinks is None else torch.empty_like(sinks)
    opts = fa.make_options(q, k, mask, (w.window_left, w.window_right), v=v, sinks=sinks,
                           dsinks=dsinks, deterministic=w.deterministic)
    stream = torch.cuda.current_stream(dev)

    def step():
        fa.fa_train_fwd_ex(q, k, v, mask, o, lse, params, opts, stream)
        fa.fa_train_bwd_ex(q, k, v, o, lse, do, mask, dq, dk, dv, params, opts, stream)

    def barrier():
        if world > 1:
            import torch.distributed as dist

            dist.barrier()

    if args.ncu:
        for _ in range(args.warmup + args.steps):
            step()
        torch.cuda.synchronize()
        rc = fa.fa_device_status(True)
        print(f"ncu mode: {args.warmup + args.steps} steps of {w.name}, status {rc}", flush=True)
        if rc != fa.FA_OK:
            raise RuntimeError("a kernel gave up a bounded wait")
        return

    clocks = ClockSampler(local)
    clocks.start()
    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    if fa.fa_device_status(True) != fa.FA_OK:
        clocks.stop()
        raise RuntimeError("a kernel gave up a bounded wait during warm-up")

    # ---------------- device-timed steps (inputs resident)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    fa.fa_profile_read()  # clear
    barrier()
    torch.cuda.synchronize()
    fa.fa_profile_enable(True)
    for s in range(args.steps):
        ev[s][0].record(stream)
        fa.fa_train_fwd_ex(q, k, v, mask, o, lse, params, opts, stream)
        ev[s][1].record(stream)
        fa.fa_train_bwd_ex(q, k, v, o, lse, do, mask, dq, dk, dv, params, opts, stream)
        ev[s][2].record(stream)
    torch.cuda.synchronize()
    fa.fa_profile_enable(False)
    barrier()
    fwd_ms = [a.elapsed_time(b) for a, b, _ in ev]
    bwd_ms = [b.elapsed_time(c) for _, b, c in ev]
    tot_ms = ev[0][0].elapsed_time(ev[-1][2]) / args.steps
    prof = fa.fa_profile_read()
    if fa.fa_device_status(True) != fa.FA_OK:
        raise RuntimeError("a kernel gave up a bounded wait during the timed steps")

    tot_ms = reduce_max(tot_ms, world, dev)
    # The same K timed steps again, until the timed regions add up to about 300 ms, so that the
    # clock samples cover the measurement and its spread is known; `value` is the median region.
    rep_ms = [tot_ms]
    n_rep = min(29, max(0, math.ceil(300.0 / (tot_ms * args.steps)) - 1))
    r0, r1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(n_rep):
        barrier()
        torch.cuda.synchronize()
        r0.record(stream)
        for _ in range(args.steps):
            step()
        r1.record(stream)
        torch.cuda.synchronize()
        rep_ms.append(reduce_max(r0.elapsed_time(r1) / args.steps, world, dev))
    clk = clocks.stop()
    if fa.fa_device_status(True) != fa.FA_OK:
        raise RuntimeError("a kernel gave up a bounded wait during the repeated steps")
    tot_ms = statistics.median(rep_ms)
    repeats = {"regions": len(rep_ms), "steps_each": args.steps,
               "ms_per_step": [round(x, 5) for x in rep_ms],
               "spread_pct": 100.0 * (max(rep_ms) - min(rep_ms)) / tot_ms,
               "ms_x_median_sm_mhz": (tot_ms * clk["sm_mhz"]) if clk and clk.get("sm_mhz")
               else None}

    fwd_f, bwd_f = w.flops()
    fwd_ex, bwd_ex = w.flops(exact=True)
    value = world * (fwd_f + bwd_f) / (tot_ms * 1e-3) / 1e12
    peaks = load_peaks()
    peak = peaks["bf16_tflops"]

    # ---------------- roofline of the dominant kernel (live CUDA-event timing)
    launches_per_step = sum(n for _, n in prof.values()) / args.steps
    dom = max(prof.items(), key=lambda kv: kv[1][0])
    dom_name, (dom_ms, dom_n) = dom
    algo = kernel_flops(w).get(dom_name, 0.0)
    dom_avg = dom_ms / max(dom_n, 1)
    achieved = algo / (dom_avg * 1e-3) / 1e12
    traffic = recorded_traffic(dom_name, w.name)
    roofline = {"bound": "tensor", "kernel": dom_name, "achieved": achieved, "peak": peak,
                "unit": "TFLOP/s", "frac": achieved / peak, "traffic": traffic,
                "peak_source": f"bf16_tflops burst, {peaks['source']}",
                "per_kernel_ms": {n: (t / max(c, 1)) for n, (t, c) in prof.items()}}
    # the secondary bound (exp2 on MUFU) beside the tensor bound, at the sampled maximum clock
    n_sm = torch.cuda.get_device_properties(dev).multi_processor_count
    clock = (clk or {}).get("sm_max_mhz") or (clk or {}).get("sm_mhz") or 2070.0
    roofline["bounds"] = kernel_bounds(w, peak, n_sm, float(clock))

    # ---------------- end to end through the C ABI with host buffers
    e2e = None
    if not args.no_e2e:
        h_dq = torch.empty(dq.shape, dtype=dq.dtype).pin_memory()
        h_dk = torch.empty(dk.shape, dtype=dk.dtype).pin_memory()
        h_dv = torch.empty(dv.shape, dtype=dv.dtype).pin_memory()

        def e2e_step():
            q.copy_(h_q, non_blocking=True)
            k.copy_(h_k, non_blocking=True)
            v.copy_(h_v, non_blocking=True)
            do.copy_(h_do, non_blocking=True)
            step()
            h_dq.copy_(dq, non_blocking=True)
            h_dk.copy_(dk, non_blocking=True)
            h_dv.copy_(dv, non_blocking=True)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        serial_ms = reduce_max(e0.elapsed_time(e1) / args.steps, world, dev)
        h2d = sum(t.numel() * t.element_size() for t in (h_q, h_k, h_v, h_do))
        d2h = sum(t.numel() * t.element_size() for t in (h_dq, h_dk, h_dv))

        ref_dk, ref_dv = h_dk.clone(), h_dv.clone()  # the serial steps' dK, dV (deterministic)

        # The same steps pipelined the way a training loop feeds the calls: two device buffer
        # sets; step i+1's inputs go up on one copy stream and step i-1's gradients come down
        # on another while step i's kernels run. Every step still copies its own inputs in and
        # its own dQ, dK, dV out inside the timed region.
        up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        sets = [(q, k, v, do, o, lse, dq, dk, dv),
                tuple(torch.empty_like(t) for t in (q, k, v, do, o, lse, dq, dk, dv))]
        ev_up = [torch.cuda.Event() for _ in range(2)]
        ev_comp = [torch.cuda.Event() for _ in range(2)]
        ev_down = [torch.cuda.Event() for _ in range(2)]

        def upload(i):
            bq, bk, bv, bdo = sets[i % 2][:4]
            with torch.cuda.stream(up):
                if i >= 2:  # step i-2 has finished reading this set's inputs
                    up.wait_event(ev_comp[i % 2])
                for dst, src in ((bq, h_q), (bk, h_k), (bv, h_v), (bdo, h_do)):
                    dst.copy_(src, non_blocking=True)
                ev_up[i % 2].record(up)

        def compute(i):
            bq, bk, bv, bdo, bo, blse, bdq, bdk, bdv = sets[i % 2]
            stream.wait_event(ev_up[i % 2])
            if i >= 2:  # step i-2's gradients in this set have been read back
                stream.wait_event(ev_down[i % 2])
            fa.fa_train_fwd_ex(bq, bk, bv, mask, bo, blse, params, opts, stream)
            fa.fa_train_bwd_ex(bq, bk, bv, bo, blse, bdo, mask, bdq, bdk, bdv, params, opts,
                               stream)
            ev_comp[i % 2].record(stream)

        def download(i):
            bdq, bdk, bdv = sets[i % 2][6:]
            with torch.cuda.stream(down):
                down.wait_event(ev_comp[i % 2])
                for dst, src in ((h_dq, bdq), (h_dk, bdk), (h_dv, bdv)):
                    dst.copy_(src, non_blocking=True)
                ev_down[i % 2].record(down)

        def pipelined(n):
            upload(0)
            for i in range(n):
                if i + 1 < n:
                    upload(i + 1)
                compute(i)
                download(i)

        e0.record(stream)
        up.wait_event(e0)
        pipelined(3)
        stream.wait_event(ev_down[2 % 2])
        torch.cuda.synchronize()
        barrier()
        e0.record(stream)
        up.wait_event(e0)
        pipelined(args.steps)
        stream.wait_event(ev_down[(args.steps - 1) % 2])
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = reduce_max(e0.elapsed_time(e1) / args.steps, world, dev)
        e2e = {"value": world * (fwd_f + bwd_f) / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
               "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "overlap": "two buffer sets: step i+1's uploads and step i-1's downloads on "
                          "copy streams during step i's kernels",
               "serial": {"value": world * (fwd_f + bwd_f) / (serial_ms * 1e-3) / 1e12,
                          "ms_per_step": serial_ms,
                          "note": "copy in, compute, copy out, one step after another on "
                                  "one stream"}}
        if fa.fa_device_status(True) != fa.FA_OK:
            raise RuntimeError("a kernel gave up a bounded wait during the end-to-end steps")
        if not (torch.equal(h_dk, ref_dk) and torch.equal(h_dv, ref_dv)):
            raise RuntimeError("the pipelined steps read back other dK / dV than the serial ones")

    # ---------------- CPU oracle baseline (rank 0, N = 1)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cores = cpu_cores()
        heads, spent, fl = [], 0.0, 0.0
        order = [(b, h) for b in range(w.batch) for h in range(w.n_heads)]
        n = 0
        while spent < 10.0 and n < len(order):
            f, dt = oracle_head_sample(w, inp, [order[n]], nthreads=cores)
            heads.append(order[n])
            spent += dt
            fl += f
            n += 1
        cpu = {"value": fl / spent / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
               "sample": f"full fwd+bwd of {len(heads)} query head(s) with their kv head "
                         f"({len(heads)}/{w.batch * w.n_heads} of the workload), f64, "
                         f"{spent:.1f} s"}

    if rank == 0:
        out = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": tot_ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic", "config": config_of(w, world),
            "pct_of_peak": 100.0 * value / (world * peak),
            "fwd_tflops": (fwd_f / (statistics.median(fwd_ms) * 1e-3)) / 1e12,
            "bwd_tflops": (bwd_f / (statistics.median(bwd_ms) * 1e-3)) / 1e12,
            "fwd_ms_median": statistics.median(fwd_ms), "bwd_ms_median": statistics.median(bwd_ms),
            "exact_visible_tflops": world * (fwd_ex + bwd_ex) / (tot_ms * 1e-3) / 1e12,
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": int(round(launches_per_step * args.steps)),
            "clocks": clk, "repeats": repeats,
        }
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


def main():
    args = parse()
    if args.workload in fa_inputs.VARLEN_BY_NAME:
        w = fa_inputs.VARLEN_BY_NAME[args.workload]
        if args.impl == "reference":
            run_varlen_reference(args, w)
        else:
            run_varlen(args, w)
        return
    if args.workload in PAGED_GRAD:
        w = fa_inputs.DECODE_BY_NAME[PAGED_GRAD[args.workload]]
        if args.impl == "reference":
            run_paged_reference(args, w, grad=True)
        else:
            run_paged(args, w, grad=True)
        return
    if args.workload in fa_inputs.DECODE_BY_NAME:
        w = fa_inputs.DECODE_BY_NAME[args.workload]
        if args.impl == "reference":
            run_paged_reference(args, w)
        else:
            run_paged(args, w)
        return
    w = fa_inputs.BY_NAME[args.workload]
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()

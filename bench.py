"""Benchmark: causal attention forward TFLOP/s on one GB300 (per rank), with
the roofline fraction, an end-to-end figure from host buffers, and the fp64
CPU oracle timed on the host as a reported baseline.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...     # the oracle alone, on host cores

A step is one attn_fwd call over the whole workload (all query rows of every
batch and head).  FLOPs per step = 4*B*Hq*S^2*D / 2 (causal).  With
--mask-density P the step is attn_fwd_block_masked with a seeded per-head
block mask keeping each 128 x 128 block with probability P, and the FLOPs are
4*D per visible (query, key) pair, counted exactly; with --window W it is
attn_fwd_elem_masked with a local window (query i keeps keys i-W < j <= i, as
keep bits) plus the block mask of the blocks the window touches, FLOPs = 4*D
per kept pair.  With --pass bwd the step
is one attn_bwd call (dQ, dK, dV for a seeded upstream gradient, O and LSE
from attn_fwd beforehand) and FLOPs = 2.5x the forward's (five products per
tile pair instead of two: the usual convention for attention backward);
--mask-density, --window and --dropout select the matching backward entry
points (attn_bwd_block_masked, attn_bwd_elem_masked, attn_bwd_dropout).
--window with --dropout runs both in one call (attn_fwd_ex / attn_bwd_ex).
With --pass proj the step is one attn_out_proj call on the workload's
attention output shape, E = Hq*D output features, FLOPs = 2*B*S*E*Hq*D.  Between timed
steps a 256 MiB buffer is written to flush L2; each step is timed with CUDA
events on the launching stream.  The forward line also carries a warm-L2
figure (the same call back to back, no flush: warm_l2) and the host time of
one asynchronous call (host_us_per_call).  With --dtype fp8 the roofline peak
is an E4M3 GEMM measured in the same run.  Under torchrun every rank runs the same
workload on its own GPU (independent problems, no collective on the data
path); rank 0 prints one JSON line with the slowest rank's time: the mean
step (ms_per_step, from which value is computed) and the median and minimum
step (ms_step_median, ms_step_min).
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import os
import platform
import re
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from causal_scaled_dot_gb300.workloads import BY_NAME, HEADLINE  # noqa: E402

DROPOUT_SEED, DROPOUT_OFFSET = 0x5EED, 0
METRIC = "causal attn fwd TFLOP/s (bf16, 1xGB300) and % of dense bf16 tensor peak"
PROJ_METRIC = "attn output projection TFLOP/s (bf16, 1xGB300) and % of dense bf16 tensor peak"
BWD_METRIC = "causal attn bwd TFLOP/s (bf16, 1xGB300; 2.5x forward FLOPs) and % of dense bf16 tensor peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 256 << 20


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def measure_fp8_peak(dev) -> float:
    """Dense E4M3 GEMM throughput of this GPU in TFLOP/s, measured here: torch's
    scaled matmul (cuBLASLt) at 8192^3 with bf16 output, best of 10 calls timed
    with CUDA events after 5 warm-up calls (burst, like the bf16 figure)."""
    import torch
    n = 8192
    a = torch.randn(n, n, device=dev).to(torch.float8_e4m3fn)
    b = torch.randn(n, n, device=dev).to(torch.float8_e4m3fn).t()  # column-major operand
    one = torch.tensor(1.0, device=dev)
    for _ in range(5):
        torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
    torch.cuda.synchronize(dev)
    best = float("inf")
    for _ in range(10):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
        e1.record()
        torch.cuda.synchronize(dev)
        best = min(best, e0.elapsed_time(e1))
    del a, b
    return 2.0 * n ** 3 / (best * 1e-3) / 1e12


def host_us_per_call(call, n: int = 200) -> float:
    """Host time of one asynchronous launch call (median of 5 batches of n calls;
    the device is synchronised only between batches)."""
    import torch
    per = []
    for _ in range(5):
        t0 = time.perf_counter()
        for _ in range(n):
            call()
        per.append((time.perf_counter() - t0) / n * 1e6)
        torch.cuda.synchronize()
    return sorted(per)[2]


# The sources of the timed kernels, per pass, with the forward's unit order
# (fwd_schedule.h), which decides what stays in L2 (the launch geometry -- one
# CTA per SM, 384 threads -- is fixed in attn_api.cu; re-take the record if it
# changes).
FWD_SOURCES = ("common.cuh", "fwd_schedule.h", "kernel_ws.cuh", "philox.cuh", "ptx.cuh")
BWD_SOURCES = ("attn_bwd.cu", "common.cuh", "kernel_bwd.cuh", "ptx.cuh")
PROJ_SOURCES = ("attn_proj.cu", "common.cuh", "kernel_proj.cuh", "ptx.cuh")


def _code_only(text: str) -> bytes:
    """Source text without comments and with whitespace runs collapsed, so that
    a comment edit leaves the hash (and the traffic record keyed by it) alone.
    String literals in these sources hold no comment markers."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split()).encode()


def kernel_source_hash(sources=FWD_SOURCES) -> str:
    csrc = os.path.join(ROOT, "causal_scaled_dot_gb300", "csrc")
    h = hashlib.sha256()
    for fn in sources:
        with open(os.path.join(csrc, fn), encoding="utf-8") as f:
            h.update(fn.encode() + b"\0" + _code_only(f.read()))
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, sources=FWD_SOURCES):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel sources; otherwise None."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    want = kernel_source_hash(sources)
    for line in open(path):
        f = line.split()
        if len(f) >= 3 and not line.startswith("#") and f[0] == want and f[1] == workload:
            return float(f[2])
    return None


class ClockSampler:
    """nvidia-smi clock/throttle sampling while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.15)
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()
        return False

    def summary(self):
        rows = [r for r in csv.reader(io.StringIO(self.out or "")) if len(r) >= 9]
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.strip() == "Active"})
        loaded = [s for s in sm if mx and s > 0.5 * max(mx)] or sm
        return {"sm_mhz": float(np.median(loaded)) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


def dist_init(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "gloo" if args.impl == "reference" else "nccl"
        dist.init_process_group(backend=backend)
    return rank, world, local


def reduce_max(value: float, world: int) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def host_cpu(cpuinfo: str = "/proc/cpuinfo") -> str:
    """The host CPU as the kernel names it (x86: the model name; Arm: implementer
    and part codes), for the CPU baseline; never raises."""
    machine = platform.machine() or "unknown"
    try:
        with open(cpuinfo) as f:
            info = f.read()
    except OSError:
        return machine
    name = re.search(r"^model name\s*:\s*(.+)$", info, re.M)
    if name:
        return f"{machine} {name.group(1).strip()}"
    impl = re.search(r"^CPU implementer\s*:\s*(\S+)", info, re.M)
    part = re.search(r"^CPU part\s*:\s*(\S+)", info, re.M)
    if impl and part:
        return f"{machine} implementer {impl.group(1)} part {part.group(1)}"
    return machine


def step_stats(per_step_ms, world: int) -> dict:
    """Median and minimum of the timed steps' CUDA-event times (the slowest rank's,
    as for ms_per_step); every rank must call it."""
    return {"ms_step_median": reduce_max(float(np.median(per_step_ms)), world),
            "ms_step_min": reduce_max(float(np.min(per_step_ms)), world)}


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# --------------------------------------------------------------------- oracle
def workload_mask(w, density: float):
    """The seeded per-head block mask of --mask-density: uint8 [Hq, nt, nt]."""
    from causal_scaled_dot_gb300.inputs import random_block_mask
    return random_block_mask(w.Hq, w.S, density, seed=w.seed)


def workload_window(w, window: int):
    """The element mask of --window: each query keeps the `window` keys ending at
    itself, shared by all heads, with the block mask of the blocks it touches."""
    from causal_scaled_dot_gb300.inputs import block_mask_of_keep_bits, window_keep_bits
    bits = window_keep_bits(w.S, window)
    return bits, block_mask_of_keep_bits(bits, w.S)


def window_keys(S: int, window: int) -> np.ndarray:
    """Keys each query row sees under the local window: [S]."""
    return np.minimum(np.arange(S) + 1, window)


def visible_keys(mask, S: int, causal: bool) -> np.ndarray:
    """Keys each query row sees under the block mask (and causality): [Hm, S]."""
    nt = mask.shape[1]
    i = np.arange(S)[:, None]
    start = (np.arange(nt) * 128)[None, :]
    end = np.minimum(i + 1, S) if causal else np.full_like(i, S)
    per_tile = np.clip(end - start, 0, 128)                     # [S, nt]
    return np.einsum("hsk,sk->hs", mask[:, i[:, 0] // 128, :].astype(np.int64), per_tile)


class OracleTimer:
    """The fp64 oracle as it stands, on all host cores, over bounded random
    samples of a workload's query rows.

    Each query row of a causal workload carries 2*S*D of the metric's FLOPs on
    average (4*B*Hq*S^2*D/2 spread over B*Hq*S rows), so a sample's FLOPs are
    rows * 2*S*D and its TFLOP/s is comparable with the GPU's.
    """

    def __init__(self, w, fp8: bool = False, mask=None, dropout_p8: int = 0, window=None):
        import oracle
        from causal_scaled_dot_gb300.inputs import qkv_bf16, qkv_e4m3
        self.oracle = oracle
        self.w = w
        self.fp8 = fp8
        gen = qkv_e4m3 if fp8 else qkv_bf16
        self.q, self.k, self.v = gen(w.B, w.Hq, w.Hkv, w.S, w.D, seed=w.seed, sigma=w.sigma)
        self.threads = oracle.default_threads()
        self.total = w.B * w.Hq * w.S
        self.row_flops = (2.0 if w.causal else 4.0) * w.S * w.D
        self.mask = mask
        self.p8 = dropout_p8
        self.window = window
        if mask is not None:
            self.keys = visible_keys(mask, w.S, w.causal)  # [mask heads, S]
            self.row_flops = 4.0 * w.D * float(self.keys.mean())
        if window is not None:
            self.bits, self.bm = workload_window(w, window)
            self.keys = window_keys(w.S, window)[None, :]
            self.row_flops = 4.0 * w.D * float(self.keys.mean())
        n = max(self.threads, 32)
        self.run(n, seed=12345)  # warm the library and the page cache
        t0 = time.perf_counter()
        self.run(n, seed=12346)
        self.sec_per_row = (time.perf_counter() - t0) / n

    def run(self, n, seed):
        rows = np.random.default_rng(seed).integers(0, self.total, n)
        if self.window is not None and self.p8:
            self.oracle.attention_ex(self.q, self.k, self.v, self.w.scale, self.w.causal, block_mask=self.bm,
                                     keep_bits=self.bits, dropout=(self.p8, DROPOUT_SEED, DROPOUT_OFFSET),
                                     rows=rows, nthreads=self.threads)
        elif self.window is not None:
            self.oracle.attention_keep(self.q, self.k, self.v, self.w.scale, self.bits, self.w.causal,
                                       block_mask=self.bm, rows=rows, nthreads=self.threads)
        elif self.mask is not None:
            self.oracle.attention_masked(self.q, self.k, self.v, self.w.scale, self.mask,
                                         self.w.causal, rows=rows, nthreads=self.threads)
        elif self.p8:
            self.oracle.attention_dropout(self.q, self.k, self.v, self.w.scale, self.p8,
                                          DROPOUT_SEED, DROPOUT_OFFSET, self.w.causal, rows=rows,
                                          nthreads=self.threads)
        elif self.fp8:
            self.oracle.attention_e4m3(self.q, self.k, self.v, self.w.scale, (1.0, 1.0, 1.0),
                                       self.w.causal, rows=rows, nthreads=self.threads)
        else:
            self.oracle.attention(self.q, self.k, self.v, self.w.scale, self.w.causal, rows=rows,
                                  nthreads=self.threads)
        return rows

    def flops_of(self, rows) -> float:
        if self.mask is None and self.window is None:
            return rows.size * self.row_flops
        S, Hq = self.w.S, self.w.Hq
        h = (rows // S) % Hq if self.keys.shape[0] > 1 else np.zeros_like(rows)
        return 4.0 * self.w.D * float(self.keys[h, rows % S].sum())

    def rows_for(self, seconds):
        return int(min(self.total, max(self.threads, seconds / max(self.sec_per_row, 1e-9))))

    def sample(self, seconds, seed):
        """Times one sample of about `seconds`; returns (TFLOP/s, rows, wall seconds)."""
        n = self.rows_for(seconds)
        t0 = time.perf_counter()
        rows = self.run(n, seed)
        dt = time.perf_counter() - t0
        return self.flops_of(rows) / dt / 1e12, n, dt


class OracleBwdTimer:
    """The fp64 oracle's gradients on a bounded sample of key/value heads (each
    with every query head of its group); a head carries 1/(B*Hkv) of the
    metric's FLOPs."""

    def __init__(self, w, mask=None, window=None, dropout_p8: int = 0):
        import oracle
        from causal_scaled_dot_gb300.inputs import gaussian_bf16, qkv_bf16
        self.oracle = oracle
        self.w = w
        self.mask = mask
        self.keep = None
        self.dropout = (dropout_p8, DROPOUT_SEED, DROPOUT_OFFSET) if dropout_p8 else None
        self.q, self.k, self.v = qkv_bf16(w.B, w.Hq, w.Hkv, w.S, w.D, seed=w.seed, sigma=w.sigma)
        self.do = gaussian_bf16((w.B, w.Hq, w.S, w.D), w.seed, 3)
        self.threads = oracle.default_threads()
        self.total = w.B * w.Hkv
        self.row_flops = 2.5 * w.flops / self.total  # per key/value head
        G = w.Hq // w.Hkv
        if mask is not None:  # per key/value head: 2.5 x 4D x its group's visible pairs
            vis = visible_keys(mask, w.S, w.causal).sum(axis=1)  # per mask head
            per_hq = vis if mask.shape[0] == w.Hq else np.repeat(vis, w.Hq)
            self.head_flops = np.array([2.5 * 4.0 * w.D * per_hq[(h % w.Hkv) * G:(h % w.Hkv + 1) * G].sum()
                                        for h in range(self.total)])
        if window is not None:  # every head: 2.5 x 4D x G x the window's kept pairs
            self.keep, self.mask = workload_window(w, window)
            self.head_flops = np.full(self.total, 2.5 * 4.0 * w.D * G * float(window_keys(w.S, window).sum()))
        t0 = time.perf_counter()
        self.run(1, seed=12345)
        self.sec_per_row = time.perf_counter() - t0

    def run(self, n, seed):
        heads = np.random.default_rng(seed).integers(0, self.total, n)
        self.oracle.attention_bwd(self.q, self.k, self.v, self.do, self.w.scale, self.w.causal,
                                  kv_heads=heads, nthreads=self.threads, block_mask=self.mask,
                                  keep_bits=self.keep, dropout=self.dropout)
        return heads

    def rows_for(self, seconds):
        return int(min(self.total, max(1, seconds / max(self.sec_per_row, 1e-9))))

    def sample(self, seconds, seed):
        n = self.rows_for(seconds)
        t0 = time.perf_counter()
        heads = self.run(n, seed)
        dt = time.perf_counter() - t0
        flops = n * self.row_flops if self.mask is None else float(self.head_flops[heads].sum())
        return flops / dt / 1e12, n, dt


def dropout_p8(args) -> int:
    return int(round(args.dropout * 256)) if args.dropout is not None else 0


def make_oracle_timer(args, w, mask=None):
    if args.pass_ == "bwd":
        return OracleBwdTimer(w, mask=mask, window=args.window, dropout_p8=dropout_p8(args))
    if args.pass_ == "proj":
        return OracleProjTimer(w)
    return OracleTimer(w, fp8=args.dtype == "fp8", mask=mask, dropout_p8=dropout_p8(args),
                       window=args.window)


def metric_name(args) -> str:
    if args.pass_ == "bwd":
        return BWD_METRIC
    if args.pass_ == "proj":
        return PROJ_METRIC
    return METRIC


def proj_inputs(w):
    """Seeded O [B, Hq, S, D], W [E, Hq*D] (E = Hq*D) and bias [E] of the projection step."""
    from causal_scaled_dot_gb300.inputs import gaussian_bf16
    E, K = w.Hq * w.D, w.Hq * w.D
    o = gaussian_bf16((w.B, w.Hq, w.S, w.D), w.seed, 0)
    wt = gaussian_bf16((E, K), w.seed, 1, sigma=1.0 / np.sqrt(K))
    bias = np.random.default_rng(w.seed).standard_normal(E).astype(np.float32)
    return o, wt, bias


class OracleProjTimer:
    """The oracle's float64 projection on a bounded sample of sequence positions."""

    def __init__(self, w):
        import oracle
        self.oracle = oracle
        self.w = w
        self.o, self.wt, self.bias = proj_inputs(w)
        self.threads = os.cpu_count() or 1
        self.total = w.S
        self.row_flops = 2.0 * w.B * (w.Hq * w.D) * (w.Hq * w.D)  # per position (all batch entries)
        t0 = time.perf_counter()
        self.run(16, seed=12345)
        self.sec_per_row = (time.perf_counter() - t0) / 16

    def run(self, n, seed):
        pos = np.sort(np.random.default_rng(seed).choice(self.w.S, size=n, replace=False))
        self.oracle.out_proj(self.o[:, :, pos], self.wt, self.bias)
        return pos

    def rows_for(self, seconds):
        return int(min(self.total, max(1, seconds / max(self.sec_per_row, 1e-9))))

    def sample(self, seconds, seed):
        n = self.rows_for(seconds)
        t0 = time.perf_counter()
        self.run(n, seed)
        dt = time.perf_counter() - t0
        return n * self.row_flops / dt / 1e12, n, dt


def window_config(w, window):
    if window is None:
        return {}
    return {"elem_mask": {"kind": "local window: query i keeps keys i-window < j <= i",
                          "window": window, "heads": 1,
                          "kept_pair_frac": float(window_keys(w.S, window).sum()) / (w.S * (w.S + 1) / 2),
                          "block_mask": "derived: the 128x128 blocks holding a kept pair"}}


def mask_config(mask, density):
    if mask is None:
        return {}
    return {"block_mask": {"density": density, "heads": int(mask.shape[0]),
                           "kept_block_frac": float(mask.mean())}}


def run_reference(args, w, rank, world):
    if rank != 0:
        return 0
    mask = workload_mask(w, args.mask_density) if args.mask_density is not None else None
    timer = make_oracle_timer(args, w, mask)
    # The whole run (warm-up and timed steps) stays within a few minutes.
    step_s = min(args.ref_step_seconds, args.ref_total_seconds / max(1, args.steps + args.warmup))
    for i in range(args.warmup):
        timer.sample(step_s, seed=1000 + i)
    samples = [timer.sample(step_s, seed=s + 1) for s in range(args.steps)]
    secs = sum(dt for _, _, dt in samples)
    value = sum(tf * dt for tf, _, dt in samples) / secs
    rows_per_step = int(np.mean([n for _, n, _ in samples]))
    what = {"bwd": "key/value heads (gradients)", "proj": "sequence positions (projection)"}.get(
        args.pass_, "query rows")
    how = "float64 numpy matmul" if args.pass_ == "proj" else "fp64 C oracle"
    sample = (f"{rows_per_step} random {what} of {w.name} per step "
              f"(of {timer.total}); {how}, {timer.threads} threads")
    line = {
        "impl": "reference", "metric": metric_name(args), "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": secs / len(samples) * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": f"synthetic (seeded N(0,1) {'e4m3' if args.dtype == 'fp8' else 'bf16'})",
        "config": {"workload": w.name, **w.shape_dict, "causal": w.causal,
                   "inputs": "e4m3" if args.dtype == "fp8" else "bf16", "pass": args.pass_,
                   **mask_config(mask, args.mask_density), **window_config(w, args.window),
                   **({"dropout_p": dropout_p8(args) / 256, "dropout_key": [DROPOUT_SEED, DROPOUT_OFFSET]}
                      if args.dropout is not None else {})},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": timer.threads, "cpu": host_cpu(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------------- ours
def run_ours(args, w, rank, world, local):
    import torch
    from causal_scaled_dot_gb300 import native
    from causal_scaled_dot_gb300.inputs import qkv_bf16, qkv_e4m3

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    native.load()
    fp8 = args.dtype == "fp8"
    if fp8:
        codes = qkv_e4m3(w.B, w.Hq, w.Hkv, w.S, w.D, seed=w.seed, sigma=w.sigma)
        qh, kh, vh = (torch.from_numpy(c).pin_memory() for c in codes)
    else:
        bits = qkv_bf16(w.B, w.Hq, w.Hkv, w.S, w.D, seed=w.seed, sigma=w.sigma)
        qh, kh, vh = (torch.from_numpy(b.view(np.int16).copy()).view(torch.bfloat16).pin_memory()
                      for b in bits)
    q, k, v = qh.to(dev), kh.to(dev), vh.to(dev)
    mask = workload_mask(w, args.mask_density) if args.mask_density is not None else None
    flops = w.flops
    if mask is not None:
        flops = 4.0 * w.D * w.B * float(visible_keys(mask, w.S, w.causal).sum())
        mask_d = torch.from_numpy(mask).to(dev)
    if args.window is not None:  # 4*D per kept (query, key) pair
        keep_bits, keep_block = workload_window(w, args.window)
        flops = 4.0 * w.D * w.B * w.Hq * float(window_keys(w.S, args.window).sum())
        keep_d, keep_block_d = torch.from_numpy(keep_bits).to(dev), torch.from_numpy(keep_block).to(dev)
        if args.dropout is not None:  # the window with dropout: one attn_fwd_ex call
            combo = native.options(block_mask=keep_block_d, keep_bits=keep_d, dropout_p=args.dropout,
                                   seed=DROPOUT_SEED, offset=DROPOUT_OFFSET)
    out = torch.empty((w.B, w.Hq, w.S, w.D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.B, w.Hq, w.S), dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step_on(q, k, v, out, lse, stream):
        if fp8:
            native.attn_fwd_fp8(q, k, v, 1.0, 1.0, 1.0, out, lse, w.B, w.Hq, w.Hkv, w.S, w.D,
                                w.scale, w.causal, stream)
        elif mask is not None:
            native.attn_fwd_block_masked(q, k, v, out, lse, w.B, w.Hq, w.Hkv, w.S, w.D, w.scale,
                                         w.causal, mask_d, mask.shape[0], stream)
        elif args.window is not None and args.dropout is not None:
            native.attn_fwd_ex(q, k, v, out, lse, w.B, w.Hq, w.Hkv, w.S, w.D, w.scale, w.causal, combo,
                               stream)
        elif args.window is not None:
            native.attn_fwd_elem_masked(q, k, v, out, lse, w.B, w.Hq, w.Hkv, w.S, w.D, w.scale,
                                        w.causal, keep_d, 1, keep_block_d, 1, stream)
        elif args.dropout is not None:
            native.attn_fwd_dropout(q, k, v, out, lse, w.B, w.Hq, w.Hkv, w.S, w.D, w.scale, w.causal,
                                    args.dropout, DROPOUT_SEED, DROPOUT_OFFSET, stream)
        else:
            native.attn_fwd(q, k, v, out, lse, w.B, w.Hq, w.Hkv, w.S, w.D, w.scale, w.causal,
                            stream)

    def step():
        step_on(q, k, v, out, lse, stream)

    for _ in range(args.warmup):
        flush.fill_(1.0)
        step()
    torch.cuda.synchronize(dev)
    native.attn_sync_status(stream)

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    launches = 0
    barrier(world)
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        wall0 = time.perf_counter()
        for i in range(args.steps):
            flush.fill_(float(i))
            starts[i].record(stream)
            step()
            launches += 1
            ends[i].record(stream)
        torch.cuda.synchronize(dev)
        wall = time.perf_counter() - wall0
    barrier(world)
    native.attn_sync_status(stream)
    per_step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms_local = float(np.mean(per_step_ms))
    ms = reduce_max(ms_local, world)
    stats = step_stats(per_step_ms, world)
    value = world * flops / (ms * 1e-3) / 1e12

    # Warm L2: the same steps back to back with no flush in between (inputs
    # resident in L2 as far as it holds them, as for consecutive layers that
    # reuse a buffer); reported beside the cold-L2 headline, not instead of it.
    warm_steps = min(args.steps, 200)
    w_starts = [torch.cuda.Event(enable_timing=True) for _ in range(warm_steps)]
    w_ends = [torch.cuda.Event(enable_timing=True) for _ in range(warm_steps)]
    for _ in range(3):
        step()
    barrier(world)
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk_warm:
        for i in range(warm_steps):
            w_starts[i].record(stream)
            step()
            w_ends[i].record(stream)
        torch.cuda.synchronize(dev)
    barrier(world)
    native.attn_sync_status(stream)
    warm_ms = reduce_max(float(np.mean([a.elapsed_time(b) for a, b in zip(w_starts, w_ends)])), world)

    # Host time per call: the Python entry point (argument checks, ctypes) and,
    # for the plain forward, the C entry point alone through ctypes.
    host_py = host_us_per_call(step)
    host_c = None
    if not fp8 and mask is None and args.window is None and args.dropout is None:
        lib = native.load()
        c_args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(), w.B, w.Hq, w.Hkv,
                  w.S, w.D, w.scale, 1 if w.causal else 0, stream.cuda_stream)
        host_c = host_us_per_call(lambda: lib.attn_fwd(*c_args))
    torch.cuda.synchronize(dev)
    native.attn_sync_status(stream)

    # End to end: every step copies its Q, K, V from pinned host buffers, runs
    # the call and copies O and LSE back, all inside the timed region.  Steps are
    # pipelined as a stream of independent requests would be: two device buffer
    # sets, uploads on one copy stream and downloads on another, so step i+1's
    # upload and step i-1's download overlap step i's kernel.  (The host link
    # carries about 190 GB/s of pinned uploads here; more upload streams did not
    # raise it.)
    e2e_steps = max(4, min(args.steps, 40))
    sets = [(q, k, v, out, lse)] + [tuple(torch.empty_like(t) for t in (q, k, v, out, lse))]
    outs_h = [(torch.empty(out.shape, dtype=out.dtype).pin_memory(),
               torch.empty(lse.shape, dtype=lse.dtype).pin_memory()) for _ in range(2)]
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = {n: [torch.cuda.Event() for _ in range(2)] for n in ("up", "run", "down")}

    def e2e_run(n):
        for i in range(n):
            b = i % 2
            qb, kb, vb, ob, lb = sets[b]
            with torch.cuda.stream(up):
                if i >= 2:
                    up.wait_event(ev["run"][b])          # step i-2 has read this set
                for dst, src in ((qb, qh), (kb, kh), (vb, vh)):
                    dst.copy_(src, non_blocking=True)
                ev["up"][b].record(up)
            stream.wait_event(ev["up"][b])
            if i >= 2:
                stream.wait_event(ev["down"][b])         # step i-2's results are on the host
            step_on(qb, kb, vb, ob, lb, stream)
            ev["run"][b].record(stream)
            with torch.cuda.stream(down):
                down.wait_event(ev["run"][b])
                outs_h[b][0].copy_(ob, non_blocking=True)
                outs_h[b][1].copy_(lb, non_blocking=True)
                ev["down"][b].record(down)

    e2e_run(2)
    torch.cuda.synchronize(dev)
    barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    up.wait_event(e0)
    e2e_run(e2e_steps)
    stream.wait_stream(up)
    stream.wait_stream(down)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = reduce_max(e0.elapsed_time(e1) / e2e_steps, world)
    h2d = sum(t.numel() * t.element_size() for t in (qh, kh, vh))
    d2h = sum(t.numel() * t.element_size() for t in outs_h[0])

    if rank != 0:
        return 0
    peaks, peak_src = load_peaks()
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    peak_what = f"{peak_src} bf16 dense (burst)"
    if fp8:  # the E4M3 GEMM peak of this GPU, measured now
        peak = measure_fp8_peak(dev)
        peak_what = "measured in this run: E4M3 GEMM (torch._scaled_mm, cuBLASLt) 8192^3, best of 10"
    achieved = flops / (ms_local * 1e-3) / 1e12
    variant = (w.name + (":fp8" if fp8 else "") + (f":mask{args.mask_density}" if mask is not None else "")
               + (f":dropout{args.dropout}" if args.dropout is not None else "")
               + (f":window{args.window}" if args.window is not None else ""))
    traffic = recorded_traffic(variant)
    # algorithmic bytes: inputs read once (1 byte per element for E4M3), O and LSE written once
    io_bytes = w.io_bytes - (w.B * (w.Hq + 2 * w.Hkv) * w.S * w.D if fp8 else 0)
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        timer = OracleTimer(w, fp8=fp8, mask=mask, dropout_p8=dropout_p8(args), window=args.window)
        tf, n, dt = timer.sample(args.cpu_seconds, seed=7)
        cpu = {"value": tf, "unit": "TFLOP/s", "cores": timer.threads, "cpu": host_cpu(), "kind": "oracle",
               "sample": f"{n} random query rows of {w.name} (of {timer.total}), "
                         f"{dt:.1f} s; fp64 C oracle"}
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, **stats,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp8 (e4m3 inputs, bf16 output)" if fp8 else "bf16",
        "data": f"synthetic (seeded N(0,1) {'e4m3' if fp8 else 'bf16'}, no weights)",
        "config": {"workload": w.name, **w.shape_dict, "causal": w.causal,
                   "inputs": "e4m3" if fp8 else "bf16", **mask_config(mask, args.mask_density),
                   **window_config(w, args.window),
                   **({"dropout_p": dropout_p8(args) / 256, "dropout_key": [DROPOUT_SEED, DROPOUT_OFFSET]}
                      if args.dropout is not None else {}),
                   "l2": "flushed between timed steps (256 MiB write)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "pct_of_peak": 100.0 * achieved / peak,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "peak_source": peak_what,
                     "hbm_gbs": io_bytes / (ms_local * 1e-3) / 1e9},
        "cpu_baseline": cpu,
        "e2e": {"value": world * flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "steps": e2e_steps,
                "pipelining": "two buffer sets; uploads and downloads on their own streams overlap "
                              "the neighbouring steps' kernels"},
        "gpu_launches": launches,
        "clocks": clk.summary(),
        "wall_s_timed_region": wall,
        "warm_l2": {"value": world * flops / (warm_ms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": warm_ms,
                    "steps": warm_steps, "l2": "not flushed: the same call back to back",
                    "clocks": clk_warm.summary()},
        "host_us_per_call": {"python_entry": host_py, "c_entry": host_c,
                             "what": "host time of one asynchronous call, median of 5 x 200 calls; "
                                     "c_entry = attn_fwd through ctypes (about 1.2 us of it is the ctypes call)"},
        "kernel_sources": kernel_source_hash(),
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours_bwd(args, w, rank, world, local):
    """attn_bwd timed like the forward: inputs (Q, K, V, O, dO, LSE) resident,
    L2 flushed between steps, CUDA events on the launching stream."""
    import torch
    from causal_scaled_dot_gb300 import native
    from causal_scaled_dot_gb300.inputs import gaussian_bf16, qkv_bf16

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    native.load()

    def host(bits):
        return torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).pin_memory()

    qh, kh, vh = (host(b) for b in qkv_bf16(w.B, w.Hq, w.Hkv, w.S, w.D, seed=w.seed, sigma=w.sigma))
    doh = host(gaussian_bf16((w.B, w.Hq, w.S, w.D), w.seed, 3))
    q, k, v, do = qh.to(dev), kh.to(dev), vh.to(dev), doh.to(dev)
    out = torch.empty_like(q)
    lse = torch.empty((w.B, w.Hq, w.S), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    mask = workload_mask(w, args.mask_density) if args.mask_density is not None else None
    if mask is not None:
        mask_d = torch.from_numpy(mask).to(dev)
        native.attn_fwd_block_masked(q, k, v, out, lse, w.B, w.Hq, w.Hkv, w.S, w.D, w.scale, w.causal,
                                     mask_d, mask.shape[0], stream)
    elif args.window is not None:
        keep_bits, keep_block = workload_window(w, args.window)
        keep_d, keep_block_d = torch.from_numpy(keep_bits).to(dev), torch.from_numpy(keep_block).to(dev)
        if args.dropout is not None:  # the window with dropout: attn_fwd_ex / attn_bwd_ex
            combo = native.options(block_mask=keep_block_d, keep_bits=keep_d, dropout_p=args.dropout,
                                   seed=DROPOUT_SEED, offset=DROPOUT_OFFSET)
            native.attn_fwd_ex(q, k, v, out, lse, w.B, w.Hq, w.Hkv, w.S, w.D, w.scale, w.causal, combo, stream)
        else:
            native.attn_fwd_elem_masked(q, k, v, out, lse, w.B, w.Hq, w.Hkv, w.S, w.D, w.scale, w.causal,
                                        keep_d, 1, keep_block_d, 1, stream)
    elif args.dropout is not None:
        native.attn_fwd_dropout(q, k, v, out, lse, w.B, w.Hq, w.Hkv, w.S, w.D, w.scale, w.causal,
                                args.dropout, DROPOUT_SEED, DROPOUT_OFFSET, stream)
    else:
        native.attn_fwd(q, k, v, out, lse, w.B, w.Hq, w.Hkv, w.S, w.D, w.scale, w.causal, stream)
    outh, lseh = out.cpu().pin_memory(), lse.cpu().pin_memory()
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    delta = torch.empty_like(lse)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flops = 2.5 * w.flops
    if mask is not None:  # 2.5x the forward's FLOPs over the visible pairs
        flops = 2.5 * 4.0 * w.D * w.B * float(visible_keys(mask, w.S, w.causal).sum())
    if args.window is not None:  # ... over the kept pairs
        flops = 2.5 * 4.0 * w.D * w.B * w.Hq * float(window_keys(w.S, args.window).sum())

    def step():
        if mask is not None:
            native.attn_bwd_block_masked(q, k, v, out, do, lse, delta, dq, dk, dv, w.B, w.Hq, w.Hkv,
                                         w.S, w.D, w.scale, w.causal, mask_d, mask.shape[0], stream)
        elif args.window is not None and args.dropout is not None:
            native.attn_bwd_ex(q, k, v, out, do, lse, delta, dq, dk, dv, w.B, w.Hq, w.Hkv, w.S, w.D,
                               w.scale, w.causal, combo, stream)
        elif args.window is not None:
            native.attn_bwd_elem_masked(q, k, v, out, do, lse, delta, dq, dk, dv, w.B, w.Hq, w.Hkv,
                                        w.S, w.D, w.scale, w.causal, keep_d, 1, keep_block_d, 1, stream)
        elif args.dropout is not None:
            native.attn_bwd_dropout(q, k, v, out, do, lse, delta, dq, dk, dv, w.B, w.Hq, w.Hkv, w.S,
                                    w.D, w.scale, w.causal, args.dropout, DROPOUT_SEED, DROPOUT_OFFSET,
                                    stream)
        else:
            native.attn_bwd(q, k, v, out, do, lse, delta, dq, dk, dv, w.B, w.Hq, w.Hkv, w.S, w.D,
                            w.scale, w.causal, stream)

    for _ in range(args.warmup):
        flush.fill_(1.0)
        step()
    torch.cuda.synchronize(dev)
    native.attn_sync_status(stream)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    launches = 0
    barrier(world)
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        wall0 = time.perf_counter()
        for i in range(args.steps):
            flush.fill_(float(i))
            starts[i].record(stream)
            step()
            launches += 2  # the dQ kernel and the dK/dV kernel
            ends[i].record(stream)
        torch.cuda.synchronize(dev)
        wall = time.perf_counter() - wall0
    barrier(world)
    native.attn_sync_status(stream)
    per_step_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    ms_local = float(np.mean(per_step_ms))
    ms = reduce_max(ms_local, world)
    stats = step_stats(per_step_ms, world)
    value = world * flops / (ms * 1e-3) / 1e12

    # End to end: Q, K, V, O, dO, LSE from pinned host buffers, dQ, dK, dV back.
    dqh, dkh, dvh = (torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in (dq, dk, dv))
    e2e_steps = max(3, min(args.steps, 20))

    def e2e_step():
        for d, h in ((q, qh), (k, kh), (v, vh), (out, outh), (do, doh), (lse, lseh)):
            d.copy_(h, non_blocking=True)
        step()
        for h, d in ((dqh, dq), (dkh, dk), (dvh, dv)):
            h.copy_(d, non_blocking=True)

    e2e_step()
    torch.cuda.synchronize(dev)
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = reduce_max(e0.elapsed_time(e1) / e2e_steps, world)
    h2d = sum(t.numel() * t.element_size() for t in (qh, kh, vh, outh, doh, lseh))
    d2h = sum(t.numel() * t.element_size() for t in (dqh, dkh, dvh))

    if rank != 0:
        return 0
    peaks, peak_src = load_peaks()
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    achieved = flops / (ms_local * 1e-3) / 1e12
    # algorithmic bytes: Q, K, V, O, dO and LSE read once; dQ, dK, dV written
    # once; delta written by the first kernel and read by the second.
    q_b = w.B * w.Hq * w.S * w.D * 2
    kv_b = w.B * w.Hkv * w.S * w.D * 2
    row_b = w.B * w.Hq * w.S * 4
    io_bytes = 3 * q_b + 2 * kv_b + row_b + q_b + 2 * kv_b + 2 * row_b
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        timer = OracleBwdTimer(w, mask=mask, window=args.window, dropout_p8=dropout_p8(args))
        tf, n, dt = timer.sample(args.cpu_seconds, seed=7)
        cpu = {"value": tf, "unit": "TFLOP/s", "cores": timer.threads, "cpu": host_cpu(), "kind": "oracle",
               "sample": f"gradients of {n} random key/value heads of {w.name} (of {timer.total}), "
                         f"{dt:.1f} s; fp64 C oracle"}
    line = {
        "metric": BWD_METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, **stats,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16 Q, K, V, dO; no weights)",
        "config": {"workload": w.name, **w.shape_dict, "causal": w.causal, "inputs": "bf16",
                   "pass": "bwd", **mask_config(mask, args.mask_density), **window_config(w, args.window),
                   **({"dropout_p": dropout_p8(args) / 256, "dropout_key": [DROPOUT_SEED, DROPOUT_OFFSET]}
                      if args.dropout is not None else {}),
                   "l2": "flushed between timed steps (256 MiB write)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "pct_of_peak": 100.0 * achieved / peak,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak,
                     "traffic": recorded_traffic(w.name + ":bwd" + (f":mask{args.mask_density}" if mask is not None
                                                                   else "")
                                                 + (f":window{args.window}" if args.window is not None else "")
                                                 + (f":dropout{args.dropout}" if args.dropout is not None else ""),
                                                 BWD_SOURCES),
                     "peak_source": f"{peak_src} bf16 dense (burst)",
                     "kernel": "attn_bwd call (dQ kernel + dK/dV kernel)",
                     "hbm_gbs": io_bytes / (ms_local * 1e-3) / 1e9},
        "cpu_baseline": cpu,
        "e2e": {"value": world * flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
        "gpu_launches": launches,
        "clocks": clk.summary(),
        "wall_s_timed_region": wall,
        "kernel_sources": kernel_source_hash(BWD_SOURCES),
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours_proj(args, w, rank, world, local):
    """attn_out_proj timed like the forward: O, W, bias resident, L2 flushed
    between steps, CUDA events on the launching stream."""
    import torch
    from causal_scaled_dot_gb300 import native

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    native.load()
    o_bits, w_bits, bias_np = proj_inputs(w)
    E, K = w.Hq * w.D, w.Hq * w.D

    def host(bits):
        return torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).pin_memory()

    oh, wh = host(o_bits), host(w_bits)
    bh = torch.from_numpy(bias_np).pin_memory()
    o, wt, bias = oh.to(dev), wh.to(dev), bh.to(dev)
    y = torch.empty((w.B, w.S, E), dtype=torch.bfloat16, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    flops = 2.0 * w.B * w.S * E * K

    def step():
        native.attn_out_proj(o, wt, bias, y, w.B, w.Hq, w.S, w.D, E, stream)

    for _ in range(args.warmup):
        flush.fill_(1.0)
        step()
    torch.cuda.synchronize(dev)
    native.attn_sync_status(stream)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    launches = 0
    barrier(world)
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        wall0 = time.perf_counter()
        for i in range(args.steps):
            flush.fill_(float(i))
            starts[i].record(stream)
            step()
            launches += 1
            ends[i].record(stream)
        torch.cuda.synchronize(dev)
        wall = time.perf_counter() - wall0
    barrier(world)
    native.attn_sync_status(stream)
    per_step_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    ms_local = float(np.mean(per_step_ms))
    ms = reduce_max(ms_local, world)
    stats = step_stats(per_step_ms, world)
    value = world * flops / (ms * 1e-3) / 1e12

    yh = torch.empty(y.shape, dtype=y.dtype).pin_memory()
    e2e_steps = max(3, min(args.steps, 20))

    def e2e_step():
        o.copy_(oh, non_blocking=True)
        wt.copy_(wh, non_blocking=True)
        bias.copy_(bh, non_blocking=True)
        step()
        yh.copy_(y, non_blocking=True)

    e2e_step()
    torch.cuda.synchronize(dev)
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = reduce_max(e0.elapsed_time(e1) / e2e_steps, world)
    h2d = sum(t.numel() * t.element_size() for t in (oh, wh, bh))
    d2h = yh.numel() * yh.element_size()

    if rank != 0:
        return 0
    peaks, peak_src = load_peaks()
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    achieved = flops / (ms_local * 1e-3) / 1e12
    io_bytes = o.numel() * 2 + wt.numel() * 2 + E * 4 + y.numel() * 2
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        timer = OracleProjTimer(w)
        tf, n, dt = timer.sample(args.cpu_seconds, seed=7)
        cpu = {"value": tf, "unit": "TFLOP/s", "cores": timer.threads, "cpu": host_cpu(), "kind": "oracle",
               "sample": f"{n} random sequence positions of {w.name} (of {timer.total}, all batch "
                         f"entries), {dt:.1f} s; float64 numpy matmul"}
    line = {
        "metric": PROJ_METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, **stats,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16 attention output, N(0, 1/(H*D)) weights; no trained weights)",
        "config": {"workload": w.name, **w.shape_dict, "E": E, "inputs": "bf16", "pass": "proj",
                   "l2": "flushed between timed steps (256 MiB write)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "pct_of_peak": 100.0 * achieved / peak,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": recorded_traffic(w.name + ":proj", PROJ_SOURCES),
                     "peak_source": f"{peak_src} bf16 dense (burst)",
                     "hbm_gbs": io_bytes / (ms_local * 1e-3) / 1e9},
        "cpu_baseline": cpu,
        "e2e": {"value": world * flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
        "gpu_launches": launches,
        "clocks": clk.summary(),
        "wall_s_timed_region": wall,
        "kernel_sources": kernel_source_hash(PROJ_SOURCES),
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=HEADLINE.name, choices=sorted(BY_NAME))
    ap.add_argument("--dtype", default="bf16", choices=["bf16", "fp8"],
                    help="input format: bf16 (attn_fwd) or E4M3 (attn_fwd_fp8, D = 128 only)")
    ap.add_argument("--pass", dest="pass_", default="fwd", choices=["fwd", "bwd", "proj"],
                    help="fwd: attn_fwd (default); bwd: attn_bwd; proj: attn_out_proj (bf16)")
    ap.add_argument("--mask-density", type=float, default=None,
                    help="bf16 only: run attn_fwd_block_masked with a seeded per-head block mask "
                         "keeping each 128x128 block with this probability")
    ap.add_argument("--dropout", type=float, default=None,
                    help="bf16 only: attn_fwd_dropout (with --pass bwd: attn_bwd_dropout) with this "
                         "drop probability (rounded to a multiple of 1/256)")
    ap.add_argument("--window", type=int, default=None,
                    help="bf16 only: attn_fwd_elem_masked (with --pass bwd: attn_bwd_elem_masked) with a "
                         "local window of this many keys per query (element mask) and the block mask it "
                         "implies")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="budget of the oracle CPU-baseline sample")
    ap.add_argument("--ref-step-seconds", type=float, default=8.0,
                    help="--impl reference: at most this many oracle seconds per step")
    ap.add_argument("--ref-total-seconds", type=float, default=120.0,
                    help="--impl reference: oracle seconds for the whole run")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.mask_density is not None and (args.dtype != "bf16" or not 0.0 <= args.mask_density <= 1.0):
        ap.error("--mask-density takes a probability in [0, 1] and bf16 inputs")
    if args.pass_ in ("bwd", "proj") and args.dtype != "bf16":
        ap.error("--pass bwd / proj take bf16 inputs")
    if args.pass_ == "proj" and args.mask_density is not None:
        ap.error("--pass proj takes no mask")
    if args.dropout is not None and (args.pass_ == "proj" or args.dtype != "bf16" or args.mask_density is not None
                                     or not 0 < round(args.dropout * 256) < 256):
        ap.error("--dropout takes 0 < p < 1 (at least 1/256), bf16 forward or backward, no mask")
    if args.window is not None and (args.window < 1 or args.pass_ == "proj" or args.dtype != "bf16"
                                    or args.mask_density is not None):
        ap.error("--window takes a positive key count, bf16 forward or backward, no other mask")
    w = BY_NAME[args.workload]
    rank, world, local = dist_init(args)
    if world != args.gpus and rank == 0:
        print(f"note: --gpus {args.gpus} but WORLD_SIZE {world}", file=sys.stderr)
    try:
        if args.impl == "reference":
            rc = run_reference(args, w, rank, world)
        else:
            rc = {"bwd": run_ours_bwd, "proj": run_ours_proj}.get(args.pass_, run_ours)(
                args, w, rank, world, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
    return rc


if __name__ == "__main__":
    sys.exit(main())

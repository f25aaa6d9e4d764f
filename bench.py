#!/usr/bin/env python
"""Benchmark of the Nyström self-attention forward pass on GB300.

Metric: tokens/s = B*H*n / time of one forward pass over one batch, with the
inputs resident in HBM (``value``), and end to end through the host-buffer
C ABI call with the host<->device copies inside the timed region (``e2e``).

One step = one full forward pass (landmarks, landmark rows, pseudo-inverse,
token rows + conv + store) over the workload's whole batch. Between timed
steps the inputs rotate over several copies whose total exceeds L2, so no
step starts with its inputs in L2.

--impl reference times the fp64 CPU oracle (the only reference there is) on
the host cores, on a bounded sample of the same workload per step.
Under torchrun every rank runs its own full replica of the workload (heads
are independent, no data-path collective: weak scaling); the time is the
max over ranks and ``value`` counts the tokens of all ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads  # noqa: E402

METRIC = "Nyström attn fwd tokens/s (B·H·n per s) at 1 GB300; % of HBM/tensor roofline"
L2_BYTES = 126 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=None,
                   help="timed steps (default: enough for about 3 s)")
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--config", default="c5", choices=workloads.ORDER,
                   help="workload (default c5, the largest: B=2 H=16 n=32768 d=128 m=256, bf16)")
    p.add_argument("--others", default="c2,c3,c4",
                   help="comma-separated workloads timed briefly after the main one and "
                        "reported under other_workloads ('' for none)")
    p.add_argument("--no-scan", action="store_true",
                   help="skip the sequence-length scan reported under linear_scan")
    p.add_argument("--no-next", action="store_true",
                   help="skip the module / variants / clustered timings reported under next_rows")
    p.add_argument("--min-region-s", type=float, default=1.0,
                   help="repeat the K-step timed region until this much wall time has passed "
                        "(so the clock sampler sees the timed work)")
    p.add_argument("--batch", type=int, default=None,
                   help="override the workload's batch size B (smaller cases for profiler captures)")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=12.0,
                   help="CPU work budget of the oracle baseline sample")
    p.add_argument("--scan-n", default=None,
                   help="comma-separated sequence lengths: time one pass at each n with the "
                        "workload's other sizes fixed, one JSON line per n (linear-time check)")
    return p.parse_args()


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def reduce_over_ranks(x, op, device, world):
    """x reduced with op (a torch.distributed ReduceOp) over all ranks; x
    itself on a single rank."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=op)
    return float(t.item())


def job_throughput(tokens_per_rank_step, world, steps, elapsed_ms):
    """Whole-job tokens/s: every rank's tokens over the slowest rank's time."""
    return tokens_per_rank_step * world * steps / (elapsed_ms / 1e3)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------ clocks ----

class ClockSampler:
    """nvidia-smi clock / throttle-reason samples every `period_ms` ms."""
    FIELDS = ["timestamp", "index", "clocks.sm", "clocks.max.sm", "power.draw",
              "clocks_event_reasons.active", "clocks_event_reasons.hw_slowdown",
              "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, gpu_index: int, period_ms: int = 50):
        self.gpu_index = gpu_index
        self.period_ms = period_ms
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={','.join(self.FIELDS)}", "--format=csv,noheader,nounits",
                 "-lms", str(self.period_ms)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) == len(self.FIELDS):
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float) -> dict:
        mine = [p for (t, p) in self.samples if p[1] == str(self.gpu_index)] or \
               [p for (t, p) in self.samples]
        inside = [p for (t, p) in self.samples if t0 <= t <= t1 and p in mine]
        use = inside if inside else mine
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[2]) for p in use if num(p[2]) is not None]
        smax = [num(p[3]) for p in use if num(p[3]) is not None]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for p in use:
            for nm, val in zip(names, p[6:10]):
                if val.strip().lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(use),
                "samples_in_timed_region": len(inside)}


REJECTING_REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown")


def clocks_rejected(clocks: dict) -> bool:
    """A timed region that saw a hardware or thermal slowdown, or whose SM
    clock sat well below its maximum with no reason given (a clock lock left
    by someone else), does not stand. sw_power_cap alone is kept."""
    if any(r in clocks.get("reasons", []) for r in REJECTING_REASONS):
        return True
    sm, smax = clocks.get("sm_mhz"), clocks.get("sm_max_mhz")
    return bool(sm and smax and sm < 0.8 * smax and not clocks.get("reasons"))


# --------------------------------------------------------------- CPU oracle ----

def oracle_sample(inp, budget_s: float, max_heads: int | None = None):
    """Run the fp64 oracle head by head until ``budget_s`` is spent (at least
    one head). Returns (tokens, seconds, heads)."""
    from oracle import nystrom_ref as R
    wl = inp.wl
    heads = [(b, h) for b in range(wl.B) for h in range(wl.H)]
    if max_heads is not None:
        heads = heads[:max_heads]
    done = 0
    t0 = time.perf_counter()
    while True:  # whole passes over the heads until the budget is spent
        for b, h in heads:
            R.nystrom_head(inp.q[b, h], inp.k[b, h], inp.v[b, h], inp.conv_w[h], wl.m, wl.iters)
            done += 1
            if time.perf_counter() - t0 >= budget_s:
                break
        if time.perf_counter() - t0 >= budget_s or max_heads is not None:
            break
    dt = time.perf_counter() - t0
    return done * wl.n, dt, done


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# --------------------------------------------------------------- reference ----

def run_reference(args, wl):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    inp = workloads.make_inputs(wl)
    # per-step sample: whole heads, sized so warmup + steps stay within ~150 s
    _, t_head, _ = oracle_sample(inp, 0.0, max_heads=1)
    steps = args.steps if args.steps is not None else 10
    per_step_budget = max(t_head, min(3.0, 150.0 / max(1, steps + args.warmup)))
    heads_per_step = max(1, min(wl.heads, int(per_step_budget / max(t_head, 1e-6))))
    for _ in range(args.warmup):
        oracle_sample(inp, 1e9, max_heads=heads_per_step)
    tokens = 0
    t0 = time.perf_counter()
    for _ in range(steps):
        tk, _, _ = oracle_sample(inp, 1e9, max_heads=heads_per_step)
        tokens += tk
    dt = time.perf_counter() - t0
    value = tokens / dt
    sample = (f"{heads_per_step} of {wl.heads} heads (n={wl.n}) per step; "
              f"fp64 numpy oracle, BLAS threads = library default")
    line = {
        "impl": "reference", "metric": METRIC, "value": value,
        "unit": "tokens/s", "n_gpus": args.gpus, "steps": steps, "warmup": args.warmup,
        "ms_per_step": dt / steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded normal draws)",
        "config": {"workload": wl.describe()},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cpu_cores(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------- ours ----

# Per-kernel roofline model: algorithmic HBM bytes in units of T*e
# (T = B*H*n*d elements, e = element bytes), or algorithmic flops.
KERNEL_BYTES = {
    "landmarks_vec": 2.0, "landmarks_small": 2.0, "landmarks_simt": 2.0,  # read Q, K
    "rows_tc": 2.0, "rows_simt": 2.0, "rows_x3": 2.0,  # read K, V
    "tokens_tc": 3.0, "tokens_simt": 3.0, "tokens_big": 3.0,  # read Q, V; write out
    "tokens_x3": 3.0,                             # read Q, V; write out (the conv fused)
    "conv_mask": 3.0,                             # read V, out; write out
}
KERNEL_SOURCES = {
    "landmarks_vec": "nys_simt.cu", "landmarks_small": "nys_simt.cu",
    "landmarks_simt": "nys_simt.cu", "rows_simt": "nys_simt.cu",
    "pinv_simt": "nys_simt.cu", "tokens_simt": "nys_simt.cu", "rows_tc": "nys_rows_tc.cu",
    "pinv_tc": "nys_pinv_tc.cu", "tokens_tc": "nys_tokens_tc.cu", "pinv_big": "nys_pinv_big.cu",
    "tokens_big": "nys_tokens_big.cu", "w_tc": "nys_pinv_tc.cu", "merge_g": "nys_simt.cu",
    "rows_x3": "nys_x3.cu", "tokens_x3": "nys_x3.cu", "conv_mask": "nys_simt.cu",
}
TF32_OVER_BF16 = 1.1 / 2.25  # nominal dense tensor rates


def pinv_flops(wl, with_w=True):
    """Algorithmic flops of the landmark kernel, the iteration and (unless a
    separate kernel forms it) W = Z G."""
    m, d = wl.m, wl.d
    return wl.heads * (2.0 * m * m * d + 8.0 * wl.iters * m ** 3 + (2.0 * m * m * d if with_w else 0.0))


def pinv_peak_time(wl, bf16_tflops, with_w=True):
    """Seconds the pseudo-inverse kernel's flops take at the tensor peaks of
    the types they run in: the scores and W = Z G in tf32; the update
    products in tf32 for m <= 128 and with fp16 operands (the bf16/fp16 rate)
    for m > 128. fp32 inputs: three tf32 products per product (a third of
    the tf32 rate)."""
    m, d = wl.m, wl.d
    tf32 = bf16_tflops * TF32_OVER_BF16 * 1e12
    if wl.dtype == "f32":  # fp32 inputs: every product is three tf32 products
        return pinv_flops(wl, with_w) / (tf32 / 3.0)
    upd = wl.heads * 8.0 * wl.iters * m ** 3
    rest = pinv_flops(wl, with_w) - upd
    return rest / tf32 + upd / (bf16_tflops * 1e12 if m > 128 else tf32)


def kernel_source_hash(kernel):
    import hashlib
    src = os.path.join(ROOT, "nystr_self_attention_gb300", "csrc", KERNEL_SOURCES.get(kernel, ""))
    if not os.path.isfile(src):
        return None
    return hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]


def measured_traffic(kernel, wl):
    """DRAM bytes per launch from profiles/dram_traffic.txt (written from an ncu
    capture), only if the kernel's source is unchanged since the capture. A
    workload captured at a smaller batch (entry "<name>b<B>") is scaled to
    this batch: every kernel streams each head once, so its bytes grow with
    the number of heads."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    h = kernel_source_hash(kernel)
    scaled = None
    for line in open(path):
        parts = line.split()
        if len(parts) != 4 or line.startswith("#") or parts[0] != kernel or parts[2] != h:
            continue
        if parts[1] == wl.name:
            return float(parts[3])
        tag = parts[1]
        if tag.startswith(wl.name + "b") and tag[len(wl.name) + 1:].isdigit():
            scaled = float(parts[3]) * wl.B / int(tag[len(wl.name) + 1:])
    return scaled


def roofline_for(kernel, ms, launches, per_step, wl, peaks, peak_src, w_separate=False):
    """Roofline of one kernel: `launches` launches took `ms` in total, and
    `per_step` launches make up one forward pass (the batch is split into
    that many head groups), so one launch covers 1/per_step of the work.
    Per-kernel times are short event-timed launches, so the tensor peak is
    the burst figure. `w_separate`: W = Z G is formed by its own kernel
    (w_tc), so the pseudo-inverse kernel is not credited with it."""
    t_launch = ms / launches / 1e3
    te = wl.B * wl.H * wl.n * wl.d * wl.elem_bytes / per_step
    traffic = measured_traffic(kernel, wl)
    if kernel in KERNEL_BYTES:
        achieved = KERNEL_BYTES[kernel] * te / t_launch / 1e9
        return {"kernel": kernel, "bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"], "traffic": traffic,
                "algorithmic_bytes": KERNEL_BYTES[kernel] * te,
                "peak_source": f"hbm_gbs ({peak_src})"}
    if kernel == "w_tc":  # W = Z G alone
        flops = wl.heads * 2.0 * wl.m * wl.m * wl.d / per_step
    elif kernel == "merge_g":  # rescale-and-add of the key-split partials
        flops = wl.heads * 2.0 * wl.m * wl.d / per_step
    else:
        flops = pinv_flops(wl, with_w=not w_separate) / per_step
    achieved = flops / t_launch / 1e12
    if kernel in ("pinv_tc", "pinv_big"):
        # the peak of this mix of tf32 and fp16 products: its flops over the
        # time they take at each type's peak
        peak = flops / (pinv_peak_time(wl, peaks["bf16_tflops"], with_w=not w_separate) / per_step) / 1e12
        return {"kernel": kernel, "bound": "tensor", "achieved": achieved, "peak": peak,
                "unit": "TFLOP/s", "frac": achieved / peak, "traffic": traffic,
                "algorithmic_flops": flops,
                "peak_source": f"bf16_tflops burst ({peak_src}); tf32 products at x 1.1/2.25 (tf32/bf16 "
                               f"nominal), fp16 update products (m > 128) at the bf16 rate; fp32 "
                               f"inputs: three tf32 products per product (tf32 rate / 3)"}
    peak = 152 * 128 * 2 * (peaks.get("sm_max_mhz", 2070.0) * 1e6) / 1e12
    return {"kernel": kernel, "bound": "alu", "achieved": achieved, "peak": peak,
            "unit": "TFLOP/s", "frac": achieved / peak, "traffic": traffic,
            "algorithmic_flops": flops,
            "peak_source": "152 SMs x 128 fp32 FMA/clk x 2 x max SM clock"}


def pass_roofline(wl, ms_per_step, peaks, peak_src):
    """Whole forward pass against its own roofline: the method's minimum
    traffic (6 T e bytes: Q and V read twice, K once, the output written once)
    at the measured HBM rate, and the dense contractions (landmark rows S and
    P V, token F and P W, the conv as a banded product, the pseudo-inverse) at
    the tensor rate; the slower of the two is the roofline time. `frac_7te`
    counts this implementation's schedule instead, which reads K twice (the
    landmark pass and the landmark rows): 7 T e bytes."""
    te = wl.B * wl.H * wl.n * wl.d * wl.elem_bytes
    nbytes = 6.0 * te
    n_tok = wl.B * wl.H * wl.n
    mm_flops = n_tok * (2.0 * wl.m * wl.d * 2 + 2.0 * wl.m * wl.d * 2 + 2.0 * wl.ks * wl.d)
    t_hbm = nbytes / (peaks["hbm_gbs"] * 1e9)
    # bf16 operands at the bf16 rate; fp32 as three tf32 products
    mma_rate = peaks["bf16_tflops"] * 1e12 * (TF32_OVER_BF16 / 3.0 if wl.dtype == "f32" else 1.0)
    t_mma = mm_flops / mma_rate + pinv_peak_time(wl, peaks["bf16_tflops"])
    t_roof = max(t_hbm, t_mma)
    t_roof7 = max(7.0 / 6.0 * t_hbm, t_mma)
    return {"bytes": nbytes, "flops": mm_flops + pinv_flops(wl), "t_hbm_us": t_hbm * 1e6,
            "t_tensor_us": t_mma * 1e6, "bound": "hbm" if t_hbm >= t_mma else "tensor",
            "t_roofline_us": t_roof * 1e6, "t_measured_us": ms_per_step * 1e3,
            "frac": t_roof / (ms_per_step / 1e3), "bytes_7te": 7.0 * te,
            "frac_7te": t_roof7 / (ms_per_step / 1e3),
            "peak_source": f"hbm_gbs, bf16_tflops ({peak_src}); tf32 = bf16 x 1.1/2.25, fp16 = bf16"}


def resident_inputs(inp, dev):
    """Device copies of one drawn workload: as many (q, k, v, out) sets as it
    takes for their total to exceed twice L2 (steps rotate over them), the
    conv weights, and the bytes of one set."""
    import torch
    wl = inp.wl

    def upload(x, bits):
        if wl.dtype == "bf16":
            return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(dev)
        return torch.from_numpy(x).to(dev)

    q0, k0, v0 = upload(inp.q, inp.q_bits), upload(inp.k, inp.k_bits), upload(inp.v, inp.v_bits)
    w = torch.from_numpy(inp.conv_w).to(dev)
    set_bytes = 4 * q0.numel() * q0.element_size()
    nsets = max(1, min(8, -(-2 * L2_BYTES // set_bytes)))
    sets = [(q0, k0, v0, torch.empty_like(q0))]
    for _ in range(nsets - 1):
        sets.append((q0.clone(), k0.clone(), v0.clone(), torch.empty_like(q0)))
    return sets, w, set_bytes


def device_inputs(wl, dev, seed):
    """Seeded device-side draws of a workload's shape (timing only: the
    sequence-length scan needs no oracle, so its inputs are drawn on the GPU
    with a seeded generator instead of on the host): rotating (q, k, v, out)
    sets whose total exceeds twice L2, conv weights, bytes of one set."""
    import torch
    tdt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    shape = (wl.B, wl.H, wl.n, wl.d)

    def draw():
        return (torch.randn(shape, generator=gen, device=dev, dtype=torch.float32) * wl.scale).to(tdt)

    ks = max(wl.ks, 1)
    w = torch.randn((wl.H, ks), generator=gen, device=dev, dtype=torch.float32) / float(np.sqrt(ks))
    set_bytes = 4 * wl.B * wl.H * wl.n * wl.d * wl.elem_bytes
    nsets = max(1, min(8, -(-2 * L2_BYTES // set_bytes)))
    sets = [(draw(), draw(), draw(), torch.empty(shape, device=dev, dtype=tdt)) for _ in range(nsets)]
    return sets, w, set_bytes


def time_regions(N, step, steps, stream, barrier, regions):
    """Exactly `regions` timed regions of `steps` steps each, back to back,
    each bracketed by a barrier + synchronize and timed with CUDA events on
    the launch stream. Returns the per-region milliseconds and the library's
    kernel launches over all regions."""
    import torch
    launches0 = N.nystrom_launch_count()
    out = []
    i0 = 0
    for _ in range(regions):
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        ev0.record(stream)
        for i in range(steps):
            step(i0 + i)
        ev1.record(stream)
        barrier()
        out.append(ev0.elapsed_time(ev1))
        i0 += steps
    return out, N.nystrom_launch_count() - launches0


def spread(vals):
    v = sorted(vals)
    q = lambda f: v[min(len(v) - 1, int(round(f * (len(v) - 1))))]
    return {"min": v[0], "p10": q(0.1), "median": statistics.median(v), "p90": q(0.9), "max": v[-1],
            "n": len(v)}


def time_brief(N, wl, sets, w, stream, steps=20, seconds=0.3):
    """Time a workload briefly (no clocks, no profile): median of K-step
    regions over about `seconds` of wall time."""
    import torch
    dt_code = N.NYS_BF16 if wl.dtype == "bf16" else N.NYS_FP32

    def step(i):
        q, k, v, out = sets[i % len(sets)]
        N.nystrom_attn_fwd(q, k, v, w, out, wl.B, wl.H, wl.n, wl.d, wl.m, wl.iters, wl.ks,
                           dt_code, stream)

    def barrier():
        torch.cuda.synchronize()

    for i in range(5):
        step(i)
    first, _ = time_regions(N, step, steps, stream, barrier, 1)
    regions = max(3, int(np.ceil(seconds / max(first[0] / 1e3, 1e-6))))
    region_ms, _ = time_regions(N, step, steps, stream, barrier, regions)
    assert N.nystrom_get_status(stream) == N.NYS_OK
    ms = statistics.median(region_ms) / steps
    return ms, spread([r / steps for r in region_ms])


def time_fn(N, step, stream, steps=20, seconds=0.3):
    """Median per-step milliseconds of an arbitrary step over ~`seconds` of
    K-step regions (CUDA events on the launch stream), after 5 warm-up steps."""
    import torch

    def barrier():
        torch.cuda.synchronize()

    for i in range(5):
        step(i)
    first, _ = time_regions(N, step, steps, stream, barrier, 1)
    regions = max(3, int(np.ceil(seconds / max(first[0] / 1e3, 1e-6))))
    region_ms, launches = time_regions(N, step, steps, stream, barrier, regions)
    assert N.nystrom_get_status(stream) == N.NYS_OK
    return statistics.median(region_ms) / steps, launches / (regions * steps)


def next_rows(N, dev, stream):
    """The rows past the core path, timed briefly on seeded device draws:
    the attention module around the op at BERT-base size, the two variants
    (padded sequences with per-channel filters) on the clustered and
    long-context shapes, and clustered attention on the clustered shape."""
    import torch
    gen = torch.Generator(device=dev)
    gen.manual_seed(4242)
    bf = torch.bfloat16
    out = {}

    def randn(*shape, scale=1.0, dtype=bf):
        return (torch.randn(shape, generator=gen, device=dev) * scale).to(dtype)

    # module: B32 n512 H12 d64 (D = 768), projections + attention
    B, n, H, d, m = 32, 512, 12, 64, 64
    D = H * d
    x, wqkv, wo = randn(B, n, D), randn(D, 3 * D, scale=D ** -0.5), randn(D, D, scale=D ** -0.5)
    bqkv, bo = randn(3 * D, scale=0.1, dtype=torch.float32), randn(D, scale=0.1, dtype=torch.float32)
    cw = randn(H, 33, scale=33 ** -0.5, dtype=torch.float32)
    y = torch.empty_like(x)
    nb = N.nystrom_mha_workspace_bytes(B, n, H, d, m, N.NYS_BF16)
    ws = torch.empty(nb, dtype=torch.uint8, device=dev)
    ms, lps = time_fn(N, lambda i: N.nystrom_mha_fwd(x, wqkv, bqkv, wo, bo, cw, y, B, n, H, d, m, 6,
                                                     33, N.NYS_BF16, ws, nb, stream), stream)
    proj_flops = 2.0 * B * n * D * (3 * D + D)
    out["module"] = {"workload": f"B={B} n={n} H={H} d={d} (D={D}) m={m} iters=6 ks=33 bf16, "
                                 "QKV and output projections (cuBLAS) + the op",
                     "ms_per_step": ms, "tokens_per_s": B * n / (ms / 1e3),
                     "projection_tflops_if_all_time": proj_flops / (ms / 1e3) / 1e12,
                     "library_launches_per_step": lps}
    del x, wqkv, wo, y, ws
    # variants: padded sequences + per-channel filters (c4 and c5 shapes)
    for name, (B, H, n, d, m, it, ks) in {"c4": (8, 8, 8192, 64, 128, 6, 33),
                                          "c5": (2, 16, 32768, 128, 256, 8, 65)}.items():
        q, k, v = randn(B, H, n, d), randn(B, H, n, d), randn(B, H, n, d)
        o = torch.empty_like(q)
        cwc = randn(H, d, ks, scale=ks ** -0.5, dtype=torch.float32)
        lengths = workloads.lengths_for(B, n, m, seed=99).tolist()
        ms, _ = time_fn(N, lambda i: N.nystrom_attn_fwd_ex(q, k, v, cwc, o, B, H, n, d, m, it, ks,
                                                           N.NYS_BF16, N.NYS_CONV_PER_CHANNEL,
                                                           lengths, None, 0, stream), stream)
        out[f"variants_{name}"] = {
            "workload": f"{name} shape B={B} H={H} n={n} d={d} m={m} iters={it} ks={ks} bf16, "
                        f"per-channel filters, lengths {lengths}",
            "ms_per_step": ms, "tokens_per_s": B * H * n / (ms / 1e3),
            "real_tokens_per_s": H * sum(lengths) / (ms / 1e3)}
        N.nystrom_profile_read()
        N.nystrom_profile_enable(True)
        for _ in range(5):
            N.nystrom_attn_fwd_ex(q, k, v, cwc, o, B, H, n, d, m, it, ks, N.NYS_BF16,
                                  N.NYS_CONV_PER_CHANNEL, lengths, None, 0, stream)
        torch.cuda.synchronize()
        N.nystrom_profile_enable(False)
        prof = N.nystrom_profile_read()
        out[f"variants_{name}"]["kernels_us_per_step"] = {kname: ms_ / 5 * 1e3 for kname, (ms_, _) in prof.items()}
        del q, k, v, o
        torch.cuda.empty_cache()
    # clustered attention: c4 shape, C = 128, 10 K-means rounds
    B, H, n, d, C, it = 8, 8, 8192, 64, 128, 10
    q, k, v = randn(B, H, n, d), randn(B, H, n, d), randn(B, H, n, d)
    o = torch.empty_like(q)
    nb = N.nystrom_clustered_workspace_bytes(B, H, n, d, C, N.NYS_BF16)
    ws = torch.empty(nb, dtype=torch.uint8, device=dev)
    ms, _ = time_fn(N, lambda i: N.nystrom_clustered_attn_fwd(q, k, v, o, B, H, n, d, C, it,
                                                              N.NYS_BF16, ws, nb, stream), stream)
    out["clustered_c4"] = {"workload": f"B={B} H={H} n={n} d={d} C={C} K-means rounds={it} bf16",
                           "ms_per_step": ms, "tokens_per_s": B * H * n / (ms / 1e3)}
    N.nystrom_profile_read()
    N.nystrom_profile_enable(True)
    for _ in range(5):
        N.nystrom_clustered_attn_fwd(q, k, v, o, B, H, n, d, C, it, N.NYS_BF16, ws, nb, stream)
    torch.cuda.synchronize()
    N.nystrom_profile_enable(False)
    prof = N.nystrom_profile_read()
    out["clustered_c4"]["kernels_us_per_step"] = {kname: ms_ / 5 * 1e3 for kname, (ms_, _) in prof.items()}
    del q, k, v, o, ws
    torch.cuda.empty_cache()
    return out


def linear_scan(N, wl, dev, stream, peaks, peak_src, ns):
    """Time of one pass against the sequence length with every other size of
    the workload fixed (linear time shows as a constant time per token), and
    a least-squares line t = a + b n over the points."""
    import dataclasses

    import torch
    points = []
    for n in ns:
        wn = dataclasses.replace(wl, n=n)
        if n % wn.m != 0:
            continue
        sets, w, _ = device_inputs(wn, dev, seed=7000 + n)
        ms, sp = time_brief(N, wn, sets, w, stream)
        points.append({"n": n, "ms_per_step": ms, "tokens_per_s": wn.tokens / (ms / 1e3),
                       "ns_per_token_per_head": ms * 1e6 / n,
                       "pass_roofline_frac": pass_roofline(wn, ms, peaks, peak_src)["frac"],
                       "spread_ms": sp})
        del sets
        torch.cuda.empty_cache()
    fit = None
    if len(points) >= 2:
        x = np.array([p_["n"] for p_ in points], dtype=np.float64)
        y = np.array([p_["ms_per_step"] * 1e3 for p_ in points])
        b, a = np.polyfit(x, y, 1)
        fit = {"intercept_us": float(a), "us_per_1k_tokens_of_n": float(b * 1e3),
               "max_rel_residual": float(np.max(np.abs(a + b * x - y) / y))}
    return {"shape": f"B={wl.B} H={wl.H} d={wl.d} m={wl.m} iters={wl.iters} ks={wl.ks} {wl.dtype}",
            "inputs": "seeded device draws (torch.Generator), rotating sets past L2",
            "points": points, "fit_t_vs_n": fit}


def run_scan(args, wl):
    """--scan-n: the sequence-length scan alone, one JSON line."""
    import torch

    from nystr_self_attention_gb300 import build as nbuild
    nbuild.build()
    import nystr_self_attention_gb300 as N

    rank, world, local = dist_env()
    if rank != 0:
        return
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    peaks, peak_src = load_peaks()
    ns = [int(x) for x in args.scan_n.split(",") if x]
    print(json.dumps({"scan": "n", **linear_scan(N, wl, dev, torch.cuda.current_stream(), peaks,
                                                 peak_src, ns)}), flush=True)


def run_ours(args, wl):
    import torch
    import torch.distributed as dist

    from nystr_self_attention_gb300 import build as nbuild
    nbuild.build()
    import nystr_self_attention_gb300 as N

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()

    inp = workloads.make_inputs(wl)
    dt_code = N.NYS_BF16 if wl.dtype == "bf16" else N.NYS_FP32
    tdt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    sets, w, set_bytes = resident_inputs(inp, dev)
    nsets = len(sets)
    q0, k0, v0 = sets[0][:3]
    B, H, n, d, m = wl.B, wl.H, wl.n, wl.d, wl.m
    plan = N.nystrom_plan_describe(B, H, n, d, m, wl.iters, wl.ks, dt_code)

    def step(i):
        q, k, v, out = sets[i % nsets]
        N.nystrom_attn_fwd(q, k, v, w, out, B, H, n, d, m, wl.iters, wl.ks, dt_code, stream)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    for i in range(args.warmup):
        step(i)
    barrier()
    # default step count: about 3 s of timed work
    steps = args.steps
    if steps is None:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(10):
            step(i)
        e1.record(stream)
        torch.cuda.synchronize()
        per = e0.elapsed_time(e1) / 10 / 1e3
        steps = int(max(20, min(200000, 3.0 / max(per, 1e-7))))
        if world > 1:
            steps = int(reduce_over_ranks(steps, dist.ReduceOp.MIN, dev, world))

    def measure():
        """The K-step timed region, repeated back to back until at least
        --min-region-s of wall time has passed (the same number of regions on
        every rank), with nvidia-smi sampling clocks throughout."""
        first, _ = time_regions(N, step, steps, stream, barrier, 1)
        regions = max(1, int(np.ceil(args.min_region_s / max(first[0] / 1e3, 1e-6))))
        if world > 1:
            regions = int(reduce_over_ranks(regions, dist.ReduceOp.MAX, dev, world))
        sampler = ClockSampler(local)
        sampler.start()
        time.sleep(0.3)
        t_wall0 = time.time()
        region_ms, n_launch = time_regions(N, step, steps, stream, barrier, regions)
        t_wall1 = time.time()
        time.sleep(0.2)
        sampler.stop()
        if world > 1:
            t = torch.tensor(region_ms, device=dev, dtype=torch.float64)
            dist.all_reduce(t, op=dist.ReduceOp.MAX)
            region_ms = t.tolist()
        return region_ms, n_launch, sampler.summary(t_wall0, t_wall1)

    region_ms, launches, clocks = measure()
    # a throttled or clock-locked run is measured once more (on every rank)
    if reduce_over_ranks(float(clocks_rejected(clocks)), dist.ReduceOp.MAX, dev, world) > 0:
        first = clocks
        region_ms, launches, clocks = measure()
        clocks["remeasured_after"] = {"reasons": first["reasons"], "sm_mhz": first["sm_mhz"]}
    assert N.nystrom_get_status(stream) == N.NYS_OK

    tokens_step = wl.tokens
    elapsed_ms = statistics.median(region_ms)  # one K-step region
    value = job_throughput(tokens_step, world, steps, elapsed_ms)
    ms_per_step = elapsed_ms / steps

    # the same steps on one input set (warm L2 where the inputs fit in it)
    def step_warm(i):
        q, k, v, out = sets[0]
        N.nystrom_attn_fwd(q, k, v, w, out, B, H, n, d, m, wl.iters, wl.ks, dt_code, stream)

    warm_ms, _ = time_fn(N, step_warm, stream)
    warm_l2 = {"ms_per_step": warm_ms, "tokens_per_s": tokens_step * world / (warm_ms / 1e3),
               "inputs": "one input set reused every step (in L2 when its 4 T e bytes fit there); "
                         "the headline value rotates sets past L2"}

    # per-kernel times (CUDA events on the launch stream) over a second pass of
    # the same steps (capped), for the roofline of the dominant kernel
    prof_steps = min(steps, 500)
    N.nystrom_profile_read()
    N.nystrom_profile_enable(True)
    for i in range(prof_steps):
        step(i)
    torch.cuda.synchronize()
    N.nystrom_profile_enable(False)
    prof = N.nystrom_profile_read()
    peaks, peak_src = load_peaks()
    w_separate = "w=w_tc" in plan
    roofline = None
    kernels = {}
    if prof:
        tot = sum(ms for ms, _ in prof.values())
        for name, (ms, cnt) in prof.items():
            kernels[name] = {"launches_per_step": cnt / prof_steps, "us_per_launch": ms / cnt * 1e3,
                             "share": ms / tot}
            per_step = max(1, round(cnt / prof_steps))
            kernels[name]["roofline"] = roofline_for(name, ms, cnt, per_step, wl, peaks, peak_src,
                                                     w_separate)
        dom = max(prof, key=lambda k: prof[k][0])
        roofline = dict(kernels[dom]["roofline"])
        for v in kernels.values():
            r = v.pop("roofline")
            v["frac"] = r["frac"]
            v["bound"] = r["bound"]

    # end to end through the host-buffer C ABI call, pinned host memory
    e2e = None
    if not args.no_e2e:
        esz = 2 if wl.dtype == "bf16" else 4
        shape = (B, H, n, d)
        hq = torch.empty(shape, dtype=tdt, pin_memory=True)
        hk = torch.empty_like(hq, pin_memory=True)
        hv = torch.empty_like(hq, pin_memory=True)
        hout = torch.empty_like(hq, pin_memory=True)
        hw = torch.from_numpy(inp.conv_w).pin_memory()
        hq.copy_(q0.cpu())
        hk.copy_(k0.cpu())
        hv.copy_(v0.cpu())
        e2e_steps = max(3, min(steps, 50))
        for _ in range(2):
            N.nystrom_attn_fwd_host(hq, hk, hv, hw, hout, B, H, n, d, m, wl.iters, wl.ks, dt_code,
                                    stream)
        barrier()
        t0 = time.perf_counter()
        for _ in range(e2e_steps):
            N.nystrom_attn_fwd_host(hq, hk, hv, hw, hout, B, H, n, d, m, wl.iters, wl.ks, dt_code,
                                    stream)
        t1 = time.perf_counter()
        dt_e2e = t1 - t0
        if world > 1:
            dt_e2e = reduce_over_ranks(dt_e2e, dist.ReduceOp.MAX, dev, world)
        e2e = {"value": tokens_step * world * e2e_steps / dt_e2e, "unit": "tokens/s",
               "h2d_bytes_per_step": 3 * wl.tokens * d * esz + wl.H * wl.ks * 4,
               "d2h_bytes_per_step": wl.tokens * d * esz, "steps": e2e_steps,
               "api": "nystrom_attn_fwd_host"}
        del hq, hk, hv, hout

    # the other workloads and the sequence-length scan ride along (one GPU)
    others = None
    scan = None
    nxt = None
    if world == 1:
        del sets, q0, k0, v0
        torch.cuda.empty_cache()
        names = [x for x in args.others.split(",") if x and x != wl.name]
        if names:
            others = {}
            for nm in names:
                wo = workloads.WORKLOADS[nm]
                so, wwo, _ = resident_inputs(workloads.make_inputs(wo), dev)
                ms, sp = time_brief(N, wo, so, wwo, stream)
                others[nm] = {"workload": wo.describe(), "tokens_per_s": wo.tokens / (ms / 1e3),
                              "ms_per_step": ms, "spread_ms": sp,
                              "pass_roofline_frac": pass_roofline(wo, ms, peaks, peak_src)["frac"],
                              "plan": N.nystrom_plan_describe(
                                  wo.B, wo.H, wo.n, wo.d, wo.m, wo.iters, wo.ks,
                                  N.NYS_BF16 if wo.dtype == "bf16" else N.NYS_FP32)}
                del so
                torch.cuda.empty_cache()
        if not args.no_scan and wl.dtype == "bf16":
            ns = sorted({max(wl.m, wl.n >> 3), max(wl.m, wl.n >> 2), max(wl.m, wl.n >> 1), wl.n})
            scan = linear_scan(N, wl, dev, stream, peaks, peak_src, ns)
        if not args.no_next:
            nxt = next_rows(N, dev, stream)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tk, secs, heads = oracle_sample(inp, args.cpu_seconds)
        cpu = {"value": tk / secs, "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
               "sample": f"{heads} head passes over the {wl.heads} heads (n={wl.n} tokens each), "
                         f"fp64 numpy, {secs:.1f} s"}

    if world > 1:
        dist.destroy_process_group()
    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": world, "steps": steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "ms_per_step_spread": spread([r / steps for r in region_ms]),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype,
        "data": "synthetic (seeded normal draws, bf16-rounded where bf16)",
        "config": {"workload": wl.describe(), "tokens_per_step": tokens_step, "plan": plan,
                   "l2": f"{nsets} rotating input sets ({nsets * set_bytes / 2**20:.0f} MiB) > L2",
                   "timed_regions": f"{len(region_ms)} back-to-back regions of {steps} steps; "
                                    "value and ms_per_step from the median region",
                   "parallelism": f"replicas x{world} (independent heads, no collective)"},
        "roofline": roofline, "pass_roofline": pass_roofline(wl, ms_per_step, peaks, peak_src),
        "warm_l2": warm_l2,
        "kernels": kernels, "cpu_baseline": cpu, "e2e": e2e,
        "clocks": clocks, "gpu_launches": launches // max(1, len(region_ms)),
        "gpu_launches_all_regions": launches,
        "other_workloads": others, "linear_scan": scan, "next_rows": nxt,
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    wl = workloads.WORKLOADS[args.config]
    if args.batch is not None:
        import dataclasses
        wl = dataclasses.replace(wl, B=args.batch)
    if args.impl == "reference":
        run_reference(args, wl)
    elif args.scan_n:
        run_scan(args, wl)
    else:
        run_ours(args, wl)


if __name__ == "__main__":
    main()

#!/usr/bin/env python
"""Throughput of the causal LLA forward (liblla, one GB300 per rank).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl lla|reference] [--workload 3]

One step is one full causal LLA forward (every stage of the hot path) over the headline workload:
B4 H8 T4096 d=dv=64, bf16 inputs and outputs, i.i.d. N(0,1) q, k, v (seed 2), h=8,
lambda=1e-2. Inputs are resident in HBM before the timed region; the 256 MiB L2 flush between
steps is outside the per-step CUDA events. Under torchrun every rank runs its own copy of the
workload (weak scaling: independent heads, no collective on the data path); the step time is
the max over ranks.

The printed JSON line carries: value (queries/s, all ranks), TFLOP/s and fraction of the
measured peak for the dominant kernel (roofline), the end-to-end rate through the C ABI on host
buffers (e2e), the float64 oracle timed on the host cores on a bounded sample of the same
workload (cpu_baseline), the number of liblla kernel launches in the timed region and the SM
clocks sampled during it.

--impl reference times the float64 oracle itself (the reference arm of this comparison) on the
host cores, on bounded samples of the same workload, and prints the same kind of line.

--op parallax measures the causal Parallax forward with a given probe instead (one kernel per
step; probe r ~ N(0, 1/d) drawn with seed + 100) on the same workload and prints the same kind
of line for it.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import multiprocessing as mp
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "LLA fwd queries/sec and TFLOP/s on 1 GB300; fraction of tensor-core peak"
METRIC_PARALLAX = "Parallax fwd queries/sec and TFLOP/s on 1 GB300; fraction of tensor-core peak"
UNIT = "queries/s"
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
SM_COUNT = 152
FP32_LANES_PER_SM = 128


# ----------------------------------------------------------------------------- accounting
def causal_pairs(w) -> int:
    return w.B * w.H * w.T * (w.T + 1) // 2


def moments_flops_per_pair(d: int) -> int:
    """Algorithmic flops per causal pair of the moments stage: the logit q.k (2d) and the
    kernel-weighted sums omega, sum w k and the upper triangle of sum w k k^T (2 each)."""
    return 2 * d + 2 * (1 + d + d * (d + 1) // 2)


def contraction_flops_per_pair(d: int) -> int:
    """Algorithmic flops per causal pair of the moment contraction alone (the tensor-core path's
    second moments kernel): omega, sum w k and the upper triangle of sum w k k^T (2 each)."""
    return 2 * (1 + d + d * (d + 1) // 2)


def tc_executed_flops_per_pair(d: int) -> int:
    """Tensor flops the tcgen05 moment contraction executes per causal pair: hi + lo over
    5 passes x 448 feature columns (2208 slots and 32 of padding); the same for d < 64, which
    runs zero-padded to d = 64."""
    return 2 * 2 * 5 * 448


def tc_weights_executed_flops_per_pair(d: int) -> int:
    """Tensor flops of the weight sweeps per causal pair: q.k twice (the exact-max sweep and the
    weight sweep)."""
    return 2 * 2 * d


def parallax_flops_per_pair(d: int, dv: int) -> int:
    """Algorithmic flops per causal pair of the Parallax forward: q.k and r.k (2d each), and the
    two value contractions P1 V and P2 V (2dv each). The exact-max sweep is not counted."""
    return 2 * d + 2 * d + 2 * dv + 2 * dv


def step_flops(w) -> int:
    """Algorithmic flops of one whole forward (keys-only dense moments + solve + readout)."""
    d, e = w.d, w.dv
    per_pair = moments_flops_per_pair(d) + 2 * d + 2 * e + 2
    per_query = d ** 3 // 3 + 2 * d * d + 2 * d * e
    return causal_pairs(w) * per_pair + w.queries * per_query


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(PEAKS_FALLBACK), "fallback"


def fp32_alu_peak_tflops(peaks) -> float:
    """FP32 FMA peak from unit counts and the maximum SM clock: SMs x lanes x 2 flop x f."""
    mhz = float(peaks.get("sm_max_mhz", 2070.0))
    return SM_COUNT * FP32_LANES_PER_SM * 2 * mhz * 1e6 / 1e12


def kernel_source_sha(name: str) -> str:
    p = os.path.join(ROOT, "local_linear_attention_gb300", "csrc", name)
    with open(p, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def shape_key(w) -> str:
    """The workload shape a traffic record belongs to, e.g. "B4 H8 T4096 d64 dv64 bf16"."""
    return f"B{w.B} H{w.H} T{w.T} d{w.d} dv{w.dv} {w.dtype}"


def recorded_traffic(kernel_file: str, w=None):
    """DRAM bytes per launch from a committed ncu summary, if it matches the current source and
    was captured on this workload's shape (bytes of one shape say nothing about another)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    ent = rec.get(kernel_file)
    if not ent or ent.get("source_sha") != kernel_source_sha(kernel_file):
        return None
    if w is not None and ent.get("shape") != shape_key(w):
        return None
    # a step that also launches kernels of other files is current only if they are unchanged too
    for other, sha in ent.get("depends", {}).items():
        if sha != kernel_source_sha(other):
            return None
    return ent.get("dram_bytes_per_launch")


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- oracle timing
_POOL_INPUTS = {}


def _pool_init(workload_index: int, op: str = "lla"):
    from local_linear_attention_gb300 import workloads as W
    w = W.WORKLOADS[workload_index]
    q, k, v = W.make_inputs(w)
    _POOL_INPUTS["qkv"] = tuple(t.float().numpy() for t in (q, k, v))
    _POOL_INPUTS["op"] = op
    if op == "parallax":
        _POOL_INPUTS["r"] = W.make_probe(w.B, w.H, w.T, w.d, w.dtype, seed=w.seed + 100).float().numpy()


def _oracle_rows(args):
    h, lam, rows = args
    from oracle import lla_forward_oracle, parallax_forward_oracle
    q, k, v = _POOL_INPUTS["qkv"]
    t0 = time.perf_counter()
    if _POOL_INPUTS["op"] == "parallax":
        parallax_forward_oracle(q, k, v, _POOL_INPUTS["r"], h, rows=rows)
    else:
        lla_forward_oracle(q, k, v, h, lam, rows=rows)
    return time.perf_counter() - t0


def _oracle_values(args):
    h, lam, rows = args
    from oracle import lla_forward_oracle
    q, k, v = _POOL_INPUTS["qkv"]
    return lla_forward_oracle(q, k, v, h, lam, rows=rows)


class OracleTimer:
    """The float64 oracle, as it stands, on bounded row samples of a workload: one chunk of rows
    per host core, in spawned single-threaded worker processes that regenerate the workload
    from its seed once."""

    def __init__(self, workload_index: int, op: str = "lla"):
        from local_linear_attention_gb300 import workloads as W
        self.W = W
        self.w = W.WORKLOADS[workload_index]
        self.op = op
        self.cores = os.cpu_count() or 1
        env = {"OMP_NUM_THREADS": "1", "OPENBLAS_NUM_THREADS": "1", "MKL_NUM_THREADS": "1"}
        old = {x: os.environ.get(x) for x in env}
        os.environ.update(env)
        try:
            self.pool = mp.get_context("spawn").Pool(self.cores, _pool_init, (workload_index, op))
        finally:
            for x, val in old.items():
                if val is None:
                    os.environ.pop(x, None)
                else:
                    os.environ[x] = val
        self.pool.map(_oracle_rows, [(1.0, 1.0, [0])] * self.cores)  # workers ready
        self.per_row = None

    def _run(self, rows):
        lam, h = self.w.points[0]
        chunks = [(h, lam, rows[i::self.cores]) for i in range(self.cores)]
        t0 = time.perf_counter()
        self.pool.map(_oracle_rows, chunks)
        return time.perf_counter() - t0

    def measure(self, budget_s: float, seed: int):
        """(queries/s, cores, sample description) for about budget_s seconds of oracle work."""
        w = self.w
        if self.per_row is None:  # the cost of a row grows with its prefix: calibrate once
            rows = self.W.sample_rows(w.B * w.H, w.T, 2 * self.cores, seed=seed)
            self.per_row = self._run(rows) / len(rows)
        for attempt in range(3):
            n = int(min(w.queries, max(self.cores, budget_s / max(self.per_row, 1e-6))))
            rows = self.W.sample_rows(w.B * w.H, w.T, n, seed=seed + 1)
            wall = self._run(rows)
            self.per_row = wall / len(rows)
            if wall >= 0.5 * budget_s or n >= w.queries:
                break
        how = ("one float64 ridge solve per row (SVD of the weighted centred keys)"
               if self.op == "lla"
               else "float64 softmax weights and explicit covariance per row")
        sample = (f"{len(rows)} uniformly sampled query rows of {w.describe()} (of {w.queries}), "
                  f"{how}, {self.cores} single-threaded processes, {wall:.1f} s")
        return len(rows) / wall, self.cores, sample

    def values(self, rows, h, lam):
        """The oracle's outputs at flat query rows (for the parity check of the timed output)."""
        import numpy as np
        chunks = [rows[i::self.cores] for i in range(self.cores)]
        parts = self.pool.map(_oracle_values, [(h, lam, c) for c in chunks if c])
        out = np.zeros((len(rows), self.w.dv))
        it = iter(parts)
        for i in range(self.cores):
            if chunks[i]:
                out[i::self.cores] = next(it)
        return out

    def close(self):
        self.pool.terminate()
        self.pool.join()


# ----------------------------------------------------------------------------- timing, parity
MIN_TIMED_S = 2.0   # device time the timed region spans at least (clock samples under load)
PARITY_ROWS = 96    # sampled rows of the timed output checked against the oracle


def max_over_ranks(x: float, world: int) -> float:
    """The largest of every rank's x (a job's time is that of its slowest rank); x itself when
    there is one rank. The reduction runs on the process group's device: CUDA under NCCL, the
    host under gloo."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], device=dev, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank: float, world: int, seconds: float) -> float:
    """Whole-job throughput: the units all ranks processed (the same on each) over the slowest
    rank's time."""
    return units_per_rank * world / seconds


def timed_repeats(warm_step_ms: float, steps: int, world: int, min_s: float = MIN_TIMED_S) -> int:
    """Repetitions of the K-step timed loop so that the timed region lasts >= min_s
    (each repetition times exactly K steps; the same count on every rank)."""
    est = max(warm_step_ms, 1e-3) * max(steps, 1)
    reps = int(min(200, max(1, math.ceil(min_s * 1e3 / est))))
    return int(max_over_ranks(reps, world))


def parity_summary(got, ref, v, bound: float, nrows: int) -> dict:
    """Relative Frobenius error and the worst row's error (||do_i|| / (||o_i|| + rms V)) of
    sampled rows of the benchmarked output against the oracle."""
    import numpy as np
    rel = float(np.linalg.norm(got - ref) / np.linalg.norm(ref))
    rms = float(np.sqrt(np.mean(v.astype(np.float64) ** 2)))
    row = float((np.linalg.norm(got - ref, axis=1) / (np.linalg.norm(ref, axis=1) + rms)).max())
    return {"rows": nrows, "rel_frob": rel, "row_max": row, "bound": bound,
            "ok": bool(rel <= bound), "sample": "uniform over (head, position), seed 77, "
            "incl. the first and last position of the first and last head"}


# ----------------------------------------------------------------------------- main
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def run_reference(args, w):
    world, rank, _ = dist_setup()
    if rank != 0:
        return 0
    budget = float(os.environ.get("LLA_ORACLE_STEP_S", "4"))
    vals, cores, sample = [], 1, ""
    timer = OracleTimer(args.workload, args.op)
    for s in range(args.warmup + args.steps):
        v, cores, sample = timer.measure(budget, seed=500 + s)
        if s >= args.warmup:
            vals.append(v)
    timer.close()
    value = statistics.median(vals)
    line = {
        "impl": "reference", "metric": METRIC_PARALLAX if args.op == "parallax" else METRIC,
        "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": w.queries / value * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": f"{w.name}: {w.describe()}, h={w.points[0][1]}, "
                               f"lambda={w.points[0][0]}, seed {w.seed}",
                   "note": "float64 CPU oracle; value extrapolated from row samples"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_parallax(args, w, cpu, world, rank):
    """One step = one lla_parallax_forward over the workload (a single kernel launch)."""
    import torch
    import torch.distributed as dist
    from local_linear_attention_gb300 import binding as lla
    from local_linear_attention_gb300 import workloads as W

    _, h = w.points[0]
    q, k, v = W.make_inputs(w)
    r = W.make_probe(w.B, w.H, w.T, w.d, w.dtype, seed=w.seed + 100)
    dq, dk, dv_, dr = q.cuda(), k.cuda(), v.cuda(), r.cuda()
    out = torch.empty(w.B, w.H, w.T, w.dv, dtype=dq.dtype, device="cuda")
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    def step():
        lla.lla_parallax_forward(dq, dk, dv_, dr, h, out=out, stream=stream)

    for _ in range(args.warmup):
        step()
    if lla.lla_stream_status() != 0:
        raise RuntimeError("liblla reported an error during warm-up")
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    n_launch0 = lla.launch_count()
    t_wall = time.perf_counter()
    for i in range(args.steps):
        flush.zero_()
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall
    if world > 1:
        dist.barrier()
    n_launch = lla.launch_count() - n_launch0
    clk = clocks.stop()
    if lla.lla_stream_status() != 0:
        raise RuntimeError("liblla reported an error during the timed steps")
    ms = sum(a.elapsed_time(b) for a, b in ev)
    ms = max_over_ranks(ms, world)
    ms_per_step = ms / args.steps
    value = job_rate(w.queries, world, ms_per_step / 1e3)

    e2e = None
    eb = q.element_size()
    if not args.no_e2e:  # pinned host inputs -> device, forward, result -> pinned host, per step
        hq, hk, hv, hr = (t.pin_memory() for t in (q, k, v, r))
        hout = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)

        def e2e_step():
            for hst, dst in ((hq, dq), (hk, dk), (hv, dv_), (hr, dr)):
                dst.copy_(hst, non_blocking=True)
            step()
            hout.copy_(out, non_blocking=True)
            torch.cuda.synchronize()

        for _ in range(2):
            e2e_step()
        e2e_steps = max(3, min(args.steps, 10))
        t0 = time.perf_counter()
        for _ in range(e2e_steps):
            e2e_step()
        e2e_s = (time.perf_counter() - t0) / e2e_steps
        e2e_s = max_over_ranks(e2e_s, world)
        e2e = {"value": job_rate(w.queries, world, e2e_s), "unit": UNIT,
               "h2d_bytes_per_step": (q.numel() + k.numel() + v.numel() + r.numel()) * eb,
               "d2h_bytes_per_step": out.numel() * eb}

    peaks, peak_src = load_peaks()
    tensor_path = w.dtype == "bf16" and w.d == 64 and w.dv == 64
    achieved = causal_pairs(w) * parallax_flops_per_pair(w.d, w.dv) / (ms_per_step / 1e3) / 1e12
    if tensor_path:
        peak = float(peaks.get("bf16_tflops", PEAKS_FALLBACK["bf16_tflops"]))
        roof = {"kernel": "parallax (lla_parallax.cu, tcgen05)", "bound": "tensor",
                "peak_source": f"bf16 dense, burst ({peak_src})"}
    else:
        peak = fp32_alu_peak_tflops(peaks)
        roof = {"kernel": "parallax (lla_parallax.cu, CUDA cores)", "bound": "alu",
                "peak_source": f"fp32 FMA: {SM_COUNT} SMs x {FP32_LANES_PER_SM} lanes x 2 x "
                               f"{peaks.get('sm_max_mhz', 2070)} MHz ({peak_src} clock)"}
    roof.update({"achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                 "traffic": recorded_traffic("lla_parallax.cu", w), "avg_launch_ms": ms_per_step})
    if rank == 0:
        line = {
            "metric": METRIC_PARALLAX, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if tensor_path else "f32", "data": "synthetic",
            "config": {"workload": f"{w.name}: {w.describe()}, {w.recipe()}, probe "
                                   f"N(0,1/d) seed {w.seed + 100}, h={h}, seed {w.seed}",
                       "B": w.B, "H": w.H, "T": w.T, "d": w.d, "dv": w.dv, "io_dtype": w.dtype,
                       "l2": "flushed between steps (256 MiB write outside the step events)",
                       "parallelism": f"replica per GPU x{world}"},
            "tflops": achieved,
            "roofline": roof,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": n_launch,
            "clocks": clk,
            "wall_s_timed": t_wall,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


METRIC_PX_BWD = ("Parallax backward queries/sec and TFLOP/s on 1 GB300; fraction of the bf16 tensor "
                 "peak (FP32 FMA peak on the CUDA-core path)")


def parallax_bwd_flops_per_pair(d: int, dv: int):
    """(algorithmic, executed) flops per causal pair of lla_parallax_backward: the forward's row
    statistics (Q K^T, R K^T, P V, P2 V: 4d + 4dv) plus the backward proper (the same logits
    and dO V^T once: 4d + 2dv; dq, dr: 4d; dk: 4d; dv: 2dv); executed (the CUDA-core passes),
    the row and column passes each recompute the logits and dO V^T (20d + 10dv). The
    tensor-core passes execute more (a max sweep in the record pass, the P2 V hi/lo pair)."""
    return 16 * d + 8 * dv, 20 * d + 10 * dv


def run_parallax_backward(args, w, world, rank):
    """One step = one lla_parallax_backward call (three launches) over the workload, with the
    Parallax probe and an i.i.d. N(0,1) upstream gradient."""
    import torch
    import torch.distributed as dist
    from local_linear_attention_gb300 import binding as lla
    from local_linear_attention_gb300 import workloads as W

    _, h = w.points[0]
    q, k, v = W.make_inputs(w)
    r = W.make_probe(w.B, w.H, w.T, w.d, w.dtype, seed=w.seed + 100)
    g = torch.Generator().manual_seed(w.seed + 200)
    do = torch.randn(w.B, w.H, w.T, w.dv, generator=g).to(q.dtype)
    xs = [x.cuda() for x in (q, k, v, r, do)]
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    grads = []

    def step():
        grads[:] = lla.lla_parallax_backward(*xs, h, stream=stream)

    for _ in range(args.warmup):
        step()
    if lla.lla_stream_status() != 0:
        raise RuntimeError("liblla reported an error during warm-up")
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    n_launch0 = lla.launch_count()
    t_wall = time.perf_counter()
    for i in range(args.steps):
        flush.zero_()
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall
    if world > 1:
        dist.barrier()
    n_launch = lla.launch_count() - n_launch0
    clk = clocks.stop()
    if lla.lla_stream_status() != 0:
        raise RuntimeError("liblla reported an error during the timed steps")
    ms = sum(a.elapsed_time(b) for a, b in ev)
    ms = max_over_ranks(ms, world)
    ms_per_step = ms / args.steps
    value = job_rate(w.queries, world, ms_per_step / 1e3)

    e2e = None
    eb = q.element_size()
    if not args.no_e2e:  # pinned host inputs -> device, backward, gradients -> pinned host
        hosts = [x.pin_memory() for x in (q, k, v, r, do)]
        houts = [torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for x in (q, k, v, r)]

        def e2e_step():
            for hst, dst in zip(hosts, xs):
                dst.copy_(hst, non_blocking=True)
            step()
            for hst, src in zip(houts, grads):
                hst.copy_(src, non_blocking=True)
            torch.cuda.synchronize()

        for _ in range(2):
            e2e_step()
        e2e_steps = max(3, min(args.steps, 10))
        t0 = time.perf_counter()
        for _ in range(e2e_steps):
            e2e_step()
        e2e_s = (time.perf_counter() - t0) / e2e_steps
        e2e_s = max_over_ranks(e2e_s, world)
        e2e = {"value": job_rate(w.queries, world, e2e_s), "unit": UNIT,
               "h2d_bytes_per_step": sum(x.numel() for x in (q, k, v, r, do)) * eb,
               "d2h_bytes_per_step": sum(x.numel() for x in (q, k, v, r)) * eb}

    peaks, peak_src = load_peaks()
    alg, exe = parallax_bwd_flops_per_pair(w.d, w.dv)
    achieved = causal_pairs(w) * alg / (ms_per_step / 1e3) / 1e12
    tensor_path = w.dtype == "bf16" and w.d == 64 and w.dv == 64
    if tensor_path:
        peak = float(peaks.get("bf16_tflops", PEAKS_FALLBACK["bf16_tflops"]))
        roof = {"kernel": "parallax backward (tcgen05: row records from the forward kernel of "
                          "lla_parallax.cu, rows and columns passes of lla_parallax_bwd_tc.cu)",
                "bound": "tensor", "peak_source": f"bf16 dense, burst ({peak_src})"}
    else:
        peak = fp32_alu_peak_tflops(peaks)
        roof = {"kernel": "parallax backward (lla_parallax_bwd.cu, CUDA cores: stats, rows, "
                          "columns)", "bound": "alu",
                "peak_source": f"fp32 FMA: {SM_COUNT} SMs x {FP32_LANES_PER_SM} lanes x 2 x "
                               f"{peaks.get('sm_max_mhz', 2070)} MHz ({peak_src} clock)"}
    roof.update({"achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                 "executed_tflops": causal_pairs(w) * exe / (ms_per_step / 1e3) / 1e12,
                 "traffic": recorded_traffic("lla_parallax_bwd_tc.cu", w) if tensor_path else None,
                 "avg_launch_ms": ms_per_step / 3})
    if rank == 0:
        line = {
            "metric": METRIC_PX_BWD, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if tensor_path else "f32", "data": "synthetic",
            "config": {"workload": f"{w.name}: {w.describe()}, {w.recipe()} and dO, probe "
                                   f"N(0,1/d) seed {w.seed + 100}, h={h}, seed {w.seed}",
                       "B": w.B, "H": w.H, "T": w.T, "d": w.d, "dv": w.dv, "io_dtype": w.dtype,
                       "l2": "flushed between steps (256 MiB write outside the step events)",
                       "parallelism": f"replica per GPU x{world}"},
            "tflops": achieved,
            "roofline": roof,
            "cpu_baseline": None,
            "e2e": e2e,
            "gpu_launches": n_launch,
            "clocks": clk,
            "wall_s_timed": t_wall,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


METRIC_DECODE = "LLA decode queries/sec (one query per head against a KV cache) on 1 GB300"
METRIC_PX_DECODE = "Parallax decode queries/sec (one query per head against a KV cache) on 1 GB300"


def run_decode(args, world, rank):
    """One step = one lla_decode / lla_parallax_decode call: every head's query against its
    cache (split-KV partials and the in-kernel last-arriver merge)."""
    import torch
    import torch.distributed as dist
    from local_linear_attention_gb300 import binding as lla

    B, H, L, d, dv, dt = args.decode_shape.split(",")
    B, H, L, d, dv = int(B), int(H), int(L), int(d), int(dv)
    tdt = torch.bfloat16 if dt == "bf16" else torch.float32
    px = args.op == "parallax_decode"
    h, lam = math.sqrt(d), 1e-2
    g = torch.Generator().manual_seed(6)
    q = torch.randn(B, H, d, generator=g).to(tdt)
    k = torch.randn(B, H, L, d, generator=g).to(tdt)
    v = torch.randn(B, H, L, dv, generator=g).to(tdt)
    r = (torch.randn(B, H, d, generator=g) / math.sqrt(d)).to(tdt)
    dq, dk, dv_, dr = q.cuda(), k.cuda(), v.cuda(), r.cuda()
    out = torch.empty(B, H, dv, dtype=tdt, device="cuda")
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    def step():
        if px:
            lla.lla_parallax_decode(dq, dk, dv_, dr, h, out=out, stream=stream)
        else:
            lla.lla_decode(dq, dk, dv_, h, lam, out=out, stream=stream)

    for _ in range(args.warmup):
        step()
    if lla.lla_stream_status() != 0:
        raise RuntimeError("liblla reported an error during warm-up")
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    n_launch0 = lla.launch_count()
    t_wall = time.perf_counter()
    for i in range(args.steps):
        flush.zero_()
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall
    if world > 1:
        dist.barrier()
    n_launch = lla.launch_count() - n_launch0
    clk = clocks.stop()
    if lla.lla_stream_status() != 0:
        raise RuntimeError("liblla reported an error during the timed steps")
    ms = sum(a.elapsed_time(b) for a, b in ev)
    ms = max_over_ranks(ms, world)
    ms_per_step = ms / args.steps
    queries = B * H
    value = job_rate(queries, world, ms_per_step / 1e3)
    eb = q.element_size()

    e2e = None
    if not args.no_e2e:  # pinned host inputs -> device, decode, result -> pinned host, per step
        hq, hk, hv, hr = (t.pin_memory() for t in (q, k, v, r))
        hout = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)

        def e2e_step():
            for hst, dst in ((hq, dq), (hk, dk), (hv, dv_)) + (((hr, dr),) if px else ()):
                dst.copy_(hst, non_blocking=True)
            step()
            hout.copy_(out, non_blocking=True)
            torch.cuda.synchronize()

        for _ in range(2):
            e2e_step()
        n_e2e = max(3, min(args.steps, 10))
        t0 = time.perf_counter()
        for _ in range(n_e2e):
            e2e_step()
        e2e_s = (time.perf_counter() - t0) / n_e2e
        e2e = {"value": job_rate(queries, world, e2e_s), "unit": UNIT,
               "h2d_bytes_per_step": (q.numel() * (2 if px else 1) + k.numel() + v.numel()) * eb,
               "d2h_bytes_per_step": out.numel() * eb}

    peaks, peak_src = load_peaks()
    kv_bytes = B * H * L * (d + dv) * eb  # the cache, read once
    gbs = kv_bytes / (ms_per_step / 1e3) / 1e9
    if px:
        peak = float(peaks.get("hbm_gbs", PEAKS_FALLBACK["hbm_gbs"]))
        roof = {"kernel": "parallax_decode_kernel (lla_decode.cu)", "bound": "hbm",
                "peak_source": f"HBM copy ({peak_src})", "achieved": gbs, "peak": peak,
                "unit": "GB/s", "frac": gbs / peak, "traffic": None,
                "note": "achieved = the K and V cache bytes (read once) per call / call time"}
    elif dt == "bf16" and d == 64 and dv == 64:
        # tensor-core decode: ~50 algorithmic flops per cache byte, below the bf16 ridge point
        # (dense peak / HBM bandwidth ~ 290 flop/B), so the cache read bounds it
        flops = B * H * L * (2 * d + 2 * (1 + d + dv + d * (d + 1) // 2 + dv * d))
        peak = float(peaks.get("hbm_gbs", PEAKS_FALLBACK["hbm_gbs"]))
        roof = {"kernel": "lla_decode_tc_kernel (lla_decode.cu)", "bound": "hbm",
                "peak_source": f"HBM copy ({peak_src})", "achieved": gbs, "peak": peak,
                "unit": "GB/s", "frac": gbs / peak, "traffic": None,
                "algorithmic_tflops": flops / (ms_per_step / 1e3) / 1e12,
                "note": "achieved = the K and V cache bytes (read once) per call / call time"}
    else:
        # algorithmic per key: the logit q.k and the moments omega, sum p k, sum p v, the upper
        # triangle of sum p k k^T and sum p v k^T
        flops = B * H * L * (2 * d + 2 * (1 + d + dv + d * (d + 1) // 2 + dv * d))
        achieved = flops / (ms_per_step / 1e3) / 1e12
        peak = fp32_alu_peak_tflops(peaks)
        roof = {"kernel": "lla_decode_kernel (lla_decode.cu)", "bound": "alu",
                "peak_source": f"fp32 FMA: {SM_COUNT} SMs x {FP32_LANES_PER_SM} lanes x 2 x "
                               f"{peaks.get('sm_max_mhz', 2070)} MHz ({peak_src} clock)",
                "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                "traffic": None, "cache_gbs": gbs}
    if rank == 0:
        line = {
            "metric": METRIC_PX_DECODE if px else METRIC_DECODE, "value": value, "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": dt, "data": "synthetic",
            "config": {"workload": f"decode: B{B} H{H} L{L} d{d} dv{dv} {dt}, i.i.d. N(0,1) "
                                   f"q/k/v" + (", probe N(0,1/d)" if px else f", lambda={lam}")
                                   + f", h={h:g}, seed 6",
                       "B": B, "H": H, "L": L, "d": d, "dv": dv, "io_dtype": dt,
                       "l2": "flushed between steps (256 MiB write outside the step events)",
                       "parallelism": f"replica per GPU x{world}"},
            "roofline": roof, "cpu_baseline": None, "e2e": e2e, "gpu_launches": n_launch,
            "clocks": clk, "wall_s_timed": t_wall,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["lla", "reference"], default="lla")
    ap.add_argument("--op", choices=["lla", "parallax", "decode", "parallax_decode",
                                     "parallax_backward"],
                    default="lla",
                    help="the operation timed: the LLA forward (default), the Parallax forward, "
                         "or LLA / Parallax decode (one query per head against a KV cache)")
    ap.add_argument("--decode-shape", default="32,8,16384,64,64,bf16",
                    help="B,H,L,d,dv,dtype of the decode workload")
    ap.add_argument("--workload", type=int, default=3)
    ap.add_argument("--strategy", choices=["dense", "cg"], default="dense",
                    help="ridge systems from dense tensor-core moments + Cholesky (default), or "
                         "matrix-free conjugate gradients (bf16 d = dv = 64 only)")
    ap.add_argument("--form", choices=["centred", "page"], default="centred",
                    help="closed form of the intercept: centred (default) or the page form with "
                         "the exact-LLA two-branch epilogue (dense strategy, bf16 d = dv = 64)")
    ap.add_argument("--cg-iters", type=int, default=1024)
    ap.add_argument("--cg-tol", type=float, default=1e-3)
    ap.add_argument("--min-timed-s", type=float, default=MIN_TIMED_S,
                    help="repeat the K-step timed loop until this much device time is timed "
                         "(0: one repetition, e.g. for profiler launch lists)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--shape", default=None,
                    help="B,H,T,d,dv,dtype: an i.i.d. N(0,1) workload of this shape instead "
                         "(for profiling captures; h = sqrt(d), lambda = 1e-2, seed 2)")
    args = ap.parse_args(argv)
    args.warmup = max(args.warmup, 3)

    from local_linear_attention_gb300 import workloads as W
    w = W.WORKLOADS[args.workload]
    if args.shape:
        B, H, T, d, dv, dt = args.shape.split(",")
        d = int(d)
        w = W.Workload("custom", int(B), int(H), int(T), d, int(dv), dt, 2, "iid",
                       h=math.sqrt(d), lam=1e-2)
        args.no_cpu_baseline = True
    if args.op in ("decode", "parallax_decode", "parallax_backward"):
        args.no_cpu_baseline = True  # the oracle leg times the prefill workloads
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable": "the oracle leg times the "
                              "prefill forward; this op has no CPU reference line"}), flush=True)
            return 0
    if args.impl == "reference":
        return run_reference(args, w)

    import torch
    import torch.distributed as dist

    world, rank, local = dist_setup()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    # The oracle's process pool is spawned before any GPU work (rank 0, one GPU only). It stays
    # up for the LLA forward, whose timed output it then checks on sampled rows (parity).
    cpu = None
    timer = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        timer = OracleTimer(args.workload, args.op)
        v, cores, sample = timer.measure(float(os.environ.get("LLA_ORACLE_BUDGET_S", "20")), 900)
        cpu = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample}
        if args.op != "lla" or args.shape:
            timer.close()
            timer = None

    from local_linear_attention_gb300 import binding as lla
    from local_linear_attention_gb300 import build as lla_build
    lla_build.build()

    if args.op == "parallax":
        return run_parallax(args, w, cpu, world, rank)
    if args.op == "parallax_backward":
        return run_parallax_backward(args, w, world, rank)
    if args.op in ("decode", "parallax_decode"):
        return run_decode(args, world, rank)

    lam, h = w.points[0]
    opts = {}
    if args.strategy == "cg":
        opts.update(path=lla.PATH_CG, cg=(args.cg_iters, args.cg_tol))
    if args.form == "page":
        opts.update(form=lla.FORM_PAGE)
    q, k, v = W.make_inputs(w)
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    out = torch.empty(w.B, w.H, w.T, w.dv, dtype=dq.dtype, device="cuda")
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    def step():
        lla.lla_forward(dq, dk, dv, h, lam, out=out, stream=stream, **opts)

    w0 = torch.cuda.Event(enable_timing=True)
    w1 = torch.cuda.Event(enable_timing=True)
    for i in range(args.warmup):
        if i == args.warmup - 1:
            w0.record(stream)
        step()
    w1.record(stream)
    if lla.lla_stream_status() != 0:
        raise RuntimeError("liblla reported an error during warm-up")
    reps = timed_repeats(w0.elapsed_time(w1), args.steps, world, args.min_timed_s)

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps * reps)]
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    n_launch0 = lla.launch_count()
    lla.profile_enable(True)
    t_wall = time.perf_counter()
    for i in range(args.steps * reps):
        flush.zero_()
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall
    lla.profile_enable(False)
    if world > 1:
        dist.barrier()
    n_launch = lla.launch_count() - n_launch0
    clk = clocks.stop()
    stage_ms, n_calls = lla.profile_collect()
    if lla.lla_stream_status() != 0:
        raise RuntimeError("liblla reported an error during the timed steps")

    # each repetition times exactly K steps; the line reports the median repetition
    rep_ms = [sum(a.elapsed_time(b) for a, b in ev[r * args.steps:(r + 1) * args.steps])
              for r in range(reps)]
    ms = statistics.median(rep_ms)
    ms = max_over_ranks(ms, world)
    ms_per_step = ms / args.steps
    value = job_rate(w.queries, world, ms_per_step / 1e3)

    parity = None
    if timer is not None:  # the oracle leg: sampled rows of the timed output vs the oracle
        rows = W.sample_rows(w.B * w.H, w.T, PARITY_ROWS, seed=77)
        ref = timer.values(rows, h, lam)
        got = out.float().reshape(-1, w.dv)[torch.tensor(rows, device=out.device)]
        parity = parity_summary(got.cpu().double().numpy(), ref, v.float().numpy(),
                                1e-3 if w.dtype == "f32" else 2e-2, len(rows))
        timer.close()

    # end to end through the C ABI on pinned host buffers (H2D + compute + D2H every step)
    e2e = None
    eb = q.element_size()
    if not args.no_e2e and not opts:  # the host entry point runs the default options only
        hq, hk, hv = (t.pin_memory() for t in (q, k, v))
        hout = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
        for _ in range(2):
            lla.lla_forward_host(hq, hk, hv, h, lam, out=hout, stream=stream)
        e2e_steps = max(3, min(args.steps, 10))
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(e2e_steps):
            lla.lla_forward_host(hq, hk, hv, h, lam, out=hout, stream=stream)
        e2e_s = (time.perf_counter() - t0) / e2e_steps
        e2e_s = max_over_ranks(e2e_s, world)
        e2e = {"value": job_rate(w.queries, world, e2e_s), "unit": UNIT,
               "h2d_bytes_per_step": (q.numel() + k.numel() + v.numel()) * eb,
               "d2h_bytes_per_step": out.numel() * eb}

    peaks, peak_src = load_peaks()
    # bf16 runs on the tensor cores (d < 64: on zero-padded d = dv = 64 copies of q, k, v)
    tensor_path = w.dtype == "bf16"
    per_call = {k_: v_ / max(n_calls, 1) for k_, v_ in stage_ms.items()}
    pairs = causal_pairs(w)
    if tensor_path:
        # the dominant kernel is the moment contraction; the weight sweeps are their own launch
        kernel_file = "lla_moments_pass_tc.cu"
        con_ms, w_ms = per_call["moments"], per_call["weights"]
        achieved = pairs * contraction_flops_per_pair(w.d) / (con_ms / 1e3) / 1e12
        peak = float(peaks.get("bf16_tflops", PEAKS_FALLBACK["bf16_tflops"]))
        stage_ms_total = con_ms + w_ms
        roof = {"kernel": "moment contraction (lla_moments_pass_tc.cu: tcgen05 cta_group::2, TMA)"
                          + (f"; d = {w.d} zero-padded to 64" if w.d < 64 else ""),
                "bound": "tensor", "peak_source": f"bf16 dense, burst ({peak_src})",
                "flops_per_unit": contraction_flops_per_pair(w.d), "unit_of_work": "causal pair",
                "units_per_launch": pairs,
                "executed_tflops": pairs * tc_executed_flops_per_pair(w.d) / (con_ms / 1e3) / 1e12,
                "moments_stage": {
                    "what": "weight sweeps (lla_weights_tc.cu) + contraction, the logit counted "
                            "once: 2d + 2(1 + d + d(d+1)/2) flop per pair",
                    "ms": stage_ms_total, "weights_ms": w_ms,
                    "tflops": pairs * moments_flops_per_pair(w.d) / (stage_ms_total / 1e3) / 1e12,
                    "frac": pairs * moments_flops_per_pair(w.d) / (stage_ms_total / 1e3) / 1e12
                    / peak}}
        avg_ms = con_ms
    else:
        kernel_file = "lla_moments_ffma.cu"
        mom_ms = per_call["moments"]
        achieved = pairs * moments_flops_per_pair(w.d) / (mom_ms / 1e3) / 1e12
        peak = fp32_alu_peak_tflops(peaks)
        roof = {"kernel": "moments (lla_moments_ffma.cu)", "bound": "alu",
                "peak_source": f"fp32 FMA: {SM_COUNT} SMs x {FP32_LANES_PER_SM} lanes x 2 x "
                               f"{peaks.get('sm_max_mhz', 2070)} MHz ({peak_src} clock)",
                "flops_per_unit": moments_flops_per_pair(w.d), "unit_of_work": "causal pair",
                "units_per_launch": pairs}
        avg_ms = mom_ms
    roof.update({"achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                 "traffic": recorded_traffic(kernel_file, w), "avg_launch_ms": avg_ms})
    if args.strategy == "cg":
        # The moments stage is reduced to its two weight sweeps; the CG passes vary in number.
        roof = None
    step_tflops = step_flops(w) * world / (ms_per_step / 1e3) / 1e12

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if tensor_path else "f32",
            "data": "synthetic",
            "config": {"workload": f"{w.name}: {w.describe()}, {w.recipe()}, h={h}, "
                                   f"lambda={lam}, seed {w.seed}",
                       "B": w.B, "H": w.H, "T": w.T, "d": w.d, "dv": w.dv, "io_dtype": w.dtype,
                       "l2": "flushed between steps (256 MiB write outside the step events)",
                       "parallelism": f"replica per GPU x{world}",
                       "strategy": (f"cg (max {args.cg_iters} passes, rel. residual "
                                    f"{args.cg_tol:g})" if args.strategy == "cg"
                                    else "dense moments + Cholesky"),
                       "form": ("page form, exact-LLA epilogue (O1 - O2) / (d1 - d2)"
                                if args.form == "page" else "centred")},
            "tflops": step_tflops,
            "bf16_peak_fraction": step_tflops / float(peaks.get("bf16_tflops", 1900.0)),
            "roofline": roof,
            "stage_ms_per_step": {k_: v_ / max(n_calls, 1) for k_, v_ in stage_ms.items()},
            "cpu_baseline": cpu,
            "parity": parity,
            "e2e": e2e,
            "gpu_launches": n_launch,
            "timed_repeats": {"repeats": reps, "steps_each": args.steps,
                              "ms_per_step_each": [x / args.steps for x in rep_ms],
                              "gpu_launches_per_repeat": n_launch // reps},
            "clocks": clk,
            "wall_s_timed": t_wall,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())

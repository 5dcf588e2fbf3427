"""Benchmark of the packed-polynomial activation kernels on GB300.

Workload (one step): the HBM-resident isolated sweep of "Fast Polynomial
Transcendentals for LLMs" (§4.2, Table 3) -- 268,435,456-element FP16
tensors (512 MiB each), x ~ N(0, 3^2) with 1 % uniform in [-40, 40],
dy ~ N(0, 1) -- through the six programs: sigmoid D3, tanh D4, SiLU D3,
GELU D5 forward and the direct sigma' D4, tanh' D4 backward.  The inputs are
four times larger than L2, so no L2 flush is needed between steps.

Reported (one JSON line, rank 0): whole-job Gelem/s of the step (all ranks),
the roofline of the dominant kernel against the measured HBM bandwidth (and
against the library's own streaming probe moving the same bytes), each of
the six programs against both MUFU-native controls (FP32 and packed
tanh.approx) and torch's native op under the paper's alternating timing
protocol (§4.2: nine rounds, order reversed every round, median of per-round
means), the SwiGLU kernels (dense [8192 x 14336] and ragged 131,072 x 2048
BF16), the L2-resident 4,194,304-element sweep with its L2 roof (a long
streaming-probe launch over the same sizes), l2_frac per program and the
launch-cost intercept / streaming-rate slope of the size curve, an
end-to-end figure through the public API with host buffers, SM clocks
sampled around the timed region, and the CPU replay oracle on bounded
samples of every configuration, on every host core (one spawned worker
process per core) and on one core.

``--impl reference`` times the CPU replay oracle itself as the reference arm,
on every host core in the same way.
Multi-GPU: one process per GPU (torchrun); every rank runs the same
per-GPU workload with no collective on the data path (weak scaling).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import threading
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "Gelem/s and achieved HBM GB/s (% of roofline) per program fwd/bwd vs MUFU control"
UNIT = "Gelem/s"
WORKLOAD = "HBM-resident isolated sweep: 268,435,456-element FP16 tensors, six programs"
SIX = [("sigmoid", 0, 3), ("tanh", 0, 4), ("silu", 0, 3), ("gelu", 0, 5),
       ("sigmoid", 1, 4), ("tanh", 1, 4)]
FN = {"sigmoid": 0, "tanh": 1, "silu": 2, "gelu": 3}
BYTES = {0: 4, 1: 6}            # algorithmic bytes per element: fwd x + y, bwd x + dy + dx
# the files that define the six programs' kernels (their DRAM traffic record
# is void once any of them changes)
KERNEL_SOURCES = ["stream_kernel.cuh", "poly_ops.cuh", "packed.cuh", "kern_act.cu"]


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def kernel_source_hash():
    """Hash of the kernel sources with comments and blank space removed, so
    that only a change to the code itself invalidates recorded counters."""
    import re
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "polynomial_activation_gb300", "csrc", name)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(kernel_key):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    src = kernel_source_hash()
    with open(path) as f:
        for line in f:
            parts = line.split()
            if len(parts) >= 3 and not line.startswith("#") and parts[0] == kernel_key:
                if parts[2] == src:
                    return int(parts[1])
    return None


def recorded_dram_peak():
    """ncu's DRAM peak for this GPU (GB/s) from the committed summary, or None."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        for line in f:
            parts = line.split()
            if len(parts) == 2 and parts[0] == "dram_peak_gbs":
                return float(parts[1])
    return None


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples every `period_ms`, each
    stamped on arrival.  start() returns once sampling is running; stop()
    waits for the first sample after it.  The record keeps every sample from
    the last one before start() to the first one after stop(), so a timed
    region shorter than the period is still bracketed by two readings."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap,clocks.mem")

    def __init__(self, index, period_ms=50):
        self.index = index
        self.period_ms = period_ms
        self.proc = None
        self.lines = []            # (monotonic arrival time, text)
        self.arrived = threading.Condition()
        self.reader = None
        self.t0 = self.t1 = None

    def _read(self):
        for line in self.proc.stdout:
            with self.arrived:
                self.lines.append((time.monotonic(), line))
                self.arrived.notify_all()
        with self.arrived:
            self.arrived.notify_all()

    def _wait_for(self, count, timeout):
        with self.arrived:
            self.arrived.wait_for(lambda: len(self.lines) >= count, timeout=timeout)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.period_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.reader = threading.Thread(target=self._read, daemon=True)
        self.reader.start()
        self._wait_for(1, 10)
        self.t0 = time.monotonic()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        self.t1 = time.monotonic()
        with self.arrived:
            n_at_stop = sum(1 for t, _ in self.lines if t <= self.t1)
        self._wait_for(n_at_stop + 1, 2.0)
        self.proc.terminate()
        self.proc.wait(timeout=10)
        self.reader.join(timeout=10)
        before = [i for i, (t, _) in enumerate(self.lines) if t <= self.t0]
        after = [i for i, (t, _) in enumerate(self.lines) if t > self.t1]
        lo = before[-1] if before else 0
        hi = after[0] if after else len(self.lines) - 1
        sm, smax, mem, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for _, line in self.lines[lo:hi + 1]:
            v = [s.strip() for s in line.split(",")]
            if len(v) < 7:
                continue
            try:
                sm.append(float(v[0]))
                smax.append(float(v[1]))
                if len(v) > 7:
                    mem.append(float(v[7]))
            except ValueError:
                continue
            for nm, flag in zip(names, v[3:7]):
                if flag.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "mem_mhz": statistics.median(mem) if mem else None,
                "samples": len(sm), "period_ms": self.period_ms,
                "window_ms": (self.t1 - self.t0) * 1e3, "reasons": sorted(reasons)}


def environment(dev):
    """GPU, driver and software the numbers were taken with."""
    import torch
    props = torch.cuda.get_device_properties(dev)
    env = {"gpu": props.name, "sms": props.multi_processor_count,
           "hbm_gib": round(props.total_memory / 2 ** 30, 1), "cuda_runtime": torch.version.cuda,
           "torch": torch.__version__, "host_cores": os.cpu_count()}
    try:
        r = subprocess.run(["nvidia-smi", "-i", str(dev.index or 0), "--query-gpu=driver_version",
                            "--format=csv,noheader"], capture_output=True, text=True, timeout=30)
        env["driver"] = r.stdout.strip() or None
    except (OSError, subprocess.TimeoutExpired):
        env["driver"] = None
    return env


def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if n_gpus > 0 else "gloo")
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world, device):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# --------------------------------------------------------------- CPU oracle

def _golden(key):
    from oracle.replay import Program
    with open(os.path.join(ROOT, "tests", "golden", "programs.json")) as f:
        v = json.load(f)[key]
    return Program(fn=v["fn"], direction=v["direction"], fmt=key.split(".")[2],
                   degree=int(key.split(".D")[1]), li=v["li"], lc=v["lc"], coef=tuple(v["coef"]),
                   lc_bits=v["lc_bits"])


def oracle_programs():
    """The oracle fitter's programs for the six (written to
    tests/golden/programs.json by a script that calls only the oracle)."""
    return [_golden(f"{name}.{'bwd' if d else 'fwd'}.f16.D{D}") for name, d, D in SIX]


_PROGS = {}


def _replay(kind, *arrays):
    """The oracle over one piece of a sample; returns the seconds it took.
    kind "six": the six FP16 programs over x (forward) and x, dy (backward),
    in pieces of 2^22 elements (which bounds the replay's FP64 temporaries);
    kind "swiglu": the BF16 SwiGLU forward and backward (D3 SiLU, centred D4
    SiLU derivative) over rows of g, u, dy."""
    from oracle.replay import backward, forward, swiglu_backward, swiglu_forward
    if kind not in _PROGS:
        _PROGS[kind] = (oracle_programs() if kind == "six" else
                        (_golden("silu.fwd.bf16.D3"), _golden("silu.bwd.bf16.D4")))
    progs = _PROGS[kind]
    t0 = time.perf_counter()
    if kind == "six":
        x, dy = arrays
        piece = 1 << 22
        for lo in range(0, x.size, piece):
            xs, dys = x[lo:lo + piece], dy[lo:lo + piece]
            for p, (name, d, D) in zip(progs, SIX):
                if d == 0:
                    forward(p, xs)
                else:
                    backward(p, xs, dys)
    else:
        g, u, dy = arrays
        piece = max(1, (1 << 21) // max(1, g.shape[-1]))
        for lo in range(0, g.shape[0], piece):
            gs, us, dys = g[lo:lo + piece], u[lo:lo + piece], dy[lo:lo + piece]
            swiglu_forward(progs[0], gs, us)
            swiglu_backward(progs[0], progs[1], gs, us, dys)
    return time.perf_counter() - t0


def _warm_worker(_):
    time.sleep(0.2)                     # one task per worker: every worker imports the oracle
    _replay("six", np.zeros(8, np.uint16), np.zeros(8, np.uint16))
    z = np.zeros((1, 8), np.uint16)
    _replay("swiglu", z, z, z)
    return os.getpid()


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


class OraclePool:
    """The CPU replay oracle, unchanged, on `workers` host cores: a sample is
    cut into one contiguous piece per worker process (along the first axis).
    Workers are spawned (no CUDA state is inherited) and import the oracle
    before any timing."""

    def __init__(self, workers):
        self.workers = max(1, int(workers))
        self.pool = None
        if self.workers > 1:
            import multiprocessing as mp
            self.pool = mp.get_context("spawn").Pool(self.workers)
            self.pool.map(_warm_worker, range(self.workers), chunksize=1)

    def run(self, kind, *arrays):
        """(wall seconds, [seconds per piece], [rows per piece])."""
        m = arrays[0].shape[0]
        if self.pool is None:
            t0 = time.perf_counter()
            t = _replay(kind, *arrays)
            return time.perf_counter() - t0, [t], [m]
        b = np.linspace(0, m, self.workers + 1).astype(np.int64)
        args = [(kind,) + tuple(a[b[i]:b[i + 1]] for a in arrays) for i in range(self.workers)]
        t0 = time.perf_counter()
        per = self.pool.starmap(_replay, args, chunksize=1)
        return time.perf_counter() - t0, per, [int(b[i + 1] - b[i]) for i in range(self.workers)]

    def close(self):
        if self.pool is not None:
            self.pool.close()
            self.pool.join()


def oracle_sample_time(n_sample, workers=1):
    """Time the CPU replay oracle on the first n_sample elements of the
    HBM-resident workload through each of the six programs, on `workers`
    processes.  Returns (wall seconds, elements x programs, CPU seconds,
    per-core Gelem/s)."""
    x, dy = workloads.isolated_hbm("f16", n=n_sample)
    pool = OraclePool(workers)
    try:
        wall, per, sizes = pool.run("six", x, dy)
    finally:
        pool.close()
    per_core = statistics.mean(6 * m / t / 1e9 for m, t in zip(sizes, per) if t > 0)
    return wall, 6 * n_sample, sum(per), per_core


def cpu_baseline_configs(cores, gpu, n_hbm_sample=1 << 24, single_scale=8):
    """The CPU replay oracle on every configuration of the GPU measurement,
    on all `cores` host cores and on one core, beside the GPU's figure for
    the same work (gpu: config -> Gelem/s).  Samples are bounded (the whole
    4,194,304-element L2 sweep; the first elements or rows of the others);
    the single-core run takes 1/single_scale of the multi-core sample.
    Gelem/s counts elements x programs for the sweeps and elements x passes
    (forward + backward) for SwiGLU."""
    out = {}
    pool = OraclePool(cores)
    one = OraclePool(1)
    try:
        cases = []
        x, dy = workloads.isolated_l2("f16")
        cases.append(("l2_resident", "six", (x, dy), 6,
                      "the whole 4,194,304-element L2-resident sweep, six FP16 programs"))
        x, dy = workloads.isolated_hbm("f16", n=n_hbm_sample)
        cases.append(("hbm_resident", "six", (x, dy), 6,
                      f"first {n_hbm_sample} elements of the HBM-resident sweep, six FP16 programs"))
        rows = 1024
        g, u, d = workloads.dense_swiglu("bf16", rows=rows)
        cases.append(("dense_swiglu", "swiglu", (g, u, d), 2,
                      f"first {rows} of 8,192 rows x 14,336 of the dense BF16 SwiGLU, forward + "
                      "backward"))
        g, u, d, _ = workloads.ragged_swiglu("bf16")
        rows = 8192
        cases.append(("ragged_swiglu", "swiglu", (g[:rows], u[:rows], d[:rows]), 2,
                      f"first {rows} of 131,072 rows x 2,048 of the ragged BF16 SwiGLU, forward "
                      "+ backward"))
        del g, u, d
        for key, kind, arrays, passes, what in cases:
            elems = arrays[0].size
            wall, per, _ = pool.run(kind, *arrays)
            m1 = max(1, arrays[0].shape[0] // single_scale)
            wall1, _, _ = one.run(kind, *(a[:m1] for a in arrays))
            e1 = arrays[0][:m1].size
            entry = {"gelem_s": passes * elems / wall / 1e9, "cores": pool.workers,
                     "single_thread_gelem_s": passes * e1 / wall1 / 1e9,
                     "elements": elems, "single_thread_elements": e1, "passes": passes,
                     "wall_s": wall, "cpu_s": sum(per), "single_thread_s": wall1,
                     "sample": what}
            if gpu.get(key):
                entry["gpu_gelem_s"] = gpu[key]
                entry["gpu_over_cpu"] = gpu[key] / entry["gelem_s"]
            out[key] = entry
    finally:
        pool.close()
        one.close()
    return out


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    cores = host_cores()
    per_step = int(np.clip(2 ** 27 // max(1, args.steps + args.warmup), 2 ** 16, 2 ** 22))
    x, dy = workloads.isolated_hbm("f16", n=per_step)
    pool = OraclePool(cores)
    try:
        for _ in range(args.warmup):
            pool.run("six", x, dy)
        t0 = time.perf_counter()
        for _ in range(args.steps):
            pool.run("six", x, dy)
        dt = time.perf_counter() - t0
    finally:
        pool.close()
    value = 6 * per_step * args.steps / dt / 1e9
    sample = (f"first {per_step} elements of x and dy per program per step, cut into {cores} "
              f"pieces on {cores} host cores (CPU replay oracle, numpy)")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f16", "data": "synthetic",
            "config": {"workload": WORKLOAD, "elements_per_program": per_step,
                       "note": "bounded sample of the workload; the oracle is a deliberately "
                               "plain CPU replay"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------- GPU arm

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-extras", action="store_true", help="only the timed step")
    ap.add_argument("--cpu-sample", type=int, default=1 << 24,
                    help="elements per program for the CPU oracle baseline (0 = skip)")
    ap.add_argument("--elements", type=int, default=workloads.N_HBM,
                    help="tensor size (a smaller case for profiling runs)")
    ap.add_argument("--no-e2e", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)

    import torch
    from polynomial_activation_gb300 import binding as B

    rank, world, local = dist_setup(args.gpus)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    peak, peak_kind = peaks()

    # ---- inputs (host generation once, then resident in HBM)
    xh, dyh = workloads.isolated_hbm("f16", n=args.elements)
    n = xh.size
    x = torch.from_numpy(xh.view(np.int16)).to(dev).view(torch.float16)
    dy = torch.from_numpy(dyh.view(np.int16)).to(dev).view(torch.float16)
    outs = [torch.empty_like(x) for _ in SIX]
    for name, d, D in SIX:                      # fit / install programs outside timing
        assert B.poly_get_program(FN[name], d, B.POLY_F16).degree == D

    def launch(i, ctrl=None):
        name, d, D = SIX[i]
        if ctrl is None:
            if d == 0:
                B.poly_act_fwd(FN[name], B.POLY_F16, x, outs[i], n)
            else:
                B.poly_act_bwd(FN[name], B.POLY_F16, x, dy, outs[i], n)
        elif d == 0:
            B.poly_ctrl_act_fwd_v(ctrl, FN[name], B.POLY_F16, x, outs[i], n)
        else:
            B.poly_ctrl_act_bwd_v(ctrl, FN[name], B.POLY_F16, x, dy, outs[i], n)

    def timed_steps(ctrl, steps, per_kernel=True):
        ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in SIX] for _ in range(steps)] if per_kernel else None
        barrier(world)
        torch.cuda.synchronize()
        t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        for s in range(steps):
            for i in range(len(SIX)):
                if per_kernel:
                    ev[s][i][0].record(stream)
                launch(i, ctrl)
                if per_kernel:
                    ev[s][i][1].record(stream)
        t_end.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        total_ms = t_start.elapsed_time(t_end)
        per = None
        if per_kernel:
            per = [sum(ev[s][i][0].elapsed_time(ev[s][i][1]) for s in range(steps)) / steps
                   for i in range(len(SIX))]
        return total_ms, per

    for _ in range(args.warmup):
        for i in range(len(SIX)):
            launch(i)
    clocks = ClockSampler(local)
    clocks.start()
    # the timed region: K steps back to back (no events between kernels)
    total_ms, _ = timed_steps(None, args.steps, per_kernel=False)
    # per-kernel durations for the roofline: a second timed pass with an event
    # pair around every launch; the clock samples cover both passes
    _, per_ms = timed_steps(None, max(50, args.steps // 4))
    clk = clocks.stop()
    total_ms = max_over_ranks(total_ms, world, dev)
    ms_per_step = total_ms / args.steps
    elems_per_step = 6 * n * world
    value = elems_per_step / (ms_per_step * 1e-3) / 1e9

    result = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
              "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
              "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
              "dtype": "f16", "data": "synthetic",
              "config": {"workload": WORKLOAD, "elements": n, "programs": [f"{a}.{'bwd' if d else 'fwd'}.D{D}" for a, d, D in SIX],
                         "inputs": "x ~ N(0, 3^2) with 1 % uniform in [-40, 40] (PCG64 seed 0), "
                                   "dy ~ N(0, 1) (seed 1), generated on the host, resident in HBM",
                         "l2": "inputs (512 MiB per tensor) larger than L2; no flush",
                         "parallelism": f"replicas x{world}, no collective"},
              "gpu_launches": len(SIX) * args.steps,
              "clocks": clk, "env": environment(dev)}

    # ---- per program: poly vs the two MUFU controls (vs torch native), the
    # paper's alternating protocol (§4.2): 9 rounds, order reversed each round
    programs = {}
    dom = max(range(len(SIX)), key=lambda i: per_ms[i])
    for i, (name, d, D) in enumerate(SIX):
        key = f"{name}.{'bwd' if d else 'fwd'}.D{D}"
        arms = {"poly": lambda i=i: launch(i),
                "ctrl_fp32": lambda i=i: launch(i, ctrl=B.POLY_CTRL_FP32),
                "ctrl_packed": lambda i=i: launch(i, ctrl=B.POLY_CTRL_PACKED)}
        if not args.no_extras:
            arms["torch"] = torch_native(name, d, x, dy)
        t = alternating(arms, stream, rounds=9, reps=20 if n >= (1 << 26) else 100,
                        warm=10 if n >= (1 << 26) else 100)
        gb = BYTES[d] * n / 1e9
        pm = t["poly"]["ms"]
        best = min(("ctrl_fp32", "ctrl_packed"), key=lambda k: t[k]["ms"])
        entry = {"poly_ms": pm, "poly_gelem_s": n / pm / 1e6, "poly_gbs": gb / pm * 1e3,
                 "poly_frac": gb / pm * 1e3 / peak,
                 "ctrl_fp32_ms": t["ctrl_fp32"]["ms"], "ctrl_packed_ms": t["ctrl_packed"]["ms"],
                 "ctrl_ms": t[best]["ms"], "ctrl_gbs": gb / t[best]["ms"] * 1e3,
                 "best_ctrl": best, "speedup_vs_ctrl": t[best]["ms"] / pm,
                 "speedup_vs_ctrl_fp32": t["ctrl_fp32"]["ms"] / pm,
                 "speedup_vs_ctrl_packed": t["ctrl_packed"]["ms"] / pm,
                 "rounds": {k: {"median_ms": v["ms"], "min_ms": v["min_ms"], "max_ms": v["max_ms"]}
                            for k, v in t.items()}}
        if "torch" in t:
            entry["torch_native_ms"] = t["torch"]["ms"]
            entry["speedup_vs_torch"] = t["torch"]["ms"] / pm
        programs[key] = entry
    result["programs"] = programs
    result["programs_protocol"] = ("9 alternating rounds (poly, FP32 control, packed control, "
                                   "torch; reversed order on odd rounds) of 20 back-to-back "
                                   "event-timed calls per arm after 10 warm-ups; median of "
                                   "per-round means, min/max kept; speedup_vs_ctrl against the "
                                   "faster control")

    # ---- the two backward rows Table 3 lost in extraction (SiLU' and GELU'
    # D4, the centred derivative fits), same protocol, against PyTorch's fused
    # backward kernels from x (the paper quotes GELU backward at 1.615x native
    # on HBM)
    if not args.no_extras:
        extra = {}
        for name in ("silu", "gelu"):
            fn = FN[name]
            arms = {"poly": lambda fn=fn: B.poly_act_bwd(fn, B.POLY_F16, x, dy, outs[0], n),
                    "ctrl_fp32": lambda fn=fn: B.poly_ctrl_act_bwd_v(B.POLY_CTRL_FP32, fn,
                                                                      B.POLY_F16, x, dy, outs[0], n),
                    "ctrl_packed": lambda fn=fn: B.poly_ctrl_act_bwd_v(B.POLY_CTRL_PACKED, fn,
                                                                        B.POLY_F16, x, dy, outs[0], n),
                    "torch": (lambda: torch.ops.aten.silu_backward(dy, x)) if name == "silu"
                             else (lambda: torch.ops.aten.gelu_backward(dy, x))}
            t = alternating(arms, stream, rounds=9, reps=20, warm=10)
            pm = t["poly"]["ms"]
            best = min(("ctrl_fp32", "ctrl_packed"), key=lambda k: t[k]["ms"])
            extra[f"{name}.bwd.D4"] = {
                "poly_ms": pm, "poly_gbs": 6 * n / pm / 1e6, "poly_frac": 6 * n / pm / 1e6 / peak,
                "ctrl_fp32_ms": t["ctrl_fp32"]["ms"], "ctrl_packed_ms": t["ctrl_packed"]["ms"],
                "torch_native_ms": t["torch"]["ms"], "best_ctrl": best,
                "speedup_vs_ctrl": t[best]["ms"] / pm, "speedup_vs_torch": t["torch"]["ms"] / pm}
        result["programs_lost_rows"] = extra

    # ---- roofline of the dominant kernel
    name, d, D = SIX[dom]
    kkey = f"{name}.{'bwd' if d else 'fwd'}.D{D}"
    nbytes = BYTES[d] * n
    ach = nbytes / (per_ms[dom] * 1e-3) / 1e9
    b2b = nbytes / (programs[kkey]["poly_ms"] * 1e-3) / 1e9
    stream_gbs, stream_rates = same_shape_stream_gbs(x, dy, outs[0], n, 2 if d else 1, stream)
    result["roofline"] = {"kernel": f"dense_kernel<OpBwd|OpFwd> {kkey}", "bound": "hbm",
                          "achieved": ach, "peak": peak, "unit": "GB/s", "frac": ach / peak,
                          "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured" else "fallback",
                          "algorithmic_bytes_per_launch": nbytes,
                          "traffic": recorded_traffic(kkey) if n == workloads.N_HBM else None,
                          "share_of_step": per_ms[dom] / sum(per_ms),
                          "above_peak": ach > peak,
                          "achieved_back_to_back": b2b, "frac_back_to_back": b2b / peak,
                          "dram_peak_gbs": recorded_dram_peak(),
                          "frac_vs_dram_peak": (ach / recorded_dram_peak()
                                                if recorded_dram_peak() else None),
                          "same_shape_stream_gbs": stream_gbs,
                          "same_shape_stream_by_inflight": stream_rates,
                          "frac_vs_same_shape_stream": ach / stream_gbs,
                          "note": "achieved: algorithmic bytes / mean event-timed launch inside "
                                  "the step (the last dirty lines of a launch are written back "
                                  "during the next); back_to_back: the same kernel launched 20 "
                                  "times in a row, so every write-back but the last falls inside "
                                  "the timed calls; peak: a torch copy_, which a streaming kernel "
                                  "can exceed; same_shape_stream: the library's own streaming "
                                  "probe moving the same bytes (reads and writes) with the "
                                  "kernels' loads and stores; dram_peak: ncu's DRAM peak for "
                                  "this GPU (profiles/dram_traffic.txt)"}

    # ---- extras: SwiGLU and the L2-resident sweep
    if not args.no_extras:
        result["programs_bf16"] = bf16_extras(x, dy, n, stream, peak)
        result["softcap"] = softcap_extras(x, dy, outs[0], n, stream, peak)
        result["exp2"] = exp2_extras(dev, stream, peak)
        result["rope"] = rope_extras(dev, stream, peak)
        result["swiglu"] = swiglu_extras(args, dev, stream, peak)
        result["components"] = component_extras(dev, stream, peak)
        result["l2_resident"] = l2_extras(dev, stream)
        result["host_us_per_call"] = host_cost_extras(dev)

    # ---- end to end through the public API with host buffers
    if not args.no_e2e:
        result["e2e"] = e2e(args, dev, stream, xh, dyh)

    # ---- CPU oracle on bounded samples (every config with the extras; the
    # step's config alone otherwise)
    if rank == 0 and args.cpu_sample > 0:
        cores = host_cores()
        if args.no_extras:
            wall, elems, cpu_s, per_core = oracle_sample_time(args.cpu_sample, cores)
            result["cpu_baseline"] = {"value": elems / wall / 1e9, "unit": UNIT, "cores": cores,
                                      "kind": "oracle", "per_core_value": per_core,
                                      "sample": f"first {args.cpu_sample} elements of the "
                                                f"workload through each of the six programs, one "
                                                f"contiguous piece per core (numpy replay, "
                                                f"{wall:.1f} s wall, {cpu_s:.1f} s of CPU work)"}
        else:
            gpu = {"hbm_resident": value / world}
            l2 = result.get("l2_resident", {})
            us = [v["poly_us"] for k, v in l2.items() if isinstance(v, dict) and "poly_us" in v
                  and k.count(".") == 2]
            if len(us) == 6:
                gpu["l2_resident"] = 6 * workloads.N_L2 / sum(us) / 1e3
            sw = result.get("swiglu", {})
            for key, fwd, bwd, rows, cols in (
                    ("dense_swiglu", "dense_fwd", "dense_bwd", workloads.DENSE_ROWS,
                     workloads.DENSE_COLS),
                    ("ragged_swiglu", "ragged_fwd", "ragged_bwd",
                     workloads.RAGGED_TOKENS * workloads.RAGGED_TOPK, workloads.RAGGED_COLS)):
                if fwd in sw and bwd in sw:
                    gpu[key] = 2 * rows * cols / (sw[fwd]["ms"] + sw[bwd]["ms"]) / 1e6
            per_config = cpu_baseline_configs(cores, gpu, n_hbm_sample=args.cpu_sample)
            h = per_config["hbm_resident"]
            result["cpu_baseline"] = {"value": h["gelem_s"], "unit": UNIT, "cores": cores,
                                      "kind": "oracle",
                                      "single_thread_value": h["single_thread_gelem_s"],
                                      "sample": h["sample"] + f" on {cores} host cores (numpy "
                                                f"replay, {h['wall_s']:.1f} s wall, "
                                                f"{h['cpu_s']:.1f} s of CPU work); the other "
                                                "configs in per_config",
                                      "per_config": per_config}
    if rank == 0:
        if args.elements != workloads.N_HBM:
            result["config"]["workload"] = f"profiling case: {args.elements} elements"
        print(json.dumps(result), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def alternating(arms, stream, rounds=9, reps=20, warm=20, graph=False):
    """The paper's isolated-timing protocol ("Fast Polynomial Transcendentals
    for LLMs", §4.2): after `warm` warm-up calls per arm, `rounds` rounds in
    which the arms run in their given order on even rounds and in reverse on
    odd rounds (polynomial first, then native first), each arm timed as
    `reps` back-to-back calls by a CUDA-event pair on the stream -- or, with
    graph=True, as one replay of a CUDA graph holding `reps` captured calls
    (microsecond kernels are otherwise bounded by the host's launch rate).
    Per arm: the median of the per-round means (ms per call), their min and
    max, and every round."""
    import torch
    for f in arms.values():
        for _ in range(warm):
            f()
    torch.cuda.synchronize()
    run = {}
    if graph:
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        for k, f in arms.items():
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(side):
                with torch.cuda.graph(g, stream=side):
                    for _ in range(reps):
                        f()
            torch.cuda.synchronize()
            g.replay()
            torch.cuda.synchronize()
            run[k] = g.replay
    else:
        for k, f in arms.items():
            def many(f=f):
                for _ in range(reps):
                    f()
            run[k] = many
    per = {k: [] for k in arms}
    order = list(arms)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(rounds * len(order))]
    i = 0
    torch.cuda.synchronize()
    for r in range(rounds):
        for k in (order if r % 2 == 0 else order[::-1]):
            e0, e1 = ev[i]
            i += 1
            e0.record(stream)
            run[k]()
            e1.record(stream)
            per[k].append((e0, e1))
    torch.cuda.synchronize()
    out = {}
    for k, pairs in per.items():
        ms = [a.elapsed_time(b) / reps for a, b in pairs]
        out[k] = {"ms": statistics.median(ms), "min_ms": min(ms), "max_ms": max(ms),
                  "round_ms": ms}
    return out


def _time(fn, stream, reps, warm=3):
    import torch
    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


def softcap_extras(x, dy, y, n, stream, peak, alpha=30.0):
    """alpha tanh(x / alpha) forward and its backward on the step's tensors,
    with the direct tanh' D4 program and with the differentiated D3 one."""
    from polynomial_activation_gb300 import binding as B
    f16 = B.POLY_F16
    res = {"alpha": alpha}
    for label, fn, nbytes in [
        ("fwd", lambda: B.poly_softcap_fwd(f16, alpha, x, y, n), 4),
        ("bwd_direct_D4", lambda: B.poly_softcap_bwd(f16, alpha, x, dy, y, n), 6),
    ]:
        ms = _time(fn, stream, 20)
        res[label] = {"ms": ms, "gbs": nbytes * n / ms / 1e6, "frac": nbytes * n / ms / 1e6 / peak}
    d = B.poly_derive_program(B.poly_get_program(B.POLY_TANH, B.POLY_FWD, f16))
    B.poly_set_program(d)
    try:
        ms = _time(lambda: B.poly_softcap_bwd(f16, alpha, x, dy, y, n), stream, 20)
        res["bwd_differentiated_D3"] = {"ms": ms, "gbs": 6 * n / ms / 1e6,
                                        "frac": 6 * n / ms / 1e6 / peak,
                                        "stated_max_abs_err": d.stated_max_abs_err}
    finally:
        B.poly_reset_programs()
        for name, dd, D in SIX:
            B.poly_get_program(FN[name], dd, f16)
    return res


def bf16_extras(x, dy, n, stream, peak, reps=30):
    """The six programs and their MUFU controls on BF16 copies of the step's
    tensors (same shapes and distribution; converted on the device)."""
    import torch
    from polynomial_activation_gb300 import binding as B
    bf = B.POLY_BF16
    xb, dyb = x.to(torch.bfloat16), dy.to(torch.bfloat16)
    y = torch.empty_like(xb)
    res = {}
    for name, d, D in SIX:
        prog = B.poly_get_program(FN[name], d, bf)
        if d == 0:
            fp = lambda: B.poly_act_fwd(FN[name], bf, xb, y, n)
            fc = lambda: B.poly_ctrl_act_fwd(FN[name], bf, xb, y, n)
            fk = lambda: B.poly_ctrl_act_fwd_v(B.POLY_CTRL_PACKED, FN[name], bf, xb, y, n)
        else:
            fp = lambda: B.poly_act_bwd(FN[name], bf, xb, dyb, y, n)
            fc = lambda: B.poly_ctrl_act_bwd(FN[name], bf, xb, dyb, y, n)
            fk = lambda: B.poly_ctrl_act_bwd_v(B.POLY_CTRL_PACKED, FN[name], bf, xb, dyb, y, n)
        tp, tc, tk = _time(fp, stream, reps), _time(fc, stream, reps), _time(fk, stream, reps)
        gb = BYTES[d] * n / 1e9
        res[f"{name}.{'bwd' if d else 'fwd'}.D{prog.degree}"] = {
            "poly_ms": tp, "poly_gbs": gb / tp * 1e3, "poly_frac": gb / tp * 1e3 / peak,
            "ctrl_ms": min(tc, tk), "ctrl_fp32_ms": tc, "ctrl_packed_ms": tk,
            "speedup_vs_ctrl": min(tc, tk) / tp}
    res["config"] = ("268,435,456 BF16 elements: the step's FP16 x and dy converted on the device; "
                     f"mean of {reps} launches each; speedup_vs_ctrl against the faster control")
    return res


def component_extras(dev, stream, peak, rounds=5, reps=100):
    """The paper's two component workloads (its B1 unary SiLU probe, 58,720,256
    BF16 values, and its B4 one-kernel expert SwiGLU activation, 24,576 rows x
    1,280), with its component protocol: 25 warm-up calls, then `rounds`
    alternating rounds of `reps` back-to-back calls per implementation, the
    median of the per-round means.  Polynomial kernel vs the MUFU control vs
    PyTorch eager (forward F.silu / F.silu(g) * u; backward aten.silu_backward
    / the two-output autograd formula)."""
    import torch
    from polynomial_activation_gb300 import binding as B
    F = torch.nn.functional
    bf = B.POLY_BF16
    gen = torch.Generator(device=dev).manual_seed(5)
    res = {}

    def run(impls, nbytes):
        for f in impls.values():
            for _ in range(25):
                f()
        per = {k: [] for k in impls}
        order = list(impls)
        for r in range(rounds):
            for k in (order if r % 2 == 0 else order[::-1]):
                per[k].append(_time(impls[k], stream, reps, warm=0))
        out = {}
        for k, v in per.items():
            ms = statistics.median(v)
            out[f"{k}_us"] = ms * 1e3
            out[f"{k}_gbs"] = nbytes / ms / 1e6
        out["poly_frac"] = out["poly_gbs"] / peak
        out["speedup_vs_ctrl"] = min(out["ctrl_us"], out["ctrl_packed_us"]) / out["poly_us"]
        out["speedup_vs_ctrl_fp32"] = out["ctrl_us"] / out["poly_us"]
        out["speedup_vs_ctrl_packed"] = out["ctrl_packed_us"] / out["poly_us"]
        out["speedup_vs_torch"] = out["torch_us"] / out["poly_us"]
        return out

    n = 58_720_256
    x = (torch.randn(n, device=dev, generator=gen) * 3).bfloat16()
    dy = torch.randn(n, device=dev, generator=gen).bfloat16()
    y = torch.empty_like(x)
    silu = FN["silu"]
    res["silu_probe_fwd"] = run({
        "poly": lambda: B.poly_act_fwd(silu, bf, x, y, n),
        "ctrl": lambda: B.poly_ctrl_act_fwd(silu, bf, x, y, n),
        "ctrl_packed": lambda: B.poly_ctrl_act_fwd_v(B.POLY_CTRL_PACKED, silu, bf, x, y, n),
        "torch": lambda: F.silu(x)}, 4 * n)
    res["silu_probe_bwd"] = run({
        "poly": lambda: B.poly_act_bwd(silu, bf, x, dy, y, n),
        "ctrl": lambda: B.poly_ctrl_act_bwd(silu, bf, x, dy, y, n),
        "ctrl_packed": lambda: B.poly_ctrl_act_bwd_v(B.POLY_CTRL_PACKED, silu, bf, x, dy, y, n),
        "torch": lambda: torch.ops.aten.silu_backward(dy, x)}, 6 * n)
    del x, dy, y
    rows, cols = 24_576, 1_280
    g = (torch.randn(rows, cols, device=dev, generator=gen) * 1.5).bfloat16()
    u = (torch.randn(rows, cols, device=dev, generator=gen) * 1.5).bfloat16()
    dy = torch.randn(rows, cols, device=dev, generator=gen).bfloat16()
    y, dg, du = torch.empty_like(g), torch.empty_like(g), torch.empty_like(g)
    m = rows * cols

    def torch_swiglu_bwd():
        du_ = dy * F.silu(g)
        dg_ = torch.ops.aten.silu_backward(dy * u, g)
        return dg_, du_

    res["expert_swiglu_fwd"] = run({
        "poly": lambda: B.poly_swiglu_fwd(bf, g, u, y),
        "ctrl": lambda: B.poly_ctrl_swiglu_fwd(bf, g, u, y),
        "ctrl_packed": lambda: B.poly_ctrl_swiglu_fwd_v(B.POLY_CTRL_PACKED, bf, g, u, y),
        "torch": lambda: F.silu(g) * u}, 6 * m)
    res["expert_swiglu_bwd"] = run({
        "poly": lambda: B.poly_swiglu_bwd(bf, g, u, dy, dg, du),
        "ctrl": lambda: B.poly_ctrl_swiglu_bwd(bf, g, u, dy, dg, du),
        "ctrl_packed": lambda: B.poly_ctrl_swiglu_bwd_v(B.POLY_CTRL_PACKED, bf, g, u, dy, dg, du),
        "torch": torch_swiglu_bwd}, 10 * m)
    res["config"] = ("BF16; SiLU probe 58,720,256 values, x ~ N(0, 3^2), dy ~ N(0, 1); expert "
                     "SwiGLU 24,576 x 1,280, g, u ~ N(0, 1.5^2), dy ~ N(0, 1); inputs drawn on the "
                     f"device (seed 5); {rounds} alternating rounds of {reps} calls, median; "
                     "no L2 flush (the paper's component protocol); GB/s = algorithmic bytes")
    return res


_COPY_MS = {}
_COPY_MS = {}
_COPY_MS = {}


def same_bytes_copy_ms(nbytes, dev, stream):
    """Time of a plain device copy that reads and writes nbytes in total: the
    attainable bandwidth at a kernel's own size (launch ramp and drain keep a
    ~50-100 us kernel below the long-copy peak)."""
    import torch
    if nbytes not in _COPY_MS:
        src = torch.empty(nbytes // 4, dtype=torch.int16, device=dev).random_(-30000, 30000)
        dst = torch.empty_like(src)
        _COPY_MS[nbytes] = _time(lambda: dst.copy_(src), stream, 20)
        del src, dst
    return _COPY_MS[nbytes]


def exp2_extras(dev, stream, peak, n=1 << 27):
    """2^x on FP32 tensors of 2^27 elements (512 MiB each, larger than L2)
    through each fractional core and the MUFU control (Appendix B.1)."""
    import torch
    from polynomial_activation_gb300 import binding as B
    x = torch.from_numpy(np.random.default_rng(7).uniform(-60, 10, n).astype(np.float32)).to(dev)
    y = torch.empty_like(x)
    res = {"config": f"{n} FP32 elements, x ~ U[-60, 10]"}
    for label, fn in [("D1", lambda: B.poly_exp2(B.POLY_EXP2_D1, x, y)),
                      ("PWL2", lambda: B.poly_exp2(B.POLY_EXP2_PWL2, x, y)),
                      ("D2", lambda: B.poly_exp2(B.POLY_EXP2_D2, x, y)),
                      ("D3", lambda: B.poly_exp2(B.POLY_EXP2_D3, x, y)),
                      ("mufu_ex2", lambda: B.poly_ctrl_exp2(x, y))]:
        ms = _time(fn, stream, 20)
        res[label] = {"ms": ms, "gbs": 8 * n / ms / 1e6, "frac": 8 * n / ms / 1e6 / peak,
                      "vs_same_bytes_copy": same_bytes_copy_ms(8 * n, dev, stream) / ms}
    return res


def rope_extras(dev, stream, peak, b=4, s=4096, hq=32, hkv=8, d=128):
    """Fused RoPE (Appendix B.2): FP16 Q [B, S, Hq, D] and K [B, S, Hkv, D] to
    the transposed layouts, with polynomial, MUFU and cached-table sine /
    cosine sharing the rotation and memory schedule."""
    import torch
    from polynomial_activation_gb300 import binding as B
    g = torch.Generator(device=dev).manual_seed(0)
    q = torch.randn((b, s, hq, d), generator=g, device=dev).to(torch.float16)
    k = torch.randn((b, s, hkv, d), generator=g, device=dev).to(torch.float16)
    qo = torch.empty((b, hq, s, d), dtype=torch.float16, device=dev)
    ko = torch.empty((b, hkv, s, d), dtype=torch.float16, device=dev)
    delta = torch.from_numpy(B.poly_rope_turn_increments(d).view(np.int32)).to(dev)
    # cached tables [S, D/2] from the polynomial variant's own values
    eye = torch.zeros((1, s, 1, d), dtype=torch.float16, device=dev)
    eye[..., 0::2] = 1.0
    cs_o = torch.empty((1, 1, s, d), dtype=torch.float16, device=dev)
    B.poly_rope_fwd(B.POLY_ROPE_POLY, eye, None, cs_o, None, delta, batch=1, seq=s, hq=1, hkv=0,
                    head_dim=d)
    cos_t, sin_t = cs_o[0, 0, :, 0::2].contiguous(), cs_o[0, 0, :, 1::2].contiguous()
    nbytes = 2 * 2 * (q.numel() + k.numel())
    res = {"config": f"FP16 B={b} S={s} Hq={hq} Hkv={hkv} D={d}, base 10000"}
    for label, fn in [
        ("poly_fwd", lambda: B.poly_rope_fwd(B.POLY_ROPE_POLY, q, k, qo, ko, delta)),
        ("mufu_fwd", lambda: B.poly_rope_fwd(B.POLY_ROPE_MUFU, q, k, qo, ko, delta)),
        ("table_fwd", lambda: B.poly_rope_fwd(B.POLY_ROPE_TABLE, q, k, qo, ko, None, cos_t, sin_t)),
        ("poly_bwd", lambda: B.poly_rope_bwd(B.POLY_ROPE_POLY, qo, ko, q, k, delta)),
    ]:
        ms = _time(fn, stream, 20)
        res[label] = {"us": ms * 1e3, "gbs": nbytes / ms / 1e6, "frac": nbytes / ms / 1e6 / peak}
    ms = same_bytes_copy_ms(nbytes, dev, stream)
    res["same_bytes_copy"] = {"us": ms * 1e3, "gbs": nbytes / ms / 1e6,
                              "frac": nbytes / ms / 1e6 / peak}
    for label in ("poly_fwd", "mufu_fwd", "table_fwd", "poly_bwd"):
        res[label]["vs_same_bytes_copy"] = ms * 1e3 / res[label]["us"]
    return res


def swiglu_extras(args, dev, stream, peak):
    import torch
    from polynomial_activation_gb300 import binding as B
    out = {}
    bf = B.POLY_BF16
    g, u, dy = workloads.dense_swiglu("bf16")
    t = lambda a: torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
    gd, ud, dyd = t(g), t(u), t(dy)
    del g, u, dy
    y, dg, du = torch.empty_like(gd), torch.empty_like(gd), torch.empty_like(gd)
    n = gd.numel()
    reps = 20
    for label, fn, nbytes in [
        ("dense_fwd", lambda: B.poly_swiglu_fwd(bf, gd, ud, y), 6),
        ("dense_fwd_ctrl", lambda: B.poly_ctrl_swiglu_fwd(bf, gd, ud, y), 6),
        ("dense_bwd", lambda: B.poly_swiglu_bwd(bf, gd, ud, dyd, dg, du), 10),
        ("dense_bwd_ctrl", lambda: B.poly_ctrl_swiglu_bwd(bf, gd, ud, dyd, dg, du), 10),
        ("dense_fwd_ctrl_packed",
         lambda: B.poly_ctrl_swiglu_fwd_v(B.POLY_CTRL_PACKED, bf, gd, ud, y), 6),
        ("dense_bwd_ctrl_packed",
         lambda: B.poly_ctrl_swiglu_bwd_v(B.POLY_CTRL_PACKED, bf, gd, ud, dyd, dg, du), 10),
        ("dense_fwd_torch", lambda: torch.nn.functional.silu(gd) * ud, 6),
        # the paper's deployed B1/B4 rule (sigmoid program recomputed), per call
        ("dense_fwd_sigmoid_rule",
         lambda: B.poly_swiglu_fwd_v(B.POLY_SWIGLU_SIGMOID, bf, gd, ud, y), 6),
        ("dense_bwd_sigmoid_rule",
         lambda: B.poly_swiglu_bwd_v(B.POLY_SWIGLU_SIGMOID, bf, gd, ud, dyd, dg, du), 10),
    ]:
        ms = _time(fn, stream, reps)
        out[label] = {"ms": ms, "gelem_s": n / ms / 1e6, "gbs": nbytes * n / ms / 1e6,
                      "frac": nbytes * n / ms / 1e6 / peak,
                      "vs_same_bytes_copy": same_bytes_copy_ms(nbytes * n, dev, stream) / ms}
    del y, dg, du
    # training step of the activation through autograd on a fused gate-up
    # buffer [8192, 2 x 14336]: forward + backward, gradient into one buffer
    from polynomial_activation_gb300 import ops
    h = gd.shape[1]
    gu = torch.cat([gd, ud], dim=1).requires_grad_(True)
    del gd, ud

    def autograd_step(f):
        def step():
            gu.grad = None
            f(gu).backward(dyd)
        return step

    for label, f in [
        ("packed_autograd_fwd_bwd", ops.swiglu_packed),
        ("chunked_autograd_fwd_bwd", lambda a: ops.swiglu(*a.chunk(2, dim=-1))),
        ("slice_gradients_autograd_fwd_bwd", lambda a: ops.PolySwiGLU.apply(a[:, :h], a[:, h:])),
        ("torch_autograd_fwd_bwd", lambda a: torch.nn.functional.silu(a[:, :h]) * a[:, h:]),
    ]:
        ms = min(_time(autograd_step(f), stream, reps, warm=6) for _ in range(3))
        out[label] = {"ms": ms, "gbs": 16 * n / ms / 1e6, "frac": 16 * n / ms / 1e6 / peak}
    del gu, dyd
    g, u, dy, seg = workloads.ragged_swiglu("bf16")
    gd, ud, dyd = t(g), t(u), t(dy)
    del g, u, dy
    segd = torch.from_numpy(seg).to(dev)
    y, dg, du = torch.empty_like(gd), torch.empty_like(gd), torch.empty_like(gd)
    n = gd.numel()
    for label, fn, nbytes in [
        ("ragged_fwd", lambda: B.poly_swiglu_fwd_ragged(bf, gd, ud, y, segd), 6),
        ("ragged_bwd", lambda: B.poly_swiglu_bwd_ragged(bf, gd, ud, dyd, dg, du, segd), 10),
    ]:
        ms = _time(fn, stream, reps)
        out[label] = {"ms": ms, "gelem_s": n / ms / 1e6, "gbs": nbytes * n / ms / 1e6,
                      "frac": nbytes * n / ms / 1e6 / peak,
                      "vs_same_bytes_copy": same_bytes_copy_ms(nbytes * n, dev, stream) / ms}
    # autograd forward + backward over the ragged rows (the offsets cover every row)
    from polynomial_activation_gb300 import ops
    gr = gd.requires_grad_(True)
    for label, pf in [("ragged_autograd_fwd_bwd", False),
                      ("ragged_autograd_fwd_bwd_padding_free", True)]:
        def step(pf=pf):
            gr.grad = None
            ops.swiglu_ragged(gr, ud, segd, padding_free=pf).backward(dyd)
        ms = min(_time(step, stream, reps, warm=6) for _ in range(3))
        out[label] = {"ms": ms, "gbs": 16 * n / ms / 1e6, "frac": 16 * n / ms / 1e6 / peak}
    out["config"] = {"dense": "BF16 [8192 x 14336], gate/up 2 N(0,1), dy N(0,1)",
                     "autograd": "forward + backward through torch.autograd on one [8192, "
                                 "28672] gate-up buffer; GB/s counts 16 bytes per element "
                                 "(fwd 6, bwd 10); best of 3 rounds of 20 steps",
                     "ragged": "BF16 131,072 x 2048 rows from 64 Zipf(1.1) segments, N(0,1.5^2)"}
    return out


def torch_native(name, d, x, dy):
    """PyTorch's own kernel for the same program: the forward activation, or
    the fused backward from the saved forward output (sigmoid_backward,
    tanh_backward) as autograd runs it."""
    import torch
    F = torch.nn.functional
    if d == 0:
        f = {"sigmoid": torch.sigmoid, "tanh": torch.tanh, "silu": F.silu, "gelu": F.gelu}[name]
        return lambda: f(x)
    ysav = torch.sigmoid(x) if name == "sigmoid" else torch.tanh(x)
    bwd = torch.ops.aten.sigmoid_backward if name == "sigmoid" else torch.ops.aten.tanh_backward
    return lambda: bwd(dy, ysav)


def _time_graph(fn, reps, replays=5):
    """Average time of fn() when `reps` calls are captured into one CUDA graph
    (removes the host launch cost, which dominates microsecond kernels)."""
    import torch
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(3):
            fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(reps):
            fn()
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(replays):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / (replays * reps)


def same_shape_stream_gbs(a, b, out, n, nin, stream, reps=10):
    """Best rate of the library's streaming probe moving the same bytes as a
    kernel with `nin` inputs and one output over n elements (reps
    back-to-back single-pass launches, for 2, 4 and 8 chunks in flight per
    thread; a, b: the kernel's inputs; out: a buffer of n elements).
    Returns (GB/s, {chunks in flight: GB/s})."""
    from polynomial_activation_gb300 import binding as B
    rates = {}
    for inflight in (2, 4, 8):
        ms = _time(lambda: B.poly_diag_stream_peak(nin, a, b if nin == 2 else None, out, n, 1,
                                                   inflight=inflight), stream, reps)
        rates[inflight] = n * 2 * (nin + 1) / ms / 1e6
    return max(rates.values()), rates


def l2_peak(dev, stream, n, passes=200, tries=3):
    """L2 streaming bandwidth of 16-byte register-staged accesses: one launch
    of the streaming probe making `passes` rotated passes over n-element
    buffers that stay in L2 (one launch's ramp and drain spread over every
    pass), with 1, 2, 4 and 8 chunks in flight per thread, for one input (4
    bytes per element and pass) and two (6 bytes); per shape the best rate
    (GB/s) and every configuration's."""
    import torch
    from polynomial_activation_gb300 import binding as B
    a = torch.randint(-30000, 30000, (n,), dtype=torch.int16, device=dev)
    b = torch.randint(-30000, 30000, (n,), dtype=torch.int16, device=dev)
    out = torch.empty_like(a)
    res = {}
    for nin in (1, 2):
        rates = {}
        for inflight in (1, 2, 4, 8):
            f = lambda: B.poly_diag_stream_peak(nin, a, b if nin == 2 else None, out, n, passes,
                                                inflight=inflight)
            f()
            torch.cuda.synchronize()
            ms = min(_time(f, stream, 1, warm=1) for _ in range(tries))
            rates[str(inflight)] = passes * n * 2 * (nin + 1) / ms / 1e6
        best = max(rates, key=rates.get)
        res[f"in{nin}"] = {"gbs": rates[best], "best_inflight": int(best), "by_inflight": rates,
                           "passes": passes}
    return res


def _fit_line(xs, ys):
    """Least-squares y = a + b x; returns (a, b)."""
    xm, ym = statistics.mean(xs), statistics.mean(ys)
    b = sum((x - xm) * (y - ym) for x, y in zip(xs, ys)) / sum((x - xm) ** 2 for x in xs)
    return ym - b * xm, b


def l2_extras(dev, stream):
    """4,194,304-element FP16 sweep, deliberately L2-resident (no flush): the
    regime where arithmetic, not HBM, can show (Table 3, first column).

    * The L2 roof (l2_roof), per shape (one input: forward; two: backward):
      the highest L2 streaming rate measured for the kernels' access
      pattern -- the streaming probe over the same buffer sizes in one long
      launch (l2_peak), or the one-pass probe's marginal rate from the size
      curve below; l2_frac = a program's algorithmic GB/s over it.
    * Per program: polynomial, FP32 control, packed control, torch and the
      probe making one pass over the same bytes (same_size_copy) under the
      paper's alternating protocol, every arm a CUDA graph of 200 launches
      (a 2-6 us kernel is otherwise bounded by the host's launch rate).
    * The size curve: time per launch of sigmoid D3 forward, the one-pass
      probe and a torch copy from 8 to 16,777,216 elements; a least-squares
      line over the L2-resident sizes 2^20..2^24 gives the fixed cost of a
      launch (intercept, us) and the streaming rate (bytes over slope)."""
    import torch
    from polynomial_activation_gb300 import binding as B
    xh, dyh = workloads.isolated_l2("f16")
    x = torch.from_numpy(xh.view(np.int16)).to(dev).view(torch.float16)
    dy = torch.from_numpy(dyh.view(np.int16)).to(dev).view(torch.float16)
    y = torch.empty_like(x)
    n = x.numel()
    res = {"l2_peak": {"n4194304": l2_peak(dev, stream, n),
                       "n8388608": l2_peak(dev, stream, 2 * n)}}
    peak = res["l2_peak"]["n4194304"]
    f16 = B.POLY_F16
    for name, d, D in SIX:
        key = f"{name}.{'bwd' if d else 'fwd'}.D{D}"
        fn = FN[name]
        if d == 0:
            arms = {"poly": lambda: B.poly_act_fwd(fn, f16, x, y, n),
                    "ctrl_fp32": lambda: B.poly_ctrl_act_fwd_v(0, fn, f16, x, y, n),
                    "ctrl_packed": lambda: B.poly_ctrl_act_fwd_v(1, fn, f16, x, y, n)}
        else:
            arms = {"poly": lambda: B.poly_act_bwd(fn, f16, x, dy, y, n),
                    "ctrl_fp32": lambda: B.poly_ctrl_act_bwd_v(0, fn, f16, x, dy, y, n),
                    "ctrl_packed": lambda: B.poly_ctrl_act_bwd_v(1, fn, f16, x, dy, y, n)}
        arms["torch"] = torch_native(name, d, x, dy)
        nin = 2 if d else 1
        arms["same_size_copy"] = lambda nin=nin: B.poly_diag_stream_peak(
            nin, x, dy if nin == 2 else None, y, n, 1)
        t = alternating(arms, stream, rounds=9, reps=200, warm=20, graph=True)
        tp = t["poly"]["ms"]
        best = min(("ctrl_fp32", "ctrl_packed"), key=lambda k: t[k]["ms"])
        gbs = BYTES[d] * n / tp / 1e6
        res[key] = {"poly_us": tp * 1e3, "ctrl_us": t[best]["ms"] * 1e3, "best_ctrl": best,
                    "ctrl_fp32_us": t["ctrl_fp32"]["ms"] * 1e3,
                    "ctrl_packed_us": t["ctrl_packed"]["ms"] * 1e3,
                    "torch_native_us": t["torch"]["ms"] * 1e3,
                    "same_size_copy_us": t["same_size_copy"]["ms"] * 1e3,
                    "speedup_vs_ctrl": t[best]["ms"] / tp,
                    "speedup_vs_ctrl_fp32": t["ctrl_fp32"]["ms"] / tp,
                    "speedup_vs_ctrl_packed": t["ctrl_packed"]["ms"] / tp,
                    "speedup_vs_torch": t["torch"]["ms"] / tp,
                    "vs_same_size_copy": t["same_size_copy"]["ms"] / tp,
                    "poly_gbs": gbs, "l2_peak_gbs": peak[f"in{nin}"]["gbs"],
                    "l2_frac": gbs / peak[f"in{nin}"]["gbs"],
                    "rounds": {k: {"median_us": v["ms"] * 1e3, "min_us": v["min_ms"] * 1e3,
                                   "max_us": v["max_ms"] * 1e3} for k, v in t.items()}}
    # the backward rows Table 3 lost (SiLU', GELU' D4; the paper's L2 maximum,
    # 2.193x against PyTorch, belongs to one of them)
    lost = {}
    for name in ("silu", "gelu"):
        fn = FN[name]
        t = alternating({
            "poly": lambda fn=fn: B.poly_act_bwd(fn, f16, x, dy, y, n),
            "ctrl_fp32": lambda fn=fn: B.poly_ctrl_act_bwd_v(0, fn, f16, x, dy, y, n),
            "ctrl_packed": lambda fn=fn: B.poly_ctrl_act_bwd_v(1, fn, f16, x, dy, y, n),
            "torch": (lambda: torch.ops.aten.silu_backward(dy, x)) if name == "silu"
                     else (lambda: torch.ops.aten.gelu_backward(dy, x))},
            stream, rounds=9, reps=200, warm=20, graph=True)
        tp = t["poly"]["ms"]
        best = min(("ctrl_fp32", "ctrl_packed"), key=lambda k: t[k]["ms"])
        lost[f"{name}.bwd.D4"] = {
            "poly_us": tp * 1e3, "ctrl_fp32_us": t["ctrl_fp32"]["ms"] * 1e3,
            "ctrl_packed_us": t["ctrl_packed"]["ms"] * 1e3,
            "torch_native_us": t["torch"]["ms"] * 1e3, "best_ctrl": best,
            "speedup_vs_ctrl": t[best]["ms"] / tp, "speedup_vs_torch": t["torch"]["ms"] / tp,
            "poly_gbs": 6 * n / tp / 1e6}
    res["lost_rows"] = lost
    res["config"] = ("4,194,304 FP16 elements, x ~ N(0, 3^2), dy ~ N(0, 1); L2-resident by "
                     "design; 9 alternating rounds per program, each arm one replay of a CUDA "
                     "graph of 200 launches; median of per-round means; l2_frac against "
                     "l2_roof")
    # launch time against size: intercept = fixed cost of a launch, slope = L2 streaming rate
    big = torch.empty(1 << 24, dtype=torch.float16, device=dev)
    big[:n].copy_(x)
    big[n:].copy_(x.repeat(3))
    out = torch.empty_like(big)
    curve = {}
    sizes = (8, 1 << 18, 1 << 20, 1 << 21, 1 << 22, 1 << 23, 1 << 24)
    arms_of = lambda m: {
        "poly": lambda: B.poly_act_fwd(FN["sigmoid"], f16, big, out, m),
        "ctrl_packed": lambda: B.poly_ctrl_act_fwd_v(1, FN["sigmoid"], f16, big, out, m),
        "ctrl_fp32": lambda: B.poly_ctrl_act_fwd_v(0, FN["sigmoid"], f16, big, out, m),
        "copy": lambda: B.poly_diag_stream_peak(1, big, None, out, -(-m // 8) * 8, 1),
        "torch_copy": lambda: out[:m].copy_(big[:m])}
    for m in sizes:
        t = alternating(arms_of(m), stream, rounds=3, reps=200, warm=5, graph=True)
        curve[str(m)] = {f"{k}_us": v["ms"] * 1e3 for k, v in t.items()}
        curve[str(m)]["poly_gbs"] = 4 * m / t["poly"]["ms"] / 1e6
    fit = {}
    xs = [m for m in sizes if m >= (1 << 20)]
    for arm in ("poly", "ctrl_packed", "ctrl_fp32", "copy", "torch_copy"):
        a, b = _fit_line(xs, [curve[str(m)][f"{arm}_us"] for m in xs])
        fit[arm] = {"intercept_us": a, "rate_gbs": 4 / (b * 1e-6) / 1e9 if b > 0 else None}
    res["size_curve_sigmoid_fwd"] = curve
    res["size_curve_fit"] = fit
    # the same for the backward shape (two inputs, one output: 6 bytes per element)
    dbig = torch.empty_like(big)
    dbig.copy_(big.flip(0))
    curve_b = {}
    for m in sizes:
        t = alternating({
            "poly": lambda m=m: B.poly_act_bwd(FN["sigmoid"], f16, big, dbig, out, m),
            "ctrl_packed": lambda m=m: B.poly_ctrl_act_bwd_v(1, FN["sigmoid"], f16, big, dbig, out, m),
            "copy": lambda m=m: B.poly_diag_stream_peak(2, big, dbig, out, -(-m // 8) * 8, 1)},
            stream, rounds=3, reps=200, warm=5, graph=True)
        curve_b[str(m)] = {f"{k}_us": v["ms"] * 1e3 for k, v in t.items()}
        curve_b[str(m)]["poly_gbs"] = 6 * m / t["poly"]["ms"] / 1e6
    fit_b = {}
    for arm in ("poly", "ctrl_packed", "copy"):
        a, b = _fit_line(xs, [curve_b[str(m)][f"{arm}_us"] for m in xs])
        fit_b[arm] = {"intercept_us": a, "rate_gbs": 6 / (b * 1e-6) / 1e9 if b > 0 else None}
    res["size_curve_sigmoid_bwd"] = curve_b
    res["size_curve_fit_bwd"] = fit_b
    # the L2 roof per shape: the highest L2 streaming rate measured for the
    # kernels' access pattern -- the long probe launch, or (one input) the
    # one-pass probe's marginal rate over 1-16 M elements, whichever is higher
    # (the backward size curve leaves L2 at its largest size, so its slope is
    # not an L2 rate)
    roof = {"in1": max(peak["in1"]["gbs"], fit["copy"]["rate_gbs"] or 0.0),
            "in2": peak["in2"]["gbs"]}
    res["l2_roof"] = {
        "fwd_gbs": roof["in1"], "bwd_gbs": roof["in2"],
        "fwd_source": "size-curve slope of the one-pass probe"
                      if roof["in1"] > peak["in1"]["gbs"] else "long probe launch",
        "bwd_source": "long probe launch",
        "note": "l2_frac = a program's algorithmic GB/s over this roof; ncu's hardware "
                "figure (lts__t_bytes.sum.peak_sustained x L2 clock) is 36 TB/s of L2 "
                "request bytes, of which the long probe reaches 48 %"}
    for name, d, D in SIX:
        e = res[f"{name}.{'bwd' if d else 'fwd'}.D{D}"]
        e["l2_peak_gbs"] = roof["in2" if d else "in1"]
        e["l2_frac"] = e["poly_gbs"] / e["l2_peak_gbs"]
    for e in res["lost_rows"].values():
        e["l2_frac"] = e["poly_gbs"] / roof["in2"]
    res["size_curve_note"] = ("least squares over 2^20..2^24 elements (4 bytes per element): "
                              "intercept = fixed cost of one launch in a graph, rate = marginal "
                              "L2 streaming rate; the arms are sigmoid D3 forward, its two MUFU "
                              "controls, the library's one-pass probe (copy) and torch copy_")
    return res


def host_cost_extras(dev, reps=5000):
    """Host time per eager call (microseconds) for a decode-sized tensor, the
    library's calls beside torch's own: the binding with a preallocated
    output, the allocating wrappers without and with an autograd node, and
    the fused SwiGLU against torch's two kernels.  The loop is host-bound
    (the kernels take ~2 us), so wall time per call is the host cost."""
    import torch
    from polynomial_activation_gb300 import binding as B, ops
    F = torch.nn.functional
    x = torch.randn(14336, device=dev).half()
    dy, y = torch.randn_like(x), torch.empty_like(x)
    xr = x.clone().requires_grad_(True)
    g = torch.randn(8, 1792, device=dev).bfloat16()
    u = torch.randn_like(g)
    cases = {
        "binding_act_fwd_preallocated": lambda: B.poly_act_fwd(B.POLY_SIGMOID, B.POLY_F16, x, y),
        "torch_sigmoid_out": lambda: torch.sigmoid(x, out=y),
        "binding_act_bwd_preallocated": lambda: B.poly_act_bwd(B.POLY_SIGMOID, B.POLY_F16, x, dy, y),
        "torch_sigmoid_backward": lambda: torch.ops.aten.sigmoid_backward(dy, x),
        "ops_sigmoid": lambda: ops.sigmoid(x),
        "torch_sigmoid": lambda: torch.sigmoid(x),
        "ops_sigmoid_recorded": lambda: ops.sigmoid(xr),
        "torch_sigmoid_recorded": lambda: torch.sigmoid(xr),
        "ops_swiglu_8x1792": lambda: ops.swiglu(g, u),
        "torch_silu_mul_8x1792": lambda: F.silu(g) * u,
    }
    res = {}
    for k, f in cases.items():
        for _ in range(200):
            f()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(reps):
            f()
        t1 = time.perf_counter()
        torch.cuda.synchronize()
        res[k] = (t1 - t0) / reps * 1e6
    res["config"] = (f"FP16 x of 14,336 elements (BF16 8 x 1,792 for SwiGLU), mean host time "
                     f"per call over {reps} eager calls, microseconds")
    return res


def e2e(args, dev, stream, xh, dyh, chunks=8):
    """Same step through the public API with host buffers.  Per step: the
    inputs are copied from pinned host memory in `chunks` pieces on a copy
    stream, and the six kernels of each piece (waiting only for that piece)
    write their outputs straight into pinned host memory over NVLink-C2C --
    the library takes any address the GPU can reach, so no device staging
    buffer and no separate device-to-host copy is needed."""
    import torch
    from polynomial_activation_gb300 import binding as B
    n = xh.size
    xp = torch.from_numpy(xh.view(np.int16)).pin_memory()
    dyp = torch.from_numpy(dyh.view(np.int16)).pin_memory()
    outs_h = [torch.empty(n, dtype=torch.int16).pin_memory().view(torch.float16) for _ in SIX]
    x = torch.empty(n, dtype=torch.int16, device=dev)
    dy = torch.empty(n, dtype=torch.int16, device=dev)
    xf, dyf = x.view(torch.float16), dy.view(torch.float16)
    copy_stream = torch.cuda.Stream(device=dev)
    step_len = -(-n // chunks)
    step_len = -(-step_len // 8) * 8                       # keep pieces 16-byte aligned
    bounds = [(lo, min(n, lo + step_len)) for lo in range(0, n, step_len)]
    ready = [torch.cuda.Event() for _ in bounds]

    def step():
        copy_stream.wait_stream(stream)                     # previous step done with x, dy
        for c, (lo, hi) in enumerate(bounds):
            with torch.cuda.stream(copy_stream):
                x[lo:hi].copy_(xp[lo:hi], non_blocking=True)
                dy[lo:hi].copy_(dyp[lo:hi], non_blocking=True)
                ready[c].record(copy_stream)
            stream.wait_event(ready[c])
            for i, (name, d, D) in enumerate(SIX):
                if d == 0:
                    B.poly_act_fwd(FN[name], B.POLY_F16, xf[lo:hi], outs_h[i][lo:hi], hi - lo,
                                   stream=stream)
                else:
                    B.poly_act_bwd(FN[name], B.POLY_F16, xf[lo:hi], dyf[lo:hi], outs_h[i][lo:hi],
                                   hi - lo, stream=stream)

    per_round = max(3, min(5, args.steps // 80))
    # five equal rounds (the first after 4 untimed passes, which touch the
    # pinned pages); the value is the median of the per-round means (the
    # statistic of the paper's timing protocol, §4.2), every round and their
    # mean are kept: the host link is shared with the machine's other GPUs and
    # a slow stretch shows as one slow round
    rounds = [_time(step, stream, per_round, 4 if r == 0 else 1) for r in range(5)]
    ms = statistics.median(rounds)
    link = link_bound(x, xp, dyf, outs_h[0], stream, copy_stream, h2d=2 * 2 * n, d2h=6 * 2 * n)
    link["frac"] = link["bound_ms"] / ms
    return {"value": 6 * n / ms / 1e6, "unit": UNIT, "h2d_bytes_per_step": 2 * 2 * n,
            "d2h_bytes_per_step": 6 * 2 * n, "ms_per_step": ms, "round_ms": rounds,
            "mean_ms": statistics.mean(rounds), "statistic": "median of 5 rounds",
            "link": link,
            "method": f"pinned host inputs copied in {len(bounds)} pieces on a second stream; "
                      "kernels write outputs directly to pinned host memory (NVLink-C2C)"}


def link_bound(xd, xp, src, out_h, stream, copy_stream, h2d, d2h):
    """The host link's rates, measured on the step's own buffers: host->device
    copies alone, kernel stores into pinned host memory alone, and both at
    once (equal bytes).  A step moving h2d bytes in and d2h >= h2d bytes out
    cannot beat h2d / r_both + (d2h - h2d) / r_store, where r_both is the
    per-direction rate while both directions are busy.  The copy fills xd
    from xp; the kernel reads src (another device buffer) into out_h."""
    import torch
    from polynomial_activation_gb300 import binding as B
    m = xd.numel()
    nb = 2 * m

    def copy_in():
        with torch.cuda.stream(copy_stream):
            xd.copy_(xp, non_blocking=True)
        stream.wait_stream(copy_stream)

    def store_out():
        B.poly_act_fwd(FN["sigmoid"], B.POLY_F16, src, out_h, m, stream=stream)

    def both():
        copy_stream.wait_stream(stream)
        with torch.cuda.stream(copy_stream):
            xd.copy_(xp, non_blocking=True)
        B.poly_act_fwd(FN["sigmoid"], B.POLY_F16, src, out_h, m, stream=stream)
        stream.wait_stream(copy_stream)

    r_in = nb / _time(copy_in, stream, 3) / 1e6
    r_out = nb / _time(store_out, stream, 3) / 1e6
    r_both = nb / _time(both, stream, 3) / 1e6          # per direction
    bound = (h2d / r_both + max(0, d2h - h2d) / r_out) / 1e6
    return {"h2d_copy_gbs": r_in, "kernel_store_to_host_gbs": r_out,
            "per_direction_when_both_gbs": r_both, "bound_ms": bound}


if __name__ == "__main__":
    sys.exit(main())

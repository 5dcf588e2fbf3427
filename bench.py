"""Benchmark of the packed-polynomial activation kernels on GB300.

Workload (one step): the HBM-resident isolated sweep of "Fast Polynomial
Transcendentals for LLMs" (§4.2, Table 3) -- 268,435,456-element FP16
tensors (512 MiB each), x ~ N(0, 3^2) with 1 % uniform in [-40, 40],
dy ~ N(0, 1) -- through the six programs: sigmoid D3, tanh D4, SiLU D3,
GELU D5 forward and the direct sigma' D4, tanh' D4 backward.  The inputs are
four times larger than L2, so no L2 flush is needed between steps.

Reported (one JSON line, rank 0): whole-job Gelem/s of the step (all ranks),
the roofline of the dominant kernel against the measured HBM bandwidth, the
same six programs through the MUFU-native control kernels, torch's native
ops, the SwiGLU kernels (dense [8192 x 14336] and ragged 131,072 x 2048 BF16)
and the L2-resident 4,194,304-element sweep as extras, an end-to-end figure
through the public API with host buffers, SM clocks sampled during the timed
region, and the CPU replay oracle's throughput on a bounded sample, run on
every host core (one spawned worker process per core).

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


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples every 200 ms.  start()
    returns once the first sample has arrived, so the sampler is running when
    the timed region begins; stop() keeps only the samples that arrived after
    start() returned."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap,clocks.mem")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []
        self.first = threading.Event()
        self.reader = None
        self.skip = 0

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line)
            self.first.set()
        self.first.set()

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.reader = threading.Thread(target=self._read, daemon=True)
        self.reader.start()
        self.first.wait(timeout=10)
        self.skip = len(self.lines)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        self.proc.terminate()
        self.proc.wait(timeout=10)
        self.reader.join(timeout=10)
        sm, smax, mem, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines[self.skip:]:
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
                "samples": len(sm), "reasons": sorted(reasons)}


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

def oracle_programs():
    """The oracle fitter's programs for the six (written to
    tests/golden/programs.json by a script that calls only the oracle)."""
    from oracle.replay import Program
    with open(os.path.join(ROOT, "tests", "golden", "programs.json")) as f:
        g = json.load(f)
    out = []
    for name, d, D in SIX:
        v = g[f"{name}.{'bwd' if d else 'fwd'}.f16.D{D}"]
        out.append(Program(fn=v["fn"], direction=v["direction"], fmt="f16", degree=D,
                           li=v["li"], lc=v["lc"], coef=tuple(v["coef"]), lc_bits=v["lc_bits"]))
    return out


_PROGS = None


def _replay_six(x, dy):
    """The oracle's six programs over one piece of the sample (in pieces of
    2^22 elements, which bounds the replay's FP64 temporaries); returns the
    seconds it took."""
    global _PROGS
    from oracle.replay import backward, forward
    if _PROGS is None:
        _PROGS = oracle_programs()
    piece = 1 << 22
    t0 = time.perf_counter()
    for lo in range(0, x.size, piece):
        xs, dys = x[lo:lo + piece], dy[lo:lo + piece]
        for p, (name, d, D) in zip(_PROGS, SIX):
            if d == 0:
                forward(p, xs)
            else:
                backward(p, xs, dys)
    return time.perf_counter() - t0


def _warm_worker(_):
    time.sleep(0.2)                     # one task per worker: every worker imports the oracle
    _replay_six(np.zeros(8, np.uint16), np.zeros(8, np.uint16))
    return os.getpid()


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


class OraclePool:
    """The CPU replay oracle, unchanged, on every host core: a sample is cut
    into one contiguous piece per worker process.  Workers are spawned (no
    CUDA state is inherited) and import the oracle before any timing."""

    def __init__(self, workers):
        self.workers = max(1, int(workers))
        self.pool = None
        if self.workers > 1:
            import multiprocessing as mp
            self.pool = mp.get_context("spawn").Pool(self.workers)
            self.pool.map(_warm_worker, range(self.workers), chunksize=1)

    def run(self, x, dy):
        """(wall seconds, [seconds per piece], [elements per piece])."""
        if self.pool is None:
            t = _replay_six(x, dy)
            return t, [t], [x.size]
        b = np.linspace(0, x.size, self.workers + 1).astype(np.int64)
        args = [(x[b[i]:b[i + 1]], dy[b[i]:b[i + 1]]) for i in range(self.workers)]
        t0 = time.perf_counter()
        per = self.pool.starmap(_replay_six, args, chunksize=1)
        return time.perf_counter() - t0, per, [int(b[i + 1] - b[i]) for i in range(self.workers)]

    def close(self):
        if self.pool is not None:
            self.pool.close()
            self.pool.join()


def oracle_sample_time(n_sample, workers=1):
    """Time the CPU replay oracle on the first n_sample elements of the
    workload through each of the six programs, on `workers` processes.
    Returns (wall seconds, elements x programs, CPU seconds, per-core
    Gelem/s)."""
    x, dy = workloads.isolated_hbm("f16", n=n_sample)
    pool = OraclePool(workers)
    try:
        wall, per, sizes = pool.run(x, dy)
    finally:
        pool.close()
    per_core = statistics.mean(6 * m / t / 1e9 for m, t in zip(sizes, per) if t > 0)
    return wall, 6 * n_sample, sum(per), per_core


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
            pool.run(x, dy)
        t0 = time.perf_counter()
        for _ in range(args.steps):
            pool.run(x, dy)
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

    def launch(i, ctrl=False):
        name, d, D = SIX[i]
        if d == 0:
            (B.poly_ctrl_act_fwd if ctrl else B.poly_act_fwd)(FN[name], B.POLY_F16, x, outs[i], n)
        else:
            (B.poly_ctrl_act_bwd if ctrl else B.poly_act_bwd)(FN[name], B.POLY_F16, x, dy, outs[i], n)

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
    total_ms, _ = timed_steps(False, args.steps, per_kernel=False)
    # per-kernel durations for the roofline: a second timed pass with an event
    # pair around every launch; the clock samples cover both passes
    _, per_ms = timed_steps(False, max(50, args.steps // 4))
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

    # ---- per program: poly vs MUFU control vs torch native
    for _ in range(args.warmup):
        for i in range(len(SIX)):
            launch(i, ctrl=True)
    ctrl_total, ctrl_ms = timed_steps(True, max(20, args.steps // 4))
    programs = {}
    for i, (name, d, D) in enumerate(SIX):
        key = f"{name}.{'bwd' if d else 'fwd'}.D{D}"
        gb = BYTES[d] * n / 1e9
        entry = {"poly_ms": per_ms[i], "poly_gelem_s": n / per_ms[i] / 1e6,
                 "poly_gbs": gb / per_ms[i] * 1e3, "poly_frac": gb / per_ms[i] * 1e3 / peak,
                 "ctrl_ms": ctrl_ms[i], "ctrl_gbs": gb / ctrl_ms[i] * 1e3,
                 "speedup_vs_ctrl": ctrl_ms[i] / per_ms[i]}
        if not args.no_extras:
            fnat = torch_native(name, d, x, dy)
            for _ in range(3):
                fnat()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            reps = 10
            torch.cuda.synchronize()
            e0.record(stream)
            for _ in range(reps):
                fnat()
            e1.record(stream)
            torch.cuda.synchronize()
            entry["torch_native_ms"] = e0.elapsed_time(e1) / reps
            entry["speedup_vs_torch"] = entry["torch_native_ms"] / per_ms[i]
        programs[key] = entry
    result["programs"] = programs

    # ---- roofline of the dominant kernel
    dom = max(range(len(SIX)), key=lambda i: per_ms[i])
    name, d, D = SIX[dom]
    kkey = f"{name}.{'bwd' if d else 'fwd'}.D{D}"
    ach = BYTES[d] * n / (per_ms[dom] * 1e-3) / 1e9
    result["roofline"] = {"kernel": f"dense_kernel<OpBwd|OpFwd> {kkey}", "bound": "hbm",
                          "achieved": ach, "peak": peak, "unit": "GB/s", "frac": ach / peak,
                          "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured" else "fallback",
                          "algorithmic_bytes_per_launch": BYTES[d] * n,
                          "traffic": recorded_traffic(kkey) if n == workloads.N_HBM else None,
                          "share_of_step": per_ms[dom] / sum(per_ms)}

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

    # ---- CPU oracle on a bounded sample
    if rank == 0 and args.cpu_sample > 0:
        cores = host_cores()
        wall, elems, cpu_s, per_core = oracle_sample_time(args.cpu_sample, cores)
        result["cpu_baseline"] = {"value": elems / wall / 1e9, "unit": UNIT, "cores": cores,
                                  "kind": "oracle", "per_core_value": per_core,
                                  "sample": f"first {args.cpu_sample} elements of the workload "
                                            f"through each of the six programs, one contiguous "
                                            f"piece per core (numpy replay, {wall:.1f} s wall, "
                                            f"{cpu_s:.1f} s of CPU work)"}
    if rank == 0:
        if args.elements != workloads.N_HBM:
            result["config"]["workload"] = f"profiling case: {args.elements} elements"
        print(json.dumps(result), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


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
        else:
            fp = lambda: B.poly_act_bwd(FN[name], bf, xb, dyb, y, n)
            fc = lambda: B.poly_ctrl_act_bwd(FN[name], bf, xb, dyb, y, n)
        tp, tc = _time(fp, stream, reps), _time(fc, stream, reps)
        gb = BYTES[d] * n / 1e9
        res[f"{name}.{'bwd' if d else 'fwd'}.D{prog.degree}"] = {
            "poly_ms": tp, "poly_gbs": gb / tp * 1e3, "poly_frac": gb / tp * 1e3 / peak,
            "ctrl_ms": tc, "speedup_vs_ctrl": tc / tp}
    res["config"] = ("268,435,456 BF16 elements: the step's FP16 x and dy converted on the device; "
                     f"mean of {reps} launches each")
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
        out["speedup_vs_ctrl"] = out["ctrl_us"] / out["poly_us"]
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
        "torch": lambda: F.silu(x)}, 4 * n)
    res["silu_probe_bwd"] = run({
        "poly": lambda: B.poly_act_bwd(silu, bf, x, dy, y, n),
        "ctrl": lambda: B.poly_ctrl_act_bwd(silu, bf, x, dy, y, n),
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
        "torch": lambda: F.silu(g) * u}, 6 * m)
    res["expert_swiglu_bwd"] = run({
        "poly": lambda: B.poly_swiglu_bwd(bf, g, u, dy, dg, du),
        "ctrl": lambda: B.poly_ctrl_swiglu_bwd(bf, g, u, dy, dg, du),
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
        ("dense_fwd_torch", lambda: torch.nn.functional.silu(gd) * ud, 6),
    ]:
        ms = _time(fn, stream, reps)
        out[label] = {"ms": ms, "gelem_s": n / ms / 1e6, "gbs": nbytes * n / ms / 1e6,
                      "frac": nbytes * n / ms / 1e6 / peak,
                      "vs_same_bytes_copy": same_bytes_copy_ms(nbytes * n, dev, stream) / ms}
    # the paper's deployed B1/B4 rule: sigmoid program recomputed
    B.poly_set_swiglu_variant(B.POLY_SWIGLU_SIGMOID)
    try:
        for label, fn, nbytes in [
            ("dense_fwd_sigmoid_rule", lambda: B.poly_swiglu_fwd(bf, gd, ud, y), 6),
            ("dense_bwd_sigmoid_rule", lambda: B.poly_swiglu_bwd(bf, gd, ud, dyd, dg, du), 10),
        ]:
            ms = _time(fn, stream, reps)
            out[label] = {"ms": ms, "gelem_s": n / ms / 1e6, "gbs": nbytes * n / ms / 1e6,
                          "frac": nbytes * n / ms / 1e6 / peak,
                          "vs_same_bytes_copy": same_bytes_copy_ms(nbytes * n, dev, stream) / ms}
    finally:
        B.poly_set_swiglu_variant(B.POLY_SWIGLU_DIRECT)
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


def l2_extras(dev, stream):
    """4,194,304-element FP16 sweep, deliberately L2-resident (no flush): the
    regime where arithmetic, not HBM, can show (Table 3, first column).
    Launches are replayed from a CUDA graph: a 4-6 us kernel is otherwise
    bounded by the host's launch rate."""
    import torch
    from polynomial_activation_gb300 import binding as B
    xh, dyh = workloads.isolated_l2("f16")
    x = torch.from_numpy(xh.view(np.int16)).to(dev).view(torch.float16)
    dy = torch.from_numpy(dyh.view(np.int16)).to(dev).view(torch.float16)
    y = torch.empty_like(x)
    n = x.numel()
    res = {}
    for name, d, D in SIX:
        key = f"{name}.{'bwd' if d else 'fwd'}.D{D}"
        if d == 0:
            fp = lambda: B.poly_act_fwd(FN[name], B.POLY_F16, x, y, n)
            fc = lambda: B.poly_ctrl_act_fwd(FN[name], B.POLY_F16, x, y, n)
        else:
            fp = lambda: B.poly_act_bwd(FN[name], B.POLY_F16, x, dy, y, n)
            fc = lambda: B.poly_ctrl_act_bwd(FN[name], B.POLY_F16, x, dy, y, n)
        tp, tc = _time_graph(fp, 200), _time_graph(fc, 200)
        tt = _time_graph(torch_native(name, d, x, dy), 200)
        res[key] = {"poly_us": tp * 1e3, "ctrl_us": tc * 1e3, "torch_native_us": tt * 1e3,
                    "speedup_vs_ctrl": tc / tp, "speedup_vs_torch": tt / tp,
                    "poly_gbs": BYTES[d] * n / tp / 1e6}
    res["config"] = ("4,194,304 FP16 elements, x ~ N(0, 3^2), dy ~ N(0, 1); L2-resident by "
                     "design; every call replayed from a CUDA graph of 200 launches")
    # launch time against size (sigmoid D3 forward and a plain copy, graph-replayed): the
    # intercept is the fixed cost of a launch, the slope the L2 streaming rate
    big = torch.empty(1 << 24, dtype=torch.float16, device=dev)
    big[:n].copy_(x)
    big[n:].copy_(x.repeat(3))
    out = torch.empty_like(big)
    curve = {}
    for m in (8, 1 << 18, 1 << 20, 1 << 22, 1 << 23, 1 << 24):
        tp = _time_graph(lambda: B.poly_act_fwd(FN["sigmoid"], B.POLY_F16, big, out, m), 200)
        tc = _time_graph(lambda: out[:m].copy_(big[:m]), 200)
        curve[str(m)] = {"poly_us": tp * 1e3, "copy_us": tc * 1e3, "poly_gbs": 4 * m / tp / 1e6}
    res["size_curve_sigmoid_fwd"] = curve
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
    # four equal rounds (the first after 4 untimed passes, which touch the
    # pinned pages); the value is their mean, the rounds show the host link's
    # variation from moment to moment
    rounds = [_time(step, stream, per_round, 4 if r == 0 else 1) for r in range(4)]
    ms = statistics.mean(rounds)
    link = link_bound(x, xp, dyf, outs_h[0], stream, copy_stream, h2d=2 * 2 * n, d2h=6 * 2 * n)
    link["frac"] = link["bound_ms"] / ms
    return {"value": 6 * n / ms / 1e6, "unit": UNIT, "h2d_bytes_per_step": 2 * 2 * n,
            "d2h_bytes_per_step": 6 * 2 * n, "ms_per_step": ms, "round_ms": rounds,
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

"""Benchmark of the per-unit FSDP cycle on GB300.

One step = one fsdp_step (gather, gather again under reshard-after-forward,
reduce-scatter, AdamW) on every unit of the workload, N virtual ranks per
unit.  Default workload: two minGPT-175B transformer blocks (d=12288,
ffn=49152; 1,812,099,072 parameters per block, one FlatParameter each), N=8
virtual ranks, bf16 per-rank gradients reduced in fp32, fp32 master weights
and Adam state.  Inputs are synthetic (seeded) and far larger than L2, so no
L2 flush is needed between steps.

Metric: counted HBM bytes per step / step time (GB/s).  Counted bytes per
unit step, every required read and write once:
    gather      R x (4P read fp32 master + 2P write bf16)          R = 2
    reduce-sc.  N*g_b*P read (N gradients) + 4P write (fp32 shards)
    AdamW       16P read (p, g, m, v) + 12P write (p, m, v)
                (+ 2P for the bf16 shadow when the unit gathers from it)

The line also carries the same step counted with every operation separate
((44 + N*g_b)P per unit, "value_survey"; the same count as above unless the
fused kernel runs), the oracle's throughput on the host cores (all cores and
one), and a "configs" object with every other workload's model step timed the
same way.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                       [--workload NAME] [--e2e-steps E] [--no-e2e] [--no-cpu-baseline]
                       [--no-configs]
With --gpus N > 1 (under torchrun) every rank runs an independent replica of
the workload on its own GPU (the N virtual ranks of a unit never span GPUs);
value = all ranks' counted bytes / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import shutil
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from fully_sharded_unit_gb300 import workloads  # noqa: E402

METRIC = "FSDP unit-step HBM GB/s (gather+reduce-scatter+AdamW) and % of GB300 HBM peak"
FALLBACK_HBM_GBS = 6800.0


# --------------------------------------------------------------------------- helpers

def counted_bytes(wl: workloads.Workload, unit: int) -> dict:
    """Algorithmic bytes of one unit step and of each kernel launch."""
    P, W = wl.unit_numel(unit), wl.world
    gb = 4 if wl.grad_dtype == "f32" else 2
    R = 2 if wl.reshard_after_forward else 1
    shadow = wl.gather_source == "shadow"   # AdamW stores the bf16 shadow only when it is gathered from
    gather = (2 if shadow else 4) * P + 2 * P
    rs = (W * gb + 4) * P
    adamw = (30 if shadow else 28) * P
    # fused: the gradient shard is written (4P) but not read back
    reduce_adamw = (W * gb + 4 + 12 + 12 + (2 if shadow else 0)) * P
    step = R * gather + (reduce_adamw if wl.fuse_reduce_adamw else rs + adamw)
    return dict(gather=gather, reduce_scatter=rs, adamw=adamw, reduce_adamw=reduce_adamw, step=step,
                gathers=R, h2d=W * gb * P, d2h=2 * P)


def survey_bytes(wl: workloads.Workload, unit: int) -> int:
    """The unit step counted with every operation separate:
    R gathers of 6P (4P when gathering the shadow), the reduce-scatter's
    (W*g_b + 4)P and AdamW's 28P (30P with the shadow gather, whose shadow
    write is then an input of the next gathers): (44 + W*g_b)P, or
    (42 + W*g_b)P from the shadow.  It differs from counted_bytes only for
    the fused kernel, which does not read the gradient shard back."""
    P, W = wl.unit_numel(unit), wl.world
    gb = 4 if wl.grad_dtype == "f32" else 2
    R = 2 if wl.reshard_after_forward else 1
    if wl.gather_source == "shadow":
        return (R * 4 + W * gb + 4 + 30) * P
    return (R * 6 + W * gb + 4 + 28) * P


L2_BYTES = 129e6   # GB300 L2 cache


def l2_statement(wl: workloads.Workload) -> str:
    """How the timed steps stand to the L2 cache (no flush is done).  A unit
    touches 20 bytes per element (fp32 master, gradient shard, m, v; bf16
    shadow and gathered output) plus its W gradients."""
    per_unit = [20 * wl.unit_numel(i) + wl.world * (4 if wl.grad_dtype == "f32" else 2) * wl.unit_numel(i)
                for i in range(wl.n_units)]
    smallest_kernel = min(min(counted_bytes(wl, i)["gather"], counted_bytes(wl, i)["reduce_scatter"])
                          for i in range(wl.n_units))
    if smallest_kernel > L2_BYTES:
        return "inputs larger than L2; no flush"
    if sum(per_unit) > L2_BYTES:
        return (f"no flush: the step touches {sum(per_unit) / 1e9:.2f} GB over {wl.n_units} units, more than "
                f"L2, so each unit step starts cold; one unit's buffers ({max(per_unit) / 1e6:.0f} MB) can "
                "partly stay in L2 between its own kernels")
    return f"no flush: the whole state ({sum(per_unit) / 1e6:.1f} MB) fits in L2 (L2-resident)"


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_sha() -> str:
    """sha256[:16] of csrc/kernels.cu with comments and whitespace removed, so
    that an edit of the comments alone keeps a capture valid."""
    with open(os.path.join(ROOT, "fully_sharded_unit_gb300", "csrc", "kernels.cu")) as f:
        code = f.read()
    code = re.sub(r"/\*.*?\*/", "", code, flags=re.S)
    code = re.sub(r"//[^\n]*", "", code)
    code = re.sub(r"\s+", " ", code).strip()
    return hashlib.sha256(code.encode()).hexdigest()[:16]


def traffic_key(wl: workloads.Workload, micro_batches: int = 1) -> str:
    """The workload name plus every option that changes a kernel's bytes per
    launch (a capture applies only to the configuration it was taken on)."""
    key = wl.name
    base = workloads.get(wl.name)
    for name in ("layout", "replicas", "reduce_dtype", "gather_source", "grad_dtype", "N"):
        if getattr(wl, name) != getattr(base, name):
            key += f"+{name}={getattr(wl, name)}"
    if micro_batches > 1:
        key += f"+micro_batches={micro_batches}"
    return key


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary line
    `kernel workload bytes_per_launch kernels_cu_sha` (workload as
    traffic_key gives it); None when absent or when the kernel source has
    changed since the capture."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    sha = kernel_source_sha()
    for line in open(path):
        f = line.split()
        if len(f) >= 4 and not line.startswith("#") and f[0] == kernel and f[1] == workload and f[3] == sha:
            return int(float(f[2]))
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""
    FIELDS = ["index", "clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, device: int):
        self.proc = None
        self.device = device

    def __enter__(self):
        smi = shutil.which("nvidia-smi")
        if smi is None:
            return self
        try:
            uuid = str(torch.cuda.get_device_properties(self.device).uuid)
            ident = uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"
        except Exception:
            ident = str(self.device)
        self.proc = subprocess.Popen([smi, "-i", ident, f"--query-gpu={','.join(self.FIELDS)}",
                                      "--format=csv,noheader,nounits", "-lms", "200"],
                                     stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.result = None
        if self.proc is None:
            return False
        time.sleep(0.25)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < len(self.FIELDS):
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if sm:
            self.result = {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                           "reasons": sorted(reasons), "samples": len(sm)}
        return False


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return world, rank, local


def dist_max(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# --------------------------------------------------------------------------- CPU oracle timing

def oracle_sample_workload(wl: workloads.Workload, S: int) -> workloads.Workload:
    """A bounded sample of the workload: one FLAT unit of S elements with the
    same N, gradient dtype, distributions and hyper-parameters."""
    largest = max(wl.units[0], key=lambda p: workloads.Workload.unit_numel(
        wl.with_(units=((p,),)), 0))
    unit = (workloads.Param("sample", (S,), largest.init),)
    return wl.with_(name=wl.name + f"_sample{S}", units=(unit,), layout="flat")


def time_oracle_steps(wl: workloads.Workload, target_s: float, n_steps: int):
    """Oracle step times on a sample sized for about target_s per step.
    Returns (list of per-step seconds, sample elements, counted bytes per step)."""
    import numpy as np
    from oracle import fsdp_oracle as O

    def one(sw, orc, grads):
        t0 = time.perf_counter()
        orc.step(grads)
        return time.perf_counter() - t0

    def make(S):
        sw = oracle_sample_workload(wl, S)
        params = [p.numpy() for p in workloads.param_tensors(sw, 0)]
        grads = []
        for r in range(sw.N):
            g = workloads.grad_tensor(sw, 0, 0, r)
            grads.append(g.numpy() if g.dtype == torch.float32 else g.view(torch.int16).numpy().view(np.uint16))
        orc = O.UnitOracle(sw.shapes(0), sw.N, "flat", O.AdamWHyper(**workloads.hyper(sw)),
                           sw.reshard_after_forward)
        orc.load(params)
        return sw, orc, grads

    S = calibrate_elements(wl, target_s, 1 << 26)
    sw, orc, grads = make(S)
    times = [one(sw, orc, grads) for _ in range(n_steps)]
    return times, S, counted_bytes(sw, 0)["step"]


def calibrate_elements(wl: workloads.Workload, target_s: float, cap: int) -> int:
    """Sample elements for which one oracle unit step takes about target_s on
    one core (from a timed step on 2^20 elements), within [2^20, cap]."""
    import numpy as np
    from oracle import fsdp_oracle as O
    S = 1 << 20
    sw = oracle_sample_workload(wl, S)
    params = [p.numpy() for p in workloads.param_tensors(sw, 0)]
    grads = []
    for r in range(sw.N):
        g = workloads.grad_tensor(sw, 0, 0, r)
        grads.append(g.numpy() if g.dtype == torch.float32 else g.view(torch.int16).numpy().view(np.uint16))
    orc = O.UnitOracle(sw.shapes(0), sw.N, "flat", O.AdamWHyper(**workloads.hyper(sw)), sw.reshard_after_forward)
    orc.load(params)
    t0 = time.perf_counter()
    orc.step(grads)
    dt = time.perf_counter() - t0
    return int(min(cap, max(1 << 20, S * target_s / max(dt, 1e-6))))


def cpu_cores_info():
    try:
        aff = len(os.sched_getaffinity(0))
    except Exception:
        aff = os.cpu_count()
    return aff


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                vendor = next((l.split(":", 1)[1].strip() for l in out.splitlines() if l.startswith("Vendor ID:")), "")
                return f"{vendor} {line.split(':', 1)[1].strip()}".strip()
    except Exception:
        pass
    try:
        info = open("/proc/cpuinfo").read()
        m = re.search(r"^model name\s*:\s*(.+)$", info, re.M)
        if m:
            return m.group(1).strip()
        imp = re.search(r"^CPU implementer\s*:\s*(\S+)", info, re.M)
        part = re.search(r"^CPU part\s*:\s*(\S+)", info, re.M)
        if imp and part:
            return f"CPU implementer {imp.group(1)} part {part.group(1)}"
    except OSError:
        pass
    return "unknown"


def _oracle_worker(wl, index, S, barrier, commands, results):
    """One spawned worker of OracleTeam: builds its own FLAT sample unit of S
    elements drawn like `wl` (its own seeds), then on every command runs one
    unchanged oracle unit step, starting together with the other workers."""
    import numpy as np
    from oracle import fsdp_oracle as O
    sw = oracle_sample_workload(wl, S).with_(name=f"{wl.name}_sample{S}_worker{index}")
    params = [p.numpy() for p in workloads.param_tensors(sw, 0)]
    grads = []
    for r in range(sw.N):
        g = workloads.grad_tensor(sw, 0, 0, r)
        grads.append(g.numpy() if g.dtype == torch.float32 else g.view(torch.int16).numpy().view(np.uint16))
    orc = O.UnitOracle(sw.shapes(0), sw.N, "flat", O.AdamWHyper(**workloads.hyper(sw)), sw.reshard_after_forward)
    orc.load(params)
    results.put(("ready", index, counted_bytes(sw, 0)["step"]))
    while commands.get() is not None:
        barrier.wait()
        t0 = time.perf_counter()
        orc.step(grads)
        results.put(("done", index, time.perf_counter() - t0))


class OracleTeam:
    """n worker processes on the host cores (spawned, so that none inherits a
    CUDA context), each holding a FLAT sample unit of `per_worker` elements
    drawn like the workload; step() runs one oracle unit step on all of them at
    once and returns the step's wall time (the slowest worker).  Every element
    of the cycle is independent, so n disjoint samples stand for one sample n
    times as large."""

    def __init__(self, wl, n: int, per_worker: int):
        import multiprocessing as mp
        ctx = mp.get_context("spawn")
        self.n = n
        self.barrier = ctx.Barrier(n)
        self.results = ctx.Queue()
        self.commands = [ctx.Queue() for _ in range(n)]
        self.procs = [ctx.Process(target=_oracle_worker, args=(wl, i, per_worker, self.barrier, self.commands[i],
                                                               self.results), daemon=True) for i in range(n)]
        for p in self.procs:
            p.start()
        ready = [self._get() for _ in range(n)]
        self.step_bytes = sum(r[2] for r in ready)
        self.elements = n * per_worker

    def _get(self, limit_s: float = 600.0):
        """The next worker message; raises if a worker died or nothing came."""
        import queue
        t0 = time.time()
        while True:
            try:
                return self.results.get(timeout=1.0)
            except queue.Empty:
                dead = [p.exitcode for p in self.procs if p.exitcode not in (None, 0)]
                if dead or time.time() - t0 > limit_s:
                    self.close()
                    raise RuntimeError(f"oracle worker failed (exit codes {dead})" if dead else
                                       "oracle workers gave no answer")

    def step(self) -> float:
        for q in self.commands:
            q.put(1)
        return max(self._get()[2] for _ in range(self.n))

    def close(self):
        for p, q in zip(self.procs, self.commands):
            if p.is_alive():
                q.put(None)
        for p in self.procs:
            p.join(timeout=60)
            if p.is_alive():
                p.terminate()


def oracle_all_cores(wl, n_steps: int, per_worker: int, cores: int | None = None, warmup: int = 0):
    """Per-step wall times of the oracle on every host core at once, after
    `warmup` untimed steps.  Returns (times, elements per step, counted bytes
    per step, workers)."""
    n = cores or cpu_cores_info() or 1
    team = OracleTeam(wl, n, per_worker)
    try:
        times = [team.step() for _ in range(warmup + n_steps)][warmup:]
    finally:
        team.close()
    return times, team.elements, team.step_bytes, n


# --------------------------------------------------------------------------- arms

def run_reference(args, world, rank):
    """The oracle as it stands, on all the host's cores: each bench step is one
    oracle unit step on every core at once, each core on its own bounded
    sample of the workload (disjoint draws; the elements are independent).
    A few one-core steps on one such sample are reported beside it."""
    if rank != 0:
        return
    wl = workloads.get(args.workload)
    per_worker = calibrate_elements(wl, args.ref_step_seconds, 1 << 24)
    times, elems, cb, n = oracle_all_cores(wl, args.warmup + args.steps, per_worker)
    timed = times[args.warmup:]
    sec = sum(timed)
    value = cb * len(timed) / sec / 1e9
    t1, S1, cb1 = time_oracle_steps(wl, target_s=args.ref_step_seconds, n_steps=2)
    cpu = {"value": value, "unit": "GB/s", "cores": n, "kind": "oracle",
           "sample": f"{n} worker processes, each one FLAT unit of {per_worker} elements drawn like {wl.name} "
                     f"(N={wl.N}, {wl.grad_dtype} grads); one oracle unit step on all of them per bench step",
           "elements_per_step": elems,
           "host": {"cpu_model": cpu_model(), "cores_available": cpu_cores_info()},
           "single_core": {"value": cb1 * len(t1) / sum(t1) / 1e9, "unit": "GB/s", "cores": 1,
                           "sample": f"2 oracle unit steps on one FLAT unit of {S1} elements"}}
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sec / len(timed),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic", "config": {"workload": wl.name, "sample_elements": elems},
            "cpu_baseline": cpu,
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def selected_workload(args) -> workloads.Workload:
    wl = workloads.get(args.workload)
    if args.units is not None:          # profiling a few units of a many-unit model
        wl = wl.with_(units=wl.units[:args.units])
    over = {k: v for k, v in (("gather_source", args.gather_source), ("layout", args.layout),
                              ("reduce_dtype", args.reduce_dtype),
                              ("fuse_reduce_adamw", None if args.fuse is None else args.fuse == "on"),
                              ("replicas", args.replicas))
            if v is not None}
    return wl.with_(**over) if over else wl


def run_ours(args, world, rank, local):
    from fully_sharded_unit_gb300 import binding as B
    from fully_sharded_unit_gb300.build import build

    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA GPU (the library has no CPU path)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    build()
    B.lib()
    wl = selected_workload(args)
    hp = workloads.hyper(wl)
    units = []
    for i in range(wl.n_units):
        u = B.Unit(wl.shapes(i), wl.layout, wl.N, wl.grad_dtype, wl.reshard_after_forward,
                   replicas=wl.replicas, reduce_dtype=wl.reduce_dtype, gather_source=wl.gather_source,
                   fuse_reduce_adamw=wl.fuse_reduce_adamw)
        params = workloads.param_tensors(wl, i, dev)
        u.load(params)
        torch.cuda.synchronize()
        del params
        units.append(u)
    P_max = max(u.numel for u in units)
    # the N ranks' full gradients (one backward's output), reused by every unit
    grads = [torch.empty(P_max, dtype=wl.torch_grad_dtype(), device=dev) for _ in range(wl.world)]
    for r in range(wl.world):
        workloads.grad_tensor(wl, 0, 0, r, dev, out=grads[r][:units[0].numel])
    out = torch.empty(P_max, dtype=torch.int16, device=dev)
    cb = [counted_bytes(wl, i) for i in range(wl.n_units)]
    if args.micro_batches > 1:
        assert not wl.fuse_reduce_adamw, "micro-batches use the separate reduce-scatter and AdamW"
        for i, c in enumerate(cb):
            acc = c["reduce_scatter"] + 4 * wl.unit_numel(i)      # also reads the shard it adds to
            c["step"] += (args.micro_batches - 1) * acc
            c["reduce_scatter"] = (c["reduce_scatter"] + (args.micro_batches - 1) * acc) / args.micro_batches
    step_bytes = sum(c["step"] for c in cb)
    stream = torch.cuda.current_stream()

    K = args.micro_batches

    def step():
        st = torch.cuda.current_stream()   # the capture stream when recording a graph
        for i, u in enumerate(units):
            g = grads if units[i].numel == P_max else [x[:u.numel] for x in grads]
            if K == 1:
                u.step(g, out, hp, st)
                continue
            u.allgather(out, st)
            if wl.reshard_after_forward:
                u.allgather(out, st)
            for k in range(K):
                u.reduce_scatter_ex(g, accumulate=k > 0, stream=st)
            u.adamw_step(hp, st)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    for u in units:
        B.fsdp_profile_reset(u.handle)
        B.fsdp_profile_enable(u.handle, True)

    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dist_barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        ev0.record(stream)
        for _ in range(args.steps):
            step()
        ev1.record(stream)
        torch.cuda.synchronize()
    dist_barrier(world)
    ms = ev0.elapsed_time(ev1)
    for u in units:
        B.fsdp_profile_enable(u.handle, False)
    ms_max = dist_max(ms, world, dev)

    # per-kernel device time over the timed region (events on the launch stream)
    per_kernel = {}
    launches = 0
    for k in ("gather", "reduce_scatter", "adamw", "reduce_adamw"):
        tot, n = 0.0, 0
        for u in units:
            t, c = B.fsdp_profile_read(u.handle, k)
            tot, n = tot + t, n + c
        per_kernel[k] = (tot, n)
        launches += n
    dom = max(per_kernel, key=lambda k: per_kernel[k][0])
    dom_ms, dom_n = per_kernel[dom]
    per_step = {"gather": lambda c: c["gather"] * c["gathers"],
                "reduce_scatter": lambda c: c["reduce_scatter"] * args.micro_batches}
    dom_bytes = sum(per_step.get(dom, lambda c: c[dom])(c) for c in cb) / \
        (dom_n / args.steps)      # counted bytes per launch
    achieved = dom_bytes / (dom_ms / dom_n * 1e-3) / 1e9
    peak, peak_kind = measured_peak()
    roofline = {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "peak_source": peak_kind,
                "traffic": recorded_traffic(dom, traffic_key(wl, args.micro_batches)),
                "per_kernel_ms_per_launch": {k: (v[0] / v[1] if v[1] else None) for k, v in per_kernel.items()},
                "per_kernel_gbs": {k: (sum(per_step.get(k, lambda c: c[k])(c) for c in cb) /
                                       (v[1] / args.steps) / (v[0] / v[1] * 1e-3) / 1e9 if v[1] else None)
                                   for k, v in per_kernel.items()}}

    value_rank = step_bytes * args.steps / (ms * 1e-3) / 1e9
    value = world * step_bytes * args.steps / (ms_max * 1e-3) / 1e9

    # the same configuration without the profiler's event pair around every
    # launch (which serialises consecutive kernels): the step as a caller runs it
    unprofiled = run_variant(args, units, step, stream, hp, world, dev, wl)
    del unprofiled["gather_source"], unprofiled["fused_reduce_adamw"]

    # the fastest configuration on the same units: bf16-shadow gather and the
    # fused reduce-scatter + AdamW (identical results, fewer bytes)
    fastest = None
    if args.fastest and K == 1 and not (wl.fuse_reduce_adamw and wl.gather_source == "shadow"):
        fastest = run_variant(args, units, step, stream, hp, world, dev,
                              wl.with_(gather_source="shadow", fuse_reduce_adamw=True))
        for u in units:
            B.fsdp_unit_set_step_options(u.handle, wl.gather_source, wl.fuse_reduce_adamw)

    graph = None
    if args.graph and K == 1:
        graph = run_graph(args, units, step, stream, step_bytes, hp, world, dev)

    # end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e and args.micro_batches == 1 and not wl.fuse_reduce_adamw:
        # the host link's speed differs from box to box, and so does which way
        # of moving the gradients in is faster: "auto" times both and reports
        # the faster, with both figures
        modes = ["pipelined", "pipelined_direct", "zero_copy"] if args.e2e_mode == "auto" else [args.e2e_mode]
        runs = [run_e2e(args, wl, units, grads, out, hp, cb, step_bytes, stream, dev, world, m) for m in modes]
        timed = [r for r in runs if r.get("value") is not None]
        e2e = min(timed, key=lambda r: r["ms_per_step"]) if timed else runs[0]
        if len(runs) > 1:
            e2e = dict(e2e, modes_ms_per_step={r["mode"]: r.get("ms_per_step") for r in runs if "mode" in r})

    cpu = None
    if not args.no_cpu_baseline and rank == 0 and world == 1:
        cpu = cpu_baseline(args, wl)

    # FSDP_KSTATUS_* bits raised by any kernel during the run (0: none)
    kstatus = 0
    for u in units:
        kstatus |= u.kernel_status(stream)
        u.close()
    del grads, out, units
    torch.cuda.empty_cache()

    # every other workload shape, timed the same way on the same GPU
    configs = None
    if args.configs and args.micro_batches == 1:
        configs = {}
        for name in CONFIG_WORKLOADS:
            if name != wl.name:
                configs[name] = run_config(args, workloads.get(name), dev, world)
                kstatus |= configs[name].pop("kernel_status")
    survey = sum(survey_bytes(wl, i) for i in range(wl.n_units))
    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "pct_of_hbm_peak": 100.0 * value_rank / peak, "hbm_peak_gbs": peak, "hbm_peak_source": peak_kind,
        "counted_bytes_per_step_survey": survey,
        "value_survey": world * survey * args.steps / (ms_max * 1e-3) / 1e9,
        "pct_of_hbm_peak_survey": 100.0 * survey * args.steps / (ms * 1e-3) / 1e9 / peak,
        "config": {"workload": wl.name, "units": wl.n_units, "params_per_unit": [u_ for u_ in
                   (wl.unit_numel(i) for i in range(wl.n_units))], "virtual_ranks": wl.N,
                   "layout": wl.layout, "grad_dtype": wl.grad_dtype,
                   "reshard_after_forward": wl.reshard_after_forward,
                   "replicas": wl.replicas, "reduce_dtype": wl.reduce_dtype,
                   "fused_reduce_adamw": wl.fuse_reduce_adamw, "micro_batches": args.micro_batches,
                   "counted_bytes_per_step": step_bytes,
                   "gather_source": "fp32 master" if wl.gather_source == "master" else "bf16 shadow",
                   "l2": l2_statement(wl), "parallelism": f"replicas x{world}"},
        "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches,
        "graph": graph, "unprofiled": unprofiled, "fastest_variant": fastest, "kernel_status": kstatus,
        "clocks": clk.result, "configs": configs,
    }
    print(json.dumps(line), flush=True)


def cpu_baseline(args, wl) -> dict:
    """The oracle on the host cores: all cores at once (the reported value)
    and one core, each over 3 unit steps of bounded samples of the workload."""
    times, S, ccb = time_oracle_steps(wl, target_s=args.cpu_seconds / 6, n_steps=3)
    single = {"value": ccb * len(times) / sum(times) / 1e9, "unit": "GB/s", "cores": 1,
              "sample": f"3 oracle unit steps on one FLAT unit of {S} elements"}
    per_worker = min(S, 1 << 24)
    at, elems, acb, n = oracle_all_cores(wl, 3, per_worker, warmup=1)
    return {"value": acb * len(at) / sum(at) / 1e9, "unit": "GB/s", "cores": n, "kind": "oracle",
            "sample": f"3 oracle unit steps on {n} worker processes at once, each one FLAT unit of "
                      f"{per_worker} elements drawn like {wl.name} (N={wl.N}, {wl.grad_dtype} grads)",
            "elements_per_step": elems,
            "host": {"cpu_model": cpu_model(), "cores_available": cpu_cores_info()},
            "single_core": single}


# the workloads timed besides the headline one, each on its own
CONFIG_WORKLOADS = ("tiny_flat", "gpt2_small_flat", "gpt2_large_dim0", "ragged_flat_n7", "ragged_dim0_n7",
                    "ragged_flat_n64", "ragged_dim0_n64", "mingpt175b_flat")


def run_config(args, wl: workloads.Workload, dev, world) -> dict:
    """One workload's model step (fsdp_step on every unit) timed with CUDA
    events around K steps on the launch stream; each kernel's time per launch
    from K back-to-back rounds of that kernel alone over every unit; and the
    step again with the per-launch profiler's event pairs (which serialise the
    launches: `profiled_ms_per_step`).  K is chosen so the timed region lasts
    about 0.2 s (at least 10 steps)."""
    from fully_sharded_unit_gb300 import binding as B
    hp = workloads.hyper(wl)
    units = []
    for i in range(wl.n_units):
        u = B.Unit(wl.shapes(i), wl.layout, wl.N, wl.grad_dtype, wl.reshard_after_forward, replicas=wl.replicas,
                   reduce_dtype=wl.reduce_dtype, gather_source=wl.gather_source,
                   fuse_reduce_adamw=wl.fuse_reduce_adamw)
        u.load(workloads.param_tensors(wl, i, dev))
        units.append(u)
    P_max = max(u.numel for u in units)
    grads = [torch.empty(P_max, dtype=wl.torch_grad_dtype(), device=dev) for _ in range(wl.world)]
    for r in range(wl.world):
        workloads.grad_tensor(wl, 0, 0, r, dev, out=grads[r][:units[0].numel])
    out = torch.empty(P_max, dtype=torch.int16, device=dev)
    stream = torch.cuda.current_stream()
    views = [grads if u.numel == P_max else [g[:u.numel] for g in grads] for u in units]
    # the C entry point with its arguments marshalled once per unit (checked by
    # one ordinary call each), so that the host's call rate does not bound the
    # small units on a slow host
    import ctypes
    lib, sh = B.lib(), stream.cuda_stream
    hp_c = B._hp(hp)
    for u, g in zip(units, views):
        u.step(g, out, hp, stream)
    torch.cuda.synchronize()
    step_args = [(u.handle, B._ptrs(g), out.data_ptr(), ctypes.byref(hp_c), sh) for u, g in zip(units, views)]

    def step():
        for a in step_args:
            rc = lib.fsdp_step(*a)
            assert rc == B.FSDP_OK, B.fsdp_last_error()

    def timed(k):
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        dist_barrier(world)
        torch.cuda.synchronize()
        ev0.record(stream)
        for _ in range(k):
            step()
        ev1.record(stream)
        torch.cuda.synchronize()
        return dist_max(ev0.elapsed_time(ev1), world, dev)

    est = timed(max(3, args.warmup)) / max(3, args.warmup)
    K = int(min(1000, max(10, round(200.0 / max(est, 1e-3)))))
    ms = timed(K) / K
    cb = [counted_bytes(wl, i) for i in range(wl.n_units)]
    # each kernel alone, launched back to back over every unit K times (no
    # events between launches, so launches overlap as in the step); AdamW
    # advances the units' state, which changes nothing in its bytes or time
    # (the C entry points with their arguments marshalled once, so that the
    # host's launch rate does not bound the small units)
    import ctypes
    lib, sh = B.lib(), stream.cuda_stream
    hp_c = B._hp(hp)
    ptrs = {id(g): B._ptrs(g) for g in views}
    calls = {"gather": lambda u, g: lib.fsdp_allgather(u.handle, out.data_ptr(), sh),
             "reduce_scatter": lambda u, g: lib.fsdp_reduce_scatter(u.handle, ptrs[id(g)], sh),
             "adamw": lambda u, g: lib.fsdp_adamw_step(u.handle, ctypes.byref(hp_c), sh)}
    kernels = {}
    for k, call in calls.items():
        def one_kernel(k_steps, call=call):
            ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            ev0.record(stream)
            for _ in range(k_steps):
                for u, g in zip(units, views):
                    rc = call(u, g)
                    assert rc == B.FSDP_OK, B.fsdp_last_error()
            ev1.record(stream)
            torch.cuda.synchronize()
            return ev0.elapsed_time(ev1)
        one_kernel(2)
        kms = one_kernel(K) / (K * wl.n_units)
        kernels[k] = {"ms_per_launch": kms, "gbs": sum(c[k] for c in cb) / wl.n_units / (kms * 1e-3) / 1e9}
    for u in units:
        B.fsdp_profile_reset(u.handle)
        B.fsdp_profile_enable(u.handle, True)
    pms = timed(K) / K
    kstatus = 0
    for u in units:
        kstatus |= u.kernel_status(stream)
        u.close()
    step_bytes = sum(c["step"] for c in cb)
    survey = sum(survey_bytes(wl, i) for i in range(wl.n_units))
    peak, _ = measured_peak()
    return {"units": wl.n_units, "params_per_unit": wl.unit_numel(0), "virtual_ranks": wl.N, "layout": wl.layout,
            "grad_dtype": wl.grad_dtype, "steps": K, "ms_per_step": ms, "ms_per_unit_step": ms / wl.n_units,
            "counted_bytes_per_step": step_bytes, "value": world * step_bytes / (ms * 1e-3) / 1e9,
            "counted_bytes_per_step_survey": survey, "value_survey": world * survey / (ms * 1e-3) / 1e9,
            "pct_of_hbm_peak_survey": 100.0 * survey / (ms * 1e-3) / 1e9 / peak, "unit": "GB/s",
            "profiled_ms_per_step": pms, "kernels": kernels, "l2": l2_statement(wl), "kernel_status": kstatus}


def run_variant(args, units, step, stream, hp, world, dev, vwl):
    """Time args.steps steps of the same units after switching them to the
    variant's gather source and fusion; same step, same counted-bytes rules."""
    from fully_sharded_unit_gb300 import binding as B
    for u in units:
        B.fsdp_unit_set_step_options(u.handle, vwl.gather_source, vwl.fuse_reduce_adamw)
    vbytes = sum(counted_bytes(vwl, i)["step"] for i in range(vwl.n_units))
    for _ in range(args.warmup):
        step()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dist_barrier(world)
    torch.cuda.synchronize()
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize()
    ms = dist_max(ev0.elapsed_time(ev1), world, dev)
    return {"gather_source": vwl.gather_source, "fused_reduce_adamw": vwl.fuse_reduce_adamw,
            "ms_per_step": ms / args.steps, "counted_bytes_per_step": vbytes,
            "value": world * vbytes * args.steps / (ms * 1e-3) / 1e9, "unit": "GB/s"}


def run_graph(args, units, step, stream, step_bytes, hp, world, dev):
    """The whole step (every unit's fsdp_step) captured once as a CUDA graph
    and replayed: each unit switches to its device-side AdamW step counter
    first, so every replay is a correct next step."""
    from fully_sharded_unit_gb300 import binding as B
    n = args.warmup + args.steps + 4
    for u in units:
        B.fsdp_adamw_device_steps(u.handle, hp, n, stream)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=torch.cuda.Stream(device=dev)):
        step()
    for _ in range(args.warmup):
        g.replay()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dist_barrier(world)
    torch.cuda.synchronize()
    ev0.record(stream)
    for _ in range(args.steps):
        g.replay()
    ev1.record(stream)
    torch.cuda.synchronize()
    ms = dist_max(ev0.elapsed_time(ev1), world, dev)
    ok = all(not B.fsdp_adamw_device_status(u.handle, stream)[1] for u in units)
    for u in units:
        B.fsdp_adamw_device_steps(u.handle, None, 0, stream)
    del g
    return {"ms_per_step": ms / args.steps, "value": world * step_bytes * args.steps / (ms * 1e-3) / 1e9,
            "unit": "GB/s", "steps": args.steps, "table_ok": ok}


def run_e2e(args, wl, units, grads, out, hp, cb, step_bytes, stream, dev, world, mode):
    """Same metric through the public API with the step's inputs and result in
    pinned host memory.  Every step, for every unit, the N gradients come from
    the host and the gathered bf16 parameters go back to the host:
      zero_copy -- the reduce-scatter reads the pinned host gradients directly
                   over the host link (device addresses from
                   fsdp_host_device_pointer);
      copy      -- cudaMemcpyAsync of each gradient host->device first, on
                   the compute stream;
      pipelined -- the same copies on a stream of their own, into two device
                   sets of gradients used by alternate units, so that a unit's
                   gradients cross the host link while the unit before it
                   computes (the first unit of the next step while this step's
                   last unit computes); the reduce-scatter waits for its unit's
                   copies.  Every timed step's copies start after the timed
                   region opens;
      pipelined_direct -- pipelined, but the first gather's kernel stores the
                   gathered parameters straight into the pinned host buffer
                   (a device address from fsdp_host_device_pointer), so no
                   device->host copy runs beside the host->device ones.
    The unit step is issued as its calls (gather, gather again, reduce-scatter,
    AdamW: the work of fsdp_step) so that the gathered parameters, final after
    the first gather, are copied to the host on a second stream while the rest
    of the unit step runs.  The timed region ends when the last copy has landed."""
    from fully_sharded_unit_gb300 import binding as B
    P_max = grads[0].numel()
    # pinned host memory: distinct gradient buffers for every virtual rank when
    # the host has room for all local ranks' copies; otherwise every virtual
    # rank reads one shared pinned buffer (the same bytes cross the host link,
    # only the values repeat)
    esz = grads[0].element_size()
    need_distinct = len(grads) * P_max * esz + len(units) * P_max * 2
    need_shared = P_max * esz + len(units) * P_max * 2
    local_ranks = int(os.environ.get("LOCAL_WORLD_SIZE", "1"))
    avail = host_mem_available()
    if avail is None or need_distinct * local_ranks <= 0.5 * avail:
        inputs = "distinct pinned host buffer per virtual rank"
        host_grads = [torch.empty(P_max, dtype=grads[0].dtype, pin_memory=True) for _ in grads]
    elif need_shared * local_ranks <= 0.5 * avail:
        inputs = "one pinned host buffer shared by all virtual ranks (host memory)"
        shared = torch.empty(P_max, dtype=grads[0].dtype, pin_memory=True)
        host_grads = [shared] * len(grads)
    else:
        return {"value": None, "unit": "GB/s", "skipped": f"host memory: {need_shared * local_ranks / 1e9:.0f} GB "
                f"of pinned buffers needed, {avail / 1e9:.0f} GB available"}
    for h, g in zip(host_grads, grads):
        h.copy_(g)
    host_out = [torch.empty(P_max, dtype=torch.int16, pin_memory=True) for _ in units]
    outs = [(out, torch.empty_like(out)), (torch.empty_like(out), torch.empty_like(out))]
    copy_stream = torch.cuda.Stream(device=dev)
    h2d_stream = torch.cuda.Stream(device=dev)
    direct = mode == "pipelined_direct"   # the first gather writes straight into pinned host memory
    if direct:
        mode = "pipelined"
        host_out_dev = [B.fsdp_host_device_pointer(h) for h in host_out]
    if mode == "zero_copy":
        unit_grads = [[B.fsdp_host_device_pointer(h[:u.numel]) for h in host_grads] for u in units]
    elif mode == "pipelined":
        # two device sets of the gradients, used by alternate units: a unit's
        # gradients are copied in while the unit before it computes
        sets = [grads] + ([[torch.empty_like(g) for g in grads]] if len(units) > 1 else [])
        unit_grads = [[g[:u.numel] for g in sets[i % len(sets)]] for i, u in enumerate(units)]
    else:
        unit_grads = [[g[:u.numel] for g in grads] for u in units]
    free = [None, None]      # events: last D2H copy out of outs[k][0] finished
    consumed = [None, None]  # events: the reduce-scatter that read gradient set k has finished
    pending = {}             # unit -> event: its gradients are on the device (pipelined)

    def issue_copy(i):
        """Unit i's gradients host->device on the copy stream, into its set,
        once the reduce-scatter that last read that set has finished."""
        u, k = units[i], i % 2
        if consumed[k] is not None:
            h2d_stream.wait_event(consumed[k])
        with torch.cuda.stream(h2d_stream):
            for h, g in zip(host_grads, unit_grads[i]):
                g.copy_(h[:u.numel], non_blocking=True)
        ev = torch.cuda.Event()
        ev.record(h2d_stream)
        pending[i] = ev

    def step(prefetch=False):
        """One e2e step; with `prefetch` (pipelined) the next step's first
        unit's gradients are queued for copying at the end."""
        done = []
        if mode == "pipelined" and 0 not in pending:
            issue_copy(0)
        for i, u in enumerate(units):
            if mode == "pipelined" and i + 1 < len(units):
                issue_copy(i + 1)           # copied while this unit computes
            first, second = outs[i % 2]
            if free[i % 2] is not None:
                stream.wait_event(free[i % 2])
            if mode == "copy":
                for h, g in zip(host_grads, grads):
                    g[:u.numel].copy_(h[:u.numel], non_blocking=True)
            if direct:   # gathered parameters stored over the host link by the kernel itself
                rc = B.lib().fsdp_allgather(u.handle, host_out_dev[i].data_ptr(), stream.cuda_stream)
                assert rc == B.FSDP_OK, B.fsdp_last_error()
            else:
                u.allgather(first[:u.numel], stream)
                ready = torch.cuda.Event()
                ready.record(stream)
                copy_stream.wait_event(ready)
                with torch.cuda.stream(copy_stream):
                    host_out[i][:u.numel].copy_(first[:u.numel], non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(copy_stream)
                free[i % 2] = ev
                done.append(ev)
            if wl.reshard_after_forward:
                u.allgather(second[:u.numel], stream)
            if mode == "pipelined":
                stream.wait_event(pending.pop(i))
            u.reduce_scatter(unit_grads[i], stream)
            if mode == "pipelined":
                ev = torch.cuda.Event()
                ev.record(stream)
                consumed[i % 2] = ev
            u.adamw_step(hp, stream)
        for ev in done:
            stream.wait_event(ev)
        if mode == "pipelined" and prefetch:
            issue_copy(0)

    step()
    torch.cuda.synchronize()
    link = host_link_rates(host_grads[0], grads[0], stream)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dist_barrier(world)
    torch.cuda.synchronize()
    ev0.record(stream)
    h2d_stream.wait_event(ev0)     # every timed step's copies start inside the timed region
    for j in range(args.e2e_steps):
        step(prefetch=j + 1 < args.e2e_steps)
    ev1.record(stream)
    torch.cuda.synchronize()
    dist_barrier(world)
    ms = dist_max(ev0.elapsed_time(ev1), world, dev)
    h2d = sum(c["h2d"] for c in cb)
    d2h = sum(c["d2h"] for c in cb)
    del host_grads, host_out, unit_grads, outs
    if mode == "pipelined":
        del sets
    return {"value": world * step_bytes * args.e2e_steps / (ms * 1e-3) / 1e9, "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": args.e2e_steps,
            "ms_per_step": ms / args.e2e_steps, "mode": "pipelined_direct" if direct else mode, "inputs": inputs,
            "host_link": link}


def host_link_rates(host: torch.Tensor, dev: torch.Tensor, stream) -> dict:
    """This machine's host link, measured just before the e2e timing: one copy of
    `host` (pinned) to the device and one back, each alone (GB/s)."""
    out = {}
    for name, dst, src in (("h2d_gbs", dev, host), ("d2h_gbs", host, dev)):
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        ev0.record(stream)
        with torch.cuda.stream(stream):
            dst.copy_(src, non_blocking=True)
        ev1.record(stream)
        torch.cuda.synchronize()
        out[name] = src.numel() * src.element_size() / (ev0.elapsed_time(ev1) * 1e-3) / 1e9
    return out


def host_mem_available():
    """MemAvailable in bytes (Linux), or None when unknown."""
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024
    except OSError:
        pass
    return None


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="mingpt175b_flat", choices=sorted(workloads.WORKLOADS))
    ap.add_argument("--e2e-steps", type=int, default=3)
    ap.add_argument("--e2e-mode", choices=["auto", "pipelined", "pipelined_direct", "zero_copy", "copy"],
                    default="auto",
                    help="pipelined: gradients copied host->device on their own stream into two "
                         "alternating device sets while the previous unit computes; zero_copy: the "
                         "reduce-scatter reads pinned host memory directly; pipelined_direct: "
                         "pipelined, with the first gather writing straight into pinned host "
                         "memory (no device->host copy); copy: copies on the compute stream; "
                         "auto: time pipelined, pipelined_direct and zero_copy, report the fastest")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-step-seconds", type=float, default=2.0)
    ap.add_argument("--gather-source", choices=["master", "shadow"], default=None,
                    help="override the workload's gather source")
    ap.add_argument("--layout", choices=["flat", "dim0", "flat_padded"], default=None)
    ap.add_argument("--reduce-dtype", choices=["f32", "bf16"], default=None)
    ap.add_argument("--replicas", type=int, default=None,
                    help="hybrid sharding: replication groups (the workload's N ranks per group)")
    ap.add_argument("--micro-batches", type=int, default=1,
                    help="gradient accumulation: reduce-scatters per step (the first overwrites, "
                         "the rest accumulate), then one AdamW")
    ap.add_argument("--no-fastest", dest="fastest", action="store_false",
                    help="skip timing the fastest configuration (shadow gather + fused step) "
                         "on the same units")
    ap.add_argument("--no-graph", dest="graph", action="store_false",
                    help="skip timing the step captured once in a CUDA graph and replayed "
                         "(device-side AdamW step counter)")
    ap.add_argument("--fuse", choices=["on", "off"], default=None,
                    help="override whether fsdp_step fuses reduce-scatter and AdamW")
    ap.add_argument("--units", type=int, default=None,
                    help="time only the first K units of the workload (for small profiling captures)")
    ap.add_argument("--no-configs", dest="configs", action="store_false",
                    help="skip timing the other workloads (the 'configs' object)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_setup()
    if world != args.gpus and world > 1:
        ap.error(f"--gpus {args.gpus} but WORLD_SIZE={world}")
    try:
        if args.impl == "reference":
            run_reference(args, world, rank)
        else:
            run_ours(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()

"""Runs a workload through the C-ABI library on the GPU and the CPU oracle on
the same seeded inputs, and compares.

Gather, cast, layout and reduce-scatter outputs must be bit-identical.
AdamW state (master, m, v) must satisfy |gpu - oracle| <= 1e-6 + 1e-5*|oracle|
elementwise (max abs err 1e-6 / max rel err 1e-5, read as an allclose bound);
the harness also reports how many elements differ at all, since the kernel
evaluates the same fp32 operation sequence as the oracle.

AdamW's stricter per-state bounds are checked as well: v within a relative
1e-5 everywhere (a sum of non-negative terms, no cancellation) and m within
1e-5 x (beta1 |m_prev| + (1 - beta1) |g|) (the size of its operands).  The
kernels evaluate the oracle's operation sequence, so the windowed checks at
the full sizes also require AdamW state to be bit-identical (``bitwise``).

Two modes:
* full   -- every element, step by step (units the host holds easily);
* window -- windows of global indices around every shard and parameter
            boundary (+-4096) plus random windows, drawn afresh for every
            step, each step's covering at least a given fraction of the unit
            (5 % by default).  Every operation after the layout is elementwise
            in the global index ("FSDP Architecture", the GPU-k boundary
            formula and backward step 3; "PyTorch FSDP ...", section 3.2.1,
            communication layout), so the oracle computes a window from the
            initial parameters and the ranks' gradients in that window; the
            union of all steps' windows is followed through every step and
            compared at every step.  The oracle runs on slices of the union in
            worker processes (spawned, so none inherits the CUDA context),
            each calling the unchanged oracle functions; the split is exact
            because every element is independent.
"""
from __future__ import annotations

import atexit
import os

import numpy as np
import torch

from fully_sharded_unit_gb300 import binding as B
from fully_sharded_unit_gb300 import workloads
from oracle import fsdp_oracle as O

ATOL, RTOL = 1e-6, 1e-5


def grad_np(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.float32:
        return t.numpy()
    return t.view(torch.int16).numpy().view(np.uint16)


def u16(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def assert_bits_equal(got: np.ndarray, want: np.ndarray, what: str) -> None:
    assert got.shape == want.shape, (what, got.shape, want.shape)
    if got.dtype == np.uint16:
        g, w = got, want
        nan_g = ((g & 0x7F80) == 0x7F80) & ((g & 0x7F) != 0)
        nan_w = ((w & 0x7F80) == 0x7F80) & ((w & 0x7F) != 0)
    else:
        g, w = got.view(np.uint32), want.view(np.uint32)
        nan_g, nan_w = np.isnan(got), np.isnan(want)
    assert np.array_equal(nan_g, nan_w), f"{what}: NaN positions differ"
    bad = (g != w) & ~nan_w
    if bad.any():
        i = int(np.flatnonzero(bad)[0])
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} elements differ; first at {i}: "
                             f"got {got[i]!r} want {want[i]!r}")


def adamw_compare(got: np.ndarray, want: np.ndarray, what: str, which: str | None = None,
                  m_prev: np.ndarray | None = None, g: np.ndarray | None = None, beta1: float = 0.9,
                  bitwise: bool = False) -> dict:
    """The AdamW tolerance on one state: |a - b| <= 1e-6 + 1e-5 |b| everywhere;
    for v (which = "exp_avg_sq") also |a - b| <= 1e-5 |b|; for m (which =
    "exp_avg", given the previous m and the last reduced gradient) also
    |a - b| <= 1e-5 (beta1 |m_prev| + (1 - beta1) |g|).  With ``bitwise`` every
    element must be bit-identical (NaN positions aside)."""
    gv = got.astype(np.float64)
    w = want.astype(np.float64)
    err = np.abs(gv - w)
    ok = err <= ATOL + RTOL * np.abs(w)
    nz = np.abs(w) > 0
    stats = dict(max_abs=float(err.max(initial=0.0)),
                 max_rel=float((err[nz] / np.abs(w[nz])).max(initial=0.0)),
                 n_diff=int((got.view(np.uint32) != want.view(np.uint32)).sum()), n=int(got.size))
    assert ok.all(), f"{what}: AdamW tolerance violated: {stats}"
    if which == "exp_avg_sq":
        assert (err <= RTOL * np.abs(w)).all(), f"{what}: v outside 1e-5 relative: {stats}"
    if which == "exp_avg" and m_prev is not None and g is not None:
        bound = RTOL * (beta1 * np.abs(m_prev.astype(np.float64)) + (1.0 - beta1) * np.abs(g.astype(np.float64)))
        assert (err <= bound).all(), f"{what}: m outside its operand bound: {stats}"
    if bitwise:
        assert stats["n_diff"] == 0, f"{what}: not bit-identical to the oracle: {stats}"
    return stats


class Comparison:
    """Collects AdamW statistics across checks."""

    def __init__(self):
        self.adamw = {}

    def add(self, key, stats):
        self.adamw[key] = stats

    @property
    def total_diff(self):
        return sum(s["n_diff"] for s in self.adamw.values())


def device_buffers(n: int, dtype, count: int, misalign: bool = False) -> list:
    """`count` CUDA tensors of n elements; with ``misalign`` each is a view that
    starts 16 bytes past a 32-byte boundary (16-byte but not 32-byte aligned)."""
    if not misalign:
        return [torch.empty(n, dtype=dtype, device="cuda") for _ in range(count)]
    k = 16 // torch.empty((), dtype=dtype).element_size()
    out = []
    for _ in range(count):
        base = torch.empty(n + 2 * k, dtype=dtype, device="cuda")
        v = base[k:k + n] if base.data_ptr() % 32 == 0 else base[:n]
        assert v.data_ptr() % 32 == 16
        out.append(v)
    return out


def run_full(wl: workloads.Workload, unit: int = 0, use_step: bool = False, steps: int | None = None,
             gen_device: str = "cpu", allocator=None, misalign: bool = False) -> Comparison:
    """Whole-unit comparison, every element, every step.  ``misalign``: the
    gradients and the gathered outputs are only 16-byte aligned."""
    shapes = wl.shapes(unit)
    N, P = wl.N, wl.unit_numel(unit)
    steps = wl.steps if steps is None else steps
    hp = workloads.hyper(wl)
    cmp = Comparison()
    params = workloads.param_tensors(wl, unit, gen_device)
    orc = O.UnitOracle(shapes, N, wl.layout, O.AdamWHyper(**hp), wl.reshard_after_forward,
                       replicas=wl.replicas, reduce_dtype=wl.reduce_dtype)
    orc.load([p.cpu().numpy() for p in params])
    u = B.Unit(shapes, wl.layout, N, wl.grad_dtype, wl.reshard_after_forward, replicas=wl.replicas,
               reduce_dtype=wl.reduce_dtype, gather_source=wl.gather_source,
               fuse_reduce_adamw=wl.fuse_reduce_adamw, allocator=allocator)
    try:
        u.load([p.cuda() for p in params])
        del params
        torch.cuda.synchronize()
        for k in range(N):   # shard-in
            assert_bits_equal(u.get_state("param", k).cpu().numpy(), orc.master[k], f"shard-in rank {k}")
            assert_bits_equal(u16(u.get_state("shadow", k)), orc.shadow[k], f"shadow rank {k}")
        outs = device_buffers(P, torch.int16, 2, misalign)
        gdev = device_buffers(P, wl.torch_grad_dtype(), wl.world, misalign)
        for s in range(steps):
            for r in range(wl.world):
                if gen_device == "cuda":
                    workloads.grad_tensor(wl, unit, s, r, "cuda", out=gdev[r])
                else:
                    gdev[r].copy_(workloads.grad_tensor(wl, unit, s, r, "cpu"))
            if s == steps - 1:       # m before the last update, for m's operand bound
                m_prev = [x.copy() for x in orc.m]
            want_outs = orc.step([grad_np(g) for g in gdev])
            if use_step:
                u.step(gdev, outs[0], hp)
                torch.cuda.synchronize()
                assert_bits_equal(u16(outs[0]), want_outs[-1], f"step {s} gathered")
            else:
                u.allgather(outs[0])
                if wl.reshard_after_forward:
                    u.allgather(outs[1])
                u.reduce_scatter(gdev)
                torch.cuda.synchronize()
                for i, w in enumerate(want_outs):
                    assert_bits_equal(u16(outs[i]), w, f"step {s} gather {i}")
                for k in range(N):
                    assert_bits_equal(u.get_state("grad", k).cpu().numpy(), orc.grad[k],
                                      f"step {s} grad shard rank {k}")
                u.adamw_step(hp)
                torch.cuda.synchronize()
            assert u.step_count == s + 1
        for k in range(N):
            for which, want in (("param", orc.master[k]), ("exp_avg", orc.m[k]), ("exp_avg_sq", orc.v[k])):
                got = u.get_state(which, k).cpu().numpy()
                cmp.add((which, k), adamw_compare(got, want, f"{which} rank {k}", which=which,
                                                  m_prev=m_prev[k] if steps else None, g=orc.grad[k],
                                                  beta1=hp["beta1"]))
            assert_bits_equal(u.get_state("grad", k).cpu().numpy(), orc.grad[k], f"final grad shard rank {k}")
            # the shadow is the cast of the GPU's own master (checked bitwise against that)
            assert_bits_equal(u16(u.get_state("shadow", k)), O.bf16_rne(u.get_state("param", k).cpu().numpy()),
                              f"shadow rank {k}")
        assert u.kernel_status() == 0, "a kernel raised its status word"
    finally:
        u.close()
    return cmp


def _merge(iv):
    iv = sorted((a, b) for a, b in iv if b > a)
    merged = []
    for a, b in iv:
        if merged and a <= merged[-1][1]:
            merged[-1] = (merged[-1][0], max(merged[-1][1], b))
        else:
            merged.append((a, b))
    return merged


def _covered(windows) -> int:
    return sum(b - a for a, b in windows)


def boundary_windows(P: int, boundaries, half: int = 4096):
    """+-half elements around every boundary, and the last half elements."""
    return _merge([(max(0, b - half), min(P, b + half)) for b in boundaries] + [(max(0, P - half), P)])


def random_windows(P: int, frac: float, length: int, rng):
    """Random windows of `length` elements (the last one shorter when needed)
    whose union covers at least frac * P elements."""
    want = min(P, int(np.ceil(frac * P)))
    wins = []
    while _covered(wins) < want:
        need = want - _covered(wins)
        n = max(1, need // length)
        for _ in range(n):
            ln = min(length, P)
            a = int(rng.integers(0, P - ln + 1))
            wins.append((a, a + ln))
        wins = _merge(wins)
    return wins


def _window_index(windows) -> torch.Tensor:
    return torch.cat([torch.arange(a, b, dtype=torch.int64) for a, b in windows])


def _flat_window(params, offsets, idx_np: np.ndarray) -> np.ndarray:
    """Values of the unsharded flat parameter buffer at the given global indices
    (parameter p's element j sits at offsets[p] + j)."""
    out = np.empty(idx_np.size, np.float32)
    bounds = list(offsets) + [offsets[-1] + params[-1].numel()]
    for p, t in enumerate(params):
        sel = (idx_np >= bounds[p]) & (idx_np < bounds[p + 1])
        if sel.any():
            local = torch.from_numpy(idx_np[sel] - bounds[p]).to(t.device)
            out[sel] = t.reshape(-1)[local].cpu().numpy()
    return out


# ---- the oracle on slices of a window, in spawned worker processes ----------

_POOL = None


def _oracle_pool():
    """A pool of spawned workers (spawned: a forked child of a process that
    holds a CUDA context can hang)."""
    global _POOL
    if _POOL is None:
        import multiprocessing as mp
        try:
            n = len(os.sched_getaffinity(0))
        except AttributeError:
            n = os.cpu_count() or 1
        _POOL = mp.get_context("spawn").Pool(max(1, min(16, n)))
        atexit.register(_POOL.terminate)
    return _POOL


def _reduce_fn(kind):
    if kind == "bf16":
        return O.reduce_full_bf16
    if isinstance(kind, tuple):          # ("hybrid", F)
        return lambda gs: O.reduce_full_hybrid(gs, kind[1])
    return O.reduce_full


def _oracle_slice(args):
    """The windowed cycle on one slice: O.run_window over all steps, and over
    all but the last (for m before the last update)."""
    p, g_steps, hp, kind = args
    reduce = _reduce_fn(kind)
    per_step, final = O.run_window(p, g_steps, O.AdamWHyper(**hp), reduce=reduce)
    if len(g_steps) > 1:
        _, (_, m_prev, _) = O.run_window(p, g_steps[:-1], O.AdamWHyper(**hp), reduce=reduce)
    else:
        m_prev = np.zeros_like(p)
    return per_step, final, m_prev


def oracle_windows(p_win, g_win, hp: dict, kind):
    """O.run_window on the whole window, computed slice by slice in worker
    processes; returns (per-step [(gathered, G)], (p, m, v), m_prev)."""
    n = p_win.size
    parts = max(1, min(64, n // (1 << 20)))
    cuts = [n * i // parts for i in range(parts + 1)]
    jobs = [(p_win[a:b], [[g[a:b] for g in gs] for gs in g_win], hp, kind) for a, b in zip(cuts, cuts[1:])]
    res = _oracle_pool().map(_oracle_slice, jobs, chunksize=1) if parts > 1 else [_oracle_slice(jobs[0])]
    steps = len(g_win)
    per_step = [(np.concatenate([r[0][s][0] for r in res]), np.concatenate([r[0][s][1] for r in res]))
                for s in range(steps)]
    final = tuple(np.concatenate([r[1][i] for r in res]) for i in range(3))
    m_prev = np.concatenate([r[2] for r in res])
    return per_step, final, m_prev


def run_windowed(wl: workloads.Workload, unit: int = 0, steps: int | None = None, frac: float = 0.05,
                 window_len: int = 1 << 20, seed: int = 0, extra_boundaries=(),
                 bitwise: bool = True) -> Comparison:
    """Full-size unit through fsdp_step (the launch configuration the bench
    times), compared on windows: +-4096 elements around every shard and
    parameter boundary, plus, for every step, random windows drawn afresh
    whose union is at least `frac` of the unit.  Every step's outputs
    (gathered bf16 parameters, gradient shards) and the final master, m, v and
    shadow are compared on the union of all of them.  ``cmp.covered`` is the
    union's size; ``cmp.step_random`` each step's random coverage.  For an
    unfused unit, step 0 runs as the separate calls (gather, gather again,
    reduce-scatter, AdamW) with the two gathers in two buffers, so both are
    compared; later steps run through fsdp_step."""
    shapes = wl.shapes(unit)
    N, P = wl.N, wl.unit_numel(unit)
    steps = wl.steps if steps is None else steps
    hp = workloads.hyper(wl)
    lay = O.Layout(shapes, N, wl.layout)
    bounds = sorted({a for segs in lay.segments for a, _ in segs} | set(lay.offsets) | set(extra_boundaries))
    rand = [random_windows(P, frac, window_len, np.random.default_rng([seed, unit, s])) for s in range(steps)]
    windows = _merge(boundary_windows(P, bounds) + [w for r in rand for w in r])
    idx = _window_index(windows)
    idx_dev = idx.cuda()
    cmp = Comparison()
    u = B.Unit(shapes, wl.layout, N, wl.grad_dtype, wl.reshard_after_forward, replicas=wl.replicas,
               reduce_dtype=wl.reduce_dtype, gather_source=wl.gather_source,
               fuse_reduce_adamw=wl.fuse_reduce_adamw)
    try:
        params = workloads.param_tensors(wl, unit, "cuda")
        p_win = _flat_window(params, lay.offsets, idx.numpy())
        u.load(params)
        torch.cuda.synchronize()
        del params
        gdev = [torch.empty(P, dtype=wl.torch_grad_dtype(), device="cuda") for _ in range(wl.world)]
        out = torch.empty(P, dtype=torch.int16, device="cuda")
        # step 0 of an unfused unit runs as its separate calls with a buffer per
        # gather, so that the first gather is compared too (fsdp_step writes
        # both into one buffer); the other steps run through fsdp_step
        split = not wl.fuse_reduce_adamw and steps > 1
        first = torch.empty(P, dtype=torch.int16, device="cuda") if split else None
        g_win, out_win, first_win, gs_win = [], [], [], []
        for s in range(steps):
            for r in range(wl.world):
                workloads.grad_tensor(wl, unit, s, r, "cuda", out=gdev[r])
            g_win.append([grad_np(g[idx_dev]) for g in gdev])
            if split and s == 0:
                u.allgather(first)
                u.allgather(out) if wl.reshard_after_forward else out.copy_(first)
                u.reduce_scatter(gdev)
                u.adamw_step(hp)
                torch.cuda.synchronize()
                first_win.append(u16(first[idx_dev]))
            else:
                u.step(gdev, out, hp)
                torch.cuda.synchronize()
            out_win.append(u16(out[idx_dev]))
            gs_win.append(np.concatenate([u.read_global("grad", a, b - a).cpu().numpy() for a, b in windows]))
        final = {w: np.concatenate([u.read_global(w, a, b - a).cpu().numpy() for a, b in windows])
                 for w in ("param", "exp_avg", "exp_avg_sq")}
        shadow = np.concatenate([u16(u.read_global("shadow", a, b - a)) for a, b in windows])
        assert u.kernel_status() == 0, "a kernel raised its status word"
        del gdev, out, idx_dev, first
    finally:
        u.close()
    kind = ("hybrid", N) if wl.replicas > 1 else ("bf16" if wl.reduce_dtype == "bf16" else "f32")
    per_step, (p, m, v), m_prev = oracle_windows(p_win, g_win, hp, kind)
    for s, (gathered, G) in enumerate(per_step):
        if s < len(first_win):
            assert_bits_equal(first_win[s], gathered, f"step {s} first gather (windows)")
        assert_bits_equal(out_win[s], gathered, f"step {s} gathered (windows)")
        assert_bits_equal(gs_win[s], G, f"step {s} grad shard (windows)")
    G_last = per_step[-1][1] if per_step else np.zeros_like(p)
    for which, want in (("param", p), ("exp_avg", m), ("exp_avg_sq", v)):
        cmp.add(which, adamw_compare(final[which], want, f"{which} (windows)", which=which, m_prev=m_prev,
                                     g=G_last, beta1=hp["beta1"], bitwise=bitwise))
    assert_bits_equal(shadow, O.bf16_rne(final["param"]), "shadow (windows)")
    cmp.covered = int(idx.numel())
    cmp.step_random = [_covered(r) for r in rand]
    cmp.P = P
    return cmp

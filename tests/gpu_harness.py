"""Runs a workload through the C-ABI library on the GPU and the CPU oracle on
the same seeded inputs, and compares.

Gather, cast, layout and reduce-scatter outputs must be bit-identical.
AdamW state (master, m, v) must satisfy |gpu - oracle| <= 1e-6 + 1e-5*|oracle|
elementwise (max abs err 1e-6 / max rel err 1e-5, read as an allclose bound);
the harness also reports how many elements differ at all, since the kernel
evaluates the same fp32 operation sequence as the oracle.

Two modes:
* full   -- every element, step by step (units the host holds easily);
* window -- windows of global indices around every shard and parameter
            boundary plus random windows.  Every operation after the layout is
            elementwise in the global index, so the oracle computes a window
            from the initial parameters and the ranks' gradients in that window.
"""
from __future__ import annotations

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


def adamw_compare(got: np.ndarray, want: np.ndarray, what: str) -> dict:
    g = got.astype(np.float64)
    w = want.astype(np.float64)
    err = np.abs(g - w)
    ok = err <= ATOL + RTOL * np.abs(w)
    nz = np.abs(w) > 0
    stats = dict(max_abs=float(err.max(initial=0.0)),
                 max_rel=float((err[nz] / np.abs(w[nz])).max(initial=0.0)),
                 n_diff=int((got.view(np.uint32) != want.view(np.uint32)).sum()), n=int(got.size))
    assert ok.all(), f"{what}: AdamW tolerance violated: {stats}"
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


def run_full(wl: workloads.Workload, unit: int = 0, use_step: bool = False, steps: int | None = None,
             gen_device: str = "cpu", allocator=None) -> Comparison:
    """Whole-unit comparison, every element, every step."""
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
        outs = [torch.empty(P, dtype=torch.int16, device="cuda") for _ in range(2)]
        gdev = [torch.empty(P, dtype=wl.torch_grad_dtype(), device="cuda") for _ in range(wl.world)]
        for s in range(steps):
            for r in range(wl.world):
                if gen_device == "cuda":
                    workloads.grad_tensor(wl, unit, s, r, "cuda", out=gdev[r])
                else:
                    gdev[r].copy_(workloads.grad_tensor(wl, unit, s, r, "cpu"))
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
                cmp.add((which, k), adamw_compare(got, want, f"{which} rank {k}"))
            assert_bits_equal(u.get_state("grad", k).cpu().numpy(), orc.grad[k], f"final grad shard rank {k}")
            # the shadow is the cast of the GPU's own master (checked bitwise against that)
            assert_bits_equal(u16(u.get_state("shadow", k)), O.bf16_rne(u.get_state("param", k).cpu().numpy()),
                              f"shadow rank {k}")
        assert u.kernel_status() == 0, "a kernel raised its status word"
    finally:
        u.close()
    return cmp


def choose_windows(P: int, boundaries, half: int = 4096, n_random: int = 16, random_len: int = 1 << 16,
                   seed: int = 0):
    rng = np.random.default_rng(seed)
    iv = [(max(0, b - half), min(P, b + half)) for b in boundaries]
    for _ in range(n_random):
        a = int(rng.integers(0, max(1, P - random_len)))
        iv.append((a, min(P, a + random_len)))
    iv.append((max(0, P - half), P))
    iv.sort()
    merged = []
    for a, b in iv:
        if b <= a:
            continue
        if merged and a <= merged[-1][1]:
            merged[-1] = (merged[-1][0], max(merged[-1][1], b))
        else:
            merged.append((a, b))
    return merged


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


def run_windowed(wl: workloads.Workload, unit: int = 0, steps: int | None = None, n_random: int = 16,
                 seed: int = 0, extra_boundaries=()) -> Comparison:
    """Full-size unit through fsdp_step (the launch configuration the bench
    times), compared on windows of global indices."""
    shapes = wl.shapes(unit)
    N, P = wl.N, wl.unit_numel(unit)
    steps = wl.steps if steps is None else steps
    hp = workloads.hyper(wl)
    lay = O.Layout(shapes, N, wl.layout)
    bounds = sorted({a for segs in lay.segments for a, _ in segs} | set(lay.offsets) | set(extra_boundaries))
    windows = choose_windows(P, bounds, n_random=n_random, seed=seed)
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
        g_win, out_win, gs_win = [], [], []
        for s in range(steps):
            for r in range(wl.world):
                workloads.grad_tensor(wl, unit, s, r, "cuda", out=gdev[r])
            g_win.append([grad_np(g[idx_dev]) for g in gdev])
            u.step(gdev, out, hp)
            torch.cuda.synchronize()
            out_win.append(u16(out[idx_dev]))
            gs_win.append(np.concatenate([u.read_global("grad", a, b - a).cpu().numpy() for a, b in windows]))
        final = {w: np.concatenate([u.read_global(w, a, b - a).cpu().numpy() for a, b in windows])
                 for w in ("param", "exp_avg", "exp_avg_sq")}
        shadow = np.concatenate([u16(u.read_global("shadow", a, b - a)) for a, b in windows])
        assert u.kernel_status() == 0, "a kernel raised its status word"
        del gdev, out
    finally:
        u.close()
    if wl.replicas > 1:
        def reduce(gs):
            return O.reduce_full_hybrid(gs, N)
    elif wl.reduce_dtype == "bf16":
        reduce = O.reduce_full_bf16
    else:
        reduce = O.reduce_full
    per_step, (p, m, v) = O.run_window(p_win, g_win, O.AdamWHyper(**hp), reduce=reduce)
    for s, (gathered, G) in enumerate(per_step):
        assert_bits_equal(out_win[s], gathered, f"step {s} gathered (windows)")
        assert_bits_equal(gs_win[s], G, f"step {s} grad shard (windows)")
    for which, want in (("param", p), ("exp_avg", m), ("exp_avg_sq", v)):
        cmp.add(which, adamw_compare(final[which], want, f"{which} (windows)"))
    assert_bits_equal(shadow, O.bf16_rne(final["param"]), "shadow (windows)")
    cmp.covered = int(idx.numel())
    return cmp

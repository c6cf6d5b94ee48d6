"""Whole-unit pins: brute force on tiny units, the pages' invariants, memory."""
import os

import numpy as np
import pytest
import torch

from fully_sharded_unit_gb300 import workloads
from oracle import brute
from oracle import fsdp_oracle as O


def _run_both(shapes, N, layout, params, grads_steps, hp, raf=True):
    u = O.UnitOracle(shapes, N, layout, hp, reshard_after_forward=raf)
    u.load(params)
    gathers, gshards = [], []
    for grads in grads_steps:
        gathers.append(u.step(grads))
        gshards.append([g.copy() for g in u.grad])
    b = brute.brute_unit_run(shapes, N, layout, [np.asarray(p, np.float32).reshape(-1).tolist() for p in params],
                             [[g.tolist() for g in gs] for gs in grads_steps],
                             dict(lr=hp.lr, beta1=hp.beta1, beta2=hp.beta2, eps=hp.eps,
                                  weight_decay=hp.weight_decay), raf=raf)
    return u, gathers, gshards, b


def _assert_same(u, gathers, gshards, b):
    for s in range(len(gathers)):
        assert len(gathers[s]) == len(b["gathers"][s])
        for g_or, g_br in zip(gathers[s], b["gathers"][s]):
            assert g_or.tolist() == g_br
        for k in range(u.N):
            assert gshards[s][k].tolist() == b["gshards"][s][k]
    for k in range(u.N):
        assert u.master[k].tolist() == b["master"][k]
        assert u.m[k].tolist() == b["m"][k]
        assert u.v[k].tolist() == b["v"][k]


def test_tiny_config_bruteforce():
    wl = workloads.get("tiny_flat")
    params = [t.numpy() for t in workloads.param_tensors(wl, 0)]
    grads = [[workloads.grad_tensor(wl, 0, s, r).numpy() for r in range(wl.N)] for s in range(wl.steps)]
    hp = O.AdamWHyper(**workloads.hyper(wl))
    _assert_same(*_run_both(wl.shapes(0), wl.N, wl.layout, params, grads, hp))


@pytest.mark.parametrize("layout", ["flat", "dim0"])
@pytest.mark.parametrize("N", [1, 3, 7, 16])
def test_odd_units_bruteforce(layout, N):
    rng = np.random.default_rng(N)
    shapes = [(7, 13), (1,), (5,), (3, 2, 2)]
    params = [rng.uniform(-0.1, 0.1, s).astype(np.float32) for s in shapes]
    P = sum(p.size for p in params)
    grads = [[rng.normal(0, 1e-2, P).astype(np.float32) for _ in range(N)] for _ in range(3)]
    hp = O.AdamWHyper(lr=1e-2, weight_decay=0.1)
    _assert_same(*_run_both(shapes, N, layout, params, grads, hp, raf=(N % 2 == 1)))


def test_fewer_elements_than_ranks_bruteforce():
    """15 elements over 16 ranks (FLAT): rank 0 owns nothing."""
    shapes = [(3, 4), (3,)]
    rng = np.random.default_rng(0)
    params = [rng.normal(0, 1, s).astype(np.float32) for s in shapes]
    grads = [[rng.normal(0, 1, 15).astype(np.float32) for _ in range(16)] for _ in range(2)]
    u, *_ = out = _run_both(shapes, 16, "flat", params, grads, O.AdamWHyper())
    _assert_same(*out)
    assert u.lay.shard_len(0) == 0 and all(u.lay.shard_len(k) == 1 for k in range(1, 16))


@pytest.mark.parametrize("layout", ["flat", "dim0"])
def test_concat_of_shards_is_the_flat_parameter(layout):
    rng = np.random.default_rng(1)
    shapes = [(50, 9), (9,), (1,), (17, 5)]
    params = [rng.normal(0, 1, s).astype(np.float32) for s in shapes]
    flat = O.flatten(params)
    for N in (1, 2, 5, 8, 64):
        lay = O.Layout(shapes, N, layout)
        sh = O.shard(flat, lay)
        assert sum(s.size for s in sh) == flat.size
        assert np.array_equal(O.unshard(sh, lay), flat)
        if layout == "flat":
            assert np.array_equal(np.concatenate(sh), flat)   # rank order = flat order
        # gather(shard(x)) == RNE(x)
        assert np.array_equal(O.allgather_cast(sh, lay), O.bf16_rne(flat))


def test_gather_of_bf16_representable_values_is_their_top_half():
    b = np.random.default_rng(2).integers(0, 0x7F00, 999).astype(np.uint16)
    x = O.bf16_to_f32(b)
    lay = O.Layout([(999,)], 7, "flat")
    assert np.array_equal(O.allgather_cast(O.shard(x, lay), lay), b)


def test_sharded_adamw_equals_unsharded_and_layouts_agree():
    """AdamW is elementwise: the sharded run reassembled equals the N=1 run
    given the same reduced gradients, bit for bit, for FLAT and DIM0."""
    rng = np.random.default_rng(3)
    shapes = [(33, 10), (10,), (7, 13), (1,)]
    params = [rng.normal(0, 0.02, s).astype(np.float32) for s in shapes]
    P = sum(p.size for p in params)
    N = 7
    grads = [[rng.normal(0, 1e-3, P).astype(np.float32) for _ in range(N)] for _ in range(4)]
    hp = O.AdamWHyper()
    runs = {}
    for layout in ("flat", "dim0"):
        u = O.UnitOracle(shapes, N, layout, hp)
        u.load(params)
        for g in grads:
            u.step(g)
        runs[layout] = {w: u.full(w) for w in ("master", "m", "v", "grad")}
    one = O.UnitOracle(shapes, 1, "flat", hp)
    one.load(params)
    for g in grads:
        one.reduce_scatter([O.reduce_full(g)])   # the reduced gradient, unsharded
        one.adamw_step()
    for w in ("master", "m", "v", "grad"):
        assert np.array_equal(runs["flat"][w], runs["dim0"][w])
        assert np.array_equal(runs["flat"][w], one.full(w))


def test_window_run_equals_unit_run():
    rng = np.random.default_rng(4)
    shapes = [(40, 11), (11,)]
    params = [rng.normal(0, 0.02, s).astype(np.float32) for s in shapes]
    P = 451
    N = 3
    grads = [[rng.normal(0, 1e-3, P).astype(np.float32) for _ in range(N)] for _ in range(3)]
    hp = O.AdamWHyper()
    u = O.UnitOracle(shapes, N, "dim0", hp)
    u.load(params)
    outs = [u.step(g) for g in grads]
    a, b = 100, 300
    flat = O.flatten(params)
    per_step, (p, m, v) = O.run_window(flat[a:b], [[g[a:b] for g in gs] for gs in grads], hp)
    for s, (gathered, G) in enumerate(per_step):
        assert np.array_equal(gathered, outs[s][0][a:b])
    assert np.array_equal(p, u.full("master")[a:b])
    assert np.array_equal(m, u.full("m")[a:b])
    assert np.array_equal(v, u.full("v")[a:b])


def _golden(name):
    path = os.path.join(os.path.dirname(__file__), "golden", name)
    return [l.split() for l in open(path) if l.strip() and not l.startswith("#")]


def test_memory_examples_printed_on_pages():
    rows = {r[0]: r for r in _golden("memory_examples.txt")}
    _, params, N, total, per_rank = rows["mbrenndoerfer_13b"]
    params, N = int(params), int(N)
    u = O.UnitOracle([(params,)], N, "flat")
    per = [u.memory_bytes(k) for k in range(N)]
    sharded = [d["param"] + d["grad"] + d["adam"] for d in per]
    assert sum(sharded) == float(total)
    assert all(s == float(per_rank) for s in sharded)
    _, psi, N, ddp_gib, fsdp_gib = rows["gpt2_large"]
    psi, N = int(psi), int(N)
    one = O.UnitOracle([(psi,)], 1, "flat").memory_bytes(0)
    assert abs((one["param"] + one["grad"] + one["adam"]) / 2**30 - float(ddp_gib)) < 0.05
    u = O.UnitOracle([(psi,)], N, "flat")
    d = u.memory_bytes(0)
    assert abs((d["param"] + d["adam"]) / 2**30 - float(fsdp_gib)) < 0.005


@pytest.mark.parametrize("replicas,reduce_dtype", [(2, "f32"), (3, "f32"), (1, "bf16")])
def test_window_run_equals_unit_run_for_hybrid_and_bf16(replicas, reduce_dtype):
    rng = np.random.default_rng(5)
    shapes = [(40, 11), (11,)]
    params = [rng.normal(0, 0.02, s).astype(np.float32) for s in shapes]
    N, P = 3, 451
    W = N * replicas
    grads = [[rng.normal(0, 1e-3, P).astype(np.float32) for _ in range(W)] for _ in range(3)]
    hp = O.AdamWHyper()
    u = O.UnitOracle(shapes, N, "flat", hp, replicas=replicas, reduce_dtype=reduce_dtype)
    u.load(params)
    outs = [u.step(g) for g in grads]
    if replicas > 1:
        def reduce(gs):
            return O.reduce_full_hybrid(gs, N)
    else:
        reduce = O.reduce_full_bf16
    a, b = 50, 400
    per_step, (p, m, v) = O.run_window(O.flatten(params)[a:b], [[g[a:b] for g in gs] for gs in grads], hp,
                                       reduce=reduce)
    for s, (gathered, G) in enumerate(per_step):
        assert np.array_equal(gathered, outs[s][0][a:b])
    assert np.array_equal(p, u.full("master")[a:b])
    assert np.array_equal(v, u.full("v")[a:b])

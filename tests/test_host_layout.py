"""The library's host-side layout tables (no GPU): equal to the oracle's layout,
aligned arenas, and host-side argument checks."""
import ctypes

import numpy as np
import pytest
import torch

from conftest import library
from fully_sharded_unit_gb300 import binding as B
from fully_sharded_unit_gb300 import workloads
from oracle import fsdp_oracle as O

SHAPE_SETS = [
    [(7, 13), (1,), (5,), (3, 2, 2)],
    [(64, 48), (64,)],
    [()],
    [(0, 4), (6,), (0,)],
    [(1,)],
    [(100003,)],
]


def _check_against_oracle(shapes, N, layout):
    P, segs = B.fsdp_plan_layout(shapes, layout, N)
    lay = O.Layout([tuple(s) for s in shapes], N, layout)
    assert P == lay.P
    by_rank = [[] for _ in range(N)]
    for s in segs:
        by_rank[s.rank].append(s)
    for k in range(N):
        got = [(s.global_off, s.global_off + s.len) for s in by_rank[k]]
        assert got == [tuple(x) for x in lay.segments[k]], (shapes, N, layout, k)
        pos = 0
        prev_end = 0
        for s in by_rank[k]:
            assert s.shard_off == pos                       # packed shard order
            pos += s.len
            assert s.arena_off % 32 == s.global_off % 32    # alignment congruence
            assert s.arena_off >= prev_end and s.arena_off - prev_end < 32
            prev_end = s.arena_off + s.len
            if layout != "dim0":
                assert s.param == -1
        assert pos == lay.shard_len(k)
    # segments listed rank-major
    assert [s.rank for s in segs] == sorted(s.rank for s in segs)


@pytest.mark.parametrize("N", [1, 2, 3, 7, 8, 16, 64, 1024])
@pytest.mark.parametrize("layout", ["flat", "dim0", "flat_padded"])
def test_plan_matches_oracle_random_shapes(N, layout):
    library()
    for shapes in SHAPE_SETS:
        if sum(O.numel(s) for s in shapes) == 0:
            continue
        _check_against_oracle(shapes, N, layout)


@pytest.mark.parametrize("name", sorted(workloads.WORKLOADS))
def test_plan_matches_oracle_workloads(name):
    library()
    wl = workloads.get(name)
    _check_against_oracle(wl.shapes(0), wl.N, wl.layout)


@pytest.mark.parametrize("name", ["ragged_flat_n7", "ragged_flat_n64", "tiny_flat", "ragged_mini_flat_n3"])
def test_padded_plan_matches_oracle_workloads(name):
    library()
    wl = workloads.get(name)
    _check_against_oracle(wl.shapes(0), wl.N, "flat_padded")


def test_plan_rejects_bad_arguments():
    library()
    for shapes, layout, N in [([(4,)], "flat", 0), ([(4,)], "flat", 1025), ([(4,)], 7, 2),
                              ([(0,)], "flat", 2), ([(-1, 3)], "dim0", 2)]:
        with pytest.raises(B.FsdpError) as e:
            B.fsdp_plan_layout(shapes, layout, N)
        assert e.value.code == B.FSDP_E_INVALID_ARG
    nd = (ctypes.c_int * 1)(9)
    dims = (ctypes.c_int64 * 9)(*([1] * 9))
    assert B.lib().fsdp_plan_layout(1, nd, dims, 0, 2, None, None, None, 0) == B.FSDP_E_INVALID_ARG
    # a too-small output array is reported with the needed count
    nd = (ctypes.c_int * 1)(1)
    dims = (ctypes.c_int64 * 1)(100)
    ns = ctypes.c_int64()
    segs = (B.Segment * 1)()
    rc = B.lib().fsdp_plan_layout(1, nd, dims, 0, 4, None, ctypes.byref(ns), segs, 1)
    assert rc == B.FSDP_E_CAPACITY and ns.value == 4


def test_create_rejects_bad_arguments_before_touching_the_gpu():
    library()
    for kw in [dict(shapes=[(4,)], layout="flat", num_ranks=0),
               dict(shapes=[(0,)], layout="dim0", num_ranks=2),
               dict(shapes=[(4,)], layout="flat", num_ranks=2, grad_dtype=5),
               dict(shapes=[(4,)], layout="flat", num_ranks=2, replicas=-1),
               dict(shapes=[(4,)], layout="flat", num_ranks=64, replicas=17),
               dict(shapes=[(4,)], layout="flat", num_ranks=2, replicas=2, reduce_dtype="bf16"),
               dict(shapes=[(4,)], layout="flat", num_ranks=2, gather_source=7)]:
        with pytest.raises(B.FsdpError) as e:
            B.fsdp_unit_create(**kw)
        assert e.value.code == B.FSDP_E_INVALID_ARG


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU error path")
def test_create_without_a_gpu_fails_loudly():
    library()
    with pytest.raises(B.FsdpError) as e:
        B.fsdp_unit_create([(8,)], "flat", 2)
    assert e.value.code == B.FSDP_E_CUDA


def test_null_unit_is_rejected():
    library()
    assert B.lib().fsdp_allgather(None, None, None) == B.FSDP_E_INVALID_ARG
    assert B.lib().fsdp_step(None, None, None, None, None) == B.FSDP_E_INVALID_ARG
    assert B.lib().fsdp_unit_destroy(None) == B.FSDP_OK


def test_new_entry_points_reject_bad_arguments_on_the_host():
    """Checks that run before any CUDA call, so they hold without a GPU."""
    import ctypes as C
    library()
    L = B.lib()
    hp = B.AdamWHp(1e-3, 0.9, 0.999, 1e-8, 0.01)
    assert L.fsdp_adamw_device_steps(None, C.byref(hp), 4, None) == B.FSDP_E_INVALID_ARG
    assert L.fsdp_adamw_device_status(None, None, None, None) == B.FSDP_E_INVALID_ARG
    assert L.fsdp_read_arena(None, 0, 0, None, None, None) == B.FSDP_E_INVALID_ARG
    assert L.fsdp_reduce_scatter_ex(None, None, None, None) == B.FSDP_E_INVALID_ARG
    assert L.fsdp_zero_grad(None, None) == B.FSDP_E_INVALID_ARG
    assert L.fsdp_host_device_pointer(None, None) == B.FSDP_E_INVALID_ARG
    d = C.c_void_p()
    assert L.fsdp_host_device_pointer(None, C.byref(d)) == B.FSDP_E_INVALID_ARG
    assert B.fsdp_last_error()          # every failure leaves a reason

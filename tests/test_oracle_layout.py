"""Pins for the oracle's layout: FLAT floor boundaries and DIM0 torch.chunk shards."""
import os

import numpy as np
import pytest

import pins
from fully_sharded_unit_gb300 import workloads
from oracle import brute
from oracle import fsdp_oracle as O


def test_flat_ranges_match_counting():
    pins.check_flat_ranges(O.flat_shard_range)


def test_flat_properties_stated_on_pages():
    cases = [(P, N) for P in (1, 2, 15, 16, 100, 3136, 7087872, 70886492, 1812099072)
             for N in (1, 2, 3, 4, 7, 8, 16, 64, 1000)]
    pins.check_flat_properties(O.flat_shard_range, cases)


RANDOM_SHAPES = [
    [(7, 13), (1,), (5,), (3, 2, 2)],
    [(1,), (1,)],
    [(9, 1), (2, 3)],
    [(64, 48), (64,)],
    [()],
    [(0, 4), (6,)],
]


@pytest.mark.parametrize("N", [1, 2, 3, 7, 8, 16, 64])
def test_dim0_matches_torch_chunk(N):
    wl3 = workloads.get("gpt2_large_dim0")
    wl5 = workloads.get("ragged_dim0_n7")
    for shapes in [wl3.shapes(0), wl5.shapes(0)] + RANDOM_SHAPES:
        pins.check_dim0_vs_torch_chunk(O.rank_segments, O.param_offsets, list(shapes), N)


@pytest.mark.parametrize("N", [1, 2, 3, 7, 16, 64])
def test_dim0_matches_bruteforce(N):
    for shapes in RANDOM_SHAPES[:4] + [workloads.get("ragged_mini_dim0_n7").shapes(0)]:
        pins.check_dim0_vs_brute(O.rank_segments, list(shapes), N)


@pytest.mark.parametrize("name", sorted(workloads.WORKLOADS))
def test_every_workload_layout_tiles_the_unit(name):
    wl = workloads.get(name)
    lay = O.Layout(wl.shapes(0), wl.N, wl.layout)
    cover = []
    for k in range(wl.N):
        cover.extend(lay.segments[k])
    cover.sort()
    pos = 0
    for a, b in cover:
        assert a == pos and b > a
        pos = b
    assert pos == lay.P == wl.unit_numel(0)


def test_ragged_dim0_chunks_as_described():
    """The stress unit at N=64: a 1-element parameter lives on rank 0 only and
    the 7-row matrix on ranks 0..6 (one row each)."""
    wl = workloads.get("ragged_dim0_n64")
    shapes = wl.shapes(0)
    offs, P = O.param_offsets(shapes)
    owners_small = [k for k in range(64) for a, b in O.rank_segments(shapes, 64, "dim0", k)
                    if offs[4] <= a < offs[5]]
    assert owners_small == list(range(7))
    owners_scalar = [k for k in range(64) for a, b in O.rank_segments(shapes, 64, "dim0", k) if a == offs[5]]
    assert owners_scalar == [0]


def test_fig3_padded_example():
    """Figure 3 of the FSDP paper (padded-equal-chunk variant): 15 elements over
    16 ranks, one element each, the pad on the last rank."""
    path = os.path.join(os.path.dirname(__file__), "golden", "fig3_padded_16ranks.txt")
    line = [l for l in open(path) if l.strip() and not l.startswith("#")][0].split()
    wshape = tuple(int(x) for x in line[0].split("x"))
    bias = int(line[1])
    N, per_rank, pad_elems, pad_rank = (int(x) for x in line[2:6])
    P = O.numel(wshape) + bias
    total_pad = 0
    for k in range(N):
        a, b, pad = O.padded_shard_range(P, N, k)
        assert (b - a) + pad == per_rank
        total_pad += pad
        if pad:
            assert k == pad_rank
    assert total_pad == pad_elems


def test_workload_sizes():
    assert workloads.get("tiny_flat").unit_numel(0) == 3136
    assert workloads.get("gpt2_small_flat").unit_numel(0) == 7_087_872
    assert workloads.get("gpt2_large_dim0").unit_numel(0) == 19_677_440
    assert workloads.get("mingpt175b_flat").unit_numel(0) == 1_812_099_072
    assert workloads.get("ragged_flat_n7").unit_numel(0) == 70_886_492

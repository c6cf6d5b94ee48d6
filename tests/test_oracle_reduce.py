"""Pins for the oracle's reduce-scatter."""
import numpy as np

import pins
from oracle import fsdp_oracle as O


def test_reduce_integer_closed_form():
    pins.check_reduce_integer_closed_form(O.reduce_full)


def test_reduce_within_fp64_bound():
    pins.check_reduce_fp64_bound(O.reduce_full)


def test_reduce_special_cases():
    pins.check_reduce_special(O.reduce_full)


def test_reduce_scatter_slices_match_reduced_gradient():
    """Rank k receives the slice of the summed gradient that matches its shard,
    checked element by element against the reduced full gradient."""
    rng = np.random.default_rng(0)
    shapes = [(31, 7), (5,), (1,), (13, 3)]
    for layout in ("flat", "dim0"):
        for N in (1, 3, 8, 40):
            lay = O.Layout(shapes, N, layout)
            grads = [rng.normal(0, 1, lay.P).astype(np.float32) for _ in range(N)]
            G = O.reduce_full(grads)
            shards = O.reduce_scatter(grads, lay)
            for k in range(N):
                got = shards[k]
                pos = 0
                for a, b in lay.segments[k]:
                    for i in range(a, b):
                        assert got[pos] == G[i]
                        pos += 1
                assert pos == got.size

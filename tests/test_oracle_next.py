"""Pins for the oracle's next-row functions: padded equal-chunk layout, hybrid
(2-D) reduction, bf16 reduction, unscale / accumulation / found-non-finite."""
import numpy as np
import pytest

import pins
from oracle import brute
from oracle import fsdp_oracle as O


def test_padded_layout_vs_torch_chunk():
    pins.check_padded_vs_torch_chunk(O.padded_shard_range,
                                     [(P, N) for P in (1, 5, 15, 16, 100, 3136, 70886492) for N in (1, 2, 3, 4, 7, 16, 64)])


def test_padded_layout_vs_brute():
    pins.check_padded_vs_brute(O.padded_shard_range)


def test_padded_layout_segments_tile_the_unit():
    for N in (1, 7, 16, 64):
        lay = O.Layout([(7, 13), (1,), (100,)], N, "flat_padded")
        cover = sorted(x for k in range(N) for x in lay.segments[k])
        pos = 0
        for a, b in cover:
            assert a == pos
            pos = b
        assert pos == lay.P
        assert sum(lay.padding(k) for k in range(N)) <= N - 1


def test_hybrid_reduction():
    pins.check_hybrid_reduce(O.reduce_full_hybrid, O.reduce_full)


def test_bf16_reduction_vs_torch():
    pins.check_bf16_reduce_vs_torch(O.reduce_full_bf16)


def test_bf16_reduction_vs_exact_rounding():
    pins.check_bf16_reduce_exact(O.reduce_full_bf16)


def test_reduce_update():
    pins.check_reduce_update(O.reduce_update)


@pytest.mark.parametrize("W,F,rd", [(8, 2, "f32"), (6, 3, "f32"), (5, 5, "f32"), (4, 4, "bf16"), (3, 3, "bf16")])
def test_reductions_vs_brute(W, F, rd):
    rng = np.random.default_rng(W * 10 + F)
    grads = [rng.normal(0, 1e-2, 200).astype(np.float32) for _ in range(W)]
    old = rng.normal(0, 1e-2, 200).astype(np.float32)
    want, want_found = brute.brute_reduce([g.tolist() for g in grads], F, rd, old.tolist(), 0.5)
    G = O.reduce_full_bf16(grads) if rd == "bf16" else O.reduce_full_hybrid(grads, F)
    got, found = O.reduce_update(G, old, 0.5)
    assert got.tolist() == want and found == want_found


def test_unit_oracle_hybrid_and_accumulation_vs_brute():
    """A hybrid unit (F = 3 shards, 2 replicas) with two accumulated
    micro-batches, element by element against brute force."""
    rng = np.random.default_rng(9)
    shapes = [(5, 7), (3,)]
    params = [rng.normal(0, 0.1, s).astype(np.float32) for s in shapes]
    u = O.UnitOracle(shapes, 3, "flat", replicas=2)
    u.load(params)
    mb = [[rng.normal(0, 1e-2, 38).astype(np.float32) for _ in range(6)] for _ in range(2)]
    u.reduce_scatter(mb[0])
    found = u.reduce_scatter(mb[1], accumulate=True, inv_scale=0.5)
    first, _ = brute.brute_reduce([g.tolist() for g in mb[0]], 3)
    want, want_found = brute.brute_reduce([g.tolist() for g in mb[1]], 3, "f32", first, 0.5)
    assert u.full("grad").tolist() == want and found == want_found

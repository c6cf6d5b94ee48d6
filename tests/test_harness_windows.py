"""The windowed comparison's own machinery, on the CPU: the random windows
cover what they claim, and the oracle computed slice by slice in worker
processes equals the oracle run once over the whole window, bit for bit (the
split is exact because every element of the cycle is independent)."""
import numpy as np
import pytest

from oracle import fsdp_oracle as O

import gpu_harness as H


@pytest.mark.parametrize("P,frac,length", [(10_000_000, 0.05, 1 << 20), (3_000, 0.5, 700), (100, 1.0, 64),
                                           (1 << 22, 0.05, 1 << 16)])
def test_random_windows_cover_the_fraction(P, frac, length):
    w = H.random_windows(P, frac, length, np.random.default_rng(1))
    assert all(0 <= a < b <= P for a, b in w)
    assert all(b1 < a2 for (_, b1), (a2, _) in zip(w, w[1:])), "windows overlap or touch after merging"
    assert H._covered(w) >= min(P, frac * P)


def test_boundary_windows_hold_every_boundary():
    P = 1_000_000
    bounds = [0, 5, 4095, 500_000, 999_999]
    w = H.boundary_windows(P, bounds, half=4096)
    for b in bounds:
        assert any(a <= b < e for a, e in w)
    assert w[-1][1] == P


def _grads(rng, W, n, bf16):
    g = [(rng.standard_normal(n) * 1e-3).astype(np.float32) for _ in range(W)]
    return [O.bf16_rne(x) for x in g] if bf16 else g


@pytest.mark.parametrize("kind,W,bf16", [("f32", 8, True), ("bf16", 4, False), (("hybrid", 3), 6, False)])
def test_pooled_oracle_equals_one_run(kind, W, bf16):
    rng = np.random.default_rng(7)
    n = (2 << 20) + 77                       # at least two slices, and a ragged one
    p = (rng.standard_normal(n) * 0.02).astype(np.float32)
    g_steps = [_grads(rng, W, n, bf16) for _ in range(3)]
    hp = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
    per_step, (pp, m, v), m_prev = H.oracle_windows(p, g_steps, hp, kind)
    reduce = H._reduce_fn(kind)
    want_steps, (wp, wm, wv) = O.run_window(p, g_steps, O.AdamWHyper(**hp), reduce=reduce)
    _, (_, wm_prev, _) = O.run_window(p, g_steps[:-1], O.AdamWHyper(**hp), reduce=reduce)
    for (a, b), (c, d) in zip(per_step, want_steps):
        assert np.array_equal(a, c) and np.array_equal(b.view(np.uint32), d.view(np.uint32))
    for a, b in ((pp, wp), (m, wm), (v, wv), (m_prev, wm_prev)):
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))

"""Each pin must catch a plausible mistake planted in a copy of the oracle."""
import numpy as np
import pytest

import pins
from oracle import fsdp_oracle as O

HP = O.AdamWHyper()


def _fails(fn, *a, **k):
    with pytest.raises(AssertionError):
        fn(*a, **k)


def test_flat_ceil_boundaries_caught():
    def ceil_range(P, N, k):
        return -(-(k * P) // N), -(-((k + 1) * P) // N)
    _fails(pins.check_flat_ranges, ceil_range, 20, 20)
    _fails(pins.check_flat_properties, ceil_range, [(7, 2), (15, 16)])


def test_flat_off_by_one_caught():
    def r(P, N, k):
        return (k * P) // N, ((k + 1) * P) // N - (1 if k == N - 1 else 0)
    _fails(pins.check_flat_ranges, r, 10, 10)


def test_dim0_floor_chunk_caught():
    def segs(shapes, N, layout, k):
        offs, _ = O.param_offsets(shapes)
        out = []
        for s, off in zip(shapes, offs):
            m, r = O.rows_and_row_len(s)
            c = max(1, m // N)                  # floor instead of ceil
            a, b = min(k * c, m), (m if k == N - 1 else min((k + 1) * c, m))
            if b > a:
                out.append((off + a * r, off + b * r))
        return out
    _fails(pins.check_dim0_vs_torch_chunk, segs, O.param_offsets, [(7, 13), (5,)], 3)


def test_cast_truncation_caught():
    def trunc(x):
        return (np.ascontiguousarray(x, np.float32).view(np.uint32) >> 16).astype(np.uint16)
    _fails(pins.check_cast_vs_torch, trunc, pins.structured_patterns())


def test_cast_ties_away_caught():
    def away(x):
        u = np.ascontiguousarray(x, np.float32).view(np.uint32)
        r = ((u + np.uint32(0x8000)) >> 16).astype(np.uint16)
        nan = np.isnan(x)
        r[nan] = (u[nan] >> 16).astype(np.uint16) | 0x40
        return r
    _fails(pins.check_cast_vs_torch, away, pins.structured_patterns())


def test_reduce_wrong_divisor_caught():
    def rf(grads):
        return (O.reduce_full(grads) * np.float32(len(grads)) / np.float32(max(1, len(grads) - 1))).astype(np.float32)
    _fails(pins.check_reduce_integer_closed_form, rf, range(2, 5))


def test_reduce_from_positive_zero_caught():
    def rf(grads):
        acc = np.zeros_like(O.upcast_grad(grads[0]))
        for g in grads:
            acc = (acc + O.upcast_grad(g)).astype(np.float32)
        return (acc / np.float32(len(grads))).astype(np.float32)
    _fails(pins.check_reduce_special, rf)


def test_reduce_reverse_order_caught():
    def rf(grads):
        return O.reduce_full(list(reversed(grads)))
    _fails(pins.check_reduce_special, rf)


def test_adamw_missing_bias_correction_caught():
    def upd(p, g, m, v, t, hp):
        c = O.adamw_scalars(t, hp)
        p1 = p * c["decay"]
        m1 = c["b1"] * m + c["c1"] * g
        v1 = c["b2"] * v + c["c2"] * (g * g)
        p2 = p1 - np.float32(hp.lr) * (m1 / (np.sqrt(v1) + c["eps"]))
        return p2.astype(np.float32), m1.astype(np.float32), v1.astype(np.float32)
    _fails(pins.check_adamw_vs_torch, upd, HP)
    _fails(pins.check_adamw_first_step_closed_form, upd, HP)


def test_adamw_weight_decay_sign_caught():
    def upd(p, g, m, v, t, hp):
        p2, m1, v1 = O.adamw_update(p, g, m, v, t, hp)
        return (p2 + np.float32(2 * hp.lr * hp.weight_decay) * p).astype(np.float32), m1, v1
    _fails(pins.check_adamw_vs_torch, upd, HP)
    _fails(pins.check_adamw_zero_grad, upd, HP)


def test_adamw_swapped_betas_caught():
    def upd(p, g, m, v, t, hp):
        return O.adamw_update(p, g, m, v, t, O.AdamWHyper(hp.lr, hp.beta2, hp.beta1, hp.eps, hp.weight_decay))
    _fails(pins.check_adamw_vs_torch, upd, HP)


def test_adamw_eps_inside_sqrt_caught():
    def upd(p, g, m, v, t, hp):
        c = O.adamw_scalars(t, hp)
        p1 = p * c["decay"]
        m1 = c["b1"] * m + c["c1"] * g
        v1 = c["b2"] * v + c["c2"] * (g * g)
        p2 = p1 - c["step"] * (m1 / np.sqrt(v1 / c["bc2"] + c["eps"]))
        return p2.astype(np.float32), m1.astype(np.float32), v1.astype(np.float32)
    _fails(pins.check_adamw_vs_torch, upd, HP)


def test_padded_floor_instead_of_ceil_caught():
    def r(P, N, k):
        a, b = O.flat_shard_range(P, N, k)
        return a, b, 0
    _fails(pins.check_padded_vs_torch_chunk, r, [(15, 16), (5, 4)])


def test_hybrid_flat_fold_caught():
    _fails(pins.check_hybrid_reduce, lambda grads, F: O.reduce_full(grads), O.reduce_full)


def test_hybrid_divide_by_group_size_caught():
    def r(grads, F):
        return (O.reduce_full_hybrid(grads, F) * np.float32(len(grads)) / np.float32(F)).astype(np.float32)
    _fails(pins.check_hybrid_reduce, r, O.reduce_full)


def test_bf16_reduce_in_fp32_caught():
    def r(grads):
        return O.bf16_to_f32(O.bf16_rne(O.reduce_full(grads)))
    _fails(pins.check_bf16_reduce_vs_torch, r)
    _fails(pins.check_bf16_reduce_exact, r)


def test_bf16_reduce_unrounded_quotient_caught():
    def r(grads):
        acc = O.bf16_to_f32(O.bf16_rne(O.upcast_grad(grads[0])))
        for g in grads[1:]:
            acc = O.bf16_to_f32(O.bf16_rne((acc + O.bf16_to_f32(O.bf16_rne(O.upcast_grad(g)))).astype(np.float32)))
        return (acc / np.float32(len(grads))).astype(np.float32)
    _fails(pins.check_bf16_reduce_exact, r)


def test_bf16_reduce_truncating_partial_sums_caught():
    def trunc(x):
        return (np.asarray(x, np.float32).view(np.uint32) & np.uint32(0xFFFF0000)).view(np.float32)
    def r(grads):
        acc = O.bf16_to_f32(O.bf16_rne(O.upcast_grad(grads[0])))
        for g in grads[1:]:
            acc = trunc((acc + O.bf16_to_f32(O.bf16_rne(O.upcast_grad(g)))).astype(np.float32))
        return O.bf16_to_f32(O.bf16_rne((acc / np.float32(len(grads))).astype(np.float32)))
    _fails(pins.check_bf16_reduce_exact, r)


def test_accumulate_overwrites_caught():
    def upd(G, old=None, inv_scale=1.0):
        return O.reduce_update(G, None, inv_scale)
    _fails(pins.check_reduce_update, upd)


def test_found_flag_misses_nan_caught():
    def upd(G, old=None, inv_scale=1.0):
        v, _ = O.reduce_update(G, old, inv_scale)
        return v, bool(np.isinf(v).any())
    _fails(pins.check_reduce_update, upd)


def _unit_vs_brute(shard_fn, unshard_fn):
    """The whole-unit brute-force pin, run against a copy of the oracle whose
    shard / unshard functions are replaced."""
    from oracle import brute
    rng = np.random.default_rng(2)
    shapes = [(7, 13), (1,), (5,)]
    params = [rng.uniform(-0.1, 0.1, s).astype(np.float32) for s in shapes]
    P = 97
    grads = [[rng.normal(0, 1e-2, P).astype(np.float32) for _ in range(3)]]
    lay = O.Layout(shapes, 3, "flat")
    flat = O.flatten(params)
    sh = shard_fn(flat, lay)
    gathered = O.bf16_rne(unshard_fn(sh, lay))
    b = brute.brute_unit_run(shapes, 3, "flat", [p.reshape(-1).tolist() for p in params],
                             [[g.tolist() for g in grads[0]]], dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8,
                                                                    weight_decay=0.01), raf=False)
    assert gathered.tolist() == b["gathers"][0][0]
    for k in range(3):
        assert sh[k].tolist() == [float(x) for x in np.asarray(flat)[[i for a, c in lay.segments[k] for i in range(a, c)]]]


def test_unit_pin_accepts_the_oracle():
    _unit_vs_brute(O.shard, O.unshard)


def test_gather_in_reverse_rank_order_caught():
    def unshard_rev(shards, lay):
        out = np.concatenate(list(reversed(shards)))
        return out
    _fails(_unit_vs_brute, O.shard, unshard_rev)


def test_shard_off_by_one_caught():
    def shard_shift(flat, lay):
        out = []
        for k in range(lay.N):
            parts = [flat[max(a - 1, 0):max(b - 1, 0)] for a, b in lay.segments[k]]
            out.append(np.concatenate(parts) if parts else np.zeros(0, flat.dtype))
        return out
    with pytest.raises((AssertionError, ValueError)):   # wrong values, or pieces that no longer fit
        _unit_vs_brute(shard_shift, O.unshard)


def test_padded_padding_count_caught():
    def r(P, N, k):
        a, b, pad = O.padded_shard_range(P, N, k)
        return a, b, 0
    _fails(pins.check_padded_vs_torch_chunk, r, [(15, 16), (5, 4)])


def test_hybrid_rank_major_grouping_caught():
    """Groups must be consecutive ranks (rank i*F + k is rank k of group i);
    grouping by stride instead changes the rounding."""
    def r(grads, F):
        W = len(grads)
        regrouped = [grads[k * (W // F) + i] for i in range(W // F) for k in range(F)]
        return O.reduce_full_hybrid(regrouped, F)
    _fails(pins.check_hybrid_reduce, r, O.reduce_full)

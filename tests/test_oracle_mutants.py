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


def test_accumulate_overwrites_caught():
    def upd(G, old=None, inv_scale=1.0):
        return O.reduce_update(G, None, inv_scale)
    _fails(pins.check_reduce_update, upd)


def test_found_flag_misses_nan_caught():
    def upd(G, old=None, inv_scale=1.0):
        v, _ = O.reduce_update(G, old, inv_scale)
        return v, bool(np.isinf(v).any())
    _fails(pins.check_reduce_update, upd)

"""Pins for the oracle's fp32 -> bf16 round-to-nearest-even cast."""
import os

import numpy as np
import pytest

import pins
from oracle import fsdp_oracle as O


def test_cast_vs_torch_structured():
    pins.check_cast_vs_torch(O.bf16_rne, pins.structured_patterns())


@pytest.mark.skipif(os.environ.get("FSDP_EXHAUSTIVE_CAST") != "1",
                    reason="all 2^32 patterns: set FSDP_EXHAUSTIVE_CAST=1")
def test_cast_vs_torch_exhaustive():
    step = 1 << 24
    for a in range(0, 1 << 32, step):
        pins.check_cast_vs_torch(O.bf16_rne, np.arange(a, a + step, dtype=np.uint64).astype(np.uint32))


def test_cast_vs_exact_rational_rounding():
    rng = np.random.default_rng(5)
    pats = np.concatenate([
        rng.integers(0, 1 << 32, 6000, dtype=np.uint64).astype(np.uint32),
        pins.structured_patterns(n_random_low=0)[::97],
        np.array([0x7F7FFFFF, 0x7F7F8000, 0x7F7F7FFF, 0xFF7F8000, 0x00000001, 0x00008000,
                  0x00018000, 0x80008000, 0x7F800000, 0xFF800000, 0x7FC00000, 0x7F800001], np.uint32)])
    pins.check_cast_vs_brute(O.bf16_rne, pats)


@pytest.mark.parametrize("bits,want", [
    (0x3F800000, 0x3F80),   # 1.0 exact
    (0x3F808000, 0x3F80),   # tie, kept half even -> down
    (0x3F818000, 0x3F82),   # tie, kept half odd -> up
    (0x3F808001, 0x3F81),   # just above half
    (0x3F807FFF, 0x3F80),   # just below half
    (0x7F7FFFFF, 0x7F80),   # largest finite fp32 rounds to +inf
    (0x00008000, 0x0000),   # subnormal tie -> even (zero)
    (0x00018000, 0x0002),   # subnormal tie -> even (up)
    (0x80000000, 0x8000),   # -0
    (0xFF800000, 0xFF80),   # -inf
])
def test_cast_examples(bits, want):
    x = np.array([bits], np.uint32).view(np.float32)
    assert int(O.bf16_rne(x)[0]) == want


def test_cast_nan_stays_nan_with_sign():
    x = np.array([0x7FC00000, 0xFFC00001, 0x7F800001], np.uint32).view(np.float32)
    b = O.bf16_rne(x)
    assert all(((v & 0x7F80) == 0x7F80) and (v & 0x7F) for v in b.tolist())
    assert [(v >> 15) for v in b.tolist()] == [0, 1, 0]


def test_widen_is_exact():
    b = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    f = O.bf16_to_f32(b)
    back = O.bf16_rne(f)
    nan = np.isnan(f)
    assert np.array_equal(back[~nan], b[~nan])

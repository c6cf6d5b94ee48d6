"""Brute-force restatement of the per-unit cycle for tiny units.

TEST INFRASTRUCTURE (same rules as ``oracle.fsdp_oracle``: only tests, the
smoke check and the bench's CPU leg may use it).  It shares no code with
``oracle.fsdp_oracle`` either: it works element by element on Python floats
and integers so that the two can check each other.

* fp32 arithmetic: each operation is carried out on Python floats (IEEE
  doubles) and the double result is rounded to the nearest fp32.  For +, -, *,
  / and sqrt of fp32 operands this gives the correctly rounded fp32 result,
  because a double carries more than 2*24+2 significand bits.
* bf16 rounding: found by comparing the input with its two neighbouring bf16
  values as exact rationals (no bit tricks).
* Layout: found by counting, not by the closed form's integer division:
  rank k's FLAT range starts at the number of integers j >= 1 with
  j <= k*P/N (tested as j*N <= k*P), and DIM0 rows are dealt out in blocks.
"""
from __future__ import annotations

import math
import struct
from fractions import Fraction


def f32(x: float) -> float:
    """Round a double to the nearest fp32 (ties to even), as a double."""
    return struct.unpack("<f", struct.pack("<f", x))[0]


def f32_bits(x: float) -> int:
    return struct.unpack("<I", struct.pack("<f", x))[0]


def bits_f32(b: int) -> float:
    return struct.unpack("<f", struct.pack("<I", b))[0]


def bf16_round(x: float) -> int:
    """bf16 pattern nearest to the fp32 value x, ties to the even pattern."""
    if math.isnan(x):
        return None  # caller compares NaN-ness only
    if math.isinf(x):
        return 0x7F80 if x > 0 else 0xFF80
    if x == 0.0:
        return 0x8000 if math.copysign(1.0, x) < 0 else 0x0000
    sign = 0x8000 if x < 0 else 0
    ax = Fraction(abs(x))
    # the bf16 value just below |x| (toward zero) is the truncated pattern;
    # the one above is the next pattern, or 2**128 past the largest finite
    # bf16 (rounding as if the exponent range were unbounded, then overflow)
    lo = f32_bits(abs(x)) >> 16
    lo_val = Fraction(bits_f32(lo << 16))
    hi = lo + 1
    hi_val = Fraction(2) ** 128 if hi == 0x7F80 else Fraction(bits_f32(hi << 16))
    d_lo = ax - lo_val
    d_hi = hi_val - ax
    if d_lo < d_hi:
        r = lo
    elif d_hi < d_lo:
        r = hi
    else:
        r = lo if lo % 2 == 0 else hi
    return sign | r


def flat_ranges(P: int, N: int):
    """Rank ranges by counting: rank k starts at the number of integers
    j >= 1 with j*N <= k*P (the floor of k*P/N, counted one at a time)."""
    starts = []
    for k in range(N + 1):
        c = 0
        while (c + 1) * N <= k * P:
            c += 1
        starts.append(c)
    return [(starts[k], starts[k + 1]) for k in range(N)]


def dim0_ranges(shapes, N: int):
    """Per rank, the global ranges of its dim-0 chunks, by handing out rows:
    rows are dealt in blocks of ceil(m/N) to ranks 0, 1, ... in turn."""
    out = [[] for _ in range(N)]
    off = 0
    for s in shapes:
        m = s[0] if len(s) else 1
        r = 1
        for d in s[1:]:
            r *= d
        block = 0
        while block * N < m:
            block += 1
        row = 0
        k = 0
        while row < m:
            take = min(block, m - row)
            out[k].append((off + row * r, off + (row + take) * r))
            row += take
            k += 1
        off += m * r
    return out


def brute_unit_run(shapes, N, layout, params, grads_per_step, hp, raf=True):
    """Whole-unit run, element by element.  ``params``: list of nested lists or
    flat lists (row-major) of floats; ``grads_per_step``: per step a list of N
    flat lists of floats (already exact fp32 values).  Returns per step the
    gathered bf16 patterns (list per gather), and final per-rank
    (master, m, v) lists and per-step per-rank gradient shards."""
    flat = []
    for p in params:
        flat.extend(f32(x) for x in p)
    P = len(flat)
    if layout == "flat":
        ranges = [[r] if r[1] > r[0] else [] for r in flat_ranges(P, N)]
    else:
        ranges = dim0_ranges(shapes, N)
    owner = [None] * P
    for k in range(N):
        pos = 0
        for a, b in ranges[k]:
            for i in range(a, b):
                assert owner[i] is None
                owner[i] = (k, pos)
                pos += 1
    assert all(o is not None for o in owner)
    shard_len = [sum(b - a for a, b in ranges[k]) for k in range(N)]
    master = [[0.0] * shard_len[k] for k in range(N)]
    for i in range(P):
        k, j = owner[i]
        master[k][j] = flat[i]
    m = [[0.0] * shard_len[k] for k in range(N)]
    v = [[0.0] * shard_len[k] for k in range(N)]
    gathers, gshards = [], []
    for t, grads in enumerate(grads_per_step, start=1):
        n_gather = 2 if raf else 1
        step_g = []
        for _ in range(n_gather):
            out = [0] * P
            for i in range(P):
                k, j = owner[i]
                out[i] = bf16_round(master[k][j])
            step_g.append(out)
        gathers.append(step_g)
        gs = [[0.0] * shard_len[k] for k in range(N)]
        for i in range(P):
            acc = f32(grads[0][i])
            for r in range(1, N):
                acc = f32(acc + f32(grads[r][i]))
            k, j = owner[i]
            gs[k][j] = f32(acc / N)
        gshards.append(gs)
        bc1 = 1.0 - hp["beta1"] ** t
        bc2 = 1.0 - hp["beta2"] ** t
        decay = f32(1.0 - hp["lr"] * hp["weight_decay"])
        b1, c1 = f32(hp["beta1"]), f32(1.0 - hp["beta1"])
        b2, c2 = f32(hp["beta2"]), f32(1.0 - hp["beta2"])
        bc2f, step, eps = f32(bc2), f32(hp["lr"] / bc1), f32(hp["eps"])
        for k in range(N):
            for j in range(shard_len[k]):
                p = master[k][j]
                g = gs[k][j]
                p = f32(p * decay)
                mm = f32(f32(b1 * m[k][j]) + f32(c1 * g))
                vv = f32(f32(b2 * v[k][j]) + f32(c2 * f32(g * g)))
                den = f32(f32(math.sqrt(f32(vv / bc2f))) + eps)
                p = f32(p - f32(step * f32(mm / den)))
                master[k][j], m[k][j], v[k][j] = p, mm, vv
    return dict(gathers=gathers, gshards=gshards, master=master, m=m, v=v, ranges=ranges)


def padded_ranges(P: int, N: int):
    """Padded equal chunks: deal the P elements to ranks 0, 1, ... in blocks of
    the smallest size c with c*N >= P; returns (begin, end, pads) per rank."""
    c = 0
    while c * N < P:
        c += 1
    out = []
    pos = 0
    for k in range(N):
        take = min(c, P - pos)
        out.append((pos, pos + take, c - take))
        pos += take
    return out


def brute_reduce(grads, F=None, reduce_dtype="f32", old=None, inv_scale=1.0):
    """Element-by-element reduction of W gradient lists of floats: group-wise
    left folds (groups of F consecutive ranks; F = W is a single group), then
    the fold over groups, then division by W; in bf16 arithmetic every result
    is rounded to bf16; then the optional unscale and accumulation.  Returns
    (values, found_nonfinite)."""
    W = len(grads)
    F = W if F is None else F
    P = len(grads[0])
    out = []
    found = False

    def rb(x):   # a double holding an fp32 value, rounded to bf16
        if math.isnan(x) or math.isinf(x):
            return x
        return bits_f32(bf16_round(f32(x)) << 16)

    for i in range(P):
        if reduce_dtype == "bf16":
            acc = rb(grads[0][i])
            for r in range(1, W):
                acc = rb(f32(acc + rb(grads[r][i])))
            val = rb(f32(acc / W))
        else:
            tot = None
            for g in range(W // F):
                acc = f32(grads[g * F][i])
                for r in range(1, F):
                    acc = f32(acc + f32(grads[g * F + r][i]))
                tot = acc if tot is None else f32(tot + acc)
            val = f32(tot / W)
        if inv_scale != 1.0:
            val = f32(val * f32(inv_scale))
        if old is not None:
            val = f32(old[i] + val)
        found = found or math.isnan(val) or math.isinf(val)
        out.append(val)
    return out, found

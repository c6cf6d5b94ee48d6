"""Checks that pin the CPU oracle to something other than itself.

Each check takes the oracle function it pins as an argument, so the same
check runs against the real oracle (``test_oracle_*.py``) and against copies
with a planted mistake (``test_oracle_mutants.py``), where it must fail.

What pins what:
* layout  -- brute-force counting (``oracle.brute``), ``torch.chunk`` on CPU,
             the properties the pages state in words (equal contiguous slices,
             rank-order concatenation), the boundary statements printed for
             GPU 0 and GPU 1 on the "FSDP Architecture" page;
* cast    -- PyTorch's CPU fp32 -> bf16 conversion (a library routine that
             rounds to nearest even) and exact rational rounding (brute);
* reduce  -- closed forms on integer-valued gradients, the fp64 sum within
             the fp32 error bound of a left fold, special cases;
* AdamW   -- ``torch.optim.AdamW`` on CPU at N = 1 (unsharded training is
             the N = 1 special case), the closed-form first step, the
             zero-gradient step, the fp64 update within tolerance.
"""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np
import torch

from oracle import brute


# ----------------------------------------------------------------- layout

def check_flat_ranges(flat_shard_range, Pmax=64, Nmax=70):
    for P in range(1, Pmax + 1):
        for N in range(1, Nmax + 1):
            want = brute.flat_ranges(P, N)
            got = [tuple(flat_shard_range(P, N, k)) for k in range(N)]
            assert got == want, (P, N, got, want)


def check_flat_properties(flat_shard_range, cases):
    """Equal contiguous slices in rank order that tile [0, P); sizes differ by
    at most one; GPU 0 holds 0 .. floor(P/N)-1 and GPU 1 starts at floor(P/N)."""
    for P, N in cases:
        rng = [flat_shard_range(P, N, k) for k in range(N)]
        assert rng[0][0] == 0 and rng[-1][1] == P
        for k in range(N - 1):
            assert rng[k][1] == rng[k + 1][0]
        sizes = [b - a for a, b in rng]
        assert min(sizes) >= P // N and max(sizes) <= -(-P // N)
        assert sum(sizes) == P
        assert rng[0] == (0, P // N)
        if N > 1:
            assert rng[1][0] == P // N
        if P % N == 0:
            assert set(sizes) == {P // N}


def check_dim0_vs_torch_chunk(rank_segments, param_offsets, shapes, N):
    """Rank k's DIM0 ranges equal the global indices of torch.chunk(., N, dim=0)[k]
    of every parameter, in parameter order."""
    offs, P = param_offsets(shapes)
    want = [[] for _ in range(N)]
    for s, off in zip(shapes, offs):
        n = 1
        for d in s:
            n *= d
        t = torch.arange(n, dtype=torch.int64).reshape(s if len(s) else (1,))
        chunks = torch.chunk(t, N, dim=0)
        for k, c in enumerate(chunks):
            idx = c.reshape(-1)
            if idx.numel() == 0:
                continue
            a, b = int(idx[0]) + off, int(idx[-1]) + off + 1
            assert b - a == idx.numel()  # a chunk of whole rows is contiguous
            want[k].append((a, b))
    for k in range(N):
        assert [tuple(x) for x in rank_segments(shapes, N, "dim0", k)] == want[k], (shapes, N, k)


def check_dim0_vs_brute(rank_segments, shapes, N):
    want = brute.dim0_ranges([tuple(s) for s in shapes], N)
    for k in range(N):
        assert [tuple(x) for x in rank_segments(shapes, N, "dim0", k)] == want[k]


# ----------------------------------------------------------------- cast

def _torch_bf16_bits(x: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def check_cast_vs_torch(bf16_rne, patterns: np.ndarray):
    x = patterns.astype(np.uint32).view(np.float32)
    got = bf16_rne(x)
    want = _torch_bf16_bits(x)
    nan_in = np.isnan(x)
    nan_got = ((got & 0x7F80) == 0x7F80) & ((got & 0x007F) != 0)
    assert np.array_equal(nan_got, nan_in)
    ok = nan_in | (got == want)
    if not ok.all():
        i = int(np.flatnonzero(~ok)[0])
        raise AssertionError(f"input {patterns[i]:#010x}: got {got[i]:#06x} want {want[i]:#06x}")


def structured_patterns(seed=0, n_random_low=8):
    """Every one of the 65536 upper halves, each with the lower halves that
    decide rounding: 0, 1, just below half, half, just above half, all ones,
    and a few random ones."""
    rng = np.random.default_rng(seed)
    lows = [0x0000, 0x0001, 0x7FFF, 0x8000, 0x8001, 0xFFFF] + list(rng.integers(0, 1 << 16, n_random_low))
    upper = np.arange(1 << 16, dtype=np.uint32) << np.uint32(16)
    return np.concatenate([upper | np.uint32(lo) for lo in lows])


def check_cast_vs_brute(bf16_rne, patterns: np.ndarray):
    x = patterns.astype(np.uint32).view(np.float32)
    got = bf16_rne(x)
    for xi, gi in zip(x.tolist(), got.tolist()):
        w = brute.bf16_round(xi)
        if w is None:
            assert (gi & 0x7F80) == 0x7F80 and (gi & 0x7F) != 0
        else:
            assert gi == w, (xi, hex(gi), hex(w))


# ----------------------------------------------------------------- reduce

def check_reduce_integer_closed_form(reduce_full, Ns=range(1, 71), P=37):
    """g_r[i] = r + 1 (exact in fp32): sum = N(N+1)/2, mean = (N+1)/2 exactly."""
    for N in Ns:
        grads = [np.full(P, r + 1, np.float32) for r in range(N)]
        G = reduce_full(grads)
        assert G.dtype == np.float32
        assert np.all(G == np.float32((N + 1) / 2)), (N, G[:3])
    # mixed signs and a per-element pattern: g_r[i] = (i - r) , exact sum
    for N in (3, 7, 8):
        i = np.arange(P)
        grads = [(i - r).astype(np.float32) for r in range(N)]
        G = reduce_full(grads)
        want = (N * i - N * (N - 1) // 2) / N
        assert np.array_equal(G, want.astype(np.float32))


def check_reduce_fp64_bound(reduce_full, seed=0):
    """|fl(sum)/N - exact mean| within the left-fold bound
    (N-1) u sum|g| / N plus one rounding of the quotient (u = 2^-24)."""
    rng = np.random.default_rng(seed)
    u = 2.0 ** -24
    for N in (2, 3, 7, 8, 64):
        grads = [rng.normal(0, 1e-3, 4096).astype(np.float32) for _ in range(N)]
        G = reduce_full(grads).astype(np.float64)
        g64 = np.stack([g.astype(np.float64) for g in grads])
        exact = g64.sum(0) / N
        bound = (N - 1) * u * np.abs(g64).sum(0) / N * (1 + 1e-6) + u * np.abs(exact) * 1.0001 + 1e-45
        assert np.all(np.abs(G - exact) <= bound), N


def check_reduce_special(reduce_full):
    # the identity at N = 1
    g = np.random.default_rng(1).normal(0, 1, 1000).astype(np.float32)
    assert np.array_equal(reduce_full([g]), g)
    # left fold from g_0 (not from +0): all-negative-zero inputs give -0
    z = np.full(4, -0.0, np.float32)
    G = reduce_full([z, z])
    assert np.all(np.signbit(G))
    # rank order 0..N-1: (1e8 + 1) - 1e8 = 0 in fp32 (1 is absorbed)
    grads = [np.array([1e8], np.float32), np.array([1.0], np.float32), np.array([-1e8], np.float32)]
    assert reduce_full(grads)[0] == 0.0
    # ... and (1e8 - 1e8) + 1 = 1, so the mean is fl(1/3); a reversed fold gives 0
    grads = [np.array([1e8], np.float32), np.array([-1e8], np.float32), np.array([1.0], np.float32)]
    assert reduce_full(grads)[0] == np.float32(1.0) / np.float32(3.0)
    # division, not a rounded reciprocal: 1/3 * 3 vs 3/3 differ when N = 3
    grads = [np.array([1.0], np.float32)] * 3
    assert reduce_full(grads)[0] == np.float32(1.0)
    # bf16 gradients widen exactly: 0x3F81 (1.0078125) from three ranks -> 1.0078125
    b = np.array([0x3F81], np.uint16)
    assert reduce_full([b, b, b])[0] == np.float32(1.0078125)


# ----------------------------------------------------------------- AdamW

def tol_ok(a, b, atol=1e-6, rtol=1e-5):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return bool(np.all(np.abs(a - b) <= atol + rtol * np.abs(b)))


def check_adamw_vs_torch(adamw_update, hp, steps=6, n=5000, seed=0):
    """N = 1 (unsharded) AdamW against torch.optim.AdamW(foreach=False) on CPU."""
    rng = np.random.default_rng(seed)
    p0 = rng.normal(0, 0.02, n).astype(np.float32)
    grads = [rng.normal(0, 1e-3, n).astype(np.float32) for _ in range(steps)]
    tp = torch.nn.Parameter(torch.from_numpy(p0.copy()))
    opt = torch.optim.AdamW([tp], lr=hp.lr, betas=(hp.beta1, hp.beta2), eps=hp.eps,
                            weight_decay=hp.weight_decay, foreach=False, fused=False)
    p, m, v = p0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    for t, g in enumerate(grads, start=1):
        tp.grad = torch.from_numpy(g.copy())
        opt.step()
        p, m, v = adamw_update(p, g, m, v, t, hp)
    st = opt.state[tp]
    assert tol_ok(p, tp.detach().numpy()), "params"
    assert tol_ok(m, st["exp_avg"].numpy(), atol=1e-9), "exp_avg"
    assert tol_ok(v, st["exp_avg_sq"].numpy(), atol=1e-14), "exp_avg_sq"


def check_adamw_first_step_closed_form(adamw_update, hp, seed=0):
    """With m = v = 0, step 1 gives m = (1-b1) g, v = (1-b2) g^2, so
    p1 = p0 (1 - lr wd) - lr g / (|g| + eps)."""
    rng = np.random.default_rng(seed)
    p0 = rng.normal(0, 0.02, 4000).astype(np.float32)
    g = rng.normal(0, 1e-3, 4000).astype(np.float32)
    z = np.zeros_like(p0)
    p1, m1, v1 = adamw_update(p0, g, z, z, 1, hp)
    pd, gd = p0.astype(np.float64), g.astype(np.float64)
    want_p = pd * (1 - hp.lr * hp.weight_decay) - hp.lr * gd / (np.abs(gd) + hp.eps)
    assert tol_ok(p1, want_p, atol=1e-8, rtol=1e-6)
    assert tol_ok(m1, (1 - hp.beta1) * gd, atol=0, rtol=1e-6)
    assert tol_ok(v1, (1 - hp.beta2) * gd * gd, atol=0, rtol=1e-6)


def check_adamw_zero_grad(adamw_update, hp):
    """g = 0 from m = v = 0: only the decay acts, p1 = fl(p0 * fl(1 - lr wd))."""
    p0 = np.random.default_rng(3).normal(0, 0.02, 1000).astype(np.float32)
    z = np.zeros_like(p0)
    p1, m1, v1 = adamw_update(p0, z, z, z, 1, hp)
    assert np.array_equal(p1, p0 * np.float32(1.0 - hp.lr * hp.weight_decay))
    assert not m1.any() and not v1.any()


def check_adamw_fp64(adamw_update, adamw_update_f64, hp, steps=5, seed=0):
    """The fp32 update stays within the stated tolerance of the same update in
    fp64.  m = b1 m + c1 g can cancel, so m's error is bounded relative to the
    magnitude of its terms, M = b1 M + c1 |g|, not to m itself; v is a sum of
    non-negative terms and gets a plain relative bound."""
    rng = np.random.default_rng(seed)
    n = 4000
    p = rng.normal(0, 0.02, n).astype(np.float32)
    m = np.zeros(n, np.float32)
    v = np.zeros(n, np.float32)
    pd, md, vd = p.astype(np.float64), m.astype(np.float64), v.astype(np.float64)
    M = np.zeros(n)
    for t in range(1, steps + 1):
        g = rng.normal(0, 1e-3, n).astype(np.float32)
        p, m, v = adamw_update(p, g, m, v, t, hp)
        pd, md, vd = adamw_update_f64(pd, g.astype(np.float64), md, vd, t, hp)
        M = hp.beta1 * M + (1 - hp.beta1) * np.abs(g.astype(np.float64))
    assert tol_ok(p, pd)
    assert np.all(np.abs(m - md) <= 1e-5 * M)
    assert tol_ok(v, vd, atol=0, rtol=1e-5)


# ----------------------------------------------------------------- next rows

def check_padded_vs_torch_chunk(padded_shard_range, cases):
    """The padded equal-chunk layout's real elements are torch.chunk of the
    flat buffer viewed as one 1-D tensor; every rank's chunk (real + pads) has
    the same size and the total padding is at most N - 1."""
    for P, N in cases:
        chunks = torch.chunk(torch.arange(P), N)
        c = chunks[0].numel()
        pads = 0
        for k in range(N):
            a, b, pad = padded_shard_range(P, N, k)
            if k < len(chunks):
                assert (a, b) == (int(chunks[k][0]), int(chunks[k][-1]) + 1), (P, N, k)
            else:
                assert a == b
            assert (b - a) + pad == c
            pads += pad
        assert pads <= N - 1 and pads == N * c - P


def check_padded_vs_brute(padded_shard_range, Pmax=40, Nmax=20):
    for P in range(1, Pmax + 1):
        for N in range(1, Nmax + 1):
            assert [tuple(padded_shard_range(P, N, k)) for k in range(N)] == brute.padded_ranges(P, N)


def check_hybrid_reduce(reduce_full_hybrid, reduce_full, seed=0):
    rng = np.random.default_rng(seed)
    # integer-valued gradients: the decomposition is exact, mean (W+1)/2
    for W, F in [(8, 2), (8, 4), (12, 3), (6, 6), (6, 1)]:
        grads = [np.full(33, r + 1, np.float32) for r in range(W)]
        assert np.all(reduce_full_hybrid(grads, F) == np.float32((W + 1) / 2))
    # F = W (one sharding group) and F = 1 (pure replication) are the plain rank-order fold
    for W in (1, 4, 7):
        grads = [rng.normal(0, 1, 500).astype(np.float32) for _ in range(W)]
        assert np.array_equal(reduce_full_hybrid(grads, W), reduce_full(grads))
        assert np.array_equal(reduce_full_hybrid(grads, 1), reduce_full(grads))
    # 1 < F < W groups the fold: ranks (1e8, 1 | -1e8, 0) with F = 2 give
    # (1e8 + 1) + (-1e8 + 0) = 0 (the 1 is absorbed inside group 0), while
    # ranks (1e8, -1e8 | 1, 0) give 0 + 1 = 1, mean 0.25
    g = [np.array([x], np.float32) for x in (1e8, 1.0, -1e8, 0.0)]
    assert reduce_full_hybrid(g, 2)[0] == np.float32(0.0)
    g = [np.array([x], np.float32) for x in (1e8, -1e8, 1.0, 0.0)]
    assert reduce_full_hybrid(g, 2)[0] == np.float32(0.25)
    # the grouping is visible: ranks (1, 1e8 | -1e8, 1): F = 2 gives
    # (1 + 1e8) + (-1e8 + 1) = 1e8 - 1e8 = 0; the plain fold gives ((1 + 1e8) - 1e8) + 1 = 1
    g = [np.array([x], np.float32) for x in (1.0, 1e8, -1e8, 1.0)]
    assert reduce_full_hybrid(g, 2)[0] == np.float32(0.0)
    assert reduce_full(g)[0] == np.float32(0.25)
    # within the fp64 bound of the exact mean
    u = 2.0 ** -24
    for W, F in [(8, 2), (16, 4)]:
        grads = [rng.normal(0, 1e-3, 2048).astype(np.float32) for _ in range(W)]
        G = reduce_full_hybrid(grads, F).astype(np.float64)
        g64 = np.stack([x.astype(np.float64) for x in grads])
        exact = g64.sum(0) / W
        bound = (W - 1) * u * np.abs(g64).sum(0) / W * (1 + 1e-6) + u * np.abs(exact) * 1.0001
        assert np.all(np.abs(G - exact) <= bound)


def check_bf16_reduce_vs_torch(reduce_full_bf16, seed=0):
    """torch CPU bfloat16 arithmetic (each op computed in fp32 and rounded to
    bf16) folded in rank order, then divided by N."""
    rng = np.random.default_rng(seed)
    for N in (1, 2, 3, 7, 8):
        grads = [rng.normal(0, 1e-2, 3000).astype(np.float32) for _ in range(N)]
        acc = torch.from_numpy(grads[0]).to(torch.bfloat16)
        for g in grads[1:]:
            acc = acc + torch.from_numpy(g).to(torch.bfloat16)
        want = (acc / N).to(torch.float32).numpy()
        got = reduce_full_bf16(grads)
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32)), N
    # small integers are exact in bf16: mean (N+1)/2
    for N in (2, 5, 8):
        grads = [np.full(10, r + 1, np.float32) for r in range(N)]
        assert np.all(reduce_full_bf16(grads) == np.float32((N + 1) / 2))


def _round_bf16_exact(x: Fraction, sign: float) -> float:
    """The bf16 value nearest to the exact rational x (ties to an even last
    significand bit; an unbounded-exponent result of 2**128 or more is
    infinity).  `sign` gives the sign of a zero result."""
    if x == 0:
        return math.copysign(0.0, sign)
    s = -1.0 if x < 0 else 1.0
    ax = abs(x)
    e = ax.numerator.bit_length() - ax.denominator.bit_length()
    while Fraction(2) ** e > ax:
        e -= 1
    while Fraction(2) ** (e + 1) <= ax:
        e += 1
    ulp = Fraction(2) ** (max(e, -126) - 7)      # 8 significand bits; subnormals below 2**-126
    q = ax / ulp
    n = q.numerator // q.denominator
    rem = q - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    val = n * ulp
    if val >= Fraction(2) ** 128:
        return s * math.inf
    return math.copysign(float(val), s)


def check_bf16_reduce_exact(reduce_full_bf16, seed=0):
    """bf16 arithmetic from its definition: each partial sum of the rank-order
    fold and the final division by N is the exact rational result rounded
    once to bf16.  Inputs are bf16 bit patterns of every exponent (subnormals,
    zeros of both signs, the largest finite values) plus pairs whose exponents
    differ by 0..20, so that sums land near bf16 rounding midpoints; a
    missing, doubled or misplaced rounding fails here."""
    rng = np.random.default_rng(seed)

    def finite_patterns(n):
        b = rng.integers(0, 1 << 16, n, dtype=np.uint32).astype(np.uint16)
        inf_nan = (b & 0x7F80) == 0x7F80
        b[inf_nan] &= 0xBFFF                     # exponent 0xFF -> 0x7F: finite
        return b

    def value(h):
        return float(np.uint32(int(h) << 16).view(np.float32))

    cases = []
    for N in (2, 3, 8):
        cases.append([finite_patterns(4000) for _ in range(N)])
    a = finite_patterns(4000) & 0x807F | (rng.integers(40, 200, 4000).astype(np.uint16) << 7)
    d = rng.integers(0, 21, 4000).astype(np.uint16)
    b = finite_patterns(4000) & 0x807F | (((a >> 7) & 0xFF) - d) << 7
    cases.append([a, b])
    cases.append([np.array([0x8000, 0x8000, 0x0000, 0x7F7F, 0xFF7F, 0x0001], np.uint16),
                  np.array([0x8000, 0x0000, 0x8000, 0x7F7F, 0x7F7F, 0x8001], np.uint16)])
    for grads in cases:
        N = len(grads)
        with np.errstate(over="ignore"):
            got = reduce_full_bf16(grads)
        for i in range(grads[0].size):
            acc = value(grads[0][i])
            for r in range(1, N):
                x = value(grads[r][i])
                if math.isinf(acc):
                    continue                     # finite inputs: inf + x stays inf
                zero_sign = -1.0 if (math.copysign(1.0, acc) < 0 and math.copysign(1.0, x) < 0) else 1.0
                acc = _round_bf16_exact(Fraction(acc) + Fraction(x), zero_sign)
            want = acc if math.isinf(acc) else _round_bf16_exact(Fraction(acc) / N, math.copysign(1.0, acc))
            w = np.float32(want).view(np.uint32)
            g = got[i].view(np.uint32)
            assert w == g, (N, i, [hex(int(gr[i])) for gr in grads], float(got[i]), want)


def check_reduce_update(reduce_update):
    # accumulation of k micro-batches: k * 2.5, exact
    old = np.zeros(50, np.float32)
    for k in range(1, 5):
        old, found = reduce_update(np.full(50, 2.5, np.float32), old)
        assert np.all(old == np.float32(2.5 * k)) and not found
    # unscale by a power of two is exact; 1.0 is the identity
    G = np.random.default_rng(0).normal(0, 1, 100).astype(np.float32)
    assert np.array_equal(reduce_update(G, None, 0.25)[0], G / np.float32(4))
    assert np.array_equal(reduce_update(G, None, 1.0)[0], G)
    # the flag is the OR over every element: one inf or NaN anywhere sets it
    for bad in (np.inf, -np.inf, np.nan):
        H = G.copy()
        H[37] = bad
        assert reduce_update(H)[1]
    assert not reduce_update(G)[1]
    # overflow created by the unscale is found too
    with np.errstate(over="ignore"):
        assert reduce_update(np.array([3e38], np.float32), None, 4.0)[1]

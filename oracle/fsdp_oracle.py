"""Plain, slow, CPU oracle for the per-FSDP-unit shard / gather / reduce-scatter / AdamW cycle.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline and reference legs may import or call this module.
The library (``fully_sharded_unit_gb300``) never imports it and never routes
through it; the two share no code.  Inputs come from
``fully_sharded_unit_gb300.workloads`` (random draws only) or from the tests.

Every step is written out from its definition, in the order the pages give:

* FSDP unit and FlatParameter -- "PyTorch FSDP: Experiences on Scaling Fully
  Sharded Data Parallel", section 3.2.1 "FlatParameter: Flattening,
  Concatenation, and Sharding" (Figure 3): each parameter is flattened to 1-D
  and the flattened parameters are concatenated in unit order.
* FLAT shard boundaries -- "FSDP Architecture" (the linear-layer example):
  rank k owns elements floor(kP/N) .. floor((k+1)P/N) - 1 of the flat buffer,
  no padding.
* DIM0 shards -- "FSDP (Fully Sharded Data Parallel)", "FSDP1 vs FSDP2", and
  "FSDP Under The Hood", section 2 "Sharding geometry": every parameter is
  chunked along dim-0 with torch.chunk semantics (ceil(m/N) rows per chunk,
  a short or empty tail); a rank's shard is its chunk of each parameter.
* All-gather -- "PyTorch FSDP ...", section 3.2.1 "Communication layout": the
  gathered buffer is the concatenation of the shards in rank order, i.e. the
  unsharded FlatParameter; section 4.4 "Native Mixed Precision": one
  full-to-low precision cast per FlatParameter when it is gathered.  Here
  fp32 -> bf16, IEEE-754 round to nearest, ties to even.
* Reduce-scatter -- "FSDP Architecture", backward step 3: sum the ranks'
  gradients and give rank k only the slice matching its parameter shard;
  "FSDP Under The Hood", section 3: fp32 reduction.  Summation is a left fold
  over ranks 0..N-1 in fp32, followed by one IEEE division by N (the average
  data-parallel gradient).
* AdamW -- "FSDP Architecture": the optimizer step is local, each rank updates
  its shard from its gradient shard and its m / v shards; "FSDP Under The
  Hood", appendix script: torch.optim.AdamW.  The update is the documented
  decoupled-weight-decay Adam (Loshchilov & Hutter) with bias correction.
* The per-unit cycle -- "FSDP Architecture" (forward: gather, compute,
  discard; backward: gather, compute, reduce-scatter, discard; then the local
  optimizer step) and "PyTorch FSDP ...", section 5.4 (reshard after forward
  re-gathers in backward).

Floating point: the pages fix the precisions (fp32 sharded master weights,
bf16 gathered parameters, fp32 gradient reduction), so the oracle computes in
fp32 with one IEEE rounding per operation, in the operation order written
below, no fused multiply-add.  numpy float32 elementwise arithmetic is IEEE
correctly rounded per operation.  ``adamw_update_f64`` is the same update in
fp64, used only as an error-bound pin.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

FLAT = "flat"
DIM0 = "dim0"
FLAT_PADDED = "flat_padded"

F32 = np.float32


# --------------------------------------------------------------------------
# Layout
# --------------------------------------------------------------------------

def numel(shape) -> int:
    """Element count of a parameter; a 0-d parameter counts as one element."""
    n = 1
    for d in shape:
        n *= int(d)
    return n


def rows_and_row_len(shape):
    """dim-0 size and the number of elements in one dim-0 row (row-major).
    A 0-d parameter is read as shape [1]."""
    if len(shape) == 0:
        return 1, 1
    m = int(shape[0])
    r = 1
    for d in shape[1:]:
        r *= int(d)
    return m, r


def param_offsets(shapes):
    """FlatParameter offsets: parameter p starts at the sum of the element
    counts of the parameters before it ("PyTorch FSDP ...", section 3.2.1,
    flatten then concatenate)."""
    offs, o = [], 0
    for s in shapes:
        offs.append(o)
        o += numel(s)
    return offs, o


def flat_shard_range(P: int, N: int, k: int):
    """Rank k's half-open element range [floor(kP/N), floor((k+1)P/N)) of the
    flat buffer ("FSDP Architecture", the GPU-k boundary formula)."""
    return (k * P) // N, ((k + 1) * P) // N


def padded_shard_range(P: int, N: int, k: int):
    """Padded-equal-chunk FLAT variant ("PyTorch FSDP ...", section 3.2.1,
    Figure 3): the flat buffer is right-padded to a multiple of N and cut into
    N equal chunks of ceil(P/N) elements.  Returns rank k's real-element range
    [begin, end) and how many padding elements follow it in its chunk."""
    c = -(-P // N)
    a, b = min(k * c, P), min((k + 1) * c, P)
    return a, b, c - (b - a)


def dim0_chunk_rows(m: int, N: int, k: int):
    """Rows [begin, end) of a dim-0 size-m parameter that rank k holds under
    torch.chunk(dim=0) semantics: chunks of ceil(m/N) rows, the last one short,
    trailing ranks empty when fewer than N chunks exist ("FSDP (Fully Sharded
    Data Parallel)", FSDP1 vs FSDP2)."""
    c = -(-m // N)
    return min(k * c, m), min((k + 1) * c, m)


def rank_segments(shapes, N: int, layout: str, k: int):
    """Rank k's shard as a list of (global_begin, global_end) ranges of the
    unsharded flat buffer, in the order the rank stores them."""
    offs, P = param_offsets(shapes)
    if layout == FLAT:
        a, b = flat_shard_range(P, N, k)
        return [(a, b)] if b > a else []
    if layout == FLAT_PADDED:
        a, b, _ = padded_shard_range(P, N, k)
        return [(a, b)] if b > a else []
    if layout == DIM0:
        segs = []
        for s, off in zip(shapes, offs):
            m, r = rows_and_row_len(s)
            r0, r1 = dim0_chunk_rows(m, N, k)
            if r1 > r0:
                segs.append((off + r0 * r, off + r1 * r))
        return segs
    raise ValueError(layout)


@dataclass
class Layout:
    shapes: list
    N: int
    layout: str

    def __post_init__(self):
        self.offsets, self.P = param_offsets(self.shapes)
        self.segments = [rank_segments(self.shapes, self.N, self.layout, k) for k in range(self.N)]

    def shard_len(self, k: int) -> int:
        return sum(b - a for a, b in self.segments[k])

    def padding(self, k: int) -> int:
        """Padding elements rank k stores after its real elements (padded
        layout only; the other layouts store none)."""
        if self.layout != FLAT_PADDED:
            return 0
        return padded_shard_range(self.P, self.N, k)[2]


# --------------------------------------------------------------------------
# FlatParameter construction and shard-in
# --------------------------------------------------------------------------

def flatten(params) -> np.ndarray:
    """The unsharded FlatParameter: every parameter flattened (row-major) and
    concatenated in unit order."""
    return np.concatenate([np.asarray(p, dtype=F32).reshape(-1) for p in params]) \
        if len(params) else np.zeros(0, F32)


def shard(flat: np.ndarray, lay: Layout):
    """Each rank's shard: the concatenation of its segments of the flat buffer."""
    out = []
    for k in range(lay.N):
        parts = [flat[a:b] for a, b in lay.segments[k]]
        out.append(np.concatenate(parts).astype(flat.dtype, copy=True) if parts
                   else np.zeros(0, flat.dtype))
    return out


def unshard(shards, lay: Layout) -> np.ndarray:
    """Rebuild the full flat buffer from the N shards (the all-gather): each
    rank's pieces go back to their global ranges."""
    dt = shards[0].dtype if shards else F32
    out = np.empty(lay.P, dtype=dt)
    written = np.zeros(lay.P, dtype=bool)
    for k in range(lay.N):
        pos = 0
        for a, b in lay.segments[k]:
            out[a:b] = shards[k][pos:pos + (b - a)]
            written[a:b] = True
            pos += b - a
        assert pos == shards[k].size
    assert written.all(), "shards do not cover the unit"
    return out


# --------------------------------------------------------------------------
# fp32 -> bf16, round to nearest, ties to even
# --------------------------------------------------------------------------

def bf16_rne(x) -> np.ndarray:
    """bf16 bit patterns (uint16) of fp32 values, IEEE-754 roundTiesToEven.

    A bf16 value is the upper 16 bits of an fp32 pattern.  For a non-NaN
    input the result is the upper half, plus one unit when the discarded
    lower half is more than half a unit, or exactly half a unit and the kept
    half is odd.  Carrying out of the mantissa steps the exponent, which is
    also correct for the largest finite values (they round to infinity).
    Infinities and subnormals need no special path.  A NaN stays a NaN of the
    same sign (quiet bit set)."""
    u = np.ascontiguousarray(x, dtype=F32).view(np.uint32)
    upper = (u >> np.uint32(16)).astype(np.uint32)
    lower = u & np.uint32(0xFFFF)
    half = np.uint32(0x8000)
    round_up = (lower > half) | ((lower == half) & ((upper & np.uint32(1)) == np.uint32(1)))
    res = upper + round_up.astype(np.uint32)
    is_nan = ((u & np.uint32(0x7F800000)) == np.uint32(0x7F800000)) & ((u & np.uint32(0x007FFFFF)) != 0)
    res = np.where(is_nan, upper | np.uint32(0x0040), res)
    return res.astype(np.uint16)


def bf16_to_f32(b) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp32 (bf16 is the top half)."""
    b = np.asarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(F32)


# --------------------------------------------------------------------------
# All-gather with the param_dtype cast
# --------------------------------------------------------------------------

def allgather_cast(master_shards, lay: Layout) -> np.ndarray:
    """The gathered bf16 unsharded FlatParameter: the shards in their global
    positions, each element cast fp32 -> bf16 (RNE)."""
    return bf16_rne(unshard(master_shards, lay))


# --------------------------------------------------------------------------
# Reduce-scatter
# --------------------------------------------------------------------------

def upcast_grad(g) -> np.ndarray:
    """A rank's gradient as fp32: fp32 stays, bf16 (given as uint16 bit
    patterns) widens exactly."""
    g = np.asarray(g)
    if g.dtype == np.uint16:
        return bf16_to_f32(g)
    assert g.dtype == F32
    return g


def reduce_full(grads) -> np.ndarray:
    """G = (((g_0 + g_1) + g_2) + ... + g_{N-1}) / N, in fp32, every
    operation rounded once.  The fold starts from g_0 itself, not from +0.0."""
    N = len(grads)
    acc = upcast_grad(grads[0]).astype(F32, copy=True)
    for r in range(1, N):
        acc = (acc + upcast_grad(grads[r])).astype(F32)
    return (acc / F32(N)).astype(F32)


def reduce_full_hybrid(grads, F: int) -> np.ndarray:
    """Hybrid sharding ("PyTorch FSDP ...", section 3.2.2, Figure 4): the W
    ranks form W/F sharding groups of F consecutive ranks; rank i*F + k is
    rank k of group i.  The global sum is decomposed as
        sum_r g_r = sum_i ( sum_{r in S_i} g_r ):
    a reduce-scatter inside each sharding group (left fold over its F ranks in
    order), then an all-reduce across groups (left fold over the group sums
    in group order), then one division by W.  With F = W or F = 1 the fold
    order is the plain rank order."""
    W = len(grads)
    assert W % F == 0
    total = None
    for i in range(W // F):
        acc = upcast_grad(grads[i * F]).astype(F32, copy=True)
        for r in range(1, F):
            acc = (acc + upcast_grad(grads[i * F + r])).astype(F32)
        total = acc if total is None else (total + acc).astype(F32)
    return (total / F32(W)).astype(F32)


def reduce_full_bf16(grads) -> np.ndarray:
    """Reduction in bf16 (reduce_dtype = bf16, "PyTorch FSDP ...", section
    4.4: collectives may run in the low precision).  Every rank's gradient is
    first rounded to bf16 (exact when it already is bf16), every partial sum
    is rounded to bf16, and so is the division by N; the result is widened
    exactly to fp32 for the fp32 gradient shard.  Each bf16 operation is the
    fp32 operation followed by one RNE rounding, which equals the correctly
    rounded bf16 operation because fp32 carries more than 2*8+2 bits."""
    N = len(grads)

    def b(x):
        return bf16_to_f32(bf16_rne(x))

    acc = b(upcast_grad(grads[0]))
    for r in range(1, N):
        acc = b((acc + b(upcast_grad(grads[r]))).astype(F32))
    return b((acc / F32(N)).astype(F32))


def reduce_update(G, old=None, inv_scale: float = 1.0):
    """Post-reduction steps on the reduced gradient G, in this order:
    unscale (G * inv_scale, skipped when inv_scale is 1, as a loss-scaling
    grad scaler does) and accumulation into the existing gradient shard
    (old + G: gradient accumulation with communication, "PyTorch FSDP ...",
    section 3.3.4: every micro-batch is reduce-scattered and each rank adds the
    result to its local gradient shard).  Returns the new gradient values and
    whether any of them is non-finite (the sharded grad scaler's global
    overflow decision, section 4.4: the OR over all ranks' shards)."""
    G = np.asarray(G, F32)
    if inv_scale != 1.0:
        G = (G * F32(inv_scale)).astype(F32)
    if old is not None:
        G = (np.asarray(old, F32) + G).astype(F32)
    return G, bool((~np.isfinite(G)).any())


def reduce_scatter(grads, lay: Layout):
    """Rank k's fp32 gradient shard: the reduced gradient restricted to rank
    k's segments (reduce, then keep only the matching slice)."""
    assert len(grads) == lay.N
    G = reduce_full(grads)
    return shard(G, lay)


# --------------------------------------------------------------------------
# AdamW
# --------------------------------------------------------------------------

@dataclass(frozen=True)
class AdamWHyper:
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.01


def adamw_scalars(t: int, hp: AdamWHyper):
    """Per-step fp32 constants of the update, each formed once from the
    double-precision hyper-parameters and rounded once to fp32:

      decay = 1 - lr*wd            (decoupled weight decay factor)
      b1, b2 = beta1, beta2;  c1, c2 = 1 - beta1, 1 - beta2
      bc2 = 1 - beta2**t           (second-moment bias correction)
      step = lr / (1 - beta1**t)   (learning rate over first-moment correction)
      eps
    """
    assert t >= 1
    bc1 = 1.0 - math.pow(hp.beta1, t)
    bc2 = 1.0 - math.pow(hp.beta2, t)
    return dict(
        decay=F32(1.0 - hp.lr * hp.weight_decay),
        b1=F32(hp.beta1), c1=F32(1.0 - hp.beta1),
        b2=F32(hp.beta2), c2=F32(1.0 - hp.beta2),
        bc2=F32(bc2), step=F32(hp.lr / bc1), eps=F32(hp.eps))


def adamw_update(p, g, m, v, t: int, hp: AdamWHyper):
    """One AdamW step at step count t (1-based), elementwise, fp32:

      p <- p * decay
      m <- b1*m + c1*g
      v <- b2*v + c2*(g*g)
      p <- p - step * (m / (sqrt(v / bc2) + eps))

    i.e. p - lr * m_hat / (sqrt(v_hat) + eps) with m_hat = m/(1-beta1^t),
    v_hat = v/(1-beta2^t), after the decoupled decay p*(1 - lr*wd).
    Returns new (p, m, v)."""
    c = adamw_scalars(t, hp)
    p = np.asarray(p, F32)
    g = np.asarray(g, F32)
    m = np.asarray(m, F32)
    v = np.asarray(v, F32)
    p1 = p * c["decay"]
    m1 = (c["b1"] * m) + (c["c1"] * g)
    v1 = (c["b2"] * v) + (c["c2"] * (g * g))
    denom = np.sqrt(v1 / c["bc2"]) + c["eps"]
    p2 = p1 - c["step"] * (m1 / denom)
    return p2.astype(F32), m1.astype(F32), v1.astype(F32)


def adamw_update_f64(p, g, m, v, t: int, hp: AdamWHyper):
    """The same update carried out in fp64 from fp64 hyper-parameters
    (used only to bound the fp32 oracle's rounding error)."""
    p = np.asarray(p, np.float64)
    g = np.asarray(g, np.float64)
    m = np.asarray(m, np.float64)
    v = np.asarray(v, np.float64)
    bc1 = 1.0 - hp.beta1 ** t
    bc2 = 1.0 - hp.beta2 ** t
    p1 = p * (1.0 - hp.lr * hp.weight_decay)
    m1 = hp.beta1 * m + (1.0 - hp.beta1) * g
    v1 = hp.beta2 * v + (1.0 - hp.beta2) * (g * g)
    p2 = p1 - (hp.lr / bc1) * (m1 / (np.sqrt(v1 / bc2) + hp.eps))
    return p2, m1, v1


# --------------------------------------------------------------------------
# The unit: N virtual ranks and the per-unit cycle
# --------------------------------------------------------------------------

class UnitOracle:
    """One FSDP unit over N virtual ranks.  Every rank keeps its own fp32
    master shard, fp32 gradient shard, fp32 m and v shards and the bf16 copy
    of its master shard; steady state is 4+4+8 bytes per owned element
    ("FSDP Architecture", memory breakdown), plus 2 for the bf16 copy."""

    def __init__(self, shapes, N: int, layout: str, hp: AdamWHyper = AdamWHyper(),
                 reshard_after_forward: bool = True, replicas: int = 1, reduce_dtype: str = "f32"):
        """N is the sharding factor F (ranks a parameter is sharded over).
        With replicas R > 1 the unit is hybrid-sharded over W = F*R ranks
        ("PyTorch FSDP ...", section 3.2.2): the R members of a replication
        group hold identical shards, so one copy of each shard is kept, and a
        reduce-scatter takes W gradients ordered group by group."""
        assert not (replicas > 1 and reduce_dtype != "f32"), "hybrid reduction is fp32"
        self.lay = Layout(list(shapes), N, layout)
        self.N = N
        self.replicas = replicas
        self.reduce_dtype = reduce_dtype
        self.hp = hp
        self.raf = reshard_after_forward
        self.t = 0
        self.master = None

    # shard-in (FlatParameter construction; optimizer state starts at zero)
    def load(self, params):
        flat = flatten(params)
        assert flat.size == self.lay.P
        self.master = shard(flat, self.lay)
        self.grad = [np.zeros(self.lay.shard_len(k), F32) for k in range(self.N)]
        self.m = [np.zeros(self.lay.shard_len(k), F32) for k in range(self.N)]
        self.v = [np.zeros(self.lay.shard_len(k), F32) for k in range(self.N)]
        self.shadow = [bf16_rne(x) for x in self.master]
        self.t = 0

    def allgather(self) -> np.ndarray:
        return allgather_cast(self.master, self.lay)

    def reduce_scatter(self, grads, accumulate: bool = False, inv_scale: float = 1.0) -> bool:
        """Reduce the W = N*replicas gradients, keep each rank's slice (added to
        its existing shard when accumulating).  Returns the found-non-finite flag."""
        assert len(grads) == self.N * self.replicas
        if self.replicas > 1:
            G = reduce_full_hybrid(grads, self.N)
        elif self.reduce_dtype == "bf16":
            G = reduce_full_bf16(grads)
        else:
            G = reduce_full(grads)
        old = unshard(self.grad, self.lay) if accumulate else None
        G, found = reduce_update(G, old, inv_scale)
        self.grad = shard(G, self.lay)
        return found

    def adamw_step(self):
        self.t += 1
        for k in range(self.N):
            self.master[k], self.m[k], self.v[k] = adamw_update(
                self.master[k], self.grad[k], self.m[k], self.v[k], self.t, self.hp)
            self.shadow[k] = bf16_rne(self.master[k])

    def step(self, grads):
        """One unit step: gather (forward), gather again when resharding after
        forward (backward), reduce-scatter, local AdamW.  Returns the list of
        gathered buffers in the order they were produced."""
        outs = [self.allgather()]
        if self.raf:
            outs.append(self.allgather())
        self.reduce_scatter(grads)
        self.adamw_step()
        return outs

    def full(self, which: str) -> np.ndarray:
        """A state reassembled in unsharded (global) order."""
        return unshard(getattr(self, which), self.lay)

    def memory_bytes(self, k: int) -> dict:
        n = self.lay.shard_len(k)
        return dict(param=4 * n, grad=4 * n, adam=8 * n, shadow=2 * n)


# --------------------------------------------------------------------------
# Element windows (for units too large to hold on the host)
# --------------------------------------------------------------------------

def run_window(params_window, grads_windows_per_step, hp: AdamWHyper, reduce=None):
    """The cycle restricted to a window of global indices.  Every operation
    after the layout is elementwise in the global index, so the master, m, v,
    gradient shard and gathered values at index i depend only on the initial
    parameter at i and the ranks' gradients at i.  ``reduce`` maps the list of
    gradient windows to the reduced gradient (default: the plain rank-order
    fold, ``reduce_full``; also ``reduce_full_bf16`` or a hybrid fold).
    Returns, per step, the (gathered bf16, reduced fp32 gradient) of the
    window and the final (master, m, v)."""
    reduce = reduce_full if reduce is None else reduce
    p = np.asarray(params_window, F32).copy()
    m = np.zeros_like(p)
    v = np.zeros_like(p)
    per_step = []
    for t, grads in enumerate(grads_windows_per_step, start=1):
        gathered = bf16_rne(p)
        G = reduce(grads)
        p, m, v = adamw_update(p, G, m, v, t, hp)
        per_step.append((gathered, G))
    return per_step, (p, m, v)

"""Seeded synthetic workloads for the per-unit FSDP cycle.

This module holds shapes and random draws only: no step of the method (no
flattening, sharding, casting, reduction or optimizer arithmetic) lives here.
It is the one module that both the CUDA path's callers and the CPU oracle's
callers use, so that both sides see the same bytes.

Workload shapes follow the models the pages measure on:

* GPT-2 blocks (the GPT-2 Large model of "FSDP Under The Hood: ZeRO-3 The
  PyTorch Way", section 5, and its GPT-2-small sibling): per block
  ln_1 w,b [d]; c_attn W[d x 3d] + b[3d]; attn c_proj W[d x d] + b[d];
  ln_2 w,b [d]; mlp c_fc W[d x ffn] + b[ffn]; mlp c_proj W[ffn x d] + b[d].
* minGPT-175B blocks (d = 12288, ffn = 49152) of "PyTorch FSDP: Experiences on
  Scaling Fully Sharded Data Parallel", section 5 (evaluation).
* A ragged stress unit whose sizes are not divisible by the rank count.

Shapes are read literally: ``W[a x b]`` has dim-0 = a, row-major.  Normal
draws are parameterised by their standard deviation.

Every tensor gets its own generator, seeded from (workload, unit, kind, step,
rank), so any one tensor can be regenerated alone and in any order.
"""
from __future__ import annotations

import dataclasses
import hashlib
from typing import Sequence

import torch

# init kinds: ("normal", std) | ("uniform", lo, hi) | ("ones",) | ("zeros",)
Init = tuple


@dataclasses.dataclass(frozen=True)
class Param:
    name: str
    shape: tuple
    init: Init


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    description: str
    units: tuple            # tuple of units; a unit is a tuple of Param
    N: int                  # virtual data-parallel ranks
    layout: str             # "flat" (FSDP1 FlatParameter) | "dim0" (FSDP2 Shard(0))
    grad_dtype: str         # "f32" | "bf16"
    steps: int
    grad_std: float
    outlier_frac: float = 0.0
    outlier_scale: float = 1.0
    reshard_after_forward: bool = True
    replicas: int = 1           # hybrid sharding: replication groups (W = N * replicas ranks)
    reduce_dtype: str = "f32"   # "f32" | "bf16"
    gather_source: str = "master"   # "master" (cast while gathering) | "shadow"
    fuse_reduce_adamw: bool = False  # fsdp_step runs reduce-scatter and AdamW as one kernel
    seed: int = 0
    # AdamW hyper-parameters (torch.optim.AdamW argument names)
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.01

    def shapes(self, unit: int) -> list:
        return [p.shape for p in self.units[unit]]

    def unit_numel(self, unit: int) -> int:
        n = 0
        for p in self.units[unit]:
            k = 1
            for d in p.shape:
                k *= d
            n += k
        return n

    @property
    def world(self) -> int:
        """Data-parallel ranks that produce gradients (N * replicas)."""
        return self.N * self.replicas

    @property
    def n_units(self) -> int:
        return len(self.units)

    def torch_grad_dtype(self):
        return torch.float32 if self.grad_dtype == "f32" else torch.bfloat16

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


def gpt_block(d: int, ffn: int, w_init: Init, ln_w_init: Init, bias_init: Init) -> tuple:
    """One GPT-2 style transformer block's parameters in registration order."""
    return (
        Param("ln_1.weight", (d,), ln_w_init),
        Param("ln_1.bias", (d,), bias_init),
        Param("attn.c_attn.weight", (d, 3 * d), w_init),
        Param("attn.c_attn.bias", (3 * d,), bias_init),
        Param("attn.c_proj.weight", (d, d), w_init),
        Param("attn.c_proj.bias", (d,), bias_init),
        Param("ln_2.weight", (d,), ln_w_init),
        Param("ln_2.bias", (d,), bias_init),
        Param("mlp.c_fc.weight", (d, ffn), w_init),
        Param("mlp.c_fc.bias", (ffn,), bias_init),
        Param("mlp.c_proj.weight", (ffn, d), w_init),
        Param("mlp.c_proj.bias", (d,), bias_init),
    )


def ragged_unit(rows_emb: int, d: int, cols: int, init: Init) -> tuple:
    """Mixed-shape unit: embedding, two LN vectors, a wide matrix with an odd
    column count, a 7x13 matrix and a one-element parameter."""
    return (
        Param("emb.weight", (rows_emb, d), init),
        Param("ln.weight", (d,), init),
        Param("ln.bias", (d,), init),
        Param("proj.weight", (d, cols), init),
        Param("small.weight", (7, 13), init),
        Param("scalar", (1,), init),
    )


def _workloads() -> dict:
    w = {}
    n002 = ("normal", 0.02)
    w["tiny_flat"] = Workload(
        name="tiny_flat",
        description="Tiny FSDP1 unit: Linear W[64x48] + bias[64] (3136 params), N=4, 3 steps",
        units=((Param("linear.weight", (64, 48), n002), Param("linear.bias", (64,), n002)),),
        N=4, layout="flat", grad_dtype="f32", steps=3, grad_std=1e-3)
    w["gpt2_small_flat"] = Workload(
        name="gpt2_small_flat",
        description="GPT-2-small FSDP1 units: 12 blocks d=768 (7,087,872 params each), N=8, 5 steps",
        units=tuple(gpt_block(768, 3072, n002, ("ones",), ("zeros",)) for _ in range(12)),
        N=8, layout="flat", grad_dtype="f32", steps=5, grad_std=1e-3)
    w["gpt2_large_dim0"] = Workload(
        name="gpt2_large_dim0",
        description="GPT-2-Large FSDP2 units: 36 blocks d=1280 ffn 5120 (19,677,440 params each), "
                    "per-parameter Shard(0), N=8, 3 steps",
        units=tuple(gpt_block(1280, 5120, n002, n002, n002) for _ in range(36)),
        N=8, layout="dim0", grad_dtype="f32", steps=3, grad_std=1e-3)
    n0006 = ("normal", 0.006)
    w["mingpt175b_flat"] = Workload(
        name="mingpt175b_flat",
        description="minGPT-175B FSDP1 units: 2 blocks d=12288 ffn 49152 (1,812,099,072 params each), "
                    "N=8, bf16 per-rank grads reduced in fp32, 2 steps",
        units=tuple(gpt_block(12288, 49152, n0006, n0006, n0006) for _ in range(2)),
        N=8, layout="flat", grad_dtype="bf16", steps=2, grad_std=1e-4,
        outlier_frac=1e-3, outlier_scale=1e3)
    u01 = ("uniform", -0.1, 0.1)
    for n in (7, 64):
        for layout in ("flat", "dim0"):
            name = f"ragged_{layout}_n{n}"
            w[name] = Workload(
                name=name,
                description=f"Ragged stress unit (70,886,492 params) {layout.upper()} at N={n}, 4 steps",
                units=(ragged_unit(50257, 1280, 5121, u01),),
                N=n, layout=layout, grad_dtype="f32", steps=4, grad_std=1e-2)
    # Reduced stand-ins the oracle finishes in seconds; same structure, several
    # kernel tiles per shard and ragged tails.
    for n in (1, 2, 3, 7, 8, 64):
        for layout in ("flat", "dim0"):
            name = f"ragged_mini_{layout}_n{n}"
            w[name] = Workload(
                name=name,
                description=f"Reduced ragged unit (46,572 params) {layout.upper()} at N={n}",
                units=(ragged_unit(1031, 40, 129, u01),),
                N=n, layout=layout, grad_dtype="f32", steps=4, grad_std=1e-2)
    w["gpt_mini_flat_bf16"] = Workload(
        name="gpt_mini_flat_bf16",
        description="Reduced GPT block d=128 ffn 512 (198,272 params) x2 units, N=8, bf16 grads with outliers",
        units=tuple(gpt_block(128, 512, n0006, n0006, n0006) for _ in range(2)),
        N=8, layout="flat", grad_dtype="bf16", steps=2, grad_std=1e-4,
        outlier_frac=1e-3, outlier_scale=1e3)
    w["gpt_d3072_flat_bf16"] = Workload(
        name="gpt_d3072_flat_bf16",
        description="Reduced minGPT-shaped block d=3072 ffn 12288 (113,286,144 params), N=8, bf16 grads "
                    "with outliers; a few GB on the device, every kernel's traffic far above L2",
        units=(gpt_block(3072, 12288, n0006, n0006, n0006),),
        N=8, layout="flat", grad_dtype="bf16", steps=2, grad_std=1e-4,
        outlier_frac=1e-3, outlier_scale=1e3)
    for layout in ("flat", "dim0"):
        name = f"huge_{layout}_n3"
        w[name] = Workload(
            name=name,
            description=f"One unit past 2^31 elements: W[46341x46341] + b[1000] (2,147,489,281 params), "
                        f"{layout.upper()} at N=3, bf16 grads",
            units=((Param("w", (46341, 46341), u01), Param("b", (1000,), u01)),),
            N=3, layout=layout, grad_dtype="bf16", steps=2, grad_std=1e-2)
    w["gpt_mini_dim0"] = Workload(
        name="gpt_mini_dim0",
        description="Reduced GPT block d=128 ffn 512 x2 units, DIM0, N=8",
        units=tuple(gpt_block(128, 512, n002, n002, n002) for _ in range(2)),
        N=8, layout="dim0", grad_dtype="f32", steps=3, grad_std=1e-3)
    return w


WORKLOADS = _workloads()


def get(name: str) -> Workload:
    return WORKLOADS[name]


def _seed(*parts) -> int:
    h = hashlib.sha256("/".join(str(p) for p in parts).encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


def _gen(device, *parts) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(_seed(*parts))
    return g


_CHUNK = 1 << 26


def _fill(out: torch.Tensor, init: Init, gen: torch.Generator) -> None:
    flat = out.view(-1)
    kind = init[0]
    if kind == "ones":
        flat.fill_(1.0)
        return
    if kind == "zeros":
        flat.zero_()
        return
    for a in range(0, flat.numel(), _CHUNK):
        part = flat[a:a + _CHUNK]
        if kind == "normal":
            part.normal_(0.0, init[1], generator=gen)
        elif kind == "uniform":
            part.uniform_(init[1], init[2], generator=gen)
        else:
            raise ValueError(f"unknown init {init}")


def param_tensors(wl: Workload, unit: int, device="cpu") -> list:
    """The unit's initial fp32 parameters, one tensor per parameter, in
    registration order, each drawn from its own seeded stream."""
    out = []
    for i, p in enumerate(wl.units[unit]):
        t = torch.empty(p.shape, dtype=torch.float32, device=device)
        _fill(t, p.init, _gen(device, wl.seed, wl.name, "param", unit, i))
        out.append(t)
    return out


def grad_tensor(wl: Workload, unit: int, step: int, rank: int, device="cpu",
                out: torch.Tensor | None = None) -> torch.Tensor:
    """Rank ``rank``'s full unsharded gradient for ``unit`` at ``step`` (0-based):
    a length-P vector indexed like the unit's unsharded parameters, fp32 or
    bf16 as the workload says.  Outliers (when the workload asks for them):
    each element independently, with probability ``outlier_frac``, is scaled by
    ``outlier_scale`` before the conversion to the gradient dtype."""
    P = wl.unit_numel(unit)
    dt = wl.torch_grad_dtype()
    if out is None:
        out = torch.empty(P, dtype=dt, device=device)
    assert out.numel() == P and out.dtype == dt
    g = _gen(device, wl.seed, wl.name, "grad", unit, step, rank)
    tmp = None
    for a in range(0, P, _CHUNK):
        n = min(_CHUNK, P - a)
        if tmp is None or tmp.numel() < n:
            tmp = torch.empty(min(_CHUNK, P), dtype=torch.float32, device=device)
        t = tmp[:n]
        t.normal_(0.0, wl.grad_std, generator=g)
        if wl.outlier_frac > 0.0:
            mask = torch.rand(n, device=device, generator=g) < wl.outlier_frac
            t[mask] *= wl.outlier_scale
        out[a:a + n].copy_(t)
    return out


def hyper(wl: Workload) -> dict:
    return dict(lr=wl.lr, beta1=wl.beta1, beta2=wl.beta2, eps=wl.eps,
                weight_decay=wl.weight_decay)


def names() -> Sequence[str]:
    return list(WORKLOADS)

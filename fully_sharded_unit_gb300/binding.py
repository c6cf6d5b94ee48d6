"""ctypes binding of the C ABI in ``include/fsdp_unit.h``.

Argument marshalling only: every function here has the C name, turns torch
tensors and Python values into pointers and sizes, checks that buffers are
large enough (the C side cannot see sizes), calls the library and raises
``FsdpError`` on a non-zero status.  No step of the per-unit cycle runs in
Python.  The library is loaded from the package's ``_lib`` directory; if it
is missing, every call raises (there is no fallback).
"""
from __future__ import annotations

import ctypes
import os
from typing import Sequence

import torch

from .build import LIB

# ---- constants (mirror include/fsdp_unit.h) ------------------------------
FSDP_OK = 0
FSDP_E_INVALID_ARG = -1
FSDP_E_OOM = -2
FSDP_E_CUDA = -3
FSDP_E_STATE = -4
FSDP_E_ALIGN = -5
FSDP_E_CAPACITY = -6

FSDP_LAYOUT_FLAT = 0
FSDP_LAYOUT_DIM0 = 1
FSDP_LAYOUT_FLAT_PADDED = 2
FSDP_DTYPE_F32 = 0
FSDP_DTYPE_BF16 = 1
FSDP_GATHER_FROM_MASTER = 0
FSDP_GATHER_FROM_SHADOW = 1

FSDP_STATE_PARAM = 0
FSDP_STATE_GRAD = 1
FSDP_STATE_EXP_AVG = 2
FSDP_STATE_EXP_AVG_SQ = 3
FSDP_STATE_SHADOW = 4

FSDP_KERNEL_SHARD_IN = 0
FSDP_KERNEL_GATHER = 1
FSDP_KERNEL_REDUCE_SCATTER = 2
FSDP_KERNEL_ADAMW = 3
FSDP_KERNEL_REDUCE_ADAMW = 4
FSDP_KERNEL_COUNT = 5

FSDP_KSTATUS_WAIT_TIMEOUT = 1
FSDP_KSTATUS_DRAIN_TIMEOUT = 2

FSDP_NOALLOC_MAX_TILES = 32768

LAYOUTS = {"flat": FSDP_LAYOUT_FLAT, "dim0": FSDP_LAYOUT_DIM0, "flat_padded": FSDP_LAYOUT_FLAT_PADDED}
GRAD_DTYPES = {"f32": FSDP_DTYPE_F32, "bf16": FSDP_DTYPE_BF16}
GATHER_SOURCES = {"master": FSDP_GATHER_FROM_MASTER, "shadow": FSDP_GATHER_FROM_SHADOW}
STATES = {"param": FSDP_STATE_PARAM, "grad": FSDP_STATE_GRAD, "exp_avg": FSDP_STATE_EXP_AVG,
          "exp_avg_sq": FSDP_STATE_EXP_AVG_SQ, "shadow": FSDP_STATE_SHADOW}
KERNELS = {"shard_in": FSDP_KERNEL_SHARD_IN, "gather": FSDP_KERNEL_GATHER,
           "reduce_scatter": FSDP_KERNEL_REDUCE_SCATTER, "adamw": FSDP_KERNEL_ADAMW,
           "reduce_adamw": FSDP_KERNEL_REDUCE_ADAMW}


class Segment(ctypes.Structure):
    _fields_ = [("rank", ctypes.c_int32), ("param", ctypes.c_int32), ("global_off", ctypes.c_int64),
                ("shard_off", ctypes.c_int64), ("arena_off", ctypes.c_int64), ("len", ctypes.c_int64)]


class AdamWHp(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_double), ("beta1", ctypes.c_double), ("beta2", ctypes.c_double),
                ("eps", ctypes.c_double), ("weight_decay", ctypes.c_double)]


class UnitConfig(ctypes.Structure):
    _fields_ = [("layout", ctypes.c_int), ("num_ranks", ctypes.c_int), ("grad_dtype", ctypes.c_int),
                ("reshard_after_forward", ctypes.c_int), ("replicas", ctypes.c_int),
                ("reduce_dtype", ctypes.c_int), ("gather_source", ctypes.c_int),
                ("fuse_reduce_adamw", ctypes.c_int)]


class RSOptions(ctypes.Structure):
    _fields_ = [("accumulate", ctypes.c_int), ("inv_scale", ctypes.c_double),
                ("found_nonfinite_dev", ctypes.c_void_p)]


_ALLOC_FN = ctypes.CFUNCTYPE(ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p)
_FREE_FN = ctypes.CFUNCTYPE(None, ctypes.c_void_p, ctypes.c_void_p)


class Allocator(ctypes.Structure):
    """fsdp_allocator: alloc(bytes, ctx) -> device pointer or NULL; free(ptr, ctx)."""
    _fields_ = [("alloc", _ALLOC_FN), ("free", _FREE_FN), ("ctx", ctypes.c_void_p)]


class FsdpError(RuntimeError):
    def __init__(self, code: int, where: str, detail: str):
        super().__init__(f"{where}: {detail} (code {code})")
        self.code = code


_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64
_PI64 = ctypes.POINTER(ctypes.c_int64)
_PI = ctypes.POINTER(ctypes.c_int)

_SIGNATURES = {
    "fsdp_plan_layout": (_I, [_I, _PI, _PI64, _I, _I, _PI64, _PI64, ctypes.POINTER(Segment), _I64]),
    "fsdp_unit_create": (_I, [_I, _PI, _PI64, ctypes.POINTER(UnitConfig), ctypes.POINTER(_P)]),
    "fsdp_unit_create_with_allocator": (_I, [_I, _PI, _PI64, ctypes.POINTER(UnitConfig),
                                             ctypes.POINTER(Allocator), ctypes.POINTER(_P)]),
    "fsdp_unit_destroy": (_I, [_P]),
    "fsdp_load_params": (_I, [_P, ctypes.POINTER(_P), _P]),
    "fsdp_allgather": (_I, [_P, _P, _P]),
    "fsdp_reduce_scatter": (_I, [_P, ctypes.POINTER(_P), _P]),
    "fsdp_reduce_scatter_ex": (_I, [_P, ctypes.POINTER(_P), ctypes.POINTER(RSOptions), _P]),
    "fsdp_zero_grad": (_I, [_P, _P]),
    "fsdp_adamw_step": (_I, [_P, ctypes.POINTER(AdamWHp), _P]),
    "fsdp_step": (_I, [_P, ctypes.POINTER(_P), _P, ctypes.POINTER(AdamWHp), _P]),
    "fsdp_reduce_scatter_flat_noalloc": (_I, [ctypes.POINTER(_P), _I, _I, _I64, _P, _P]),
    "fsdp_get_state": (_I, [_P, _I, _I, _P, _P]),
    "fsdp_set_state": (_I, [_P, _I, _I, _P, _P]),
    "fsdp_read_global": (_I, [_P, _I, _I64, _I64, _P, _P]),
    "fsdp_read_arena": (_I, [_P, _I, _I, _P, _PI64, _P]),
    "fsdp_unit_set_step_options": (_I, [_P, _I, _I]),
    "fsdp_adamw_device_steps": (_I, [_P, ctypes.POINTER(AdamWHp), _I64, _P]),
    "fsdp_adamw_device_status": (_I, [_P, _PI64, ctypes.POINTER(ctypes.c_int32), _P]),
    "fsdp_get_step_count": (_I, [_P, _PI64]),
    "fsdp_set_step_count": (_I, [_P, _I64]),
    "fsdp_unit_info": (_I, [_P, _PI64, ctypes.POINTER(UnitConfig)]),
    "fsdp_unit_segments": (_I, [_P, ctypes.POINTER(Segment), _I64, _PI64]),
    "fsdp_memory_report": (_I, [_P, _I, _PI64, _PI64, _PI64, _PI64, _PI64]),
    "fsdp_profile_enable": (_I, [_P, _I]),
    "fsdp_profile_read": (_I, [_P, _I, ctypes.POINTER(ctypes.c_double), _PI64]),
    "fsdp_profile_reset": (_I, [_P]),
    "fsdp_kernel_status": (_I, [_P, ctypes.POINTER(ctypes.c_int32), _P]),
    "fsdp_unit_set_wait_limit": (_I, [_P, ctypes.c_double, _I]),
    "fsdp_selftest_bounded_wait": (_I, [ctypes.c_double, ctypes.POINTER(ctypes.c_int32), _P]),
    "fsdp_host_device_pointer": (_I, [_P, ctypes.POINTER(_P)]),
    "fsdp_strerror": (ctypes.c_char_p, [_I]),
    "fsdp_last_error": (ctypes.c_char_p, []),
}

_lib = None


def lib() -> ctypes.CDLL:
    """The loaded CUDA library.  Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            raise RuntimeError(
                f"CUDA library {LIB} is not built; run fully_sharded_unit_gb300.build.build() "
                "(there is no CPU fallback)")
        l = ctypes.CDLL(LIB)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(l, name)
            fn.restype = res
            fn.argtypes = args
        _lib = l
    return _lib


def _check(rc: int, where: str) -> None:
    if rc != FSDP_OK:
        detail = lib().fsdp_last_error().decode() or lib().fsdp_strerror(rc).decode()
        raise FsdpError(rc, where, detail)


def _shape_args(shapes: Sequence[Sequence[int]]):
    nd = (ctypes.c_int * len(shapes))(*[len(s) for s in shapes])
    flat = [int(d) for s in shapes for d in s]
    dims = (ctypes.c_int64 * max(1, len(flat)))(*flat)
    return len(shapes), nd, dims


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _hp(hp) -> AdamWHp:
    if isinstance(hp, AdamWHp):
        return hp
    return AdamWHp(float(hp["lr"]), float(hp["beta1"]), float(hp["beta2"]), float(hp["eps"]),
                   float(hp["weight_decay"]))


def _ptrs(tensors) -> ctypes.Array:
    return (_P * len(tensors))(*[t.data_ptr() if t is not None else None for t in tensors])


# ---- C entry points -----------------------------------------------------

def fsdp_plan_layout(shapes, layout, num_ranks):
    """(P, [Segment, ...]) for a unit; host only."""
    n, nd, dims = _shape_args(shapes)
    P = ctypes.c_int64()
    ns = ctypes.c_int64()
    _check(lib().fsdp_plan_layout(n, nd, dims, LAYOUTS.get(layout, layout), num_ranks,
                                  ctypes.byref(P), ctypes.byref(ns), None, 0), "fsdp_plan_layout")
    segs = (Segment * max(1, ns.value))()
    _check(lib().fsdp_plan_layout(n, nd, dims, LAYOUTS.get(layout, layout), num_ranks,
                                  ctypes.byref(P), ctypes.byref(ns), segs, ns.value), "fsdp_plan_layout")
    return P.value, list(segs)[:ns.value]


def _unit_config(layout, num_ranks, grad_dtype, reshard_after_forward, replicas, reduce_dtype,
                 gather_source, fuse_reduce_adamw) -> UnitConfig:
    return UnitConfig(LAYOUTS.get(layout, layout), int(num_ranks), GRAD_DTYPES.get(grad_dtype, grad_dtype),
                      1 if reshard_after_forward else 0, int(replicas),
                      GRAD_DTYPES.get(reduce_dtype, reduce_dtype), GATHER_SOURCES.get(gather_source, gather_source),
                      1 if fuse_reduce_adamw else 0)


def fsdp_unit_create(shapes, layout, num_ranks, grad_dtype="f32", reshard_after_forward=True,
                     replicas=1, reduce_dtype="f32", gather_source="master", fuse_reduce_adamw=False):
    n, nd, dims = _shape_args(shapes)
    cfg = _unit_config(layout, num_ranks, grad_dtype, reshard_after_forward, replicas, reduce_dtype,
                       gather_source, fuse_reduce_adamw)
    h = _P()
    _check(lib().fsdp_unit_create(n, nd, dims, ctypes.byref(cfg), ctypes.byref(h)), "fsdp_unit_create")
    return h


def fsdp_unit_create_with_allocator(shapes, layout, num_ranks, allocator: Allocator, grad_dtype="f32",
                                    reshard_after_forward=True, replicas=1, reduce_dtype="f32",
                                    gather_source="master", fuse_reduce_adamw=False):
    """`allocator` is an ``Allocator`` struct; the caller keeps it (and the
    callbacks it holds) alive until the unit is destroyed."""
    n, nd, dims = _shape_args(shapes)
    cfg = _unit_config(layout, num_ranks, grad_dtype, reshard_after_forward, replicas, reduce_dtype,
                       gather_source, fuse_reduce_adamw)
    h = _P()
    _check(lib().fsdp_unit_create_with_allocator(n, nd, dims, ctypes.byref(cfg), ctypes.byref(allocator),
                                                 ctypes.byref(h)), "fsdp_unit_create_with_allocator")
    return h


class TorchAllocator:
    """Device memory for units from torch's caching allocator: each block is a
    torch uint8 tensor on the current device (torch aligns blocks to 512
    bytes), so torch.cuda.memory_allocated() counts the units' arenas and the
    memory returns to torch's pool when a unit is destroyed.  Keep this object
    alive while any unit made with it exists.  ``allocs`` / ``frees`` count the
    calls; ``live`` holds the blocks not yet freed."""

    def __init__(self):
        self.live = {}
        self.allocs = 0
        self.frees = 0

        def _alloc(nbytes, ctx):
            try:
                t = torch.empty(int(nbytes), dtype=torch.uint8, device="cuda")
            except RuntimeError:                  # out of memory: the library reports FSDP_E_OOM
                return None
            self.live[t.data_ptr()] = t
            self.allocs += 1
            return t.data_ptr()

        def _free(ptr, ctx):
            self.live.pop(ptr, None)
            self.frees += 1

        self._callbacks = (_ALLOC_FN(_alloc), _FREE_FN(_free))
        self.struct = Allocator(self._callbacks[0], self._callbacks[1], None)


def fsdp_unit_destroy(h) -> None:
    _check(lib().fsdp_unit_destroy(h), "fsdp_unit_destroy")


def fsdp_unit_info(h):
    P = ctypes.c_int64()
    cfg = UnitConfig()
    _check(lib().fsdp_unit_info(h, ctypes.byref(P), ctypes.byref(cfg)), "fsdp_unit_info")
    return dict(numel=P.value, num_ranks=cfg.num_ranks, layout=cfg.layout, grad_dtype=cfg.grad_dtype,
                reshard_after_forward=bool(cfg.reshard_after_forward), replicas=cfg.replicas,
                reduce_dtype=cfg.reduce_dtype, gather_source=cfg.gather_source,
                fuse_reduce_adamw=bool(cfg.fuse_reduce_adamw))


def fsdp_unit_segments(h):
    ns = ctypes.c_int64()
    _check(lib().fsdp_unit_segments(h, None, 0, ctypes.byref(ns)), "fsdp_unit_segments")
    segs = (Segment * max(1, ns.value))()
    _check(lib().fsdp_unit_segments(h, segs, ns.value, ctypes.byref(ns)), "fsdp_unit_segments")
    return list(segs)[:ns.value]


def fsdp_load_params(h, params, stream=None) -> None:
    for p in params:
        assert p.dtype == torch.float32 and p.is_contiguous() and (p.numel() == 0 or p.is_cuda)
    _check(lib().fsdp_load_params(h, _ptrs(params), _stream(stream)), "fsdp_load_params")


def fsdp_allgather(h, out: torch.Tensor, stream=None) -> None:
    P = fsdp_unit_info(h)["numel"]
    assert out.is_cuda and out.element_size() == 2 and out.is_contiguous() and out.numel() >= P
    _check(lib().fsdp_allgather(h, out.data_ptr(), _stream(stream)), "fsdp_allgather")


def _check_grads(h, grads):
    info = fsdp_unit_info(h)
    assert len(grads) == info["num_ranks"] * info["replicas"]
    want = torch.float32 if info["grad_dtype"] == FSDP_DTYPE_F32 else torch.bfloat16
    for g in grads:
        assert g.is_cuda and g.is_contiguous() and g.numel() >= info["numel"]
        assert g.dtype == want, f"gradient dtype {g.dtype}, unit expects {want}"


def fsdp_reduce_scatter(h, grads, stream=None) -> None:
    _check_grads(h, grads)
    _check(lib().fsdp_reduce_scatter(h, _ptrs(grads), _stream(stream)), "fsdp_reduce_scatter")


def fsdp_reduce_scatter_ex(h, grads, accumulate=False, inv_scale=1.0, found: torch.Tensor | None = None,
                           stream=None) -> None:
    """``found``: optional one-element int32 CUDA tensor for the found-non-finite flag."""
    _check_grads(h, grads)
    if found is not None:
        assert found.is_cuda and found.dtype == torch.int32 and found.numel() >= 1
    opt = RSOptions(1 if accumulate else 0, float(inv_scale), found.data_ptr() if found is not None else None)
    _check(lib().fsdp_reduce_scatter_ex(h, _ptrs(grads), ctypes.byref(opt), _stream(stream)),
           "fsdp_reduce_scatter_ex")


def fsdp_zero_grad(h, stream=None) -> None:
    _check(lib().fsdp_zero_grad(h, _stream(stream)), "fsdp_zero_grad")


def fsdp_adamw_step(h, hp, stream=None) -> None:
    hp = _hp(hp)
    _check(lib().fsdp_adamw_step(h, ctypes.byref(hp), _stream(stream)), "fsdp_adamw_step")


def fsdp_step(h, grads, out: torch.Tensor, hp, stream=None) -> None:
    _check_grads(h, grads)
    P = fsdp_unit_info(h)["numel"]
    assert out.is_cuda and out.element_size() == 2 and out.is_contiguous() and out.numel() >= P
    hp = _hp(hp)
    _check(lib().fsdp_step(h, _ptrs(grads), out.data_ptr(), ctypes.byref(hp), _stream(stream)),
           "fsdp_step")


def fsdp_reduce_scatter_flat_noalloc(grads, out: torch.Tensor, numel: int | None = None, stream=None) -> None:
    """The FLAT reduce-scatter that allocates nothing: ``grads`` are the N
    ranks' full gradients (fp32 or bf16 CUDA tensors of one dtype), ``out`` an
    fp32 CUDA tensor that receives every rank's shard back to back (rank k's at
    [floor(k*numel/N), floor((k+1)*numel/N))).  ``numel`` defaults to
    out.numel()."""
    numel = out.numel() if numel is None else int(numel)
    assert len(grads) >= 1 and len({g.dtype for g in grads}) == 1
    dt = grads[0].dtype
    assert dt in (torch.float32, torch.bfloat16), f"gradient dtype {dt}"
    for g in grads:
        assert g.is_cuda and g.is_contiguous() and g.numel() >= numel
    assert out.is_cuda and out.is_contiguous() and out.dtype == torch.float32 and out.numel() >= numel
    gd = FSDP_DTYPE_F32 if dt == torch.float32 else FSDP_DTYPE_BF16
    _check(lib().fsdp_reduce_scatter_flat_noalloc(_ptrs(grads), len(grads), gd, numel, out.data_ptr(),
                                                  _stream(stream)), "fsdp_reduce_scatter_flat_noalloc")


def _shard_len(h, rank):
    return sum(s.len for s in fsdp_unit_segments(h) if s.rank == rank)


def fsdp_get_state(h, which, rank, dst: torch.Tensor, stream=None) -> None:
    which = STATES.get(which, which)
    assert dst.is_contiguous() and dst.element_size() == (2 if which == FSDP_STATE_SHADOW else 4)
    assert dst.numel() >= _shard_len(h, rank)
    _check(lib().fsdp_get_state(h, which, rank, dst.data_ptr(), _stream(stream)), "fsdp_get_state")


def fsdp_set_state(h, which, rank, src: torch.Tensor, stream=None) -> None:
    which = STATES.get(which, which)
    assert src.is_contiguous() and src.element_size() == (2 if which == FSDP_STATE_SHADOW else 4)
    assert src.numel() >= _shard_len(h, rank)
    _check(lib().fsdp_set_state(h, which, rank, src.data_ptr(), _stream(stream)), "fsdp_set_state")


def fsdp_read_global(h, which, begin, count, dst: torch.Tensor, stream=None) -> None:
    which = STATES.get(which, which)
    assert dst.is_contiguous() and dst.element_size() == (2 if which == FSDP_STATE_SHADOW else 4)
    assert dst.numel() >= count
    _check(lib().fsdp_read_global(h, which, int(begin), int(count), dst.data_ptr(), _stream(stream)),
           "fsdp_read_global")


def fsdp_read_arena(h, which, rank, stream=None) -> torch.Tensor:
    """Rank ``rank``'s whole arena of state ``which`` (pads included), on the device."""
    which = STATES.get(which, which)
    n = ctypes.c_int64()
    _check(lib().fsdp_read_arena(h, which, rank, None, ctypes.byref(n), _stream(stream)), "fsdp_read_arena")
    dt = torch.int16 if which == FSDP_STATE_SHADOW else torch.float32
    dst = torch.empty(n.value, dtype=dt, device="cuda")
    if n.value:
        _check(lib().fsdp_read_arena(h, which, rank, dst.data_ptr(), None, _stream(stream)), "fsdp_read_arena")
    return dst


def fsdp_unit_set_step_options(h, gather_source="master", fuse_reduce_adamw=False) -> None:
    _check(lib().fsdp_unit_set_step_options(h, GATHER_SOURCES.get(gather_source, gather_source),
                                            1 if fuse_reduce_adamw else 0), "fsdp_unit_set_step_options")


def fsdp_adamw_device_steps(h, hp, count, stream=None) -> None:
    hpv = _hp(hp) if hp is not None else None
    _check(lib().fsdp_adamw_device_steps(h, ctypes.byref(hpv) if hpv is not None else None, int(count),
                                         _stream(stream)), "fsdp_adamw_device_steps")


def fsdp_adamw_device_status(h, stream=None):
    t = ctypes.c_int64()
    ex = ctypes.c_int32()
    _check(lib().fsdp_adamw_device_status(h, ctypes.byref(t), ctypes.byref(ex), _stream(stream)),
           "fsdp_adamw_device_status")
    return t.value, bool(ex.value)


def fsdp_get_step_count(h) -> int:
    t = ctypes.c_int64()
    _check(lib().fsdp_get_step_count(h, ctypes.byref(t)), "fsdp_get_step_count")
    return t.value


def fsdp_set_step_count(h, t: int) -> None:
    _check(lib().fsdp_set_step_count(h, int(t)), "fsdp_set_step_count")


def fsdp_memory_report(h, rank):
    vals = [ctypes.c_int64() for _ in range(5)]
    _check(lib().fsdp_memory_report(h, rank, *[ctypes.byref(v) for v in vals]), "fsdp_memory_report")
    return dict(zip(("param", "grad", "adam", "shadow", "pad"), (v.value for v in vals)))


def fsdp_kernel_status(h, stream=None) -> int:
    """FSDP_KSTATUS_* bits raised since the last call (0: none); clears them."""
    f = ctypes.c_int32()
    _check(lib().fsdp_kernel_status(h, ctypes.byref(f), _stream(stream)), "fsdp_kernel_status")
    return f.value


def fsdp_unit_set_wait_limit(h, seconds=10.0, withhold_next=0) -> None:
    """``withhold_next``: 0, 1 (one wait runs out) or 2 (the drain's wait too)."""
    _check(lib().fsdp_unit_set_wait_limit(h, float(seconds), int(withhold_next)), "fsdp_unit_set_wait_limit")


def fsdp_selftest_bounded_wait(limit_seconds=0.05, stream=None) -> bool:
    """True when a wait that nothing completes ran out and reported it."""
    t = ctypes.c_int32()
    _check(lib().fsdp_selftest_bounded_wait(float(limit_seconds), ctypes.byref(t), _stream(stream)),
           "fsdp_selftest_bounded_wait")
    return bool(t.value)


def fsdp_profile_enable(h, on=True) -> None:
    _check(lib().fsdp_profile_enable(h, 1 if on else 0), "fsdp_profile_enable")


def fsdp_profile_read(h, kernel):
    ms = ctypes.c_double()
    n = ctypes.c_int64()
    _check(lib().fsdp_profile_read(h, KERNELS.get(kernel, kernel), ctypes.byref(ms), ctypes.byref(n)),
           "fsdp_profile_read")
    return ms.value, n.value


def fsdp_profile_reset(h) -> None:
    _check(lib().fsdp_profile_reset(h), "fsdp_profile_reset")


class DevicePtr:
    """A raw device address standing in for a tensor in calls that take buffers."""

    def __init__(self, addr: int, like: torch.Tensor):
        self.addr = addr
        self.dtype = like.dtype
        self.is_cuda = True
        self._like = like          # keeps the host memory alive

    def data_ptr(self) -> int:
        return self.addr

    def numel(self) -> int:
        return self._like.numel()

    def is_contiguous(self) -> bool:
        return self._like.is_contiguous()


def fsdp_host_device_pointer(host: torch.Tensor) -> DevicePtr:
    """Device view of a pinned host tensor (read over the host link)."""
    d = _P()
    _check(lib().fsdp_host_device_pointer(host.data_ptr(), ctypes.byref(d)), "fsdp_host_device_pointer")
    return DevicePtr(d.value, host)


def fsdp_strerror(code: int) -> str:
    return lib().fsdp_strerror(code).decode()


def fsdp_last_error() -> str:
    return lib().fsdp_last_error().decode()


# ---- a small owning wrapper ----------------------------------------------

class Unit:
    """Owns one ``fsdp_unit`` handle; methods call the C entry points."""

    def __init__(self, shapes, layout="flat", num_ranks=1, grad_dtype="f32", reshard_after_forward=True,
                 replicas=1, reduce_dtype="f32", gather_source="master", fuse_reduce_adamw=False,
                 allocator=None):
        """`allocator`: None (the library's cudaMalloc) or an object with an
        ``Allocator`` in its ``struct`` attribute, e.g. ``TorchAllocator()``."""
        self.shapes = [tuple(int(d) for d in s) for s in shapes]
        self.allocator = allocator
        if allocator is None:
            self.handle = fsdp_unit_create(self.shapes, layout, num_ranks, grad_dtype, reshard_after_forward,
                                           replicas, reduce_dtype, gather_source, fuse_reduce_adamw)
        else:
            self.handle = fsdp_unit_create_with_allocator(self.shapes, layout, num_ranks, allocator.struct,
                                                          grad_dtype, reshard_after_forward, replicas,
                                                          reduce_dtype, gather_source, fuse_reduce_adamw)
        info = fsdp_unit_info(self.handle)
        self.numel = info["numel"]
        self.N = info["num_ranks"]
        self.replicas = info["replicas"]
        self.grad_dtype = grad_dtype
        self.segments = fsdp_unit_segments(self.handle)
        self._step_key = None
        self._hp_key = None
        self.shard_len = [0] * self.N
        for s in self.segments:
            self.shard_len[s.rank] += s.len

    def close(self):
        if self.handle is not None:
            fsdp_unit_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def load(self, params, stream=None):
        fsdp_load_params(self.handle, params, stream)

    def allgather(self, out, stream=None):
        fsdp_allgather(self.handle, out, stream)

    def reduce_scatter(self, grads, stream=None):
        fsdp_reduce_scatter(self.handle, grads, stream)

    def reduce_scatter_ex(self, grads, accumulate=False, inv_scale=1.0, found=None, stream=None):
        fsdp_reduce_scatter_ex(self.handle, grads, accumulate, inv_scale, found, stream)

    def zero_grad(self, stream=None):
        fsdp_zero_grad(self.handle, stream)

    def adamw_step(self, hp, stream=None):
        fsdp_adamw_step(self.handle, hp, stream)

    def step(self, grads, out, hp, stream=None):
        """fsdp_step.  The pointer array and the hyper-parameter struct are
        cached by buffer address and values, so repeated steps over the same
        buffers skip re-validation and re-marshalling."""
        key = (out.data_ptr(), out.numel(), out.dtype, *[(g.data_ptr(), g.numel(), g.dtype) for g in grads])
        if key != self._step_key:
            _check_grads(self.handle, grads)
            assert out.is_cuda and out.element_size() == 2 and out.is_contiguous() and out.numel() >= self.numel
            self._step_ptrs = _ptrs(grads)
            self._step_key = key
        hkey = tuple(hp.values()) if isinstance(hp, dict) else id(hp)
        if hkey != self._hp_key:
            self._hp_struct = _hp(hp)
            self._hp_key = hkey
        _check(lib().fsdp_step(self.handle, self._step_ptrs, out.data_ptr(), ctypes.byref(self._hp_struct),
                               _stream(stream)), "fsdp_step")

    def get_state(self, which, rank, device="cuda"):
        dt = torch.int16 if STATES.get(which, which) == FSDP_STATE_SHADOW else torch.float32
        dst = torch.empty(self.shard_len[rank], dtype=dt, device=device)
        if dst.numel():
            fsdp_get_state(self.handle, which, rank, dst)
        return dst

    def set_state(self, which, rank, src, stream=None):
        fsdp_set_state(self.handle, which, rank, src, stream)

    def read_global(self, which, begin=0, count=None, device="cuda"):
        count = self.numel - begin if count is None else count
        dt = torch.int16 if STATES.get(which, which) == FSDP_STATE_SHADOW else torch.float32
        dst = torch.empty(count, dtype=dt, device=device)
        fsdp_read_global(self.handle, which, begin, count, dst)
        return dst

    @property
    def step_count(self):
        return fsdp_get_step_count(self.handle)

    @step_count.setter
    def step_count(self, t):
        fsdp_set_step_count(self.handle, t)

    def memory_report(self, rank):
        return fsdp_memory_report(self.handle, rank)

    def kernel_status(self, stream=None) -> int:
        return fsdp_kernel_status(self.handle, stream)

    def set_wait_limit(self, seconds=10.0, withhold_next=0) -> None:
        fsdp_unit_set_wait_limit(self.handle, seconds, withhold_next)

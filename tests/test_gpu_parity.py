"""GPU parity on the reduced workloads: every element, every step, through the C ABI."""
import numpy as np
import pytest
import torch

from fully_sharded_unit_gb300 import binding as B
from fully_sharded_unit_gb300 import workloads
from oracle import fsdp_oracle as O

import gpu_harness as H

pytestmark = pytest.mark.gpu

MINI = sorted(n for n in workloads.WORKLOADS if n.startswith("ragged_mini"))


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from conftest import library
    library()


def test_tiny_config_individual_calls():
    cmp = H.run_full(workloads.get("tiny_flat"))
    assert cmp.total_diff == 0


def test_tiny_config_through_fsdp_step():
    H.run_full(workloads.get("tiny_flat"), use_step=True)


@pytest.mark.parametrize("name", MINI)
def test_ragged_mini(name):
    H.run_full(workloads.get(name))


@pytest.mark.parametrize("name", ["gpt_mini_flat_bf16", "gpt_mini_dim0"])
def test_gpt_mini(name):
    H.run_full(workloads.get(name))
    H.run_full(workloads.get(name), unit=1, use_step=True)


def test_adamw_is_bit_identical_to_the_oracle():
    """The kernel evaluates the oracle's fp32 operation sequence with explicitly
    rounded operations, so beyond the tolerance it matches bit for bit."""
    for name in ("ragged_mini_dim0_n7", "gpt_mini_flat_bf16"):
        cmp = H.run_full(workloads.get(name))
        assert cmp.total_diff == 0, cmp.adamw


def _custom(shapes, N, layout, grad_dtype="f32", steps=3, raf=True, name="custom"):
    init = ("uniform", -0.5, 0.5)
    units = (tuple(workloads.Param(f"p{i}", tuple(s), init) for i, s in enumerate(shapes)),)
    return workloads.Workload(name=name, description=name, units=units, N=N, layout=layout,
                              grad_dtype=grad_dtype, steps=steps, grad_std=1e-2,
                              reshard_after_forward=raf)


@pytest.mark.parametrize("layout", ["flat", "dim0"])
@pytest.mark.parametrize("shapes,N", [
    ([(1,)], 1), ([(1,)], 5), ([(3, 4), (3,)], 16), ([(5,)], 64), ([(2, 3), ()], 3),
    ([(0, 7), (9, 2), (0,)], 4), ([(8193,)], 3), ([(16384 + 5, 3)], 7), ([(40, 50)], 100),
])
def test_edge_shapes(shapes, N, layout):
    """Fewer elements than ranks (empty ranks), one element, zero-size
    parameters, more than 64 ranks, shards that straddle tile boundaries."""
    H.run_full(_custom(shapes, N, layout, raf=(N % 2 == 1)))
    H.run_full(_custom(shapes, N, layout, grad_dtype="bf16", name="custom_bf16"), use_step=True)


@pytest.mark.parametrize("layout,N,R,grad_dtype,kw", [
    ("flat", 1024, 1, "f32", {}),                                   # the most ranks a unit takes
    ("dim0", 1024, 1, "bf16", {}),                                  # fewer dim-0 rows than ranks
    ("flat", 1024, 1, "bf16", {"reduce_dtype": "bf16"}),
    ("flat", 1024, 1, "f32", {"fuse_reduce_adamw": True}),          # register-staged fused kernel
    ("flat", 64, 16, "f32", {}),                                    # hybrid: W = 1024 gradients
    ("dim0", 128, 8, "bf16", {"fuse_reduce_adamw": True}),          # hybrid fused, W = 1024
])
def test_maximum_rank_count(layout, N, R, grad_dtype, kw):
    """W = N * replicas = 1024, the library's maximum: 1024 gradient pointers
    per launch, ranks whose shards are a few elements or empty."""
    wl = _custom([(300, 257), (1000,), (7, 3)], N, layout, grad_dtype=grad_dtype, steps=2,
                 name=f"max_ranks_{grad_dtype}").with_(replicas=R, **kw)
    cmp = H.run_full(wl, use_step=True)
    assert cmp.total_diff == 0


def test_no_reshard_after_forward_gathers_once():
    H.run_full(_custom([(77, 5)], 4, "flat", raf=False), use_step=True)
    H.run_full(_custom([(77, 5)], 4, "dim0", raf=False))


def test_special_values_cast_and_reduce():
    """Gather of inf, NaN, -0, subnormals and ties; reduce-scatter of infinities."""
    vals = np.array([0x7F800000, 0xFF800000, 0x7FC00000, 0x80000000, 0x00000001, 0x00008000,
                     0x00018000, 0x3F808000, 0x3F818000, 0x7F7FFFFF, 0xFF7FFFFF, 0x0080FFFF] * 11,
                    np.uint32)
    x = vals.view(np.float32)
    u = B.Unit([(x.size,)], "flat", 5)
    try:
        u.load([torch.from_numpy(x.copy()).cuda()])
        out = torch.empty(x.size, dtype=torch.int16, device="cuda")
        u.allgather(out)
        torch.cuda.synchronize()
        H.assert_bits_equal(H.u16(out), O.bf16_rne(x), "special-value gather")
        grads = [torch.from_numpy(np.full(x.size, v, np.float32)).cuda() for v in (1.0, np.inf, -np.inf, 2.0, 0.5)]
        u.reduce_scatter(grads)
        torch.cuda.synchronize()
        got = u.read_global("grad").cpu().numpy()
        with np.errstate(invalid="ignore"):                  # inf + (-inf) is NaN, as intended
            want = O.reduce_full([g.cpu().numpy() for g in grads])
        assert np.isnan(want).all() and np.isnan(got).all()
    finally:
        u.close()


def test_checkpoint_resume_equals_uninterrupted_run():
    """k steps, export every rank's state, import into a new unit, continue:
    identical to an uninterrupted run, bit for bit."""
    wl = workloads.get("ragged_mini_dim0_n7")
    shapes, N, P = wl.shapes(0), wl.N, wl.unit_numel(0)
    hp = workloads.hyper(wl)
    params = [p.cuda() for p in workloads.param_tensors(wl, 0)]
    grads = [[workloads.grad_tensor(wl, 0, s, r).cuda() for r in range(N)] for s in range(4)]
    out = torch.empty(P, dtype=torch.int16, device="cuda")
    a = B.Unit(shapes, "dim0", N)
    a.load(params)
    for s in range(4):
        a.step(grads[s], out, hp)
    b = B.Unit(shapes, "dim0", N)
    b.load(params)
    for s in range(2):
        b.step(grads[s], out, hp)
    saved = {(w, k): b.get_state(w, k).clone() for w in B.STATES for k in range(N)}
    t = b.step_count
    b.close()
    c = B.Unit(shapes, "dim0", N)
    c.load(params)
    for (w, k), v in saved.items():
        if v.numel():
            c.set_state(w, k, v)
    c.step_count = t
    for s in range(2, 4):
        c.step(grads[s], out, hp)
    torch.cuda.synchronize()
    for w in B.STATES:
        for k in range(N):
            assert torch.equal(a.get_state(w, k), c.get_state(w, k)), (w, k)
    a.close()
    c.close()


def test_memory_report_is_16_bytes_per_owned_element():
    wl = workloads.get("ragged_mini_flat_n7")
    u = B.Unit(wl.shapes(0), "flat", 7)
    orc = O.UnitOracle(wl.shapes(0), 7, "flat")
    try:
        tot = 0
        for k in range(7):
            r = u.memory_report(k)
            want = orc.memory_bytes(k)
            assert (r["param"], r["grad"], r["adam"], r["shadow"]) == \
                (want["param"], want["grad"], want["adam"], want["shadow"])
            tot += r["param"] + r["grad"] + r["adam"]
            assert 0 <= r["pad"] < 2 * 32 * 18
        assert tot == 16 * wl.unit_numel(0)
    finally:
        u.close()


def test_host_checks_reject_bad_calls():
    u = B.Unit([(100,)], "flat", 2)
    try:
        out = torch.empty(128, dtype=torch.int16, device="cuda")
        with pytest.raises(B.FsdpError) as e:
            u.allgather(out)                           # before load
        assert e.value.code == B.FSDP_E_STATE
        u.load([torch.zeros(100, device="cuda")])
        with pytest.raises(B.FsdpError) as e:
            B.fsdp_allgather(u.handle, out[4:])        # 8-byte offset: not 32-byte aligned
        assert e.value.code == B.FSDP_E_ALIGN
        g = torch.zeros(2, 136, device="cuda")
        with pytest.raises(B.FsdpError) as e:
            B.fsdp_reduce_scatter(u.handle, [g[0], g[1, 1:]])
        assert e.value.code == B.FSDP_E_ALIGN
        with pytest.raises(B.FsdpError) as e:
            u.adamw_step(dict(lr=1e-3, beta1=1.0, beta2=0.999, eps=1e-8, weight_decay=0.0))
        assert e.value.code == B.FSDP_E_INVALID_ARG
        assert u.step_count == 0                        # nothing was enqueued
    finally:
        u.close()


def test_profiler_counts_launches():
    wl = workloads.get("ragged_mini_flat_n8")
    u = B.Unit(wl.shapes(0), "flat", 8)
    try:
        u.load([p.cuda() for p in workloads.param_tensors(wl, 0)])
        grads = [workloads.grad_tensor(wl, 0, 0, r).cuda() for r in range(8)]
        out = torch.empty(wl.unit_numel(0), dtype=torch.int16, device="cuda")
        B.fsdp_profile_enable(u.handle, True)
        for _ in range(3):
            u.step(grads, out, workloads.hyper(wl))
        counts = {k: B.fsdp_profile_read(u.handle, k) for k in B.KERNELS}
        assert counts["gather"][1] == 6 and counts["reduce_scatter"][1] == 3 and counts["adamw"][1] == 3
        assert all(ms > 0 for ms, n in counts.values() if n)
        B.fsdp_profile_reset(u.handle)
        assert B.fsdp_profile_read(u.handle, "adamw") == (0.0, 0)
    finally:
        u.close()

"""The shared-memory staged kernels' give-up path, run for real without any
fault: a one-shot test request (fsdp_unit_set_wait_limit) makes CTA 0 arm the
barrier of its first stage without issuing that stage's copies, so its wait
runs out after a short limit exactly as for a copy that never arrives.  The
kernel must raise FSDP_KSTATUS_WAIT_TIMEOUT (and, when the drain is made to
wait on the same stage, FSDP_KSTATUS_DRAIN_TIMEOUT), return, leave the context
usable, and the library must then refuse further steps on the unit until it
is reloaded (or, after a drain timeout, destroyed).  A reloaded unit must step
bit for bit like the oracle."""
import pytest
import torch

from fully_sharded_unit_gb300 import binding as B
from fully_sharded_unit_gb300 import workloads
from oracle import fsdp_oracle as O

import gpu_harness as H

pytestmark = pytest.mark.gpu

LIMIT_S = 0.02


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from conftest import library
    library()


# each case runs a different staged kernel: the fused reduce-scatter + AdamW of
# fsdp_step, the staged reduce-scatter accumulating, and under hybrid sharding
CASES = {
    "fused_step": dict(kw=dict(fuse_reduce_adamw=True), call="step"),
    "reduce_scatter_accumulate": dict(kw={}, call="accumulate"),
    "reduce_scatter_hybrid": dict(kw=dict(N=4, replicas=2), call="reduce_scatter"),
}


def _workload(case):
    base = workloads.get("gpt_mini_flat_bf16")
    return base.with_(units=(base.units[0],), **CASES[case]["kw"])


def _unit(wl):
    return B.Unit(wl.shapes(0), wl.layout, wl.N, wl.grad_dtype, wl.reshard_after_forward, replicas=wl.replicas,
                  fuse_reduce_adamw=wl.fuse_reduce_adamw)


def _launch(case, u, grads, out, hp):
    call = CASES[case]["call"]
    if call == "step":
        u.step(grads, out, hp)
    elif call == "accumulate":
        u.reduce_scatter_ex(grads, accumulate=True)
    else:
        u.reduce_scatter(grads)


@pytest.mark.parametrize("mode", [1, 2])
@pytest.mark.parametrize("case", list(CASES))
def test_a_wait_that_runs_out_is_reported_and_blocks_the_unit(case, mode):
    wl = _workload(case)
    hp = workloads.hyper(wl)
    params = [p.cuda() for p in workloads.param_tensors(wl, 0)]
    grads = [workloads.grad_tensor(wl, 0, 0, r, "cuda") for r in range(wl.world)]
    out = torch.empty(wl.unit_numel(0), dtype=torch.int16, device="cuda")
    u = _unit(wl)
    try:
        u.load(params)
        u.set_wait_limit(LIMIT_S, withhold_next=mode)
        _launch(case, u, grads, out, hp)
        flags = u.kernel_status()
        want = B.FSDP_KSTATUS_WAIT_TIMEOUT | (B.FSDP_KSTATUS_DRAIN_TIMEOUT if mode == 2 else 0)
        assert flags == want, f"status {flags}, expected {want}"
        assert u.kernel_status() == 0, "reading the status clears it"
        for refused in (lambda: u.step(grads, out, hp), lambda: u.reduce_scatter(grads),
                        lambda: u.allgather(out), lambda: u.adamw_step(hp)):
            with pytest.raises(B.FsdpError) as e:
                refused()
            assert e.value.code == B.FSDP_E_STATE
        if mode == 2:
            with pytest.raises(B.FsdpError) as e:      # only destroy (and queries) after a drain timeout
                u.load(params)
            assert e.value.code == B.FSDP_E_STATE
            assert u.numel == wl.unit_numel(0)
    finally:
        u.close()
    # the context is still usable: a fresh unit steps normally
    torch.cuda.synchronize()


@pytest.mark.parametrize("case", list(CASES))
def test_a_reloaded_unit_steps_like_the_oracle(case):
    wl = _workload(case).with_(steps=2)
    hp = workloads.hyper(wl)
    params = workloads.param_tensors(wl, 0)
    u = _unit(wl)
    try:
        u.load([p.cuda() for p in params])
        g0 = [workloads.grad_tensor(wl, 0, 0, r, "cuda") for r in range(wl.world)]
        out = torch.empty(wl.unit_numel(0), dtype=torch.int16, device="cuda")
        u.set_wait_limit(LIMIT_S, withhold_next=1)
        _launch(case, u, g0, out, hp)
        assert u.kernel_status() == B.FSDP_KSTATUS_WAIT_TIMEOUT
        u.load([p.cuda() for p in params])                  # reload: the unit is usable again
        u.set_wait_limit(10.0)
        orc = O.UnitOracle(wl.shapes(0), wl.N, wl.layout, O.AdamWHyper(**hp), wl.reshard_after_forward,
                           replicas=wl.replicas)
        orc.load([p.numpy() for p in params])
        for s in range(wl.steps):
            grads = [workloads.grad_tensor(wl, 0, s, r, "cuda") for r in range(wl.world)]
            want = orc.step([H.grad_np(g) for g in grads])
            u.step(grads, out, hp)
            torch.cuda.synchronize()
            H.assert_bits_equal(H.u16(out), want[-1], f"step {s} gathered")
        for k in range(wl.N):
            for which, ref in (("param", orc.master[k]), ("grad", orc.grad[k]), ("exp_avg", orc.m[k]),
                               ("exp_avg_sq", orc.v[k])):
                H.assert_bits_equal(u.get_state(which, k).cpu().numpy(), ref, f"{which} rank {k}")
        assert u.kernel_status() == 0
        assert u.step_count == wl.steps
    finally:
        u.close()


def test_wait_limit_arguments_are_checked():
    wl = _workload("fused_step")
    u = _unit(wl)
    try:
        for bad in (0.0, 1e-7, 61.0, float("nan")):
            with pytest.raises(B.FsdpError) as e:
                u.set_wait_limit(bad)
            assert e.value.code == B.FSDP_E_INVALID_ARG
        with pytest.raises(B.FsdpError):
            u.set_wait_limit(1.0, withhold_next=3)
        u.set_wait_limit(1.0)
    finally:
        u.close()

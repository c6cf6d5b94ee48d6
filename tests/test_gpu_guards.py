"""Guard bands: every arena element outside a rank's segments (alignment pads
and the padded layout's chunk padding) is zero from creation and must still be
zero after any sequence of calls, and nothing is written past the end of the
gathered output.  A non-zero pad or a changed canary means a kernel wrote
outside its range."""
import pytest
import torch

from fully_sharded_unit_gb300 import binding as B
from fully_sharded_unit_gb300 import workloads

pytestmark = pytest.mark.gpu

CANARY = 0x5A5A


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from conftest import library
    library()


def _pads_are_zero(u):
    for which in B.STATES:
        for k in range(u.N):
            arena = B.fsdp_read_arena(u.handle, which, k)
            mask = torch.ones(arena.numel(), dtype=torch.bool, device="cuda")
            for s in u.segments:
                if s.rank == k:
                    mask[s.arena_off:s.arena_off + s.len] = False
            bad = arena[mask] != 0
            assert not bad.any(), f"{which} rank {k}: {int(bad.sum())} non-zero pad elements"


@pytest.mark.parametrize("name,kw", [
    ("ragged_mini_flat_n7", {}), ("ragged_mini_dim0_n64", {}), ("gpt_mini_flat_bf16", {"fuse_reduce_adamw": True}),
    ("ragged_mini_flat_n3", {"layout": "flat_padded", "gather_source": "shadow"}),
    ("ragged_mini_dim0_n7", {"replicas": 2, "reduce_dtype": "f32"}),
    ("ragged_mini_flat_n8", {"reduce_dtype": "bf16", "fuse_reduce_adamw": True}),
    ("ragged_mini_dim0_n3", {"fuse_reduce_adamw": True}),           # fp32, W = 3: shared-memory staged
])
def test_pads_stay_zero_and_output_canary_holds(name, kw):
    wl = workloads.get(name).with_(**kw)
    u = B.Unit(wl.shapes(0), wl.layout, wl.N, wl.grad_dtype, wl.reshard_after_forward, replicas=wl.replicas,
               reduce_dtype=wl.reduce_dtype, gather_source=wl.gather_source,
               fuse_reduce_adamw=wl.fuse_reduce_adamw)
    try:
        P = u.numel
        u.load([p.cuda() for p in workloads.param_tensors(wl, 0)])
        torch.cuda.synchronize()
        _pads_are_zero(u)
        out = torch.full((P + 64,), CANARY, dtype=torch.int16, device="cuda")
        found = torch.zeros(1, dtype=torch.int32, device="cuda")
        for s in range(3):
            grads = [workloads.grad_tensor(wl, 0, s, r).cuda() for r in range(wl.world)]
            u.step(grads, out[:P], workloads.hyper(wl))
            u.allgather(out[:P])
            u.reduce_scatter_ex(grads, accumulate=True, inv_scale=0.5, found=found)
            if wl.replicas == 1:
                u.set_state("param", 0, u.get_state("param", 0))
            u.adamw_step(workloads.hyper(wl))
        torch.cuda.synchronize()
        assert torch.all(out[P:] == CANARY), "gathered output overran its P elements"
        _pads_are_zero(u)
    finally:
        u.close()


def test_bounded_wait_runs_out_and_reports():
    """A wait that nothing completes gives up after its limit, the status
    comes back to the host, and the context stays usable."""
    import time
    t0 = time.perf_counter()
    assert B.fsdp_selftest_bounded_wait(0.05)
    assert time.perf_counter() - t0 >= 0.05
    wl = workloads.get("gpt_mini_flat_bf16").with_(fuse_reduce_adamw=True)
    u = B.Unit(wl.shapes(0), "flat", wl.N, "bf16", fuse_reduce_adamw=True)
    try:
        u.load([p.cuda() for p in workloads.param_tensors(wl, 0)])
        grads = [workloads.grad_tensor(wl, 0, 0, r).cuda() for r in range(wl.N)]
        out = torch.empty(wl.unit_numel(0), dtype=torch.int16, device="cuda")
        u.step(grads, out, workloads.hyper(wl))
        assert u.kernel_status() == 0
        assert torch.isfinite(u.read_global("param")).all()
    finally:
        u.close()

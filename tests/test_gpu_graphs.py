"""CUDA-graph replay of fsdp_step with the device-side AdamW step counter:
replays give exactly the results of ordinary calls, an exhausted constant
table leaves the state untouched and raises the status, and leaving the mode
hands the step count back to the host."""
import pytest
import torch

from fully_sharded_unit_gb300 import binding as B
from fully_sharded_unit_gb300 import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from conftest import library
    library()


def _units(wl, **kw):
    return [B.Unit(wl.shapes(i), wl.layout, wl.N, wl.grad_dtype, wl.reshard_after_forward, **kw)
            for i in range(wl.n_units)]


def _state(u):
    return {w: u.read_global(w).clone() for w in B.STATES}


@pytest.mark.parametrize("name,kw", [("gpt_mini_flat_bf16", {}), ("gpt_mini_dim0", {"fuse_reduce_adamw": True}),
                                     ("ragged_mini_flat_n7", {"gather_source": "shadow"}),
                                     ("gpt_mini_flat_bf16", {"replicas": 2}),
                                     ("gpt_mini_flat_bf16", {"replicas": 2, "fuse_reduce_adamw": True})])
def test_graph_replay_equals_ordinary_steps(name, kw):
    """Also with the shared-memory staged kernels inside the graph (the fused
    step, and the reduce-scatter of hybrid sharding)."""
    wl = workloads.get(name).with_(replicas=kw.get("replicas", 1))
    hp = workloads.hyper(wl)
    steps = 4
    ref, gra = _units(wl, **kw), _units(wl, **kw)
    P = max(u.numel for u in ref)
    grads = [[[workloads.grad_tensor(wl, i, s, r).cuda() for r in range(wl.world)] for i in range(wl.n_units)]
             for s in range(steps + 1)]
    bufs = [[torch.empty_like(g) for g in grads[0][i]] for i in range(wl.n_units)]
    out_r = torch.empty(P, dtype=torch.int16, device="cuda")
    out_g = torch.empty(P, dtype=torch.int16, device="cuda")
    try:
        for i in range(wl.n_units):
            params = [p.cuda() for p in workloads.param_tensors(wl, i)]
            ref[i].load(params)
            gra[i].load(params)
        # one ordinary step on both (also loads every kernel before capture)
        for i in range(wl.n_units):
            ref[i].step(grads[0][i], out_r[:ref[i].numel], hp)
            gra[i].step(grads[0][i], out_g[:gra[i].numel], hp)
        for u in gra:
            B.fsdp_adamw_device_steps(u.handle, hp, steps)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for i, u in enumerate(gra):
                u.step(bufs[i], out_g[:u.numel], hp)
        for s in range(1, steps + 1):
            for i in range(wl.n_units):
                ref[i].step(grads[s][i], out_r[:ref[i].numel], hp)
                for b, g in zip(bufs[i], grads[s][i]):
                    b.copy_(g)
            graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out_r, out_g)
        for r, g in zip(ref, gra):
            assert B.fsdp_adamw_device_status(g.handle) == (1 + steps, False)
            sr, sg = _state(r), _state(g)
            for w in B.STATES:
                assert torch.equal(sr[w], sg[w]), w
        for g in gra:   # leaving the mode hands the count back to the host
            B.fsdp_adamw_device_steps(g.handle, None, 0)
            assert g.step_count == 1 + steps
    finally:
        for u in ref + gra:
            u.close()


def test_exhausted_table_changes_nothing_and_reports():
    wl = workloads.get("ragged_mini_flat_n3")
    hp = workloads.hyper(wl)
    u = _units(wl)[0]
    try:
        u.load([p.cuda() for p in workloads.param_tensors(wl, 0)])
        grads = [workloads.grad_tensor(wl, 0, 0, r).cuda() for r in range(wl.N)]
        out = torch.empty(u.numel, dtype=torch.int16, device="cuda")
        B.fsdp_adamw_device_steps(u.handle, hp, 2)
        u.step(grads, out, hp)
        u.step(grads, out, hp)
        torch.cuda.synchronize()
        before = {w: u.read_global(w).clone() for w in ("param", "exp_avg", "exp_avg_sq", "shadow")}
        assert B.fsdp_adamw_device_status(u.handle) == (2, False)
        u.adamw_step(hp)                                   # a third step: the table is used up
        torch.cuda.synchronize()
        assert B.fsdp_adamw_device_status(u.handle) == (2, True)
        for w, v in before.items():
            assert torch.equal(u.read_global(w), v), w
        with pytest.raises(B.FsdpError) as e:
            B.fsdp_set_step_count(u.handle, 0)
        assert e.value.code == B.FSDP_E_STATE
        B.fsdp_adamw_device_steps(u.handle, None, 0)
        assert u.step_count == 2
    finally:
        u.close()

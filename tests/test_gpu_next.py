"""GPU parity for the rows beyond the basic cycle: padded equal-chunk FLAT
layout, hybrid sharding, bf16 reduction, gather from the bf16 shadow,
gradient accumulation with unscale and the found-non-finite flag."""
import numpy as np
import pytest
import torch

from fully_sharded_unit_gb300 import binding as B
from fully_sharded_unit_gb300 import workloads
from oracle import fsdp_oracle as O

import gpu_harness as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from conftest import library
    library()


def _mini(layout="flat", N=7, **kw):
    return workloads.get(f"ragged_mini_{'dim0' if layout == 'dim0' else 'flat'}_n{N}").with_(layout=layout, **kw)


@pytest.mark.parametrize("N", [1, 3, 7, 64])
def test_padded_layout(N):
    H.run_full(_mini("flat_padded", N))
    H.run_full(_mini("flat_padded", N), use_step=True, steps=2)


def test_padded_layout_figure3_unit():
    """Figure 3's Linear (12 weights + 3 bias) over 16 ranks: one element each."""
    wl = workloads.Workload(
        name="fig3", description="fig3",
        units=((workloads.Param("w", (3, 4), ("normal", 0.1)), workloads.Param("b", (3,), ("normal", 0.1))),),
        N=16, layout="flat_padded", grad_dtype="f32", steps=2, grad_std=1e-2)
    H.run_full(wl)
    u = B.Unit(wl.shapes(0), "flat_padded", 16)
    try:
        assert u.shard_len == [1] * 15 + [0]
        assert [u.memory_report(k)["pad"] > 0 for k in range(16)][-1]
    finally:
        u.close()


@pytest.mark.parametrize("layout,N,R", [("flat", 4, 2), ("dim0", 4, 2), ("flat", 8, 8), ("dim0", 3, 22),
                                        ("flat", 1, 5)])
def test_hybrid_sharding(layout, N, R):
    H.run_full(_mini(layout, 7).with_(N=N, replicas=R))


def test_hybrid_sharding_bf16_grads_through_step():
    H.run_full(workloads.get("gpt_mini_flat_bf16").with_(N=4, replicas=2), use_step=True)


@pytest.mark.parametrize("name", ["ragged_mini_flat_n8", "ragged_mini_dim0_n7", "gpt_mini_flat_bf16"])
def test_bf16_reduction(name):
    H.run_full(workloads.get(name).with_(reduce_dtype="bf16"))


def _finite_bf16_patterns(rng, n):
    b = rng.integers(0, 1 << 16, n, dtype=np.uint32).astype(np.uint16)
    b[(b & 0x7F80) == 0x7F80] &= 0xBFFF          # exponent 0xFF -> 0x7F: finite
    return b


@pytest.mark.parametrize("grad_dtype", ["bf16", "f32"])
@pytest.mark.parametrize("N", [2, 3, 8])
@pytest.mark.parametrize("fused", [False, True])
def test_bf16_reduction_on_every_exponent(grad_dtype, N, fused):
    """bf16 reduction of gradients drawn from every bf16 exponent (subnormals,
    zeros of both signs, the largest finite values, sums that overflow) and of
    rank pairs whose exponents differ by 0..20, so that partial sums fall on
    and near bf16 rounding midpoints; fp32 gradients also carry random low
    halves that the input rounding must handle.  The gradient shard must equal
    the oracle's bit for bit, through the plain and the fused kernels."""
    rng = np.random.default_rng(1000 * N + (grad_dtype == "f32"))
    P = 3 * 8192 + 37                             # several tiles and a ragged tail
    pats = [_finite_bf16_patterns(rng, P) for _ in range(N)]
    e0 = (pats[0] >> 7) & 0xFF
    gap = rng.integers(0, 21, P).astype(np.uint16)
    near = (e0 > 21) & (rng.random(P) < 0.5)
    pats[1] = np.where(near, (pats[1] & 0x807F) | ((e0 - gap) << 7), pats[1]).astype(np.uint16)
    if grad_dtype == "f32":
        low = rng.integers(0, 1 << 16, (N, P), dtype=np.uint32)
        host = [(p.astype(np.uint32) << 16 | lo).view(np.float32) for p, lo in zip(pats, low)]
        host = [np.where(np.isfinite(h), h, np.float32(1.5)) for h in host]
        grads = [torch.from_numpy(h).cuda() for h in host]
    else:
        host = pats
        grads = [torch.from_numpy(h.view(np.int16)).view(torch.bfloat16).cuda() for h in host]
    with np.errstate(over="ignore", invalid="ignore"):
        want = O.reduce_full_bf16(host)
    u = B.Unit([(P,)], "flat", N, grad_dtype, reduce_dtype="bf16", fuse_reduce_adamw=fused)
    try:
        u.load([torch.zeros(P, device="cuda")])
        if fused:
            out = torch.empty(P, dtype=torch.int16, device="cuda")
            u.step(grads, out, dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01))
        else:
            u.reduce_scatter(grads)
        torch.cuda.synchronize()
        H.assert_bits_equal(u.read_global("grad").cpu().numpy(), want, f"bf16 reduction N={N}")
    finally:
        u.close()


@pytest.mark.parametrize("name", ["ragged_mini_flat_n7", "ragged_mini_dim0_n64", "gpt_mini_flat_bf16"])
def test_gather_from_shadow(name):
    H.run_full(workloads.get(name).with_(gather_source="shadow"))
    H.run_full(workloads.get(name).with_(gather_source="shadow"), use_step=True)


def test_set_param_refreshes_the_shadow_gather():
    wl = workloads.get("ragged_mini_flat_n7")
    u = B.Unit(wl.shapes(0), "flat", 7, gather_source="shadow")
    try:
        u.load([p.cuda() for p in workloads.param_tensors(wl, 0)])
        new = [torch.randn(u.shard_len[k], device="cuda") for k in range(7)]
        for k in range(7):
            u.set_state("param", k, new[k])
        out = torch.empty(u.numel, dtype=torch.int16, device="cuda")
        u.allgather(out)
        torch.cuda.synchronize()
        lay = O.Layout(wl.shapes(0), 7, "flat")
        want = O.allgather_cast([x.cpu().numpy() for x in new], lay)
        H.assert_bits_equal(H.u16(out), want, "gather after set_state")
    finally:
        u.close()


@pytest.mark.parametrize("name,R", [("ragged_mini_flat_n7", 1), ("ragged_mini_dim0_n3", 1),
                                    ("gpt_mini_flat_bf16", 1), ("ragged_mini_flat_n3", 2)])
def test_accumulation_unscale_and_found_flag(name, R):
    """Three micro-batches: the first overwrites, the next two accumulate with
    an unscale; the flag reports non-finite values, including a planted NaN."""
    wl = workloads.get(name).with_(replicas=R)
    shapes, N, P = wl.shapes(0), wl.N, wl.unit_numel(0)
    u = B.Unit(shapes, wl.layout, N, wl.grad_dtype, replicas=R)
    orc = O.UnitOracle(shapes, N, wl.layout, replicas=R)
    params = workloads.param_tensors(wl, 0)
    orc.load([p.numpy() for p in params])
    found = torch.empty(1, dtype=torch.int32, device="cuda")
    try:
        u.load([p.cuda() for p in params])
        u.zero_grad()
        for mb, (acc, scale) in enumerate([(False, 1.0), (True, 0.5), (True, 0.125)]):
            grads = [workloads.grad_tensor(wl, 0, mb, r).cuda() for r in range(wl.world)]
            if mb == 2:
                grads[1][P // 2] = float("nan")
            want_found = orc.reduce_scatter([H.grad_np(g) for g in grads], accumulate=acc, inv_scale=scale)
            found.fill_(7)
            u.reduce_scatter_ex(grads, accumulate=acc, inv_scale=scale, found=found)
            torch.cuda.synchronize()
            assert int(found.item()) == int(want_found), mb
            for k in range(N):
                H.assert_bits_equal(u.get_state("grad", k).cpu().numpy(), orc.grad[k], f"mb {mb} rank {k}")
        assert want_found
        u.zero_grad()
        torch.cuda.synchronize()
        assert not u.read_global("grad").any()
    finally:
        u.close()


def test_overflow_from_unscale_sets_the_flag():
    u = B.Unit([(1000,)], "flat", 2)
    try:
        u.load([torch.zeros(1000, device="cuda")])
        g = [torch.full((1000,), 1e38, device="cuda"), torch.full((1000,), 1e38, device="cuda")]   # sum 2e38, mean 1e38
        found = torch.zeros(1, dtype=torch.int32, device="cuda")
        u.reduce_scatter_ex(g, inv_scale=0.5, found=found)
        torch.cuda.synchronize()
        assert int(found.item()) == 0
        u.reduce_scatter_ex(g, inv_scale=4.0, found=found)
        torch.cuda.synchronize()
        assert int(found.item()) == 1
    finally:
        u.close()


@pytest.mark.parametrize("name,kw", [
    ("ragged_mini_flat_n7", {}), ("ragged_mini_dim0_n64", {}), ("gpt_mini_flat_bf16", {}),
    ("ragged_mini_flat_n3", {"replicas": 2}), ("ragged_mini_dim0_n8", {"reduce_dtype": "bf16"}),
    ("ragged_mini_flat_n7", {"gather_source": "shadow", "layout": "flat_padded"}),
    ("ragged_mini_flat_n64", {"reshard_after_forward": False}),
])
def test_fused_reduce_adamw_step(name, kw):
    """fsdp_step with the reduce-scatter and AdamW fused into one kernel gives
    the oracle's results bit for bit (the same operation sequence)."""
    cmp = H.run_full(workloads.get(name).with_(fuse_reduce_adamw=True, **kw), use_step=True)
    assert cmp.total_diff == 0


def _staged_eligible(wl):
    """The shared-memory staged fused kernel takes W x gradient bytes <= 100."""
    return wl.world * (2 if wl.grad_dtype == "bf16" else 4) <= 100


@pytest.mark.parametrize("name,kw", [
    ("ragged_mini_flat_n3", {}), ("ragged_mini_dim0_n2", {}), ("ragged_mini_flat_n1", {}),
    ("gpt_mini_flat_bf16", {"N": 4, "replicas": 2}),
    ("gpt_mini_dim0", {"grad_dtype": "bf16"}),
    ("ragged_mini_flat_n8", {"grad_dtype": "bf16", "layout": "flat_padded", "gather_source": "shadow"}),
    ("ragged_mini_dim0_n7", {"grad_dtype": "bf16", "reduce_dtype": "bf16"}),
    ("ragged_mini_flat_n2", {"replicas": 2}),
    ("ragged_mini_flat_n8", {}),                                  # 1024-element chunks
    ("gpt_mini_flat_bf16", {"N": 8, "replicas": 2}),              # W = 16, 1024-element chunks
    ("ragged_mini_dim0_n7", {"replicas": 3}),                     # fp32, W = 21, 512-element chunks
    ("ragged_mini_flat_n3", {"N": 25}),                           # fp32, W = 25: the widest staged unit
])
def test_fused_staged_kernel(name, kw):
    """Units with W x gradient bytes <= 100 take the fused kernel that stages
    its inputs in shared memory with bulk asynchronous copies: bit-identical
    to the oracle, status word clear."""
    wl = workloads.get(name).with_(fuse_reduce_adamw=True, **kw)
    assert _staged_eligible(wl)
    cmp = H.run_full(wl, use_step=True)
    assert cmp.total_diff == 0


def _custom(shapes, N, layout, grad_dtype="bf16", steps=3):
    init = ("uniform", -0.5, 0.5)
    units = (tuple(workloads.Param(f"p{i}", tuple(s), init) for i, s in enumerate(shapes)),)
    return workloads.Workload(name="custom", description="custom", units=units, N=N, layout=layout,
                              grad_dtype=grad_dtype, steps=steps, grad_std=1e-2, fuse_reduce_adamw=True)


@pytest.mark.parametrize("layout", ["flat", "dim0"])
@pytest.mark.parametrize("shapes,N", [
    ([(1,)], 1), ([(3, 4), (3,)], 8), ([(2, 3), ()], 3), ([(0, 7), (9, 2), (0,)], 4), ([(8193,)], 3),
    ([(16384 + 5, 3)], 7), ([(2049,), (15,), (17,)], 2), ([(40, 50)], 8), ([(4096 + 16,)], 1),
])
def test_fused_staged_edge_shapes(shapes, N, layout):
    """Tiles with no aligned body, bodies shorter than one chunk, chunks that
    end mid-tile, empty ranks, one element."""
    wl = _custom(shapes, N, layout)
    assert _staged_eligible(wl)
    H.run_full(wl, use_step=True)
    H.run_full(wl.with_(grad_dtype="f32"), use_step=True)


def test_fused_step_profiles_one_kernel():
    wl = workloads.get("ragged_mini_flat_n8")
    u = B.Unit(wl.shapes(0), "flat", 8, fuse_reduce_adamw=True)
    try:
        u.load([p.cuda() for p in workloads.param_tensors(wl, 0)])
        grads = [workloads.grad_tensor(wl, 0, 0, r).cuda() for r in range(8)]
        out = torch.empty(wl.unit_numel(0), dtype=torch.int16, device="cuda")
        B.fsdp_profile_enable(u.handle, True)
        u.step(grads, out, workloads.hyper(wl))
        counts = {k: B.fsdp_profile_read(u.handle, k)[1] for k in B.KERNELS}
        assert counts == {"shard_in": 0, "gather": 2, "reduce_scatter": 0, "adamw": 0, "reduce_adamw": 1}
        assert u.step_count == 1
    finally:
        u.close()


def test_gradients_in_pinned_host_memory():
    """Gradients read straight from pinned host memory give the same reduce-
    scatter and step as device-resident ones."""
    wl = workloads.get("gpt_mini_flat_bf16")
    shapes, N, P = wl.shapes(0), wl.N, wl.unit_numel(0)
    params = [p.cuda() for p in workloads.param_tensors(wl, 0)]
    grads = [workloads.grad_tensor(wl, 0, 0, r) for r in range(N)]
    host = [g.pin_memory() for g in grads]
    views = [B.fsdp_host_device_pointer(h) for h in host]
    a = B.Unit(shapes, "flat", N, "bf16", fuse_reduce_adamw=True)
    b = B.Unit(shapes, "flat", N, "bf16", fuse_reduce_adamw=True)
    try:
        a.load(params)
        b.load(params)
        out_a = torch.empty(P, dtype=torch.int16, device="cuda")
        out_b = torch.empty(P, dtype=torch.int16, device="cuda")
        a.step([g.cuda() for g in grads], out_a, workloads.hyper(wl))
        b.step(views, out_b, workloads.hyper(wl))
        torch.cuda.synchronize()
        for w in ("param", "grad", "exp_avg", "exp_avg_sq", "shadow"):
            assert torch.equal(a.read_global(w), b.read_global(w)), w
    finally:
        a.close()
        b.close()
    with pytest.raises(B.FsdpError) as e:
        B.fsdp_host_device_pointer(torch.zeros(16))          # pageable, not pinned
    assert e.value.code == B.FSDP_E_INVALID_ARG


def test_switching_step_options_mid_run_changes_nothing():
    """fsdp_unit_set_step_options between steps (shadow gather, fused
    reduce-scatter + AdamW, and back) gives the same bytes as never switching."""
    wl = workloads.get("ragged_mini_dim0_n7")
    hp = workloads.hyper(wl)
    a = B.Unit(wl.shapes(0), "dim0", wl.N)
    b = B.Unit(wl.shapes(0), "dim0", wl.N)
    try:
        params = [p.cuda() for p in workloads.param_tensors(wl, 0)]
        a.load(params)
        b.load(params)
        oa = torch.empty(a.numel, dtype=torch.int16, device="cuda")
        ob = torch.empty(b.numel, dtype=torch.int16, device="cuda")
        for s, opts in enumerate([("master", False), ("shadow", True), ("shadow", False), ("master", True)]):
            B.fsdp_unit_set_step_options(b.handle, *opts)
            grads = [workloads.grad_tensor(wl, 0, s, r).cuda() for r in range(wl.N)]
            a.step(grads, oa, hp)
            b.step(grads, ob, hp)
            torch.cuda.synchronize()
            assert torch.equal(oa, ob), s
        for w in B.STATES:
            assert torch.equal(a.read_global(w), b.read_global(w)), w
    finally:
        a.close()
        b.close()


def test_shadow_is_rne_of_master_whenever_read():
    """AdamW stores the bf16 shadow only when the unit gathers from it; every
    read of the shadow (state export, arena, a gather from it) must still see
    RNE(master).  The hard case: the shadow is stale, the unit switches to the
    shadow gather, and the next (shadow-storing) AdamW is skipped on the device
    because its step table is used up; the library refreshes the shadow before
    that launch, so it is right either way."""
    wl = workloads.get("ragged_mini_flat_n7")
    hp = workloads.hyper(wl)
    u = B.Unit(wl.shapes(0), wl.layout, wl.N)                 # gathers from the fp32 master
    try:
        u.load([p.cuda() for p in workloads.param_tensors(wl, 0)])
        grads = [workloads.grad_tensor(wl, 0, 0, r).cuda() for r in range(wl.N)]
        out = torch.empty(u.numel, dtype=torch.int16, device="cuda")

        def check(what):
            torch.cuda.synchronize()
            master = u.read_global("param").cpu().numpy()
            H.assert_bits_equal(H.u16(u.read_global("shadow")), O.bf16_rne(master), what)
            for k in range(u.N):
                H.assert_bits_equal(H.u16(u.get_state("shadow", k)),
                                    O.bf16_rne(u.get_state("param", k).cpu().numpy()), f"{what} rank {k}")

        u.step(grads, out, hp)                                 # AdamW leaves the shadow stale
        check("after a master-gather step")
        u.step(grads, out, hp)
        B.fsdp_adamw_device_steps(u.handle, hp, 1)
        u.adamw_step(hp)                                       # uses the table's only step, no shadow store
        B.fsdp_unit_set_step_options(u.handle, "shadow", False)
        u.adamw_step(hp)                                       # shadow-storing, skipped: table used up
        assert B.fsdp_adamw_device_status(u.handle)[1]
        check("after a skipped shadow-storing step")
        B.fsdp_adamw_device_steps(u.handle, None, 0)
        u.step(grads, out, hp)                                 # gathers from the shadow
        torch.cuda.synchronize()
        # the gathered buffer is RNE of the master before this step's AdamW:
        # compare against a fresh master-gather of the same state instead
        B.fsdp_unit_set_step_options(u.handle, "master", False)
        ref = torch.empty_like(out)
        u.allgather(ref)
        B.fsdp_unit_set_step_options(u.handle, "shadow", False)
        got = torch.empty_like(out)
        u.allgather(got)
        torch.cuda.synchronize()
        assert torch.equal(ref, got)
        check("after a shadow-gather step")
    finally:
        u.close()

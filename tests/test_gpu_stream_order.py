"""Stream order with programmatic dependent launch: the library's kernels
interleaved with torch kernels on one stream and no host synchronisation.
Before every unit step a torch copy writes the gradients the step reads, and
after it a torch copy takes the gathered parameters the step wrote; several
units share those buffers, and the bf16 output buffer is rewritten by the next
unit while torch has just read it.  Any reordering shows up as a difference
from the oracle."""
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


@pytest.mark.parametrize("grad_dtype,fuse", [("f32", False), ("bf16", False), ("bf16", True)])
def test_interleaved_with_torch_kernels(grad_dtype, fuse):
    shapes_per_unit = [[(37, 11), (37,)], [(300, 7)], [(5,), (8193,)]]
    N, S = 4, 12
    hp = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
    rng = np.random.default_rng(7)
    tdt = torch.float32 if grad_dtype == "f32" else torch.bfloat16
    units, oracles, host_grads = [], [], []
    P_max = max(sum(int(np.prod(s)) for s in shp) for shp in shapes_per_unit)
    for shp in shapes_per_unit:
        params = [rng.uniform(-0.5, 0.5, s).astype(np.float32) for s in shp]
        P = sum(p.size for p in params)
        u = B.Unit(shp, "flat", N, grad_dtype, fuse_reduce_adamw=fuse)
        u.load([torch.from_numpy(p).cuda() for p in params])
        orc = O.UnitOracle(shp, N, "flat", O.AdamWHyper(**hp))
        orc.load(params)
        units.append(u)
        oracles.append(orc)
        g = torch.from_numpy(rng.normal(0, 1e-2, (S, N, P)).astype(np.float32)).to(tdt)
        host_grads.append(g)
    dev_grads = [g.cuda() for g in host_grads]                 # every step's gradients, resident
    work = [torch.empty(P_max, dtype=tdt, device="cuda") for _ in range(N)]   # shared per-step inputs
    out = torch.empty(P_max, dtype=torch.int16, device="cuda")                # shared output
    hist = [[torch.empty(u.numel, dtype=torch.int16, device="cuda") for u in units] for _ in range(S)]
    torch.cuda.synchronize()
    for s in range(S):
        for i, u in enumerate(units):
            for r in range(N):
                work[r][:u.numel].copy_(dev_grads[i][s, r])    # torch writes what the step reads
            u.step([w[:u.numel] for w in work], out, hp)
            hist[s][i].copy_(out[:u.numel])                     # torch reads what the step wrote
    torch.cuda.synchronize()
    for s in range(S):
        for i, orc in enumerate(oracles):
            want = orc.step([H.grad_np(host_grads[i][s, r]) for r in range(N)])
            H.assert_bits_equal(H.u16(hist[s][i]), want[-1], f"step {s} unit {i} gathered")
    for u, orc in zip(units, oracles):
        for which in ("param", "exp_avg", "exp_avg_sq"):
            H.assert_bits_equal(u.read_global(which).cpu().numpy(), orc.full(
                {"param": "master", "exp_avg": "m", "exp_avg_sq": "v"}[which]), which)
        u.close()

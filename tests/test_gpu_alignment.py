"""Gradient and output buffers that are 16-byte but not 32-byte aligned (a
torch view 16 bytes into an allocation): the library accepts them and every
kernel path gives the oracle's results bit for bit; buffers aligned to less
than 16 bytes are refused with FSDP_E_ALIGN before anything is enqueued."""
import pytest
import torch

from fully_sharded_unit_gb300 import binding as B
from fully_sharded_unit_gb300 import workloads

import gpu_harness as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from conftest import library
    library()


@pytest.mark.parametrize("name,kw,use_step", [
    ("ragged_mini_flat_n7", {}, False),                              # fp32 plain reduce-scatter
    ("ragged_mini_flat_n7", {}, True),                               # fsdp_step, separate kernels
    ("ragged_mini_dim0_n7", {"fuse_reduce_adamw": True}, True),      # fp32 fused, shared-memory staged
    ("ragged_mini_flat_n64", {"fuse_reduce_adamw": True}, True),     # fp32 fused, register-staged
    ("gpt_mini_flat_bf16", {}, False),                               # bf16 plain (8-wide instead of 16)
    ("gpt_mini_flat_bf16", {"N": 66}, False),                        # bf16 plain, more than 64 ranks
    ("gpt_mini_flat_bf16", {"fuse_reduce_adamw": True}, True),       # bf16 fused, staged
    ("ragged_mini_flat_n8", {"replicas": 2}, False),                 # fp32 hybrid, staged
    ("ragged_mini_flat_n64", {"replicas": 2}, False),                # fp32 hybrid, register, 128 ranks
    ("ragged_mini_flat_n8", {"reduce_dtype": "bf16"}, True),         # bf16 reduction of fp32 gradients
    ("ragged_mini_dim0_n3", {"gather_source": "shadow"}, True),      # gather from the bf16 shadow
])
def test_16_byte_aligned_buffers_match_the_oracle(name, kw, use_step):
    wl = workloads.get(name).with_(**kw)
    cmp = H.run_full(wl, use_step=use_step, steps=2, misalign=True)
    assert cmp.total_diff == 0


def test_buffers_below_16_bytes_are_refused():
    wl = workloads.get("ragged_mini_flat_n3")
    u = B.Unit(wl.shapes(0), wl.layout, wl.N, wl.grad_dtype)
    try:
        P = u.numel
        u.load([p.cuda() for p in workloads.param_tensors(wl, 0)])
        grads = [torch.zeros(P + 8, dtype=torch.float32, device="cuda") for _ in range(wl.N)]
        out = torch.zeros(P + 8, dtype=torch.int16, device="cuda")
        ok = [g[:P] for g in grads]
        bad = [g[2:P + 2] for g in grads[:1]] + ok[1:]          # 8 bytes past a 32-byte boundary
        with pytest.raises(B.FsdpError) as e:
            u.reduce_scatter(bad)
        assert e.value.code == B.FSDP_E_ALIGN
        with pytest.raises(B.FsdpError) as e:
            u.step(bad, out[:P], workloads.hyper(wl))
        assert e.value.code == B.FSDP_E_ALIGN
        with pytest.raises(B.FsdpError) as e:
            u.allgather(out[4:P + 4])                              # 8-byte aligned output
        assert e.value.code == B.FSDP_E_ALIGN
        assert u.step_count == 0, "a refused call advanced the step count"
        u.allgather(out[8:P + 8])                                  # 16-byte aligned: accepted
        torch.cuda.synchronize()
    finally:
        u.close()

"""fsdp_unit_create_with_allocator: the unit's device memory from a caller's
allocator (here torch's caching allocator), the same results as with the
library's own allocations, and every block handed back on success and on
each failure path."""
import gc

import pytest
import torch

from fully_sharded_unit_gb300 import binding as B
from fully_sharded_unit_gb300 import workloads

import gpu_harness as H

pytestmark = pytest.mark.gpu

# master, gradient shard, m, v, shadow, the two tile tables, the parameter
# table, the kernel status word
BLOCKS_PER_UNIT = 9


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from conftest import library
    library()


@pytest.mark.parametrize("name,use_step", [("ragged_mini_dim0_n7", False), ("gpt_mini_flat_bf16", True)])
def test_torch_allocator_parity_and_accounting(name, use_step):
    wl = workloads.get(name)
    torch.cuda.synchronize()
    gc.collect()          # tensors of earlier tests held in reference cycles would be freed mid-count
    base = torch.cuda.memory_allocated()
    alloc = B.TorchAllocator()
    cmp = H.run_full(wl, use_step=use_step, allocator=alloc)
    assert cmp.total_diff == 0
    assert alloc.allocs == BLOCKS_PER_UNIT and alloc.frees == BLOCKS_PER_UNIT and not alloc.live
    torch.cuda.synchronize()
    assert torch.cuda.memory_allocated() == base


def test_torch_allocator_holds_the_arenas_while_the_unit_lives():
    wl = workloads.get("ragged_mini_flat_n7")
    alloc = B.TorchAllocator()
    gc.collect()
    before = torch.cuda.memory_allocated()
    u = B.Unit(wl.shapes(0), "flat", wl.N, allocator=alloc)
    try:
        arena = sum(sum(u.memory_report(k).values()) for k in range(wl.N))   # states + shadow + pads
        grown = torch.cuda.memory_allocated() - before
        assert arena >= 18 * wl.unit_numel(0)          # 4 fp32 states + the bf16 shadow per element
        assert grown >= arena                          # all of it (and the tile tables) held by torch
        assert len(alloc.live) == BLOCKS_PER_UNIT
        # device-step mode takes its table and counters from the same allocator
        u.load([p.cuda() for p in workloads.param_tensors(wl, 0)])
        B.fsdp_adamw_device_steps(u.handle, workloads.hyper(wl), 5)
        assert alloc.allocs == BLOCKS_PER_UNIT + 3
        B.fsdp_adamw_device_steps(u.handle, workloads.hyper(wl), 50)   # a larger table replaces the old one
        assert alloc.allocs == BLOCKS_PER_UNIT + 4 and alloc.frees == 1
    finally:
        u.close()
    assert alloc.allocs == alloc.frees and not alloc.live
    assert torch.cuda.memory_allocated() == before


class _Faulty:
    """Hands out torch blocks, but the k-th request returns NULL or a block
    offset by 16 bytes (not 256-byte aligned)."""

    def __init__(self, k, mode):
        self.k, self.mode, self.n = k, mode, 0
        self.live = {}
        self.frees = []

        def _alloc(nbytes, ctx):
            i = self.n
            self.n += 1
            if i == self.k and self.mode == "null":
                return None
            t = torch.empty(int(nbytes) + 256, dtype=torch.uint8, device="cuda")
            p = t.data_ptr() + (16 if i == self.k else 0)
            self.live[p] = t
            return p

        def _free(ptr, ctx):
            assert ptr in self.live, "freed a block the allocator did not hand out"
            self.live.pop(ptr)
            self.frees.append(ptr)

        self._cb = (B._ALLOC_FN(_alloc), B._FREE_FN(_free))
        self.struct = B.Allocator(self._cb[0], self._cb[1], None)


@pytest.mark.parametrize("mode,code", [("null", B.FSDP_E_OOM), ("misaligned", B.FSDP_E_ALIGN)])
@pytest.mark.parametrize("k", range(BLOCKS_PER_UNIT))
def test_failed_allocation_returns_every_block(mode, code, k):
    wl = workloads.get("ragged_mini_flat_n7")
    a = _Faulty(k, mode)
    with pytest.raises(B.FsdpError) as e:
        B.Unit(wl.shapes(0), "flat", wl.N, allocator=a)
    assert e.value.code == code
    assert not a.live                                   # nothing leaked
    assert len(a.frees) == (k if mode == "null" else k + 1)


def test_allocator_without_free_is_rejected():
    a = B.Allocator(B._ALLOC_FN(lambda n, c: None), B._FREE_FN(0), None)
    with pytest.raises(B.FsdpError) as e:
        B.fsdp_unit_create_with_allocator([(10,)], "flat", 2, a)
    assert e.value.code == B.FSDP_E_INVALID_ARG

"""fsdp_reduce_scatter_flat_noalloc: the reduce-scatter for callers that cannot
allocate device memory (a plug-in inside a framework that owns the GPU's
memory pool, or a process whose HBM is already given to shards).  It needs no
unit; its only scratch, the kernel's table of work tiles, is a fixed array in
the library's device image.

Each check calls it through the C ABI and compares its output with what the
unit-based fsdp_reduce_scatter writes for a FLAT unit of the same size and
rank count: bit for bit, the reduce-scatter's tolerance.  Two calls run in a
row (the second smaller than the first, so stale tiles of the first are left
in the shared scratch), and sizes beyond the scratch are refused before any
work is enqueued.

This file sorts last so that a run stopping at its first failure has already
run every other test."""
import pytest
import torch

from fully_sharded_unit_gb300 import binding as B
from fully_sharded_unit_gb300 import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from conftest import library
    library()


def _unit_reduce_scatter(wl, grads):
    """The existing entry point: a FLAT unit's reduce-scatter, its shards read
    back and concatenated in rank order (the unsharded reduced gradient)."""
    u = B.Unit(wl.shapes(0), "flat", wl.N, wl.grad_dtype)
    try:
        u.load([p.cuda() for p in workloads.param_tensors(wl, 0)])
        u.reduce_scatter(grads)
        torch.cuda.synchronize()
        return torch.cat([u.get_state("grad", k) for k in range(wl.N)])
    finally:
        u.close()


def _noalloc(wl, grads):
    out = torch.full((wl.unit_numel(0),), float("nan"), dtype=torch.float32, device="cuda")
    B.fsdp_reduce_scatter_flat_noalloc(grads, out)
    torch.cuda.synchronize()
    return out


def _same_bits(a, b, what):
    assert a.shape == b.shape, what
    diff = a.view(torch.int32) != b.view(torch.int32)
    assert not bool(diff.any()), f"{what}: {int(diff.sum())} of {a.numel()} elements differ"


def test_two_calls_in_a_row_match_the_unit_reduce_scatter():
    # first call: 70.9 M elements at N = 7 (8,660 tiles, fp32 gradients)
    big = workloads.get("ragged_flat_n7")
    # second call: 0.4 M elements at N = 8 (bf16 gradients with outliers), far
    # fewer tiles, so most of the table still holds the first call's tiles
    small = workloads.get("gpt_mini_flat_bf16").with_(units=(workloads.get("gpt_mini_flat_bf16").units[0],))
    for wl in (big, small):
        grads = [workloads.grad_tensor(wl, 0, 0, r, "cuda") for r in range(wl.N)]
        _same_bits(_noalloc(wl, grads), _unit_reduce_scatter(wl, grads), wl.name)
        del grads


def test_repeated_calls_on_one_stream_stay_ordered():
    """Calls queued back to back on one stream, each rewriting the shared
    table before its kernel, with no host synchronisation between them."""
    wls = [workloads.get("ragged_mini_flat_n64"), workloads.get("ragged_mini_flat_n3"),
           workloads.get("ragged_flat_n7")]
    st = torch.cuda.Stream()
    results = []
    with torch.cuda.stream(st):
        for wl in wls:
            grads = [workloads.grad_tensor(wl, 0, 1, r, "cuda") for r in range(wl.N)]
            out = torch.empty(wl.unit_numel(0), dtype=torch.float32, device="cuda")
            B.fsdp_reduce_scatter_flat_noalloc(grads, out, stream=st)
            results.append((wl, grads, out))
    st.synchronize()
    for wl, grads, out in results:
        _same_bits(out, _unit_reduce_scatter(wl, grads), wl.name)


def test_sizes_beyond_the_scratch_are_refused():
    g = [torch.zeros(64, dtype=torch.float32, device="cuda") for _ in range(3)]
    out = torch.zeros(64, dtype=torch.float32, device="cuda")
    ptrs = B._ptrs(g)
    tile = 8192
    # more whole tiles than the table holds
    rc = B.lib().fsdp_reduce_scatter_flat_noalloc(ptrs, 1, B.FSDP_DTYPE_F32, tile * B.FSDP_NOALLOC_MAX_TILES + 1,
                                                   out.data_ptr(), None)
    assert rc == B.FSDP_E_INVALID_ARG
    assert "tiles" in B.fsdp_last_error()
    # exactly the table's whole tiles, but three ranks cut two tiles in two
    rc = B.lib().fsdp_reduce_scatter_flat_noalloc(ptrs, 3, B.FSDP_DTYPE_F32, tile * B.FSDP_NOALLOC_MAX_TILES,
                                                   out.data_ptr(), None)
    assert rc == B.FSDP_E_INVALID_ARG
    assert "32770 work tiles" in B.fsdp_last_error()
    torch.cuda.synchronize()
    assert bool(torch.all(out == 0)), "a refused call wrote its output"

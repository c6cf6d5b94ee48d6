"""GPU parity at the full workload sizes, through fsdp_step (the call the bench
times): whole units where the host holds them, windows otherwise.  Windowed
checks cover every shard and parameter boundary (+-4096 elements) and, for
every step, random windows drawn afresh totalling at least 5 % of the unit;
the AdamW state must be bit-identical to the oracle there."""
import pytest
import torch

from fully_sharded_unit_gb300 import workloads

import gpu_harness as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from conftest import library
    library()
    yield
    torch.cuda.empty_cache()


@pytest.mark.parametrize("unit", [0, 11])
def test_gpt2_small_flat_full(unit):
    H.run_full(workloads.get("gpt2_small_flat"), unit=unit, use_step=True, gen_device="cuda")


@pytest.mark.parametrize("unit", [0, 35])
def test_gpt2_large_dim0_full(unit):
    H.run_full(workloads.get("gpt2_large_dim0"), unit=unit, use_step=True, gen_device="cuda")


@pytest.mark.parametrize("name", ["ragged_flat_n7", "ragged_dim0_n7"])
def test_ragged_n7_full(name):
    H.run_full(workloads.get(name), use_step=True, gen_device="cuda")


@pytest.mark.parametrize("name", ["ragged_flat_n64", "ragged_dim0_n64"])
def test_ragged_n64_full(name):
    """Every element of the 70.9 M-element unit at N = 64 (57 empty DIM0
    chunks of the 7x13 parameter, ragged FLAT shards), every step."""
    cmp = H.run_full(workloads.get(name), use_step=True, gen_device="cuda")
    assert cmp.total_diff == 0


def _coverage(cmp, frac=0.05):
    """At least `frac` of the unit in fresh random windows at every step, and
    in the union compared at every step."""
    assert min(cmp.step_random) >= frac * cmp.P, (cmp.step_random, cmp.P)
    assert cmp.covered >= frac * cmp.P


@pytest.mark.parametrize("unit", [0, 1])
def test_mingpt175b_windows(unit):
    cmp = H.run_windowed(workloads.get("mingpt175b_flat"), unit=unit)
    _coverage(cmp)


def test_mingpt175b_windows_fused_shadow_gather():
    """The fastest configuration of the bench workload: fsdp_step with the fused
    reduce-scatter + AdamW kernel and the gather from the bf16 shadow."""
    wl = workloads.get("mingpt175b_flat").with_(fuse_reduce_adamw=True, gather_source="shadow")
    cmp = H.run_windowed(wl, unit=0)
    _coverage(cmp)


@pytest.mark.parametrize("name", ["huge_flat_n3", "huge_dim0_n3"])
def test_unit_past_2_31_elements(name):
    """P = 2,147,489,281 > 2^31: offsets, tiles and slab indices are 64-bit;
    windows cover every shard boundary and the 2^31 element boundary."""
    wl = workloads.get(name)
    assert wl.unit_numel(0) > 2 ** 31
    cmp = H.run_windowed(wl, extra_boundaries=(2 ** 31, 2 ** 31 - 8192))
    _coverage(cmp)
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name,kw", [("huge_flat_n3", dict(fuse_reduce_adamw=True)),
                                     ("huge_dim0_n3", dict(replicas=2)),
                                     ("huge_flat_n3", dict(replicas=2, fuse_reduce_adamw=True))])
def test_staged_kernels_past_2_31_elements(name, kw):
    """The shared-memory staged kernels (fused step; reduce-scatter of hybrid
    sharding) on a unit past 2^31 elements: 64-bit chunk offsets and copy
    addresses, windows at every shard boundary and at 2^31."""
    wl = workloads.get(name).with_(**kw)
    cmp = H.run_windowed(wl, extra_boundaries=(2 ** 31, 2 ** 31 - 8192))
    _coverage(cmp)
    torch.cuda.empty_cache()


@pytest.mark.parametrize("kw", [
    dict(replicas=2),                                   # hybrid: 2 sharding groups of 8, W = 16 gradients
    dict(reduce_dtype="bf16"),                          # reductions in bf16
    dict(layout="flat_padded", gather_source="shadow"),  # the paper's padded FlatParameter, bf16 gather
    dict(layout="dim0", fuse_reduce_adamw=True, replicas=2),
])
def test_mingpt175b_next_rows_windows(kw):
    """The rows beyond the basic cycle at the full minGPT-175B unit size,
    through fsdp_step, compared on windows."""
    wl = workloads.get("mingpt175b_flat").with_(**kw)
    cmp = H.run_windowed(wl, unit=0)
    _coverage(cmp)
    torch.cuda.empty_cache()

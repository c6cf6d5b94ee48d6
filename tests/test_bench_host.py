"""bench.py's host-side bookkeeping: the configuration key that recorded ncu
traffic is tied to, and the counted bytes of each kernel (no GPU needed)."""
import os

from conftest import ROOT

import bench
from fully_sharded_unit_gb300 import workloads


def test_traffic_key_names_every_option_that_changes_kernel_bytes():
    wl = workloads.get("mingpt175b_flat")
    assert bench.traffic_key(wl) == "mingpt175b_flat"
    assert bench.traffic_key(wl.with_(fuse_reduce_adamw=True)) == "mingpt175b_flat"   # separate kernel kinds
    assert bench.traffic_key(wl.with_(replicas=2)) == "mingpt175b_flat+replicas=2"
    assert bench.traffic_key(wl.with_(gather_source="shadow")) == "mingpt175b_flat+gather_source=shadow"
    assert bench.traffic_key(wl.with_(reduce_dtype="bf16")) == "mingpt175b_flat+reduce_dtype=bf16"
    assert bench.traffic_key(wl.with_(layout="dim0")) == "mingpt175b_flat+layout=dim0"
    assert bench.traffic_key(wl, 4) == "mingpt175b_flat+micro_batches=4"


def test_recorded_traffic_file_parses_and_unknown_keys_give_none():
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    for line in open(path):
        if line.startswith("#") or not line.strip():
            continue
        kernel, key, nbytes, sha = line.split()
        assert kernel in ("gather", "reduce_scatter", "adamw", "reduce_adamw")
        assert key.split("+")[0] in workloads.names()
        assert int(nbytes) > 0 and len(sha) == 16
    assert bench.recorded_traffic("adamw", "no_such_workload") is None


def test_counted_bytes_per_launch():
    """Algorithmic bytes per element: gather 6 (4 from the shadow), reduce-scatter
    W*g_b + 4, AdamW 28 (30 when it also stores the shadow the gathers read),
    fused W*g_b + 28 (+2); a unit step sums them, and with the separate kernels
    it equals the every-operation-separate (44 + W*g_b) count."""
    wl = workloads.get("mingpt175b_flat")
    P = wl.unit_numel(0)
    c = bench.counted_bytes(wl, 0)
    assert (c["gather"], c["reduce_scatter"], c["adamw"], c["reduce_adamw"]) == (6 * P, 20 * P, 28 * P, 44 * P)
    assert c["step"] == 2 * 6 * P + 20 * P + 28 * P == bench.survey_bytes(wl, 0) == (44 + 16) * P
    f = bench.counted_bytes(wl.with_(fuse_reduce_adamw=True, gather_source="shadow"), 0)
    assert f["gather"] == 4 * P and f["adamw"] == 30 * P and f["step"] == 2 * 4 * P + 46 * P
    assert bench.survey_bytes(wl.with_(gather_source="shadow"), 0) == (42 + 16) * P
    h = bench.counted_bytes(wl.with_(replicas=2), 0)
    assert h["reduce_scatter"] == (16 * 2 + 4) * P


def test_oracle_on_several_cores_times_every_worker():
    """The all-core CPU baseline: two spawned workers, each with its own
    sample, run one oracle unit step at once per bench step."""
    wl = workloads.get("mingpt175b_flat")
    times, elements, step_bytes, workers = bench.oracle_all_cores(wl, 2, 1 << 20, cores=2, warmup=1)
    assert workers == 2 and elements == 2 << 20 and len(times) == 2 and min(times) > 0
    sample = bench.oracle_sample_workload(wl, 1 << 20)
    assert step_bytes == 2 * bench.counted_bytes(sample, 0)["step"]
    assert bench.cpu_model()

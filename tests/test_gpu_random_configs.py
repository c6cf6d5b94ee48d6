"""A seeded sweep over the configuration space, each case compared with the
oracle on every element of every step: random ragged shapes (0-d, empty and
odd dims), N from 1 to 70, every layout, fp32 and bf16 gradients, replicas,
bf16 reduction, the fused step (staged and register-staged forms), the
bf16-shadow gather, both resharding modes, and (drawn separately, so the
configurations themselves stay as they were) gradient and output buffers
that are only 16-byte aligned."""
import numpy as np
import pytest

from fully_sharded_unit_gb300 import workloads

import gpu_harness as H

pytestmark = pytest.mark.gpu

N_CASES = 100


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from conftest import library
    library()


def random_config(seed: int) -> workloads.Workload:
    rng = np.random.default_rng(10_000 + seed)
    nparams = int(rng.integers(1, 5))
    shapes = []
    for _ in range(nparams):
        kind = rng.random()
        if kind < 0.1:
            shapes.append(())                                   # 0-d
        elif kind < 0.15:
            shapes.append((0, int(rng.integers(1, 9))))         # empty
        elif kind < 0.55:
            shapes.append((int(rng.integers(1, 9000)),))
        else:
            shapes.append((int(rng.integers(1, 400)), int(rng.integers(1, 60))))
    if sum(int(np.prod(s)) if s else 1 for s in shapes) == 0:
        shapes.append((17,))
    N = int(rng.choice([1, 2, 3, 4, 5, 7, 8, 13, 16, 31, 64, 70]))
    layout = str(rng.choice(["flat", "dim0", "flat_padded"]))
    grad_dtype = str(rng.choice(["f32", "bf16"]))
    replicas = int(rng.choice([1, 1, 2, 3])) if N * 3 <= 1024 else 1
    reduce_dtype = "bf16" if (replicas == 1 and rng.random() < 0.25) else "f32"
    units = (tuple(workloads.Param(f"p{i}", tuple(s), ("uniform", -0.5, 0.5)) for i, s in enumerate(shapes)),)
    return workloads.Workload(
        name=f"random{seed}", description="random configuration", units=units, N=N, layout=layout,
        grad_dtype=grad_dtype, steps=2, grad_std=1e-2, replicas=replicas, reduce_dtype=reduce_dtype,
        reshard_after_forward=bool(rng.random() < 0.7),
        fuse_reduce_adamw=bool(rng.random() < 0.5),
        gather_source="shadow" if rng.random() < 0.3 else "master")


@pytest.mark.parametrize("seed", range(N_CASES))
def test_random_configuration(seed):
    wl = random_config(seed)
    misalign = bool(np.random.default_rng(20_000 + seed).random() < 0.3)
    cmp = H.run_full(wl, use_step=bool(seed % 2), misalign=misalign)
    assert cmp.total_diff == 0, (wl, cmp.adamw)

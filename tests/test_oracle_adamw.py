"""Pins for the oracle's AdamW step."""
import numpy as np
import pytest

import pins
from oracle import fsdp_oracle as O

HP = O.AdamWHyper(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
HP2 = O.AdamWHyper(lr=3e-4, beta1=0.9, beta2=0.95, eps=1e-6, weight_decay=0.1)


@pytest.mark.parametrize("hp", [HP, HP2])
def test_adamw_matches_torch_at_n1(hp):
    pins.check_adamw_vs_torch(O.adamw_update, hp)


@pytest.mark.parametrize("hp", [HP, HP2])
def test_adamw_first_step_closed_form(hp):
    pins.check_adamw_first_step_closed_form(O.adamw_update, hp)


def test_adamw_zero_gradient_only_decays():
    pins.check_adamw_zero_grad(O.adamw_update, HP)


@pytest.mark.parametrize("hp", [HP, HP2])
def test_adamw_within_fp64_reference(hp):
    pins.check_adamw_fp64(O.adamw_update, O.adamw_update_f64, hp)


def test_adamw_zero_is_a_fixed_point():
    z = np.zeros(64, np.float32)
    p, m, v = O.adamw_update(z, z, z, z, 3, HP)
    assert not p.any() and not m.any() and not v.any()

"""The rounding allowance the GPU parity checks grant the 16-bit outputs:
half an ulp of each exact value, i.e. exactly what one round-to-nearest
conversion to the output dtype may cost (checked against torch's own
conversions), and no more (the bound is attained)."""

import numpy as np
import pytest
import torch

from tests.helpers import rounding_allowance

DT = {"bf16": torch.bfloat16, "f16": torch.float16}


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_allowance_bounds_one_rounding(dtype):
    x = np.random.default_rng(3).normal(0.0, 3.0, 200000).astype(np.float32).astype(np.float64)
    r = torch.from_numpy(x).to(torch.float32).to(DT[dtype]).to(torch.float64).numpy()
    excess = np.abs(r - x) - rounding_allowance(x, dtype)
    assert np.max(excess) <= 0.0
    # attained: some value lands (almost) half an ulp away
    assert np.max(np.abs(r - x) / rounding_allowance(x, dtype)) > 0.99


def test_allowance_values():
    ref = np.array([1.0, 1.5, 2.0, 3.99, 4.0, -2.5])
    assert np.array_equal(rounding_allowance(ref, "bf16"), [2.0 ** -8, 2.0 ** -8, 2.0 ** -7, 2.0 ** -7, 2.0 ** -6, 2.0 ** -7])
    assert np.array_equal(rounding_allowance(ref, "f16"), [2.0 ** -11, 2.0 ** -11, 2.0 ** -10, 2.0 ** -10, 2.0 ** -9, 2.0 ** -10])
    assert np.all(rounding_allowance(ref, "f32") == 0)

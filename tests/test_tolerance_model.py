"""Derivation of the bf16 Newton-Schulz tolerance from the arithmetic.

A NumPy model of the tensor-core path's rounding is compared with the fp64
oracle. In the model, X, A and B are bf16, rounded to nearest even. Products
accumulate exactly, standing in for the fp32 accumulator. X is kept in bf16
between steps, and the aX term is folded into the polynomial matrix,
B = aI + bA + cA^2, so each step is X' = B X.

The measured errors justify the tolerances the GPU tests use. Under both
normalisations the model stays inside the 2e-2 bound that the workload
specification states for bf16 NS:

* Frobenius scale (X0 = M/||M||_F): about 1.0e-2.
* Spectral scale (X0 = M/(||M||_F sigma_hat)): about 1.3e-2. The singular
  values start near 1, where the quintic is more sensitive to rounding.

The model also records why this form was chosen over two others. In both,
the aX term is added in fp32 outside the product:
* with X's bf16 operand: 1.3e-2 Frobenius, 1.7e-2 spectral;
* with an fp32 master of X: 1.6e-2 Frobenius, 2.2e-2 spectral.
Both are less accurate than the folded, consistent bf16 operator.
"""
import numpy as np
import pytest

from oracle import muon as om
from tests.gpu_helpers import NS_BF16_SPECTRAL_TOL, NS_BF16_TOL
from tests.ns_rounding_model import ns_bf16_model


@pytest.mark.parametrize("shape", [(96, 200), (256, 512)])
def test_bf16_model_error_levels(shape):
    forms = ("folded", "bf16_ax", "fp32_master")
    worst = {}
    for seed in range(3):
        M = np.random.default_rng(seed).standard_normal(shape)
        F = M / np.linalg.norm(M)
        s = om.spectral_estimate(F, 8)
        for key, X0 in (("f", F), ("s", F / s)):
            ref = om.ns_iterate(X0)
            for form in forms:
                err = np.linalg.norm(ns_bf16_model(X0, form=form) - ref) / np.linalg.norm(ref)
                worst[key, form] = max(worst.get((key, form), 0.0), err)
    assert worst["f", "folded"] < 0.65 * NS_BF16_TOL
    assert worst["s", "folded"] < 0.8 * NS_BF16_SPECTRAL_TOL
    # the design choice: the folded, consistent bf16 operator is the most accurate
    for key in ("f", "s"):
        assert worst[key, "folded"] < worst[key, "bf16_ax"] < worst[key, "fp32_master"]

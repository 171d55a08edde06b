"""Derivation of the bf16 Newton-Schulz tolerance from the arithmetic.

A NumPy model of the tensor-core path's rounding is compared with the fp64
oracle. In the model, X, A and B are bf16, rounded to nearest even. Products
accumulate exactly, standing in for the fp32 accumulator. X is kept in bf16
between steps, and the aX term is folded into the polynomial matrix,
B = aI + bA + cA^2, so each step is X' = B X. B's diagonal lies near
a = 3.44, where the bf16 spacing is 2^-6; the kernels keep that diagonal's
rounding residual in fp32 and add it back in the apply epilogue.

The measured errors justify the tolerance the GPU tests use: the model stays
inside the 2e-2 bound that the workload specification states for bf16 NS,
with margin, under both normalisations and on the inputs where the plain
folded operator misses it (a tight spectrum, whose singular values all start
at 1/sqrt(m)).

The model also records why this form was chosen over three others:
* the folded operator without the diagonal residual reaches 2.3e-2 to 2.5e-2
  on tight spectra at m = 32 to 48 and 2.2e-2 at m = 384;
* aX added in fp32 outside the product (from X's bf16 operand, or from an
  fp32 master of X) is less accurate than the folded operator.
"""
import numpy as np
import pytest

from oracle import muon as om
from tests.gpu_helpers import NS_BF16_SPECTRAL_TOL, NS_BF16_TOL
from tests.ns_rounding_model import f32, model_rel_err, ns_bf16_model
from workloads import matrix_set_inputs, tight_spectrum_matrix


@pytest.mark.parametrize("shape", [(96, 200), (256, 512)])
def test_bf16_model_error_levels(shape):
    forms = ("folded_diag", "folded", "bf16_ax", "fp32_master")
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
    assert worst["f", "folded_diag"] < 0.5 * NS_BF16_TOL
    assert worst["s", "folded_diag"] < 0.6 * NS_BF16_SPECTRAL_TOL
    # the design choice: the folded operator with its diagonal residual is the
    # most accurate form
    for key in ("f", "s"):
        assert worst[key, "folded_diag"] < worst[key, "folded"] < worst[key, "bf16_ax"] < worst[key, "fp32_master"]


@pytest.mark.parametrize("m,n,kind", [(32, 256, "tight"), (48, 256, "tight"), (384, 768, "tight"),
                                      (32, 200, "gauss"), (32, 240, "gauss")])
def test_diagonal_residual_keeps_tight_spectra_inside_bound(m, n, kind):
    M = f32(tight_spectrum_matrix(m, n, 0)) if kind == "tight" else f32(np.random.default_rng(0).standard_normal((m, n)))
    plain, fixed = model_rel_err(M, form="folded"), model_rel_err(M)
    assert plain > 0.9 * NS_BF16_TOL          # the inputs where the plain operator is at or above the bound
    assert fixed < 0.75 * NS_BF16_TOL


def test_model_inside_bound_on_tiny_batch_draw():
    """The draw of the GPU batch test of 300 matrices (8 to 64 rows, 8 to 256
    columns): the kernels' form stays inside 2e-2 on every matrix."""
    rng = np.random.default_rng(12)
    shapes = [(8 * int(rng.integers(1, 9)), 8 * int(rng.integers(1, 33))) for _ in range(300)]
    worst = max(model_rel_err(inp["G"].astype(np.float64)) for inp in matrix_set_inputs(shapes))
    assert worst < 0.8 * NS_BF16_TOL, worst

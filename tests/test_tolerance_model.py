"""Derivation of the bf16 Newton-Schulz tolerance from the arithmetic.

A NumPy model of the tensor-core path's rounding is compared with the fp64
oracle.  In the model, the operands X, A and B are bf16, rounded to nearest
even. Products accumulate exactly, standing in for the fp32 accumulator. X is
kept in bf16 between steps, and the aX term uses that same operand.

The measured errors justify the tolerances the GPU tests use. Under both
normalisations the model stays inside the 2e-2 bound that the workload
specification states for bf16 NS:

* Frobenius scale (X0 = M/||M||_F): about 1.3e-2.
* Spectral scale (X0 = M/(||M||_F sigma_hat)): about 1.7e-2. The singular
  values start near 1, where the quintic is more sensitive to rounding.

The model also records the reason X is not carried in fp32. An fp32 master
of X in the aX term, while the products use its bf16 rounding, measures a
larger error (1.6e-2 Frobenius, 2.2e-2 spectral): it breaks the consistency
between the aX term and the products.
"""
import numpy as np
import pytest
import torch

from oracle import muon as om
from tests.gpu_helpers import NS_BF16_SPECTRAL_TOL, NS_BF16_TOL

A, B, C = om.NS_A, om.NS_B, om.NS_C


def _bf(x):
    return torch.from_numpy(np.asarray(x, np.float32)).bfloat16().double().numpy()


def _f32(x):
    return np.asarray(x, np.float32).astype(np.float64)


def _ns_bf16_model(X0, steps=5, fp32_master=False):
    Xf = _f32(X0)
    Xb = _bf(Xf)
    for _ in range(steps):
        Ab = _bf(_f32(Xb @ Xb.T))
        Bb = _bf(_f32(B * Ab + C * _f32(Ab @ Ab)))
        Xf = _f32(A * (Xf if fp32_master else Xb) + Bb @ Xb)
        Xb = _bf(Xf)
    return Xf


@pytest.mark.parametrize("shape", [(96, 200), (256, 512)])
def test_bf16_model_error_levels(shape):
    worst = {"f": 0.0, "s": 0.0, "f_master": 0.0, "s_master": 0.0}
    for seed in range(3):
        M = np.random.default_rng(seed).standard_normal(shape)
        F = M / np.linalg.norm(M)
        s = om.spectral_estimate(F, 8)
        for key, X0 in (("f", F), ("s", F / s)):
            ref = om.ns_iterate(X0)
            for suffix, master in (("", False), ("_master", True)):
                err = np.linalg.norm(_ns_bf16_model(X0, fp32_master=master) - ref) / np.linalg.norm(ref)
                worst[key + suffix] = max(worst[key + suffix], err)
    assert worst["f"] < 0.75 * NS_BF16_TOL
    assert worst["s"] < 0.9 * NS_BF16_SPECTRAL_TOL
    # the design choice: the bf16-consistent aX term is the more accurate one
    assert worst["f"] < worst["f_master"] and worst["s"] < worst["s_master"]

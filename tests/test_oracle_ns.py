"""Pins of the oracle's Muon math against mathematics independent of it.

Newton-Schulz: for X0 = U S V^T the k-step quintic is U p^k(S) V^T with
p(s) = a s + b s^3 + c s^5 (each step maps every singular value through p and
keeps the singular vectors).  The cubic special case (a, b, c) = (3/2, -1/2, 0)
is the classical NS iteration, which converges to the polar factor U V^T.
"""
from fractions import Fraction

import numpy as np
import pytest
import scipy.linalg

from oracle import muon as om

A, B, C = om.NS_A, om.NS_B, om.NS_C


def _p(s, a=A, b=B, c=C):
    return a * s + b * s ** 3 + c * s ** 5


def _closed_form(M, steps, a=A, b=B, c=C):
    """U p^k(S) V^T from an SVD of M/||M||_F (no orientation needed: the
    identity holds for either orientation)."""
    X0 = M / np.linalg.norm(M)
    U, S, Vt = np.linalg.svd(X0, full_matrices=False)
    for _ in range(steps):
        S = _p(S, a, b, c)
    return (U * S) @ Vt


@pytest.mark.parametrize("shape", [(5, 9), (9, 5), (16, 16), (40, 70), (70, 40)])
@pytest.mark.parametrize("steps", [0, 1, 2, 5])
def test_ns_matches_svd_closed_form(shape, steps):
    M = np.random.default_rng(hash(shape) % 1000).standard_normal(shape)
    O = om.newton_schulz(M, steps)
    assert O.shape == M.shape
    np.testing.assert_allclose(O, _closed_form(M, steps), rtol=0, atol=1e-11)


def test_ns_closed_form_other_coefficients():
    rng = np.random.default_rng(3)
    M = rng.standard_normal((12, 20))
    coeffs = (2.0, -1.5, 0.5)
    O = om.newton_schulz(M, 3, *coeffs)
    np.testing.assert_allclose(O, _closed_form(M, 3, *coeffs), atol=1e-11)


def test_ns_hand_example_exact():
    # M = [[3,0,0],[0,4,0]] -> ||M||_F = 5, singular values 0.6, 0.8 on the
    # coordinate axes.  One step maps them through p exactly.
    M = np.array([[3.0, 0, 0], [0, 4.0, 0]])
    a, b, c = Fraction("3.4445"), Fraction("-4.7750"), Fraction("2.0315")
    def p(s):
        return a * s + b * s ** 3 + c * s ** 5
    want = np.zeros((2, 3))
    want[0, 0] = float(p(Fraction(3, 5)))
    want[1, 1] = float(p(Fraction(4, 5)))
    np.testing.assert_allclose(om.newton_schulz(M, 1), want, rtol=1e-14, atol=1e-15)
    # p(1) = a + b + c = 0.701 exactly
    assert a + b + c == Fraction("0.701")


def test_cubic_ns_reaches_polar_factor():
    rng = np.random.default_rng(5)
    Q1, _ = np.linalg.qr(rng.standard_normal((24, 24)))
    Q2, _ = np.linalg.qr(rng.standard_normal((40, 40)))
    S = np.linspace(0.3, 1.0, 24)
    M = (Q1 * S) @ Q2[:24]
    X0 = M / np.linalg.norm(M)
    O = om.ns_iterate(X0, 80, 1.5, -0.5, 0.0)
    # scipy's polar decomposition of the wide matrix through its transpose
    Up, _ = scipy.linalg.polar(M.T)
    np.testing.assert_allclose(O, Up.T, atol=1e-10)


def test_ns_polar_distance_equals_band_gap():
    rng = np.random.default_rng(11)
    M = rng.standard_normal((30, 50))
    O = om.newton_schulz(M, 5)
    U, S, Vt = np.linalg.svd(M / np.linalg.norm(M), full_matrices=False)
    s = S.copy()
    for _ in range(5):
        s = _p(s)
    dist = np.linalg.norm(O - U @ Vt, 2)
    assert abs(dist - np.max(np.abs(s - 1.0))) < 1e-10


def test_ns_output_band_on_gaussian_256x512():
    rng = np.random.default_rng(0)
    M = rng.standard_normal((256, 512))
    O = om.newton_schulz(M, 5)
    sv = np.linalg.svd(O, compute_uv=False)
    grid = np.linspace(1e-7, 1.0, 2_000_001)
    g = grid.copy()
    for _ in range(5):
        g = _p(g)
    hi = g.max()
    lo = g[grid >= 0.0015].min()
    # max of p^5 over (0, 1] is ~1.20237; over [0.0015, 1] p^5 stays above ~0.6799
    assert 1.2023 < hi < 1.2025 and 0.679 < lo < 0.681
    assert sv.max() <= hi + 1e-12 and sv.min() >= lo - 1e-12
    # input singular values of M/||M|| lie well inside [0.0015, 1]
    sin = np.linalg.svd(M / np.linalg.norm(M), compute_uv=False)
    assert sin.min() > 0.0015


@pytest.mark.parametrize("j", [-7, -1, 1, 5, 40])
def test_ns_power_of_two_scale_is_bitwise(j):
    M = np.random.default_rng(2).standard_normal((20, 33))
    assert np.array_equal(om.newton_schulz(M * 2.0 ** j), om.newton_schulz(M))


def test_ns_positive_scale_invariance():
    M = np.random.default_rng(4).standard_normal((20, 33))
    np.testing.assert_allclose(om.newton_schulz(3.7 * M), om.newton_schulz(M), atol=1e-12)


def test_ns_transpose_equivariance():
    M = np.random.default_rng(6).standard_normal((17, 29))
    np.testing.assert_allclose(om.newton_schulz(M.T), om.newton_schulz(M).T, atol=1e-12)


def test_ns_orientation_is_result_neutral():
    # iterating on the tall matrix directly gives the same result as the m<=n
    # orientation (X(X^TX) = (XX^T)X), so the transpose is a cost choice only
    M = np.random.default_rng(8).standard_normal((29, 17))
    X0 = M / np.linalg.norm(M)
    tall = X0
    for _ in range(5):
        Gm = tall.T @ tall
        tall = A * tall + tall @ (B * Gm + C * Gm @ Gm)
    np.testing.assert_allclose(om.newton_schulz(M), tall, atol=1e-12)


def test_ns_orthogonal_equivariance():
    rng = np.random.default_rng(9)
    M = rng.standard_normal((12, 18))
    Q1, _ = np.linalg.qr(rng.standard_normal((12, 12)))
    Q2, _ = np.linalg.qr(rng.standard_normal((18, 18)))
    np.testing.assert_allclose(om.newton_schulz(Q1 @ M @ Q2), Q1 @ om.newton_schulz(M) @ Q2,
                               atol=1e-12)


def test_ns_degenerate_cases():
    M = np.random.default_rng(10).standard_normal((8, 13))
    np.testing.assert_allclose(om.newton_schulz(M, 0), M / np.linalg.norm(M), atol=1e-15)
    np.testing.assert_allclose(om.newton_schulz(M, 4, 1.0, 0.0, 0.0), M / np.linalg.norm(M),
                               atol=1e-15)
    Z = np.zeros((6, 4))
    assert np.array_equal(om.newton_schulz(Z), Z)


def test_spectral_estimate_converges_to_sigma_max():
    rng = np.random.default_rng(14)
    Q1, _ = np.linalg.qr(rng.standard_normal((16, 16)))
    Q2, _ = np.linalg.qr(rng.standard_normal((30, 30)))
    s = np.array([3.0] + list(np.linspace(0.2, 1.5, 15)))    # a clear spectral gap
    M = (Q1 * s) @ Q2[:16]
    assert abs(om.spectral_estimate(M, 60) - 3.0) < 1e-10
    # power iteration from below: each iterate's Rayleigh quotient is <= sigma_max^2
    assert all(om.spectral_estimate(M, q) <= 3.0 + 1e-12 for q in range(0, 8))
    X0, scale = om.spectral_normalize(M, 60)
    np.testing.assert_allclose(X0, M / 3.0, atol=1e-12)
    assert abs(scale - 3.0) < 1e-10


def test_spectral_scaled_ns_closed_form_and_invariance():
    rng = np.random.default_rng(15)
    M = rng.standard_normal((20, 36))
    O = om.newton_schulz(M, 5, spectral_iters=8)
    F = M / np.linalg.norm(M)
    sig = om.spectral_estimate(F, 8)
    U, S, Vt = np.linalg.svd(F / sig, full_matrices=False)
    for _ in range(5):
        S = _p(S)
    np.testing.assert_allclose(O, (U * S) @ Vt, atol=1e-11)
    np.testing.assert_allclose(om.newton_schulz(2.5 * M, 5, spectral_iters=8), O, atol=1e-12)
    np.testing.assert_allclose(om.newton_schulz(M.T, 5, spectral_iters=8), O.T, atol=1e-12)


def test_momentum_special_cases():
    rng = np.random.default_rng(12)
    M0, G = rng.standard_normal((5, 7)), rng.standard_normal((5, 7))
    assert np.array_equal(om.momentum(M0, G, 0.0), G)
    assert np.array_equal(om.momentum(M0, np.zeros_like(G), 0.95), 0.95 * M0)
    G2 = rng.standard_normal((5, 7))
    M2 = om.momentum(om.momentum(M0, G, 0.9), G2, 0.9)
    np.testing.assert_allclose(M2, 0.81 * M0 + 0.9 * G + G2, atol=1e-14)


def test_muon_step_composes_momentum_ns_update():
    rng = np.random.default_rng(13)
    W, M0, G = (rng.standard_normal((10, 6)) for _ in range(3))
    W1, M1, O = om.muon_step(W, M0, G, mu=0.95, lr=0.02, update_scale=1.5, weight_decay=0.1)
    np.testing.assert_allclose(M1, 0.95 * M0 + G, atol=1e-15)
    np.testing.assert_allclose(O, _closed_form(0.95 * M0 + G, 5), atol=1e-11)
    np.testing.assert_allclose(W1, W * (1 - 0.02 * 0.1) - 0.02 * 1.5 * O, atol=1e-13)
    W2, _, _ = om.muon_step(W, M0, G, mu=0.95, lr=0.02, apply_update=False)
    assert np.array_equal(W2, W)


def test_muon_update_pins():
    """The update against facts its formula does not restate.
    * Descent: for a linear loss <G, W> and mu = 0, the step changes the loss
      by -lr * s * <G, O> = -lr * s * sum_i sigma_i p^5(sigma_i / ||G||_F),
      computed here from the singular values of G alone (negative: a wrong
      sign, scale or operand of the update fails).
    * Decoupled decay: a zero gradient gives a zero direction, so the step
      only shrinks W by the factor (1 - lr * wd), and leaves it as is at wd = 0.
    * Size: the step's spectral norm over lr * s lies in the NS output band."""
    rng = np.random.default_rng(17)
    W, G = rng.standard_normal((12, 30)), rng.standard_normal((12, 30))
    lr, s = 0.02, 1.5
    W1, _, _ = om.muon_step(W, np.zeros_like(W), G, mu=0.0, lr=lr, update_scale=s)
    sv = np.linalg.svd(G, compute_uv=False)
    q = sv / np.linalg.norm(G)
    for _ in range(5):
        q = _p(q)
    want = -lr * s * float(np.sum(sv * q))
    assert want < 0
    np.testing.assert_allclose(float(np.sum(G * (W1 - W))), want, rtol=1e-10)
    Z = np.zeros_like(G)
    Wd, _, _ = om.muon_step(W, Z, Z, mu=0.9, lr=lr, weight_decay=0.3)
    np.testing.assert_allclose(Wd, (1 - lr * 0.3) * W, rtol=1e-15)
    W0, _, _ = om.muon_step(W, Z, Z, mu=0.9, lr=lr)
    assert np.array_equal(W0, W)
    step_norm = np.linalg.norm(W1 - W, 2) / (lr * s)
    assert 0.68 < step_norm < 1.2024


def test_ns_flops_count():
    assert om.ns_flops(4096, 4096) == 5 * 6 * 4096 ** 3
    assert om.ns_flops(11008, 4096) == om.ns_flops(4096, 11008) == \
        5 * (4 * 4096 ** 2 * 11008 + 2 * 4096 ** 3)

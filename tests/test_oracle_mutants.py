"""The NS and vote pins must catch plausible slips in the oracle.

Each mutant below is a plausible mistake planted into a copy of the oracle's
arithmetic on the CPU; the closed-form / brute-force checks used by the pin
tests must reject every one of them.
"""
import itertools

import numpy as np

from oracle import muon as om
from oracle import sign as osg

A, B, C = om.NS_A, om.NS_B, om.NS_C


def _closed_form(M, steps):
    U, S, Vt = np.linalg.svd(M / np.linalg.norm(M), full_matrices=False)
    for _ in range(steps):
        S = A * S + B * S ** 3 + C * S ** 5
    return (U * S) @ Vt


def _mutant_ns(M, kind, steps=5):
    X, tr = (M.T, True) if M.shape[0] > M.shape[1] else (M, False)
    X = X / np.linalg.norm(X)
    for _ in range(steps):
        G = X @ X.T
        if kind == "dropped_quintic":
            P = B * G
        elif kind == "sign_flip_b":
            P = -B * G + C * G @ G
        elif kind == "swapped_bc":
            P = C * G + B * G @ G
        elif kind == "left_right":
            P = B * G + C * G @ G
            X = A * X + (P @ X) @ (X.T @ X) / np.trace(X.T @ X)
            continue
        elif kind == "no_transpose_back":
            P = B * G + C * G @ G
        else:
            P = B * G + C * G @ G
        X = A * X + P @ X
    if tr and kind != "no_transpose_back":
        X = X.T
    return X


def test_ns_pins_reject_mutants():
    rng = np.random.default_rng(0)
    for shape in [(12, 20), (20, 12)]:
        M = rng.standard_normal(shape)
        ref = _closed_form(M, 5)
        assert np.allclose(_mutant_ns(M, "none"), ref, atol=1e-10)
        kinds = ["dropped_quintic", "sign_flip_b", "swapped_bc", "left_right"]
        if shape[0] > shape[1]:
            kinds.append("no_transpose_back")      # only tall matrices are transposed
        for kind in kinds:
            out = _mutant_ns(M, kind)
            assert out.shape != ref.shape or not np.allclose(out, ref, atol=1e-6), kind


def test_vote_brute_force_rejects_tie_and_order_mutants():
    M = 4
    pats = list(itertools.product([-1.0, 1.0], repeat=M))
    S = np.array(pats)
    bufs = [osg.pack_bits(S[:, m]) for m in range(M)]
    want = np.array([1.0 if sum(p) >= 0 else -1.0 for p in pats])
    assert np.array_equal(osg.majority_vote(bufs, len(pats)), want)
    c = osg.vote_counts(bufs, len(pats))
    ties_down = np.where(2 * c > M, 1.0, -1.0)              # ties -> -1
    assert not np.array_equal(ties_down, want)
    be = [np.array([int('{:032b}'.format(int(w))[::-1], 2) for w in b], dtype=np.uint32)
          for b in bufs]                                      # bit order reversed
    assert not np.array_equal(osg.majority_vote(be, len(pats)), want)

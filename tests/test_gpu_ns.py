"""GPU parity of the Newton-Schulz path through the C ABI: each phase alone
(via the workspace view), ns_orthogonalize in bf16 and fp32 modes, the
degenerate cases, and the invariances the oracle is pinned to."""
import numpy as np
import pytest
import torch

import matrix_optimizers_gb300 as mo
from matrix_optimizers_gb300 import _binding as B
from oracle import bf16 as ob
from oracle import muon as om
from workloads import tight_spectrum_matrix
from tests.gpu_helpers import NS_BF16_TOL, NS_FP32_TOL, dev, rel_fro, to_dev, to_np, workspace, ws_view

pytestmark = pytest.mark.gpu

A, Bc, C = om.NS_A, om.NS_B, om.NS_C


def _ns(X_list, steps=5, precision=mo.MO_NS_BF16, out_dtype=torch.float32, coeffs=(A, Bc, C), lds=None):
    shapes = [tuple(x.shape) for x in X_list]
    ws = workspace(mo.ns_workspace_bytes(shapes, precision))
    # the ABI wants ld * element size a multiple of 16 bytes: pad odd widths
    # (the padding is NaN-filled, so a kernel reading it would show)
    lds = lds or [None if s[1] % 8 == 0 else (s[1] + 7) // 8 * 8 for s in shapes]
    Xt = [to_dev(x, torch.float32, ld) for x, ld in zip(X_list, lds)]
    outs = []
    for x, ld in zip(X_list, lds):
        o = to_dev(np.zeros(x.shape), out_dtype, ld)
        outs.append(o)
    mo.ns_orthogonalize(Xt, outs, steps, ws, *coeffs, precision=precision)
    torch.cuda.synchronize()
    assert mo.mo_check_device_status(ws) == 0
    return [to_np(o) for o in outs], ws, Xt


@pytest.mark.parametrize("shape", [(256, 512), (128, 256), (200, 300), (300, 200), (64, 64), (640, 700)])
def test_phases_individually(shape):
    """steps = 1: the Gram, polynomial and apply buffers each match the oracle
    computed from the bf16 operands the kernels used.  m = 200, 256 and 640
    include tiles whose first 128 columns lie below the diagonal (computed
    as half tiles), 640 two of them per phase."""
    X = np.random.default_rng(1).standard_normal(shape)
    outs, ws, _ = _ns([X], steps=1)
    v = B.mo_debug_ns_view([shape], 0)
    m, n = v.m, v.n
    Xo = X.T if v.transposed else X
    s = np.linalg.norm(Xo.astype(np.float32).astype(np.float64))
    Xb = ob.round_bf16(Xo.astype(np.float32).astype(np.float64))        # operand the kernels read
    # the bf16 operand lives in 8-column blocks of v.ldx rows: [block][row][8]
    nb = -(-n // 8)
    blk = ws[v.x_op[0]: v.x_op[0] + nb * v.ldx * 16].view(torch.bfloat16).view(nb, v.ldx, 8)
    xb_dev = to_np(blk[:, :m, :].permute(1, 0, 2).reshape(m, nb * 8)[:, :n])
    assert np.array_equal(xb_dev, Xb)
    gram = to_np(ws_view(ws, v.gram, (m, m), torch.bfloat16, v.lda))
    want_gram = Xb @ Xb.T / s ** 2
    assert rel_fro(gram, want_gram) < 4e-3                                # bf16 storage of A
    for r0 in range(0, m, 128):                                           # every 128-row block, on its own
        assert rel_fro(gram[r0:r0 + 128], want_gram[r0:r0 + 128]) < 4e-3
    assert np.array_equal(gram, gram.T)                                   # mirrored exactly
    poly = to_np(ws_view(ws, v.poly, (m, m), torch.bfloat16, v.lda))
    want_poly = A * np.eye(m) + Bc * gram + C * gram @ gram              # a folded onto the diagonal
    assert rel_fro(poly, want_poly) < 4e-3
    assert np.array_equal(poly, poly.T)
    # the diagonal's bf16 rounding residual, kept in fp32: within half a bf16
    # spacing of the stored diagonal, and restoring it to fp32 accuracy
    res = to_np(ws[v.diag_res: v.diag_res + 4 * m].view(torch.float32))
    d = np.diag(poly)
    assert np.all(np.abs(res) <= np.spacing(np.abs(d).astype(np.float32)) * 2.0 ** 15)
    np.testing.assert_allclose(d + res, np.diag(want_poly), rtol=2e-6, atol=1e-6)
    want_x1 = (poly + np.diag(res)) @ Xb / s                              # X1 = (aI + bA + cA^2) X0
    got = outs[0].T if v.transposed else outs[0]
    assert rel_fro(got, want_x1) < 1e-5


@pytest.mark.parametrize("shape", [(256, 512), (768, 768), (768, 3072), (3072, 768), (100, 300),
                                   (300, 100), (64, 64), (8, 40), (1, 33), (200, 1000), (1000, 200),
                                   (520, 1032), (136, 2056)])
def test_ns_bf16_vs_oracle(shape):
    X = np.random.default_rng(sum(shape)).standard_normal(shape)
    got = _ns([X])[0][0]
    want = om.newton_schulz(X.astype(np.float32).astype(np.float64))
    assert rel_fro(got, want) < NS_BF16_TOL


@pytest.mark.parametrize("m,n,kind", [(32, 256, "tight"), (48, 256, "tight"), (384, 768, "tight"),
                                      (768, 384, "tight"), (32, 200, "gauss"), (32, 240, "gauss")])
def test_ns_bf16_tight_spectrum(m, n, kind):
    """Inputs whose singular values all start near 1/sqrt(m), where bf16 NS is
    most sensitive to the rounding of B's diagonal (without its fp32 residual
    these land at 2.1e-2 to 2.5e-2): inside the plain bound."""
    if kind == "tight":
        X = tight_spectrum_matrix(min(m, n), max(m, n), 0).astype(np.float64)
        X = X if m <= n else X.T
    else:
        X = np.random.default_rng(0).standard_normal((m, n)).astype(np.float32).astype(np.float64)
    got = _ns([X])[0][0]
    assert rel_fro(got, om.newton_schulz(X)) < NS_BF16_TOL


@pytest.mark.parametrize("shape", [(64, 8192), (8192, 64), (72, 4104)])
def test_ns_bf16_extreme_aspect(shape):
    """One row tile against a K of thousands in the Gram phase, and dozens of
    apply tiles per row tile (aspect ratios up to 1:128)."""
    X = np.random.default_rng(sum(shape) + 2).standard_normal(shape)
    got = _ns([X])[0][0]
    want = om.newton_schulz(X.astype(np.float32).astype(np.float64))
    assert rel_fro(got, want) < NS_BF16_TOL


@pytest.mark.parametrize("precision", [mo.MO_NS_BF16, mo.MO_NS_FP32])
def test_ns_rank_deficient(precision):
    """Rank-5 input.  Zero is a fixed point of the quintic, but an unstable one
    (slope a = 3.4445), so rounding noise in the null space grows step by step.
    In fp32 the output matches the oracle in full.  In bf16 that noise reaches
    singular values near 0.16 (the rounding model puts it at 0.158), so the
    check is on the part of the output in the input's row and column spaces,
    which carries the result, with the null-space part bounded."""
    rng = np.random.default_rng(8)
    X = rng.standard_normal((192, 5)) @ rng.standard_normal((5, 320))
    x32 = X.astype(np.float32).astype(np.float64)
    got = _ns([X], precision=precision)[0][0]
    want = om.newton_schulz(x32)
    if precision == mo.MO_NS_FP32:
        assert rel_fro(got, want) < NS_FP32_TOL
        return
    U, _, Vt = np.linalg.svd(x32, full_matrices=False)
    Q, P = U[:, :5] @ U[:, :5].T, Vt[:5].T @ Vt[:5]
    assert rel_fro(Q @ got @ P, want) < NS_BF16_TOL
    sv = np.linalg.svd(got, compute_uv=False)
    assert sv[5] < 0.4 * sv[0]


def test_ns_bf16_batch_mixed_shapes_and_ld():
    rng = np.random.default_rng(7)
    shapes = [(256, 512), (512, 256), (96, 160), (384, 384), (72, 576)]
    lds = [520, 264, 168, None, 584]
    X = [rng.standard_normal(s) for s in shapes]
    outs, _, _ = _ns(X, lds=lds)
    for x, o in zip(X, outs):
        assert rel_fro(o, om.newton_schulz(x.astype(np.float32).astype(np.float64))) < NS_BF16_TOL


@pytest.mark.parametrize("shape", [(256, 512), (300, 200), (64, 64), (130, 70), (1, 9)])
def test_ns_fp32_vs_oracle(shape):
    X = np.random.default_rng(sum(shape) + 1).standard_normal(shape)
    got = _ns([X], precision=mo.MO_NS_FP32)[0][0]
    want = om.newton_schulz(X.astype(np.float32).astype(np.float64))
    assert rel_fro(got, want) < NS_FP32_TOL


@pytest.mark.parametrize("precision", [mo.MO_NS_BF16, mo.MO_NS_FP32])
def test_ns_degenerate(precision):
    rng = np.random.default_rng(3)
    X = rng.standard_normal((96, 200))
    got0 = _ns([X], steps=0, precision=precision)[0][0]
    x32 = X.astype(np.float32).astype(np.float64)
    assert rel_fro(got0, x32 / np.linalg.norm(x32)) < 1e-6
    Z = np.zeros((64, 128))
    assert np.all(_ns([Z], precision=precision)[0][0] == 0)
    ident = _ns([X], steps=3, precision=precision, coeffs=(1.0, 0.0, 0.0))[0][0]
    assert rel_fro(ident, x32 / np.linalg.norm(x32)) < (3e-3 if precision == mo.MO_NS_BF16 else 1e-6)


@pytest.mark.parametrize("precision", [mo.MO_NS_BF16, mo.MO_NS_FP32])
def test_ns_power_of_two_scale_is_bitwise(precision):
    X = np.random.default_rng(4).standard_normal((192, 320))
    a = _ns([X], precision=precision)[0][0]
    b = _ns([X * 2.0 ** 5], precision=precision)[0][0]
    c = _ns([X * 2.0 ** -9], precision=precision)[0][0]
    assert np.array_equal(a, b) and np.array_equal(a, c)


def test_ns_transpose_equivariance():
    # the bf16 operand is the same matrix either way; only the order of the
    # norm's partial sums differs, so agreement is to bf16 noise, not bitwise
    X = np.random.default_rng(5).standard_normal((160, 288))
    a = _ns([X])[0][0]
    b = _ns([np.ascontiguousarray(X.T)])[0][0]
    assert rel_fro(b.T, a) < 5e-3


def test_ns_output_band():
    X = np.random.default_rng(0).standard_normal((256, 512))
    got = _ns([X])[0][0]
    sv = np.linalg.svd(got, compute_uv=False)
    assert sv.max() < 1.2024 * 1.03 and sv.min() > 0.6799 * 0.97


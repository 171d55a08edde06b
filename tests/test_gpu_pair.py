"""The CTA-pair geometry of the NS kernel (256 x 256 tiles, tcgen05
cta_group::2 across a cluster of two CTAs) against the single-CTA geometry
(128 x 256 tiles) and the oracle, over ragged shapes, tails below one tile,
transposed matrices and every output form.  The two geometries schedule
different tiles and each walks K backwards on every other tile of a CTA's
list, so their fp32 sums differ in order: they agree to accumulation noise,
not bit for bit."""
import numpy as np
import pytest
import torch

import matrix_optimizers_gb300 as mo
from matrix_optimizers_gb300 import _binding as B
from oracle import muon as om
from tests.gpu_helpers import NS_BF16_SPECTRAL_TOL, NS_BF16_TOL, dev, rel_fro, to_np, workspace

pytestmark = pytest.mark.gpu

CASES = [
    ([(256, 512)], {}),
    ([(64, 64), (96, 200), (130, 132), (200, 96)], {}),
    ([(512, 256), (768, 3072), (1000, 1200), (2048, 2048)], {}),
    ([(300, 700), (4096, 1024)], {"ns_steps": 2}),
    ([(512, 1536), (200, 96)], {"spectral_iters": 6}),
    ([(384, 640), (640, 384)], {"apply_update": False, "out_dtype": mo.MO_BF16}),
]


def _inputs(shapes, seed):
    rng = np.random.default_rng(seed)
    return [{"W": (0.02 * rng.standard_normal(s)).astype(np.float32),
             "G": rng.standard_normal(s).astype(np.float32)} for s in shapes]


def _step(inputs, kw, pair, fused=3):
    prev_p = B.mo_debug_set_ns_pair(pair)
    prev_f = B.mo_debug_set_ns_fused(fused)
    try:
        Ws = [torch.from_numpy(x["W"]).to(dev()) for x in inputs]
        Ms = [torch.zeros_like(w) for w in Ws]
        Gs = [torch.from_numpy(x["G"]).to(dev()) for x in inputs]
        mats = [mo.make_matrix(w, m, g) for w, m, g in zip(Ws, Ms, Gs)]
        cfg = mo.make_cfg(mu=0.95, lr=0.02, **kw)
        out = None
        if kw.get("apply_update", True) is False:
            out = [torch.full(w.shape, float("nan"), dtype=torch.bfloat16, device=dev()) for w in Ws]
        ws = workspace(mo.mo_workspace_bytes(mats, cfg))
        mo.muon_step_batched(mats, cfg, ws, out=out)
        torch.cuda.synchronize()
        assert mo.mo_check_device_status(ws) == 0
        return out if out is not None else Ws
    finally:
        B.mo_debug_set_ns_fused(prev_f)
        B.mo_debug_set_ns_pair(prev_p)


def _diff(a, b):
    return rel_fro(to_np(a), to_np(b))


@pytest.mark.parametrize("fused", [0, 3])
@pytest.mark.parametrize("case", range(len(CASES)))
def test_pair_vs_single_and_oracle(case, fused):
    shapes, kw = CASES[case]
    inputs = _inputs(shapes, 300 + case)
    Rp = _step(inputs, kw, True, fused)
    Rs = _step(inputs, kw, False, fused)
    spectral = kw.get("spectral_iters", 0)
    tol = NS_BF16_SPECTRAL_TOL if spectral else NS_BF16_TOL
    for a, b, inp, s in zip(Rp, Rs, inputs, shapes):
        assert torch.isfinite(a.float()).all(), s
        W0 = inp["W"].astype(np.float64)
        Wn, _, _ = om.muon_step(W0, np.zeros_like(W0), inp["G"], mu=0.95, lr=0.02,
                                spectral_iters=spectral, steps=kw.get("ns_steps", 5))
        if kw.get("apply_update", True) is False:
            O = om.newton_schulz(om.momentum(np.zeros_like(W0), inp["G"], 0.95), kw.get("ns_steps", 5))
            assert rel_fro(to_np(a), O) < tol, s
        else:
            assert rel_fro(to_np(a) - W0, Wn - W0) < tol, s
        # the same products, summed in another K order
        if kw.get("apply_update", True) is False:
            assert _diff(a, b) < 2e-3, s
        else:
            W0t = torch.from_numpy(inp["W"]).to(dev())
            assert _diff(a - W0t, b - W0t) < 2e-3, s


def test_pair_sign_packed_equals_single():
    shapes = [(256, 512), (96, 160), (160, 96), (2048, 2048)]
    rng = np.random.default_rng(77)
    G = [rng.standard_normal(s).astype(np.float32) for s in shapes]
    cfg = mo.make_cfg(mu=0.95, apply_update=False, out_dtype=mo.MO_BF16)
    res = []
    for pair in (True, False):
        prev = B.mo_debug_set_ns_pair(pair)
        try:
            Ms = [torch.zeros(s, dtype=torch.bfloat16, device=dev()) for s in shapes]
            Gs = [torch.from_numpy(g).to(dev()) for g in G]
            mats = [mo.make_matrix(m, m, g) for m, g in zip(Ms, Gs)]
            words = [torch.full(((s[0] * s[1] + 31) // 32,), -7, dtype=torch.int32, device=dev()) for s in shapes]
            ws = workspace(mo.mo_workspace_bytes(mats, cfg))
            mo.muon_step_sign_packed(mats, cfg, words, ws)
            torch.cuda.synchronize()
            assert mo.mo_check_device_status(ws) == 0
            res.append(words)
        finally:
            B.mo_debug_set_ns_pair(prev)
    # a sign can differ only where the two accumulation orders straddle zero
    for a, b, s in zip(res[0], res[1], shapes):
        flips = int(torch.sum(torch.bitwise_xor(a, b) != 0).item())
        assert flips <= max(2, a.numel() // 500), (s, flips)

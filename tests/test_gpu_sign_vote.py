"""GPU parity of muon_step_sign_vote, the whole Sign-Muon step of the M
workers held on one GPU in one call ("Riepilogo Tecnico: SignMuon" §2
"Flusso Algoritmico" steps 1-4): momentum, NS with the sign + 1-bit pack fused
into the last epilogue, and the majority vote with W <- W - lr * vote.  The
updated W must equal, bit for bit, the oracle's vote update over the packed
signs the call wrote; those signs must agree with the signs of the oracle's
NS direction wherever that direction is not within rounding of zero; and the
fused and per-phase NS launches must give W from their signs alike."""
import numpy as np
import pytest
import torch

import matrix_optimizers_gb300 as mo
from matrix_optimizers_gb300 import _binding as B
from oracle import muon as om
from oracle import sign as osg
from tests.gpu_helpers import NS_BF16_TOL, dev, rel_fro, to_np, workspace
from workloads import sign_muon_inputs

pytestmark = pytest.mark.gpu


def _run(G, W0, lr, w_dtype=torch.float32, fused=3, ld=None, spectral=0, off=0):
    shape = G[0].shape
    prev = B.mo_debug_set_ns_fused(fused)
    try:
        Ms = [torch.zeros(shape, dtype=torch.bfloat16, device=dev()) for _ in G]
        Gs = [torch.from_numpy(g).to(dev()) for g in G]
        mats = [mo.make_matrix(m, m, g) for m, g in zip(Ms, Gs)]
        words = [torch.full(((shape[0] * shape[1] + 31) // 32,), -7, dtype=torch.int32, device=dev()) for _ in G]
        if ld is None:
            W = torch.from_numpy(W0).to(dev()).to(w_dtype)
        else:
            buf = torch.full((shape[0], ld), float("nan"), dtype=w_dtype, device=dev())
            buf[:, off: off + shape[1]] = torch.from_numpy(W0).to(dev()).to(w_dtype)
            W = buf[:, off: off + shape[1]]
        cfg = mo.make_cfg(mu=0.95, apply_update=False, out_dtype=mo.MO_BF16, spectral_iters=spectral)
        ws = workspace(mo.mo_workspace_bytes(mats, cfg))
        mo.muon_step_sign_vote(mats, cfg, words, W, lr, ws)
        torch.cuda.synchronize()
        assert mo.mo_check_device_status(ws) == 0
        if ld is not None:
            assert torch.isnan(buf[:, off + shape[1]:].float()).all()      # the padding is untouched
            assert torch.isnan(buf[:, :off].float()).all()
        return W, words, Ms
    finally:
        B.mo_debug_set_ns_fused(prev)


def _check(G, W0, lr, W, words, Ms, w_dtype=torch.float32, spectral=0, ns_check=(0,)):
    wn = [w.cpu().numpy().view(np.uint32) for w in words]
    want = osg.vote_update(W0.astype(np.float64), wn, lr,
                           w_dtype="bf16" if w_dtype == torch.bfloat16 else "f32")
    assert np.array_equal(to_np(W), want)
    # the packed signs are those of directions within the NS bound: rebuild the
    # bf16 direction of worker k with the unfused step and pack it in the oracle
    for k in ns_check:
        _, Mst, O = om.muon_step(np.zeros(G[k].shape), np.zeros(G[k].shape), G[k], mu=0.95, lr=lr, m_dtype="bf16",
                                 apply_update=False, spectral_iters=spectral)
        assert rel_fro(to_np(Ms[k]), Mst) < 1e-7
        agree = np.mean(osg.unpack_bits(wn[k], G[k].size) == (O.reshape(-1) >= 0))
        assert agree > 0.99, agree


def test_sign_muon_m8_step_in_one_call():
    inp = sign_muon_inputs()
    W, words, Ms = _run(inp["G"], inp["W"], 1e-3)
    _check(inp["G"], inp["W"], 1e-3, W, words, Ms, ns_check=(0, 7))


@pytest.mark.parametrize("shape,M,w_dtype,ld,off", [((256, 512), 3, torch.float32, None, 0),
                                                     ((512, 256), 5, torch.float32, 264, 0),
                                                     ((320, 640), 7, torch.bfloat16, None, 0),
                                                     ((96, 160), 2, torch.float32, None, 0),
                                                     ((1000, 1024), 4, torch.float32, 1032, 0),
                                                     ((100, 128), 3, torch.float32, None, 0),
                                                     ((98, 128), 2, torch.float32, None, 0),
                                                     # W rows off 16-byte boundaries (element alignment)
                                                     ((256, 512), 3, torch.float32, 520, 1),
                                                     ((320, 640), 4, torch.bfloat16, 650, 3)])
def test_vote_step_shapes(shape, M, w_dtype, ld, off):
    rng = np.random.default_rng(shape[0] + M)
    G0 = rng.standard_normal(shape)
    G = [(G0 + 0.7 * rng.standard_normal(shape)).astype(np.float32) for _ in range(M)]
    W0 = (0.02 * rng.standard_normal(shape)).astype(np.float32)
    if w_dtype == torch.bfloat16:
        W0 = torch.from_numpy(W0).bfloat16().float().numpy()
    W, words, Ms = _run(G, W0, 2e-3, w_dtype=w_dtype, ld=ld, off=off)
    _check(G, W0, 2e-3, W, words, Ms, w_dtype=w_dtype)


def test_fused_and_per_phase_ns_give_the_same_step():
    """The fused NS launch and one launch per phase compute the same tiles in
    the same order: the same packed signs and the same W, bit for bit."""
    rng = np.random.default_rng(5)
    shape = (384, 768)
    G = [rng.standard_normal(shape).astype(np.float32) for _ in range(6)]
    W0 = (0.02 * rng.standard_normal(shape)).astype(np.float32)
    Wf, wf, _ = _run(G, W0, 1e-3, fused=3)
    Wp, wp, _ = _run(G, W0, 1e-3, fused=0)
    for W, words in ((Wf, wf), (Wp, wp)):
        wn = [w.cpu().numpy().view(np.uint32) for w in words]
        assert np.array_equal(to_np(W), osg.vote_update(W0.astype(np.float64), wn, 1e-3))
    assert all(torch.equal(a, b) for a, b in zip(wf, wp))
    assert torch.equal(Wf, Wp)


def test_vote_step_spectral_scale():
    rng = np.random.default_rng(9)
    shape = (256, 768)
    G = [rng.standard_normal(shape).astype(np.float32) for _ in range(4)]
    W0 = (0.02 * rng.standard_normal(shape)).astype(np.float32)
    W, words, Ms = _run(G, W0, 1e-3, spectral=6)
    _check(G, W0, 1e-3, W, words, Ms, spectral=6)

"""The fused Newton-Schulz launch (every (step, phase) of a call in one
cooperative persistent grid ordered by per-matrix completion counters)
against the per-phase launches: the same tiles with the same arithmetic, so
the results must agree bit for bit; plus the launch structure and the final
counter values."""
import numpy as np
import pytest
import torch

import matrix_optimizers_gb300 as mo
from matrix_optimizers_gb300 import _binding as B
from oracle import muon as om
from tests.gpu_helpers import NS_BF16_TOL, dev, rel_fro, to_np, workspace

pytestmark = pytest.mark.gpu

CASES = [
    ([(256, 512)], {}),
    ([(512, 256), (96, 200), (768, 3072), (130, 132)], {}),
    ([(1024, 4096), (4096, 1024), (64, 64)], {"ns_steps": 1}),
    ([(300, 700), (2048, 2048)], {"ns_steps": 2}),
    ([(512, 1536), (200, 96)], {"spectral_iters": 6}),
    ([(384, 640), (640, 384)], {"apply_update": False, "out_dtype": mo.MO_BF16}),
    ([(128 * k, 256 * (k + 1)) for k in range(1, 9)], {}),
]


def _inputs(shapes, seed):
    rng = np.random.default_rng(seed)
    return [{"W": (0.02 * rng.standard_normal(s)).astype(np.float32),
             "G": rng.standard_normal(s).astype(np.float32)} for s in shapes]


def _step(inputs, cfg_kw, fused):
    prev = B.mo_debug_set_ns_fused(fused)
    try:
        Ws = [torch.from_numpy(x["W"]).to(dev()) for x in inputs]
        Ms = [torch.zeros_like(w) for w in Ws]
        Gs = [torch.from_numpy(x["G"]).to(dev()) for x in inputs]
        mats = [mo.make_matrix(w, m, g) for w, m, g in zip(Ws, Ms, Gs)]
        cfg = mo.make_cfg(mu=0.95, lr=0.02, **cfg_kw)
        out = None
        if cfg_kw.get("apply_update", True) is False:
            out = [torch.full(w.shape, float("nan"), dtype=torch.bfloat16, device=dev()) for w in Ws]
        ws = workspace(mo.mo_workspace_bytes(mats, cfg))
        mo.mo_trace_enable(64)
        mo.muon_step_batched(mats, cfg, ws, out=out)
        trace = mo.mo_trace_read(64)
        mo.mo_trace_enable(0)
        torch.cuda.synchronize()
        assert mo.mo_check_device_status(ws) == 0
        return (out if out is not None else Ws), Ms, ws, [k for k, _ in trace]
    finally:
        B.mo_debug_set_ns_fused(prev)


@pytest.mark.parametrize("mode", [1, 2])
@pytest.mark.parametrize("case", range(len(CASES)))
def test_fused_equals_per_phase_bitwise(case, mode):
    shapes, kw = CASES[case]
    inputs = _inputs(shapes, 100 + case)
    Rf, Mf, _, kinds_f = _step(inputs, kw, mode)
    Rp, Mp, _, kinds_p = _step(inputs, kw, 0)
    for a, b, s in zip(Rf, Rp, shapes):
        assert torch.equal(a, b), s
    for a, b in zip(Mf, Mp):
        assert torch.equal(a, b)
    steps = kw.get("ns_steps", 5)
    assert kinds_p.count("ns_gram") == steps and kinds_p.count("ns_apply") == steps
    assert "ns_fused" not in kinds_p
    if kw.get("spectral_iters", 0):
        assert kinds_f.count("ns_gram") == 1 and kinds_f.count("spectral_estimate") == 1
    else:
        assert "ns_gram" not in kinds_f
    assert kinds_f.count("ns_fused") == 1 and "ns_apply" not in kinds_f and "ns_poly" not in kinds_f


def test_fused_step_vs_oracle():
    shapes, kw = CASES[1]
    inputs = _inputs(shapes, 7)
    R, _, _, _ = _step(inputs, kw, True)
    for w, inp in zip(R, inputs):
        W0 = inp["W"].astype(np.float64)
        Wn, _, _ = om.muon_step(W0, np.zeros_like(W0), inp["G"], mu=0.95, lr=0.02)
        assert rel_fro(to_np(w) - W0, Wn - W0) < NS_BF16_TOL


@pytest.mark.parametrize("case", [1, 3, 4])
def test_fused_counters_reach_totals(case):
    """Every epilogue warp released every tile of every fused level once."""
    shapes, kw = CASES[case]
    _, _, ws, _ = _step(_inputs(shapes, 5), kw, True)
    steps = kw.get("ns_steps", 5)
    spectral = kw.get("spectral_iters", 0) > 0
    for i in range(len(shapes)):
        v = B.mo_debug_ns_view(shapes, i)
        cnt = ws[v.deps: v.deps + 12].view(torch.int32).cpu().tolist()
        gram_steps = steps - 1 if spectral else steps
        r = v.releases_per_tile
        assert cnt == [r * v.tiles_sym * gram_steps, r * v.tiles_sym * steps, r * v.tiles_apply * steps], i
    views = [B.mo_debug_ns_view(shapes, i) for i in range(len(shapes))]
    lvl = views[-1].deps + 16                          # the grid-wide set follows the last matrix
    assert ws[lvl: lvl + 12].view(torch.int32).cpu().tolist() == [0, 0, 0]
    # grid-wide counters: the per-matrix ones stay 0, the shared set holds the sums
    _, _, ws, _ = _step(_inputs(shapes, 5), kw, 2)
    for v in views:
        assert ws[v.deps: v.deps + 12].view(torch.int32).cpu().tolist() == [0, 0, 0]
    ts, ta = sum(v.tiles_sym for v in views), sum(v.tiles_apply for v in views)
    gram_steps = steps - 1 if spectral else steps
    r = views[0].releases_per_tile
    assert ws[lvl: lvl + 12].view(torch.int32).cpu().tolist() == [r * ts * gram_steps, r * ts * steps,
                                                                 r * ta * steps]
    _, _, ws, _ = _step(_inputs(shapes, 5), kw, 0)
    for v in views:
        assert ws[v.deps: v.deps + 12].view(torch.int32).cpu().tolist() == [0, 0, 0]
    assert ws[lvl: lvl + 12].view(torch.int32).cpu().tolist() == [0, 0, 0]


def test_fused_repeated_calls_reset_counters():
    """The counters are re-zeroed by every call's control-block upload, so a
    second call on the same workspace (cached plan) is fused correctly."""
    shapes, kw = CASES[1]
    inputs = _inputs(shapes, 9)
    prev = B.mo_debug_set_ns_fused(True)
    try:
        Ws = [torch.from_numpy(x["W"]).to(dev()) for x in inputs]
        Ms = [torch.zeros_like(w) for w in Ws]
        Gs = [torch.from_numpy(x["G"]).to(dev()) for x in inputs]
        mats = [mo.make_matrix(w, m, g) for w, m, g in zip(Ws, Ms, Gs)]
        cfg = mo.make_cfg(mu=0.95, lr=0.02)
        ws = workspace(mo.mo_workspace_bytes(mats, cfg))
        for _ in range(3):
            mo.muon_step_batched(mats, cfg, ws)
        torch.cuda.synchronize()
        assert mo.mo_check_device_status(ws) == 0
    finally:
        B.mo_debug_set_ns_fused(prev)
    # the per-phase path from the same initial state, three times
    Rp = [torch.from_numpy(x["W"]).to(dev()) for x in inputs]
    Mp = [torch.zeros_like(w) for w in Rp]
    mats_p = [mo.make_matrix(w, m, g) for w, m, g in zip(Rp, Mp, Gs)]
    prev = B.mo_debug_set_ns_fused(False)
    try:
        ws2 = workspace(mo.mo_workspace_bytes(mats_p, cfg))
        for _ in range(3):
            mo.muon_step_batched(mats_p, cfg, ws2)
        torch.cuda.synchronize()
    finally:
        B.mo_debug_set_ns_fused(prev)
    for a, b in zip(Ws, Rp):
        assert torch.equal(a, b)

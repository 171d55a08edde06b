"""GPU parity of the whole Muon step (muon_step_batched) on the workloads:
momentum, NS, update and the AdamW tail, against the oracle."""
import numpy as np
import pytest
import torch

import matrix_optimizers_gb300 as mo
from oracle import adamw as oa
from oracle.bf16 import round_bf16
from oracle import muon as om
from oracle import planner as oplan
from oracle import sign as osg
from tests.gpu_helpers import (MOM_TOL, NS_BF16_SPECTRAL_TOL, NS_BF16_TOL, NS_FP32_TOL, dev, rel_fro, to_dev,
                               to_np, workspace)
from workloads import (CONFIGS, llama7b_shapes, matrix_inputs, matrix_set_inputs, ragged_shapes,
                       sign_muon_inputs,
                       single_matrix_inputs, tail_inputs)

pytestmark = pytest.mark.gpu


def _run(inputs, cfg, tail=None, out=None, m_dtype=torch.float32):
    Ws = [to_dev(x["W"]) for x in inputs]
    Ms = [to_dev(x["M0"], m_dtype) if "M0" in x else
          torch.zeros(x["W"].shape, dtype=m_dtype, device=dev()) for x in inputs]
    Gs = [to_dev(x["G"]) for x in inputs]
    mats = [mo.make_matrix(w, m, g) for w, m, g in zip(Ws, Ms, Gs)]
    ws = workspace(mo.mo_workspace_bytes(mats, cfg))
    mo.muon_step_batched(mats, cfg, ws, tail=tail, out=out)
    torch.cuda.synchronize()
    assert mo.mo_check_device_status(ws) == 0
    return Ws, Ms


def _check_update(W_gpu, inp, mu, lr, tol, m_dtype="f32"):
    W0 = inp["W"].astype(np.float64)
    M0 = inp["M0"].astype(np.float64) if "M0" in inp else np.zeros_like(W0)
    Wn, _, _ = om.muon_step(W0, M0, inp["G"].astype(np.float64), mu=mu, lr=lr, m_dtype=m_dtype)
    err = rel_fro(to_np(W_gpu) - W0, Wn - W0)
    assert err < tol, err
    return err


def test_single_256x512_fp32_mode():
    cfg_d = CONFIGS["single_256x512"]
    inp = single_matrix_inputs()
    cfg = mo.make_cfg(mu=cfg_d["mu"], lr=cfg_d["lr"], precision=mo.MO_NS_FP32)
    Ws, Ms = _run([inp], cfg)
    M1 = om.momentum(inp["M0"], inp["G"], cfg_d["mu"])
    assert rel_fro(to_np(Ms[0]), M1) < MOM_TOL
    _check_update(Ws[0], inp, cfg_d["mu"], cfg_d["lr"], NS_FP32_TOL)


def test_single_256x512_bf16_mode():
    inp = single_matrix_inputs()
    cfg = mo.make_cfg(mu=0.95, lr=0.02)
    Ws, _ = _run([inp], cfg)
    _check_update(Ws[0], inp, 0.95, 0.02, NS_BF16_TOL)


def test_gpt_small_full_step_with_tail():
    c = CONFIGS["gpt_small"]
    shapes = c["shapes"]
    inputs = [matrix_inputs(shapes, i) for i in range(len(shapes))]
    # a second step with non-zero momentum: run step 1 on the oracle for M0
    for inp in inputs:
        inp["M0"] = (0.5 * inp["G"]).astype(np.float32)
    t = tail_inputs(c["tail_numel"])
    tW, tg, tm_, tv = (torch.from_numpy(t[k]).to(dev()) for k in ("W", "g", "m", "v"))
    tail = mo.make_tail(tW, tg, tm_, tv, step=1, lr=c["tail_lr"])
    cfg = mo.make_cfg(mu=c["mu"], lr=c["lr"])
    Ws, Ms = _run(inputs, cfg, tail=tail)
    worst = 0.0
    for i, inp in enumerate(inputs):
        M1 = om.momentum(inp["M0"], inp["G"], c["mu"])
        assert rel_fro(to_np(Ms[i]), M1) < MOM_TOL
        worst = max(worst, _check_update(Ws[i], inp, c["mu"], c["lr"], NS_BF16_TOL))
    Wt, _, _ = oa.adamw_step(t["W"], t["g"], t["m"], t["v"], 1, lr=c["tail_lr"])
    assert np.max(np.abs(tW.cpu().numpy() - Wt)) < 1e-8


def test_many_tiny_matrices_one_step():
    """300 matrices of 8 to 256 rows and columns, each one or a few tiles, so
    that every CTA holds tiles of many matrices.  This exercises the grouped
    launch, its per-matrix counters and the transposed frame."""
    rng = np.random.default_rng(12)
    shapes = [(8 * int(rng.integers(1, 9)), 8 * int(rng.integers(1, 33))) for _ in range(300)]
    inputs = matrix_set_inputs(shapes)
    cfg = mo.make_cfg(mu=0.95, lr=0.02)
    Ws, _ = _run(inputs, cfg)
    for w, inp in zip(Ws, inputs):
        _check_update(w, inp, 0.95, 0.02, NS_BF16_TOL)


def test_weight_decay_and_update_scale():
    rng = np.random.default_rng(9)
    inp = {"W": rng.standard_normal((128, 384)).astype(np.float32),
           "G": rng.standard_normal((128, 384)).astype(np.float32),
           "M0": rng.standard_normal((128, 384)).astype(np.float32)}
    cfg = mo.make_cfg(mu=0.9, lr=0.05, update_scale=1.7, weight_decay=0.2)
    Ws, _ = _run([inp], cfg)
    W0 = inp["W"].astype(np.float64)
    Wn, _, _ = om.muon_step(W0, inp["M0"], inp["G"], mu=0.9, lr=0.05, update_scale=1.7, weight_decay=0.2)
    assert rel_fro(to_np(Ws[0]) - W0, Wn - W0) < NS_BF16_TOL


def test_bf16_state_dtypes():
    # W starts at 0 so that bf16 storage keeps the update at bf16 relative
    # precision (a unit-scale W would have a bf16 spacing above the update)
    rng = np.random.default_rng(10)
    inp = {"W": np.zeros((192, 256), dtype=np.float32),
           "G": rng.standard_normal((192, 256)).astype(np.float32),
           "M0": rng.standard_normal((192, 256)).astype(np.float32)}
    W = to_dev(inp["W"], torch.bfloat16)
    M = to_dev(inp["M0"], torch.bfloat16)
    G = to_dev(inp["G"], torch.bfloat16)
    W0, M0, G0 = to_np(W), to_np(M), to_np(G)
    mats = [mo.make_matrix(W, M, G)]
    cfg = mo.make_cfg(mu=0.95, lr=0.05)
    ws = workspace(mo.mo_workspace_bytes(mats, cfg))
    mo.muon_step_batched(mats, cfg, ws)
    torch.cuda.synchronize()
    Wn, Mn, _ = om.muon_step(W0, M0, G0, mu=0.95, lr=0.05, m_dtype="bf16")
    # W is stored in bf16: compare the update with bf16 storage noise allowed
    assert rel_fro(to_np(W) - W0, Wn - W0) < 3e-2
    assert rel_fro(to_np(M), Mn) < 4e-3


def _bf16_ulp(x):
    """Spacing of bfloat16 at |x| (8 significant bits)."""
    e = np.floor(np.log2(np.maximum(np.abs(x), np.finfo(np.float32).tiny)))
    return np.exp2(e - 7)


@pytest.mark.parametrize("shapes", [
    # every matrix untransposed with ld % 8 == 0: the 16-byte momentum kernel
    [(192, 256, 256), (70, 203, 208), (130, 130, 136), (64, 1000, 1000)],
    # a transposed matrix in the batch: the general kernel for all of them
    [(192, 256, 256), (70, 203, 208), (300, 100, 104)],
])
def test_bf16_momentum_fp32_gradient(shapes):
    """bf16 momentum with an fp32 gradient (the Sign-Muon workers' state):
    the stored momentum is bf16(mu*M + G), the oracle's value or the bf16
    neighbour that the fp32 fma's double rounding can give, and the update
    matches the oracle's Muon step on that momentum.  Ragged columns (the last
    8-column group partly valid), padded leading dimensions and tiles cut at
    the matrix edge, and a batch that the 16-byte kernel does not take."""
    rng = np.random.default_rng(sum(r * c for r, c, _ in shapes))
    mats, keep = [], []
    for rows, cols, ld in shapes:
        W0 = (0.02 * rng.standard_normal((rows, cols))).astype(np.float32)
        M0 = round_bf16(rng.standard_normal((rows, cols))).astype(np.float32)
        G0 = rng.standard_normal((rows, cols)).astype(np.float32)

        def padded(a, dtype):
            big = torch.zeros((rows, ld), dtype=dtype, device=dev())
            big[:, :cols] = to_dev(a, dtype)
            return big[:, :cols]

        W, M, G = padded(W0, torch.float32), padded(M0, torch.bfloat16), padded(G0, torch.float32)
        assert np.array_equal(to_np(M), M0)
        mats.append(mo.make_matrix(W, M, G))
        keep.append((W, M, G, W0, M0, G0))
    cfg = mo.make_cfg(mu=0.95, lr=0.05)
    ws = workspace(mo.mo_workspace_bytes(mats, cfg))
    mo.muon_step_batched(mats, cfg, ws)
    torch.cuda.synchronize()
    assert mo.mo_check_device_status(ws) == 0
    for (rows, cols, _), (W, M, G, W0, M0, G0) in zip(shapes, keep):
        Wn, Mn, _ = om.muon_step(W0.astype(np.float64), M0.astype(np.float64), G0.astype(np.float64),
                                 mu=0.95, lr=0.05, m_dtype="bf16")
        got = to_np(M).astype(np.float64)
        assert np.all(np.abs(got - Mn) <= _bf16_ulp(Mn)), (rows, cols)
        assert np.mean(got == Mn) > 0.99, (rows, cols)
        assert rel_fro(to_np(W) - W0, Wn - W0) < NS_BF16_TOL, (rows, cols)


@pytest.mark.parametrize("rows,cols,ld,wdt", [
    (100, 264, 268, "f32"),     # ragged 32-row boxes, padded rows
    (264, 100, 104, "f32"),     # transposed frame
    (96, 320, 328, "bf16"),
    (320, 96, 104, "bf16"),
])
def test_update_through_w_boxes(rows, cols, ld, wdt):
    """The last-step update loads and stores W in 32-row boxes: partial boxes at
    the matrix edge, padded rows and the transposed frame give the oracle's
    update, and the padding columns keep their values."""
    rng = np.random.default_rng(rows + 3 * cols)
    W0 = (0.02 * rng.standard_normal((rows, cols))).astype(np.float32) if wdt == "f32" else \
        np.zeros((rows, cols), dtype=np.float32)       # bf16 W: see test_bf16_state_dtypes
    G0 = rng.standard_normal((rows, cols)).astype(np.float32)
    wt = torch.float32 if wdt == "f32" else torch.bfloat16
    sentinel = 7.0

    def padded(a, dtype):
        big = torch.full((rows, ld), sentinel, dtype=dtype, device=dev())
        big[:, :cols] = to_dev(a, dtype)
        return big, big[:, :cols]

    Wb, W = padded(W0, wt)
    Mb, M = padded(np.zeros_like(G0), torch.float32)
    Gb, G = padded(G0, torch.float32)
    W0q = to_np(W)
    mats = [mo.make_matrix(W, M, G)]
    cfg = mo.make_cfg(mu=0.95, lr=0.05)
    ws = workspace(mo.mo_workspace_bytes(mats, cfg))
    mo.muon_step_batched(mats, cfg, ws)
    torch.cuda.synchronize()
    assert mo.mo_check_device_status(ws) == 0
    Wn, _, _ = om.muon_step(W0q.astype(np.float64), np.zeros_like(W0q, dtype=np.float64), G0.astype(np.float64),
                            mu=0.95, lr=0.05)
    tol = NS_BF16_TOL if wdt == "f32" else 3e-2
    assert rel_fro(to_np(W) - W0q, Wn - W0q) < tol
    assert bool((Wb[:, cols:] == sentinel).all())


def test_apply_update_off_writes_output():
    rng = np.random.default_rng(11)
    shapes = [(256, 384), (384, 256)]
    inputs = [{"W": np.zeros(s, np.float32), "G": rng.standard_normal(s).astype(np.float32),
               "M0": np.zeros(s, np.float32)} for s in shapes]
    outs = [torch.zeros(s, dtype=torch.bfloat16, device=dev()) for s in shapes]
    cfg = mo.make_cfg(mu=0.95, lr=0.02, apply_update=False, out_dtype=mo.MO_BF16)
    Ws, _ = _run(inputs, cfg, out=outs)
    for inp, o, w in zip(inputs, outs, Ws):
        assert torch.all(w == 0)
        want = om.newton_schulz(om.momentum(inp["M0"], inp["G"], 0.95))
        assert rel_fro(to_np(o), want) < NS_BF16_TOL


def test_sign_muon_m8_step_bit_exact_vote():
    c = CONFIGS["sign_muon_m8"]
    inp = sign_muon_inputs()
    n = 2048
    Ms = [torch.zeros(n, n, dtype=torch.bfloat16, device=dev()) for _ in range(8)]
    Gs = [torch.from_numpy(g).to(dev()) for g in inp["G"]]
    dummyW = [torch.zeros(1, dtype=torch.float32, device=dev()) for _ in range(8)]
    U = [torch.zeros(n, n, dtype=torch.bfloat16, device=dev()) for _ in range(8)]
    mats = [mo.make_matrix(M, M, G) for M, G in zip(Ms, Gs)]      # W unused without update
    cfg = mo.make_cfg(mu=c["mu"], lr=c["lr"], apply_update=False, out_dtype=mo.MO_BF16)
    ws = workspace(mo.mo_workspace_bytes(mats, cfg))
    mo.muon_step_batched(mats, cfg, ws, out=U)
    words = [torch.empty((n * n + 31) // 32, dtype=torch.int32, device=dev()) for _ in range(8)]
    for u, w in zip(U, words):
        mo.sign_pack(u, w)
    W = torch.from_numpy(inp["W"]).to(dev())
    W0 = inp["W"].astype(np.float64)
    mo.sign_vote_update(words, W, c["lr"])
    torch.cuda.synchronize()
    del dummyW
    # NS outputs vs the oracle (momentum stored in bf16)
    for m in (0, 5):
        _, Mst, O = om.muon_step(np.zeros((n, n)), np.zeros((n, n)), inp["G"][m], mu=c["mu"], lr=c["lr"],
                                 m_dtype="bf16", apply_update=False)
        assert rel_fro(to_np(Ms[m]), Mst) < 1e-7
        assert rel_fro(to_np(U[m]), O) < NS_BF16_TOL
    # pack and vote: bit-exact on the GPU's own sign buffers
    ref_words = [osg.pack_bits(to_np(u)) for u in U]
    for w, r in zip(words, ref_words):
        assert np.array_equal(w.cpu().numpy().view(np.uint32), r)
    assert np.array_equal(to_np(W), osg.vote_update(W0, ref_words, c["lr"]))


@pytest.mark.parametrize("shapes", [[(256, 512), (512, 256)], [(96, 160), (160, 96), (2048, 2048)],
                                    [(200, 64), (64, 224), (320, 320)]])
def test_sign_packed_step_equals_separate_pack(shapes):
    """Fused sign + pack in the last NS epilogue: bit for bit the oracle's
    packing (sign(0) = +1, bit j % 32 of word j / 32) of the bf16 direction
    that the unfused step writes, that direction within the NS bound of the
    oracle's, and equal to sign_pack of it."""
    rng = np.random.default_rng(len(shapes))
    G = [rng.standard_normal(s).astype(np.float32) for s in shapes]
    cfg_out = mo.make_cfg(mu=0.95, apply_update=False, out_dtype=mo.MO_BF16)

    def fresh():
        Ms = [torch.zeros(s, dtype=torch.bfloat16, device=dev()) for s in shapes]
        Gs = [torch.from_numpy(g).to(dev()) for g in G]
        return Ms, Gs, [mo.make_matrix(m, m, g) for m, g in zip(Ms, Gs)]

    Ms, Gs, mats = fresh()
    U = [torch.zeros(s, dtype=torch.bfloat16, device=dev()) for s in shapes]
    ws = workspace(mo.mo_workspace_bytes(mats, cfg_out))
    mo.muon_step_batched(mats, cfg_out, ws, out=U)
    ref = [torch.empty((s[0] * s[1] + 31) // 32, dtype=torch.int32, device=dev()) for s in shapes]
    for u, w in zip(U, ref):
        mo.sign_pack(u, w)
    Ms2, Gs2, mats2 = fresh()
    fused = [torch.full_like(w, -7) for w in ref]
    mo.muon_step_sign_packed(mats2, cfg_out, fused, ws)
    torch.cuda.synchronize()
    for a, b, s in zip(fused, ref, shapes):
        assert torch.equal(a, b), s
    for m1, m2 in zip(Ms, Ms2):
        assert torch.equal(m1, m2)                       # same momentum state update
    for a, u, g in zip(fused, U, G):
        assert np.array_equal(a.cpu().numpy().view(np.uint32), osg.pack_bits(to_np(u)))
        _, _, O = om.muon_step(np.zeros(g.shape), np.zeros(g.shape), g, mu=0.95, lr=0.02, m_dtype="bf16",
                               apply_update=False)
        assert rel_fro(to_np(u), O) < NS_BF16_TOL


def test_sign_packed_step_rejects_unaligned_columns():
    M = torch.zeros(64, 40, device=dev())
    G = torch.ones(64, 40, device=dev())
    words = [torch.empty(80, dtype=torch.int32, device=dev())]
    cfg = mo.make_cfg(apply_update=False)
    ws = workspace(mo.mo_workspace_bytes([mo.make_matrix(M, M, G)], cfg))
    with pytest.raises(mo.MoError) as e:
        mo.muon_step_sign_packed([mo.make_matrix(M, M, G)], cfg, words, ws)
    assert e.value.status == -6


@pytest.mark.parametrize("shapes", [[(256, 512)], [(512, 256), (768, 3072), (96, 200)]])
def test_spectral_scale_vs_oracle(shapes):
    rng = np.random.default_rng(31 + len(shapes))
    inputs = [{"W": (0.02 * rng.standard_normal(s)).astype(np.float32),
               "G": rng.standard_normal(s).astype(np.float32)} for s in shapes]
    cfg = mo.make_cfg(mu=0.95, lr=0.02, spectral_iters=8)
    Ws, _ = _run(inputs, cfg)
    for w, inp in zip(Ws, inputs):
        W0 = inp["W"].astype(np.float64)
        Wn, _, _ = om.muon_step(W0, np.zeros_like(W0), inp["G"], mu=0.95, lr=0.02, spectral_iters=8)
        Wf, _, _ = om.muon_step(W0, np.zeros_like(W0), inp["G"], mu=0.95, lr=0.02)
        d = to_np(w) - W0
        assert rel_fro(d, Wn - W0) < NS_BF16_SPECTRAL_TOL
        assert rel_fro(d, Wf - W0) > 5 * NS_BF16_SPECTRAL_TOL  # the spectral path is really taken


@pytest.mark.slow
def test_llama7b_owner0_sampled():
    c = CONFIGS["llama7b_owner0"]
    shapes = llama7b_shapes()
    owner, _ = oplan.plan_owners(shapes, 8, 5)
    mine = [i for i in range(len(shapes)) if owner[i] == 0]
    assert len(mine) == 28
    inputs = matrix_set_inputs(shapes, mine)
    cfg = mo.make_cfg(mu=c["mu"], lr=c["lr"])
    Ws, Ms = _run(inputs, cfg)
    # elementwise against the oracle: the first and the last matrix of each
    # shape class (4096 x 4096; 4096 x 11008 as is; 11008 x 4096 transposed)
    classes = [lambda s: s[0] == s[1], lambda s: s[0] < s[1], lambda s: s[0] > s[1]]
    for cls in classes:
        ks = [k for k, i in enumerate(mine) if cls(shapes[i])]
        for k in (ks[0], ks[-1]):
            _check_update(Ws[k], inputs[k], c["mu"], c["lr"], NS_BF16_TOL)
    # every matrix: the update is finite and its Frobenius norm lies in the
    # NS band: ||O||_F^2 = sum sigma_i^2 with each sigma in [0.68, 1.21]
    for k, i in enumerate(mine):
        d = (to_np(Ws[k]) - inputs[k]["W"]) / c["lr"]
        m = min(shapes[i])
        f2 = float(np.sum(d * d)) / m
        assert np.isfinite(f2) and 0.68 ** 2 * 0.95 < f2 < 1.21 ** 2 * 1.05
        assert rel_fro(to_np(Ms[k]), inputs[k]["G"]) < MOM_TOL


@pytest.mark.slow
def test_ns_8192_square_vs_oracle():
    """The largest matrix the workloads draw, alone: 8192 x 8192 (128 K-blocks
    in every phase, 64 x 32 apply tiles), elementwise against the oracle."""
    X = np.random.default_rng(81).standard_normal((8192, 8192), dtype=np.float32)
    Xt = torch.from_numpy(X).to(dev())
    out = torch.zeros_like(Xt)
    ws = workspace(mo.ns_workspace_bytes([(8192, 8192)]))
    mo.ns_orthogonalize([Xt], [out], 5, ws)
    torch.cuda.synchronize()
    assert mo.mo_check_device_status(ws) == 0
    assert rel_fro(to_np(out), om.newton_schulz(X.astype(np.float64))) < NS_BF16_TOL


@pytest.mark.slow
def test_ragged500_sampled():
    c = CONFIGS["ragged500"]
    shapes = ragged_shapes()
    inputs = matrix_set_inputs(shapes)
    cfg = mo.make_cfg(mu=c["mu"], lr=c["lr"])
    Ws, _ = _run(inputs, cfg)
    sizes = [r * cc for r, cc in shapes]
    # the smallest matrix, the one with the largest m (about 8000: 125 Gram
    # K-blocks of 64 and 63 apply row tiles), the largest, and three more
    picks = {int(np.argmin(sizes)), int(np.argmax([min(s) for s in shapes])), int(np.argmax(sizes)), 17, 250, 499}
    assert max(min(shapes[k]) for k in picks) > 4096
    for k in sorted(picks):
        _check_update(Ws[k], inputs[k], c["mu"], c["lr"], NS_BF16_TOL)
    for k in range(len(shapes)):
        d = (to_np(Ws[k]) - inputs[k]["W"]) / c["lr"]
        assert np.all(np.isfinite(d))

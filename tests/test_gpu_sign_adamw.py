"""GPU parity: sign_pack and sign_vote_update (bit-exact) and the AdamW tail,
through the C ABI, against the oracle on seeded inputs."""
import numpy as np
import pytest
import torch

import matrix_optimizers_gb300 as mo
from oracle import adamw as oa
from oracle import sign as osg
from tests.gpu_helpers import dev, to_dev, to_np

pytestmark = pytest.mark.gpu


def _words_np(t):
    return t.cpu().numpy().view(np.uint32)


def _signed_input(shape, seed):
    rng = np.random.default_rng(seed)
    U = rng.standard_normal(shape).astype(np.float32)
    flat = U.reshape(-1)
    flat[::7] = 0.0
    flat[3::11] = -0.0
    flat[5::13] = np.nan
    flat[1::17] = -1e-30
    return U


@pytest.mark.parametrize("shape,ld", [((1, 1), None), ((3, 7), 8), ((5, 33), 40), ((64, 64), None),
                                      ((100, 257), 264), ((1, 4097), None), ((513, 1), 8),
                                      ((3, 8), None), ((5, 40), 48), ((77, 1000), 1024), ((1, 8), None),
                                      ((2048, 2048), None)])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_sign_pack_bit_exact(shape, ld, dtype):
    U = _signed_input(shape, sum(shape))
    Ut = to_dev(U, dtype, ld)
    nw = (U.size + 31) // 32
    words = torch.full((nw + 4,), -1, dtype=torch.int32, device=dev())    # canary after the end
    mo.sign_pack(Ut, words[:nw])
    torch.cuda.synchronize()
    stored = to_np(Ut)        # the values the kernel saw (bf16-rounded for bf16)
    want = osg.pack_bits(stored)
    got = _words_np(words)
    assert np.array_equal(got[:nw], want)
    assert np.all(got[nw:] == 0xFFFFFFFF)


@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 7, 8, 13, 64, 128])
@pytest.mark.parametrize("shape,ld", [((1, 5), 8), ((33, 95), 96), ((64, 64), None), ((7, 12), 16),
                                      ((31, 100), 104), ((2048, 2048), None)])
@pytest.mark.parametrize("wdtype", [torch.float32, torch.bfloat16])
def test_vote_update_bit_exact(M, shape, ld, wdtype):
    if M > 13 and shape[0] * shape[1] > 100_000:
        pytest.skip("large voter counts are covered on the smaller shapes")
    rng = np.random.default_rng(M * 1000 + shape[0])
    numel = shape[0] * shape[1]
    nw = (numel + 31) // 32
    bufs = [rng.integers(0, 2 ** 32, size=nw, dtype=np.uint64).astype(np.uint32) for _ in range(M)]
    # tail bits beyond numel are zero in a packed buffer
    if numel % 32:
        for b in bufs:
            b[-1] &= np.uint32((1 << (numel % 32)) - 1)
    words = [torch.from_numpy(b.view(np.int32).copy()).to(dev()) for b in bufs]
    W = (0.02 * rng.standard_normal(shape)).astype(np.float32)
    Wt = to_dev(W, wdtype, ld)
    W_stored = to_np(Wt)
    lr = 1e-3
    mo.sign_vote_update(words, Wt, lr)
    torch.cuda.synchronize()
    want = osg.vote_update(W_stored, bufs, lr, "bf16" if wdtype == torch.bfloat16 else "f32")
    got = to_np(Wt)
    assert np.array_equal(got, want)
    if ld is not None:   # padding columns (NaN-filled) are left untouched
        full = Wt.as_strided((shape[0], ld), (ld, 1))
        assert torch.isnan(full[:, shape[1]:].float()).all()


@pytest.mark.parametrize("M", [1, 2, 8, 16, 17])
@pytest.mark.parametrize("shape", [(64, 64), (64, 192), (64, 128), (256, 512), (2048, 2048)])
@pytest.mark.parametrize("wdtype", [torch.float32, torch.bfloat16])
def test_vote_update_chunked_path_bit_exact(M, shape, wdtype):
    """Contiguous W with whole 4096-element chunks (one, an odd three, ...) and
    up to 16 workers takes the shared-memory streaming path (17 workers fall
    back); bit-exact both ways."""
    rng = np.random.default_rng(7 * M + shape[1])
    numel = shape[0] * shape[1]
    bufs = [rng.integers(0, 2 ** 32, size=numel // 32, dtype=np.uint64).astype(np.uint32) for _ in range(M)]
    words = [torch.from_numpy(b.view(np.int32).copy()).to(dev()) for b in bufs]
    W = (0.02 * rng.standard_normal(shape)).astype(np.float32)
    Wt = to_dev(W, wdtype)
    W_stored = to_np(Wt)
    mo.sign_vote_update(words, Wt, 1e-3)
    torch.cuda.synchronize()
    want = osg.vote_update(W_stored, bufs, 1e-3, "bf16" if wdtype == torch.bfloat16 else "f32")
    assert np.array_equal(to_np(Wt), want)


@pytest.mark.parametrize("wdtype", [torch.float32, torch.bfloat16])
def test_vote_update_chunked_path_ring_wraps(wdtype):
    """4096^2 with 8 workers: 4096 chunks of 4096 elements over one resident
    wave of blocks, so every block reuses both stages of its ring several
    times; bit-exact."""
    rng = np.random.default_rng(41)
    shape = (4096, 4096)
    numel = shape[0] * shape[1]
    bufs = [rng.integers(0, 2 ** 32, size=numel // 32, dtype=np.uint64).astype(np.uint32) for _ in range(8)]
    words = [torch.from_numpy(b.view(np.int32).copy()).to(dev()) for b in bufs]
    Wt = to_dev((0.02 * rng.standard_normal(shape)).astype(np.float32), wdtype)
    W_stored = to_np(Wt)
    mo.sign_vote_update(words, Wt, 1e-3)
    torch.cuda.synchronize()
    want = osg.vote_update(W_stored, bufs, 1e-3, "bf16" if wdtype == torch.bfloat16 else "f32")
    assert np.array_equal(to_np(Wt), want)


def test_vote_ties_go_plus():
    # M = 2 with opposite signs everywhere: every vote is a tie -> +1
    numel = 64 * 64
    a = np.full((numel + 31) // 32, 0xFFFFFFFF, dtype=np.uint32)
    b = np.zeros_like(a)
    words = [torch.from_numpy(x.view(np.int32).copy()).to(dev()) for x in (a, b)]
    W = torch.zeros(64, 64, device=dev())
    mo.sign_vote_update(words, W, 0.5)
    torch.cuda.synchronize()
    assert torch.all(W == -0.5)


@pytest.mark.parametrize("numel", [1, 3, 1001, 36_864, 4_000_003])
@pytest.mark.parametrize("wd", [0.0, 0.1])
def test_adamw_tail_matches_oracle(numel, wd):
    rng = np.random.default_rng(numel)
    W = (0.02 * rng.standard_normal(numel)).astype(np.float32)
    m = np.zeros(numel)
    v = np.zeros(numel)
    tW, tm_, tv = (torch.from_numpy(x.astype(np.float32)).to(dev()) for x in (W, m, v))
    Wr, mr, vr = W.astype(np.float64), m, v
    for t in range(1, 4):
        g = (1e-3 * rng.standard_normal(numel)).astype(np.float32)
        tg = torch.from_numpy(g).to(dev())
        tail = mo.make_tail(tW, tg, tm_, tv, step=t, lr=1e-3, weight_decay=wd)
        cfg = mo.make_cfg()
        mo.muon_step_batched([], cfg, None, tail=tail)
        Wr, mr, vr = oa.adamw_step(Wr, g, mr, vr, t, lr=1e-3, weight_decay=wd)
    torch.cuda.synchronize()
    gotW = tW.cpu().numpy().astype(np.float64)
    # float32 state: |dW| error ~ float32 rounding of W plus ~1e-6 relative of each update
    assert np.max(np.abs(gotW - Wr)) <= 1e-5 * 1e-3 * 3 + 4 * np.max(np.abs(Wr)) * 2 ** -23
    # m is a signed running sum: elements near zero carry the float32 rounding of
    # terms of size ~|g|, so the bound is relative to the terms, not to m itself
    gm, gv = tm_.cpu().numpy().astype(np.float64), tv.cpu().numpy().astype(np.float64)
    assert np.max(np.abs(gm - mr)) <= 16 * 2 ** -24 * np.max(np.abs(mr))
    assert np.max(np.abs(gv - vr) / vr.clip(min=1e-300)) <= 16 * 2 ** -24


@pytest.mark.parametrize("shape,ld", [((1, 1), None), ((3, 7), 8), ((5, 40), 48), ((64, 64), None),
                                      ((33, 95), 96), ((2048, 2048), None)])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_sign_int8_bit_exact(shape, ld, dtype):
    U = _signed_input(shape, sum(shape) + 3)
    Ut = to_dev(U, dtype, ld)
    numel = U.size
    out = torch.full((numel + 16,), 7, dtype=torch.int8, device=dev())      # canary tail
    mo.sign_int8(Ut, out[:numel])
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    assert np.array_equal(got[:numel], osg.sign_int8(to_np(Ut)))
    assert np.all(got[numel:] == 7)


@pytest.mark.parametrize("M", [1, 2, 3, 8, 13, 127])
@pytest.mark.parametrize("shape,ld", [((1, 5), 8), ((33, 95), 96), ((64, 64), None), ((7, 32), 36),
                                      ((2048, 2048), None)])
@pytest.mark.parametrize("wdtype", [torch.float32, torch.bfloat16])
def test_int8_vote_update_bit_exact(M, shape, ld, wdtype):
    if M > 13 and shape[0] * shape[1] > 100_000:
        pytest.skip("large voter counts are covered on the smaller shapes")
    rng = np.random.default_rng(M * 7 + shape[1])
    numel = shape[0] * shape[1]
    signs = [np.where(rng.random(numel) < 0.5, -1, 1).astype(np.int8) for _ in range(M)]
    sig_t = [torch.from_numpy(s).to(dev()) for s in signs]
    W = (0.02 * rng.standard_normal(shape)).astype(np.float32)
    Wt = to_dev(W, wdtype, ld)
    W_stored = to_np(Wt)
    mo.sign_vote_update_int8(sig_t, Wt, 1e-3)
    torch.cuda.synchronize()
    want = osg.int8_vote_update(W_stored, signs, 1e-3, "bf16" if wdtype == torch.bfloat16 else "f32")
    assert np.array_equal(to_np(Wt), want)


def test_int8_and_packed_votes_agree_on_gpu():
    rng = np.random.default_rng(42)
    U = [rng.standard_normal((256, 512)).astype(np.float32) for _ in range(6)]
    Ut = [torch.from_numpy(u).to(dev()) for u in U]
    words = [torch.empty(256 * 512 // 32, dtype=torch.int32, device=dev()) for _ in U]
    signs = [torch.empty(256 * 512, dtype=torch.int8, device=dev()) for _ in U]
    for u, w, s in zip(Ut, words, signs):
        mo.sign_pack(u, w)
        mo.sign_int8(u, s)
    W1 = torch.zeros(256, 512, device=dev())
    W2 = torch.zeros(256, 512, device=dev())
    mo.sign_vote_update(words, W1, 0.25)
    mo.sign_vote_update_int8(signs, W2, 0.25)
    torch.cuda.synchronize()
    assert torch.equal(W1, W2)


@pytest.mark.parametrize("shape,ld", [((64, 64), None), ((5, 40), 48), ((33, 95), 96), ((2048, 2048), None),
                                      ((64, 128), None), ((64, 192), None), ((256, 512), None)])
@pytest.mark.parametrize("M", [1, 3, 8])
def test_sign_pack_batched_bit_exact(shape, ld, M):
    Us = [_signed_input(shape, 100 + m) for m in range(M)]
    Ut = [to_dev(u, torch.bfloat16, ld) for u in Us]
    nw = (Us[0].size + 31) // 32
    words = [torch.full((nw + 4,), -1, dtype=torch.int32, device=dev()) for _ in range(M)]
    mo.sign_pack_batched(Ut, [w[:nw] for w in words])
    torch.cuda.synchronize()
    for u, w in zip(Ut, words):
        got = _words_np(w)
        assert np.array_equal(got[:nw], osg.pack_bits(to_np(u)))
        assert np.all(got[nw:] == 0xFFFFFFFF)


@pytest.mark.parametrize("shape,ld", [((256, 512), None), ((512, 256), None), ((200, 300), 304),
                                      ((2048, 2048), None)])
@pytest.mark.parametrize("M", [3, 8])
def test_vote_polar_update_vs_oracle(shape, ld, M):
    """The local polar step on the vote: W - lr * NS(S_bar) within the bf16 NS tolerance."""
    from tests.gpu_helpers import NS_BF16_TOL, rel_fro, workspace
    rng = np.random.default_rng(M + shape[0])
    numel = shape[0] * shape[1]
    bufs = [osg.pack_bits(rng.standard_normal(shape)) for _ in range(M)]
    words = [torch.from_numpy(b.view(np.int32).copy()).to(dev()) for b in bufs]
    W = (0.02 * rng.standard_normal(shape)).astype(np.float32)
    Wt = to_dev(W, torch.float32, ld)
    W0 = to_np(Wt)
    ws = workspace(mo.sign_vote_polar_workspace_bytes(Wt))
    mo.sign_vote_polar_update(words, Wt, 1e-2, ws)
    torch.cuda.synchronize()
    want = osg.vote_polar_update(W0, bufs, 1e-2)
    assert rel_fro(to_np(Wt) - W0, want - W0) < NS_BF16_TOL
    assert numel == W.size

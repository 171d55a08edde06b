"""Pins of the oracle's sign / pack / vote, AdamW, planner and bf16 rounding."""
import itertools

import numpy as np
import pytest
import torch

from oracle import adamw as oa
from oracle import bf16 as ob
from oracle import planner as op
from oracle import sign as osg
from workloads import llama7b_shapes


# ---------------------------------------------------------------- bf16 ------
def _torch_bf16(x32):
    return torch.from_numpy(np.asarray(x32, dtype=np.float32)).to(torch.bfloat16) \
        .to(torch.float64).numpy()


def test_bf16_matches_torch_cast_on_float32_inputs():
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.standard_normal(100_000).astype(np.float32),
        (rng.standard_normal(10_000) * 1e-38).astype(np.float32),   # subnormal range
        (rng.standard_normal(10_000) * 1e30).astype(np.float32),
        np.array([0.0, -0.0, 1.0, -1.0, 3.0e38, -3.39e38], dtype=np.float32),
    ])
    got = ob.round_bf16(x.astype(np.float64))
    want = _torch_bf16(x)
    assert np.array_equal(got, want)
    assert np.array_equal(np.signbit(got), np.signbit(want))


def test_bf16_ties_to_even():
    one = 1.0
    assert ob.round_bf16(one + 2.0 ** -8) == 1.0                   # tie -> even (1.0)
    assert ob.round_bf16(one + 3 * 2.0 ** -8) == one + 2.0 ** -6   # tie -> even (up)
    assert ob.round_bf16(one + 2.0 ** -8 + 2.0 ** -30) == one + 2.0 ** -7
    assert ob.round_bf16(2.0 ** 128 * (1 - 2.0 ** -9)) == np.inf
    assert ob.round_bf16(-(2.0 ** 127) * (2 - 2.0 ** -7)) == -(2.0 ** 127) * (2 - 2.0 ** -7)


# ---------------------------------------------------------------- sign ------
@pytest.mark.parametrize("shape", [(1, 1), (3, 7), (4, 8), (5, 33), (64, 64), (7, 100)])
def test_pack_numpy_equals_python_loop(shape):
    rng = np.random.default_rng(sum(shape))
    U = rng.standard_normal(shape)
    U.reshape(-1)[:: 5] = 0.0
    U.reshape(-1)[1:: 7] = -0.0
    U.reshape(-1)[2:: 11] = np.nan
    w1, w2 = osg.pack_bits(U), osg.pack_bits_loop(U)
    assert w1.dtype == np.uint32 and np.array_equal(w1, w2)
    assert w1.size == (U.size + 31) // 32
    # unused bits of the last word are zero
    tail = U.size % 32
    if tail:
        assert int(w1[-1]) >> tail == 0


def test_sign_tie_rule():
    U = np.array([[-1.0, 0.0, -0.0, np.nan, 2.0, -1e-30]])
    assert np.array_equal(osg.sign(U), np.array([[-1, 1, 1, 1, 1, -1.0]]))
    assert osg.pack_bits(U)[0] == 0b011110


@pytest.mark.parametrize("M", range(1, 9))
def test_majority_vote_brute_force_all_patterns(M):
    # element e carries the sign pattern given by the bits of e: every one of
    # the 2^M patterns appears once
    numel = 2 ** M
    pats = list(itertools.product([-1.0, 1.0], repeat=M))
    S = np.array(pats)                  # numel x M
    bufs = [osg.pack_bits(S[:, m]) for m in range(M)]
    vote = osg.majority_vote(bufs, numel)
    for e, pat in enumerate(pats):
        total = sum(pat)
        want = 1.0 if total >= 0 else -1.0      # sign(sum) with sign(0) = +1
        assert vote[e] == want


@pytest.mark.parametrize("M", range(1, 9))
def test_int8_sum_vote_brute_force_all_patterns(M):
    pats = list(itertools.product([-1.0, 1.0], repeat=M))
    S = np.array(pats)
    signs = [osg.sign_int8(S[:, m]) for m in range(M)]
    assert all(s.dtype == np.int8 and set(np.unique(s)) <= {-1, 1} for s in signs)
    vote = osg.int8_vote(signs)
    for e, pat in enumerate(pats):
        assert vote[e] == (1.0 if sum(pat) >= 0 else -1.0)
    # both payloads (1-bit all-gather, int8 all-reduce) give the same vote
    bufs = [osg.pack_bits(S[:, m]) for m in range(M)]
    assert np.array_equal(vote, osg.majority_vote(bufs, len(pats)))


def test_vote_polar_update_composes_vote_and_closed_form_ns():
    rng = np.random.default_rng(21)
    shape = (12, 20)
    bufs = [osg.pack_bits(rng.standard_normal(shape)) for _ in range(5)]
    W = rng.standard_normal(shape)
    got = osg.vote_polar_update(W, bufs, 0.1)
    S = osg.majority_vote(bufs, W.size).reshape(shape)
    U, s, Vt = np.linalg.svd(S / np.linalg.norm(S), full_matrices=False)
    for _ in range(5):
        s = 3.4445 * s - 4.7750 * s ** 3 + 2.0315 * s ** 5
    np.testing.assert_allclose(got, W - 0.1 * (U * s) @ Vt, atol=1e-12)
    # ||S_bar||_F = sqrt(numel): every entry is +-1
    assert np.linalg.norm(S) == np.sqrt(S.size)


def test_int8_sign_tie_rule():
    U = np.array([[-1.0, 0.0, -0.0, np.nan, 2.0, -1e-30]])
    assert np.array_equal(osg.sign_int8(U), np.array([-1, 1, 1, 1, 1, -1], dtype=np.int8))


def test_vote_update_single_float32_rounding():
    rng = np.random.default_rng(3)
    W = rng.standard_normal((9, 13)).astype(np.float32)
    bufs = [osg.pack_bits(rng.standard_normal((9, 13))) for _ in range(5)]
    lr = 1e-3
    got = osg.vote_update(W, bufs, lr)
    vote = osg.majority_vote(bufs, W.size).reshape(W.shape)
    # float32 operands subtract exactly in float64; one rounding to float32
    want = (W.astype(np.float64) - np.float64(np.float32(lr)) * vote).astype(np.float32)
    assert np.array_equal(got, want.astype(np.float64))
    gotb = osg.vote_update(ob.round_bf16(W), bufs, lr, "bf16")
    assert np.array_equal(gotb, _torch_bf16(
        (ob.round_bf16(W) - np.float64(np.float32(lr)) * vote).astype(np.float32)))


# ---------------------------------------------------------------- AdamW -----
def test_adamw_first_step_closed_form():
    rng = np.random.default_rng(4)
    W, g = rng.standard_normal(1000), rng.standard_normal(1000) * 1e-3
    Wn, m, v = oa.adamw_step(W, g, np.zeros(1000), np.zeros(1000), 1, lr=1e-3)
    np.testing.assert_allclose(Wn, W - 1e-3 * g / (np.abs(g) + 1e-8), rtol=0, atol=1e-15)
    np.testing.assert_allclose(m, 0.1 * g, atol=1e-18)
    np.testing.assert_allclose(v, 0.05 * g * g, atol=1e-22)


def test_adamw_matches_torch_optim():
    rng = np.random.default_rng(5)
    W0 = rng.standard_normal(257)
    p = torch.nn.Parameter(torch.from_numpy(W0.copy()))
    opt = torch.optim.AdamW([p], lr=3e-3, betas=(0.9, 0.95), eps=1e-8, weight_decay=0.05)
    W, m, v = W0.copy(), np.zeros(257), np.zeros(257)
    for t in range(1, 5):
        g = rng.standard_normal(257) * 1e-2
        p.grad = torch.from_numpy(g.copy())
        opt.step()
        W, m, v = oa.adamw_step(W, g, m, v, t, lr=3e-3, weight_decay=0.05)
    np.testing.assert_allclose(W, p.detach().numpy(), rtol=0, atol=1e-14)


# ---------------------------------------------------------------- planner ---
def test_plan_7b_deals_each_shape_class_round_robin():
    shapes = llama7b_shapes()
    owner, load = op.plan_owners(shapes, 8, 5)
    square = [i for i, s in enumerate(shapes) if s[0] == s[1]]
    big = [i for i, s in enumerate(shapes) if s[0] != s[1]]
    # every big matrix has one and the same cost, above every square one, so
    # LPT deals the bigs first, in index order, to ranks 0..7 in turn, then
    # the squares the same way
    for j, i in enumerate(big):
        assert owner[i] == j % 8
    for j, i in enumerate(square):
        assert owner[i] == j % 8
    assert len(set(load)) == 1
    mine = [i for i in range(len(shapes)) if owner[i] == 0]
    assert len(mine) == 28
    assert sum(1 for i in mine if shapes[i][0] == shapes[i][1]) == 16


def test_plan_hand_example():
    owner, load = op.plan_owners([(8, 8), (8, 8), (16, 16)], 2, 5)
    # costs 4/15, 4/15, 22/15: the big one to rank 0, the two small ones to rank 1
    assert owner == [1, 1, 0]
    assert abs(load[0] - 22 / 15) < 1e-15 and abs(load[1] - 8 / 15) < 1e-15


def test_plan_lpt_within_graham_bound_of_brute_force():
    rng = np.random.default_rng(6)
    for trial in range(20):
        n, world = int(rng.integers(2, 9)), int(rng.integers(2, 4))
        shapes = [(int(rng.integers(1, 40)) * 8, int(rng.integers(1, 40)) * 8) for _ in range(n)]
        cost = op.costs(shapes, 5)
        _, load = op.plan_owners(shapes, world, 5)
        best = min(max(sum(cost[i] for i in range(n) if a[i] == r) for r in range(world))
                   for a in itertools.product(range(world), repeat=n))
        assert max(load) <= (4 / 3 - 1 / (3 * world)) * best + 1e-12
        assert abs(sum(load) - sum(cost)) < 1e-12


def test_plan_rejects_empty_world():
    with pytest.raises(ValueError):
        op.plan_owners([(8, 8)], 0, 5)

"""Host-side checks of the C ABI (no GPU): the library loads, exports every
symbol the headers declare, validates arguments, and its owner planner equals
the oracle's bit for bit."""
import ctypes
import os
import re

import numpy as np
import pytest

from matrix_optimizers_gb300 import _binding as B
from oracle import planner as oplan
from workloads import gpt_small_shapes, llama7b_shapes, ragged_shapes

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_symbols():
    names = set()
    for h in ("matrixopt.h", "matrixopt_debug.h"):
        src = open(os.path.join(ROOT, "include", h)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(\w+)\s*\(", src, flags=re.M):
            names.add(m.group(1))
    return names


def test_library_exports_every_declared_symbol(lib):
    declared = _declared_symbols()
    assert {"muon_step_batched", "ns_orthogonalize", "sign_pack", "sign_vote_update",
            "plan_owners", "mo_workspace_bytes", "mo_check_device_status"} <= declared
    for name in declared:
        assert hasattr(lib, name), name
    bound = {n for n, _, _ in B._SIGNATURES}
    assert declared == bound


def test_struct_sizes_match_header():
    assert ctypes.sizeof(B.mo_matrix) == 64
    assert ctypes.sizeof(B.mo_muon_cfg) == 48
    assert ctypes.sizeof(B.mo_adamw_tail) == 72
    assert ctypes.sizeof(B.mo_ns_view) == 104


def test_status_strings(lib):
    for code in range(-6, 1):
        assert lib.mo_status_string(code).startswith(b"MO_")
    assert lib.mo_version() == 0x000100


@pytest.mark.parametrize("shapes,world", [
    (llama7b_shapes(), 8), (gpt_small_shapes(), 3), (ragged_shapes(), 8), (ragged_shapes(), 5),
    ([(8, 8), (8, 8), (16, 16)], 2), ([(3, 5)], 4), ([], 2)])
def test_plan_owners_bit_exact_vs_oracle(shapes, world):
    got, gload = B.plan_owners(shapes, world, 5)
    want, wload = oplan.plan_owners(shapes, world, 5)
    assert got == want
    assert np.array_equal(np.array(gload), np.array(wload))   # bitwise-equal doubles


def test_plan_owners_weights_and_golden():
    shapes = ragged_shapes()[:40]
    for wb, wf in [(1.0, 0.0), (0.0, 1.0), (0.3, 1.7)]:
        assert B.plan_owners(shapes, 6, 5, wb, wf)[0] == oplan.plan_owners(shapes, 6, 5, wb, wf)[0]
    golden = open(os.path.join(ROOT, "tests", "golden", "plan_llama7b_world8.txt")).read().split("\n")[1]
    assert B.plan_owners(llama7b_shapes(), 8, 5)[0] == [int(x) for x in golden.split()]


def test_plan_owners_rejects_bad_args(lib):
    with pytest.raises(B.MoError) as e:
        B.plan_owners([(4, 4)], 0)
    assert e.value.status == B.MO_ERR_INVALID_ARG
    rows = (ctypes.c_int64 * 1)(-1)
    cols = (ctypes.c_int64 * 1)(4)
    owner = (ctypes.c_int32 * 1)()
    assert lib.plan_owners(rows, cols, 1, 2, 5, 1.0, 1.0, owner, None) == B.MO_ERR_INVALID_ARG
    assert lib.plan_owners(None, None, 0, 2, 5, 1.0, 1.0, None, None) == B.MO_OK


def test_workspace_bytes_host_only():
    mats = [B.mo_matrix(768, 3072, 3072, 0, 0, 0, 0, 16, 16, 16),
            B.mo_matrix(3072, 768, 768, 0, 0, 0, 0, 16, 16, 16)]
    cfg = B.make_cfg()
    ws = B.mo_workspace_bytes(mats, cfg)
    # both orient to 768 x 3072: operands 2 x bf16 X + 2 x 768^2 bf16 each
    per = 768 * 3072 * (2 + 2) + 2 * 768 * 768 * 2
    assert 2 * per <= ws < 2 * per + (1 << 20)
    assert ws == B.ns_workspace_bytes([(768, 3072), (3072, 768)])
    cfg32 = B.make_cfg(precision=B.MO_NS_FP32)
    assert B.mo_workspace_bytes(mats, cfg32) >= 2 * (768 * 3072 * 8 + 2 * 768 * 768 * 4)


def test_validation_errors_without_device(lib):
    cfg = B.make_cfg()
    good = B.mo_matrix(64, 64, 64, 0, 0, 0, 0, 256, 256, 256)
    bad_ld = B.mo_matrix(64, 64, 32, 0, 0, 0, 0, 256, 256, 256)
    bad_al = B.mo_matrix(64, 64, 64, 0, 0, 0, 0, 260, 256, 256)
    bad_ld_al = B.mo_matrix(64, 60, 62, 0, 0, 0, 0, 256, 256, 256)
    bad_dt = B.mo_matrix(64, 64, 64, 7, 0, 0, 0, 256, 256, 256)
    big = B.mo_matrix(40000, 40000, 40000, 0, 0, 0, 0, 256, 256, 256)

    def step(m, ws=1 << 20, wsb=1 << 40, c=cfg):
        arr = (B.mo_matrix * 1)(m)
        return lib.muon_step_batched(arr, 1, ctypes.byref(c), None, None, ctypes.c_void_p(ws), wsb, None)

    assert step(bad_ld) == B.MO_ERR_INVALID_ARG
    assert step(bad_al) == B.MO_ERR_ALIGNMENT
    assert step(bad_ld_al) == B.MO_ERR_ALIGNMENT
    assert step(bad_dt) == B.MO_ERR_INVALID_ARG
    assert step(big) == B.MO_ERR_UNSUPPORTED
    assert step(good, ws=0) == B.MO_ERR_WORKSPACE
    assert step(good, ws=(1 << 20) + 64) == B.MO_ERR_WORKSPACE
    assert step(good, wsb=1024) == B.MO_ERR_WORKSPACE
    neg = B.make_cfg(ns_steps=-1)
    assert step(good, c=neg) == B.MO_ERR_INVALID_ARG
    badp = B.make_cfg(precision=3)
    assert step(good, c=badp) == B.MO_ERR_INVALID_ARG
    noout = B.make_cfg(apply_update=False)
    assert step(good, c=noout) == B.MO_ERR_INVALID_ARG
    # zero-size matrices and n = 0 are no-ops
    empty = B.mo_matrix(0, 64, 64, 0, 0, 0, 0, 0, 0, 0)
    assert step(empty, ws=0, wsb=0) == B.MO_OK
    assert lib.muon_step_batched(None, 0, ctypes.byref(cfg), None, None, None, 0, None) == B.MO_OK
    # tail validation
    tail = B.mo_adamw_tail(10, 256, 256, 256, 256, 1e-3, 0.9, 0.95, 1e-8, 0.0, 0, 0)
    assert lib.muon_step_batched(None, 0, ctypes.byref(cfg), ctypes.byref(tail), None, None, 0,
                                 None) == B.MO_ERR_INVALID_ARG
    tail.step = 1
    tail.g = 258
    assert lib.muon_step_batched(None, 0, ctypes.byref(cfg), ctypes.byref(tail), None, None, 0,
                                 None) == B.MO_ERR_ALIGNMENT


def test_sign_vote_step_validation_without_device(lib):
    cfg = B.make_cfg(apply_update=False)

    def call(mats, W=256, w_dtype=0, ld=64, words=(256, 512)):
        arr = (B.mo_matrix * len(mats))(*mats)
        wp = (ctypes.c_void_p * len(words))(*words)
        return lib.muon_step_sign_vote(arr, len(mats), ctypes.byref(cfg), wp, ctypes.c_void_p(W), w_dtype, ld,
                                       1e-3, ctypes.c_void_p(1 << 20), 1 << 40, None)

    a = B.mo_matrix(32, 64, 64, 0, 0, 0, 0, 256, 256, 256)
    b = B.mo_matrix(64, 32, 32, 0, 0, 0, 0, 256, 256, 256)          # another shape
    c = B.mo_matrix(32, 48, 48, 0, 0, 0, 0, 256, 256, 256)          # cols not a multiple of 32
    assert call([a, b]) == B.MO_ERR_INVALID_ARG
    assert call([c, c], ld=48) == B.MO_ERR_UNSUPPORTED
    assert call([a, a], W=0) == B.MO_ERR_INVALID_ARG
    assert call([a, a], ld=32) == B.MO_ERR_INVALID_ARG                # ld below cols
    assert call([a, a], W=258) == B.MO_ERR_ALIGNMENT                  # fp32 W on a 2-byte boundary
    assert call([a, a], words=(256, 0)) == B.MO_ERR_INVALID_ARG
    assert call([a, a], words=(256, 514)) == B.MO_ERR_ALIGNMENT
    fp32 = B.make_cfg(apply_update=False, precision=B.MO_NS_FP32)
    arr = (B.mo_matrix * 1)(a)
    wp = (ctypes.c_void_p * 1)(256)
    assert lib.muon_step_sign_vote(arr, 1, ctypes.byref(fp32), wp, ctypes.c_void_p(256), 0, 64, 1e-3,
                                   ctypes.c_void_p(1 << 20), 1 << 40, None) == B.MO_ERR_UNSUPPORTED
    empty = (B.mo_matrix * 1)(B.mo_matrix(0, 64, 64, 0, 0, 0, 0, 0, 0, 0))
    assert lib.muon_step_sign_vote(empty, 1, ctypes.byref(cfg), wp, None, 0, 64, 1e-3, None, 0, None) == B.MO_OK


def test_sign_call_validation_without_device(lib):
    assert lib.sign_pack(None, 0, 4, 4, 4, None, None) == B.MO_ERR_INVALID_ARG
    assert lib.sign_pack(ctypes.c_void_p(256), 5, 4, 4, 4, ctypes.c_void_p(256), None) == B.MO_ERR_INVALID_ARG
    assert lib.sign_pack(ctypes.c_void_p(258), 0, 4, 4, 4, ctypes.c_void_p(256), None) == B.MO_ERR_ALIGNMENT
    assert lib.sign_pack(ctypes.c_void_p(257), 1, 4, 4, 4, ctypes.c_void_p(256), None) == B.MO_ERR_ALIGNMENT
    assert lib.sign_pack(ctypes.c_void_p(256), 0, 4, 4, 4, ctypes.c_void_p(258), None) == B.MO_ERR_ALIGNMENT
    assert lib.sign_pack(ctypes.c_void_p(256), 0, 4, 4, 3, ctypes.c_void_p(256), None) == B.MO_ERR_INVALID_ARG
    assert lib.sign_pack(ctypes.c_void_p(256), 0, 0, 4, 4, ctypes.c_void_p(256), None) == B.MO_OK
    words = (ctypes.c_void_p * 2)(256, 512)
    assert lib.sign_vote_update(words, 0, 4, 4, ctypes.c_void_p(256), 0, 4, 1e-3, None) == B.MO_ERR_INVALID_ARG
    assert lib.sign_vote_update(words, 129, 4, 4, ctypes.c_void_p(256), 0, 4, 1e-3, None) == \
        B.MO_ERR_UNSUPPORTED
    bad = (ctypes.c_void_p * 2)(256, 0)
    assert lib.sign_vote_update(bad, 2, 4, 4, ctypes.c_void_p(256), 0, 4, 1e-3, None) == B.MO_ERR_INVALID_ARG
    assert lib.sign_vote_update(words, 2, 4, 4, ctypes.c_void_p(258), 0, 4, 1e-3, None) == B.MO_ERR_ALIGNMENT
    odd = (ctypes.c_void_p * 2)(256, 514)
    assert lib.sign_vote_update(odd, 2, 4, 4, ctypes.c_void_p(256), 0, 4, 1e-3, None) == B.MO_ERR_ALIGNMENT


def test_debug_view_offsets_are_disjoint():
    shapes = [(100, 300), (300, 100), (64, 64)]
    spans, res = [], []
    for i in range(3):
        v = B.mo_debug_ns_view(shapes, i)
        assert (v.m, v.n) == ((100, 300) if i < 2 else (64, 64))
        assert v.transposed == (1 if i == 1 else 0)
        assert v.ldx % 8 == 0 and v.ldx >= v.m and v.lda % 64 == 0     # bf16 operand: 8-column blocks
        xb = -(-v.n // 8) * v.ldx * 16
        spans += [(v.x_op[0], xb), (v.x_op[1], xb),
                  (v.gram, v.m * v.lda * 2), (v.poly, v.m * v.lda * 2)]
        res.append((v.diag_res, v.m * 4))
    spans.sort()
    for (a, la), (b, _) in zip(spans, spans[1:]):
        assert a + la <= b and a % 1024 == 0
    assert spans[-1][0] + spans[-1][1] <= B.ns_workspace_bytes(shapes)
    # the diagonal residual vectors: disjoint, ahead of the NS buffers
    res.sort()
    for (a, la), (b, _) in zip(res, res[1:]):
        assert a + la <= b and a % 128 == 0
    assert res[-1][0] + res[-1][1] <= spans[0][0]


def test_debug_view_dependency_counters():
    """Counter slots: one 16-byte slot per matrix, ahead of the NS buffers;
    tile counts equal a brute-force count of 128 x 256 tiles (upper-triangle
    tiles for the symmetric phases)."""
    shapes = [(100, 300), (300, 100), (64, 64), (1000, 2000)]
    views = [B.mo_debug_ns_view(shapes, i) for i in range(len(shapes))]
    deps = [v.deps for v in views]
    assert all(d % 16 == 0 for d in deps)
    assert sorted(deps) == deps and all(b - a == 16 for a, b in zip(deps, deps[1:]))
    assert max(deps) + 16 <= min(v.x_op[0] for v in views)
    for v in views:
        m, n = v.m, v.n
        sym = sum(1 for I in range(-(-m // 128)) for J in range(-(-m // 256))
                  if min(J * 256 + 255, m - 1) >= I * 128)
        assert v.tiles_sym == sym
        assert v.tiles_apply == -(-m // 128) * -(-n // 256)
    lib = B.load()
    assert lib.mo_debug_set_ns_fused(4) == B.MO_ERR_INVALID_ARG
    assert lib.mo_debug_set_ns_fused(-1) == B.MO_ERR_INVALID_ARG
    prev = B.mo_debug_set_ns_fused(0)
    assert B.mo_debug_set_ns_fused(2) == 0
    assert B.mo_debug_set_ns_fused(prev) == 2


def test_missing_library_raises_instead_of_falling_back(monkeypatch, tmp_path):
    # with no built library every entry point must fail loudly: there is no
    # CPU or PyTorch fallback behind the binding
    monkeypatch.setattr(B, "_lib", None)
    monkeypatch.setattr(B, "library_path", lambda: str(tmp_path / "libmatrixopt.so"))
    with pytest.raises(ImportError):
        B.load()
    with pytest.raises(ImportError):
        B.plan_owners([(64, 64), (128, 64)], 2, 5)

"""The fused Newton-Schulz launch's failure path, driven the allowed way: a
debug hook makes one matrix's dependency waits impossible to meet and shortens
their budget to about 1 ms.  The wait runs out, the launch unwinds (other CTAs
see the error word and stop at their next dependency wait; armed copies and
issued MMAs drain, TMEM is freed) and mo_check_device_status reports
MO_ERR_TIMEOUT well within a second.  The next call on the same workspace,
without the hook, matches the oracle."""
import time

import numpy as np
import pytest
import torch

import matrix_optimizers_gb300 as mo
from matrix_optimizers_gb300 import _binding as B
from oracle import muon as om
from tests.gpu_helpers import NS_BF16_TOL, dev, rel_fro, to_np, workspace

pytestmark = pytest.mark.gpu

CASES = [
    ([(512, 1024)], 0, 1),                        # the only matrix stalls at its first wait (per-matrix counters)
    ([(256, 512), (384, 768), (200, 96)], 1, 1),  # the others run on, then stop on the error word
    ([(256, 512), (384, 768), (200, 96)], 2, 2),  # grid-wide counters
]


@pytest.mark.parametrize("shapes,stall,mode", CASES)
def test_dependency_wait_runs_out_and_reports_timeout(shapes, stall, mode):
    rng = np.random.default_rng(40 + stall)
    X = [rng.standard_normal(s).astype(np.float32) for s in shapes]
    Xt = [torch.from_numpy(x).to(dev()) for x in X]
    ws = workspace(mo.ns_workspace_bytes(shapes))
    prev_pair = B.mo_debug_set_ns_pair(0)          # the single-CTA geometry
    prev_mode = B.mo_debug_set_ns_fused(mode)
    try:
        outs = [torch.zeros_like(x) for x in Xt]
        torch.cuda.synchronize()
        B.mo_trace_enable(64)
        B.mo_debug_inject_dep_stall(stall, 2_000_000)
        try:
            t0 = time.perf_counter()
            mo.ns_orthogonalize(Xt, outs, 5, ws)
            status = mo.mo_check_device_status(ws)  # synchronises
            elapsed = time.perf_counter() - t0
        finally:
            B.mo_debug_inject_dep_stall(-1)
        kinds = [k for k, _ in B.mo_trace_read()]
        B.mo_trace_enable(0)
        assert "ns_fused" in kinds                  # the launch with dependency waits ran
        assert status == B.MO_ERR_TIMEOUT
        assert elapsed < 1.0
        # the device and the workspace are usable: a normal call matches the oracle
        outs2 = [torch.zeros_like(x) for x in Xt]
        mo.ns_orthogonalize(Xt, outs2, 5, ws)
        assert mo.mo_check_device_status(ws) == 0
        for x, o in zip(X, outs2):
            assert rel_fro(to_np(o), om.newton_schulz(x.astype(np.float64))) < NS_BF16_TOL
    finally:
        B.mo_debug_set_ns_fused(prev_mode)
        B.mo_debug_set_ns_pair(prev_pair)


def test_stall_hook_rejects_bad_arguments():
    with pytest.raises(B.MoError):
        B.mo_debug_inject_dep_stall(-2)
    with pytest.raises(B.MoError):
        B.mo_debug_inject_dep_stall(0, 10)

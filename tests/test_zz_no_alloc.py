"""The allocation-free Newton-Schulz entry point, ns_orthogonalize_noalloc.

Some callers cannot allocate device memory: a plugin that a host framework
hands only its input and output buffers (the framework owns and accounts for
all device memory), or a latency-critical loop where a cudaMalloc would
synchronise the device.  For them the library runs Newton-Schulz on a fixed
scratch array compiled into it.  These tests call that entry point through the
C ABI and check it against ns_orthogonalize with a caller workspace, on two
calls in a row of the same shape and then of another shape, so each later
call runs over an earlier call's leftovers in the shared scratch.  This file
is collected last on purpose.
"""
import numpy as np
import pytest
import torch

import matrix_optimizers_gb300 as mo
from matrix_optimizers_gb300 import _binding as B
from oracle import muon as om
from tests.gpu_helpers import NS_BF16_TOL, dev, rel_fro, to_np, workspace

pytestmark = pytest.mark.gpu


def _with_workspace(Xt, out_dtype):
    ref = torch.zeros(Xt.shape, dtype=out_dtype, device=dev())
    ws = workspace(mo.ns_workspace_bytes([tuple(Xt.shape)]))
    mo.ns_orthogonalize([Xt], [ref], 5, ws)
    return ref


def test_noalloc_matches_workspace_entry_two_calls_in_a_row():
    cases = [((768, 3072), torch.float32, torch.float32, 1),
             ((1000, 520), torch.bfloat16, torch.float32, 2)]
    for shape, in_dt, out_dt, seed in cases:
        X = np.random.default_rng(seed).standard_normal(shape).astype(np.float32)
        Xt = torch.from_numpy(X).to(dev()).to(in_dt)
        ref = _with_workspace(Xt, out_dt)
        want = to_np(ref)
        # two calls back to back on the same input: the second starts from the
        # first call's leftovers in the shared scratch
        outs = [torch.full(shape, float("nan"), dtype=out_dt, device=dev()) for _ in range(2)]
        B.ns_orthogonalize_noalloc(Xt, outs[0], 5)
        torch.cuda.synchronize()
        free_after_first = torch.cuda.mem_get_info()[0]
        B.ns_orthogonalize_noalloc(Xt, outs[1], 5)
        torch.cuda.synchronize()
        # the second call takes no device memory at all (the first may have
        # loaded the library's module and its scratch array)
        assert torch.cuda.mem_get_info()[0] == free_after_first
        # the runs' device status: no bounded wait gave up
        assert B.ns_orthogonalize_noalloc_status() == B.MO_OK
        for out in outs:
            got = to_np(out)
            assert np.all(np.isfinite(got))
            assert rel_fro(got, want) < NS_BF16_TOL
            assert rel_fro(got, om.newton_schulz(to_np(Xt))) < NS_BF16_TOL


def test_noalloc_rejects_a_matrix_beyond_the_scratch():
    X = torch.zeros(2048, 2048, device=dev())
    out = torch.zeros_like(X)
    with pytest.raises(B.MoError) as e:
        B.ns_orthogonalize_noalloc(X, out, 5)
    assert e.value.status == B.MO_ERR_UNSUPPORTED

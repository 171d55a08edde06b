"""matrix_optimizers_gb300: the Muon owner step for GB300 (sm_103a).

The compute lives in ``libmatrixopt.so`` (C ABI in ``include/matrixopt.h``);
this package is its ctypes binding.  Calls fail loudly when the library has not
been built; there is no CPU fallback.
"""
from ._binding import (  # noqa: F401
    MO_BF16, MO_F32, MO_NS_BF16, MO_NS_FP32, MoError,
    load, make_cfg, make_matrix, make_tail,
    mo_check_device_status, mo_trace_enable, mo_trace_read, mo_workspace_bytes, muon_step_batched,
    muon_step_sign_packed, muon_step_sign_vote,
    sign_int8, sign_pack_batched, sign_vote_polar_update, sign_vote_polar_workspace_bytes,
    sign_vote_update_int8,
    ns_orthogonalize, ns_workspace_bytes, plan_owners, sign_pack, sign_vote_update,
)

__version__ = "0.1.0"

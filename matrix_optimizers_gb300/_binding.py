"""ctypes binding of libmatrixopt (include/matrixopt.h): argument marshalling only.

Every function here has the name of the C entry point it calls, converts
torch tensors / Python values into the C structures and pointers, and raises
``MoError`` on a non-zero status.  No arithmetic of the method happens here:
every step runs in the library's CUDA kernels (or, for ``plan_owners``, in
its host C++).  If the library has not been built the first call raises.
"""
import ctypes
import os
import threading

import torch  # loads the CUDA runtime the library links against

from . import build as _build

c_int32, c_int64, c_float, c_double, c_void_p, c_size_t = (
    ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_double, ctypes.c_void_p, ctypes.c_size_t)

MO_OK, MO_ERR_INVALID_ARG, MO_ERR_ALIGNMENT, MO_ERR_WORKSPACE, MO_ERR_CUDA, MO_ERR_TIMEOUT, \
    MO_ERR_UNSUPPORTED = 0, -1, -2, -3, -4, -5, -6
MO_F32, MO_BF16 = 0, 1
MO_NS_BF16, MO_NS_FP32 = 0, 1


class MoError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__(f"{msg} (status {status})")
        self.status = status


class mo_matrix(ctypes.Structure):
    _fields_ = [("rows", c_int64), ("cols", c_int64), ("ld", c_int64),
                ("w_dtype", c_int32), ("m_dtype", c_int32), ("g_dtype", c_int32),
                ("reserved", c_int32),
                ("W", c_void_p), ("M", c_void_p), ("G", c_void_p)]


class mo_muon_cfg(ctypes.Structure):
    _fields_ = [("mu", c_float), ("lr", c_float), ("update_scale", c_float),
                ("weight_decay", c_float), ("ns_steps", c_int32),
                ("a", c_float), ("b", c_float), ("c", c_float),
                ("ns_precision", c_int32), ("apply_update", c_int32),
                ("out_dtype", c_int32), ("spectral_iters", c_int32)]


class mo_adamw_tail(ctypes.Structure):
    _fields_ = [("numel", c_int64), ("W", c_void_p), ("g", c_void_p), ("m", c_void_p),
                ("v", c_void_p), ("lr", c_float), ("beta1", c_float), ("beta2", c_float),
                ("eps", c_float), ("weight_decay", c_float), ("reserved", c_int32),
                ("step", c_int64)]


class mo_ns_view(ctypes.Structure):
    _fields_ = [("m", c_int64), ("n", c_int64), ("ldx", c_int64), ("lda", c_int64),
                ("transposed", c_int32), ("precision", c_int32),
                ("x_op", c_int64 * 2), ("diag_res", c_int64), ("gram", c_int64),
                ("poly", c_int64), ("deps", c_int64), ("tiles_sym", c_int32), ("tiles_apply", c_int32),
                ("releases_per_tile", c_int32), ("reserved", c_int32)]


# (name, restype, argtypes) of every exported symbol declared in include/*.h
_SIGNATURES = [
    ("mo_workspace_bytes", c_int32, [ctypes.POINTER(mo_matrix), c_int32, ctypes.POINTER(mo_muon_cfg),
                                     ctypes.POINTER(c_size_t)]),
    ("muon_step_batched", c_int32, [ctypes.POINTER(mo_matrix), c_int32, ctypes.POINTER(mo_muon_cfg),
                                    ctypes.POINTER(mo_adamw_tail), ctypes.POINTER(c_void_p),
                                    c_void_p, c_size_t, c_void_p]),
    ("muon_step_sign_packed", c_int32, [ctypes.POINTER(mo_matrix), c_int32, ctypes.POINTER(mo_muon_cfg),
                                        ctypes.POINTER(c_void_p), c_void_p, c_size_t, c_void_p]),
    ("muon_step_sign_vote", c_int32, [ctypes.POINTER(mo_matrix), c_int32, ctypes.POINTER(mo_muon_cfg),
                                      ctypes.POINTER(c_void_p), c_void_p, c_int32, c_int64, c_float, c_void_p,
                                      c_size_t, c_void_p]),
    ("ns_workspace_bytes", c_int32, [ctypes.POINTER(c_int64), ctypes.POINTER(c_int64), c_int32, c_int32,
                                     ctypes.POINTER(c_size_t)]),
    ("ns_orthogonalize", c_int32, [ctypes.POINTER(c_void_p), ctypes.POINTER(c_void_p),
                                   ctypes.POINTER(c_int64), ctypes.POINTER(c_int64),
                                   ctypes.POINTER(c_int64), c_int32, c_int32, c_int32, c_int32,
                                   c_float, c_float, c_float, c_int32, c_void_p, c_size_t, c_void_p]),
    ("ns_orthogonalize_noalloc", c_int32, [c_void_p, c_void_p, c_int64, c_int64, c_int64, c_int32, c_int32,
                                           c_int32, c_float, c_float, c_float, c_void_p]),
    ("ns_orthogonalize_noalloc_status", c_int32, [c_void_p]),
    ("sign_pack", c_int32, [c_void_p, c_int32, c_int64, c_int64, c_int64, c_void_p, c_void_p]),
    ("sign_vote_update", c_int32, [ctypes.POINTER(c_void_p), c_int32, c_int64, c_int64, c_void_p,
                                   c_int32, c_int64, c_float, c_void_p]),
    ("sign_vote_polar_workspace_bytes", c_int32, [c_int64, c_int64, c_int64, ctypes.POINTER(c_size_t)]),
    ("sign_vote_polar_update", c_int32, [ctypes.POINTER(c_void_p), c_int32, c_int64, c_int64, c_void_p, c_int32,
                                         c_int64, c_float, c_int32, c_float, c_float, c_float, c_void_p,
                                         c_size_t, c_void_p]),
    ("sign_pack_batched", c_int32, [ctypes.POINTER(c_void_p), c_int32, c_int32, c_int64, c_int64, c_int64,
                                    ctypes.POINTER(c_void_p), c_void_p]),
    ("sign_int8", c_int32, [c_void_p, c_int32, c_int64, c_int64, c_int64, c_void_p, c_void_p]),
    ("sign_vote_update_int8", c_int32, [ctypes.POINTER(c_void_p), c_int32, c_int64, c_int64, c_void_p,
                                        c_int32, c_int64, c_float, c_void_p]),
    ("plan_owners", c_int32, [ctypes.POINTER(c_int64), ctypes.POINTER(c_int64), c_int32, c_int32,
                              c_int32, c_double, c_double, ctypes.POINTER(c_int32),
                              ctypes.POINTER(c_double)]),
    ("mo_check_device_status", c_int32, [c_void_p, c_void_p]),
    ("mo_status_string", ctypes.c_char_p, [c_int32]),
    ("mo_version", c_int32, []),
    ("mo_debug_ns_view", c_int32, [ctypes.POINTER(c_int64), ctypes.POINTER(c_int64), c_int32, c_int32,
                                   c_int32, ctypes.POINTER(mo_ns_view)]),
    ("mo_debug_sm_count", c_int32, []),
    ("mo_debug_set_ns_fused", c_int32, [c_int32]),
    ("mo_debug_inject_dep_stall", c_int32, [c_int32, c_int64]),
    ("mo_debug_set_ns_pair", c_int32, [c_int32]),
    ("mo_debug_cta_stamps", c_int32, [c_void_p, c_int32, c_int32, ctypes.POINTER(c_int32)]),
    ("mo_trace_enable", c_int32, [c_int32]),
    ("mo_trace_read", c_int32, [ctypes.POINTER(c_int32), ctypes.POINTER(c_float), c_int32,
                                ctypes.POINTER(c_int32)]),
]

TRACE_KINDS = {1: "momentum_norm", 2: "norm_finalize", 3: "ns_gram", 4: "ns_poly", 5: "ns_apply",
               6: "ns_k0", 7: "adamw", 8: "sign_pack", 9: "vote_update", 10: "spectral_estimate",
               11: "ns_fused"}

_lib = None
_lock = threading.Lock()


def library_path():
    return _build.lib_path()


def load():
    """Load libmatrixopt.so (built in-tree by ``matrix_optimizers_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise ImportError(
                f"{path} is missing: build the CUDA library first "
                "(python -m matrix_optimizers_gb300.build or __graft_entry__.build())")
        lib = ctypes.CDLL(path)
        for name, res, args in _SIGNATURES:
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _check(status):
    if status != MO_OK:
        msg = load().mo_status_string(status).decode()
        raise MoError(status, msg)


def dtype_code(dt):
    if dt == torch.float32:
        return MO_F32
    if dt == torch.bfloat16:
        return MO_BF16
    raise MoError(MO_ERR_INVALID_ARG, f"unsupported dtype {dt}")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _ld(t):
    if t.dim() != 2 or (t.size(1) > 1 and t.stride(1) != 1):
        raise MoError(MO_ERR_INVALID_ARG, "matrices must be 2D with unit column stride")
    return t.stride(0) if t.size(0) > 1 else max(t.size(1), t.stride(0))


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def make_matrix(W, M, G):
    """mo_matrix for one parameter: W, M, G same shape and leading dimension."""
    if not (W.shape == M.shape == G.shape):
        raise MoError(MO_ERR_INVALID_ARG, "W, M and G must have one shape")
    ld = _ld(W)
    if _ld(M) != ld or _ld(G) != ld:
        raise MoError(MO_ERR_INVALID_ARG, "W, M and G must share the leading dimension")
    return mo_matrix(W.size(0), W.size(1), ld, dtype_code(W.dtype), dtype_code(M.dtype),
                     dtype_code(G.dtype), 0, W.data_ptr(), M.data_ptr(), G.data_ptr())


def make_cfg(mu=0.95, lr=0.02, ns_steps=5, a=3.4445, b=-4.7750, c=2.0315,
             precision=MO_NS_BF16, update_scale=1.0, weight_decay=0.0, apply_update=True,
             out_dtype=MO_BF16, spectral_iters=0):
    return mo_muon_cfg(mu, lr, update_scale, weight_decay, ns_steps, a, b, c, precision,
                       1 if apply_update else 0, out_dtype, spectral_iters)


def make_tail(W, g, m, v, step, lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.0):
    for t in (W, g, m, v):
        if t.dtype != torch.float32 or not t.is_contiguous():
            raise MoError(MO_ERR_INVALID_ARG, "the AdamW tail is contiguous float32")
    return mo_adamw_tail(W.numel(), W.data_ptr(), g.data_ptr(), m.data_ptr(), v.data_ptr(),
                         lr, beta1, beta2, eps, weight_decay, 0, step)


def _mat_array(mats):
    arr = (mo_matrix * max(1, len(mats)))()
    for i, m in enumerate(mats):
        arr[i] = m
    return arr


def mo_workspace_bytes(mats, cfg):
    out = c_size_t(0)
    _check(load().mo_workspace_bytes(_mat_array(mats), len(mats), ctypes.byref(cfg), ctypes.byref(out)))
    return out.value


def muon_step_batched(mats, cfg, ws, tail=None, out=None, stream=None):
    """One Muon step over ``mats`` (list of mo_matrix); ``ws`` a CUDA uint8
    tensor of at least mo_workspace_bytes(); ``out`` a list of tensors when
    cfg.apply_update is 0."""
    outs = None
    if out is not None:
        outs = (c_void_p * max(1, len(out)))(*[o.data_ptr() for o in out])
    _check(load().muon_step_batched(
        _mat_array(mats), len(mats), ctypes.byref(cfg),
        ctypes.byref(tail) if tail is not None else None, outs,
        _ptr(ws), ws.numel() if ws is not None else 0, _stream(stream)))


def muon_step_sign_packed(mats, cfg, words, ws, stream=None):
    """Sign-Muon worker step: momentum + NS with the packed signs of the
    direction written to ``words`` (list of int32 tensors) in the last epilogue."""
    arr = (c_void_p * max(1, len(words)))(*[w.data_ptr() for w in words])
    _check(load().muon_step_sign_packed(_mat_array(mats), len(mats), ctypes.byref(cfg), arr, _ptr(ws),
                                        ws.numel() if ws is not None else 0, _stream(stream)))


def muon_step_sign_vote(mats, cfg, words, W, lr, ws, stream=None):
    """The Sign-Muon step of the M workers ``mats``: momentum + NS with fused
    sign packing into ``words``, then the majority vote W <- W - lr * vote."""
    arr = (c_void_p * max(1, len(words)))(*[w.data_ptr() for w in words])
    _check(load().muon_step_sign_vote(_mat_array(mats), len(mats), ctypes.byref(cfg), arr, _ptr(W),
                                      dtype_code(W.dtype), _ld(W), lr, _ptr(ws),
                                      ws.numel() if ws is not None else 0, _stream(stream)))


def ns_workspace_bytes(shapes, precision=MO_NS_BF16):
    n = len(shapes)
    rows = (c_int64 * max(1, n))(*[s[0] for s in shapes])
    cols = (c_int64 * max(1, n))(*[s[1] for s in shapes])
    out = c_size_t(0)
    _check(load().ns_workspace_bytes(rows, cols, n, precision, ctypes.byref(out)))
    return out.value


def ns_orthogonalize(X, out, steps, ws, a=3.4445, b=-4.7750, c=2.0315, precision=MO_NS_BF16,
                     stream=None):
    """out[i] = NS_steps(X[i]/||X[i]||_F) for lists of tensors (one dtype each)."""
    n = len(X)
    xs = (c_void_p * max(1, n))(*[x.data_ptr() for x in X])
    os_ = (c_void_p * max(1, n))(*[o.data_ptr() for o in out])
    rows = (c_int64 * max(1, n))(*[x.size(0) for x in X])
    cols = (c_int64 * max(1, n))(*[x.size(1) for x in X])
    lds = []
    for x, o in zip(X, out):
        if _ld(x) != _ld(o):
            raise MoError(MO_ERR_INVALID_ARG, "X[i] and out[i] must share the leading dimension")
        lds.append(_ld(x))
    ld = (c_int64 * max(1, n))(*lds)
    in_dt = dtype_code(X[0].dtype) if n else MO_F32
    out_dt = dtype_code(out[0].dtype) if n else MO_F32
    _check(load().ns_orthogonalize(xs, os_, rows, cols, ld, n, in_dt, out_dt, steps, a, b, c,
                                   precision, _ptr(ws), ws.numel() if ws is not None else 0,
                                   _stream(stream)))


def ns_orthogonalize_noalloc(X, out, steps, a=3.4445, b=-4.7750, c=2.0315, stream=None):
    """out = NS_steps(X/||X||_F) for one matrix, using the library's fixed
    device scratch instead of a workspace (for callers that cannot allocate
    device memory; see include/matrixopt.h for the size limit)."""
    if _ld(X) != _ld(out):
        raise MoError(MO_ERR_INVALID_ARG, "X and out must share the leading dimension")
    _check(load().ns_orthogonalize_noalloc(_ptr(X), _ptr(out), X.size(0), X.size(1), _ld(X),
                                           dtype_code(X.dtype), dtype_code(out.dtype), steps, a, b, c,
                                           _stream(stream)))


def ns_orthogonalize_noalloc_status(stream=None):
    """MO_OK, or MO_ERR_TIMEOUT if an allocation-free run's bounded device
    wait gave up since the last check (the record is then cleared)."""
    return load().ns_orthogonalize_noalloc_status(_stream(stream))


def sign_pack(U, words, stream=None):
    """Pack the signs of U (2D float32/bf16) into the uint32 words tensor
    (int32 storage, ceil(numel/32) entries)."""
    _check(load().sign_pack(_ptr(U), dtype_code(U.dtype), U.size(0), U.size(1), _ld(U),
                            _ptr(words), _stream(stream)))


def sign_vote_update(words, W, lr, stream=None):
    """W -= lr * majority_vote(words) for a list of packed word tensors."""
    M = len(words)
    arr = (c_void_p * max(1, M))(*[w.data_ptr() for w in words])
    _check(load().sign_vote_update(arr, M, W.size(0), W.size(1), _ptr(W), dtype_code(W.dtype),
                                   _ld(W), lr, _stream(stream)))


def sign_vote_polar_workspace_bytes(W):
    out = c_size_t(0)
    _check(load().sign_vote_polar_workspace_bytes(W.size(0), W.size(1), _ld(W), ctypes.byref(out)))
    return out.value


def sign_vote_polar_update(words, W, lr, ws, steps=5, a=3.4445, b=-4.7750, c=2.0315, stream=None):
    """W -= lr * NS(majority_vote(words)): the vote followed by the local polar step."""
    M = len(words)
    arr = (c_void_p * max(1, M))(*[w.data_ptr() for w in words])
    _check(load().sign_vote_polar_update(arr, M, W.size(0), W.size(1), _ptr(W), dtype_code(W.dtype), _ld(W),
                                         lr, steps, a, b, c, _ptr(ws), ws.numel() if ws is not None else 0,
                                         _stream(stream)))


def sign_pack_batched(U, words, stream=None):
    """sign_pack of M same-shaped matrices (lists U, words) in one launch."""
    M = len(U)
    us = (c_void_p * max(1, M))(*[u.data_ptr() for u in U])
    ws = (c_void_p * max(1, M))(*[w.data_ptr() for w in words])
    lds = {_ld(u) for u in U}
    if len(lds) != 1 or len({tuple(u.shape) for u in U}) != 1 or len({u.dtype for u in U}) != 1:
        raise MoError(MO_ERR_INVALID_ARG, "sign_pack_batched wants one shape, dtype and ld")
    _check(load().sign_pack_batched(us, M, dtype_code(U[0].dtype), U[0].size(0), U[0].size(1), lds.pop(),
                                    ws, _stream(stream)))


def sign_int8(U, out, stream=None):
    """int8 signs (-1/+1) of U into ``out`` (int8, rows*cols entries)."""
    _check(load().sign_int8(_ptr(U), dtype_code(U.dtype), U.size(0), U.size(1), _ld(U), _ptr(out),
                            _stream(stream)))


def sign_vote_update_int8(signs, W, lr, stream=None):
    """W -= lr * sign(sum of the workers' int8 signs), ties -> +1."""
    M = len(signs)
    arr = (c_void_p * max(1, M))(*[s.data_ptr() for s in signs])
    _check(load().sign_vote_update_int8(arr, M, W.size(0), W.size(1), _ptr(W), dtype_code(W.dtype),
                                        _ld(W), lr, _stream(stream)))


def plan_owners(shapes, world, ns_steps=5, w_bytes=1.0, w_flops=1.0):
    """Host-only owner plan: returns (owner list, per-rank load list)."""
    n = len(shapes)
    rows = (c_int64 * max(1, n))(*[s[0] for s in shapes])
    cols = (c_int64 * max(1, n))(*[s[1] for s in shapes])
    owner = (c_int32 * max(1, n))()
    load_ = (c_double * max(1, world))() if world > 0 else None
    _check(load().plan_owners(rows, cols, n, world, ns_steps, w_bytes, w_flops, owner, load_))
    return list(owner)[:n], list(load_)[:world]


def mo_check_device_status(ws, stream=None):
    """Returns the status word the kernels left in ``ws`` (and clears it)."""
    return load().mo_check_device_status(_ptr(ws), _stream(stream))


def mo_debug_ns_view(shapes, index, precision=MO_NS_BF16):
    n = len(shapes)
    rows = (c_int64 * max(1, n))(*[s[0] for s in shapes])
    cols = (c_int64 * max(1, n))(*[s[1] for s in shapes])
    v = mo_ns_view()
    _check(load().mo_debug_ns_view(rows, cols, n, precision, index, ctypes.byref(v)))
    return v


def mo_debug_inject_dep_stall(matrix, wait_cycles=2_000_000):
    """Makes the fused NS launch's dependency waits of matrix `matrix` run out
    after `wait_cycles` SM cycles (matrix -1 turns it off)."""
    _check(load().mo_debug_inject_dep_stall(matrix, wait_cycles))


def mo_debug_set_ns_pair(on):
    """Selects 256 x 256 CTA-pair tiles (True) or 128 x 256 single-CTA tiles
    (False) for the NS kernel; returns the previous setting."""
    prev = load().mo_debug_set_ns_pair(1 if on else 0)
    _check(prev if prev < 0 else 0)
    return bool(prev)


def mo_debug_set_ns_fused(on):
    """Selects the NS launch schedule: 1 / True fused with per-matrix
    counters, 2 fused with grid-wide counters, 3 (default) either by size,
    0 / False one launch per phase; returns the previous setting."""
    prev = load().mo_debug_set_ns_fused(int(on))
    _check(prev if prev < 0 else 0)
    return prev


def mo_debug_cta_stamps(buf, capacity, max_ctas):
    """Start recording per-CTA stamps (start, end, dependency-wait ns,
    spinning waits) into ``buf`` (int64 CUDA tensor of 4*capacity*max_ctas
    entries); ``buf=None`` stops.  Returns the number of launches recorded
    since the previous call."""
    rec = c_int32(0)
    _check(load().mo_debug_cta_stamps(_ptr(buf), capacity, max_ctas, ctypes.byref(rec)))
    return rec.value


def mo_trace_enable(capacity):
    """Record a CUDA event pair around each of the next ``capacity`` launches
    issued from this thread (0 disables)."""
    _check(load().mo_trace_enable(capacity))


def mo_trace_read(cap=1 << 16):
    """[(kind name, milliseconds), ...] of the launches traced since the last read."""
    kinds = (c_int32 * cap)()
    ms = (c_float * cap)()
    count = c_int32(0)
    _check(load().mo_trace_read(kinds, ms, cap, ctypes.byref(count)))
    return [(TRACE_KINDS.get(kinds[i], str(kinds[i])), ms[i]) for i in range(min(cap, count.value))]

"""Shapes, seeds and seeded inputs of the five synthetic workloads.

Recipe (every array is drawn on the CPU with NumPy's PCG64 ``default_rng``):

* per-matrix streams: matrix ``i`` of a set draws from ``default_rng([seed, i])``
  so that one matrix can be regenerated alone (sampled checks at full size);
* normals are drawn in float32 (``standard_normal(dtype=float32)``) and scaled
  by the stated standard deviation in float32; bf16 state is the float32 value
  cast to bf16 by torch (round to nearest even);
* momentum starts at zero unless a workload says otherwise.

Workloads (name -> what it is):

* ``single_256x512``   one 256x512 float32 matrix; M0 and G i.i.d. N(0,1) drawn
                       in that order from ``default_rng(0)`` in float64 then
                       cast; W0 = 0; mu 0.95, lr 0.02, fp32 NS, k = 5.
* ``gpt_small``        12 layers x {Wq, Wk, Wv, Wo 768x768, W_up 768x3072,
                       W_down 3072x768} = 72 matrices; W ~ N(0, 0.02^2) (seed 0),
                       G ~ N(0, 1e-3^2) (seed 1); bf16 NS; plus a 36,864-value
                       float32 tail (12 x 4 x 768) for AdamW.
* ``llama7b_owner0``   32 layers x {4 x 4096x4096, 4096x11008 (gate, up),
                       11008x4096 (down)} = 224 matrices planned onto 8 ranks;
                       this GPU steps rank 0's share; W ~ N(0, 0.02^2) (seed 0),
                       G ~ N(0, 1e-3^2) (seed 1); bf16 NS.
* ``sign_muon_m8``     8 workers x 2048x2048; G ~ N(0,1) (seed 0) shared,
                       noise_m ~ N(0, 0.5^2) (seed 1+m); worker gradient
                       G + noise_m (float32); bf16 momentum starting at 0;
                       W ~ N(0, 0.02^2) (seed 100) float32; lr 1e-3.
* ``ragged500``        500 shapes, each side log-uniform on [64, 8192]
                       (``default_rng(0)``, m then n), rejected when the aspect
                       exceeds 8, each side rounded to the nearest multiple of
                       8; W ~ N(0, 0.02^2) (seed 0), G ~ N(0, 1e-3^2) (seed 1);
                       plus a 50,000,000-value float32 AdamW tail.
"""
import math

import numpy as np

NS_COEFFS = (3.4445, -4.7750, 2.0315)
NS_STEPS = 5
MU = 0.95


def gpt_small_shapes(layers=12, d=768, ff=3072):
    out = []
    for _ in range(layers):
        out += [(d, d)] * 4 + [(d, ff), (ff, d)]
    return out


def llama7b_shapes(layers=32, d=4096, ff=11008):
    out = []
    for _ in range(layers):
        out += [(d, d)] * 4 + [(d, ff), (d, ff), (ff, d)]
    return out


def ragged_shapes(count=500, seed=0, lo=64, hi=8192, max_aspect=8, multiple=8):
    rng = np.random.default_rng(seed)
    la, lb = math.log(lo), math.log(hi)
    out = []
    while len(out) < count:
        m = math.exp(rng.uniform(la, lb))
        n = math.exp(rng.uniform(la, lb))
        if max(m, n) / min(m, n) > max_aspect:
            continue
        m = max(multiple, int(round(m / multiple)) * multiple)
        n = max(multiple, int(round(n / multiple)) * multiple)
        out.append((m, n))
    return out


def _normal(key, shape, std):
    x = np.random.default_rng(key).standard_normal(shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return x


def matrix_inputs(shapes, index, seed_w=0, seed_g=1, w_std=0.02, g_std=1e-3):
    """Inputs of matrix ``index`` of a set: dict of float32 W and G; the
    momentum starts at zero (no array is stored for it)."""
    r, c = shapes[index]
    return {
        "W": _normal([seed_w, index], (r, c), w_std),
        "G": _normal([seed_g, index], (r, c), g_std),
    }


def matrix_set_inputs(shapes, indices=None, threads=None, **kw):
    """matrix_inputs for many matrices, drawn in parallel threads (each matrix
    has its own generator, so the result does not depend on the threading)."""
    from concurrent.futures import ThreadPoolExecutor
    import os
    idx = list(range(len(shapes))) if indices is None else list(indices)
    threads = threads or min(16, len(os.sched_getaffinity(0)))
    with ThreadPoolExecutor(max_workers=threads) as ex:
        return list(ex.map(lambda i: matrix_inputs(shapes, i, **kw), idx))


def single_matrix_inputs(rows=256, cols=512, seed=0):
    """single_256x512: M0 then G from one default_rng(seed) stream, float64 ->
    float32; W0 = 0."""
    rng = np.random.default_rng(seed)
    M0 = rng.standard_normal((rows, cols)).astype(np.float32)
    G = rng.standard_normal((rows, cols)).astype(np.float32)
    return {"W": np.zeros((rows, cols), dtype=np.float32), "G": G, "M0": M0}


def sign_muon_inputs(workers=8, n=2048, seed_g=0, noise_std=0.5, seed_w=100):
    """sign_muon_m8: per-worker float32 gradients, shared W (float32)."""
    G = np.random.default_rng(seed_g).standard_normal((n, n))
    grads = []
    for m in range(workers):
        noise = noise_std * np.random.default_rng(1 + m).standard_normal((n, n))
        grads.append((G + noise).astype(np.float32))
    W = (0.02 * np.random.default_rng(seed_w).standard_normal((n, n))).astype(np.float32)
    return {"G": grads, "W": W}


def tight_spectrum_matrix(m, n, seed=0, spread=0.01):
    """An m x n (m <= n) float32 matrix whose singular values all lie within
    +-`spread` of 1: orthonormal rows (QR of an n x m N(0,1) draw from
    default_rng(seed)) scaled per row by 1 + spread * N(0,1) (default_rng(seed + 9)).
    Normalised by its Frobenius norm, every singular value starts near
    1/sqrt(m): the hardest start for bf16 Newton-Schulz."""
    Q, _ = np.linalg.qr(np.random.default_rng(seed).standard_normal((n, m)))
    scale = 1.0 + spread * np.random.default_rng(seed + 9).standard_normal((m, 1))
    return (Q.T * scale).astype(np.float32)


def tail_inputs(numel, seed=7, w_std=0.02, g_std=1e-3):
    """AdamW tail: float32 W, g; m = v = 0."""
    return {
        "W": _normal([seed, 0], (numel,), w_std),
        "g": _normal([seed, 1], (numel,), g_std),
        "m": np.zeros(numel, dtype=np.float32),
        "v": np.zeros(numel, dtype=np.float32),
    }


CONFIGS = {
    "single_256x512": dict(shapes=[(256, 512)], mu=MU, lr=0.02, precision="fp32"),
    "gpt_small": dict(shapes=gpt_small_shapes(), mu=MU, lr=0.02, precision="bf16",
                      tail_numel=12 * 4 * 768, tail_lr=1e-3),
    "llama7b_owner0": dict(shapes=llama7b_shapes(), world=8, owner=0, mu=MU, lr=0.02,
                           precision="bf16"),
    "sign_muon_m8": dict(shapes=[(2048, 2048)] * 8, mu=MU, lr=1e-3, precision="bf16"),
    "ragged500": dict(shapes=None, mu=MU, lr=0.02, precision="bf16",
                      tail_numel=50_000_000, tail_lr=1e-3),
}

"""Muon owner step in float64: momentum, normalisation, orientation,
quintic Newton-Schulz, scaled weight update.

Oracle module: test infrastructure only.

Passages followed
-----------------
* "Riepilogo Tecnico: SignMuon" §2 "Meccanismo Principale" item 1: each worker
  forms a momentum matrix and takes the polar direction of it, approximated by
  a Newton-Schulz iteration that orthogonalises the momentum;
  §2 "Flusso Algoritmico" step 1: gradient -> momentum M_{t+1} -> polar factor
  U_t by NS; step 4: the update is W_{t+1} = W_t - eta_t * (direction).
* "Riassunto Tecnico: MatrixFSDP" §Metodologia 1: the owner of a full 2D
  matrix runs that NS update locally, with no matrix communication.
* SignMuon §3 "Geometria": the normalised direction has spectral norm at most 1
  (the quintic below keeps it within ~1.2024; see the NS band pin).

The pages name the iteration but print neither its polynomial nor its
constants.  Readings taken (each one a parameter):
  momentum    heavy-ball M <- mu*M + G, no Nesterov term;
  X0          M / ||M||_F, no epsilon, and X0 = 0 when ||M||_F = 0;
  orientation if rows > cols iterate on M^T (m <= n), transpose back after;
              for rows == cols no transpose;
  NS step     A = X X^T ; B = b*A + c*A@A ; X <- a*X + B@X, repeated k times,
              (a, b, c) = (3.4445, -4.7750, 2.0315), k = 5;
  update      W <- W - lr*weight_decay*W - lr*update_scale*O,
              update_scale = 1 and weight_decay = 0 by default.
"""
import numpy as np

from .bf16 import round_bf16

NS_A, NS_B, NS_C = 3.4445, -4.7750, 2.0315
NS_STEPS = 5


def momentum(M0, G, mu):
    """Heavy-ball momentum M1 = mu*M0 + G (float64)."""
    return mu * np.asarray(M0, dtype=np.float64) + np.asarray(G, dtype=np.float64)


def orient(M):
    """Return (X, transposed): X = M^T when M has more rows than columns."""
    M = np.asarray(M, dtype=np.float64)
    if M.shape[0] > M.shape[1]:
        return M.T, True
    return M, False


def frobenius_normalize(X):
    """Return (X / ||X||_F, ||X||_F); the zero matrix maps to zeros."""
    X = np.asarray(X, dtype=np.float64)
    s = float(np.sqrt(np.sum(X * X)))
    if s == 0.0:
        return np.zeros_like(X), 0.0
    return X / s, s


def spectral_estimate(F, iters):
    """Largest singular value of F by power iteration on the Gram matrix
    F F^T: v0 = ones/sqrt(m); repeat iters times y = (F F^T) v, v = y/||y||;
    then sigma^2 = v^T (F F^T) v (the Rayleigh quotient)."""
    F = np.asarray(F, dtype=np.float64)
    Gm = F @ F.T
    m = Gm.shape[0]
    v = np.ones(m) / np.sqrt(m)
    for _ in range(iters):
        y = Gm @ v
        nrm = np.linalg.norm(y)
        if nrm == 0.0:
            return 0.0
        v = y / nrm
    lam = float(v @ (Gm @ v))
    return float(np.sqrt(max(lam, 0.0)))


def spectral_normalize(X, iters):
    """X / sigma_hat: the spectral scale the pages contrast with the
    Frobenius scale ("Riepilogo Tecnico: SignMuon" §4, nanoGPT).  Reading:
    sigma_hat is estimated by `iters` power iterations (spectral_estimate) on
    the Frobenius-normalised matrix, so the result is X/||X||_F/sigma_hat."""
    F, s = frobenius_normalize(X)
    if s == 0.0:
        return F, 0.0
    sig = spectral_estimate(F, iters)
    return (F / sig if sig > 0 else np.zeros_like(F)), s * sig


def ns_iterate(X0, steps=NS_STEPS, a=NS_A, b=NS_B, c=NS_C):
    """k quintic NS steps on an m x n matrix (any m, n): the pages' local
    orthogonalisation, with the Gram matrix formed on the rows of X."""
    X = np.asarray(X0, dtype=np.float64)
    for _ in range(steps):
        A = X @ X.T                     # m x m Gram matrix
        B = b * A + c * (A @ A)         # polynomial part, m x m
        X = a * X + B @ X               # apply to X
    return X


def newton_schulz(M, steps=NS_STEPS, a=NS_A, b=NS_B, c=NS_C, spectral_iters=0):
    """Orthogonalised direction O of a 2D matrix M, in M's own orientation:
    orient to m <= n, normalise (Frobenius norm, or the spectral estimate
    when spectral_iters > 0), iterate, orient back."""
    X, transposed = orient(M)
    if spectral_iters > 0:
        X0, _ = spectral_normalize(X, spectral_iters)
    else:
        X0, _ = frobenius_normalize(X)
    O = ns_iterate(X0, steps, a, b, c)
    return O.T if transposed else O


def muon_update(W, O, lr, update_scale=1.0, weight_decay=0.0):
    """W - lr*weight_decay*W - lr*update_scale*O (float64)."""
    W = np.asarray(W, dtype=np.float64)
    return W - lr * weight_decay * W - lr * update_scale * np.asarray(O, dtype=np.float64)


def muon_step(W, M0, G, mu, lr, steps=NS_STEPS, a=NS_A, b=NS_B, c=NS_C,
              update_scale=1.0, weight_decay=0.0, m_dtype="f32", apply_update=True, spectral_iters=0):
    """One Muon step on one matrix.

    Returns (W_new, M_stored, O): O is the NS output the update uses.
    ``m_dtype="bf16"`` models momentum state held in bfloat16: the stored
    momentum is bf16_rne(mu*M0 + G) and NS runs on that stored value.
    With ``apply_update=False`` W is returned unchanged.
    """
    M1 = momentum(M0, G, mu)
    if m_dtype == "bf16":
        M1 = round_bf16(M1)
    O = newton_schulz(M1, steps, a, b, c, spectral_iters)
    W_new = muon_update(W, O, lr, update_scale, weight_decay) if apply_update \
        else np.asarray(W, dtype=np.float64)
    return W_new, M1, O


def ns_flops(rows, cols, steps=NS_STEPS):
    """Nominal NS work: 4 m^2 n + 2 m^3 flops per step with m = min, n = max
    (the Gram product 2m^2n, the square 2m^3, the apply 2m^2n)."""
    m, n = min(rows, cols), max(rows, cols)
    return steps * (4 * m * m * n + 2 * m ** 3)

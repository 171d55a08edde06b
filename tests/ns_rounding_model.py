"""NumPy model of the tensor-core Newton-Schulz path's rounding (CPU only).

X, A and B are bf16, rounded to nearest even.  Products accumulate exactly,
standing in for the fp32 accumulator.  X is kept in bf16 between steps.

Forms:
* "folded_diag" (the kernels'): B = aI + bA + cA^2 as one bf16 operator, and
  X' = B X + d X with d = diag(B) - bf16(diag(B)) held in fp32.  B's diagonal
  sits near a = 3.44, where the bf16 spacing is 2^-6, so its rounding is the
  largest error of the step; the residual row scale removes it.
* "folded": the same operator without the diagonal residual.
* "bf16_ax", "fp32_master": aX added in fp32 outside the product, from X's
  bf16 operand or from an fp32 master of X."""
import numpy as np
import torch

from oracle import muon as om

A, B, C = om.NS_A, om.NS_B, om.NS_C


def bf(x):
    return torch.from_numpy(np.asarray(x, np.float32)).bfloat16().double().numpy()


def f32(x):
    return np.asarray(x, np.float32).astype(np.float64)


def ns_bf16_model(X0, steps=5, form="folded_diag"):
    Xf = f32(X0)
    Xb = bf(Xf)
    for _ in range(steps):
        Ab = bf(f32(Xb @ Xb.T))
        P = f32(B * Ab + C * f32(Ab @ Ab))
        if form in ("folded", "folded_diag"):
            Pa = f32(P + A * np.eye(len(P)))
            Pb = bf(Pa)
            Y = Pb @ Xb
            if form == "folded_diag":
                Y = Y + f32(np.diag(Pa) - np.diag(Pb))[:, None] * Xb
            Xf = f32(Y)
        else:
            Xf = f32(A * (Xf if form == "fp32_master" else Xb) + bf(P) @ Xb)
        Xb = bf(Xf)
    return Xf


def model_rel_err(M, form="folded_diag"):
    """Relative Frobenius error of a bf16 model form against the fp64 oracle
    for the NS of M (Frobenius scaling; M in any orientation)."""
    Y = M if M.shape[0] <= M.shape[1] else M.T
    ref = om.ns_iterate(Y / np.linalg.norm(Y))
    return float(np.linalg.norm(ns_bf16_model(Y / np.linalg.norm(Y), form=form) - ref) / np.linalg.norm(ref))

"""NumPy model of the tensor-core Newton-Schulz path's rounding (CPU only).

X, A and B are bf16, rounded to nearest even.  Products accumulate exactly,
standing in for the fp32 accumulator.  X is kept in bf16 between steps.  The
"folded" form is the kernels': B = aI + bA + cA^2 as one bf16 operator, then
X' = B X.  Two alternative forms add aX in fp32 outside the product, from X's
bf16 operand or from an fp32 master of X."""
import numpy as np
import torch

from oracle import muon as om

A, B, C = om.NS_A, om.NS_B, om.NS_C


def bf(x):
    return torch.from_numpy(np.asarray(x, np.float32)).bfloat16().double().numpy()


def f32(x):
    return np.asarray(x, np.float32).astype(np.float64)


def ns_bf16_model(X0, steps=5, form="folded"):
    Xf = f32(X0)
    Xb = bf(Xf)
    for _ in range(steps):
        Ab = bf(f32(Xb @ Xb.T))
        P = f32(B * Ab + C * f32(Ab @ Ab))
        if form == "folded":
            Xf = f32(bf(P + A * np.eye(len(P))) @ Xb)
        else:
            Xf = f32(A * (Xf if form == "fp32_master" else Xb) + bf(P) @ Xb)
        Xb = bf(Xf)
    return Xf


def model_rel_err(M):
    """Relative Frobenius error of the folded bf16 model against the fp64
    oracle for the NS of M (Frobenius scaling; M in any orientation)."""
    Y = M if M.shape[0] <= M.shape[1] else M.T
    ref = om.ns_iterate(Y / np.linalg.norm(Y))
    return float(np.linalg.norm(ns_bf16_model(Y / np.linalg.norm(Y)) - ref) / np.linalg.norm(ref))

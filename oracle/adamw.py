"""Decoupled AdamW for the 1D tail, in float64.

Oracle module: test infrastructure only.

"Riassunto Tecnico: MatrixFSDP" §Metodologia 1 ("Tensori Non-Matriciali"): the
1D and other non-2D tensors are packed into a tail on a separate owner and keep
standard AdamW.  The pages give no hyper-parameters; betas (0.9, 0.95) and
eps 1e-8 are the workload's, and the reading for the rest is textbook AdamW
with bias correction and decoupled weight decay, step counter t starting at 1:

    m <- beta1*m + (1-beta1)*g
    v <- beta2*v + (1-beta2)*g^2
    W <- W - lr*wd*W - lr * (m/(1-beta1^t)) / (sqrt(v/(1-beta2^t)) + eps)
"""
import numpy as np


def adamw_step(W, g, m, v, t, lr, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.0):
    """One AdamW step at step number t (>= 1).  Returns (W, m, v) in float64."""
    W = np.asarray(W, dtype=np.float64)
    g = np.asarray(g, dtype=np.float64)
    m = beta1 * np.asarray(m, dtype=np.float64) + (1.0 - beta1) * g
    v = beta2 * np.asarray(v, dtype=np.float64) + (1.0 - beta2) * g * g
    m_hat = m / (1.0 - beta1 ** t)
    v_hat = v / (1.0 - beta2 ** t)
    W = W - lr * weight_decay * W - lr * m_hat / (np.sqrt(v_hat) + eps)
    return W, m, v

"""Helpers for the GPU parity tests: device tensors from seeded NumPy inputs,
relative Frobenius errors, and the tolerances the tests hold the kernels to.

Tolerances (each stated where it is used):
  NS_BF16_TOL  2e-2 relative Frobenius error of a bf16-operand NS output (or of
               the Muon update it drives) against the fp64 oracle;
  NS_BF16_SPECTRAL_TOL  2e-2 for bf16 NS under spectral scaling as well (the
               bf16 rounding model in test_tolerance_model.py reaches ~1.7e-2);
  NS_FP32_TOL  1e-4 for the fp32 NS mode;
  MOM_TOL      1e-6 relative error of float32 momentum (one fp32 FMA vs fp64);
  bit-exact    sign, pack, vote, voted update, owner plan.
"""
import numpy as np
import torch

NS_BF16_TOL = 2e-2
NS_BF16_SPECTRAL_TOL = 2e-2      # spectral scale: the model in tests/test_tolerance_model.py stays below it
NS_FP32_TOL = 1e-4
MOM_TOL = 1e-6


def dev():
    return torch.device("cuda:0")


def to_dev(a, dtype=torch.float32, ld=None):
    """Upload a 2D array; with ``ld`` > cols the tensor is a column slice of a
    wider buffer (leading dimension ld)."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    if ld is None or ld == a.shape[1]:
        return t.to(dtype).to(dev())
    buf = torch.full((a.shape[0], ld), float("nan"), dtype=dtype, device=dev())
    buf[:, : a.shape[1]] = t.to(dtype).to(dev())
    return buf[:, : a.shape[1]]


def to_np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def rel_fro(got, want):
    want = np.asarray(want, dtype=np.float64)
    den = np.linalg.norm(want)
    return float(np.linalg.norm(np.asarray(got, dtype=np.float64) - want) / (den if den > 0 else 1.0))


def workspace(nbytes):
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=dev())


def ws_view(ws, offset, shape, dtype, ld):
    """A 2D view (rows x cols, leading dimension ld) into the workspace."""
    esz = torch.tensor([], dtype=dtype).element_size()
    rows, cols = shape
    flat = ws[offset: offset + rows * ld * esz].view(dtype)
    return flat.view(rows, ld)[:, :cols]

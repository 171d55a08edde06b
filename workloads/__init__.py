"""Seeded synthetic workloads shared by the library's tests/bench and the oracle.

This package draws inputs only: shapes, seeds, random matrices and their
storage-type casts.  It holds none of the method's arithmetic, and imports
neither ``oracle`` nor ``matrix_optimizers_gb300``.
"""
from .configs import (  # noqa: F401
    NS_COEFFS, gpt_small_shapes, llama7b_shapes, ragged_shapes,
    matrix_inputs, matrix_set_inputs, sign_muon_inputs, tail_inputs, single_matrix_inputs,
    tight_spectrum_matrix,
    CONFIGS,
)

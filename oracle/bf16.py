"""bfloat16 round-to-nearest-even, written from the format's definition.

bfloat16 keeps the float32 exponent range (8 exponent bits) and 8 significant
bits (7 stored + the implicit one).  Normal values are rounded to the nearest
multiple of 2**(e-7) where 2**e <= |x| < 2**(e+1); values below the smallest
normal (2**-126) are rounded on the subnormal grid 2**-133.  Ties go to the
even significand.  Values at or above 2**128 * (1 - 2**-9) overflow to inf.

Oracle module: test infrastructure only.
"""
import numpy as np

_MIN_EXP_SPACING = -133        # spacing of bf16 subnormals
_OVERFLOW = 2.0 ** 128 * (1.0 - 2.0 ** -9)   # halfway above the largest finite


def round_bf16(x):
    """Return float64 array holding bf16_rne(x) for each element of ``x``.

    Rounds directly from the float64 value (no intermediate float32 step).
    NaN stays NaN; +-inf stay; signed zero keeps its sign.
    """
    x = np.asarray(x, dtype=np.float64)
    out = np.array(x, dtype=np.float64, copy=True)
    finite = np.isfinite(x) & (x != 0.0)
    xf = x[finite]
    # |x| = mant * 2**exp with 0.5 <= mant < 1  ->  2**(exp-1) <= |x| < 2**exp
    _, exp = np.frexp(xf)
    # grid spacing for 8 significant bits: 2**(exp-1-7) ; clamp to subnormal grid
    spacing_exp = np.maximum(exp - 8, _MIN_EXP_SPACING)
    scaled = np.ldexp(xf, -spacing_exp)          # exact (power-of-two scaling)
    q = np.rint(scaled)                          # round-half-even
    r = np.ldexp(q, spacing_exp)
    r = np.where(np.abs(xf) >= _OVERFLOW, np.copysign(np.inf, xf), r)
    # keep the sign of values that rounded to zero
    r = np.where(r == 0.0, np.copysign(0.0, xf), r)
    out[finite] = r
    return out

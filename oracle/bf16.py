"""bfloat16 helpers for the oracle (test infrastructure only).

bfloat16 is the upper half of an IEEE-754 binary32: 1 sign bit, 8 exponent
bits, 7 stored fraction bits. The oracle keeps bf16 tensors as their raw
uint16 bit patterns, widens them exactly to float64 for arithmetic, and rounds
an exact float64 result to bf16 ONCE, directly (round to nearest, ties to
even). Rounding float64 -> float32 -> bf16 would round twice and can land one
ulp off on values just beside a bf16 tie, so it is not used.
"""

import numpy as np

# bf16 has 8 significant bits (1 implicit + 7 stored). For |x| in
# [2**(e-1), 2**e) the spacing of bf16 values is 2**(e-8). The smallest
# spacing is that of the subnormals, 2**-133 (= 2**-126 * 2**-7).
_BF16_SIG_BITS = 8
_BF16_MIN_EXP_SPACING = -133
_BF16_OVERFLOW = 2.0 ** 128  # first power of two past the largest finite bf16


def bf16_bits_to_f64(bits):
    """Widen bf16 bit patterns (uint16) exactly to float64."""
    b = np.asarray(bits, dtype=np.uint16)
    with np.errstate(invalid="ignore"):  # signalling-NaN patterns stay NaN
        return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def to_bf16_rne(x):
    """Round float64 values to bf16 (nearest, ties to even) in one step.

    Returns the uint16 bit patterns. NaN maps to the canonical quiet NaN 0x7FC0;
    values whose rounding reaches 2**128 in magnitude become +-inf.
    """
    x = np.asarray(x, dtype=np.float64)
    with np.errstate(invalid="ignore", over="ignore"):
        _, e = np.frexp(x)  # x = m * 2**e with 0.5 <= |m| < 1 (e = 0 for x = 0)
        q = np.maximum(e - _BF16_SIG_BITS, _BF16_MIN_EXP_SPACING)
        # x / 2**q is exact (power-of-two scaling); np.rint rounds half to even.
        r = np.ldexp(np.rint(np.ldexp(x, -q)), q)
        r = np.where(np.abs(r) >= _BF16_OVERFLOW, np.copysign(np.inf, x), r)
        r = np.where(np.isfinite(x), r, x)  # +-inf and NaN pass through
    # r is exactly representable in bf16, hence in float32: its top 16 bits
    # are the bf16 pattern.
    bits = (r.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    return np.where(np.isnan(x), np.uint16(0x7FC0), bits).astype(np.uint16)

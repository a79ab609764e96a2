"""FP8 E4M3 ("e4m3fn") and UE8M0 codecs, written from the format definitions.

Test infrastructure only (see the package docstring).

The pages name the operand type ``torch.float8_e4m3fn`` (How to Use DeepGEMM
Weight Gradient Kernels for Training Backward Passes, "FP8 Implementation
Example") and power-of-two UE8M0 scale bytes (DeepGEMM knowledge-base index,
"UE8M0 Format in DeepGEMM").  Neither page spells out the bit layouts; they are
the standard ones:

E4M3 (OCP 8-bit floating point, "fn" variant): sign bit, 4 exponent bits with
bias 7, 3 mantissa bits.  Exponent field 0 holds subnormals ``m * 2^-9``; the
only non-finite codes are 0x7F / 0xFF (NaN); there is no infinity.  The largest
finite magnitude is 1.75 * 2^8 = 448.

UE8M0: an unsigned byte ``b`` holding the value ``2^(b - 127)``; 0xFF is NaN.
"""
import numpy as np

E4M3_MAX = 448.0
E4M3_MIN_NORMAL_EXP = -6       # smallest normal is 2^-6
E4M3_SUBNORMAL_QUANTUM = 2.0 ** -9


def e4m3_decode(codes) -> np.ndarray:
    """Value of each E4M3 code as float64 (NaN for 0x7F / 0xFF)."""
    c = np.asarray(codes, dtype=np.uint8)
    sign = np.where(c & 0x80, -1.0, 1.0)
    ef = ((c >> 3) & 0xF).astype(np.int64)
    mf = (c & 0x7).astype(np.float64)
    sub = mf * E4M3_SUBNORMAL_QUANTUM
    norm = (1.0 + mf / 8.0) * np.ldexp(1.0, ef - 7)
    v = sign * np.where(ef == 0, sub, norm)
    return np.where((c & 0x7F) == 0x7F, np.nan, v)


def e4m3_encode(y) -> np.ndarray:
    """Round each finite float64 ``y`` to the nearest E4M3 value, ties to even,
    saturating magnitudes above 448 to 448 (never producing NaN).

    Zero and values that round to zero keep their sign (0x00 / 0x80).
    """
    y = np.asarray(y, dtype=np.float64)
    neg = np.signbit(y)
    a = np.abs(y)
    # frexp: a = f * 2^p with f in [0.5, 1); unbiased exponent E = p - 1.
    _, p = np.frexp(a)
    E = p.astype(np.int64) - 1
    normal = (a >= 2.0 ** E4M3_MIN_NORMAL_EXP)
    # Normal range: mantissa step 2^(E-3); subnormal range: fixed step 2^-9.
    step_exp = np.where(normal, E - 3, -9)
    q = np.rint(np.ldexp(a, -step_exp))          # integer multiple of the step, ties-to-even
    val = np.ldexp(q, step_exp)                  # rounded magnitude (exact in float64)
    val = np.minimum(val, E4M3_MAX)
    # Re-derive the code from the rounded magnitude.
    _, p2 = np.frexp(val)
    E2 = p2.astype(np.int64) - 1
    is_norm = val >= 2.0 ** E4M3_MIN_NORMAL_EXP
    mant_norm = np.rint(np.ldexp(val, -(E2 - 3))).astype(np.int64) - 8    # 0..7
    code_norm = ((E2 + 7) << 3) | mant_norm
    code_sub = np.rint(val / E4M3_SUBNORMAL_QUANTUM).astype(np.int64)     # 0..7
    code = np.where(is_norm, code_norm, code_sub)
    code = np.where(val == 0.0, 0, code)
    return (code | np.where(neg, 0x80, 0)).astype(np.uint8)


def ue8m0_to_float(b) -> np.ndarray:
    """2^(b - 127) as float64 for each scale byte (NaN for 0xFF)."""
    b = np.asarray(b, dtype=np.int64)
    v = np.ldexp(1.0, b - 127)
    return np.where(b == 0xFF, np.nan, v)

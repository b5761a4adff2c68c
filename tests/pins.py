"""Independent statements used to pin the oracle (test code only).

Nothing here calls the oracle or the CUDA library.  These are the format's
closed form written with exact rationals, a brute-force nearest-code search,
and an exact round-to-float32 of a rational -- the "something other than
itself" each oracle function is checked against.
"""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np


def e4m3_exact(code: int):
    """Exact value of an E4M3 code as a Fraction (None for the NaN codes).

    Closed form of the OCP E4M3 format: bias 7, three mantissa bits, exponent
    field 0 is the subnormal range with step 2^-9, magnitude 0x7F is NaN.
    """
    mag = code & 0x7F
    if mag == 0x7F:
        return None
    e, m = mag >> 3, mag & 7
    if e == 0:
        v = Fraction(m, 512)
    else:
        v = Fraction(8 + m, 8) * (Fraction(2) ** (e - 7))
    return -v if code & 0x80 else v


# Positive finite codes 0x00..0x7E in increasing order of value.
POS_CODES = np.arange(0x7F, dtype=np.int64)
POS_VALUES = np.array([float(e4m3_exact(int(c))) for c in POS_CODES], dtype=np.float64)
assert np.all(np.diff(POS_VALUES) > 0)


def brute_encode(x: np.ndarray) -> np.ndarray:
    """Nearest finite E4M3 code by direct search; ties to the even code; clamp at 448.

    Works on float32 inputs.  For |x| inside [0, 448] the two candidate
    distances are exact in float64 (an 8- or 24-bit value minus a 4-bit value
    of the same or a neighbouring binade, or minus zero), so the comparison is
    exact.  NaN keeps its sign bit and maps to 0x7F; +-0 keep the sign.
    """
    x = np.asarray(x, dtype=np.float32).ravel()
    with np.errstate(invalid="ignore"):
        a = np.abs(x.astype(np.float64))
    sign = np.signbit(x).astype(np.uint8) << 7
    out = np.empty(x.size, dtype=np.uint8)
    nan = np.isnan(x)
    big = ~nan & (a >= 448.0)
    mid = ~nan & ~big
    am = a[mid]
    hi = np.searchsorted(POS_VALUES, am, side="left")  # first value >= am
    hi = np.clip(hi, 0, len(POS_VALUES) - 1)
    lo = np.clip(hi - 1, 0, len(POS_VALUES) - 1)
    d_lo = am - POS_VALUES[lo]
    d_hi = POS_VALUES[hi] - am
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (POS_CODES[hi] % 2 == 0))
    exact_hit = POS_VALUES[hi] == am
    code = np.where(exact_hit | pick_hi, POS_CODES[hi], POS_CODES[lo]).astype(np.uint8)
    out[mid] = code | sign[mid]
    out[big] = 0x7E | sign[big]
    out[nan] = 0x7F | sign[nan]
    return out


def rn_f32(v: Fraction) -> float:
    """Round an exact rational to the nearest float32 (ties to even), as a Python float.

    Handles the subnormal range (quantum 2^-149) and overflow to +-inf.
    """
    if v == 0:
        return 0.0
    neg = v < 0
    a = -v if neg else v
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    q_exp = max(e, -126) - 23
    scaled = a / (Fraction(2) ** q_exp)
    k = math.floor(scaled)
    rem = scaled - k
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and k % 2 == 1):
        k += 1
    r = Fraction(k) * (Fraction(2) ** q_exp)
    if r >= Fraction(2) ** 128:
        f = math.inf
    else:
        f = float(r)  # exact: r has at most 24 significant bits
    return -f if neg else f


def all_bf16_as_f32() -> np.ndarray:
    """All 65536 bf16 bit patterns widened (exactly) to float32."""
    bits = np.arange(1 << 16, dtype=np.uint32) << 16
    return bits.view(np.float32)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32)

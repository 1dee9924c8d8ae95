"""Oracle e4m3 quantiser (test infrastructure; see the package docstring).

The pages define no 8-bit path (they mention low-precision training only as
context: "Scaling Video Training with Parallelism", §Key claims, NVFP4).  The
e4m3 format is the published OCP 8-bit floating-point format E4M3: 1 sign
bit, 4 exponent bits with bias 7, 3 mantissa bits; exponent field 0 holds the
subnormals m * 2^-9; field 15 with mantissa 7 is NaN (no infinities), so the
largest finite magnitude is 1.75 * 2^8 = 448.

The quantiser of the e4m3 attention path is

    code = e4m3(fp32(x) * inv_scale)

(one float32 multiply rounded to nearest even, then the nearest e4m3 value,
ties to the even code, magnitudes beyond 448 saturated to 448).  Written
here from that definition, by brute force: every code is decoded once, and a
value is encoded by choosing the nearest decoded value.
"""
import numpy as np


def decode_table():
    """float64 value of each of the 256 codes (NaN for the two NaN codes)."""
    vals = np.empty(256, dtype=np.float64)
    for code in range(256):
        sign = -1.0 if code & 0x80 else 1.0
        e = (code >> 3) & 0xF
        m = code & 0x7
        if e == 0xF and m == 0x7:
            vals[code] = np.nan
        elif e == 0:
            vals[code] = sign * m * 2.0 ** -9
        else:
            vals[code] = sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return vals


_TABLE = decode_table()
_POS = _TABLE[:0x7F]           # codes 0x00 .. 0x7E: 0 .. 448, increasing


def decode(codes):
    return _TABLE[np.asarray(codes, dtype=np.uint8)]


def encode(x):
    """Nearest e4m3 code of each value of x (float), ties to the even code,
    saturating at +-448.  NaN is not expected."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), 448.0)
    hi = np.searchsorted(_POS, a, side="left")           # first code with value >= a
    hi = np.minimum(hi, 0x7E)
    lo = np.maximum(hi - 1, 0)
    d_lo, d_hi = a - _POS[lo], _POS[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    mag = np.where(pick_hi, hi, lo).astype(np.uint8)
    return np.where(np.signbit(x), mag | 0x80, mag).astype(np.uint8)


def quantize(x_bf16_as_f32, inv_scale):
    """code = e4m3(fp32(x) * inv_scale) with the product in float32."""
    prod = np.asarray(x_bf16_as_f32, dtype=np.float32) * np.float32(inv_scale)
    return encode(prod)

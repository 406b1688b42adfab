"""Oracle: FP8 E4M3 codec written from the OCP 8-bit floating-point definition.

TEST INFRASTRUCTURE (see ``oracle/__init__``): only tests, ``smoke()`` and the
CPU-baseline legs of ``bench.py`` may use it.

The FP8 cache variant ("PagedAttention" glossary, section "Các kỹ thuật liên
quan", item on FP8 cache quantisation) stores each K/V element in 8 bits. The
pages name no encoding; the reading taken is OCP E4M3 ("e4m3fn"): 1 sign bit,
4 exponent bits with bias 7, 3 mantissa bits, no infinities, and the single NaN
pattern S.1111.111 per sign. Hence:

* normal   (1 <= e <= 15, not NaN): (-1)^s * 2^(e-7) * (1 + m/8)
* subnormal (e == 0):               (-1)^s * 2^(-6)  * (m/8)
* largest finite magnitude: code 0x7E = 2^8 * 1.75 = 448.

Quantisation of a value x with a per-tensor scale (the reading for the FP8
variant): q = x / scale computed as an IEEE float32 division, then rounded to
the nearest E4M3 value, ties to the even code, with magnitudes of 448 or more
saturating to 448 ("satfinite"). The sign of the input is kept, so a negative
value that rounds to zero gives -0 (code 0x80).
"""
import numpy as np

E4M3_MAX = 448.0


def e4m3_decode(codes):
    """Exact value of each E4M3 code (uint8 array) as float64; NaN codes give nan."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    s = c >> 7
    e = (c >> 3) & 0xF
    m = c & 0x7
    sign = np.where(s == 1, -1.0, 1.0)
    normal = np.ldexp(1.0 + m / 8.0, e - 7)
    subnormal = np.ldexp(m / 8.0, -6)
    mag = np.where(e == 0, subnormal, normal)
    out = sign * mag
    return np.where((e == 15) & (m == 7), np.nan, out)


# The 127 non-negative finite magnitudes, indexed by their code 0x00..0x7E.
# They increase strictly with the code, so a code is also a rank.
_MAGNITUDES = e4m3_decode(np.arange(127, dtype=np.uint8))


def e4m3_encode(x):
    """Round float32 values to E4M3 codes: nearest, ties to even code, saturating.

    ``x`` must hold finite float32 values (NaN is not a supported input).
    """
    x32 = np.asarray(x, dtype=np.float32)
    if not np.all(np.isfinite(x32)):
        raise ValueError("e4m3_encode: non-finite input")
    a = np.abs(x32).astype(np.float64)          # exact widening
    a = np.minimum(a, E4M3_MAX)                 # satfinite: everything above 448 -> 448
    hi = np.searchsorted(_MAGNITUDES, a, side="left")   # _M[hi-1] < a <= _M[hi]
    hi = np.minimum(hi, 126)
    lo = np.maximum(hi - 1, 0)
    d_lo = a - _MAGNITUDES[lo]
    d_hi = _MAGNITUDES[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo)
    code = np.where(a == _MAGNITUDES[hi], hi, code)
    sign = np.signbit(x32).astype(np.int64) << 7
    return (code | sign).astype(np.uint8)


def e4m3_quantize(x, scale):
    """Codes for x / scale: float32 division first, then ``e4m3_encode``."""
    q = np.asarray(x, dtype=np.float32) / np.float32(scale)
    return e4m3_encode(q)

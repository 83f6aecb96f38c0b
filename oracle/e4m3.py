"""E4M3 codec written from the FP8 format definition.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

The pages quantize activations and weights to the "(4, 3) bit" FP8 format
([P1] *Logs*: ``TensorQuantizer((4, 3) bit ... per-tensor amax=...)``), i.e.
E4M3 with 4 exponent bits (bias 7) and 3 mantissa bits, the ``fn`` variant
that has no infinities and one NaN pattern per sign (S.1111.111).  Values
beyond the largest finite magnitude 448 saturate to +-448 (the static-FP8
quantizer clamps before rounding: [P2] *Verification*, ``aten::clamp``).

Reading taken where the pages are silent: a NaN input keeps its sign
(``sign | 0x7F``) so that every one of the 256 codes round-trips; a negative
value that underflows to zero encodes as negative zero (0x80).
"""

import numpy as np

E4M3_MAX = 448.0          # 1.75 * 2**8, the largest finite E4M3 magnitude
_MANT_BITS = 3
_EXP_BIAS = 7
_EMIN = 1 - _EXP_BIAS     # exponent of the smallest normal, 2**-6


def round_to_grid(a, mant_bits, emin):
    """Round non-negative float64 magnitudes ``a`` to the nearest value that
    has ``mant_bits`` fraction bits, ties to even, with gradual underflow
    below ``2**emin`` and no upper bound.

    Works for any binary floating-point format whose values are all float64
    numbers; the scaling by powers of two below is exact in float64.
    """
    a = np.asarray(a, dtype=np.float64)
    frac, ex = np.frexp(a)                       # a = frac * 2**ex, frac in [0.5, 1)
    e = np.maximum(ex.astype(np.int64) - 1, emin)  # binade exponent, clamped for subnormals
    quantum = np.ldexp(1.0, (e - mant_bits).astype(np.int32))
    return np.rint(a / quantum) * quantum        # np.rint rounds half to even


def _decode_formula(codes):
    """Exact value of each E4M3 code from the format definition."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    sub = m * 2.0 ** (_EMIN - _MANT_BITS)                       # e == 0: m * 2**-9
    nor = (1.0 + m / 8.0) * np.ldexp(1.0, (e - _EXP_BIAS).astype(np.int32))
    val = np.where(e == 0, sub, nor) * sign
    val = np.where((e == 15) & (m == 7), np.copysign(np.nan, sign), val)
    return val.astype(np.float32)


# The 256 values, each computed by the formula above; decoding a large array
# is then a table look-up of the same values.
_TABLE = _decode_formula(np.arange(256, dtype=np.uint8))


def e4m3_decode(codes):
    """Exact value of each E4M3 code as float32 (NaN for S.1111.111)."""
    return _TABLE[np.asarray(codes, dtype=np.uint8)]


def e4m3_encode(v):
    """Saturating round-to-nearest-even of float32 values to E4M3 codes."""
    v = np.asarray(v, dtype=np.float32)
    bits = v.view(np.uint32)
    sign = ((bits >> 31) & 1).astype(np.uint8) << 7
    nan = np.isnan(v)
    a = np.abs(v.astype(np.float64))
    a = np.where(nan, 0.0, np.minimum(a, 1e6))  # inf and huge values saturate below
    r = np.minimum(round_to_grid(a, _MANT_BITS, _EMIN), E4M3_MAX)
    code = np.zeros(v.shape, dtype=np.int64)
    sub = r < 2.0 ** _EMIN
    code = np.where(sub, np.rint(r / 2.0 ** (_EMIN - _MANT_BITS)), code)
    frac, ex = np.frexp(np.where(sub, 1.0, r))
    e = ex.astype(np.int64) - 1
    m = np.rint((frac * 2.0 - 1.0) * 8.0).astype(np.int64)
    code = np.where(sub, code, ((e + _EXP_BIAS) << 3) | m).astype(np.int64)
    code = code.astype(np.uint8) | sign
    code = np.where(nan, sign | 0x7F, code)
    return code.astype(np.uint8)


def e4m3_all_values():
    """All 256 codes and their decoded values (NaN for the two NaN codes)."""
    codes = np.arange(256, dtype=np.uint8)
    return codes, e4m3_decode(codes)

"""IEEE binary16 (half) rounding and decoding, written from the format
definition.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

binary16: 5 exponent bits (bias 15), 10 fraction bits, gradual underflow
below 2**-14, largest finite value 65504.  [P4] *Test Coverage*: the
two-input SwiGLU takes FP16 inputs as well as BF16.  Rounding is to nearest,
ties to even, once, from the exact value; magnitudes at or above 65520 (the
midpoint between 65504 and 2**16) become infinity.
"""

import numpy as np

from .e4m3 import round_to_grid

_F16_MANT = 10
_F16_EMIN = -14
_F16_MAX = 65504.0


def fp16_decode(bits):
    """binary16 bit patterns (uint16) -> exact float32 values."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.int64)
    sign = np.where(b & 0x8000, -1.0, 1.0)
    e = (b >> 10) & 0x1F
    m = b & 0x3FF
    sub = m * 2.0 ** (_F16_EMIN - _F16_MANT)
    nor = (1.0 + m / 1024.0) * np.ldexp(1.0, (e - 15).astype(np.int32))
    val = np.where(e == 0, sub, nor)
    val = np.where((e == 31) & (m == 0), np.inf, val)
    val = np.where((e == 31) & (m != 0), np.nan, val)
    return (val * sign).astype(np.float32)


def fp16_round(v):
    """Round float32 or float64 values once to binary16; returns uint16 bits."""
    v64 = np.asarray(v).astype(np.float64)
    nan = np.isnan(v64)
    neg = np.signbit(v64)
    a = np.abs(np.where(nan, 0.0, v64))
    inf_in = np.isinf(a)
    r = round_to_grid(np.where(inf_in, 0.0, a), _F16_MANT, _F16_EMIN)
    over = inf_in | (r > _F16_MAX)
    r = np.where(over, 0.0, r)
    frac, ex = np.frexp(r)                                   # r = frac * 2**ex
    e = np.where(r == 0, 0, ex.astype(np.int64) - 1)
    normal = r >= 2.0 ** _F16_EMIN
    m = np.where(normal, np.rint((r / np.ldexp(1.0, e.astype(np.int32)) - 1.0) * 1024.0),
                 np.rint(r / 2.0 ** (_F16_EMIN - _F16_MANT)))
    exp_field = np.where(normal, e + 15, 0)
    bits = (exp_field << 10) | m.astype(np.int64)
    bits = np.where(over, 0x7C00, bits)
    bits = bits | (neg.astype(np.int64) << 15)
    bits = np.where(nan, 0x7E00 | (neg.astype(np.int64) << 15), bits)
    return bits.astype(np.uint16)

"""bfloat16 rounding and decoding, written from the format definition.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

bf16 is the upper half of an IEEE binary32: 8 exponent bits, 7 fraction
bits.  Activations and GEMM outputs of the path are bf16 ([P2]
*Verification*; [P3] *Behavior*).  Rounding is to nearest, ties to even,
with overflow to infinity (IEEE default), applied once to the exact value.
"""

import numpy as np

from .e4m3 import round_to_grid

_BF16_MANT = 7
_BF16_EMIN = -126
_BF16_MAX = float.fromhex("0x1.fep127")     # largest finite bf16


def bf16_decode(bits):
    """bf16 bit patterns (uint16) -> exact float32 values."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32)


def bf16_round(v):
    """Round float32 or float64 values once to bf16; returns uint16 bits."""
    v = np.asarray(v)
    v64 = v.astype(np.float64)
    nan = np.isnan(v64)
    neg = np.signbit(v64)
    a = np.abs(np.where(nan, 0.0, v64))
    inf_in = np.isinf(a)
    r = round_to_grid(np.where(inf_in, 0.0, a), _BF16_MANT, _BF16_EMIN)
    # Values at or beyond the rounding threshold above the largest finite
    # bf16 become infinity, as IEEE round-to-nearest prescribes.
    r = np.where(inf_in | (r > _BF16_MAX), np.inf, r)
    r32 = np.where(neg, -r, r).astype(np.float32)
    out = (r32.view(np.uint32) >> 16).astype(np.uint16)
    out = np.where(nan, np.uint16(0x7FC0) | (neg.astype(np.uint16) << 15), out)
    return out.astype(np.uint16)

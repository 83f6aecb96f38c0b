"""Two-input SwiGLU with FP8 or bf16 output.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

[P4] *What changed*: ``swiglu_2in`` computes ``SiLU(G) * U`` from two
separate tensors and quantizes the result directly for the FP8 down
projection with that projection's static input scale.  The pages fix
neither the order of the operations nor the exponential; FP8 codes have to
agree bit for bit, so this file fixes one binary32 specification, and the
GPU kernel implements the same specification independently:

1. ``g``, ``u``: bf16 widened exactly to binary32.
2. ``p = g * u`` (exact: two 8-bit significands).
3. ``e = exp_spec(-g)``.
4. ``h = p / (1 + e)``: one binary32 addition, one correctly rounded
   binary32 division.
5. FP8 output: ``E4M3_satRNE(h / s_out)`` (one binary32 division, as in
   the static activation quantization); bf16 output: ``bf16_rne(h)``.

``exp_spec`` is a Cody-Waite range reduction (W. J. Cody and W. Waite,
*Software Manual for the Elementary Functions*, 1980) followed by the
degree-7 Taylor polynomial of ``exp`` on the reduced argument, every
operation a separately rounded binary32 multiply or add (no FMA):

* ``t`` is clamped to ``[-88, 88]``; ``t > 88`` gives ``+inf`` and
  ``t < -88`` gives ``0``.
* ``n = rint(t * L2E)`` with ``L2E = fl32(1/ln 2)`` and ties to even.
* ``r = (t - n * LN2_HI) - n * LN2_LO``; ``LN2_HI`` is ``ln 2`` with the
  low 12 significand bits of its binary32 rounding cleared (so
  ``n * LN2_HI`` is exact), ``LN2_LO = fl32(ln 2 - LN2_HI)``.
* ``q = c7; q = q*r + c_k`` for k = 6..0 with ``c_k = fl32(1/k!)``.
* ``exp_spec(t) = (q * 2**(n >> 1)) * 2**(n - (n >> 1))`` (two scalings by
  powers of two, arithmetic shift).

NaN inputs are outside the specification (``p`` is NaN and so is ``h``).

Variants ([P4] *Test Coverage*: the op is tested "for BF16 / FP16 /
swiglu_limit / swiglu_alpha+swiglu_beta / FP8 output").  The pages name the
options and no formula.  Reading (the plainest one the names support, the
clamped and shifted SwiGLU of the public gpt-oss MLP):

* FP16 inputs: ``g``, ``u`` are binary16, widened exactly; the 16-bit output
  is binary16 as well.
* ``swiglu_limit = L``: ``g = min(g, L)``, ``u = clamp(u, -L, L)`` before
  anything else (a NaN stays NaN).
* ``swiglu_alpha = a``: the sigmoid's argument is ``t = fl32(a * g)``.
* ``swiglu_beta = b``: ``u`` becomes ``fl32(u + b)``; the addition is
  omitted when ``b == 0``, so that ``-0`` keeps its sign and the defaults
  reproduce the base op bit for bit.

Then ``p = fl32(g * u)``, ``e = exp_spec(-t)``, ``h = fl32(p / fl32(1 + e))``
as above.  With ``a = 1``, ``b = 0`` and no limit, ``t = g`` and ``p`` is
the exact product, i.e. the base specification.
"""

import math

import numpy as np

from .e4m3 import e4m3_encode
from .bf16 import bf16_decode, bf16_round
from .fp16 import fp16_decode, fp16_round


def _bits_to_f32(u):
    return np.array([u], dtype=np.uint32).view(np.float32)[0]


L2E = _bits_to_f32(0x3FB8AA3B)          # fl32(1 / ln 2)
LN2_HI = _bits_to_f32(0x3F317000)       # ln 2, 12 low significand bits cleared
LN2_LO = _bits_to_f32(0x3805FDF4)       # fl32(ln 2 - LN2_HI)
TAYLOR = [np.float32(1.0 / math.factorial(k)) for k in range(8)]
T_MAX = np.float32(88.0)


def exp_spec(t):
    """The binary32 exponential of the SwiGLU specification (see module doc)."""
    t = np.asarray(t, dtype=np.float32)
    hi = t > T_MAX
    lo = t < -T_MAX
    tc = np.clip(np.where(np.isnan(t), np.float32(0), t), -T_MAX, T_MAX).astype(np.float32)
    n = np.rint(tc * L2E).astype(np.float32)
    r = (tc - n * LN2_HI) - n * LN2_LO
    q = np.full_like(r, TAYLOR[7])
    for k in range(6, -1, -1):
        q = q * r
        q = q + TAYLOR[k]
    ni = n.astype(np.int32)
    h1 = ni >> 1
    h2 = ni - h1
    res = q * np.ldexp(np.float32(1), h1).astype(np.float32)
    res = res * np.ldexp(np.float32(1), h2).astype(np.float32)
    assert res.dtype == np.float32
    res = np.where(hi, np.float32(np.inf), res)
    res = np.where(lo, np.float32(0), res)
    res = np.where(np.isnan(t), np.float32(np.nan), res)
    return res.astype(np.float32)


def swiglu_h(g_bits, u_bits):
    """``h = (g * u) / (1 + exp_spec(-g))`` in binary32 (steps 1-4)."""
    g = bf16_decode(g_bits)
    u = bf16_decode(u_bits)
    p = g * u
    e = exp_spec(-g)
    d = np.float32(1) + e
    h = p / d
    assert h.dtype == np.float32
    return h


def swiglu_2in_fp8(g_bits, u_bits, s_out):
    """FP8 output for the down projection, quantized with its static scale."""
    h = swiglu_h(g_bits, u_bits)
    return e4m3_encode(h / np.float32(s_out))


def swiglu_2in_bf16(g_bits, u_bits):
    """bf16 output, used when a 16-bit step stands the FP8 output down."""
    return bf16_round(swiglu_h(g_bits, u_bits))


def _decode16(bits, in_dtype):
    if in_dtype == "bf16":
        return bf16_decode(bits)
    if in_dtype == "fp16":
        return fp16_decode(bits)
    raise ValueError(in_dtype)


def swiglu_h_ex(g_bits, u_bits, in_dtype="bf16", limit=None, alpha=1.0, beta=0.0):
    """``h`` of the variant specification (module doc): clamp, then
    ``fl32(g * (u + b)) / fl32(1 + exp_spec(-fl32(a * g)))``."""
    g = _decode16(g_bits, in_dtype)
    u = _decode16(u_bits, in_dtype)
    if limit is not None:
        lim = np.float32(limit)
        g = np.where(g > lim, lim, g).astype(np.float32)
        u = np.where(u > lim, lim, np.where(u < -lim, -lim, u)).astype(np.float32)
    t = np.float32(alpha) * g
    v = u if beta == 0 else u + np.float32(beta)
    p = g * v
    d = np.float32(1) + exp_spec(-t)
    h = p / d
    assert h.dtype == np.float32
    return h


def swiglu_2in_ex_fp8(g_bits, u_bits, s_out, in_dtype="bf16", limit=None, alpha=1.0, beta=0.0):
    """Variant with FP8 output: ``E4M3_satRNE(fl32(h / s_out))``."""
    h = swiglu_h_ex(g_bits, u_bits, in_dtype, limit, alpha, beta)
    return e4m3_encode(h / np.float32(s_out))


def swiglu_2in_ex_16(g_bits, u_bits, in_dtype="bf16", limit=None, alpha=1.0, beta=0.0):
    """Variant with 16-bit output in the input's format (bf16 or binary16)."""
    h = swiglu_h_ex(g_bits, u_bits, in_dtype, limit, alpha, beta)
    return bf16_round(h) if in_dtype == "bf16" else fp16_round(h)

"""Static per-tensor FP8 linear: activation quantization, W8A8, W8A16, the
shared-quantization group, and the max(s) re-quantization it replaces.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Layouts follow an exported checkpoint: a weight is ``[N, K]`` row-major E4M3
(``nn.Linear.weight``) with a scalar ``weight_scale``; the activation is
``[M, K]`` row-major bf16 with a scalar ``input_scale``; there is no bias
([P1] *Logs*: ``in_features=4096, out_features=4096, bias=False``).
"""

import numpy as np

from .e4m3 import e4m3_decode, e4m3_encode
from .bf16 import bf16_decode, bf16_round


def _f32(s):
    return np.float32(s)


def quant_static(x_bits, s_in):
    """Static per-tensor activation quantization.

    [P2] *Verification*: activation quantization is ``aten::div ->
    aten::clamp -> _RoundToFloat8`` with the exported ``input_scale``.
    Reading: the bf16 activation is widened exactly to binary32, divided by
    ``s_in`` with one correctly rounded binary32 division, then rounded once
    to E4M3 with saturation at +-448 (clamp, then round to nearest even).

    x_bits: uint16 bf16 bit patterns, any shape.  Returns uint8 codes.
    """
    x = bf16_decode(x_bits)
    with np.errstate(invalid="ignore", divide="ignore", over="ignore"):
        q = x / _f32(s_in)                   # float32 / float32: IEEE division
    assert q.dtype == np.float32
    return e4m3_encode(q)


def linear_w8a8(qx, qw, s_in, s_w, rows=None):
    """W8A8 FP8 linear, the definition written out in float64.

    ``y[m, n] = s_in * s_w * sum_k dec(qx[m, k]) * dec(qw[n, k])``
    ([P2] *Verification*: ``aten::_scaled_mm`` with the two per-tensor
    scales; [P3] *Behavior*: "native ModelOpt W8A8").  Every product of two
    E4M3 values is exact in float64 and the sums of K <= 2**16 such products
    carry only float64 rounding, far below any bf16 tolerance.

    Returns ``(y64, y_bf16)``: the exact-as-possible float64 value and its
    single rounding to bf16 (uint16 bits).  ``rows`` restricts the output
    to a subset of rows (for sampled checks at full size).
    """
    qx = np.asarray(qx, dtype=np.uint8)
    if rows is not None:
        qx = qx[np.asarray(rows)]
    a = e4m3_decode(qx).astype(np.float64)
    b = e4m3_decode(qw).astype(np.float64)
    alpha = np.float64(_f32(s_in)) * np.float64(_f32(s_w))
    y64 = alpha * (a @ b.T)
    return y64, bf16_round(y64)


def dequant_weight_bf16(qw, s_w):
    """Dequantized weight of the W8A16 path.

    [P3] *Behavior*: W8A16 steps run "dequant + F.linear"; [P4]
    *Denoising-step activation precision*: the resident FP8 weight is
    dequantized with its own ``weight_scale`` and ``input_scale`` goes
    unused.  Reading: E4M3 -> bf16 is exact, the product with the binary32
    scale is formed in binary32 and rounded once to bf16 (what a bf16 tensor
    times a float32 scalar yields).  Returns uint16 bf16 bits ``[N, K]``.
    """
    w = e4m3_decode(qw) * _f32(s_w)          # float32 * float32, one rounding
    assert w.dtype == np.float32
    return bf16_round(w)


def linear_w8a16(x_bits, qw, s_w, rows=None):
    """W8A16 linear: a bf16 GEMM on the dequantized weight, float64 sums.

    ``y = x @ Wd.T`` with ``Wd = dequant_weight_bf16(qw, s_w)``; the static
    ``input_scale`` is not used ([P4] *Denoising-step activation
    precision*).  Returns ``(y64, y_bf16)`` as ``linear_w8a8``.
    """
    x_bits = np.asarray(x_bits, dtype=np.uint16)
    if rows is not None:
        x_bits = x_bits[np.asarray(rows)]
    x = bf16_decode(x_bits).astype(np.float64)
    wd = bf16_decode(dequant_weight_bf16(qw, s_w)).astype(np.float64)
    y64 = x @ wd.T
    return y64, bf16_round(y64)


def requant_onto_max_scale(qws, s_ws):
    """The fused-group re-quantization the split topology removes.

    [P4] *Description*: a per-tensor FP8 Linear holding one scale kept
    ``max(s)`` and re-quantized each member as
    ``qW_i' = FP8-round((s_i * qW_i) / max(s))``.  Reading: the product and
    the quotient are binary32 operations, the FP8 rounding is the saturating
    round-to-nearest-even of ``e4m3_encode``.

    Returns ``(list of re-quantized codes, max scale)``.
    """
    s_max = _f32(max(_f32(s) for s in s_ws))
    out = []
    for qw, s in zip(qws, s_ws):
        v = e4m3_decode(qw) * _f32(s)
        out.append(e4m3_encode(v / s_max))
    return out, s_max


def qkv_shared_quant_gemm(mode, x_bits, s_in, qws, s_ws, rows=None):
    """A projection group sharing one activation quantization.

    [P4] *What changed*: q/k/v (and gate/up) quantize the shared activation
    once and hand the same FP8 tensor to every projection, each of which
    keeps its own weight and weight scale.  [P4] *Denoising-step activation
    precision*: on a 16-bit step the sharing stands down and every
    projection runs the W8A16 path.

    mode: "A8" or "A16".  Returns a list of ``(y64, y_bf16)``.
    """
    if mode == "A8":
        qx = quant_static(x_bits if rows is None else np.asarray(x_bits)[np.asarray(rows)], s_in)
        return [linear_w8a8(qx, qw, s_in, s) for qw, s in zip(qws, s_ws)]
    if mode == "A16":
        return [linear_w8a16(x_bits, qw, s, rows=rows) for qw, s in zip(qws, s_ws)]
    raise ValueError(f"unknown mode {mode!r}")

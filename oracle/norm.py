"""The producer of a linear layer's input: a modulated LayerNorm, and the
static activation quantization fused after it.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

The pages place the static quantization right after the block's pre-attention
(and pre-MLP) norm/modulation and give that step no formula ([P2]
*Verification* shows only the ``aten::div -> aten::clamp -> _RoundToFloat8``
that follows it).  Reading taken here, the plainest one for a diffusion
transformer block: a LayerNorm without learned affine over the hidden
dimension, then a per-sample shift/scale modulation,

    mu    = (1/K) sum_k x_k
    var   = (1/K) sum_k (x_k - mu)^2            (biased, as LayerNorm)
    n_k   = (x_k - mu) / sqrt(var + eps)
    h_k   = n_k * (1 + scale_k) + shift_k

with x, shift and scale bf16 and h handed on in bf16 (the activation dtype of
the path, [P3] *Behavior*).  Rows are grouped into samples of
``rows_per_sample`` consecutive tokens; row m uses the modulation vectors of
sample ``m // rows_per_sample``.  The quantization that follows is the
path's own (``linear.quant_static``) applied to the bf16 h.

The values here are the definition written out in float64 on exactly decoded
inputs; h is rounded once to bf16.  A binary32 implementation can land on
another bf16 where the exact h lies within its rounding error of a bf16
rounding boundary (several bf16 steps away where h is small against its
terms); the tests accept the bf16 values within that error there, and only
there.
"""

import numpy as np

from .bf16 import bf16_decode, bf16_round
from .linear import quant_static


def layer_norm_stats(x_bits):
    """Per-row mean and 1/sqrt-free variance of a bf16 ``[M, K]`` activation
    in float64: returns ``(mu, var)``, each ``[M]``."""
    x = bf16_decode(x_bits).astype(np.float64)
    mu = x.mean(axis=1)
    d = x - mu[:, None]
    var = (d * d).mean(axis=1)
    return mu, var


def ln_modulate(x_bits, shift_bits, scale_bits, eps, rows_per_sample):
    """Modulated LayerNorm in float64 (the definition above).

    x_bits: uint16 bf16 ``[M, K]``; shift_bits, scale_bits: uint16 bf16
    ``[S, K]`` with ``S * rows_per_sample == M``; eps: the LayerNorm epsilon
    (a float32 value).  Returns ``(h64, mu, var)``: h in float64 ``[M, K]``
    and the per-row statistics.
    """
    x = bf16_decode(x_bits).astype(np.float64)
    M, K = x.shape
    shift = bf16_decode(shift_bits).astype(np.float64).reshape(-1, K)
    scale = bf16_decode(scale_bits).astype(np.float64).reshape(-1, K)
    T = int(rows_per_sample)
    assert T > 0 and shift.shape[0] * T == M and scale.shape == shift.shape
    mu, var = layer_norm_stats(x_bits)
    n = (x - mu[:, None]) / np.sqrt(var + np.float64(np.float32(eps)))[:, None]
    sample = np.arange(M) // T
    h = n * (1.0 + scale[sample]) + shift[sample]
    return h, mu, var


def ln_modulate_bf16(x_bits, shift_bits, scale_bits, eps, rows_per_sample):
    """h rounded once to bf16 (uint16 bits)."""
    return bf16_round(ln_modulate(x_bits, shift_bits, scale_bits, eps, rows_per_sample)[0])


def ln_modulate_quant(x_bits, shift_bits, scale_bits, eps, rows_per_sample, s_in):
    """E4M3 codes of the fused producer: the path's static quantization of
    the bf16 h.  Returns ``(q, h_bf16)``."""
    h = ln_modulate_bf16(x_bits, shift_bits, scale_bits, eps, rows_per_sample)
    return quant_static(h, s_in), h


def bf16_neighbours(h64, tol):
    """The bf16 roundings of ``h64 - tol`` and ``h64 + tol`` (uint16 bits):
    equal where every value within ``tol`` of h rounds to the same bf16;
    otherwise every bf16 between the two (inclusive) is the rounding of some
    value within ``tol``."""
    return bf16_round(h64 - tol), bf16_round(h64 + tol)


def bf16_value(bits):
    """float64 value of bf16 bit patterns."""
    return bf16_decode(bits).astype(np.float64)

"""CPU check of the fused producer's binary32 error bound (tests/norm_bound.py),
independent of the GPU: a float32 emulation of the kernel's arithmetic must
stay within the bound itself (margin 1, not the GPU test's 2) on every
element, including rows with a large common offset, outliers, small
variance against eps, and the reciprocal square root off by 2 ulps either
way.  The emulation restates the arithmetic the kernel documents; it shares
no code with the kernel."""

import numpy as np
import pytest

import oracle as O
from oracle import norm as N
from norm_bound import bound_terms
from w8a16_linear_gb300 import synth

f32 = np.float32


def _tree_sum(v):
    """Pairwise float32 sum over the last axis (depth log2 K <= 13)."""
    v = v.astype(np.float32)
    while v.shape[-1] > 1:
        if v.shape[-1] % 2:
            v = np.concatenate([v, np.zeros(v.shape[:-1] + (1,), np.float32)], axis=-1)
        v = (v[..., 0::2] + v[..., 1::2]).astype(np.float32)
    return v[..., 0]


def _fma(a, b, c):
    """fl32(a * b + c) with one rounding (the float64 product of two float32
    values is exact; the sum's float64 rounding is far below 2^-24)."""
    return (a.astype(np.float64) * b.astype(np.float64) + c.astype(np.float64)).astype(np.float32)


def _ulp_shift(v, k):
    """v moved k float32 ulps (v > 0)."""
    return (v.view(np.uint32) + np.uint32(k) if k >= 0 else v.view(np.uint32) - np.uint32(-k)).view(np.float32)


def _emulate(x, shift, scale, eps, T, rsqrt_ulps):
    xf = O.bf16_decode(x).astype(np.float32)
    M, K = xf.shape
    p = xf[:, :1]
    a = (xf - p).astype(np.float32)
    inv_k = f32(1.0) / f32(K)
    m = (_tree_sum(a) * inv_k).astype(np.float32)[:, None]
    d = (a - m).astype(np.float32)
    var = (_tree_sum((d * d).astype(np.float32)) * inv_k).astype(np.float32)
    ve = (var + f32(eps)).astype(np.float32)
    r = (1.0 / np.sqrt(ve.astype(np.float64))).astype(np.float32)   # correctly rounded 1/sqrt
    r = _ulp_shift(r, rsqrt_ulps)[:, None]
    mr = (m * r).astype(np.float32)
    n = _fma(a, np.broadcast_to(r, a.shape), np.broadcast_to(-mr, a.shape))
    smp = np.arange(M) // T
    g = (f32(1.0) + O.bf16_decode(scale).astype(np.float32)[smp]).astype(np.float32)
    h = _fma(n, g, O.bf16_decode(shift).astype(np.float32)[smp])
    return h.astype(np.float64)


@pytest.mark.parametrize("K,mean,std,eps", [(4096, 0.0, 1.0, 1e-6), (4096, -30.0, 0.25, 1e-6), (8192, 4.0, 0.5, 1e-6),
                                            (1000, 0.0, 1e-3, 1e-5), (2048, 1.0, 3.0, 0.0), (256, 0.0, 0.05, 1e-2)])
@pytest.mark.parametrize("rsqrt_ulps", [-2, 0, 2])
def test_emulation_within_bound(K, mean, std, eps, rsqrt_ulps):
    M, S = 24, 2
    x = synth.activations_bf16(31 + K, (M, K), std, outlier_frac=0.01, mean=mean)
    shift = synth.activations_bf16(32, (S, K), 0.5)
    scale = synth.activations_bf16(33, (S, K), 0.5)
    h_emul = _emulate(x, shift, scale, eps, M // S, rsqrt_ulps)
    h64, bound = bound_terms(x, shift, scale, eps, M // S)
    err = np.abs(h_emul - h64)
    assert np.all(err <= bound), float((err / bound).max())
    # and the bound is not vacuous: the emulation's worst error uses a
    # visible part of it
    assert (err / bound).max() > 1e-3


def test_emulation_rounds_like_the_oracle_mostly():
    """Away from the bound's band the emulated bf16 h is the oracle's."""
    M, K, S = 16, 4096, 1
    x = synth.activations_bf16(40, (M, K), 1.0, outlier_frac=0.001)
    shift = synth.activations_bf16(41, (S, K), 0.5)
    scale = synth.activations_bf16(42, (S, K), 0.5)
    h_emul = O.bf16_round(_emulate(x, shift, scale, 1e-6, M, 0))
    h64, bound = bound_terms(x, shift, scale, 1e-6, M)
    lo, hi = N.bf16_neighbours(h64, bound)
    settled = lo == hi
    assert np.array_equal(h_emul[settled], lo[settled])
    v = N.bf16_value(h_emul)
    assert np.all((N.bf16_value(lo) <= v) & (v <= N.bf16_value(hi)))

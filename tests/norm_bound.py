"""The binary32 error bound of the fused producer's bf16 h (shared by its
GPU parity test and the CPU check of the bound itself).

With u = 2^-24, n and r the exact normalised value and 1/sqrt(var + eps),
p = x_0 the row's first element and rho = rms(x - p) r, the kernel's
arithmetic (summation trees of depth <= 13, sums scaled by fl32(1/K),
rsqrt within 2 ulps, n = fma(a, r, -fl32(m r)), h = fma(n, fl32(1 + scale),
shift)) gives

    |h^ - h| <= [u r (|x_k - p| + 16 mean|x - p| + |m|) + u |n| (15.5 + rho)] |1 + scale|
                + u |h|

(the derivation is in tests/test_gpu_norm.py).  `window` returns the exact h
and `margin` times that bound.
"""

import numpy as np

import oracle as O
from oracle import norm as N

U = 2.0 ** -24


def bound_terms(x, shift, scale, eps, T):
    """(h64, bound) per element: the exact h and the bound above (margin 1)."""
    h64, mu, var = N.ln_modulate(x, shift, scale, eps, T)
    xf = O.bf16_decode(x).astype(np.float64)
    r = 1.0 / np.sqrt(var + float(np.float32(eps)))
    n = (xf - mu[:, None]) * r[:, None]
    smp = np.arange(x.shape[0]) // T
    sc = N.bf16_value(scale)[smp]
    xp = np.abs(xf - xf[:, :1])                  # |x_k - p|, p = the row's first element
    rho = np.sqrt((xp * xp).mean(axis=1)) * r
    m_abs = np.abs(mu - xf[:, 0])                # |m| = |mean - p|
    lead = r[:, None] * (xp + (16 * xp.mean(axis=1) + m_abs)[:, None])
    bound = U * ((lead + np.abs(n) * (15.5 + rho)[:, None]) * (1 + np.abs(sc)) + np.abs(h64))
    return h64, bound


def window(x, shift, scale, eps, T, margin=2.0):
    """Exact h and the tolerance the GPU test applies (twice the bound)."""
    h64, bound = bound_terms(x, shift, scale, eps, T)
    return h64, margin * bound

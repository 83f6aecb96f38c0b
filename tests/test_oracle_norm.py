"""Pins of the modulated-LayerNorm producer oracle (``oracle/norm.py``)
against closed forms, invariants and an independent library routine."""

import numpy as np
import torch

import oracle as O
from oracle import norm as N
from w8a16_linear_gb300 import synth


def _bits(v):
    return O.bf16_round(np.asarray(v, dtype=np.float64))


def _zeros(S, K):
    return np.zeros((S, K), dtype=np.uint16)   # bf16 +0.0


def test_constant_row_gives_shift():
    """var = 0: n = 0 whatever eps, so h is the shift vector exactly."""
    K = 64
    x = np.full((3, K), _bits(1.75), dtype=np.uint16)
    shift = synth.activations_bf16(1, (1, K), 0.5)
    scale = synth.activations_bf16(2, (1, K), 0.5)
    h64, mu, var = N.ln_modulate(x, shift, scale, 1e-6, 3)
    assert np.all(mu == 1.75) and np.all(var == 0)
    assert np.array_equal(O.bf16_round(h64), np.repeat(shift, 3, axis=0))
    q, _ = N.ln_modulate_quant(x, shift, scale, 1e-6, 3, np.float32(0.01))
    assert np.array_equal(q, O.quant_static(np.repeat(shift, 3, axis=0), np.float32(0.01)))


def test_two_value_row_closed_form():
    """Half the row at a, half at b: mu = (a+b)/2, var = ((a-b)/2)^2 and
    n = +-d / sqrt(d^2 + eps) with d = (a-b)/2 (biased variance)."""
    K, a, b, eps = 128, 3.0, -0.5, 0.25
    x = np.empty((1, K), dtype=np.uint16)
    x[0, ::2], x[0, 1::2] = _bits(a), _bits(b)
    h64, mu, var = N.ln_modulate(x, _zeros(1, K), _zeros(1, K), eps, 1)
    d = (a - b) / 2
    assert mu[0] == (a + b) / 2 and var[0] == d * d
    want = d / np.sqrt(d * d + float(np.float32(eps)))
    np.testing.assert_allclose(h64[0, ::2], want, rtol=1e-15)
    np.testing.assert_allclose(h64[0, 1::2], -want, rtol=1e-15)


def test_against_torch_layer_norm_float64():
    """With zero modulation h is LayerNorm(x) without affine: compare with
    torch's own float64 layer_norm (a routine the oracle does not call)."""
    for K, eps in ((4096, 1e-6), (1000, 1e-5), (16, 0.5)):
        x = synth.activations_bf16(3, (7, K), 0.7, outlier_frac=0.01)
        h64, _, _ = N.ln_modulate(x, _zeros(1, K), _zeros(1, K), eps, 7)
        xt = torch.from_numpy(O.bf16_decode(x).astype(np.float64))
        ref = torch.nn.functional.layer_norm(xt, (K,), eps=float(np.float32(eps))).numpy()
        np.testing.assert_allclose(h64, ref, rtol=1e-12, atol=1e-12)


def test_normalised_invariants():
    """mean(n) = 0 and mean(n^2) = var / (var + eps) on every row."""
    K, eps = 512, 1e-3
    x = synth.activations_bf16(4, (9, K), 0.05)
    h64, _, var = N.ln_modulate(x, _zeros(1, K), _zeros(1, K), eps, 9)
    np.testing.assert_allclose(h64.mean(axis=1), 0.0, atol=1e-13)
    np.testing.assert_allclose((h64 * h64).mean(axis=1), var / (var + float(np.float32(eps))), rtol=1e-12)


def test_power_of_two_rescale_invariant():
    """With eps = 0, LayerNorm(2^j x) = LayerNorm(x) (2^j x is exact in bf16)."""
    K = 256
    x = synth.activations_bf16(5, (4, K), 1.0)
    x8 = _bits(O.bf16_decode(x).astype(np.float64) * 8.0)
    h1, _, _ = N.ln_modulate(x, _zeros(1, K), _zeros(1, K), 0.0, 4)
    h8, _, _ = N.ln_modulate(x8, _zeros(1, K), _zeros(1, K), 0.0, 4)
    np.testing.assert_allclose(h1, h8, rtol=1e-14, atol=1e-14)


def test_modulation_uses_each_rows_sample():
    """Rows m use sample m // rows_per_sample: h - shift[s] = n * (1 + scale[s])
    with n from a modulation-free run; scale = -1 leaves the shift alone."""
    S, T, K = 3, 5, 64
    x = synth.activations_bf16(6, (S * T, K), 1.0)
    shift = synth.activations_bf16(7, (S, K), 0.3)
    scale = synth.activations_bf16(8, (S, K), 0.3)
    h64, _, _ = N.ln_modulate(x, shift, scale, 1e-6, T)
    n, _, _ = N.ln_modulate(x, _zeros(1, K), _zeros(1, K), 1e-6, S * T)
    for m in range(S * T):
        s = m // T
        want = n[m] * (1.0 + N.bf16_value(scale[s])) + N.bf16_value(shift[s])
        np.testing.assert_allclose(h64[m], want, rtol=1e-15, atol=1e-15)
    minus1 = np.full((S, K), _bits(-1.0), dtype=np.uint16)
    h64, _, _ = N.ln_modulate(x, shift, minus1, 1e-6, T)
    assert np.array_equal(O.bf16_round(h64), np.repeat(shift, T, axis=0))


def test_neighbours_bracket_the_rounding():
    """bf16_neighbours: equal away from a rounding boundary, the two
    adjacent bf16 values across one."""
    one_plus_half_ulp = 1.0 + 2.0 ** -8          # midpoint between 1 and 1 + 2^-7
    lo, hi = N.bf16_neighbours(np.array([1.0 + 2.0 ** -10, one_plus_half_ulp]), 2.0 ** -12)
    assert lo[0] == hi[0] == _bits(1.0)
    assert lo[1] == _bits(1.0) and hi[1] == _bits(1.0 + 2.0 ** -7)


def test_brute_force_decimal():
    """Tiny rows in 50-digit decimal arithmetic (exact mean and variance of
    the decoded bf16 values, a 50-digit square root), against the float64
    oracle."""
    from decimal import Decimal, getcontext
    getcontext().prec = 50
    M, K, S = 4, 8, 2
    x = synth.activations_bf16(50, (M, K), 1.3, mean=0.7)
    shift = synth.activations_bf16(51, (S, K), 0.5)
    scale = synth.activations_bf16(52, (S, K), 0.5)
    eps = 1e-3
    h64, _, _ = N.ln_modulate(x, shift, scale, eps, M // S)
    e = Decimal(float(np.float32(eps)))
    for m in range(M):
        xs = [Decimal(float(v)) for v in O.bf16_decode(x[m])]
        mu = sum(xs) / K
        var = sum((v - mu) ** 2 for v in xs) / K
        root = (var + e).sqrt()
        s = m // (M // S)
        for k in range(K):
            sc = Decimal(float(O.bf16_decode(scale[s, k])))
            sh = Decimal(float(O.bf16_decode(shift[s, k])))
            want = (xs[k] - mu) / root * (1 + sc) + sh
            assert abs(Decimal(float(h64[m, k])) - want) <= Decimal("1e-14") * (abs(want) + 1)

"""Pins of the oracle's SwiGLU specification: the exponential against
float64 exp, the activation against a float64 SiLU(g)*u, and the special
cases that reduce to closed forms."""

import numpy as np
import pytest
import torch

import oracle as O
from w8a16_linear_gb300 import synth


def test_exp_spec_accuracy_dense_sweep():
    t = np.linspace(-87.0, 88.0, 3_000_001).astype(np.float32)
    e = O.exp_spec(t).astype(np.float64)
    ref = np.exp(t.astype(np.float64))
    ulp = np.spacing(np.abs(ref).astype(np.float32)).astype(np.float64)
    normal = ref > 2.0 ** -126
    assert (np.abs(e - ref) / ulp)[normal].max() <= 2.0


def test_denominator_within_1p5_ulp_on_every_bf16_argument():
    """fl(1 + exp_spec(t)) against 1 + e^t for every finite bf16 t in [-88, 88]
    (the arguments the SwiGLU meets): within 1.5 * 2^-24 relative.  The fast
    FP8 SwiGLU's error budget counts on this figure."""
    bits = np.arange(1 << 16, dtype=np.uint32)
    t = (bits << 16).view(np.float32)
    t = t[np.isfinite(t) & (np.abs(t) <= 88.0)]
    d = (np.float32(1.0) + O.exp_spec(t)).astype(np.float64)
    ref = 1.0 + np.exp(t.astype(np.float64))
    assert np.max(np.abs(d / ref - 1.0)) <= 1.5 * 2.0 ** -24


def test_exp_spec_special_values():
    t = np.array([0.0, -0.0, 88.5, np.inf, -88.5, -np.inf], np.float32)
    e = O.exp_spec(t)
    assert e[0] == 1.0 and e[1] == 1.0
    assert np.isinf(e[2]) and np.isinf(e[3])
    assert e[4] == 0.0 and e[5] == 0.0


def test_swiglu_against_float64_silu():
    g = synth.random_bf16_bits(0, (200_000,))
    u = synth.activations_bf16(1, (200_000,), 1.0)
    gf, uf = O.bf16_decode(g), O.bf16_decode(u)
    ok = np.isfinite(gf) & (np.abs(gf) < 1e30) & np.isfinite(uf)
    g, u, gf, uf = g[ok], u[ok], gf[ok].astype(np.float64), uf[ok].astype(np.float64)
    with np.errstate(over="ignore"):
        ref = gf * uf / (1.0 + np.exp(-gf))
    h = O.swiglu_h(g, u).astype(np.float64)
    fin = np.isfinite(ref) & (np.abs(ref) > 2.0 ** -120) & (np.abs(ref) < 3e38)
    ulp = np.spacing(np.abs(ref[fin]).astype(np.float32)).astype(np.float64)
    assert (np.abs(h[fin] - ref[fin]) / ulp).max() <= 4.0


def test_swiglu_closed_forms():
    def bits(v):
        return torch.tensor(v, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    g = bits([0.0, 20.0, 100.0, -100.0, 30.0])
    u = bits([5.0, 1.5, -0.75, 3.0, 2.0])
    h = O.swiglu_h(g, u)
    assert h[0] == 0.0                       # silu(0) = 0
    assert h[1] == np.float32(30.0)          # exp(-20) < 2^-24: 1 + e rounds to 1
    assert h[2] == np.float32(-75.0)
    assert h[3] == 0.0                       # exp(100) = inf: p / inf
    s = np.float32(0.25)
    assert O.swiglu_2in_fp8(g, u, s)[4] == O.e4m3_encode(np.array([240.0], np.float32))[0]


def test_swiglu_fp8_codes_agree_with_float64_away_from_midpoints():
    """FP8 codes equal those of the float64 value except where that value is
    within 2^-18 (relative) of an E4M3 rounding boundary."""
    g = synth.activations_bf16(3, (300_000,), 2.0)
    u = synth.activations_bf16(4, (300_000,), 1.0)
    s = np.float32(0.01)
    gf, uf = O.bf16_decode(g).astype(np.float64), O.bf16_decode(u).astype(np.float64)
    v = gf * uf / (1.0 + np.exp(-gf)) / float(s)
    code64 = O.e4m3_encode(v.astype(np.float32))  # the float32 rounding of v is within 2^-24
    got = O.swiglu_2in_fp8(g, u, s)
    # distance of v to the nearest E4M3 decision midpoint
    codes, vals = O.e4m3_all_values()
    fv = np.sort(np.unique(np.abs(vals[~np.isnan(vals)])).astype(np.float64))
    mids = (fv[1:] + fv[:-1]) / 2
    idx = np.clip(np.searchsorted(mids, np.abs(v)), 1, len(mids) - 1)
    dist = np.minimum(np.abs(np.abs(v) - mids[idx]), np.abs(np.abs(v) - mids[idx - 1]))
    near = dist <= np.abs(v) * 2.0 ** -18
    assert np.array_equal(got[~near], code64[~near])
    assert near.mean() < 1e-3


def test_swiglu_bf16_output_is_rounded_h():
    g = synth.activations_bf16(5, (1000,), 2.0)
    u = synth.activations_bf16(6, (1000,), 1.0)
    assert np.array_equal(O.swiglu_2in_bf16(g, u), O.bf16_round(O.swiglu_h(g, u)))
    ref = torch.from_numpy(O.swiglu_h(g, u)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(O.swiglu_2in_bf16(g, u), ref)


# ---------------------------------------------------------------- variants

def _bits_with_specials(seed, n, scale):
    rng = np.random.default_rng(seed)
    v = (rng.standard_normal(n) * scale).astype(np.float32)
    v[:8] = [0.0, -0.0, np.inf, -np.inf, 1e30, -1e30, 7.0, -7.0]
    return v


def test_variant_defaults_reduce_to_the_base_specification():
    g = O.bf16_round(_bits_with_specials(1, 20000, 4.0))
    u = O.bf16_round(_bits_with_specials(2, 20000, 2.0))
    a, b = O.swiglu_h_ex(g, u), O.swiglu_h(g, u)
    assert np.array_equal(a.view(np.uint32)[~np.isnan(a)], b.view(np.uint32)[~np.isnan(b)])
    assert np.array_equal(np.isnan(a), np.isnan(b))


@pytest.mark.parametrize("in_dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("limit,alpha,beta", [(7.0, 1.702, 1.0), (None, 1.702, 0.0), (3.0, 1.0, 0.5),
                                              (None, 0.75, -1.0)])
def test_variant_against_float64_formula(in_dtype, limit, alpha, beta):
    """h against g * sigmoid(alpha g) * (u + beta) in float64 with the clamps
    written independently: relative error below 2^-19 wherever |h| is a
    normal binary32 number (argument rounding of alpha*g at |alpha g| <= 16,
    four roundings, the exponential's own 1.5 ulp)."""
    rng = np.random.default_rng(3)
    gv = (rng.standard_normal(50000) * 3.0).astype(np.float32)
    uv = (rng.standard_normal(50000) * 3.0).astype(np.float32)
    gv, uv = np.clip(gv, -9, 9), np.clip(uv, -9, 9)
    enc = O.bf16_round if in_dtype == "bf16" else O.fp16_round
    dec = O.bf16_decode if in_dtype == "bf16" else O.fp16_decode
    g, u = enc(gv), enc(uv)
    h = O.swiglu_h_ex(g, u, in_dtype, limit, alpha, beta).astype(np.float64)
    g64, u64 = dec(g).astype(np.float64), dec(u).astype(np.float64)
    if limit is not None:
        g64 = np.minimum(g64, limit)
        u64 = np.clip(u64, -limit, limit)
    ref = g64 * (u64 + beta) / (1.0 + np.exp(-alpha * g64))
    ok = np.abs(ref) > 1e-30
    assert np.max(np.abs(h[ok] / ref[ok] - 1.0)) < 2.0 ** -19


def test_variant_limit_closed_forms():
    """With a limit L every gate above L acts as L (also +inf) and up is held
    to [-L, L] (also +-inf); below the limit the clamp changes nothing."""
    L = 7.0
    g = O.bf16_round(np.array([7.0, 8.0, 1e30, np.inf, 3.0, 3.0, 3.0, 3.0], np.float32))
    u = O.bf16_round(np.array([1.0, 1.0, 1.0, 1.0, 7.0, 100.0, np.inf, -np.inf], np.float32))
    h = O.swiglu_h_ex(g, u, limit=L, alpha=1.702, beta=1.0)
    assert h[0] == h[1] == h[2] == h[3] and np.isfinite(h[0])
    assert h[4] == h[5] == h[6]
    assert h[7] == O.swiglu_h_ex(g[7:], O.bf16_round(np.float32(-7.0)).reshape(1), limit=L, alpha=1.702,
                                 beta=1.0)[0]
    # -inf gate: the clamp is one-sided, so p = -inf and d = inf: NaN
    assert np.isnan(O.swiglu_h_ex(O.bf16_round(np.float32(-np.inf)).reshape(1),
                                  O.bf16_round(np.float32(1.0)).reshape(1), limit=L)[0])


def test_variant_bf16_and_fp16_inputs_agree_where_both_represent_the_value():
    v = np.array([0.5, -1.25, 3.0, -6.5, 0.0078125, 100.0, -0.375], np.float32)
    gb, ub = O.bf16_round(v), O.bf16_round(v[::-1].copy())
    gf, uf = O.fp16_round(v), O.fp16_round(v[::-1].copy())
    for kw in ({}, {"limit": 7.0, "alpha": 1.702, "beta": 1.0}):
        hb = O.swiglu_h_ex(gb, ub, "bf16", **kw)
        hf = O.swiglu_h_ex(gf, uf, "fp16", **kw)
        assert np.array_equal(hb, hf)

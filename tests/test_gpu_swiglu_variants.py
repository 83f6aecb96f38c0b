"""GPU parity of the SwiGLU variants (swiglu_2in_ex_fp8 / swiglu_2in_ex_16:
limit, alpha, beta; bf16 or binary16 inputs) against the oracle's binary32
specification: bit-exact codes and 16-bit values."""

import numpy as np
import pytest
import torch

import oracle as O
from gpu_util import W, dev_bf16, dev_f32, host_bits, host_u8  # noqa: F401
from w8a16_linear_gb300 import synth

pytestmark = pytest.mark.gpu

PARAMS = [(7.0, 1.702, 1.0), (None, 1.702, 0.0), (3.0, 1.0, 0.5), (None, 0.75, -1.0)]


def dev16(bits, in_dtype):
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda()
    return t.view(torch.bfloat16 if in_dtype == "bf16" else torch.float16)


def _decode(bits, in_dtype):
    return O.bf16_decode(bits) if in_dtype == "bf16" else O.fp16_decode(bits)


def _fp8_equal(got, want):
    gn, wn = (got & 0x7F) == 0x7F, (want & 0x7F) == 0x7F
    assert np.array_equal(gn, wn), int(np.sum(gn != wn))
    bad = np.nonzero(got[~gn] != want[~wn])[0]
    assert bad.size == 0, (bad.size, got[~gn][bad[:5]], want[~wn][bad[:5]])


def _16_equal(got, want, in_dtype):
    gn, wn = np.isnan(_decode(got, in_dtype)), np.isnan(_decode(want, in_dtype))
    assert np.array_equal(gn, wn), int(np.sum(gn != wn))
    bad = np.nonzero(got[~gn] != want[~wn])[0]
    assert bad.size == 0, (bad.size, got[~gn][bad[:5]], want[~wn][bad[:5]])


def _all_finite_gates(in_dtype, copies):
    g = np.arange(1 << 16, dtype=np.uint16)
    g = g[np.isfinite(_decode(g, in_dtype))]
    g = np.tile(g, copies)
    n = (g.size // 16) * 16
    return g[:n].reshape(-1, 16)


def _ups(in_dtype, seed, shape, std):
    return (synth.activations_bf16(seed, shape, std) if in_dtype == "bf16"
            else synth.activations_f16(seed, shape, std))


def test_defaults_equal_the_plain_swiglu(W):
    g = _all_finite_gates("bf16", 2)
    u = _ups("bf16", 1, g.shape, 1.5)
    gd, ud = dev_bf16(g), dev_bf16(u)
    s = dev_f32(0.02)
    assert np.array_equal(host_u8(W.swiglu_2in_ex_fp8(gd, ud, s)), host_u8(W.swiglu_2in_fp8(gd, ud, s)))
    assert np.array_equal(host_bits(W.swiglu_2in_ex_16(gd, ud)), host_bits(W.swiglu_2in_bf16(gd, ud)))


@pytest.mark.parametrize("in_dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("limit,alpha,beta", PARAMS)
def test_all_gate_values(W, in_dtype, limit, alpha, beta):
    """Every finite 16-bit gate value against a spread of up values."""
    g = _all_finite_gates(in_dtype, 2)
    u = _ups(in_dtype, 2, g.shape, 3.0)
    gd, ud = dev16(g, in_dtype), dev16(u, in_dtype)
    kw = dict(limit=limit, alpha=alpha, beta=beta)
    for s in (0.02, 1.0):
        got = host_u8(W.swiglu_2in_ex_fp8(gd, ud, dev_f32(s), **kw))
        _fp8_equal(got, O.swiglu_2in_ex_fp8(g, u, np.float32(s), in_dtype, **kw))
    got16 = host_bits(W.swiglu_2in_ex_16(gd, ud, **kw))
    _16_equal(got16, O.swiglu_2in_ex_16(g, u, in_dtype, **kw), in_dtype)


def _rel_to_midpoint(v, frac_bits):
    """Relative distance of v to the nearest rounding midpoint of a format with
    `frac_bits` fraction bits (normal range)."""
    m, _ = np.frexp(np.abs(v).astype(np.float64))
    f = m * 2.0 ** (frac_bits + 1)
    return np.abs(f - np.floor(f) - 0.5) / f


@pytest.mark.parametrize("in_dtype", ["bf16", "fp16"])
def test_near_rounding_boundaries(W, in_dtype):
    """Inputs whose specified result lies within 2^-16 (FP8) / 2^-19 (16-bit)
    of a rounding midpoint of the output format: the fast value cannot settle
    them alone."""
    limit, alpha, beta = 7.0, 1.702, 1.0
    s = np.float32(0.02)
    gb = np.arange(1 << 16, dtype=np.uint16)
    gv = _decode(gb, in_dtype)
    gb = gb[np.isfinite(gv) & (np.abs(gv) <= 12.0) & (np.abs(gv) >= 2.0 ** -10)]
    ub = _ups(in_dtype, 9, (640 if in_dtype == "bf16" else 160,), 3.0)
    G, U = np.repeat(gb, ub.size), np.tile(ub, gb.size)
    h = O.swiglu_h_ex(G, U, in_dtype, limit, alpha, beta)
    q = h / s
    pick8 = (np.abs(q) >= 2.0 ** -6) & (np.abs(q) <= 400.0) & (_rel_to_midpoint(q, 3) < 2.0 ** -16)
    frac16 = 7 if in_dtype == "bf16" else 10
    pick16 = (np.abs(h) >= 2.0 ** -14) & (np.abs(h) <= 6e4) & (_rel_to_midpoint(h, frac16) < 2.0 ** -19)
    for pick, fp8 in ((pick8, True), (pick16, False)):
        Gs, Us = G[pick], U[pick]
        assert Gs.size >= 256, Gs.size
        n = (Gs.size // 16) * 16
        Gs, Us = Gs[:n].reshape(-1, 16), Us[:n].reshape(-1, 16)
        gd, ud = dev16(Gs, in_dtype), dev16(Us, in_dtype)
        kw = dict(limit=limit, alpha=alpha, beta=beta)
        if fp8:
            got = host_u8(W.swiglu_2in_ex_fp8(gd, ud, dev_f32(s), **kw))
            _fp8_equal(got, O.swiglu_2in_ex_fp8(Gs, Us, s, in_dtype, **kw))
        else:
            got = host_bits(W.swiglu_2in_ex_16(gd, ud, **kw))
            _16_equal(got, O.swiglu_2in_ex_16(Gs, Us, in_dtype, **kw), in_dtype)


@pytest.mark.parametrize("M,I", [(1, 16), (7, 16400), (333, 4096)])
def test_shapes(W, M, I):
    for in_dtype in ("bf16", "fp16"):
        g = _ups(in_dtype, 3, (M, I), 2.0)
        u = _ups(in_dtype, 4, (M, I), 1.0)
        gd, ud = dev16(g, in_dtype), dev16(u, in_dtype)
        kw = dict(limit=7.0, alpha=1.702, beta=1.0)
        got = host_u8(W.swiglu_2in_ex_fp8(gd, ud, dev_f32(0.02), **kw))
        assert np.array_equal(got, O.swiglu_2in_ex_fp8(g, u, np.float32(0.02), in_dtype, **kw))
        got16 = host_bits(W.swiglu_2in_ex_16(gd, ud, **kw))
        assert np.array_equal(got16, O.swiglu_2in_ex_16(g, u, in_dtype, **kw))


def test_zero_rows_and_refusals(W):
    e = torch.empty((0, 16), dtype=torch.float16, device="cuda")
    assert W.swiglu_2in_ex_16(e, e, limit=1.0).shape == (0, 16)
    x = torch.zeros((4, 16), dtype=torch.float16, device="cuda")
    with pytest.raises(W.W8Error) as ei:
        W.swiglu_2in_ex_16(x, x, limit=0.0)
    assert ei.value.status == 11
    with pytest.raises(W.W8Error):
        W.swiglu_2in_ex_16(x, x.to(torch.bfloat16))


def test_full_size_sampled(W):
    """20670 x 16384 binary16 inputs with the limit/alpha/beta options; sampled
    rows (and the last ones) against the oracle."""
    M, I = 20670, 16384
    gen = torch.Generator("cuda").manual_seed(0)
    gd = (torch.randn((M, I), generator=gen, device="cuda") * 2.0).to(torch.float16)
    ud = torch.randn((M, I), generator=gen, device="cuda").to(torch.float16)
    kw = dict(limit=7.0, alpha=1.702, beta=1.0)
    s = np.float32(0.02)
    out = W.swiglu_2in_ex_fp8(gd, ud, dev_f32(s), **kw)
    out16 = W.swiglu_2in_ex_16(gd, ud, **kw)
    rows = np.concatenate([synth.random_rows(6, M, 96), np.arange(M - 8, M)])
    ri = torch.from_numpy(rows).cuda()
    g, u = host_bits(gd[ri]), host_bits(ud[ri])
    assert np.array_equal(host_u8(out[ri]), O.swiglu_2in_ex_fp8(g, u, s, "fp16", **kw))
    assert np.array_equal(host_bits(out16[ri]), O.swiglu_2in_ex_16(g, u, "fp16", **kw))

"""GPU parity of swiglu_2in_fp8 / swiglu_2in_bf16 against the oracle's
binary32 specification: bit-exact codes and bf16 bits."""

import numpy as np
import pytest
import torch

import oracle as O
from gpu_util import W, dev_bf16, dev_f32, host_bits, host_u8, amax_scale  # noqa: F401
from w8a16_linear_gb300 import synth

pytestmark = pytest.mark.gpu


def _finite(bits):
    return np.isfinite(O.bf16_decode(bits))


def _bf16_equal(got, want):
    """Bit-equal, except that any NaN pattern matches any NaN pattern (inf/inf
    and 0*inf give a NaN whose payload is not specified)."""
    gn, wn = np.isnan(O.bf16_decode(got)), np.isnan(O.bf16_decode(want))
    assert np.array_equal(gn, wn), int(np.sum(gn != wn))
    bad = np.nonzero(got[~gn] != want[~wn])[0]
    assert bad.size == 0, (bad.size, got[~gn][bad[:5]], want[~wn][bad[:5]])


def _fp8_equal(got, want):
    gn, wn = (got & 0x7F) == 0x7F, (want & 0x7F) == 0x7F
    assert np.array_equal(gn, wn), int(np.sum(gn != wn))
    assert np.array_equal(got[~gn], want[~wn])


def test_swiglu_all_gate_values(W):
    """Every finite bf16 gate value against a spread of up values."""
    g = np.arange(1 << 16, dtype=np.uint16)
    g = g[_finite(g)]
    g = np.tile(g, 4)
    n = (g.size // 16) * 16
    g = g[:n]
    u = synth.activations_bf16(1, (n,), 1.5)
    g2, u2 = g.reshape(-1, 16), u.reshape(-1, 16)
    for s in [0.01, 0.5430 / 448, 1.0]:
        got = host_u8(W.swiglu_2in_fp8(dev_bf16(g2), dev_bf16(u2), dev_f32(s)))
        _fp8_equal(got, O.swiglu_2in_fp8(g2, u2, np.float32(s)))
    got16 = host_bits(W.swiglu_2in_bf16(dev_bf16(g2), dev_bf16(u2)))
    _bf16_equal(got16, O.swiglu_2in_bf16(g2, u2))


@pytest.mark.parametrize("s", [2.0 ** -20, 2.0 ** -22, 2e38])
def test_swiglu_scales_at_and_outside_the_fast_range(W, s):
    """|1/s| = 2^20 is the last scale of the fast path; 2^-22 (|1/s| > 2^20)
    and 2e38 (1/s not normal) send every element to the exact divisions."""
    g = np.arange(1 << 16, dtype=np.uint16)
    g = g[_finite(g)]
    n = (g.size // 16) * 16
    g = g[:n].reshape(-1, 16)
    u = synth.activations_bf16(2, g.shape, 1.5)
    got = host_u8(W.swiglu_2in_fp8(dev_bf16(g), dev_bf16(u), dev_f32(s)))
    _fp8_equal(got, O.swiglu_2in_fp8(g, u, np.float32(s)))


def _rel_to_e4m3_midpoint(q):
    """Relative distance of binary32 q (normal E4M3 range) to the nearest
    rounding midpoint of E4M3 (three fraction bits)."""
    m, e = np.frexp(np.abs(q).astype(np.float64))       # |q| = m * 2^e, m in [0.5, 1)
    f = m * 16.0                                        # 8..16: the grid step is 1
    return np.abs(f - np.floor(f) - 0.5) / f


def test_swiglu_near_midpoint_cases(W):
    """Pairs (g, u) whose specified h / s lies within 2^-16 (relative) of an
    E4M3 rounding midpoint: the fast value cannot settle them alone, so this
    exercises the bracket and the exact path on the cases that matter."""
    s = np.float32(0.02)
    gb = np.arange(1 << 16, dtype=np.uint16)
    gv = O.bf16_decode(gb)
    gb = gb[np.isfinite(gv) & (np.abs(gv) <= 16.0) & (np.abs(gv) >= 2.0 ** -12)]
    ub = synth.activations_bf16(9, (1024,), 3.0)
    G = np.repeat(gb, ub.size)
    U = np.tile(ub, gb.size)
    h = O.swiglu_h(G, U)
    q = h / s
    aq = np.abs(q)
    keep = (aq >= 2.0 ** -6) & (aq <= 400.0) & (_rel_to_e4m3_midpoint(q) < 2.0 ** -16)
    G, U = G[keep], U[keep]
    assert G.size >= 512, G.size
    n = (G.size // 16) * 16
    G, U = G[:n].reshape(-1, 16), U[:n].reshape(-1, 16)
    got = host_u8(W.swiglu_2in_fp8(dev_bf16(G), dev_bf16(U), dev_f32(s)))
    _fp8_equal(got, O.swiglu_2in_fp8(G, U, s))


def _rel_to_bf16_midpoint(h):
    m, _ = np.frexp(np.abs(h).astype(np.float64))
    f = m * 256.0                                       # 128..256: one bf16 step is 1
    return np.abs(f - np.floor(f) - 0.5) / f


def test_swiglu_exact_path_near_ties(W):
    """(g, u) pairs whose specified h lies within 2^-22 (relative) of a bf16
    rounding midpoint, and whose h / s lies within 2^-20 of an E4M3 one:
    only a denominator equal to the specification's, bit for bit, gives the
    specified result there (a 1-ulp error in d flips these)."""
    gb = np.arange(1 << 16, dtype=np.uint16)
    gv = O.bf16_decode(gb)
    gb = gb[np.isfinite(gv) & (np.abs(gv) <= 16.0) & (np.abs(gv) >= 2.0 ** -12)]
    ub = synth.activations_bf16(11, (2048,), 3.0)
    G, U = np.repeat(gb, ub.size), np.tile(ub, gb.size)
    h = O.swiglu_h(G, U)
    s = np.float32(0.02)
    q = h / s
    pick16 = (np.abs(h) >= 2.0 ** -100) & np.isfinite(h) & (_rel_to_bf16_midpoint(h) < 2.0 ** -22)
    pick8 = (np.abs(q) >= 2.0 ** -6) & (np.abs(q) <= 400.0) & (_rel_to_e4m3_midpoint(q) < 2.0 ** -20)
    for pick, fp8 in ((pick16, False), (pick8, True)):
        Gs, Us = G[pick], U[pick]
        assert Gs.size >= 64, Gs.size
        n = (Gs.size // 16) * 16
        Gs, Us = Gs[:n].reshape(-1, 16), Us[:n].reshape(-1, 16)
        if fp8:
            got = host_u8(W.swiglu_2in_fp8(dev_bf16(Gs), dev_bf16(Us), dev_f32(s)))
            _fp8_equal(got, O.swiglu_2in_fp8(Gs, Us, s))
        else:
            got = host_bits(W.swiglu_2in_bf16(dev_bf16(Gs), dev_bf16(Us)))
            _bf16_equal(got, O.swiglu_2in_bf16(Gs, Us))


@pytest.mark.parametrize("M,I", [(64, 256), (333, 4096), (1, 16), (7, 16400)])
def test_swiglu_shapes(W, M, I):
    g = synth.activations_bf16(3, (M, I), 2.0)
    u = synth.activations_bf16(4, (M, I), 1.0)
    s = amax_scale(O.swiglu_h(g, u)) if M * I > 0 else np.float32(1)
    got = host_u8(W.swiglu_2in_fp8(dev_bf16(g), dev_bf16(u), dev_f32(s)))
    assert np.array_equal(got, O.swiglu_2in_fp8(g, u, s))
    got16 = host_bits(W.swiglu_2in_bf16(dev_bf16(g), dev_bf16(u)))
    assert np.array_equal(got16, O.swiglu_2in_bf16(g, u))


def test_swiglu_full_size_sampled(W):
    M, I = 20670, 16384
    gd = torch.randn((M, I), generator=torch.Generator("cuda").manual_seed(0), device="cuda") * 2.0
    ud = torch.randn((M, I), generator=torch.Generator("cuda").manual_seed(1), device="cuda")
    gd, ud = gd.to(torch.bfloat16), ud.to(torch.bfloat16)
    s = np.float32(0.02)
    out = W.swiglu_2in_fp8(gd, ud, dev_f32(s))
    out16 = W.swiglu_2in_bf16(gd, ud)
    rows = np.concatenate([synth.random_rows(6, M, 128), np.arange(M - 8, M)])
    ri = torch.from_numpy(rows).cuda()
    g, u = host_bits(gd[ri]), host_bits(ud[ri])
    assert np.array_equal(host_u8(out[ri]), O.swiglu_2in_fp8(g, u, s))
    assert np.array_equal(host_bits(out16[ri]), O.swiglu_2in_bf16(g, u))

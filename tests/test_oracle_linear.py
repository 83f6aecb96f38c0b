"""Pins of the oracle's quantization, W8A8, W8A16 and max(s) re-quantization
against closed forms, exact rational brute force, torch's own ops and the
properties the pages state."""

from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle as O
from conftest import golden_lines
from w8a16_linear_gb300 import synth


def _calib():
    d = {k: float(v) for k, v in golden_lines("calibration.txt")}
    return d["input_amax"], d["weight_amax"]


# ---------------------------------------------------------------- quant_static

def test_quant_matches_torch_div_clamp_cast_exhaustive():
    """All 65,536 bf16 inputs x several scales against the chain
    div -> clamp -> round-to-float8 written with torch CPU ops."""
    ia, wa = _calib()
    bits = np.arange(1 << 16, dtype=np.uint16)
    x = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float()
    finite = torch.isfinite(x).numpy()
    for s in [ia / 448, wa / 448, 2.0 ** -10, 1.0, 0.0123, 3.7]:
        s32 = np.float32(s)
        ref = (x / torch.tensor(s32)).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        got = O.quant_static(bits, s32)
        assert np.array_equal(got[finite], ref[finite]), s


def test_quant_representable_values_exact():
    """s * dec(c) with s a power of two quantizes back to c."""
    codes, vals = O.e4m3_all_values()
    fin = ~np.isnan(vals)
    for k in [-8, -3, 0, 2]:
        s = np.float32(2.0 ** k)
        x = torch.from_numpy(vals[fin] * s).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(O.quant_static(x, s), codes[fin])


def test_quant_calibrated_amax_and_saturation():
    ia, _ = _calib()
    s = np.float32(ia / 448)
    x = torch.tensor([ia, -ia, 2 * ia, -100.0, 0.0]).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert list(O.quant_static(x, s)) == [0x7E, 0xFE, 0x7E, 0xFE, 0x00]


# ---------------------------------------------------------------- W8A8 / W8A16

def _codes_from_values(vals):
    return O.e4m3_encode(np.asarray(vals, np.float32))


def test_w8a8_selection_matrix_closed_form():
    """W = a 0/1 selection matrix (N < K, non-square): y[m, n] = s_in * s_w * x[m, pi(n)]."""
    rng = np.random.default_rng(3)
    M, K, N = 7, 48, 20
    qx = _codes_from_values(rng.choice([-2.0, -1.5, -0.5, 0.0, 0.25, 1.0, 3.0, 6.0], size=(M, K)))
    pi = rng.permutation(K)[:N]
    w = np.zeros((N, K), np.float32)
    w[np.arange(N), pi] = 1.0
    qw = _codes_from_values(w)
    s_in, s_w = np.float32(2.0 ** -2), np.float32(2.0 ** -3)
    y64, y16 = O.linear_w8a8(qx, qw, s_in, s_w)
    expect = O.e4m3_decode(qx)[:, pi].astype(np.float64) * 2.0 ** -5
    assert np.array_equal(y64, expect)
    assert np.array_equal(O.bf16_decode(y16), expect.astype(np.float32))


def test_w8a8_exact_rational_brute_force():
    """Random codes and non-power-of-two scales on a tiny non-square problem,
    checked against exact rational arithmetic."""
    rng = np.random.default_rng(4)
    M, N, K = 3, 5, 11
    qx = rng.integers(0, 256, (M, K)).astype(np.uint8)
    qw = rng.integers(0, 256, (N, K)).astype(np.uint8)
    qx[(qx & 0x7F) == 0x7F] = 0x3C       # no NaN codes
    qw[(qw & 0x7F) == 0x7F] = 0xC4
    s_in, s_w = np.float32(0.5430 / 448), np.float32(0.5039 / 448)
    y64, _ = O.linear_w8a8(qx, qw, s_in, s_w)
    dx, dw = O.e4m3_decode(qx), O.e4m3_decode(qw)
    for m in range(M):
        for n in range(N):
            acc = sum(Fraction(float(dx[m, k])) * Fraction(float(dw[n, k])) for k in range(K))
            exact = Fraction(float(s_in)) * Fraction(float(s_w)) * acc
            assert abs(Fraction(float(y64[m, n])) - exact) <= abs(exact) * Fraction(1, 2 ** 50) + Fraction(1, 2 ** 200)


def test_w8a16_dequant_power_of_two_scale_exact_and_closed_form():
    rng = np.random.default_rng(5)
    M, K, N = 6, 32, 9
    x = synth.activations_bf16(7, (M, K), 0.5)
    w = rng.standard_normal((N, K)).astype(np.float32) * 50
    qw = O.e4m3_encode(w)
    s_w = np.float32(2.0 ** -7)
    wd = O.bf16_decode(O.dequant_weight_bf16(qw, s_w))
    assert np.array_equal(wd, O.e4m3_decode(qw) * s_w)      # exact scaling
    # selection matrix: y[m, n] = x[m, pi(n)] * s_w
    pi = rng.permutation(K)[:N]
    sel = np.zeros((N, K), np.float32)
    sel[np.arange(N), pi] = 1.0
    y64, _ = O.linear_w8a16(x, O.e4m3_encode(sel), s_w)
    assert np.array_equal(y64, O.bf16_decode(x)[:, pi].astype(np.float64) * float(s_w))


def test_w8a16_dequant_rounds_product_once():
    """Non-power-of-two scale: Wd is the product rounded to binary32 then to
    bf16, compared with torch's bf16-tensor-times-float32-scalar."""
    codes, vals = O.e4m3_all_values()
    fin = ~np.isnan(vals)
    s_w = np.float32(0.5039 / 448)
    wd = O.dequant_weight_bf16(codes[fin], s_w)
    ref = (torch.from_numpy(vals[fin]).to(torch.bfloat16) * torch.tensor(s_w)).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(wd, ref)


def test_w8a16_equals_bf16_gemm_on_dequantized_weight():
    rng = np.random.default_rng(6)
    M, K, N = 16, 64, 24
    x = synth.activations_bf16(8, (M, K), 0.25)
    qw = O.e4m3_encode(rng.standard_normal((N, K)).astype(np.float32) * 100)
    s_w = np.float32(0.02 / 448 * 4)
    y64, _ = O.linear_w8a16(x, qw, s_w)
    xt = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).double()
    wt = torch.from_numpy(O.dequant_weight_bf16(qw, s_w).view(np.int16)).view(torch.bfloat16).double()
    assert np.allclose(y64, (xt @ wt.T).numpy(), rtol=1e-13, atol=1e-300)


def test_w8a8_equals_w8a16_when_both_exact():
    """x exactly s_in * dec(c) and s_w a power of two: quantization and
    dequantization are lossless, so both paths compute the same product."""
    rng = np.random.default_rng(9)
    M, K, N = 5, 40, 7
    cx = O.e4m3_encode(rng.choice([-3.0, -1.0, -0.375, 0.0, 0.5, 2.0, 12.0], size=(M, K)).astype(np.float32))
    s_in = np.float32(2.0 ** -4)
    x = torch.from_numpy(O.e4m3_decode(cx) * s_in).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    qw = O.e4m3_encode(rng.standard_normal((N, K)).astype(np.float32) * 30)
    s_w = np.float32(2.0 ** -6)
    assert np.array_equal(O.quant_static(x, s_in), cx)
    y8, _ = O.linear_w8a8(O.quant_static(x, s_in), qw, s_in, s_w)
    y16, _ = O.linear_w8a16(x, qw, s_w)
    assert np.allclose(y8, y16, rtol=1e-14, atol=0)


def test_group_a8_quantizes_once_and_a16_stands_down():
    x = synth.activations_bf16(10, (8, 32), 0.25)
    rng = np.random.default_rng(11)
    qws = [O.e4m3_encode(rng.standard_normal((16, 32)).astype(np.float32) * 40) for _ in range(3)]
    s_ws = [np.float32(0.01), np.float32(0.013), np.float32(0.02)]
    s_in = np.float32(0.004)
    outs = O.qkv_shared_quant_gemm("A8", x, s_in, qws, s_ws)
    qx = O.quant_static(x, s_in)
    for (y, _), qw, s in zip(outs, qws, s_ws):
        assert np.array_equal(y, O.linear_w8a8(qx, qw, s_in, s)[0])
    outs16 = O.qkv_shared_quant_gemm("A16", x, s_in, qws, s_ws)
    for (y, _), qw, s in zip(outs16, qws, s_ws):
        assert np.array_equal(y, O.linear_w8a16(x, qw, s)[0])
    assert not np.allclose(outs[0][0], outs16[0][0])      # the two paths differ


def test_a16_closer_to_unquantized_than_a8():
    """The 16-bit path lands closer to the unquantized reference than the
    quantized path (same weights, same scales)."""
    M, K, N = 64, 256, 128
    x = synth.activations_bf16(0, (M, K), 0.5, outlier_frac=0.001)
    w = synth.normal_f32(1, (N, K), 0.02)
    xc = synth.activations_bf16(2, (M, K), 0.5, outlier_frac=0.001)
    s_in = np.float32(np.abs(O.bf16_decode(xc)).max() / 448)
    s_w = np.float32(np.abs(w).max() / 448)
    qw = O.e4m3_encode(w / s_w)
    ref = O.bf16_decode(x).astype(np.float64) @ w.astype(np.float64).T
    y8, _ = O.linear_w8a8(O.quant_static(x, s_in), qw, s_in, s_w)
    y16, _ = O.linear_w8a16(x, qw, s_w)
    assert np.linalg.norm(y16 - ref) < np.linalg.norm(y8 - ref)


# ---------------------------------------------------------------- max(s) re-quant

def test_requant_onto_max_scale():
    """Split: each projection keeps (qW_i, s_i), so s_i * dec(qW_i) is
    reproduced exactly; fused: every member with s_i < max(s) loses codes,
    the member holding max(s) is untouched."""
    K = 4096
    qws, s_ws = [], []
    for i, c in enumerate([0.55, 1.0, 0.8]):
        w = synth.normal_f32(10 + i, (64, K), 0.02) * np.float32(c)
        s = np.float32(np.abs(w).max() / 448)
        qws.append(O.e4m3_encode(w / s))
        s_ws.append(s)
    assert len(set(float(s) for s in s_ws)) == 3          # scales genuinely differ
    fused, s_max = O.requant_onto_max_scale(qws, s_ws)
    assert s_max == max(s_ws)
    for qw, qf, s in zip(qws, fused, s_ws):
        if s == s_max:
            assert np.array_equal(qw, qf)
        else:
            assert np.mean(qw != qf) > 0.05
            # and the dequantized value moved
            assert not np.array_equal(O.e4m3_decode(qw) * s, O.e4m3_decode(qf) * s_max)


def test_requant_by_exact_half_is_lossless_above_subnormals():
    codes, vals = O.e4m3_all_values()
    fin = ~np.isnan(vals) & (np.abs(vals) >= 2.0 ** -5)
    s1, s2 = np.float32(0.25), np.float32(0.5)
    fused, _ = O.requant_onto_max_scale([codes[fin], codes[fin]], [s1, s2])
    assert np.array_equal(O.e4m3_decode(fused[0]) * s2, vals[fin] * s1)


def test_fused_requant_error_against_the_numerical_floor():
    """Context, not a target ([P4] Description: re-quantizing onto max(s)
    added error several times the numerical floor).  Reference: the float64
    product on the exact checkpoint weights s_i * dec(qW_i) with the same
    quantized activation; the split path's only error is then the bf16 output
    rounding (the floor).  The fused variant re-rounds the weights of every
    member whose scale is below max(s): its error is many times the floor,
    while the max-scale member is unchanged (ratio exactly 1)."""
    M, K, N = 256, 1024, 512
    x = synth.activations_bf16(0, (M, K), 0.25, outlier_frac=0.001)
    s_in = np.float32(np.abs(O.bf16_decode(x)).max() / 448)
    qx = O.quant_static(x, s_in)
    c = synth.uniform_f32(3, (3,), 0.5, 1.0)
    qws, s_ws = [], []
    for i in range(3):
        w = synth.normal_f32(10 + i, (N, K), 0.02) * c[i]
        s = np.float32(np.abs(w).max() / 448)
        qws.append(O.e4m3_encode(w / s))
        s_ws.append(s)
    fused, s_max = O.requant_onto_max_scale(qws, s_ws)
    ratios = []
    for q, s, qf in zip(qws, s_ws, fused):
        y64, yb = O.linear_w8a8(qx, q, s_in, s)
        _, fb = O.linear_w8a8(qx, qf, s_in, s_max)
        floor = np.linalg.norm(O.bf16_decode(yb).astype(np.float64) - y64)
        err = np.linalg.norm(O.bf16_decode(fb).astype(np.float64) - y64)
        ratios.append(err / floor)
    print("fused-requant error / floor:", [round(r, 2) for r in ratios])
    for r, s in zip(ratios, s_ws):
        if s == s_max:
            assert r == 1.0
        else:
            assert r > 3.0

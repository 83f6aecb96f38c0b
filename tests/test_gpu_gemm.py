"""GPU parity of fp8_linear_w8a8 / fp8_linear_w8a16 against the oracle:
the stated relative tolerance everywhere, bit-exact bf16 where every partial
sum is exact, sampled rows (plus the ragged tail) at full size."""

import numpy as np
import pytest
import torch

import oracle as O
from gpu_util import (W, GEMM_TOL, dev_bf16, dev_f32, dev_u8, host_bits, host_u8,  # noqa: F401
                      gemm_err, frac_rounded_equal, linear_problem)
from w8a16_linear_gb300 import synth

pytestmark = pytest.mark.gpu


def _run_both(W, x, qw, s_in, s_w):
    xd, wd = dev_bf16(x), dev_u8(qw)
    y8 = host_bits(W.fp8_linear_w8a8(xd, wd, dev_f32(s_in), dev_f32(s_w)))
    y16 = host_bits(W.fp8_linear_w8a16(xd, wd, dev_f32(s_w)))
    torch.cuda.synchronize()
    W.poll_device_error()
    return y8, y16


@pytest.mark.parametrize("M,K,N,kw", [
    (64, 256, 256, dict(x_std=0.5, outliers=0.0)),       # single static-FP8 linear, small
    (4096, 4096, 4096, {}),                               # 4096 -> 4096 linear, 4096 tokens
])
def test_linear_configs(W, M, K, N, kw):
    x, qw, s_in, s_w = linear_problem(M, K, N, **kw)
    y8, y16 = _run_both(W, x, qw, s_in, s_w)
    r8, _ = O.linear_w8a8(O.quant_static(x, s_in), qw, s_in, s_w)
    r16, _ = O.linear_w8a16(x, qw, s_w)
    e8, e16 = gemm_err(y8, r8), gemm_err(y16, r16)
    print(f"M={M} K={K} N={N}: w8a8 err {e8:.3e} eq {frac_rounded_equal(y8, r8):.4f}; "
          f"w8a16 err {e16:.3e} eq {frac_rounded_equal(y16, r16):.4f}")
    assert e8 <= GEMM_TOL and e16 <= GEMM_TOL
    assert frac_rounded_equal(y8, r8) >= 0.98 and frac_rounded_equal(y16, r16) >= 0.98


@pytest.mark.parametrize("M,K,N", [
    (1, 16, 16), (3, 48, 16), (127, 128, 256), (129, 144, 272), (200, 4112, 48),
    (333, 384, 512), (130, 64, 16 * 33),
    # ragged M, N and K against the W8A16 kernels' tiles (the fused kernel's
    # 128 weight rows x 320 tokens, the bf16 GEMM's 256 x 256)
    (1000, 256, 400), (777, 4112, 272), (385, 64, 16 * 17),
])
def test_linear_ragged_shapes(W, M, K, N):
    x, qw, s_in, s_w = linear_problem(M, K, N, seed_x=M, seed_w=N)
    y8, y16 = _run_both(W, x, qw, s_in, s_w)
    r8, _ = O.linear_w8a8(O.quant_static(x, s_in), qw, s_in, s_w)
    r16, _ = O.linear_w8a16(x, qw, s_w)
    assert gemm_err(y8, r8) <= GEMM_TOL
    assert gemm_err(y16, r16) <= GEMM_TOL


def test_pages_calibrated_scale_magnitudes(W):
    """The calibrated maxima of one 4096 -> 4096 linear on the pages
    (diffusers issue #15170, Logs: input amax 0.5430, weight amax 0.5039,
    MaxCalibrator): s_in = 0.5430 / 448 and s_w = 0.5039 / 448, with the
    activation and the weight drawn to exactly those maxima."""
    M, K, N = 512, 4096, 4096
    s_in, s_w = np.float32(0.5430 / 448), np.float32(0.5039 / 448)
    xf = synth.normal_f32(41, (M, K), 0.12)
    x = O.bf16_round(xf * np.float32(0.5430 / np.abs(xf).max()))
    wf = synth.normal_f32(42, (N, K), 0.02)
    qw = O.e4m3_encode((wf * np.float32(0.5039 / np.abs(wf).max())) / s_w)
    y8, y16 = _run_both(W, x, qw, s_in, s_w)
    r8, _ = O.linear_w8a8(O.quant_static(x, s_in), qw, s_in, s_w)
    r16, _ = O.linear_w8a16(x, qw, s_w)
    assert gemm_err(y8, r8) <= GEMM_TOL and gemm_err(y16, r16) <= GEMM_TOL
    assert frac_rounded_equal(y8, r8) >= 0.98 and frac_rounded_equal(y16, r16) >= 0.98


def test_w8a8_exact_sums_bit_exact(W):
    """Codes in {0, +-0.5, +-1, +-1.5, +-2} and power-of-two scales: every
    partial sum is a multiple of 2^-2 below 2^22, exact in any order, so the
    bf16 output must equal the oracle's bit for bit."""
    rng = np.random.default_rng(0)
    M, K, N = 300, 4096, 512
    vals = np.array([0.0, 0.5, -0.5, 1.0, -1.0, 1.5, -1.5, 2.0, -2.0], np.float32)
    qx = O.e4m3_encode(rng.choice(vals, size=(M, K)))
    qw = O.e4m3_encode(rng.choice(vals, size=(N, K)))
    s_in, s_w = np.float32(2.0 ** -3), np.float32(2.0 ** -5)
    y = host_bits(W.fp8_linear_w8a8(dev_u8(qx), dev_u8(qw), dev_f32(s_in), dev_f32(s_w)))
    _, want = O.linear_w8a8(qx, qw, s_in, s_w)
    assert np.array_equal(y, want)


@pytest.mark.parametrize("M,N", [(260, 384), (900, 400)])
def test_w8a16_exact_sums_bit_exact(W, M, N):
    rng = np.random.default_rng(1)
    K = 2048
    xv = np.array([0.0, 0.25, -0.25, 0.5, -1.0, 1.5, 2.0, -3.0], np.float32)
    x = torch.from_numpy(rng.choice(xv, size=(M, K))).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    qw = O.e4m3_encode(rng.choice(np.array([0.0, 1.0, -1.0, 2.0, -0.5, 3.0], np.float32), size=(N, K)))
    s_w = np.float32(2.0 ** -4)
    y = host_bits(W.fp8_linear_w8a16(dev_bf16(x), dev_u8(qw), dev_f32(s_w)))
    _, want = O.linear_w8a16(x, qw, s_w)
    assert np.array_equal(y, want)


def test_w8a8_e4m3_input_passthrough(W):
    """A pre-quantized activation goes straight to the GEMM and matches the
    bf16-input call that quantizes internally."""
    x, qw, s_in, s_w = linear_problem(256, 512, 256)
    xd, wd, si, sw = dev_bf16(x), dev_u8(qw), dev_f32(s_in), dev_f32(s_w)
    ws = torch.empty((256, 512), dtype=torch.uint8, device="cuda")
    y_a = W.fp8_linear_w8a8(xd, wd, si, sw, ws=ws)
    q = W.fp8_quant_static(xd, si)
    y_b = W.fp8_linear_w8a8(q, wd, si, sw)
    assert torch.equal(ws, q)
    assert torch.equal(y_a.view(torch.int16), y_b.view(torch.int16))


def test_w8a16_refuses_quantized_input(W):
    q = torch.zeros((16, 64), dtype=torch.uint8, device="cuda")
    w = torch.zeros((16, 64), dtype=torch.uint8, device="cuda")
    with pytest.raises(W.W8Error) as ei:
        W.fp8_linear_w8a16(q, w, dev_f32(1.0))
    assert ei.value.status == 5


def test_full_size_sampled_rows(W):
    """20670 tokens x 4096 -> 4096: sampled rows plus the 62-row tail tile."""
    M, K, N = 20670, 4096, 4096
    x, qw, s_in, s_w = linear_problem(M, K, N)
    y8, y16 = _run_both(W, x, qw, s_in, s_w)
    rows = np.concatenate([synth.random_rows(7, M, 256), np.arange(M - 62, M)])
    r8, _ = O.linear_w8a8(O.quant_static(x[rows], s_in), qw, s_in, s_w)
    r16, _ = O.linear_w8a16(x, qw, s_w, rows=rows)
    assert gemm_err(y8[rows], r8) <= GEMM_TOL
    assert gemm_err(y16[rows], r16) <= GEMM_TOL


def test_zero_rows(W):
    x = torch.empty((0, 256), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((256, 256), dtype=torch.uint8, device="cuda")
    assert W.fp8_linear_w8a8(x, w, dev_f32(1.0), dev_f32(1.0)).shape == (0, 256)
    assert W.fp8_linear_w8a16(x, w, dev_f32(1.0)).shape == (0, 256)


def test_scaled_mm_through_the_same_checker(W):
    """Calibration of the checker: torch's own FP8 GEMM on the same inputs,
    passed through the same metric (informational)."""
    M, K, N = 4096, 4096, 4096
    x, qw, s_in, s_w = linear_problem(M, K, N)
    qx = O.quant_static(x, s_in)
    r8, _ = O.linear_w8a8(qx, qw, s_in, s_w)
    try:
        a = dev_u8(qx).view(torch.float8_e4m3fn)
        b = dev_u8(qw).view(torch.float8_e4m3fn).t()
        y = torch._scaled_mm(a, b, scale_a=dev_f32(s_in), scale_b=dev_f32(s_w), out_dtype=torch.bfloat16)
    except Exception as e:  # noqa: BLE001
        pytest.skip(f"torch._scaled_mm unavailable: {e}")
    e_lib = gemm_err(host_bits(y), r8)
    print(f"torch._scaled_mm err {e_lib:.3e} eq {frac_rounded_equal(host_bits(y), r8):.4f}")
    assert e_lib <= GEMM_TOL

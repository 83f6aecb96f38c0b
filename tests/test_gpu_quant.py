"""GPU parity of fp8_quant_static against the oracle: bit-exact E4M3 codes."""

import numpy as np
import pytest
import torch

import oracle as O
from gpu_util import W, dev_bf16, dev_f32, host_u8, linear_problem, amax_scale  # noqa: F401
from w8a16_linear_gb300 import synth

pytestmark = pytest.mark.gpu


def _nan_ok(got, want, x_bits):
    """Codes equal; for NaN inputs any NaN code is accepted."""
    isnan = np.isnan(O.bf16_decode(x_bits))
    assert np.array_equal(got[~isnan], want[~isnan])
    assert np.all((got[isnan] & 0x7F) == 0x7F)


@pytest.mark.parametrize("s", [0.5430 / 448, 0.5039 / 448, 2.0 ** -10, 1.0, 0.0123, 3.7, 1e-30, 2e38,
                               2.0 ** 125, 2.0 ** 126, 2.0 ** -126, 6e37, 3e37])
def test_quant_exhaustive_bf16(W, s):
    bits = np.arange(1 << 16, dtype=np.uint16).reshape(4096, 16)
    got = host_u8(W.fp8_quant_static(dev_bf16(bits), dev_f32(s)))
    _nan_ok(got, O.quant_static(bits, np.float32(s)), bits)


@pytest.mark.parametrize("M,K", [(64, 256), (4096, 4096), (1, 16), (3, 48), (129, 272), (1000, 4112)])
def test_quant_shapes(W, M, K):
    x, _, s_in, _ = linear_problem(M, K, 16)
    got = host_u8(W.fp8_quant_static(dev_bf16(x), dev_f32(s_in)))
    assert np.array_equal(got, O.quant_static(x, s_in))


def test_quant_full_size_sampled(W):
    M, K = 20670, 4096
    x, _, s_in, _ = linear_problem(M, K, 16)
    got = host_u8(W.fp8_quant_static(dev_bf16(x), dev_f32(s_in)))
    rows = np.concatenate([synth.random_rows(5, M, 512), np.arange(M - 62, M)])
    assert np.array_equal(got[rows], O.quant_static(x[rows], s_in))


def test_quant_saturates_on_the_live_batch(W):
    """With a static scale calibrated on another batch, live values beyond
    448 s_in saturate to +-448 (codes 0x7E / 0xFE) instead of overflowing:
    here the scale is half the live batch's amax/448, so every outlier above
    half the amax saturates.  The rows holding them are checked bit for bit."""
    M, K = 4096, 4096
    x, _, _, _ = linear_problem(M, K, 16, seed_x=21)
    xv = np.abs(O.bf16_decode(x).astype(np.float64))
    s_sat = np.float32(xv.max() / 448 / 2)
    got = host_u8(W.fp8_quant_static(dev_bf16(x), dev_f32(s_sat)))
    sat_rows = np.unique(np.nonzero(xv > 448.0 * float(s_sat))[0])
    assert sat_rows.size > 0
    assert np.any(got[sat_rows] == 0x7E) and np.any(got[sat_rows] == 0xFE)
    rows = np.unique(np.concatenate([sat_rows[:256], synth.random_rows(6, M, 64)]))
    assert np.array_equal(got[rows], O.quant_static(x[rows], s_sat))


def test_quant_refuses_strided_rows(W):
    """A view whose rows are not dense reaches the library with its real row
    pitch and is refused (W8_ERR_STRIDE), not quantized with the wrong pitch."""
    x = torch.zeros((64, 512), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(W.W8Error) as ei:
        W.fp8_quant_static(x[:, :256], dev_f32(1.0))
    assert ei.value.status == 4
    out = torch.empty((64, 512), dtype=torch.uint8, device="cuda")
    with pytest.raises(W.W8Error) as ei:
        W.fp8_quant_static(x[:, :256], dev_f32(1.0), out=out[:, :256])
    assert ei.value.status == 4


def test_quant_zero_rows(W):
    x = torch.empty((0, 256), dtype=torch.bfloat16, device="cuda")
    assert W.fp8_quant_static(x, dev_f32(1.0)).shape == (0, 256)

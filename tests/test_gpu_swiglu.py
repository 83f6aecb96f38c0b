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

"""Seeded random shapes across every GEMM mode of the path: ragged M (1 ..
3000), K and N / I multiples of 16 that are rarely multiples of the tile
sizes.  W8A8 and both W8A16 forms against the oracle on sampled rows; the
fused gate/up + SwiGLU kernels (E4M3 and bf16 out) bit for bit against their
separate paths; the elementwise kernels bit for bit against the oracle."""

import numpy as np
import pytest
import torch

import oracle as O
from gpu_util import W, GEMM_TOL, dev_bf16, dev_f32, dev_u8, host_bits, host_u8, gemm_err, linear_problem  # noqa: F401
from w8a16_linear_gb300 import synth

pytestmark = pytest.mark.gpu

_rng = np.random.default_rng(2024)
SHAPES = [(int(_rng.integers(1, 3000)), 16 * int(_rng.integers(1, 129)), 16 * int(_rng.integers(1, 129)))
          for _ in range(12)]


@pytest.mark.parametrize("M,K,N", SHAPES)
def test_random_linear(W, M, K, N):
    x, qw, s_in, s_w = linear_problem(M, K, N, seed_x=M, seed_w=K + N)
    xd, wd = dev_bf16(x), dev_u8(qw)
    y8 = host_bits(W.fp8_linear_w8a8(xd, wd, dev_f32(s_in), dev_f32(s_w)))
    y16 = host_bits(W.fp8_linear_w8a16(xd, wd, dev_f32(s_w)))
    y16w = host_bits(W.qkv_shared_quant_gemm(W.MODE_A16, xd, None, [wd], [dev_f32(s_w)],
                                             ws=W.w8a16_workspace([wd]))[0])
    torch.cuda.synchronize()
    W.poll_device_error()
    rows = np.unique(np.concatenate([synth.random_rows(M, M, min(M, 48)), np.arange(max(0, M - 3), M)]))
    r8, _ = O.linear_w8a8(O.quant_static(x[rows], s_in), qw, s_in, s_w)
    r16, _ = O.linear_w8a16(x, qw, s_w, rows=rows)
    assert gemm_err(y8[rows], r8) <= GEMM_TOL
    assert gemm_err(y16[rows], r16) <= GEMM_TOL
    assert gemm_err(y16w[rows], r16) <= GEMM_TOL


@pytest.mark.parametrize("M,K,I", [(m, k, n) for m, k, n in SHAPES[:6]])
def test_random_gate_up_swiglu(W, M, K, I):
    gen = torch.Generator(device="cuda").manual_seed(M * 7 + I)
    x = (torch.randn((M, K), generator=gen, device="cuda") * 0.25).to(torch.bfloat16)

    def weight():
        w = torch.randn((I, K), generator=gen, device="cuda") * 0.02
        sc = (w.abs().amax() / 448).reshape(1).contiguous()
        return (w / sc).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).contiguous(), sc
    (wg, sg), (wu, su) = weight(), weight()
    s_x = (x.float().abs().amax() / 448).reshape(1).contiguous()
    s_h = dev_f32(0.02)
    # W8A8 step: fused vs group GEMM + swiglu_2in_fp8
    h = W.gate_up_swiglu_fp8(x, s_x, wg, wu, sg, su, s_h)
    g, u = W.qkv_shared_quant_gemm(W.MODE_A8, x, s_x, [wg, wu], [sg, su])
    assert torch.equal(h, W.swiglu_2in_fp8(g, u, s_h))
    # W8A16 step: fused bf16 vs bf16 group GEMM + swiglu_2in_bf16
    dg, du = W.fp8_dequant_weight(wg, sg), W.fp8_dequant_weight(wu, su)
    h16 = W.bf16_gate_up_swiglu(x, dg, du)
    g16, u16 = W.bf16_linear_group(x, [dg, du])
    assert torch.equal(h16.view(torch.int16), W.swiglu_2in_bf16(g16, u16).view(torch.int16))
    torch.cuda.synchronize()
    W.poll_device_error()


@pytest.mark.parametrize("M,K,N", SHAPES[:6])
def test_random_elementwise(W, M, K, N):
    x = synth.activations_bf16(M + K, (M, K), 0.25, outlier_frac=0.001)
    s = np.float32(0.25 * 4 / 448)
    assert np.array_equal(host_u8(W.fp8_quant_static(dev_bf16(x), dev_f32(s))), O.quant_static(x, s))
    g = synth.activations_bf16(N, (M, N), 2.0)
    u = synth.activations_bf16(N + 1, (M, N), 1.0)
    gd, ud = dev_bf16(g), dev_bf16(u)
    assert np.array_equal(host_u8(W.swiglu_2in_fp8(gd, ud, dev_f32(0.02))), O.swiglu_2in_fp8(g, u, np.float32(0.02)))
    assert np.array_equal(host_bits(W.swiglu_2in_bf16(gd, ud)), O.swiglu_2in_bf16(g, u))

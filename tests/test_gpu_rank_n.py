"""Rank-N activations (the op contract tested in TensorRT-LLM PR #17476,
Test Coverage): every entry point takes [..., K] and returns [..., N]; the
binding flattens the leading dimensions, so the results equal the 2-D call
bit for bit."""

import pytest
import torch

from gpu_util import W  # noqa: F401

pytestmark = pytest.mark.gpu

M, K, N, I = 600, 512, 256, 512


def _eq(a, b):
    return a.shape == b.shape and torch.equal(a.reshape(-1).view(torch.uint8), b.reshape(-1).view(torch.uint8))


def test_rank3_equals_rank2(W):
    g = torch.Generator(device="cuda").manual_seed(5)
    x2 = (torch.randn((M, K), generator=g, device="cuda") * 0.25).to(torch.bfloat16)
    x3 = x2.view(2, M // 2, K)
    ws = [(torch.randn((N, K), generator=g, device="cuda") * 200).clamp(-448, 448)
          .to(torch.float8_e4m3fn).view(torch.uint8) for _ in range(3)]
    wg = [(torch.randn((I, K), generator=g, device="cuda") * 200).clamp(-448, 448)
          .to(torch.float8_e4m3fn).view(torch.uint8) for _ in range(2)]
    ss = [torch.tensor([0.02 * (i + 1) / 448], device="cuda") for i in range(3)]
    s_in = torch.tensor([1.0 / 448], device="cuda")
    s_o = torch.tensor([0.01], device="cuda")
    sh, sc = ((torch.randn((2, K), generator=g, device="cuda") * 0.5).to(torch.bfloat16) for _ in range(2))
    gu2 = (torch.randn((M, I), generator=g, device="cuda") * 2).to(torch.bfloat16)
    uu2 = torch.randn((M, I), generator=g, device="cuda").to(torch.bfloat16)

    cases = [
        (lambda x: W.fp8_quant_static(x, s_in), K),
        (lambda x: W.fp8_linear_w8a8(x, ws[0], s_in, ss[0]), N),
        (lambda x: W.fp8_linear_w8a16(x, ws[0], ss[0]), N),
        (lambda x: W.qkv_shared_quant_gemm(W.MODE_A8, x, s_in, ws, ss)[2], N),
        (lambda x: W.qkv_shared_quant_gemm(W.MODE_A16, x, None, ws, ss)[1], N),
        (lambda x: W.gate_up_swiglu_fp8(x, s_in, wg[0], wg[1], ss[0], ss[1], s_o), I),
        (lambda x: W.ln_modulate_quant(x, sh, sc, s_in), K),
    ]
    for fn, n_out in cases:
        a, b = fn(x2), fn(x3)
        torch.cuda.synchronize()
        assert b.shape == (2, M // 2, n_out)
        assert _eq(a.reshape(b.shape), b)
    for fn in (lambda g_, u_: W.swiglu_2in_fp8(g_, u_, s_o), lambda g_, u_: W.swiglu_2in_bf16(g_, u_)):
        a, b = fn(gu2, uu2), fn(gu2.view(2, M // 2, I), uu2.view(2, M // 2, I))
        torch.cuda.synchronize()
        assert b.shape == (2, M // 2, I) and _eq(a.reshape(b.shape), b)
    W.poll_device_error()

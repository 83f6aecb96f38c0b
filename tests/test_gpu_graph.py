"""The path's entry points only enqueue work on the caller's stream, so a
whole W8A8 block (shared-quant Q/K/V group, out-projection, fused gate/up +
SwiGLU, down projection), a W8A16 block (fused, and through the
dequantization workspace), the fused gate/up GEMMs with the SwiGLU options
and the input producer (modulated LayerNorm with the quantization fused)
can be captured in a CUDA graph;
replaying the graph reproduces the eager results bit for bit."""

import numpy as np
import pytest
import torch

from gpu_util import W, dev_f32  # noqa: F401

pytestmark = pytest.mark.gpu


def _weights(gen, n, k):
    w = torch.randn((n, k), generator=gen, device="cuda") * 0.02
    s = (w.abs().amax() / 448).reshape(1).contiguous()
    return (w / s).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).contiguous(), s


def test_block_in_cuda_graph(W):
    M, H, I = 1000, 512, 1024
    gen = torch.Generator(device="cuda").manual_seed(2)
    x = (torch.randn((M, H), generator=gen, device="cuda") * 0.25).to(torch.bfloat16)
    s_in = (x.float().abs().amax() / 448).reshape(1).contiguous()
    wq = [_weights(gen, H, H) for _ in range(3)]
    wo = _weights(gen, H, H)
    wg, wu = _weights(gen, I, H), _weights(gen, I, H)
    wd = _weights(gen, H, I)
    s_h = dev_f32(0.01)
    bf = dict(dtype=torch.bfloat16, device="cuda")
    outs = {
        "qkv": [torch.empty((M, H), **bf) for _ in range(3)],
        "o": torch.empty((M, H), **bf),
        "h8": torch.empty((M, I), dtype=torch.uint8, device="cuda"),
        "y8": torch.empty((M, H), **bf),
        "qkv16": [torch.empty((M, H), **bf) for _ in range(3)],
        "gu16": [torch.empty((M, I), **bf) for _ in range(2)],
        "h16": torch.empty((M, I), **bf),
        "y16": torch.empty((M, H), **bf),
        "qkv16w": [torch.empty((M, H), **bf) for _ in range(3)],
        "y16w": torch.empty((M, H), **bf),
        "h16f": torch.empty((M, I), **bf),
        "h8x": torch.empty((M, I), dtype=torch.uint8, device="cuda"),
        "h16x": torch.empty((M, I), **bf),
        "qn": torch.empty((M, H), dtype=torch.uint8, device="cuda"),
        "hn": torch.empty((M, H), **bf),
    }
    mod = [(torch.randn((2, H), generator=gen, device="cuda") * 0.5).to(torch.bfloat16) for _ in range(2)]
    wdg, wdu = W.fp8_dequant_weight(wg[0], wg[1]), W.fp8_dequant_weight(wu[0], wu[1])
    wsd = W.w8a16_workspace([wg[0], wu[0]])
    ws = torch.empty((M, H), dtype=torch.uint8, device="cuda")
    ws2 = torch.empty((M, H), dtype=torch.uint8, device="cuda")

    def block():
        W.qkv_shared_quant_gemm(W.MODE_A8, x, s_in, [q for q, _ in wq], [s for _, s in wq], outs=outs["qkv"], ws=ws)
        W.fp8_linear_w8a8(x, wo[0], s_in, wo[1], out=outs["o"], ws=ws2)
        W.gate_up_swiglu_fp8(x, s_in, wg[0], wu[0], wg[1], wu[1], s_h, out=outs["h8"], ws=ws)
        W.fp8_linear_w8a8(outs["h8"], wd[0], s_h, wd[1], out=outs["y8"])
        W.qkv_shared_quant_gemm(W.MODE_A16, x, None, [q for q, _ in wq], [s for _, s in wq], outs=outs["qkv16"])
        W.qkv_shared_quant_gemm(W.MODE_A16, x, None, [wg[0], wu[0]], [wg[1], wu[1]], outs=outs["gu16"])
        W.swiglu_2in_bf16(outs["gu16"][0], outs["gu16"][1], out=outs["h16"])
        W.fp8_linear_w8a16(outs["h16"], wd[0], wd[1], out=outs["y16"])
        # W8A16 through the workspace (dequantization + bf16 group GEMM)
        W.qkv_shared_quant_gemm(W.MODE_A16, x, None, [q for q, _ in wq], [s for _, s in wq], outs=outs["qkv16w"],
                                ws=wsd)
        W.qkv_shared_quant_gemm(W.MODE_A16, outs["h16"], None, [wd[0]], [wd[1]], outs=[outs["y16w"]], ws=wsd)
        W.bf16_gate_up_swiglu(x, wdg, wdu, out=outs["h16f"])
        # the fused gate/up with the SwiGLU options, both forms
        W.gate_up_swiglu_fp8(x, s_in, wg[0], wu[0], wg[1], wu[1], s_h, out=outs["h8x"], ws=ws,
                             limit=7.0, alpha=1.702, beta=1.0)
        W.bf16_gate_up_swiglu(x, wdg, wdu, out=outs["h16x"], limit=3.0, alpha=1.0, beta=0.5)
        # the input producer with the quantization fused (two samples of 500 rows)
        W.ln_modulate_quant(x, mod[0], mod[1], s_in, out=outs["qn"], h_out=outs["hn"])

    def snapshot():
        flat = []
        for v in outs.values():
            flat += v if isinstance(v, list) else [v]
        return [t.clone() for t in flat]

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        block()                                  # eager, also initialises every entry point
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    eager = snapshot()
    for v in outs.values():
        for t in (v if isinstance(v, list) else [v]):
            t.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        block()
    graph.replay()
    torch.cuda.synchronize()
    W.poll_device_error()
    for a, b in zip(eager, snapshot()):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))

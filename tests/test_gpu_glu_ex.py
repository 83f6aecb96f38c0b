"""GPU parity of the fused gate/up GEMMs with the SwiGLU options in their
epilogue (gate_up_swiglu_ex_fp8, bf16_gate_up_swiglu_ex; TensorRT-LLM PR
#17476, section Test Coverage: swiglu_limit, swiglu_alpha + swiglu_beta):
the same outputs as the separate path (group GEMM -> bf16 gate and up ->
swiglu_2in_ex_fp8 / swiglu_2in_ex_16), the plain options equal to the plain
fused calls, and the codes equal to the oracle's SwiGLU with options on the
kernel's own bf16 gate and up values."""

import numpy as np
import pytest
import torch

import oracle as O
from gpu_util import W, dev_bf16, dev_f32, dev_u8, host_bits, host_u8, amax_scale  # noqa: F401
from w8a16_linear_gb300 import synth

pytestmark = pytest.mark.gpu

OPTIONS = [dict(limit=7.0, alpha=1.702, beta=1.0), dict(limit=None, alpha=1.702, beta=0.0),
           dict(limit=3.0, alpha=1.0, beta=0.5), dict(limit=None, alpha=0.75, beta=-1.0)]


def _problem(M, K, I, seed=0):
    x = synth.activations_bf16(seed, (M, K), 0.25, outlier_frac=0.001)
    xc = synth.activations_bf16(seed + 1, (min(M, 2048), K), 0.25, outlier_frac=0.001)
    s_in = amax_scale(O.bf16_decode(xc))
    ws, ss = [], []
    for i, c in enumerate((0.7, 1.0)):
        w = synth.normal_f32(seed + 10 + i, (I, K), 0.02) * np.float32(c)
        s = amax_scale(w)
        ws.append(O.e4m3_encode(w / s))
        ss.append(s)
    return x, s_in, ws, ss


def _s_out(g, u, kw):
    """The down projection's input scale, calibrated on this batch: amax / 448
    of the oracle's SwiGLU with the options on the GPU's bf16 gate and up."""
    h = O.swiglu_h_ex(host_bits(g), host_bits(u), "bf16", **kw)
    h = h[np.isfinite(h)]
    return dev_f32(amax_scale(h) if h.size and np.max(np.abs(h)) > 0 else 1.0)


@pytest.mark.parametrize("kw", OPTIONS)
@pytest.mark.parametrize("M,K,I", [(64, 256, 256), (1, 16, 16), (129, 144, 272), (300, 512, 1024),
                                   (2048, 4096, 4096)])
def test_fp8_fused_options_equal_separate_path(W, M, K, I, kw):
    x, s_in, ws, ss = _problem(M, K, I, seed=M + I)
    xd, si = dev_bf16(x), dev_f32(s_in)
    wd, sd = [dev_u8(w) for w in ws], [dev_f32(s) for s in ss]
    g, u = W.qkv_shared_quant_gemm(W.MODE_A8, xd, si, wd, sd)
    s_out = _s_out(g, u, kw)
    sep = W.swiglu_2in_ex_fp8(g, u, s_out, **kw)
    fused = W.gate_up_swiglu_fp8(xd, si, wd[0], wd[1], sd[0], sd[1], s_out, **kw)
    torch.cuda.synchronize()
    W.poll_device_error()
    assert torch.equal(fused, sep)
    if M * I <= 300 * 1024:
        assert np.array_equal(host_u8(fused), O.swiglu_2in_ex_fp8(host_bits(g), host_bits(u),
                                                                 np.float32(s_out.item()), "bf16", **kw))


@pytest.mark.parametrize("kw", OPTIONS)
@pytest.mark.parametrize("M,K,I", [(64, 256, 256), (129, 144, 272), (300, 512, 1024), (1024, 4096, 4096)])
def test_bf16_fused_options_equal_separate_path(W, M, K, I, kw):
    x, _, ws, ss = _problem(M, K, I, seed=3 * M + I)
    xd = dev_bf16(x)
    wdg, wdu = (W.fp8_dequant_weight(dev_u8(w), dev_f32(s)) for w, s in zip(ws, ss))
    g, u = W.bf16_linear_group(xd, [wdg, wdu])
    sep = W.swiglu_2in_ex_16(g, u, **kw)
    fused = W.bf16_gate_up_swiglu(xd, wdg, wdu, **kw)
    torch.cuda.synchronize()
    W.poll_device_error()
    assert torch.equal(fused.view(torch.int16), sep.view(torch.int16))
    if M * I <= 300 * 1024:
        assert np.array_equal(host_bits(fused), O.swiglu_2in_ex_16(host_bits(g), host_bits(u), "bf16", **kw))


def test_plain_options_equal_plain_fused_calls(W):
    """{no limit, alpha 1, beta 0} through the options entries gives the plain
    entries' outputs bit for bit."""
    M, K, I = 777, 1024, 2048
    x, s_in, ws, ss = _problem(M, K, I, seed=5)
    xd, si = dev_bf16(x), dev_f32(s_in)
    wd, sd = [dev_u8(w) for w in ws], [dev_f32(s) for s in ss]
    s_out = dev_f32(0.02)
    plain = W.gate_up_swiglu_fp8(xd, si, wd[0], wd[1], sd[0], sd[1], s_out)
    opt = W.gate_up_swiglu_fp8(xd, si, wd[0], wd[1], sd[0], sd[1], s_out, alpha=1.0)
    wdg, wdu = (W.fp8_dequant_weight(w, s) for w, s in zip(wd, sd))
    plain16 = W.bf16_gate_up_swiglu(xd, wdg, wdu)
    opt16 = W.bf16_gate_up_swiglu(xd, wdg, wdu, beta=0.0)
    torch.cuda.synchronize()
    assert torch.equal(plain, opt)
    assert torch.equal(plain16.view(torch.int16), opt16.view(torch.int16))


def test_full_size_gate_up_with_limit(W):
    """The bench's gated-MLP shape at 8192 tokens (20670 x 4096 -> 2 x 16384
    cut to 8192 rows) with the clamp: fused = separate, and sampled rows plus
    the last ones against the oracle."""
    M, K, I = 8192, 4096, 16384
    kw = OPTIONS[0]
    x, s_in, ws, ss = _problem(M, K, I, seed=11)
    xd, si = dev_bf16(x), dev_f32(s_in)
    wd, sd = [dev_u8(w) for w in ws], [dev_f32(s) for s in ss]
    g, u = W.qkv_shared_quant_gemm(W.MODE_A8, xd, si, wd, sd)
    rows = np.concatenate([synth.random_rows(12, M - 40, 96), np.arange(M - 40, M)])
    s_out = _s_out(g[rows], u[rows], kw)
    sep = W.swiglu_2in_ex_fp8(g, u, s_out, **kw)
    fused = W.gate_up_swiglu_fp8(xd, si, wd[0], wd[1], sd[0], sd[1], s_out, **kw)
    torch.cuda.synchronize()
    W.poll_device_error()
    assert torch.equal(fused, sep)
    assert np.array_equal(host_u8(fused[rows]), O.swiglu_2in_ex_fp8(host_bits(g[rows]), host_bits(u[rows]),
                                                                    np.float32(s_out.item()), "bf16", **kw))

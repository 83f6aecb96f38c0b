"""GPU parity of gate_up_swiglu_fp8, the fused gate/up GEMMs with the SwiGLU
epilogue: the same E4M3 codes as the separate path (group GEMM -> bf16 gate
and up -> swiglu_2in_fp8), bit-exact against the oracle where every partial
sum is exact, and against the oracle chain elsewhere."""

import numpy as np
import pytest
import torch

import oracle as O
from gpu_util import (W, dev_bf16, dev_f32, dev_u8, host_bits, host_u8, amax_scale,  # noqa: F401
                      abs_product_sums, accumulation_window, assert_swiglu_consistent)
from w8a16_linear_gb300 import synth

pytestmark = pytest.mark.gpu


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


@pytest.mark.parametrize("M,K,I", [(64, 256, 256), (1, 16, 16), (129, 144, 272), (300, 512, 1024),
                                   (2048, 4096, 4096)])
def test_fused_equals_separate_path(W, M, K, I):
    x, s_in, ws, ss = _problem(M, K, I, seed=M)
    xd, si = dev_bf16(x), dev_f32(s_in)
    wd, sd = [dev_u8(w) for w in ws], [dev_f32(s) for s in ss]
    # calibrate the down projection's input scale on this batch's SwiGLU output
    g, u = W.qkv_shared_quant_gemm(W.MODE_A8, xd, si, wd, sd)
    h = O.swiglu_h(host_bits(g), host_bits(u))
    s_out = dev_f32(amax_scale(h) if h.size else 1.0)
    sep = W.swiglu_2in_fp8(g, u, s_out)
    fused = W.gate_up_swiglu_fp8(xd, si, wd[0], wd[1], sd[0], sd[1], s_out)
    torch.cuda.synchronize()
    W.poll_device_error()
    assert torch.equal(fused, sep)


def test_fused_exact_sums_bit_exact_vs_oracle(W):
    rng = np.random.default_rng(3)
    M, K, I = 300, 2048, 512
    vals = np.array([0.0, 0.5, -0.5, 1.0, -1.0, 1.5, -2.0], np.float32)
    qx = O.e4m3_encode(rng.choice(vals, size=(M, K)))
    wg = O.e4m3_encode(rng.choice(vals, size=(I, K)))
    wu = O.e4m3_encode(rng.choice(vals, size=(I, K)))
    s_in, s_g, s_u, s_out = (np.float32(2.0 ** -3), np.float32(2.0 ** -5), np.float32(2.0 ** -4),
                             np.float32(0.0123))
    out = W.gate_up_swiglu_fp8(dev_u8(qx), dev_f32(s_in), dev_u8(wg), dev_u8(wu), dev_f32(s_g),
                               dev_f32(s_u), dev_f32(s_out))
    _, gb = O.linear_w8a8(qx, wg, s_in, s_g)
    _, ub = O.linear_w8a8(qx, wu, s_in, s_u)
    assert np.array_equal(host_u8(out), O.swiglu_2in_fp8(gb, ub, s_out))


def test_fused_vs_oracle_chain(W):
    M, K, I = 512, 1024, 2048
    x, s_in, ws, ss = _problem(M, K, I, seed=7)
    s_out = np.float32(0.004)
    out = host_u8(W.gate_up_swiglu_fp8(dev_bf16(x), dev_f32(s_in), dev_u8(ws[0]), dev_u8(ws[1]),
                                       dev_f32(ss[0]), dev_f32(ss[1]), dev_f32(s_out)))
    (g64, gb), (u64, ub) = O.qkv_shared_quant_gemm("A8", x, s_in, ws, ss)
    # codes can differ from the oracle's only where the kernel's own bf16
    # gate/up differ from the correctly rounded ones, within the binary32
    # accumulation window of the exact sums
    wg = accumulation_window(g64, abs_product_sums("A8", x, s_in, ws[0], ss[0]), K)
    wu = accumulation_window(u64, abs_product_sums("A8", x, s_in, ws[1], ss[1]), K)
    assert_swiglu_consistent(out, O.swiglu_2in_fp8(gb, ub, s_out), g64, u64, wg, wu, "e4m3", s_out, 2e-3)


def test_fused_full_size(W):
    """20670 tokens, 4096 -> 2 x 16384: the fused kernel equals the separate
    path everywhere, and the oracle chain on sampled rows plus the tail."""
    M, K, I = 20670, 4096, 16384
    gen = torch.Generator(device="cuda").manual_seed(5)
    x = (torch.randn((M, K), generator=gen, device="cuda") * 0.25).to(torch.bfloat16)
    wq, sw = [], []
    for c in (0.6, 1.0):
        w = torch.randn((I, K), generator=gen, device="cuda") * (0.02 * c)
        s = (w.abs().amax() / 448).reshape(1)
        wq.append((w / s).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).contiguous())
        sw.append(s.contiguous())
    s_in = (x.float().abs().amax() / 448).reshape(1).contiguous()
    s_out = dev_f32(0.02)
    fused = W.gate_up_swiglu_fp8(x, s_in, wq[0], wq[1], sw[0], sw[1], s_out)
    g, u = W.qkv_shared_quant_gemm(W.MODE_A8, x, s_in, wq, sw)
    sep = W.swiglu_2in_fp8(g, u, s_out)
    torch.cuda.synchronize()
    W.poll_device_error()
    assert torch.equal(fused, sep)
    rows = np.concatenate([synth.random_rows(9, M, 48), np.arange(M - 62, M)])
    ri = torch.from_numpy(rows).cuda()
    xs = host_bits(x[ri])
    qws = [host_u8(w) for w in wq]
    sws = [np.float32(s.item()) for s in sw]
    si = np.float32(s_in.item())
    (g64, gb), (u64, ub) = O.qkv_shared_quant_gemm("A8", xs, si, qws, sws)
    want = O.swiglu_2in_fp8(gb, ub, np.float32(0.02))
    wg = accumulation_window(g64, abs_product_sums("A8", xs, si, qws[0], sws[0]), K)
    wu = accumulation_window(u64, abs_product_sums("A8", xs, si, qws[1], sws[1]), K)
    assert_swiglu_consistent(host_u8(fused[ri]), want, g64, u64, wg, wu, "e4m3", np.float32(0.02), 2e-3)

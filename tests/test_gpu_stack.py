"""The step-scheduled block at the CFG batch size (M = 2 x 20670 = 41340):
the policy picks W8A16 for step 2 and W8A8 for step 3 of 8; every row of the
block (Q/K/V group, out-projection, gate/up + SwiGLU, down) is checked on
sampled rows plus the ragged tail against the oracle."""

import numpy as np
import pytest
import torch

import oracle as O
from gpu_util import W, GEMM_TOL, dev_f32, host_bits, host_u8, gemm_err  # noqa: F401
from w8a16_linear_gb300 import synth

pytestmark = pytest.mark.gpu

M, H, I = 41340, 4096, 16384


def _weight(gen, n, k, c):
    w = torch.randn((n, k), generator=gen, device="cuda") * (0.02 * c)
    s = (w.abs().amax() / 448).reshape(1).contiguous()
    q = (w / s).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).contiguous()
    return q, s


@pytest.fixture(scope="module")
def block(W):
    gen = torch.Generator(device="cuda").manual_seed(11)
    x = (torch.randn((M, H), generator=gen, device="cuda") * 0.25).to(torch.bfloat16)
    s_in = (x.float().abs().amax() / 448).reshape(1).contiguous()
    wqkv = [_weight(gen, H, H, c) for c in (0.6, 0.8, 1.0)]
    wout = _weight(gen, H, H, 0.9)
    wgu = [_weight(gen, I, H, c) for c in (0.7, 1.0)]
    wdown = _weight(gen, H, I, 0.8)
    return dict(x=x, s_in=s_in, wqkv=wqkv, wout=wout, wgu=wgu, wdown=wdown,
                s_h=dev_f32(0.02), rows=np.concatenate([synth.random_rows(12, M, 24), np.arange(M - 124, M)]))


def _run(W, b, step):
    pol = W.StepPolicy(1, 1, 3, 3)
    mode = W.step_policy_dispatch(pol, step, 8)
    x = b["x"]
    if mode == W.MODE_A8:
        qkv = W.qkv_shared_quant_gemm(W.MODE_A8, x, b["s_in"], [q for q, _ in b["wqkv"]], [s for _, s in b["wqkv"]])
        out = W.fp8_linear_w8a8(x, b["wout"][0], b["s_in"], b["wout"][1])
        h = W.gate_up_swiglu_fp8(x, b["s_in"], b["wgu"][0][0], b["wgu"][1][0], b["wgu"][0][1], b["wgu"][1][1], b["s_h"])
        y = W.fp8_linear_w8a8(h, b["wdown"][0], b["s_h"], b["wdown"][1])
    else:
        qkv = W.qkv_shared_quant_gemm(W.MODE_A16, x, None, [q for q, _ in b["wqkv"]], [s for _, s in b["wqkv"]])
        out = W.fp8_linear_w8a16(x, b["wout"][0], b["wout"][1])
        g, u = W.qkv_shared_quant_gemm(W.MODE_A16, x, None, [q for q, _ in b["wgu"]], [s for _, s in b["wgu"]])
        h = W.swiglu_2in_bf16(g, u)
        y = W.fp8_linear_w8a16(h, b["wdown"][0], b["wdown"][1])
    torch.cuda.synchronize()
    W.poll_device_error()
    return mode, qkv, out, h, y


@pytest.mark.parametrize("step", [2, 3])
def test_block_step_at_cfg_batch(W, block, step):
    mode, qkv, out, h, y = _run(W, block, step)
    rows = block["rows"]
    ri = torch.from_numpy(rows).cuda()
    xs = host_bits(block["x"][ri])
    s_in = np.float32(block["s_in"].item())
    sc = lambda t: np.float32(t.item())  # noqa: E731
    qkv_w = [host_u8(q) for q, _ in block["wqkv"]]
    qkv_s = [sc(s) for _, s in block["wqkv"]]
    om = "A8" if mode == W.MODE_A8 else "A16"
    assert om == ("A16" if step == 2 else "A8")
    for yg, (r64, _) in zip(qkv, O.qkv_shared_quant_gemm(om, xs, s_in, qkv_w, qkv_s)):
        assert gemm_err(host_bits(yg[ri]), r64) <= GEMM_TOL
    wo, so = host_u8(block["wout"][0]), sc(block["wout"][1])
    r_out = (O.linear_w8a8(O.quant_static(xs, s_in), wo, s_in, so) if om == "A8"
             else O.linear_w8a16(xs, wo, so))[0]
    assert gemm_err(host_bits(out[ri]), r_out) <= GEMM_TOL
    gu_w = [host_u8(q) for q, _ in block["wgu"]]
    gu_s = [sc(s) for _, s in block["wgu"]]
    (_, gb), (_, ub) = O.qkv_shared_quant_gemm(om, xs, s_in, gu_w, gu_s)
    wd, sd = host_u8(block["wdown"][0]), sc(block["wdown"][1])
    if om == "A8":
        want = O.swiglu_2in_fp8(gb, ub, np.float32(0.02))
        got = host_u8(h[ri])
        assert (got != want).mean() < 2e-3
        r_y, _ = O.linear_w8a8(got, wd, np.float32(0.02), sd)      # down on the GPU's own codes
    else:
        want = O.swiglu_2in_bf16(gb, ub)
        got = host_bits(h[ri])
        assert (got != want).mean() < 2e-2                           # bf16 gate/up may differ by an ulp
        r_y, _ = O.linear_w8a16(got, wd, sd)
    assert gemm_err(host_bits(y[ri]), r_y) <= GEMM_TOL

"""GPU parity of the W8A16 "dequant + F.linear" path: fp8_dequant_weight
(bit-exact dequantized weight) and qkv_shared_quant_gemm in A16 mode with a
workspace (the group's weights dequantized there, then one bf16 GEMM launch)
against the oracle and against the path that dequantizes inside the GEMM."""

import numpy as np
import pytest
import torch

import oracle as O
from gpu_util import W, GEMM_TOL, dev_bf16, dev_f32, dev_u8, host_bits, gemm_err, amax_scale  # noqa: F401
from w8a16_linear_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("s_w", [0.5039 / 448, 2.0 ** -12, 1.0, 3.7e-3, 1e-30, 2e30])
def test_dequant_every_code(W, s_w):
    """All 256 codes (both NaN codes included) against the oracle's
    bf16(fl32(dec(q) * s_w)); NaN codes may give any NaN pattern."""
    q = np.tile(np.arange(256, dtype=np.uint8), 64).reshape(64, 256)
    got = host_bits(W.fp8_dequant_weight(dev_u8(q), dev_f32(s_w)))
    want = O.dequant_weight_bf16(q, np.float32(s_w))
    nan = np.isnan(O.bf16_decode(want))
    assert np.array_equal(np.isnan(O.bf16_decode(got)), nan)
    assert np.array_equal(got[~nan], want[~nan])


@pytest.mark.parametrize("N,K", [(1, 16), (3, 592), (33, 48), (2000, 4112)])
def test_dequant_ragged_sizes(W, N, K):
    """Sizes that end inside a warp's 512-element block, and one that takes
    two grid-stride iterations: every element bit-exact against the oracle."""
    rng = np.random.default_rng(N + K)
    q = rng.integers(0, 256, (N, K), dtype=np.uint8)
    q[(q & 0x7F) == 0x7F] = 0x10          # no NaN codes: compare bit for bit
    s_w = np.float32(0.37)
    got = host_bits(W.fp8_dequant_weight(dev_u8(q), dev_f32(s_w)))
    assert np.array_equal(got, O.dequant_weight_bf16(q, s_w))


def _group(M, K, Ns, seed=0):
    x = synth.activations_bf16(seed, (M, K), 0.25, outlier_frac=0.001)
    c = synth.uniform_f32(3, (len(Ns),), 0.5, 1.0)
    qws, s_ws = [], []
    for i, N in enumerate(Ns):
        w = synth.normal_f32(10 + i, (N, K), 0.02) * c[i]
        s = amax_scale(w)
        qws.append(O.e4m3_encode(w / s))
        s_ws.append(s)
    return x, qws, s_ws


@pytest.mark.parametrize("M,K,Ns", [(1000, 512, (512, 512, 512)), (257, 256, (1024, 1024)),
                                    (64, 256, (256,)), (129, 4112, (272,)), (777, 384, (400, 16 * 17))])
def test_a16_workspace_vs_oracle_and_fused(W, M, K, Ns):
    x, qws, s_ws = _group(M, K, Ns)
    xd, wd, sd = dev_bf16(x), [dev_u8(q) for q in qws], [dev_f32(s) for s in s_ws]
    ws = W.w8a16_workspace(wd)
    ys = W.qkv_shared_quant_gemm(W.MODE_A16, xd, None, wd, sd, ws=ws)
    yf = W.qkv_shared_quant_gemm(W.MODE_A16, xd, None, wd, sd)
    torch.cuda.synchronize()
    W.poll_device_error()
    ref = O.qkv_shared_quant_gemm("A16", x, None, qws, s_ws)
    off = 0
    for y, f, (r64, _), q, s in zip(ys, yf, ref, qws, s_ws):
        assert gemm_err(host_bits(y), r64) <= GEMM_TOL
        assert gemm_err(host_bits(f), r64) <= GEMM_TOL
        # the workspace holds the dequantized weight, bit for bit
        n = q.size
        assert np.array_equal(host_bits(ws[off:off + n]).reshape(q.shape), O.dequant_weight_bf16(q, s))
        off += n


def test_a16_workspace_exact_sums_bit_exact(W):
    """Operands whose partial sums are exact in any order: the two-pass
    result equals the oracle bit for bit (pair and single-CTA tiles)."""
    rng = np.random.default_rng(1)
    for M in (100, 900):
        K, N = 2048, 400
        xv = np.array([0.0, 0.25, -0.25, 0.5, -1.0, 1.5, 2.0, -3.0], np.float32)
        x = torch.from_numpy(rng.choice(xv, size=(M, K))).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        qw = O.e4m3_encode(rng.choice(np.array([0.0, 1.0, -1.0, 2.0, -0.5, 3.0], np.float32), size=(N, K)))
        s_w = np.float32(2.0 ** -4)
        wd = [dev_u8(qw)]
        y = W.qkv_shared_quant_gemm(W.MODE_A16, dev_bf16(x), None, wd, [dev_f32(s_w)], ws=W.w8a16_workspace(wd))
        _, want = O.linear_w8a16(x, qw, s_w)
        assert np.array_equal(host_bits(y[0]), want)


def test_a16_workspace_full_size_sampled(W):
    """20670 tokens, the Q/K/V group: sampled rows and the tail."""
    M, K = 20670, 4096
    x, qws, s_ws = _group(M, K, (4096, 4096, 4096))
    xd, wd, sd = dev_bf16(x), [dev_u8(q) for q in qws], [dev_f32(s) for s in s_ws]
    ys = W.qkv_shared_quant_gemm(W.MODE_A16, xd, None, wd, sd, ws=W.w8a16_workspace(wd))
    rows = np.concatenate([synth.random_rows(8, M, 128), np.arange(M - 62, M)])
    for y, q, s in zip(ys, qws, s_ws):
        r16, _ = O.linear_w8a16(x, q, s, rows=rows)
        assert gemm_err(host_bits(y)[rows], r16) <= GEMM_TOL


def test_workspace_too_small_is_refused(W):
    x = torch.zeros((64, 256), dtype=torch.bfloat16, device="cuda")
    w = [torch.zeros((256, 256), dtype=torch.uint8, device="cuda")]
    with pytest.raises(W.W8Error):
        W.qkv_shared_quant_gemm(W.MODE_A16, x, None, w, [dev_f32(1.0)],
                                ws=torch.empty((100,), dtype=torch.bfloat16, device="cuda"))


def test_bf16_linear_group_on_dequantized_weights(W):
    """The F.linear half on its own: dequantize each weight, then one group
    launch; equals qkv_shared_quant_gemm(A16, ws) bit for bit."""
    x, qws, s_ws = _group(1000, 512, (512, 256, 768))
    xd, wd, sd = dev_bf16(x), [dev_u8(q) for q in qws], [dev_f32(s) for s in s_ws]
    wdq = [W.fp8_dequant_weight(w, s) for w, s in zip(wd, sd)]
    ys = W.bf16_linear_group(xd, wdq)
    yw = W.qkv_shared_quant_gemm(W.MODE_A16, xd, None, wd, sd, ws=W.w8a16_workspace(wd))
    ref = O.qkv_shared_quant_gemm("A16", x, None, qws, s_ws)
    for y, y2, (r64, _) in zip(ys, yw, ref):
        assert gemm_err(host_bits(y), r64) <= GEMM_TOL
        assert torch.equal(y.view(torch.int16), y2.view(torch.int16))


@pytest.mark.parametrize("M,K,I", [(1000, 512, 1024), (100, 256, 512), (257, 4112, 16 * 33),
                                   (20670, 4096, 16384)])
def test_bf16_gate_up_swiglu_equals_separate_path(W, M, K, I):
    """The fused 16-bit gate/up + SwiGLU launch against bf16_linear_group ->
    swiglu_2in_bf16 on the same dequantized weights: bit for bit (the
    epilogue rounds gate and up to bf16 exactly as the GEMM would write
    them)."""
    gen = torch.Generator(device="cuda").manual_seed(M + I)
    x = (torch.randn((M, K), generator=gen, device="cuda") * 0.25).to(torch.bfloat16)
    wg = (torch.randn((I, K), generator=gen, device="cuda") * 0.02 * 448 / 0.1).clamp(-448, 448)
    wu = (torch.randn((I, K), generator=gen, device="cuda") * 0.02 * 448 / 0.1).clamp(-448, 448)
    qg = wg.to(torch.float8_e4m3fn).view(torch.uint8)
    qu = wu.to(torch.float8_e4m3fn).view(torch.uint8)
    sg, su = dev_f32(0.1 / 448), dev_f32(0.08 / 448)
    dg, du = W.fp8_dequant_weight(qg, sg), W.fp8_dequant_weight(qu, su)
    h = W.bf16_gate_up_swiglu(x, dg, du)
    g, u = W.bf16_linear_group(x, [dg, du])
    h_sep = W.swiglu_2in_bf16(g, u)
    torch.cuda.synchronize()
    W.poll_device_error()
    assert torch.equal(h.view(torch.int16), h_sep.view(torch.int16))


def test_bf16_gate_up_swiglu_exact_sums_vs_oracle(W):
    """Operands whose partial sums are exact in any order: gate and up are
    then the oracle's bit for bit, and so is the SwiGLU."""
    rng = np.random.default_rng(3)
    M, K, I = 300, 1024, 512
    xv = np.array([0.0, 0.25, -0.25, 0.5, -1.0, 1.5, 2.0, -3.0], np.float32)
    x = torch.from_numpy(rng.choice(xv, size=(M, K))).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    cv = np.array([0.0, 1.0, -1.0, 2.0, -0.5, 3.0], np.float32)
    qg = O.e4m3_encode(rng.choice(cv, size=(I, K)))
    qu = O.e4m3_encode(rng.choice(cv, size=(I, K)))
    s_w = np.float32(2.0 ** -6)
    dg, du = W.fp8_dequant_weight(dev_u8(qg), dev_f32(s_w)), W.fp8_dequant_weight(dev_u8(qu), dev_f32(s_w))
    h = host_bits(W.bf16_gate_up_swiglu(dev_bf16(x), dg, du))
    _, gb = O.linear_w8a16(x, qg, s_w)
    _, ub = O.linear_w8a16(x, qu, s_w)
    want = O.swiglu_2in_bf16(gb, ub)
    nan = np.isnan(O.bf16_decode(want))
    assert np.array_equal(np.isnan(O.bf16_decode(h)), nan)
    assert np.array_equal(h[~nan], want[~nan])


@pytest.mark.parametrize("M,K,N", [(64, 256, 256), (300, 512, 1024), (4096, 4096, 4096), (20670, 4096, 4096)])
def test_exported_linear_with_workspace(W, M, K, N):
    """fp8_linear_w8a16 with its optional workspace: the weight dequantized
    into the workspace, then the bf16 GEMM.  Against the oracle (sampled rows
    plus the tail at full size), bit for bit against the A16 group call with
    a workspace (the same two kernels), and within the tolerance of the form
    without a workspace (same operand bits, other accumulation order); the
    workspace holds the dequantized weight afterwards."""
    x, qws, s_ws = _group(M, K, (N,), seed=M)
    xd, wd, sd = dev_bf16(x), dev_u8(qws[0]), dev_f32(s_ws[0])
    ws = torch.empty((N * K,), dtype=torch.bfloat16, device="cuda")
    y = W.fp8_linear_w8a16(xd, wd, sd, ws=ws)
    y_group = W.qkv_shared_quant_gemm(W.MODE_A16, xd, None, [wd], [sd], ws=W.w8a16_workspace([wd]))[0]
    y_fused = W.fp8_linear_w8a16(xd, wd, sd)
    torch.cuda.synchronize()
    W.poll_device_error()
    assert torch.equal(y.view(torch.int16), y_group.view(torch.int16))
    assert np.array_equal(host_bits(ws.view(N, K)), O.dequant_weight_bf16(qws[0], s_ws[0]))
    rows = (np.arange(M) if M <= 4096 else
            np.concatenate([synth.random_rows(M, M, 64), np.arange(M - 62, M)]))
    y64, _ = O.linear_w8a16(x, qws[0], s_ws[0], rows=rows)
    assert gemm_err(host_bits(y)[rows], y64) <= GEMM_TOL
    yf = O.bf16_decode(host_bits(y_fused)[rows]).astype(np.float64)
    assert np.abs(yf - y64).max() / np.abs(y64).max() <= GEMM_TOL

"""GPU parity of qkv_shared_quant_gemm (split Q/K/V and gate/up groups) and
of the gated-MLP chain gate/up -> swiglu_2in -> down."""

import numpy as np
import pytest
import torch

import oracle as O
from gpu_util import (W, GEMM_TOL, dev_bf16, dev_f32, dev_u8, host_bits, host_u8,  # noqa: F401
                      gemm_err, amax_scale, linear_problem)
from w8a16_linear_gb300 import synth

pytestmark = pytest.mark.gpu


def _group(M, K, Ns, seed=0):
    x = synth.activations_bf16(seed, (M, K), 0.25, outlier_frac=0.001)
    xc = synth.activations_bf16(seed + 2, (min(M, 4096), K), 0.25, outlier_frac=0.001)
    s_in = amax_scale(O.bf16_decode(xc))
    c = synth.uniform_f32(3, (len(Ns),), 0.5, 1.0)
    qws, s_ws = [], []
    for i, N in enumerate(Ns):
        w = synth.normal_f32(10 + i, (N, K), 0.02) * c[i]
        s = amax_scale(w)
        qws.append(O.e4m3_encode(w / s))
        s_ws.append(s)
    return x, s_in, qws, s_ws


@pytest.mark.parametrize("M,K,Ns", [(1000, 512, (512, 512, 512)), (257, 256, (1024, 1024)),
                                    (64, 256, (256,))])
def test_group_vs_oracle(W, M, K, Ns):
    x, s_in, qws, s_ws = _group(M, K, Ns)
    assert len(set(float(s) for s in s_ws)) == len(Ns)       # scales genuinely differ
    xd, wd, sd = dev_bf16(x), [dev_u8(q) for q in qws], [dev_f32(s) for s in s_ws]
    for mode, om in ((W.MODE_A8, "A8"), (W.MODE_A16, "A16")):
        ys = W.qkv_shared_quant_gemm(mode, xd, dev_f32(s_in), wd, sd)
        torch.cuda.synchronize()
        W.poll_device_error()
        ref = O.qkv_shared_quant_gemm(om, x, s_in, qws, s_ws)
        for y, (r64, _) in zip(ys, ref):
            assert gemm_err(host_bits(y), r64) <= GEMM_TOL, om


def test_a8_single_quantization_by_storage(W):
    """One quantization into the workspace; every projection reads that same
    storage: outputs equal separate W8A8 calls fed with the workspace."""
    x, s_in, qws, s_ws = _group(512, 512, (512, 512, 512))
    xd, wd, sd, si = dev_bf16(x), [dev_u8(q) for q in qws], [dev_f32(s) for s in s_ws], dev_f32(s_in)
    ws = torch.full((512, 512), 0xAA, dtype=torch.uint8, device="cuda")
    ys = W.qkv_shared_quant_gemm(W.MODE_A8, xd, si, wd, sd, ws=ws)
    assert np.array_equal(host_u8(ws), O.quant_static(x, s_in))
    for y, w, s in zip(ys, wd, sd):
        y1 = W.fp8_linear_w8a8(ws, w, si, s)
        assert torch.equal(y.view(torch.int16), y1.view(torch.int16))


def test_a16_stands_down_and_differs(W):
    """A16 needs no workspace (no quantization runs), matches the single
    W8A16 call bit for bit, and differs from the A8 result."""
    x, s_in, qws, s_ws = _group(300, 256, (256, 256, 256))
    xd, wd, sd = dev_bf16(x), [dev_u8(q) for q in qws], [dev_f32(s) for s in s_ws]
    ys16 = W.qkv_shared_quant_gemm(W.MODE_A16, xd, None, wd, sd, ws=None)
    ys8 = W.qkv_shared_quant_gemm(W.MODE_A8, xd, dev_f32(s_in), wd, sd)
    for y16, y8, w, s in zip(ys16, ys8, wd, sd):
        assert torch.equal(y16.view(torch.int16), W.fp8_linear_w8a16(xd, w, s).view(torch.int16))
        assert not torch.equal(y16.view(torch.int16), y8.view(torch.int16))


def test_a16_closer_to_unquantized_reference(W):
    M, K, N = 4096, 4096, 4096
    x = synth.activations_bf16(0, (M, K), 0.25, outlier_frac=0.001)
    xc = synth.activations_bf16(2, (M, K), 0.25, outlier_frac=0.001)
    s_in = amax_scale(O.bf16_decode(xc))
    w = synth.normal_f32(1, (N, K), 0.02)
    s_w = amax_scale(w)
    qw = O.e4m3_encode(w / s_w)
    xd, wd = dev_bf16(x), dev_u8(qw)
    y8 = O.bf16_decode(host_bits(W.fp8_linear_w8a8(xd, wd, dev_f32(s_in), dev_f32(s_w)))).astype(np.float64)
    y16 = O.bf16_decode(host_bits(W.fp8_linear_w8a16(xd, wd, dev_f32(s_w)))).astype(np.float64)
    rows = synth.random_rows(1, M, 256)
    ref = O.bf16_decode(x[rows]).astype(np.float64) @ w.astype(np.float64).T
    assert np.linalg.norm(y16[rows] - ref) < np.linalg.norm(y8[rows] - ref)


def test_qkv_full_size_sampled_and_fused_requant_context(W):
    """20670 tokens, three 4096x4096 projections with scales differing up to
    2x and one shared input scale; the max(s)-re-quantized fused variant is
    reported beside the split result (it is the defect, not a target)."""
    M, K = 20670, 4096
    x, s_in, qws, s_ws = _group(M, K, (4096, 4096, 4096))
    xd, wd, sd = dev_bf16(x), [dev_u8(q) for q in qws], [dev_f32(s) for s in s_ws]
    ys = W.qkv_shared_quant_gemm(W.MODE_A8, xd, dev_f32(s_in), wd, sd)
    torch.cuda.synchronize()
    rows = np.concatenate([synth.random_rows(8, M, 128), np.arange(M - 62, M)])
    qx = O.quant_static(x[rows], s_in)
    fused, s_max = O.requant_onto_max_scale(qws, s_ws)
    for y, qw, s, qf in zip(ys, qws, s_ws, fused):
        r64, _ = O.linear_w8a8(qx, qw, s_in, s)
        assert gemm_err(host_bits(y)[rows], r64) <= GEMM_TOL
        if s != s_max:
            assert np.mean(qf != qw) > 0.05      # the fused variant visibly re-rounds


def test_gated_mlp_chain(W):
    """gate/up (G=2, distinct scales) -> swiglu_2in_fp8 -> down on the FP8
    codes, against the oracle chain on sampled rows."""
    M, K, I = 2048, 512, 2048
    x, s_in, qws, s_ws = _group(M, K, (I, I), seed=20)
    wdn = synth.normal_f32(30, (K, I), 0.02)
    s_dn = amax_scale(wdn)
    q_dn = O.e4m3_encode(wdn / s_dn)
    # calibration of the down projection's input scale on a separate batch
    xc = synth.activations_bf16(22, (M, K), 0.25, outlier_frac=0.001)
    gc, uc = O.qkv_shared_quant_gemm("A8", xc, s_in, qws, s_ws)
    s_out = amax_scale(O.swiglu_h(gc[1], uc[1]))
    xd = dev_bf16(x)
    g, u = W.qkv_shared_quant_gemm(W.MODE_A8, xd, dev_f32(s_in), [dev_u8(q) for q in qws],
                                   [dev_f32(s) for s in s_ws])
    h = W.swiglu_2in_fp8(g, u, dev_f32(s_out))
    y = W.fp8_linear_w8a8(h, dev_u8(q_dn), dev_f32(s_out), dev_f32(s_dn))
    torch.cuda.synchronize()
    # the SwiGLU codes are bit-exact given the GPU's gate/up outputs
    gb, ub = host_bits(g), host_bits(u)
    assert np.array_equal(host_u8(h), O.swiglu_2in_fp8(gb, ub, s_out))
    # the down projection is within tolerance given those codes
    r64, _ = O.linear_w8a8(host_u8(h), q_dn, s_out, s_dn)
    assert gemm_err(host_bits(y), r64) <= GEMM_TOL


def test_full_size_group_equals_separate_calls_bit_for_bit(W):
    """M = 20670, 3 x 4096 x 4096: the group launch (3888 tiles) cuts its last
    wave's 12 tiles into four column slices each, the single-projection
    launches (1296 tiles) cut their last 4 tiles; every output element is
    accumulated in the same order either way, so the outputs are identical."""
    M, K, N = 20670, 4096, 4096
    gen = torch.Generator(device="cuda").manual_seed(21)
    q = (torch.randn((M, K), generator=gen, device="cuda") * 40).clamp(-448, 448).to(torch.float8_e4m3fn)
    q = q.view(torch.uint8).contiguous()
    ws, ss = [], []
    for i in range(3):
        w = torch.randn((N, K), generator=gen, device="cuda") * (0.02 * (0.5 + 0.25 * i))
        s = (w.abs().amax() / 448).reshape(1).contiguous()
        ws.append((w / s).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).contiguous())
        ss.append(s)
    s_in = dev_f32(0.003)
    group = W.fp8_linear_w8a8_group(q, s_in, ws, ss)
    for y, w, s in zip(group, ws, ss):
        y1 = W.fp8_linear_w8a8(q, w, s_in, s)
        assert torch.equal(y.view(torch.int16), y1.view(torch.int16))
    torch.cuda.synchronize()
    W.poll_device_error()


@pytest.mark.parametrize("M,Ns", [(2600, (4096,)),          # 11 x 16 = 176 tiles: 2 x 76 + 24 -> halves
                                  (4990, (2048, 2048)),     # 20 x 16 = 320 tiles: 4 x 76 + 16 -> quarters
                                  (8192, (4096, 1024)),     # 32 x 20 = 640 tiles: 8 x 76 + 32 -> halves
                                  (3000, (1024, 1024, 1024))])  # 12 x 12 = 144 tiles: 76 + 68 -> not cut
def test_tail_slices_against_oracle(W, M, Ns):
    """Launches whose last wave is cut into column slices: every projection
    against the oracle on sampled rows plus the ragged tail, and against its
    own single-projection launch (cut differently, or not at all) bit for bit."""
    K = 1024
    x, s_in, qws, s_ws = _group(M, K, Ns)
    xd, wd, sd, si = dev_bf16(x), [dev_u8(q) for q in qws], [dev_f32(s) for s in s_ws], dev_f32(s_in)
    q = W.fp8_quant_static(xd, si)
    ys = W.fp8_linear_w8a8_group(q, si, wd, sd)
    rows = np.concatenate([synth.random_rows(M, M - 300, 40), np.arange(M - 300, M)])
    qx = host_u8(q)[rows]
    for y, w, s, qw, sw in zip(ys, wd, sd, qws, s_ws):
        y64, _ = O.linear_w8a8(qx, qw, s_in, sw)
        assert gemm_err(host_bits(y)[rows], y64) <= GEMM_TOL
        assert torch.equal(y.view(torch.int16), W.fp8_linear_w8a8(q, w, si, s).view(torch.int16))
    torch.cuda.synchronize()
    W.poll_device_error()


def test_tail_slices_bf16_group(W):
    """The bf16 GEMM of the W8A16 path cuts its tail the same way (N = 128 or
    64 kind::f16 MMAs): a 3-projection group (20 x 48 = 960 tiles, 12 x 76 +
    48: not cut) against single projections (320 tiles, 4 x 76 + 16: cut in
    four) bit for bit, and against the oracle."""
    M, K, Ns = 4990, 1024, (4096, 4096, 4096)
    x, _, qws, s_ws = _group(M, K, Ns, seed=3)
    xd = dev_bf16(x)
    wds = [W.fp8_dequant_weight(dev_u8(q), dev_f32(s)) for q, s in zip(qws, s_ws)]
    ys = W.bf16_linear_group(xd, wds)
    rows = np.concatenate([synth.random_rows(8, M - 200, 32), np.arange(M - 200, M)])
    for y, wd, qw, sw in zip(ys, wds, qws, s_ws):
        assert torch.equal(y.view(torch.int16), W.bf16_linear_group(xd, [wd])[0].view(torch.int16))
        y64, _ = O.linear_w8a16(x, qw, sw, rows=rows)
        assert gemm_err(host_bits(y)[rows], y64) <= GEMM_TOL
    torch.cuda.synchronize()
    W.poll_device_error()

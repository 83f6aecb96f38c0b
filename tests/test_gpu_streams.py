"""The entry points keep no state between calls besides what the caller
passes (fp8_linear_w8a8_noalloc, whose shared scratch its header documents,
aside): work issued on two streams at once gives, bit for bit, what the
same calls give one after the other."""

import pytest
import torch

from gpu_util import W  # noqa: F401

pytestmark = pytest.mark.gpu


def _inputs(seed, M, K, N):
    g = torch.Generator(device="cuda").manual_seed(seed)
    x = (torch.randn((M, K), generator=g, device="cuda") * 0.25).to(torch.bfloat16)
    ws = [(torch.randn((N, K), generator=g, device="cuda") * 200).clamp(-448, 448)
          .to(torch.float8_e4m3fn).view(torch.uint8) for _ in range(3)]
    ss = [torch.tensor([0.02 * (1 + i) / 448], device="cuda") for i in range(3)]
    s_in = torch.tensor([1.0 / 448], device="cuda")
    sh, sc = ((torch.randn((2, K), generator=g, device="cuda") * 0.5).to(torch.bfloat16) for _ in range(2))
    return x, ws, ss, s_in, sh, sc


def _calls(W, inp):
    x, ws, ss, s_in, sh, sc = inp
    a8 = W.qkv_shared_quant_gemm(W.MODE_A8, x, s_in, ws, ss)
    a16 = W.qkv_shared_quant_gemm(W.MODE_A16, x, None, ws, ss, ws=W.w8a16_workspace(ws))
    q = W.ln_modulate_quant(x, sh, sc, s_in)
    return [t.view(torch.uint8) for t in a8 + a16 + [q]]


def test_two_streams_at_once_equal_serial(W):
    inps = [_inputs(1, 3000, 1024, 1024), _inputs(2, 2500, 1024, 1024)]
    serial = [_calls(W, inp) for inp in inps]
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = [None, None]
    for _ in range(3):  # interleave the two streams' launches
        for i, st in enumerate(streams):
            with torch.cuda.stream(st):
                outs[i] = _calls(W, inps[i])
    torch.cuda.synchronize()
    W.poll_device_error()
    for got, want in zip(outs, serial):
        for a, b in zip(got, want):
            assert torch.equal(a, b)

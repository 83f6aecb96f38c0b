"""The allocation-free W8A8 entry point, for callers that cannot allocate
device memory (operator/plugin interfaces that pass only inputs and outputs,
fixed memory pools, code that may not call cudaMalloc during a stream
capture).  It is called through the C ABI on consecutive calls and must give
exactly the output of the workspace-based entry point (the same quantization
and GEMM kernels on the same bits), and the oracle's on sampled rows.  This
file is collected last on purpose."""

import ctypes

import numpy as np
import pytest
import torch

import oracle as O
from gpu_util import W, GEMM_TOL, dev_bf16, dev_f32, dev_u8, host_bits, linear_problem, gemm_err  # noqa: F401
from w8a16_linear_gb300 import synth

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 32 << 20            # the entry point's fixed limit on M * K


def _noalloc(L, xd, M, K, wd, N, si, sw, y, stream):
    return L.fp8_linear_w8a8_noalloc(ctypes.c_void_p(xd.data_ptr()), M, K, ctypes.c_void_p(wd.data_ptr()), N,
                                     ctypes.c_void_p(si.data_ptr()), ctypes.c_void_p(sw.data_ptr()),
                                     ctypes.c_void_p(y.data_ptr()), stream)


def test_noalloc_matches_workspace_entry_point_consecutive_calls(W):
    from w8a16_linear_gb300 import binding
    L = binding.lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    # consecutive calls: one that fills the scratch array exactly (M*K = 32 MiB),
    # then smaller ones, so scratch left by an earlier call must not leak into
    # a later result
    cases = [(8192, 4096, 256, 0), (2048, 4096, 512, 1), (333, 1024, 256, 2)]
    assert cases[0][0] * cases[0][1] == SCRATCH_BYTES
    for (M, K, N, seed) in cases:
        x, qw, s_in, s_w = linear_problem(M, K, N, seed_x=seed, seed_w=seed + 10)
        xd, wd, si, sw = dev_bf16(x), dev_u8(qw), dev_f32(s_in), dev_f32(s_w)
        y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        st = _noalloc(L, xd, M, K, wd, N, si, sw, y, stream)
        assert st == 0, L.w8_last_error()
        ref = W.fp8_linear_w8a8(xd, wd, si, sw)
        torch.cuda.synchronize()
        W.poll_device_error()
        assert torch.equal(y.view(torch.int16), ref.view(torch.int16))
        rows = np.concatenate([synth.random_rows(40 + seed, M, min(M, 24)), np.arange(max(M - 8, 0), M)])
        y64, _ = O.linear_w8a8(O.quant_static(x[rows], s_in), qw, s_in, s_w)
        assert gemm_err(host_bits(y)[rows], y64) <= GEMM_TOL


def test_noalloc_refuses_more_than_its_scratch(W):
    from w8a16_linear_gb300 import binding
    L = binding.lib()
    p = ctypes.c_void_p(0x10000)
    assert L.fp8_linear_w8a8_noalloc(p, 8193, 4096, p, 256, p, p, p, None) == 2
    assert b"scratch" in L.w8_last_error()

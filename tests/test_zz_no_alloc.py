"""The allocation-free W8A8 entry point, for callers that cannot allocate
device memory (operator/plugin interfaces that pass only inputs and outputs,
fixed memory pools, code that may not call cudaMalloc during a stream
capture).  It is called through the C ABI and compared with the existing
workspace-based entry point on two calls in a row.  This file is collected
last on purpose."""

import ctypes

import numpy as np
import pytest
import torch

from gpu_util import W, GEMM_TOL, dev_bf16, dev_f32, dev_u8, linear_problem  # noqa: F401

pytestmark = pytest.mark.gpu


def _rel(a, b):
    a, b = a.float(), b.float()
    return float((a - b).abs().max() / b.abs().max().clamp_min(1e-30))


def test_noalloc_matches_workspace_entry_point_twice(W):
    from w8a16_linear_gb300 import binding
    L = binding.lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    # two calls in a row, the second smaller than the first, so that scratch
    # left by the first call must not leak into the second result
    for (M, K, N, seed) in [(2048, 4096, 512, 0), (333, 1024, 256, 1)]:
        x, qw, s_in, s_w = linear_problem(M, K, N, seed_x=seed, seed_w=seed + 10)
        xd, wd, si, sw = dev_bf16(x), dev_u8(qw), dev_f32(s_in), dev_f32(s_w)
        y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        st = L.fp8_linear_w8a8_noalloc(ctypes.c_void_p(xd.data_ptr()), M, K, ctypes.c_void_p(wd.data_ptr()), N,
                                       ctypes.c_void_p(si.data_ptr()), ctypes.c_void_p(sw.data_ptr()),
                                       ctypes.c_void_p(y.data_ptr()), stream)
        assert st == 0, L.w8_last_error()
        ref = W.fp8_linear_w8a8(xd, wd, si, sw)
        torch.cuda.synchronize()
        W.poll_device_error()
        assert _rel(y, ref) <= GEMM_TOL


def test_noalloc_refuses_more_than_its_scratch(W):
    from w8a16_linear_gb300 import binding
    L = binding.lib()
    p = ctypes.c_void_p(0x10000)
    assert L.fp8_linear_w8a8_noalloc(p, 8193, 4096, p, 256, p, p, p, None) == 2
    assert b"scratch" in L.w8_last_error()

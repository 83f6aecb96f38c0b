"""Failure detection on the GPU without a fault: a pipeline wait that nothing
satisfies times out, the host reads W8_ERR_TIMEOUT, and the context keeps
working (the next GEMM is correct)."""

import numpy as np
import pytest
import torch

import oracle as O
from gpu_util import W, GEMM_TOL, dev_bf16, dev_f32, dev_u8, host_bits, gemm_err, linear_problem  # noqa: F401

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives(W):
    W.poll_device_error()                       # clean slate
    W.selftest_timeout()
    with pytest.raises(W.W8Error) as ei:
        W.poll_device_error()
    assert ei.value.status == 8                 # W8_ERR_TIMEOUT
    W.poll_device_error()                       # cleared by the read
    x, qw, s_in, s_w = linear_problem(300, 256, 256)
    y = host_bits(W.fp8_linear_w8a8(dev_bf16(x), dev_u8(qw), dev_f32(s_in), dev_f32(s_w)))
    torch.cuda.synchronize()
    W.poll_device_error()
    r64, _ = O.linear_w8a8(O.quant_static(x, s_in), qw, s_in, s_w)
    assert gemm_err(y, r64) <= GEMM_TOL

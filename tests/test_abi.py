"""CPU tests of the C ABI: the library builds and loads, exports every
symbol the header declares, and its host-side logic (argument validation,
step policy, M == 0) behaves as the header states.  No call here reaches
the GPU."""

import ctypes
import os
import re

import numpy as np
import pytest

import oracle as O
from conftest import ROOT


@pytest.fixture(scope="module")
def L():
    from w8a16_linear_gb300 import build as B
    from w8a16_linear_gb300 import binding
    B.build()
    return binding.lib()


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "w8lin.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", src, flags=re.M)))


def test_header_symbols_exported(L):
    from w8a16_linear_gb300 import binding
    names = _declared_functions()
    assert set(names) == set(binding.SIGNATURES), names
    for n in names:
        assert hasattr(L, n), n
        assert n in binding.SIGNATURES, n
    assert L.w8_abi_version() == 6


def test_policy_matches_oracle_everywhere(L):
    from w8a16_linear_gb300 import binding as b
    for first in range(0, 5):
        for last in range(0, 5):
            pol = b.StepPolicy(1, 1, first, last)
            opol = O.StepPolicy(1, True, first, last)
            for n in range(1, 40):
                for s in range(n):
                    got = b.step_policy_dispatch(pol, s, n)
                    want = O.step_mode(opol, s, n)
                    assert got == (b.MODE_A16 if want == "A16" else b.MODE_A8)


def test_policy_refusals(L):
    from w8a16_linear_gb300 import binding as b
    for pol, step, n in [(b.StepPolicy(2, 1, 3, 3), 0, 8), (b.StepPolicy(1, 1, -1, 3), 0, 8),
                         (b.StepPolicy(1, 1, 3, -1), 0, 8), (b.StepPolicy(1, 1, 3, 3), 8, 8),
                         (b.StepPolicy(1, 1, 3, 3), -1, 8), (b.StepPolicy(1, 1, 3, 3), 0, 0)]:
        with pytest.raises(b.W8Error) as ei:
            b.step_policy_dispatch(pol, step, n)
        assert ei.value.status == 7
    assert all(b.step_policy_dispatch(None, s, 8) == b.MODE_A8 for s in range(8))
    assert L.step_policy_dispatch(None, 0, 8, None) == 1          # NULL mode_out


def _u(v):
    return ctypes.c_void_p(v)


def test_validation_before_any_cuda_call(L):
    # Non-null fake device addresses; validation must reject before use.
    p16 = _u(0x10000)
    # NULL pointers
    assert L.fp8_quant_static(None, 4, 16, 16, p16, p16, 16, None) == 1
    # K not a multiple of 16 / negative M
    assert L.fp8_quant_static(p16, 4, 24, 24, p16, p16, 24, None) == 2
    assert L.fp8_quant_static(p16, -1, 16, 16, p16, p16, 16, None) == 2
    # misaligned
    assert L.fp8_quant_static(_u(0x10008), 4, 16, 16, p16, p16, 16, None) == 3
    # W8A16 refuses an already-quantized (E4M3) activation
    assert L.fp8_linear_w8a16(p16, 1, 4, 16, p16, 16, p16, p16, None, None) == 5
    assert b"already-quantized" in L.w8_last_error()
    # unknown dtype, N not a multiple of 16, missing workspace for bf16 input
    assert L.fp8_linear_w8a8(p16, 7, 4, 16, p16, 16, p16, p16, p16, None, None) == 5
    assert L.fp8_linear_w8a8(p16, 1, 4, 16, p16, 24, p16, p16, p16, None, None) == 2
    assert L.fp8_linear_w8a8(p16, 0, 4, 16, p16, 16, p16, p16, p16, None, None) == 1
    # group size and mode
    arr = (ctypes.c_void_p * 3)(0x10000, 0x10000, 0x10000)
    ns = (ctypes.c_int64 * 3)(16, 16, 16)
    assert L.qkv_shared_quant_gemm(0, p16, 4, 16, p16, 4, arr, ns, arr, arr, p16, None) == 2
    assert L.qkv_shared_quant_gemm(5, p16, 4, 16, p16, 3, arr, ns, arr, arr, p16, None) == 2
    assert L.qkv_shared_quant_gemm(0, p16, 4, 16, p16, 3, arr, ns, arr, arr, None, None) == 1
    # swiglu
    assert L.swiglu_2in_fp8(p16, p16, 4, 24, p16, p16, None) == 2
    assert L.swiglu_2in_fp8(p16, p16, 4, 16, None, p16, None) == 1
    assert L.swiglu_2in_bf16(p16, _u(0x10004), 4, 16, p16, None) == 3
    # dequantization and the bf16 group GEMM
    assert L.fp8_dequant_weight(p16, 16, 24, p16, p16, None) == 2
    assert L.fp8_dequant_weight(None, 16, 16, p16, p16, None) == 1
    assert L.fp8_dequant_weight(p16, 0, 16, p16, p16, None) == 0
    assert L.bf16_linear_group(p16, 4, 16, 4, arr, ns, arr, None) == 2
    assert L.bf16_linear_group(p16, 4, 16, 3, None, ns, arr, None) == 1
    assert L.bf16_linear_group(p16, 0, 16, 3, arr, ns, arr, None) == 0
    # binary32 -> E4M3 encoding: size, NULL and alignment checks
    assert L.fp8_e4m3_from_f32(p16, -1, p16, None) == 2
    assert L.fp8_e4m3_from_f32(None, 0, None, None) == 0
    assert L.fp8_e4m3_from_f32(None, 8, p16, None) == 1
    assert L.fp8_e4m3_from_f32(p16, 8, None, None) == 1
    assert L.fp8_e4m3_from_f32(_u(0x10004), 8, p16, None) == 3
    assert L.fp8_e4m3_from_f32(p16, 8, _u(0x10002), None) == 3
    # group-scale check arguments
    assert L.w8_check_group_scales(None, 3) == 1
    assert L.w8_check_group_scales(arr, 0) == 2


def test_zero_rows_is_a_noop(L):
    p16 = _u(0x10000)
    arr = (ctypes.c_void_p * 3)(0x10000, 0x10000, 0x10000)
    ns = (ctypes.c_int64 * 3)(16, 16, 16)
    assert L.fp8_quant_static(p16, 0, 16, 16, p16, p16, 16, None) == 0
    assert L.fp8_linear_w8a8(p16, 0, 0, 16, p16, 16, p16, p16, p16, None, None) == 0
    assert L.fp8_linear_w8a16(p16, 0, 0, 16, p16, 16, p16, p16, None, None) == 0
    assert L.qkv_shared_quant_gemm(0, p16, 0, 16, p16, 3, arr, ns, arr, arr, None, None) == 0
    assert L.swiglu_2in_fp8(p16, p16, 0, 16, p16, p16, None) == 0
    assert L.swiglu_2in_bf16(p16, p16, 0, 16, p16, None) == 0


def test_non_dense_rows_are_refused(L):
    """A row pitch other than the row length is refused with W8_ERR_STRIDE
    before anything else is looked at (TensorRT-LLM PR #17476, Test
    Coverage: the op rejects non-contiguous inputs)."""
    p16 = _u(0x10000)
    for ldx, ldq in ((32, 16), (16, 32), (8, 16), (16, 0), (-1, 16), (16, -1)):
        assert L.fp8_quant_static(p16, 4, 16, ldx, p16, p16, ldq, None) == 4
        assert b"dense" in L.w8_last_error()
    # refused even for zero rows and before the NULL check
    assert L.fp8_quant_static(None, 0, 16, 32, None, None, 16, None) == 4
    # dense rows pass validation (M == 0: nothing is launched)
    assert L.fp8_quant_static(p16, 0, 4096, 4096, p16, p16, 4096, None) == 0


def test_binding_reports_row_pitch():
    """The binding hands the library the tensor's real row pitch (or -1 for
    a layout that has none), so a strided view reaches the library's refusal."""
    import torch
    from w8a16_linear_gb300.binding import _row_pitch
    x = torch.empty((6, 64), dtype=torch.bfloat16)
    assert _row_pitch(x) == 64
    assert _row_pitch(x[:, :32]) == 64          # a column slice keeps the parent's pitch
    assert _row_pitch(x.t()) == -1              # columns not contiguous
    assert _row_pitch(x.view(2, 3, 64)) == 64
    assert _row_pitch(torch.empty((2, 3, 80))[:, :, :64]) == 80
    assert _row_pitch(torch.empty((4, 3, 64))[::2]) == -1   # every other batch: rows not packed


def test_swiglu_variant_validation_before_any_cuda_call(L):
    from w8a16_linear_gb300 import binding as b
    p16 = _u(0x10000)
    ok = b.SwigluParams(1, 7.0, 1.702, 1.0)
    ref = ctypes.byref
    # shape, NULL, alignment as the plain SwiGLU
    assert L.swiglu_2in_ex_fp8(p16, p16, 0, 4, 24, ref(ok), p16, p16, None) == 2
    assert L.swiglu_2in_ex_fp8(p16, p16, 0, 4, 16, ref(ok), None, p16, None) == 1
    assert L.swiglu_2in_ex_16(p16, _u(0x10004), 0, 4, 16, ref(ok), p16, None) == 3
    # input dtype: bf16 (0) or f16 (2) only
    assert L.swiglu_2in_ex_16(p16, p16, 1, 4, 16, ref(ok), p16, None) == 5
    # parameters
    assert L.swiglu_2in_ex_16(p16, p16, 0, 4, 16, None, p16, None) == 1
    for bad in (b.SwigluParams(1, 0.0, 1.0, 0.0), b.SwigluParams(1, -1.0, 1.0, 0.0),
                b.SwigluParams(1, float("inf"), 1.0, 0.0), b.SwigluParams(0, 0.0, float("nan"), 0.0),
                b.SwigluParams(0, 0.0, 1.0, float("inf"))):
        assert L.swiglu_2in_ex_fp8(p16, p16, 2, 4, 16, ref(bad), p16, p16, None) == 11
    assert b"swiglu_2in_ex_fp8" in L.w8_last_error()
    # a limit that is not applied is not checked
    assert L.swiglu_2in_ex_16(p16, p16, 2, 0, 16, ref(b.SwigluParams(0, -5.0, 1.0, 0.0)), p16, None) == 0
    # zero rows: no launch
    assert L.swiglu_2in_ex_fp8(p16, p16, 0, 0, 16, ref(ok), p16, p16, None) == 0
    assert L.swiglu_2in_ex_16(p16, p16, 2, 0, 16, ref(ok), p16, None) == 0


def test_ln_modulate_quant_validation_before_any_cuda_call(L):
    p16, nul = _u(0x10000), None
    f = L.ln_modulate_quant
    # (x, M, K, shift, scale, rows_per_sample, eps, s_in, q, h, stream)
    assert f(p16, 4, 12, p16, p16, 4, 1e-6, p16, p16, nul, nul) == 2        # K % 8
    assert f(p16, 4, 8200, p16, p16, 4, 1e-6, p16, p16, nul, nul) == 2      # K > 8192
    assert f(p16, 4, 0, p16, p16, 4, 1e-6, p16, p16, nul, nul) == 2
    assert f(p16, -1, 16, p16, p16, 1, 1e-6, p16, p16, nul, nul) == 2
    assert f(p16, 6, 16, p16, p16, 4, 1e-6, p16, p16, nul, nul) == 2        # 4 does not divide 6
    assert f(p16, 6, 16, p16, p16, 0, 1e-6, p16, p16, nul, nul) == 2
    for eps in (-1e-6, float("nan"), float("inf")):
        assert f(p16, 4, 16, p16, p16, 4, eps, p16, p16, nul, nul) == 11
    assert f(nul, 4, 16, p16, p16, 4, 1e-6, p16, p16, nul, nul) == 1
    assert f(p16, 4, 16, nul, p16, 4, 1e-6, p16, p16, nul, nul) == 1
    assert f(p16, 4, 16, p16, p16, 4, 1e-6, p16, nul, nul, nul) == 1        # no output
    assert f(p16, 4, 16, p16, p16, 4, 1e-6, nul, p16, nul, nul) == 1        # q without s_in
    assert f(p16, 4, 16, p16, _u(0x10008), 4, 1e-6, p16, p16, nul, nul) == 3
    assert f(p16, 4, 16, p16, p16, 4, 1e-6, nul, nul, _u(0x10004), nul) == 3
    assert b"ln_modulate_quant" in L.w8_last_error()
    assert f(p16, 0, 16, p16, p16, 1, 1e-6, p16, p16, nul, nul) == 0        # zero rows: no launch
    assert f(p16, 0, 4096, nul, nul, 7, 0.0, nul, nul, nul, nul) == 0


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    """No fallback: with the library absent every entry point raises."""
    from w8a16_linear_gb300 import binding as b
    monkeypatch.setattr(b, "_lib", None)
    monkeypatch.setattr(b, "LIB_PATH", str(tmp_path / "libw8lin.so"))
    with pytest.raises(ImportError):
        b.abi_version()
    with pytest.raises(ImportError):
        b.step_policy_dispatch(None, 0, 8)


def test_fused_swiglu_options_validation_before_any_cuda_call(L):
    """The fused gate/up entries with SwiGLU options refuse NULL or
    out-of-range options (W8_ERR_NULL, W8_ERR_PARAM) before touching the
    operands, and a zero-row call with valid options launches nothing."""
    from w8a16_linear_gb300 import binding as b
    p16 = _u(0x10000)
    ref = ctypes.byref
    ok = b.SwigluParams(1, 7.0, 1.702, 1.0)
    bad = b.SwigluParams(1, -1.0, 1.0, 0.0)

    def fp8(prm, M):
        return L.gate_up_swiglu_ex_fp8(p16, 1, M, 16, p16, p16, p16, 16, p16, p16, prm, p16, p16, p16, None)

    def bf16(prm, M):
        return L.bf16_gate_up_swiglu_ex(p16, M, 16, p16, p16, 16, prm, p16, None)

    assert fp8(None, 4) == 1
    assert fp8(ref(bad), 4) == 11
    assert b"gate_up_swiglu_ex_fp8" in L.w8_last_error()
    assert fp8(ref(b.SwigluParams(0, 0.0, float("nan"), 0.0)), 4) == 11
    assert fp8(ref(ok), 0) == 0
    assert bf16(None, 4) == 1
    assert bf16(ref(bad), 4) == 11
    assert b"bf16_gate_up_swiglu_ex" in L.w8_last_error()
    assert bf16(ref(ok), 0) == 0
    # operand checks as the plain entries: K not a multiple of 16
    assert L.gate_up_swiglu_ex_fp8(p16, 1, 4, 24, p16, p16, p16, 16, p16, p16, ref(ok), p16, p16, p16,
                                   None) == L.gate_up_swiglu_fp8(p16, 1, 4, 24, p16, p16, p16, 16, p16, p16, p16,
                                                                 p16, p16, None)

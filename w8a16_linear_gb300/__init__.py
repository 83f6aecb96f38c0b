"""Static per-tensor FP8 linear layer (W8A8 / W8A16) for GB300, sm_103a.

The compute runs in ``libw8lin.so`` (CUDA kernels behind the C ABI of
``include/w8lin.h``); this package holds its ctypes binding, the build
script and the seeded synthetic-input generators.
"""

from .binding import (  # noqa: F401
    W8Error, StepPolicy, SwigluParams, DTYPE_BF16, DTYPE_E4M3, DTYPE_F16, MODE_A8, MODE_A16,
    abi_version, device_check, poll_device_error, selftest_timeout,
    fp8_quant_static, fp8_linear_w8a8, fp8_linear_w8a16, qkv_shared_quant_gemm, fp8_linear_w8a8_group, gate_up_swiglu_fp8, fp8_linear_w8a8_noalloc,
    fp8_e4m3_from_f32, fp8_dequant_weight, w8a16_workspace, bf16_linear_group, bf16_gate_up_swiglu,
    ln_modulate_quant, ln_modulate_bf16,
    swiglu_2in_fp8, swiglu_2in_bf16, swiglu_2in_ex_fp8, swiglu_2in_ex_16, step_policy_dispatch, step_policy_parse, check_group_scales,
)

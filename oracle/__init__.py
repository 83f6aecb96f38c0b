"""CPU oracle for the static per-tensor FP8 linear path.

TEST INFRASTRUCTURE ONLY.  Nothing in the product package imports this
package.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may call it.

Every function is written from the pages that describe the method and cites
the passage it follows:

* [P1] diffusers issue #15170, "Cosmos 3 docs: FP8 snippet fails at the first
  W8A8 step without importing ModelOpt's FP8 GEMM backend" (section *Logs*:
  the ``(4, 3) bit`` per-tensor quantizers and their calibrated amax).
* [P2] cosmos-framework PR #157, "feat: load ModelOpt static-FP8 checkpoints
  via TorchAO" (section *Verification*: ``aten::div -> aten::clamp ->
  _RoundToFloat8`` with the exported ``input_scale``; ``aten::_scaled_mm``).
* [P3] diffusers PR #14664, "[Cosmos3] Mixed W8A8/W8A16 denoising for ModelOpt
  FP8 checkpoints" (section *Behavior*: first 3 + last 3 steps W8A16 as
  "dequant + F.linear", middle steps W8A8; section *Tests*: "1-step stays
  native", the 8- and 35-step traces).
* [P4] TensorRT-LLM PR #17476, "Load static FP8 Cosmos3 Nano/Super checkpoints
  without re-quantizing them" (sections *Description*, *What changed*,
  *Denoising-step activation precision*, *Test Coverage*).

Modules: ``e4m3`` (the FP8 codec), ``bf16`` and ``fp16`` (16-bit codecs),
``linear`` (quantization, W8A8 / W8A16, the dequantized weight, the max(s)
re-quantization, the sharing group), ``swiglu`` (the SwiGLU specification
and its options), ``policy`` (the per-step precision policy and its JSON),
``norm`` (the modulated LayerNorm that produces a linear layer's input, and
the static quantization fused after it).

Floating point: the GEMM oracles work in float64 on exactly decoded
operands (the definition written out).  Where a floating-point value decides
an integer -- an E4M3 code or a bf16 bit pattern -- the oracle takes that
decision in IEEE binary32, the precision of the kernel, as a plain sequence
of numpy float32 operations (no fused multiply-add anywhere).
"""

from .e4m3 import (E4M3_MAX, e4m3_decode, e4m3_encode, e4m3_all_values)
from .bf16 import bf16_decode, bf16_round
from .fp16 import fp16_decode, fp16_round
from .linear import (quant_static, linear_w8a8, linear_w8a16,
                     dequant_weight_bf16, requant_onto_max_scale,
                     qkv_shared_quant_gemm)
from .swiglu import (exp_spec, swiglu_2in_fp8, swiglu_2in_bf16, swiglu_h, swiglu_h_ex,
                     swiglu_2in_ex_fp8, swiglu_2in_ex_16)
from .policy import StepPolicy, PolicyError, step_mode, parse_policy, A8, A16
from .norm import ln_modulate, ln_modulate_bf16, ln_modulate_quant

__all__ = [
    "E4M3_MAX", "e4m3_decode", "e4m3_encode", "e4m3_all_values",
    "bf16_decode", "bf16_round", "fp16_decode", "fp16_round",
    "quant_static", "linear_w8a8", "linear_w8a16", "dequant_weight_bf16",
    "requant_onto_max_scale", "qkv_shared_quant_gemm",
    "exp_spec", "swiglu_2in_fp8", "swiglu_2in_bf16", "swiglu_h", "swiglu_h_ex",
    "swiglu_2in_ex_fp8", "swiglu_2in_ex_16",
    "StepPolicy", "PolicyError", "step_mode", "parse_policy", "A8", "A16",
    "ln_modulate", "ln_modulate_bf16", "ln_modulate_quant",
]

// Device-side static per-tensor activation quantization, shared by the
// standalone quantization kernel, the fused LayerNorm producer and the
// W8A8 GEMM that quantizes its own activation ahead of its tiles:
// q = E4M3_satRNE(fl32(x / s_in)), one correctly rounded binary32 division
// then one saturating round-to-nearest-even to E4M3 (cosmos-framework PR
// #157, "feat: load ModelOpt static-FP8 checkpoints via TorchAO", section
// Verification: div -> clamp -> round-to-float8 with the exported
// input_scale).
#pragma once

#include <cstdint>

#include "ptx.cuh"
#include "swiglu_spec.cuh"

namespace w8 {
namespace {

// q = E4M3(fl32(x / s)).  Fast value f = fl32(x * fl32(1/s)): two roundings
// of 2^-24 on the exact quotient against the specification's one, so
// |f / fl32(x / s) - 1| <= 3 * 2^-24 when s and 1/s are normal (a binary32
// subnormal f is below every E4M3 rounding boundary, as is the specified
// value).  The bracket of 2^-21 (swiglu_spec.cuh) settles every pair whose
// code cannot differ; the rest take the correctly rounded division.

constexpr float kQuantBracketLo = 0.99999952316284180f;   // 1 - 2^-21
constexpr float kQuantBracketHi = 1.00000047683715820f;   // 1 + 2^-21

__device__ __forceinline__ uint32_t quant_pair(uint32_t w, float s, float r, bool exact_only) {
  const float v0 = bf16_lo(w), v1 = bf16_hi(w);
  bool unsettled;
  const uint32_t code = e4m3x2_bracket(mul2(F2{v0, v1}, splat(r)), kQuantBracketLo,
                                       kQuantBracketHi, unsettled);
  if (exact_only | unsettled) return cvt_e4m3x2(__fdiv_rn(v0, s), __fdiv_rn(v1, s));
  return code;
}

// The specification's codes of one packed bf16 pair: correctly rounded
// division, then the E4M3 rounding.  Kept out of line: it is the rare path of
// the fused producer's row fix-up.
__device__ __noinline__ uint32_t quant_pair_exact(uint32_t w, float s) {
  return cvt_e4m3x2(__fdiv_rn(bf16_lo(w), s), __fdiv_rn(bf16_hi(w), s));
}

}  // namespace
}  // namespace w8

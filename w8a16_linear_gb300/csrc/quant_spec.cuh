// Device-side static per-tensor activation quantization, shared by the
// standalone quantization kernel and the fused LayerNorm producer:
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

// q = E4M3(fl32(x / s)) from products with r = fl32(1/s).  The two ends of
// the bracket are fl(x * fl(r (1 - 2^-21))) and fl(x * fl(r (1 + 2^-21))):
// against the exact quotient, r, the scaled reciprocal and the product each
// round once (2^-24), the specification's quotient once more, so the ends lie
// on either side of fl32(x / s) while 4 * 2^-24 < 2^-21.  That holds when s and
// r are normal and r >= 2^-125, which keeps the scaled reciprocals normal (a
// product in the binary32 subnormal range is below every E4M3 rounding
// boundary, as is the specified value).  Equal codes at both ends are the
// specified code; the rest take the correctly rounded division.
//
// When s = +-2^k, x * r is the same real number as x / s, so fl32(x * r) is
// the specified value itself and both ends are r: no pair is ever unsettled.
// At such scales one bf16 x in 16 is an E4M3 midpoint, which the bracket
// could never settle.

constexpr float kQuantBracketLo = 0.99999952316284180f;   // 1 - 2^-21
constexpr float kQuantBracketHi = 1.00000047683715820f;   // 1 + 2^-21

struct QuantBracket {
  float lo, hi;       // reciprocal of s times the bracket's ends
  bool exact_only;    // s outside the range above: every pair divides
};

__device__ __forceinline__ QuantBracket quant_bracket(float s) {
  const float r = __frcp_rn(s);
  const bool pow2 = (__float_as_uint(s) & 0x007FFFFFu) == 0u;   // with s normal: s = +-2^k
  QuantBracket b;
  b.exact_only = !scale_is_fast(s, r) || fabsf(r) < 2.35098870e-38f;   // 2^-125
  b.lo = pow2 ? r : __fmul_rn(r, kQuantBracketLo);
  b.hi = pow2 ? r : __fmul_rn(r, kQuantBracketHi);
  return b;
}

__device__ __forceinline__ uint32_t quant_pair(uint32_t w, float s, const QuantBracket& b) {
  const float v0 = bf16_lo(w), v1 = bf16_hi(w);
  bool unsettled;
  const uint32_t code = e4m3x2_bracket(F2{v0, v1}, b.lo, b.hi, unsettled);
  if (b.exact_only | unsettled) return cvt_e4m3x2(__fdiv_rn(v0, s), __fdiv_rn(v1, s));
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

// Device-side binary32 specification of the two-input SwiGLU and its
// exactness-guarded fast evaluation, shared by the elementwise SwiGLU
// kernels and the fused gate/up GEMM epilogue (TensorRT-LLM PR #17476,
// "Load static FP8 Cosmos3 Nano/Super checkpoints without re-quantizing
// them", section What changed: SiLU(G) * U from two tensors, quantized
// directly for the FP8 down projection).
//
// Specification (the pages fix only SiLU(G) * U and the FP8 output):
//   p = g * u;  e = exp_spec(-g);  h = p / (1 + e)
//   FP8 out:  E4M3_satRNE(h / s_out);  bf16 out: bf16_RNE(h)
// exp_spec: Cody-Waite reduction (Cody and Waite, Software Manual for the
// Elementary Functions, 1980) with n = rint(t * fl32(1/ln2)),
// r = (t - n*LN2_HI) - n*LN2_LO, LN2_HI = ln 2 with 12 low significand bits
// cleared, LN2_LO = fl32(ln 2 - LN2_HI); degree-7 Taylor polynomial of exp(r)
// in Horner form with coefficients fl32(1/k!), separate multiply and add;
// result scaled by 2^(n>>1) then 2^(n-(n>>1)); t > 88 gives +inf, t < -88
// gives 0.
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace w8 {

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// ---- packed binary32 pairs: two independent round-to-nearest operations per
// instruction.  A packed multiply whose result feeds a packed add may come out
// fused (one rounding); the exact specification therefore never uses them in
// that pattern (exp_spec1 is scalar), and the fast paths use explicit fused
// multiply-adds where they want them.
struct F2 {
  float x, y;
};

__device__ __forceinline__ F2 mul2(F2 a, F2 b) {
  F2 r;
  asm("{.reg .b64 p, q, d;\n\tmov.b64 p, {%2, %3};\n\tmov.b64 q, {%4, %5};\n\t"
      "mul.rn.f32x2 d, p, q;\n\tmov.b64 {%0, %1}, d;}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}

__device__ __forceinline__ F2 add2(F2 a, F2 b) {
  F2 r;
  asm("{.reg .b64 p, q, d;\n\tmov.b64 p, {%2, %3};\n\tmov.b64 q, {%4, %5};\n\t"
      "add.rn.f32x2 d, p, q;\n\tmov.b64 {%0, %1}, d;}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}

// a * b + c with one rounding per element (the fast paths only).
__device__ __forceinline__ F2 fma2(F2 a, F2 b, F2 c) {
  F2 r;
  asm("{.reg .b64 p, q, s, d;\n\tmov.b64 p, {%2, %3};\n\tmov.b64 q, {%4, %5};\n\t"
      "mov.b64 s, {%6, %7};\n\tfma.rn.f32x2 d, p, q, s;\n\tmov.b64 {%0, %1}, d;}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return r;
}

__device__ __forceinline__ F2 splat(float v) { return F2{v, v}; }
__device__ __forceinline__ F2 neg(F2 a) { return F2{-a.x, -a.y}; }

__device__ __forceinline__ float pow2i(int k) { return __int_as_float((k + 127) << 23); }

// exp_spec of one argument, exactly as specified: every multiply and add is a
// separately rounded __fmul_rn / __fadd_rn, which the compiler never merges
// into a fused multiply-add.  (The packed f32x2 multiply and add are not used
// here: a multiply feeding an add was observed to come out fused, i.e. with
// one rounding instead of two.)
__device__ __forceinline__ float exp_spec1(float t) {
  const float kL2E = __uint_as_float(0x3FB8AA3Bu);
  const float kLn2Hi = __uint_as_float(0x3F317000u);
  const float kLn2Lo = __uint_as_float(0x3805FDF4u);
  const float tc = fminf(fmaxf(t, -88.0f), 88.0f);
  const float n = rintf(__fmul_rn(tc, kL2E));
  float r = __fadd_rn(tc, -__fmul_rn(n, kLn2Hi));
  r = __fadd_rn(r, -__fmul_rn(n, kLn2Lo));
  float q = __uint_as_float(0x39500D01u);                     // 1/k!, k = 7 .. 0
  q = __fadd_rn(__fmul_rn(q, r), __uint_as_float(0x3AB60B61u));
  q = __fadd_rn(__fmul_rn(q, r), __uint_as_float(0x3C088889u));
  q = __fadd_rn(__fmul_rn(q, r), __uint_as_float(0x3D2AAAABu));
  q = __fadd_rn(__fmul_rn(q, r), __uint_as_float(0x3E2AAAABu));
  q = __fadd_rn(__fmul_rn(q, r), 0.5f);
  q = __fadd_rn(__fmul_rn(q, r), 1.0f);
  q = __fadd_rn(__fmul_rn(q, r), 1.0f);
  const int ni = __float2int_rn(n);
  const int a = ni >> 1;
  const float res = __fmul_rn(__fmul_rn(q, pow2i(a)), pow2i(ni - a));
  return (t > 88.0f) ? __int_as_float(0x7F800000) : ((t < -88.0f) ? 0.0f : res);
}

__device__ __forceinline__ F2 exp_spec2(F2 t) { return F2{exp_spec1(t.x), exp_spec1(t.y)}; }

// d' ~ 1 + exp_spec(t) for the fast paths: the specification's reduction and
// polynomial evaluated with fused multiply-adds, the argument clamped to
// [-17, 88] and the final 2^n scaling done by adding n to the exponent field.
// Checked exhaustively on the host over every binary32 t in [-17, 88]: d' is
// within 2 ulp (4 * 2^-24 relative) of the specified d, and equal to it on
// 99.6% of the arguments; for t <= -17 the specified d is exactly 1, as is
// d'.  Arguments above 88 are clamped too; they give d' >= 2^126, which the
// guard sends to the exact path (h_needs_exact).
__device__ __forceinline__ F2 dplus1_fast(F2 t) {
  const float kL2E = __uint_as_float(0x3FB8AA3Bu);
  const float kLn2Hi = __uint_as_float(0x3F317000u);
  const float kLn2Lo = __uint_as_float(0x3805FDF4u);
  const F2 tc{fminf(fmaxf(t.x, -17.0f), 88.0f), fminf(fmaxf(t.y, -17.0f), 88.0f)};
  const F2 nl = mul2(tc, splat(kL2E));
  const F2 n{rintf(nl.x), rintf(nl.y)};
  F2 r = fma2(neg(n), splat(kLn2Hi), tc);
  r = fma2(neg(n), splat(kLn2Lo), r);
  F2 q = splat(__uint_as_float(0x39500D01u));
  q = fma2(q, r, splat(__uint_as_float(0x3AB60B61u)));
  q = fma2(q, r, splat(__uint_as_float(0x3C088889u)));
  q = fma2(q, r, splat(__uint_as_float(0x3D2AAAABu)));
  q = fma2(q, r, splat(__uint_as_float(0x3E2AAAABu)));
  q = fma2(q, r, splat(0.5f));
  q = fma2(q, r, splat(1.0f));
  q = fma2(q, r, splat(1.0f));
  const F2 e{__int_as_float(__float_as_int(q.x) + (__float2int_rn(n.x) << 23)),
             __int_as_float(__float_as_int(q.y) + (__float2int_rn(n.y) << 23))};
  return add2(splat(1.0f), e);
}

__device__ __forceinline__ float rcp_approx(float d) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(d));
  return r;
}

// ---- exactness guards.
//
// E4M3 (bracket test): a fast value f with |f / v - 1| <= E of the specified
// value v, E < eps - 2^-24, gives the specified code unless a rounding
// boundary of the saturating round-to-nearest-even conversion lies between
// f (1 - eps) and f (1 + eps).  Conversion is monotonic, so converting both
// ends (each rounded to binary32, hence the 2^-24) and comparing the codes
// settles it: equal codes are the code of every value in between, v
// included.  This holds in the normal and the subnormal E4M3 range, at
// saturation, for zeros (sign kept) and NaN.  A pair of elements is settled
// together (one packed conversion per end).
__device__ __forceinline__ uint32_t e4m3x2_bracket(F2 f, float lo_factor, float hi_factor,
                                                   bool& unsettled) {
  const F2 lo = mul2(f, splat(lo_factor));
  const F2 hi = mul2(f, splat(hi_factor));
  const uint32_t clo = cvt_e4m3x2(lo.x, lo.y);
  const uint32_t chi = cvt_e4m3x2(hi.x, hi.y);
  unsettled = clo != chi;
  return chi;
}

// bf16 (window test): in the normal range every bf16 rounding midpoint has
// the low 16 significand bits of the binary32 value equal to 0x8000, so a
// fast value within W binary32 ulps of the specified one needs the exact path
// only when its low bits are within W of that pattern.
template <int W>
__device__ __forceinline__ bool near_bf16_midpoint(float f) {
  const uint32_t b = __float_as_uint(f);
  return ((b & 0xFFFFu) + (uint32_t)W - 0x8000u) <= (uint32_t)(2 * W);
}

__device__ __forceinline__ uint4 ldg16(const void* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}

__device__ __forceinline__ bool scale_is_fast(float s, float r) {
  const float kMinNormal = 1.17549435e-38f;
  return fabsf(s) >= kMinNormal && fabsf(r) >= kMinNormal && fabsf(r) < __int_as_float(0x7F800000);
}

// ------------------------------------------------------------------ swiglu
//
// FP8 output.  Fast value, elementwise: p = g * u (exact, as specified),
// d' = fl(1 + __expf(-g)), q' = fl(fl(p * rcp.approx(d')) * fl(1/s)).
// Error budget against the specified q = fl(fl(p / d) / s), relative, in
// units of 2^-24, for gates g >= -16 (x = -g <= 16):
//   __expf(x): documented within 2 + floor(|1.173 x|) ulp of e^x, at most 20
//     ulp (40) for 0 < x <= 16; for x <= 0 its share of d = 1 + e is below
//     2^-23 (2) because e / (1 + e) shrinks faster than the bound grows;
//     plus the rounding of 1 + e (1)                                      <= 41
//   the specified d against 1 + e^x (exp_spec checked exhaustively on
//     every bf16 argument on the host: within 1.5)                       <= 1.5
//   rcp.approx: documented within 1 ulp                                    <= 2
//   roundings of p * r, of fl(1/s), of q' and the specification's two      <= 5
// in all below 50, under the bracket's 2^-18 - 2^-24 (63).  Gates below
// -16 (and -inf) take the exact path.  A scale with |1/s| > 2^20 (or 1/s not
// normal) sends every element to the exact path: with |1/s| <= 2^20 a
// binary32-subnormal h' (absolute error 2^-149, not relative) maps to
// |q| < 2^-106, code 0 either way, with the same sign.
//
// bf16 output.  hf = fl(p * rcp.approx(d')) with d' = dplus1_fast (within
// 4 * 2^-24 of the specified d), for d' < 2^126: relative error against the
// specified h at most 4 (d') + 2 (rcp.approx, 1 ulp) + 1 + 1 (the two
// roundings) = 8 * 2^-24, i.e. at most 8 ulp of hf; the window is 12 ulp.
// Elements where hf is within the window of a bf16 midpoint, where
// d' >= 2^126 (the reciprocal flushes) or where hf is tiny (binary32
// subnormal range) take the correctly rounded division with the exactly
// specified denominator.

constexpr float kFp8BracketLo = 0.999996185302734375f;   // 1 - 2^-18
constexpr float kFp8BracketHi = 1.000003814697265625f;   // 1 + 2^-18

__device__ __forceinline__ bool swiglu_fp8_scale_is_fast(float s, float rs) {
  return scale_is_fast(s, rs) && fabsf(rs) <= 1048576.0f;            // |1/s| <= 2^20
}

__device__ __forceinline__ bool h_needs_exact(float p, float d, float hf) {
  const float ah = fabsf(hf);
  return !(d < 8.507059e37f)                                       // d >= 2^126 (or NaN)
         | ((ah < 7.888609e-31f) & ((ah != 0.0f) | (p != 0.0f)));  // |hf| < 2^-100
}

// Two elements: gate word and up word each hold a bf16 pair.  p exact, d the
// fast form of 1 + exp_spec(-g) (exact except where the guards catch it).
__device__ __forceinline__ void swiglu_pd(uint32_t gw, uint32_t uw, F2& p, F2& d) {
  const F2 g{bf16_lo(gw), bf16_hi(gw)};
  p = mul2(g, F2{bf16_lo(uw), bf16_hi(uw)});
  d = dplus1_fast(neg(g));
}

// 1 + exp_spec(-g) exactly as specified (every argument), for the exact path.
__device__ __forceinline__ F2 swiglu_d_exact(uint32_t gw) {
  const F2 g{bf16_lo(gw), bf16_hi(gw)};
  return add2(splat(1.0f), exp_spec2(neg(g)));
}

// The specified E4M3 codes of a pair, by correctly rounded divisions.
__device__ __forceinline__ uint32_t swiglu_fp8_exact_pair(uint32_t gw, uint32_t uw, float s) {
  const F2 p = mul2(F2{bf16_lo(gw), bf16_hi(gw)}, F2{bf16_lo(uw), bf16_hi(uw)});
  const F2 d = swiglu_d_exact(gw);
  return cvt_e4m3x2(__fdiv_rn(__fdiv_rn(p.x, d.x), s), __fdiv_rn(__fdiv_rn(p.y, d.y), s));
}

// Fast codes of a pair; `unsettled` when the bracket does not settle them or
// a gate is below -16.
__device__ __forceinline__ uint32_t swiglu_fp8_fast_pair(uint32_t gw, uint32_t uw, float rs,
                                                         bool& unsettled) {
  const F2 g{bf16_lo(gw), bf16_hi(gw)};
  const F2 p = mul2(g, F2{bf16_lo(uw), bf16_hi(uw)});
  const F2 d = add2(splat(1.0f), F2{__expf(-g.x), __expf(-g.y)});
  const F2 hf = mul2(p, F2{rcp_approx(d.x), rcp_approx(d.y)});
  const uint32_t code = e4m3x2_bracket(mul2(hf, splat(rs)), kFp8BracketLo, kFp8BracketHi, unsettled);
  unsettled |= (g.x < -16.0f) | (g.y < -16.0f);
  return code;
}

__device__ __forceinline__ uint32_t swiglu_fp8_pair(uint32_t gw, uint32_t uw, float s, float rs,
                                                    bool exact_only) {
  bool unsettled;
  const uint32_t code = swiglu_fp8_fast_pair(gw, uw, rs, unsettled);
  if (exact_only | unsettled) return swiglu_fp8_exact_pair(gw, uw, s);   // rare
  return code;
}

__device__ __forceinline__ uint32_t swiglu_bf16_pair(uint32_t gw, uint32_t uw) {
  F2 p, d;
  swiglu_pd(gw, uw, p, d);
  F2 h = mul2(p, F2{rcp_approx(d.x), rcp_approx(d.y)});
  if (h_needs_exact(p.x, d.x, h.x) | h_needs_exact(p.y, d.y, h.y) | near_bf16_midpoint<12>(h.x) |
      near_bf16_midpoint<12>(h.y)) {
    const F2 de = swiglu_d_exact(gw);
    if (h_needs_exact(p.x, d.x, h.x) || near_bf16_midpoint<12>(h.x)) h.x = __fdiv_rn(p.x, de.x);
    if (h_needs_exact(p.y, d.y, h.y) || near_bf16_midpoint<12>(h.y)) h.y = __fdiv_rn(p.y, de.y);
  }
  return cvt_bf16x2(h.x, h.y);
}

// 16 elements at once (the fused gate/up epilogue): the fast codes of all 8
// pairs are computed straight-line so that independent pairs interleave, a
// bitmask records the unsettled pairs, and a single, rarely taken branch
// recomputes those exactly.  gw/uw: 8 words of two bf16 each; codes: 16 E4M3
// codes, element 0 in the low byte of codes[0].
__device__ __forceinline__ void swiglu_fp8_x16(const uint32_t (&gw)[8], const uint32_t (&uw)[8],
                                               float s, float rs, bool exact_only,
                                               uint32_t (&codes)[4]) {
  uint32_t c[8];
  uint32_t bad = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    bool unsettled;
    c[j] = swiglu_fp8_fast_pair(gw[j], uw[j], rs, unsettled);
    bad |= (uint32_t)unsettled << j;
  }
  if (exact_only) bad = 0xFFu;
  if (bad) {
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (bad & (1u << j)) c[j] = swiglu_fp8_exact_pair(gw[j], uw[j], s);
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) codes[j] = c[2 * j] | (c[2 * j + 1] << 16);
}

// ------------------------------------------------------------------ variants
//
// The options the two-input SwiGLU is tested with besides the plain form
// (TensorRT-LLM PR #17476, section Test Coverage: BF16 / FP16 inputs,
// swiglu_limit, swiglu_alpha + swiglu_beta, FP8 output).  The pages name them
// only; the specification here is the clamped, shifted SwiGLU of the public
// gpt-oss MLP:
//   g = min(g, L), u = clamp(u, -L, L)            (limit L; a NaN stays NaN)
//   t = fl32(a * g)                               (alpha a)
//   u = fl32(u + b)                               (beta b; skipped when b == 0)
//   p = fl32(g * u), h = fl32(p / fl32(1 + exp_spec(-t)))
// With a = 1, b = 0 and no limit this is the base specification bit for bit.
// The fast paths are the base ones with t in place of g: FP8 output through
// __expf and the 2^-18 bracket (exact path for t < -16); 16-bit output with
// p * rcp.approx(d'), d' = dplus1_fast (within 8 * 2^-24 of the specified h,
// as for the bf16 output above) and a 2^-20 bracket on the packed 16-bit
// conversion, plus the d' >= 2^126 and tiny-h guards.

struct SwigluParams {
  float limit;     // used when has_limit
  float alpha;
  float beta;      // added to up when has_beta
  int has_limit;
  int has_beta;
};

constexpr float k16BracketLo = 0.99999904632568359375f;   // 1 - 2^-20
constexpr float k16BracketHi = 1.00000095367431640625f;   // 1 + 2^-20

template <bool kF16>
__device__ __forceinline__ F2 unpack16(uint32_t w) {
  if constexpr (kF16) {
    F2 r;
    f16x2_to_f32(w, r.x, r.y);
    return r;
  } else {
    return F2{bf16_lo(w), bf16_hi(w)};
  }
}

// NaN-propagating min / max (a NaN input gives NaN, as the clamps specify).
__device__ __forceinline__ float min_nan(float a, float b) {
  float r;
  asm("min.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ float max_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ float clamp_hi(float v, float lim) { return min_nan(v, lim); }
__device__ __forceinline__ float clamp_sym(float v, float lim) { return min_nan(max_nan(v, -lim), lim); }

// t = fl32(a * g) and p = fl32(g * (u + b)) of a pair, after the clamps.
template <bool kF16>
__device__ __forceinline__ void swiglu_ex_operands(uint32_t gw, uint32_t uw, const SwigluParams& pr,
                                                   F2& t, F2& p) {
  F2 g = unpack16<kF16>(gw), u = unpack16<kF16>(uw);
  if (pr.has_limit) {
    g = F2{clamp_hi(g.x, pr.limit), clamp_hi(g.y, pr.limit)};
    u = F2{clamp_sym(u.x, pr.limit), clamp_sym(u.y, pr.limit)};
  }
  t = mul2(g, splat(pr.alpha));
  if (pr.has_beta) u = add2(u, splat(pr.beta));
  p = mul2(g, u);
}

template <bool kF16>
__device__ __forceinline__ uint32_t swiglu_ex_fp8_pair(uint32_t gw, uint32_t uw, const SwigluParams& pr,
                                                       float s, float rs, bool exact_only) {
  F2 t, p;
  swiglu_ex_operands<kF16>(gw, uw, pr, t, p);
  const F2 d = add2(splat(1.0f), F2{__expf(-t.x), __expf(-t.y)});
  const F2 hf = mul2(p, F2{rcp_approx(d.x), rcp_approx(d.y)});
  bool unsettled;
  const uint32_t code = e4m3x2_bracket(mul2(hf, splat(rs)), kFp8BracketLo, kFp8BracketHi, unsettled);
  if (exact_only | unsettled | (t.x < -16.0f) | (t.y < -16.0f)) {   // rare
    const F2 de = add2(splat(1.0f), exp_spec2(neg(t)));
    return cvt_e4m3x2(__fdiv_rn(__fdiv_rn(p.x, de.x), s), __fdiv_rn(__fdiv_rn(p.y, de.y), s));
  }
  return code;
}

// The specification's codes of one pair with the options (the rare path of
// swiglu_ex_fp8_x16): the operands again, the specified denominator, the
// correctly rounded divisions.
template <bool kF16>
__device__ __forceinline__ uint32_t swiglu_ex_fp8_exact_pair(uint32_t gw, uint32_t uw, const SwigluParams& pr,
                                                             float s) {
  F2 t, p;
  swiglu_ex_operands<kF16>(gw, uw, pr, t, p);
  const F2 de = add2(splat(1.0f), exp_spec2(neg(t)));
  return cvt_e4m3x2(__fdiv_rn(__fdiv_rn(p.x, de.x), s), __fdiv_rn(__fdiv_rn(p.y, de.y), s));
}

// swiglu_ex_fp8_pair over 8 packed pairs: the fast codes of all of them,
// then one rarely taken branch for the pairs the bracket cannot settle (or
// whose gate is below -16), as swiglu_fp8_x16 does for the plain form.  The
// codes are swiglu_ex_fp8_pair's, bit for bit.  For callers with registers to
// spare (the fused gate/up GEMM's epilogue).
template <bool kF16>
__device__ __forceinline__ void swiglu_ex_fp8_x16(const uint32_t (&gw)[8], const uint32_t (&uw)[8],
                                                  const SwigluParams& pr, float s, float rs, bool exact_only,
                                                  uint32_t (&codes)[4]) {
  uint32_t c[8];
  uint32_t bad = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    F2 t, p;
    swiglu_ex_operands<kF16>(gw[j], uw[j], pr, t, p);
    const F2 d = add2(splat(1.0f), F2{__expf(-t.x), __expf(-t.y)});
    const F2 hf = mul2(p, F2{rcp_approx(d.x), rcp_approx(d.y)});
    bool unsettled;
    c[j] = e4m3x2_bracket(mul2(hf, splat(rs)), kFp8BracketLo, kFp8BracketHi, unsettled);
    bad |= (uint32_t)(unsettled | (t.x < -16.0f) | (t.y < -16.0f)) << j;
  }
  if (exact_only) bad = 0xFFu;
  if (bad) {
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (bad & (1u << j)) c[j] = swiglu_ex_fp8_exact_pair<kF16>(gw[j], uw[j], pr, s);
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) codes[j] = c[2 * j] | (c[2 * j + 1] << 16);
}

__device__ __forceinline__ uint32_t cvt16x2(bool f16, float lo, float hi) {
  return f16 ? cvt_f16x2(lo, hi) : cvt_bf16x2(lo, hi);
}

template <bool kF16>
__device__ __forceinline__ uint32_t swiglu_ex_16_pair(uint32_t gw, uint32_t uw, const SwigluParams& pr) {
  F2 t, p;
  swiglu_ex_operands<kF16>(gw, uw, pr, t, p);
  const F2 d = dplus1_fast(neg(t));
  const F2 hf = mul2(p, F2{rcp_approx(d.x), rcp_approx(d.y)});
  const F2 lo = mul2(hf, splat(k16BracketLo));
  const F2 hi = mul2(hf, splat(k16BracketHi));
  const uint32_t clo = cvt16x2(kF16, lo.x, lo.y);
  const uint32_t chi = cvt16x2(kF16, hi.x, hi.y);
  if ((clo != chi) | h_needs_exact(p.x, d.x, hf.x) | h_needs_exact(p.y, d.y, hf.y)) {   // rare
    const F2 de = add2(splat(1.0f), exp_spec2(neg(t)));
    return cvt16x2(kF16, __fdiv_rn(p.x, de.x), __fdiv_rn(p.y, de.y));
  }
  return chi;
}

}  // namespace w8

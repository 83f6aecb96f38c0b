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
// instruction (never contracted into a fused multiply-add).
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

__device__ __forceinline__ F2 splat(float v) { return F2{v, v}; }
__device__ __forceinline__ F2 neg(F2 a) { return F2{-a.x, -a.y}; }

__device__ __forceinline__ float pow2i(int k) { return __int_as_float((k + 127) << 23); }

// exp_spec on two arguments at once (see the specification at the top).
__device__ __forceinline__ F2 exp_spec2(F2 t) {
  const float kL2E = __uint_as_float(0x3FB8AA3Bu);
  const float kLn2Hi = __uint_as_float(0x3F317000u);
  const float kLn2Lo = __uint_as_float(0x3805FDF4u);
  const F2 tc{fminf(fmaxf(t.x, -88.0f), 88.0f), fminf(fmaxf(t.y, -88.0f), 88.0f)};
  const F2 nl = mul2(tc, splat(kL2E));
  const F2 n{rintf(nl.x), rintf(nl.y)};
  F2 r = add2(tc, neg(mul2(n, splat(kLn2Hi))));
  r = add2(r, neg(mul2(n, splat(kLn2Lo))));
  // 1/k! rounded to binary32, k = 7 .. 0, Horner with separate multiply and add
  F2 q = splat(__uint_as_float(0x39500D01u));
  q = add2(mul2(q, r), splat(__uint_as_float(0x3AB60B61u)));
  q = add2(mul2(q, r), splat(__uint_as_float(0x3C088889u)));
  q = add2(mul2(q, r), splat(__uint_as_float(0x3D2AAAABu)));
  q = add2(mul2(q, r), splat(__uint_as_float(0x3E2AAAABu)));
  q = add2(mul2(q, r), splat(0.5f));
  q = add2(mul2(q, r), splat(1.0f));
  q = add2(mul2(q, r), splat(1.0f));
  const int n0 = __float2int_rn(n.x), n1 = __float2int_rn(n.y);
  const int a0 = n0 >> 1, a1 = n1 >> 1;
  F2 res = mul2(q, F2{pow2i(a0), pow2i(a1)});
  res = mul2(res, F2{pow2i(n0 - a0), pow2i(n1 - a1)});
  const float kInf = __int_as_float(0x7F800000);
  res.x = (t.x > 88.0f) ? kInf : ((t.x < -88.0f) ? 0.0f : res.x);
  res.y = (t.y > 88.0f) ? kInf : ((t.y < -88.0f) ? 0.0f : res.y);
  return res;
}

// d = 1 + exp_spec(t) on the fast path.  For every binary32 t <= -17 the
// specification's exp_spec(t) is below 2^-24, so 1 + e rounds to exactly 1:
// clamping t at -17 leaves d unchanged.  For t in [-17, 88] the specified
// result q * 2^(n>>1) * 2^(n-(n>>1)) is a normal binary32 number, so both
// power-of-two multiplications are exact and equal one add of n to the
// exponent field.  Arguments above 88 are clamped too; they give d >= 2^126,
// which the guards send to the exact path (h_needs_exact / h_maybe_bad).
__device__ __forceinline__ F2 dplus1_fast(F2 t) {
  const float kL2E = __uint_as_float(0x3FB8AA3Bu);
  const float kLn2Hi = __uint_as_float(0x3F317000u);
  const float kLn2Lo = __uint_as_float(0x3805FDF4u);
  const F2 tc{fminf(fmaxf(t.x, -17.0f), 88.0f), fminf(fmaxf(t.y, -17.0f), 88.0f)};
  const F2 nl = mul2(tc, splat(kL2E));
  const F2 n{rintf(nl.x), rintf(nl.y)};
  F2 r = add2(tc, neg(mul2(n, splat(kLn2Hi))));
  r = add2(r, neg(mul2(n, splat(kLn2Lo))));
  F2 q = splat(__uint_as_float(0x39500D01u));
  q = add2(mul2(q, r), splat(__uint_as_float(0x3AB60B61u)));
  q = add2(mul2(q, r), splat(__uint_as_float(0x3C088889u)));
  q = add2(mul2(q, r), splat(__uint_as_float(0x3D2AAAABu)));
  q = add2(mul2(q, r), splat(__uint_as_float(0x3E2AAAABu)));
  q = add2(mul2(q, r), splat(0.5f));
  q = add2(mul2(q, r), splat(1.0f));
  q = add2(mul2(q, r), splat(1.0f));
  const F2 e{__int_as_float(__float_as_int(q.x) + (__float2int_rn(n.x) << 23)),
             __int_as_float(__float_as_int(q.y) + (__float2int_rn(n.y) << 23))};
  return add2(splat(1.0f), e);
}

__device__ __forceinline__ float rcp_approx(float d) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(d));
  return r;
}

// ---- exactness guards.  A fast result f within a known number of binary32
// ulps of the specified value v gives the same E4M3 code (bf16 bits) as v
// unless a rounding midpoint of the narrow format lies between them.  In the
// normal E4M3 range every midpoint has the low 20 significand bits equal to
// 0x80000 (bf16: low 16 bits equal to 0x8000), so f needs the exact path only
// when its low bits are within `W` of that pattern.  In the E4M3 subnormal
// range (|f| < 2^-6) the midpoints are the odd multiples of 2^-10: there f
// needs the exact path only when f * 2^9 is within 2^-14 of a half-integer
// (far more than W binary32 ulps of f at that scale).
// Cheap pre-test: true near a midpoint of the normal E4M3 range and for every
// value in the subnormal range (a superset of near_e4m3_midpoint).
template <int W>
__device__ __forceinline__ bool maybe_near_e4m3_midpoint(float f) {
  const uint32_t b = __float_as_uint(f);
  const uint32_t a = b & 0x7FFFFFFFu;
  const bool sub = (a != 0u) & (a < 0x3C800000u);                   // 0 < |f| < 2^-6
  const bool mid = ((b & 0xFFFFFu) + (uint32_t)W - 0x80000u) <= (uint32_t)(2 * W);
  return sub | mid;
}

template <int W>
__device__ __forceinline__ bool near_e4m3_midpoint(float f) {
  const float a = fabsf(f);
  const float t = a * 512.0f;                                       // exact scaling
  const bool near_sub = fabsf((t - floorf(t)) - 0.5f) < 6.103515625e-05f;   // 2^-14
  const uint32_t b = __float_as_uint(f);
  const bool mid = ((b & 0xFFFFFu) + (uint32_t)W - 0x80000u) <= (uint32_t)(2 * W);
  return (a < 0.015625f) ? near_sub : mid;                          // |f| < 2^-6: subnormal E4M3
}

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
// h = p / d with p = g * u and d = 1 + exp_spec(-g), both exact to the
// specification.  Fast path: hf = fl32(p * rcp(d)) (rcp: the hardware
// reciprocal approximation), within a few ulp of fl32(p / d) for d < 2^126;
// FP8: qf = fl32(hf * fl32(1/s)).  Elements where the fast value is within the
// guard window of a midpoint, where d >= 2^126 (the reciprocal flushes), or
// where hf is tiny (binary32 subnormal range) take the correctly rounded
// divisions.

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

__device__ __forceinline__ uint32_t swiglu_fp8_pair(uint32_t gw, uint32_t uw, float s, float rs,
                                                    bool exact_only) {
  F2 p, d;
  swiglu_pd(gw, uw, p, d);
  const F2 hf = mul2(p, F2{rcp_approx(d.x), rcp_approx(d.y)});
  F2 q = mul2(hf, splat(rs));
  const bool fx = exact_only | h_needs_exact(p.x, d.x, hf.x) | near_e4m3_midpoint<32>(q.x);
  const bool fy = exact_only | h_needs_exact(p.y, d.y, hf.y) | near_e4m3_midpoint<32>(q.y);
  if (fx | fy) {                       // rare: a rounding decision the fast value cannot settle
    const F2 de = swiglu_d_exact(gw);
    if (fx) q.x = __fdiv_rn(__fdiv_rn(p.x, de.x), s);
    if (fy) q.y = __fdiv_rn(__fdiv_rn(p.y, de.y), s);
  }
  return cvt_e4m3x2(q.x, q.y);
}

__device__ __forceinline__ uint32_t swiglu_bf16_pair(uint32_t gw, uint32_t uw) {
  F2 p, d;
  swiglu_pd(gw, uw, p, d);
  F2 h = mul2(p, F2{rcp_approx(d.x), rcp_approx(d.y)});
  if (h_needs_exact(p.x, d.x, h.x) | h_needs_exact(p.y, d.y, h.y) | near_bf16_midpoint<8>(h.x) |
      near_bf16_midpoint<8>(h.y)) {
    const F2 de = swiglu_d_exact(gw);
    if (h_needs_exact(p.x, d.x, h.x) || near_bf16_midpoint<8>(h.x)) h.x = __fdiv_rn(p.x, de.x);
    if (h_needs_exact(p.y, d.y, h.y) || near_bf16_midpoint<8>(h.y)) h.y = __fdiv_rn(p.y, de.y);
  }
  return cvt_bf16x2(h.x, h.y);
}

// ---- 16 elements at once (the fused gate/up epilogue): the fast values of all
// 16 are computed straight-line so that independent pairs interleave, a
// bitmask records the elements whose rounding decision the fast value cannot
// settle, and a single, rarely taken branch recomputes those exactly.
// gw/uw: 8 words of two bf16 each.

// Cheap integer form of h_needs_exact for the straight-line pass:
// d >= 2^126 (or NaN), or |hf| < 2^-100 while p != 0.
__device__ __forceinline__ bool h_maybe_bad(float p, float d, float hf) {
  const uint32_t db = __float_as_uint(d);
  const uint32_t hb = __float_as_uint(hf) & 0x7FFFFFFFu;
  return (db >= 0x7E800000u) | ((hb < 0x0D800000u) & ((__float_as_uint(p) << 1) != 0u));
}

__device__ __forceinline__ void swiglu_fp8_x16(const uint32_t (&gw)[8], const uint32_t (&uw)[8],
                                               float s, float rs, bool exact_only,
                                               uint32_t (&codes)[4]) {
  float q[16], pp[16], dd[16];
  uint32_t maybe = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    F2 p, d;
    swiglu_pd(gw[j], uw[j], p, d);
    const F2 hf = mul2(p, F2{rcp_approx(d.x), rcp_approx(d.y)});
    const F2 qf = mul2(hf, splat(rs));
    q[2 * j] = qf.x;
    q[2 * j + 1] = qf.y;
    pp[2 * j] = p.x;
    pp[2 * j + 1] = p.y;
    dd[2 * j] = d.x;
    dd[2 * j + 1] = d.y;
    maybe |= (uint32_t)(h_maybe_bad(p.x, d.x, hf.x) | maybe_near_e4m3_midpoint<32>(qf.x)) << (2 * j);
    maybe |= (uint32_t)(h_maybe_bad(p.y, d.y, hf.y) | maybe_near_e4m3_midpoint<32>(qf.y)) << (2 * j + 1);
  }
  if (exact_only) maybe = 0xFFFFu;
  if (maybe) {                         // the precise tests, then the rare exact divisions
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      if (maybe & (1u << e)) {
        const float hf = __fmul_rn(pp[e], rcp_approx(dd[e]));
        if (exact_only || h_needs_exact(pp[e], dd[e], hf) || near_e4m3_midpoint<32>(q[e])) {
          const F2 de = swiglu_d_exact(gw[e >> 1]);
          q[e] = __fdiv_rn(__fdiv_rn(pp[e], (e & 1) ? de.y : de.x), s);
        }
      }
    }
  }
#pragma unroll
  for (int j = 0; j < 4; ++j)
    codes[j] = cvt_e4m3x2(q[4 * j], q[4 * j + 1]) | (cvt_e4m3x2(q[4 * j + 2], q[4 * j + 3]) << 16);
}

}  // namespace w8

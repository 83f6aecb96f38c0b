// HBM-bound elementwise kernels of the static-FP8 linear path:
//
//  * static per-tensor activation quantization, x / s_in rounded once to
//    E4M3 with saturation (cosmos-framework PR #157, "feat: load ModelOpt
//    static-FP8 checkpoints via TorchAO", section Verification: div -> clamp
//    -> round-to-float8 with the exported input_scale);
//  * the two-input SwiGLU, SiLU(gate) * up, written straight to E4M3 with the
//    down projection's static input scale, or to bf16 on 16-bit steps
//    (TensorRT-LLM PR #17476, "Load static FP8 Cosmos3 Nano/Super checkpoints
//    without re-quantizing them", sections What changed and Denoising-step
//    activation precision).
//
// Each thread moves 16 elements per step with 128-bit loads and stores in a
// grid-stride loop over a grid sized to the SM count.  All arithmetic is
// IEEE binary32 with explicit round-to-nearest intrinsics, so that no
// multiply-add is contracted and the result is the same bit pattern as the
// specification below on any compiler setting.
//
// SwiGLU specification (the pages fix only SiLU(G) * U and the FP8 output):
//   p = g * u;  e = exp_spec(-g);  h = p / (1 + e)
//   FP8 out:  E4M3_satRNE(h / s_out);  bf16 out: bf16_RNE(h)
// exp_spec: Cody-Waite reduction (Cody and Waite, Software Manual for the
// Elementary Functions, 1980) with n = rint(t * fl32(1/ln2)),
// r = (t - n*LN2_HI) - n*LN2_LO, LN2_HI = ln 2 with 12 low significand bits
// cleared, LN2_LO = fl32(ln 2 - LN2_HI); degree-7 Taylor polynomial of exp(r)
// in Horner form with coefficients fl32(1/k!), separate multiply and add;
// result scaled by 2^(n>>1) then 2^(n-(n>>1)); t > 88 gives +inf, t < -88
// gives 0.
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace w8 {
namespace {

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ float exp_spec(float t) {
  const float kL2E = __uint_as_float(0x3FB8AA3Bu);
  const float kLn2Hi = __uint_as_float(0x3F317000u);
  const float kLn2Lo = __uint_as_float(0x3805FDF4u);
  const float tc = fminf(fmaxf(t, -88.0f), 88.0f);
  const float n = rintf(__fmul_rn(tc, kL2E));
  const float r = __fsub_rn(__fsub_rn(tc, __fmul_rn(n, kLn2Hi)), __fmul_rn(n, kLn2Lo));
  // 1/k! rounded to binary32, k = 7 .. 0
  float q = __uint_as_float(0x39500D01u);
  q = __fadd_rn(__fmul_rn(q, r), __uint_as_float(0x3AB60B61u));
  q = __fadd_rn(__fmul_rn(q, r), __uint_as_float(0x3C088889u));
  q = __fadd_rn(__fmul_rn(q, r), __uint_as_float(0x3D2AAAABu));
  q = __fadd_rn(__fmul_rn(q, r), __uint_as_float(0x3E2AAAABu));
  q = __fadd_rn(__fmul_rn(q, r), 0.5f);
  q = __fadd_rn(__fmul_rn(q, r), 1.0f);
  q = __fadd_rn(__fmul_rn(q, r), 1.0f);
  const int ni = __float2int_rn(n);
  const int h1 = ni >> 1;
  const int h2 = ni - h1;
  float res = __fmul_rn(q, __int_as_float((h1 + 127) << 23));
  res = __fmul_rn(res, __int_as_float((h2 + 127) << 23));
  res = (t > 88.0f) ? __int_as_float(0x7F800000) : res;
  res = (t < -88.0f) ? 0.0f : res;
  return res;
}

__device__ __forceinline__ float swiglu_h(float g, float u) {
  const float p = __fmul_rn(g, u);
  const float e = exp_spec(-g);
  return __fdiv_rn(p, __fadd_rn(1.0f, e));
}

__device__ __forceinline__ uint4 ldg16(const void* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}

// ------------------------------------------------------------------ quant

__global__ void __launch_bounds__(256) quant_static_kernel(const uint16_t* __restrict__ x,
                                                           int64_t n16,
                                                           const float* __restrict__ s_in,
                                                           uint8_t* __restrict__ q) {
  const float s = __ldg(s_in);
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += stride) {
    const uint4 a = ldg16(x + i * 16);
    const uint4 b = ldg16(x + i * 16 + 8);
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t c0 = cvt_e4m3x2(__fdiv_rn(bf16_lo(w[2 * j]), s), __fdiv_rn(bf16_hi(w[2 * j]), s));
      const uint32_t c1 =
          cvt_e4m3x2(__fdiv_rn(bf16_lo(w[2 * j + 1]), s), __fdiv_rn(bf16_hi(w[2 * j + 1]), s));
      o[j] = c0 | (c1 << 16);
    }
    *reinterpret_cast<uint4*>(q + i * 16) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// ------------------------------------------------------------------ swiglu

__global__ void __launch_bounds__(256) swiglu_fp8_kernel(const uint16_t* __restrict__ g,
                                                         const uint16_t* __restrict__ u,
                                                         int64_t n16,
                                                         const float* __restrict__ s_out,
                                                         uint8_t* __restrict__ out) {
  const float s = __ldg(s_out);
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += stride) {
    const uint4 ga = ldg16(g + i * 16), gb = ldg16(g + i * 16 + 8);
    const uint4 ua = ldg16(u + i * 16), ub = ldg16(u + i * 16 + 8);
    const uint32_t gw[8] = {ga.x, ga.y, ga.z, ga.w, gb.x, gb.y, gb.z, gb.w};
    const uint32_t uw[8] = {ua.x, ua.y, ua.z, ua.w, ub.x, ub.y, ub.z, ub.w};
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float h0 = swiglu_h(bf16_lo(gw[2 * j]), bf16_lo(uw[2 * j]));
      const float h1 = swiglu_h(bf16_hi(gw[2 * j]), bf16_hi(uw[2 * j]));
      const float h2 = swiglu_h(bf16_lo(gw[2 * j + 1]), bf16_lo(uw[2 * j + 1]));
      const float h3 = swiglu_h(bf16_hi(gw[2 * j + 1]), bf16_hi(uw[2 * j + 1]));
      const uint32_t c0 = cvt_e4m3x2(__fdiv_rn(h0, s), __fdiv_rn(h1, s));
      const uint32_t c1 = cvt_e4m3x2(__fdiv_rn(h2, s), __fdiv_rn(h3, s));
      o[j] = c0 | (c1 << 16);
    }
    *reinterpret_cast<uint4*>(out + i * 16) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

__global__ void __launch_bounds__(256) swiglu_bf16_kernel(const uint16_t* __restrict__ g,
                                                          const uint16_t* __restrict__ u,
                                                          int64_t n16,
                                                          uint16_t* __restrict__ out) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += stride) {
    const uint4 ga = ldg16(g + i * 16), gb = ldg16(g + i * 16 + 8);
    const uint4 ua = ldg16(u + i * 16), ub = ldg16(u + i * 16 + 8);
    const uint32_t gw[8] = {ga.x, ga.y, ga.z, ga.w, gb.x, gb.y, gb.z, gb.w};
    const uint32_t uw[8] = {ua.x, ua.y, ua.z, ua.w, ub.x, ub.y, ub.z, ub.w};
    uint32_t o[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      o[j] = cvt_bf16x2(swiglu_h(bf16_lo(gw[j]), bf16_lo(uw[j])),
                        swiglu_h(bf16_hi(gw[j]), bf16_hi(uw[j])));
    }
    uint4* dst = reinterpret_cast<uint4*>(out + i * 16);
    dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
    dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
  }
}

int grid_for(int64_t n16, int sms) {
  const int64_t want = (n16 + 255) / 256;
  const int64_t cap = (int64_t)sms * 8;   // 8 resident 256-thread blocks per SM
  return (int)(want < cap ? (want > 0 ? want : 1) : cap);
}

}  // namespace

cudaError_t launch_quant_static(const uint16_t* x, int64_t n, const float* s_in, uint8_t* q,
                                int sms, cudaStream_t st) {
  const int64_t n16 = n / 16;
  quant_static_kernel<<<grid_for(n16, sms), 256, 0, st>>>(x, n16, s_in, q);
  return cudaGetLastError();
}

cudaError_t launch_swiglu_fp8(const uint16_t* g, const uint16_t* u, int64_t n, const float* s_out,
                              uint8_t* out, int sms, cudaStream_t st) {
  const int64_t n16 = n / 16;
  swiglu_fp8_kernel<<<grid_for(n16, sms), 256, 0, st>>>(g, u, n16, s_out, out);
  return cudaGetLastError();
}

cudaError_t launch_swiglu_bf16(const uint16_t* g, const uint16_t* u, int64_t n, uint16_t* out,
                               int sms, cudaStream_t st) {
  const int64_t n16 = n / 16;
  swiglu_bf16_kernel<<<grid_for(n16, sms), 256, 0, st>>>(g, u, n16, out);
  return cudaGetLastError();
}

}  // namespace w8

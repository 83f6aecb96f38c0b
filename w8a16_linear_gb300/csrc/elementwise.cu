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
//    activation precision), and its tested options (limit, alpha, beta;
//    bf16 or binary16 inputs; section Test Coverage);
//  * the W8A16 weight dequantization, bf16(fl32(dec(q) * s_w)) (diffusers PR
//    #14664, "[Cosmos3] Mixed W8A8/W8A16 denoising for ModelOpt FP8
//    checkpoints", section Behavior: dequant + F.linear).
//
// Each thread moves 16 elements per step with 128-bit loads and stores in a
// grid-stride loop over a grid of as many blocks as fit on the GPU at once.
// Every output is the specification's bit pattern: a fast value with a
// proven error bound is kept only where it provably rounds to the same code,
// everything else is recomputed with correctly rounded, never-fused scalar
// operations.
//
// The SwiGLU specification and its guarded fast evaluation live in
// swiglu_spec.cuh.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"
#include "swiglu_spec.cuh"

namespace w8 {
namespace {

// ------------------------------------------------------------------ quant
//
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

__global__ void __launch_bounds__(256, 8) quant_static_kernel(const uint16_t* __restrict__ x,
                                                              int64_t n16,
                                                              const float* __restrict__ s_in,
                                                              uint8_t* __restrict__ q) {
  const float s = __ldg(s_in);
  const float r = __frcp_rn(s);
  const bool exact_only = !scale_is_fast(s, r);
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += stride) {
    const uint4 a = ldg16(x + i * 16);
    const uint4 b = ldg16(x + i * 16 + 8);
    uint4 o;
    o.x = quant_pair(a.x, s, r, exact_only) | (quant_pair(a.y, s, r, exact_only) << 16);
    o.y = quant_pair(a.z, s, r, exact_only) | (quant_pair(a.w, s, r, exact_only) << 16);
    o.z = quant_pair(b.x, s, r, exact_only) | (quant_pair(b.y, s, r, exact_only) << 16);
    o.w = quant_pair(b.z, s, r, exact_only) | (quant_pair(b.w, s, r, exact_only) << 16);
    *reinterpret_cast<uint4*>(q + i * 16) = o;
  }
}

__global__ void __launch_bounds__(256, 6) swiglu_fp8_kernel(const uint16_t* __restrict__ g,
                                                            const uint16_t* __restrict__ u,
                                                            int64_t n16,
                                                            const float* __restrict__ s_out,
                                                            uint8_t* __restrict__ out) {
  const float s = __ldg(s_out);
  const float rs = __frcp_rn(s);
  const bool exact_only = !swiglu_fp8_scale_is_fast(s, rs);
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += stride) {
    const uint4 ga = ldg16(g + i * 16), gb = ldg16(g + i * 16 + 8);
    const uint4 ua = ldg16(u + i * 16), ub = ldg16(u + i * 16 + 8);
    uint4 o;
    o.x = swiglu_fp8_pair(ga.x, ua.x, s, rs, exact_only) |
          (swiglu_fp8_pair(ga.y, ua.y, s, rs, exact_only) << 16);
    o.y = swiglu_fp8_pair(ga.z, ua.z, s, rs, exact_only) |
          (swiglu_fp8_pair(ga.w, ua.w, s, rs, exact_only) << 16);
    o.z = swiglu_fp8_pair(gb.x, ub.x, s, rs, exact_only) |
          (swiglu_fp8_pair(gb.y, ub.y, s, rs, exact_only) << 16);
    o.w = swiglu_fp8_pair(gb.z, ub.z, s, rs, exact_only) |
          (swiglu_fp8_pair(gb.w, ub.w, s, rs, exact_only) << 16);
    *reinterpret_cast<uint4*>(out + i * 16) = o;
  }
}

__global__ void __launch_bounds__(256, 6) swiglu_bf16_kernel(const uint16_t* __restrict__ g,
                                                             const uint16_t* __restrict__ u,
                                                             int64_t n16,
                                                             uint16_t* __restrict__ out) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += stride) {
    const uint4 ga = ldg16(g + i * 16), gb = ldg16(g + i * 16 + 8);
    const uint4 ua = ldg16(u + i * 16), ub = ldg16(u + i * 16 + 8);
    uint4* dst = reinterpret_cast<uint4*>(out + i * 16);
    dst[0] = make_uint4(swiglu_bf16_pair(ga.x, ua.x), swiglu_bf16_pair(ga.y, ua.y),
                        swiglu_bf16_pair(ga.z, ua.z), swiglu_bf16_pair(ga.w, ua.w));
    dst[1] = make_uint4(swiglu_bf16_pair(gb.x, ub.x), swiglu_bf16_pair(gb.y, ub.y),
                        swiglu_bf16_pair(gb.z, ub.z), swiglu_bf16_pair(gb.w, ub.w));
  }
}

// ------------------------------------------------------------------ weight dequantization
//
// Wd = bf16_RNE(fl32(dec(q) * s_w)): the W8A16 step's transient bf16 weight
// ("dequant + F.linear").  E4M3 -> f16 is exact (cvt e4m3x2 -> f16x2), f16 ->
// f32 exact, one correctly rounded binary32 multiply, one bf16 rounding.

__global__ void __launch_bounds__(256, 8) dequant_weight_kernel(const uint8_t* __restrict__ q, int64_t n16,
                                                                const float* __restrict__ s_w,
                                                                uint16_t* __restrict__ wd) {
  const float sw = __ldg(s_w);
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += stride) {
    const uint4 c = ldg16(q + i * 16);
    const uint32_t cw[4] = {c.x, c.y, c.z, c.w};
    uint32_t o[8];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t f01 = cvt_e4m3x2_to_f16x2((uint16_t)(cw[e] & 0xFFFF));
      const uint32_t f23 = cvt_e4m3x2_to_f16x2((uint16_t)(cw[e] >> 16));
      F2 a, b;
      f16x2_to_f32(f01, a.x, a.y);
      f16x2_to_f32(f23, b.x, b.y);
      a = mul2(a, splat(sw));
      b = mul2(b, splat(sw));
      o[2 * e] = cvt_bf16x2(a.x, a.y);
      o[2 * e + 1] = cvt_bf16x2(b.x, b.y);
    }
    uint4* dst = reinterpret_cast<uint4*>(wd + i * 16);
    dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
    dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
  }
}

// The SwiGLU variants (swiglu_spec.cuh): bf16 or binary16 inputs, FP8 output
// or a 16-bit output in the input's format.
template <bool kF16, bool kFp8>
__global__ void __launch_bounds__(256, 6) swiglu_ex_kernel(const uint16_t* __restrict__ g,
                                                           const uint16_t* __restrict__ u,
                                                           int64_t n16, SwigluParams pr,
                                                           const float* __restrict__ s_out,
                                                           void* __restrict__ out) {
  float s = 1.0f, rs = 1.0f;
  bool exact_only = false;
  if constexpr (kFp8) {
    s = __ldg(s_out);
    rs = __frcp_rn(s);
    exact_only = !swiglu_fp8_scale_is_fast(s, rs);
  }
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += stride) {
    const uint4 ga = ldg16(g + i * 16), gb = ldg16(g + i * 16 + 8);
    const uint4 ua = ldg16(u + i * 16), ub = ldg16(u + i * 16 + 8);
    const uint32_t gw[8] = {ga.x, ga.y, ga.z, ga.w, gb.x, gb.y, gb.z, gb.w};
    const uint32_t uw[8] = {ua.x, ua.y, ua.z, ua.w, ub.x, ub.y, ub.z, ub.w};
    if constexpr (kFp8) {
      uint32_t c[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) c[j] = swiglu_ex_fp8_pair<kF16>(gw[j], uw[j], pr, s, rs, exact_only);
      *reinterpret_cast<uint4*>(static_cast<uint8_t*>(out) + i * 16) =
          make_uint4(c[0] | (c[1] << 16), c[2] | (c[3] << 16), c[4] | (c[5] << 16), c[6] | (c[7] << 16));
    } else {
      uint32_t h[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) h[j] = swiglu_ex_16_pair<kF16>(gw[j], uw[j], pr);
      uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(out) + i * 16);
      dst[0] = make_uint4(h[0], h[1], h[2], h[3]);
      dst[1] = make_uint4(h[4], h[5], h[6], h[7]);
    }
  }
}

// Grid of 256-thread blocks for a grid-stride kernel: as many blocks as fit
// on the GPU at once (blocks beyond that would run as a second, partly
// occupied wave, which an HBM-bound kernel cannot afford), fewer for small
// inputs.  The per-SM figure is the occupancy of `kern`, looked up once.
int grid_for(const void* kern, std::atomic<int>* per_sm, int64_t n16, int sms) {
  int b = per_sm->load(std::memory_order_relaxed);
  if (b == 0) {   // first call: look the figure up (threads racing here store the same value)
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, kern, 256, 0) != cudaSuccess || b < 1) b = 1;
    per_sm->store(b, std::memory_order_relaxed);
  }
  const int64_t want = (n16 + 255) / 256;
  const int64_t cap = (int64_t)sms * b;
  return (int)(want < cap ? (want > 0 ? want : 1) : cap);
}

}  // namespace

cudaError_t launch_swiglu_ex(const uint16_t* g, const uint16_t* u, int64_t n, bool in_f16, bool out_fp8,
                             const SwigluExArgs& a, const float* s_out, void* out, int sms,
                             cudaStream_t st) {
  const int64_t n16 = n / 16;
  const SwigluParams pr{a.limit, a.alpha, a.beta, a.has_limit ? 1 : 0, a.beta != 0.0f ? 1 : 0};
  static std::atomic<int> occ[4];
  if (in_f16) {
    if (out_fp8) {
      auto k = swiglu_ex_kernel<true, true>;
      k<<<grid_for((const void*)k, &occ[0], n16, sms), 256, 0, st>>>(g, u, n16, pr, s_out, out);
    } else {
      auto k = swiglu_ex_kernel<true, false>;
      k<<<grid_for((const void*)k, &occ[1], n16, sms), 256, 0, st>>>(g, u, n16, pr, s_out, out);
    }
  } else {
    if (out_fp8) {
      auto k = swiglu_ex_kernel<false, true>;
      k<<<grid_for((const void*)k, &occ[2], n16, sms), 256, 0, st>>>(g, u, n16, pr, s_out, out);
    } else {
      auto k = swiglu_ex_kernel<false, false>;
      k<<<grid_for((const void*)k, &occ[3], n16, sms), 256, 0, st>>>(g, u, n16, pr, s_out, out);
    }
  }
  return cudaGetLastError();
}

cudaError_t launch_dequant_weight(const uint8_t* q, int64_t n, const float* s_w, uint16_t* wd, int sms,
                                  cudaStream_t st) {
  const int64_t n16 = n / 16;
  static std::atomic<int> occ{0};
  dequant_weight_kernel<<<grid_for((const void*)dequant_weight_kernel, &occ, n16, sms), 256, 0, st>>>(q, n16, s_w,
                                                                                                  wd);
  return cudaGetLastError();
}

cudaError_t launch_quant_static(const uint16_t* x, int64_t n, const float* s_in, uint8_t* q,
                                int sms, cudaStream_t st) {
  const int64_t n16 = n / 16;
  static std::atomic<int> occ{0};
  quant_static_kernel<<<grid_for((const void*)quant_static_kernel, &occ, n16, sms), 256, 0, st>>>(x, n16, s_in, q);
  return cudaGetLastError();
}

cudaError_t launch_swiglu_fp8(const uint16_t* g, const uint16_t* u, int64_t n, const float* s_out,
                              uint8_t* out, int sms, cudaStream_t st) {
  const int64_t n16 = n / 16;
  static std::atomic<int> occ{0};
  swiglu_fp8_kernel<<<grid_for((const void*)swiglu_fp8_kernel, &occ, n16, sms), 256, 0, st>>>(g, u, n16, s_out, out);
  return cudaGetLastError();
}

cudaError_t launch_swiglu_bf16(const uint16_t* g, const uint16_t* u, int64_t n, uint16_t* out,
                               int sms, cudaStream_t st) {
  const int64_t n16 = n / 16;
  static std::atomic<int> occ{0};
  swiglu_bf16_kernel<<<grid_for((const void*)swiglu_bf16_kernel, &occ, n16, sms), 256, 0, st>>>(g, u, n16, out);
  return cudaGetLastError();
}

}  // namespace w8

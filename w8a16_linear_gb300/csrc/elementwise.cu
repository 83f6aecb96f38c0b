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
//    checkpoints", section Behavior: dequant + F.linear);
//  * the producer of a linear layer's input with the static quantization
//    fused after it: LayerNorm (no affine) over each row, a per-sample
//    shift/scale modulation, bf16 rounding, then the quantization above
//    (the pages name the block's norm/modulation before the quantization
//    without a formula; this is the diffusion-transformer form).
//
// Each thread moves 16 elements per step (the dequantization: two 8-element
// chunks of its warp's 512-element block) with 64- or 128-bit loads and
// 128-bit stores in a grid-stride loop over a grid of as many blocks as fit
// on the GPU at once.
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
#include "quant_spec.cuh"

namespace w8 {
namespace {

// ------------------------------------------------------------------ quant
//
// quant_pair / quant_pair_exact (quant_spec.cuh): the specification's codes
// of one packed bf16 pair.

// Work distribution of the elementwise kernels: 16-element vectors, U per
// thread per iteration, taken a grid stride apart (vector i + j * stride for
// j < U), so each load instruction of a warp covers contiguous memory and a
// thread has all U vectors' loads in flight before it converts any of them.
// Blocks per SM that each kernel's launch bounds are written for.  Measured
// at the bench's sizes (20670x4096, 16384x4096, 20670x16384): one vector per
// iteration with 4 blocks per SM for the quantization and the two SwiGLU
// kernels, two with 4 blocks for the (write-heavy) dequantization, one with 6
// blocks for the SwiGLU options; 2-4 vectors per iteration, or the full
// 8 / 6 blocks per SM, measured 1-10% slower.
constexpr int kQuantU = 1, kQuantBlocks = 4;
constexpr int kDequantU = 2, kDequantBlocks = 4;
constexpr int kSwigluU = 1, kSwigluBlocks = 4;
constexpr int kSwigluExU = 1, kSwigluExBlocks = 6;

// A 16-byte streaming load that leaves no line in L1.  The quantization reads
// each byte of x once; without L1 allocation it measured 36.9 against 38.9 µs
// at 20670x4096 (same process, L2 flushed, both orders).  The two-input
// SwiGLU kernels measured 0-1.6% slower with it and keep the plain load.
__device__ __forceinline__ uint4 ldg16_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

template <int U>
__global__ void __launch_bounds__(256, kQuantBlocks) quant_static_kernel(const uint16_t* __restrict__ x, int64_t n16,
                                                              const float* __restrict__ s_in,
                                                              uint8_t* __restrict__ q) {
  griddep_launch_dependents();   // a GEMM launched next may start its prologue
  const float s = __ldg(s_in);
  const QuantBracket br = quant_bracket(s);
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += U * stride) {
    uint4 a[U], b[U];
#pragma unroll
    for (int j = 0; j < U; ++j) {
      const int64_t v = i + j * stride;
      if (v < n16) {
        a[j] = ldg16_stream(x + v * 16);
        b[j] = ldg16_stream(x + v * 16 + 8);
      }
    }
#pragma unroll
    for (int j = 0; j < U; ++j) {
      const int64_t v = i + j * stride;
      if (v >= n16) break;
      uint4 o;
      o.x = quant_pair(a[j].x, s, br) | (quant_pair(a[j].y, s, br) << 16);
      o.y = quant_pair(a[j].z, s, br) | (quant_pair(a[j].w, s, br) << 16);
      o.z = quant_pair(b[j].x, s, br) | (quant_pair(b[j].y, s, br) << 16);
      o.w = quant_pair(b[j].z, s, br) | (quant_pair(b[j].w, s, br) << 16);
      *reinterpret_cast<uint4*>(q + v * 16) = o;
    }
  }
}

template <int U>
__global__ void __launch_bounds__(256, kSwigluBlocks) swiglu_fp8_kernel(const uint16_t* __restrict__ g,
                                                            const uint16_t* __restrict__ u, int64_t n16,
                                                            const float* __restrict__ s_out,
                                                            uint8_t* __restrict__ out) {
  griddep_launch_dependents();   // a GEMM launched next may start its prologue
  const float s = __ldg(s_out);
  const float rs = __frcp_rn(s);
  const bool exact_only = !swiglu_fp8_scale_is_fast(s, rs);
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += U * stride) {
    uint4 ga[U], gb[U], ua[U], ub[U];
#pragma unroll
    for (int j = 0; j < U; ++j) {
      const int64_t v = i + j * stride;
      if (v < n16) {
        ga[j] = ldg16(g + v * 16);
        gb[j] = ldg16(g + v * 16 + 8);
        ua[j] = ldg16(u + v * 16);
        ub[j] = ldg16(u + v * 16 + 8);
      }
    }
#pragma unroll
    for (int j = 0; j < U; ++j) {
      const int64_t v = i + j * stride;
      if (v >= n16) break;
      uint4 o;
      o.x = swiglu_fp8_pair(ga[j].x, ua[j].x, s, rs, exact_only) |
            (swiglu_fp8_pair(ga[j].y, ua[j].y, s, rs, exact_only) << 16);
      o.y = swiglu_fp8_pair(ga[j].z, ua[j].z, s, rs, exact_only) |
            (swiglu_fp8_pair(ga[j].w, ua[j].w, s, rs, exact_only) << 16);
      o.z = swiglu_fp8_pair(gb[j].x, ub[j].x, s, rs, exact_only) |
            (swiglu_fp8_pair(gb[j].y, ub[j].y, s, rs, exact_only) << 16);
      o.w = swiglu_fp8_pair(gb[j].z, ub[j].z, s, rs, exact_only) |
            (swiglu_fp8_pair(gb[j].w, ub[j].w, s, rs, exact_only) << 16);
      *reinterpret_cast<uint4*>(out + v * 16) = o;
    }
  }
}

template <int U>
__global__ void __launch_bounds__(256, kSwigluBlocks) swiglu_bf16_kernel(const uint16_t* __restrict__ g,
                                                             const uint16_t* __restrict__ u, int64_t n16,
                                                             uint16_t* __restrict__ out) {
  griddep_launch_dependents();   // a GEMM launched next may start its prologue
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += U * stride) {
    uint4 ga[U], gb[U], ua[U], ub[U];
#pragma unroll
    for (int j = 0; j < U; ++j) {
      const int64_t v = i + j * stride;
      if (v < n16) {
        ga[j] = ldg16(g + v * 16);
        gb[j] = ldg16(g + v * 16 + 8);
        ua[j] = ldg16(u + v * 16);
        ub[j] = ldg16(u + v * 16 + 8);
      }
    }
#pragma unroll
    for (int j = 0; j < U; ++j) {
      const int64_t v = i + j * stride;
      if (v >= n16) break;
      uint4* dst = reinterpret_cast<uint4*>(out + v * 16);
      dst[0] = make_uint4(swiglu_bf16_pair(ga[j].x, ua[j].x), swiglu_bf16_pair(ga[j].y, ua[j].y),
                          swiglu_bf16_pair(ga[j].z, ua[j].z), swiglu_bf16_pair(ga[j].w, ua[j].w));
      dst[1] = make_uint4(swiglu_bf16_pair(gb[j].x, ub[j].x), swiglu_bf16_pair(gb[j].y, ub[j].y),
                          swiglu_bf16_pair(gb[j].z, ub[j].z), swiglu_bf16_pair(gb[j].w, ub[j].w));
    }
  }
}

// ------------------------------------------------------------------ weight dequantization
//
// Wd = bf16_RNE(fl32(dec(q) * s_w)): the W8A16 step's transient bf16 weight
// ("dequant + F.linear").  E4M3 -> f16 is exact (cvt e4m3x2 -> f16x2), f16 ->
// f32 exact, one correctly rounded binary32 multiply, one bf16 rounding.

// Element layout by warp: a warp covers 512 consecutive elements per
// iteration, lane t the 8-element chunks at 8 t and 256 + 8 t, so that every
// 16-byte store instruction of the warp writes 512 contiguous bytes (whole
// 32-byte sectors) and every 8-byte load of codes reads 256.  Two 16-byte
// stores per thread 32 bytes apart (a thread's 16 consecutive outputs) left
// each store instruction writing half of every sector it touched: 43.0
// against 32.8 µs for a 16384 x 4096 weight.  (The read-heavy SwiGLU kernels
// with 16-bit outputs measured 8-11% slower in this layout and keep theirs.)
__device__ __forceinline__ int64_t chunk16_first(int64_t b, int64_t j, int64_t warps, int hh, int lane) {
  return (b + j * warps) * 512 + hh * 256 + 8 * lane;
}

template <int U>
__global__ void __launch_bounds__(256, kDequantBlocks) dequant_weight_kernel(const uint8_t* __restrict__ q, int64_t n16,
                                                                const float* __restrict__ s_w,
                                                                uint16_t* __restrict__ wd) {
  griddep_launch_dependents();   // a GEMM launched next may start its prologue
  const float sw = __ldg(s_w);
  const int64_t n = n16 * 16;
  const int lane = (int)(threadIdx.x & 31);
  const int64_t nblk = (n + 511) / 512;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x / 32);
  for (int64_t b = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) / 32; b < nblk; b += U * warps) {
    uint2 c[U][2];   // 8 codes per chunk
#pragma unroll
    for (int j = 0; j < U; ++j) {
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int64_t e0 = chunk16_first(b, j, warps, hh, lane);
        if (e0 + 8 <= n) c[j][hh] = __ldg(reinterpret_cast<const uint2*>(q + e0));
      }
    }
#pragma unroll
    for (int j = 0; j < U; ++j) {
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int64_t e0 = chunk16_first(b, j, warps, hh, lane);
        if (e0 + 8 > n) continue;
        const uint32_t cw[2] = {c[j][hh].x, c[j][hh].y};
        uint32_t o[4];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const uint32_t f01 = cvt_e4m3x2_to_f16x2((uint16_t)(cw[e] & 0xFFFF));
          const uint32_t f23 = cvt_e4m3x2_to_f16x2((uint16_t)(cw[e] >> 16));
          F2 a, bq;
          f16x2_to_f32(f01, a.x, a.y);
          f16x2_to_f32(f23, bq.x, bq.y);
          a = mul2(a, splat(sw));
          bq = mul2(bq, splat(sw));
          o[2 * e] = cvt_bf16x2(a.x, a.y);
          o[2 * e + 1] = cvt_bf16x2(bq.x, bq.y);
        }
        *reinterpret_cast<uint4*>(wd + e0) = make_uint4(o[0], o[1], o[2], o[3]);
      }
    }
  }
}

// The SwiGLU variants (swiglu_spec.cuh): bf16 or binary16 inputs, FP8 output
// or a 16-bit output in the input's format.
template <bool kF16, bool kFp8, int U>
__global__ void __launch_bounds__(256, kSwigluExBlocks) swiglu_ex_kernel(const uint16_t* __restrict__ g,
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
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += U * stride) {
    uint4 ga[U], gb[U], ua[U], ub[U];
#pragma unroll
    for (int j = 0; j < U; ++j) {
      const int64_t v = i + j * stride;
      if (v < n16) {
        ga[j] = ldg16(g + v * 16);
        gb[j] = ldg16(g + v * 16 + 8);
        ua[j] = ldg16(u + v * 16);
        ub[j] = ldg16(u + v * 16 + 8);
      }
    }
#pragma unroll
    for (int j = 0; j < U; ++j) {
      const int64_t v = i + j * stride;
      if (v >= n16) break;
      const uint32_t gw[8] = {ga[j].x, ga[j].y, ga[j].z, ga[j].w, gb[j].x, gb[j].y, gb[j].z, gb[j].w};
      const uint32_t uw[8] = {ua[j].x, ua[j].y, ua[j].z, ua[j].w, ub[j].x, ub[j].y, ub[j].z, ub[j].w};
      if constexpr (kFp8) {
        uint32_t c[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) c[e] = swiglu_ex_fp8_pair<kF16>(gw[e], uw[e], pr, s, rs, exact_only);
        *reinterpret_cast<uint4*>(static_cast<uint8_t*>(out) + v * 16) =
            make_uint4(c[0] | (c[1] << 16), c[2] | (c[3] << 16), c[4] | (c[5] << 16), c[6] | (c[7] << 16));
      } else {
        uint32_t h[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) h[e] = swiglu_ex_16_pair<kF16>(gw[e], uw[e], pr);
        uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(out) + v * 16);
        dst[0] = make_uint4(h[0], h[1], h[2], h[3]);
        dst[1] = make_uint4(h[4], h[5], h[6], h[7]);
      }
    }
  }
}

// ------------------------------------------------------------ norm + quant
//
// A block of 256 threads works on kG = 256 / kT rows at a time: row group g
// (threads g kT .. g kT + kT - 1, kT = 64 for K <= 4096, else 128) takes row
// blockIdx.x kG + g, then every gridDim.x kG-th row after it, with its own
// named barrier, its own shared-memory ring of row buffers and its own
// reduction slots, so the groups of a block never wait for one another.  A
// group's coming rows stream into its ring by bulk copies (cp.async.bulk,
// one mbarrier per buffer), several rows ahead of the one being worked on;
// a buffer is refilled after the row's first reduction, when every thread
// of the group holds its part of the row in registers.  Thread t of a group
// takes the row's 16-byte vectors t, t + kT, ... (kV of them, K <= 8 kT kV):
// 64 elements per thread at K = 4096, so the per-row reductions and barriers
// are spread over many elements.  For K <= 4096 the block keeps a table of
// fl32(1 + scale) and shift in binary32 for one sample (shared memory,
// filled once); with several samples and enough blocks each block works on
// the rows of its table's sample only, otherwise rows of another sample
// (and all rows when K > 4096) read the bf16 modulation from global memory
// where h is formed.  Statistics in binary32, taken about the row's first
// element p = x_0 (so that a large common offset of the row does not enter their
// rounding errors), with summation trees of depth <= 13 (the thread's 4 kV
// pairs pairwise, the last pair's two halves, five butterfly levels, the
// group's 2 or 4 warp sums pairwise):
//   a   = fl32(x - p),   m = fl32(sum a * fl32(1/K))    (m = mean - p)
//   var = fl32(sum fl32(a - m)^2 * fl32(1/K)),
//   r   = rsqrt(fl32(var + eps))                        (within 2 ulps),
//   n   = fma(a, r, -fl32(m r)),
//   h   = bf16(fma(n, fl32(1 + scale), shift)).
// h differs from the exactly computed value by a few binary32 ulps of its
// terms, so it is the correctly rounded bf16 except where the exact value is
// that close to a bf16 rounding boundary.  The E4M3 codes are the static
// quantization of this bf16 h, bit for bit: the bracket test of quant_pair
// in a branch-free per-pair loop that only marks, in a per-thread mask, the
// pairs it cannot settle; after the row, a thread with marked pairs (rare:
// values within 2^-21 of an E4M3 rounding boundary, or every pair when the
// scale is outside the fast range) recomputes each of them from the row in
// global memory by the same operations and stores the correctly rounded
// division's code over the fast one.

constexpr int kLnMaxStages = 8;
constexpr int kLnRingBytes = 64 * 1024;       // row buffers per block, split among its row groups
constexpr uint64_t kLnWaitLimitNs = 2000000000ull;

int ln_group_threads(int K) { return K <= 4096 ? 64 : 128; }

int ln_stages(int K) {
  const int groups = 256 / ln_group_threads(K);
  const int s = kLnRingBytes / groups / (2 * K);
  return s < kLnMaxStages ? s : kLnMaxStages;   // >= 2 for K <= 8192
}

// Bytes of the modulation table (fl32(1 + scale), shift) of the kT = 64 forms.
int ln_table_bytes(int K) { return K <= 4096 ? 8 * K : 0; }

__device__ uint32_t g_elem_err;                // kErrTimeout when a row-buffer wait gives up

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o >= 1; o /= 2) v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

__device__ __forceinline__ void group_bar(uint32_t id, uint32_t threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Sum over a row group of kW warps: each warp's butterfly total, then the
// warp totals pairwise in a fixed order, so every thread gets the same value.
template <int kW>
__device__ __forceinline__ float group_sum(float v, float* slot, uint32_t bar_id) {
  v = warp_sum(v);
  if ((threadIdx.x & 31) == 0) slot[(threadIdx.x >> 5) % kW] = v;
  group_bar(bar_id, 32 * kW);
  if constexpr (kW == 2) return __fadd_rn(slot[0], slot[1]);
  else return __fadd_rn(__fadd_rn(slot[0], slot[1]), __fadd_rn(slot[2], slot[3]));
}

// fl32(1 + scale) and shift of the 8 columns of vector j, as 4 packed pairs:
// from the block's table, or from the bf16 rows in global memory.
template <bool kTable>
__device__ __forceinline__ void ln_modulation(bool from_table, const float4* table, int nvec, const uint16_t* sh_row,
                                              const uint16_t* sc_row, int j, F2 (&gc)[4], F2 (&sf)[4]) {
  if (kTable && from_table) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const float4 v = table[c * nvec + j];    // columns 8j + 2c, + 1: (1 + scale) x2, shift x2
      gc[c] = F2{v.x, v.y};
      sf[c] = F2{v.z, v.w};
    }
  } else {
    const uint4 shv = ldg16(sh_row + 8 * j);
    const uint4 scv = ldg16(sc_row + 8 * j);
    const uint32_t sw[4] = {shv.x, shv.y, shv.z, shv.w};
    const uint32_t cw[4] = {scv.x, scv.y, scv.z, scv.w};
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      gc[c] = add2(splat(1.0f), F2{bf16_lo(cw[c]), bf16_hi(cw[c])});
      sf[c] = F2{bf16_lo(sw[c]), bf16_hi(sw[c])};
    }
  }
}

// The exact codes of a thread's unsettled pairs (bit 4 i + c of `mask`: pair
// c of its vector i) of one row: h recomputed from the row in global memory
// by the main pass's operations (so it is the same bf16), then the correctly
// rounded division.  This thread stored the fast codes of these pairs
// before, so its own program order puts these stores after them.
template <int kT, bool kTable>
__device__ __noinline__ void ln_fix_pairs(uint32_t mask, const uint16_t* xrow, uint8_t* qrow, int lt, int nvec,
                                          float minus_p, float r, float minus_mr, bool from_table,
                                          const float4* table, const uint16_t* sh_row, const uint16_t* sc_row,
                                          float s) {
  while (mask != 0u) {
    const int b = __ffs(mask) - 1;
    mask &= mask - 1u;
    const int j = lt + kT * (b >> 2), c = b & 3;
    const int col = 8 * j + 2 * c;
    const uint32_t xw = *reinterpret_cast<const uint32_t*>(xrow + col);
    const F2 a = add2(F2{bf16_lo(xw), bf16_hi(xw)}, splat(minus_p));
    F2 gc, sf;
    if (kTable && from_table) {
      const float4 v = table[c * nvec + j];
      gc = F2{v.x, v.y};
      sf = F2{v.z, v.w};
    } else {
      const uint32_t sw = *reinterpret_cast<const uint32_t*>(sh_row + col);
      const uint32_t cw = *reinterpret_cast<const uint32_t*>(sc_row + col);
      gc = add2(splat(1.0f), F2{bf16_lo(cw), bf16_hi(cw)});
      sf = F2{bf16_lo(sw), bf16_hi(sw)};
    }
    const F2 hv = fma2(fma2(a, splat(r), splat(minus_mr)), gc, sf);
    *reinterpret_cast<uint16_t*>(qrow + col) = (uint16_t)quant_pair_exact(cvt_bf16x2(hv.x, hv.y), s);
  }
}

// kFull: K == 8 kT kV, every vector slot of every thread holds row data.
// kOut: bit 0 the E4M3 codes q, bit 1 the bf16 h.
template <int kT, int kV, bool kFull, int kOut>
__global__ void __launch_bounds__(256, 2) ln_modulate_quant_kernel(
    const uint16_t* __restrict__ x, int64_t M, int K, const uint16_t* __restrict__ shift,
    const uint16_t* __restrict__ scale, int64_t rows_per_sample, float eps, int stages,
    const float* __restrict__ s_in, uint8_t* __restrict__ q, uint16_t* __restrict__ h) {
  constexpr int kG = 256 / kT;                 // row groups per block
  constexpr int kW = kT / 32;                  // warps per row group
  constexpr int kP = 4 * kV;                   // binary32 pairs per thread
  constexpr bool kTable = (kT == 64);          // modulation table in shared memory
  constexpr bool kQ = (kOut & 1) != 0, kH = (kOut & 2) != 0;
  static_assert(kP <= 32, "one mask bit per pair");
  // dynamic shared memory: [table: K x (1 + scale, shift) binary32] then the
  // row rings, kG x stages x K bf16
  extern __shared__ __align__(128) uint8_t ln_smem[];
  __shared__ __align__(8) uint64_t full[kG][kLnMaxStages];
  // [group][row parity][statistic][warp]: a row's two reductions and the
  // next row's use different slots, so the row's own barriers keep them apart.
  __shared__ float red[kG][2][2][kW];
  __shared__ int bad[kG];
  const int g = (int)threadIdx.x / kT;
  const int lt = (int)threadIdx.x % kT;
  const uint32_t bar_id = 1u + (uint32_t)g;
  const int nvec = K / 8;                      // 16-byte vectors per row
  const uint32_t row_bytes = 2u * (uint32_t)K;
  // Rows of the group: first, first + G, ... below row_end.  With several
  // samples and at least as many blocks, each block takes the rows of one
  // sample (blocks [s bps, (s + 1) bps) sample s), so that its modulation
  // table serves every row it works on; else the whole grid strides over M.
  const int64_t nsmp = (M + rows_per_sample - 1) / rows_per_sample;
  int64_t G, first, row_end, table_smp;
  if (nsmp > 1 && (int64_t)gridDim.x >= nsmp) {
    const int64_t bps = (int64_t)gridDim.x / nsmp;   // blocks per sample
    table_smp = (int64_t)blockIdx.x / bps;
    if (table_smp >= nsmp) return;             // the grid's remainder blocks (uniform per block)
    G = bps * kG;
    first = table_smp * rows_per_sample + ((int64_t)blockIdx.x % bps) * kG + g;
    row_end = (table_smp + 1) * rows_per_sample < M ? (table_smp + 1) * rows_per_sample : M;
  } else {
    G = (int64_t)gridDim.x * kG;
    first = (int64_t)blockIdx.x * kG + g;
    row_end = M;
    table_smp = ((int64_t)blockIdx.x * kG) / rows_per_sample;   // the sample of the block's first row
  }
  const uint32_t table_bytes = kTable ? 8u * (uint32_t)K : 0u;
  float4* table = reinterpret_cast<float4*>(ln_smem);
  uint8_t* ln_ring = ln_smem + table_bytes;
  // The table holds the modulation of sample table_smp: entry c * nvec + j
  // = (1 + scale) of columns 8 j + 2 c and 8 j + 2 c + 1, then their shift
  // (each pair lands in an aligned register pair for the packed FMAs), so that
  // the lanes of a warp (consecutive j) read consecutive 16-byte words.
  if constexpr (kTable) {
    const uint32_t* sh0 = reinterpret_cast<const uint32_t*>(shift + table_smp * K);
    const uint32_t* sc0 = reinterpret_cast<const uint32_t*>(scale + table_smp * K);
    for (int pi = (int)threadIdx.x; pi < K / 2; pi += 256) {
      const uint32_t sw = __ldg(sh0 + pi), cw = __ldg(sc0 + pi);
      table[(pi & 3) * nvec + (pi >> 2)] = make_float4(__fadd_rn(1.0f, bf16_lo(cw)), __fadd_rn(1.0f, bf16_hi(cw)),
                                                       bf16_lo(sw), bf16_hi(sw));
    }
    __syncthreads();
  }
  if (first >= row_end) return;                // uniform over the group
  const int64_t nrows = (row_end - 1 - first) / G + 1;
  const uint32_t ring = smem_u32(ln_ring) + (uint32_t)(g * stages) * row_bytes;
  if (lt == 0) {
    for (int st = 0; st < stages; ++st) mbar_init(smem_u32(&full[g][st]), 1);
    fence_mbar_init();
    bad[g] = 0;
  }
  group_bar(bar_id, kT);
  int64_t issued = 0;                          // rows whose copy is out (lt 0's count)
  if (lt == 0) {
    for (; issued < nrows && issued < stages; ++issued) {
      const uint32_t bar = smem_u32(&full[g][issued]);
      mbar_arrive_expect_tx(bar, row_bytes);
      bulk_load(ring + (uint32_t)issued * row_bytes, x + (first + issued * G) * K, row_bytes, bar);
    }
  }
  // the codes' bracket ends, the reciprocal of s folded in (quant_spec.cuh)
  float s = 1.0f, rlo = 1.0f, rhi = 1.0f;
  bool exact_only = false;
  if constexpr (kQ) {
    s = __ldg(s_in);
    const QuantBracket br = quant_bracket(s);
    rlo = br.lo;
    rhi = br.hi;
    exact_only = br.exact_only;
  }
  uint32_t live = 0;                           // mask bits of the thread's pairs that hold row data
#pragma unroll
  for (int i = 0; i < kV; ++i)
    if (kFull || lt + kT * i < nvec) live |= 0xFu << (4 * i);
  const float inv_k = __frcp_rn((float)K);     // exact when K is a power of two
  int never = 0;                               // nothing aborts these waits early
  int64_t k = 0;
  for (; k < nrows; ++k) {
    const int par = (int)(k & 1);
    const int64_t row = first + k * G;
    const int st = (int)(k % stages);
    const int64_t smp = row / rows_per_sample;
    const uint16_t* sh_row = shift + smp * K;
    const uint16_t* sc_row = scale + smp * K;
    if (!mbar_wait_warp(smem_u32(&full[g][st]), (uint32_t)((k / stages) & 1), &never, kLnWaitLimitNs))
      bad[g] = 1;
    // the row into registers: a = x - p as packed pairs (padding pairs 0)
    const uint16_t* rb = reinterpret_cast<const uint16_t*>(ln_ring + (size_t)(g * stages + st) * row_bytes);
    const float p = bf16_lo((uint32_t)rb[0]);
    const F2 minus_p = splat(-p);
    F2 a[kP];
#pragma unroll
    for (int i = 0; i < kV; ++i) {
      const int j = lt + kT * i;
      const bool live = kFull || j < nvec;
      const uint4 v = live ? *reinterpret_cast<const uint4*>(rb + 8 * j) : make_uint4(0u, 0u, 0u, 0u);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int c = 0; c < 4; ++c)
        a[4 * i + c] = live ? add2(F2{bf16_lo(w[c]), bf16_hi(w[c])}, minus_p) : F2{0.0f, 0.0f};
    }
    // mean about the pivot: the thread's pairs pairwise, then the group
    F2 t[kP / 2];
#pragma unroll
    for (int i = 0; i < kP / 2; ++i) t[i] = add2(a[i], a[i + kP / 2]);
#pragma unroll
    for (int w = kP / 4; w >= 1; w /= 2) {
#pragma unroll
      for (int i = 0; i < w; ++i) t[i] = add2(t[i], t[i + w]);
    }
    const float m = __fmul_rn(group_sum<kW>(__fadd_rn(t[0].x, t[0].y), red[g][par][0], bar_id), inv_k);
    // every thread has its part of the row: the buffer takes the group's
    // row k + stages
    if (bad[g]) break;                         // uniform: set before the barrier above
    if (lt == 0 && issued < nrows) {
      const uint32_t bar = smem_u32(&full[g][st]);
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(bar, row_bytes);
      bulk_load(ring + (uint32_t)st * row_bytes, x + (first + issued * G) * K, row_bytes, bar);
      ++issued;
    }
    // variance (two-pass: squared deviations from the mean)
    const F2 minus_m = splat(-m);
#pragma unroll
    for (int i = 0; i < kP / 2; ++i) {
      const bool live_lo = kFull || lt + kT * (i / 4) < nvec;
      const bool live_hi = kFull || lt + kT * ((i + kP / 2) / 4) < nvec;
      const F2 d0 = add2(a[i], minus_m), d1 = add2(a[i + kP / 2], minus_m);
      const F2 q0 = live_lo ? mul2(d0, d0) : F2{0.0f, 0.0f};
      const F2 q1 = live_hi ? mul2(d1, d1) : F2{0.0f, 0.0f};
      t[i] = add2(q0, q1);
    }
#pragma unroll
    for (int w = kP / 4; w >= 1; w /= 2) {
#pragma unroll
      for (int i = 0; i < w; ++i) t[i] = add2(t[i], t[i + w]);
    }
    const float var = __fmul_rn(group_sum<kW>(__fadd_rn(t[0].x, t[0].y), red[g][par][1], bar_id), inv_k);
    const float r = rsqrtf(__fadd_rn(var, eps));   // within 2 ulps of 1 / sqrt
    // n = a r - m r in one rounding, h = bf16(n g + shift), then the codes
    const F2 r2 = splat(r), mr2 = splat(-__fmul_rn(m, r));
    const bool from_table = kTable && smp == table_smp;   // uniform over the group
    uint32_t unsettled_mask = 0;
#pragma unroll
    for (int i = 0; i < kV; ++i) {
      const int j = lt + kT * i;
      if (!kFull && j >= nvec) break;
      F2 gc[4], sf[4];
      ln_modulation<kTable>(from_table, table, nvec, sh_row, sc_row, j, gc, sf);
      uint32_t hb[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const F2 hv = fma2(fma2(a[4 * i + c], r2, mr2), gc[c], sf[c]);
        hb[c] = cvt_bf16x2(hv.x, hv.y);
      }
      if constexpr (kH) *reinterpret_cast<uint4*>(h + row * K + 8 * j) = make_uint4(hb[0], hb[1], hb[2], hb[3]);
      if constexpr (kQ) {
        uint32_t code[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          bool unsettled;
          code[c] = e4m3x2_bracket(F2{bf16_lo(hb[c]), bf16_hi(hb[c])}, rlo, rhi, unsettled);
          unsettled_mask |= (uint32_t)unsettled << (4 * i + c);
        }
        *reinterpret_cast<uint2*>(q + row * K + 8 * j) =
            make_uint2(code[0] | (code[1] << 16), code[2] | (code[3] << 16));
      }
    }
    if constexpr (kQ) {
      if (exact_only) unsettled_mask = live;
      if (unsettled_mask != 0u)
        ln_fix_pairs<kT, kTable>(unsettled_mask, x + row * K, q + row * K, lt, nvec, -p, r, mr2.x, from_table,
                                 table, sh_row, sc_row, s);
    }
  }
  if (bad[g] && lt == 0) {
    // a wait gave up at row k: record it, then let the copies of rows k ..
    // issued - 1, still in flight, land (each wait bounded) before the
    // block's shared memory is released
    atomicOr(&g_elem_err, kErrTimeout);
    for (; k < issued; ++k)
      mbar_wait(smem_u32(&full[g][k % stages]), (uint32_t)((k / stages) & 1), &never, kLnWaitLimitNs);
  }
}

// Grid of 256-thread blocks for a grid-stride kernel: as many blocks as fit
// on the GPU at once (blocks beyond that would run as a second, partly
// occupied wave, which an HBM-bound kernel cannot afford), fewer for small
// inputs.  The per-SM figure is the occupancy of `kern`, looked up once.
int grid_for(const void* kern, std::atomic<int>* per_sm, int64_t n16, int sms, int u = 1) {
  int b = per_sm->load(std::memory_order_relaxed);
  if (b == 0) {   // first call: look the figure up (threads racing here store the same value)
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, kern, 256, 0) != cudaSuccess || b < 1) b = 1;
    per_sm->store(b, std::memory_order_relaxed);
  }
  const int64_t want = (n16 + 256 * u - 1) / (256 * u);
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
      auto k = swiglu_ex_kernel<true, true, kSwigluExU>;
      k<<<grid_for((const void*)k, &occ[0], n16, sms, kSwigluExU), 256, 0, st>>>(g, u, n16, pr, s_out, out);
    } else {
      auto k = swiglu_ex_kernel<true, false, kSwigluExU>;
      k<<<grid_for((const void*)k, &occ[1], n16, sms, kSwigluExU), 256, 0, st>>>(g, u, n16, pr, s_out, out);
    }
  } else {
    if (out_fp8) {
      auto k = swiglu_ex_kernel<false, true, kSwigluExU>;
      k<<<grid_for((const void*)k, &occ[2], n16, sms, kSwigluExU), 256, 0, st>>>(g, u, n16, pr, s_out, out);
    } else {
      auto k = swiglu_ex_kernel<false, false, kSwigluExU>;
      k<<<grid_for((const void*)k, &occ[3], n16, sms, kSwigluExU), 256, 0, st>>>(g, u, n16, pr, s_out, out);
    }
  }
  return cudaGetLastError();
}

// Binary32 -> E4M3, four values per thread per iteration (one 16-byte load,
// one 4-byte store); the last n % 4 values by a second, one-thread-per-value
// launch.
__global__ void __launch_bounds__(256) e4m3_from_f32_kernel(const float4* __restrict__ x, int64_t n4,
                                                            uint32_t* __restrict__ q) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += stride) {
    const float4 v = x[i];
    q[i] = cvt_e4m3x2(v.x, v.y) | (cvt_e4m3x2(v.z, v.w) << 16);
  }
}

__global__ void e4m3_from_f32_tail_kernel(const float* __restrict__ x, int64_t from, int64_t n,
                                          uint8_t* __restrict__ q) {
  const int64_t i = from + threadIdx.x;
  if (i < n) q[i] = (uint8_t)(cvt_e4m3x2(x[i], 0.0f) & 0xFFu);
}

cudaError_t launch_e4m3_from_f32(const float* x, int64_t n, uint8_t* q, int sms, cudaStream_t st) {
  const int64_t n4 = n / 4;
  if (n4 > 0) {
    static std::atomic<int> occ{0};
    auto k = e4m3_from_f32_kernel;
    k<<<grid_for((const void*)k, &occ, n4, sms), 256, 0, st>>>(reinterpret_cast<const float4*>(x), n4,
                                                                reinterpret_cast<uint32_t*>(q));
  }
  if (n % 4) e4m3_from_f32_tail_kernel<<<1, 4, 0, st>>>(x, 4 * n4, n, q);
  return cudaGetLastError();
}

cudaError_t launch_dequant_weight(const uint8_t* q, int64_t n, const float* s_w, uint16_t* wd, int sms,
                                  cudaStream_t st) {
  const int64_t n16 = n / 16;
  static std::atomic<int> occ{0};
  auto k = dequant_weight_kernel<kDequantU>;
  k<<<grid_for((const void*)k, &occ, n16, sms, kDequantU), 256, 0, st>>>(q, n16, s_w, wd);
  return cudaGetLastError();
}

cudaError_t launch_quant_static(const uint16_t* x, int64_t n, const float* s_in, uint8_t* q,
                                int sms, cudaStream_t st) {
  const int64_t n16 = n / 16;
  static std::atomic<int> occ{0};
  auto k = quant_static_kernel<kQuantU>;
  k<<<grid_for((const void*)k, &occ, n16, sms, kQuantU), 256, 0, st>>>(x, n16, s_in, q);
  return cudaGetLastError();
}

cudaError_t launch_swiglu_fp8(const uint16_t* g, const uint16_t* u, int64_t n, const float* s_out,
                              uint8_t* out, int sms, cudaStream_t st) {
  const int64_t n16 = n / 16;
  static std::atomic<int> occ{0};
  auto k = swiglu_fp8_kernel<kSwigluU>;
  k<<<grid_for((const void*)k, &occ, n16, sms, kSwigluU), 256, 0, st>>>(g, u, n16, s_out, out);
  return cudaGetLastError();
}

cudaError_t launch_ln_modulate_quant(const uint16_t* x, int64_t M, int K, const uint16_t* shift,
                                     const uint16_t* scale, int64_t rows_per_sample, float eps,
                                     const float* s_in, uint8_t* q, uint16_t* h, int sms, cudaStream_t st) {
  // kG = 256 / kT rows per block at a time; as many blocks as fit at once
  // (the ring is the kernel's dynamic shared memory, opted in above the
  // default per-block limit).
  static std::atomic<int> occ[15];
  const int kt = ln_group_threads(K);
  const int groups = 256 / kt;
  const int stages = ln_stages(K);
  const int ring = ln_table_bytes(K) + groups * stages * 2 * K;
  const int64_t blocks_wanted = (M + groups - 1) / groups;
  const int out = (q != nullptr ? 1 : 0) | (h != nullptr ? 2 : 0);
  if (out == 0) return cudaErrorInvalidValue;   // the entry point refuses this first
#define W8_LN_KERNEL(T, V, F)                                                                        \
  (out == 1 ? ln_modulate_quant_kernel<T, V, F, 1>                                                   \
            : out == 2 ? ln_modulate_quant_kernel<T, V, F, 2> : ln_modulate_quant_kernel<T, V, F, 3>)
#define W8_LN_LAUNCH(T, V, SLOT)                                                                      \
  {                                                                                                  \
    auto k = K == 8 * T * V ? W8_LN_KERNEL(T, V, true) : W8_LN_KERNEL(T, V, false);                   \
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, ring);      \
    if (e != cudaSuccess) return e;                                                                  \
    std::atomic<int>& o = occ[3 * (SLOT) + out - 1];                                                 \
    int b = o.load(std::memory_order_relaxed);                                                       \
    if (b == 0) {                                                                                    \
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, k, 256, ring) != cudaSuccess || b < 1) b = 1; \
      o.store(b, std::memory_order_relaxed);                                                         \
    }                                                                                                \
    const int64_t cap = (int64_t)sms * b;                                                            \
    const int grid = (int)(blocks_wanted < cap ? blocks_wanted : cap);                               \
    k<<<grid, 256, ring, st>>>(x, M, K, shift, scale, rows_per_sample, eps, stages, s_in, q, h);     \
  }
  if (K <= 512) W8_LN_LAUNCH(64, 1, 0)
  else if (K <= 1024) W8_LN_LAUNCH(64, 2, 1)
  else if (K <= 2048) W8_LN_LAUNCH(64, 4, 2)
  else if (K <= 4096) W8_LN_LAUNCH(64, 8, 3)
  else W8_LN_LAUNCH(128, 8, 4)
#undef W8_LN_LAUNCH
#undef W8_LN_KERNEL
  return cudaGetLastError();
}

cudaError_t elementwise_read_error(cudaStream_t st, uint32_t* err) {
  *err = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(err, g_elem_err, sizeof(uint32_t), 0, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e == cudaSuccess && *err != 0) {
    const uint32_t zero = 0;
    e = cudaMemcpyToSymbolAsync(g_elem_err, &zero, sizeof(uint32_t), 0, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  }
  return e;
}

cudaError_t launch_swiglu_bf16(const uint16_t* g, const uint16_t* u, int64_t n, uint16_t* out,
                               int sms, cudaStream_t st) {
  const int64_t n16 = n / 16;
  static std::atomic<int> occ{0};
  auto k = swiglu_bf16_kernel<kSwigluU>;
  k<<<grid_for((const void*)k, &occ, n16, sms, kSwigluU), 256, 0, st>>>(g, u, n16, out);
  return cudaGetLastError();
}

}  // namespace w8

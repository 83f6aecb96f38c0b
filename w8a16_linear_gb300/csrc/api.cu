// C-ABI entry points (include/w8lin.h): host-side argument validation, device
// checks, and dispatch to the kernels.  Validation happens before any CUDA
// call so that a bad argument never touches the GPU.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "../../include/w8lin.h"
#include "internal.h"

namespace {

thread_local char g_last_error[512] = "";

w8_status fail(w8_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return st;
}

w8_status ok() {
  g_last_error[0] = '\0';
  return W8_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

constexpr int kMaxDevices = 64;
int g_sms[kMaxDevices];      // 0 = not yet queried
int g_arch_ok[kMaxDevices];  // 0 = unknown, 1 = sm_103, -1 = other
std::mutex g_dev_mu;

// Checks that the current device is sm_103 and returns its SM count.
w8_status device_info(int* sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(W8_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(W8_ERR_CUDA, "device index %d out of range", dev);
  std::lock_guard<std::mutex> lk(g_dev_mu);
  if (g_arch_ok[dev] == 0) {
    int major = 0, minor = 0, n = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return fail(W8_ERR_CUDA, "cudaDeviceGetAttribute: %s", cudaGetErrorString(e));
    g_arch_ok[dev] = (major == 10 && minor == 3) ? 1 : -1;
    g_sms[dev] = n;
    if (g_arch_ok[dev] < 0)
      return fail(W8_ERR_ARCH, "device %d is sm_%d%d; this library is built for sm_103a", dev,
                  major, minor);
  }
  if (g_arch_ok[dev] < 0) return fail(W8_ERR_ARCH, "device %d is not sm_103", dev);
  *sms = g_sms[dev];
  return W8_OK;
}

w8_status cuda_status(cudaError_t e, const char* what) {
  if (e != cudaSuccess) return fail(W8_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  return ok();
}

}  // namespace

namespace w8 {

EncodeTiledFn get_encode_tiled() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

void set_last_error(const char* msg) {
  snprintf(g_last_error, sizeof(g_last_error), "%s", msg);
}

int query_device(int* sms) { return device_info(sms); }

}  // namespace w8

extern "C" {

int w8_abi_version(void) { return 6; }

const char* w8_last_error(void) { return g_last_error; }

w8_status w8_device_check(void) {
  int sms = 0;
  w8_status st = device_info(&sms);
  return st == W8_OK ? ok() : st;
}

w8_status w8_poll_device_error(void* stream) {
  uint32_t err = 0, err2 = 0;
  cudaError_t e = w8::gemm_read_error(static_cast<cudaStream_t>(stream), &err);
  if (e == cudaSuccess) e = w8::elementwise_read_error(static_cast<cudaStream_t>(stream), &err2);
  if (e != cudaSuccess) return fail(W8_ERR_CUDA, "reading device error word: %s", cudaGetErrorString(e));
  if (err & w8::kErrTimeout) return fail(W8_ERR_TIMEOUT, "a GEMM pipeline wait timed out");
  if (err2 & w8::kErrTimeout) return fail(W8_ERR_TIMEOUT, "a row-buffer wait of ln_modulate_quant timed out");
  return ok();
}

w8_status w8_selftest_timeout(void* stream) {
  int sms = 0;
  w8_status st = device_info(&sms);
  if (st != W8_OK) return st;
  return cuda_status(w8::launch_selftest_timeout(static_cast<cudaStream_t>(stream)),
                     "w8_selftest_timeout launch");
}

w8_status fp8_quant_static(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, const float* s_in,
                           uint8_t* q, int64_t ldq, void* stream) {
  if (M < 0 || K <= 0) return fail(W8_ERR_SHAPE, "fp8_quant_static: M=%lld K=%lld", (long long)M, (long long)K);
  if (K % 16) return fail(W8_ERR_SHAPE, "fp8_quant_static: K=%lld is not a multiple of 16", (long long)K);
  // Rows must be dense: a padded or strided activation is refused rather
  // than read with the wrong pitch.
  if (ldx != K || ldq != K)
    return fail(W8_ERR_STRIDE, "fp8_quant_static: ldx=%lld ldq=%lld, both must equal K=%lld (dense rows)",
                (long long)ldx, (long long)ldq, (long long)K);
  if (M == 0) return ok();
  if (!x || !s_in || !q) return fail(W8_ERR_NULL, "fp8_quant_static: NULL pointer");
  if (!aligned16(x) || !aligned16(q) || (reinterpret_cast<uintptr_t>(s_in) & 3u))
    return fail(W8_ERR_ALIGN, "fp8_quant_static: x and q must be 16-byte aligned");
  int sms = 0;
  w8_status st = device_info(&sms);
  if (st != W8_OK) return st;
  return cuda_status(w8::launch_quant_static(x, M * K, s_in, q, sms, static_cast<cudaStream_t>(stream)),
                     "fp8_quant_static launch");
}

static w8_status check_linear_common(const char* fn, const void* x, int64_t M, int64_t K,
                                     const uint8_t* w, int64_t N, const float* s_w, const uint16_t* y) {
  if (M < 0 || K <= 0 || N <= 0)
    return fail(W8_ERR_SHAPE, "%s: M=%lld K=%lld N=%lld", fn, (long long)M, (long long)K, (long long)N);
  if (K % 16 || N % 16)
    return fail(W8_ERR_SHAPE, "%s: K=%lld and N=%lld must be multiples of 16", fn, (long long)K, (long long)N);
  if (M > INT32_MAX / 2 || K > INT32_MAX / 2 || N > INT32_MAX / 2)
    return fail(W8_ERR_SHAPE, "%s: dimension too large", fn);
  if (M == 0) return W8_OK;
  if (!x || !w || !s_w || !y) return fail(W8_ERR_NULL, "%s: NULL pointer", fn);
  if (!aligned16(x) || !aligned16(w) || !aligned16(y) || (reinterpret_cast<uintptr_t>(s_w) & 3u))
    return fail(W8_ERR_ALIGN, "%s: x, w and y must be 16-byte aligned", fn);
  return W8_OK;
}

w8_status fp8_linear_w8a8(const void* x, int32_t x_dtype, int64_t M, int64_t K, const uint8_t* w,
                          int64_t N, const float* s_in, const float* s_w, uint16_t* y, uint8_t* ws,
                          void* stream) {
  if (x_dtype != W8_DTYPE_BF16 && x_dtype != W8_DTYPE_E4M3)
    return fail(W8_ERR_DTYPE, "fp8_linear_w8a8: unknown activation dtype %d", x_dtype);
  w8_status st = check_linear_common("fp8_linear_w8a8", x, M, K, w, N, s_w, y);
  if (st != W8_OK) return st;
  if (M == 0) return ok();
  if (!s_in) return fail(W8_ERR_NULL, "fp8_linear_w8a8: NULL s_in");
  if (x_dtype == W8_DTYPE_BF16) {
    if (!ws) return fail(W8_ERR_NULL, "fp8_linear_w8a8: bf16 input needs the [M,K] E4M3 workspace");
    if (!aligned16(ws)) return fail(W8_ERR_ALIGN, "fp8_linear_w8a8: ws must be 16-byte aligned");
  }
  int sms = 0;
  if ((st = device_info(&sms)) != W8_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const uint8_t* qx = static_cast<const uint8_t*>(x);
  if (x_dtype == W8_DTYPE_BF16) {
    cudaError_t e = w8::launch_quant_static(static_cast<const uint16_t*>(x), M * K, s_in, ws, sms, s);
    if (e != cudaSuccess) return cuda_status(e, "fp8_linear_w8a8: quant launch");
    qx = ws;
  }
  w8::GemmProblem p{};
  p.M = M;
  p.K = K;
  p.G = 1;
  p.x = qx;
  p.w[0] = w;
  p.N[0] = N;
  p.s_in = s_in;
  p.s_w[0] = s_w;
  p.y[0] = y;
  int terr = 0;
  cudaError_t e = w8::launch_gemm_w8a8(p, sms, s, &terr);
  if (terr) return fail(W8_ERR_ALIGN, "fp8_linear_w8a8: tensor map encoding rejected the operands");
  return cuda_status(e, "fp8_linear_w8a8: GEMM launch");
}

w8_status fp8_linear_w8a16(const void* x, int32_t x_dtype, int64_t M, int64_t K, const uint8_t* w,
                           int64_t N, const float* s_w, uint16_t* y, uint16_t* ws, void* stream) {
  if (x_dtype != W8_DTYPE_BF16)
    return fail(W8_ERR_DTYPE,
                "fp8_linear_w8a16: activation must be bf16; an already-quantized input is refused");
  w8_status st = check_linear_common("fp8_linear_w8a16", x, M, K, w, N, s_w, y);
  if (st != W8_OK) return st;
  if (M == 0) return ok();
  if (ws && !aligned16(ws)) return fail(W8_ERR_ALIGN, "fp8_linear_w8a16: ws must be 16-byte aligned");
  int sms = 0;
  if ((st = device_info(&sms)) != W8_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  w8::GemmProblem p{};
  p.M = M;
  p.K = K;
  p.G = 1;
  p.x = x;
  p.w[0] = w;
  p.N[0] = N;
  p.s_w[0] = s_w;
  p.y[0] = y;
  int terr = 0;
  cudaError_t e;
  if (ws) {
    // dequant + F.linear: the weight into ws, then the bf16 GEMM on it
    e = w8::launch_dequant_weight(w, N * K, s_w, ws, sms, s);
    if (e != cudaSuccess) return cuda_status(e, "fp8_linear_w8a16: dequantization launch");
    p.w[0] = reinterpret_cast<const uint8_t*>(ws);
    e = w8::launch_gemm_bf16(p, sms, s, &terr);
  } else {
    e = w8::launch_gemm_w8a16(p, sms, s, &terr);
  }
  if (terr) return fail(W8_ERR_ALIGN, "fp8_linear_w8a16: tensor map encoding rejected the operands");
  return cuda_status(e, "fp8_linear_w8a16: GEMM launch");
}

w8_status qkv_shared_quant_gemm(int32_t mode, const uint16_t* x, int64_t M, int64_t K,
                                const float* s_in, int32_t G, const uint8_t* const* w,
                                const int64_t* N, const float* const* s_w, uint16_t* const* y,
                                uint8_t* ws, void* stream) {
  if (mode != W8_MODE_A8 && mode != W8_MODE_A16)
    return fail(W8_ERR_SHAPE, "qkv_shared_quant_gemm: unknown mode %d", mode);
  if (G < 1 || G > w8::kMaxGroup)
    return fail(W8_ERR_SHAPE, "qkv_shared_quant_gemm: group size %d outside 1..3", G);
  if (!w || !N || !s_w || !y) return fail(W8_ERR_NULL, "qkv_shared_quant_gemm: NULL host array");
  for (int g = 0; g < G; ++g) {
    w8_status st = check_linear_common("qkv_shared_quant_gemm", x, M, K, w[g], N[g], s_w[g], y[g]);
    if (st != W8_OK) return st;
  }
  if (M == 0) return ok();
  if (mode == W8_MODE_A8) {
    if (!s_in) return fail(W8_ERR_NULL, "qkv_shared_quant_gemm: NULL s_in");
    if (!ws) return fail(W8_ERR_NULL, "qkv_shared_quant_gemm: A8 needs the [M,K] E4M3 workspace");
  }
  if (ws && !aligned16(ws)) return fail(W8_ERR_ALIGN, "qkv_shared_quant_gemm: ws must be 16-byte aligned");
  int sms = 0;
  w8_status st = device_info(&sms);
  if (st != W8_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  w8::GemmProblem p{};
  p.M = M;
  p.K = K;
  p.G = G;
  for (int g = 0; g < G; ++g) {
    p.w[g] = w[g];
    p.N[g] = N[g];
    p.s_w[g] = s_w[g];
    p.y[g] = y[g];
  }
  int terr = 0;
  cudaError_t e;
  if (mode == W8_MODE_A8) {
    e = w8::launch_quant_static(x, M * K, s_in, ws, sms, s);
    if (e != cudaSuccess) return cuda_status(e, "qkv_shared_quant_gemm: quant launch");
    p.x = ws;
    p.s_in = s_in;
    e = w8::launch_gemm_w8a8(p, sms, s, &terr);
  } else if (ws) {
    // dequant + F.linear: the group's weights into ws, then one bf16 launch
    uint16_t* wd = reinterpret_cast<uint16_t*>(ws);
    for (int g = 0; g < G; ++g) {
      e = w8::launch_dequant_weight(w[g], N[g] * K, s_w[g], wd, sms, s);
      if (e != cudaSuccess) return cuda_status(e, "qkv_shared_quant_gemm: dequantization launch");
      p.w[g] = reinterpret_cast<const uint8_t*>(wd);
      wd += N[g] * K;
    }
    p.x = x;
    e = w8::launch_gemm_bf16(p, sms, s, &terr);
  } else {
    p.x = x;
    e = w8::launch_gemm_w8a16(p, sms, s, &terr);
  }
  if (terr) return fail(W8_ERR_ALIGN, "qkv_shared_quant_gemm: tensor map encoding rejected the operands");
  return cuda_status(e, "qkv_shared_quant_gemm: GEMM launch");
}

w8_status fp8_e4m3_from_f32(const float* x, int64_t n, uint8_t* q, void* stream) {
  if (n < 0) return fail(W8_ERR_SHAPE, "fp8_e4m3_from_f32: n=%lld", (long long)n);
  if (n == 0) return ok();
  if (!x || !q) return fail(W8_ERR_NULL, "fp8_e4m3_from_f32: NULL pointer");
  if (!aligned16(x) || (reinterpret_cast<uintptr_t>(q) & 3u))
    return fail(W8_ERR_ALIGN, "fp8_e4m3_from_f32: x must be 16-byte and q 4-byte aligned");
  int sms = 0;
  w8_status st = device_info(&sms);
  if (st != W8_OK) return st;
  return cuda_status(w8::launch_e4m3_from_f32(x, n, q, sms, static_cast<cudaStream_t>(stream)),
                     "fp8_e4m3_from_f32 launch");
}

w8_status fp8_dequant_weight(const uint8_t* w, int64_t N, int64_t K, const float* s_w, uint16_t* wd,
                             void* stream) {
  if (N < 0 || K < 0) return fail(W8_ERR_SHAPE, "fp8_dequant_weight: N=%lld K=%lld", (long long)N, (long long)K);
  if (K % 16) return fail(W8_ERR_SHAPE, "fp8_dequant_weight: K=%lld is not a multiple of 16", (long long)K);
  if (N == 0 || K == 0) return ok();
  if (!w || !s_w || !wd) return fail(W8_ERR_NULL, "fp8_dequant_weight: NULL pointer");
  if (!aligned16(w) || !aligned16(wd)) return fail(W8_ERR_ALIGN, "fp8_dequant_weight: w and wd must be 16-byte aligned");
  int sms = 0;
  w8_status st = device_info(&sms);
  if (st != W8_OK) return st;
  return cuda_status(w8::launch_dequant_weight(w, N * K, s_w, wd, sms, static_cast<cudaStream_t>(stream)),
                     "fp8_dequant_weight launch");
}

w8_status bf16_linear_group(const uint16_t* x, int64_t M, int64_t K, int32_t G, const uint16_t* const* wd,
                            const int64_t* N, uint16_t* const* y, void* stream) {
  if (G < 1 || G > w8::kMaxGroup)
    return fail(W8_ERR_SHAPE, "bf16_linear_group: group size %d outside 1..3", G);
  if (!wd || !N || !y) return fail(W8_ERR_NULL, "bf16_linear_group: NULL host array");
  static const float kOne = 1.0f;  // placeholder scale: the common check wants a pointer
  for (int g = 0; g < G; ++g) {
    w8_status st = check_linear_common("bf16_linear_group", x, M, K, reinterpret_cast<const uint8_t*>(wd[g]),
                                       N[g], &kOne, y[g]);
    if (st != W8_OK) return st;
  }
  if (M == 0) return ok();
  int sms = 0;
  w8_status st = device_info(&sms);
  if (st != W8_OK) return st;
  w8::GemmProblem p{};
  p.M = M;
  p.K = K;
  p.G = G;
  p.x = x;
  for (int g = 0; g < G; ++g) {
    p.w[g] = reinterpret_cast<const uint8_t*>(wd[g]);
    p.N[g] = N[g];
    p.y[g] = y[g];
  }
  int terr = 0;
  cudaError_t e = w8::launch_gemm_bf16(p, sms, static_cast<cudaStream_t>(stream), &terr);
  if (terr) return fail(W8_ERR_ALIGN, "bf16_linear_group: tensor map encoding rejected the operands");
  return cuda_status(e, "bf16_linear_group: GEMM launch");
}

// The SwiGLU options, checked and copied (the standalone and the fused
// forms share them).
static w8_status check_swiglu_params(const char* fn, const w8_swiglu_params* prm, w8::SwigluExArgs* a) {
  if (!prm) return fail(W8_ERR_NULL, "%s: NULL params", fn);
  if (!std::isfinite(prm->alpha) || !std::isfinite(prm->beta))
    return fail(W8_ERR_PARAM, "%s: alpha and beta must be finite", fn);
  if (prm->has_limit && !(std::isfinite(prm->limit) && prm->limit > 0.0f))
    return fail(W8_ERR_PARAM, "%s: limit must be finite and > 0", fn);
  a->has_limit = prm->has_limit != 0;
  a->limit = prm->limit;
  a->alpha = prm->alpha;
  a->beta = prm->beta;
  return W8_OK;
}

static w8_status bf16_gate_up_swiglu_impl(const char* fn, const uint16_t* x, int64_t M, int64_t K,
                                          const uint16_t* wd_gate, const uint16_t* wd_up, int64_t I,
                                          const w8::SwigluExArgs* ex, uint16_t* out, void* stream) {
  static const float kOne = 1.0f;  // placeholder scale: the common check wants a pointer
  const uint8_t* wg = reinterpret_cast<const uint8_t*>(wd_gate);
  const uint8_t* wu = reinterpret_cast<const uint8_t*>(wd_up);
  w8_status st = check_linear_common(fn, x, M, K, wg, I, &kOne, out);
  if (st != W8_OK) return st;
  if ((st = check_linear_common(fn, x, M, K, wu, I, &kOne, out)) != W8_OK) return st;
  if (M == 0) return ok();
  int sms = 0;
  if ((st = device_info(&sms)) != W8_OK) return st;
  w8::GemmProblem p{};
  p.M = M;
  p.K = K;
  p.G = 1;
  p.x = x;
  p.w[0] = wg;
  p.w[1] = wu;
  p.N[0] = I;
  p.N[1] = I;
  p.y[0] = out;
  p.ex = ex;
  int terr = 0;
  cudaError_t e = w8::launch_gemm_glu16(p, sms, static_cast<cudaStream_t>(stream), &terr);
  if (terr) return fail(W8_ERR_ALIGN, "%s: tensor map encoding rejected the operands", fn);
  return cuda_status(e, "bf16_gate_up_swiglu: GEMM launch");
}

w8_status bf16_gate_up_swiglu(const uint16_t* x, int64_t M, int64_t K, const uint16_t* wd_gate,
                              const uint16_t* wd_up, int64_t I, uint16_t* out, void* stream) {
  return bf16_gate_up_swiglu_impl("bf16_gate_up_swiglu", x, M, K, wd_gate, wd_up, I, nullptr, out, stream);
}

w8_status bf16_gate_up_swiglu_ex(const uint16_t* x, int64_t M, int64_t K, const uint16_t* wd_gate,
                                 const uint16_t* wd_up, int64_t I, const w8_swiglu_params* prm,
                                 uint16_t* out, void* stream) {
  w8::SwigluExArgs a{};
  w8_status st = check_swiglu_params("bf16_gate_up_swiglu_ex", prm, &a);
  if (st != W8_OK) return st;
  return bf16_gate_up_swiglu_impl("bf16_gate_up_swiglu_ex", x, M, K, wd_gate, wd_up, I, &a, out, stream);
}

w8_status fp8_linear_w8a8_group(const uint8_t* qx, int64_t M, int64_t K, const float* s_in,
                                int32_t G, const uint8_t* const* w, const int64_t* N,
                                const float* const* s_w, uint16_t* const* y, void* stream) {
  if (G < 1 || G > w8::kMaxGroup)
    return fail(W8_ERR_SHAPE, "fp8_linear_w8a8_group: group size %d outside 1..3", G);
  if (!w || !N || !s_w || !y) return fail(W8_ERR_NULL, "fp8_linear_w8a8_group: NULL host array");
  for (int g = 0; g < G; ++g) {
    w8_status st = check_linear_common("fp8_linear_w8a8_group", qx, M, K, w[g], N[g], s_w[g], y[g]);
    if (st != W8_OK) return st;
  }
  if (M == 0) return ok();
  if (!s_in) return fail(W8_ERR_NULL, "fp8_linear_w8a8_group: NULL s_in");
  int sms = 0;
  w8_status st = device_info(&sms);
  if (st != W8_OK) return st;
  w8::GemmProblem p{};
  p.M = M;
  p.K = K;
  p.G = G;
  p.x = qx;
  p.s_in = s_in;
  for (int g = 0; g < G; ++g) {
    p.w[g] = w[g];
    p.N[g] = N[g];
    p.s_w[g] = s_w[g];
    p.y[g] = y[g];
  }
  int terr = 0;
  cudaError_t e = w8::launch_gemm_w8a8(p, sms, static_cast<cudaStream_t>(stream), &terr);
  if (terr) return fail(W8_ERR_ALIGN, "fp8_linear_w8a8_group: tensor map encoding rejected the operands");
  return cuda_status(e, "fp8_linear_w8a8_group: GEMM launch");
}

static w8_status gate_up_swiglu_fp8_impl(const char* fn, const void* x, int32_t x_dtype, int64_t M,
                                         int64_t K, const float* s_in, const uint8_t* w_gate,
                                         const uint8_t* w_up, int64_t I, const float* s_w_gate,
                                         const float* s_w_up, const w8::SwigluExArgs* ex, const float* s_out,
                                         uint8_t* out, uint8_t* ws, void* stream) {
  if (x_dtype != W8_DTYPE_BF16 && x_dtype != W8_DTYPE_E4M3)
    return fail(W8_ERR_DTYPE, "%s: unknown activation dtype %d", fn, x_dtype);
  w8_status st = check_linear_common(fn, x, M, K, w_gate, I, s_w_gate, reinterpret_cast<const uint16_t*>(out));
  if (st != W8_OK) return st;
  if (M == 0) return ok();
  if (!w_up || !s_w_up || !s_in || !s_out) return fail(W8_ERR_NULL, "%s: NULL pointer", fn);
  if (!aligned16(w_up)) return fail(W8_ERR_ALIGN, "%s: w_up must be 16-byte aligned", fn);
  if (x_dtype == W8_DTYPE_BF16) {
    if (!ws) return fail(W8_ERR_NULL, "%s: bf16 input needs the [M,K] E4M3 workspace", fn);
    if (!aligned16(ws)) return fail(W8_ERR_ALIGN, "%s: ws must be 16-byte aligned", fn);
  }
  int sms = 0;
  if ((st = device_info(&sms)) != W8_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const uint8_t* qx = static_cast<const uint8_t*>(x);
  if (x_dtype == W8_DTYPE_BF16) {
    cudaError_t e = w8::launch_quant_static(static_cast<const uint16_t*>(x), M * K, s_in, ws, sms, s);
    if (e != cudaSuccess) return cuda_status(e, "gate_up_swiglu_fp8: quant launch");
    qx = ws;
  }
  w8::GemmProblem p{};
  p.M = M;
  p.K = K;
  p.G = 1;
  p.x = qx;
  p.w[0] = w_gate;
  p.w[1] = w_up;
  p.N[0] = I;
  p.s_in = s_in;
  p.s_w[0] = s_w_gate;
  p.s_w[1] = s_w_up;
  p.y[0] = out;
  p.s_out = s_out;
  p.ex = ex;
  int terr = 0;
  cudaError_t e = w8::launch_gemm_glu(p, sms, s, &terr);
  if (terr) return fail(W8_ERR_ALIGN, "%s: tensor map encoding rejected the operands", fn);
  return cuda_status(e, "gate_up_swiglu_fp8: GEMM launch");
}

w8_status gate_up_swiglu_fp8(const void* x, int32_t x_dtype, int64_t M, int64_t K,
                             const float* s_in, const uint8_t* w_gate, const uint8_t* w_up,
                             int64_t I, const float* s_w_gate, const float* s_w_up,
                             const float* s_out, uint8_t* out, uint8_t* ws, void* stream) {
  return gate_up_swiglu_fp8_impl("gate_up_swiglu_fp8", x, x_dtype, M, K, s_in, w_gate, w_up, I, s_w_gate,
                                 s_w_up, nullptr, s_out, out, ws, stream);
}

w8_status gate_up_swiglu_ex_fp8(const void* x, int32_t x_dtype, int64_t M, int64_t K,
                                const float* s_in, const uint8_t* w_gate, const uint8_t* w_up,
                                int64_t I, const float* s_w_gate, const float* s_w_up,
                                const w8_swiglu_params* prm, const float* s_out, uint8_t* out,
                                uint8_t* ws, void* stream) {
  w8::SwigluExArgs a{};
  w8_status st = check_swiglu_params("gate_up_swiglu_ex_fp8", prm, &a);
  if (st != W8_OK) return st;
  return gate_up_swiglu_fp8_impl("gate_up_swiglu_ex_fp8", x, x_dtype, M, K, s_in, w_gate, w_up, I, s_w_gate,
                                 s_w_up, &a, s_out, out, ws, stream);
}

static w8_status check_swiglu(const char* fn, const uint16_t* g, const uint16_t* u, int64_t M,
                              int64_t I, const void* out) {
  if (M < 0 || I <= 0) return fail(W8_ERR_SHAPE, "%s: M=%lld I=%lld", fn, (long long)M, (long long)I);
  if (I % 16) return fail(W8_ERR_SHAPE, "%s: I=%lld is not a multiple of 16", fn, (long long)I);
  if (M == 0) return W8_OK;
  if (!g || !u || !out) return fail(W8_ERR_NULL, "%s: NULL pointer", fn);
  if (!aligned16(g) || !aligned16(u) || !aligned16(out))
    return fail(W8_ERR_ALIGN, "%s: gate, up and out must be 16-byte aligned", fn);
  return W8_OK;
}

w8_status swiglu_2in_fp8(const uint16_t* gate, const uint16_t* up, int64_t M, int64_t I,
                         const float* s_out, uint8_t* out, void* stream) {
  w8_status st = check_swiglu("swiglu_2in_fp8", gate, up, M, I, out);
  if (st != W8_OK) return st;
  if (M == 0) return ok();
  if (!s_out) return fail(W8_ERR_NULL, "swiglu_2in_fp8: NULL s_out");
  int sms = 0;
  if ((st = device_info(&sms)) != W8_OK) return st;
  return cuda_status(w8::launch_swiglu_fp8(gate, up, M * I, s_out, out, sms,
                                           static_cast<cudaStream_t>(stream)),
                     "swiglu_2in_fp8 launch");
}

w8_status swiglu_2in_bf16(const uint16_t* gate, const uint16_t* up, int64_t M, int64_t I,
                          uint16_t* out, void* stream) {
  w8_status st = check_swiglu("swiglu_2in_bf16", gate, up, M, I, out);
  if (st != W8_OK) return st;
  if (M == 0) return ok();
  int sms = 0;
  if ((st = device_info(&sms)) != W8_OK) return st;
  return cuda_status(w8::launch_swiglu_bf16(gate, up, M * I, out, sms, static_cast<cudaStream_t>(stream)),
                     "swiglu_2in_bf16 launch");
}

static w8_status check_swiglu_ex(const char* fn, const void* g, const void* u, int32_t in_dtype,
                                 int64_t M, int64_t I, const w8_swiglu_params* prm, const void* out,
                                 w8::SwigluExArgs* a) {
  w8_status st = check_swiglu(fn, static_cast<const uint16_t*>(g), static_cast<const uint16_t*>(u), M, I,
                              out);
  if (st != W8_OK) return st;
  if (in_dtype != W8_DTYPE_BF16 && in_dtype != W8_DTYPE_F16)
    return fail(W8_ERR_DTYPE, "%s: in_dtype %d is neither bf16 nor f16", fn, in_dtype);
  return check_swiglu_params(fn, prm, a);
}

w8_status swiglu_2in_ex_fp8(const void* gate, const void* up, int32_t in_dtype, int64_t M, int64_t I,
                            const w8_swiglu_params* prm, const float* s_out, uint8_t* out,
                            void* stream) {
  w8::SwigluExArgs a{};
  w8_status st = check_swiglu_ex("swiglu_2in_ex_fp8", gate, up, in_dtype, M, I, prm, out, &a);
  if (st != W8_OK) return st;
  if (M == 0) return ok();
  if (!s_out) return fail(W8_ERR_NULL, "swiglu_2in_ex_fp8: NULL s_out");
  int sms = 0;
  if ((st = device_info(&sms)) != W8_OK) return st;
  return cuda_status(w8::launch_swiglu_ex(static_cast<const uint16_t*>(gate), static_cast<const uint16_t*>(up),
                                          M * I, in_dtype == W8_DTYPE_F16, true, a, s_out, out, sms,
                                          static_cast<cudaStream_t>(stream)),
                     "swiglu_2in_ex_fp8 launch");
}

w8_status swiglu_2in_ex_16(const void* gate, const void* up, int32_t in_dtype, int64_t M, int64_t I,
                           const w8_swiglu_params* prm, void* out, void* stream) {
  w8::SwigluExArgs a{};
  w8_status st = check_swiglu_ex("swiglu_2in_ex_16", gate, up, in_dtype, M, I, prm, out, &a);
  if (st != W8_OK) return st;
  if (M == 0) return ok();
  int sms = 0;
  if ((st = device_info(&sms)) != W8_OK) return st;
  return cuda_status(w8::launch_swiglu_ex(static_cast<const uint16_t*>(gate), static_cast<const uint16_t*>(up),
                                          M * I, in_dtype == W8_DTYPE_F16, false, a, nullptr, out, sms,
                                          static_cast<cudaStream_t>(stream)),
                     "swiglu_2in_ex_16 launch");
}

w8_status ln_modulate_quant(const uint16_t* x, int64_t M, int64_t K, const uint16_t* shift,
                            const uint16_t* scale, int64_t rows_per_sample, float eps,
                            const float* s_in, uint8_t* q, uint16_t* h, void* stream) {
  if (M < 0 || K < 8 || K > 8192 || K % 8)
    return fail(W8_ERR_SHAPE, "ln_modulate_quant: M=%lld K=%lld (need 8 <= K <= 8192, K %% 8 == 0)",
                (long long)M, (long long)K);
  if (rows_per_sample < 1 || (M % rows_per_sample) != 0)
    return fail(W8_ERR_SHAPE, "ln_modulate_quant: rows_per_sample=%lld does not divide M=%lld",
                (long long)rows_per_sample, (long long)M);
  if (!std::isfinite(eps) || eps < 0.0f) return fail(W8_ERR_PARAM, "ln_modulate_quant: eps=%g", (double)eps);
  if (M == 0) return ok();
  if (!x || !shift || !scale) return fail(W8_ERR_NULL, "ln_modulate_quant: NULL input");
  if (!q && !h) return fail(W8_ERR_NULL, "ln_modulate_quant: neither q nor h given");
  if (q && !s_in) return fail(W8_ERR_NULL, "ln_modulate_quant: q needs s_in");
  if (!aligned16(x) || !aligned16(shift) || !aligned16(scale) || (q && !aligned16(q)) || (h && !aligned16(h)) ||
      (q && (reinterpret_cast<uintptr_t>(s_in) & 3u)))
    return fail(W8_ERR_ALIGN, "ln_modulate_quant: arrays must be 16-byte aligned");
  int sms = 0;
  w8_status st = device_info(&sms);
  if (st != W8_OK) return st;
  return cuda_status(w8::launch_ln_modulate_quant(x, M, (int)K, shift, scale, rows_per_sample, eps, s_in, q, h,
                                                  sms, static_cast<cudaStream_t>(stream)),
                     "ln_modulate_quant launch");
}

w8_status step_policy_dispatch(const w8_step_policy* policy, int32_t step, int32_t num_steps,
                               int32_t* mode_out) {
  if (!mode_out) return fail(W8_ERR_NULL, "step_policy_dispatch: NULL mode_out");
  if (num_steps < 1 || step < 0 || step >= num_steps)
    return fail(W8_ERR_POLICY, "step_policy_dispatch: step %d outside [0, %d)", step, num_steps);
  if (!policy || !policy->enabled) {
    *mode_out = W8_MODE_A8;
    return ok();
  }
  if (policy->schema_version != 1)
    return fail(W8_ERR_POLICY, "step_policy_dispatch: schema_version %d is not 1", policy->schema_version);
  if (policy->first_steps < 0 || policy->last_steps < 0)
    return fail(W8_ERR_POLICY, "step_policy_dispatch: negative step window");
  if (num_steps == 1) {
    *mode_out = W8_MODE_A8;
    return ok();
  }
  const bool edge = step < policy->first_steps || step >= num_steps - policy->last_steps;
  *mode_out = edge ? W8_MODE_A16 : W8_MODE_A8;
  return ok();
}

w8_status w8_check_group_scales(const float* const* s_in, int32_t G) {
  if (G < 1) return fail(W8_ERR_SHAPE, "w8_check_group_scales: G=%d", G);
  if (!s_in) return fail(W8_ERR_NULL, "w8_check_group_scales: NULL array");
  for (int g = 0; g < G; ++g)
    if (!s_in[g]) return fail(W8_ERR_NULL, "w8_check_group_scales: NULL scale %d", g);
  uint32_t first = 0;
  for (int g = 0; g < G; ++g) {
    uint32_t v = 0;
    cudaError_t e = cudaMemcpy(&v, s_in[g], sizeof(float), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_status(e, "w8_check_group_scales: read scale");
    if (g == 0) first = v;
    else if (v != first)
      return fail(W8_ERR_SCALE, "w8_check_group_scales: input scale %d differs from scale 0", g);
  }
  return ok();
}

}  // extern "C"

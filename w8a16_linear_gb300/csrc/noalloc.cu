// fp8_linear_w8a8_noalloc: the bf16-input W8A8 linear for callers that cannot
// allocate device memory.
//
// fp8_linear_w8a8 quantizes a bf16 activation into a caller-provided E4M3
// workspace before the GEMM reads it.  Some callers have no way to provide
// one: a plugin or operator interface that hands the kernel only its inputs
// and outputs, a runtime whose device memory is owned by a pool it cannot
// grow, or code that must not call cudaMalloc (which can synchronise the
// device and is not allowed while a stream is being captured).  This entry
// point instead uses a fixed scratch array that lives in this file as a
// device global, so it allocates nothing at all.
//
// Costs and rules of that choice:
//  * Every GPU that loads the library holds kScratchBytes (32 MiB) of device
//    memory for this array until the process exits.
//  * One array per device is shared by every call on that device: two calls
//    whose work overlaps on the GPU (different streams, no ordering between
//    them) race on it.  Calls on one stream, or otherwise ordered, are safe.
//  * Nothing in the array needs to start at zero: the quantization kernel
//    writes all M*K bytes it uses before the GEMM reads them, so contents
//    left by an earlier call are never read.
//  * The device address of the array is looked up once per device, with that
//    device current, by the first call on it (cudaGetSymbolAddress).  Make
//    that first call before any stream capture begins.
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <mutex>

#include "../../include/w8lin.h"
#include "internal.h"

namespace {

constexpr int64_t kScratchBytes = int64_t(32) << 20;  // 32 MiB: M*K E4M3 codes
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_noalloc_scratch[kScratchBytes];

uint8_t* g_scratch_ptr[kMaxDevices];  // device address per device, set up once
std::mutex g_scratch_mu;

w8_status nfail(w8_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  w8::set_last_error(buf);
  return st;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Looks up (once per device, with that device current) the device address of
// the scratch array; also checks the device architecture and SM count.
w8_status scratch_for_current_device(uint8_t** ptr, int* sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return nfail(W8_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return nfail(W8_ERR_CUDA, "device index %d out of range", dev);
  w8_status st = static_cast<w8_status>(w8::query_device(sms));
  if (st != W8_OK) return st;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p)
      return nfail(W8_ERR_CUDA, "fp8_linear_w8a8_noalloc: cudaGetSymbolAddress: %s",
                   cudaGetErrorString(e));
    g_scratch_ptr[dev] = static_cast<uint8_t*>(p);
  }
  *ptr = g_scratch_ptr[dev];
  return W8_OK;
}

}  // namespace

extern "C" w8_status fp8_linear_w8a8_noalloc(const uint16_t* x, int64_t M, int64_t K,
                                             const uint8_t* w, int64_t N, const float* s_in,
                                             const float* s_w, uint16_t* y, void* stream) {
  if (M < 0 || K <= 0 || N <= 0)
    return nfail(W8_ERR_SHAPE, "fp8_linear_w8a8_noalloc: M=%lld K=%lld N=%lld", (long long)M,
                 (long long)K, (long long)N);
  if (K % 16 || N % 16)
    return nfail(W8_ERR_SHAPE, "fp8_linear_w8a8_noalloc: K=%lld and N=%lld must be multiples of 16",
                 (long long)K, (long long)N);
  if (K > kScratchBytes || M > kScratchBytes / K)
    return nfail(W8_ERR_SHAPE,
                 "fp8_linear_w8a8_noalloc: M*K = %lld*%lld exceeds the fixed scratch of %lld bytes "
                 "(use fp8_linear_w8a8 with a workspace for larger activations)",
                 (long long)M, (long long)K, (long long)kScratchBytes);
  if (N > INT32_MAX / 2) return nfail(W8_ERR_SHAPE, "fp8_linear_w8a8_noalloc: N too large");
  if (M == 0) {
    w8::set_last_error("");
    return W8_OK;
  }
  if (!x || !w || !s_in || !s_w || !y) return nfail(W8_ERR_NULL, "fp8_linear_w8a8_noalloc: NULL pointer");
  if (!aligned16(x) || !aligned16(w) || !aligned16(y) || (reinterpret_cast<uintptr_t>(s_in) & 3u) ||
      (reinterpret_cast<uintptr_t>(s_w) & 3u))
    return nfail(W8_ERR_ALIGN, "fp8_linear_w8a8_noalloc: x, w and y must be 16-byte aligned");
  uint8_t* scratch = nullptr;
  int sms = 0;
  w8_status st = scratch_for_current_device(&scratch, &sms);
  if (st != W8_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = w8::launch_quant_static(x, M * K, s_in, scratch, sms, s);
  if (e != cudaSuccess)
    return nfail(W8_ERR_CUDA, "fp8_linear_w8a8_noalloc: quant launch: %s", cudaGetErrorString(e));
  w8::GemmProblem p{};
  p.M = M;
  p.K = K;
  p.G = 1;
  p.x = scratch;
  p.w[0] = w;
  p.N[0] = N;
  p.s_in = s_in;
  p.s_w[0] = s_w;
  p.y[0] = y;
  int terr = 0;
  e = w8::launch_gemm_w8a8(p, sms, s, &terr);
  if (terr) return nfail(W8_ERR_ALIGN, "fp8_linear_w8a8_noalloc: tensor map encoding rejected the operands");
  if (e != cudaSuccess)
    return nfail(W8_ERR_CUDA, "fp8_linear_w8a8_noalloc: GEMM launch: %s", cudaGetErrorString(e));
  w8::set_last_error("");
  return W8_OK;
}

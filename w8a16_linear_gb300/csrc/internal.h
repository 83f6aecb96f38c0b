// Internal launcher interface between the C-ABI layer (api.cu) and the
// kernel translation units.  Not part of the public header.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace w8 {

// Error word bits set by kernels that wait on mbarriers.
enum : uint32_t {
  kErrTimeout = 1u,   // an mbarrier wait ran past its deadline
};

// ---- elementwise (elementwise.cu)
cudaError_t launch_quant_static(const uint16_t* x, int64_t n, const float* s_in, uint8_t* q,
                                int sms, cudaStream_t st);
cudaError_t launch_swiglu_fp8(const uint16_t* g, const uint16_t* u, int64_t n, const float* s_out,
                              uint8_t* out, int sms, cudaStream_t st);
cudaError_t launch_swiglu_bf16(const uint16_t* g, const uint16_t* u, int64_t n, uint16_t* out,
                               int sms, cudaStream_t st);

// Binary32 -> E4M3 codes (x 16-byte aligned, q 4-byte aligned).
cudaError_t launch_e4m3_from_f32(const float* x, int64_t n, uint8_t* q, int sms, cudaStream_t st);

cudaError_t launch_dequant_weight(const uint8_t* q, int64_t n, const float* s_w, uint16_t* wd, int sms,
                                  cudaStream_t st);

// Modulated LayerNorm of each [K] row, rounded to bf16 (h) and/or quantized
// to E4M3 with s_in (q); either output may be null, not both; 8 <= K <= 8192,
// K % 8 == 0; row m uses shift/scale row m / rows_per_sample.
// Reads and clears the elementwise kernels' device error word (synchronises `st`).
cudaError_t elementwise_read_error(cudaStream_t st, uint32_t* err);

cudaError_t launch_ln_modulate_quant(const uint16_t* x, int64_t M, int K, const uint16_t* shift,
                                     const uint16_t* scale, int64_t rows_per_sample, float eps,
                                     const float* s_in, uint8_t* q, uint16_t* h, int sms, cudaStream_t st);

struct SwigluExArgs {            // validated by the caller
  bool has_limit;
  float limit, alpha, beta;
};
cudaError_t launch_swiglu_ex(const uint16_t* g, const uint16_t* u, int64_t n, bool in_f16, bool out_fp8,
                             const SwigluExArgs& a, const float* s_out, void* out, int sms,
                             cudaStream_t st);

// ---- GEMMs (gemm.cu)
constexpr int kMaxGroup = 3;

struct GemmProblem {
  int64_t M, K;
  int G;                         // projections sharing the activation (1..3)
  const void* x;                 // E4M3 [M,K] (W8A8) or bf16 [M,K] (W8A16)
  const uint8_t* w[kMaxGroup];   // E4M3 [N_g, K]
  int64_t N[kMaxGroup];
  const float* s_in;             // W8A8 only
  const float* s_w[kMaxGroup];
  void* y[kMaxGroup];            // bf16 [M, N_g] (GLU: E4M3 [M, I])
  const float* s_out;            // GLU: input scale of the down projection
  const SwigluExArgs* ex;        // GLU / GLU16: SwiGLU options, or nullptr for the plain form
};

// Returns cudaSuccess or the CUDA error; *tmap_err is set non-zero when a
// tensor map could not be encoded.
cudaError_t launch_gemm_w8a8(const GemmProblem& p, int sms, cudaStream_t st, int* tmap_err);
cudaError_t launch_gemm_w8a16(const GemmProblem& p, int sms, cudaStream_t st, int* tmap_err);
// Gate/up W8A8 GEMMs with the SwiGLU-to-E4M3 epilogue: x E4M3 [M,K], w[0] gate
// and w[1] up [I,K] with s_w[0], s_w[1]; N[0] = I; y[0] E4M3 [M,I]; s_out.
// bf16 x bf16 GEMM of the W8A16 step on weights dequantized beforehand:
// y_g = bf16(x . Wd_g^T), x bf16 [M,K], Wd_g bf16 [N_g,K] in w[g] (s_w unused).
cudaError_t launch_gemm_bf16(const GemmProblem& p, int sms, cudaStream_t st, int* tmap_err);
// The gate/up pair of a 16-bit step on dequantized bf16 weights w[0] (gate)
// and w[1] (up), [I, K] each, with h = SwiGLU written as bf16 into y[0] [M, I].
cudaError_t launch_gemm_glu16(const GemmProblem& p, int sms, cudaStream_t st, int* tmap_err);
cudaError_t launch_gemm_glu(const GemmProblem& p, int sms, cudaStream_t st, int* tmap_err);

// Launches a one-thread kernel whose mbarrier wait times out (0.2 s).
cudaError_t launch_selftest_timeout(cudaStream_t st);

// Reads and clears the GEMM kernels' device error word (synchronises `st`).
cudaError_t gemm_read_error(cudaStream_t st, uint32_t* err);

// Thread-local error text shared with the C-ABI layer, and the device check
// (sm_103 and SM count of the current device) for entry points defined
// outside api.cu.
void set_last_error(const char* msg);
int query_device(int* sms);  // returns a w8_status

// Driver entry point for tensor-map encoding (resolved once).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn get_encode_tiled();

}  // namespace w8

/*
 * w8lin.h — C ABI of the static per-tensor FP8 linear layer for GB300 (sm_103a).
 *
 * Sources of the operations (web pages; cited by title and section):
 *  [P1] diffusers issue #15170, "Cosmos 3 docs: FP8 snippet fails at the first
 *       W8A8 step without importing ModelOpt's FP8 GEMM backend".
 *  [P2] cosmos-framework PR #157, "feat: load ModelOpt static-FP8 checkpoints
 *       via TorchAO".
 *  [P3] diffusers PR #14664, "[Cosmos3] Mixed W8A8/W8A16 denoising for
 *       ModelOpt FP8 checkpoints".
 *  [P4] TensorRT-LLM PR #17476, "Load static FP8 Cosmos3 Nano/Super
 *       checkpoints without re-quantizing them".
 *
 * Conventions shared by every entry point
 *  - Data pointers are DEVICE pointers owned by the caller; the library never
 *    allocates, frees or retains them.  Tensors are dense row-major:
 *    activations [M, K], weights [N, K] (the exported nn.Linear.weight),
 *    outputs [M, N].  There is no bias ([P1] Logs: bias=False).
 *  - bf16 values travel as uint16_t bit patterns, E4M3 codes as uint8_t
 *    (OCP E4M3 "fn": 4 exponent bits, bias 7, 3 mantissa bits, max 448).
 *  - Scales are `const float*` to ONE float in device memory, never read on
 *    the host: reading a scale on the hot path would synchronise the device
 *    ([P4] What changed: the shared-scale invariant is checked at load, never
 *    in forward).
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  Every compute
 *    entry point only enqueues work on it and returns; results are ready when
 *    the stream reaches that point.
 *  - Base pointers must be 16-byte aligned and K (and N for outputs) multiples
 *    of 16 (E4M3 rows) / 8 (bf16 rows) so that every row starts on a 16-byte
 *    boundary, as the tensor-memory-accelerator copies require.
 *  - M == 0 is a no-op that returns W8_OK without launching anything (zero-row
 *    inputs; [P2] Commits: the zero-row limitation it works around).
 *    Tensors of rank > 2 are flattened to [M, K] by the caller.
 *  - Arguments are validated on the host before any CUDA call; an invalid
 *    argument returns its error code and enqueues nothing.  Thread-local
 *    detail is available from w8_last_error().
 *  - Kernels never trap.  A GEMM whose internal pipeline wait runs past its
 *    deadline (2 s), or an ln_modulate_quant block whose row-buffer wait
 *    does, stops, records W8_ERR_TIMEOUT in a device error word and
 *    returns; w8_poll_device_error() reports and clears it.
 */
#ifndef W8LIN_H
#define W8LIN_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  W8_OK = 0,
  W8_ERR_NULL = 1,     /* a required pointer is NULL */
  W8_ERR_SHAPE = 2,    /* negative or unsupported size, or group size outside 1..3 */
  W8_ERR_ALIGN = 3,    /* a pointer or row pitch is not 16-byte aligned */
  W8_ERR_STRIDE = 4,   /* a row pitch differs from the row length (non-dense layout) */
  W8_ERR_DTYPE = 5,    /* activation dtype not accepted by this path */
  W8_ERR_ARCH = 6,     /* current device is not sm_103 */
  W8_ERR_POLICY = 7,   /* step policy refused (schema, window, step range) */
  W8_ERR_TIMEOUT = 8,  /* a kernel's bounded pipeline wait expired */
  W8_ERR_CUDA = 9,     /* a CUDA runtime/driver call failed */
  W8_ERR_SCALE = 10,   /* projections of a sharing group carry different input scales */
  W8_ERR_PARAM = 11    /* a scalar parameter is out of its range (not finite, limit <= 0) */
} w8_status;

typedef enum { W8_DTYPE_BF16 = 0, W8_DTYPE_E4M3 = 1, W8_DTYPE_F16 = 2 } w8_dtype;

/* Activation precision of one denoising step ([P3] Behavior). */
typedef enum { W8_MODE_A8 = 0, W8_MODE_A16 = 1 } w8_mode;

/* Per-denoising-step precision policy ([P4] Denoising-step activation
 * precision: quantization_config.runtime.diffusion_step_policy). */
typedef struct {
  int32_t schema_version; /* must be 1 */
  int32_t enabled;        /* 0 = the checkpoint carries no policy: every step W8A8 */
  int32_t first_steps;    /* leading steps run W8A16 (published policy: 3) */
  int32_t last_steps;     /* trailing steps run W8A16 (published policy: 3) */
} w8_step_policy;

/* Version of this ABI (bumped on any signature change). */
int w8_abi_version(void);

/* Thread-local text of the last error returned on this thread ("" if none). */
const char* w8_last_error(void);

/* W8_OK if the current CUDA device is an sm_103 part, else W8_ERR_ARCH. */
w8_status w8_device_check(void);

/* Synchronises `stream`, then returns W8_ERR_TIMEOUT (and clears the word)
 * if any GEMM launched so far on the current device recorded a pipeline
 * timeout, else W8_OK. */
w8_status w8_poll_device_error(void* stream);

/* Self-test of the failure path (no counterpart on the pages): enqueues a
 * one-thread kernel that waits on a pipeline barrier nothing arrives on; the
 * wait gives up after 0.2 s and records the same timeout bit a stalled GEMM
 * would, so that the next w8_poll_device_error() returns W8_ERR_TIMEOUT and
 * clears it.  The CUDA context stays usable.  Errors: ARCH, CUDA. */
w8_status w8_selftest_timeout(void* stream);

/*
 * fp8_quant_static — static per-tensor activation quantization.
 * q[i] = E4M3_satRNE( fl32( x[i] / s_in ) ) for all M*K elements: one
 * correctly rounded binary32 division, then one round-to-nearest-even to
 * E4M3 with saturation at +-448 ([P2] Verification: div -> clamp ->
 * round-to-float8 with the exported input_scale).  NaN inputs give a NaN code.
 *   x    bf16 [M, K], device, read-only; ldx = elements between row starts
 *   s_in float scalar, device
 *   q    E4M3 [M, K], device, written; ldq = bytes between row starts
 * Rows must be dense: ldx and ldq must both equal K.  A padded or strided
 * (non-contiguous) tensor is refused with W8_ERR_STRIDE rather than read or
 * written with the wrong pitch ([P4] Test Coverage: the op rejects
 * non-contiguous inputs).
 * Errors: SHAPE (M<0, K<=0, K%16), STRIDE (ldx != K or ldq != K), NULL,
 * ALIGN, ARCH, CUDA.
 */
w8_status fp8_quant_static(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, const float* s_in,
                           uint8_t* q, int64_t ldq, void* stream);

/*
 * fp8_linear_w8a8 — W8A8 FP8 linear.
 * y = bf16_RNE( fl32(s_in * s_w) * sum_k dec(qx[m,k]) * dec(w[n,k]) ), F32
 * accumulation on the tcgen05 tensor cores ([P2] Verification: _scaled_mm
 * with the two per-tensor scales; [P3] Behavior: native W8A8 on middle steps).
 *   x       activation [M, K]: bf16 if x_dtype == W8_DTYPE_BF16 (quantized
 *           first with s_in into `ws`), or E4M3 codes already quantized with
 *           s_in if x_dtype == W8_DTYPE_E4M3 (pass-through: [P4] What changed,
 *           a pre-quantized input goes straight to the GEMM)
 *   w       E4M3 weight [N, K]; s_in, s_w device float scalars
 *   y       bf16 output [M, N], written
 *   ws      E4M3 scratch [M, K], required iff x_dtype == W8_DTYPE_BF16,
 *           else ignored (may be NULL)
 * Errors: NULL, SHAPE (K%16, N%16), DTYPE, ALIGN, ARCH, CUDA.
 */
w8_status fp8_linear_w8a8(const void* x, int32_t x_dtype, int64_t M, int64_t K, const uint8_t* w,
                          int64_t N, const float* s_in, const float* s_w, uint16_t* y, uint8_t* ws,
                          void* stream);

/*
 * fp8_linear_w8a16 — W8A16 linear on the same E4M3 weight.
 * y = bf16_RNE( sum_k x[m,k] * Wd[n,k] ), Wd = bf16_RNE( fl32(dec(w) * s_w) );
 * input_scale is unused ([P3] Behavior: dequant + F.linear; [P4]
 * Denoising-step activation precision: same weights, same scales).
 *   x_dtype must be W8_DTYPE_BF16: an already-quantized activation is refused
 *   with W8_ERR_DTYPE ([P4] Denoising-step activation precision: the W8A16
 *   linear raises rather than accept an already-quantized activation).
 *   ws   optional bf16 scratch of N*K values (16-byte aligned), device.  With
 *        ws the weight is dequantized into it (a transient copy, overwritten
 *        by the next call that is given the same ws) and a bf16 tensor-core
 *        GEMM runs on it: the faster form.  With ws == NULL the dequantization
 *        happens inside the GEMM and nothing is written besides y.  Both forms
 *        use the same operand bits; they may differ in accumulation order only.
 * Errors: NULL, SHAPE (K%16, N%16), DTYPE, ALIGN, ARCH, CUDA.
 */
w8_status fp8_linear_w8a16(const void* x, int32_t x_dtype, int64_t M, int64_t K, const uint8_t* w,
                           int64_t N, const float* s_w, uint16_t* y, uint16_t* ws, void* stream);

/*
 * qkv_shared_quant_gemm — a group of G projections sharing one activation
 * (G = 3: split Q/K/V; G = 2: split gate/up), each with its own weight,
 * weight scale and contiguous output ([P4] Description and What changed:
 * projections stay split, the shared activation is quantized once and the
 * same FP8 tensor is handed to every projection).
 *   mode == W8_MODE_A8:  one fp8_quant_static of x into ws, then one
 *                        persistent W8A8 launch over the tiles of all G
 *                        projections, all reading ws.
 *   mode == W8_MODE_A16: no quantization (sharing stands down on 16-bit
 *                        steps, [P4] Denoising-step activation precision).
 *                        With ws: each weight is dequantized into ws
 *                        (Wd_g = bf16_RNE(fl32(dec(w_g) * s_w[g])), [P3]
 *                        Behavior: dequant + F.linear; a transient copy,
 *                        overwritten by the next call) and one bf16 GEMM
 *                        launch covers all G projections.  Without ws: one
 *                        launch that dequantizes inside the GEMM.  Both give
 *                        the same operand bits; they may differ in the
 *                        accumulation order only.
 *   x          bf16 [M, K], device
 *   s_in       device float scalar shared by the group (A8 only)
 *   w, N, s_w, y  HOST arrays of G entries: device weight [N_g, K], its row
 *              count, device weight scale, device output [M, N_g]
 *   ws         A8: E4M3 scratch [M, K], required.  A16: optional bf16
 *              scratch of sum_g N_g * K values (2 bytes each), the
 *              dequantized weights of the group in order; 16-byte aligned.
 * Errors: NULL, SHAPE (G outside 2..3 or 1, K%16, N_g%16), ALIGN, ARCH, CUDA.
 */
w8_status qkv_shared_quant_gemm(int32_t mode, const uint16_t* x, int64_t M, int64_t K,
                                const float* s_in, int32_t G, const uint8_t* const* w,
                                const int64_t* N, const float* const* s_w, uint16_t* const* y,
                                uint8_t* ws, void* stream);

/*
 * fp8_e4m3_from_f32 — the E4M3 encoding step on its own: q[i] =
 * E4M3_satRNE(x[i]) for binary32 x, the round-to-nearest-even to E4M3 with
 * saturation at +-448 that ends the static quantization ([P2] Verification:
 * div -> clamp -> round-to-float8) and every other code-producing kernel
 * here (the same hardware conversion).  Infinities saturate to +-448; NaN
 * gives a NaN code (0x7F or 0xFF); the sign of zero is kept.
 *   x   binary32 [n], device, 16-byte aligned
 *   q   E4M3 codes [n], device (written), 4-byte aligned
 * n == 0 launches nothing.
 * Errors: SHAPE (n < 0), NULL, ALIGN, ARCH, CUDA.
 */
w8_status fp8_e4m3_from_f32(const float* x, int64_t n, uint8_t* q, void* stream);

/*
 * fp8_dequant_weight — the dequantization step of the W8A16 path on its own
 * ([P3] Behavior: "dequant + F.linear"): Wd = bf16_RNE(fl32(dec(w) * s_w)).
 *   w    E4M3 weight [N, K], device;  s_w device float scalar
 *   wd   bf16 output [N, K], device (written)
 * Errors: NULL, SHAPE (K%16, negative sizes), ALIGN, ARCH, CUDA.
 */
w8_status fp8_dequant_weight(const uint8_t* w, int64_t N, int64_t K, const float* s_w, uint16_t* wd,
                             void* stream);

/*
 * bf16_linear_group — the "F.linear" half of the W8A16 path ([P3] Behavior:
 * dequant + F.linear) on weights already dequantized by fp8_dequant_weight:
 * G projections (1..3) of one bf16 activation in one launch,
 * y_g = bf16_RNE( x . Wd_g^T ) with fp32 accumulation.
 *   x    bf16 [M, K], device;  wd, N, y: HOST arrays of G entries: device
 *   bf16 weight [N_g, K], its row count, device bf16 output [M, N_g]
 * Errors: NULL, SHAPE (G outside 1..3, K%16, N_g%16), ALIGN, ARCH, CUDA.
 */
w8_status bf16_linear_group(const uint16_t* x, int64_t M, int64_t K, int32_t G, const uint16_t* const* wd,
                            const int64_t* N, uint16_t* const* y, void* stream);

/*
 * bf16_gate_up_swiglu — the gate/up pair of a 16-bit step with its SwiGLU,
 * on weights dequantized by fp8_dequant_weight, in one launch: out =
 * bf16_RNE(h) with h the SwiGLU of swiglu_2in_bf16 applied to g =
 * bf16_RNE(x . Wd_gate^T) and u = bf16_RNE(x . Wd_up^T) -- bit for bit the
 * result of bf16_linear_group followed by swiglu_2in_bf16, without writing
 * g and u ([P3] Behavior: dequant + F.linear; [P4] What changed: SiLU(G) * U
 * from the split gate and up projections).
 *   x        bf16 [M, K], device;  wd_gate, wd_up  bf16 [I, K], device
 *   out      bf16 [M, I], device
 * Errors: NULL, SHAPE (K%16, I%16), ALIGN, ARCH, CUDA.
 */
w8_status bf16_gate_up_swiglu(const uint16_t* x, int64_t M, int64_t K, const uint16_t* wd_gate,
                              const uint16_t* wd_up, int64_t I, uint16_t* out, void* stream);

/*
 * fp8_linear_w8a8_group — the GEMM half of qkv_shared_quant_gemm in A8 mode:
 * G projections (1..3) over an activation that is ALREADY E4M3, quantized
 * with s_in (for example by fp8_quant_static or swiglu_2in_fp8), in one
 * persistent launch.  y_g = bf16_RNE( fl32(s_in * s_w[g]) * qx . w_g^T ).
 *   qx   E4M3 [M, K], device;  w, N, s_w, y: HOST arrays of G entries as in
 *   qkv_shared_quant_gemm.
 * Errors: NULL, SHAPE, ALIGN, ARCH, CUDA.
 */
w8_status fp8_linear_w8a8_group(const uint8_t* qx, int64_t M, int64_t K, const float* s_in,
                                int32_t G, const uint8_t* const* w, const int64_t* N,
                                const float* const* s_w, uint16_t* const* y, void* stream);

/*
 * gate_up_swiglu_fp8 — the split gated MLP's gate and up projections and the
 * two-input SwiGLU in one pass, writing the down projection's E4M3 input:
 *   g = bf16_RNE( fl32(s_in * s_w_gate) * qx . w_gate^T )
 *   u = bf16_RNE( fl32(s_in * s_w_up)   * qx . w_up^T )
 *   out = swiglu_2in_fp8(g, u, s_out)   (same specification, same codes)
 * The gate and up accumulators live side by side in TMEM and never go to
 * global memory; each projection keeps its own weight scale ([P4] What
 * changed: split gate/up, one shared activation quantization, SiLU(G) * U
 * quantized directly for the FP8 down projection).
 *   x      activation [M, K]: bf16 if x_dtype == W8_DTYPE_BF16 (quantized
 *          first with s_in into `ws`), or E4M3 codes quantized with s_in
 *   w_gate, w_up  E4M3 [I, K];  s_in, s_w_gate, s_w_up, s_out device floats
 *   out    E4M3 [M, I], written;  ws E4M3 [M, K] scratch (bf16 input only)
 * Errors: NULL, SHAPE (K%16, I%16), DTYPE, ALIGN, ARCH, CUDA.
 */
w8_status gate_up_swiglu_fp8(const void* x, int32_t x_dtype, int64_t M, int64_t K,
                             const float* s_in, const uint8_t* w_gate, const uint8_t* w_up,
                             int64_t I, const float* s_w_gate, const float* s_w_up,
                             const float* s_out, uint8_t* out, uint8_t* ws, void* stream);

/*
 * fp8_linear_w8a8_noalloc — fp8_linear_w8a8 on a bf16 activation for callers
 * that cannot allocate device memory (the web pages have no counterpart: this
 * entry point exists for integration, not for the method).  Some callers can
 * neither allocate nor be handed a workspace: operator or plugin interfaces
 * that pass only inputs and outputs, runtimes whose memory belongs to a fixed
 * pool, or code that may not call cudaMalloc because it can synchronise the
 * device or because a stream capture is in progress.  The E4M3 copy of the
 * activation goes instead into a fixed 32 MiB device array inside the
 * library, so this call allocates nothing.
 *   x bf16 [M, K]; w E4M3 [N, K]; s_in, s_w device float scalars; y bf16 [M, N].
 *   Limit: M*K <= 33,554,432 (32 MiB of E4M3 codes); larger activations are
 *   refused with W8_ERR_SHAPE (use fp8_linear_w8a8 with a workspace).
 *   Every GPU that loads the library keeps the 32 MiB array until exit.
 *   The first call on a device looks up the array's device address (with
 *   that device current); make that first call before any stream capture.
 *   All calls on a device share the one array: calls that overlap on the GPU
 *   race; calls ordered on one stream do not.  Nothing in the array needs to
 *   start zeroed (every byte read was written by the same call).
 * Errors: NULL, SHAPE, ALIGN, ARCH, CUDA.
 */
w8_status fp8_linear_w8a8_noalloc(const uint16_t* x, int64_t M, int64_t K, const uint8_t* w,
                                  int64_t N, const float* s_in, const float* s_w, uint16_t* y,
                                  void* stream);

/*
 * swiglu_2in_fp8 — out = E4M3_satRNE( fl32( h / s_out ) ) with
 * h = fl32( fl32(g * u) / fl32(1 + exp_spec(-g)) ), SiLU(gate) * up from two
 * separate tensors written straight to FP8 for the down projection
 * ([P4] What changed: two-input SwiGLU quantizing directly for the FP8
 * down_proj).  exp_spec is the library's binary32 exponential (Cody-Waite
 * reduction, degree-7 Taylor polynomial; stated in the kernel source).
 *   gate, up  bf16 [M, I], device;  s_out device float scalar (the down
 *   projection's input_scale);  out E4M3 [M, I], device.
 * Errors: NULL, SHAPE (I%16), ALIGN, ARCH, CUDA.
 */
w8_status swiglu_2in_fp8(const uint16_t* gate, const uint16_t* up, int64_t M, int64_t I,
                         const float* s_out, uint8_t* out, void* stream);

/* swiglu_2in_bf16 — bf16_RNE(h) with h as above; the 16-bit-step variant in
 * which the FP8 output stands down ([P4] Denoising-step activation precision). */
w8_status swiglu_2in_bf16(const uint16_t* gate, const uint16_t* up, int64_t M, int64_t I,
                          uint16_t* out, void* stream);

/* Options of the two-input SwiGLU ([P4] Test Coverage: swiglu_limit,
 * swiglu_alpha + swiglu_beta).  The pages name the options and no formula; the
 * reading is the clamped, shifted SwiGLU of the public gpt-oss MLP:
 *   g = min(g, limit), u = clamp(u, -limit, limit)   (if has_limit)
 *   h = fl32( fl32(g * fl32(u + beta)) / fl32(1 + exp_spec(-fl32(alpha * g))) )
 * with the addition of beta skipped when beta == 0.  {0, 0, 1, 0} is the
 * plain SwiGLU of swiglu_2in_fp8 / swiglu_2in_bf16, bit for bit. */
typedef struct {
  int32_t has_limit; /* nonzero: apply `limit` */
  float limit;       /* finite, > 0 when has_limit */
  float alpha;       /* finite; 1 = plain SiLU */
  float beta;        /* finite; 0 = none */
} w8_swiglu_params;

/*
 * swiglu_2in_ex_fp8 — the SwiGLU with options and bf16 or binary16 inputs
 * ([P4] Test Coverage: BF16 / FP16 inputs, swiglu_limit, swiglu_alpha +
 * swiglu_beta, FP8 output), written as E4M3_satRNE(fl32(h / s_out)).
 *   gate, up   [M, I] of in_dtype (W8_DTYPE_BF16 or W8_DTYPE_F16), device;
 *   prm        host struct, read during the call only;
 *   s_out      device float scalar;  out E4M3 [M, I], device.
 * Errors: NULL, SHAPE (I%16), ALIGN, DTYPE, PARAM, ARCH, CUDA.
 */
w8_status swiglu_2in_ex_fp8(const void* gate, const void* up, int32_t in_dtype, int64_t M, int64_t I,
                            const w8_swiglu_params* prm, const float* s_out, uint8_t* out,
                            void* stream);

/* swiglu_2in_ex_16 — as swiglu_2in_ex_fp8 with a 16-bit output in the input's
 * format (bf16_RNE(h) or binary16_RNE(h), overflow to infinity): the
 * 16-bit-step form. */
w8_status swiglu_2in_ex_16(const void* gate, const void* up, int32_t in_dtype, int64_t M, int64_t I,
                           const w8_swiglu_params* prm, void* out, void* stream);

/*
 * gate_up_swiglu_ex_fp8 — gate_up_swiglu_fp8 with the SwiGLU options in its
 * epilogue ([P4] Test Coverage: swiglu_limit, swiglu_alpha + swiglu_beta).
 * The bf16 gate and up values are those of the separate projections (as in
 * gate_up_swiglu_fp8); the codes are swiglu_2in_ex_fp8's on them, bit for bit.
 *   prm   host struct, read during the call only; {0, 0, 1, 0} gives
 *         gate_up_swiglu_fp8's codes.
 * Other arguments, layouts and errors as gate_up_swiglu_fp8, plus PARAM.
 */
w8_status gate_up_swiglu_ex_fp8(const void* x, int32_t x_dtype, int64_t M, int64_t K,
                                const float* s_in, const uint8_t* w_gate, const uint8_t* w_up,
                                int64_t I, const float* s_w_gate, const float* s_w_up,
                                const w8_swiglu_params* prm, const float* s_out, uint8_t* out,
                                uint8_t* ws, void* stream);

/*
 * bf16_gate_up_swiglu_ex — bf16_gate_up_swiglu with the SwiGLU options: the
 * bf16 outputs are swiglu_2in_ex_16's (bf16 inputs) on the bf16 gate and up
 * values of the separate projections, bit for bit.  prm as above.
 * Other arguments, layouts and errors as bf16_gate_up_swiglu, plus PARAM.
 */
w8_status bf16_gate_up_swiglu_ex(const uint16_t* x, int64_t M, int64_t K, const uint16_t* wd_gate,
                                 const uint16_t* wd_up, int64_t I, const w8_swiglu_params* prm,
                                 uint16_t* out, void* stream);

/*
 * ln_modulate_quant — the producer of a linear layer's input with the static
 * quantization fused after it.  The pages place the quantization right after
 * the block's norm/modulation ([P2] Verification: div -> clamp ->
 * round-to-float8 on the activation) and give the norm no formula; this
 * entry takes the diffusion-transformer form: per row of x,
 *   n = (x - mean(x)) / sqrt(var(x) + eps)     (LayerNorm without affine,
 *                                              biased variance over K)
 *   h = bf16_RNE( n * (1 + scale[s]) + shift[s] ),   s = row / rows_per_sample
 *   q = E4M3_satRNE( fl32(h / s_in) )          (exactly fp8_quant_static of h)
 * Statistics in binary32: h equals the correctly rounded bf16 of the exact
 * value except where that value lies within the binary32 rounding error of
 * its terms (a few ulps of |n (1 + scale)| and |h|) of a bf16 rounding
 * boundary, where it may be another bf16 within that error.  q is always the
 * quantization of the h this call produces (written or not).
 *   x      bf16 [M, K], device, read-only; 8 <= K <= 8192, K % 8 == 0
 *   shift, scale  bf16 [M / rows_per_sample, K], device, read-only
 *   rows_per_sample  tokens per sample (>= 1, divides M)
 *   eps    LayerNorm epsilon, finite and >= 0 (eps = 0 on a constant row
 *          gives NaN, as the formula does)
 *   s_in   device float scalar; required iff q is given
 *   q      E4M3 [M, K], device, written; may be NULL (bf16 h only)
 *   h      bf16 [M, K], device, written; may be NULL (codes only)
 * All arrays 16-byte aligned.  M == 0 launches nothing.
 * Errors: NULL (x, shift, scale, both outputs, s_in with q), SHAPE, ALIGN,
 * PARAM (eps), ARCH, CUDA.
 */
w8_status ln_modulate_quant(const uint16_t* x, int64_t M, int64_t K, const uint16_t* shift,
                            const uint16_t* scale, int64_t rows_per_sample, float eps,
                            const float* s_in, uint8_t* q, uint16_t* h, void* stream);

/*
 * step_policy_dispatch — host-only, pure function of (policy, step, num_steps).
 * policy == NULL or enabled == 0: W8_MODE_A8 on every step (a checkpoint with
 * no policy runs fully quantized).  num_steps == 1: W8_MODE_A8 (the one-step
 * carve-out, [P3] Tests: 1-step stays native).  Otherwise W8_MODE_A16 iff
 * step < first_steps or step >= num_steps - last_steps ([P3] Behavior: first
 * 3 + last 3 steps W8A16).  Steps are zero-based.
 * Errors: NULL (mode_out), POLICY (schema_version != 1, negative window,
 * step outside [0, num_steps)) — refused rather than partially honoured
 * ([P4] Denoising-step activation precision).
 */
w8_status step_policy_dispatch(const w8_step_policy* policy, int32_t step, int32_t num_steps,
                               int32_t* mode_out);

/*
 * w8_step_policy_parse — host-only, fail-closed parse of a checkpoint's
 * quantization_config.runtime.diffusion_step_policy JSON text into a
 * w8_step_policy ([P4] Denoising-step activation precision: unknown or
 * missing fields, schema_version other than 1, and any other type,
 * index_space, default_mode or overlap value are refused rather than
 * partially honoured; overlap is validated, not acted on; [P3] Behavior:
 * "runtime: null" means no policy).
 *   json   NUL-terminated text: `null`, or an object with exactly the keys
 *          schema_version (1), type ("first_last_n"), index_space
 *          ("scheduler_step"), default_mode ("w8a8"), overlap ("w8a16"),
 *          first_steps and last_steps (integers >= 0), reasoner ("a16" or
 *          "a8").  The pages name the fields but not the value spellings;
 *          these spellings are this library's reading.
 *   policy_out        filled on success (`null` gives enabled = 0)
 *   reasoner_mode_out W8_MODE_A16 / W8_MODE_A8 as stated, -1 for `null`
 *                     (the reasoner is not step-gated; its precision is
 *                     stated by the policy)
 * Errors: NULL, POLICY (with the reason in w8_last_error()).
 */
w8_status w8_step_policy_parse(const char* json, w8_step_policy* policy_out,
                               int32_t* reasoner_mode_out);

/*
 * w8_check_group_scales — load-time check that the G projections of a
 * sharing group carry bit-identical input scales ([P4] What changed: the
 * invariant the sharing rests on, validated in post_load_weights(), never
 * in forward).  Reads the G device scalars and synchronises the device.
 *   s_in  HOST array of G device pointers.
 * Errors: NULL, SHAPE (G < 1), SCALE (scales differ), CUDA.
 */
w8_status w8_check_group_scales(const float* const* s_in, int32_t G);

#ifdef __cplusplus
}
#endif

#endif /* W8LIN_H */

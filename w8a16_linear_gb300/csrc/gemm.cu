// Persistent tcgen05 GEMMs of the static per-tensor FP8 linear layer.
//
//  W8A8  (kind::f8f6f4): y = bf16( s_in * s_w * sum_k qx[m,k] * qw[n,k] ),
//        E4M3 activations and weights, F32 accumulation in TMEM
//        (cosmos-framework PR #157, "feat: load ModelOpt static-FP8
//        checkpoints via TorchAO", section Verification: _scaled_mm on the
//        two per-tensor scales).  One launch serves a group of up to three
//        projections that share the same activation (split Q/K/V or gate/up,
//        each with its own weight and weight scale and its own contiguous
//        output; TensorRT-LLM PR #17476, "Load static FP8 Cosmos3 Nano/Super
//        checkpoints without re-quantizing them", sections Description and
//        What changed).
//  GLU   (kind::f8f6f4): the gate and up projections of a split gated MLP in
//        one pass, followed in the epilogue by the two-input SwiGLU written
//        straight to E4M3 for the down projection: out = E4M3(SwiGLU(g, u) /
//        s_out) with g = bf16(s_in s_wg acc_g), u = bf16(s_in s_wu acc_u) --
//        the same bf16 values the separate GEMMs would write, so the codes are
//        those of swiglu_2in_fp8 applied to them; each projection keeps its
//        own weight scale (TensorRT-LLM PR #17476, section What changed).
//  BF16  (kind::f16): the "F.linear" half of the W8A16 path, y = bf16( sum_k
//        x[m,k] * Wd[n,k] ) on a weight dequantized beforehand, Wd =
//        bf16( fl32(dec(qw) * s_w) ); the static input scale is not used
//        (TensorRT-LLM PR #17476, section Denoising-step activation precision;
//        diffusers PR #14664, "[Cosmos3] Mixed W8A8/W8A16 denoising for
//        ModelOpt FP8 checkpoints", section Behavior: dequant + F.linear).
//  GLU16 (kind::f16): the gate and up projections of a 16-bit step on
//        dequantized weights, with the SwiGLU written as bf16 -- the values
//        swiglu_2in_bf16 would produce from the bf16 outputs of BF16.
//  GLUX / GLU16X: GLU / GLU16 with the SwiGLU options (limit, alpha, beta;
//        TensorRT-LLM PR #17476, section Test Coverage) in the epilogue -- the
//        values swiglu_2in_ex_fp8 / swiglu_2in_ex_16 would produce from the
//        same bf16 gate and up.
//  W8A16 (kind::f16, gemm_a16t_kernel below): the same product with the
//        dequantized weight formed in TMEM inside the GEMM, for calls that
//        provide no workspace.
//
// W8A8 / GLU / BF16 / GLU16 (and GLUX / GLU16X) kernel shapes (template parameter CG):
//   CG = 1  one CTA per SM computes a 128-row output tile.
//   CG = 2  a cluster of two CTAs on two SMs computes a 256-row tile with
//           CTA-pair MMAs (tcgen05 cta_group::2): each CTA stages its 128
//           activation rows and half of the weight rows of the tile, the even
//           CTA issues the MMAs, each CTA's TMEM receives its 128 output rows.
//           Per SM this halves the weight bytes staged per FLOP.
//
// Roles (per CTA, one CTA per SM, static round-robin over output tiles):
//   warp 0      TMA producer: activation and weight tiles into a smem ring
//   warp 1      TMEM allocator; MMA issuer (one thread of the even CTA)
//   warps 2-5   epilogue, one warp per TMEM lane quadrant: TMEM -> registers
//               -> scale -> bf16 (or SwiGLU -> E4M3 / bf16) -> swizzled smem ->
//               TMA store; double-buffered TMEM accumulators let it overlap
//               the next tile's main loop
// Every mbarrier wait is bounded: on a timeout the kernel records an error
// bit, the other roles stop at their next wait, in-flight copies and MMAs
// are drained with bounded waits, TMEM is freed and the kernel returns.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include "internal.h"
#include "ptx.cuh"
#include "swiglu_spec.cuh"

namespace w8 {

__device__ uint32_t g_gemm_err;

namespace {

constexpr int BM = 128;                           // output rows per CTA
constexpr uint32_t kTmemCols = 512;               // two 256-column F32 accumulator buffers
constexpr uint32_t kAccCols = 256;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per wait
constexpr int kEpiBufBytes = 32 * 128;            // W8A8 staging: 32 rows x 64 bf16

enum class Mode { W8A8, GLU, BF16, GLU16, GLUX, GLU16X };

template <Mode MODE, int CG>
struct Cfg {
  // GLUX / GLU16X: GLU / GLU16 with the SwiGLU options (limit, alpha, beta)
  // in the epilogue; separate kernels, so that the plain forms keep theirs.
  static constexpr bool kEx = (MODE == Mode::GLUX || MODE == Mode::GLU16X);
  static constexpr bool kGlu = (MODE == Mode::GLU || MODE == Mode::GLU16 || kEx);
  // BF16: the W8A16 product on an already dequantized weight (bf16 x bf16,
  // kind::f16): the same tiles and pipeline (a 128-byte swizzle atom holds
  // 64 K-values instead of 128) and an unscaled epilogue.  GLU16: the gate/up pair of a 16-bit
  // step on dequantized weights, with the SwiGLU written as bf16.
  static constexpr bool kBf16 = (MODE == Mode::BF16 || MODE == Mode::GLU16 || MODE == Mode::GLU16X);
  static constexpr bool kOut16 = (MODE == Mode::GLU16 || MODE == Mode::GLU16X);
  // W8A8: 256 output columns per tile.  GLU: 128 intermediate columns per
  // tile, computed by one N = 256 MMA whose B operand is [128 gate rows | 128
  // up rows] of the slice: D columns 0-127 hold gate, 128-255 hold up, and
  // the activation operand is read once for both.  In the CTA pair the even
  // CTA stages the gate rows and the odd CTA the up rows.
  static constexpr int kBN = kGlu ? 128 : 256;              // output columns per tile
  static constexpr int kMmaN = 256;
  static constexpr int kBRows = kMmaN / CG;                 // weight rows staged per CTA
  // A stage holds kAtoms 128-byte-wide K slices ("atoms", the span of the
  // 128-byte swizzle) of each operand: more K per barrier round trip, fewer
  // and larger stages in the same shared memory.  Two atoms (256 bytes of K,
  // 8 MMAs per stage) measured 3-7% faster than one for W8A8, 14% for GLU,
  // 8% for GLU16 and the same for BF16.
  static constexpr int kAtoms = 2;
  static constexpr int kAtomK = kBf16 ? 64 : 128;           // K elements per atom
  static constexpr int kBK = kAtomK * kAtoms;               // K per stage
  static constexpr int kABytes = BM * 128 * kAtoms;
  static constexpr int kBBytes = kBRows * 128 * kAtoms;
  static constexpr int kStages = (CG == 1 ? 4 : 6) / kAtoms;
  static constexpr uint32_t kIdesc =                        // E4M3 x E4M3 or BF16 x BF16 -> F32
      kBf16 ? make_idesc(1, 1, BM * CG, kMmaN) : make_idesc(0, 0, BM * CG, kMmaN);
  // One epilogue warp per TMEM lane quadrant: more warps (each taking fewer
  // columns) measured slower for the SwiGLU epilogues, their instruction
  // issue competing with the producer and MMA threads.
  static constexpr int kEpiWarps = 4;
  // GLU staging per warp: 32 rows x 64 E4M3 codes (64 bytes) or, GLU16,
  // 32 rows x 64 bf16 (128 bytes), double-buffered.
  static constexpr int kEpiBuf = kOut16 ? 32 * 128 : (kGlu ? 32 * 64 : kEpiBufBytes);
  static constexpr int kEpiNBuf = 2;
  static constexpr int kEpiBytes = kEpiWarps * kEpiNBuf * kEpiBuf;
};

template <Mode MODE, int CG>
struct Layout {
  using C = Cfg<MODE, CG>;
  static constexpr int kA = 0;
  static constexpr int kB = kA + C::kStages * C::kABytes;
  static constexpr int kEpi = kB + C::kStages * C::kBBytes;
  static constexpr int kBar = kEpi + C::kEpiBytes;
  // barriers: full[S], empty[S], tfull[2], tempty[2], drain
  static constexpr int kNumBars = 2 * C::kStages + 5;
  static constexpr int kTmemSlot = kBar + kNumBars * 8;
  static constexpr int kAbort = kTmemSlot + 4;
  static constexpr int kEnd = kAbort + 4;
  static constexpr int kAlloc = kEnd + 1024;  // slack for 1024-byte alignment
  static constexpr int kThreads = (2 + C::kEpiWarps) * 32;
  static_assert(kAlloc <= 232448, "shared memory budget");
};

struct Maps {
  CUtensorMap a;
  CUtensorMap b[kMaxGroup];
  CUtensorMap y[kMaxGroup];
};

struct Args {
  int G;
  int M, K;
  int N[kMaxGroup];
  int tiles_n[kMaxGroup];
  int tiles_per_m;
  int tiles_m;
  int group_m;   // m-blocks swept together down each column of tiles
  int num_tiles;
  // Work units of gemm_kernel: tiles [0, num_full) whole, then each of the
  // num_tiles - num_full tail tiles cut into tail_split column slices (of
  // kBN / tail_split columns) that separate CTAs (pairs) compute, so that the
  // last, partly filled wave is short.  num_units = num_full + tail tiles x
  // tail_split.  Every output element is accumulated over the same k order
  // whichever way its tile is cut.
  int num_full;
  int tail_split;
  int num_units;
  int num_kb;
  const float* s_in;
  const float* s_w[kMaxGroup];
  const float* s_out;  // GLU: the down projection's input scale
  SwigluParams pr;     // GLUX / GLU16X: the SwiGLU options
  // L2 policies of the operand loads and the output stores (kL2Normal,
  // kL2Keep, kL2Stream), chosen per launch from what fits in L2
  int l2_a, l2_b, l2_y;
};

enum : int { kL2Normal = 0, kL2Keep = 1, kL2Stream = 2 };

__device__ __forceinline__ uint64_t l2_policy(int kind) {
  return kind == kL2Keep ? l2_policy_evict_last()
                         : (kind == kL2Stream ? l2_policy_evict_first() : l2_policy_evict_normal());
}

// Tile t -> first output row of the (cluster) tile, projection, first column.
// Tiles are rasterised in groups of `group_m` m-blocks: within a group the
// m-block varies fastest, then the column of tiles (projection, n-block), so
// the CTAs running at the same time share each weight tile through L2 and
// the group's activation rows stay L2-resident while it sweeps the columns.
__device__ __forceinline__ void decode_tile(const Args& a, int t, int rows_per_tile, int cols_per_tile,
                                            int& m0, int& g, int& n0) {
  const int per_group = a.group_m * a.tiles_per_m;
  const int grp = t / per_group;
  const int mb0 = grp * a.group_m;
  const int gm = min(a.group_m, a.tiles_m - mb0);
  const int rr = t - grp * per_group;
  int r = rr / gm;                       // column of tiles
  const int mb = mb0 + (rr - r * gm);
  g = 0;
  while (g < a.G - 1 && r >= a.tiles_n[g]) {
    r -= a.tiles_n[g];
    ++g;
  }
  m0 = mb * rows_per_tile;
  n0 = r * cols_per_tile;
}

// Work unit u -> its tile's first row, projection, first column, and width.
__device__ __forceinline__ void decode_unit(const Args& a, int u, int rows_per_tile, int cols_per_tile,
                                            int& m0, int& g, int& n0, int& width) {
  if (u < a.num_full) {
    decode_tile(a, u, rows_per_tile, cols_per_tile, m0, g, n0);
    width = cols_per_tile;
  } else {
    const int v = u - a.num_full;
    const int piece = v % a.tail_split;
    decode_tile(a, a.num_full + v / a.tail_split, rows_per_tile, cols_per_tile, m0, g, n0);
    width = cols_per_tile / a.tail_split;
    n0 += piece * width;
  }
}

__device__ __forceinline__ const CUtensorMap* map_b(const Maps& m, int g) {
  return g == 0 ? &m.b[0] : (g == 1 ? &m.b[1] : &m.b[2]);
}
__device__ __forceinline__ const CUtensorMap* map_y(const Maps& m, int g) {
  return g == 0 ? &m.y[0] : (g == 1 ? &m.y[1] : &m.y[2]);
}
__device__ __forceinline__ const float* scale_w(const Args& a, int g) {
  return g == 0 ? a.s_w[0] : (g == 1 ? a.s_w[1] : a.s_w[2]);
}

__device__ __forceinline__ void record_timeout(volatile int* abort) {
  *abort = 1;
  atomicOr(&g_gemm_err, kErrTimeout);
}

template <Mode MODE, int CG>
__global__ void __launch_bounds__(Layout<MODE, CG>::kThreads, 1)
    gemm_kernel(const __grid_constant__ Maps maps, const __grid_constant__ Args args) {
  using C = Cfg<MODE, CG>;
  using L = Layout<MODE, CG>;
  constexpr int S = C::kStages;
  constexpr bool kGlu = C::kGlu;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + L::kBar;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (S + s); };
  auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * S + b); };
  auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * S + 2 + b); };
  const uint32_t drain_bar = bar0 + 8u * (2 * S + 4);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + L::kAbort);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kTmemSlot);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = (CG == 2) ? cluster_ctarank() : 0u;
  const bool leader = (rank == 0);
  const int cluster_id = blockIdx.x / CG;
  const int num_clusters = gridDim.x / CG;
  // Barriers that live in the even CTA, as shared::cluster addresses.
  auto leader_addr = [&](uint32_t a) { return (CG == 2) ? mapa_shared(a, 0) : a; };

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), C::kEpiWarps * CG);
    }
    mbar_init(drain_bar, 1);
    *abort = 0;
    fence_mbar_init();
    prefetch_tensormap(&maps.a);
    for (int g = 0; g < (kGlu ? 2 : args.G); ++g) prefetch_tensormap(map_b(maps, g));
    for (int g = 0; g < args.G; ++g) prefetch_tensormap(map_y(maps, g));
  }
  if (warp == 1) {
    if constexpr (CG == 2) {
      tmem_alloc_pair(sbase + L::kTmemSlot, kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(sbase + L::kTmemSlot, kTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (CG == 2) cluster_sync();  // peer barriers initialised before any remote use
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // Everything above overlaps the previous kernel on the stream; from here
  // on every thread may read what it wrote (activations, scales) and write
  // what it may still read (outputs).
  griddep_wait();

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0;
      uint32_t issued = 0;
      bool ok = true;
      const uint64_t pol_a = l2_policy(args.l2_a);
      const uint64_t pol_b = l2_policy(args.l2_b);
      for (int t = cluster_id; ok && t < args.num_units; t += num_clusters) {
        int m0, g, n0, width;
        decode_unit(args, t, BM * CG, C::kBN, m0, g, n0, width);
        const int a_row = m0 + (int)rank * BM;
        // W8A8: this CTA's half (pair) or all of the unit's weight rows (a
        // tail slice uses the first width / CG rows of the box it loads).
        // GLU: the slice's rows n0 .. n0+127 of gate (even CTA / first half)
        // and of up (odd CTA / second half).
        const int b_row = kGlu ? n0 : n0 + (int)rank * (width / CG);
        for (int kb = 0; kb < args.num_kb; ++kb) {
          if (!mbar_wait(empty_bar(s), ph ^ 1, abort, kWaitLimitNs)) {
            record_timeout(abort);
            ok = false;
            break;
          }
          const uint32_t a_dst = sbase + L::kA + s * C::kABytes;
          const uint32_t b_dst = sbase + L::kB + s * C::kBBytes;
          const int kc = kb * C::kBK;
          if (leader) mbar_arrive_expect_tx(full_bar(s), CG * (C::kABytes + C::kBBytes));
          const uint32_t fb = leader_addr(full_bar(s));
          const CUtensorMap* mb0 = kGlu ? (rank == 0 ? &maps.b[0] : &maps.b[1]) : map_b(maps, g);
#pragma unroll
          for (int at = 0; at < C::kAtoms; ++at) {
            const uint32_t ad = a_dst + (uint32_t)(at * BM * 128);
            const uint32_t bd = b_dst + (uint32_t)(at * C::kBRows * 128);
            const int kx = kc + at * C::kAtomK;
            if constexpr (CG == 2) {
              tma_load_2d_pair_hint(ad, &maps.a, fb, kx, a_row, pol_a);
              tma_load_2d_pair_hint(bd, mb0, fb, kx, b_row, pol_b);
            } else {
              tma_load_2d_hint(ad, &maps.a, fb, kx, a_row, pol_a);
              tma_load_2d_hint(bd, mb0, fb, kx, b_row, pol_b);
              if constexpr (kGlu) tma_load_2d_hint(bd + 128 * 128, &maps.b[1], fb, kx, b_row, pol_b);
            }
          }
          ++issued;
          if (++s == S) {
            s = 0;
            ph ^= 1;
          }
        }
      }
      // Drain: every stage's most recent loads must have landed before exit.
      // (The odd CTA of a pair has no armed full barriers; its loads are
      // covered by the even CTA's MMA drain and the closing cluster sync.)
      if (leader) {
        for (int j = 0; j < S && (uint32_t)j < issued; ++j) {
          const uint32_t l = issued - 1 - j;
          volatile int never = 0;
          if (!mbar_wait(full_bar((int)(l % S)), (l / S) & 1, &never, kWaitLimitNs))
            atomicOr(&g_gemm_err, kErrTimeout);
        }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0 && leader) {
      int s = 0;
      uint32_t ph = 0;
      int acc = 0;
      uint32_t acc_ph = 0;
      bool ok = true;
      for (int t = cluster_id; ok && t < args.num_units; t += num_clusters) {
        // a tail slice of width w: an N = w MMA (its descriptor), else the tile's
        const int w = t < args.num_full ? C::kMmaN : C::kMmaN / args.tail_split;
        const uint32_t idesc = w == C::kMmaN ? C::kIdesc
                                             : (C::kBf16 ? make_idesc(1, 1, BM * CG, w) : make_idesc(0, 0, BM * CG, w));
        if (!mbar_wait(tempty_bar(acc), acc_ph ^ 1, abort, kWaitLimitNs)) {
          record_timeout(abort);
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(acc * kAccCols);
        for (int kb = 0; kb < args.num_kb; ++kb) {
          if (!mbar_wait(full_bar(s), ph, abort, kWaitLimitNs)) {
            record_timeout(abort);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = sbase + L::kA + s * C::kABytes;
          const uint32_t b_addr = sbase + L::kB + s * C::kBBytes;
#pragma unroll
          for (int k = 0; k < 4 * C::kAtoms; ++k) {  // MMAs of 32 bytes of K each, 4 per atom
            const uint64_t ad = sw128_kmajor_desc(a_addr + (k >> 2) * BM * 128 + 32 * (k & 3));
            const uint64_t bd = sw128_kmajor_desc(b_addr + (k >> 2) * C::kBRows * 128 + 32 * (k & 3));
            const uint32_t accum = (kb | k) != 0;
            if constexpr (C::kBf16) {  // K = 16 per MMA: 32 bytes, as for E4M3
              if constexpr (CG == 2) mma_f16_pair(d, ad, bd, idesc, accum);
              else mma_f16(d, ad, bd, idesc, accum);
            } else {
              if constexpr (CG == 2) mma_f8f6f4_pair(d, ad, bd, idesc, accum);
              else mma_f8f6f4(d, ad, bd, idesc, accum);
            }
          }
          if constexpr (CG == 2) mma_commit_pair_mc(empty_bar(s), 0x3);
          else mma_commit(empty_bar(s));
          if (++s == S) {
            s = 0;
            ph ^= 1;
          }
        }
        if (!ok) break;
        if constexpr (CG == 2) mma_commit_pair_mc(tfull_bar(acc), 0x3);
        else mma_commit(tfull_bar(acc));
        if (++acc == 2) {
          acc = 0;
          acc_ph ^= 1;
        }
      }
      // Drain: all MMAs issued by this thread complete before TMEM is freed.
      if constexpr (CG == 2) mma_commit_pair(drain_bar);
      else mma_commit(drain_bar);
      volatile int never = 0;
      if (!mbar_wait(drain_bar, 0, &never, kWaitLimitNs)) atomicOr(&g_gemm_err, kErrTimeout);
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    const int wq = warp & 3;              // TMEM lane quadrant this warp may access
    constexpr int EB = C::kEpiBuf;
    const uint32_t buf0 = sbase + L::kEpi + (uint32_t)((warp - 2) * C::kEpiNBuf * EB);
    uint8_t* buf0_ptr = smem + L::kEpi + (warp - 2) * C::kEpiNBuf * EB;
    int acc = 0;
    uint32_t acc_ph = 0;
    int nbuf = 0;
    float s_out = 1.0f, rs_out = 1.0f;
    bool exact_only = false;
    const uint64_t pol_y = l2_policy(args.l2_y);
    if constexpr (kGlu && !C::kOut16) {
      s_out = __ldg(args.s_out);
      rs_out = __frcp_rn(s_out);
      exact_only = !swiglu_fp8_scale_is_fast(s_out, rs_out);
    }
    for (int t = cluster_id; t < args.num_units; t += num_clusters) {
      int m0, g, n0, width;
      decode_unit(args, t, BM * CG, C::kBN, m0, g, n0, width);
      float alpha = 1.0f, alpha_u = 1.0f;
      // BF16: the scale is already in the dequantized weight; y = bf16(acc).
      if constexpr (!C::kBf16) alpha = __fmul_rn(__ldg(args.s_in), __ldg(scale_w(args, kGlu ? 0 : g)));
      if constexpr (kGlu && !C::kBf16) alpha_u = __fmul_rn(__ldg(args.s_in), __ldg(args.s_w[1]));
      // Warp-uniform wait: the TMEM loads below are .sync.aligned.
      if (!mbar_wait_warp(tfull_bar(acc), acc_ph, abort, kWaitLimitNs)) {
        if (lane == 0) record_timeout(abort);
        break;
      }
      tc_fence_after();
      const int row0 = m0 + (int)rank * BM + wq * 32;
      const int ng = args.N[g];
      const uint32_t tbase = tmem_base + ((uint32_t)(wq * 32) << 16) + (uint32_t)(acc * kAccCols);
      if constexpr (!kGlu) {
        const int chunks = width / 64;
#pragma unroll 1
        for (int c = 0; c < chunks; ++c) {
          uint32_t r0[32], r1[32];
          tmem_ld_32x32b_x32(tbase + c * 64, r0);
          tmem_ld_32x32b_x32(tbase + c * 64 + 32, r1);
          tmem_ld_wait();
          if (c == chunks - 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
              if constexpr (CG == 2) mbar_arrive_cluster(leader_addr(tempty_bar(acc)));
              else mbar_arrive(tempty_bar(acc));
            }
          }
          uint32_t packed[32];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            packed[j] = cvt_bf16x2(__fmul_rn(__uint_as_float(r0[2 * j]), alpha),
                                   __fmul_rn(__uint_as_float(r0[2 * j + 1]), alpha));
            packed[16 + j] = cvt_bf16x2(__fmul_rn(__uint_as_float(r1[2 * j]), alpha),
                                        __fmul_rn(__uint_as_float(r1[2 * j + 1]), alpha));
          }
          const int col0 = n0 + c * 64;
          if (col0 >= ng || row0 >= args.M) continue;  // nothing of this chunk is in range
          // The store issued two chunks ago from this buffer must have read it.
          if (lane == 0) tma_store_wait_read<1>();
          __syncwarp();
          uint8_t* bp = buf0_ptr + nbuf * EB + lane * 128;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int pj = j ^ (lane & 7);  // 128-byte swizzle within the 1024-byte atom
            *reinterpret_cast<uint4*>(bp + pj * 16) =
                make_uint4(packed[4 * j], packed[4 * j + 1], packed[4 * j + 2], packed[4 * j + 3]);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d_hint(map_y(maps, g), buf0 + nbuf * EB, col0, row0, pol_y);
            tma_store_commit();
          }
          nbuf ^= 1;
        }
      } else if constexpr (C::kOut16) {
        // 16-bit step: bf16 SwiGLU of the bf16-rounded gate / up values.  The
        // tile's 128 columns in two halves of 64 (two 32-column chunks each),
        // each staged as one 128-byte row per lane with the 128-byte swizzle
        // (16-byte chunk j at j ^ (row & 7)) and stored with one TMA store.
#pragma unroll 1
        for (int cp = 0; cp < 2; ++cp) {
          if (lane == 0) tma_store_wait_read<1>();
          __syncwarp();
          uint8_t* bp = buf0_ptr + nbuf * EB + lane * 128;
#pragma unroll 1
          for (int lc = 0; lc < 2; ++lc) {
            const int c = 2 * cp + lc;
            uint32_t rg[32], ru[32];
            tmem_ld_32x32b_x32(tbase + c * 32, rg);
            tmem_ld_32x32b_x32(tbase + C::kBN + c * 32, ru);
            tmem_ld_wait();
            if (c == 3) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) {
                if constexpr (CG == 2) mbar_arrive_cluster(leader_addr(tempty_bar(acc)));
                else mbar_arrive(tempty_bar(acc));
              }
            }
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              uint32_t hw[8];
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                const int e = 16 * hh + 2 * j;
                // the bf16 values the separate gate / up GEMMs would have written
                const uint32_t gw = cvt_bf16x2(__uint_as_float(rg[e]), __uint_as_float(rg[e + 1]));
                const uint32_t uw = cvt_bf16x2(__uint_as_float(ru[e]), __uint_as_float(ru[e + 1]));
                if constexpr (C::kEx) hw[j] = swiglu_ex_16_pair<false>(gw, uw, args.pr);
                else hw[j] = swiglu_bf16_pair(gw, uw);
              }
              const int j0 = 4 * lc + 2 * hh;
              *reinterpret_cast<uint4*>(bp + ((j0 ^ (lane & 7)) * 16)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
              *reinterpret_cast<uint4*>(bp + (((j0 + 1) ^ (lane & 7)) * 16)) =
                  make_uint4(hw[4], hw[5], hw[6], hw[7]);
            }
          }
          fence_proxy_async_smem();
          __syncwarp();
          const int col0 = n0 + cp * 64;
          if (lane == 0 && col0 < ng && row0 < args.M) {
            tma_store_2d_hint(map_y(maps, 0), buf0 + nbuf * EB, col0, row0, pol_y);
            tma_store_commit();
          }
          nbuf ^= 1;
        }
      } else {
        // 128 intermediate columns per tile: gate at tbase, up at tbase + 128,
        // in two halves of 64 columns (two 32-column chunks of 32 E4M3 codes
        // each), each staged as one 64-byte row per lane with the 64-byte
        // swizzle (16-byte chunk j at j ^ ((row >> 1) & 3)) and stored with
        // one TMA store.
#pragma unroll 1
        for (int cp = 0; cp < 2; ++cp) {
          if (lane == 0) tma_store_wait_read<1>();
          __syncwarp();
          uint8_t* bp = buf0_ptr + nbuf * EB + lane * 64;
          const int sw = (lane >> 1) & 3;
#pragma unroll 1
          for (int lc = 0; lc < 2; ++lc) {
            const int c = 2 * cp + lc;
            uint32_t rg[32], ru[32];
            tmem_ld_32x32b_x32(tbase + c * 32, rg);
            tmem_ld_32x32b_x32(tbase + C::kBN + c * 32, ru);
            tmem_ld_wait();
            if (c == 3) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) {
                if constexpr (CG == 2) mbar_arrive_cluster(leader_addr(tempty_bar(acc)));
                else mbar_arrive(tempty_bar(acc));
              }
            }
            uint32_t codes[8];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              // the bf16 values the separate gate / up GEMMs would have written
              uint32_t gw[8], uw[8];
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                const int e = 16 * hh + 2 * j;
                gw[j] = cvt_bf16x2(__fmul_rn(__uint_as_float(rg[e]), alpha),
                                   __fmul_rn(__uint_as_float(rg[e + 1]), alpha));
                uw[j] = cvt_bf16x2(__fmul_rn(__uint_as_float(ru[e]), alpha_u),
                                   __fmul_rn(__uint_as_float(ru[e + 1]), alpha_u));
              }
              uint32_t c4[4];
              if constexpr (C::kEx) {   // the options' specification, 8 pairs at a time
                swiglu_ex_fp8_x16<false>(gw, uw, args.pr, s_out, rs_out, exact_only, c4);
              } else {
                swiglu_fp8_x16(gw, uw, s_out, rs_out, exact_only, c4);
              }
#pragma unroll
              for (int j = 0; j < 4; ++j) codes[4 * hh + j] = c4[j];
            }
            *reinterpret_cast<uint4*>(bp + (((2 * lc) ^ sw) * 16)) =
                make_uint4(codes[0], codes[1], codes[2], codes[3]);
            *reinterpret_cast<uint4*>(bp + (((2 * lc + 1) ^ sw) * 16)) =
                make_uint4(codes[4], codes[5], codes[6], codes[7]);
          }
          fence_proxy_async_smem();
          __syncwarp();
          const int col0 = n0 + cp * 64;
          if (lane == 0 && col0 < ng && row0 < args.M) {
            tma_store_2d_hint(map_y(maps, 0), buf0 + nbuf * EB, col0, row0, pol_y);
            tma_store_commit();
          }
          nbuf ^= 1;
        }
      }
      if (++acc == 2) {
        acc = 0;
        acc_ph ^= 1;
      }
    }
    if (lane == 0) tma_store_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  // A pair leaves together: no remote arrive or MMA may target an exited CTA.
  if constexpr (CG == 2) cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    if constexpr (CG == 2) tmem_dealloc_pair(tmem_base, kTmemCols);
    else tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ------------------------------------------------------------------ W8A16, weights in TMEM
//
// The W8A16 product computed transposed, D[n, m] = sum_k Wd[n, k] * x[m, k]:
// the dequantized weight is the MMA's A operand and lives in TMEM, written
// there by the transform warps with tcgen05.st (it never passes through
// shared memory); the activation tile is the B operand, staged by TMA into a
// 128-byte-swizzled K-major shared-memory buffer.  A tile is 128 weight rows
// x 320 tokens, computed as two N = 160 MMAs that share each dequantized
// weight stage, so every weight element is converted once per 320 tokens.
// D has the weight rows across the TMEM lanes and the tokens across columns;
// the epilogue turns each 32-token x 32-feature block into row-major y
// through a small staging buffer and a TMA store.
//
// TMEM columns: D (tokens 0-159) 0-159, D (tokens 160-319) 160-319, A stages
// 320 + 32 s (64 K-values of 128 rows, two bf16 per column).
namespace a16t {
constexpr int NH = 160;                      // tokens per MMA (MMA N)
constexpr int BT = 2 * NH;                   // tokens per tile
constexpr int BW = 128;                      // weight rows per tile (MMA M)
constexpr int BK = 64;                       // K per stage
constexpr int S = 4;                         // stages
constexpr int kXHalf = NH * 128;             // bf16 activation rows of one MMA, 128-byte rows
constexpr int kXBytes = 2 * kXHalf;
constexpr int kRawBytes = BW * 64;           // raw E4M3 weight rows
constexpr int kEpiBuf = 32 * 64;             // 32 tokens x 32 features bf16
constexpr int kEpiWarps = 8;                 // 2 per TMEM lane quadrant, 6 token chunks each
constexpr int kOffX = 0;
constexpr int kOffRaw = kOffX + S * kXBytes;
constexpr int kOffEpi = kOffRaw + S * kRawBytes;
constexpr int kOffBar = kOffEpi + kEpiWarps * 2 * kEpiBuf;
constexpr int kNumBars = 3 * S + 3;          // full[S], empty[S], ready[S], tfull, tempty, drain
constexpr int kOffTmemSlot = kOffBar + kNumBars * 8;
constexpr int kOffAbort = kOffTmemSlot + 4;
constexpr int kAlloc = kOffAbort + 4 + 1024;
constexpr int kTransformWarps = 8;           // 2 per TMEM lane quadrant, 32 K-values each
constexpr int kThreads = (2 + kEpiWarps + kTransformWarps) * 32;
constexpr uint32_t kTmemA = 2 * NH;          // first A-stage column
constexpr uint32_t kIdesc = make_idesc(1, 1, BW, NH);
static_assert(kTmemA + S * 32 <= kTmemCols, "TMEM budget");
static_assert(kAlloc <= 232448, "shared memory budget");
}  // namespace a16t

__global__ void __launch_bounds__(a16t::kThreads, 1)
    gemm_a16t_kernel(const __grid_constant__ Maps maps, const __grid_constant__ Args args) {
  using namespace a16t;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + kOffBar;
  auto full_bar = [&](int st) { return bar0 + 8u * st; };
  auto empty_bar = [&](int st) { return bar0 + 8u * (S + st); };
  auto ready_bar = [&](int st) { return bar0 + 8u * (2 * S + st); };
  const uint32_t tfull_bar = bar0 + 8u * (3 * S);
  const uint32_t tempty_bar = bar0 + 8u * (3 * S + 1);
  const uint32_t drain_bar = bar0 + 8u * (3 * S + 2);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + kOffAbort);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffTmemSlot);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int st = 0; st < S; ++st) {
      mbar_init(full_bar(st), 1);
      mbar_init(empty_bar(st), 1);
      mbar_init(ready_bar(st), kTransformWarps);
    }
    mbar_init(tfull_bar, 1);
    mbar_init(tempty_bar, kEpiWarps);
    mbar_init(drain_bar, 1);
    *abort = 0;
    fence_mbar_init();
    prefetch_tensormap(&maps.a);
    for (int g = 0; g < args.G; ++g) {
      prefetch_tensormap(map_b(maps, g));
      prefetch_tensormap(map_y(maps, g));
    }
  }
  if (warp == 1) {
    tmem_alloc(sbase + kOffTmemSlot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      int st = 0;
      uint32_t ph = 0, issued = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < args.num_tiles; t += gridDim.x) {
        int m0, g, n0;
        decode_tile(args, t, BT, BW, m0, g, n0);
        for (int kb = 0; kb < args.num_kb; ++kb) {
          if (!mbar_wait(empty_bar(st), ph ^ 1, abort, kWaitLimitNs)) {
            record_timeout(abort);
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(full_bar(st), kXBytes + kRawBytes);
          const uint32_t xd = sbase + kOffX + st * kXBytes;
          tma_load_2d(xd, &maps.a, full_bar(st), kb * BK, m0);
          tma_load_2d(xd + kXHalf, &maps.a, full_bar(st), kb * BK, m0 + NH);
          tma_load_2d(sbase + kOffRaw + st * kRawBytes, map_b(maps, g), full_bar(st), kb * BK, n0);
          ++issued;
          if (++st == S) {
            st = 0;
            ph ^= 1;
          }
        }
      }
      for (int j = 0; j < S && (uint32_t)j < issued; ++j) {
        const uint32_t l = issued - 1 - j;
        volatile int never = 0;
        if (!mbar_wait(full_bar((int)(l % S)), (l / S) & 1, &never, kWaitLimitNs))
          atomicOr(&g_gemm_err, kErrTimeout);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int st = 0;
      uint32_t ph = 0, acc_ph = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < args.num_tiles; t += gridDim.x) {
        if (!mbar_wait(tempty_bar, acc_ph ^ 1, abort, kWaitLimitNs)) {
          record_timeout(abort);
          break;
        }
        tc_fence_after();
        for (int kb = 0; kb < args.num_kb; ++kb) {
          if (!mbar_wait(ready_bar(st), ph, abort, kWaitLimitNs)) {
            record_timeout(abort);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t x_addr = sbase + kOffX + st * kXBytes;
          const uint32_t a_col = tmem_base + kTmemA + (uint32_t)(st * 32);
#pragma unroll
          for (int k = 0; k < 4; ++k) {  // K = 16 per MMA: 8 TMEM columns, 32 smem bytes
#pragma unroll
            for (int h = 0; h < 2; ++h)
              mma_f16_tmem_a(tmem_base + (uint32_t)(h * NH), a_col + 8 * k,
                             sw128_kmajor_desc(x_addr + h * kXHalf + 32 * k), kIdesc, (kb | k) != 0);
          }
          mma_commit(empty_bar(st));
          if (++st == S) {
            st = 0;
            ph ^= 1;
          }
        }
        if (!ok) break;
        mma_commit(tfull_bar);
        acc_ph ^= 1;
      }
      mma_commit(drain_bar);
      volatile int never = 0;
      if (!mbar_wait(drain_bar, 0, &never, kWaitLimitNs)) atomicOr(&g_gemm_err, kErrTimeout);
    }
  } else if (warp < 2 + kEpiWarps) {
    // ---------------------------------------------------------------- epilogue
    const int q = warp & 3;  // TMEM lane quadrant: weight rows (features) q*32 .. q*32+31
    const int eh = (warp - 2) >> 2;  // which half of the tile's 384 tokens
    uint8_t* bufp = smem + kOffEpi + (warp - 2) * 2 * kEpiBuf;
    const uint32_t bufs = sbase + kOffEpi + (uint32_t)((warp - 2) * 2 * kEpiBuf);
    int nbuf = 0;
    uint32_t acc_ph = 0;
    for (int t = blockIdx.x; t < args.num_tiles; t += gridDim.x) {
      int m0, g, n0;
      decode_tile(args, t, BT, BW, m0, g, n0);
      if (!mbar_wait_warp(tfull_bar, acc_ph, abort, kWaitLimitNs)) {
        if (lane == 0) record_timeout(abort);
        break;
      }
      tc_fence_after();
      const int f0 = n0 + q * 32;
      const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16);
#pragma unroll 1
      for (int c = eh * (NH / 32); c < (eh + 1) * (NH / 32); ++c) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(tbase + c * 32, r);  // feature f0+lane, tokens m0+c*32 .. +31
        tmem_ld_wait();
        if (c == (eh + 1) * (NH / 32) - 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(tempty_bar);
        }
        const int tok0 = m0 + c * 32;
        if (tok0 >= args.M || f0 >= args.N[g]) continue;
        if (lane == 0) tma_store_wait_read<1>();
        __syncwarp();
        uint16_t* bp = reinterpret_cast<uint16_t*>(bufp + nbuf * kEpiBuf);
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          const uint32_t pk = cvt_bf16x2(__uint_as_float(r[j]), __uint_as_float(r[j + 1]));
          bp[j * 32 + lane] = (uint16_t)(pk & 0xFFFF);        // token j, feature lane
          bp[(j + 1) * 32 + lane] = (uint16_t)(pk >> 16);     // token j+1
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(map_y(maps, g), bufs + nbuf * kEpiBuf, f0, tok0);
          tma_store_commit();
        }
        nbuf ^= 1;
      }
      acc_ph ^= 1;
    }
    if (lane == 0) tma_store_wait_all();
  } else {
    // ---------------------------------------------------------------- weight transform
    const int q = warp & 3;              // TMEM lane quadrant of this warp
    const int h = (warp - 2 - kEpiWarps) >> 2;  // which 32 of the stage's 64 K-values
    const int r = q * 32 + lane;         // weight row of the tile = TMEM lane
    int st = 0;
    uint32_t ph = 0;
    bool ok = true;
    for (int t = blockIdx.x; ok && t < args.num_tiles; t += gridDim.x) {
      int m0, g, n0;
      decode_tile(args, t, BT, BW, m0, g, n0);
      const float sw = __ldg(scale_w(args, g));
      for (int kb = 0; kb < args.num_kb; ++kb) {
        if (!mbar_wait_warp(full_bar(st), ph, abort, kWaitLimitNs)) {
          if (lane == 0) record_timeout(abort);
          ok = false;
          break;
        }
        // Raw row: 64 bytes with the 64-byte swizzle (chunk j at j ^ ((r >> 1) & 3)).
        const uint8_t* raw = smem + kOffRaw + st * kRawBytes + r * 64;
        const uint4 v0 = *reinterpret_cast<const uint4*>(raw + (((2 * h) ^ ((r >> 1) & 3)) * 16));
        const uint4 v1 = *reinterpret_cast<const uint4*>(raw + (((2 * h + 1) ^ ((r >> 1) & 3)) * 16));
        const uint32_t w8[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
        uint32_t o[16];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const uint32_t f01 = cvt_e4m3x2_to_f16x2((uint16_t)(w8[e] & 0xFFFF));
          const uint32_t f23 = cvt_e4m3x2_to_f16x2((uint16_t)(w8[e] >> 16));
          const F2 lo = mul2(F2{__half2float(__ushort_as_half((unsigned short)(f01 & 0xFFFF))),
                                __half2float(__ushort_as_half((unsigned short)(f01 >> 16)))},
                             splat(sw));
          const F2 hi = mul2(F2{__half2float(__ushort_as_half((unsigned short)(f23 & 0xFFFF))),
                                __half2float(__ushort_as_half((unsigned short)(f23 >> 16)))},
                             splat(sw));
          o[2 * e] = cvt_bf16x2(lo.x, lo.y);
          o[2 * e + 1] = cvt_bf16x2(hi.x, hi.y);
        }
        tmem_st_32x32b_x16(tmem_base + ((uint32_t)(q * 32) << 16) + kTmemA + (uint32_t)(st * 32 + h * 16), o);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(ready_bar(st));
        if (++st == S) {
          st = 0;
          ph ^= 1;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ------------------------------------------------------------------ host side

// m-blocks per rasterisation group: as many as keep the group's activation
// rows within ~32 MB of L2, between 1 and 16.
int group_rows(int rows_per_tile, int64_t K, int elem_bytes, int tiles_m) {
  const int64_t per_block = (int64_t)rows_per_tile * K * elem_bytes;
  int gm = (int)((32ll << 20) / (per_block > 0 ? per_block : 1));
  gm = gm < 1 ? 1 : (gm > 16 ? 16 : gm);
  return gm < tiles_m ? gm : tiles_m;
}

// What a launch asks L2 to keep.  The outputs are written once and never
// read back by the launch: streamed.  When all weights and a group of
// activation rows fit in kL2KeepBytes (of the 129 MB L2; the rest holds the
// output stream and the tiles in flight), both are kept -- the group made
// smaller if that makes them fit.  Otherwise the group's rows are kept and
// the weights streamed, with groups of up to kL2GroupBytes of rows, split
// evenly, so that the weights are swept as few times as possible (once per
// group).  The policies are hints: each die's L2 slice keeps its own copy of
// lines that SMs on both dies read, and the measured DRAM reads stay at
// 1.3-3.8x the operands' bytes (the plan measured fastest of those tried).
constexpr int64_t kL2KeepBytes = 96ll << 20;
constexpr int64_t kL2GroupBytes = 48ll << 20;

void l2_plan(int64_t w_bytes, int64_t a_block_bytes, int tiles_m, Args& a) {
  int gm = a.group_m;
  a.l2_y = kL2Stream;
  if (w_bytes + gm * a_block_bytes <= kL2KeepBytes) {
    a.l2_a = a.l2_b = kL2Keep;
  } else if (kL2KeepBytes - w_bytes >= 2 * a_block_bytes) {
    gm = (int)((kL2KeepBytes - w_bytes) / a_block_bytes);
    a.l2_a = a.l2_b = kL2Keep;
  } else {
    int gmax = (int)(kL2GroupBytes / a_block_bytes);
    gmax = gmax < 1 ? 1 : gmax;
    const int ngroups = (tiles_m + gmax - 1) / gmax;
    gm = (tiles_m + ngroups - 1) / ngroups;
    a.l2_a = kL2Keep;
    a.l2_b = kL2Stream;
  }
  a.group_m = gm < tiles_m ? gm : tiles_m;
}

bool encode_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner,
               uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
               CUtensorMapSwizzle sw) {
  EncodeTiledFn fn = get_encode_tiled();
  if (!fn) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

cudaError_t launch_cluster(void (*kern)(Maps, Args), int grid, int threads, int smem, int cg,
                           cudaStream_t st, const Maps& maps, const Args& args) {
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cg;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // The prologue (barriers, TMEM allocation, tensor-map prefetch) may run
  // while the previous kernel finishes; the kernel waits for it before
  // touching global memory.
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  e = cudaLaunchKernelEx(&cfg, kern, maps, args);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <Mode MODE, int CG>
cudaError_t launch(const GemmProblem& p, int sms, cudaStream_t st, int* tmap_err) {
  using C = Cfg<MODE, CG>;
  using L = Layout<MODE, CG>;
  constexpr bool kGlu = C::kGlu;
  *tmap_err = 0;
  Maps maps;
  Args args;
  std::memset(&maps, 0, sizeof(maps));
  std::memset(&args, 0, sizeof(args));
  args.G = kGlu ? 1 : p.G;
  args.M = (int)p.M;
  args.K = (int)p.K;
  args.num_kb = (int)((p.K + C::kBK - 1) / C::kBK);
  args.s_in = p.s_in;
  args.s_out = p.s_out;
  if (C::kEx)
    args.pr = SwigluParams{p.ex->limit, p.ex->alpha, p.ex->beta, p.ex->has_limit ? 1 : 0,
                           p.ex->beta != 0.0f ? 1 : 0};
  const int tiles_m = (int)((p.M + BM * CG - 1) / (BM * CG));
  constexpr int kEl = C::kBf16 ? 2 : 1;  // operand element bytes
  const CUtensorMapDataType dt = C::kBf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  bool ok = encode_2d(&maps.a, dt, p.x, p.K, p.M, p.K * kEl, C::kAtomK, BM, CU_TENSOR_MAP_SWIZZLE_128B);
  const int nb = kGlu ? 2 : p.G;  // weight maps: GLU gate and up
  for (int g = 0; g < nb; ++g) {
    args.s_w[g] = p.s_w[g];
    ok &= encode_2d(&maps.b[g], dt, p.w[g], p.K, p.N[kGlu ? 0 : g], p.K * kEl, C::kAtomK,
                    kGlu ? 128 : C::kBRows, CU_TENSOR_MAP_SWIZZLE_128B);
  }
  for (int g = 0; g < args.G; ++g) {
    args.N[g] = (int)p.N[g];
    args.tiles_n[g] = (int)((p.N[g] + C::kBN - 1) / C::kBN);
    args.tiles_per_m += args.tiles_n[g];
    if (kGlu && !C::kOut16)  // E4M3 output [M, I]: 32 rows x 64 codes per epilogue warp
      ok &= encode_2d(&maps.y[g], CU_TENSOR_MAP_DATA_TYPE_UINT8, p.y[g], p.N[g], p.M, p.N[g], 64,
                      32, CU_TENSOR_MAP_SWIZZLE_64B);
    else
      ok &= encode_2d(&maps.y[g], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.y[g], p.N[g], p.M, p.N[g] * 2,
                      64, 32, CU_TENSOR_MAP_SWIZZLE_128B);
  }
  for (int g = nb; g < kMaxGroup; ++g) args.s_w[g] = p.s_w[0];
  if (!ok) {
    *tmap_err = 1;
    return cudaSuccess;
  }
  args.num_tiles = tiles_m * args.tiles_per_m;
  args.tiles_m = tiles_m;
  args.group_m = group_rows(BM * CG, p.K, kEl, tiles_m);
  int64_t w_bytes = 0;
  for (int g = 0; g < nb; ++g) w_bytes += p.N[kGlu ? 0 : g] * p.K * kEl;
  l2_plan(w_bytes, (int64_t)BM * CG * p.K * kEl, tiles_m, args);
  const int max_clusters = sms / CG;
  const int clusters = args.num_tiles < max_clusters ? args.num_tiles : max_clusters;
  // The last wave's tiles, if they fill at most half of the clusters, are
  // cut in two column slices (not GLU, whose tile columns pair gate with up;
  // not single CTAs).  A slice is an N = 128 MMA, which does half a tile's
  // work in about 0.8 of its time; N = 64 quarter slices took almost a whole
  // tile's time, so cutting in four measured slower than in two (the Q/K/V
  // group at M = 20670: 555 against 549-551 us) and is not used.
  const int tail = args.num_tiles % clusters;
  args.tail_split = 1;
  if (!kGlu && CG == 2 && tail > 0 && 2 * tail <= clusters) args.tail_split = 2;
  args.num_full = args.num_tiles - (args.tail_split > 1 ? tail : 0);
  args.num_units = args.num_full + (args.num_tiles - args.num_full) * args.tail_split;
  return launch_cluster(gemm_kernel<MODE, CG>, clusters * CG, L::kThreads, L::kAlloc, CG, st, maps,
                        args);
}

// The CTA pair needs M above one 128-row tile to pay off.
bool use_pair(const GemmProblem& p) { return p.M > BM; }

cudaError_t launch_a16t(const GemmProblem& p, int sms, cudaStream_t st, int* tmap_err) {
  using namespace a16t;
  *tmap_err = 0;
  Maps maps;
  Args args;
  std::memset(&maps, 0, sizeof(maps));
  std::memset(&args, 0, sizeof(args));
  args.G = p.G;
  args.M = (int)p.M;
  args.K = (int)p.K;
  args.num_kb = (int)((p.K + BK - 1) / BK);
  const int tiles_m = (int)((p.M + BT - 1) / BT);
  bool ok = encode_2d(&maps.a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.x, p.K, p.M, p.K * 2, 64, NH,
                      CU_TENSOR_MAP_SWIZZLE_128B);
  for (int g = 0; g < p.G; ++g) {
    args.N[g] = (int)p.N[g];
    args.s_w[g] = p.s_w[g];
    args.tiles_n[g] = (int)((p.N[g] + BW - 1) / BW);
    args.tiles_per_m += args.tiles_n[g];
    ok &= encode_2d(&maps.b[g], CU_TENSOR_MAP_DATA_TYPE_UINT8, p.w[g], p.K, p.N[g], p.K, 64, BW,
                    CU_TENSOR_MAP_SWIZZLE_64B);
    ok &= encode_2d(&maps.y[g], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.y[g], p.N[g], p.M, p.N[g] * 2,
                    32, 32, CU_TENSOR_MAP_SWIZZLE_NONE);
  }
  for (int g = p.G; g < kMaxGroup; ++g) args.s_w[g] = p.s_w[0];
  if (!ok) {
    *tmap_err = 1;
    return cudaSuccess;
  }
  args.num_tiles = tiles_m * args.tiles_per_m;
  args.num_full = args.num_units = args.num_tiles;
  args.tail_split = 1;
  args.tiles_m = tiles_m;
  args.group_m = group_rows(BT, p.K, 2, tiles_m);
  const int grid = args.num_tiles < sms ? args.num_tiles : sms;
  cudaError_t e =
      cudaFuncSetAttribute(gemm_a16t_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kAlloc);
  if (e != cudaSuccess) return e;
  gemm_a16t_kernel<<<grid, kThreads, kAlloc, st>>>(maps, args);
  return cudaGetLastError();
}

// Self-test of the bounded wait: one thread waits on an mbarrier that nothing
// arrives on, gives up after `limit_ns` and records the timeout bit exactly as
// the GEMM roles do.  No other memory is touched.
__global__ void selftest_timeout_kernel(uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    volatile int* ab = &abort_flag;
    if (!mbar_wait(smem_u32(&bar), 0, ab, limit_ns)) record_timeout(ab);
  }
  __syncthreads();
}


}  // namespace

cudaError_t launch_gemm_w8a8(const GemmProblem& p, int sms, cudaStream_t st, int* tmap_err) {
  return use_pair(p) ? launch<Mode::W8A8, 2>(p, sms, st, tmap_err)
                     : launch<Mode::W8A8, 1>(p, sms, st, tmap_err);
}

cudaError_t launch_gemm_bf16(const GemmProblem& p, int sms, cudaStream_t st, int* tmap_err) {
  return use_pair(p) ? launch<Mode::BF16, 2>(p, sms, st, tmap_err)
                     : launch<Mode::BF16, 1>(p, sms, st, tmap_err);
}

cudaError_t launch_gemm_glu16(const GemmProblem& p, int sms, cudaStream_t st, int* tmap_err) {
  if (p.ex)
    return use_pair(p) ? launch<Mode::GLU16X, 2>(p, sms, st, tmap_err)
                       : launch<Mode::GLU16X, 1>(p, sms, st, tmap_err);
  return use_pair(p) ? launch<Mode::GLU16, 2>(p, sms, st, tmap_err)
                     : launch<Mode::GLU16, 1>(p, sms, st, tmap_err);
}

cudaError_t launch_gemm_glu(const GemmProblem& p, int sms, cudaStream_t st, int* tmap_err) {
  if (p.ex)
    return use_pair(p) ? launch<Mode::GLUX, 2>(p, sms, st, tmap_err)
                       : launch<Mode::GLUX, 1>(p, sms, st, tmap_err);
  return use_pair(p) ? launch<Mode::GLU, 2>(p, sms, st, tmap_err)
                     : launch<Mode::GLU, 1>(p, sms, st, tmap_err);
}

// W8A16 runs one CTA per tile with the dequantized weight in TMEM.  A CTA
// pair (cta_group::2 MMAs reading each CTA's 128 dequantized rows from its
// own TMEM, 6 stages with half the activation bytes per CTA, the odd CTA's
// conversions signalled to the even CTA every stage) gave bit-identical
// results but ran 1.65-1.7x slower at M = 4096 .. 20670, whether its waits
// spun or slept and at either acquire scope.
cudaError_t launch_gemm_w8a16(const GemmProblem& p, int sms, cudaStream_t st, int* tmap_err) {
  return launch_a16t(p, sms, st, tmap_err);
}

cudaError_t launch_selftest_timeout(cudaStream_t st) {
  selftest_timeout_kernel<<<1, 32, 0, st>>>(200000000ull);  // 0.2 s
  return cudaGetLastError();
}

cudaError_t gemm_read_error(cudaStream_t st, uint32_t* err) {
  uint32_t zero = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(err, g_gemm_err, sizeof(uint32_t), 0,
                                            cudaMemcpyDeviceToHost, st);
  if (e != cudaSuccess) return e;
  e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return e;
  if (*err) {
    e = cudaMemcpyToSymbolAsync(g_gemm_err, &zero, sizeof(uint32_t), 0, cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(st);
  }
  return e;
}

}  // namespace w8

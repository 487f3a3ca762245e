// Chunked (WY / UT-transform) prefill of the Gated DeltaNet recurrence on the
// 5th-generation tensor cores of sm_103a (tcgen05.mma kind::f16 with split
// operands, or kind::tf32; TMEM accumulators), for D_k = D_v = 128.
//
// The recurrence is the token-by-token one of the capture kernel page
// ("gated_delta_net_decode_capture.metal", mlx-native 0.9.2, decay-first) or
// of the module doc of "gated_delta_net.rs" (mlx-native 0.4.0, decay-after).
// Over a chunk of C = 64 tokens it is rewritten exactly (up to rounding) in
// matrix form.  With S the state entering the chunk (D_v x D_k, row = d_v),
// G_r = sum_{tau<=r} g_tau, gamma_r = exp(-G_r), Gam_{r,i} = exp(G_i - G_r):
//
//   A_{r,i}  = beta_r * Gam_{r,i} * (k_r . k_i)       (i < r; decay-after:
//              Gam_{r-1,i} and gamma_{r-1} below)      T = (I + A)^-1
//   U        = T diag(beta) V  -  T diag(beta gamma) K S^T       (C x D_v)
//   Y        = q_scale [diag(gamma) Q S^T + (Q K^T o Gam)_{i<=r} U]
//   S_next   = gamma_C S + U^T diag(Gam_{C,.}) K
//
// (the pseudo-values U are the per-token delta's; substituting the recurrence
// into itself gives exactly these sums).  Every product with a dimension of
// 128 runs on the tensor cores with M = 128 (D_v or the stacked [K;Q]):
//
//   G   = [K;Q] K^T              (Gram: rows 0..63 = K K^T, 64..127 = Q K^T)
//   [X | Yt] = S [K; Q']^T        Q' = c q_scale diag(gamma) Q (A = S from TMEM)
//   Ut  = V^T  T''^T + X (-T')^T  T''= T diag(beta), T' = c T diag(beta gamma)
//                                 (A = V^T and X from TMEM, one batch)
//   [Yt | S] += Ut [P'; K'^T]^T   P' = q_scale (Q K^T o Gam), K' = diag(Gam_C /
//                                 c_next) K (A = Ut from TMEM, one product)
//
// where Ut = U^T, Yt = Y^T (D_v x C) live in TMEM, and S is kept lazily as
// c * S (c = product of the chunk decays since the last fold), so the decay
// never needs a read-modify-write of TMEM; c is folded into S when it leaves
// [2^-30, 2^30], and a chunk whose |G| exceeds 40 (extreme gates) folds its
// decay into S before the update instead.  Accumulation is f32.  Operands are
// either rounded to TF32 (round-to-nearest) when staged, or split into bf16
// hi and lo halves with every product taken as three bf16 MMAs
// (chunked_common.cuh); the split form computes Yt = S Q^T and scales its
// columns by c q_scale gamma_r in TMEM instead of scaling Q, and splits X
// into hi and lo before the Ut batch.  The triangular inverse (64 x 64) is
// blocked 16 x 16: the diagonal blocks by substitution on the CUDA cores, the
// block products on the warp-level MMA with 3xTF32 operands.
//
// One CTA (8 warps) owns one segment of a (seq, value head) chain, with 512
// TMEM columns, X, Yt and S adjacent: TF32: X (and G) 0, Yt 64, S 128, Ut 256,
// V^T 320; split: X (and G) 0, Yt 64, S 128, S hi 256 (then X hi | lo), S lo
// 320 (then Ut hi | lo), V^T hi | lo 384, Ut 448.  Shared-memory operands use the
// canonical K-major no-swizzle layout: 8-row x 16-byte core matrices, cores
// adjacent along K (LBO = 128 B), core rows SBO = (K bytes / 16) * 128 B
// apart; a split operand is its hi image followed by its lo image.  Every
// mbarrier wait is bounded; on a timeout the CTA writes NaN to its
// state_out, frees its TMEM and returns.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <type_traits>

#include "chunked_common.cuh"
#include "gdn_internal.h"

namespace gdn {
namespace {

using namespace chunked;


// TMEM columns
template <bool SPLIT> struct Tm;
// X, Y^T and S are adjacent: [X | Y^T] is one N = 128 accumulator and
// [Y^T | S] one N = 192 accumulator; the Gram takes X's columns, which are
// dead from the previous chunk's U^T product on
template <> struct Tm<false> {
  static constexpr uint32_t X = 0, Y = 64, S = 128, G = 0, U = 256, V = 320;
};
template <> struct Tm<true> {  // SH / SL: S~ hi and lo, then X hi | lo and Ut hi | lo
  static constexpr uint32_t X = 0, Y = 64, S = 128, G = 0, SH = 256, SL = 320, V = 384, U = 448;
};
static_assert(Tm<false>::Y == Tm<false>::X + 64 && Tm<true>::Y == Tm<true>::X + 64 &&
              Tm<false>::S == Tm<false>::Y + 64 && Tm<true>::S == Tm<true>::Y + 64, "[X | Y^T | S] contiguous");
constexpr uint32_t TM_COLS = 512;

// shared memory map (bytes)
constexpr uint32_t SM_STACK = 0;                     // [K;Q] 128 x 128 canonical, 64 KB (split:
                                                     // hi 32 KB, then lo; Q rows from 16 KB on)
constexpr uint32_t SM_P = SM_STACK + 65536;          // [P'; K'^T]: P' 64 x 64 canonical, then K'^T
                                                     // 128 x 64 canonical, rows continuing (one B
                                                     // operand of 192 rows), 48 KB; split: the hi
                                                     // images, then the lo images from SM_P + PK_LO
constexpr uint32_t PK_LO = 24576;
constexpr uint32_t SM_A = SM_P + 49152;              // A plain 64 x LD; then -T' (canonical)
constexpr uint32_t SM_T = SM_A + 64 * LD * 4;        // T plain 64 x LD; then T'' (canonical)
constexpr uint32_t SM_M = SM_T + 64 * LD * 4;        // block products, 4 x 256 f32
constexpr uint32_t SM_SC = SM_M + 4 * 256 * 4;       // per-token scalars
constexpr int NSC = 11;                              // scalar arrays of 64
constexpr uint32_t SM_MISC = SM_SC + NSC * 64 * 4;   // mbarrier, tmem base, flags
constexpr int LDS = 132;                             // staging row stride (floats): 528 B, so the
                                                     // 8 rows of a core matrix hit distinct banks
constexpr uint32_t SM_KS = SM_MISC + 64;             // next chunk's K rows (natural), 64 x LDS
constexpr uint32_t SM_VS = SM_KS + 64 * LDS * 4;     // next chunk's V rows (natural), 64 x LDS
constexpr uint32_t SMEM_BYTES = SM_VS + 64 * LDS * 4;
constexpr uint32_t SM_TP = SM_A;                     // -T' canonical (16 KB) over the dead A
constexpr uint32_t SM_TPP = SM_T;                    // T''  canonical (16 KB) over the dead T

// scalar array slots
enum { SC_G = 0, SC_GAM, SC_GAMP, SC_BETA, SC_KTS, SC_TPS, SC_QS, SC_GPREV, SC_EG, SC_GRAW, SC_BRAW };

struct ChunkArgs {
  const void *__restrict__ q;  // q, k, v and output: f32, or bf16 with bf16 activations
  const void *__restrict__ k;
  const void *__restrict__ v;
  const float *__restrict__ g;
  const float *__restrict__ beta;
  const float *state_in;
  void *__restrict__ output;
  float *state_out;
  uint32_t nk, nv, nt, group, khead_div, nchunks;
  float q_scale;
  // the chain of each (seq, value head) runs as segments of seg_len chunks,
  // one launch per group of segments: CTA b of the launch takes segment
  // (seg_base + b) / heads of head (seg_base + b) % heads
  uint32_t heads, seg_len, seg_base;
};

struct Misc {
  unsigned long long mbar;   // MMA commits within a chunk
  unsigned long long mbar2;  // batch 2 (output and state update), waited in the next chunk
  uint32_t tmem_base;
  int failed;
  float c_renorm;   // factor folded into S at the chunk start (if do_renorm)
  float c_fold;     // factor folded into S before the update (if do_fold)
  float c_next;     // scale after this chunk
  int do_renorm;
  int do_fold;
};
static_assert(sizeof(Misc) <= 64, "misc area");

// bf16 activations: staged rows of 128 bf16 at a stride of 136 (272 bytes)
constexpr int LDSB = 136;

// Asynchronous copies of one chunk's Q rows; tokens past the chunk's end
// are zero-filled.  f32: into the stack's Q half (rows 64..127) in the TF32
// canonical order; bf16 activations: straight into the bf16 canonical image
// of the stack's Q rows (a 16-byte row of a core is 8 consecutive d_k of one
// token).  Issued by NT threads, tid counted from the first of them.
template <bool BF16IN, int NT>
__device__ __forceinline__ void stage_q_async(uint32_t sbase, const void *qv, size_t kq_tok, int nc, int tid) {
  if constexpr (BF16IN) {
    const uint16_t *qbase = static_cast<const uint16_t *>(qv);
#pragma unroll
    for (int it = 0; it < (64 * 16 + NT - 1) / NT; ++it) {
      const int cc = tid + NT * it;       // token cc >> 4, d_k 8 (cc & 15) .. +7
      if ((64 * 16) % NT != 0 && cc >= 64 * 16) break;
      const int r = cc >> 4, d0 = 8 * (cc & 15);
      cp_async16(sbase + SM_STACK + canon16(64 + r, d0, 128), qbase + (r < nc ? r : 0) * kq_tok + d0,
                 r < nc ? 16u : 0u);
    }
  } else {
    const float *qbase = static_cast<const float *>(qv);
#pragma unroll
    for (int it = 0; it < (64 * 32 + NT - 1) / NT; ++it) {
      const int cc = tid + NT * it;       // 16-byte chunk within the Q half
      if ((64 * 32) % NT != 0 && cc >= 64 * 32) break;
      const int core = cc >> 3, r = (core >> 5) * 8 + (cc & 7), c4 = core & 31;
      cp_async16(sbase + SM_STACK + 32768 + cc * 16, qbase + (r < nc ? r : 0) * kq_tok + 4 * c4,
                 r < nc ? 16u : 0u);
    }
  }
  cp_async_commit();
}

// Asynchronous copies of one chunk's gates and betas into the scalar area,
// by warp 0, which reads them (and waits for them) alone; tokens past the
// chunk's end are zero-filled.
__device__ __forceinline__ void stage_gates_async(uint32_t sbase, const float *g, const float *beta, size_t sc0,
                                                  size_t nv, int nc, int lane) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int i = lane + 32 * h;
    const size_t src = sc0 + static_cast<size_t>(i < nc ? i : 0) * nv;
    cp_async4(sbase + SM_SC + (SC_GRAW * 64 + i) * 4, g + src, i < nc ? 4u : 0u);
    cp_async4(sbase + SM_SC + (SC_BRAW * 64 + i) * 4, beta + src, i < nc ? 4u : 0u);
  }
  cp_async_commit();
}

// Asynchronous copies of one chunk's K and V rows (natural layout, row
// stride LDS floats, or LDSB bf16 with bf16 activations) into the staging
// buffers; rows past the end are zeros.  Issued by NT threads, tid counted
// from the first of them.
template <bool BF16IN, int NT = NTH>
__device__ __forceinline__ void stage_kv_async(uint32_t sbase, const void *kv, size_t kq_tok, const void *vv,
                                               size_t v_tok, int nc, int tid) {
  if constexpr (BF16IN) {
    const uint16_t *kbase = static_cast<const uint16_t *>(kv), *vbase = static_cast<const uint16_t *>(vv);
#pragma unroll
    for (int it = 0; it < (64 * 16 + NT - 1) / NT; ++it) {
      const int ci = tid + NT * it;       // 16-byte chunk: row ci/16, 8 bf16 at 8 (ci%16)
      if ((64 * 16) % NT != 0 && ci >= 64 * 16) break;
      const int r = ci >> 4, c8 = ci & 15;
      const uint32_t n = r < nc ? 16u : 0u;
      const int rr = r < nc ? r : 0;
      const uint32_t dst = static_cast<uint32_t>((r * LDSB + 8 * c8) * 2);
      cp_async16(sbase + SM_KS + dst, kbase + rr * kq_tok + 8 * c8, n);
      cp_async16(sbase + SM_VS + dst, vbase + rr * v_tok + 8 * c8, n);
    }
  } else {
    const float *kbase = static_cast<const float *>(kv), *vbase = static_cast<const float *>(vv);
#pragma unroll
    for (int it = 0; it < (64 * 32 + NT - 1) / NT; ++it) {
      const int ci = tid + NT * it;       // 16-byte chunk: row ci/32, float4 ci%32
      if ((64 * 32) % NT != 0 && ci >= 64 * 32) break;
      const int r = ci >> 5, c4 = ci & 31;
      const uint32_t n = r < nc ? 16u : 0u;
      const int rr = r < nc ? r : 0;
      const uint32_t dst = static_cast<uint32_t>((r * LDS + 4 * c4) * 4);
      cp_async16(sbase + SM_KS + dst, kbase + rr * kq_tok + 4 * c4, n);
      cp_async16(sbase + SM_VS + dst, vbase + rr * v_tok + 4 * c4, n);
    }
  }
  cp_async_commit();
}

// A bf16 bit pattern widened to f32 (exact).
__device__ __forceinline__ float bf16_bits_to_f32(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }

// BF16IN: q, k, v and output hold bf16 (split operands only): the inputs
// are exact bf16 values, so K, Q and V^T are their own hi halves with zero
// lo halves, and the products leave out the terms with a zero lo (the Gram
// is one bf16 product per K step, X, Y^T and V^T T''^T two); every other
// step is the f32 form's, and y is rounded to bf16 once when stored.
template <bool DECAY_AFTER, bool SPLIT, bool BF16IN>
__global__ void __launch_bounds__(NTH, 1) gdn_chunked_kernel(const ChunkArgs a) {
  static_assert(SPLIT || !BF16IN, "bf16 activations take split operands");
  using TM = Tm<SPLIT>;
  constexpr uint32_t SM_KT = SM_P + (SPLIT ? 8192 : 16384);  // K'^T: after P''s 64 rows
  using In = typename std::conditional<BF16IN, uint16_t, float>::type;
  extern __shared__ __align__(1024) unsigned char smem[];
  float *sA = reinterpret_cast<float *>(smem + SM_A);
  float *sT = reinterpret_cast<float *>(smem + SM_T);
  float *sM = reinterpret_cast<float *>(smem + SM_M);
  float *sc = reinterpret_cast<float *>(smem + SM_SC);
  const float *sKS = reinterpret_cast<const float *>(smem + SM_KS);
  const float *sVS = reinterpret_cast<const float *>(smem + SM_VS);
  Misc *misc = reinterpret_cast<Misc *>(smem + SM_MISC);
  const uint32_t sbase = smem_addr(smem);
  const uint32_t mbar = smem_addr(&misc->mbar), mbar2 = smem_addr(&misc->mbar2);

  const int tid = static_cast<int>(threadIdx.x);
  const int warp = tid >> 5, lane = tid & 31;
  const int row = tid & 127;          // TMEM lane of this thread (= d_v or a Gram row)
  const int half = tid >> 7;          // which half of a 64-column group this thread handles
  const uint32_t lane_field = static_cast<uint32_t>(32 * (warp & 3)) << 16;

  const uint32_t task = a.seg_base + blockIdx.x;
  const uint32_t seg = task / a.heads;
  const uint32_t head = task % a.heads;  // = s * nv + vh
  const uint32_t vh = head % a.nv, s = head / a.nv;
  const uint32_t kh = a.khead_div ? vh / a.group : vh % a.nk;
  // this segment: chunks [cb, cb + nchunks) of the window, tokens from tb on;
  // below, chunk and token indices count from the segment's start, and nt is
  // the number of tokens from there to the window's end
  const uint32_t cb = seg * a.seg_len;
  const uint32_t nchunks = min(a.seg_len, a.nchunks - cb);
  const uint32_t tb = cb * C;
  const uint32_t nt = a.nt - tb;
  const size_t state_head = static_cast<size_t>(head) * D * D;
  const size_t kq_tok = static_cast<size_t>(a.nk) * D;
  const size_t v_tok = static_cast<size_t>(a.nv) * D;
  const size_t tok0 = static_cast<size_t>(s) * a.nt + tb;  // the segment's first token of this seq
  const In *kseq = static_cast<const In *>(a.k) + (tok0 * a.nk + kh) * D;
  const In *qseq = static_cast<const In *>(a.q) + (tok0 * a.nk + kh) * D;
  const In *vseq = static_cast<const In *>(a.v) + (tok0 * a.nv + vh) * D;
  const uint16_t *sKSb = reinterpret_cast<const uint16_t *>(smem + SM_KS);  // bf16 staging views
  const uint16_t *sVSb = reinterpret_cast<const uint16_t *>(smem + SM_VS);
  const size_t sc_first = tok0 * a.nv + vh;
  // the state enters from state_in, or, after an earlier segment, from
  // state_out, where that segment left it (an earlier launch)
  const float *state_src = seg == 0 ? a.state_in : a.state_out;

  if (tid == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" :: "r"(mbar));
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" :: "r"(mbar2));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    misc->failed = 0;
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(smem_addr(&misc->tmem_base)), "r"(TM_COLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  // chunk 0's inputs start arriving while the state is loaded
  {
    const int nc0 = static_cast<int>(min(nt, static_cast<uint32_t>(C)));
    stage_kv_async<BF16IN>(sbase, kseq, kq_tok, vseq, v_tok, nc0, tid);
    stage_q_async<BF16IN, NTH>(sbase, qseq, kq_tok, nc0, tid);
    if (warp == 0) stage_gates_async(sbase, a.g, a.beta, sc_first, a.nv, nc0, lane);
  }
  cta_sync();
  const uint32_t tmem = misc->tmem_base;
  const uint32_t tl = tmem + lane_field;  // this warp's lane quarter

  // S <- state_in (c = 1).  Thread: row d_v, columns [64*half, 64*half + 64).
  {
    const float4 *src = reinterpret_cast<const float4 *>(state_src + state_head + row * D + 64 * half);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t v[32];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float4 x = __ldcs(src + 8 * h + j);
        v[4 * j] = __float_as_uint(x.x); v[4 * j + 1] = __float_as_uint(x.y);
        v[4 * j + 2] = __float_as_uint(x.z); v[4 * j + 3] = __float_as_uint(x.w);
      }
      GDN_TMEM_ST32(tl + TM::S + 64 * half + 32 * h, v);
    }
    tmem_wait_st();
  }

  // chunk 0's copies (issued by every thread) have landed; in the loop, warp
  // 0 waits for its own copies (the gates) and warps 1-7 for theirs (the rows)
  cp_async_wait_all();
  __syncthreads();

  float c = 1.f;          // S = c * (TMEM S), carried by warp 0 (the others read c_next at the end)
  uint32_t phase = 0, phase2 = 0;
  bool pending2 = false;  // a batch 2 committed and not yet waited for (uniform over the CTA)
  bool failed = false;
  // Y^T of the chunk starting at token tt0 (ncc tokens) to the output:
  // thread = d_v, tokens [32*half, +32)
  auto write_outputs = [&](uint32_t tt0, int ncc) {
    uint32_t yv[32];
    GDN_TMEM_LD32(tl + TM::Y + 32 * half, yv);
    tmem_wait_ld();
    In *obase = static_cast<In *>(a.output) + ((tok0 + tt0) * a.nv + vh) * D + row;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const int i = 32 * half + j;
      if (i < ncc) {
        if constexpr (BF16IN)
          obase[static_cast<size_t>(i) * v_tok] = __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(yv[j])));
        else
          obase[static_cast<size_t>(i) * v_tok] = __uint_as_float(yv[j]);
      }
    }
  };

  for (uint32_t ch = 0; ch < nchunks && !failed; ++ch) {
    const uint32_t t0 = ch * C;

    // ---- 1. per-token scalars (warp 0, once its own copies, the gates, have
    // landed; it has just issued the previous chunk's batch 2): prefix sums
    // of g, decays, scalings.  Meanwhile, 3., warps 1-7 build the stack.
    if (warp == 0) {
      cp_async_wait_all();
      __syncwarp();
      float g0 = sc[SC_GRAW * 64 + lane], g1 = sc[SC_GRAW * 64 + lane + 32];
      const float b0 = sc[SC_BRAW * 64 + lane], b1 = sc[SC_BRAW * 64 + lane + 32];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float u0 = __shfl_up_sync(0xffffffffu, g0, o), u1 = __shfl_up_sync(0xffffffffu, g1, o);
        if (lane >= o) { g0 += u0; g1 += u1; }
      }
      g1 += __shfl_sync(0xffffffffu, g0, 31);
      const float G0 = g0, G1 = g1;               // inclusive prefix sums, tokens lane, lane+32
      const float GC = __shfl_sync(0xffffffffu, G1, 31);  // = G of the last (or padded) token
      float Gp0 = __shfl_up_sync(0xffffffffu, G0, 1);
      if (lane == 0) Gp0 = 0.f;
      float Gp1 = __shfl_up_sync(0xffffffffu, G1, 1);
      const float G0_last = __shfl_sync(0xffffffffu, G0, 31);  // every lane takes part
      if (lane == 0) Gp1 = G0_last;
      const bool extreme = __any_sync(0xffffffffu, fabsf(G0) > kMaxLogScale || fabsf(G1) > kMaxLogScale);
      // fold c into S at the chunk start if it left [2^-30, 2^30]
      float cc = c, renorm = 1.f;
      const bool do_renorm = cc < kRenormLo || cc > kRenormHi;
      if (do_renorm) { renorm = cc; cc = 1.f; }
      const float gamC = __expf(-GC);
      float cnext, fold = 1.f;
      if (extreme) { fold = cc * gamC; cnext = 1.f; }
      else { cnext = cc * gamC; }
      const float gam0 = __expf(-G0), gam1 = __expf(-G1);
      const float gp0 = __expf(-Gp0), gp1 = __expf(-Gp1);
      sc[SC_G * 64 + lane] = G0; sc[SC_G * 64 + lane + 32] = G1;
      sc[SC_GPREV * 64 + lane] = Gp0; sc[SC_GPREV * 64 + lane + 32] = Gp1;
      sc[SC_GAM * 64 + lane] = gam0; sc[SC_GAM * 64 + lane + 32] = gam1;
      sc[SC_GAMP * 64 + lane] = gp0; sc[SC_GAMP * 64 + lane + 32] = gp1;
      sc[SC_BETA * 64 + lane] = b0; sc[SC_BETA * 64 + lane + 32] = b1;
      // e^{G_i} (only used when |G| <= 40, where it cannot overflow)
      sc[SC_EG * 64 + lane] = __expf(G0); sc[SC_EG * 64 + lane + 32] = __expf(G1);
      // K' row scale: Gam_{C,i} / c_next (lazy) or Gam_{C,i} (after a fold)
      sc[SC_KTS * 64 + lane] = __expf(G0 - GC) / cnext;
      sc[SC_KTS * 64 + lane + 32] = __expf(G1 - GC) / cnext;
      // -T' column scale: -c beta_i gamma_i (decay-after: gamma_{i-1})
      sc[SC_TPS * 64 + lane] = -cc * b0 * (DECAY_AFTER ? gp0 : gam0);
      sc[SC_TPS * 64 + lane + 32] = -cc * b1 * (DECAY_AFTER ? gp1 : gam1);
      // Q' row scale: c q_scale gamma_r
      sc[SC_QS * 64 + lane] = cc * a.q_scale * gam0;
      sc[SC_QS * 64 + lane + 32] = cc * a.q_scale * gam1;
      if (lane == 0) {
        misc->c_renorm = renorm; misc->c_fold = fold; misc->c_next = cnext;
        misc->do_renorm = do_renorm; misc->do_fold = extreme;
      }
      c = cnext;  // warp 0 carries c from chunk to chunk
    } else {
      // ---- 3. the stack from the staged rows (warps 1-7, once their own
      // copies -- the K, V and Q rows -- have landed): K (canonical) and Q
      // (the staged Q rows), rounded to TF32 in place or as bf16 hi and lo
      // images (bf16 activations: Q is in place already, K's rows are copied)
      constexpr int NS = NTH - 32;
      const int vt = tid - 32;
      cp_async_wait_all();
      asm volatile("bar.sync 3, %0;" :: "n"(NS) : "memory");  // warps 1-7
      if constexpr (BF16IN) {
#pragma unroll
        for (int it = 0; it < (64 * 16 + NS - 1) / NS; ++it) {
          const int ci = vt + NS * it;        // token ci >> 4, d_k 8 (ci & 15) .. +7
          if (ci >= 64 * 16) break;
          const int r = ci >> 4, d0 = 8 * (ci & 15);
          *reinterpret_cast<uint4 *>(smem + SM_STACK + canon16(r, d0, 128)) =
              *reinterpret_cast<const uint4 *>(sKSb + r * LDSB + d0);
        }
      } else if constexpr (SPLIT) {
        // the staged Q rows (f32, in the TF32 canonical order of the Q half),
        // read before the bf16 images overwrite them
        constexpr int NIT = (64 * 32 + NS - 1) / NS;
        float4 qv[NIT];
#pragma unroll
        for (int it = 0; it < NIT; ++it) {
          const int cc = vt + NS * it;
          if (cc < 64 * 32) qv[it] = *reinterpret_cast<const float4 *>(smem + SM_STACK + 32768 + cc * 16);
        }
        asm volatile("bar.sync 3, %0;" :: "n"(NS) : "memory");
#pragma unroll
        for (int it = 0; it < NIT; ++it) {
          const int cc = vt + NS * it;        // element group: row r, d_k 4 c4 .. +3
          if (cc >= 64 * 32) break;
          const int core = cc >> 3, r = (core >> 5) * 8 + (cc & 7), d0 = 4 * (core & 31);
          const float4 x = *reinterpret_cast<const float4 *>(sKS + r * LDS + d0);
          uint2 h, l;
          split2(x.x, x.y, h.x, l.x); split2(x.z, x.w, h.y, l.y);
          *reinterpret_cast<uint2 *>(smem + SM_STACK + canon16(r, d0, 128)) = h;
          *reinterpret_cast<uint2 *>(smem + SM_STACK + 32768 + canon16(r, d0, 128)) = l;
          split2(qv[it].x, qv[it].y, h.x, l.x); split2(qv[it].z, qv[it].w, h.y, l.y);
          *reinterpret_cast<uint2 *>(smem + SM_STACK + canon16(64 + r, d0, 128)) = h;
          *reinterpret_cast<uint2 *>(smem + SM_STACK + 32768 + canon16(64 + r, d0, 128)) = l;
        }
      } else {
#pragma unroll
        for (int it = 0; it < (64 * 32 + NS - 1) / NS; ++it) {
          const int ci = vt + NS * it;        // 16-byte chunk of the K half
          if (ci >= 64 * 32) break;
          const int core = ci >> 3, r = (core >> 5) * 8 + (ci & 7), c4 = core & 31;
          float4 x = *reinterpret_cast<const float4 *>(sKS + r * LDS + 4 * c4);
          x.x = tf32_rn(x.x); x.y = tf32_rn(x.y); x.z = tf32_rn(x.z); x.w = tf32_rn(x.w);
          *reinterpret_cast<float4 *>(smem + SM_STACK + ci * 16) = x;
          float4 *pq = reinterpret_cast<float4 *>(smem + SM_STACK + 32768 + ci * 16);
          float4 y = *pq;
          y.x = tf32_rn(y.x); y.y = tf32_rn(y.y); y.z = tf32_rn(y.z); y.w = tf32_rn(y.w);
          *pq = y;
        }
      }
    }
    fence_async_smem();
    cta_sync();
    const float c_renorm = misc->c_renorm, c_fold = misc->c_fold;
    const bool do_renorm = misc->do_renorm != 0, do_fold = misc->do_fold != 0;

    // ---- 4. Gram [K;Q] K^T -> TMEM G.  Meanwhile, once the previous chunk's
    // batch 2 is done (it ran beside this chunk's first steps): c folded
    // into S if needed, and the other operands from the staged rows -- K'^T
    // (smem, over the image batch 2 read), V^T (TMEM), split: S~ as hi and lo
    // (TMEM).  The previous chunk's outputs stay in Y^T until step 6.
    if (tid == 0) {
      if constexpr (BF16IN) {
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint64_t dh = sdesc(sbase + SM_STACK + ks * 256, 2048);
          mma_ss<true>(tmem + TM::G, dh, dh, idesc_bf16(128, 64), ks > 0);
        }
      } else if constexpr (SPLIT) {
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint64_t dh = sdesc(sbase + SM_STACK + ks * 256, 2048), dl = sdesc(sbase + SM_STACK + 32768 + ks * 256, 2048);
          mma_ss<true>(tmem + TM::G, dh, dh, idesc_bf16(128, 64), ks > 0);
          mma_ss<true>(tmem + TM::G, dh, dl, idesc_bf16(128, 64), 1);
          mma_ss<true>(tmem + TM::G, dl, dh, idesc_bf16(128, 64), 1);
        }
      } else {
#pragma unroll
        for (int ks = 0; ks < D / 8; ++ks) {
          const uint64_t d = sdesc(sbase + SM_STACK + ks * 256, 4096);
          mma_ss(tmem + TM::G, d, d, idesc_tf32(128, 64), ks > 0);
        }
      }
      mma_commit(mbar);
    }
    if (pending2) {
      if (!mbar_wait(mbar2, phase2)) misc->failed = 1;
      phase2 ^= 1;
      pending2 = false;
      fence_after();
    }
    if (do_renorm) tmem_scale64(tl + TM::S + 64 * half, c_renorm);  // c left [2^-30, 2^30] (rare)
    if constexpr (SPLIT) {
      // K'^T [d_k][i] (K extent 64): thread owns column d_k = row, tokens
      // [32*hf, +32) for hf = half; warp 0, which issues the Gram, leaves
      // its share to warp 4
      const float *kts = sc + SC_KTS * 64;
#pragma unroll 1
      for (int hf = warp == 4 ? 0 : (warp == 0 ? 2 : half); hf <= (warp == 0 ? 1 : half); ++hf)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int i = 32 * hf + 8 * j;
        float e[8];
#pragma unroll
        for (int u = 0; u < 8; ++u)
          e[u] = (BF16IN ? bf16_bits_to_f32(sKSb[(i + u) * LDSB + row]) : sKS[(i + u) * LDS + row]) * kts[i + u];
        uint4 h, l;
        split2(e[0], e[1], h.x, l.x); split2(e[2], e[3], h.y, l.y);
        split2(e[4], e[5], h.z, l.z); split2(e[6], e[7], h.w, l.w);
        *reinterpret_cast<uint4 *>(smem + SM_KT + canon16(row, i, 64)) = h;
        *reinterpret_cast<uint4 *>(smem + SM_KT + PK_LO + canon16(row, i, 64)) = l;
      }
      // V^T -> TMEM as hi | lo (lane d_v = row, token pairs of [32*half, +32));
      // bf16 activations: V^T is its own hi half
      if constexpr (BF16IN) {
        uint32_t vh[16];
#pragma unroll
        for (int j = 0; j < 16; ++j)
          vh[j] = static_cast<uint32_t>(sVSb[(32 * half + 2 * j) * LDSB + row]) |
                  (static_cast<uint32_t>(sVSb[(32 * half + 2 * j + 1) * LDSB + row]) << 16);
        GDN_TMEM_ST16(tl + TM::V + 16 * half, vh);
      } else {
        uint32_t vh[16], vl[16];
#pragma unroll
        for (int j = 0; j < 16; ++j)
          split2(sVS[(32 * half + 2 * j) * LDS + row], sVS[(32 * half + 2 * j + 1) * LDS + row], vh[j], vl[j]);
        GDN_TMEM_ST16(tl + TM::V + 16 * half, vh);
        GDN_TMEM_ST16(tl + TM::V + 32 + 16 * half, vl);
      }
      // S~ -> hi and lo (the previous chunk's products are done)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t v[32], sh[16], sl[16];
        GDN_TMEM_LD32(tl + TM::S + 64 * half + 32 * h, v);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 16; ++j) split2(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]), sh[j], sl[j]);
        GDN_TMEM_ST16(tl + TM::SH + 32 * half + 16 * h, sh);
        GDN_TMEM_ST16(tl + TM::SL + 32 * half + 16 * h, sl);
      }
    } else {
      // K'^T [d_k][i] (K extent 64): thread owns column d_k = row, tokens
      // [32*hf, +32) for hf = half; warp 0 leaves its share to warp 4
      const float *kts = sc + SC_KTS * 64;
#pragma unroll 1
      for (int hf = warp == 4 ? 0 : (warp == 0 ? 2 : half); hf <= (warp == 0 ? 1 : half); ++hf)
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int i = 32 * hf + 4 * j;
        *reinterpret_cast<float4 *>(smem + SM_KT + canon(row, i, 64)) =
            make_float4(tf32_rn(sKS[(i + 0) * LDS + row] * kts[i + 0]),
                        tf32_rn(sKS[(i + 1) * LDS + row] * kts[i + 1]),
                        tf32_rn(sKS[(i + 2) * LDS + row] * kts[i + 2]),
                        tf32_rn(sKS[(i + 3) * LDS + row] * kts[i + 3]));
      }
      // V^T -> TMEM (lane d_v = row, columns = tokens [32*half, +32))
      uint32_t vv[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) vv[j] = __float_as_uint(tf32_rn(sVS[(32 * half + j) * LDS + row]));
      GDN_TMEM_ST32(tl + TM::V + 32 * half, vv);
    }
    tmem_wait_st();
    fence_async_smem();
    if (!mbar_wait(mbar, phase)) misc->failed = 1;
    phase ^= 1;
    fence_after();

    // ---- 5. A (plain), P' (canonical), Q' (in place)
    {
      uint32_t gv[32];
      GDN_TMEM_LD32(tl + TM::G + 32 * half, gv);
      tmem_wait_ld();
      const float *G = sc + SC_G * 64, *eG = sc + SC_EG * 64;
      if (row < 64) {
        const int r = row;
        const float br = sc[SC_BETA * 64 + r];
        // Gam_{r,i} = e^{G_i - G_r} (decay-after: G_{r-1}); products of e^{G_i}
        // and e^{-G_r} when |G| <= 40, exponentials of differences otherwise
        const float Gr = DECAY_AFTER ? sc[SC_GPREV * 64 + r] : G[r];
        const float bgr = br * (DECAY_AFTER ? sc[SC_GAMP * 64 + r] : sc[SC_GAM * 64 + r]);
        // the branch on do_fold (uniform) stays outside the loop, so that the
        // common case evaluates no exponential
        auto a_row = [&](auto gamf) {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            float e[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int i = 32 * half + 4 * j + u;
              e[u] = i < r ? gamf(i) * __uint_as_float(gv[4 * j + u]) : 0.f;
            }
            *reinterpret_cast<float4 *>(sA + r * LD + 32 * half + 4 * j) = make_float4(e[0], e[1], e[2], e[3]);
          }
        };
        if (do_fold) a_row([&](int i) { return br * __expf(G[i] - Gr); });
        else a_row([&](int i) { return bgr * eG[i]; });
      } else {
        const int r = row - 64;
        const float Gr = G[r];
        const float qgr = a.q_scale * sc[SC_GAM * 64 + r];
        auto p_row = [&](auto gamf) {
          if constexpr (SPLIT) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              float e[8];
#pragma unroll
              for (int u = 0; u < 8; ++u) {
                const int i = 32 * half + 8 * j + u;
                e[u] = i <= r ? gamf(i) * __uint_as_float(gv[8 * j + u]) : 0.f;
              }
              uint4 h, l;
              split2(e[0], e[1], h.x, l.x); split2(e[2], e[3], h.y, l.y);
              split2(e[4], e[5], h.z, l.z); split2(e[6], e[7], h.w, l.w);
              *reinterpret_cast<uint4 *>(smem + SM_P + canon16(r, 32 * half + 8 * j, 64)) = h;
              *reinterpret_cast<uint4 *>(smem + SM_P + PK_LO + canon16(r, 32 * half + 8 * j, 64)) = l;
            }
          } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              float e[4];
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const int i = 32 * half + 4 * j + u;
                e[u] = i <= r ? tf32_rn(gamf(i) * __uint_as_float(gv[4 * j + u])) : 0.f;
              }
              *reinterpret_cast<float4 *>(smem + SM_P + canon(r, 32 * half + 4 * j, 64)) =
                  make_float4(e[0], e[1], e[2], e[3]);
            }
          }
        };
        if (do_fold) p_row([&](int i) { return a.q_scale * __expf(G[i] - Gr); });
        else p_row([&](int i) { return qgr * eG[i]; });
      }
      if constexpr (!SPLIT) {
        // Q' = c q_scale gamma_r Q, in place in the stack's Q half (rows 64..127)
        const float *qs = sc + SC_QS * 64;
#pragma unroll
        for (int it = 0; it < 8; ++it) {
          const int cc = tid + NTH * it;        // chunk within the Q half
          const int core = cc >> 3, r = (core >> 5) * 8 + (cc & 7);
          float4 *p = reinterpret_cast<float4 *>(smem + SM_STACK + 32768 + cc * 16);
          float4 x = *p;
          const float f = qs[r];
          x.x = tf32_rn(x.x * f); x.y = tf32_rn(x.y * f); x.z = tf32_rn(x.z * f); x.w = tf32_rn(x.w * f);
          *p = x;
        }
      }
    }
    cta_sync();

    // ---- 6. [X | Y^T] = S~ [K; Q]^T (TF32: S [K; Q']^T), one N = 128
    // product (the stack's K rows, then its Q rows), which needs no T, runs
    // on the tensor cores while warps 0-3 invert I + A; with split operands
    // warps 4-7 then split X into hi | lo over S~ hi and scale Y^T's columns
    // by c q_scale gamma_r.  Warps 4-7 first write the previous chunk's
    // outputs from Y^T (off the Gram step, where thread 0's issuing held up
    // its warp); warp 4 then issues the product (issuing takes about 44
    // cycles an instruction), so the inverse starts at once, and warps 4-7
    // stage the next chunk's K and V rows (their copies are issued off the
    // inverse's path).
    const bool next = ch + 1 < nchunks;
    const int ncn = next ? static_cast<int>(min(static_cast<uint32_t>(C), nt - t0 - C)) : 0;
    if (warp < 4) {
      tri_inverse<128>(sA, sT, sM, tid);
      if (!mbar_wait(mbar, phase)) misc->failed = 1;
    } else {
      // the previous chunk's outputs (this warp's d_v rows, all 64 tokens)
      // leave Y^T before [X | Y^T] overwrites it
      if (ch > 0) {
        In *obase = static_cast<In *>(a.output) + ((tok0 + t0 - C) * a.nv + vh) * D + row;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t yv[32];
          GDN_TMEM_LD32(tl + TM::Y + 32 * h, yv);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            if constexpr (BF16IN)
              obase[static_cast<size_t>(32 * h + j) * v_tok] = __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(yv[j])));
            else
              obase[static_cast<size_t>(32 * h + j) * v_tok] = __uint_as_float(yv[j]);
          }
        }
        fence_before();
        asm volatile("bar.sync 2, %0;" :: "n"(NTH / 2) : "memory");  // warps 4-7
        fence_after();
      }
      if (tid == NTH / 2) {
        if constexpr (SPLIT) {
          const uint32_t i128 = idesc_bf16(128, 128);
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {  // [X | Yt] = S~ [K; Q]^T
            const uint64_t bh = sdesc(sbase + SM_STACK + ks * 256, 2048), bl = sdesc(sbase + SM_STACK + 32768 + ks * 256, 2048);
            mma_ts<true>(tmem + TM::X, tmem + TM::SH + 8 * ks, bh, i128, ks > 0);
            if constexpr (!BF16IN) mma_ts<true>(tmem + TM::X, tmem + TM::SH + 8 * ks, bl, i128, 1);
            mma_ts<true>(tmem + TM::X, tmem + TM::SL + 8 * ks, bh, i128, 1);
          }
        } else {
#pragma unroll
          for (int ks = 0; ks < D / 8; ++ks)   // [X | Yt] = S [K; Q']^T
            mma_ts(tmem + TM::X, tmem + TM::S + 8 * ks, sdesc(sbase + SM_STACK + ks * 256, 4096), idesc_tf32(128, 128),
                   ks > 0);
        }
        mma_commit(mbar);
      }
      // the staging buffers are free (every thread took its operands from
      // them before step 5's barrier): the next chunk's K and V rows, issued
      // here so that warps 0-3 start the inverse at once
      if (next && warp > 4)  // warps 5-7 (warp 4 issues the product)
        stage_kv_async<BF16IN, NTH / 2 - 32>(sbase, kseq + (t0 + C) * kq_tok, kq_tok, vseq + (t0 + C) * v_tok,
                                             v_tok, ncn, tid - NTH / 2 - 32);
      if (!mbar_wait(mbar, phase)) misc->failed = 1;
      if constexpr (SPLIT) {
        __syncwarp();
        fence_after();
        const float *qs = sc + SC_QS * 64;
#pragma unroll
        for (int h = 0; h < 2; ++h) {  // this warp's lanes, all 64 columns
          uint32_t xv[32], xh[16], xl[16];
          GDN_TMEM_LD32(tl + TM::X + 32 * h, xv);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 16; ++j) split2(__uint_as_float(xv[2 * j]), __uint_as_float(xv[2 * j + 1]), xh[j], xl[j]);
          GDN_TMEM_ST16(tl + TM::SH + 16 * h, xh);
          GDN_TMEM_ST16(tl + TM::SH + 32 + 16 * h, xl);
          GDN_TMEM_LD32(tl + TM::Y + 32 * h, xv);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 32; ++j) xv[j] = __float_as_uint(__uint_as_float(xv[j]) * qs[32 * h + j]);
          GDN_TMEM_ST32(tl + TM::Y + 32 * h, xv);
        }
        tmem_wait_st();
      }
    }
    phase ^= 1;
    cta_sync();
    if (misc->failed) { failed = true; break; }

    // ---- 7. -T' (over A) and T'' (over T), canonical images
    if constexpr (SPLIT) {
      const float *tps = sc + SC_TPS * 64, *bet = sc + SC_BETA * 64;
      float4 t0[2], t1[2];
      int ci[2];
#pragma unroll
      for (int it = 0; it < 2; ++it) {
        ci[it] = tid + NTH * it;              // 16-byte row ci & 7 of bf16 core ci >> 3 = (R, Kc)
        const int core = ci[it] >> 3, r = (core >> 3) * 8 + (ci[it] & 7), i0 = 8 * (core & 7);
        t0[it] = *reinterpret_cast<const float4 *>(sT + r * LD + i0);
        t1[it] = *reinterpret_cast<const float4 *>(sT + r * LD + i0 + 4);
      }
      __syncthreads();                        // every thread has read T before it is overwritten
#pragma unroll
      for (int it = 0; it < 2; ++it) {
        const int i0 = 8 * ((ci[it] >> 3) & 7);
        const float t[8] = {t0[it].x, t0[it].y, t0[it].z, t0[it].w, t1[it].x, t1[it].y, t1[it].z, t1[it].w};
        uint4 h, l;
        split2(t[0] * tps[i0], t[1] * tps[i0 + 1], h.x, l.x); split2(t[2] * tps[i0 + 2], t[3] * tps[i0 + 3], h.y, l.y);
        split2(t[4] * tps[i0 + 4], t[5] * tps[i0 + 5], h.z, l.z); split2(t[6] * tps[i0 + 6], t[7] * tps[i0 + 7], h.w, l.w);
        *reinterpret_cast<uint4 *>(smem + SM_TP + ci[it] * 16) = h;
        *reinterpret_cast<uint4 *>(smem + SM_TP + 8192 + ci[it] * 16) = l;
        split2(t[0] * bet[i0], t[1] * bet[i0 + 1], h.x, l.x); split2(t[2] * bet[i0 + 2], t[3] * bet[i0 + 3], h.y, l.y);
        split2(t[4] * bet[i0 + 4], t[5] * bet[i0 + 5], h.z, l.z); split2(t[6] * bet[i0 + 6], t[7] * bet[i0 + 7], h.w, l.w);
        *reinterpret_cast<uint4 *>(smem + SM_TPP + ci[it] * 16) = h;
        *reinterpret_cast<uint4 *>(smem + SM_TPP + 8192 + ci[it] * 16) = l;
      }
    } else {
      const float *tps = sc + SC_TPS * 64, *bet = sc + SC_BETA * 64;
      float4 t[4];
      int ci[4];
#pragma unroll
      for (int it = 0; it < 4; ++it) {
        ci[it] = tid + NTH * it;              // 16-byte chunk of a 64 x 64 canonical image
        const int core = ci[it] >> 3, r = (core >> 4) * 8 + (ci[it] & 7), i0 = 4 * (core & 15);
        t[it] = *reinterpret_cast<const float4 *>(sT + r * LD + i0);
      }
      __syncthreads();                        // every thread has read T before it is overwritten
#pragma unroll
      for (int it = 0; it < 4; ++it) {
        const int i0 = 4 * ((ci[it] >> 3) & 15);
        *reinterpret_cast<float4 *>(smem + SM_TP + ci[it] * 16) =
            make_float4(tf32_rn(t[it].x * tps[i0]), tf32_rn(t[it].y * tps[i0 + 1]),
                        tf32_rn(t[it].z * tps[i0 + 2]), tf32_rn(t[it].w * tps[i0 + 3]));
        *reinterpret_cast<float4 *>(smem + SM_TPP + ci[it] * 16) =
            make_float4(tf32_rn(t[it].x * bet[i0]), tf32_rn(t[it].y * bet[i0 + 1]),
                        tf32_rn(t[it].z * bet[i0 + 2]), tf32_rn(t[it].w * bet[i0 + 3]));
      }
    }
    fence_async_smem();
    cta_sync();

    // ---- 8. U^T = V^T T''^T + X (-T')^T; then U^T made an A operand
    // (rounded to TF32 in place -- the tensor core would otherwise truncate
    // it -- or split over S~ lo) and, for an extreme-gate chunk, the chunk's
    // decay folded into S; batch 2 adds the intra-chunk output and updates S.
    if (tid == 0) {
      if constexpr (SPLIT) {
        const uint32_t i64 = idesc_bf16(128, 64);
#pragma unroll
        for (int ks = 0; ks < C / 16; ++ks) {  // Ut = V^T T''^T
          const uint64_t bh = sdesc(sbase + SM_TPP + ks * 256, 1024), bl = sdesc(sbase + SM_TPP + 8192 + ks * 256, 1024);
          mma_ts<true>(tmem + TM::U, tmem + TM::V + 8 * ks, bh, i64, ks > 0);
          mma_ts<true>(tmem + TM::U, tmem + TM::V + 8 * ks, bl, i64, 1);
          if constexpr (!BF16IN) mma_ts<true>(tmem + TM::U, tmem + TM::V + 32 + 8 * ks, bh, i64, 1);
        }
#pragma unroll
        for (int ks = 0; ks < C / 16; ++ks) {  // Ut += X (-T')^T
          const uint64_t bh = sdesc(sbase + SM_TP + ks * 256, 1024), bl = sdesc(sbase + SM_TP + 8192 + ks * 256, 1024);
          mma_ts<true>(tmem + TM::U, tmem + TM::SH + 8 * ks, bh, idesc_bf16(128, 64), 1);
          mma_ts<true>(tmem + TM::U, tmem + TM::SH + 8 * ks, bl, idesc_bf16(128, 64), 1);
          mma_ts<true>(tmem + TM::U, tmem + TM::SH + 32 + 8 * ks, bh, idesc_bf16(128, 64), 1);
        }
      } else {
        const uint32_t i64 = idesc_tf32(128, 64);
#pragma unroll
        for (int ks = 0; ks < C / 8; ++ks)   // Ut = V^T T''^T
          mma_ts(tmem + TM::U, tmem + TM::V + 8 * ks, sdesc(sbase + SM_TPP + ks * 256, 2048), i64, ks > 0);
#pragma unroll
        for (int ks = 0; ks < C / 8; ++ks)   // Ut += X (-T')^T
          mma_ts(tmem + TM::U, tmem + TM::X + 8 * ks, sdesc(sbase + SM_TP + ks * 256, 2048), i64, 1);
      }
      mma_commit(mbar);
    }
    // while U^T runs (the stack is free: X and Y^T are done): the next chunk's Q rows and gates
    if (next) {
      if (warp == 0)
        stage_gates_async(sbase, a.g, a.beta, sc_first + static_cast<size_t>(t0 + C) * a.nv, a.nv, ncn, lane);
      else
        stage_q_async<BF16IN, NTH - 32>(sbase, qseq + (t0 + C) * kq_tok, kq_tok, ncn, tid - 32);
    }
    if (!mbar_wait(mbar, phase)) misc->failed = 1;
    phase ^= 1;
    fence_after();
    if constexpr (SPLIT) {
      {  // Ut -> hi | lo over S~ lo
        uint32_t uv[32], uh[16], ul[16];
        GDN_TMEM_LD32(tl + TM::U + 32 * half, uv);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 16; ++j) split2(__uint_as_float(uv[2 * j]), __uint_as_float(uv[2 * j + 1]), uh[j], ul[j]);
        GDN_TMEM_ST16(tl + TM::SL + 16 * half, uh);
        GDN_TMEM_ST16(tl + TM::SL + 32 + 16 * half, ul);
        tmem_wait_st();
      }
    } else {
      {
        uint32_t uv[32];
        GDN_TMEM_LD32(tl + TM::U + 32 * half, uv);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j) uv[j] = __float_as_uint(tf32_rn(__uint_as_float(uv[j])));
        GDN_TMEM_ST32(tl + TM::U + 32 * half, uv);
        tmem_wait_st();
      }
    }
    if (do_fold) tmem_scale64(tl + TM::S + 64 * half, c_fold);  // extreme gates: decay S now
    cta_sync();
    if (tid == 0) {  // [Yt | S] += Ut [P'; K'^T]^T, one N = 192 product
      if constexpr (SPLIT) {
        const uint32_t i192 = idesc_bf16(128, 192);
#pragma unroll
        for (int ks = 0; ks < C / 16; ++ks) {
          const uint64_t bh = sdesc(sbase + SM_P + ks * 256, 1024), bl = sdesc(sbase + SM_P + PK_LO + ks * 256, 1024);
          mma_ts<true>(tmem + TM::Y, tmem + TM::SL + 8 * ks, bh, i192, 1);
          mma_ts<true>(tmem + TM::Y, tmem + TM::SL + 8 * ks, bl, i192, 1);
          mma_ts<true>(tmem + TM::Y, tmem + TM::SL + 32 + 8 * ks, bh, i192, 1);
        }
      } else {
#pragma unroll
        for (int ks = 0; ks < C / 8; ++ks)
          mma_ts(tmem + TM::Y, tmem + TM::U + 8 * ks, sdesc(sbase + SM_P + ks * 256, 2048), idesc_tf32(128, 192), 1);
      }
      mma_commit(mbar2);
    }
    pending2 = true;

    // (batch 2 runs beside the next chunk's first steps, which wait for it
    // before they touch S, K'^T or Y^T; this chunk's outputs are written
    // by warps 4-7 in the next chunk's step 6, the last chunk's after the
    // loop)
    if (misc->failed) failed = true;
  }

  if (pending2) {
    if (!mbar_wait(mbar2, phase2)) misc->failed = 1;
    fence_after();
  }
  cta_sync();
  if (misc->failed) failed = true;
  if (!failed && nchunks > 0) {
    const uint32_t tl0 = (nchunks - 1) * C;
    write_outputs(tl0, static_cast<int>(nt - tl0));
  }
  cp_async_wait_all();  // no copy may still be landing in shared memory at exit
  if (failed && tid == 0) report_wait_timeout();

  // ---- state_out = c * S (or NaN if a wait timed out)
  {
    float4 *dst = reinterpret_cast<float4 *>(a.state_out + state_head + row * D + 64 * half);
    const float f = failed ? __int_as_float(0x7fc00000) : (nchunks > 0 ? misc->c_next : 1.f);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t v[32];
      GDN_TMEM_LD32(tl + TM::S + 64 * half + 32 * h, v);
      tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < 8; ++j)
        __stcs(dst + 8 * h + j, make_float4(__uint_as_float(v[4 * j]) * f, __uint_as_float(v[4 * j + 1]) * f,
                                            __uint_as_float(v[4 * j + 2]) * f, __uint_as_float(v[4 * j + 3]) * f));
    }
  }
  cta_sync();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(tmem), "r"(TM_COLS));
}

template <bool DA, bool SPLIT, bool BF16IN>
cudaError_t launch(const Problem &p, cudaStream_t stream) {
  ChunkArgs a;
  a.q = p.q; a.k = p.k; a.v = p.v; a.g = p.g; a.beta = p.beta;
  a.state_in = p.state_in; a.output = p.output; a.state_out = p.state_out;
  a.nk = p.nk; a.nv = p.nv; a.nt = p.nt;
  a.group = p.nv / p.nk;
  a.khead_div = p.khead_div ? 1u : 0u;
  a.q_scale = p.q_scale;
  const uint32_t nchunks = (p.nt + C - 1) / C;
  const unsigned long long heads = static_cast<unsigned long long>(p.nv) * p.ns;
  if (heads == 0 || heads * nchunks > 0x7fffffffull) return cudaErrorInvalidConfiguration;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const unsigned long long want = static_cast<unsigned long long>(sms > 0 ? sms : 1);
  a.nchunks = nchunks;
  a.heads = static_cast<uint32_t>(heads);
  const uint32_t segs = state_segments(heads, nchunks, want);
  a.seg_len = (nchunks + segs - 1) / segs;
  const unsigned long long tasks = heads * ((nchunks + a.seg_len - 1) / a.seg_len);
  auto kern = gdn_chunked_kernel<DA, SPLIT, BF16IN>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(SMEM_BYTES));
  if (e != cudaSuccess) return e;
  // one launch per group of up to `want` (one CTA per SM) segments, in the
  // order segment-major: a head's segment j + 1 lies at least `heads` >=
  // `want` tasks after its segment j, so in a later launch
  const unsigned long long per_launch = segs > 1 ? want : tasks;
  for (unsigned long long base = 0; base < tasks; base += per_launch) {
    a.seg_base = static_cast<uint32_t>(base);
    const unsigned long long n = min(per_launch, tasks - base);
    kern<<<static_cast<unsigned>(n), NTH, SMEM_BYTES, stream>>>(a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace

bool chunked_supported(const Problem &p) {
  return p.dk == 128 && p.dv == 128 && p.capture == nullptr && !(p.io_bf16 && p.tf32);
}

cudaError_t launch_chunked(const Problem &p, cudaStream_t stream) {
  if (!chunked_supported(p)) return cudaErrorInvalidValue;
  if (p.tf32) return p.decay_after ? launch<true, false, false>(p, stream) : launch<false, false, false>(p, stream);
  if (p.io_bf16) return p.decay_after ? launch<true, true, true>(p, stream) : launch<false, true, true>(p, stream);
  return p.decay_after ? launch<true, true, false>(p, stream) : launch<false, true, false>(p, stream);
}

cudaError_t chunked_wait_status(unsigned int *bits, bool reset, cudaStream_t stream) {
  return chunked::read_wait_status(bits, reset, stream);
}

}  // namespace gdn

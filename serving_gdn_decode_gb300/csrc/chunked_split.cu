// Two-pass chunked (WY / UT-transform) prefill of the Gated DeltaNet
// recurrence on sm_103a, D_k = D_v = 128: the same chunk equations as the
// single-pass kernel (chunked.cu), split at the state.
//
// Pass 1, one CTA per (seq, chunk, key head), computes everything that does
// not depend on the state and writes it to a caller-provided workspace.  It
// turns the key head's K and Q into tensor-core operands once and stores them
// in the 128-byte-swizzled layout the MMA reads (exactly its shared-memory
// stack), stores K^T as a canonical image, and forms the Gram products K K^T
// and Q K^T once; then, for each value head that reads the key head, that
// head's gates give A, T = (I + A)^-1 (chunked_common.cuh), T'' = T diag(beta) and
// P' = q_scale (Q K^T o Gam)_{i<=r}, stored as canonical images.  The state
// pass loads every operand ready-made and converts nothing but its own TMEM
// products.
//
// Pass 2, one CTA per segment of a (seq, value head) chain (with more chains
// than SMs the chains are cut into segments run by consecutive launches,
// which hand the state on through state_out), runs the state-dependent chain
// per chunk with the state in TMEM as S = c * S~ (c a lazy scalar): [X | Z] =
// S~ [K; Q]^T, W = V^T - X diag(c gamma), U^T = W T''^T, Y^T = Z diag(c
// q_scale gamma) + U^T P'^T, S~ += U~^T K^T.  Its loads are bulk copies
// (images) and one TMA box per chunk (V rows), each on its own mbarrier.
//
// Operands are either split bf16 (every product as three bf16 MMAs of the
// halves, chunked_common.cuh) or TF32 (one MMA, rounded to nearest); both
// take four bytes per element, so the layouts below have the same sizes.
//
// Workspace layout (floats):
//   ws[head][chunk][8192], head = s * n_v + vh:
//     TF32:  [0, 4096) T'' and [4096, 8192) P' (64 x 64 canonical images);
//     split: T'' hi, T'' lo, P' hi, P' lo (2048 floats each, 64 x 64 bf16
//            canonical images);
//   then ws_k[s * n_k + kh][chunk][24576]:
//     TF32:  [0, 16384) the [K; Q] stack (column block cb = 16 KB: K's 64
//            rows, then Q's, 128-byte swizzled, 32 d_k each),
//            [16384, 24576) K^T (128 x 64 canonical);
//     split: [0, 16384) the stack as blocks hi(d_k 0-63), lo(0-63),
//            hi(64-127), lo(64-127) of 16 KB (128 rows x 64 bf16, swizzled),
//            [16384, 20480) K^T hi, [20480, 24576) K^T lo (128 x 64 bf16
//            canonical);
//     bf16 activations (split operands; K and Q are their own hi halves):
//            [0, 8192) the stack as hi(d_k 0-63), hi(64-127), [8192, 12288)
//            K^T; the rest of the slot is unused.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>
#include <type_traits>

#include "chunked_common.cuh"
#include "gdn_internal.h"

namespace gdn {
namespace {

using namespace chunked;

constexpr uint32_t kWsFloats = 8192;    // per (head, chunk): T'' and P'
constexpr uint32_t kWsKFloats = 24576;  // per (seq, key head, chunk): [K; Q] and K^T images

// per-token scalar slots (64 floats each)
enum { Q_G = 0, Q_GAM, Q_GAMP, Q_BETA, Q_GPREV, Q_EG, Q_GRAW, Q_BRAW, Q_KTS, Q_WS, Q_QS, Q_NSC };

// Per-chunk scalars of one warp (warp 0): inclusive prefix sums of g over the
// chunk (G), exclusive ones (Gp), the decays e^-G, e^-Gp, e^G and whether any
// |G| exceeds kMaxLogScale.  Reads raw g/beta from sc, writes the slots.
__device__ __forceinline__ bool chunk_scalars(float *sc, int lane, float *GC_out) {
  float g0 = sc[Q_GRAW * 64 + lane], g1 = sc[Q_GRAW * 64 + lane + 32];
  const float b0 = sc[Q_BRAW * 64 + lane], b1 = sc[Q_BRAW * 64 + lane + 32];
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float u0 = __shfl_up_sync(0xffffffffu, g0, o), u1 = __shfl_up_sync(0xffffffffu, g1, o);
    if (lane >= o) { g0 += u0; g1 += u1; }
  }
  g1 += __shfl_sync(0xffffffffu, g0, 31);
  const float G0 = g0, G1 = g1;
  const float GC = __shfl_sync(0xffffffffu, G1, 31);
  float Gp0 = __shfl_up_sync(0xffffffffu, G0, 1);
  if (lane == 0) Gp0 = 0.f;
  float Gp1 = __shfl_up_sync(0xffffffffu, G1, 1);
  const float G0_last = __shfl_sync(0xffffffffu, G0, 31);
  if (lane == 0) Gp1 = G0_last;
  const bool extreme = __any_sync(0xffffffffu, fabsf(G0) > kMaxLogScale || fabsf(G1) > kMaxLogScale);
  sc[Q_G * 64 + lane] = G0; sc[Q_G * 64 + lane + 32] = G1;
  sc[Q_GPREV * 64 + lane] = Gp0; sc[Q_GPREV * 64 + lane + 32] = Gp1;
  sc[Q_GAM * 64 + lane] = __expf(-G0); sc[Q_GAM * 64 + lane + 32] = __expf(-G1);
  sc[Q_GAMP * 64 + lane] = __expf(-Gp0); sc[Q_GAMP * 64 + lane + 32] = __expf(-Gp1);
  sc[Q_EG * 64 + lane] = __expf(G0); sc[Q_EG * 64 + lane + 32] = __expf(G1);
  sc[Q_BETA * 64 + lane] = b0; sc[Q_BETA * 64 + lane + 32] = b1;
  *GC_out = GC;
  return extreme;
}

// ---------------------------------------------------------------- TMA

// One box of a 4-D tensor map (coordinates innermost first) into shared memory.
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap *tm, int c0, int c1, int c2, int c3,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], [%6];"
      :: "r"(dst), "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
      : "memory");
}
// K-major SWIZZLE_128B operand descriptor: 8-row x 128-byte atoms 1024 bytes apart.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) {
  return static_cast<uint64_t>((saddr >> 4) & 0x3FFF) | (1ull << 16) |
         (static_cast<uint64_t>(1024 >> 4) << 32) | (1ull << 46) | (2ull << 61);
}
// T'' and P' are lower triangular (diagonal included).  In the canonical
// K-major image of a 64 x 64 matrix the 8 x 4 core block (R, Kc) -- rows
// 8R .. 8R+7, columns 4Kc .. 4Kc+3 -- holds a nonzero only if Kc <= 2R + 1,
// so the used cores of each 8-row group (2 KB) are a prefix of 2R + 2 cores
// (128 bytes each): 72 of 128.  Pass 1 writes only those, pass 2 copies only
// those into image buffers whose other cores it zeroed once.
__host__ __device__ constexpr bool tri_core_used(int R, int Kc) { return Kc <= 2 * R + 1; }
constexpr uint32_t kTriBytes = 72 * 128;  // the used cores of one image
// The used cores of the image at src (global) into the image at dst (shared).
__device__ __forceinline__ void load_tri(uint32_t dst, const float *src, uint32_t bar) {
  mbar_expect_tx(bar, kTriBytes);
#pragma unroll
  for (int R = 0; R < 8; ++R) bulk_load(dst + R * 2048, src + R * 512, (2 * R + 2) * 128, bar);
}
// The same for a bf16 image (8 x 8-element cores, 1 KB per 8-row group):
// core (R, Kc) is used if Kc <= R, 36 of 64.  The hi and lo images of a
// matrix (8 KB apart, both sides) come on one barrier.
__host__ __device__ constexpr bool tri16_used(int R, int Kc) { return Kc <= R; }
constexpr uint32_t kTri16Bytes = 36 * 128;
__device__ __forceinline__ void load_tri16_pair(uint32_t dst, const float *src, uint32_t bar) {
  mbar_expect_tx(bar, 2 * kTri16Bytes);
#pragma unroll
  for (int h = 0; h < 2; ++h)
#pragma unroll
    for (int R = 0; R < 8; ++R) bulk_load(dst + h * 8192 + R * 1024, src + h * 2048 + R * 256, (R + 1) * 128, bar);
}
template <bool SPLIT>
__device__ __forceinline__ void load_image(uint32_t dst, const float *src, uint32_t bar) {
  if constexpr (SPLIT) load_tri16_pair(dst, src, bar);
  else load_tri(dst, src, bar);
}

// ================================================================ pass 1

// shared memory (bytes): the [K;Q] stack for the Gram, then, once the Gram
// is in TMEM, A, T and the block products overlaid on it; one set of
// per-token scalars per value head of the key head (group x Q_NSC slots);
// the raw g and beta of those heads (group x 128 floats); the barriers and
// one "extreme gates" flag per head.
constexpr uint32_t P1_STACK = 0;
constexpr uint32_t P1_A = 0;
constexpr uint32_t P1_T = 64 * LD * 4;
constexpr uint32_t P1_M = 2 * 64 * LD * 4;
constexpr uint32_t P1_SC = 65536;
constexpr uint32_t kScSet = Q_NSC * 64;  // floats of one head's scalar set
static_assert(P1_M + 4 * 256 * 4 <= P1_SC, "pass-1 overlay must fit in the stack");
__host__ __device__ constexpr uint32_t p1_rg(uint32_t group) { return P1_SC + group * kScSet * 4u; }
__host__ __device__ constexpr uint32_t p1_misc(uint32_t group) { return p1_rg(group) + group * 512u; }
__host__ __device__ constexpr uint32_t p1_smem(uint32_t group) {  // + room to align the base to 1024
  return p1_misc(group) + 32u + 4u * group + 1024u;
}

struct PrepArgs {
  const float *__restrict__ q;
  const float *__restrict__ k;
  const float *__restrict__ g;
  const float *__restrict__ beta;
  float *__restrict__ ws;    // per (head, chunk) images
  float *__restrict__ ws_k;  // per (seq, key head, chunk) images
  uint32_t nk, nv, nt, group, khead_div, nchunks;
  uint32_t hpc, parts;       // value heads per CTA; CTAs per (seq, chunk, key head)
  float q_scale;
};

struct P1Misc {
  unsigned long long mbar;    // Gram MMA commit
  unsigned long long bar_ld;  // TMA: the chunk's K and Q rows
  uint32_t tmem_base;
  int failed;
};
static_assert(sizeof(P1Misc) <= 32, "pass-1 misc area");  // then one int per value head: extreme gates

// One CTA per (seq, chunk, key head) -- or per part of its value heads when
// there are fewer of those than SMs.  The stack [K;Q] arrives by TMA,
// 128-byte swizzled: column block cb (32 floats) holds K's 64 rows then Q's
// 64 rows (16 KB), so A = [K;Q] (M = 128) and B = K (N = 64) of the Gram are
// K-major SWIZZLE_128B operands.  K and Q are rounded and the Gram formed
// once for the key head; the key-head images ([K; Q] stack and K^T) are
// stored; then, for each value head that reads this key head in turn, its
// gates turn the Gram into A and P', and T'' follows from T = (I + A)^-1.
// SPLIT: split-bf16 operands, else TF32.  BF16IN: bf16 activations (with
// SPLIT): the TMA boxes land as the bf16 hi blocks, the Gram is one product
// per K step, and only hi images are stored.
template <bool DECAY_AFTER, bool SPLIT, bool BF16IN>
__global__ void __launch_bounds__(NTH, 3)
    gdn_chunk_prep_kernel(const PrepArgs a, const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_q) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t raw_addr = smem_addr(smem_raw);
  unsigned char *smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  float *sA = reinterpret_cast<float *>(smem + P1_A);
  float *sT = reinterpret_cast<float *>(smem + P1_T);
  float *sM = reinterpret_cast<float *>(smem + P1_M);
  float *sc = reinterpret_cast<float *>(smem + P1_SC);
  const float *rg = reinterpret_cast<const float *>(smem + p1_rg(a.hpc));
  P1Misc *misc = reinterpret_cast<P1Misc *>(smem + p1_misc(a.hpc));
  int *extreme_of = reinterpret_cast<int *>(smem + p1_misc(a.hpc) + 32);  // [hpc]
  const uint32_t sbase = smem_addr(smem);
  const uint32_t mbar = smem_addr(&misc->mbar), bar_ld = smem_addr(&misc->bar_ld);
  const int tid = static_cast<int>(threadIdx.x);
  const int warp = tid >> 5, lane = tid & 31;
  const int row = tid & 127, half = tid >> 7;
  const uint32_t lane_field = static_cast<uint32_t>(32 * (warp & 3)) << 16;

  // block -> (seq, chunk, key head, part), part fastest; this CTA takes the
  // key head's value heads j0 .. j0 + nh - 1
  const uint32_t part = blockIdx.x % a.parts;
  const uint32_t kh = (blockIdx.x / a.parts) % a.nk;
  const uint32_t rest = blockIdx.x / a.parts / a.nk;
  const uint32_t ch = rest % a.nchunks, s = rest / a.nchunks;
  const uint32_t j0 = part * a.hpc, nh = min(a.hpc, a.group - j0);
  const bool store_k = part == 0;  // the first part stores the key-head images
  const uint32_t t0 = ch * C;
  const int nc = static_cast<int>(min(static_cast<uint32_t>(C), a.nt - t0));
  float *wk = a.ws_k + ((static_cast<size_t>(s) * a.nk + kh) * a.nchunks + ch) * kWsKFloats;
  // value head jl of this CTA (j0 + jl of the key head)
  auto vhead = [&](uint32_t jl) {
    const uint32_t j = j0 + jl;
    return a.khead_div ? kh * a.group + j : kh + j * a.nk;
  };

  // raw g and beta of this CTA's value heads (tokens past the chunk's end
  // read as zero)
  for (uint32_t e = static_cast<uint32_t>(tid); e < nh * 128u; e += NTH) {
    const uint32_t jl = e >> 7, w = e & 127, i = w & 63;
    const size_t src = (static_cast<size_t>(s) * a.nt + t0 + (static_cast<int>(i) < nc ? i : 0)) * a.nv + vhead(jl);
    cp_async4(sbase + p1_rg(a.hpc) + e * 4, (w < 64 ? a.g : a.beta) + src, static_cast<int>(i) < nc ? 4u : 0u);
  }
  cp_async_commit();
  if (tid == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" :: "r"(mbar));
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" :: "r"(bar_ld));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    misc->failed = 0;
    constexpr int kBlocks = BF16IN ? 2 : 4;  // 128-byte column blocks of d_k: 64 bf16 or 32 f32
    mbar_expect_tx(bar_ld, kBlocks * 16384);
#pragma unroll
    for (int cb = 0; cb < kBlocks; ++cb) {
      tma_load_4d(sbase + P1_STACK + cb * 16384, &tm_k, (128 / kBlocks) * cb, static_cast<int>(kh),
                  static_cast<int>(t0), static_cast<int>(s), bar_ld);
      tma_load_4d(sbase + P1_STACK + cb * 16384 + 8192, &tm_q, (128 / kBlocks) * cb, static_cast<int>(kh),
                  static_cast<int>(t0), static_cast<int>(s), bar_ld);
    }
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(smem_addr(&misc->tmem_base)), "r"(64));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  __syncthreads();  // the load barrier is initialised before anyone waits on it
  const bool loaded = mbar_wait(bar_ld, 0);
  if (!loaded) misc->failed = 1;
  cp_async_wait_all();
  cta_sync();
  const uint32_t tmem = misc->tmem_base;

  if constexpr (BF16IN) {
    // Gram [K;Q] K^T -> TMEM: exact bf16 inputs, one product per K step
    if (tid == 0) {
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const uint64_t d = sdesc_sw128(sbase + P1_STACK + (ks >> 2) * 16384 + (ks & 3) * 32);
        mma_ss<true>(tmem, d, d, idesc_bf16(128, 64), ks > 0);
      }
      mma_commit(mbar);
    }
    // while it runs (by the first part): the stack as the workspace image,
    // and K^T (d_k rows x 64 tokens, bf16 canonical) from it
    if (store_k) {
#pragma unroll
      for (int it = 0; it < 8; ++it)
        __stcg(reinterpret_cast<uint4 *>(wk) + tid + NTH * it,
               reinterpret_cast<const uint4 *>(smem + P1_STACK)[tid + NTH * it]);
      unsigned char *wkb = reinterpret_cast<unsigned char *>(wk);
      for (int oc = tid; oc < 1024; oc += NTH) {  // d_k = oc % 128, tokens 8 (oc / 128) .. +7
        const int dk = oc & 127, i0 = (oc >> 7) * 8;
        const unsigned char *kb = smem + P1_STACK + (dk >> 6) * 16384 + (dk & 7) * 2;
        uint32_t e[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int i = i0 + u;
          e[u] = *reinterpret_cast<const uint16_t *>(kb + i * 128 + ((((dk & 63) >> 3) ^ (i & 7)) << 4));
        }
        __stcg(reinterpret_cast<uint4 *>(wkb + 32768 + canon16(dk, i0, 64)),
               make_uint4(e[0] | (e[1] << 16), e[2] | (e[3] << 16), e[4] | (e[5] << 16), e[6] | (e[7] << 16)));
      }
    }
  } else if constexpr (SPLIT) {
    // K^T (d_k rows x 64 tokens) as bf16 hi and lo canonical images, from
    // the f32 stack (by the first part)
    unsigned char *wkb = reinterpret_cast<unsigned char *>(wk);
    for (int oc = store_k ? tid : 1024; oc < 1024; oc += NTH) {  // d_k = oc % 128, tokens 8 (oc / 128) .. +7
      const int dk = oc & 127, i0 = (oc >> 7) * 8;
      const unsigned char *kb = smem + P1_STACK + (dk >> 5) * 16384 + (dk & 3) * 4;
      float e[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = i0 + u;
        e[u] = *reinterpret_cast<const float *>(kb + i * 128 + ((((dk & 31) >> 2) ^ (i & 7)) << 4));
      }
      uint4 h, l;
      split2(e[0], e[1], h.x, l.x); split2(e[2], e[3], h.y, l.y);
      split2(e[4], e[5], h.z, l.z); split2(e[6], e[7], h.w, l.w);
      __stcg(reinterpret_cast<uint4 *>(wkb + 65536 + canon16(dk, i0, 64)), h);
      __stcg(reinterpret_cast<uint4 *>(wkb + 81920 + canon16(dk, i0, 64)), l);
    }
    // The stack to bf16 hi and lo in place, 32 KB at a time: f32 column
    // blocks 2p and 2p+1 (d_k 64p .. 64p+63) become the hi block (128 rows x
    // 128 bytes, swizzled like the f32 ones) and the lo block after it.
    // Every thread reads its elements before any writes (the barrier), and
    // the first part stores the same bytes as the workspace image.
#pragma unroll 1
    for (int p = 0; p < 2; ++p) {
      unsigned char *reg = smem + P1_STACK + 32768 * p;
      uint2 hv[8], lv[8];
      uint32_t dst[8];
#pragma unroll
      for (int it = 0; it < 8; ++it) {
        const int f = tid + NTH * it;  // float4 of the region: block f >> 10, row (f >> 3) & 127, chunk f & 7
        const int rr = (f >> 3) & 127;
        const int dkb = 32 * (f >> 10) + 4 * ((f & 7) ^ (rr & 7));  // d_k - 64p of its first element
        const float4 x = reinterpret_cast<const float4 *>(reg)[f];
        split2(x.x, x.y, hv[it].x, lv[it].x);
        split2(x.z, x.w, hv[it].y, lv[it].y);
        dst[it] = static_cast<uint32_t>(rr * 128 + (((dkb >> 3) ^ (rr & 7)) << 4) + (dkb & 7) * 2);
      }
      __syncthreads();
#pragma unroll
      for (int it = 0; it < 8; ++it) {
        *reinterpret_cast<uint2 *>(reg + dst[it]) = hv[it];
        *reinterpret_cast<uint2 *>(reg + 16384 + dst[it]) = lv[it];
        if (store_k) {
          __stcg(reinterpret_cast<uint2 *>(wkb + 32768 * p + dst[it]), hv[it]);
          __stcg(reinterpret_cast<uint2 *>(wkb + 32768 * p + 16384 + dst[it]), lv[it]);
        }
      }
    }
    fence_async_smem();
    cta_sync();
    // Gram [K;Q] K^T -> TMEM (128 lanes x 64 columns), three bf16 terms per K step
    if (tid == 0) {
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const uint32_t ah = sbase + P1_STACK + (ks >> 2) * 32768 + (ks & 3) * 32;
        const uint64_t dh = sdesc_sw128(ah), dl = sdesc_sw128(ah + 16384);
        mma_ss<true>(tmem, dh, dh, idesc_bf16(128, 64), ks > 0);
        mma_ss<true>(tmem, dh, dl, idesc_bf16(128, 64), 1);
        mma_ss<true>(tmem, dl, dh, idesc_bf16(128, 64), 1);
      }
      mma_commit(mbar);
    }
  } else {
    // K and Q to TF32 (round to nearest) in place, stored as the [K; Q] image
    // (by the first part)
#pragma unroll
    for (int it = 0; it < 16; ++it) {
      float4 *p = reinterpret_cast<float4 *>(smem + P1_STACK) + tid + NTH * it;
      float4 x = *p;
      x.x = tf32_rn(x.x); x.y = tf32_rn(x.y); x.z = tf32_rn(x.z); x.w = tf32_rn(x.w);
      *p = x;
      if (store_k) __stcg(reinterpret_cast<float4 *>(wk) + tid + NTH * it, x);
    }
    fence_async_smem();
    cta_sync();

    // Gram [K;Q] K^T -> TMEM (128 lanes x 64 columns)
    if (tid == 0) {
#pragma unroll
      for (int ks = 0; ks < D / 8; ++ks) {
        const uint64_t d = sdesc_sw128(sbase + P1_STACK + (ks >> 2) * 16384 + (ks & 3) * 32);
        mma_ss(tmem, d, d, idesc_tf32(128, 64), ks > 0);
      }
      mma_commit(mbar);
    }
    // while the Gram runs, K^T (d_k rows x 64 tokens, canonical K-major image)
    // from the TF32 stack (by the first part)
    for (int oc = store_k ? tid : 2048; oc < 2048; oc += NTH) {  // d_k = oc % 128, tokens 4 (oc / 128) .. +3
      const int dk = oc & 127, i0 = (oc >> 7) * 4;
      const unsigned char *kb = smem + P1_STACK + (dk >> 5) * 16384 + (dk & 3) * 4;
      float e[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = i0 + u;
        e[u] = *reinterpret_cast<const float *>(kb + i * 128 + ((((dk & 31) >> 2) ^ (i & 7)) << 4));
      }
      __stcg(reinterpret_cast<float4 *>(wk + 16384 + canon(dk, i0, 64) / 4), make_float4(e[0], e[1], e[2], e[3]));
    }
  }
  // and every value head's per-token scalars, one warp per head
  for (uint32_t jl = static_cast<uint32_t>(warp); jl < nh; jl += NTH / 32) {
    float *scj = sc + jl * kScSet;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      scj[Q_GRAW * 64 + lane + 32 * h] = rg[jl * 128 + lane + 32 * h];
      scj[Q_BRAW * 64 + lane + 32 * h] = rg[jl * 128 + 64 + lane + 32 * h];
    }
    __syncwarp();
    float GC;
    const bool ex = chunk_scalars(scj, lane, &GC);
    if (lane == 0) extreme_of[jl] = ex;
  }
  if (!mbar_wait(mbar, 0)) misc->failed = 1;
  fence_after();
  cta_sync();  // the stack is dead: A, T and M may overlay it

  // A (plain, over the dead stack) and P' (straight to the workspace) of
  // value head j, from the Gram in TMEM and that head's gates
  auto epilogue = [&](uint32_t j) {
    const float *scj = sc + j * kScSet;
    const bool extreme = extreme_of[j] != 0;
    float *ws = a.ws + ((static_cast<size_t>(s) * a.nv + vhead(j)) * a.nchunks + ch) * kWsFloats;
    uint32_t gv[32];
    GDN_TMEM_LD32(tmem + lane_field + 32 * half, gv);
    tmem_wait_ld();
    const float *G = scj + Q_G * 64, *eG = scj + Q_EG * 64;
    if (row < 64) {
      const int r = row;
      const float br = scj[Q_BETA * 64 + r];
      const float Gr = DECAY_AFTER ? scj[Q_GPREV * 64 + r] : G[r];
      const float bgr = br * (DECAY_AFTER ? scj[Q_GAMP * 64 + r] : scj[Q_GAM * 64 + r]);
      // the branch on extreme (uniform) stays outside the loop, so that the
      // common case evaluates no exponential
      auto a_row = [&](auto gamf) {
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          float e[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int i = 32 * half + 4 * jj + u;
            e[u] = i < r ? gamf(i) * __uint_as_float(gv[4 * jj + u]) : 0.f;
          }
          *reinterpret_cast<float4 *>(sA + r * LD + 32 * half + 4 * jj) = make_float4(e[0], e[1], e[2], e[3]);
        }
      };
      if (extreme) a_row([&](int i) { return br * __expf(G[i] - Gr); });
      else a_row([&](int i) { return bgr * eG[i]; });
    } else {
      const int r = row - 64;
      const float Gr = G[r];
      const float qgr = a.q_scale * scj[Q_GAM * 64 + r];
      float *wp = ws + 4096;
      auto p_row = [&](auto gamf) {
        if constexpr (SPLIT) {
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            if (!tri16_used(r >> 3, 4 * half + jj)) continue;  // the rest of the image stays unwritten (zeros)
            float e[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const int i = 32 * half + 8 * jj + u;
              e[u] = i <= r ? gamf(i) * __uint_as_float(gv[8 * jj + u]) : 0.f;
            }
            uint4 h, l;
            split2(e[0], e[1], h.x, l.x); split2(e[2], e[3], h.y, l.y);
            split2(e[4], e[5], h.z, l.z); split2(e[6], e[7], h.w, l.w);
            unsigned char *wb = reinterpret_cast<unsigned char *>(wp) + canon16(r, 32 * half + 8 * jj, 64);
            *reinterpret_cast<uint4 *>(wb) = h;
            *reinterpret_cast<uint4 *>(wb + 8192) = l;
          }
        } else {
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) {
            float e[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int i = 32 * half + 4 * jj + u;
              e[u] = i <= r ? tf32_rn(gamf(i) * __uint_as_float(gv[4 * jj + u])) : 0.f;
            }
            if (tri_core_used(r >> 3, 8 * half + jj))  // the rest of the image stays unwritten (zeros)
              *reinterpret_cast<float4 *>(wp + canon(r, 32 * half + 4 * jj, 64) / 4) =
                  make_float4(e[0], e[1], e[2], e[3]);
          }
        }
      };
      if (extreme) p_row([&](int i) { return a.q_scale * __expf(G[i] - Gr); });
      else p_row([&](int i) { return qgr * eG[i]; });
    }
  };
  // T'' = T diag(beta) of value head j as canonical images (NaN if a wait
  // timed out)
  auto store_tpp = [&](uint32_t j) {
    const float nan = __int_as_float(0x7fc00000);
    const float *bet = sc + j * kScSet + Q_BETA * 64;
    const bool failed = misc->failed != 0;
    float *ws = a.ws + ((static_cast<size_t>(s) * a.nv + vhead(j)) * a.nchunks + ch) * kWsFloats;
    if constexpr (SPLIT) {
#pragma unroll
      for (int it = 0; it < 2; ++it) {
        const int ci = tid + NTH * it;  // 16-byte row ci & 7 of core ci >> 3 = (R, Kc)
        const int core = ci >> 3, r = (core >> 3) * 8 + (ci & 7), i0 = 8 * (core & 7);
        if (!tri16_used(core >> 3, core & 7)) continue;
        const float4 t0 = *reinterpret_cast<const float4 *>(sT + r * LD + i0);
        const float4 t1 = *reinterpret_cast<const float4 *>(sT + r * LD + i0 + 4);
        uint4 h, l;
        split2(t0.x * bet[i0], t0.y * bet[i0 + 1], h.x, l.x);
        split2(t0.z * bet[i0 + 2], t0.w * bet[i0 + 3], h.y, l.y);
        split2(t1.x * bet[i0 + 4], t1.y * bet[i0 + 5], h.z, l.z);
        split2(t1.z * bet[i0 + 6], t1.w * bet[i0 + 7], h.w, l.w);
        if (failed) { h = make_uint4(0x7fc07fc0u, 0x7fc07fc0u, 0x7fc07fc0u, 0x7fc07fc0u); l = h; }
        reinterpret_cast<uint4 *>(ws)[ci] = h;
        reinterpret_cast<uint4 *>(ws + 2048)[ci] = l;
      }
    } else {
#pragma unroll
      for (int it = 0; it < 4; ++it) {
        const int ci = tid + NTH * it;
        const int core = ci >> 3, r = (core >> 4) * 8 + (ci & 7), i0 = 4 * (core & 15);
        float4 t = *reinterpret_cast<const float4 *>(sT + r * LD + i0);
        t = make_float4(tf32_rn(t.x * bet[i0]), tf32_rn(t.y * bet[i0 + 1]), tf32_rn(t.z * bet[i0 + 2]),
                        tf32_rn(t.w * bet[i0 + 3]));
        if (failed) t = make_float4(nan, nan, nan, nan);
        if (tri_core_used(core >> 4, core & 15)) reinterpret_cast<float4 *>(ws)[ci] = t;
      }
    }
  };

  // per value head: T = (I + A)^-1, then its T'' is stored while the next
  // head's A and P' are formed (different buffers)
  epilogue(0);
  cta_sync();
  for (uint32_t jl = 0; jl < nh; ++jl) {
    tri_inverse(sA, sT, sM, tid);  // ends with a barrier: A is consumed
    store_tpp(jl);
    if (jl + 1 < nh) epilogue(jl + 1);
    cta_sync();
  }
  // a load that timed out may still land: wait for it (bounded) before exit
  if (tid == 0 && !loaded) (void)mbar_wait(bar_ld, 0);
  if (tid == 0 && misc->failed) report_wait_timeout();
  cta_sync();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(tmem), "r"(64));
}

// ================================================================ pass 2

// TMEM columns: the state, U^T, W (then U~^T), and [X | Z -> Y^T] in two
// regions that alternate by chunk, so a chunk's outputs are read out while
// the next chunk's products run.  With split-bf16 operands every A operand
// is a hi and a lo half of packed bf16 pairs: S~ as hi over W's columns and
// lo over U's at the chunk start, W as hi | lo (32 columns each) in W's,
// U^T as hi | lo over X (dead once W is formed) and U~^T as hi | lo in W's.
constexpr uint32_t P2_TM_S = 0, P2_TM_XY0 = 128, P2_TM_U = 256, P2_TM_W = 320, P2_TM_XY1 = 384;
constexpr uint32_t P2_TM_COLS = 512;

// Shared memory (bytes from a 1024-aligned base).  The [K; Q] image is the
// swizzled stack pass 1 stored (column block cb = 16 KB: K's 64 rows, then
// Q's), one 128-row K-major SWIZZLE_128B operand.
constexpr uint32_t P2_KQ = 0;                 // [K; Q] image (bulk copy)
constexpr uint32_t P2_KT = P2_KQ + 65536;     // K^T image (bulk copy), 128 x 64 canonical
constexpr uint32_t P2_TPP = P2_KT + 32768;    // T'' image (bulk copy)
constexpr uint32_t P2_P = P2_TPP + 16384;     // P' image (bulk copy)
constexpr uint32_t P2_VS = P2_P + 16384;      // V rows (TMA), 64 x 128 natural
constexpr uint32_t P2_SC = P2_VS + 32768;     // per-token scalars
constexpr uint32_t P2_MISC = P2_SC + Q_NSC * 64 * 4;
constexpr uint32_t P2_SMEM = P2_MISC + 128 + 1024;  // + room to align the base to 1024
static_assert(P2_SMEM <= 232448, "pass-2 shared memory");
constexpr uint32_t kImgBytes = 16384;   // one 64 x 64 workspace image

struct StateArgs {
  const float *__restrict__ g;
  const float *__restrict__ beta;
  const float *state_in;
  const float *__restrict__ ws;    // per (head, chunk) images
  const float *__restrict__ ws_k;  // per (seq, key head, chunk) images
  void *__restrict__ output;  // f32, or bf16 with bf16 activations
  float *state_out;
  uint32_t nk, nv, nt, group, khead_div, nchunks;
  float q_scale;
  // the chain of each (seq, value head) runs as segments of seg_len chunks,
  // one launch per group of segments: CTA b of the launch takes segment
  // (seg_base + b) / heads of head (seg_base + b) % heads
  uint32_t heads, seg_len, seg_base;
};

struct P2Misc {
  unsigned long long mbar_xy;  // [X | Z] MMA commit
  unsigned long long mbar1;    // U^T MMA commit
  unsigned long long mbar2;    // batch-2 MMA commit
  unsigned long long mbar2s;   // split operands: batch 2's state update (issued first) done
  unsigned long long bar_kq;   // bulk copy: the [K; Q] image of a chunk
  unsigned long long bar_kt;   // bulk copy: the K^T image of a chunk
  unsigned long long bar_t;    // bulk copy: the T'' image of a chunk
  unsigned long long bar_v;    // TMA: V rows of a chunk
  unsigned long long bar_p;    // bulk copy: the P' image of a chunk
  uint32_t tmem_base;
  int failed;
  float c_renorm, c_fold, c_next;
  int do_renorm, do_fold;
};
static_assert(sizeof(P2Misc) <= 128, "pass-2 misc area");

// An output value from its f32 bits: f32, or rounded to bf16 (nearest even).
template <bool BF16>
__device__ __forceinline__ typename std::conditional<BF16, uint16_t, float>::type to_out(uint32_t bits) {
  if constexpr (BF16) return __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(bits)));
  else return __uint_as_float(bits);
}

// One warp: a chunk's raw g and beta into the scalar area by 4-byte
// asynchronous copies; tokens past the chunk's end read as zero.
__device__ __forceinline__ void stage_gates_warp(uint32_t sc_addr, const float *g, const float *beta, size_t sc0,
                                                 size_t nv, int nc, int lane) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int i = lane + 32 * h;
    const size_t src = sc0 + static_cast<size_t>(i < nc ? i : 0) * nv;
    const uint32_t n = i < nc ? 4u : 0u;
    cp_async4(sc_addr + (Q_GRAW * 64 + i) * 4, g + src, n);
    cp_async4(sc_addr + (Q_BRAW * 64 + i) * 4, beta + src, n);
  }
}

// One warp, once the chunk's raw gates have landed: the per-token scalars,
// the lazy-scale bookkeeping of the chunk (S = c * TMEM S enters with scale
// c) and the column scales of W, U~ and Z (below).  Returns the scale the
// chunk hands on.
template <bool DECAY_AFTER>
__device__ __forceinline__ float p2_chunk_setup(float *sc, P2Misc *misc, float c, float q_scale, int lane) {
  float GC;
  const bool extreme = chunk_scalars(sc, lane, &GC);
  float cc = c, renorm = 1.f;
  const bool do_renorm = cc < kRenormLo || cc > kRenormHi;
  if (do_renorm) { renorm = cc; cc = 1.f; }
  const float gamC = __expf(-GC);
  float cnext, fold = 1.f;
  if (extreme) { fold = cc * gamC; cnext = 1.f; }
  else { cnext = cc * gamC; }
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int i = lane + 32 * h;
    const float Gi = sc[Q_G * 64 + i];
    sc[Q_KTS * 64 + i] = __expf(Gi - GC) / cnext;                                      // U~ column
    sc[Q_WS * 64 + i] = cc * (DECAY_AFTER ? sc[Q_GAMP * 64 + i] : sc[Q_GAM * 64 + i]);  // W column
    sc[Q_QS * 64 + i] = cc * q_scale * sc[Q_GAM * 64 + i];                             // Z column
  }
  if (lane == 0) {
    misc->c_renorm = renorm; misc->c_fold = fold; misc->c_next = cnext;
    misc->do_renorm = do_renorm; misc->do_fold = extreme;
  }
  return cnext;
}

// The state pass: one CTA per (seq, value head) over all chunks, the state
// in TMEM as S = c * S~.  Per chunk, with everything state-free read from
// the workspace:
//   [X | Z] = S~ [K; Q]^T                 (one N = 128 product)
//   W  = V^T - X diag(c gamma)            (TMEM pass; gamma' with decay-after)
//   U^T = W T''^T                         (T'' = T diag(beta), so this is
//                                          V^T T''^T + X (-T')^T of the chunk
//                                          equations, -T' = -c T diag(beta gamma))
//   Y^T = Z diag(c q_scale gamma) + U^T P'^T
//   S~ <- S~ + U~^T K^T,  U~ = U diag(e^(G_i - G_C) / c_next)
// The serial chain is [X | Z] -> W -> U^T -> rounding -> batch 2; the
// outputs, Z's scaling and the next chunk's V come in beside it.  Thread 32
// issues the MMAs, thread 0 the copies, warp 2 sets up the next chunk's
// scalars while batch 2 runs.  Waits are bounded.
// BF16IN: bf16 activations (with SPLIT): hi-only [K; Q] and K^T images,
// [X | Z] and the state update two products per K step (the terms with a
// zero lo half left out), V rows as bf16, y rounded to bf16 when stored.
template <bool DECAY_AFTER, bool SPLIT, bool BF16IN>
__global__ void __launch_bounds__(NTH, 1)
    gdn_chunk_state_kernel(const StateArgs a, const __grid_constant__ CUtensorMap tm_v) {
  static_assert(SPLIT || !BF16IN, "bf16 activations take split operands");
  using Out = typename std::conditional<BF16IN, uint16_t, float>::type;
  constexpr uint32_t kKqBytes = BF16IN ? 32768 : 65536;   // the [K; Q] image
  constexpr uint32_t kKtBytes = BF16IN ? 16384 : 32768;   // the K^T image
  constexpr uint32_t kKtOff = BF16IN ? 8192 : 16384;      // K^T in the key-head slot (floats)
  constexpr uint32_t kVBytes = BF16IN ? 16384 : 32768;    // a chunk's V rows
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // operate from a 1024-byte aligned base (the swizzled image needs it)
  const uint32_t raw_addr = smem_addr(smem_raw);
  const uint32_t pad = ((raw_addr + 1023u) & ~1023u) - raw_addr;
  unsigned char *smem = smem_raw + pad;
  float *sc = reinterpret_cast<float *>(smem + P2_SC);
  const float *sVS = reinterpret_cast<const float *>(smem + P2_VS);
  P2Misc *misc = reinterpret_cast<P2Misc *>(smem + P2_MISC);
  const uint32_t sbase = raw_addr + pad;
  const uint32_t mbar_xy = smem_addr(&misc->mbar_xy), mbar1 = smem_addr(&misc->mbar1),
                 mbar2 = smem_addr(&misc->mbar2), mbar2s = smem_addr(&misc->mbar2s);
  const uint32_t bar_kq = smem_addr(&misc->bar_kq), bar_kt = smem_addr(&misc->bar_kt),
                 bar_t = smem_addr(&misc->bar_t), bar_v = smem_addr(&misc->bar_v), bar_p = smem_addr(&misc->bar_p);

  const int tid = static_cast<int>(threadIdx.x);
  const int warp = tid >> 5, lane = tid & 31;
  const int row = tid & 127;
  const int half = tid >> 7;
  const uint32_t lane_field = static_cast<uint32_t>(32 * (warp & 3)) << 16;
  constexpr int ISSUER = 32;  // thread that issues (and commits) every MMA

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
  const size_t v_tok = static_cast<size_t>(a.nv) * D;
  const float *wseq = a.ws + (static_cast<size_t>(head) * a.nchunks + cb) * kWsFloats;
  const float *wkseq = a.ws_k + ((static_cast<size_t>(s) * a.nk + kh) * a.nchunks + cb) * kWsKFloats;
  const size_t sc_first = (static_cast<size_t>(s) * a.nt + tb) * a.nv + vh;
  // the state enters from state_in, or, after an earlier segment, from
  // state_out, where that segment left it (an earlier launch)
  const float *state_src = seg == 0 ? a.state_in : a.state_out;

  if (tid == 0) {
    const uint32_t bars[9] = {mbar_xy, mbar1, mbar2, mbar2s, bar_kq, bar_kt, bar_t, bar_v, bar_p};
#pragma unroll
    for (int b = 0; b < 9; ++b) asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" :: "r"(bars[b]));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    misc->failed = 0;
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(smem_addr(&misc->tmem_base)), "r"(P2_TM_COLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  // the T'' and P' buffers (adjacent): zeros where the copies write nothing
  for (int i = tid; i < 2 * static_cast<int>(kImgBytes) / 16; i += NTH)
    reinterpret_cast<float4 *>(smem + P2_TPP)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  fence_async_smem();
  __syncthreads();  // barriers initialised and buffers zeroed before anyone uses them
  // chunk 0's inputs start arriving while the state is loaded
  if (tid == 0) {
    mbar_expect_tx(bar_kq, kKqBytes);
    bulk_load(sbase + P2_KQ, wkseq, kKqBytes, bar_kq);
    mbar_expect_tx(bar_kt, kKtBytes);
    bulk_load(sbase + P2_KT, wkseq + kKtOff, kKtBytes, bar_kt);
    load_image<SPLIT>(sbase + P2_TPP, wseq, bar_t);
    load_image<SPLIT>(sbase + P2_P, wseq + 4096, bar_p);
    mbar_expect_tx(bar_v, kVBytes);
    tma_load_4d(sbase + P2_VS, &tm_v, 0, static_cast<int>(vh), static_cast<int>(tb), static_cast<int>(s), bar_v);
  }
  // copies armed and MMA batches committed per barrier (uniform over the
  // CTA), for the bounded waits at exit
  uint32_t n_ld = 1, n_v = 1, n_mma = 0;
  float c_carry = 1.f;  // warp 2: the scale the next chunk starts with
  if (warp == 2) {
    stage_gates_warp(sbase + P2_SC, a.g, a.beta, sc_first, a.nv, static_cast<int>(min(nt, static_cast<uint32_t>(C))),
                     lane);
    cp_async_commit();
    cp_async_wait_all();
    __syncwarp();
    c_carry = p2_chunk_setup<DECAY_AFTER>(sc, misc, 1.f, a.q_scale, lane);
    __syncwarp();  // every lane is done with the raw gates
    if (nchunks > 1) {
      stage_gates_warp(sbase + P2_SC, a.g, a.beta, sc_first + static_cast<size_t>(C) * a.nv, a.nv,
                       static_cast<int>(min(nt - C, static_cast<uint32_t>(C))), lane);
      cp_async_commit();
    }
  }
  cta_sync();
  const uint32_t tmem = misc->tmem_base;
  const uint32_t tl = tmem + lane_field;
  // split operands: S~ as the A operand hi (over W's columns) and lo (over
  // U's) from the state in TMEM; this thread's row, its 64 columns
  auto split_state = [&]() {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t v[32], sh[16], sl[16];
      GDN_TMEM_LD32(tl + P2_TM_S + 64 * half + 32 * h, v);
      tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < 16; ++j) split2(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]), sh[j], sl[j]);
      GDN_TMEM_ST16(tl + P2_TM_W + 32 * half + 16 * h, sh);
      GDN_TMEM_ST16(tl + P2_TM_U + 32 * half + 16 * h, sl);
    }
  };

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
      GDN_TMEM_ST32(tl + P2_TM_S + 64 * half + 32 * h, v);
      if constexpr (SPLIT) {  // chunk 0's A operand S~ = S
        uint32_t sh[16], sl[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) split2(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]), sh[j], sl[j]);
        GDN_TMEM_ST16(tl + P2_TM_W + 32 * half + 16 * h, sh);
        GDN_TMEM_ST16(tl + P2_TM_U + 32 * half + 16 * h, sl);
      }
    }
    tmem_wait_st();
  }
  // This thread's V^T values of a chunk: row d_v, tokens 32*half .. +31.
  float vr[32];
  if (!mbar_wait(bar_v, 0)) misc->failed = 1;
#pragma unroll
  for (int j = 0; j < 32; ++j)
    vr[j] = BF16IN ? __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t *>(sVS)[(32 * half + j) * D + row]) << 16)
                   : sVS[(32 * half + j) * D + row];

  bool failed = false;
  for (uint32_t ch = 0; ch < nchunks; ++ch) {
    const uint32_t t0 = ch * C;
    const bool more = ch + 1 < nchunks;
    const uint32_t par = ch & 1;                         // phase parity of this chunk's barriers
    const uint32_t tm_x = par ? P2_TM_XY1 : P2_TM_XY0;  // X; Z -> Y^T at tm_x + 64
    const uint32_t tm_y = tm_x + 64;

    // ---- 0. the previous chunk's batch 2 is done (thread 0 waited), this
    // chunk's scalars are set and its V is in registers
    cta_sync();
    if (misc->failed) { failed = true; break; }
    if (misc->do_renorm) {  // c left [2^-30, 2^30]: fold it into S (rare)
      if (ch > 0 && !mbar_wait(mbar2, par ^ 1)) misc->failed = 1;
      __syncwarp();
      fence_after();
      tmem_scale64(tl + P2_TM_S + 64 * half, misc->c_renorm);
      if constexpr (SPLIT) {  // and the A operand again from the folded state
        split_state();
        tmem_wait_st();
      }
      cta_sync();
    }
    if (tid == 0 && more) {  // V rows are free: the next chunk's
      fence_async_smem();
      mbar_expect_tx(bar_v, kVBytes);
      tma_load_4d(sbase + P2_VS, &tm_v, 0, static_cast<int>(vh), static_cast<int>(tb + t0 + C), static_cast<int>(s),
                  bar_v);
    }

    // ---- 1. [X | Z] = S~ [K; Q]^T
    if (tid == ISSUER) {
      if (!mbar_wait(bar_kq, par)) misc->failed = 1;
      if constexpr (BF16IN) {
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint64_t bh = sdesc_sw128(sbase + P2_KQ + (ks >> 2) * 16384 + (ks & 3) * 32);
          mma_ts<true>(tmem + tm_x, tmem + P2_TM_W + 8 * ks, bh, idesc_bf16(128, 128), ks > 0);
          mma_ts<true>(tmem + tm_x, tmem + P2_TM_U + 8 * ks, bh, idesc_bf16(128, 128), 1);
        }
      } else if constexpr (SPLIT) {
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t b = sbase + P2_KQ + (ks >> 2) * 32768 + (ks & 3) * 32;
          const uint64_t bh = sdesc_sw128(b), bl = sdesc_sw128(b + 16384);
          mma_ts<true>(tmem + tm_x, tmem + P2_TM_W + 8 * ks, bh, idesc_bf16(128, 128), ks > 0);
          mma_ts<true>(tmem + tm_x, tmem + P2_TM_W + 8 * ks, bl, idesc_bf16(128, 128), 1);
          mma_ts<true>(tmem + tm_x, tmem + P2_TM_U + 8 * ks, bh, idesc_bf16(128, 128), 1);
        }
      } else {
#pragma unroll
        for (int ks = 0; ks < D / 8; ++ks)
          mma_ts(tmem + tm_x, tmem + P2_TM_S + 8 * ks,
                 sdesc_sw128(sbase + P2_KQ + (ks >> 2) * 16384 + (ks & 3) * 32), idesc_tf32(128, 128), ks > 0);
      }
      mma_commit(mbar_xy);
    }
    // meanwhile warps 4-7: the previous chunk's outputs (every chunk but the
    // last is full)
    if (warp >= 4 && ch > 0) {
      if (!mbar_wait(mbar2, par ^ 1)) misc->failed = 1;
      __syncwarp();
      fence_after();
      const uint32_t tm_yp = (par ? P2_TM_XY0 : P2_TM_XY1) + 64;
      Out *obase = static_cast<Out *>(a.output) + ((static_cast<size_t>(s) * a.nt + tb + (t0 - C)) * a.nv + vh) * D + row;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t yv[32];
        GDN_TMEM_LD32(tl + tm_yp + 32 * h, yv);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j) obase[static_cast<size_t>(32 * h + j) * v_tok] = to_out<BF16IN>(yv[j]);
      }
    }

    // ---- 2. W = V^T - X diag(c gamma), as an A operand, into TMEM
    if (!mbar_wait(mbar_xy, par)) misc->failed = 1;
    __syncwarp();
    fence_after();
    {
      const float *wsc = sc + Q_WS * 64 + 32 * half;
      uint32_t xv[32];
      GDN_TMEM_LD32(tl + tm_x + 32 * half, xv);
      tmem_wait_ld();
      if constexpr (SPLIT) {
        uint32_t wh[16], wl[16];
#pragma unroll
        for (int j = 0; j < 16; ++j)
          split2(fmaf(-wsc[2 * j], __uint_as_float(xv[2 * j]), vr[2 * j]),
                 fmaf(-wsc[2 * j + 1], __uint_as_float(xv[2 * j + 1]), vr[2 * j + 1]), wh[j], wl[j]);
        GDN_TMEM_ST16(tl + P2_TM_W + 16 * half, wh);
        GDN_TMEM_ST16(tl + P2_TM_W + 32 + 16 * half, wl);
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          xv[j] = __float_as_uint(tf32_rn(fmaf(-wsc[j], __uint_as_float(xv[j]), vr[j])));
        GDN_TMEM_ST32(tl + P2_TM_W + 32 * half, xv);
      }
      tmem_wait_st();
    }
    cta_sync();

    // ---- 3. U^T = W T''^T; [K; Q] is free for the next chunk's
    if (tid == 0 && more) {
      mbar_expect_tx(bar_kq, kKqBytes);
      bulk_load(sbase + P2_KQ, wkseq + static_cast<size_t>(ch + 1) * kWsKFloats, kKqBytes, bar_kq);
    }
    if (tid == ISSUER) {
      if (!mbar_wait(bar_t, par)) misc->failed = 1;
      if constexpr (SPLIT) {
#pragma unroll
        for (int ks = 0; ks < C / 16; ++ks) {
          const uint64_t bh = sdesc(sbase + P2_TPP + ks * 256, 1024), bl = sdesc(sbase + P2_TPP + 8192 + ks * 256, 1024);
          mma_ts<true>(tmem + P2_TM_U, tmem + P2_TM_W + 8 * ks, bh, idesc_bf16(128, 64), ks > 0);
          mma_ts<true>(tmem + P2_TM_U, tmem + P2_TM_W + 8 * ks, bl, idesc_bf16(128, 64), 1);
          mma_ts<true>(tmem + P2_TM_U, tmem + P2_TM_W + 32 + 8 * ks, bh, idesc_bf16(128, 64), 1);
        }
      } else {
#pragma unroll
        for (int ks = 0; ks < C / 8; ++ks)
          mma_ts(tmem + P2_TM_U, tmem + P2_TM_W + 8 * ks, sdesc(sbase + P2_TPP + ks * 256, 2048),
                 idesc_tf32(128, 64), ks > 0);
      }
      mma_commit(mbar1);
    }
    // meanwhile warps 4-7: Y^T = Z diag(c q_scale gamma)
    __syncwarp();
    if (warp >= 4) {
      const float *qs = sc + Q_QS * 64;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t zv[32];
        GDN_TMEM_LD32(tl + tm_y + 32 * h, zv);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j) zv[j] = __float_as_uint(__uint_as_float(zv[j]) * qs[32 * h + j]);
        GDN_TMEM_ST32(tl + tm_y + 32 * h, zv);
      }
      tmem_wait_st();
    }

    // ---- 4. U^T and U~^T as A operands: TF32 (nearest) in place and over W,
    // or split over X and W; extreme gates: decay S now
    if (!mbar_wait(mbar1, par)) misc->failed = 1;
    __syncwarp();
    fence_after();
    {
      const float *kts = sc + Q_KTS * 64 + 32 * half;
      uint32_t uv[32];
      GDN_TMEM_LD32(tl + P2_TM_U + 32 * half, uv);
      tmem_wait_ld();
      if constexpr (SPLIT) {
        uint32_t uh[16], ul[16], th[16], tlo[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float u0 = __uint_as_float(uv[2 * j]), u1 = __uint_as_float(uv[2 * j + 1]);
          split2(u0, u1, uh[j], ul[j]);
          split2(u0 * kts[2 * j], u1 * kts[2 * j + 1], th[j], tlo[j]);
        }
        GDN_TMEM_ST16(tl + tm_x + 16 * half, uh);
        GDN_TMEM_ST16(tl + tm_x + 32 + 16 * half, ul);
        GDN_TMEM_ST16(tl + P2_TM_W + 16 * half, th);
        GDN_TMEM_ST16(tl + P2_TM_W + 32 + 16 * half, tlo);
      } else {
        uint32_t us[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float u = __uint_as_float(uv[j]);
          uv[j] = __float_as_uint(tf32_rn(u));
          us[j] = __float_as_uint(tf32_rn(u * kts[j]));
        }
        GDN_TMEM_ST32(tl + P2_TM_U + 32 * half, uv);
        GDN_TMEM_ST32(tl + P2_TM_W + 32 * half, us);
      }
      tmem_wait_st();
    }
    if (misc->do_fold) tmem_scale64(tl + P2_TM_S + 64 * half, misc->c_fold);
    cta_sync();

    // ---- 5. batch 2: Yt += Ut P'^T; S~ += U~t K^T.  Meanwhile warp 2 sets up
    // the next chunk's scalars and every thread takes the next chunk's V.
    if (tid == 0 && more) {  // U^T is done: T'' is free
      load_image<SPLIT>(sbase + P2_TPP, wseq + static_cast<size_t>(ch + 1) * kWsFloats, bar_t);
    }
    if (tid == ISSUER) {
      if (!mbar_wait(bar_p, par)) misc->failed = 1;
      if (!mbar_wait(bar_kt, par)) misc->failed = 1;
      if constexpr (SPLIT) {
        // the state update first, on its own barrier, so that the next
        // chunk's S~ split runs beside the output product
#pragma unroll
        for (int ks = 0; ks < C / 16; ++ks) {
          const uint64_t bh = sdesc(sbase + P2_KT + ks * 256, 1024), bl = sdesc(sbase + P2_KT + 16384 + ks * 256, 1024);
          mma_ts<true>(tmem + P2_TM_S, tmem + P2_TM_W + 8 * ks, bh, idesc_bf16(128, 128), 1);
          if constexpr (!BF16IN) mma_ts<true>(tmem + P2_TM_S, tmem + P2_TM_W + 8 * ks, bl, idesc_bf16(128, 128), 1);
          mma_ts<true>(tmem + P2_TM_S, tmem + P2_TM_W + 32 + 8 * ks, bh, idesc_bf16(128, 128), 1);
        }
        mma_commit(mbar2s);
#pragma unroll
        for (int ks = 0; ks < C / 16; ++ks) {
          const uint64_t bh = sdesc(sbase + P2_P + ks * 256, 1024), bl = sdesc(sbase + P2_P + 8192 + ks * 256, 1024);
          mma_ts<true>(tmem + tm_y, tmem + tm_x + 8 * ks, bh, idesc_bf16(128, 64), 1);
          mma_ts<true>(tmem + tm_y, tmem + tm_x + 8 * ks, bl, idesc_bf16(128, 64), 1);
          mma_ts<true>(tmem + tm_y, tmem + tm_x + 32 + 8 * ks, bh, idesc_bf16(128, 64), 1);
        }
      } else {
#pragma unroll
        for (int ks = 0; ks < C / 8; ++ks)
          mma_ts(tmem + tm_y, tmem + P2_TM_U + 8 * ks, sdesc(sbase + P2_P + ks * 256, 2048), idesc_tf32(128, 64),
                 1);
#pragma unroll
        for (int ks = 0; ks < C / 8; ++ks)
          mma_ts(tmem + P2_TM_S, tmem + P2_TM_W + 8 * ks, sdesc(sbase + P2_KT + ks * 256, 2048),
                 idesc_tf32(128, 128), 1);
      }
      mma_commit(mbar2);
    }
    ++n_mma;
    if (more) {
      if (warp == 2) {
        cp_async_wait_all();
        __syncwarp();
        c_carry = p2_chunk_setup<DECAY_AFTER>(sc, misc, c_carry, a.q_scale, lane);
        __syncwarp();
        if (ch + 2 < nchunks) {
          stage_gates_warp(sbase + P2_SC, a.g, a.beta, sc_first + static_cast<size_t>(t0 + 2 * C) * a.nv, a.nv,
                           static_cast<int>(min(nt - t0 - 2 * C, static_cast<uint32_t>(C))), lane);
          cp_async_commit();
        }
      }
      if (!mbar_wait(bar_v, par ^ 1)) misc->failed = 1;
#pragma unroll
      for (int j = 0; j < 32; ++j)
        vr[j] = BF16IN ? __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t *>(sVS)[(32 * half + j) * D + row]) << 16)
                       : sVS[(32 * half + j) * D + row];
      if constexpr (SPLIT) {  // the next chunk's A operand S~ = hi + lo, once the update is done
        if (!mbar_wait(mbar2s, par)) misc->failed = 1;
        __syncwarp();
        fence_after();
        split_state();
        tmem_wait_st();
      }
    }
    if (tid == 0) {  // batch 2 done: P' and K^T are free for the next chunk's
      if (!mbar_wait(mbar2, par)) misc->failed = 1;
      if (more) {
        load_image<SPLIT>(sbase + P2_P, wseq + static_cast<size_t>(ch + 1) * kWsFloats + 4096, bar_p);
        mbar_expect_tx(bar_kt, kKtBytes);
        bulk_load(sbase + P2_KT, wkseq + static_cast<size_t>(ch + 1) * kWsKFloats + kKtOff, kKtBytes, bar_kt);
      }
    }
    if (more) { ++n_ld; ++n_v; }
  }

  // ---- the last chunk's outputs
  cta_sync();
  if (!failed && !misc->failed) {
    const uint32_t cl = nchunks - 1;
    if (!mbar_wait(mbar2, cl & 1)) misc->failed = 1;
    __syncwarp();
    fence_after();
    const uint32_t tm_yl = ((cl & 1) ? P2_TM_XY1 : P2_TM_XY0) + 64;
    const int ncl = static_cast<int>(nt - cl * C);
    uint32_t yv[32];
    GDN_TMEM_LD32(tl + tm_yl + 32 * half, yv);
    tmem_wait_ld();
    Out *obase = static_cast<Out *>(a.output) + ((static_cast<size_t>(s) * a.nt + tb + cl * C) * a.nv + vh) * D + row;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const int i = 32 * half + j;
      if (i < ncl) obase[static_cast<size_t>(i) * v_tok] = to_out<BF16IN>(yv[j]);
    }
  }

  // Nothing may still be in flight when TMEM is read or released or the
  // CTA's shared memory is freed: after a failure, wait (bounded) for the
  // last MMA batch and the last copy on every barrier.
  cp_async_wait_all();
  if (tid == 0) {
    if (n_mma > 0) {  // every chunk commits once on each MMA barrier
      (void)mbar_wait(mbar_xy, (n_mma - 1) & 1);
      (void)mbar_wait(mbar1, (n_mma - 1) & 1);
      (void)mbar_wait(mbar2, (n_mma - 1) & 1);
      if (SPLIT) (void)mbar_wait(mbar2s, (n_mma - 1) & 1);
    }
    const uint32_t pl = (n_ld - 1) & 1;  // every image barrier is armed once per chunk
    (void)mbar_wait(bar_kq, pl);
    (void)mbar_wait(bar_kt, pl);
    (void)mbar_wait(bar_t, pl);
    (void)mbar_wait(bar_p, pl);
    (void)mbar_wait(bar_v, (n_v - 1) & 1);
  }
  fence_before();
  __syncthreads();
  fence_after();
  failed = failed || misc->failed != 0;
  if (failed && tid == 0) report_wait_timeout();

  // ---- state_out = c * S~ (or NaN if a wait timed out)
  {
    const float f = failed ? __int_as_float(0x7fc00000) : misc->c_next;
    float4 *dst = reinterpret_cast<float4 *>(a.state_out + state_head + row * D + 64 * half);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t v[32];
      GDN_TMEM_LD32(tl + P2_TM_S + 64 * half + 32 * h, v);
      tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < 8; ++j)
        __stcs(dst + 8 * h + j, make_float4(__uint_as_float(v[4 * j]) * f, __uint_as_float(v[4 * j + 1]) * f,
                                            __uint_as_float(v[4 * j + 2]) * f, __uint_as_float(v[4 * j + 3]) * f));
    }
  }
  cta_sync();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(tmem), "r"(P2_TM_COLS));
}

// cuTensorMapEncodeTiled from the driver, looked up once through the runtime.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// A [128, heads, n_tokens, n_seqs] f32 (or bf16) tensor (128 contiguous) as a
// 4-D map whose box is `inner` elements x 1 head x 64 tokens x 1 seq.
cudaError_t rows_map(CUtensorMap *tm, const void *base, uint32_t heads, uint32_t nt, uint32_t ns,
                     uint32_t inner, CUtensorMapSwizzle swizzle, bool bf16 = false) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (enc == nullptr) return cudaErrorNotSupported;
  const cuuint64_t row = bf16 ? 256 : 512;  // bytes of one 128-element row
  const cuuint64_t dims[4] = {128, heads, nt, ns};
  const cuuint64_t strides[3] = {row, row * heads, row * heads * nt};
  const cuuint32_t box[4] = {inner, 1, 64, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = enc(tm, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4,
                         const_cast<void *>(base), dims, strides, box,
                         estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <bool DA, bool SPLIT, bool BF16IN>
cudaError_t launch_split(const Problem &p, float *ws, cudaStream_t stream) {
  const uint32_t nchunks = (p.nt + C - 1) / C;
  const unsigned long long heads = static_cast<unsigned long long>(p.nv) * p.ns;
  if (heads == 0 || heads * nchunks > 0x7fffffffull) return cudaErrorInvalidConfiguration;
  const uint32_t group = p.nv / p.nk;
  // one CTA per (seq, chunk, key head) takes all its value heads, unless
  // there are fewer of those than SMs: then the value heads are split into
  // parts, one CTA each (measured: one sequence of 256 tokens 43.3 -> 38.8
  // us; splitting already at 1024 tokens cost more in repeated K, Q and Gram
  // work than it gained)
  const unsigned long long tasks = static_cast<unsigned long long>(p.nk) * p.ns * nchunks;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const unsigned long long want = static_cast<unsigned long long>(sms > 0 ? sms : 1);
  uint32_t parts = tasks >= want ? 1u : static_cast<uint32_t>(min(static_cast<unsigned long long>(group),
                                                                   (want + tasks - 1) / tasks));
  const uint32_t hpc = (group + parts - 1) / parts;
  parts = (group + hpc - 1) / hpc;
  const unsigned long long prep_blocks = tasks * parts;
  if (p1_smem(hpc) > 232448u) return cudaErrorInvalidConfiguration;  // raw gates of the heads in a CTA
  if (reinterpret_cast<uintptr_t>(p.v) % 16 != 0) return cudaErrorMisalignedAddress;  // TMA source
  CUtensorMap tm_k, tm_q, tm_v;
  // K and Q boxes: 128-byte rows (32 f32 or 64 bf16), swizzled like the MMA's operand
  const uint32_t kq_inner = BF16IN ? 64 : 32;
  e = rows_map(&tm_k, p.k, p.nk, p.nt, p.ns, kq_inner, CU_TENSOR_MAP_SWIZZLE_128B, BF16IN);
  if (e == cudaSuccess) e = rows_map(&tm_q, p.q, p.nk, p.nt, p.ns, kq_inner, CU_TENSOR_MAP_SWIZZLE_128B, BF16IN);
  if (e == cudaSuccess) e = rows_map(&tm_v, p.v, p.nv, p.nt, p.ns, 128, CU_TENSOR_MAP_SWIZZLE_NONE, BF16IN);
  if (e != cudaSuccess) return e;

  float *ws_k = ws + static_cast<size_t>(p.nv) * p.ns * nchunks * kWsFloats;
  PrepArgs pa;
  pa.q = static_cast<const float *>(p.q); pa.k = static_cast<const float *>(p.k);
  pa.g = p.g; pa.beta = p.beta; pa.ws = ws; pa.ws_k = ws_k;
  pa.nk = p.nk; pa.nv = p.nv; pa.nt = p.nt; pa.group = group; pa.hpc = hpc; pa.parts = parts;
  pa.khead_div = p.khead_div ? 1u : 0u; pa.nchunks = nchunks; pa.q_scale = p.q_scale;
  auto prep = gdn_chunk_prep_kernel<DA, SPLIT, BF16IN>;
  e = cudaFuncSetAttribute(prep, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(p1_smem(hpc)));
  if (e != cudaSuccess) return e;
  prep<<<static_cast<unsigned>(prep_blocks), NTH, p1_smem(hpc), stream>>>(pa, tm_k, tm_q);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  StateArgs sa;
  sa.g = p.g; sa.beta = p.beta;
  sa.state_in = p.state_in; sa.ws = ws; sa.ws_k = ws_k; sa.output = p.output;
  sa.state_out = p.state_out;
  sa.nk = p.nk; sa.nv = p.nv; sa.nt = p.nt; sa.group = pa.group; sa.khead_div = pa.khead_div;
  sa.nchunks = nchunks; sa.q_scale = p.q_scale;
  sa.heads = static_cast<uint32_t>(heads);
  const uint32_t segs = state_segments(heads, nchunks, want);
  sa.seg_len = (nchunks + segs - 1) / segs;
  const unsigned long long tasks2 = heads * ((nchunks + sa.seg_len - 1) / sa.seg_len);
  auto state = gdn_chunk_state_kernel<DA, SPLIT, BF16IN>;
  e = cudaFuncSetAttribute(state, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(P2_SMEM));
  if (e != cudaSuccess) return e;
  // one launch per group of up to `want` (one CTA per SM) segments, in the
  // order segment-major: a head's segment j + 1 lies at least `heads` >=
  // `want` tasks after its segment j, so in a later launch
  const unsigned long long per_launch = segs > 1 ? want : tasks2;
  for (unsigned long long base = 0; base < tasks2; base += per_launch) {
    sa.seg_base = static_cast<uint32_t>(base);
    const unsigned long long n = min(per_launch, tasks2 - base);
    state<<<static_cast<unsigned>(n), NTH, P2_SMEM, stream>>>(sa, tm_v);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace

bool chunked_split_supported(const Problem &p) {
  return chunked_supported(p) && p.nk > 0 && p.nv / p.nk <= kMaxSplitGroup;
}

size_t chunked_split_workspace_bytes(const Problem &p) {
  const size_t nchunks = (static_cast<size_t>(p.nt) + C - 1) / C;
  return (static_cast<size_t>(p.nv) * kWsFloats + static_cast<size_t>(p.nk) * kWsKFloats) * p.ns * nchunks *
         sizeof(float);
}

cudaError_t launch_chunked_split(const Problem &p, float *workspace, cudaStream_t stream) {
  if (!chunked_split_supported(p)) return cudaErrorInvalidValue;
  if (p.tf32)
    return p.decay_after ? launch_split<true, false, false>(p, workspace, stream)
                         : launch_split<false, false, false>(p, workspace, stream);
  if (p.io_bf16)
    return p.decay_after ? launch_split<true, true, true>(p, workspace, stream)
                         : launch_split<false, true, true>(p, workspace, stream);
  return p.decay_after ? launch_split<true, true, false>(p, workspace, stream)
                       : launch_split<false, true, false>(p, workspace, stream);
}

// ---------------------------------------------------------------- fixed scratch
//
// The two-pass workspace in a fixed device array, for callers that cannot
// allocate device memory (gdn_forward_chunked_noalloc).  Every call on a
// device uses the same array.  Pass 1 writes every workspace element pass 2
// reads, so nothing needs clearing between calls; two calls that overlap on
// the GPU (different streams) would race on it.

static __device__ __align__(256) float g_noalloc_ws[kNoallocWorkspaceBytes / sizeof(float)];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
// Device address of g_noalloc_ws per device, with the id of the context it
// was looked up in (0: none yet).  A context torn down and created again
// (cudaDeviceReset) gets a new id, so the address is looked up again.
struct NoallocAddr {
  unsigned long long ctx_id;
  float *addr;
};
NoallocAddr g_noalloc_addr[kMaxDevices] = {};

using CtxGetCurrentFn = CUresult (*)(CUcontext *);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long *);

// Unique id of the calling thread's current context (never reused within a
// process), or 0 when there is none or the driver cannot say.
unsigned long long current_context_id() {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(f);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current == nullptr || get_id == nullptr || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr ||
      get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}
}  // namespace

cudaError_t launch_chunked_split_noalloc(const Problem &p, cudaStream_t stream) {
  if (!chunked_split_supported(p) || chunked_split_workspace_bytes(p) > kNoallocWorkspaceBytes)
    return cudaErrorInvalidValue;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  float *ws = nullptr;
  {
    // Once per device and context, with that device current: the array's
    // name is only a host-side stand-in, so its device address comes from
    // the runtime.
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    NoallocAddr &c = g_noalloc_addr[dev];
    const unsigned long long id = current_context_id();
    if (c.addr == nullptr || id == 0 || c.ctx_id != id) {
      void *addr = nullptr;
      e = cudaGetSymbolAddress(&addr, g_noalloc_ws);
      if (e != cudaSuccess) return e;
      c.addr = static_cast<float *>(addr);
      c.ctx_id = current_context_id();  // the lookup made the context current if there was none
    }
    ws = c.addr;
  }
  return launch_chunked_split(p, ws, stream);
}

cudaError_t chunked_split_wait_status(unsigned int *bits, bool reset, cudaStream_t stream) {
  return chunked::read_wait_status(bits, reset, stream);
}

}  // namespace gdn

// Two-pass chunked (WY / UT-transform) prefill of the Gated DeltaNet
// recurrence on sm_103a, D_k = D_v = 128: the same chunk equations as the
// single-pass kernel (chunked.cu), split at the state.
//
// Everything the chunk equations need that does not depend on the state --
// the Gram products K K^T and Q K^T, A, T = (I + A)^-1 and
// P' = q_scale (Q K^T o Gam)_{i<=r} -- is computed for every (seq, value
// head, chunk) at once by pass 1, one CTA per chunk, and written to a
// caller-provided workspace (32 KB per chunk: T as an f32 canonical image,
// P' as a TF32 canonical image).  Pass 2 keeps one CTA per (seq, value head)
// for the whole token range and runs only the state-dependent part per
// chunk: operand building, U^T = V^T T''^T + X (-T')^T with X = S K^T,
// Y^T = S Q'^T + U^T P'^T, S += U^T K'^T.  The serial chain per chunk loses
// the Gram epilogue and the triangular inverse.  Pass 2 loads by TMA: K and
// Q rows land 128-byte swizzled, which is both the MMA's K-major SWIZZLE_128B
// operand layout and conflict-free for the transposed reads that build K'^T;
// V rows, the T image and P' land as plain boxes and bulk copies, each group
// on its own mbarrier, so no thread stalls issuing copies.
//
// Pass 1 is free of the lazy state scale c (S = c * TMEM S): T'' = T diag(beta)
// and -T' = -T diag(beta gamma) are built by pass 2 from T, and c enters
// pass 2 through the K operand of X (K_img = c K, so X = (c S~) K^T exactly as
// in the single-pass kernel), through Q' and through K'.
//
// Workspace layout: float ws[head][chunk][8192], head = s * n_v + vh:
// [0, 4096) T (64 x 64, canonical K-major image, unrounded f32),
// [4096, 8192) P' (canonical image, rounded to TF32).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

#include "chunked_common.cuh"
#include "gdn_internal.h"

namespace gdn {
namespace {

using namespace chunked;

constexpr uint32_t kWsFloats = 8192;  // per (head, chunk)

// per-token scalar slots (64 floats each)
enum { Q_G = 0, Q_GAM, Q_GAMP, Q_BETA, Q_GPREV, Q_EG, Q_GRAW, Q_BRAW, Q_KTS, Q_TPS, Q_QS, Q_NSC };

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

// Asynchronous copies of one chunk's raw g and beta into the scalar area
// (threads 0..127); tokens past the chunk's end read as zero.
__device__ __forceinline__ void stage_gates_async(uint32_t sc_addr, const float *g, const float *beta,
                                                  size_t sc0, size_t nv, int nc, int tid) {
  if (tid < 128) {
    const int i = tid & 63;
    const size_t src = sc0 + static_cast<size_t>(i < nc ? i : 0) * nv;
    cp_async4(sc_addr + ((tid < 64 ? Q_GRAW : Q_BRAW) * 64 + i) * 4, (tid < 64 ? g : beta) + src,
              i < nc ? 4u : 0u);
  }
}

// ---------------------------------------------------------------- TMA

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" :: "r"(bar), "r"(bytes) : "memory");
}
// One box of a 4-D tensor map (coordinates innermost first) into shared memory.
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap *tm, int c0, int c1, int c2, int c3,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], [%6];"
      :: "r"(dst), "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
      : "memory");
}
// A contiguous global block into shared memory (16-byte aligned, multiple of 16 bytes).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               :: "r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}
// Named barriers (ids 1..15): arrive without waiting, or wait for `n` threads.
__device__ __forceinline__ void named_arrive(int id, int n) {
  asm volatile("bar.arrive %0, %1;" :: "r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ void named_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(n) : "memory");
}
// K-major SWIZZLE_128B operand descriptor: 8-row x 128-byte atoms 1024 bytes apart.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) {
  return static_cast<uint64_t>((saddr >> 4) & 0x3FFF) | (1ull << 16) |
         (static_cast<uint64_t>(1024 >> 4) << 32) | (1ull << 46) | (2ull << 61);
}
// ================================================================ pass 1

// shared memory (bytes): the [K;Q] stack for the Gram, then, once the Gram
// is in TMEM, A, T and the block products overlaid on it
constexpr uint32_t P1_STACK = 0;
constexpr uint32_t P1_A = 0;
constexpr uint32_t P1_T = 64 * LD * 4;
constexpr uint32_t P1_M = 2 * 64 * LD * 4;
constexpr uint32_t P1_SC = 65536;
constexpr uint32_t P1_MISC = P1_SC + Q_NSC * 64 * 4;
constexpr uint32_t P1_SMEM = P1_MISC + 64 + 1024;  // + room to align the base to 1024
static_assert(P1_M + 4 * 256 * 4 <= P1_SC, "pass-1 overlay must fit in the stack");

struct PrepArgs {
  const float *__restrict__ q;
  const float *__restrict__ k;
  const float *__restrict__ g;
  const float *__restrict__ beta;
  float *__restrict__ ws;
  uint32_t nk, nv, nt, group, khead_div, nchunks;
  float q_scale;
};

struct P1Misc {
  unsigned long long mbar;    // Gram MMA commit
  unsigned long long bar_ld;  // TMA: the chunk's K and Q rows
  uint32_t tmem_base;
  int failed;
  int extreme;
};

// The stack [K;Q] arrives by TMA, 128-byte swizzled: column block cb (32
// floats) holds K's 64 rows then Q's 64 rows (16 KB), so A = [K;Q] (M = 128)
// and B = K (N = 64) of the Gram are K-major SWIZZLE_128B operands.
template <bool DECAY_AFTER>
__global__ void __launch_bounds__(NTH, 2)
    gdn_chunk_prep_kernel(const PrepArgs a, const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_q) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t raw_addr = smem_addr(smem_raw);
  unsigned char *smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  float *sA = reinterpret_cast<float *>(smem + P1_A);
  float *sT = reinterpret_cast<float *>(smem + P1_T);
  float *sM = reinterpret_cast<float *>(smem + P1_M);
  float *sc = reinterpret_cast<float *>(smem + P1_SC);
  P1Misc *misc = reinterpret_cast<P1Misc *>(smem + P1_MISC);
  const uint32_t sbase = smem_addr(smem);
  const uint32_t mbar = smem_addr(&misc->mbar), bar_ld = smem_addr(&misc->bar_ld);
  const int tid = static_cast<int>(threadIdx.x);
  const int warp = tid >> 5, lane = tid & 31;
  const int row = tid & 127, half = tid >> 7;
  const uint32_t lane_field = static_cast<uint32_t>(32 * (warp & 3)) << 16;

  // block -> (seq, chunk, value head), value head fastest: the value heads
  // that read one key head run side by side and share its K and Q in L2
  const uint32_t vh = blockIdx.x % a.nv;
  const uint32_t rest = blockIdx.x / a.nv;
  const uint32_t ch = rest % a.nchunks, s = rest / a.nchunks;
  const uint32_t kh = a.khead_div ? vh / a.group : vh % a.nk;
  const uint32_t t0 = ch * C;
  const int nc = static_cast<int>(min(static_cast<uint32_t>(C), a.nt - t0));
  const size_t sc0 = (static_cast<size_t>(s) * a.nt + t0) * a.nv + vh;
  float *ws = a.ws + ((static_cast<size_t>(s) * a.nv + vh) * a.nchunks + ch) * kWsFloats;

  stage_gates_async(sbase + P1_SC, a.g, a.beta, sc0, a.nv, nc, tid);
  cp_async_commit();
  if (tid == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" :: "r"(mbar));
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" :: "r"(bar_ld));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    misc->failed = 0;
    mbar_expect_tx(bar_ld, 65536);
#pragma unroll
    for (int cb = 0; cb < 4; ++cb) {
      tma_load_4d(sbase + P1_STACK + cb * 16384, &tm_k, 32 * cb, static_cast<int>(kh), static_cast<int>(t0),
                  static_cast<int>(s), bar_ld);
      tma_load_4d(sbase + P1_STACK + cb * 16384 + 8192, &tm_q, 32 * cb, static_cast<int>(kh),
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

  // K and Q to TF32 (round to nearest) in place; per-token scalars (warp 0)
#pragma unroll
  for (int it = 0; it < 16; ++it) {
    float4 *p = reinterpret_cast<float4 *>(smem + P1_STACK) + tid + NTH * it;
    float4 x = *p;
    x.x = tf32_rna(x.x); x.y = tf32_rna(x.y); x.z = tf32_rna(x.z); x.w = tf32_rna(x.w);
    *p = x;
  }
  if (warp == 0) {
    float GC;
    const bool extreme = chunk_scalars(sc, lane, &GC);
    if (lane == 0) misc->extreme = extreme;
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
  const bool ok = mbar_wait(mbar, 0);
  if (!ok) misc->failed = 1;
  fence_after();
  const bool extreme = misc->extreme != 0;

  // A (plain, over the dead stack) and P' (straight to the workspace)
  {
    uint32_t gv[32];
    GDN_TMEM_LD32(tmem + lane_field + 32 * half, gv);
    tmem_wait_ld();
    __syncthreads();  // every Gram row is in registers before A overwrites the stack
    const float *G = sc + Q_G * 64, *eG = sc + Q_EG * 64;
    if (row < 64) {
      const int r = row;
      const float br = sc[Q_BETA * 64 + r];
      const float Gr = DECAY_AFTER ? sc[Q_GPREV * 64 + r] : G[r];
      const float bgr = br * (DECAY_AFTER ? sc[Q_GAMP * 64 + r] : sc[Q_GAM * 64 + r]);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        float e[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int i = 32 * half + 4 * j + u;
          const float gam = extreme ? br * __expf(G[i] - Gr) : bgr * eG[i];
          e[u] = i < r ? gam * __uint_as_float(gv[4 * j + u]) : 0.f;
        }
        *reinterpret_cast<float4 *>(sA + r * LD + 32 * half + 4 * j) = make_float4(e[0], e[1], e[2], e[3]);
      }
    } else {
      const int r = row - 64;
      const float Gr = G[r];
      const float qgr = a.q_scale * sc[Q_GAM * 64 + r];
      float *wp = ws + 4096;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        float e[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int i = 32 * half + 4 * j + u;
          const float gam = extreme ? a.q_scale * __expf(G[i] - Gr) : qgr * eG[i];
          e[u] = i <= r ? tf32_rna(gam * __uint_as_float(gv[4 * j + u])) : 0.f;
        }
        *reinterpret_cast<float4 *>(wp + canon(r, 32 * half + 4 * j, 64) / 4) =
            make_float4(e[0], e[1], e[2], e[3]);
      }
    }
  }
  cta_sync();

  // T = (I + A)^-1, written as a canonical image (NaN if the Gram wait timed out)
  tri_inverse(sA, sT, sM, tid);
  {
    const float nan = __int_as_float(0x7fc00000);
#pragma unroll
    for (int it = 0; it < 4; ++it) {
      const int ci = tid + NTH * it;
      const int core = ci >> 3, r = (core >> 4) * 8 + (ci & 7), i0 = 4 * (core & 15);
      float4 t = *reinterpret_cast<const float4 *>(sT + r * LD + i0);
      if (misc->failed) t = make_float4(nan, nan, nan, nan);
      reinterpret_cast<float4 *>(ws)[ci] = t;
    }
  }
  // a load that timed out may still land: wait for it (bounded) before exit
  if (tid == 0 && !loaded) (void)mbar_wait(bar_ld, 0);
  cta_sync();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(tmem), "r"(64));
}

// ================================================================ pass 2

// TMEM columns (Y^T alternates between two regions so a chunk's outputs are
// read out while the next chunk's products run)
// [X | Y^T] is one N = 128 product; its two regions alternate by chunk.
constexpr uint32_t P2_TM_S = 0, P2_TM_XY0 = 128, P2_TM_U = 256, P2_TM_V = 320, P2_TM_XY1 = 384;
constexpr uint32_t P2_TM_COLS = 512;

// Shared memory (bytes from a 1024-aligned base).  K and Q arrive by TMA as
// four 64-row x 128-byte boxes each, 128-byte swizzled, interleaved so that
// column block cb (32 floats) holds K's 64 rows then Q's (16 KB): [K; Q'] is
// then one 128-row K-major SWIZZLE_128B operand, and a warp reading either a
// row or a column of K touches distinct banks.
constexpr uint32_t P2_KQ = 0;                      // [K; Q] (TMA) -> [K; Q'] in TF32, in place
constexpr uint32_t P2_KT = P2_KQ + 65536;          // K'^T, 128 x 64 canonical (no swizzle)
constexpr uint32_t P2_TPP = P2_KT + 32768;         // T image (bulk copy) -> T'' in place
constexpr uint32_t P2_TP = P2_TPP + 16384;         // -T'
constexpr uint32_t P2_P = P2_TP + 16384;           // P' image (bulk copy), used as is
constexpr uint32_t P2_VS = P2_P + 16384;           // V rows (TMA), 64 x 128 natural
constexpr uint32_t P2_SC = P2_VS + 32768;          // per-token scalars
constexpr uint32_t P2_MISC = P2_SC + Q_NSC * 64 * 4;
constexpr uint32_t P2_SMEM = P2_MISC + 128 + 1024;  // + room to align the base to 1024
static_assert(P2_SMEM <= 232448, "pass-2 shared memory");
constexpr uint32_t kImgBytes = 16384;   // one 64 x 64 workspace image
constexpr uint32_t kRowsBytes = 32768;  // 64 rows of 128 floats

struct StateArgs {
  const float *__restrict__ g;
  const float *__restrict__ beta;
  const float *state_in;
  const float *__restrict__ ws;
  float *__restrict__ output;
  float *state_out;
  uint32_t nk, nv, nt, group, khead_div, nchunks;
  float q_scale;
};

struct P2Misc {
  unsigned long long mbar1;   // batch-1 MMA commits
  unsigned long long mbar2;   // batch-2 MMA commits
  unsigned long long bar_in;  // TMA: K, Q rows and the T image of a chunk
  unsigned long long bar_v;   // TMA: V rows of a chunk
  unsigned long long bar_p;   // TMA: P' image of a chunk
  uint32_t tmem_base;
  int failed;
  float c_renorm, c_fold, c_next;
  int do_renorm, do_fold;
};

// Thread 0: this chunk's K and Q rows (4 boxes each) and T image, on bar_in.
__device__ __forceinline__ void p2_load_in(uint32_t sbase, const CUtensorMap *tm_k, const CUtensorMap *tm_q,
                                           int kh, int t0, int s, const float *timg, uint32_t bar) {
  mbar_expect_tx(bar, 2 * kRowsBytes + kImgBytes);
#pragma unroll
  for (int cb = 0; cb < 4; ++cb) {
    tma_load_4d(sbase + P2_KQ + cb * 16384, tm_k, 32 * cb, kh, t0, s, bar);
    tma_load_4d(sbase + P2_KQ + cb * 16384 + 8192, tm_q, 32 * cb, kh, t0, s, bar);
  }
  bulk_load(sbase + P2_TPP, timg, kImgBytes, bar);
}

// The state pass (see the file comment); loads by TMA, waits bounded.
template <bool DECAY_AFTER>
__global__ void __launch_bounds__(NTH, 1)
    gdn_chunk_state_kernel(const StateArgs a, const __grid_constant__ CUtensorMap tm_k,
                           const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_v) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // operate from a 1024-byte aligned base (the swizzled boxes need it)
  const uint32_t raw_addr = smem_addr(smem_raw);
  const uint32_t pad = ((raw_addr + 1023u) & ~1023u) - raw_addr;
  unsigned char *smem = smem_raw + pad;
  float *sc = reinterpret_cast<float *>(smem + P2_SC);
  const float *sVS = reinterpret_cast<const float *>(smem + P2_VS);
  P2Misc *misc = reinterpret_cast<P2Misc *>(smem + P2_MISC);
  const uint32_t sbase = raw_addr + pad;
  const uint32_t mbar1 = smem_addr(&misc->mbar1), mbar2 = smem_addr(&misc->mbar2);
  const uint32_t bar_in = smem_addr(&misc->bar_in), bar_v = smem_addr(&misc->bar_v),
                 bar_p = smem_addr(&misc->bar_p);

  const int tid = static_cast<int>(threadIdx.x);
  const int warp = tid >> 5, lane = tid & 31;
  const int row = tid & 127;
  const int half = tid >> 7;
  const uint32_t lane_field = static_cast<uint32_t>(32 * (warp & 3)) << 16;

  const uint32_t head = blockIdx.x;  // = s * nv + vh
  const uint32_t vh = head % a.nv, s = head / a.nv;
  const uint32_t kh = a.khead_div ? vh / a.group : vh % a.nk;
  const uint32_t nt = a.nt;
  const size_t state_head = static_cast<size_t>(head) * D * D;
  const size_t v_tok = static_cast<size_t>(a.nv) * D;
  const float *wseq = a.ws + static_cast<size_t>(head) * a.nchunks * kWsFloats;
  const size_t sc_first = static_cast<size_t>(s) * nt * a.nv + vh;
  const uint32_t nchunks = a.nchunks;

  if (tid == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" :: "r"(mbar1));
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" :: "r"(mbar2));
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" :: "r"(bar_in));
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" :: "r"(bar_v));
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" :: "r"(bar_p));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    misc->failed = 0;
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(smem_addr(&misc->tmem_base)), "r"(P2_TM_COLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  __syncthreads();  // barriers initialised before anyone waits on them
  // chunk 0's inputs start arriving while the state is loaded
  {
    const int nc0 = static_cast<int>(min(nt, static_cast<uint32_t>(C)));
    if (tid == 0) {
      p2_load_in(sbase, &tm_k, &tm_q, static_cast<int>(kh), 0, static_cast<int>(s), wseq, bar_in);
      mbar_expect_tx(bar_v, kRowsBytes);
      tma_load_4d(sbase + P2_VS, &tm_v, 0, static_cast<int>(vh), 0, static_cast<int>(s), bar_v);
      mbar_expect_tx(bar_p, kImgBytes);
      bulk_load(sbase + P2_P, wseq + 4096, kImgBytes, bar_p);
    }
    stage_gates_async(sbase + P2_SC, a.g, a.beta, sc_first, a.nv, nc0, tid);
    cp_async_commit();
  }
  cta_sync();
  const uint32_t tmem = misc->tmem_base;
  const uint32_t tl = tmem + lane_field;

  // S <- state_in (c = 1).  Thread: row d_v, columns [64*half, 64*half + 64).
  {
    const float4 *src = reinterpret_cast<const float4 *>(a.state_in + state_head + row * D + 64 * half);
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
    }
    tmem_wait_st();
  }

  float c = 1.f;
  uint32_t ph1 = 0, ph2 = 0;
  bool failed = false;
  bool b2_pending = false;  // a batch 2 was issued and not yet waited for
  // TMA arms and waits per barrier (uniform over the CTA): a copy is in
  // flight while a barrier has been armed more often than waited on
  uint32_t armed_in = 1, armed_v = 1, armed_p = 1, waited_in = 0, waited_v = 0, waited_p = 0;
  const int wt = tid - 32;  // worker index of warps 1..7 (steps 5-7)
  constexpr int NW = NTH - 32;

  for (uint32_t ch = 0; ch < nchunks && !failed; ++ch) {
    const uint32_t t0 = ch * C;
    const int nc = static_cast<int>(min(static_cast<uint32_t>(C), nt - t0));
    const bool more = ch + 1 < nchunks;
    const int ncn = more ? static_cast<int>(min(static_cast<uint32_t>(C), nt - t0 - C)) : 0;
    const uint32_t tm_x = (ch & 1) ? P2_TM_XY1 : P2_TM_XY0;  // X; Y^T at tm_x + 64
    const uint32_t tm_y = tm_x + 64;
    const uint32_t par = ch & 1;  // phase parity of this chunk's TMA barriers

    // ---- 0. this chunk's V rows (TMA) and gates (cp.async) have landed; its
    // K, Q rows and T image may still be on the way, and the previous chunk's
    // batch 2 may still be running
    if (!mbar_wait(bar_v, par)) misc->failed = 1;
    ++waited_v;
    cp_async_wait_all();
    __syncthreads();
    if (misc->failed) { failed = true; break; }

    // ---- 1. warp 0: per-token scalars and the lazy-scale bookkeeping.
    // Meanwhile V^T -> TMEM (lane d_v, columns = tokens), warp 4 taking both
    // halves of the lane quarter it shares with warp 0.
    if (warp == 0) {
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
        const float bi = sc[Q_BETA * 64 + i];
        sc[Q_KTS * 64 + i] = __expf(Gi - GC) / cnext;                       // K' row scale
        sc[Q_TPS * 64 + i] = -cc * bi * (DECAY_AFTER ? sc[Q_GAMP * 64 + i] : sc[Q_GAM * 64 + i]);  // -T' column
        sc[Q_QS * 64 + i] = cc * a.q_scale * sc[Q_GAM * 64 + i];           // Q' row scale
      }
      if (lane == 0) {
        misc->c_renorm = renorm; misc->c_fold = fold; misc->c_next = cnext;
        misc->do_renorm = do_renorm; misc->do_fold = extreme;
      }
    } else {
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int h = warp == 4 ? hh : half;
        if (hh == 1 && warp != 4) break;
        uint32_t vv[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) vv[j] = __float_as_uint(tf32_rna(sVS[(32 * h + j) * D + row]));
        GDN_TMEM_ST32(tl + P2_TM_V + 32 * h, vv);
      }
      tmem_wait_st();
    }
    cta_sync();
    if (more) {  // the V buffer is free: the next chunk's V rows
      if (tid == 0) {
        fence_async_smem();
        mbar_expect_tx(bar_v, kRowsBytes);
        tma_load_4d(sbase + P2_VS, &tm_v, 0, static_cast<int>(vh), static_cast<int>(t0 + C),
                    static_cast<int>(s), bar_v);
      }
      ++armed_v;
    }
    const float c_renorm = misc->c_renorm, c_fold = misc->c_fold;
    const bool do_renorm = misc->do_renorm != 0, do_fold = misc->do_fold != 0;

    // ---- 2. the previous chunk's batch 2 is done: S, Y, K'^T and P' are
    // settled; this chunk's P' may load
    if (b2_pending) {
      if (!mbar_wait(mbar2, ph2)) misc->failed = 1;
      ph2 ^= 1;
      b2_pending = false;
      fence_after();
      __syncthreads();
      if (misc->failed) { failed = true; break; }
      if (tid == 0) {
        mbar_expect_tx(bar_p, kImgBytes);
        bulk_load(sbase + P2_P, wseq + ch * kWsFloats + 4096, kImgBytes, bar_p);
      }
      ++armed_p;
    }

    // ---- 3. fold c into S if it left [2^-30, 2^30] (no MMA in flight here)
    if (do_renorm) tmem_scale64(tl + P2_TM_S + 64 * half, c_renorm);

    // ---- 4. K, Q rows and the T image
    if (!mbar_wait(bar_in, par)) misc->failed = 1;
    ++waited_in;
    __syncthreads();
    if (misc->failed) { failed = true; break; }

    // ---- 5. all warps: K to TF32 and Q' in place (row = chunk / 8 in its box)
    {
      const float *qs = sc + Q_QS * 64;
#pragma unroll
      for (int it = 0; it < 8; ++it) {
        const int ci = tid + NTH * it;
        const int off = (ci >> 9) * 16384 + (ci & 511) * 16;
        float4 *pk = reinterpret_cast<float4 *>(smem + P2_KQ + off);
        float4 x = *pk;
        x.x = tf32_rna(x.x); x.y = tf32_rna(x.y); x.z = tf32_rna(x.z); x.w = tf32_rna(x.w);
        *pk = x;
        float4 *pq = reinterpret_cast<float4 *>(smem + P2_KQ + 8192 + off);
        float4 y = *pq;
        const float f = qs[(ci & 511) >> 3];
        y.x = tf32_rna(y.x * f); y.y = tf32_rna(y.y * f); y.z = tf32_rna(y.z * f); y.w = tf32_rna(y.w * f);
        *pq = y;
      }
    }
    fence_async_smem();
    cta_sync();

    // ---- 6-7. warp 0 issues [X | Y^T] = S [K; Q']^T (one N = 128 product),
    // then, once warps 1-7 have built T'' and -T' (named barrier),
    // Ut = V^T T''^T + X (-T')^T; warps 1-7 then build K'^T from the TF32 K
    // while those run (only batch 2 reads it).  The scale c rides on -T' and Q'.
    if (warp == 0) {
      if (lane == 0) {
#pragma unroll
        for (int ks = 0; ks < D / 8; ++ks)
          mma_ts(tmem + tm_x, tmem + P2_TM_S + 8 * ks,
                 sdesc_sw128(sbase + P2_KQ + (ks >> 2) * 16384 + (ks & 3) * 32), idesc_tf32(128, 128),
                 ks > 0);
      }
      __syncwarp();
      named_sync(1, NTH);
      fence_after();
      if (lane == 0) {
        const uint32_t i64 = idesc_tf32(128, 64);
#pragma unroll
        for (int ks = 0; ks < C / 8; ++ks)   // Ut = V^T T''^T
          mma_ts(tmem + P2_TM_U, tmem + P2_TM_V + 8 * ks, sdesc(sbase + P2_TPP + ks * 256, 2048), i64, ks > 0);
#pragma unroll
        for (int ks = 0; ks < C / 8; ++ks)   // Ut += X (-T')^T
          mma_ts(tmem + P2_TM_U, tmem + tm_x + 8 * ks, sdesc(sbase + P2_TP + ks * 256, 2048), i64, 1);
        mma_commit(mbar1);
      }
      __syncwarp();
    } else {
      const float *tps = sc + Q_TPS * 64, *bet = sc + Q_BETA * 64;
      for (int ci = wt; ci < 1024; ci += NW) {  // T'' in place, -T' beside it
        const int i0 = 4 * ((ci >> 3) & 15);
        float4 *pt = reinterpret_cast<float4 *>(smem + P2_TPP + ci * 16);
        const float4 t = *pt;
        *reinterpret_cast<float4 *>(smem + P2_TP + ci * 16) =
            make_float4(tf32_rna(t.x * tps[i0]), tf32_rna(t.y * tps[i0 + 1]),
                        tf32_rna(t.z * tps[i0 + 2]), tf32_rna(t.w * tps[i0 + 3]));
        *pt = make_float4(tf32_rna(t.x * bet[i0]), tf32_rna(t.y * bet[i0 + 1]),
                          tf32_rna(t.z * bet[i0 + 2]), tf32_rna(t.w * bet[i0 + 3]));
      }
      fence_async_smem();
      fence_before();
      named_arrive(1, NTH);
      const float *kts = sc + Q_KTS * 64;
      for (int oc = wt; oc < 2048; oc += NW) {  // K'^T: d_k = oc % 128, tokens 4 (oc / 128) .. +3
        const int dk = oc & 127, i0 = (oc >> 7) * 4;
        const unsigned char *kb = smem + P2_KQ + (dk >> 5) * 16384 + (dk & 3) * 4;
        float e[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int i = i0 + u;
          e[u] = tf32_rna(*reinterpret_cast<const float *>(kb + i * 128 + ((((dk & 31) >> 2) ^ (i & 7)) << 4)) *
                          kts[i]);
        }
        *reinterpret_cast<float4 *>(smem + P2_KT + canon(dk, i0, 64)) = make_float4(e[0], e[1], e[2], e[3]);
      }
      fence_async_smem();
    }

    // ---- the previous chunk's outputs, from its Y^T region, while these run
    if (ch > 0) {
      const uint32_t tm_yp = ((ch & 1) ? P2_TM_XY0 : P2_TM_XY1) + 64;
      uint32_t yv[32];
      GDN_TMEM_LD32(tl + tm_yp + 32 * half, yv);
      tmem_wait_ld();
      float *obase = a.output + ((static_cast<size_t>(s) * nt + (t0 - C)) * a.nv + vh) * D + row;
#pragma unroll
      for (int j = 0; j < 32; ++j)  // every chunk but the last is full
        obase[static_cast<size_t>(32 * half + j) * v_tok] = __uint_as_float(yv[j]);
    }

    if (!mbar_wait(mbar1, ph1)) misc->failed = 1;
    ph1 ^= 1;
    fence_after();
    __syncthreads();
    if (misc->failed) { failed = true; break; }
    // K, Q and the T image are free: the next chunk's (TMA) and its gates
    if (more) {
      if (tid == 0) {
        fence_async_smem();
        p2_load_in(sbase, &tm_k, &tm_q, static_cast<int>(kh), static_cast<int>(t0 + C), static_cast<int>(s),
                   wseq + (ch + 1) * kWsFloats, bar_in);
      }
      ++armed_in;
      stage_gates_async(sbase + P2_SC, a.g, a.beta, sc_first + static_cast<size_t>(t0 + C) * a.nv, a.nv,
                        ncn, tid);
      cp_async_commit();
    }

    // ---- 8. U^T to TF32 (nearest) in place; extreme gates: decay S now
    {
      uint32_t uv[32];
      GDN_TMEM_LD32(tl + P2_TM_U + 32 * half, uv);
      tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < 32; ++j) uv[j] = __float_as_uint(tf32_rna(__uint_as_float(uv[j])));
      GDN_TMEM_ST32(tl + P2_TM_U + 32 * half, uv);
      tmem_wait_st();
    }
    if (do_fold) tmem_scale64(tl + P2_TM_S + 64 * half, c_fold);
    if (!mbar_wait(bar_p, par)) misc->failed = 1;  // this chunk's P'
    ++waited_p;
    cta_sync();

    // ---- 9. batch 2: Yt += Ut P'^T; S += Ut K'^T.  Not waited for here unless
    // this is the last chunk: the next chunk's first steps overlap it.
    if (tid == 0) {
#pragma unroll
      for (int ks = 0; ks < C / 8; ++ks)
        mma_ts(tmem + tm_y, tmem + P2_TM_U + 8 * ks, sdesc(sbase + P2_P + ks * 256, 2048),
               idesc_tf32(128, 64), 1);
#pragma unroll
      for (int ks = 0; ks < C / 8; ++ks)
        mma_ts(tmem + P2_TM_S, tmem + P2_TM_U + 8 * ks, sdesc(sbase + P2_KT + ks * 256, 2048),
               idesc_tf32(128, 128), 1);
      mma_commit(mbar2);
    }
    b2_pending = true;
    if (!more) {  // ---- 10. the last chunk: wait, then its outputs
      if (!mbar_wait(mbar2, ph2)) misc->failed = 1;
      ph2 ^= 1;
      b2_pending = false;
      fence_after();
      __syncthreads();
      if (misc->failed) { failed = true; break; }
      uint32_t yv[32];
      GDN_TMEM_LD32(tl + tm_y + 32 * half, yv);
      tmem_wait_ld();
      float *obase = a.output + ((static_cast<size_t>(s) * nt + t0) * a.nv + vh) * D + row;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int i = 32 * half + j;
        if (i < nc) obase[static_cast<size_t>(i) * v_tok] = __uint_as_float(yv[j]);
      }
    }
    c = misc->c_next;
  }

  // an MMA batch still in flight after a failure finishes (bounded) before
  // TMEM is read or released
  if (b2_pending && tid == 0) (void)mbar_wait(mbar2, ph2);
  fence_after();
  __syncthreads();
  cp_async_wait_all();  // no cp.async may still be landing in shared memory at exit
  // after a failure, let any TMA copy still in flight land (bounded waits)
  // before the CTA's shared memory is released
  if (tid == 0) {
    if (armed_in > waited_in) (void)mbar_wait(bar_in, waited_in & 1);
    if (armed_v > waited_v) (void)mbar_wait(bar_v, waited_v & 1);
    if (armed_p > waited_p) (void)mbar_wait(bar_p, waited_p & 1);
  }

  // ---- state_out = c * S (or NaN if a wait timed out)
  {
    float4 *dst = reinterpret_cast<float4 *>(a.state_out + state_head + row * D + 64 * half);
    const float f = failed ? __int_as_float(0x7fc00000) : c;
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

// A [128, heads, n_tokens, n_seqs] f32 tensor (128 contiguous) as a 4-D map
// whose box is `inner` floats x 1 head x 64 tokens x 1 seq.
cudaError_t rows_map(CUtensorMap *tm, const void *base, uint32_t heads, uint32_t nt, uint32_t ns,
                     uint32_t inner, CUtensorMapSwizzle swizzle) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (enc == nullptr) return cudaErrorNotSupported;
  const cuuint64_t dims[4] = {128, heads, nt, ns};
  const cuuint64_t strides[3] = {512, 512ull * heads, 512ull * heads * nt};
  const cuuint32_t box[4] = {inner, 1, 64, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<void *>(base), dims, strides, box,
                         estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <bool DA>
cudaError_t launch_split(const Problem &p, float *ws, cudaStream_t stream) {
  const uint32_t nchunks = (p.nt + C - 1) / C;
  const unsigned long long heads = static_cast<unsigned long long>(p.nv) * p.ns;
  const unsigned long long prep_blocks = heads * nchunks;
  if (heads == 0 || prep_blocks > 0x7fffffffull) return cudaErrorInvalidConfiguration;
  if (reinterpret_cast<uintptr_t>(p.v) % 16 != 0) return cudaErrorMisalignedAddress;  // TMA source
  CUtensorMap tm_k, tm_q, tm_v;
  cudaError_t e = rows_map(&tm_k, p.k, p.nk, p.nt, p.ns, 32, CU_TENSOR_MAP_SWIZZLE_128B);
  if (e == cudaSuccess) e = rows_map(&tm_q, p.q, p.nk, p.nt, p.ns, 32, CU_TENSOR_MAP_SWIZZLE_128B);
  if (e == cudaSuccess) e = rows_map(&tm_v, p.v, p.nv, p.nt, p.ns, 128, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (e != cudaSuccess) return e;

  PrepArgs pa;
  pa.q = static_cast<const float *>(p.q); pa.k = static_cast<const float *>(p.k);
  pa.g = p.g; pa.beta = p.beta; pa.ws = ws;
  pa.nk = p.nk; pa.nv = p.nv; pa.nt = p.nt; pa.group = p.nv / p.nk;
  pa.khead_div = p.khead_div ? 1u : 0u; pa.nchunks = nchunks; pa.q_scale = p.q_scale;
  auto prep = gdn_chunk_prep_kernel<DA>;
  e = cudaFuncSetAttribute(prep, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(P1_SMEM));
  if (e != cudaSuccess) return e;
  prep<<<static_cast<unsigned>(prep_blocks), NTH, P1_SMEM, stream>>>(pa, tm_k, tm_q);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  StateArgs sa;
  sa.g = p.g; sa.beta = p.beta;
  sa.state_in = p.state_in; sa.ws = ws; sa.output = static_cast<float *>(p.output);
  sa.state_out = p.state_out;
  sa.nk = p.nk; sa.nv = p.nv; sa.nt = p.nt; sa.group = pa.group; sa.khead_div = pa.khead_div;
  sa.nchunks = nchunks; sa.q_scale = p.q_scale;
  auto state = gdn_chunk_state_kernel<DA>;
  e = cudaFuncSetAttribute(state, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(P2_SMEM));
  if (e != cudaSuccess) return e;
  state<<<static_cast<unsigned>(heads), NTH, P2_SMEM, stream>>>(sa, tm_k, tm_q, tm_v);
  return cudaGetLastError();
}

}  // namespace

size_t chunked_split_workspace_bytes(const Problem &p) {
  const size_t nchunks = (static_cast<size_t>(p.nt) + C - 1) / C;
  return static_cast<size_t>(p.nv) * p.ns * nchunks * kWsFloats * sizeof(float);
}

cudaError_t launch_chunked_split(const Problem &p, float *workspace, cudaStream_t stream) {
  if (!chunked_supported(p)) return cudaErrorInvalidValue;
  return p.decay_after ? launch_split<true>(p, workspace, stream) : launch_split<false>(p, workspace, stream);
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
float *g_noalloc_addr[kMaxDevices] = {};  // device address of g_noalloc_ws, per device
}  // namespace

cudaError_t launch_chunked_split_noalloc(const Problem &p, cudaStream_t stream) {
  if (!chunked_supported(p) || chunked_split_workspace_bytes(p) > kNoallocWorkspaceBytes)
    return cudaErrorInvalidValue;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  float *ws = nullptr;
  {
    // Once per device, with that device current: the array's name is only a
    // host-side stand-in, so its device address comes from the runtime.
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (g_noalloc_addr[dev] == nullptr) {
      void *addr = nullptr;
      e = cudaGetSymbolAddress(&addr, g_noalloc_ws);
      if (e != cudaSuccess) return e;
      g_noalloc_addr[dev] = static_cast<float *>(addr);
    }
    ws = g_noalloc_addr[dev];
  }
  return launch_chunked_split(p, ws, stream);
}

}  // namespace gdn

// Shared pieces of the chunked (WY / UT-transform) prefill kernels on
// sm_103a: chunk geometry, inline-PTX wrappers for tcgen05 (MMA issue,
// commit, TMEM load/store, fences), cp.async, a bounded mbarrier wait, and
// the 64 x 64 unit-lower-triangular inverse on the CUDA cores.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace gdn {
namespace chunked {
namespace {

constexpr int C = 64;     // tokens per chunk
constexpr int D = 128;    // D_k = D_v
constexpr int NTH = 256;  // threads per CTA
constexpr int LD = 68;    // row stride (floats) of the plain 64 x 64 work matrices
constexpr float kMaxLogScale = 40.f;
constexpr float kRenormLo = 9.3132257e-10f;  // 2^-30
constexpr float kRenormHi = 1.0737418e+09f;  // 2^30

// ---------------------------------------------------------------- PTX helpers

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
// Round to the nearest TF32 value (10 mantissa bits), ties to even; NaN
// stays NaN, infinities stay infinite.  The rounding-to-nearest conversion
// is one instruction here, cheaper than the ties-away form.
__device__ __forceinline__ float tf32_rn(float x) {
  uint32_t r;
  asm("cvt.rn.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return __uint_as_float(r);
}
// canonical K-major no-swizzle byte offset of element (row, k) in a matrix
// whose K extent is KE elements
__device__ __forceinline__ uint32_t canon(int row, int kk, int KE) {
  return static_cast<uint32_t>(((row >> 3) * (KE >> 2) + (kk >> 2)) * 128 + (row & 7) * 16 + (kk & 3) * 4);
}
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t sbo) {
  return static_cast<uint64_t>((saddr >> 4) & 0x3FFF) | (static_cast<uint64_t>(128 >> 4) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFF) << 32) | (1ull << 46);
}
__host__ __device__ constexpr uint32_t idesc_tf32(int M, int N) {
  return (1u << 4) | (2u << 7) | (2u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}
// bf16 A and B, f32 accumulator (kind::f16): 16 K elements per instruction,
// the same 32 bytes of a K-major row as the 8 of a TF32 instruction.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}
// D (+)= A B with both operands in shared memory; BF16 selects kind::f16
// (bf16 operands) over kind::tf32.
template <bool BF16 = false>
__device__ __forceinline__ void mma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  if constexpr (BF16)
    asm volatile("{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n"
                 :: "r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc));
  else
    asm volatile("{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
                 "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}\n"
                 :: "r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc));
}
// The same with A in tensor memory (lane = row; a bf16 A packs two K
// elements per 32-bit column, the lower K index in the low half).
template <bool BF16 = false>
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc) {
  if constexpr (BF16)
    asm volatile("{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n"
                 :: "r"(d), "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc));
  else
    asm volatile("{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
                 "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n}\n"
                 :: "r"(d), "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc));
}

// Split-bf16 operands.  x = hi + lo with hi = bf16(x) and lo = bf16(x - hi),
// both rounded to nearest (x - hi is exact in f32), so |x - hi - lo| <=
// 2^-18 |x|; a product is taken as A_hi B_hi + A_hi B_lo + A_lo B_hi with
// f32 accumulation -- the three-term bf16 scheme of Henry, Tang and Heinecke
// ("Leveraging the bfloat16 artificial intelligence datatype for
// higher-precision computations", 2019).  The dropped A_lo B_lo and the
// remainders are about 2^-16 of each term, against 2^-11 for TF32 operands.
// NaN stays NaN in both halves.
//
// pack_bf16x2(a, b): a in the low 16 bits, b in the high, each rounded to nearest.
__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));
  return r;
}
__device__ __forceinline__ void split2(float a, float b, uint32_t &hi, uint32_t &lo) {
  hi = pack_bf16x2(a, b);
  lo = pack_bf16x2(a - __uint_as_float(hi << 16), b - __uint_as_float(hi & 0xFFFF0000u));
}
// canonical K-major no-swizzle byte offset of bf16 element (row, k) in a
// matrix whose K extent is KE elements (8 x 8-element cores of 128 bytes)
__host__ __device__ constexpr uint32_t canon16(int row, int kk, int KE) {
  return static_cast<uint32_t>(((row >> 3) * (KE >> 3) + (kk >> 3)) * 128 + (row & 7) * 16 + (kk & 7) * 2);
}
__device__ __forceinline__ void mma_commit(uint32_t mbar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
               :: "r"(mbar) : "memory");
}
__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void cta_sync() {
  fence_before();
  __syncthreads();
  fence_after();
}

// 16-byte global -> shared copy; src_bytes = 0 fills the 16 bytes with zeros.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void *src, uint32_t src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;\n" ::: "memory"); }
// Wait until at most N of this thread's most recent cp.async groups are pending.
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// Arrive on an mbarrier and expect `bytes` of asynchronous copies on it.
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" :: "r"(bar), "r"(bytes) : "memory");
}
// A contiguous global block into shared memory (16-byte aligned, multiple of 16 bytes).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               :: "r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}

// Failure bits of the kernels of one translation unit, one word per device
// (a module global), read and cleared by read_wait_status.  A kernel whose
// bounded wait ran out ORs in kWaitTimeoutBit (the value of
// GDN_DEVICE_WAIT_TIMEOUT in gdn.h) besides writing NaN into its outputs.
constexpr unsigned int kWaitTimeoutBit = 0x1u;
__device__ unsigned int g_wait_status = 0u;
__device__ __forceinline__ void report_wait_timeout() { atomicOr(&g_wait_status, kWaitTimeoutBit); }

// Host: after all work on `stream` so far, *bits = this translation unit's
// word on the current device; cleared afterwards when `reset`.  Symbol
// copies only (no allocation); synchronises `stream`.
inline cudaError_t read_wait_status(unsigned int *bits, bool reset, cudaStream_t stream) {
  unsigned int h = 0u;
  cudaError_t e = cudaMemcpyFromSymbolAsync(&h, g_wait_status, sizeof h, 0, cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess && reset) {
    static const unsigned int zero = 0u;
    e = cudaMemcpyToSymbolAsync(g_wait_status, &zero, sizeof zero, 0, cudaMemcpyHostToDevice, stream);
  }
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  *bits = e == cudaSuccess ? h : 0u;
  return e;
}

// How many segments each (seq, value head) chain of a state-carrying kernel
// (the one-pass kernel, the two-pass state pass) is cut into.  Both run one
// CTA per SM (their shared memory and tensor memory fill one), so `heads`
// chains of `nchunks` chunks on `sms` SMs take
// ceil(heads / sms) rounds of the whole chain.  Cut into m segments, run in
// ceil(m heads / sms) launches of ceil(nchunks / m) chunks each, with about
// kRestartChunks chunks' worth of extra time per launch (the launch, the
// state load and the first chunk's copies).  A segment must land in a later
// launch than the one before it, which holds when heads >= sms.
constexpr double kRestartChunks = 1.5;
uint32_t state_segments(unsigned long long heads, uint32_t nchunks, unsigned long long sms) {
  auto cost = [&](uint32_t m) {
    const unsigned long long len = (nchunks + m - 1) / m, segs = (nchunks + len - 1) / len;
    return static_cast<double>((segs * heads + sms - 1) / sms) * (static_cast<double>(len) + kRestartChunks);
  };
  uint32_t best = 1;
  if (heads < sms) return best;
  for (uint32_t m = 2; m <= 8 && m <= nchunks; ++m)
    if (cost(m) < cost(best)) best = m;
  return best;
}

// Bounded wait on an mbarrier phase: about a second of clock at most.
__device__ __forceinline__ bool mbar_wait(uint32_t mbar, uint32_t phase) {
  const long long t0 = clock64();
  for (;;) {
    uint32_t done;
    asm volatile("{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
                 "selp.u32 %0, 1, 0, p;\n}\n" : "=r"(done) : "r"(mbar), "r"(phase) : "memory");
    if (done) return true;
    if (clock64() - t0 > 2000000000LL) return false;
  }
}

#define GDN_TMEM_LD32(taddr, v)                                                                \
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11," \
               "%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,"   \
               "%31}, [%32];\n"                                                                 \
               : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]),        \
                 "=r"(v[6]), "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]),      \
                 "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]),  \
                 "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),  \
                 "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]),  \
                 "=r"(v[30]), "=r"(v[31])                                                       \
               : "r"(taddr))
#define GDN_TMEM_ST32(taddr, v)                                                                 \
  asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10," \
               "%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,"  \
               "%30,%31,%32};\n"                                                               \
               :: "r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), \
                  "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]),          \
                  "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]),      \
                  "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]),      \
                  "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]),      \
                  "r"(v[30]), "r"(v[31]))
#define GDN_TMEM_ST16(taddr, v)                                                                 \
  asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10," \
               "%11,%12,%13,%14,%15,%16};\n"                                                   \
               :: "r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), \
                  "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]),          \
                  "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]))
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Scale the 64 TMEM columns [col, col+64) of this warp's 32 lanes by f.
__device__ __forceinline__ void tmem_scale64(uint32_t taddr, float f) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint32_t v[32];
    GDN_TMEM_LD32(taddr + 32 * h, v);
    tmem_wait_ld();
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * f);
    GDN_TMEM_ST32(taddr + 32 * h, v);
  }
  tmem_wait_st();
}

// The 16 x 16 block products of the triangular inverse run on the warp's
// tensor-core MMA (m16n8k8, TF32 operands) with each operand split as
// x = hi + lo, hi = tf32(x), lo = tf32(x - hi) (both to nearest; x - hi is
// exact), and C += A_lo B_hi + A_hi B_lo + A_hi B_hi, the small terms first:
// the three-term split of the same scheme the chunk products use in bf16,
// here with 11-bit halves, so each product keeps about 22 bits (the dropped
// A_lo B_lo term is below 2^-22 of it).  Per lane and block product that is
// 16 four-byte shared loads, one element each, against 24 sixteen-byte
// loads (each fetched by four or eight lanes) of a 2 x 4 tile of fma.
__device__ __forceinline__ void split_tf32(float x, uint32_t &hi, uint32_t &lo) {
  const float h = tf32_rn(x);
  hi = __float_as_uint(h);
  lo = __float_as_uint(tf32_rn(x - h));
}
__device__ __forceinline__ void mma_m16n8k8_tf32(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile("mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
               "{%0, %1, %2, %3};"
               : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
               : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// Column of element (r, c) in the product scratch M (16 x 16 blocks, row
// stride 16): columns swapped in halves of 8 on rows with bit 1 set, so
// that the B-fragment loads (rows t, t + 4, columns g) hit distinct banks.
__device__ __forceinline__ int mcol(int r, int c) { return c ^ (((r >> 1) & 1) << 3); }
// One warp accumulates C += L R for 16 x 16 blocks (L rows at stride ldl; R
// rows at stride ldr, or R = a block of M with ldr = 16 and RSWZ); C as two
// m16n8 accumulator fragments: c[nb] holds rows g, g + 8 and columns
// 8 nb + 2t, + 1 (g = lane / 4, t = lane % 4).  Where L is triangular its
// other half is stored zeros and multiplied like the rest.
template <bool RSWZ>
__device__ __forceinline__ void blk_mma(float (&c)[2][4], const float *L, int ldl, const float *R, int ldr,
                                        int lane) {
  const int g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int kb = 0; kb < 2; ++kb) {
    uint32_t ah[4], al[4];
    split_tf32(L[g * ldl + 8 * kb + t], ah[0], al[0]);
    split_tf32(L[(g + 8) * ldl + 8 * kb + t], ah[1], al[1]);
    split_tf32(L[g * ldl + 8 * kb + t + 4], ah[2], al[2]);
    split_tf32(L[(g + 8) * ldl + 8 * kb + t + 4], ah[3], al[3]);
#pragma unroll
    for (int nb = 0; nb < 2; ++nb) {
      const int r0 = 8 * kb + t, r1 = 8 * kb + t + 4, cn = 8 * nb + g;
      uint32_t b0h, b0l, b1h, b1l;
      split_tf32(R[r0 * ldr + (RSWZ ? mcol(r0, cn) : cn)], b0h, b0l);
      split_tf32(R[r1 * ldr + (RSWZ ? mcol(r1, cn) : cn)], b1h, b1l);
      mma_m16n8k8_tf32(c[nb], al, b0h, b1h);
      mma_m16n8k8_tf32(c[nb], ah, b0l, b1l);
      mma_m16n8k8_tf32(c[nb], ah, b0h, b1h);
    }
  }
}
// sign * C (fragments as above) to the 16 x 16 block at dst (row stride ld,
// or a block of M with SWZ).
template <bool SWZ>
__device__ __forceinline__ void blk_store(float *dst, int ld, const float (&c)[2][4], float sign, int lane) {
  const int g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int nb = 0; nb < 2; ++nb)
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int r = g + 8 * hh, cn = 8 * nb + 2 * t;
      *reinterpret_cast<float2 *>(dst + r * ld + (SWZ ? mcol(r, cn) : cn)) =
          make_float2(sign * c[nb][2 * hh], sign * c[nb][2 * hh + 1]);
    }
}

// Barrier of the NT threads running tri_inverse: the whole CTA, or warps
// 0-3 alone (named barrier 1) while the other warps do other work.
template <int NT>
__device__ __forceinline__ void tri_sync() {
  if constexpr (NT == NTH) __syncthreads();
  else asm volatile("bar.sync 1, %0;" :: "n"(NT) : "memory");
}

// T = (I + A)^-1 for a strictly lower 64 x 64 A (plain, row stride LD), by
// doubling over 16 x 16 blocks: the four diagonal blocks by forward
// substitution (one thread per column); then the two 32 x 32 diagonal blocks,
// T_{j+1,j} = -T_{j+1,j+1} (A_{j+1,j} T_jj) for j = 0, 2; then the lower-left
// 32 x 32 quarter, -T[hi] (A[hi,lo] T[lo]), as four 16 x 16 output blocks per
// product, one warp each (tensor-core fragments).  M is 4 x 256 floats of
// scratch for the inner products.  Run by threads 0 .. NT-1 (NT = 128: warps
// 0-3, which do all the work; NT = NTH: the whole CTA).
template <int NT = NTH>
__device__ void tri_inverse(const float *A, float *T, float *M, int tid) {
  static_assert(NT == NTH || NT == 128, "tri_inverse runs on the CTA or on warps 0-3");
  // the six blocks above the diagonal stay zero
  for (int e = tid; e < 6 * 256; e += NT) {
    const int b = e >> 8, rr = (e & 255) >> 4, cc = e & 15;
    const int bi = b < 3 ? 0 : (b < 5 ? 1 : 2), bj = b < 3 ? b + 1 : (b < 5 ? b - 1 : 3);
    T[(16 * bi + rr) * LD + 16 * bj + cc] = 0.f;
  }
  if (tid < 64) {
    const int base = 16 * (tid >> 4), cl = tid & 15;
    float x[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      float acc = (r == cl) ? 1.f : 0.f;
#pragma unroll
      for (int i = 0; i < r; ++i) acc = fmaf(-A[(base + r) * LD + base + i], x[i], acc);
      x[r] = acc;
    }
#pragma unroll
    for (int r = 0; r < 16; ++r) T[(base + r) * LD + base + cl] = x[r];
  }
  tri_sync<NT>();
  const int warp = tid >> 5, lane = tid & 31;
  float *mw = M + warp * 256;

  // 32 x 32 diagonal blocks: warp 0 builds T_10, warp 1 builds T_32
  if (warp < 2) {
    const int j = 2 * warp, i = j + 1;
    float m[2][4] = {};
    blk_mma<false>(m, A + (16 * i) * LD + 16 * j, LD, T + (16 * j) * LD + 16 * j, LD, lane);
    blk_store<true>(mw, 16, m, 1.f, lane);
    __syncwarp();
    float t[2][4] = {};
    blk_mma<true>(t, T + (16 * i) * LD + 16 * i, LD, mw, 16, lane);
    blk_store<false>(T + (16 * i) * LD + 16 * j, LD, t, -1.f, lane);
  }
  tri_sync<NT>();

  // lower-left quarter, rows r = 2, 3 and columns c = 0, 1 (16-blocks): warp
  // 2(r-2) + c first forms M'_rc = sum_{k=c}^{1} A_rk T_kc ...
  const int r = 2 + (warp >> 1), cb = warp & 1;
  if (warp < 4) {
    float m[2][4] = {};
    for (int k = cb; k <= 1; ++k)
      blk_mma<false>(m, A + (16 * r) * LD + 16 * k, LD, T + (16 * k) * LD + 16 * cb, LD, lane);
    blk_store<true>(mw, 16, m, 1.f, lane);
  }
  tri_sync<NT>();
  // ... then T_rc = -sum_{k=2}^{r} T_rk M'_kc (T_rr lower triangular)
  if (warp < 4) {
    float t[2][4] = {};
    if (r == 3)
      blk_mma<true>(t, T + (16 * r) * LD + 32, LD, M + cb * 256, 16, lane);  // T_32 M'_2c
    blk_mma<true>(t, T + (16 * r) * LD + 16 * r, LD, M + (2 * (r - 2) + cb) * 256, 16, lane);
    blk_store<false>(T + (16 * r) * LD + 16 * cb, LD, t, -1.f, lane);
  }
  tri_sync<NT>();
}

}  // namespace
}  // namespace chunked
}  // namespace gdn

// Sequential-scan kernel for long token ranges (prefill) on sm_103a.
//
// Same recurrence as the token-loop decode kernel (decay-first by default,
// the step order of the kernel body of "gated_delta_net_decode_capture.metal",
// mlx-native 0.9.2; decay-after as in the module-doc recurrence of
// "gated_delta_net.rs", mlx-native 0.4.0), laid out for arithmetic throughput
// instead of memory throughput:
//
// * P lanes share a state row (P = 2 or 4), each holding D_k/P cells in
//   registers (float4 chunks at d_k offsets 4P*i + 4*(lane%P)), so a row's
//   S@k and S@q take log2(P) shuffles each and a warp owns 32/P rows.  k_t is
//   held in registers for the token (used by S@k and by the update); lanes
//   with the same lane%P read the same k/q addresses from shared memory
//   (broadcast).
//
// * Lazy decay.  The state is kept as S = c * St, with c the product of the
//   decays since the last fold.  Then, per token t (c_t = c_{t-1} * alpha_t):
//       x     = St @ k_t
//       delta = (v_t - c_sk * x) * beta_t          c_sk = c_t (decay-first),
//                                                 c_{t-1} (decay-after)
//       St   += (delta / c_t) k_t^T
//       y_t   = q_scale * c_t * (St @ q_t)
//   which is the same recurrence with 3 FMAs per state cell instead of 4.
//   The c_t of a chunk of tokens come from a lane-parallel prefix sum of g
//   (c_t = exp(-G_t)); at the end of each chunk c is folded back into St.
//   If |G| would leave [-40, 40] inside a chunk (extreme gates, where c or
//   1/c could overflow), that chunk runs with the decay applied explicitly.
//
// * k, q, v (the CTA's rows), g and beta are staged into shared memory with
//   cp.async in chunks of TC tokens, double-buffered.  q, k, v and output
//   are f32 or bf16 (IO).  bf16 k and q are widened once per chunk into an
//   f32 copy in shared memory (every lane pair of a warp reads all of them,
//   so widening on each read would repeat the work 32/P times); v is widened
//   on its one read per row, and y is rounded once on store.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "device_io.cuh"
#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int TC = 16;            // tokens per staged chunk (<= 32: one lane per token)
constexpr float kMaxLogScale = 40.f;

struct ScanArgs {
  const void *__restrict__ q;
  const void *__restrict__ k;
  const void *__restrict__ v;
  const float *__restrict__ g;
  const float *__restrict__ beta;
  const float *state_in;  // may be the same buffer as state_out
  void *__restrict__ output;
  float *state_out;
  float *__restrict__ capture;
  uint32_t dv, nk, nv, nt, group, khead_div;
  float q_scale;
  uint32_t row_blocks;
};

__device__ __forceinline__ float dot4(const float4 a, const float4 b, float acc) {
  acc = fmaf(a.x, b.x, acc);
  acc = fmaf(a.y, b.y, acc);
  acc = fmaf(a.z, b.z, acc);
  return fmaf(a.w, b.w, acc);
}
__device__ __forceinline__ void axpy4(float a, const float4 x, float4 &y) {
  y.x = fmaf(a, x.x, y.x);
  y.y = fmaf(a, x.y, y.y);
  y.z = fmaf(a, x.z, y.z);
  y.w = fmaf(a, x.w, y.w);
}
__device__ __forceinline__ void scale4(float a, float4 &y) {
  y.x *= a; y.y *= a; y.z *= a; y.w *= a;
}
// Pairwise sum of N partials (N a power of two): ((a0 + a1) + (a2 + a3)) ...
template <int N>
__device__ __forceinline__ float tree_sum(float (&a)[N]) {
#pragma unroll
  for (int h = N / 2; h >= 1; h >>= 1) {
#pragma unroll
    for (int i = 0; i < h; ++i) a[i] = a[2 * i] + a[2 * i + 1];
  }
  return a[0];
}

constexpr int kScanP = 2;    // lanes per state row (4 measured slower at D_k = 128)
constexpr int kScanAcc = 4;  // independent partial sums per dot product

// Bytes of one staging buffer: k[TC][DK] q[TC][DK] v[TC][ROWS] (IO), then
// g[TC] beta[TC] (f32); a multiple of 16 for every DK and ROWS used here.
template <typename IO, int DK, int ROWS>
constexpr int scan_staging_bytes() {
  return TC * ((2 * DK + ROWS) * static_cast<int>(sizeof(IO)) + 8);
}
// Bytes of the f32 copy of one chunk's k and q (bf16 activations only).
template <typename IO, int DK>
constexpr int scan_widened_bytes() {
  return sizeof(IO) == sizeof(float) ? 0 : TC * 2 * DK * static_cast<int>(sizeof(float));
}

template <typename IO, int NSG, int P, int WARPS, bool CAPTURE, bool DECAY_AFTER>
__global__ void __launch_bounds__(WARPS * 32, P == 2 ? 3 : 5) gdn_scan_kernel(const ScanArgs a) {
  constexpr int DK = 32 * NSG;
  constexpr int NC = DK / (4 * P);      // 4-cell chunks per lane (each lane holds DK/P cells)
  constexpr int NA = NC < kScanAcc ? NC : kScanAcc;  // accumulators per dot product
  constexpr int RPW = 32 / P;           // rows per warp
  constexpr int ROWS = WARPS * RPW;     // rows per CTA
  constexpr int E16 = 16 / static_cast<int>(sizeof(IO));  // elements per 16-byte copy
  constexpr int E4 = Act<IO>::kPer4B;                      // elements per 4-byte copy
  static_assert(P == 2 || P == 4, "two or four lanes per row");
  constexpr int BUF = scan_staging_bytes<IO, DK, ROWS>();
  static_assert(BUF % 16 == 0, "staging buffers must stay 16-byte aligned");
  static_assert(DK % E16 == 0 && ROWS % E4 == 0, "staging granularity");
  constexpr bool WIDEN = sizeof(IO) != sizeof(float);

  extern __shared__ __align__(16) unsigned char smem[];
  float *const kq32 = reinterpret_cast<float *>(smem + 2 * BUF);  // WIDEN: k[TC][DK] q[TC][DK]
  const uint32_t rb = blockIdx.x % a.row_blocks;
  const uint32_t head = blockIdx.x / a.row_blocks;  // = s * nv + vh
  const uint32_t vh = head % a.nv;
  const uint32_t s = head / a.nv;
  const uint32_t kh = a.khead_div ? vh / a.group : vh % a.nk;
  const int warp = static_cast<int>(threadIdx.x >> 5);
  const int lane = static_cast<int>(threadIdx.x & 31);
  const int part = lane % P;
  const int row_in_cta = warp * RPW + lane / P;
  const uint32_t row_cta0 = rb * ROWS;
  const uint32_t row = row_cta0 + row_in_cta;
  const bool row_ok = row < a.dv;
  const uint32_t nt = a.nt;

  // This lane's cells of its state row, loaded first.
  const size_t state_row = (static_cast<size_t>(head) * a.dv + row) * DK;
  float4 st[NC];
#pragma unroll
  for (int i = 0; i < NC; ++i)
    st[i] = row_ok ? __ldcs(reinterpret_cast<const float4 *>(a.state_in + state_row + 4 * P * i + 4 * part))
                   : make_float4(0.f, 0.f, 0.f, 0.f);

  const size_t kq_tok = static_cast<size_t>(a.nk) * DK;
  const size_t kq_first = (static_cast<size_t>(s) * nt * a.nk + kh) * DK;
  const size_t v_tok = static_cast<size_t>(a.nv) * a.dv;
  const size_t v_first = (static_cast<size_t>(s) * nt * a.nv + vh) * a.dv + row_cta0;
  const size_t sc_first = static_cast<size_t>(s) * nt * a.nv + vh;

  const IO *gk = static_cast<const IO *>(a.k);
  const IO *gq = static_cast<const IO *>(a.q);
  const IO *gv = static_cast<const IO *>(a.v);
  IO *gout = static_cast<IO *>(a.output);

  auto stage = [&](uint32_t chunk, int buf) {
    IO *ks = reinterpret_cast<IO *>(smem + buf * BUF);
    IO *qs = ks + TC * DK;
    IO *vs = qs + TC * DK;
    float *gs = reinterpret_cast<float *>(vs + TC * ROWS);
    float *bs = gs + TC;
    const uint32_t t0 = chunk * TC;
    const int n = static_cast<int>(min(static_cast<uint32_t>(TC), nt - t0));
    for (int i = threadIdx.x; i < n * (DK / E16); i += WARPS * 32) {
      const int t = i / (DK / E16), e = E16 * (i % (DK / E16));
      const size_t src = kq_first + (t0 + t) * kq_tok + e;
      cp_async_16(ks + t * DK + e, gk + src);
      cp_async_16(qs + t * DK + e, gq + src);
    }
    // v in 4-byte units (one f32 or two bf16 rows; D_v is even for bf16)
    for (int i = threadIdx.x; i < n * (ROWS / E4); i += WARPS * 32) {
      const int t = i / (ROWS / E4), r = E4 * (i % (ROWS / E4));
      if (row_cta0 + r < a.dv) {
        cp_async_4(vs + t * ROWS + r, gv + v_first + (t0 + t) * v_tok + r);
      } else {
#pragma unroll
        for (int u = 0; u < E4; ++u) Act<IO>::put(vs + t * ROWS + r + u, 0.f);
      }
    }
    for (int i = threadIdx.x; i < n; i += WARPS * 32) {
      const size_t src = sc_first + static_cast<size_t>(t0 + i) * a.nv;
      cp_async_4(gs + i, a.g + src);
      cp_async_4(bs + i, a.beta + src);
    }
    cp_async_commit();
  };

  const uint32_t nchunks = (nt + TC - 1) / TC;
  stage(0, 0);
  for (uint32_t c = 0; c < nchunks; ++c) {
    if (c + 1 < nchunks) {
      stage(c + 1, (c + 1) & 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();

    const IO *ks = reinterpret_cast<const IO *>(smem + (c & 1) * BUF);
    const IO *qs = ks + TC * DK;
    const IO *vs = qs + TC * DK;
    const float *gs = reinterpret_cast<const float *>(vs + TC * ROWS);
    const float *bs = gs + TC;
    const uint32_t t0 = c * TC;
    const int n = static_cast<int>(min(static_cast<uint32_t>(TC), nt - t0));

    const float *kf;  // this chunk's k and q as f32
    const float *qf;
    if constexpr (WIDEN) {
      // k and q are adjacent in the staging buffer and in kq32
      for (int i = threadIdx.x; i < 2 * TC * DK / 4; i += WARPS * 32) {
        float c4[4];
        Act<IO>::template get_n<4>(ks + 4 * i, c4);
        *reinterpret_cast<float4 *>(kq32 + 4 * i) = make_float4(c4[0], c4[1], c4[2], c4[3]);
      }
      __syncthreads();
      kf = kq32;
      qf = kq32 + TC * DK;
    } else {
      kf = reinterpret_cast<const float *>(ks);
      qf = reinterpret_cast<const float *>(qs);
    }

    // Per-token scalars of this chunk: lane t holds those of token t.
    const float gl = lane < n ? gs[lane] : 0.f;
    const float bl = lane < n ? bs[lane] : 0.f;
    float G = gl;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float up = __shfl_up_sync(kFull, G, o);
      if (lane >= o) G += up;
    }
    const bool direct = __any_sync(kFull, fabsf(G) > kMaxLogScale);
    const float cl = direct ? 1.f : expf(-G);
    float cprev = __shfl_up_sync(kFull, cl, 1);
    if (lane == 0) cprev = 1.f;
    const float csk_l = DECAY_AFTER ? cprev : cl;
    const float binv_l = bl / cl;
    const float alpha_l = direct ? expf(-gl) : 1.f;
    const float c_last = __shfl_sync(kFull, cl, n - 1);

    for (int tt = 0; tt < n; ++tt) {
      const float c_t = __shfl_sync(kFull, cl, tt);
      const float csk = __shfl_sync(kFull, csk_l, tt);
      const float binv = __shfl_sync(kFull, binv_l, tt);
      const float4 *kr = reinterpret_cast<const float4 *>(kf + tt * DK + 4 * part);
      const float4 *qr = reinterpret_cast<const float4 *>(qf + tt * DK + 4 * part);
      float4 kk[NC];
#pragma unroll
      for (int i = 0; i < NC; ++i) kk[i] = kr[P * i];
      if (direct && !DECAY_AFTER) {
        const float at = __shfl_sync(kFull, alpha_l, tt);
#pragma unroll
        for (int i = 0; i < NC; ++i) scale4(at, st[i]);
      }
      float pa[NA];
#pragma unroll
      for (int j = 0; j < NA; ++j) pa[j] = 0.f;
#pragma unroll
      for (int i = 0; i < NC; ++i) pa[i % NA] = dot4(st[i], kk[i], pa[i % NA]);
      float x = tree_sum<NA>(pa);
#pragma unroll
      for (int o = 1; o < P; o <<= 1) x += __shfl_xor_sync(kFull, x, o);
      if (direct && DECAY_AFTER) {
        const float at = __shfl_sync(kFull, alpha_l, tt);
#pragma unroll
        for (int i = 0; i < NC; ++i) scale4(at, st[i]);
      }
      const float d = (Act<IO>::get(vs + tt * ROWS + row_in_cta) - csk * x) * binv;
      float ya[NA];
#pragma unroll
      for (int j = 0; j < NA; ++j) ya[j] = 0.f;
#pragma unroll
      for (int i = 0; i < NC; ++i) {
        axpy4(d, kk[i], st[i]);
        ya[i % NA] = dot4(st[i], qr[P * i], ya[i % NA]);
      }
      float y = tree_sum<NA>(ya);
#pragma unroll
      for (int o = 1; o < P; o <<= 1) y += __shfl_xor_sync(kFull, y, o);
      const size_t tok_head = (static_cast<size_t>(s) * nt + t0 + tt) * a.nv + vh;
      if (part == 0 && row_ok) Act<IO>::put(gout + tok_head * a.dv + row, y * (c_t * a.q_scale));
      if (CAPTURE && row_ok) {
        float *cap = a.capture + (tok_head * a.dv + row) * DK + 4 * part;
#pragma unroll
        for (int i = 0; i < NC; ++i) {
          float4 o = st[i];
          scale4(c_t, o);
          __stcs(reinterpret_cast<float4 *>(cap + 4 * P * i), o);
        }
      }
    }
    if (!direct) {
#pragma unroll
      for (int i = 0; i < NC; ++i) scale4(c_last, st[i]);
    }
    __syncthreads();  // this buffer is refilled by the stage() of chunk c+2
  }

  if (row_ok) {
#pragma unroll
    for (int i = 0; i < NC; ++i)
      __stcs(reinterpret_cast<float4 *>(a.state_out + state_row + 4 * P * i + 4 * part), st[i]);
  }
}

// Lanes per row (kScanP, above) and warps per CTA: 4 warps (64 rows) for
// D_k >= 64; at D_k = 32 (D_v = 32 rows per head) 2 warps, so no warp of the
// CTA lies past the head's rows (measured: 0.286 -> 0.238 ms on 1024 tokens;
// 4 lanes per row was slower at every D_k).
template <int NSG> constexpr int kScanPFor = kScanP;
template <int NSG> constexpr int kScanWarpsFor = NSG == 1 ? 2 : 4;

template <typename IO, int NSG, bool CAPTURE, bool DA>
cudaError_t launch(const Problem &p, cudaStream_t stream) {
  constexpr int DK = 32 * NSG;
  constexpr int kP = kScanPFor<NSG>, kW = kScanWarpsFor<NSG>;
  constexpr int ROWS = kW * (32 / kP);
  ScanArgs a;
  a.q = p.q; a.k = p.k; a.v = p.v; a.g = p.g; a.beta = p.beta;
  a.state_in = p.state_in; a.output = p.output; a.state_out = p.state_out; a.capture = p.capture;
  a.dv = p.dv; a.nk = p.nk; a.nv = p.nv; a.nt = p.nt;
  a.group = p.nv / p.nk;
  a.khead_div = p.khead_div ? 1u : 0u;
  a.q_scale = p.q_scale;
  a.row_blocks = (p.dv + ROWS - 1) / ROWS;
  const unsigned long long blocks =
      static_cast<unsigned long long>(a.row_blocks) * p.nv * static_cast<unsigned long long>(p.ns);
  if (blocks == 0 || blocks > 0x7fffffffull) return cudaErrorInvalidConfiguration;
  const size_t smem = 2u * scan_staging_bytes<IO, DK, ROWS>() + scan_widened_bytes<IO, DK>();
  auto kern = gdn_scan_kernel<IO, NSG, kP, kW, CAPTURE, DA>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  kern<<<static_cast<unsigned>(blocks), kW * 32, smem, stream>>>(a);
  return cudaGetLastError();
}

template <typename IO, int NSG>
cudaError_t launch_nsg(const Problem &p, cudaStream_t stream) {
  const bool cap = p.capture != nullptr;
  if (cap)
    return p.decay_after ? launch<IO, NSG, true, true>(p, stream) : launch<IO, NSG, true, false>(p, stream);
  return p.decay_after ? launch<IO, NSG, false, true>(p, stream) : launch<IO, NSG, false, false>(p, stream);
}

template <typename IO>
cudaError_t launch_io(const Problem &p, cudaStream_t stream) {
  switch (p.dk) {
    case 32: return launch_nsg<IO, 1>(p, stream);
    case 64: return launch_nsg<IO, 2>(p, stream);
    case 128: return launch_nsg<IO, 4>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_scan(const Problem &p, cudaStream_t stream) {
  if (p.io_bf16) {
    if (p.dv % 2 != 0) return cudaErrorInvalidValue;  // v is staged two bf16 rows at a time
    return launch_io<__nv_bfloat16>(p, stream);
  }
  return launch_io<float>(p, stream);
}

}  // namespace gdn

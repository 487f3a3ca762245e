// Token-loop kernel for the Gated DeltaNet recurrence on sm_103a: decode and
// short multi-token windows, with optional per-token state capture.  Long
// token ranges use the scan kernel (scan.cu) instead.
//
// Work decomposition.  The D_v rows of a (seq, value head) state are
// independent (each row i only meets v_t[i] and the shared k_t, q_t), so a
// warp owns R consecutive rows and a CTA owns WARPS*R rows of one pair.
// Lane l keeps the D_k/32 contiguous f32 cells [l*NSG, l*NSG+NSG) of each of
// its R rows in registers for the whole token range (NSG = D_k/32), as the
// capture kernel of "gated_delta_net_decode_capture.metal" (mlx-native 0.9.2)
// keeps NSG cells per lane; state therefore crosses HBM once in and once out
// per call whatever n_tokens is ("Threading" section of gated_delta_net.rs,
// mlx-native 0.4.0).  Loads and stores of state are coalesced 128-bit
// (D_k = 128) streaming accesses.
//
// Per token (decay-first; the kernel body's steps "decay + partial s_k" and
// "state update + output partial"):
//     S *= alpha;  sk = S@k;  delta = (v - sk)*beta;  S += delta k^T;  y = S@q
// The two row reductions (S@k, S@q) are warp reductions over the 32 lanes.
// Reducing R rows at once uses a transpose-reduce: at each of log2(R)
// butterfly stages a lane keeps half of its remaining row partials and
// trades the other half with its partner, so R rows cost R-1+5-log2(R)
// shuffles instead of 5R; lane l ends with the total of row l/(32/R).
//
// k_t, q_t (shared by every row of the CTA), v_t for the CTA's rows, g_t and
// beta_t are staged into shared memory with cp.async, in chunks of `tc`
// tokens, double-buffered so the next chunk loads while this one computes.
// q, k, v and output are f32 or bf16 (IO); staging keeps the stored type and
// widens to f32 on the shared-memory read, and y is rounded once on store.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "device_io.cuh"
#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr unsigned kFull = 0xffffffffu;

struct LayerPtrs {
  const void *q, *k, *v;
  const float *g, *beta, *state_in;
  void *output;
  float *state_out, *capture;
};

struct LoopArgs {
  uint32_t dv, nk, nv, nt, group, khead_div;
  float q_scale;
  uint32_t row_blocks;    // CTAs per (seq, value head) pair
  uint32_t layer_blocks;  // CTAs per layer = row_blocks * nv * ns
  uint32_t tc;            // tokens per staged chunk
};

// ---- NSG contiguous floats per lane: streaming global and plain shared I/O

template <int NSG>
struct Cells;
template <>
struct Cells<4> {
  static __device__ __forceinline__ void load_cs(const float *p, float (&c)[4]) {
    const float4 x = __ldcs(reinterpret_cast<const float4 *>(p));
    c[0] = x.x; c[1] = x.y; c[2] = x.z; c[3] = x.w;
  }
  static __device__ __forceinline__ void store_cs(float *p, const float (&c)[4]) {
    __stcs(reinterpret_cast<float4 *>(p), make_float4(c[0], c[1], c[2], c[3]));
  }
};
template <>
struct Cells<2> {
  static __device__ __forceinline__ void load_cs(const float *p, float (&c)[2]) {
    const float2 x = __ldcs(reinterpret_cast<const float2 *>(p));
    c[0] = x.x; c[1] = x.y;
  }
  static __device__ __forceinline__ void store_cs(float *p, const float (&c)[2]) {
    __stcs(reinterpret_cast<float2 *>(p), make_float2(c[0], c[1]));
  }
};
template <>
struct Cells<1> {
  static __device__ __forceinline__ void load_cs(const float *p, float (&c)[1]) { c[0] = __ldcs(p); }
  static __device__ __forceinline__ void store_cs(float *p, const float (&c)[1]) { __stcs(p, c[0]); }
};

// Transpose-reduce R per-lane partials over the warp.  Returns, in every
// lane l, the warp-wide total of row l / (32/R).
template <int R>
__device__ __forceinline__ float reduce_rows(float (&a)[R], int lane) {
#pragma unroll
  for (int m = R, o = 16; m > 1; m >>= 1, o >>= 1) {
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < m / 2; ++i) {
      const float send = upper ? a[i] : a[i + m / 2];
      const float keep = upper ? a[i + m / 2] : a[i];
      a[i] = keep + __shfl_xor_sync(kFull, send, o);
    }
  }
  float x = a[0];
#pragma unroll
  for (int o = 16 / R; o >= 1; o >>= 1) x += __shfl_xor_sync(kFull, x, o);
  return x;
}

// Up to MAXL problems of the same shape (e.g. the linear-attention layers of
// one forward pass) in one launch: CTA blocks are layer-major, and each CTA
// reads its layer's buffers from this table in the kernel parameters.
template <int MAXL>
struct LayerTable {
  LayerPtrs l[MAXL];
};

// Bytes of one staging buffer: k[tc][DK] q[tc][DK] v[tc][ROWS] (IO) then
// g[tc] beta[tc] (f32), padded so both buffers start 16-byte aligned.
template <typename IO, int DK, int ROWS>
__host__ __device__ constexpr int staging_bytes(int tc) {
  return (tc * ((2 * DK + ROWS) * static_cast<int>(sizeof(IO)) + 8) + 15) & ~15;
}

// Single-layer launches leave the register count to the compiler (48 at
// D_k = 128: five 8-warp CTAs per SM); multi-layer launches are held to 64.
template <typename IO, int NSG, int R, int WARPS, bool CAPTURE, bool DECAY_AFTER, int MAXL>
__global__ void __launch_bounds__(WARPS * 32, MAXL == 1 ? 0 : 32 / WARPS)
    gdn_token_loop_kernel(const LoopArgs a, const LayerPtrs one,
                          const __grid_constant__ LayerTable<MAXL> tab) {
  constexpr int DK = 32 * NSG;
  constexpr int ROWS = WARPS * R;  // rows per CTA
  constexpr int LPR = 32 / R;      // lanes that end up holding one row's total
  constexpr int E16 = 16 / static_cast<int>(sizeof(IO));  // elements per 16-byte copy
  constexpr int E4 = Act<IO>::kPer4B;                      // elements per 4-byte copy
  static_assert(R >= 1 && R <= 32 && (R & (R - 1)) == 0, "R must be a power of two <= 32");
  static_assert(DK % E16 == 0 && ROWS % E4 == 0, "staging granularity");

  extern __shared__ __align__(16) unsigned char smem[];
  const int tc = static_cast<int>(a.tc);
  const int buf_bytes = staging_bytes<IO, DK, ROWS>(tc);

  const uint32_t layer = MAXL == 1 ? 0u : blockIdx.x / a.layer_blocks;
  const uint32_t bid = blockIdx.x - layer * a.layer_blocks;
  // Buffer pointers: `one` when the launch has a single layer, else this
  // CTA's entry of the table.
#define GDN_LAYER(field) (MAXL == 1 ? one.field : tab.l[layer].field)
  const uint32_t rb = bid % a.row_blocks;
  const uint32_t head = bid / a.row_blocks;  // = s * nv + vh
  const uint32_t vh = head % a.nv;
  const uint32_t s = head / a.nv;
  const uint32_t kh = a.khead_div ? vh / a.group : vh % a.nk;
  const int warp = static_cast<int>(threadIdx.x >> 5);
  const int lane = static_cast<int>(threadIdx.x & 31);
  const uint32_t row_cta0 = rb * ROWS;
  const uint32_t row0 = row_cta0 + static_cast<uint32_t>(warp * R);
  const uint32_t nt = a.nt;

  // 1. Issue the state loads first: they are the bulk of the HBM traffic.
  const size_t state_head = static_cast<size_t>(head) * a.dv * DK;
  float st[R][NSG];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    if (row0 + r < a.dv) {
      Cells<NSG>::load_cs(GDN_LAYER(state_in) + state_head + static_cast<size_t>(row0 + r) * DK + lane * NSG,
                          st[r]);
    } else {
#pragma unroll
      for (int j = 0; j < NSG; ++j) st[r][j] = 0.f;
    }
  }

  // 2. Staging of per-token inputs.
  const size_t kq_tok = static_cast<size_t>(a.nk) * DK;
  const size_t kq_first = (static_cast<size_t>(s) * nt * a.nk + kh) * DK;
  const size_t v_tok = static_cast<size_t>(a.nv) * a.dv;
  const size_t v_first = (static_cast<size_t>(s) * nt * a.nv + vh) * a.dv + row_cta0;
  const size_t sc_first = static_cast<size_t>(s) * nt * a.nv + vh;  // token stride nv

  const IO *gk = static_cast<const IO *>(GDN_LAYER(k));
  const IO *gq = static_cast<const IO *>(GDN_LAYER(q));
  const IO *gv = static_cast<const IO *>(GDN_LAYER(v));
  IO *gout = static_cast<IO *>(GDN_LAYER(output));

  auto stage = [&](uint32_t chunk, int buf) {
    IO *ks = reinterpret_cast<IO *>(smem + buf * buf_bytes);
    IO *qs = ks + tc * DK;
    IO *vs = qs + tc * DK;
    float *gs = reinterpret_cast<float *>(vs + tc * ROWS);
    float *bs = gs + tc;
    const uint32_t t0 = chunk * static_cast<uint32_t>(tc);
    const int n = static_cast<int>(min(static_cast<uint32_t>(tc), nt - t0));
    for (int i = threadIdx.x; i < n * (DK / E16); i += WARPS * 32) {
      const int t = i / (DK / E16), e = E16 * (i % (DK / E16));
      const size_t src = kq_first + (t0 + t) * kq_tok + e;
      cp_async_16(ks + t * DK + e, gk + src);
      cp_async_16(qs + t * DK + e, gq + src);
    }
    // v in 4-byte units (one f32 or two bf16 rows; D_v is even for bf16, so a
    // unit is either wholly inside the head or wholly past its last row)
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
      cp_async_4(gs + i, GDN_LAYER(g) + src);
      cp_async_4(bs + i, GDN_LAYER(beta) + src);
    }
    cp_async_commit();
  };

  const uint32_t nchunks = (nt + tc - 1) / tc;
  const int my_r = lane / LPR;  // the row whose totals this lane ends up holding
  const uint32_t my_row = row0 + my_r;

  stage(0, 0);
  for (uint32_t c = 0; c < nchunks; ++c) {
    if (c + 1 < nchunks) {
      stage(c + 1, (c + 1) & 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();

    const IO *ks = reinterpret_cast<const IO *>(smem + (c & 1) * buf_bytes);
    const IO *qs = ks + tc * DK;
    const IO *vs = qs + tc * DK;
    const float *gs = reinterpret_cast<const float *>(vs + tc * ROWS);
    const float *bs = gs + tc;
    const int n = static_cast<int>(min(static_cast<uint32_t>(tc), nt - c * tc));

    for (int tt = 0; tt < n; ++tt) {
      const uint32_t t = c * tc + tt;
      float kk[NSG], qq[NSG];
      Act<IO>::template get_n<NSG>(ks + tt * DK + lane * NSG, kk);
      Act<IO>::template get_n<NSG>(qs + tt * DK + lane * NSG, qq);
      const float alpha = expf(-gs[tt]);
      const float b = bs[tt];

      // S@k (on the decayed state for decay-first, the old one for decay-after)
      float part[R];
#pragma unroll
      for (int r = 0; r < R; ++r) {
        part[r] = 0.f;
#pragma unroll
        for (int j = 0; j < NSG; ++j) {
          if (!DECAY_AFTER) st[r][j] *= alpha;
          part[r] = fmaf(st[r][j], kk[j], part[r]);
        }
      }
      const float sk = reduce_rows<R>(part, lane);
      const float d = (Act<IO>::get(vs + tt * ROWS + warp * R + my_r) - sk) * b;

      // rank-1 update and S@q
      float py[R];
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const float dr = __shfl_sync(kFull, d, r * LPR);
        py[r] = 0.f;
#pragma unroll
        for (int j = 0; j < NSG; ++j) {
          if (DECAY_AFTER)
            st[r][j] = fmaf(alpha, st[r][j], dr * kk[j]);
          else
            st[r][j] = fmaf(dr, kk[j], st[r][j]);
          py[r] = fmaf(st[r][j], qq[j], py[r]);
        }
      }
      const float y = reduce_rows<R>(py, lane);
      const size_t tok_head = (static_cast<size_t>(s) * nt + t) * a.nv + vh;
      if ((lane % LPR) == 0 && my_row < a.dv) Act<IO>::put(gout + tok_head * a.dv + my_row, y * a.q_scale);

      if (CAPTURE) {
        float *cap = GDN_LAYER(capture) + tok_head * a.dv * DK;
#pragma unroll
        for (int r = 0; r < R; ++r)
          if (row0 + r < a.dv)
            Cells<NSG>::store_cs(cap + static_cast<size_t>(row0 + r) * DK + lane * NSG, st[r]);
      }
    }
    __syncthreads();  // this buffer is refilled by the stage() of chunk c+2
  }

  // 3. Final state, from the same registers as the last capture slice.
#pragma unroll
  for (int r = 0; r < R; ++r)
    if (row0 + r < a.dv)
      Cells<NSG>::store_cs(GDN_LAYER(state_out) + state_head + static_cast<size_t>(row0 + r) * DK + lane * NSG,
                           st[r]);
#undef GDN_LAYER
}

// ---- launch shape: several rows per warp (R = 16/NSG, 64 B of state per
// lane) and small CTAs (8 KB of state per CTA), so each SM keeps tens of KB
// of state loads in flight across many CTAs and the fixed cost of a CTA is
// shared by few rows; tokens are staged 8 at a time.  4 warps for
// D_k >= 64; at D_k = 32 a warp already holds 16 rows, so 2 warps (32 rows:
// one value head of D_v = 32 per CTA).  (Measured: at D_k = 128, 4 warps beat
// 8 by 8 % on 32 one-sequence layers per launch and by 1 % on 64-sequence
// decode; at D_k = 32, 2 warps reach 0.88 of the HBM roofline where 4 reach
// 0.55, half their rows lying past D_v.)

template <int NSG>
constexpr int kWarpsFor = NSG == 1 ? 2 : 4;
constexpr int kTcMax = 8;

template <typename IO, int NSG, bool CAPTURE, bool DA, int MAXL>
cudaError_t launch_layers(const Problem &p, const Problem *layers, uint32_t n_layers,
                          cudaStream_t stream) {
  constexpr int R = 16 / NSG;
  constexpr int kWarps = kWarpsFor<NSG>;
  constexpr int ROWS = kWarps * R;
  constexpr int DK = 32 * NSG;
  LoopArgs a;
  a.dv = p.dv; a.nk = p.nk; a.nv = p.nv; a.nt = p.nt;
  a.group = p.nv / p.nk;
  a.khead_div = p.khead_div ? 1u : 0u;
  a.q_scale = p.q_scale;
  a.row_blocks = (p.dv + ROWS - 1) / ROWS;
  a.tc = static_cast<uint32_t>(p.nt < static_cast<uint32_t>(kTcMax) ? p.nt : kTcMax);
  const unsigned long long per_layer =
      static_cast<unsigned long long>(a.row_blocks) * p.nv * static_cast<unsigned long long>(p.ns);
  if (per_layer == 0 || per_layer * n_layers > 0x7fffffffull || n_layers == 0 || n_layers > MAXL)
    return cudaErrorInvalidConfiguration;
  a.layer_blocks = static_cast<uint32_t>(per_layer);
  LayerTable<MAXL> t;
  for (uint32_t i = 0; i < n_layers; ++i) {
    const Problem &x = layers[i];
    t.l[i] = LayerPtrs{x.q, x.k, x.v, x.g, x.beta, x.state_in, x.output, x.state_out, x.capture};
  }
  const LayerPtrs one = t.l[0];
  const size_t smem = 2u * static_cast<size_t>(staging_bytes<IO, DK, ROWS>(static_cast<int>(a.tc)));
  gdn_token_loop_kernel<IO, NSG, R, kWarps, CAPTURE, DA, MAXL>
      <<<static_cast<unsigned>(per_layer * n_layers), kWarps * 32, smem, stream>>>(a, one, t);
  return cudaGetLastError();
}

template <typename IO, int NSG, int MAXL>
cudaError_t launch_nsg(const Problem &p, const Problem *layers, uint32_t n, cudaStream_t stream) {
  const bool cap = p.capture != nullptr;
  if (cap)
    return p.decay_after ? launch_layers<IO, NSG, true, true, MAXL>(p, layers, n, stream)
                         : launch_layers<IO, NSG, true, false, MAXL>(p, layers, n, stream);
  return p.decay_after ? launch_layers<IO, NSG, false, true, MAXL>(p, layers, n, stream)
                       : launch_layers<IO, NSG, false, false, MAXL>(p, layers, n, stream);
}

template <typename IO, int MAXL>
cudaError_t launch_io(const Problem &p, const Problem *layers, uint32_t n, cudaStream_t stream) {
  switch (p.dk) {
    case 32: return launch_nsg<IO, 1, MAXL>(p, layers, n, stream);
    case 64: return launch_nsg<IO, 2, MAXL>(p, layers, n, stream);
    case 128: return launch_nsg<IO, 4, MAXL>(p, layers, n, stream);
    default: return cudaErrorInvalidValue;
  }
}

template <int MAXL>
cudaError_t launch_dk(const Problem &p, const Problem *layers, uint32_t n, cudaStream_t stream) {
  if (p.io_bf16) {
    if (p.dv % 2 != 0) return cudaErrorInvalidValue;  // v is staged two bf16 rows at a time
    return launch_io<__nv_bfloat16, MAXL>(p, layers, n, stream);
  }
  return launch_io<float, MAXL>(p, layers, n, stream);
}

}  // namespace

cudaError_t launch_token_loop(const Problem &p, cudaStream_t stream) {
  return launch_dk<1>(p, &p, 1, stream);
}

cudaError_t launch_token_loop_layers(const Problem *layers, uint32_t n_layers, cudaStream_t stream) {
  for (uint32_t i = 0; i < n_layers; i += kMaxLayersPerLaunch) {
    const uint32_t n = n_layers - i < kMaxLayersPerLaunch ? n_layers - i : kMaxLayersPerLaunch;
    const cudaError_t e = launch_dk<kMaxLayersPerLaunch>(layers[i], layers + i, n, stream);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace gdn

// Token-loop kernel for the Gated DeltaNet recurrence on sm_103a: decode and
// short multi-token windows, with optional per-token state capture.  Long
// token ranges use the scan kernel (scan.cu) instead.
//
// Work decomposition.  The D_v rows of a (seq, value head) state are
// independent (each row i only meets v_t[i] and the shared k_t, q_t), so a
// warp owns R consecutive rows and a CTA owns WARPS*R rows of one pair.
// A row is spread over LR = D_k/CW lanes, each keeping CW contiguous f32
// cells of it in registers for the whole token range; one warp-wide access
// thus covers RPI = 32/LR consecutive rows, and a lane holds J = R/RPI rows
// (slots), row j*RPI + lane/LR of the warp's R in slot j.  With CW = D_k/32
// (one row per access, the D_k = 128 and 64 shapes) this is the layout of the
// capture kernel of "gated_delta_net_decode_capture.metal" (mlx-native
// 0.9.2), NSG cells per lane; at D_k = 32, CW = 4 puts a row on 8 lanes so
// that state moves in 128-bit accesses there too.  State crosses HBM once in
// and once out per call whatever n_tokens is ("Threading" section of
// gated_delta_net.rs, mlx-native 0.4.0).
//
// Per token (decay-first; the kernel body's steps "decay + partial s_k" and
// "state update + output partial"):
//     S *= alpha;  sk = S@k;  delta = (v - sk)*beta;  S += delta k^T;  y = S@q
// The two row reductions (S@k, S@q) are reductions over a row's LR lanes.
// Reducing J slots at once uses a transpose-reduce: at each of log2(J)
// butterfly stages a lane keeps half of its remaining slot partials and
// trades the other half with its partner, so J slots cost
// J-1+log2(LR)-log2(J) shuffles instead of J*log2(LR); lane l ends with the
// total of slot (l % LR)/(LR/J) of its row group l/LR.
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

// Transpose-reduce J per-lane partials over groups of LR lanes.  Returns, in
// every lane l, the total over its group of slot (l % LR) / (LR/J).
template <int J, int LR>
__device__ __forceinline__ float reduce_slots(float (&a)[J], int lane) {
#pragma unroll
  for (int m = J, o = LR / 2; m > 1; m >>= 1, o >>= 1) {
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
  for (int o = LR / (2 * J); o >= 1; o >>= 1) x += __shfl_xor_sync(kFull, x, o);
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
template <typename IO, int NSG, int CW, int R, int WARPS, bool CAPTURE, bool DECAY_AFTER, int MAXL>
__global__ void __launch_bounds__(WARPS * 32, MAXL == 1 ? 0 : 32 / WARPS)
    gdn_token_loop_kernel(const LoopArgs a, const LayerPtrs one,
                          const __grid_constant__ LayerTable<MAXL> tab) {
  constexpr int DK = 32 * NSG;
  constexpr int ROWS = WARPS * R;  // rows per CTA
  constexpr int LR = DK / CW;      // lanes per row
  constexpr int RPI = 32 / LR;     // rows per warp-wide access
  constexpr int J = R / RPI;       // rows (slots) per lane
  constexpr int LPS = LR / J;      // lanes that end up holding one slot's total
  constexpr int E16 = 16 / static_cast<int>(sizeof(IO));  // elements per 16-byte copy
  constexpr int E4 = Act<IO>::kPer4B;                      // elements per 4-byte copy
  static_assert(R >= 1 && R <= 32 && (R & (R - 1)) == 0, "R must be a power of two <= 32");
  static_assert(CW * LR == DK && LR <= 32 && (LR & (LR - 1)) == 0, "a row spans a power of two of lanes");
  static_assert(J >= 1 && J * RPI == R && J <= LR, "whole slots, at most one per lane of a row");
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
  const int rg = lane / LR;  // this lane's row within each access: slot j holds row row0 + j*RPI + rg
  const int cell0 = (lane % LR) * CW;

  // 1. Issue the state loads first: they are the bulk of the HBM traffic.
  //    Slot j of lane l is at (row0 + j*RPI)*DK + l*CW: the warp's lanes
  //    read RPI whole rows, contiguous.
  const size_t state_head = static_cast<size_t>(head) * a.dv * DK;
  float st[J][CW];
#pragma unroll
  for (int j = 0; j < J; ++j) {
    if (row0 + j * RPI + rg < a.dv) {
      Cells<CW>::load_cs(
          GDN_LAYER(state_in) + state_head + static_cast<size_t>(row0 + j * RPI) * DK + lane * CW, st[j]);
    } else {
#pragma unroll
      for (int c = 0; c < CW; ++c) st[j][c] = 0.f;
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
  const int my_r = ((lane % LR) / LPS) * RPI + rg;  // the row (within the warp's R) whose totals this lane holds
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
      float kk[CW], qq[CW];
      Act<IO>::template get_n<CW>(ks + tt * DK + cell0, kk);
      Act<IO>::template get_n<CW>(qs + tt * DK + cell0, qq);
      const float alpha = expf(-gs[tt]);
      const float b = bs[tt];

      // S@k (on the decayed state for decay-first, the old one for decay-after)
      float part[J];
#pragma unroll
      for (int j = 0; j < J; ++j) {
        part[j] = 0.f;
#pragma unroll
        for (int c = 0; c < CW; ++c) {
          if (!DECAY_AFTER) st[j][c] *= alpha;
          part[j] = fmaf(st[j][c], kk[c], part[j]);
        }
      }
      const float sk = reduce_slots<J, LR>(part, lane);
      const float d = (Act<IO>::get(vs + tt * ROWS + warp * R + my_r) - sk) * b;

      // rank-1 update and S@q
      float py[J];
#pragma unroll
      for (int j = 0; j < J; ++j) {
        const float dr = __shfl_sync(kFull, d, rg * LR + j * LPS);
        py[j] = 0.f;
#pragma unroll
        for (int c = 0; c < CW; ++c) {
          if (DECAY_AFTER)
            st[j][c] = fmaf(alpha, st[j][c], dr * kk[c]);
          else
            st[j][c] = fmaf(dr, kk[c], st[j][c]);
          py[j] = fmaf(st[j][c], qq[c], py[j]);
        }
      }
      const float y = reduce_slots<J, LR>(py, lane);
      const size_t tok_head = (static_cast<size_t>(s) * nt + t) * a.nv + vh;
      if ((lane % LPS) == 0 && my_row < a.dv) Act<IO>::put(gout + tok_head * a.dv + my_row, y * a.q_scale);

      if (CAPTURE) {
        float *cap = GDN_LAYER(capture) + tok_head * a.dv * DK;
#pragma unroll
        for (int j = 0; j < J; ++j)
          if (row0 + j * RPI + rg < a.dv)
            Cells<CW>::store_cs(cap + static_cast<size_t>(row0 + j * RPI) * DK + lane * CW, st[j]);
      }
    }
    __syncthreads();  // this buffer is refilled by the stage() of chunk c+2
  }

  // 3. Final state, from the same registers as the last capture slice.
#pragma unroll
  for (int j = 0; j < J; ++j)
    if (row0 + j * RPI + rg < a.dv)
      Cells<CW>::store_cs(GDN_LAYER(state_out) + state_head + static_cast<size_t>(row0 + j * RPI) * DK + lane * CW,
                          st[j]);
#undef GDN_LAYER
}

// ---- launch shape: several rows per warp (R = 16/NSG, 64 B of state per
// lane) and small CTAs (8 KB of state per CTA), so each SM keeps tens of KB
// of state loads in flight across many CTAs and the fixed cost of a CTA is
// shared by few rows; tokens are staged 8 at a time.  4 warps for
// D_k >= 64; at D_k = 32 a warp already holds 16 rows, so 2 warps (32 rows:
// one value head of D_v = 32 per CTA), each row on 8 lanes of 4 cells.
// (Measured on decode with 134 MB of state: at D_k = 128, 4 warps beat 8 by
// 8 % on 32 one-sequence layers per launch and by 1 % on 64-sequence decode.
// At D_k = 32, rows on 8 lanes (128-bit accesses, 4-shuffle reductions, 48
// registers) move 6738 GB/s where one cell of every row per lane (16 scalar
// accesses and 16-shuffle reductions a lane, 96 registers) moved 5989; 8 rows
// per warp and 4 warps 5688; two 2-warp value heads per CTA 4586.  4 cells
// per lane at D_k = 64 measured the same as 2.)

template <int NSG>
constexpr int kWarpsFor = NSG == 1 ? 2 : 4;
template <int NSG>
constexpr int kCellsFor = NSG == 1 ? 4 : NSG;  // cells of a row per lane
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
  gdn_token_loop_kernel<IO, NSG, kCellsFor<NSG>, R, kWarps, CAPTURE, DA, MAXL>
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

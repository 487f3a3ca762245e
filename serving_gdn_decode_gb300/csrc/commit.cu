// Speculative-decode rollback commit: make the captured state after each
// sequence's last accepted token the active state.
//
// "dispatch_gated_delta_net_decode_with_capture" (gated_delta_net_decode.rs,
// mlx-native 0.21.1) leaves this step to the caller: on a partial reject it
// reads state_capture[..., accepted_idx, ...] as the new state.  Here it is
// one launch that gathers, for every sequence s, the contiguous slice
// state_capture[:, :, :, idx_s, s] (D_k*D_v*n_v f32) into state[:, :, :, s],
// reading idx_s from device memory so the whole verify-and-commit step can be
// enqueued (or graph-captured) without a host round trip.
#include <cuda_runtime.h>

#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;  // independent 16-byte copies in flight per thread

// grid.y = sequence, grid.x = 4 KiB pieces of that sequence's slice: the
// accepted index is read once per CTA and a CTA whose sequence keeps its
// state exits at once.
__global__ void __launch_bounds__(kThreads)
    gdn_commit_kernel(const float4 *__restrict__ capture, const int32_t *__restrict__ accepted,
                      float4 *__restrict__ state, uint32_t nt,
                      uint64_t slice4 /* float4s per (token, seq) slice */, uint32_t s0) {
  const uint32_t s = s0 + blockIdx.y;
  const int32_t idx = __ldg(accepted + s);
  if (idx < 0 || static_cast<uint32_t>(idx) >= nt) return;  // nothing accepted: keep the state
  const float4 *src = capture + (static_cast<uint64_t>(s) * nt + static_cast<uint32_t>(idx)) * slice4;
  float4 *dst = state + static_cast<uint64_t>(s) * slice4;
  const uint64_t base = static_cast<uint64_t>(blockIdx.x) * (kThreads * kUnroll) + threadIdx.x;
  float4 x[kUnroll];
#pragma unroll
  for (int u = 0; u < kUnroll; ++u) {
    const uint64_t e = base + u * kThreads;
    if (e < slice4) x[u] = __ldcs(src + e);
  }
#pragma unroll
  for (int u = 0; u < kUnroll; ++u) {
    const uint64_t e = base + u * kThreads;
    if (e < slice4) __stcs(dst + e, x[u]);
  }
}

}  // namespace

cudaError_t launch_commit(const float *capture, const int32_t *accepted, float *state,
                          uint32_t nt, uint32_t ns, uint64_t slice_elems, cudaStream_t stream) {
  constexpr uint32_t kMaxGridY = 65535;
  const uint64_t slice4 = slice_elems / 4;
  const uint64_t bx = (slice4 + kThreads * kUnroll - 1) / (kThreads * kUnroll);
  if (bx == 0 || bx > 0x7fffffffull) return cudaErrorInvalidConfiguration;
  for (uint32_t s0 = 0; s0 < ns; s0 += kMaxGridY) {  // grid.y holds at most 65535 sequences
    const uint32_t n = ns - s0 < kMaxGridY ? ns - s0 : kMaxGridY;
    gdn_commit_kernel<<<dim3(static_cast<unsigned>(bx), n), kThreads, 0, stream>>>(
        reinterpret_cast<const float4 *>(capture), accepted, reinterpret_cast<float4 *>(state), nt,
        slice4, s0);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace gdn

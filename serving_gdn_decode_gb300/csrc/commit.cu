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

__global__ void __launch_bounds__(256)
    gdn_commit_kernel(const float4 *__restrict__ capture, const int32_t *__restrict__ accepted,
                      float4 *__restrict__ state, uint32_t nt, uint32_t ns,
                      uint64_t slice4 /* float4s per (token, seq) slice */) {
  const uint64_t total = slice4 * ns;
  for (uint64_t i = blockIdx.x * static_cast<uint64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<uint64_t>(gridDim.x) * blockDim.x) {
    const uint64_t s = i / slice4;
    const uint64_t e = i - s * slice4;
    const int32_t idx = __ldg(accepted + s);
    if (idx < 0 || static_cast<uint32_t>(idx) >= nt) continue;  // keep this sequence's state
    __stcs(state + i, __ldcs(capture + (s * nt + static_cast<uint32_t>(idx)) * slice4 + e));
  }
}

}  // namespace

cudaError_t launch_commit(const float *capture, const int32_t *accepted, float *state,
                          uint32_t nt, uint32_t ns, uint64_t slice_elems, int sm_count,
                          cudaStream_t stream) {
  const uint64_t slice4 = slice_elems / 4;
  const uint64_t total = slice4 * ns;
  uint64_t blocks = (total + 255) / 256;
  const uint64_t cap = static_cast<uint64_t>(sm_count > 0 ? sm_count : 152) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks == 0) blocks = 1;
  gdn_commit_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
      reinterpret_cast<const float4 *>(capture), accepted, reinterpret_cast<float4 *>(state), nt,
      ns, slice4);
  return cudaGetLastError();
}

}  // namespace gdn

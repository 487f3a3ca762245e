// Internal interface between the C-ABI host code and the kernel launchers.
// Nothing here is exported from the shared library.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace gdn {

// One validated problem.  Pointers are device pointers in the layouts of
// gdn.h; sizes are the decoded params.  q, k, v and output hold f32, or
// bf16 when io_bf16 is set; every other buffer is f32.
struct Problem {
  const void *q, *k, *v;
  const float *g, *beta, *state_in;
  void *output;
  float *state_out, *capture;  // capture == nullptr: no capture
  uint32_t dk, dv, nk, nv, nt, ns;
  bool decay_after;
  bool khead_div;
  bool io_bf16;
  bool tf32;  // chunked forms: TF32 operands instead of split bf16
  float q_scale;
};

// Decode / multi-token-window kernel (token_loop.cu): every (seq, value head)
// state row stays in registers across the call; shaped for HBM throughput.
cudaError_t launch_token_loop(const Problem &p, cudaStream_t stream);

// The same kernel over several problems of one shape (the layers of a
// forward pass) in ceil(n / kMaxLayersPerLaunch) launches; layers[i] share
// every field but the buffer pointers.
constexpr uint32_t kMaxLayersPerLaunch = 64;
cudaError_t launch_token_loop_layers(const Problem *layers, uint32_t n_layers, cudaStream_t stream);

// Sequential-scan kernel for long token ranges (scan.cu): two lanes per row,
// lazy decay; shaped for FP32 issue throughput.
cudaError_t launch_scan(const Problem &p, cudaStream_t stream);

// Chunked tensor-core prefill (chunked.cu): D_k = D_v = 128, no capture; f32
// activations, or bf16 ones with split operands (not with tf32).
bool chunked_supported(const Problem &p);
cudaError_t launch_chunked(const Problem &p, cudaStream_t stream);

// The same chunk equations in two passes (chunked_split.cu): a parallel pass
// over every (seq, chunk, key head) writes the state-independent chunk
// matrices to `workspace` (device, chunked_split_workspace_bytes(p) bytes,
// 16-byte aligned), then one CTA per (seq, value head) runs the state pass.
// The chunk pass holds the gate scalars of all value heads of a key head in
// shared memory, so the form takes at most kMaxSplitGroup of them.
constexpr uint32_t kMaxSplitGroup = 32;
bool chunked_split_supported(const Problem &p);  // chunked_supported, f32 activations, n_v / n_k <= kMaxSplitGroup
size_t chunked_split_workspace_bytes(const Problem &p);
cudaError_t launch_chunked_split(const Problem &p, float *workspace, cudaStream_t stream);

// The two-pass form with its workspace in a fixed 32 MiB device array of
// chunked_split.cu instead of caller memory (no allocation anywhere).
constexpr size_t kNoallocWorkspaceBytes = static_cast<size_t>(32) << 20;
cudaError_t launch_chunked_split_noalloc(const Problem &p, cudaStream_t stream);

// Failure bits of the chunked kernels (chunked.cu, chunked_split.cu): each
// file's word on the current device after all work on `stream` so far
// (synchronises the stream); cleared afterwards when `reset`.
cudaError_t chunked_wait_status(unsigned int *bits, bool reset, cudaStream_t stream);
cudaError_t chunked_split_wait_status(unsigned int *bits, bool reset, cudaStream_t stream);

// Rollback commit (commit.cu): state[.., s] = capture[.., accepted[s], s] for
// every sequence whose accepted index lies in [0, nt).
cudaError_t launch_commit(const float *capture, const int32_t *accepted, float *state,
                          uint32_t nt, uint32_t ns, uint64_t slice_elems, cudaStream_t stream);

}  // namespace gdn

// Internal interface between the C-ABI host code and the kernel launchers.
// Nothing here is exported from the shared library.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace gdn {

// One validated problem.  Pointers are device pointers in the layouts of
// gdn.h; sizes are the decoded params.
struct Problem {
  const float *q, *k, *v, *g, *beta, *state_in;
  float *output, *state_out, *capture;  // capture == nullptr: no capture
  uint32_t dk, dv, nk, nv, nt, ns;
  bool decay_after;
  bool khead_div;
  float q_scale;
};

// Token-loop kernels: the state rows of every (seq, value head) pair stay in
// registers across the whole token range.  `geometry` picks the decode
// launch shape (few tokens, HBM-bound) or the scan shape (many tokens).
enum class LoopGeometry { kDecode, kScan };
cudaError_t launch_token_loop(const Problem &p, LoopGeometry geometry, cudaStream_t stream);

// Kernel name of the token-loop launch that `launch_token_loop` would use.
const char *token_loop_name(LoopGeometry geometry, bool capture);

}  // namespace gdn

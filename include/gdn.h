/*
 * gdn.h -- C ABI of the GB300 (sm_103a) Gated DeltaNet recurrence library
 *          (libgdn_gb300.so).
 *
 * The operation.  For every sequence s and value head vh, with the D_v x D_k
 * f32 state S of that pair (row i = d_v index, column j = d_k index) and for
 * tokens t = 0 .. n_tokens-1 in order:
 *
 *     alpha    = exp(-g_t)
 *     S        = alpha * S                       (decay-first, flags bit0 = 0)
 *     sk[i]    = sum_j S[i][j] * k_t[j]
 *     delta[i] = (v_t[i] - sk[i]) * beta_t
 *     S[i][j] += delta[i] * k_t[j]
 *     y_t[i]   = q_scale * sum_j S[i][j] * q_t[j]
 *
 * This is the step order of the kernel body of
 * "gated_delta_net_decode_capture.metal" (mlx-native 0.9.2), steps
 * "decay + partial s_k" and "state update + output partial".  With flags
 * bit0 = 1 the state is decayed after S@k instead, as in the recurrence of
 * the module doc of "gated_delta_net.rs" (mlx-native 0.4.0):
 * S' = alpha*S + beta*outer(v - S@k, k), y = S'@q.
 *
 * k_head, the key/query head read by value head vh ("GQA broadcast",
 * gated_delta_net.rs): vh % n_k_heads (flags bit1 = 0, the capture kernel's
 * head setup) or vh / (n_v_heads / n_k_heads) (flags bit1 = 1).
 *
 * Layouts, innermost (fastest) dimension first, all f32, densely packed
 * ("Memory layouts" table of gated_delta_net.rs; "Memory layout for
 * state_capture" section of the capture kernel page):
 *     q, k            [D_k, n_k_heads, n_tokens, n_seqs]
 *     v, output       [D_v, n_v_heads, n_tokens, n_seqs]
 *     g, beta         [n_v_heads, n_tokens, n_seqs]
 *     state_in/out    [D_k, D_v, n_v_heads, n_seqs]
 *     state_capture   [D_k, D_v, n_v_heads, n_tokens, n_seqs]
 *
 * Parameters: a HOST array of at least 9 uint32 ("Buffer bindings" section of
 * the capture kernel page; "Buffer / params contract" of
 * gated_delta_net_decode.rs, mlx-native 0.21.1):
 *     params[0..5] = D_k, D_v, n_k_heads, n_v_heads, n_tokens, n_seqs
 *     params[6]    = flags (the pages always write 0 here; see GDN_FLAG_*)
 *     params[7]    = reserved, must be 0
 *     params[8]    = q_scale_bits: the f32 bit pattern of q_scale, applied to
 *                    y at writeback; 0 means q_scale = 1.0.
 *
 * Ownership and lifetime.  Every buffer pointer is a DEVICE pointer owned by
 * the caller; the library allocates no memory, keeps no state between calls
 * (apart from the device status word of gdn_device_status) and never
 * synchronises (apart from gdn_device_status).  All work is enqueued on `stream` (NULL = the
 * legacy default stream) and is asynchronous: buffers must stay valid until
 * the stream reaches the call.  Calls on different streams with disjoint
 * buffers may run concurrently.
 *
 * Errors.  Arguments are checked on the host before anything is enqueued; a
 * failed check returns GDN_ERR_INVALID_ARGUMENT or GDN_ERR_UNSUPPORTED and
 * enqueues nothing.  A failed launch returns GDN_ERR_CUDA.  Faults during
 * kernel execution surface through the stream like any CUDA error.  After a
 * non-OK status, gdn_last_error() gives a message (per calling thread).
 *
 * Device-side failures.  The chunked prefill kernels (the chunked path of
 * gdn_forward, gdn_forward_ws, gdn_forward_chunked_noalloc) wait on
 * asynchronous copies and tensor-core work through barriers, and every such
 * wait is bounded (about a second of GPU clock).  A wait that runs out does
 * not hang or fault the GPU: the kernel writes NaN into the affected
 * (seq, value head) state_out (the two-pass form also into its chunk
 * matrices, so the outputs that depend on them become NaN), releases its
 * tensor memory, returns, and sets GDN_DEVICE_WAIT_TIMEOUT in the library's
 * device status word.  The call itself has already returned GDN_OK by then;
 * gdn_device_status() reads the word, which tells a timed-out wait from NaN
 * inputs.  The other kernels have no waits of this kind.
 */
#ifndef GDN_GB300_H
#define GDN_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as CUDA's cudaStream_t / CUstream. */
typedef struct CUstream_st *gdn_stream_t;

typedef enum gdn_status {
  GDN_OK = 0,
  GDN_ERR_INVALID_ARGUMENT = 1, /* the pages' InvalidArgument cases, and ours */
  GDN_ERR_UNSUPPORTED = 2,      /* valid for the method, no kernel for it here */
  GDN_ERR_CUDA = 3              /* a CUDA runtime call failed */
} gdn_status;

#define GDN_N_PARAMS 9

/* params[6] flag bits.  0 selects the behaviour of the pages' kernel. */
#define GDN_FLAG_DECAY_AFTER 0x1u /* decay after S@k (gated_delta_net.rs)  */
#define GDN_FLAG_KHEAD_DIV 0x2u   /* k_head = vh / (n_v/n_k)               */
#define GDN_PATH_SHIFT 2u         /* bits 2-3: path choice                 */
#define GDN_PATH_MASK 0xCu
#define GDN_PATH_AUTO 0u          /* the library picks by shape            */
#define GDN_PATH_SCAN 1u          /* token-by-token scan kernel            */
#define GDN_PATH_CHUNKED 2u       /* chunked tensor-core prefill, split-bf16
                                     operands                              */
#define GDN_PATH_CHUNKED_TF32 3u  /* the same with TF32 operands (faster,
                                     about 1e-3 less accurate)             */

/*
 * gdn_forward -- run the recurrence over n_tokens tokens for every
 * (seq, value head) pair, write y to `output` and the final state to
 * `state_out`.  Follows dispatch_gated_delta_net_decode
 * (gated_delta_net_decode.rs, mlx-native 0.21.1) and dispatch_gated_delta_net
 * (gated_delta_net.rs, mlx-native 0.4.0); buffer order is the pages' buffer
 * slots 0-8.
 *
 * Checks (mirroring `validate` and `validate_params_buf` of
 * gated_delta_net_decode.rs):
 *   INVALID_ARGUMENT: params == NULL or n_params < 9; any of D_k, D_v,
 *     n_k_heads, n_v_heads, n_tokens, n_seqs == 0; n_v_heads % n_k_heads != 0;
 *     D_k % 32 != 0 or D_k > 128; D_v % (D_k/32) != 0; params[7] != 0;
 *     unknown flag bits; a NULL buffer; q, k, state_in or state_out
 *     not 16-byte aligned, or v, g, beta, output not 4-byte aligned;
 *     state_in and state_out overlapping without being the same pointer
 *     (state_in == state_out, an in-place update, is allowed); output
 *     overlapping any other buffer; on a forced chunked path, v not 16-byte
 *     aligned (its rows are copied 16 bytes at a time).
 *   UNSUPPORTED: D_k = 96 (D_k/32 = 3 has no kernel, as on the pages);
 *     the chunked path forced for a shape it does not cover.
 *
 * Path choice (params[6] bits 2-3).  GDN_PATH_AUTO runs the token-loop
 * kernel for n_tokens <= 16 and for every capture call; for longer windows
 * without capture it runs the tensor-core
 * chunked form when that form covers the call (D_k = D_v = 128, f32
 * activations, no capture, v 16-byte aligned) and n_tokens >= 48, and the
 * token-by-token FP32 scan otherwise.  GDN_PATH_SCAN forces the scan;
 * GDN_PATH_CHUNKED and GDN_PATH_CHUNKED_TF32 force the chunked form
 * (UNSUPPORTED for a shape it does not cover).
 * Accuracy against a double-precision evaluation of the recurrence (rel-L2,
 * 4 x 4096-token windows): the token-loop kernel and the scan compute every
 * product in f32, about 1e-7; the chunked form takes each tensor-core
 * product as three bf16 products of split operands (x = hi + lo), about
 * 1e-5 (3e-5 for negative gates, whose states grow by e^20 over the
 * window); GDN_PATH_CHUNKED_TF32 rounds the operands to TF32 instead, one
 * product each, about 5e-4 (3e-3 for those negative gates).
 * gdn_forward runs the chunked form in one pass; gdn_forward_ws, given a
 * workspace, in two (faster from about 512 tokens on; under GDN_PATH_AUTO it
 * keeps the one pass below that).
 * Buffer sizes cannot be checked through raw pointers: each buffer must hold
 * the element count its layout above gives.
 */
gdn_status gdn_forward(const float *q, const float *k, const float *v, const float *g,
                       const float *beta, const float *state_in, float *output,
                       float *state_out, const uint32_t *params, size_t n_params,
                       gdn_stream_t stream);

/*
 * gdn_forward_capture -- gdn_forward, plus the state after every token
 * written to `state_capture` (slot 9 of the capture kernel page):
 * state_capture[:, :, vh, t, s] = S after token t.  Slice n_tokens-1 is
 * bit-identical to state_out (the "Determinism contract" of
 * dispatch_gated_delta_net_decode_with_capture).  For speculative-decode
 * rollback the caller takes slice `accepted_idx` as the new state.
 *
 * Extra checks (dispatch_gated_delta_net_decode_with_capture):
 *   INVALID_ARGUMENT: state_capture == NULL or not 16-byte aligned, or
 *     overlapping any other buffer; state_capture_elems !=
 *     n_tokens*D_k*D_v*n_v_heads*n_seqs when n_seqs > 1, or smaller than it
 *     when n_seqs == 1 (elements past that count are left untouched).
 *   UNSUPPORTED: the chunked path forced (it keeps no per-token state).
 */
gdn_status gdn_forward_capture(const float *q, const float *k, const float *v, const float *g,
                               const float *beta, const float *state_in, float *output,
                               float *state_out, const uint32_t *params, size_t n_params,
                               float *state_capture, size_t state_capture_elems,
                               gdn_stream_t stream);

/* The buffers of one problem (e.g. one linear-attention layer) for
 * gdn_forward_layers; every pointer is a DEVICE pointer, as in gdn_forward. */
typedef struct gdn_layer_buffers {
  const float *q, *k, *v, *g, *beta, *state_in;
  float *output, *state_out;
  float *state_capture; /* read only when with_capture != 0 */
} gdn_layer_buffers;

/*
 * gdn_forward_layers -- gdn_forward (or gdn_forward_capture when with_capture
 * != 0) on n_layers problems of the same shape and flags (`params`), such as
 * the linear-attention layers of one forward pass, which the pages run one
 * dispatch per layer ("Memory cost" of gated_delta_net_decode_capture.metal:
 * 30+ linear-attention layers per forward).  On the decode path (n_tokens <=
 * 16, automatic path) all layers run in one launch per 64 layers, so a
 * small-batch decode step is not paid for in launch latency; otherwise the
 * layers are launched one after another.  `layers` is a HOST array of
 * n_layers entries (1 <= n_layers <= 1024) that the call reads before it
 * returns.
 *
 * Checks: those of gdn_forward / gdn_forward_capture for every layer (the
 * message names the layer), plus INVALID_ARGUMENT when a layer's output,
 * state_out or state_capture overlaps any buffer of another layer.
 * Results are bit-identical to calling gdn_forward once per layer.
 */
gdn_status gdn_forward_layers(const gdn_layer_buffers *layers, size_t n_layers,
                              const uint32_t *params, size_t n_params, int with_capture,
                              size_t state_capture_elems, gdn_stream_t stream);

/*
 * gdn_commit_capture -- speculative-decode rollback.  After gdn_forward_capture
 * verified n_tokens tokens, make the state after each sequence's last
 * accepted token the active state:
 *     for every s with 0 <= accepted_idx[s] < n_tokens:
 *         state[:, :, :, s] = state_capture[:, :, :, accepted_idx[s], s]
 * Sequences with an index outside [0, n_tokens) (e.g. -1: nothing accepted)
 * keep their state.  The pages leave this step to the caller
 * (dispatch_gated_delta_net_decode_with_capture, gated_delta_net_decode.rs:
 * "the caller reads state_capture[..., accepted_idx, ...] as the new active
 * state"); here it is one launch that reads the indices on the device.
 *
 * state_capture: DEVICE, [D_k, D_v, n_v_heads, n_tokens, n_seqs] f32 as written by
 *   gdn_forward_capture with the same params; state_capture_elems as there.
 * accepted_idx:  DEVICE, n_seqs int32.
 * state:         DEVICE, [D_k, D_v, n_v_heads, n_seqs] f32, updated in place.
 * params:        HOST, the same 9-u32 block as the capture call (n_k_heads and
 *   the flags are checked but not used).
 * Checks: the params checks of gdn_forward; NULL pointers; state_capture and
 *   state 16-byte aligned, accepted_idx 4-byte aligned; the capture size rule
 *   of gdn_forward_capture; state overlapping state_capture or accepted_idx.
 */
gdn_status gdn_commit_capture(const float *state_capture, size_t state_capture_elems,
                              const int32_t *accepted_idx, float *state, const uint32_t *params,
                              size_t n_params, gdn_stream_t stream);

/*
 * bf16 activations with f32 state.  The prefill page ("Dtype / precision" of
 * gated_delta_net.rs, mlx-native 0.4.0) keeps all accumulation in f32 and
 * names bf16 inputs and outputs as a later variant.  These entry points are
 * that variant: q, k, v and output hold bfloat16 (the upper half of an f32
 * bit pattern, as torch.bfloat16 / __nv_bfloat16), in the same layouts as
 * above; g, beta, state_in, state_out and state_capture stay f32.  Each
 * bf16 value is widened exactly to f32 on load, every product and sum is f32
 * as in gdn_forward, and y is rounded once, to nearest-even bf16, when it is
 * stored.  Results for the same widened inputs therefore equal gdn_forward's
 * up to that final rounding of y (state and capture are bit-identical).
 *
 * Extra checks: v 4-byte aligned and output 2-byte aligned (q and k stay
 * 16-byte); UNSUPPORTED when D_v is odd (v is staged two rows at a time) or
 * when the TF32 chunked path is forced.  The chunked path (forced, or chosen
 * by GDN_PATH_AUTO) runs with split operands; bf16 inputs are their own hi
 * halves, so its products leave out the terms with a zero lo half, which
 * add nothing in the f32 form: results keep the equalities above.
 */
typedef uint16_t gdn_bf16; /* bfloat16 bit pattern */

gdn_status gdn_forward_bf16(const gdn_bf16 *q, const gdn_bf16 *k, const gdn_bf16 *v,
                            const float *g, const float *beta, const float *state_in,
                            gdn_bf16 *output, float *state_out, const uint32_t *params,
                            size_t n_params, gdn_stream_t stream);

gdn_status gdn_forward_capture_bf16(const gdn_bf16 *q, const gdn_bf16 *k, const gdn_bf16 *v,
                                    const float *g, const float *beta, const float *state_in,
                                    gdn_bf16 *output, float *state_out, const uint32_t *params,
                                    size_t n_params, float *state_capture,
                                    size_t state_capture_elems, gdn_stream_t stream);

/*
 * Two-pass chunked prefill with a caller-provided workspace.
 *
 * The chunked (WY / UT) form of the recurrence over 64-token chunks splits
 * into a part that does not depend on the state -- per chunk, the Gram
 * products, A, T = (I + A)^-1 and the masked decay-weighted Q K^T -- and the
 * state pass.  gdn_forward_ws runs the first part for every (seq, chunk) in
 * parallel -- the products of K and Q once per key head, the gated parts per
 * value head -- writes it to `workspace`, then runs the state pass (one CTA
 * per (seq, value head)).  The pages have no chunked kernel:
 * the chunk equations are the delta rule's published chunkwise form derived
 * from the recurrence of gated_delta_net.rs (mlx-native 0.4.0) and of the
 * capture kernel page, with the operands of the path bits (split bf16 for
 * GDN_PATH_AUTO and GDN_PATH_CHUNKED, TF32 for GDN_PATH_CHUNKED_TF32).
 *
 * gdn_workspace_size: *bytes = the workspace gdn_forward_ws needs for
 *   `params` -- on the chunked path (forced, or chosen by GDN_PATH_AUTO for
 *   the shape, assuming a 16-byte-aligned v, with at least 512 tokens: the
 *   automatic choice keeps the one-pass form for shorter windows, where it
 *   is the faster one), per (seq, 64-token chunk),
 *   32 KB per value head plus 96 KB per key head (the K and Q operands and K^T,
 *   shared by the value heads that read the key head); 0 on every other
 *   path, and 0 when a key head has more than 32 value heads (the two-pass
 *   form takes at most 32; gdn_forward_ws then runs the one-pass chunked
 *   form of gdn_forward).  Same params checks and status as gdn_path_name.
 *
 * gdn_forward_ws: gdn_forward, plus `workspace` (DEVICE, caller-owned,
 *   at least gdn_workspace_size bytes, 16-byte aligned, overlapping no other
 *   buffer; may be NULL when the size is 0).  The call overwrites the
 *   workspace; its contents afterwards are unspecified.  On the chunked
 *   path (forced, or chosen by GDN_PATH_AUTO for 512 tokens or more) the
 *   two-pass form runs; otherwise the call runs exactly as gdn_forward and
 *   does not touch the workspace.  Extra checks: INVALID_ARGUMENT for a NULL, misaligned,
 *   short or overlapping workspace when the size is > 0.
 */
gdn_status gdn_workspace_size(const uint32_t *params, size_t n_params, size_t *bytes);

gdn_status gdn_forward_ws(const float *q, const float *k, const float *v, const float *g,
                          const float *beta, const float *state_in, float *output,
                          float *state_out, const uint32_t *params, size_t n_params,
                          void *workspace, size_t workspace_bytes, gdn_stream_t stream);

/*
 * gdn_forward_ws_bf16 -- gdn_forward_ws with bf16 q, k, v and output, as
 * gdn_forward_bf16 is to gdn_forward (same layouts, f32 g, beta and state;
 * y rounded once to nearest-even bf16 when stored).  The workspace size is
 * gdn_workspace_size's for the same params; the two-pass form stores only
 * the hi halves of K, Q and K^T (bf16 inputs are exact), using part of it.
 * Results: the state equals gdn_forward_ws's on the same widened inputs bit
 * for bit, and the output equals its output rounded to bf16.  Checks as
 * gdn_forward_bf16 plus the workspace checks of gdn_forward_ws; the TF32
 * chunked path (GDN_PATH_CHUNKED_TF32) is UNSUPPORTED with bf16 activations.
 */
gdn_status gdn_forward_ws_bf16(const gdn_bf16 *q, const gdn_bf16 *k, const gdn_bf16 *v,
                               const float *g, const float *beta, const float *state_in,
                               gdn_bf16 *output, float *state_out, const uint32_t *params,
                               size_t n_params, void *workspace, size_t workspace_bytes,
                               gdn_stream_t stream);

/*
 * gdn_forward_chunked_noalloc -- the two-pass chunked prefill of
 * gdn_forward_ws, for callers that cannot allocate device memory: its chunk
 * scratch lives in a fixed array inside this library instead of a
 * caller-provided workspace.  The pages have no counterpart; it exists for
 * code that only ever receives device buffers from a host framework that
 * owns all device memory (a plugin or an embedded runtime whose memory pool
 * offers it no allocation hook), and for loops that must not pay for
 * cudaMalloc, which can synchronise the device.  Nothing here allocates:
 * no cudaMalloc, no cudaFree, no allocating library routine.
 *
 * Limit: the fixed scratch is 32 MiB, and a problem needs, per (seq,
 * 64-token chunk), 32 KB per value head plus 96 KB per key head (what
 * gdn_workspace_size reports) -- e.g. one sequence of 1024 tokens with 16
 * value and 16 key heads, or of 640 tokens with 48 value and 16 key heads;
 * every GPU on which the library's chunked kernels are loaded holds it until
 * the process exits.  Larger problems return
 * GDN_ERR_INVALID_ARGUMENT with the numbers; use gdn_forward_ws for them.
 *
 * Arguments, layouts and checks as gdn_forward (f32 activations), for the
 * chunked path: the params path bits must not be GDN_PATH_SCAN
 * (GDN_PATH_AUTO means GDN_PATH_CHUNKED here), the chunked path's shape rules apply (D_k = D_v = 128,
 * else GDN_ERR_UNSUPPORTED), and v must be 16-byte aligned as for
 * gdn_forward_ws (INVALID_ARGUMENT otherwise).  Results equal
 * gdn_forward_ws's on the chunked path.  With more than 32 value heads per
 * key head it runs the one-pass chunked form of gdn_forward, which needs no
 * scratch (as gdn_forward_ws does).
 *
 * The first call on a device looks up the device address of the scratch
 * (once per device and context, with that device current; if the context is
 * destroyed and created again, e.g. by cudaDeviceReset, the next call looks
 * it up again); make that first call before any stream capture.  Every call
 * on a device shares the one scratch array:
 * each call writes all of it that it reads, so nothing carries over between
 * calls, but calls that overlap on the GPU (e.g. on two streams at once)
 * race on it and must be ordered by the caller.
 */
gdn_status gdn_forward_chunked_noalloc(const float *q, const float *k, const float *v,
                                       const float *g, const float *beta, const float *state_in,
                                       float *output, float *state_out, const uint32_t *params,
                                       size_t n_params, gdn_stream_t stream);

/* gdn_layer_buffers with bf16 q, k, v and output. */
typedef struct gdn_layer_buffers_bf16 {
  const gdn_bf16 *q, *k, *v;
  const float *g, *beta, *state_in;
  gdn_bf16 *output;
  float *state_out;
  float *state_capture; /* read only when with_capture != 0 */
} gdn_layer_buffers_bf16;

/* gdn_forward_layers on bf16 activations (gdn_forward_bf16 per layer). */
gdn_status gdn_forward_layers_bf16(const gdn_layer_buffers_bf16 *layers, size_t n_layers,
                                   const uint32_t *params, size_t n_params, int with_capture,
                                   size_t state_capture_elems, gdn_stream_t stream);

/* Message for the last non-OK status returned on the calling thread ("" if
 * none).  The pointer stays valid until the thread's next call. */
const char *gdn_last_error(void);

/* Bits of the device status word. */
#define GDN_DEVICE_WAIT_TIMEOUT 0x1u /* a chunked kernel's bounded wait ran out */

/*
 * gdn_device_status -- the library's device-side failure channel (see
 * "Device-side failures" above).  The pages report errors as a Result from
 * validation on the host ("validate", gated_delta_net_decode.rs); a failure
 * that can only happen while a kernel runs needs a channel of its own, and
 * this is it.
 *
 * Waits for all work enqueued on `stream` so far (it synchronises the
 * stream), then stores in *status (HOST pointer) the OR of the GDN_DEVICE_*
 * bits set by any kernel of this library on the CURRENT device since the
 * word was last cleared (0 = no failure); with reset != 0 the word is
 * cleared afterwards.  One word per device, shared by every stream and
 * thread: read it after the calls of interest have been enqueued on
 * `stream`, and order work on other streams yourself.  Allocates nothing.
 * Returns INVALID_ARGUMENT for status == NULL, GDN_ERR_CUDA if the read
 * fails (e.g. an earlier fault left the context unusable).
 */
gdn_status gdn_device_status(uint32_t *status, int reset, gdn_stream_t stream);

/* The kernel path the library would run for `params` (with or without
 * capture): on GDN_OK, *name points to a static string such as
 * "token_loop_decode".  Runs the same params checks as gdn_forward and returns
 * the same status for invalid params.  Host-only: enqueues nothing. */
gdn_status gdn_path_name(const uint32_t *params, size_t n_params, int capture,
                         const char **name);

#ifdef __cplusplus
}
#endif

#endif /* GDN_GB300_H */

// C-ABI entry points of libgdn_gb300.so: argument checks, path choice and
// dispatch.  The checks mirror `validate`, `validate_params_buf` and the
// capture-size rule of gated_delta_net_decode.rs (mlx-native 0.21.1); the
// alias and alignment rules are this library's own (the pages are silent).
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "../../include/gdn.h"
#include "gdn_internal.h"

namespace {

thread_local char g_last_error[512] = "";

gdn_status fail(gdn_status st, const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
  va_end(ap);
  return st;
}

// Largest n_tokens that runs on the decode launch shape under GDN_PATH_AUTO.
constexpr uint32_t kDecodeMaxTokens = 16;
// Shortest window GDN_PATH_AUTO runs on the chunked form where it covers
// the call.  Measured on GB300 for 16 to 256 (seq, value head) chains: the
// one-pass and two-pass forms overtake the scan between 32 and 64 tokens
// (at 64 tokens, 4 x 48 chains: 41.7 / 42.6 against 51.9 us).
constexpr uint32_t kChunkedMinTokens = 48;
// Under GDN_PATH_AUTO a workspace turns the chunked form into two passes from
// this window length on; below it the one-pass form is the faster one
// (measured over 48 to 768 chains: at 256 tokens the one pass leads by 2-5 %
// with 48 or 192 chains, the two passes by 7 % with 768; from 512 tokens on
// the two passes lead in every case).
constexpr uint32_t kTwoPassMinTokens = 512;
// Upper bound on any buffer's element count (keeps byte counts far from
// 64-bit overflow).
constexpr unsigned long long kMaxElems = 1ull << 60;
// Most layers one gdn_forward_layers call takes (the cross-layer overlap check
// is quadratic in it).
constexpr size_t kMaxLayers = 1024;

bool mul_ok(unsigned long long a, unsigned long long b, unsigned long long *out) {
  const unsigned __int128 r = static_cast<unsigned __int128>(a) * b;
  if (r > kMaxElems) return false;
  *out = static_cast<unsigned long long>(r);
  return true;
}

struct Span {
  const void *p;
  unsigned long long bytes;
  const char *name;
};

bool overlap(const Span &a, const Span &b) {
  const auto a0 = reinterpret_cast<uintptr_t>(a.p), b0 = reinterpret_cast<uintptr_t>(b.p);
  return a0 < b0 + b.bytes && b0 < a0 + a.bytes;
}

bool aligned(const void *p, uintptr_t n) { return (reinterpret_cast<uintptr_t>(p) % n) == 0; }

struct Decoded {
  gdn::Problem prob;
  unsigned long long qk_elems, v_elems, sc_elems, state_elems, capture_elems;
  uint32_t path;
};

// Params block checks (no buffers).
gdn_status decode_params(const uint32_t *params, size_t n_params, Decoded *d) {
  if (params == nullptr)
    return fail(GDN_ERR_INVALID_ARGUMENT, "gdn: params is NULL");
  if (n_params < GDN_N_PARAMS)
    return fail(GDN_ERR_INVALID_ARGUMENT,
                "gdn: params has %zu u32, expected >= 9 (index 8 = q_scale_bits)", n_params);
  gdn::Problem &p = d->prob;
  std::memset(&p, 0, sizeof p);
  p.dk = params[0]; p.dv = params[1]; p.nk = params[2]; p.nv = params[3];
  p.nt = params[4]; p.ns = params[5];
  const uint32_t flags = params[6];
  if (p.dk == 0 || p.dv == 0 || p.nk == 0 || p.nv == 0)
    return fail(GDN_ERR_INVALID_ARGUMENT, "gdn: dims must all be > 0");
  if (p.nt == 0 || p.ns == 0)
    return fail(GDN_ERR_INVALID_ARGUMENT, "gdn: n_tokens and n_seqs must be > 0");
  if (p.nv % p.nk != 0)
    return fail(GDN_ERR_INVALID_ARGUMENT,
                "gdn: n_v_heads (%u) must be a multiple of n_k_heads (%u)", p.nv, p.nk);
  if (p.dk % 32 != 0)
    return fail(GDN_ERR_INVALID_ARGUMENT, "gdn: D_k (%u) must be a multiple of 32", p.dk);
  if (p.dk > 128)
    return fail(GDN_ERR_INVALID_ARGUMENT, "gdn: D_k (%u) must be <= 128 (D_k/32 <= 4)", p.dk);
  if (p.dk == 96)
    return fail(GDN_ERR_UNSUPPORTED, "gdn: D_k = 96 (D_k/32 = 3) has no kernel; use 32, 64 or 128");
  const uint32_t nsg = p.dk / 32;
  if (p.dv % nsg != 0)
    return fail(GDN_ERR_INVALID_ARGUMENT, "gdn: D_v (%u) must be a multiple of D_k/32 (%u)", p.dv,
                nsg);
  if (params[7] != 0)
    return fail(GDN_ERR_INVALID_ARGUMENT, "gdn: params[7] is reserved and must be 0 (got %u)",
                params[7]);
  if (flags & ~(GDN_FLAG_DECAY_AFTER | GDN_FLAG_KHEAD_DIV | GDN_PATH_MASK))
    return fail(GDN_ERR_INVALID_ARGUMENT, "gdn: unknown flag bits 0x%x in params[6]", flags);
  d->path = (flags & GDN_PATH_MASK) >> GDN_PATH_SHIFT;
  p.tf32 = d->path == GDN_PATH_CHUNKED_TF32;
  p.decay_after = (flags & GDN_FLAG_DECAY_AFTER) != 0;
  p.khead_div = (flags & GDN_FLAG_KHEAD_DIV) != 0;
  if (params[8] == 0) {
    p.q_scale = 1.0f;
  } else {
    std::memcpy(&p.q_scale, &params[8], sizeof(float));
  }
  unsigned long long x;
  if (!mul_ok(p.dk, p.nk, &x) || !mul_ok(x, p.nt, &x) || !mul_ok(x, p.ns, &d->qk_elems) ||
      !mul_ok(p.dv, p.nv, &x) || !mul_ok(x, p.nt, &x) || !mul_ok(x, p.ns, &d->v_elems) ||
      !mul_ok(p.nv, p.nt, &x) || !mul_ok(x, p.ns, &d->sc_elems) ||
      !mul_ok(p.dk, p.dv, &x) || !mul_ok(x, p.nv, &x) || !mul_ok(x, p.ns, &d->state_elems) ||
      !mul_ok(d->state_elems, p.nt, &d->capture_elems))
    return fail(GDN_ERR_INVALID_ARGUMENT, "gdn: buffer sizes overflow");
  return GDN_OK;
}

enum class Path { kDecode, kScan, kChunked };

const char *path_name(Path path, bool capture, bool tf32) {
  switch (path) {
    case Path::kDecode: return capture ? "token_loop_decode_capture" : "token_loop_decode";
    case Path::kChunked: return tf32 ? "chunked_tf32" : "chunked";
    default: return capture ? "scan_capture" : "scan";
  }
}

gdn_status choose_path(const Decoded &d, bool capture, bool bf16, Path *out) {
  if (bf16 && d.prob.dv % 2 != 0)
    return fail(GDN_ERR_UNSUPPORTED, "gdn: bf16 activations need an even D_v (got %u)", d.prob.dv);
  switch (d.path) {
    case GDN_PATH_SCAN:
      *out = Path::kScan;
      return GDN_OK;
    case GDN_PATH_CHUNKED:
    case GDN_PATH_CHUNKED_TF32:
      if (capture)
        return fail(GDN_ERR_UNSUPPORTED, "gdn: the chunked path keeps no per-token state (capture)");
      if (d.prob.dk != 128 || d.prob.dv != 128)
        return fail(GDN_ERR_UNSUPPORTED, "gdn: the chunked path needs D_k = D_v = 128");
      if (bf16 && d.path == GDN_PATH_CHUNKED_TF32)
        return fail(GDN_ERR_UNSUPPORTED, "gdn: the TF32 chunked path takes f32 activations only");
      *out = Path::kChunked;
      return GDN_OK;
    default:
      // the token loop also takes every capture window: writing each token's
      // state from the registers that hold it was measured faster than the
      // scan's capture from 24 to 256 tokens (by 2-11 % with 192 or 768
      // chains, 37 % with 48)
      if (d.prob.nt <= kDecodeMaxTokens || capture)
        *out = Path::kDecode;
      else if (!capture && d.prob.dk == 128 && d.prob.dv == 128 && d.prob.nt >= kChunkedMinTokens)
        *out = Path::kChunked;
      else
        *out = Path::kScan;
      return GDN_OK;
  }
}

// The automatic choice falls back to the scan where the chunked form cannot
// take v (rows copied 16 bytes at a time); a forced chunked path is refused
// instead (below).
Path fit_auto(const Decoded &d, Path path, const void *v) {
  return d.path == GDN_PATH_AUTO && path == Path::kChunked && !aligned(v, 16) ? Path::kScan : path;
}

// The buffers of one call, in slot order; q, k, v and output hold f32 or bf16.
struct Buffers {
  const void *q, *k, *v;
  const float *g, *beta, *state_in;
  void *output;
  float *state_out, *capture;
};

template <typename L>
Buffers buffers_of(const L &x, bool with_capture) {
  return Buffers{x.q, x.k, x.v, x.g, x.beta, x.state_in, x.output, x.state_out,
                 with_capture ? x.state_capture : nullptr};
}

// Byte spans of every buffer of one call (capture: zero bytes when absent).
struct Spans {
  Span in[6];  // q, k, v, g, beta, state_in
  Span output, state_out, capture;
};

Spans spans_of(const Decoded &d, const Buffers &b, bool bf16) {
  const unsigned long long io = bf16 ? 2 : 4;
  return Spans{{{b.q, d.qk_elems * io, "q"},
                {b.k, d.qk_elems * io, "k"},
                {b.v, d.v_elems * io, "v"},
                {b.g, d.sc_elems * 4, "g"},
                {b.beta, d.sc_elems * 4, "beta"},
                {b.state_in, d.state_elems * 4, "state_in"}},
               {b.output, d.v_elems * io, "output"},
               {b.state_out, d.state_elems * 4, "state_out"},
               {b.capture, b.capture ? d.capture_elems * 4 : 0, "state_capture"}};
}

gdn_status check_buffers(const Decoded &d, const Buffers &b, size_t capture_elems,
                         bool with_capture, bool bf16) {
  const Spans sp = spans_of(d, b, bf16);
  for (const Span &s : sp.in)
    if (s.p == nullptr) return fail(GDN_ERR_INVALID_ARGUMENT, "gdn: %s is NULL", s.name);
  if (b.output == nullptr) return fail(GDN_ERR_INVALID_ARGUMENT, "gdn: output is NULL");
  if (b.state_out == nullptr) return fail(GDN_ERR_INVALID_ARGUMENT, "gdn: state_out is NULL");
  if (with_capture && b.capture == nullptr)
    return fail(GDN_ERR_INVALID_ARGUMENT, "gdn: state_capture is NULL");

  const struct { const void *p; uintptr_t a; const char *name; } al[] = {
      {b.q, 16, "q"},        {b.k, 16, "k"},         {b.state_in, 16, "state_in"},
      {b.state_out, 16, "state_out"}, {b.v, 4, "v"}, {b.g, 4, "g"},
      {b.beta, 4, "beta"},   {b.output, bf16 ? 2u : 4u, "output"}};
  for (const auto &x : al)
    if (!aligned(x.p, x.a))
      return fail(GDN_ERR_INVALID_ARGUMENT, "gdn: %s must be %u-byte aligned", x.name,
                  static_cast<unsigned>(x.a));
  if (with_capture && !aligned(b.capture, 16))
    return fail(GDN_ERR_INVALID_ARGUMENT, "gdn: state_capture must be 16-byte aligned");

  if (with_capture) {
    if (d.prob.ns > 1 && capture_elems != d.capture_elems)
      return fail(GDN_ERR_INVALID_ARGUMENT,
                  "gdn: state_capture element count %zu != required %llu (n_tokens x state "
                  "elements); equality is required when n_seqs > 1",
                  capture_elems, d.capture_elems);
    if (d.prob.ns == 1 && capture_elems < d.capture_elems)
      return fail(GDN_ERR_INVALID_ARGUMENT, "gdn: state_capture element count %zu < required %llu",
                  capture_elems, d.capture_elems);
  }

  if (b.state_out != b.state_in && overlap(sp.state_out, sp.in[5]))
    return fail(GDN_ERR_INVALID_ARGUMENT,
                "gdn: state_in and state_out overlap without being the same buffer");
  for (const Span &s : sp.in)
    if (overlap(sp.output, s)) return fail(GDN_ERR_INVALID_ARGUMENT, "gdn: output overlaps %s", s.name);
  if (overlap(sp.output, sp.state_out))
    return fail(GDN_ERR_INVALID_ARGUMENT, "gdn: output overlaps state_out");
  for (int i = 0; i < 5; ++i)
    if (overlap(sp.state_out, sp.in[i]))
      return fail(GDN_ERR_INVALID_ARGUMENT, "gdn: state_out overlaps %s", sp.in[i].name);
  if (with_capture) {
    for (const Span &s : sp.in)
      if (overlap(sp.capture, s))
        return fail(GDN_ERR_INVALID_ARGUMENT, "gdn: state_capture overlaps %s", s.name);
    if (overlap(sp.capture, sp.output) || overlap(sp.capture, sp.state_out))
      return fail(GDN_ERR_INVALID_ARGUMENT, "gdn: state_capture overlaps an output buffer");
  }
  return GDN_OK;
}

void fill_problem(gdn::Problem &p, const Buffers &b, bool bf16) {
  p.q = b.q; p.k = b.k; p.v = b.v; p.g = b.g; p.beta = b.beta; p.state_in = b.state_in;
  p.output = b.output; p.state_out = b.state_out; p.capture = b.capture;
  p.io_bf16 = bf16;
}

// Workspace bytes of a decoded, path-checked problem (two-pass chunked only).
// The two-pass form's workspace; 0 (the one-pass form runs) off the chunked
// path, for more than kMaxSplitGroup value heads per key head, and under
// GDN_PATH_AUTO for windows shorter than kTwoPassMinTokens.
size_t workspace_bytes_of(const Decoded &d, Path path) {
  const bool two_pass = path == Path::kChunked && gdn::chunked_split_supported(d.prob) &&
                        (d.path != GDN_PATH_AUTO || d.prob.nt >= kTwoPassMinTokens);
  return two_pass ? gdn::chunked_split_workspace_bytes(d.prob) : 0;
}

// with_ws: the caller passed a workspace argument (gdn_forward_ws); the
// chunked path then runs in two passes.
gdn_status run(const Buffers &b, const uint32_t *params, size_t n_params, size_t capture_elems,
               bool with_capture, bool bf16, gdn_stream_t stream, bool with_ws = false,
               void *workspace = nullptr, size_t workspace_bytes = 0) {
  g_last_error[0] = '\0';
  Decoded d;
  gdn_status st = decode_params(params, n_params, &d);
  if (st != GDN_OK) return st;
  st = check_buffers(d, b, capture_elems, with_capture, bf16);
  if (st != GDN_OK) return st;
  Path path;
  st = choose_path(d, with_capture, bf16, &path);
  if (st != GDN_OK) return st;
  path = fit_auto(d, path, b.v);
  if (path == Path::kChunked && !aligned(b.v, 16))
    return fail(GDN_ERR_INVALID_ARGUMENT,
                "gdn: the chunked path needs v 16-byte aligned (its rows are copied 16 bytes at a time)");
  const size_t ws_need = with_ws ? workspace_bytes_of(d, path) : 0;
  if (ws_need > 0) {
    if (workspace == nullptr) return fail(GDN_ERR_INVALID_ARGUMENT, "gdn: workspace is NULL");
    if (!aligned(workspace, 16))
      return fail(GDN_ERR_INVALID_ARGUMENT, "gdn: workspace must be 16-byte aligned");
    if (workspace_bytes < ws_need)
      return fail(GDN_ERR_INVALID_ARGUMENT, "gdn: workspace has %zu bytes, %zu needed",
                  workspace_bytes, ws_need);
    const Spans sp = spans_of(d, b, bf16);
    const Span w{workspace, ws_need, "workspace"};
    const Span all[8] = {sp.in[0], sp.in[1], sp.in[2], sp.in[3], sp.in[4], sp.in[5], sp.output,
                         sp.state_out};
    for (const Span &x : all)
      if (overlap(w, x)) return fail(GDN_ERR_INVALID_ARGUMENT, "gdn: workspace overlaps %s", x.name);
  }

  gdn::Problem &p = d.prob;
  fill_problem(p, b, bf16);
  const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  const cudaError_t err =
      path == Path::kDecode    ? gdn::launch_token_loop(p, cs)
      : path == Path::kChunked ? (ws_need > 0 ? gdn::launch_chunked_split(p, static_cast<float *>(workspace), cs)
                                              : gdn::launch_chunked(p, cs))
                               : gdn::launch_scan(p, cs);
  if (err != cudaSuccess)
    return fail(GDN_ERR_CUDA, "gdn: kernel launch failed: %s", cudaGetErrorString(err));
  return GDN_OK;
}

// gdn_forward_layers and its bf16 twin: L is gdn_layer_buffers or
// gdn_layer_buffers_bf16 (same field names).
template <typename L>
gdn_status run_layers(const L *layers, size_t n_layers, const uint32_t *params, size_t n_params,
                      int with_capture, size_t state_capture_elems, bool bf16,
                      gdn_stream_t stream) {
  g_last_error[0] = '\0';
  if (layers == nullptr || n_layers == 0)
    return fail(GDN_ERR_INVALID_ARGUMENT, "gdn: layers is NULL or n_layers is 0");
  if (n_layers > kMaxLayers)
    return fail(GDN_ERR_INVALID_ARGUMENT, "gdn: n_layers %zu > %zu", n_layers, kMaxLayers);
  Decoded d;
  gdn_status st = decode_params(params, n_params, &d);
  if (st != GDN_OK) return st;
  const bool cap = with_capture != 0;
  Path path;
  st = choose_path(d, cap, bf16, &path);
  if (st != GDN_OK) return st;
  for (size_t i = 0; i < n_layers; ++i)
    path = fit_auto(d, path, layers[i].v);
  for (size_t i = 0; i < n_layers; ++i) {
    st = check_buffers(d, buffers_of(layers[i], cap), state_capture_elems, cap, bf16);
    if (st != GDN_OK) {
      char msg[sizeof g_last_error];
      std::snprintf(msg, sizeof msg, "%s", g_last_error);
      return fail(st, "%s (layer %zu)", msg, i);
    }
    if (path == Path::kChunked && !aligned(layers[i].v, 16))
      return fail(GDN_ERR_INVALID_ARGUMENT,
                  "gdn: the chunked path needs v 16-byte aligned (its rows are copied 16 bytes at a time) "
                  "(layer %zu)", i);
  }
  // No layer may write where another layer reads or writes.
  for (size_t i = 0; i < n_layers; ++i) {
    const Spans A = spans_of(d, buffers_of(layers[i], cap), bf16);
    const Span outs[3] = {A.output, A.state_out, A.capture};
    for (size_t j = 0; j < n_layers; ++j) {
      if (j == i) continue;
      const Spans B = spans_of(d, buffers_of(layers[j], cap), bf16);
      const Span all[9] = {B.in[0], B.in[1], B.in[2], B.in[3], B.in[4], B.in[5],
                           B.output, B.state_out, B.capture};
      for (const Span &o : outs) {
        if (o.p == nullptr) continue;
        for (const Span &x : all)
          if (x.p != nullptr && overlap(o, x))
            return fail(GDN_ERR_INVALID_ARGUMENT, "gdn: %s of layer %zu overlaps %s of layer %zu",
                        o.name, i, x.name, j);
      }
    }
  }
  const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  gdn::Problem batch[gdn::kMaxLayersPerLaunch];
  for (size_t i0 = 0; i0 < n_layers; i0 += gdn::kMaxLayersPerLaunch) {
    const size_t n = n_layers - i0 < gdn::kMaxLayersPerLaunch ? n_layers - i0 : gdn::kMaxLayersPerLaunch;
    for (size_t i = 0; i < n; ++i) {
      batch[i] = d.prob;
      fill_problem(batch[i], buffers_of(layers[i0 + i], cap), bf16);
    }
    cudaError_t err = cudaSuccess;
    if (path == Path::kDecode) {
      err = gdn::launch_token_loop_layers(batch, static_cast<uint32_t>(n), cs);
    } else {
      for (size_t i = 0; i < n && err == cudaSuccess; ++i)
        err = path == Path::kChunked ? gdn::launch_chunked(batch[i], cs) : gdn::launch_scan(batch[i], cs);
    }
    if (err != cudaSuccess)
      return fail(GDN_ERR_CUDA, "gdn: kernel launch failed: %s", cudaGetErrorString(err));
  }
  return GDN_OK;
}

}  // namespace

extern "C" {

gdn_status gdn_forward(const float *q, const float *k, const float *v, const float *g,
                       const float *beta, const float *state_in, float *output, float *state_out,
                       const uint32_t *params, size_t n_params, gdn_stream_t stream) {
  return run(Buffers{q, k, v, g, beta, state_in, output, state_out, nullptr}, params, n_params, 0,
             false, false, stream);
}

gdn_status gdn_forward_capture(const float *q, const float *k, const float *v, const float *g,
                               const float *beta, const float *state_in, float *output,
                               float *state_out, const uint32_t *params, size_t n_params,
                               float *state_capture, size_t state_capture_elems,
                               gdn_stream_t stream) {
  return run(Buffers{q, k, v, g, beta, state_in, output, state_out, state_capture}, params,
             n_params, state_capture_elems, true, false, stream);
}

gdn_status gdn_forward_ws(const float *q, const float *k, const float *v, const float *g,
                          const float *beta, const float *state_in, float *output,
                          float *state_out, const uint32_t *params, size_t n_params,
                          void *workspace, size_t workspace_bytes, gdn_stream_t stream) {
  return run(Buffers{q, k, v, g, beta, state_in, output, state_out, nullptr}, params, n_params, 0,
             false, false, stream, true, workspace, workspace_bytes);
}

gdn_status gdn_forward_ws_bf16(const gdn_bf16 *q, const gdn_bf16 *k, const gdn_bf16 *v,
                               const float *g, const float *beta, const float *state_in,
                               gdn_bf16 *output, float *state_out, const uint32_t *params,
                               size_t n_params, void *workspace, size_t workspace_bytes,
                               gdn_stream_t stream) {
  return run(Buffers{q, k, v, g, beta, state_in, output, state_out, nullptr}, params, n_params, 0,
             false, true, stream, true, workspace, workspace_bytes);
}

gdn_status gdn_forward_chunked_noalloc(const float *q, const float *k, const float *v,
                                       const float *g, const float *beta, const float *state_in,
                                       float *output, float *state_out, const uint32_t *params,
                                       size_t n_params, gdn_stream_t stream) {
  g_last_error[0] = '\0';
  Decoded d;
  gdn_status st = decode_params(params, n_params, &d);
  if (st != GDN_OK) return st;
  if (d.path == GDN_PATH_SCAN)
    return fail(GDN_ERR_INVALID_ARGUMENT,
                "gdn: gdn_forward_chunked_noalloc runs the chunked path only (path bits 0, 2 or 3)");
  if (d.path == GDN_PATH_AUTO) d.path = GDN_PATH_CHUNKED;
  const Buffers b{q, k, v, g, beta, state_in, output, state_out, nullptr};
  st = check_buffers(d, b, 0, false, false);
  if (st != GDN_OK) return st;
  Path path;
  st = choose_path(d, false, false, &path);
  if (st != GDN_OK) return st;
  if (!aligned(v, 16))
    return fail(GDN_ERR_INVALID_ARGUMENT,
                "gdn: the chunked path needs v 16-byte aligned (its rows are copied 16 bytes at a time)");
  gdn::Problem &p = d.prob;
  if (!gdn::chunked_split_supported(p)) {  // more value heads per key head than the two-pass form takes
    fill_problem(p, b, false);
    const cudaError_t err = gdn::launch_chunked(p, reinterpret_cast<cudaStream_t>(stream));
    if (err != cudaSuccess)
      return fail(GDN_ERR_CUDA, "gdn: kernel launch failed: %s", cudaGetErrorString(err));
    return GDN_OK;
  }
  const size_t need = gdn::chunked_split_workspace_bytes(d.prob);
  if (need > gdn::kNoallocWorkspaceBytes)
    return fail(GDN_ERR_INVALID_ARGUMENT,
                "gdn: this problem needs %zu bytes of chunk scratch; the fixed scratch of "
                "gdn_forward_chunked_noalloc holds %zu (per seq and 64-token chunk the problem "
                "takes 32 KB per value head and 96 KB per key head): use gdn_forward_ws with "
                "your own workspace",
                need, gdn::kNoallocWorkspaceBytes);
  fill_problem(p, b, false);
  const cudaError_t err = gdn::launch_chunked_split_noalloc(p, reinterpret_cast<cudaStream_t>(stream));
  if (err != cudaSuccess)
    return fail(GDN_ERR_CUDA, "gdn: kernel launch failed: %s", cudaGetErrorString(err));
  return GDN_OK;
}

gdn_status gdn_workspace_size(const uint32_t *params, size_t n_params, size_t *bytes) {
  g_last_error[0] = '\0';
  if (bytes == nullptr) return fail(GDN_ERR_INVALID_ARGUMENT, "gdn: bytes is NULL");
  *bytes = 0;
  Decoded d;
  gdn_status st = decode_params(params, n_params, &d);
  if (st != GDN_OK) return st;
  Path path;
  st = choose_path(d, false, false, &path);
  if (st != GDN_OK) return st;
  *bytes = workspace_bytes_of(d, path);
  return GDN_OK;
}

gdn_status gdn_forward_bf16(const gdn_bf16 *q, const gdn_bf16 *k, const gdn_bf16 *v,
                            const float *g, const float *beta, const float *state_in,
                            gdn_bf16 *output, float *state_out, const uint32_t *params,
                            size_t n_params, gdn_stream_t stream) {
  return run(Buffers{q, k, v, g, beta, state_in, output, state_out, nullptr}, params, n_params, 0,
             false, true, stream);
}

gdn_status gdn_forward_capture_bf16(const gdn_bf16 *q, const gdn_bf16 *k, const gdn_bf16 *v,
                                    const float *g, const float *beta, const float *state_in,
                                    gdn_bf16 *output, float *state_out, const uint32_t *params,
                                    size_t n_params, float *state_capture,
                                    size_t state_capture_elems, gdn_stream_t stream) {
  return run(Buffers{q, k, v, g, beta, state_in, output, state_out, state_capture}, params,
             n_params, state_capture_elems, true, true, stream);
}

gdn_status gdn_forward_layers(const gdn_layer_buffers *layers, size_t n_layers,
                              const uint32_t *params, size_t n_params, int with_capture,
                              size_t state_capture_elems, gdn_stream_t stream) {
  return run_layers(layers, n_layers, params, n_params, with_capture, state_capture_elems, false,
                    stream);
}

gdn_status gdn_forward_layers_bf16(const gdn_layer_buffers_bf16 *layers, size_t n_layers,
                                   const uint32_t *params, size_t n_params, int with_capture,
                                   size_t state_capture_elems, gdn_stream_t stream) {
  return run_layers(layers, n_layers, params, n_params, with_capture, state_capture_elems, true,
                    stream);
}

gdn_status gdn_commit_capture(const float *state_capture, size_t state_capture_elems,
                              const int32_t *accepted_idx, float *state, const uint32_t *params,
                              size_t n_params, gdn_stream_t stream) {
  g_last_error[0] = '\0';
  Decoded d;
  gdn_status st = decode_params(params, n_params, &d);
  if (st != GDN_OK) return st;
  if (state_capture == nullptr || accepted_idx == nullptr || state == nullptr)
    return fail(GDN_ERR_INVALID_ARGUMENT, "gdn: NULL buffer");
  if (!aligned(state_capture, 16) || !aligned(state, 16) || !aligned(accepted_idx, 4))
    return fail(GDN_ERR_INVALID_ARGUMENT,
                "gdn: state_capture and state must be 16-byte aligned, accepted_idx 4-byte");
  if (d.prob.ns > 1 && state_capture_elems != d.capture_elems)
    return fail(GDN_ERR_INVALID_ARGUMENT, "gdn: state_capture element count %zu != required %llu",
                state_capture_elems, d.capture_elems);
  if (d.prob.ns == 1 && state_capture_elems < d.capture_elems)
    return fail(GDN_ERR_INVALID_ARGUMENT, "gdn: state_capture element count %zu < required %llu",
                state_capture_elems, d.capture_elems);
  const Span cap{state_capture, d.capture_elems * 4, "state_capture"};
  const Span stt{state, d.state_elems * 4, "state"};
  const Span idx{accepted_idx, static_cast<unsigned long long>(d.prob.ns) * 4, "accepted_idx"};
  if (overlap(stt, cap) || overlap(stt, idx))
    return fail(GDN_ERR_INVALID_ARGUMENT, "gdn: state overlaps state_capture or accepted_idx");
  const cudaError_t err = gdn::launch_commit(
      state_capture, accepted_idx, state, d.prob.nt, d.prob.ns,
      static_cast<uint64_t>(d.prob.dk) * d.prob.dv * d.prob.nv,
      reinterpret_cast<cudaStream_t>(stream));
  if (err != cudaSuccess)
    return fail(GDN_ERR_CUDA, "gdn: commit launch failed: %s", cudaGetErrorString(err));
  return GDN_OK;
}

const char *gdn_last_error(void) { return g_last_error; }

gdn_status gdn_device_status(uint32_t *status, int reset, gdn_stream_t stream) {
  g_last_error[0] = '\0';
  if (status == nullptr) return fail(GDN_ERR_INVALID_ARGUMENT, "gdn: status is NULL");
  *status = 0;
  const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  unsigned int one = 0, two = 0;
  cudaError_t err = gdn::chunked_wait_status(&one, reset != 0, cs);
  if (err == cudaSuccess) err = gdn::chunked_split_wait_status(&two, reset != 0, cs);
  if (err != cudaSuccess)
    return fail(GDN_ERR_CUDA, "gdn: reading the device status failed: %s", cudaGetErrorString(err));
  *status = one | two;
  return GDN_OK;
}

gdn_status gdn_path_name(const uint32_t *params, size_t n_params, int capture,
                         const char **name) {
  g_last_error[0] = '\0';
  if (name == nullptr) return fail(GDN_ERR_INVALID_ARGUMENT, "gdn: name is NULL");
  *name = nullptr;
  Decoded d;
  gdn_status st = decode_params(params, n_params, &d);
  if (st != GDN_OK) return st;
  Path path;
  st = choose_path(d, capture != 0, false, &path);
  if (st != GDN_OK) return st;
  *name = path_name(path, capture != 0, d.prob.tf32);
  return GDN_OK;
}

}  // extern "C"

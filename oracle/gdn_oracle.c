/*
 * gdn_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously-correct CPU oracle of the Gated DeltaNet
 * recurrence, in double precision.  Only the test suite, the smoke check and
 * the benchmark's CPU-baseline leg load it.  The CUDA library never links,
 * includes or calls anything in this directory, and this file includes no
 * header of that library: the two share no code.
 *
 * What it computes (one (seq s, value head vh) pair at a time, tokens in
 * order), following the pages:
 *
 *   decay-first (the default, flags bit0 = 0) -- the step order of the
 *   kernel body in "gated_delta_net_decode_capture.metal" (mlx-native 0.9.2),
 *   steps "decay + partial s_k" and "state update + output partial":
 *       alpha   = exp(-g_t)
 *       S       = alpha * S
 *       sk[i]   = sum_j S[i][j] * k_t[j]
 *       delta[i]= (v_t[i] - sk[i]) * beta_t
 *       S[i][j] = S[i][j] + delta[i] * k_t[j]
 *       y_t[i]  = q_scale * sum_j S[i][j] * q_t[j]
 *
 *   decay-after (flags bit0 = 1) -- the recurrence in the module doc of
 *   "gated_delta_net.rs" (mlx-native 0.4.0) and its cpu_reference_f32:
 *       alpha   = exp(-g_t)
 *       delta[i]= v_t[i] - sum_j S[i][j] * k_t[j]        (S not yet decayed)
 *       S[i][j] = alpha * S[i][j] + beta_t * delta[i] * k_t[j]
 *       y_t[i]  = q_scale * sum_j S[i][j] * q_t[j]
 *
 *   S is the D_v x D_k state of the pair, row i = d_v index, column j = d_k
 *   index.  With capture, the state after token t is written to slice t of
 *   state_capture.  After the last token, S is written to state_out.
 *
 * Parameters: the 9-u32 params array of the "Buffer bindings" section of the
 * capture kernel page, (D_k, D_v, n_k_heads, n_v_heads, n_tokens, n_seqs,
 * 0, 0, q_scale_bits), where q_scale_bits == 0 means q_scale = 1.0.  Slot 6
 * carries flag bits (bit0 decay-after, bit1 k_head by division, bits 2-3 a
 * GPU path choice that the oracle ignores); slot 7 is reserved and must be 0.
 *
 * k_head mapping (the "GQA broadcast" section of gated_delta_net.rs and the
 * capture kernel's head setup): flags bit1 = 0 -> vh % n_k_heads (the
 * capture kernel), bit1 = 1 -> vh / (n_v_heads / n_k_heads) (gated_delta_net.rs).
 *
 * Layouts (innermost first), from the "Memory layouts" table of
 * gated_delta_net.rs and the "Memory layout for state_capture" section of the
 * capture kernel page:
 *   q, k           [D_k, n_k_heads, n_tokens, n_seqs]
 *   v, output      [D_v, n_v_heads, n_tokens, n_seqs]
 *   g, beta        [n_v_heads, n_tokens, n_seqs]
 *   state_in/out   [D_k, D_v, n_v_heads, n_seqs]
 *   state_capture  [D_k, D_v, n_v_heads, n_tokens, n_seqs]
 *
 * Precision: q, k, v, g, beta are f32 (as the pages' buffers are); all
 * arithmetic is double; exp is libm's double exp.  state_in may be given
 * as f32 or f64 (f64 lets chained calls be compared exactly).
 */
#include <math.h>
#include <pthread.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_BAD_ARGUMENT 1
#define ORACLE_NO_MEMORY 2

#define FLAG_DECAY_AFTER 0x1u
#define FLAG_KHEAD_DIV 0x2u
#define FLAG_PATH_MASK 0xCu
#define FLAG_KNOWN (FLAG_DECAY_AFTER | FLAG_KHEAD_DIV | FLAG_PATH_MASK)

typedef struct {
  size_t dk, dv, nk, nv, nt, ns;
  uint32_t flags;
  double q_scale;
} problem_t;

typedef struct {
  const problem_t *p;
  const float *q, *k, *v, *g, *beta;
  const void *state_in;
  int state_in_f64;
  /* Which heads to run: heads[h] = s * n_v + vh, or all heads in order when
   * heads == NULL. */
  const uint32_t *heads;
  size_t n_heads;
  /* Full-layout outputs (compact == 0) or per-listed-head outputs
   * (compact == 1: output [n][T][D_v], state [n][D_v][D_k],
   * capture [n][T][D_v][D_k]). */
  int compact;
  double *output, *state_out, *capture;
  size_t next; /* work counter, taken atomically */
} job_t;

static int decode_params(const uint32_t *params, size_t n_params, problem_t *p) {
  if (params == NULL || n_params < 9) return ORACLE_BAD_ARGUMENT;
  p->dk = params[0];
  p->dv = params[1];
  p->nk = params[2];
  p->nv = params[3];
  p->nt = params[4];
  p->ns = params[5];
  p->flags = params[6];
  if (p->dk == 0 || p->dv == 0 || p->nk == 0 || p->nv == 0 || p->nt == 0 || p->ns == 0)
    return ORACLE_BAD_ARGUMENT;
  if (p->nv % p->nk != 0) return ORACLE_BAD_ARGUMENT;
  if ((p->flags & ~FLAG_KNOWN) != 0) return ORACLE_BAD_ARGUMENT;
  if (params[7] != 0) return ORACLE_BAD_ARGUMENT;
  if (params[8] == 0) {
    p->q_scale = 1.0;
  } else {
    float f;
    uint32_t bits = params[8];
    memcpy(&f, &bits, sizeof f);
    p->q_scale = (double)f;
  }
  return ORACLE_OK;
}

/* Runs the recurrence for one (s, vh) pair.  S is D_v*D_k doubles of work
 * space, sk is D_v doubles. */
static void run_head(const job_t *job, size_t slot, size_t s, size_t vh, double *S, double *sk) {
  const problem_t *p = job->p;
  const size_t dk = p->dk, dv = p->dv, nk = p->nk, nv = p->nv, nt = p->nt;
  const int decay_after = (p->flags & FLAG_DECAY_AFTER) != 0;
  const size_t kh = (p->flags & FLAG_KHEAD_DIV) ? vh / (nv / nk) : vh % nk;

  /* state_in[j, i, vh, s] -> S[i][j] */
  const size_t state_base = dk * dv * (vh + nv * s);
  for (size_t i = 0; i < dv; ++i)
    for (size_t j = 0; j < dk; ++j) {
      const size_t src = state_base + j + dk * i;
      S[i * dk + j] = job->state_in_f64 ? ((const double *)job->state_in)[src]
                                        : (double)((const float *)job->state_in)[src];
    }

  for (size_t t = 0; t < nt; ++t) {
    const float *kt = job->k + dk * (kh + nk * (t + nt * s));
    const float *qt = job->q + dk * (kh + nk * (t + nt * s));
    const float *vt = job->v + dv * (vh + nv * (t + nt * s));
    const size_t sc = vh + nv * (t + nt * s);
    const double g = (double)job->g[sc];
    const double beta = (double)job->beta[sc];
    const double alpha = exp(-g);

    if (!decay_after) {
      for (size_t i = 0; i < dv * dk; ++i) S[i] = alpha * S[i];
      for (size_t i = 0; i < dv; ++i) {
        double acc = 0.0;
        for (size_t j = 0; j < dk; ++j) acc += S[i * dk + j] * (double)kt[j];
        sk[i] = acc;
      }
      for (size_t i = 0; i < dv; ++i) {
        const double delta = ((double)vt[i] - sk[i]) * beta;
        for (size_t j = 0; j < dk; ++j) S[i * dk + j] = S[i * dk + j] + delta * (double)kt[j];
      }
    } else {
      for (size_t i = 0; i < dv; ++i) {
        double acc = 0.0;
        for (size_t j = 0; j < dk; ++j) acc += S[i * dk + j] * (double)kt[j];
        sk[i] = acc;
      }
      for (size_t i = 0; i < dv; ++i) {
        const double delta = (double)vt[i] - sk[i];
        for (size_t j = 0; j < dk; ++j)
          S[i * dk + j] = alpha * S[i * dk + j] + beta * delta * (double)kt[j];
      }
    }

    /* y_t[i] = q_scale * sum_j S[i][j] q_t[j] on the updated state */
    for (size_t i = 0; i < dv; ++i) {
      double acc = 0.0;
      for (size_t j = 0; j < dk; ++j) acc += S[i * dk + j] * (double)qt[j];
      const double y = p->q_scale * acc;
      if (job->compact)
        job->output[(slot * nt + t) * dv + i] = y;
      else
        job->output[i + dv * (vh + nv * (t + nt * s))] = y;
    }

    if (job->capture != NULL) {
      for (size_t i = 0; i < dv; ++i)
        for (size_t j = 0; j < dk; ++j) {
          const size_t dst = job->compact ? ((slot * nt + t) * dv + i) * dk + j
                                          : j + dk * (i + dv * (vh + nv * (t + nt * s)));
          job->capture[dst] = S[i * dk + j];
        }
    }
  }

  for (size_t i = 0; i < dv; ++i)
    for (size_t j = 0; j < dk; ++j) {
      const size_t dst = job->compact ? (slot * dv + i) * dk + j : state_base + j + dk * i;
      job->state_out[dst] = S[i * dk + j];
    }
}

static void *worker(void *arg) {
  job_t *job = (job_t *)arg;
  const problem_t *p = job->p;
  double *S = (double *)malloc(sizeof(double) * p->dv * p->dk);
  double *sk = (double *)malloc(sizeof(double) * p->dv);
  if (S == NULL || sk == NULL) {
    free(S);
    free(sk);
    return (void *)1;
  }
  for (;;) {
    const size_t slot = __atomic_fetch_add(&job->next, 1, __ATOMIC_RELAXED);
    if (slot >= job->n_heads) break;
    const size_t h = job->heads ? job->heads[slot] : slot;
    run_head(job, slot, h / p->nv, h % p->nv, S, sk);
  }
  free(S);
  free(sk);
  return NULL;
}

static int run_job(job_t *job, int n_threads) {
  if (n_threads < 1) n_threads = 1;
  if ((size_t)n_threads > job->n_heads) n_threads = (int)job->n_heads;
  pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)n_threads);
  if (tid == NULL) return ORACLE_NO_MEMORY;
  int started = 0, failed = 0;
  for (int i = 1; i < n_threads; ++i) {
    if (pthread_create(&tid[i], NULL, worker, job) != 0) break;
    started = i;
  }
  if (worker(job) != NULL) failed = 1;
  for (int i = 1; i <= started; ++i) {
    void *ret = NULL;
    pthread_join(tid[i], &ret);
    if (ret != NULL) failed = 1;
  }
  free(tid);
  return failed ? ORACLE_NO_MEMORY : ORACLE_OK;
}

/* Full problem.  Inputs in the pages' layouts; outputs in the same layouts,
 * as doubles.  state_capture may be NULL (no capture).  Returns 0, or 1 for
 * parameters the pages reject, or 2 when memory runs out. */
int gdn_oracle_forward(const uint32_t *params, size_t n_params, const float *q, const float *k,
                       const float *v, const float *g, const float *beta, const void *state_in,
                       int state_in_f64, double *output, double *state_out, double *state_capture,
                       int n_threads) {
  problem_t p;
  const int rc = decode_params(params, n_params, &p);
  if (rc != ORACLE_OK) return rc;
  if (!q || !k || !v || !g || !beta || !state_in || !output || !state_out)
    return ORACLE_BAD_ARGUMENT;
  job_t job = {&p, q, k, v, g, beta, state_in, state_in_f64, NULL, p.ns * p.nv, 0,
               output, state_out, state_capture, 0};
  return run_job(&job, n_threads);
}

/* A listed subset of heads (head = s * n_v_heads + vh), for sampled checks
 * of full-size problems.  Inputs are the full-layout buffers; outputs are
 * compact: output [n_heads][T][D_v], state_out [n_heads][D_v][D_k],
 * state_capture [n_heads][T][D_v][D_k] (or NULL). */
int gdn_oracle_forward_heads(const uint32_t *params, size_t n_params, const float *q,
                             const float *k, const float *v, const float *g, const float *beta,
                             const void *state_in, int state_in_f64, const uint32_t *heads,
                             size_t n_heads, double *output, double *state_out,
                             double *state_capture, int n_threads) {
  problem_t p;
  const int rc = decode_params(params, n_params, &p);
  if (rc != ORACLE_OK) return rc;
  if (!q || !k || !v || !g || !beta || !state_in || !output || !state_out || !heads)
    return ORACLE_BAD_ARGUMENT;
  for (size_t h = 0; h < n_heads; ++h)
    if (heads[h] >= p.ns * p.nv) return ORACLE_BAD_ARGUMENT;
  job_t job = {&p, q, k, v, g, beta, state_in, state_in_f64, heads, n_heads, 1,
               output, state_out, state_capture, 0};
  return run_job(&job, n_threads);
}

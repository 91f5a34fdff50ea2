/*
 * fp64 CPU oracle for the gated delta rule prefill over packed sequences.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path links, loads or calls
 * this file; only the tests, the smoke check and the bench's CPU-baseline /
 * reference arm do. It shares no code, header or constant with the CUDA
 * library.
 *
 * What it computes (one independent chain per sequence n and value head h):
 *
 *   S_t = exp(g_t) (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T
 *   o_t = scale * S_t^T q_t
 *
 * the gated delta rule of "Gated Delta Networks: Improving Mamba2 with Delta
 * Rule" (Yang, Kautz, Hatamizadeh, ICLR 2025), the model's recurrent
 * linear-attention layer in System1-Omni PR #186 ("Purpose and summary") and
 * reference [5] of the open-jev-fast README. k_t and q_t are L2-normalised
 * first, as x / sqrt(|x|^2 + eps); that README does the normalisation in its
 * linear-attention input-prep kernel (Phase 2 item 1).
 *
 * Readings taken where the pages are silent:
 *  - the decay multiplies the whole (I - beta k k^T) S term, so the delta
 *    correction uses the decayed state: S' = e^g S; u = beta (v - S'^T k);
 *    S = S' + k u^T, which expands to the formula above;
 *  - value head h uses q/k head h / (h_v / h_qk) (contiguous groups);
 *  - scale defaults to d_k^-1/2 (the caller passes it);
 *  - a sequence of length 0 returns its initial state unchanged;
 *  - state_index[n] < 0 selects a zero initial state.
 *
 * Two independent routines:
 *  gdn_oracle_recurrent  - the token-by-token definition above (parity oracle);
 *  gdn_oracle_chunked    - the chunked (WY/UT) form the pages' kernel follows
 *                          (open-jev-fast README, Phase 3 item 1: gate cumsum,
 *                          K K^T, the (I + A)^-1 solve, u and w, the chunk
 *                          output and the state update), derived from the
 *                          recurrence; used only to cross-check the recurrence.
 *
 * Inputs are float32 arrays holding the exact stored values (bf16 values widen
 * exactly); every operation is carried out in double. No fast-math.
 *
 * Layouts (row-major): q, k [T, h_qk, d_k]; v [T, h_v, d_v]; g, beta [T, h_v];
 * cu_seqlens [N+1]; initial_state [n_slots, h_v, d_k, d_v];
 * state_index [N] (or NULL: sequence n reads slot n); out [T, h_v, d_v];
 * final_state [N, h_v, d_k, d_v]. unit_mask [N * h_v] (or NULL: all): units
 * with mask 0 are skipped and their outputs left untouched.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
  int n_seqs;
  const int64_t *cu;
  int h_qk, h_v, d_k, d_v;
  const float *q, *k, *v, *g, *beta, *s0;
  int n_slots;
  const int64_t *sidx;
  double scale;
  int l2norm;
  double eps;
  const unsigned char *mask;
  double *out, *fs;
  int chunk; /* 0: recurrent */
  int next;
  int err;
  pthread_mutex_t mu;
} job_t;

static void load_row(const float *src, int n, double *dst, int l2norm, double eps) {
  double ss = 0.0;
  for (int i = 0; i < n; ++i) {
    dst[i] = (double)src[i];
    ss += dst[i] * dst[i];
  }
  if (l2norm) {
    double r = 1.0 / sqrt(ss + eps);
    for (int i = 0; i < n; ++i) dst[i] *= r;
  }
}

/* Initial state of one unit into S [d_k][d_v]; returns 0 or -1 (bad slot). */
static int load_state(const job_t *J, int n, int h, double *S) {
  const int dk = J->d_k, dv = J->d_v;
  memset(S, 0, sizeof(double) * (size_t)dk * dv);
  if (!J->s0) return 0;
  int64_t slot = J->sidx ? J->sidx[n] : n;
  if (slot < 0) return 0;
  if (slot >= J->n_slots) return -1;
  const float *src = J->s0 + ((size_t)slot * J->h_v + h) * (size_t)dk * dv;
  for (size_t i = 0; i < (size_t)dk * dv; ++i) S[i] = (double)src[i];
  return 0;
}

static void store_state(const job_t *J, int n, int h, const double *S) {
  if (!J->fs) return;
  const size_t sz = (size_t)J->d_k * J->d_v;
  memcpy(J->fs + ((size_t)n * J->h_v + h) * sz, S, sizeof(double) * sz);
}

/* The definition, one token at a time. */
static int unit_recurrent(const job_t *J, int n, int h, double *S, double *kk, double *qq,
                          double *u) {
  const int dk = J->d_k, dv = J->d_v, hq = h / (J->h_v / J->h_qk);
  if (load_state(J, n, h, S)) return -1;
  for (int64_t t = J->cu[n]; t < J->cu[n + 1]; ++t) {
    load_row(J->k + ((size_t)t * J->h_qk + hq) * dk, dk, kk, J->l2norm, J->eps);
    load_row(J->q + ((size_t)t * J->h_qk + hq) * dk, dk, qq, J->l2norm, J->eps);
    const float *vt = J->v + ((size_t)t * J->h_v + h) * dv;
    const double a = exp((double)J->g[(size_t)t * J->h_v + h]);
    const double b = (double)J->beta[(size_t)t * J->h_v + h];
    /* S <- e^g S */
    for (size_t i = 0; i < (size_t)dk * dv; ++i) S[i] *= a;
    /* u = beta (v - S^T k) */
    for (int j = 0; j < dv; ++j) u[j] = 0.0;
    for (int i = 0; i < dk; ++i)
      for (int j = 0; j < dv; ++j) u[j] += S[(size_t)i * dv + j] * kk[i];
    for (int j = 0; j < dv; ++j) u[j] = b * ((double)vt[j] - u[j]);
    /* S <- S + k u^T */
    for (int i = 0; i < dk; ++i)
      for (int j = 0; j < dv; ++j) S[(size_t)i * dv + j] += kk[i] * u[j];
    /* o = scale S^T q */
    if (J->out) {
      double *o = J->out + ((size_t)t * J->h_v + h) * dv;
      for (int j = 0; j < dv; ++j) o[j] = 0.0;
      for (int i = 0; i < dk; ++i)
        for (int j = 0; j < dv; ++j) o[j] += S[(size_t)i * dv + j] * qq[i];
      for (int j = 0; j < dv; ++j) o[j] *= J->scale;
    }
  }
  store_state(J, n, h, S);
  return 0;
}

/*
 * The chunked form, derived from the recurrence. Inside a chunk that starts
 * from state S0 with G_i = sum_{s<=i} g_s:
 *   (I + A) U' = diag(beta) V - diag(beta e^G) K S0,  A_ij = beta_i e^{G_i-G_j} k_i.k_j (j<i)
 *   T = (I + A)^-1, U = T diag(beta) V, W = T diag(beta e^G) K, U' = U - W S0
 *   o_i = scale (e^{G_i} S0^T q_i + sum_{j<=i} e^{G_i-G_j} (q_i.k_j) u'_j)
 *   S_C = e^{G_C} S0 + sum_j e^{G_C-G_j} k_j u'_j^T
 */
typedef struct {
  double *K, *Q, *V, *G, *B, *A, *T, *U, *W, *Up, *S2;
} chunk_ws_t;

static int unit_chunked(const job_t *J, int n, int h, double *S, chunk_ws_t *w) {
  const int dk = J->d_k, dv = J->d_v, C = J->chunk, hq = h / (J->h_v / J->h_qk);
  if (load_state(J, n, h, S)) return -1;
  for (int64_t c0 = J->cu[n]; c0 < J->cu[n + 1]; c0 += C) {
    const int m = (int)((J->cu[n + 1] - c0) < C ? (J->cu[n + 1] - c0) : C);
    double acc = 0.0;
    for (int i = 0; i < m; ++i) {
      const int64_t t = c0 + i;
      load_row(J->k + ((size_t)t * J->h_qk + hq) * dk, dk, w->K + (size_t)i * dk, J->l2norm,
               J->eps);
      load_row(J->q + ((size_t)t * J->h_qk + hq) * dk, dk, w->Q + (size_t)i * dk, J->l2norm,
               J->eps);
      for (int j = 0; j < dv; ++j) w->V[(size_t)i * dv + j] = J->v[((size_t)t * J->h_v + h) * dv + j];
      acc += (double)J->g[(size_t)t * J->h_v + h];
      w->G[i] = acc; /* gate cumsum */
      w->B[i] = J->beta[(size_t)t * J->h_v + h];
    }
    /* A (strictly lower) */
    for (int i = 0; i < m; ++i)
      for (int j = 0; j < m; ++j) {
        double a = 0.0;
        if (j < i) {
          double kk = 0.0;
          for (int x = 0; x < dk; ++x) kk += w->K[(size_t)i * dk + x] * w->K[(size_t)j * dk + x];
          a = w->B[i] * exp(w->G[i] - w->G[j]) * kk;
        }
        w->A[(size_t)i * m + j] = a;
      }
    /* T = (I + A)^-1 by forward substitution, row by row */
    for (int i = 0; i < m; ++i)
      for (int j = 0; j < m; ++j) {
        double s = (i == j) ? 1.0 : 0.0;
        for (int x = 0; x < i; ++x) s -= w->A[(size_t)i * m + x] * w->T[(size_t)x * m + j];
        w->T[(size_t)i * m + j] = s;
      }
    /* U = T diag(beta) V ; W = T diag(beta e^G) K */
    for (int i = 0; i < m; ++i) {
      for (int j = 0; j < dv; ++j) {
        double s = 0.0;
        for (int x = 0; x < m; ++x) s += w->T[(size_t)i * m + x] * w->B[x] * w->V[(size_t)x * dv + j];
        w->U[(size_t)i * dv + j] = s;
      }
      for (int j = 0; j < dk; ++j) {
        double s = 0.0;
        for (int x = 0; x < m; ++x)
          s += w->T[(size_t)i * m + x] * w->B[x] * exp(w->G[x]) * w->K[(size_t)x * dk + j];
        w->W[(size_t)i * dk + j] = s;
      }
    }
    /* U' = U - W S0 */
    for (int i = 0; i < m; ++i)
      for (int j = 0; j < dv; ++j) {
        double s = w->U[(size_t)i * dv + j];
        for (int x = 0; x < dk; ++x) s -= w->W[(size_t)i * dk + x] * S[(size_t)x * dv + j];
        w->Up[(size_t)i * dv + j] = s;
      }
    /* chunk output */
    if (J->out) {
      for (int i = 0; i < m; ++i) {
        double *o = J->out + ((size_t)(c0 + i) * J->h_v + h) * dv;
        const double eg = exp(w->G[i]);
        for (int j = 0; j < dv; ++j) {
          double s = 0.0;
          for (int x = 0; x < dk; ++x) s += S[(size_t)x * dv + j] * w->Q[(size_t)i * dk + x];
          o[j] = eg * s;
        }
        for (int jj = 0; jj <= i; ++jj) {
          double qk = 0.0;
          for (int x = 0; x < dk; ++x) qk += w->Q[(size_t)i * dk + x] * w->K[(size_t)jj * dk + x];
          const double p = exp(w->G[i] - w->G[jj]) * qk;
          for (int j = 0; j < dv; ++j) o[j] += p * w->Up[(size_t)jj * dv + j];
        }
        for (int j = 0; j < dv; ++j) o[j] *= J->scale;
      }
    }
    /* state update */
    const double gc = w->G[m - 1];
    for (size_t i = 0; i < (size_t)dk * dv; ++i) w->S2[i] = exp(gc) * S[i];
    for (int jj = 0; jj < m; ++jj) {
      const double d = exp(gc - w->G[jj]);
      for (int x = 0; x < dk; ++x) {
        const double kx = d * w->K[(size_t)jj * dk + x];
        for (int j = 0; j < dv; ++j) w->S2[(size_t)x * dv + j] += kx * w->Up[(size_t)jj * dv + j];
      }
    }
    memcpy(S, w->S2, sizeof(double) * (size_t)dk * dv);
  }
  store_state(J, n, h, S);
  return 0;
}

static void *worker(void *arg) {
  job_t *J = (job_t *)arg;
  const int dk = J->d_k, dv = J->d_v, C = J->chunk > 0 ? J->chunk : 1;
  double *S = (double *)malloc(sizeof(double) * (size_t)dk * dv);
  double *kk = (double *)malloc(sizeof(double) * (size_t)dk);
  double *qq = (double *)malloc(sizeof(double) * (size_t)dk);
  double *u = (double *)malloc(sizeof(double) * (size_t)dv);
  chunk_ws_t w;
  memset(&w, 0, sizeof(w));
  if (J->chunk > 0) {
    w.K = (double *)malloc(sizeof(double) * (size_t)C * dk);
    w.Q = (double *)malloc(sizeof(double) * (size_t)C * dk);
    w.V = (double *)malloc(sizeof(double) * (size_t)C * dv);
    w.G = (double *)malloc(sizeof(double) * (size_t)C);
    w.B = (double *)malloc(sizeof(double) * (size_t)C);
    w.A = (double *)malloc(sizeof(double) * (size_t)C * C);
    w.T = (double *)malloc(sizeof(double) * (size_t)C * C);
    w.U = (double *)malloc(sizeof(double) * (size_t)C * dv);
    w.W = (double *)malloc(sizeof(double) * (size_t)C * dk);
    w.Up = (double *)malloc(sizeof(double) * (size_t)C * dv);
    w.S2 = (double *)malloc(sizeof(double) * (size_t)dk * dv);
  }
  const int total = J->n_seqs * J->h_v;
  for (;;) {
    pthread_mutex_lock(&J->mu);
    const int idx = J->next++;
    pthread_mutex_unlock(&J->mu);
    if (idx >= total) break;
    if (J->mask && !J->mask[idx]) continue;
    const int n = idx / J->h_v, h = idx % J->h_v;
    const int rc = J->chunk > 0 ? unit_chunked(J, n, h, S, &w) : unit_recurrent(J, n, h, S, kk, qq, u);
    if (rc) {
      pthread_mutex_lock(&J->mu);
      J->err = rc;
      pthread_mutex_unlock(&J->mu);
    }
  }
  free(S); free(kk); free(qq); free(u);
  free(w.K); free(w.Q); free(w.V); free(w.G); free(w.B); free(w.A); free(w.T);
  free(w.U); free(w.W); free(w.Up); free(w.S2);
  return NULL;
}

static int run(job_t *J, int n_threads) {
  if (J->n_seqs < 0 || J->h_qk <= 0 || J->h_v <= 0 || J->d_k <= 0 || J->d_v <= 0) return -2;
  if (J->h_v % J->h_qk) return -3;
  for (int n = 0; n < J->n_seqs; ++n)
    if (J->cu[n + 1] < J->cu[n]) return -4;
  if (n_threads < 1) n_threads = 1;
  if (n_threads > 256) n_threads = 256;
  pthread_mutex_init(&J->mu, NULL);
  J->next = 0;
  J->err = 0;
  pthread_t th[256];
  for (int i = 0; i < n_threads; ++i) pthread_create(&th[i], NULL, worker, J);
  for (int i = 0; i < n_threads; ++i) pthread_join(th[i], NULL);
  pthread_mutex_destroy(&J->mu);
  return J->err;
}

#define FILL_JOB                                                                              \
  job_t J;                                                                                    \
  memset(&J, 0, sizeof(J));                                                                   \
  J.n_seqs = n_seqs; J.cu = cu_seqlens; J.h_qk = h_qk; J.h_v = h_v; J.d_k = d_k; J.d_v = d_v; \
  J.q = q; J.k = k; J.v = v; J.g = g; J.beta = beta; J.s0 = initial_state;                   \
  J.n_slots = n_slots; J.sidx = state_index; J.scale = scale; J.l2norm = l2norm; J.eps = eps; \
  J.mask = unit_mask; J.out = out; J.fs = final_state;

/* Returns 0, or a negative code: -1 state slot out of range, -2 bad sizes,
 * -3 h_v not a multiple of h_qk, -4 decreasing cu_seqlens, -5 bad chunk. */
int gdn_oracle_recurrent(int n_seqs, const int64_t *cu_seqlens, int h_qk, int h_v, int d_k,
                         int d_v, const float *q, const float *k, const float *v, const float *g,
                         const float *beta, const float *initial_state, int n_slots,
                         const int64_t *state_index, double scale, int l2norm, double eps,
                         const unsigned char *unit_mask, double *out, double *final_state,
                         int n_threads) {
  FILL_JOB
  J.chunk = 0;
  return run(&J, n_threads);
}

int gdn_oracle_chunked(int n_seqs, const int64_t *cu_seqlens, int h_qk, int h_v, int d_k,
                       int d_v, const float *q, const float *k, const float *v, const float *g,
                       const float *beta, const float *initial_state, int n_slots,
                       const int64_t *state_index, double scale, int l2norm, double eps,
                       const unsigned char *unit_mask, double *out, double *final_state,
                       int chunk, int n_threads) {
  if (chunk < 1) return -5;
  FILL_JOB
  J.chunk = chunk;
  return run(&J, n_threads);
}

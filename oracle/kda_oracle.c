/*
 * Kimi Delta Attention (KDA): fp64 CPU oracle.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path loads this library:
 * only the test suite, the smoke check and the benchmark's CPU-baseline leg
 * do.  It shares no code, header, table or helper with the CUDA library.
 *
 * Source of the operation: "[Paper Review] Kimi K3: Open Frontier
 * Intelligence" (baba9811.github.io), section "Kimi Delta Attention (KDA)".
 * The display equation of that section was lost from the page text; its prose
 * fixes the form used here: Diag(alpha_t) is a per-channel forget gate that
 * decays the prior state, and (I - beta_t k_t k_t^T) erases the key-direction
 * component before the new key-value pair is written.  Per head:
 *
 *     S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T
 *     o_t = S_t^T q_t            S_t in R^{dk x dv},  alpha_t = exp(g_t)
 *
 * The oracle evaluates this one token at a time in the algebraically identical
 * expanded form
 *     S' = Diag(alpha_t) S_{t-1};  u = S'^T k_t;
 *     S_t = S' + beta_t k_t (v_t - u)^T;   o_t = S_t^T q_t
 * with no chunking, blocking or reordering.  Sequences are packed token-major
 * and delimited by cu_seqlens (the state restarts from init_state at every
 * sequence start).
 *
 * Layouts (row-major, token-major packed):
 *   q, k, g : [T_total, H, dk]      v, out : [T_total, H, dv]
 *   beta    : [T_total, H]          state  : [N, H, dk, dv]  (dv fastest)
 * Inputs may be fp32, bf16 (raw 16-bit patterns) or fp64; each element is
 * widened to fp64 exactly before use, so the oracle sees the same bytes the
 * GPU sees.  All arithmetic is fp64.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

enum { ORC_F32 = 0, ORC_BF16 = 1, ORC_F64 = 2 };

/* Widen one stored element to fp64 (exact for all three formats). */
static double orc_read(const void* base, int dtype, long long idx) {
  if (dtype == ORC_F64) return ((const double*)base)[idx];
  if (dtype == ORC_F32) return (double)((const float*)base)[idx];
  uint32_t bits = (uint32_t)((const uint16_t*)base)[idx] << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

typedef struct {
  const void *q, *k, *v, *g, *beta;
  int dtype;
  const double* init_state; /* nullable: zero initial state */
  const long long* cu_seqlens; /* [n_seqs + 1] */
  int n_seqs, heads, dk, dv;
  double* out;              /* [T_total, H, dv] */
  double* final_state;      /* nullable */
  double* checkpoints;      /* nullable: [n_ckpt, H, dk, dv] */
  const long long* ckpt_offsets; /* [n_seqs + 1] when checkpoints != NULL */
  long long ckpt_interval;  /* tokens between checkpoints */
  int next_job;             /* shared work counter */
} orc_job_t;

/* One (sequence, head): the token-by-token recurrence. */
static void orc_run_pair(const orc_job_t* J, int n, int h, double* S, double* kk,
                         double* qq, double* alpha, double* u) {
  const int H = J->heads, dk = J->dk, dv = J->dv;
  const long long state_off = ((long long)n * H + h) * dk * dv;
  if (J->init_state)
    memcpy(S, J->init_state + state_off, sizeof(double) * dk * dv);
  else
    memset(S, 0, sizeof(double) * dk * dv);

  for (long long t = J->cu_seqlens[n]; t < J->cu_seqlens[n + 1]; ++t) {
    const long long rk = (t * H + h) * dk, rv = (t * H + h) * dv;
    for (int c = 0; c < dk; ++c) {
      kk[c] = orc_read(J->k, J->dtype, rk + c);
      qq[c] = orc_read(J->q, J->dtype, rk + c);
      alpha[c] = exp(orc_read(J->g, J->dtype, rk + c));
    }
    const double b = orc_read(J->beta, J->dtype, t * H + h);

    /* S' = Diag(alpha) S : channel c of the key dimension keeps alpha_c. */
    for (int c = 0; c < dk; ++c)
      for (int j = 0; j < dv; ++j) S[c * dv + j] *= alpha[c];

    /* u = S'^T k : what the decayed state currently returns for key k. */
    for (int j = 0; j < dv; ++j) u[j] = 0.0;
    for (int c = 0; c < dk; ++c)
      for (int j = 0; j < dv; ++j) u[j] += S[c * dv + j] * kk[c];

    /* S = S' + beta k (v - u)^T : the delta-rule write. */
    for (int j = 0; j < dv; ++j) u[j] = b * (orc_read(J->v, J->dtype, rv + j) - u[j]);
    for (int c = 0; c < dk; ++c)
      for (int j = 0; j < dv; ++j) S[c * dv + j] += kk[c] * u[j];

    /* o = S^T q, read from the updated state (includes token t). */
    for (int j = 0; j < dv; ++j) u[j] = 0.0;
    for (int c = 0; c < dk; ++c)
      for (int j = 0; j < dv; ++j) u[j] += S[c * dv + j] * qq[c];
    memcpy(J->out + rv, u, sizeof(double) * dv);

    /* Prefix-cache checkpoint: the state after every ckpt_interval tokens. */
    const long long done = t - J->cu_seqlens[n] + 1;
    if (J->checkpoints && done % J->ckpt_interval == 0) {
      const long long row = J->ckpt_offsets[n] + done / J->ckpt_interval - 1;
      memcpy(J->checkpoints + (row * H + h) * dk * dv, S, sizeof(double) * dk * dv);
    }
  }
  if (J->final_state) memcpy(J->final_state + state_off, S, sizeof(double) * dk * dv);
}

static void* orc_worker(void* arg) {
  orc_job_t* J = (orc_job_t*)arg;
  const int dk = J->dk, dv = J->dv;
  double* S = (double*)malloc(sizeof(double) * ((size_t)dk * dv + 3 * (size_t)dk + (size_t)dv));
  if (!S) return (void*)1;
  double* kk = S + (size_t)dk * dv;
  double* qq = kk + dk;
  double* alpha = qq + dk;
  double* u = alpha + dk;
  const int n_jobs = J->n_seqs * J->heads;
  for (;;) {
    int job = __atomic_fetch_add(&J->next_job, 1, __ATOMIC_RELAXED);
    if (job >= n_jobs) break;
    orc_run_pair(J, job / J->heads, job % J->heads, S, kk, qq, alpha, u);
  }
  free(S);
  return NULL;
}

/* Number of threads the oracle uses when the caller passes n_threads <= 0. */
int kda_oracle_default_threads(void) {
  long n = sysconf(_SC_NPROCESSORS_ONLN);
  return n > 0 ? (int)n : 1;
}

/*
 * Prefill over packed sequences, optionally also writing the state after every
 * ckpt_interval tokens of each sequence (the prefix-cache checkpoints of the
 * paper review's serving description): checkpoint k of sequence n (state after
 * (k+1) * ckpt_interval tokens) is row ckpt_offsets[n] + k of `checkpoints`.
 * Returns the number of threads used, or a negative value on bad arguments /
 * allocation failure.
 */
int kda_oracle_prefill_ckpt(const void* q, const void* k, const void* v, const void* g,
                            const void* beta, int dtype, const double* init_state,
                            const long long* cu_seqlens, int n_seqs, int heads, int dk, int dv,
                            double* out, double* final_state, double* checkpoints,
                            const long long* ckpt_offsets, long long ckpt_interval,
                            int n_threads) {
  if (!q || !k || !v || !g || !beta || !cu_seqlens || !out) return -1;
  if (n_seqs < 0 || heads <= 0 || dk <= 0 || dv <= 0) return -1;
  if (dtype != ORC_F32 && dtype != ORC_BF16 && dtype != ORC_F64) return -1;
  for (int n = 0; n < n_seqs; ++n)
    if (cu_seqlens[n + 1] < cu_seqlens[n]) return -1;
  if (checkpoints && (!ckpt_offsets || ckpt_interval <= 0)) return -1;
  orc_job_t J = {q, k, v, g, beta, dtype, init_state, cu_seqlens, n_seqs, heads, dk, dv,
                 out, final_state, checkpoints, ckpt_offsets, ckpt_interval, 0};
  const int n_jobs = n_seqs * heads;
  if (n_threads <= 0) n_threads = kda_oracle_default_threads();
  if (n_threads > n_jobs) n_threads = n_jobs > 0 ? n_jobs : 1;
  if (n_threads == 1) return orc_worker(&J) ? -2 : 1;
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * n_threads);
  if (!th) return -2;
  int started = 0, failed = 0;
  for (; started < n_threads; ++started)
    if (pthread_create(&th[started], NULL, orc_worker, &J) != 0) break;
  if (started == 0) failed = orc_worker(&J) != NULL;
  for (int i = 0; i < started; ++i) {
    void* rc = NULL;
    pthread_join(th[i], &rc);
    failed |= rc != NULL;
  }
  free(th);
  return failed ? -2 : (started ? started : 1);
}

/* Prefill over packed sequences without checkpoints. */
int kda_oracle_prefill(const void* q, const void* k, const void* v, const void* g,
                       const void* beta, int dtype, const double* init_state,
                       const long long* cu_seqlens, int n_seqs, int heads, int dk, int dv,
                       double* out, double* final_state, int n_threads) {
  return kda_oracle_prefill_ckpt(q, k, v, g, beta, dtype, init_state, cu_seqlens, n_seqs, heads,
                                 dk, dv, out, final_state, NULL, NULL, 0, n_threads);
}

/*
 * One decode step: every sequence n advances by exactly one token (token n of
 * the [N, H, d] inputs).  `state` [N, H, dk, dv] is read and overwritten.
 */
int kda_oracle_decode(const void* q, const void* k, const void* v, const void* g,
                      const void* beta, int dtype, double* state, int n_seqs, int heads,
                      int dk, int dv, double* out, int n_threads) {
  if (!state || n_seqs < 0) return -1;
  long long* cu = (long long*)malloc(sizeof(long long) * ((size_t)n_seqs + 1));
  if (!cu) return -2;
  for (int n = 0; n <= n_seqs; ++n) cu[n] = n;
  /* Each pair copies its state in before it writes it back, so in == out is safe. */
  int rc = kda_oracle_prefill(q, k, v, g, beta, dtype, state, cu, n_seqs, heads, dk, dv, out,
                              state, n_threads);
  free(cu);
  return rc;
}

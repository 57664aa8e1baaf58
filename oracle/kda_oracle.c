/*
 * kda_oracle.c -- fp64 CPU oracle for the Kimi Delta Attention (KDA) forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or calls
 * this file: only the tests, __graft_entry__.smoke() and the benchmark's CPU
 * baseline leg use it.  It shares no code with the CUDA library.
 *
 * What it computes (plain definitions, token by token, in double precision):
 *
 *  kda_oracle_gate  -- the bounded log-decay
 *        g = g_min * Sigmoid(exp(A_h) * z),  alpha = exp(g)
 *      ("Kimi K3 technical report review" (devpress/CSDN), section 3.2, Eq. 5;
 *       "Kimi K3: architecture, training and inference systems" (weigao.cc),
 *       section 3.2).  A_h is one scalar per head, z and g are per key channel.
 *
 *  kda_oracle_recurrence -- the KDA state recurrence and read-out
 *        S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T
 *        o_t = S_t^T q_t
 *      ("Kimi K3 technical report review", section 3.1, Eq. 1;
 *       "Kimi K3: architecture, training and inference systems", section 3.1).
 *      The product form is applied as operators: first X = Diag(alpha) S,
 *      then (I - beta k k^T) X = X - beta k (k^T X), then + beta k v^T.
 *      With form = 1 the same step is taken in the delta (error-correction)
 *      form of the same section:
 *        S_t = D_t S_{t-1} + beta_t k_t (v_t^T - k_t^T D_t S_{t-1}).
 *
 * Layouts (row-major, fp64):
 *   q, k, g : [NT][H][dk]     v : [NT][H][dv]     beta : [NT][H]
 *   h0, hT  : [N][H][dv][dk]  (the state S in R^{dk x dv} stored transposed,
 *                              i.e. element (c, j) of S at [j][c])
 *   o       : [NT][H][dv]
 *   cu_seqlens : [N+1] int64, sequence n = tokens cu[n] .. cu[n+1]-1.
 * h0 may be NULL (zero initial state); hT may be NULL.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

void kda_oracle_gate(const double* z, const double* A, double g_min, int64_t n_tokens, int H,
                     int dk, double* g) {
  for (int64_t t = 0; t < n_tokens; ++t)
    for (int h = 0; h < H; ++h) {
      const double scale = exp(A[h]);
      for (int c = 0; c < dk; ++c) {
        const int64_t i = (t * H + h) * (int64_t)dk + c;
        const double x = scale * z[i];
        g[i] = g_min / (1.0 + exp(-x)); /* g_min * Sigmoid(x) */
      }
    }
}

typedef struct {
  const double *q, *k, *v, *g, *beta, *h0;
  const int64_t* cu;
  int n_seqs, H, dk, dv, form;
  double *o, *hT;
  int64_t next_unit; /* shared work counter, guarded by mu */
  pthread_mutex_t mu;
} rec_job;

/* One (sequence, head) unit: the recurrence over that sequence's tokens. */
static void rec_unit(const rec_job* J, int n, int h, double* S, double* X, double* kX) {
  const int H = J->H, dk = J->dk, dv = J->dv;
  /* S is the math state, S[c*dv + j] = S_{c,j}, c < dk, j < dv. */
  for (int c = 0; c < dk; ++c)
    for (int j = 0; j < dv; ++j)
      S[c * dv + j] = J->h0 ? J->h0[(((int64_t)n * H + h) * dv + j) * dk + c] : 0.0;

  for (int64_t t = J->cu[n]; t < J->cu[n + 1]; ++t) {
    const double* qt = J->q + (t * H + h) * (int64_t)dk;
    const double* kt = J->k + (t * H + h) * (int64_t)dk;
    const double* gt = J->g + (t * H + h) * (int64_t)dk;
    const double* vt = J->v + (t * H + h) * (int64_t)dv;
    const double bt = J->beta[t * H + h];
    /* X = Diag(alpha_t) S_{t-1} : row c of S scaled by alpha_{t,c} = exp(g_{t,c}) */
    for (int c = 0; c < dk; ++c) {
      const double alpha = exp(gt[c]);
      for (int j = 0; j < dv; ++j) X[c * dv + j] = alpha * S[c * dv + j];
    }
    /* kX = k_t^T X  (a row vector of length dv) */
    for (int j = 0; j < dv; ++j) kX[j] = 0.0;
    for (int c = 0; c < dk; ++c)
      for (int j = 0; j < dv; ++j) kX[j] += kt[c] * X[c * dv + j];
    if (J->form == 0) {
      /* product form: S_t = X - beta k (k^T X) + beta k v^T */
      for (int c = 0; c < dk; ++c)
        for (int j = 0; j < dv; ++j)
          S[c * dv + j] = X[c * dv + j] - bt * kt[c] * kX[j] + bt * kt[c] * vt[j];
    } else {
      /* delta form: S_t = X + beta k (v^T - k^T X) */
      for (int c = 0; c < dk; ++c)
        for (int j = 0; j < dv; ++j)
          S[c * dv + j] = X[c * dv + j] + bt * kt[c] * (vt[j] - kX[j]);
    }
    /* o_t = S_t^T q_t */
    double* ot = J->o + (t * H + h) * (int64_t)dv;
    for (int j = 0; j < dv; ++j) {
      double acc = 0.0;
      for (int c = 0; c < dk; ++c) acc += S[c * dv + j] * qt[c];
      ot[j] = acc;
    }
  }
  if (J->hT)
    for (int c = 0; c < dk; ++c)
      for (int j = 0; j < dv; ++j)
        J->hT[(((int64_t)n * H + h) * dv + j) * dk + c] = S[c * dv + j];
}

static void* rec_worker(void* arg) {
  rec_job* J = (rec_job*)arg;
  double* S = (double*)malloc(sizeof(double) * (size_t)J->dk * J->dv);
  double* X = (double*)malloc(sizeof(double) * (size_t)J->dk * J->dv);
  double* kX = (double*)malloc(sizeof(double) * (size_t)J->dv);
  const int64_t n_units = (int64_t)J->n_seqs * J->H;
  for (;;) {
    pthread_mutex_lock(&J->mu);
    const int64_t u = J->next_unit++;
    pthread_mutex_unlock(&J->mu);
    if (u >= n_units) break;
    rec_unit(J, (int)(u / J->H), (int)(u % J->H), S, X, kX);
  }
  free(S);
  free(X);
  free(kX);
  return NULL;
}

/* Returns 0 on success, -1 on bad arguments or allocation failure. */
int kda_oracle_recurrence(const double* q, const double* k, const double* v, const double* g,
                          const double* beta, const double* h0, const int64_t* cu_seqlens,
                          int n_seqs, int H, int dk, int dv, int form, double* o, double* hT,
                          int n_threads) {
  if (!q || !k || !v || !g || !beta || !cu_seqlens || !o || n_seqs < 0 || H <= 0 || dk <= 0 ||
      dv <= 0)
    return -1;
  for (int n = 0; n < n_seqs; ++n)
    if (cu_seqlens[n + 1] < cu_seqlens[n]) return -1;
  rec_job J;
  J.q = q; J.k = k; J.v = v; J.g = g; J.beta = beta; J.h0 = h0; J.cu = cu_seqlens;
  J.n_seqs = n_seqs; J.H = H; J.dk = dk; J.dv = dv; J.form = form; J.o = o; J.hT = hT;
  J.next_unit = 0;
  pthread_mutex_init(&J.mu, NULL);
  if (n_threads < 1) n_threads = 1;
  if (n_threads > 256) n_threads = 256;
  pthread_t th[256];
  int started = 0;
  for (int i = 1; i < n_threads; ++i)
    if (pthread_create(&th[started], NULL, rec_worker, &J) == 0) ++started;
  rec_worker(&J);
  for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
  pthread_mutex_destroy(&J.mu);
  return 0;
}

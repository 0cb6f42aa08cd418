/*
 * oracle.c -- plain, slow, token-by-token fp64 CPU oracle for the gated
 * linear attention recurrence (GLA and Mamba-2 SSD), forward and backward.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline leg of bench.py may load this library.  It shares no code,
 * header, table or helper with the CUDA path (package csrc/), and the CUDA
 * path never calls it.
 *
 * What it computes (the plain definition, one token at a time, in double):
 *
 *   S_t = diag(exp(g_t)) S_{t-1} + k_t v_t^T          (S is K x V)
 *   o_t = scale * S_t^T q_t
 *
 * Sources:
 *  - "FLAT" blog (trainstation-project.github.io/blog/flat), section
 *    "Linear Attention / Forward Recurrence": the recurrent form, the
 *    architecture table (GLA = diagonal per-key-channel forget gate,
 *    Mamba-2 = one scalar gate per head), and the note that the output at
 *    position t reads the state that already contains token t (the causal
 *    mask M_C includes the diagonal).
 *  - same page, "Backward Recurrence": the state gradient runs backwards in
 *    time with q_t and dL/dy_t in the roles of k_t and v_t, the gate also
 *    scales the state gradient at every step, and the forget-gate gradient
 *    is (dL/dH_t (.) H_{t-1}) 1_V; for the log gate g = log f this becomes
 *    dL/dg_t = f_t * dL/df_t.
 *  - "JLA" product page (karlex.ai/jla): segment_ids make a packed batch
 *    train exactly as its documents would one by one; optional initial and
 *    final states.
 *
 * Readings taken where the pages are silent (all listed in the design
 * notes of the repository):
 *  - the first token's gate also decays the initial state:
 *    S_{t0} = diag(exp(g_{t0})) h0 + k v^T;
 *  - a document starts at t = 0 of every batch row and wherever
 *    segment_ids[b,t] != segment_ids[b,t-1]; documents are numbered in
 *    row-major order of their first token and index h0 / final states;
 *  - Mamba-2 (gate_kind = 1): g is [B,T,H], the same decay for every key
 *    channel; dg sums the per-channel gate gradient over K; q and k may be
 *    shared by H/Hqk heads and their gradients are summed over the heads of
 *    the group.
 *
 * Backward: hand-derived reverse-time recurrence.  The states S_t are
 * needed in reverse order; the oracle keeps a checkpoint every CKPT tokens
 * and recomputes each block forward into a buffer (storing every state of a
 * long sequence is what makes per-step references run out of memory).
 *
 * Layouts (row-major, contiguous):
 *   q, k  [B,T,Hqk,K]   v, o  [B,T,H,V]   g  [B,T,H,K] (gate_kind 0) or
 *   [B,T,H] (gate_kind 1)   segment_ids [B,T] int32 or NULL
 *   h0, ht, dht, dh0 [n_docs,H,K,V]   do [B,T,H,V]   dq, dk [B,T,Hqk,K]
 *   dv [B,T,H,V]   dg like g.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define CKPT 256

typedef struct {
  int64_t B, T, H, Hqk, K, V;
  int gate_kind;
  double scale;
  const double *q, *k, *v, *g, *h0, *dO, *dht;
  double *o, *ht, *dq, *dk, *dv, *dg, *dh0;
  /* document table */
  int64_t n_docs;
  const int64_t *doc_row, *doc_t0, *doc_t1;
  /* work distribution */
  int64_t n_units; /* n_docs * Hqk */
  int64_t next_unit;
  pthread_mutex_t lock;
  int backward;
} job_t;

/* ---- document table --------------------------------------------------- */

/* Number of documents: one starts at t = 0 of every row and wherever the id
 * changes from the previous token of the same row. */
int64_t oracle_count_docs(int64_t B, int64_t T, const int32_t *seg) {
  if (T <= 0 || B <= 0) return 0;
  if (!seg) return B;
  int64_t n = 0;
  for (int64_t b = 0; b < B; ++b)
    for (int64_t t = 0; t < T; ++t)
      if (t == 0 || seg[b * T + t] != seg[b * T + t - 1]) ++n;
  return n;
}

static void build_docs(int64_t B, int64_t T, const int32_t *seg, int64_t n,
                       int64_t *row, int64_t *t0, int64_t *t1) {
  int64_t d = 0;
  for (int64_t b = 0; b < B; ++b) {
    for (int64_t t = 0; t < T; ++t) {
      int start = (t == 0) || (seg && seg[b * T + t] != seg[b * T + t - 1]);
      if (start) {
        if (d > 0 && row[d - 1] == b) t1[d - 1] = t;
        row[d] = b;
        t0[d] = t;
        t1[d] = T;
        ++d;
      }
    }
  }
  (void)n;
}

/* ---- index helpers ---------------------------------------------------- */

static inline const double *QK(const job_t *j, const double *base, int64_t b,
                               int64_t t, int64_t hk) {
  return base + ((b * j->T + t) * j->Hqk + hk) * j->K;
}
static inline int64_t VOFF(const job_t *j, int64_t b, int64_t t, int64_t h) {
  return ((b * j->T + t) * j->H + h) * j->V;
}
/* exp of the gate of key channel c at (b,t,h) */
static inline double gate_log(const job_t *j, int64_t b, int64_t t, int64_t h,
                              int64_t c) {
  if (j->gate_kind == 0) return j->g[((b * j->T + t) * j->H + h) * j->K + c];
  return j->g[(b * j->T + t) * j->H + h];
}

/* One step of the recurrence: S <- diag(exp(g_t)) S + k_t v_t^T. */
static void step(const job_t *j, double *S, int64_t b, int64_t t, int64_t h,
                 int64_t hk) {
  const int64_t K = j->K, V = j->V;
  const double *kt = QK(j, j->k, b, t, hk);
  const double *vt = j->v + VOFF(j, b, t, h);
  for (int64_t c = 0; c < K; ++c) {
    double f = exp(gate_log(j, b, t, h, c));
    double *row = S + c * V;
    for (int64_t e = 0; e < V; ++e) row[e] = f * row[e] + kt[c] * vt[e];
  }
}

/* ---- forward ---------------------------------------------------------- */

static void fwd_unit(job_t *j, int64_t d, int64_t h, int64_t hk, double *S) {
  const int64_t K = j->K, V = j->V;
  const int64_t b = j->doc_row[d];
  if (j->h0)
    memcpy(S, j->h0 + (d * j->H + h) * K * V, sizeof(double) * K * V);
  else
    memset(S, 0, sizeof(double) * K * V);
  for (int64_t t = j->doc_t0[d]; t < j->doc_t1[d]; ++t) {
    step(j, S, b, t, h, hk);
    const double *qt = QK(j, j->q, b, t, hk);
    double *ot = j->o + VOFF(j, b, t, h);
    for (int64_t e = 0; e < V; ++e) ot[e] = 0.0;
    for (int64_t c = 0; c < K; ++c) {
      const double *row = S + c * V;
      for (int64_t e = 0; e < V; ++e) ot[e] += qt[c] * row[e];
    }
    for (int64_t e = 0; e < V; ++e) ot[e] *= j->scale;
  }
  if (j->ht) memcpy(j->ht + (d * j->H + h) * K * V, S, sizeof(double) * K * V);
}

/* ---- backward --------------------------------------------------------- */

/* Reverse-time recurrence for one (document, head).  dq/dk are accumulated
 * (+=) because heads of one q/k group share them; the caller zeroes them. */
static void bwd_unit(job_t *j, int64_t d, int64_t h, int64_t hk, double *ckpt,
                     double *blk, double *dH, double *Sprev) {
  const int64_t K = j->K, V = j->V, KV = K * V;
  const int64_t b = j->doc_row[d], t0 = j->doc_t0[d], t1 = j->doc_t1[d];
  const int64_t L = t1 - t0;
  const int64_t nb = (L + CKPT - 1) / CKPT;
  /* forward sweep: checkpoint the state entering every block */
  double *S = Sprev; /* scratch */
  if (j->h0)
    memcpy(S, j->h0 + (d * j->H + h) * KV, sizeof(double) * KV);
  else
    memset(S, 0, sizeof(double) * KV);
  for (int64_t i = 0; i < nb; ++i) {
    memcpy(ckpt + i * KV, S, sizeof(double) * KV);
    int64_t te = t0 + (i + 1) * CKPT < t1 ? t0 + (i + 1) * CKPT : t1;
    for (int64_t t = t0 + i * CKPT; t < te; ++t) step(j, S, b, t, h, hk);
  }
  if (j->dht)
    memcpy(dH, j->dht + (d * j->H + h) * KV, sizeof(double) * KV);
  else
    memset(dH, 0, sizeof(double) * KV);
  for (int64_t i = nb - 1; i >= 0; --i) {
    const int64_t ts = t0 + i * CKPT;
    const int64_t te = ts + CKPT < t1 ? ts + CKPT : t1;
    /* recompute the block: blk[r] = state after token ts + r */
    memcpy(S, ckpt + i * KV, sizeof(double) * KV);
    for (int64_t t = ts; t < te; ++t) {
      step(j, S, b, t, h, hk);
      memcpy(blk + (t - ts) * KV, S, sizeof(double) * KV);
    }
    for (int64_t t = te - 1; t >= ts; --t) {
      const double *St = blk + (t - ts) * KV;
      const double *Sm = (t > ts) ? blk + (t - ts - 1) * KV : ckpt + i * KV;
      const double *qt = QK(j, j->q, b, t, hk);
      const double *kt = QK(j, j->k, b, t, hk);
      const double *vt = j->v + VOFF(j, b, t, h);
      const double *dot = j->dO + VOFF(j, b, t, h);
      double *dqt = j->dq + ((b * j->T + t) * j->Hqk + hk) * K;
      double *dkt = j->dk + ((b * j->T + t) * j->Hqk + hk) * K;
      double *dvt = j->dv + VOFF(j, b, t, h);
      /* dL/dS_t gets the readout of token t */
      for (int64_t c = 0; c < K; ++c)
        for (int64_t e = 0; e < V; ++e)
          dH[c * V + e] += j->scale * qt[c] * dot[e];
      for (int64_t e = 0; e < V; ++e) dvt[e] = 0.0;
      double dg_head = 0.0;
      for (int64_t c = 0; c < K; ++c) {
        double aq = 0.0, ak = 0.0, ag = 0.0;
        for (int64_t e = 0; e < V; ++e) {
          aq += St[c * V + e] * dot[e];
          ak += dH[c * V + e] * vt[e];
          ag += Sm[c * V + e] * dH[c * V + e];
          dvt[e] += dH[c * V + e] * kt[c];
        }
        dqt[c] += j->scale * aq;
        dkt[c] += ak;
        double f = exp(gate_log(j, b, t, h, c));
        /* dL/dg_tc = exp(g_tc) * sum_v S_{t-1}[c,v] dH_t[c,v] */
        if (j->gate_kind == 0)
          j->dg[((b * j->T + t) * j->H + h) * K + c] = f * ag;
        else
          dg_head += f * ag;
        /* dL/dS_{t-1} = diag(exp(g_t)) dL/dS_t */
        for (int64_t e = 0; e < V; ++e) dH[c * V + e] *= f;
      }
      if (j->gate_kind == 1) j->dg[(b * j->T + t) * j->H + h] = dg_head;
    }
  }
  if (j->dh0) memcpy(j->dh0 + (d * j->H + h) * KV, dH, sizeof(double) * KV);
}

static void *worker(void *arg) {
  job_t *j = (job_t *)arg;
  const int64_t KV = j->K * j->V;
  double *S = (double *)malloc(sizeof(double) * KV);
  double *dH = NULL, *ckpt = NULL, *blk = NULL;
  int64_t maxlen = 0;
  if (j->backward) {
    for (int64_t d = 0; d < j->n_docs; ++d)
      if (j->doc_t1[d] - j->doc_t0[d] > maxlen) maxlen = j->doc_t1[d] - j->doc_t0[d];
    dH = (double *)malloc(sizeof(double) * KV);
    ckpt = (double *)malloc(sizeof(double) * KV * ((maxlen + CKPT - 1) / CKPT + 1));
    blk = (double *)malloc(sizeof(double) * KV * CKPT);
  }
  const int64_t G = j->H / j->Hqk;
  for (;;) {
    pthread_mutex_lock(&j->lock);
    int64_t u = j->next_unit++;
    pthread_mutex_unlock(&j->lock);
    if (u >= j->n_units) break;
    const int64_t d = u / j->Hqk, hk = u % j->Hqk;
    for (int64_t h = hk * G; h < (hk + 1) * G; ++h) {
      if (j->backward)
        bwd_unit(j, d, h, hk, ckpt, blk, dH, S);
      else
        fwd_unit(j, d, h, hk, S);
    }
  }
  free(S);
  free(dH);
  free(ckpt);
  free(blk);
  return NULL;
}

static int run(job_t *j, int64_t B, int64_t T, const int32_t *seg,
               int64_t n_seqs, int nthreads) {
  if (B < 0 || T < 0 || j->H <= 0 || j->Hqk <= 0 || j->K <= 0 || j->V <= 0) return -1;
  if (j->H % j->Hqk) return -1;
  if (j->gate_kind != 0 && j->gate_kind != 1) return -1;
  int64_t n = oracle_count_docs(B, T, seg);
  if (n_seqs >= 0 && n != n_seqs) return -2;
  int64_t *row = (int64_t *)malloc(sizeof(int64_t) * (n + 1));
  int64_t *t0 = (int64_t *)malloc(sizeof(int64_t) * (n + 1));
  int64_t *t1 = (int64_t *)malloc(sizeof(int64_t) * (n + 1));
  build_docs(B, T, seg, n, row, t0, t1);
  j->B = B;
  j->T = T;
  j->n_docs = n;
  j->doc_row = row;
  j->doc_t0 = t0;
  j->doc_t1 = t1;
  j->n_units = n * j->Hqk;
  j->next_unit = 0;
  pthread_mutex_init(&j->lock, NULL);
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  pthread_t th[256];
  for (int i = 0; i < nthreads; ++i) pthread_create(&th[i], NULL, worker, j);
  for (int i = 0; i < nthreads; ++i) pthread_join(th[i], NULL);
  pthread_mutex_destroy(&j->lock);
  free(row);
  free(t0);
  free(t1);
  return 0;
}

/* Forward.  Returns 0, -1 on bad sizes, -2 if n_seqs (when >= 0) differs
 * from the number of documents in segment_ids. */
int oracle_fwd(int64_t B, int64_t T, int64_t H, int64_t Hqk, int64_t K,
               int64_t V, int gate_kind, double scale, const double *q,
               const double *k, const double *v, const double *g,
               const int32_t *segment_ids, int64_t n_seqs, const double *h0,
               double *o, double *ht, int nthreads) {
  job_t j;
  memset(&j, 0, sizeof(j));
  j.H = H; j.Hqk = Hqk; j.K = K; j.V = V; j.gate_kind = gate_kind;
  j.scale = scale; j.q = q; j.k = k; j.v = v; j.g = g; j.h0 = h0;
  j.o = o; j.ht = ht; j.backward = 0;
  return run(&j, B, T, segment_ids, n_seqs, nthreads);
}

/* Backward.  dq, dk, dv, dg are fully written; dh0 (if non-NULL) too. */
int oracle_bwd(int64_t B, int64_t T, int64_t H, int64_t Hqk, int64_t K,
               int64_t V, int gate_kind, double scale, const double *q,
               const double *k, const double *v, const double *g,
               const int32_t *segment_ids, int64_t n_seqs, const double *h0,
               const double *dO, const double *dht, double *dq, double *dk,
               double *dv, double *dg, double *dh0, int nthreads) {
  job_t j;
  memset(&j, 0, sizeof(j));
  j.H = H; j.Hqk = Hqk; j.K = K; j.V = V; j.gate_kind = gate_kind;
  j.scale = scale; j.q = q; j.k = k; j.v = v; j.g = g; j.h0 = h0;
  j.dO = dO; j.dht = dht; j.dq = dq; j.dk = dk; j.dv = dv; j.dg = dg;
  j.dh0 = dh0; j.backward = 1;
  memset(dq, 0, sizeof(double) * B * T * Hqk * K);
  memset(dk, 0, sizeof(double) * B * T * Hqk * K);
  return run(&j, B, T, segment_ids, n_seqs, nthreads);
}

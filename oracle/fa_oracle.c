/*
 * fa_oracle.c -- plain fp64 CPU reference for the no-cache multi-head attention
 * forward (the `mo.mha.no_cache` operator). TEST INFRASTRUCTURE ONLY: it is
 * called by the tests, by the smoke check and by the benchmark's CPU-baseline
 * leg, never by the product path. It shares no code with the CUDA library.
 *
 * What it computes, step by step as the MAX API page "FlashAttentionGPU"
 * (method `execute`, Steps -1 to 4) describes the operator, for every batch b,
 * query head h and query position i:
 *
 *   Step -1 (grouped attention): K and V may carry Hkv < H heads (BShD). The
 *            page says only "G groups, h = H/G"; query head h reads KV head
 *            h / G (consecutive query heads share one KV head, G = H / Hkv).
 *            The alternative reading (KV head h % Hkv, a literal head-axis
 *            concatenation) is selectable with head_map = 1.
 *   Step 0  : the BSHD -> BHSD / BHDS transposes are index arithmetic here.
 *   Step 1-3: s_j = scale * sum_d q[b,i,h,d] * k[b,j,hk,d]; keys the mask
 *            hides get s_j = -inf (they are simply skipped below).
 *   Step 4  : p_j = exp(s_j - m) / sum_j' exp(s_j' - m), m = max_j s_j;
 *            out[b,i,h,:] = sum_j p_j v[b,j,hk,:]. This is the classic
 *            attention of the Modular recipe "Custom Operations: Applications
 *            in AI Models" (section "Limitations of classic attention"): bmm,
 *            softmax, bmm, computed here one query row at a time.
 *   LSE     : lse[b,h,i] = m + ln(sum_j exp(s_j - m)) (natural log, scale
 *            included). The pages define no LSE output; this is its plain
 *            definition.
 *
 * Mask (the page's `mask_str` / `local_window_size` parameters): key j is
 * visible to query i iff (not causal or j <= i) and (window < 1 or
 * i - j < window) and (causal or window < 1 or j - i < window): a causal
 * window holds the W keys ending at the query, a window without the causal
 * mask the keys within distance W - 1 on either side. window = -1 (or 0)
 * means no window.
 *
 * KV-cache form (fa_oracle_forward_kvcache): the same operator when the keys
 * and values of batch b are the first L_b rows of a cache of capacity S and
 * the Sq queries are the last Sq tokens of that sequence, so query row r sits
 * at position L_b - Sq + r. The pages name only the no-cache operator; this
 * is the plainest reading of its cached sibling: every step above is
 * unchanged, the mask is evaluated at the query's position, and keys at
 * positions >= L_b do not exist (they are never read). A query that sees no
 * key at all (possible only here, e.g. a causal row whose position is
 * negative because L_b < Sq) gets out = 0 and lse = -inf.
 *
 * Everything is fp64. Inputs are fp64 arrays (bf16 / fp32 values widen to
 * fp64 exactly). The score row of one query is materialised (length S); the
 * S x S matrix is not, which changes nothing in the arithmetic.
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

#define FA_ORACLE_OK 0
#define FA_ORACLE_BAD_ARG 1
#define FA_ORACLE_NO_MEM 2

typedef struct {
  const double *q, *k, *v;
  double *out, *lse;
  long B, S, H, Hkv, D;
  double scale;
  int causal;
  long window;
  int head_map;
  const long *rows;
  long nrows;
  const long *lens; /* KV-cache form: keys per batch (NULL: S keys) */
  int from_end;     /* KV-cache form: row r sits at position lens[b] - nrows + r */
  long first, last; /* this worker's half-open range of (b, h, r) items */
  int status;
} fa_oracle_job;

static int key_visible(long i, long j, int causal, long window) {
  if (causal && j > i) return 0;
  if (window > 0 && i - j >= window) return 0;
  if (!causal && window > 0 && j - i >= window) return 0;
  return 1;
}

static void *fa_oracle_worker(void *arg) {
  fa_oracle_job *job = (fa_oracle_job *)arg;
  const long S = job->S, H = job->H, Hkv = job->Hkv, D = job->D;
  const long G = H / Hkv;
  double *score = (double *)malloc(sizeof(double) * (size_t)S);
  char *seen = (char *)malloc((size_t)S);
  double *acc = (double *)malloc(sizeof(double) * (size_t)D);
  if (!score || !seen || !acc) {
    job->status = FA_ORACLE_NO_MEM;
    free(score);
    free(seen);
    free(acc);
    return NULL;
  }
  for (long item = job->first; item < job->last; ++item) {
    /* item enumerates (b, h, r) with r fastest. */
    const long r = item % job->nrows;
    const long h = (item / job->nrows) % H;
    const long b = item / (job->nrows * H);
    const long L = job->lens ? job->lens[b] : S; /* keys 0 .. L-1 exist */
    const long i = job->from_end ? L - job->nrows + r : (job->rows ? job->rows[r] : r);
    const long hk = job->head_map == 0 ? h / G : h % Hkv;

    const double *qrow = job->q + ((b * job->nrows + r) * H + h) * D;

    /* Steps 1-3: scaled scores of the visible keys, and their maximum. */
    double m = -INFINITY;
    for (long j = 0; j < L; ++j) {
      seen[j] = (char)key_visible(i, j, job->causal, job->window);
      if (!seen[j]) continue;
      const double *krow = job->k + ((b * S + j) * Hkv + hk) * D;
      double dot = 0.0;
      for (long d = 0; d < D; ++d) dot += qrow[d] * krow[d];
      score[j] = job->scale * dot;
      if (score[j] > m) m = score[j];
    }

    /* Step 4: max-subtracted softmax, then the weighted sum of V rows. */
    double denom = 0.0;
    for (long d = 0; d < D; ++d) acc[d] = 0.0;
    for (long j = 0; j < L; ++j) {
      if (!seen[j]) continue;
      const double e = exp(score[j] - m);
      denom += e;
      const double *vrow = job->v + ((b * S + j) * Hkv + hk) * D;
      for (long d = 0; d < D; ++d) acc[d] += e * vrow[d];
    }
    double *orow = job->out + ((b * job->nrows + r) * H + h) * D;
    if (denom > 0.0) {
      for (long d = 0; d < D; ++d) orow[d] = acc[d] / denom;
      if (job->lse) job->lse[(b * H + h) * job->nrows + r] = m + log(denom);
    } else { /* no visible key (KV-cache form only) */
      for (long d = 0; d < D; ++d) orow[d] = 0.0;
      if (job->lse) job->lse[(b * H + h) * job->nrows + r] = -INFINITY;
    }
  }
  free(score);
  free(seen);
  free(acc);
  return NULL;
}

/* Runs the B * H * nrows row jobs on nthreads threads. */
static int fa_oracle_run(const fa_oracle_job *tmpl, int nthreads) {
  const long items = tmpl->B * tmpl->H * tmpl->nrows;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > items) nthreads = (int)items;
  fa_oracle_job *jobs = (fa_oracle_job *)calloc((size_t)nthreads, sizeof(fa_oracle_job));
  pthread_t *tids = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
  char *started = (char *)calloc((size_t)nthreads, 1);
  if (!jobs || !tids || !started) {
    free(jobs);
    free(tids);
    free(started);
    return FA_ORACLE_NO_MEM;
  }
  for (int t = 0; t < nthreads; ++t) {
    jobs[t] = *tmpl;
    jobs[t].first = items * t / nthreads;
    jobs[t].last = items * (t + 1) / nthreads;
    jobs[t].status = FA_ORACLE_OK;
  }
  for (int t = 1; t < nthreads; ++t)
    started[t] = pthread_create(&tids[t], NULL, fa_oracle_worker, &jobs[t]) == 0;
  fa_oracle_worker(&jobs[0]);
  int status = jobs[0].status;
  for (int t = 1; t < nthreads; ++t) {
    if (started[t]) {
      pthread_join(tids[t], NULL);
    } else {
      fa_oracle_worker(&jobs[t]); /* thread creation failed: run inline */
    }
    if (jobs[t].status != FA_ORACLE_OK) status = jobs[t].status;
  }
  free(jobs);
  free(tids);
  free(started);
  return status;
}

/*
 * fa_oracle_forward
 *   q    : [B, nrows, H, D] fp64 -- the query rows to evaluate. With rows ==
 *          NULL, nrows must equal S and q is the whole BSHD query tensor.
 *   k, v : [B, S, Hkv, D] fp64 (BSHD, or BShD when Hkv < H).
 *   out  : [B, nrows, H, D] fp64, written.
 *   lse  : [B, H, nrows] fp64 or NULL.
 *   rows : NULL, or nrows query positions in [0, S) (the positions of q's rows).
 *   causal, window: the mask (window <= 0 means no window).
 *   head_map: 0 = grouped (h / G), 1 = tiled (h % Hkv).
 *   nthreads: worker threads (>= 1).
 * Returns 0 on success, 1 on a bad argument, 2 when memory runs out.
 */
int fa_oracle_forward(const double *q, const double *k, const double *v, double *out,
                      double *lse, long B, long S, long H, long Hkv, long D, double scale,
                      int causal, long window, int head_map, const long *rows, long nrows,
                      int nthreads) {
  if (!q || !k || !v || !out) return FA_ORACLE_BAD_ARG;
  if (B < 1 || S < 1 || H < 1 || Hkv < 1 || D < 1 || H % Hkv != 0) return FA_ORACLE_BAD_ARG;
  if (head_map != 0 && head_map != 1) return FA_ORACLE_BAD_ARG;
  if (!rows) nrows = S;
  if (nrows < 1) return FA_ORACLE_BAD_ARG;
  if (rows)
    for (long r = 0; r < nrows; ++r)
      if (rows[r] < 0 || rows[r] >= S) return FA_ORACLE_BAD_ARG;

  fa_oracle_job job;
  memset(&job, 0, sizeof(job));
  job.q = q;
  job.k = k;
  job.v = v;
  job.out = out;
  job.lse = lse;
  job.B = B;
  job.S = S;
  job.H = H;
  job.Hkv = Hkv;
  job.D = D;
  job.scale = scale;
  job.causal = causal;
  job.window = window;
  job.head_map = head_map;
  job.rows = rows;
  job.nrows = nrows;
  return fa_oracle_run(&job, nthreads);
}

/*
 * fa_oracle_forward_kvcache -- the KV-cache form (see the header).
 *   q     : [B, Sq, H, D] fp64, the last Sq tokens of each sequence.
 *   k, v  : [B, S, Hkv, D] fp64 caches of capacity S; rows >= lens[b] are
 *           never read.
 *   lens  : B key counts in [0, S], or NULL for S keys in every batch.
 *   out   : [B, Sq, H, D] fp64, written; lse: [B, H, Sq] fp64 or NULL.
 *   Other arguments as fa_oracle_forward (grouped head map).
 * Returns 0 on success, 1 on a bad argument, 2 when memory runs out.
 */
int fa_oracle_forward_kvcache(const double *q, const double *k, const double *v, double *out,
                              double *lse, long B, long Sq, long S, const long *lens, long H,
                              long Hkv, long D, double scale, int causal, long window,
                              int nthreads) {
  if (!q || !k || !v || !out) return FA_ORACLE_BAD_ARG;
  if (B < 1 || Sq < 1 || S < 1 || H < 1 || Hkv < 1 || D < 1 || H % Hkv != 0)
    return FA_ORACLE_BAD_ARG;
  if (lens)
    for (long b = 0; b < B; ++b)
      if (lens[b] < 0 || lens[b] > S) return FA_ORACLE_BAD_ARG;

  fa_oracle_job job;
  memset(&job, 0, sizeof(job));
  job.q = q;
  job.k = k;
  job.v = v;
  job.out = out;
  job.lse = lse;
  job.B = B;
  job.S = S;
  job.H = H;
  job.Hkv = Hkv;
  job.D = D;
  job.scale = scale;
  job.causal = causal;
  job.window = window;
  job.head_map = 0;
  job.nrows = Sq;
  job.lens = lens;
  job.from_end = 1;
  return fa_oracle_run(&job, nthreads);
}

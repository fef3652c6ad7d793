/*
 * Dense-attention oracle in fp64 -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg may
 * load this file.  The CUDA library never calls it, and it shares no code,
 * header, table or helper with the CUDA library.
 *
 * What it computes is the plain definition of attention, not the blockwise
 * ring algorithm.  The definition comes from "RingAttention: Scaling LLM
 * Context to 10M Tokens", section "1. Incremental Online Softmax
 * Accumulation", first display: O = softmax(Q K^T / sqrt(d)) V.  The
 * max-shift used here comes from "Ring Attention Math Deep", section "The
 * online-softmax identity that makes streaming legal": the ratio does not
 * change when any constant m is subtracted from every score, and m = max is
 * the safe choice.
 *
 * For every requested query row r and query head h it returns the partial
 * state of that row against the whole key set handed in:
 *   m = max_t s_rt                 over the allowed keys t
 *   l = sum_t exp(s_rt - m)
 *   o = sum_t exp(s_rt - m) v_t    (a vector of length d)
 * where s_rt = (q_r . k_t) * scale.  Key t is allowed for row r unless
 *   - `causal` is set and k_pos[t] > q_pos[r], or
 *   - `window` > 0 and |q_pos[r] - k_pos[t]| >= window, or
 *   - document ids are given and q_doc[r] < 0 or k_doc[t] != q_doc[r].
 * Causal masking on global token positions follows "Ring Attention：把超长
 * 序列沿设备环流动", section "位置编码必须使用全局位置" (positions are
 * global, device p local index i maps to p * N_local + i).  The window, the
 * packed documents that must not see each other, and the padding rows of
 * the last rank (document id -1: they see nothing and nobody sees them)
 * are the cases the same page lists under "正确性测试应覆盖哪些边界".  A
 * row with no allowed key returns m = -inf, l = 0, o = 0.
 *
 * Query head h reads KV head h / (hq / hkv).  The pages only name GQA, so
 * this maps consecutive groups of query heads to one KV head.
 *
 * The work per row takes two passes.  The first pass computes and stores
 * every allowed score and finds the max.  The second pass sums the
 * exponentials and the weighted values.  Everything runs in fp64.  The
 * inputs are either fp32 or bf16 (raw 16-bit patterns).  A bf16 value is
 * widened exactly: its bits become the high half of an IEEE binary32.
 *
 * Layout is token-major: q is [nq, hq, d], and k and v are [nk, hkv, d].
 * Outputs are indexed by position in `rows`: m and l are [nrows, hq], and
 * o is [nrows, hq, d].
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_F32 0
#define ORACLE_BF16 1

typedef struct {
  const void* q;
  const void* k;
  const void* v;
  int dtype;
  long long nq, nk;
  int hq, hkv, d;
  double scale;
  int causal;
  long long window;
  const long long* q_doc;
  const long long* k_doc;
  const long long* q_pos;
  const long long* k_pos;
  const long long* rows;
  long long nrows;
  double* m_out;
  double* l_out;
  double* o_out;
  long long next; /* next (row, head) work item, taken atomically */
  int failed;
} job_t;

static double widen(const void* base, int dtype, size_t idx) {
  if (dtype == ORACLE_F32) return (double)((const float*)base)[idx];
  uint32_t bits = ((uint32_t)((const uint16_t*)base)[idx]) << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

static void one_row(job_t* J, long long item, double* score, char* allowed, double* qrow,
                    double* acc) {
  const long long ri = item / J->hq;
  const int h = (int)(item % J->hq);
  const int d = J->d;
  const int group = J->hq / J->hkv;
  const int kh = h / group;
  const long long r = J->rows[ri];
  const long long qp = J->q_pos ? J->q_pos[r] : r;
  const long long qd = J->q_doc ? J->q_doc[r] : 0;

  for (int x = 0; x < d; ++x) qrow[x] = widen(J->q, J->dtype, ((size_t)r * J->hq + h) * d + x);

  /* pass 1: scores of the allowed keys, and their max */
  double m = -INFINITY;
  long long n_allowed = 0;
  for (long long t = 0; t < J->nk; ++t) {
    const long long kp = J->k_pos ? J->k_pos[t] : t;
    int ok = !(J->causal && kp > qp);
    if (J->window > 0 && (qp - kp >= J->window || kp - qp >= J->window)) ok = 0;
    if (J->q_doc && (qd < 0 || J->k_doc[t] != qd)) ok = 0;
    allowed[t] = (char)ok;
    if (!ok) continue;
    const size_t kb = ((size_t)t * J->hkv + kh) * d;
    double s = 0.0;
    for (int x = 0; x < d; ++x) s += qrow[x] * widen(J->k, J->dtype, kb + x);
    s *= J->scale;
    score[t] = s;
    if (s > m) m = s;
    ++n_allowed;
  }

  /* pass 2: l = sum exp(s - m), o = sum exp(s - m) v */
  double l = 0.0;
  for (int x = 0; x < d; ++x) acc[x] = 0.0;
  if (n_allowed > 0) {
    for (long long t = 0; t < J->nk; ++t) {
      if (!allowed[t]) continue;
      const double e = exp(score[t] - m);
      l += e;
      const size_t vb = ((size_t)t * J->hkv + kh) * d;
      for (int x = 0; x < d; ++x) acc[x] += e * widen(J->v, J->dtype, vb + x);
    }
  }
  J->m_out[ri * J->hq + h] = m;
  J->l_out[ri * J->hq + h] = l;
  for (int x = 0; x < d; ++x) J->o_out[((size_t)ri * J->hq + h) * d + x] = acc[x];
}

static void* worker(void* arg) {
  job_t* J = (job_t*)arg;
  const size_t nk1 = (size_t)(J->nk > 0 ? J->nk : 1);
  double* score = (double*)malloc(sizeof(double) * nk1);
  char* allowed = (char*)malloc(nk1);
  double* qrow = (double*)malloc(sizeof(double) * (size_t)J->d);
  double* acc = (double*)malloc(sizeof(double) * (size_t)J->d);
  if (!score || !allowed || !qrow || !acc) {
    __atomic_store_n(&J->failed, 1, __ATOMIC_SEQ_CST);
  } else {
    const long long total = J->nrows * (long long)J->hq;
    for (;;) {
      const long long item = __atomic_fetch_add(&J->next, 1, __ATOMIC_RELAXED);
      if (item >= total) break;
      one_row(J, item, score, allowed, qrow, acc);
    }
  }
  free(score);
  free(allowed);
  free(qrow);
  free(acc);
  return NULL;
}

/*
 * Returns 0 on success, -1 on a bad argument, -2 when memory or threads
 * could not be had.  q_pos / k_pos may be NULL (position = index).  q_doc
 * and k_doc are both NULL (one document) or both given.
 */
int oracle_partial_state_masked(const void* q, const void* k, const void* v, int dtype,
                                long long nq, long long nk, int hq, int hkv, int d,
                                double scale, int causal, long long window,
                                const long long* q_pos, const long long* k_pos,
                                const long long* q_doc, const long long* k_doc,
                                const long long* rows, long long nrows, double* m_out,
                                double* l_out, double* o_out, int nthreads) {
  if (dtype != ORACLE_F32 && dtype != ORACLE_BF16) return -1;
  if (window < 0 || (!q_doc) != (!k_doc)) return -1;
  if (hq <= 0 || hkv <= 0 || d <= 0 || hq % hkv != 0 || nq < 0 || nk < 0 || nrows < 0) return -1;
  if (nrows > 0 && (!q || !rows || !m_out || !l_out || !o_out)) return -1;
  if (nk > 0 && (!k || !v)) return -1;
  for (long long i = 0; i < nrows; ++i)
    if (rows[i] < 0 || rows[i] >= nq) return -1;
  if (nthreads < 1) nthreads = 1;

  job_t J;
  memset(&J, 0, sizeof J);
  J.q = q; J.k = k; J.v = v; J.dtype = dtype;
  J.nq = nq; J.nk = nk; J.hq = hq; J.hkv = hkv; J.d = d;
  J.scale = scale; J.causal = causal; J.window = window;
  J.q_doc = q_doc; J.k_doc = k_doc;
  J.q_pos = q_pos; J.k_pos = k_pos; J.rows = rows; J.nrows = nrows;
  J.m_out = m_out; J.l_out = l_out; J.o_out = o_out;

  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
  if (!th) return -2;
  int started = 0;
  for (int i = 0; i < nthreads; ++i) {
    if (pthread_create(&th[i], NULL, worker, &J) != 0) break;
    ++started;
  }
  if (started == 0) worker(&J);
  for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
  free(th);
  return J.failed ? -2 : 0;
}

/* The causal-only form: no window, one document. */
int oracle_partial_state(const void* q, const void* k, const void* v, int dtype,
                         long long nq, long long nk, int hq, int hkv, int d, double scale,
                         int causal, const long long* q_pos, const long long* k_pos,
                         const long long* rows, long long nrows, double* m_out,
                         double* l_out, double* o_out, int nthreads) {
  return oracle_partial_state_masked(q, k, v, dtype, nq, nk, hq, hkv, d, scale, causal, 0, q_pos,
                                     k_pos, NULL, NULL, rows, nrows, m_out, l_out, o_out,
                                     nthreads);
}

/* Version tag so the Python side can tell a stale build. */
int oracle_abi_version(void) { return 2; }

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

/*
 * Gradients of dense attention -- the backward pass the ring runs again
 * ("Ring Attention：把超长序列沿设备环流动", section "Backward 需要让梯度也
 * 沿环传播": every (Q block, K/V block) pair adds to dQ, dK and dV, and the
 * softmax statistics are recomputed from the saved log-sum-exp).  What is
 * computed here is the plain calculus of O = softmax(S) V with S = scale *
 * Q K^T over the allowed keys, for the loss L = sum(dO * O):
 *   P_rt  = exp(s_rt - LSE_r)               (the row softmax)
 *   dP_rt = dO_r . v_t
 *   D_r   = sum_t P_rt dP_rt
 *   dS_rt = P_rt (dP_rt - D_r)
 *   dQ_r  = scale * sum_t dS_rt k_t
 *   dK_t  = scale * sum over (r, query heads of t's KV head) dS_rt q_r
 *   dV_t  = sum over (r, query heads of t's KV head) P_rt dO_r
 * Everything in fp64.  Rows with no allowed key have P = 0 and contribute
 * nothing.
 *
 * oracle_grad_q: for the listed query rows and every head, LSE, D and dQ.
 * oracle_grad_kv: for the listed keys and every KV head, dK and dV; it
 * needs LSE and D of every query row (from oracle_grad_q over all rows).
 *
 * Absolute-term sums (optional outputs; NULL skips them).  These are not a
 * step of the method and the pages have no counterpart: they are the
 * magnitudes that bound rounding error in the standard forward error
 * analysis of a sum (Higham, "Accuracy and Stability of Numerical
 * Algorithms", ch. 3: fl(sum x_i) - sum x_i is at most a multiple of the
 * unit roundoff times sum |x_i|).  Each is the same sum as above with
 * every product and every term replaced by its absolute value:
 *   |dP|_rt = sum_x |dO_rx| |v_tx|
 *   A_D,r   = sum_t P_rt |dP|_rt
 *   A_S,rt  = P_rt (|dP|_rt + A_D,r)
 *   A_dQ,r  = scale * sum_t A_S,rt |k_t|
 *   A_dK,t  = scale * sum over (r, query heads) A_S,rt |q_r|
 *   A_dV,t  = sum over (r, query heads) P_rt |dO_r|
 * A rounding of relative size u in any operand of a product (P or dS
 * rounded to bf16, D taken from a rounded O) moves an output element by at
 * most a small multiple of u times its A.  Elementwise A >= |gradient|.
 * oracle_grad_q writes A_dQ and A_D; oracle_grad_kv takes A_D of every
 * query row and writes A_dK and A_dV.
 */
typedef struct {
  job_t base;  /* inputs, mask, positions, rows, threads */
  const void* dout;
  double* dq;   /* [nrows, hq, d] */
  double* lse;  /* [nrows, hq] (grad_q: out; grad_kv: in, all nq rows) */
  double* dvec; /* [nrows, hq] (same) */
  double* dk;   /* [nkeys, hkv, d] */
  double* dv;
  const long long* keys;
  long long nkeys;
  /* absolute-term sums, NULL when not asked for */
  double* dq_abs;   /* [nrows, hq, d] */
  double* dvec_abs; /* [nrows, hq] (grad_q: out; grad_kv: in, all nq rows) */
  double* dk_abs;   /* [nkeys, hkv, d] */
  double* dv_abs;
} gjob_t;

static int pair_allowed(const job_t* J, long long r, long long t) {
  const long long qp = J->q_pos ? J->q_pos[r] : r;
  const long long kp = J->k_pos ? J->k_pos[t] : t;
  if (J->causal && kp > qp) return 0;
  if (J->window > 0 && (qp - kp >= J->window || kp - qp >= J->window)) return 0;
  if (J->q_doc && (J->q_doc[r] < 0 || J->k_doc[t] != J->q_doc[r])) return 0;
  return 1;
}

static double dot_rows(const job_t* J, const void* a, size_t ia, const void* b, size_t ib) {
  double s = 0.0;
  for (int x = 0; x < J->d; ++x) s += widen(a, J->dtype, ia + x) * widen(b, J->dtype, ib + x);
  return s;
}

/* sum_x |a_x| |b_x| */
static double dot_abs(const job_t* J, const void* a, size_t ia, const void* b, size_t ib) {
  double s = 0.0;
  for (int x = 0; x < J->d; ++x)
    s += fabs(widen(a, J->dtype, ia + x)) * fabs(widen(b, J->dtype, ib + x));
  return s;
}

static void grad_q_item(gjob_t* G, long long item, double* sc) {
  job_t* J = &G->base;
  const long long ri = item / J->hq;
  const int h = (int)(item % J->hq);
  const int d = J->d, kh = h / (J->hq / J->hkv);
  const long long r = J->rows[ri];
  const size_t qb = ((size_t)r * J->hq + h) * d;
  /* scores and their max */
  double m = -INFINITY;
  for (long long t = 0; t < J->nk; ++t) {
    if (!pair_allowed(J, r, t)) { sc[t] = NAN; continue; }
    sc[t] = dot_rows(J, J->q, qb, J->k, ((size_t)t * J->hkv + kh) * d) * J->scale;
    if (sc[t] > m) m = sc[t];
  }
  double l = 0.0;
  if (m > -INFINITY)
    for (long long t = 0; t < J->nk; ++t)
      if (!isnan(sc[t])) l += exp(sc[t] - m);
  const double lse = l > 0.0 ? m + log(l) : -INFINITY;
  /* D = sum P dP, then dQ */
  double D = 0.0, Da = 0.0;
  double* dq = G->dq + ((size_t)ri * J->hq + h) * d;
  double* dqa = G->dq_abs ? G->dq_abs + ((size_t)ri * J->hq + h) * d : NULL;
  for (int x = 0; x < d; ++x) dq[x] = 0.0;
  if (dqa)
    for (int x = 0; x < d; ++x) dqa[x] = 0.0;
  if (l > 0.0) {
    for (long long t = 0; t < J->nk; ++t) {
      if (isnan(sc[t])) continue;
      const double p = exp(sc[t] - lse);
      const size_t vb = ((size_t)t * J->hkv + kh) * d;
      D += p * dot_rows(J, G->dout, qb, J->v, vb);
      if (dqa) Da += p * dot_abs(J, G->dout, qb, J->v, vb);
    }
    for (long long t = 0; t < J->nk; ++t) {
      if (isnan(sc[t])) continue;
      const double p = exp(sc[t] - lse);
      const size_t kb = ((size_t)t * J->hkv + kh) * d;
      const double dp = dot_rows(J, G->dout, qb, J->v, kb);
      const double ds = p * (dp - D);
      for (int x = 0; x < d; ++x) dq[x] += J->scale * ds * widen(J->k, J->dtype, kb + x);
      if (dqa) {
        const double dsa = p * (dot_abs(J, G->dout, qb, J->v, kb) + Da);
        for (int x = 0; x < d; ++x) dqa[x] += J->scale * dsa * fabs(widen(J->k, J->dtype, kb + x));
      }
    }
  }
  G->lse[ri * J->hq + h] = lse;
  G->dvec[ri * J->hq + h] = D;
  if (G->dvec_abs) G->dvec_abs[ri * J->hq + h] = Da;
}

static void grad_kv_item(gjob_t* G, long long item) {
  job_t* J = &G->base;
  const long long ti = item / J->hkv;
  const int kh = (int)(item % J->hkv);
  const int d = J->d, g = J->hq / J->hkv;
  const long long t = G->keys[ti];
  const size_t kb = ((size_t)t * J->hkv + kh) * d;
  double* dk = G->dk + ((size_t)ti * J->hkv + kh) * d;
  double* dv = G->dv + ((size_t)ti * J->hkv + kh) * d;
  double* dka = G->dk_abs ? G->dk_abs + ((size_t)ti * J->hkv + kh) * d : NULL;
  double* dva = G->dv_abs ? G->dv_abs + ((size_t)ti * J->hkv + kh) * d : NULL;
  for (int x = 0; x < d; ++x) dk[x] = dv[x] = 0.0;
  if (dka)
    for (int x = 0; x < d; ++x) dka[x] = dva[x] = 0.0;
  for (int hl = 0; hl < g; ++hl) {
    const int h = kh * g + hl;
    for (long long r = 0; r < J->nq; ++r) {
      const double lse = G->lse[r * J->hq + h];
      if (lse == -INFINITY || !pair_allowed(J, r, t)) continue;
      const size_t qb = ((size_t)r * J->hq + h) * d;
      const double s = dot_rows(J, J->q, qb, J->k, kb) * J->scale;
      const double p = exp(s - lse);
      const double dp = dot_rows(J, G->dout, qb, J->v, kb);
      const double ds = p * (dp - G->dvec[r * J->hq + h]);
      for (int x = 0; x < d; ++x) {
        dk[x] += J->scale * ds * widen(J->q, J->dtype, qb + x);
        dv[x] += p * widen(G->dout, J->dtype, qb + x);
      }
      if (dka) {
        const double dsa = p * (dot_abs(J, G->dout, qb, J->v, kb) + G->dvec_abs[r * J->hq + h]);
        for (int x = 0; x < d; ++x) {
          dka[x] += J->scale * dsa * fabs(widen(J->q, J->dtype, qb + x));
          dva[x] += p * fabs(widen(G->dout, J->dtype, qb + x));
        }
      }
    }
  }
}

static void* gq_worker(void* arg) {
  gjob_t* G = (gjob_t*)arg;
  job_t* J = &G->base;
  double* sc = (double*)malloc(sizeof(double) * (size_t)(J->nk > 0 ? J->nk : 1));
  if (!sc) {
    __atomic_store_n(&J->failed, 1, __ATOMIC_SEQ_CST);
    return NULL;
  }
  const long long total = J->nrows * (long long)J->hq;
  for (;;) {
    const long long item = __atomic_fetch_add(&J->next, 1, __ATOMIC_RELAXED);
    if (item >= total) break;
    grad_q_item(G, item, sc);
  }
  free(sc);
  return NULL;
}

static void* gkv_worker(void* arg) {
  gjob_t* G = (gjob_t*)arg;
  job_t* J = &G->base;
  const long long total = G->nkeys * (long long)J->hkv;
  for (;;) {
    const long long item = __atomic_fetch_add(&J->next, 1, __ATOMIC_RELAXED);
    if (item >= total) break;
    grad_kv_item(G, item);
  }
  return NULL;
}

static int run_threads(void* (*fn)(void*), void* arg, int nthreads) {
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
  if (!th) return -2;
  int started = 0;
  for (int i = 0; i < nthreads; ++i) {
    if (pthread_create(&th[i], NULL, fn, arg) != 0) break;
    ++started;
  }
  if (started == 0) fn(arg);
  for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
  free(th);
  return 0;
}

static int grad_setup(gjob_t* G, const void* q, const void* k, const void* v, const void* dout,
                      int dtype, long long nq, long long nk, int hq, int hkv, int d,
                      double scale, int causal, long long window, const long long* q_pos,
                      const long long* k_pos, const long long* q_doc, const long long* k_doc) {
  if (dtype != ORACLE_F32 && dtype != ORACLE_BF16) return -1;
  if (hq <= 0 || hkv <= 0 || d <= 0 || hq % hkv != 0 || nq < 0 || nk < 0) return -1;
  if (window < 0 || (!q_doc) != (!k_doc)) return -1;
  if ((nq > 0 && (!q || !dout)) || (nk > 0 && (!k || !v))) return -1;
  memset(G, 0, sizeof *G);
  job_t* J = &G->base;
  J->q = q; J->k = k; J->v = v; J->dtype = dtype;
  J->nq = nq; J->nk = nk; J->hq = hq; J->hkv = hkv; J->d = d;
  J->scale = scale; J->causal = causal; J->window = window;
  J->q_pos = q_pos; J->k_pos = k_pos; J->q_doc = q_doc; J->k_doc = k_doc;
  G->dout = dout;
  return 0;
}

int oracle_grad_q(const void* q, const void* k, const void* v, const void* dout, int dtype,
                  long long nq, long long nk, int hq, int hkv, int d, double scale, int causal,
                  long long window, const long long* q_pos, const long long* k_pos,
                  const long long* q_doc, const long long* k_doc, const long long* rows,
                  long long nrows, double* dq_out, double* lse_out, double* d_out,
                  double* dq_abs_out, double* d_abs_out, int nthreads) {
  gjob_t G;
  int rc = grad_setup(&G, q, k, v, dout, dtype, nq, nk, hq, hkv, d, scale, causal, window, q_pos,
                      k_pos, q_doc, k_doc);
  if (rc != 0) return rc;
  if (nrows < 0 || (nrows > 0 && (!rows || !dq_out || !lse_out || !d_out))) return -1;
  for (long long i = 0; i < nrows; ++i)
    if (rows[i] < 0 || rows[i] >= nq) return -1;
  G.base.rows = rows;
  G.base.nrows = nrows;
  if ((!dq_abs_out) != (!d_abs_out)) return -1;
  G.dq = dq_out;
  G.lse = lse_out;
  G.dvec = d_out;
  G.dq_abs = dq_abs_out;
  G.dvec_abs = d_abs_out;
  if (run_threads(gq_worker, &G, nthreads < 1 ? 1 : nthreads) != 0) return -2;
  return G.base.failed ? -2 : 0;
}

int oracle_grad_kv(const void* q, const void* k, const void* v, const void* dout, int dtype,
                   long long nq, long long nk, int hq, int hkv, int d, double scale, int causal,
                   long long window, const long long* q_pos, const long long* k_pos,
                   const long long* q_doc, const long long* k_doc, const double* lse_all,
                   const double* d_all, const long long* keys, long long nkeys, double* dk_out,
                   double* dv_out, const double* d_abs_all, double* dk_abs_out,
                   double* dv_abs_out, int nthreads) {
  gjob_t G;
  int rc = grad_setup(&G, q, k, v, dout, dtype, nq, nk, hq, hkv, d, scale, causal, window, q_pos,
                      k_pos, q_doc, k_doc);
  if (rc != 0) return rc;
  if (nkeys < 0 || (nkeys > 0 && (!keys || !dk_out || !dv_out || !lse_all || !d_all))) return -1;
  for (long long i = 0; i < nkeys; ++i)
    if (keys[i] < 0 || keys[i] >= nk) return -1;
  G.lse = (double*)lse_all;
  G.dvec = (double*)d_all;
  G.keys = keys;
  G.nkeys = nkeys;
  if ((!d_abs_all) != (!dk_abs_out) || (!d_abs_all) != (!dv_abs_out)) return -1;
  G.dk = dk_out;
  G.dv = dv_out;
  G.dvec_abs = (double*)d_abs_all;
  G.dk_abs = dk_abs_out;
  G.dv_abs = dv_abs_out;
  if (run_threads(gkv_worker, &G, nthreads < 1 ? 1 : nthreads) != 0) return -2;
  return G.base.failed ? -2 : 0;
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
int oracle_abi_version(void) { return 4; }

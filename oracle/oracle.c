/*
 * oracle.c -- fp64 CPU oracle for decode-step top-K sparse attention.
 *
 * TEST INFRASTRUCTURE ONLY (see oracle.h).  Plain definitions, written in
 * the order the pages state them; sorting uses the C library's qsort as a
 * primitive.  Nothing here is blocked, fused or reordered for speed.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

double orc_bf16_to_f64(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* ---- a1: static window (RetrievalAttention, "CPU-GPU Co-Execution",
 * W = initial tokens + most recent tokens, clipped to the cache). ------- */
int orc_in_window(int64_t i, int64_t L, int64_t n_init, int64_t n_recent) {
  if (i < 0 || i >= L) return 0;
  if (i < n_init) return 1;
  if (i >= L - n_recent) return 1;
  return 0;
}

/* ---- a2: logits z_i = q . k_i / sqrt(d) (RetrievalAttention Eq. 1;
 * ReTopK "Exact Top-K" e_{t,i}). ---------------------------------------- */
void orc_scores(const uint16_t* q, const uint16_t* k, int64_t L, int d,
                int64_t ld, double scale, double* z) {
  for (int64_t i = 0; i < L; ++i) {
    double acc = 0.0;
    for (int j = 0; j < d; ++j)
      acc += orc_bf16_to_f64(q[j]) * orc_bf16_to_f64(k[i * ld + j]);
    z[i] = scale * acc;
  }
}

/* ---- a3: exact top-K by (z desc, index asc) --------------------------- */
typedef struct { double z; int64_t i; } zi_pair;

static int cmp_rank(const void* a, const void* b) {
  const zi_pair* x = (const zi_pair*)a;
  const zi_pair* y = (const zi_pair*)b;
  if (x->z > y->z) return -1;
  if (x->z < y->z) return 1;
  if (x->i < y->i) return -1;
  if (x->i > y->i) return 1;
  return 0;
}

/* Whole pool in rank order (caller frees). */
static zi_pair* rank_pool(const double* z, const int64_t* pool, int64_t n) {
  zi_pair* r = (zi_pair*)malloc((size_t)(n > 0 ? n : 1) * sizeof(zi_pair));
  for (int64_t s = 0; s < n; ++s) {
    r[s].z = z[pool[s]];
    r[s].i = pool[s];
  }
  qsort(r, (size_t)n, sizeof(zi_pair), cmp_rank);
  return r;
}

int64_t orc_topk(const double* z, const int64_t* pool, int64_t n, int64_t K,
                 int64_t* out) {
  if (K <= 0 || n <= 0) return 0;
  zi_pair* r = rank_pool(z, pool, n);
  int64_t m = K < n ? K : n;
  for (int64_t s = 0; s < m; ++s) out[s] = r[s].i;
  free(r);
  return m;
}

static int cmp_i64(const void* a, const void* b) {
  int64_t x = *(const int64_t*)a, y = *(const int64_t*)b;
  return (x > y) - (x < y);
}

int orc_topk_check(const double* z, const int64_t* pool, int64_t n, int64_t K,
                   const int64_t* got, int64_t n_got, double rel) {
  int64_t want = K < n ? K : n;
  if (want < 0) want = 0;
  if (n_got != want) return 0;
  if (want == 0) return 1;

  /* got must be distinct members of the pool */
  int64_t* pool_sorted = (int64_t*)malloc((size_t)n * sizeof(int64_t));
  int64_t* got_sorted = (int64_t*)malloc((size_t)n_got * sizeof(int64_t));
  memcpy(pool_sorted, pool, (size_t)n * sizeof(int64_t));
  memcpy(got_sorted, got, (size_t)n_got * sizeof(int64_t));
  qsort(pool_sorted, (size_t)n, sizeof(int64_t), cmp_i64);
  qsort(got_sorted, (size_t)n_got, sizeof(int64_t), cmp_i64);
  int ok = 1;
  for (int64_t s = 0; s < n_got && ok; ++s) {
    if (s > 0 && got_sorted[s] == got_sorted[s - 1]) ok = 0;
    if (ok && bsearch(&got_sorted[s], pool_sorted, (size_t)n, sizeof(int64_t),
                      cmp_i64) == NULL)
      ok = 0;
  }
  if (!ok) {
    free(pool_sorted);
    free(got_sorted);
    return 0;
  }

  zi_pair* r = rank_pool(z, pool, n);
  int64_t* own = (int64_t*)malloc((size_t)want * sizeof(int64_t));
  for (int64_t s = 0; s < want; ++s) own[s] = r[s].i;
  qsort(own, (size_t)want, sizeof(int64_t), cmp_i64);
  int same = memcmp(own, got_sorted, (size_t)want * sizeof(int64_t)) == 0;
  int result = 0;
  if (same) {
    result = 1;
  } else if (want < n) {
    double zk = r[want - 1].z, zk1 = r[want].z;
    double margin = rel * fabs(zk);
    if (fabs(zk - zk1) < margin) {
      result = 2;
      for (int64_t s = 0; s < n_got; ++s)
        if (z[got_sorted[s]] < zk - margin) result = 0;
    }
  }
  free(own);
  free(r);
  free(pool_sorted);
  free(got_sorted);
  return result;
}

/* ---- a4/a5: partial attention with local max (RetrievalAttention Eq. 3,
 * o_W with z~1 and o_Omega with z~2). ----------------------------------- */
void orc_partial(const double* z, const int64_t* idx, int64_t n,
                 const uint16_t* v, int d, int64_t ld,
                 double* o, double* m, double* l, double* lse) {
  for (int j = 0; j < d; ++j) o[j] = 0.0;
  if (n <= 0) {
    *m = -INFINITY;
    *l = 0.0;
    *lse = -INFINITY;
    return;
  }
  double mx = -INFINITY;
  for (int64_t s = 0; s < n; ++s)
    if (z[idx[s]] > mx) mx = z[idx[s]];
  double sum = 0.0;
  for (int64_t s = 0; s < n; ++s) {
    double w = exp(z[idx[s]] - mx);
    sum += w;
    for (int j = 0; j < d; ++j) o[j] += w * orc_bf16_to_f64(v[idx[s] * ld + j]);
  }
  for (int j = 0; j < d; ++j) o[j] /= sum;
  *m = mx;
  *l = sum;
  *lse = mx + log(sum);
}

/* ---- a6: gamma1/gamma2 rescale (RetrievalAttention Eq. 4-5). ---------- */
void orc_merge(const double* o1, double m1, double l1,
               const double* o2, double m2, double l2, int d,
               double* o, double* lse) {
  int e1 = !(l1 > 0.0), e2 = !(l2 > 0.0); /* empty partials carry no mass */
  if (e1 && e2) {
    for (int j = 0; j < d; ++j) o[j] = 0.0;
    *lse = -INFINITY;
    return;
  }
  double zt = e1 ? m2 : (e2 ? m1 : (m1 > m2 ? m1 : m2));
  double a1 = e1 ? 0.0 : exp(m1 - zt) * l1; /* e^(z~1 - z~) sum_W e^(z - z~1) */
  double a2 = e2 ? 0.0 : exp(m2 - zt) * l2;
  double den = a1 + a2; /* sum over W u Omega of e^(z - z~) */
  double g1 = a1 / den, g2 = a2 / den;
  for (int j = 0; j < d; ++j) o[j] = g1 * o1[j] + g2 * o2[j];
  *lse = zt + log(den);
}

/* ---- one head of the decode step -------------------------------------- */
static int64_t window_list(int64_t L, int64_t n_init, int64_t n_recent,
                           int64_t* w) {
  int64_t c = 0;
  for (int64_t i = 0; i < L; ++i)
    if (orc_in_window(i, L, n_init, n_recent)) w[c++] = i;
  return c;
}

void orc_decode_eval_set(const double* z, const uint16_t* v, int64_t L, int d,
                         int64_t ld, int64_t n_init, int64_t n_recent,
                         const int64_t* given, int64_t n_given, double* out,
                         double* lse) {
  int64_t* w = (int64_t*)malloc((size_t)(L > 0 ? L : 1) * sizeof(int64_t));
  int64_t nw = window_list(L, n_init, n_recent, w);
  double* oW = (double*)malloc((size_t)d * sizeof(double));
  double* oS = (double*)malloc((size_t)d * sizeof(double));
  double mW, lW, lseW, mS, lS, lseS;
  orc_partial(z, w, nw, v, d, ld, oW, &mW, &lW, &lseW);
  orc_partial(z, given, n_given, v, d, ld, oS, &mS, &lS, &lseS);
  orc_merge(oW, mW, lW, oS, mS, lS, d, out, lse);
  free(oS);
  free(oW);
  free(w);
}

void orc_decode_head(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                     int64_t L, int d, int64_t ld, double scale, int64_t K,
                     int64_t n_init, int64_t n_recent, double* out,
                     double* lse, int64_t* sel, int64_t* n_sel, double* z) {
  orc_scores(q, k, L, d, ld, scale, z);
  /* pool P = [0, L) \ W_t (W and Omega disjoint, Eq. 3) */
  int64_t* pool = (int64_t*)malloc((size_t)(L > 0 ? L : 1) * sizeof(int64_t));
  int64_t np = 0;
  for (int64_t i = 0; i < L; ++i)
    if (!orc_in_window(i, L, n_init, n_recent)) pool[np++] = i;
  *n_sel = orc_topk(z, pool, np, K, sel);
  orc_decode_eval_set(z, v, L, d, ld, n_init, n_recent, sel, *n_sel, out, lse);
  free(pool);
}

/* ------------------------------------------------------------------ */
/* ReTopK                                                               */

int orc_retopk_create(orc_retopk* st, int Hq, int d, int64_t K, int C, int R,
                      int64_t W, double tau, int64_t T_r) {
  memset(st, 0, sizeof *st);
  if (Hq <= 0 || d <= 0 || K < 0 || C <= 0 || R <= 0 || R > C || W < 0 ||
      T_r <= 0)
    return -1;
  st->Hq = Hq;
  st->d = d;
  st->K = K;
  st->C = C;
  st->R = R;
  st->W = W;
  st->tau = tau;
  st->T_r = T_r;
  st->t = 0;
  st->stamp = 0;
  size_t kk = (size_t)(K > 0 ? K : 1);
  st->qbar = (double*)calloc((size_t)Hq * C * d, sizeof(double));
  st->sup = (int64_t*)calloc((size_t)Hq * C * kk, sizeof(int64_t));
  st->sup_n = (int64_t*)calloc((size_t)Hq * C, sizeof(int64_t));
  st->age = (int64_t*)calloc((size_t)Hq * C, sizeof(int64_t));
  return 0;
}

void orc_retopk_destroy(orc_retopk* st) {
  free(st->qbar);
  free(st->sup);
  free(st->sup_n);
  free(st->age);
  memset(st, 0, sizeof *st);
}

static void normalise(const uint16_t* q, int d, double* out) {
  double nn = 0.0;
  for (int j = 0; j < d; ++j) {
    double x = orc_bf16_to_f64(q[j]);
    nn += x * x;
  }
  double nrm = sqrt(nn);
  for (int j = 0; j < d; ++j)
    out[j] = nrm > 0.0 ? orc_bf16_to_f64(q[j]) / nrm : 0.0;
}

void orc_retopk_set_slot(orc_retopk* st, int h, int c, const uint16_t* q,
                         const int64_t* support, int64_t n) {
  size_t hc = (size_t)h * st->C + c;
  normalise(q, st->d, st->qbar + hc * st->d);
  int64_t m = n < st->K ? n : st->K;
  for (int64_t s = 0; s < m; ++s) st->sup[hc * st->K + s] = support[s];
  st->sup_n[hc] = m;
  /* slot c of the initial cache holds prefill query L0-C+c: c=0 oldest */
  st->age[hc] = c;
  if (st->stamp < st->C) st->stamp = st->C;
}

/* slot order for recall: rho descending, older slot first on equal rho */
typedef struct { double rho; int64_t age; int slot; } slot_rank;

static int cmp_slot(const void* a, const void* b) {
  const slot_rank* x = (const slot_rank*)a;
  const slot_rank* y = (const slot_rank*)b;
  if (x->rho > y->rho) return -1;
  if (x->rho < y->rho) return 1;
  if (x->age < y->age) return -1;
  if (x->age > y->age) return 1;
  return 0;
}

/* A_t = Unique(U_{c in chosen} S_c  u  [max(0, L-W), L)), ascending. */
static int64_t candidate_union(const orc_retopk* st, int h, const int* chosen,
                               int n_chosen, int64_t L, int64_t* cand) {
  int64_t cap = (int64_t)n_chosen * st->K + st->W;
  int64_t* tmp = (int64_t*)malloc((size_t)(cap > 0 ? cap : 1) * sizeof(int64_t));
  int64_t c = 0;
  for (int r = 0; r < n_chosen; ++r) {
    size_t hc = (size_t)h * st->C + chosen[r];
    for (int64_t s = 0; s < st->sup_n[hc]; ++s) tmp[c++] = st->sup[hc * st->K + s];
  }
  int64_t lo = L - st->W > 0 ? L - st->W : 0;
  for (int64_t i = lo; i < L; ++i) tmp[c++] = i;
  qsort(tmp, (size_t)c, sizeof(int64_t), cmp_i64);
  int64_t u = 0;
  for (int64_t s = 0; s < c; ++s)
    if (u == 0 || tmp[s] != cand[u - 1]) cand[u++] = tmp[s];
  free(tmp);
  return u;
}

static int same_list(const int64_t* a, int64_t na, const int64_t* b, int64_t nb) {
  if (na != nb) return 0;
  return na == 0 || memcmp(a, b, (size_t)na * sizeof(int64_t)) == 0;
}

void orc_retopk_step_head(orc_retopk* st, int h, const uint16_t* q,
                          const uint16_t* k, const uint16_t* v, int64_t L,
                          int64_t ld, double scale,
                          const orc_retopk_margins* mg, int other_path,
                          const int64_t* other_cand, int64_t other_n_cand,
                          const int64_t* other_sup, int64_t other_n_sup,
                          int64_t* cand, int64_t* sup, double* out,
                          orc_retopk_result* res) {
  const int d = st->d, C = st->C, R = st->R;
  const int64_t K = st->K;
  memset(res, 0, sizeof *res);
  res->cand_ok = -1;
  res->sup_ok = -1;

  /* 1. normalise the query; 2. cosine against every cached query */
  double* qb = (double*)malloc((size_t)d * sizeof(double));
  normalise(q, d, qb);
  slot_rank* sr = (slot_rank*)malloc((size_t)C * sizeof(slot_rank));
  double max_rho = -INFINITY;
  for (int c = 0; c < C; ++c) {
    const double* qc = st->qbar + ((size_t)h * C + c) * d;
    double rho = 0.0;
    for (int j = 0; j < d; ++j) rho += qb[j] * qc[j];
    sr[c].rho = rho;
    sr[c].age = st->age[(size_t)h * C + c];
    sr[c].slot = c;
    if (rho > max_rho) max_rho = rho;
  }
  res->max_rho = max_rho;

  /* 3. fallback / refresh decision */
  int refresh = (st->t % st->T_r) == 0;
  int own_exact = (max_rho < st->tau) || refresh;
  int exact = own_exact;
  if (!refresh && other_path >= 0 && fabs(max_rho - st->tau) < mg->path_abs &&
      (other_path == 1) != own_exact) {
    exact = other_path == 1;
    res->adopt_path = 1;
  }
  res->own_path = own_exact;
  res->path = exact;

  double* z = (double*)malloc((size_t)(L > 0 ? L : 1) * sizeof(double));
  int64_t* pool;
  int64_t npool;
  if (exact) {
    /* exact Top-K over every key in the cache (no window) */
    orc_scores(q, k, L, d, ld, scale, z);
    pool = (int64_t*)malloc((size_t)(L > 0 ? L : 1) * sizeof(int64_t));
    for (int64_t i = 0; i < L; ++i) pool[i] = i;
    npool = L;
    res->n_cand = L;
  } else {
    /* recall the R most similar cached queries */
    qsort(sr, (size_t)C, sizeof(slot_rank), cmp_slot);
    int* chosen = (int*)malloc((size_t)R * sizeof(int));
    for (int r = 0; r < R; ++r) chosen[r] = sr[r].slot;
    int64_t ncand = candidate_union(st, h, chosen, R, L, cand);
    res->cand_ok = -1;
    if (other_cand != NULL) {
      res->cand_ok = same_list(cand, ncand, other_cand, other_n_cand) ? 1 : 0;
      /* near-tie at the R boundary: accept the other side's union if it is
       * the union for some admissible choice of the tied slots */
      if (!res->cand_ok && R < C &&
          fabs(sr[R - 1].rho - sr[R].rho) < mg->rho_abs) {
        double edge = sr[R - 1].rho;
        int sure[64], tied[64], ns = 0, nt = 0;
        for (int c = 0; c < C && c < 64; ++c) {
          if (sr[c].rho > edge + mg->rho_abs) sure[ns++] = sr[c].slot;
          else if (fabs(sr[c].rho - edge) <= mg->rho_abs) tied[nt++] = sr[c].slot;
        }
        int need = R - ns;
        int64_t* alt = (int64_t*)malloc((size_t)(R * K + st->W + 1) * sizeof(int64_t));
        if (need >= 0 && nt <= 16) {
          for (uint32_t mask = 0; mask < (1u << nt) && !res->cand_ok; ++mask) {
            if (__builtin_popcount(mask) != need) continue;
            int pick[64], np = 0;
            for (int s = 0; s < ns; ++s) pick[np++] = sure[s];
            for (int s = 0; s < nt; ++s)
              if (mask & (1u << s)) pick[np++] = tied[s];
            int64_t na = candidate_union(st, h, pick, np, L, alt);
            if (same_list(alt, na, other_cand, other_n_cand)) {
              res->cand_ok = 2;
              res->adopt_cand = 1;
              memcpy(cand, alt, (size_t)na * sizeof(int64_t));
              ncand = na;
            }
          }
        }
        free(alt);
      }
    }
    free(chosen);
    res->n_cand = ncand;
    /* exact rescoring of every candidate with the current query */
    for (int64_t s = 0; s < ncand; ++s)
      orc_scores(q, k + cand[s] * ld, 1, d, ld, scale, &z[cand[s]]);
    pool = (int64_t*)malloc((size_t)(ncand > 0 ? ncand : 1) * sizeof(int64_t));
    memcpy(pool, cand, (size_t)ncand * sizeof(int64_t));
    npool = ncand;
  }

  /* re-top-K over the pool (|A_t| <= K keeps all of it) */
  int64_t nsup = orc_topk(z, pool, npool, K, sup);
  if (other_sup != NULL) {
    res->sup_ok = orc_topk_check(z, pool, npool, K, other_sup, other_n_sup,
                                 mg->topk_rel);
    if (res->sup_ok == 2) { /* evaluate and push the other side's valid set */
      memcpy(sup, other_sup, (size_t)other_n_sup * sizeof(int64_t));
      nsup = other_n_sup;
    }
  }
  res->n_sup = nsup;

  /* sparse softmax . V over the support (no window merge) */
  double m, l, lse;
  orc_partial(z, sup, nsup, v, d, ld, out, &m, &l, &lse);
  res->lse = lse;

  /* push (q_bar, support) into the FIFO, evicting the oldest entry */
  int oldest = 0;
  for (int c = 1; c < C; ++c)
    if (st->age[(size_t)h * C + c] < st->age[(size_t)h * C + oldest]) oldest = c;
  size_t hc = (size_t)h * C + oldest;
  memcpy(st->qbar + hc * d, qb, (size_t)d * sizeof(double));
  for (int64_t s = 0; s < nsup; ++s) st->sup[hc * K + s] = sup[s];
  st->sup_n[hc] = nsup;
  st->age[hc] = st->stamp++;

  free(pool);
  free(z);
  free(sr);
  free(qb);
}

void orc_retopk_advance(orc_retopk* st) { st->t += 1; }

/* ------------------------------------------------------------------ */
/* f4. Scalar int8 key quantisation (see oracle.h for the definitions). */

/* One code and its exact error; s is the channel's binary32 scale. */
static uint8_t q8_code(uint16_t kbits, float s, double* e) {
  const double kd = orc_bf16_to_f64(kbits);
  long c = 0;
  if (s != 0.0f) {
    const float r = (float)kd / s; /* binary32 division */
    double cr = rint((double)r);   /* nearest, ties to even */
    if (cr > 127.0) cr = 127.0;
    if (cr < -127.0) cr = -127.0;
    c = (long)cr;
  }
  *e = fabs(kd - (double)s * (double)c); /* exact: 24 x 8 bit product */
  return (uint8_t)(c + 128);
}

void orc_q8_fit(const uint16_t* k, int64_t L, int d, int64_t ld,
                float* scale, uint8_t* codes, double* err) {
  for (int j = 0; j < d; ++j) {
    double m = 0.0;
    for (int64_t i = 0; i < L; ++i) {
      const double a = fabs(orc_bf16_to_f64(k[i * ld + j]));
      if (a > m) m = a;
    }
    scale[j] = (float)m / 127.0f; /* m is a bf16 value: exact as float */
    err[j] = 0.0;
  }
  orc_q8_append(k, L, d, ld, scale, codes, err);
}

void orc_q8_append(const uint16_t* k, int64_t n, int d, int64_t ld,
                   const float* scale, uint8_t* codes, double* err) {
  for (int64_t i = 0; i < n; ++i)
    for (int j = 0; j < d; ++j) {
      double e;
      codes[i * d + j] = q8_code(k[i * ld + j], scale[j], &e);
      if (e > err[j]) err[j] = e;
    }
}

double orc_q8_bound(const uint16_t* q, int d, double scale, const double* err) {
  double acc = 0.0;
  for (int j = 0; j < d; ++j) acc += fabs(orc_bf16_to_f64(q[j])) * err[j];
  return scale * acc;
}

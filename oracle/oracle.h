/*
 * oracle.h -- fp64 CPU oracle for decode-step top-K sparse attention.
 *
 * TEST INFRASTRUCTURE ONLY.  This is a plain, slow, single-threaded C
 * restatement of what the decode path computes, written from the method's
 * definitions so that the CUDA path can be checked against it.  Only the
 * tests, the smoke check and the benchmark's CPU-baseline leg may load it.
 * It shares no code, header, table or helper with the CUDA library.
 *
 * Sources (page title, section / equation):
 *   [RA]  "RetrievalAttention: Accelerating Long-Context LLM Inference via
 *         Vector Retrieval" -- Eq. 1 (logits z_i = q.k_i/sqrt(d), softmax),
 *         Eq. 2 (renormalised sparse attention over a selected set),
 *         Eq. 3 (I = W u Omega, W = initial + recent tokens, disjoint),
 *         Eq. 4-5 (o_t = g1 o_W + g2 o_Omega with the max/sum rescale),
 *         "Flat" baseline (scan every key, exact top-k by inner product).
 *   [RTK] "Recall Before You Rank: Similarity-Guided Top-K Reuse for
 *         Efficient Long-Context Attention" (ReTopK) -- exact Top-K
 *         definition, per-head query-support FIFO cache, cosine recall of
 *         the top-R cached queries, candidate set A_t = Unique(U S_c u L_t),
 *         exact rescoring + re-top-K, tau fallback and T_r refresh,
 *         sparse softmax-V, cache push on both paths.
 *
 * Conventions
 *   - Every bf16 input is a uint16 bit pattern; it is widened exactly to
 *     double (bf16 is the upper half of an IEEE binary32).
 *   - Arithmetic is IEEE double, summed in index order, no fusion.
 *   - Indices are int64.  Token positions are 0-based: the cache holds
 *     positions 0 .. L-1 and position L-1 is the newest token.
 *   - lse = -INFINITY with o = 0 denotes attention over an empty set.
 *
 * Readings of points the pages leave open (each also listed in the
 * design notes):
 *   - d is the head dimension; the scale is supplied by the caller
 *     (1/sqrt(d) on every workload).
 *   - Window W_t = [0, n_init) u [L - n_recent, L), clipped to [0, L).
 *   - Top-K order is (z descending, index ascending); K >= |pool| selects
 *     the whole pool, K = 0 selects nothing.
 *   - ReTopK: t counts decode steps from 0 (step 0 is a refresh step);
 *     the fallback is strict (max rho < tau -> exact); top-R ties go to
 *     the older cache slot; the recent window is the last W positions
 *     including the newest token; |A_t| <= K keeps all of A_t.
 */
#ifndef TSA_ORACLE_H
#define TSA_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Exact widening of a bf16 bit pattern. */
double orc_bf16_to_f64(uint16_t h);

/* a1. 1 if position i lies in W_t = [0,n_init) u [L-n_recent, L). */
int orc_in_window(int64_t i, int64_t L, int64_t n_init, int64_t n_recent);

/* a2. z[i] = scale * sum_j q[j] * k[i*ld + j] for i < L (Eq. 1 logits).
 * q: [d] bf16; k: L rows of d bf16 with row stride ld elements. */
void orc_scores(const uint16_t* q, const uint16_t* k, int64_t L, int d,
                int64_t ld, double scale, double* z);

/* a3. Exact top-K of pool (n indices into z): the K entries of largest z,
 * ties broken by smaller index.  Writes min(K,n) indices to out in rank
 * order and returns that count. */
int64_t orc_topk(const double* z, const int64_t* pool, int64_t n, int64_t K,
                 int64_t* out);

/* Check a top-K set produced elsewhere against the exact one.
 * Returns  1: same set as orc_topk;
 *          2: different set, accepted by the near-tie rule (the fp64 K-th
 *             and (K+1)-th scores differ by less than rel*|z_(K)| and every
 *             chosen index scores at least z_(K) - rel*|z_(K)|);
 *          0: rejected (wrong size, duplicate, outside the pool, or a
 *             difference not covered by the near-tie rule). */
int orc_topk_check(const double* z, const int64_t* pool, int64_t n, int64_t K,
                   const int64_t* got, int64_t n_got, double rel);

/* a4/a5. Partial attention over the index set idx (Eq. 3 form):
 * m = max z, l = sum exp(z - m), o = sum exp(z - m) v / l, lse = m + ln l.
 * z is indexed by position (z[idx[s]]); v: rows of d bf16, stride ld.
 * Empty set: o = 0, m = lse = -inf, l = 0. */
void orc_partial(const double* z, const int64_t* idx, int64_t n,
                 const uint16_t* v, int d, int64_t ld,
                 double* o, double* m, double* l, double* lse);

/* a6. Eq. 4-5 rescale merge of two disjoint partials given as (o, m, l):
 * zt = max(m1, m2); den = l1 e^(m1-zt) + l2 e^(m2-zt);
 * g1 = e^(m1-zt) l1 / den; g2 = e^(m2-zt) l2 / den; o = g1 o1 + g2 o2.
 * Writes o (may alias neither input) and lse = zt + ln den. */
void orc_merge(const double* o1, double m1, double l1,
               const double* o2, double m2, double l2, int d,
               double* o, double* lse);

/* One query head of the decode step: scores over [0,L), pool
 * P = [0,L) \ W_t, S = top-K of P, partials over W_t and S, Eq. 4-5 merge.
 * q: [d]; k, v: L rows (stride ld).  Outputs: out[d], *lse, sel[<=K] in
 * rank order with *n_sel, z[L] (all logits; caller-allocated). */
void orc_decode_head(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                     int64_t L, int d, int64_t ld, double scale, int64_t K,
                     int64_t n_init, int64_t n_recent, double* out,
                     double* lse, int64_t* sel, int64_t* n_sel, double* z);

/* Attention output over W_t u given_set (given_set must avoid W_t): lets a
 * test evaluate the oracle on a set chosen elsewhere.  z: logits [L]. */
void orc_decode_eval_set(const double* z, const uint16_t* v, int64_t L, int d,
                         int64_t ld, int64_t n_init, int64_t n_recent,
                         const int64_t* given, int64_t n_given, double* out,
                         double* lse);

/* ------------------------------------------------------------------ */
/* ReTopK per-head query-support cache and decode step.                */

typedef struct orc_retopk {
  int Hq, d;
  int64_t K;       /* top-K budget */
  int C, R;        /* cache capacity, recalled entries */
  int64_t W;       /* recent window */
  double tau;      /* cosine fallback threshold */
  int64_t T_r;     /* refresh interval */
  int64_t t;       /* decode step counter, starts at 0 */
  int64_t stamp;   /* next insertion stamp */
  double* qbar;    /* [Hq][C][d] normalised cached queries */
  int64_t* sup;    /* [Hq][C][K] cached supports */
  int64_t* sup_n;  /* [Hq][C] support sizes */
  int64_t* age;    /* [Hq][C] insertion stamp (smaller = older) */
} orc_retopk;

int orc_retopk_create(orc_retopk* st, int Hq, int d, int64_t K, int C, int R,
                      int64_t W, double tau, int64_t T_r);
void orc_retopk_destroy(orc_retopk* st);

/* Fill slot c of head h (c = 0 is the oldest) with normalise(q) and the
 * given support.  Used to initialise the cache from the last C prefill
 * queries. */
void orc_retopk_set_slot(orc_retopk* st, int h, int c, const uint16_t* q,
                         const int64_t* support, int64_t n);

/* Decision margins used for lockstep adoption (see orc_retopk_step_head). */
typedef struct orc_retopk_margins {
  double path_abs;   /* |max rho - tau| below this: path is a near-tie  */
  double rho_abs;    /* |rho_(R) - rho_(R+1)| below this: top-R near-tie */
  double topk_rel;   /* near-tie rule for the top-K sets                 */
} orc_retopk_margins;

/* Result of one head's step. */
typedef struct orc_retopk_result {
  int path;          /* 1 = exact, 0 = reuse (the path actually taken)  */
  int own_path;      /* the oracle's own decision                       */
  double max_rho;    /* max cosine against the cache                    */
  int adopt_path;    /* 1 if the path was adopted from `other`          */
  int adopt_cand;    /* 1 if the candidate set was adopted (top-R tie)  */
  int cand_ok;       /* other's candidates: 1 equal, 2 tie-valid, 0 bad */
  int sup_ok;        /* other's support: 1 equal, 2 tie-valid, 0 bad    */
  int64_t n_cand;    /* |A_t| (reuse path) or L (exact path)            */
  int64_t n_sup;     /* |S_t|                                           */
  double lse;        /* log-sum-exp of the support logits               */
} orc_retopk_result;

/* One decode step of ReTopK for query head h (does not advance t).
 * q: [d] bf16 query; k, v: L rows (stride ld) of this head's KV head.
 * `other_*` describe another implementation's decisions for the same step
 * (pass other_path < 0 to run free).  When the oracle's own decision lies
 * within a margin it adopts the other side's choice, and records it, so
 * that one rounding-level tie does not diverge the cache state.
 * Outputs: cand (capacity R*K+W, ascending), sup (capacity K), out[d].
 * The pushed support is `other_sup` when it passes the near-tie rule,
 * else the oracle's own. */
void orc_retopk_step_head(orc_retopk* st, int h, const uint16_t* q,
                          const uint16_t* k, const uint16_t* v, int64_t L,
                          int64_t ld, double scale,
                          const orc_retopk_margins* mg, int other_path,
                          const int64_t* other_cand, int64_t other_n_cand,
                          const int64_t* other_sup, int64_t other_n_sup,
                          int64_t* cand, int64_t* sup, double* out,
                          orc_retopk_result* res);

/* Advance the shared step counter after all heads ran step t. */
void orc_retopk_advance(orc_retopk* st);

/* ------------------------------------------------------------------ */
/* f4. Scalar int8 key quantisation (RetrievalAttention review, Appendix
 * C "CPU memory minimization" and "Scalar quantization of KV vectors with
 * accuracy-preservation guarantees": 8-bit scalar quantisation of the key
 * vectors, scheme left open; per-channel symmetric is the reading).
 *
 * One scale per channel j of one (sequence, KV head):
 *   s_j  = fl32(maxabs_j / 127)       (binary32 division; maxabs over the
 *                                      fitted rows, exact as a bf16 value)
 *   c_ij = clamp(rint(fl32(k_ij / s_j)), -127, 127)   (rint: nearest, ties
 *                                      to even; c = 0 where s_j = 0)
 *   stored as the offset-binary byte u_ij = c_ij + 128
 *   e_j  = max_i |k_ij - s_j c_ij|    (exact, in double)
 * Rows appended later use the fitted s_j; a value past 127 s_j saturates
 * and its larger error enters e_j.  The decisions that produce integers
 * (s_j and the rounding of k/s) are taken in binary32, the precision of
 * the quantiser under test; the error is exact. */

/* Fit: scales over rows [0, L) and codes/errors of those rows.
 * k: L rows of d bf16, stride ld; scale[d] (binary32), codes: L rows of d
 * bytes (stride d), err[d]. */
void orc_q8_fit(const uint16_t* k, int64_t L, int d, int64_t ld,
                float* scale, uint8_t* codes, double* err);

/* Append: codes of n more rows with the given scales; err[d] is updated in
 * place (running maximum). */
void orc_q8_append(const uint16_t* k, int64_t n, int d, int64_t ld,
                   const float* scale, uint8_t* codes, double* err);

/* The logit error bound of a quantised key: for every row i,
 *   |scale * sum_j q_j k_ij - scale * sum_j q_j s_j c_ij|
 *     <= scale * sum_j |q_j| e_j.
 * Returns the right-hand side (double arithmetic). */
double orc_q8_bound(const uint16_t* q, int d, double scale, const double* err);

#ifdef __cplusplus
}
#endif
#endif

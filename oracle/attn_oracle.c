/*
 * attn_oracle.c -- plain, slow CPU oracle for fused exact attention (fp64).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call this code:
 * only the tests, the smoke check and the benchmark's CPU-baseline leg use it.
 * It shares no code, header, table or constant with the CUDA library.
 *
 * What it computes (FlashAttention-4 pages, "The Asymmetric Hardware Scaling
 * Wall on NVIDIA Blackwell", the three phases GEMM 1 / Softmax / GEMM 2, and the
 * functional validation harness, which calls the result "mathematically
 * exact"): attention is exact, so the oracle is the plain definition
 *
 *     s_ij  = scale * sum_d q_id k_jd            (j allowed; causal: j <= i)
 *     LSE_i = M_i + ln sum_j exp(s_ij - M_i),   M_i = max_j s_ij
 *     P_ij  = exp(s_ij - LSE_i)
 *     O_id  = sum_j P_ij v_jd
 *
 * with the causal mask q_idx >= kv_idx (top-left, the only form the pages'
 * simulator prints) and grouped heads: q head h reads kv head floor(h*Hkv/Hq).
 *
 * The backward pass is the textbook gradient of that definition (the pages give
 * none):  dV_j = sum_i P_ij dO_i,  dP_ij = dO_i . v_j,  D_i = dO_i . O_i,
 *         dS_ij = P_ij (dP_ij - D_i),  dQ_i = scale sum_j dS_ij k_j,
 *         dK_j = scale sum_i dS_ij q_i  (dK, dV summed over the q heads of a group).
 *
 * A second entry point restates the tiled online-softmax loop of the pages'
 * simulator ("End-to-End Implementation" section): q-tile outer loop, kv-tile
 * inner loop, running max and sum, accumulator rescale, final O/l.  Mode 0
 * rescales on every tile as the simulator does; mode 1 is the conditional
 * rescale of the pages' key contribution #2 (skip unless the running max grows
 * by more than log2(256) = 8.0), taken in the base-2 domain.  It exists to pin
 * that the tiled algorithm reaches the plain definition.
 *
 * Tensors are dense row-major [B, H, S, D] (the simulator's docstring layout),
 * LSE is [B, Hq, Sq], natural log.  Every routine returns 0 on success and a
 * negative value on a bad argument.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int oracle_version(void) { return 1; }

int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

void oracle_set_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

/* Grouped heads: contiguous groups of Hq/Hkv query heads share one kv head. */
static int kv_head_of(int h, int Hq, int Hkv) { return (int)(((long long)h * Hkv) / Hq); }

/* Number of keys row i may attend to (top-left causal: j <= i). */
static long allowed_keys(long i, long Sk, int causal) {
  if (!causal) return Sk;
  return (i + 1 < Sk) ? i + 1 : Sk;
}

static double dot(const double* a, const double* b, long D) {
  double acc = 0.0;
  for (long d = 0; d < D; ++d) acc += a[d] * b[d];
  return acc;
}

static int check_dims(int B, int Hq, int Hkv, int Sq, int Sk, int D) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Sq < 0 || Sk < 0 || D < 1) return -1;
  if (Hq % Hkv != 0) return -2;
  return 0;
}

/*
 * Forward pass of one query row from the definition.  s is scratch of Sk
 * doubles.  Writes D values of O and the row's LSE.
 */
static void fwd_one_row(const double* q_row, const double* k_head, const double* v_head,
                        long Sk, long D, long n_allowed, double scale, double* s,
                        double* o_row, double* lse_out) {
  if (n_allowed <= 0) { /* fully masked row: empty softmax */
    for (long d = 0; d < D; ++d) o_row[d] = 0.0;
    *lse_out = -INFINITY;
    return;
  }
  double M = -INFINITY;
  for (long j = 0; j < n_allowed; ++j) {
    s[j] = scale * dot(q_row, k_head + j * D, D);
    if (s[j] > M) M = s[j];
  }
  double sum = 0.0;
  for (long j = 0; j < n_allowed; ++j) sum += exp(s[j] - M);
  const double lse = M + log(sum);
  for (long d = 0; d < D; ++d) o_row[d] = 0.0;
  for (long j = 0; j < n_allowed; ++j) {
    const double p = exp(s[j] - lse);
    const double* vj = v_head + j * D;
    for (long d = 0; d < D; ++d) o_row[d] += p * vj[d];
  }
  *lse_out = lse;
  (void)Sk;
}

/*
 * Forward for a list of rows.  rows[r] is a flat row index (b*Hq + h)*Sq + i.
 * o_rows is [n_rows, D], lse_rows is [n_rows].
 */
int oracle_fwd_rows(const double* q, const double* k, const double* v, int B, int Hq, int Hkv,
                    int Sq, int Sk, int D, int causal, double scale, const int64_t* rows,
                    int64_t n_rows, double* o_rows, double* lse_rows) {
  int rc = check_dims(B, Hq, Hkv, Sq, Sk, D);
  if (rc) return rc;
  const long total = (long)B * Hq * Sq;
  for (int64_t r = 0; r < n_rows; ++r)
    if (rows[r] < 0 || rows[r] >= total) return -3;
#pragma omp parallel
  {
    double* s = (double*)malloc(sizeof(double) * (size_t)(Sk > 0 ? Sk : 1));
#pragma omp for schedule(dynamic, 4)
    for (int64_t r = 0; r < n_rows; ++r) {
      const long flat = (long)rows[r];
      const long i = flat % Sq;
      const long bh = flat / Sq;
      const long b = bh / Hq, h = bh % Hq;
      const long hk = kv_head_of((int)h, Hq, Hkv);
      const double* q_row = q + flat * D;
      const double* k_head = k + ((b * Hkv + hk) * (long)Sk) * D;
      const double* v_head = v + ((b * Hkv + hk) * (long)Sk) * D;
      fwd_one_row(q_row, k_head, v_head, Sk, D, allowed_keys(i, Sk, causal), scale, s,
                  o_rows + r * D, lse_rows + r);
    }
    free(s);
  }
  return 0;
}

/* Full forward: O [B,Hq,Sq,D], LSE [B,Hq,Sq]. */
int oracle_fwd(const double* q, const double* k, const double* v, int B, int Hq, int Hkv, int Sq,
               int Sk, int D, int causal, double scale, double* o, double* lse) {
  int rc = check_dims(B, Hq, Hkv, Sq, Sk, D);
  if (rc) return rc;
  const long total = (long)B * Hq * Sq;
#pragma omp parallel
  {
    double* s = (double*)malloc(sizeof(double) * (size_t)(Sk > 0 ? Sk : 1));
#pragma omp for schedule(dynamic, 4)
    for (long flat = 0; flat < total; ++flat) {
      const long i = flat % Sq;
      const long bh = flat / Sq;
      const long b = bh / Hq, h = bh % Hq;
      const long hk = kv_head_of((int)h, Hq, Hkv);
      fwd_one_row(q + flat * D, k + ((b * Hkv + hk) * (long)Sk) * D,
                  v + ((b * Hkv + hk) * (long)Sk) * D, Sk, D, allowed_keys(i, Sk, causal),
                  scale, s, o + flat * D, lse + flat);
    }
    free(s);
  }
  return 0;
}

/*
 * Backward from the definition for a list of kv-head units u = b*Hkv + hk.
 * For each unit it writes dK, dV of that kv head and dQ, O, LSE of every q head
 * in its group; other slices of the (full-size) outputs are left untouched.
 * O and LSE come from this oracle's own forward.
 */
int oracle_bwd_units(const double* q, const double* k, const double* v, const double* dO, int B,
                     int Hq, int Hkv, int Sq, int Sk, int D, int causal, double scale,
                     const int64_t* units, int64_t n_units, double* dq, double* dk, double* dv,
                     double* o, double* lse) {
  int rc = check_dims(B, Hq, Hkv, Sq, Sk, D);
  if (rc) return rc;
  for (int64_t u = 0; u < n_units; ++u)
    if (units[u] < 0 || units[u] >= (int64_t)B * Hkv) return -3;
  const int g = Hq / Hkv;
  double* delta = (double*)malloc(sizeof(double) * (size_t)(Sq > 0 ? Sq : 1) * (size_t)g);
  if (!delta) return -4;

  for (int64_t u = 0; u < n_units; ++u) {
    const long b = (long)(units[u] / Hkv), hk = (long)(units[u] % Hkv);
    const double* k_head = k + ((b * Hkv + hk) * (long)Sk) * D;
    const double* v_head = v + ((b * Hkv + hk) * (long)Sk) * D;
    double* dk_head = dk + ((b * Hkv + hk) * (long)Sk) * D;
    double* dv_head = dv + ((b * Hkv + hk) * (long)Sk) * D;

    /* Pass 1, per query row: O, LSE, D_i = dO_i . O_i, dQ_i. */
    for (int gi = 0; gi < g; ++gi) {
      const long h = hk * g + gi;
      const long base = (b * Hq + h) * (long)Sq;
#pragma omp parallel
      {
        double* s = (double*)malloc(sizeof(double) * (size_t)(Sk > 0 ? Sk : 1));
#pragma omp for schedule(dynamic, 4)
        for (long i = 0; i < Sq; ++i) {
          const long na = allowed_keys(i, Sk, causal);
          const double* qi = q + (base + i) * D;
          const double* doi = dO + (base + i) * D;
          double* oi = o + (base + i) * D;
          double* dqi = dq + (base + i) * D;
          fwd_one_row(qi, k_head, v_head, Sk, D, na, scale, s, oi, lse + base + i);
          const double Di = dot(doi, oi, D);
          delta[gi * (long)Sq + i] = Di;
          for (long d = 0; d < D; ++d) dqi[d] = 0.0;
          for (long j = 0; j < na; ++j) {
            const double p = exp(s[j] - lse[base + i]);
            const double dp = dot(doi, v_head + j * D, D);
            const double ds = p * (dp - Di);
            const double* kj = k_head + j * D;
            for (long d = 0; d < D; ++d) dqi[d] += scale * ds * kj[d];
          }
        }
        free(s);
      }
    }

    /* Pass 2, per key row: dK_j, dV_j summed over the group's q heads and rows. */
#pragma omp parallel for schedule(dynamic, 4)
    for (long j = 0; j < Sk; ++j) {
      double* dkj = dk_head + j * D;
      double* dvj = dv_head + j * D;
      for (long d = 0; d < D; ++d) { dkj[d] = 0.0; dvj[d] = 0.0; }
      const double* kj = k_head + j * D;
      const double* vj = v_head + j * D;
      for (int gi = 0; gi < g; ++gi) {
        const long h = hk * g + gi;
        const long base = (b * Hq + h) * (long)Sq;
        for (long i = causal ? j : 0; i < Sq; ++i) {
          const double* qi = q + (base + i) * D;
          const double* doi = dO + (base + i) * D;
          const double sij = scale * dot(qi, kj, D);
          const double p = exp(sij - lse[base + i]);
          const double dp = dot(doi, vj, D);
          const double ds = p * (dp - delta[gi * (long)Sq + i]);
          for (long d = 0; d < D; ++d) {
            dkj[d] += scale * ds * qi[d];
            dvj[d] += p * doi[d];
          }
        }
      }
    }
  }
  free(delta);
  return 0;
}

/* ---- tiled online-softmax restatement, fp64 and fp32 ---- */
#define REAL double
#define EXP exp
#define EXP2 exp2
#define LOG log
#define LOG2 log2
#define TILED_NAME oracle_tiled_fwd_f64
#include "tiled_body.h"
#undef REAL
#undef EXP
#undef EXP2
#undef LOG
#undef LOG2
#undef TILED_NAME

#define REAL float
#define EXP expf
#define EXP2 exp2f
#define LOG logf
#define LOG2 log2f
#define TILED_NAME oracle_tiled_fwd_f32
#include "tiled_body.h"

/* ---- score modification: a sliding window and a linear relative-position bias ----
 *
 * The pages name score modifications, relative position biases and custom masks
 * (FlexAttention integration) without defining any.  Reading taken: key j is
 * visible to query i iff (wl < 0 || j >= i - wl) && (wr < 0 || j <= i + wr), so
 * wl = -1, wr = 0 is the causal mask and wl = wr = -1 no mask; the score of a
 * visible pair in query head h is scale * q_i . k_j + slope[h] * (j - i) (slopes
 * NULL: no bias).  A custom key padding mask: with per-batch key lengths
 * seqlens_k (NULL: none), keys j >= seqlens_k[b] are invisible in batch b.  The
 * row's softmax, LSE and the gradients follow the plain definition with that
 * score over the visible keys; a row with none has O = 0 and LSE = -inf and
 * contributes no gradient.
 */

/* Visible keys of query i: the interval [*lo, *hi) (empty when *hi <= *lo). */
static void mod_key_range(long i, long Sk, int wl, int wr, long* lo, long* hi) {
  long a = 0, b = Sk;
  if (wl >= 0 && i - wl > a) a = i - wl;
  if (wr >= 0 && i + wr + 1 < b) b = i + wr + 1;
  *lo = a;
  *hi = (b > a) ? b : a;
}

/* Score of (i, j) with the bias. */
static double mod_score(const double* qi, const double* kj, long D, double scale, double slope,
                        long i, long j) {
  return scale * dot(qi, kj, D) + slope * (double)(j - i);
}

/* One query row: O (D values) and LSE over the visible keys; s is scratch [Sk]. */
static void mod_fwd_row(const double* qi, const double* k_head, const double* v_head, long D,
                        long i, long lo, long hi, double scale, double slope, double* s,
                        double* oi, double* lse_out) {
  for (long d = 0; d < D; ++d) oi[d] = 0.0;
  if (hi <= lo) {
    *lse_out = -INFINITY;
    return;
  }
  double top = -INFINITY;
  for (long j = lo; j < hi; ++j) {
    s[j] = mod_score(qi, k_head + j * D, D, scale, slope, i, j);
    top = fmax(top, s[j]);
  }
  double z = 0.0;
  for (long j = lo; j < hi; ++j) z += exp(s[j] - top);
  const double row_lse = top + log(z);
  for (long j = lo; j < hi; ++j) {
    const double w = exp(s[j] - row_lse);
    for (long d = 0; d < D; ++d) oi[d] += w * v_head[j * D + d];
  }
  *lse_out = row_lse;
}

static double head_slope(const double* slopes, long h) { return slopes ? slopes[h] : 0.0; }

/* Keys of batch b that exist: the first seqlens_k[b] (clamped to [0, Sk]);
 * all Sk without lengths.  Keys past it are invisible to every query. */
static long batch_keys(const int* seqlens_k, long b, long Sk) {
  if (!seqlens_k) return Sk;
  const long L = seqlens_k[b];
  return L < 0 ? 0 : (L > Sk ? Sk : L);
}

/* Full forward with the score modification: O [B,Hq,Sq,D], LSE [B,Hq,Sq]. */
int oracle_fwd_mod(const double* q, const double* k, const double* v, int B, int Hq, int Hkv,
                   int Sq, int Sk, int D, double scale, int wl, int wr, const double* slopes,
                   const int* seqlens_k, double* o, double* lse) {
  int rc = check_dims(B, Hq, Hkv, Sq, Sk, D);
  if (rc) return rc;
  const long total = (long)B * Hq * Sq;
#pragma omp parallel
  {
    double* s = (double*)malloc(sizeof(double) * (size_t)(Sk > 0 ? Sk : 1));
#pragma omp for schedule(dynamic, 4)
    for (long flat = 0; flat < total; ++flat) {
      const long i = flat % Sq, bh = flat / Sq;
      const long b = bh / Hq, h = bh % Hq;
      const long kvh = b * Hkv + kv_head_of((int)h, Hq, Hkv);
      long lo, hi;
      mod_key_range(i, batch_keys(seqlens_k, b, Sk), wl, wr, &lo, &hi);
      mod_fwd_row(q + flat * D, k + kvh * (long)Sk * D, v + kvh * (long)Sk * D, D, i, lo, hi,
                  scale, head_slope(slopes, h), s, o + flat * D, lse + flat);
    }
    free(s);
  }
  return 0;
}

/* Forward with the score modification for selected flat rows (b*Hq + h)*Sq + i. */
int oracle_fwd_rows_mod(const double* q, const double* k, const double* v, int B, int Hq,
                        int Hkv, int Sq, int Sk, int D, double scale, int wl, int wr,
                        const double* slopes, const int* seqlens_k, const int64_t* rows,
                        int64_t n_rows, double* o_rows, double* lse_rows) {
  int rc = check_dims(B, Hq, Hkv, Sq, Sk, D);
  if (rc) return rc;
  const long total = (long)B * Hq * Sq;
  for (int64_t r = 0; r < n_rows; ++r)
    if (rows[r] < 0 || rows[r] >= total) return -3;
#pragma omp parallel
  {
    double* s = (double*)malloc(sizeof(double) * (size_t)(Sk > 0 ? Sk : 1));
#pragma omp for schedule(dynamic, 4)
    for (int64_t r = 0; r < n_rows; ++r) {
      const long flat = (long)rows[r];
      const long i = flat % Sq, bh = flat / Sq;
      const long b = bh / Hq, h = bh % Hq;
      const long kvh = b * Hkv + kv_head_of((int)h, Hq, Hkv);
      long lo, hi;
      mod_key_range(i, batch_keys(seqlens_k, b, Sk), wl, wr, &lo, &hi);
      mod_fwd_row(q + flat * D, k + kvh * (long)Sk * D, v + kvh * (long)Sk * D, D, i, lo, hi,
                  scale, head_slope(slopes, h), s, o_rows + r * D, lse_rows + r);
    }
    free(s);
  }
  return 0;
}

/*
 * Backward with the score modification for kv-head units u = b*Hkv + hk: dK, dV
 * of the unit and dQ, O, LSE of its group's q heads.  The bias does not depend
 * on q or k, so it enters the gradients only through P.
 */
int oracle_bwd_units_mod(const double* q, const double* k, const double* v, const double* dO,
                         int B, int Hq, int Hkv, int Sq, int Sk, int D, double scale, int wl,
                         int wr, const double* slopes, const int* seqlens_k,
                         const int64_t* units, int64_t n_units, double* dq, double* dk,
                         double* dv, double* o, double* lse) {
  int rc = check_dims(B, Hq, Hkv, Sq, Sk, D);
  if (rc) return rc;
  for (int64_t u = 0; u < n_units; ++u)
    if (units[u] < 0 || units[u] >= (int64_t)B * Hkv) return -3;
  const int g = Hq / Hkv;
  double* dsum = (double*)malloc(sizeof(double) * (size_t)(Sq > 0 ? Sq : 1) * (size_t)g);
  if (!dsum) return -4;
  for (int64_t u = 0; u < n_units; ++u) {
    const long b = (long)(units[u] / Hkv), hk = (long)(units[u] % Hkv);
    const long kvh = b * Hkv + hk;
    const double* kh = k + kvh * (long)Sk * D;
    const double* vh = v + kvh * (long)Sk * D;
    /* per query row of the group: O, LSE, the row term sum_d dO O, and dQ */
    for (int gi = 0; gi < g; ++gi) {
      const long h = hk * g + gi;
      const long row0 = (b * Hq + h) * (long)Sq;
      const double slope = head_slope(slopes, h);
#pragma omp parallel
      {
        double* s = (double*)malloc(sizeof(double) * (size_t)(Sk > 0 ? Sk : 1));
#pragma omp for schedule(dynamic, 4)
        for (long i = 0; i < Sq; ++i) {
          long lo, hi;
          mod_key_range(i, batch_keys(seqlens_k, b, Sk), wl, wr, &lo, &hi);
          const double* qi = q + (row0 + i) * D;
          const double* gi_row = dO + (row0 + i) * D;
          double* oi = o + (row0 + i) * D;
          double* dqi = dq + (row0 + i) * D;
          mod_fwd_row(qi, kh, vh, D, i, lo, hi, scale, slope, s, oi, lse + row0 + i);
          const double rterm = dot(gi_row, oi, D);
          dsum[gi * (long)Sq + i] = rterm;
          for (long d = 0; d < D; ++d) dqi[d] = 0.0;
          for (long j = lo; j < hi; ++j) {
            const double w = exp(s[j] - lse[row0 + i]);
            const double g_w = w * (dot(gi_row, vh + j * D, D) - rterm);
            for (long d = 0; d < D; ++d) dqi[d] += scale * g_w * kh[j * D + d];
          }
        }
        free(s);
      }
    }
    /* per key row: dK_j, dV_j over the queries that see key j */
#pragma omp parallel for schedule(dynamic, 4)
    for (long j = 0; j < Sk; ++j) {
      double* dkj = dk + (kvh * (long)Sk + j) * D;
      double* dvj = dv + (kvh * (long)Sk + j) * D;
      for (long d = 0; d < D; ++d) dkj[d] = dvj[d] = 0.0;
      for (int gi = 0; gi < g; ++gi) {
        const long h = hk * g + gi;
        const long row0 = (b * Hq + h) * (long)Sq;
        const double slope = head_slope(slopes, h);
        for (long i = 0; i < Sq; ++i) {
          long lo, hi;
          mod_key_range(i, batch_keys(seqlens_k, b, Sk), wl, wr, &lo, &hi);
          if (j < lo || j >= hi) continue;
          const double* qi = q + (row0 + i) * D;
          const double* gi_row = dO + (row0 + i) * D;
          const double w = exp(mod_score(qi, kh + j * D, D, scale, slope, i, j) - lse[row0 + i]);
          const double g_w = w * (dot(gi_row, vh + j * D, D) - dsum[gi * (long)Sq + i]);
          for (long d = 0; d < D; ++d) {
            dkj[d] += scale * g_w * qi[d];
            dvj[d] += w * gi_row[d];
          }
        }
      }
    }
  }
  free(dsum);
  return 0;
}

/*
 * Split-KV: attention over part of the keys, and the merge of such parts.
 *
 * The FlashAttention-4 pages name sequence parallelism ("Production Deployment Guide")
 * without a mechanism; the step it rests on is the identity behind the online
 * softmax of the three phases ("The Asymmetric Hardware Scaling Wall"): the
 * softmax over a union of disjoint key sets K_1 .. K_n follows from each set's
 * own normalised output O_c and log-sum-exp LSE_c,
 *
 *     LSE = M + ln sum_c exp(LSE_c - M),   M = max_c LSE_c
 *     O   = sum_c exp(LSE_c - LSE) O_c
 *
 * An empty part has LSE_c = -inf and weight 0; a row with no non-empty part
 * gets O = 0 and LSE = -inf.
 */

/*
 * Forward with the score modification restricted to the keys [k0, k1) (window
 * and bias still use the absolute key index j).  Rows with no visible key in
 * the range get O = 0, LSE = -inf.
 */
int oracle_fwd_mod_range(const double* q, const double* k, const double* v, int B, int Hq,
                         int Hkv, int Sq, int Sk, int D, double scale, int wl, int wr,
                         const double* slopes, const int* seqlens_k, int k0, int k1, double* o,
                         double* lse) {
  int rc = check_dims(B, Hq, Hkv, Sq, Sk, D);
  if (rc) return rc;
  if (k0 < 0 || k1 < k0 || k1 > Sk) return -3;
  const long total = (long)B * Hq * Sq;
#pragma omp parallel
  {
    double* s = (double*)malloc(sizeof(double) * (size_t)(Sk > 0 ? Sk : 1));
#pragma omp for schedule(dynamic, 4)
    for (long flat = 0; flat < total; ++flat) {
      const long i = flat % Sq, bh = flat / Sq;
      const long b = bh / Hq, h = bh % Hq;
      const long kvh = b * Hkv + kv_head_of((int)h, Hq, Hkv);
      long lo, hi;
      mod_key_range(i, batch_keys(seqlens_k, b, Sk), wl, wr, &lo, &hi);
      if (lo < k0) lo = k0;
      if (hi > k1) hi = k1;
      mod_fwd_row(q + flat * D, k + kvh * (long)Sk * D, v + kvh * (long)Sk * D, D, i, lo, hi,
                  scale, head_slope(slopes, h), s, o + flat * D, lse + flat);
    }
    free(s);
  }
  return 0;
}

/*
 * Merge n parts: o_parts [n, rows, D], lse_parts [n, rows] -> o [rows, D],
 * lse [rows].
 */
int oracle_lse_merge(const double* o_parts, const double* lse_parts, int n, long rows, int D,
                     double* o, double* lse) {
  if (n < 1 || rows < 0 || D < 1) return -1;
#pragma omp parallel for schedule(static)
  for (long r = 0; r < rows; ++r) {
    double M = -INFINITY;
    for (int c = 0; c < n; ++c) M = fmax(M, lse_parts[(long)c * rows + r]);
    double* orow = o + r * D;
    for (long d = 0; d < D; ++d) orow[d] = 0.0;
    if (M == -INFINITY) {
      lse[r] = -INFINITY;
      continue;
    }
    double z = 0.0;
    for (int c = 0; c < n; ++c) z += exp(lse_parts[(long)c * rows + r] - M);
    const double row_lse = M + log(z);
    for (int c = 0; c < n; ++c) {
      const double w = exp(lse_parts[(long)c * rows + r] - row_lse);
      const double* oc = o_parts + ((long)c * rows + r) * D;
      for (long d = 0; d < D; ++d) orow[d] += w * oc[d];
    }
    lse[r] = row_lse;
  }
  return 0;
}

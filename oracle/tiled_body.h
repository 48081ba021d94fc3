/*
 * tiled_body.h -- body of the tiled online-softmax restatement, included by
 * attn_oracle.c once with REAL = double and once with REAL = float.
 * TEST INFRASTRUCTURE ONLY (see attn_oracle.c).
 *
 * Loop order follows the FlashAttention-4 pages' simulator ("End-to-End
 * Implementation: Simulating the FA4 Pipelined Tiling Algorithm"): for every
 * query tile, walk the key/value tiles; per tile form the scaled scores, mask
 * (causal q_idx >= kv_idx), take the tile's row max, update the running max m,
 * exponentiate, rescale the running sum l and accumulator, add P.V; at the end
 * divide by l.
 *
 * mode 0 -- the simulator as printed: natural exp, rescale on every tile.
 * mode 1 -- conditional rescale (key contribution #2): scores in base 2
 *           (t = s*log2 e); the running max moves only when the tile's max
 *           exceeds it by more than `threshold` (8.0 = log2 256); otherwise the
 *           stale max is kept and P = 2^(t - m) may reach 2^threshold.  The
 *           first tile always sets m.  LSE = ln2 * (m + log2 l) with the same
 *           (possibly stale) m, which is exact.
 *
 * Causal tile skip: a kv tile starting at or after the query tile's exclusive
 * end is skipped (the printed loop skips only when it starts strictly after;
 * the extra tile it keeps is fully masked and changes nothing).
 *
 * Counters: n_rescaled counts (row, tile) steps where the running max had been
 * set and the accumulator was rescaled; n_skipped counts steps in mode 1 where
 * the tile max grew the running max by a positive amount no larger than the
 * threshold, so the rescale was skipped.
 */
int TILED_NAME(const double* q, const double* k, const double* v, int B, int Hq, int Hkv, int Sq,
               int Sk, int D, int causal, double scale, int block_q, int block_kv, int mode,
               double threshold, double* o, double* lse, int64_t* n_rescaled,
               int64_t* n_skipped) {
  int rc = check_dims(B, Hq, Hkv, Sq, Sk, D);
  if (rc) return rc;
  if (block_q < 1 || block_kv < 1 || (mode != 0 && mode != 1)) return -5;
  const REAL log2e = (REAL)1.4426950408889634;
  const REAL ln2 = (REAL)0.6931471805599453;
  int64_t cnt_rescaled = 0, cnt_skipped = 0;

#pragma omp parallel for schedule(dynamic, 1) reduction(+ : cnt_rescaled, cnt_skipped)
  for (long bh = 0; bh < (long)B * Hq; ++bh) {
    const long b = bh / Hq, h = bh % Hq;
    const long hk = kv_head_of((int)h, Hq, Hkv);
    const double* k_head = k + ((b * Hkv + hk) * (long)Sk) * D;
    const double* v_head = v + ((b * Hkv + hk) * (long)Sk) * D;
    REAL* m = (REAL*)malloc(sizeof(REAL) * (size_t)block_q);
    REAL* l = (REAL*)malloc(sizeof(REAL) * (size_t)block_q);
    REAL* acc = (REAL*)malloc(sizeof(REAL) * (size_t)block_q * (size_t)D);
    REAL* st = (REAL*)malloc(sizeof(REAL) * (size_t)block_q * (size_t)block_kv);

    for (long q0 = 0; q0 < Sq; q0 += block_q) {
      const long q1 = (q0 + block_q < Sq) ? q0 + block_q : Sq;
      const long nq = q1 - q0;
      for (long r = 0; r < nq; ++r) {
        m[r] = -INFINITY;
        l[r] = 0;
        for (long d = 0; d < D; ++d) acc[r * D + d] = 0;
      }
      for (long k0 = 0; k0 < Sk; k0 += block_kv) {
        const long k1 = (k0 + block_kv < Sk) ? k0 + block_kv : Sk;
        if (causal && k0 >= q1) continue;
        const long nk = k1 - k0;
        for (long r = 0; r < nq; ++r) {
          const long i = q0 + r;
          const double* qi = q + ((bh * Sq) + i) * D;
          REAL* srow = st + r * block_kv;
          REAL tile_max = -INFINITY;
          /* GEMM 1 and the mask */
          for (long c = 0; c < nk; ++c) {
            const long j = k0 + c;
            REAL sv;
            if (causal && j > i) {
              sv = -INFINITY;
            } else {
              REAL dotv = 0;
              const double* kj = k_head + j * D;
              for (long d = 0; d < D; ++d) dotv += (REAL)qi[d] * (REAL)kj[d];
              sv = (REAL)scale * dotv;
              if (mode == 1) sv = sv * log2e;
            }
            srow[c] = sv;
            if (sv > tile_max) tile_max = sv;
          }
          /* online softmax update */
          REAL alpha = 1;
          if (tile_max == -INFINITY) {
            /* fully masked for this row: contributes nothing */
            for (long c = 0; c < nk; ++c) srow[c] = 0;
            continue;
          }
          if (mode == 0) {
            const REAL new_m = (tile_max > m[r]) ? tile_max : m[r];
            alpha = (m[r] == -INFINITY) ? (REAL)0 : EXP(m[r] - new_m);
            if (m[r] != -INFINITY) ++cnt_rescaled;
            m[r] = new_m;
            for (long c = 0; c < nk; ++c) srow[c] = EXP(srow[c] - new_m);
          } else {
            if (m[r] == -INFINITY) {
              alpha = 0;
              m[r] = tile_max;
            } else if (tile_max - m[r] > (REAL)threshold) {
              alpha = EXP2(m[r] - tile_max);
              m[r] = tile_max;
              ++cnt_rescaled;
            } else if (tile_max > m[r]) {
              ++cnt_skipped;
            }
            for (long c = 0; c < nk; ++c) srow[c] = EXP2(srow[c] - m[r]);
          }
          REAL tile_l = 0;
          for (long c = 0; c < nk; ++c) tile_l += srow[c];
          l[r] = l[r] * alpha + tile_l;
          /* GEMM 2 */
          for (long d = 0; d < D; ++d) {
            REAL pv = 0;
            for (long c = 0; c < nk; ++c) pv += srow[c] * (REAL)v_head[(k0 + c) * D + d];
            acc[r * D + d] = acc[r * D + d] * alpha + pv;
          }
        }
      }
      for (long r = 0; r < nq; ++r) {
        const long flat = bh * Sq + q0 + r;
        for (long d = 0; d < D; ++d) o[flat * D + d] = (double)(acc[r * D + d] / l[r]);
        if (mode == 0)
          lse[flat] = (double)(m[r] + LOG(l[r]));
        else
          lse[flat] = (double)(ln2 * (m[r] + LOG2(l[r])));
      }
    }
    free(m);
    free(l);
    free(acc);
    free(st);
  }
  if (n_rescaled) *n_rescaled = cnt_rescaled;
  if (n_skipped) *n_skipped = cnt_skipped;
  return 0;
}

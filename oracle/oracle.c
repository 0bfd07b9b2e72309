/*
 * fp64 CPU oracle for softmax-threshold block skipping.
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the package's smoke check and the
 * CPU-baseline leg of the benchmark load this library.  It shares no code,
 * header or constant with the CUDA path, and the CUDA path never calls it.
 *
 * Source: the web page "BLASST：一个标量阈值实现的动态块稀疏注意力（MLSys 2026）"
 * (BLASST, arXiv 2512.12087), sections
 *   "铺垫：FlashAttention 的在线 softmax"  -- the online-softmax tile loop, Eqs. (2)-(4);
 *   "BLASST 的判定准则"                    -- the skip test, Eq. (5);
 *   "判定本身：几乎零成本的秘密"            -- a tile skips only when all its rows agree;
 *   "Decode 内核：砍带宽"                   -- decode skips the value load of a skipped block;
 * and FlashDecoding's split-KV merge (the SANTA page, "FlashDecoding" baseline).
 * The sampled decode output at the end of this file follows the web page
 * "Stochastic Sparse Attention for Memory-Bound Inference" (SANTA), section
 * "关键设计" (the unbiased estimator and its stratified / systematic forms).
 *
 * Arithmetic: every input is an fp32 array holding exactly the values the GPU
 * reads (bf16 inputs are widened exactly); all arithmetic is fp64, in the
 * order the page's algorithm states.  Scores are the SCALED dot products
 * s = scale * <q, k>; logs are natural.
 *
 * Readings where the page is silent or its equations were lost (each one is
 * also listed in the design notes):
 *   - the test compares the block's row max with the UPDATED running max and is
 *     strict: skip iff  rowmax(S_ij) - m_new < ln(lambda);  lambda = 0 never skips;
 *   - a row with no visible key in the block has rowmax = -inf and votes "skip";
 *   - prefill: a block is skipped iff every valid row of the query tile votes skip;
 *     decode: iff every query head sharing the KV head votes skip;
 *   - causal masking is top-left with T_q = T_k: key c is visible to row r iff c <= r,
 *     and blocks past the tile's last row are not traversed (bit 0, margin NaN);
 *   - decode split s owns blocks [floor(s*nb/n), floor((s+1)*nb/n)) and restarts its
 *     running max at -inf; an empty split has LSE = -inf and O = 0;
 *   - the running max is updated on skipped blocks too (it cannot change there).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define NEG_INF (-INFINITY)

static double dot_f32(const float *a, const float *b, int n) {
  double acc = 0.0;
  for (int i = 0; i < n; ++i) acc += (double)a[i] * (double)b[i];
  return acc;
}

int bsa_oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* ------------------------------------------------------------------------ */
/* Dense softmax attention: the plain definition y = softmax(s) V, with      */
/* M = max s, Z = sum exp(s - M), LSE = M + ln Z, over all visible keys.     */
/* ------------------------------------------------------------------------ */

/* q:[B,Hq,T,dk] k:[B,Hkv,T,dk] v:[B,Hkv,T,dv]; rows = flat indices into
 * [B,Hq,T] (NULL = all); y:[B,Hq,T,dv], lse:[B,Hq,T]. */
int bsa_oracle_dense_prefill(const float *q, const float *k, const float *v, int B, int Hq,
                             int Hkv, int T, int dk, int dv, double scale, int causal,
                             const int64_t *rows, int64_t n_rows, double *y, double *lse) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || T <= 0 || dk <= 0 || dv <= 0 || Hq % Hkv) return -1;
  const int G = Hq / Hkv;
  const int64_t total = rows ? n_rows : (int64_t)B * Hq * T;
#pragma omp parallel
  {
    double *s = (double *)malloc(sizeof(double) * (size_t)T);
#pragma omp for schedule(dynamic, 16)
    for (int64_t it = 0; it < total; ++it) {
      const int64_t idx = rows ? rows[it] : it;
      const int r = (int)(idx % T);
      const int h = (int)((idx / T) % Hq);
      const int b = (int)(idx / ((int64_t)T * Hq));
      const int hk = h / G;
      const float *qr = q + (((int64_t)b * Hq + h) * T + r) * dk;
      const float *kb = k + ((int64_t)b * Hkv + hk) * T * dk;
      const float *vb = v + ((int64_t)b * Hkv + hk) * T * dv;
      const int nvis = causal ? r + 1 : T;
      double M = NEG_INF;
      for (int c = 0; c < nvis; ++c) {
        s[c] = scale * dot_f32(qr, kb + (int64_t)c * dk, dk);
        if (s[c] > M) M = s[c];
      }
      double Z = 0.0;
      for (int c = 0; c < nvis; ++c) Z += exp(s[c] - M);
      double *yr = y + idx * dv;
      for (int e = 0; e < dv; ++e) yr[e] = 0.0;
      for (int c = 0; c < nvis; ++c) {
        const double p = exp(s[c] - M) / Z;
        const float *vc = vb + (int64_t)c * dv;
        for (int e = 0; e < dv; ++e) yr[e] += p * (double)vc[e];
      }
      lse[idx] = M + log(Z);
    }
    free(s);
  }
  return 0;
}

/* Decode: q:[B,Hq,dk]; key c of (b,hk) at k + ((b*Hkv+hk)*L + c)*k_row_stride, value at
 * v + ((b*Hkv+hk)*L + c)*v_row_stride.  y:[B,Hq,dv], lse:[B,Hq]. */
int bsa_oracle_dense_decode(const float *q, const float *k, const float *v, int B, int Hq,
                            int Hkv, int L, int dk, int dv, int64_t k_row_stride,
                            int64_t v_row_stride, double scale, double *y, double *lse) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || L <= 0 || dk <= 0 || dv <= 0 || Hq % Hkv) return -1;
  const int G = Hq / Hkv;
#pragma omp parallel
  {
    double *s = (double *)malloc(sizeof(double) * (size_t)L);
#pragma omp for schedule(dynamic, 1)
    for (int64_t idx = 0; idx < (int64_t)B * Hq; ++idx) {
      const int h = (int)(idx % Hq), b = (int)(idx / Hq), hk = h / G;
      const float *qr = q + idx * dk;
      const int64_t base = ((int64_t)b * Hkv + hk) * L;
      double M = NEG_INF;
      for (int c = 0; c < L; ++c) {
        s[c] = scale * dot_f32(qr, k + (base + c) * k_row_stride, dk);
        if (s[c] > M) M = s[c];
      }
      double Z = 0.0;
      for (int c = 0; c < L; ++c) Z += exp(s[c] - M);
      double *yr = y + idx * dv;
      for (int e = 0; e < dv; ++e) yr[e] = 0.0;
      for (int c = 0; c < L; ++c) {
        const double p = exp(s[c] - M) / Z;
        const float *vc = v + (base + c) * v_row_stride;
        for (int e = 0; e < dv; ++e) yr[e] += p * (double)vc[e];
      }
      lse[idx] = M + log(Z);
    }
    free(s);
  }
  return 0;
}

/* ------------------------------------------------------------------------ */
/* The thresholded online-softmax loop over one group of query rows.         */
/* ------------------------------------------------------------------------ */

/* State of the loop for nr query rows: running max m, row sum l, output acc. */
typedef struct {
  int nr, dv;
  double *m, *l, *acc;
  double *s;    /* nr x Bc scores of the current block */
  double *mt;   /* per-row block max  rowmax(S_ij)     */
  double *mnew; /* per-row updated running max          */
} loop_state;

static void state_init(loop_state *st, int nr, int Bc, int dv) {
  st->nr = nr;
  st->dv = dv;
  st->m = (double *)malloc(sizeof(double) * nr);
  st->l = (double *)calloc((size_t)nr, sizeof(double));
  st->acc = (double *)calloc((size_t)nr * dv, sizeof(double));
  st->s = (double *)malloc(sizeof(double) * (size_t)nr * Bc);
  st->mt = (double *)malloc(sizeof(double) * nr);
  st->mnew = (double *)malloc(sizeof(double) * nr);
  for (int r = 0; r < nr; ++r) st->m[r] = NEG_INF; /* m^(0) = -inf, l^(0) = 0, O^(0) = 0 */
}

static void state_free(loop_state *st) {
  free(st->m); free(st->l); free(st->acc); free(st->s); free(st->mt); free(st->mnew);
}

/* One step j of the loop, once st->s holds S_ij for the block's nc keys (masked
 * scores are -inf).  Returns 1 if the block is skipped.  *margin receives the
 * tile statistic max_r (rowmax_r - m_new_r): the block is skipped iff that
 * statistic is below ln(lambda) (and lambda > 0).  forced >= 0 replaces the
 * decision by the caller's (0 keep, 1 skip); the arithmetic is unchanged. */
static int loop_step(loop_state *st, int nc, int Bc, const float *vblk, int64_t v_row_stride,
                     double lambda, double ln_lambda, int forced, double *margin) {
  const int nr = st->nr, dv = st->dv;
  double mu = NEG_INF;
  int all_vote_skip = 1;
  for (int r = 0; r < nr; ++r) {
    const double *sr = st->s + (size_t)r * Bc;
    double mt = NEG_INF;                     /* block row max, rowmax(S_ij) */
    for (int c = 0; c < nc; ++c) if (sr[c] > mt) mt = sr[c];
    const double mnew = st->m[r] > mt ? st->m[r] : mt; /* updated running max m^(j) */
    st->mt[r] = mt;
    st->mnew[r] = mnew;
    /* Eq. (5): the difference is taken against the updated running max. */
    const double diff = (mt == NEG_INF) ? NEG_INF : mt - mnew;
    if (diff > mu) mu = diff;
    const int vote = (lambda > 0.0) && (diff < ln_lambda);
    if (!vote) all_vote_skip = 0;
  }
  *margin = mu;
  if (forced >= 0) all_vote_skip = forced;
  if (!all_vote_skip) {
    /* Eqs. (2)-(4): rescale the history to the new max, add this block. */
    for (int r = 0; r < nr; ++r) {
      const double mnew = st->mnew[r];
      const double alpha = (st->m[r] == NEG_INF) ? 0.0 : exp(st->m[r] - mnew);
      double *accr = st->acc + (size_t)r * dv;
      double rowsum = 0.0;
      for (int e = 0; e < dv; ++e) accr[e] *= alpha;
      const double *sr = st->s + (size_t)r * Bc;
      for (int c = 0; c < nc; ++c) {
        if (sr[c] == NEG_INF) continue;
        const double p = exp(sr[c] - mnew);
        rowsum += p;
        const float *vc = vblk + (int64_t)c * v_row_stride;
        for (int e = 0; e < dv; ++e) accr[e] += p * (double)vc[e];
      }
      st->l[r] = alpha * st->l[r] + rowsum;
    }
  }
  /* The running max always advances; on a skipped block mt < m so it is unchanged. */
  for (int r = 0; r < nr; ++r) st->m[r] = st->mnew[r];
  return !all_vote_skip ? 0 : 1;
}

/* Prefill.  q:[B,Hq,T,dk], k:[B,Hkv,T,dk], v:[B,Hkv,T,dv] (fp32), query head h reads
 * KV head h / (Hq/Hkv).  units: flat indices into [B,Hq,n_t] (NULL = all).
 * Outputs (only the chosen units' entries are written):
 *   o:[B,Hq,T,dv], lse:[B,Hq,T]   final O = acc / l and LSE = m + ln l;
 *   skip:[B,Hq,n_t,n_b] (1 = skipped), margin:[B,Hq,n_t,n_b] (NaN = not traversed).
 * force_skip (NULL = none), same layout as skip: the decisions to take instead of
 * the test's, for evaluating the loop under another valid set of decisions.
 * allow (NULL = every block), same layout as skip: an explicit block set per
 * query tile (the SparDA page, section 2.1: an access set such as
 * B_init u B_local u B_topk); blocks outside it are not traversed -- no scores,
 * no running-max update, skip 0, margin NaN -- and the threshold test applies
 * among the blocks inside it.  A row with no visible key in its tile's set gets
 * O = 0 and LSE = -inf (no mass at all). */
int bsa_oracle_prefill(const float *q, const float *k, const float *v, int B, int Hq, int Hkv,
                       int T, int dk, int dv, double scale, double lambda, int Br, int Bc,
                       int causal, const int64_t *units, int64_t n_units,
                       const uint8_t *force_skip, const uint8_t *allow, double *o, double *lse,
                       uint8_t *skip, double *margin) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || T <= 0 || dk <= 0 || dv <= 0 || Br <= 0 || Bc <= 0 ||
      Hq % Hkv || !(lambda >= 0.0 && lambda < 1.0))
    return -1;
  const int G = Hq / Hkv;
  const int n_t = (T + Br - 1) / Br, n_b = (T + Bc - 1) / Bc;
  const double ln_lambda = lambda > 0.0 ? log(lambda) : NEG_INF;
  const int64_t total = units ? n_units : (int64_t)B * Hq * n_t;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t it = 0; it < total; ++it) {
    const int64_t u = units ? units[it] : it;
    const int t = (int)(u % n_t);
    const int h = (int)((u / n_t) % Hq);
    const int b = (int)(u / ((int64_t)n_t * Hq));
    const int hk = h / G;
    const int r0 = t * Br, r1 = (r0 + Br < T) ? r0 + Br : T, nr = r1 - r0;
    const float *qb = q + ((int64_t)b * Hq + h) * T * dk;
    const float *kb = k + ((int64_t)b * Hkv + hk) * T * dk;
    const float *vb = v + ((int64_t)b * Hkv + hk) * T * dv;
    uint8_t *sk = skip + u * n_b;
    double *mg = margin + u * n_b;
    const int jmax = causal ? (r1 - 1) / Bc : n_b - 1;
    for (int j = 0; j < n_b; ++j) { sk[j] = 0; mg[j] = NAN; }
    loop_state st;
    state_init(&st, nr, Bc, dv);
    for (int j = 0; j <= jmax; ++j) { /* KV blocks in ascending order */
      if (allow && !allow[u * n_b + j]) continue; /* outside the tile's block set */
      const int c0 = j * Bc, c1 = (c0 + Bc < T) ? c0 + Bc : T, nc = c1 - c0;
      for (int r = 0; r < nr; ++r) {
        const int row = r0 + r;
        for (int c = 0; c < nc; ++c) {
          const int col = c0 + c;
          st.s[(size_t)r * Bc + c] = (causal && col > row)
              ? NEG_INF
              : scale * dot_f32(qb + (int64_t)row * dk, kb + (int64_t)col * dk, dk);
        }
      }
      const int forced = force_skip ? (int)force_skip[u * n_b + j] : -1;
      sk[j] = (uint8_t)loop_step(&st, nc, Bc, vb + (int64_t)c0 * dv, dv, lambda, ln_lambda,
                                 forced, &mg[j]);
    }
    for (int r = 0; r < nr; ++r) {
      const int64_t orow = ((int64_t)b * Hq + h) * T + r0 + r;
      const int empty = !(st.l[r] > 0.0); /* no visible key in the block set */
      for (int e = 0; e < dv; ++e) o[orow * dv + e] = empty ? 0.0 : st.acc[(size_t)r * dv + e] / st.l[r];
      lse[orow] = empty ? NEG_INF : st.m[r] + log(st.l[r]);
    }
    state_free(&st);
  }
  return 0;
}

/* Split-KV decode, one query token per sequence.  q:[B,Hq,dk]; key c of (b,hk) at
 * k + ((b*Hkv+hk)*L + c)*k_row_stride, value at v + (...)*v_row_stride (an absorbed
 * latent cache passes v == k).  The G query heads of a KV head form one group.
 * units: flat indices into [B,Hkv,n_splits] (NULL = all).  Outputs:
 *   o_part:[B,Hq,n_splits,dv], lse_part:[B,Hq,n_splits] (-inf for an empty split);
 *   skip, margin:[B,Hkv,n_splits,bps] with bps = ceil(n_b/n_splits), block j of split s
 *   at position j - floor(s*n_b/n_splits).
 * force_skip (NULL = none), same layout as skip: decisions to take instead of the test's.
 * per_head != 0: each query head decides for itself instead of the G heads ANDing their
 * votes (the per-head variant of the group reading); skip, margin and force_skip are then
 * [B,Hq,n_splits,bps]. */
int bsa_oracle_decode(const float *q, const float *k, const float *v, int B, int Hq, int Hkv,
                      int L, int dk, int dv, int64_t k_row_stride, int64_t v_row_stride,
                      double scale, double lambda, int Bc, int n_splits, const int64_t *units,
                      int64_t n_units, const uint8_t *force_skip, int per_head, double *o_part,
                      double *lse_part, uint8_t *skip, double *margin) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || L <= 0 || dk <= 0 || dv <= 0 || Bc <= 0 ||
      n_splits <= 0 || Hq % Hkv || !(lambda >= 0.0 && lambda < 1.0))
    return -1;
  const int G = Hq / Hkv;
  const int n_b = (L + Bc - 1) / Bc;
  const int bps = (n_b + n_splits - 1) / n_splits;
  const double ln_lambda = lambda > 0.0 ? log(lambda) : NEG_INF;
  const int64_t total = units ? n_units : (int64_t)B * Hkv * n_splits;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t it = 0; it < total; ++it) {
    const int64_t u = units ? units[it] : it;
    const int sp = (int)(u % n_splits);
    const int hk = (int)((u / n_splits) % Hkv);
    const int b = (int)(u / ((int64_t)n_splits * Hkv));
    const int j0 = (int)((int64_t)sp * n_b / n_splits);
    const int j1 = (int)((int64_t)(sp + 1) * n_b / n_splits);
    const int64_t base = ((int64_t)b * Hkv + hk) * L;
    if (per_head) {
      /* Each query head is its own decision unit (one row): its own skip
       * decisions, statistic and bits, rows of skip/margin [B,Hq,n_splits,bps]. */
      for (int g = 0; g < G; ++g) {
        const int64_t hrow = ((int64_t)b * Hq + hk * G + g) * n_splits + sp;
        uint8_t *skh = skip + hrow * bps;
        double *mgh = margin + hrow * bps;
        for (int j = 0; j < bps; ++j) { skh[j] = 0; mgh[j] = NAN; }
        loop_state st;
        state_init(&st, 1, Bc, dv);
        const float *qr = q + ((int64_t)b * Hq + hk * G + g) * dk;
        for (int j = j0; j < j1; ++j) {
          const int c0 = j * Bc, c1 = (c0 + Bc < L) ? c0 + Bc : L, nc = c1 - c0;
          for (int c = 0; c < nc; ++c)
            st.s[c] = scale * dot_f32(qr, k + (base + c0 + c) * k_row_stride, dk);
          const int forced = force_skip ? (int)force_skip[hrow * bps + (j - j0)] : -1;
          skh[j - j0] = (uint8_t)loop_step(&st, nc, Bc, v + (base + c0) * v_row_stride,
                                           v_row_stride, lambda, ln_lambda, forced,
                                           &mgh[j - j0]);
        }
        if (j1 == j0) { /* empty split */
          for (int e = 0; e < dv; ++e) o_part[hrow * dv + e] = 0.0;
          lse_part[hrow] = NEG_INF;
        } else {
          for (int e = 0; e < dv; ++e) o_part[hrow * dv + e] = st.acc[e] / st.l[0];
          lse_part[hrow] = st.m[0] + log(st.l[0]);
        }
        state_free(&st);
      }
      continue;
    }
    uint8_t *sk = skip + u * bps;
    double *mg = margin + u * bps;
    for (int j = 0; j < bps; ++j) { sk[j] = 0; mg[j] = NAN; }
    loop_state st;
    state_init(&st, G, Bc, dv);
    for (int j = j0; j < j1; ++j) {
      const int c0 = j * Bc, c1 = (c0 + Bc < L) ? c0 + Bc : L, nc = c1 - c0;
      for (int g = 0; g < G; ++g) {
        const float *qr = q + ((int64_t)b * Hq + hk * G + g) * dk;
        for (int c = 0; c < nc; ++c)
          st.s[(size_t)g * Bc + c] = scale * dot_f32(qr, k + (base + c0 + c) * k_row_stride, dk);
      }
      const int forced = force_skip ? (int)force_skip[u * bps + (j - j0)] : -1;
      sk[j - j0] = (uint8_t)loop_step(&st, nc, Bc, v + (base + c0) * v_row_stride,
                                      v_row_stride, lambda, ln_lambda, forced, &mg[j - j0]);
    }
    for (int g = 0; g < G; ++g) {
      const int64_t row = ((int64_t)b * Hq + hk * G + g) * n_splits + sp;
      if (j1 == j0) { /* empty split */
        for (int e = 0; e < dv; ++e) o_part[row * dv + e] = 0.0;
        lse_part[row] = NEG_INF;
      } else {
        for (int e = 0; e < dv; ++e) o_part[row * dv + e] = st.acc[(size_t)g * dv + e] / st.l[g];
        lse_part[row] = st.m[g] + log(st.l[g]);
      }
    }
    state_free(&st);
  }
  return 0;
}

/* Merge of split partials by their log-sum-exp: LSE = ln sum_s exp(LSE_s) and
 * O = sum_s exp(LSE_s - LSE) O_s.  Empty splits (LSE_s = -inf) weigh zero. */
int bsa_oracle_combine(const double *o_part, const double *lse_part, int B, int Hq, int n_splits,
                       int dv, double *o, double *lse) {
  if (B <= 0 || Hq <= 0 || n_splits <= 0 || dv <= 0) return -1;
  for (int64_t idx = 0; idx < (int64_t)B * Hq; ++idx) {
    const double *ls = lse_part + idx * n_splits;
    double M = NEG_INF;
    for (int s = 0; s < n_splits; ++s) if (ls[s] > M) M = ls[s];
    double *orow = o + idx * dv;
    for (int e = 0; e < dv; ++e) orow[e] = 0.0;
    if (M == NEG_INF) { lse[idx] = NEG_INF; continue; }
    double Z = 0.0;
    for (int s = 0; s < n_splits; ++s) Z += exp(ls[s] - M);
    const double LSE = M + log(Z);
    for (int s = 0; s < n_splits; ++s) {
      if (ls[s] == NEG_INF) continue;
      const double w = exp(ls[s] - LSE);
      const double *op = o_part + (idx * n_splits + s) * dv;
      for (int e = 0; e < dv; ++e) orow[e] += w * op[e];
    }
    lse[idx] = LSE;
  }
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Sampled attention output for one decode token: the web page "Stochastic   */
/* Sparse Attention for Memory-Bound Inference" (SANTA), section "关键设计",  */
/* items "SANTA 无偏估计 + Stratified/Systematic 降方差" and "S²ANTA-prop"    */
/* (the sampling that the kernel's second pass carries out).                */
/*                                                                          */
/* The attention weights of a query over its L keys form a categorical      */
/* distribution p_i = exp(s_i - M) / Z.  With the cumulative weights         */
/* W_i = sum_{j<=i} exp(s_j - M) (so W_{L-1} = Z), the inverse CDF of a      */
/* threshold T in [0, 1) is the smallest i with W_i > T * Z.  The estimate   */
/* of p V is the mean of the S value rows V_{J_m}, J_m the inverse CDF of   */
/* threshold T_m:                                                           */
/*   mode 0 (SANTA, i.i.d.):      T_m = u[b,h,m]                            */
/*   mode 1 (S²ANTA-sys):         T_m = (m + u[b,h]) / S   (one offset; the  */
/*                                page's U ~ Unif[0,1/S) is u / S)           */
/*   mode 2 (S²ANTA-strat):       T_m = (m + u[b,h,m]) / S (one uniform     */
/*                                draw inside each of the S equal-mass strata)*/
/* with every u in [0, 1).  Outputs: y [B,Hq,dv] = (1/S) sum_m V_{J_m};      */
/* idx [B,Hq,S] = J_m; gap [B,Hq,S] = the distance, in probability units,   */
/* from T_m to the nearer end of J_m's interval [W_{J-1}, W_J) / Z; and,     */
/* when cdf is not NULL, cdf [B,Hq,L] = W_i / Z.                             */
/* A threshold that rounds to T*Z >= Z (possible only within rounding of 1) */
/* takes the last key of positive weight.                                   */
/* Returns -1 on invalid shapes, mode, or a u outside [0, 1).               */
/* ------------------------------------------------------------------------ */
static int64_t first_above(const double *W, int64_t n, double R, int strict) {
  /* Bisection for the smallest i in [0, n) with W_i > R (strict) or W_i >= R;
   * W is nondecreasing.  Returns n when no element qualifies. */
  int64_t lo = 0, hi = n;
  while (lo < hi) {
    const int64_t mid = lo + (hi - lo) / 2;
    const int ok = strict ? (W[mid] > R) : (W[mid] >= R);
    if (ok) hi = mid; else lo = mid + 1;
  }
  return lo;
}

int bsa_oracle_santa_decode(const float *q, const float *k, const float *v, int B, int Hq,
                            int Hkv, int L, int dk, int dv, int64_t k_row_stride,
                            int64_t v_row_stride, double scale, int S, int mode,
                            const float *u, double *y, int32_t *idx, double *gap, double *cdf) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || L <= 0 || dk <= 0 || dv <= 0 || Hq % Hkv || S <= 0)
    return -1;
  if (mode < 0 || mode > 2 || !u) return -1;
  const int64_t n_u = (int64_t)B * Hq * (mode == 1 ? 1 : S);
  for (int64_t i = 0; i < n_u; ++i)
    if (!(u[i] >= 0.0f && u[i] < 1.0f)) return -1;
  const int G = Hq / Hkv;
#pragma omp parallel
  {
    double *W = (double *)malloc(sizeof(double) * (size_t)L);
#pragma omp for schedule(dynamic, 1)
    for (int64_t bh = 0; bh < (int64_t)B * Hq; ++bh) {
      const int h = (int)(bh % Hq), b = (int)(bh / Hq), hk = h / G;
      const float *qr = q + bh * dk;
      const int64_t base = ((int64_t)b * Hkv + hk) * L;
      /* Scores s_i, then W_i = running sum of exp(s_i - M) in key order. */
      double M = NEG_INF;
      for (int c = 0; c < L; ++c) {
        W[c] = scale * dot_f32(qr, k + (base + c) * k_row_stride, dk);
        if (W[c] > M) M = W[c];
      }
      double run = 0.0;
      for (int c = 0; c < L; ++c) {
        run += exp(W[c] - M);
        W[c] = run;
      }
      const double Z = run;
      if (cdf)
        for (int c = 0; c < L; ++c) cdf[bh * L + c] = W[c] / Z;
      double *yr = y + bh * dv;
      for (int e = 0; e < dv; ++e) yr[e] = 0.0;
      for (int m = 0; m < S; ++m) {
        double T;
        if (mode == 0) T = (double)u[bh * S + m];
        else if (mode == 1) T = ((double)m + (double)u[bh]) / S;
        else T = ((double)m + (double)u[bh * S + m]) / S;
        const double R = T * Z;
        int64_t J = first_above(W, L, R, 1);
        if (J == L) J = first_above(W, L, Z, 0); /* R rounded up to Z */
        const double lo = J > 0 ? W[J - 1] : 0.0, hi = W[J];
        double g = fmin(hi - R, R - lo) / Z;
        if (g < 0.0) g = 0.0;
        idx[bh * S + m] = (int32_t)J;
        gap[bh * S + m] = g;
        const float *vr = v + (base + J) * v_row_stride;
        for (int e = 0; e < dv; ++e) yr[e] += (double)vr[e];
      }
      for (int e = 0; e < dv; ++e) yr[e] /= S;
    }
    free(W);
  }
  return 0;
}

/*
 * oracle.c -- plain fp64 CPU reference for masked attention (forward and
 * backward) with a per-head attention sink and GQA head sharing.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the oracle that the CUDA path is
 * compared against.  Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may load it.  It shares no code, header, table or constant
 * with the CUDA library, and the CUDA library never calls it.
 *
 * What it computes (sources are the pages this project restates):
 *   - tilelang-ascend PR #1 "Add GQA Sink Backward BHSD", Summary ("online
 *     softmax with attention sink + sliding window mask") and the commit notes
 *     of the 2-kernel design: Phase0 Delta = sum(O*dO), a KV loop of five
 *     contractions + softmax + dS, Phase5 dSink.
 *   - cannbot-knowledge PR #174, BlockSparseAttentionGrad runbook:
 *     task features (uint8 block mask [B,N,ceil(Sq/bx),ceil(Skv/by)], bx and by
 *     independent and not necessarily dividing S) and the precision notes
 *     (p = exp(s - lse), ds = p * (dp - delta); lse/delta given in fp32; a row
 *     with no visible key yields zeros, no division in the backward).
 *
 * Everything is the plain definition, evaluated in double precision, one
 * output row (or column) at a time:
 *
 *   s_ij    = scale * <q_i, k_j>                 (only where vis(i,j))
 *   m_i     = max(max_j s_ij, sink_h)            (sink term only if present)
 *   l_i     = sum_j exp(s_ij - m_i) + exp(sink_h - m_i)
 *   LSE_i   = m_i + log(l_i)          (no visible key and no sink: +inf)
 *   O_i     = sum_j exp(s_ij - LSE_i) v_j
 *
 *   variable lengths (optional per-batch lengths Lq[b] <= Sq, Lk[b] <= Skv):
 *   rows i >= Lq[b] and keys j >= Lk[b] are outside the problem -- no pair
 *   with either is visible, such a row has O = 0, LSE = +inf, Delta = 0 and
 *   no part in dSink, whatever O, dO and LSE the caller passes for it.
 *
 *   backward, given O_in, LSE_in (whatever the caller passes):
 *   Delta_i = <dO_i, O_in_i>
 *   P_ij    = exp(s_ij - LSE_in_i),  dP_ij = <dO_i, v_j>
 *   dS_ij   = P_ij (dP_ij - Delta_i)
 *   dQ_i    = scale * sum_j dS_ij k_j
 *   dK_j    = scale * sum_{h in group(c)} sum_i dS_ij q_i
 *   dV_j    =         sum_{h in group(c)} sum_i P_ij dO_i
 *   dSink_h = - sum_b sum_i exp(sink_h - LSE_in_i) Delta_i
 *
 * The sink is an extra logit whose value row is zero: it joins only the
 * softmax denominator.  q-head h reads kv-head floor(h / (Hq/Hkv)).
 *
 * Layout: every tensor is contiguous row-major; q, O, dO, dQ are
 * [B,Hq,Sq,D]; k, v, dK, dV are [B,Hkv,Skv,D]; LSE and Delta are [B,Hq,Sq].
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

enum {
  OM_MASK_NONE = 0,
  OM_MASK_CAUSAL = 1,
  OM_MASK_SLIDING = 2, /* causal and i - j < window */
  OM_MASK_BLOCK = 3,   /* uint8 block mask [B,Hq,ceil(Sq/bx),ceil(Skv/by)] */
  OM_MASK_TOKEN = 4    /* uint8 token mask [B,Hq,Sq,Skv] (pins only) */
};

typedef struct {
  int64_t B, Hq, Hkv, Sq, Skv, D;
  int64_t mask_kind;
  int64_t window;
  int64_t bx, by;
  const uint8_t* block_mask;
  const uint8_t* token_mask;
  const double* sink; /* [Hq] or NULL for "no sink" */
  double scale;
  const int64_t* seqlen_q; /* [B] valid query rows per batch, or NULL (= Sq) */
  const int64_t* seqlen_k; /* [B] valid keys per batch, or NULL (= Skv) */
} om_problem;

/* Valid rows / keys of batch b (lengths outside [0, S] are clamped). */
static int64_t om_len(const int64_t* len, int64_t b, int64_t S) {
  if (!len) return S;
  return len[b] < 0 ? 0 : (len[b] > S ? S : len[b]);
}

/* Token-level visibility of key j for query i of (b, h). */
static int om_visible(const om_problem* p, int64_t b, int64_t h, int64_t i,
                      int64_t j) {
  if (i >= om_len(p->seqlen_q, b, p->Sq) || j >= om_len(p->seqlen_k, b, p->Skv)) return 0;
  switch (p->mask_kind) {
    case OM_MASK_NONE:
      return 1;
    case OM_MASK_CAUSAL:
      return j <= i;
    case OM_MASK_SLIDING:
      return j <= i && i - j < p->window;
    case OM_MASK_BLOCK: {
      int64_t nqb = (p->Sq + p->bx - 1) / p->bx;
      int64_t nkb = (p->Skv + p->by - 1) / p->by;
      return p->block_mask[((b * p->Hq + h) * nqb + i / p->bx) * nkb +
                           j / p->by] != 0;
    }
    case OM_MASK_TOKEN:
      return p->token_mask[((b * p->Hq + h) * p->Sq + i) * p->Skv + j] != 0;
    default:
      return 0;
  }
}

static double om_dot(const double* x, const double* y, int64_t n) {
  double acc = 0.0;
  for (int64_t d = 0; d < n; ++d) acc += x[d] * y[d];
  return acc;
}

static const double* om_row(const double* base, int64_t heads, int64_t seq,
                            int64_t D, int64_t b, int64_t h, int64_t i) {
  return base + ((b * heads + h) * seq + i) * D;
}

/*
 * Forward for a list of query rows.  rows[r] is a flat index into [B,Hq,Sq].
 * Writes O_out[r*D .. r*D+D) and LSE_out[r].
 */
void om_forward_rows(const om_problem* p, const double* q, const double* k,
                     const double* v, int64_t nrows, const int64_t* rows,
                     double* O_out, double* LSE_out) {
  const int64_t D = p->D, group = p->Hq / p->Hkv;
#pragma omp parallel
  {
    double* s = (double*)malloc(sizeof(double) * (size_t)p->Skv);
    uint8_t* vis = (uint8_t*)malloc((size_t)p->Skv);
#pragma omp for schedule(dynamic, 1)
    for (int64_t r = 0; r < nrows; ++r) {
      int64_t flat = rows[r];
      int64_t i = flat % p->Sq, h = (flat / p->Sq) % p->Hq,
              b = flat / (p->Sq * p->Hq);
      int64_t c = h / group;
      const double* qi = om_row(q, p->Hq, p->Sq, D, b, h, i);
      if (i >= om_len(p->seqlen_q, b, p->Sq)) { /* outside the problem */
        for (int64_t d = 0; d < D; ++d) O_out[r * D + d] = 0.0;
        LSE_out[r] = INFINITY;
        continue;
      }
      double m = -INFINITY;
      for (int64_t j = 0; j < p->Skv; ++j) {
        vis[j] = (uint8_t)om_visible(p, b, h, i, j);
        if (!vis[j]) continue;
        s[j] = p->scale * om_dot(qi, om_row(k, p->Hkv, p->Skv, D, b, c, j), D);
        if (s[j] > m) m = s[j];
      }
      double sink = p->sink ? p->sink[h] : -INFINITY;
      if (sink > m) m = sink;
      double* Oi = O_out + r * D;
      for (int64_t d = 0; d < D; ++d) Oi[d] = 0.0;
      if (m == -INFINITY) { /* nothing to attend to: P = 0 everywhere */
        LSE_out[r] = INFINITY;
        continue;
      }
      double l = 0.0;
      for (int64_t j = 0; j < p->Skv; ++j)
        if (vis[j]) l += exp(s[j] - m);
      if (p->sink) l += exp(sink - m);
      double lse = m + log(l);
      LSE_out[r] = lse;
      for (int64_t j = 0; j < p->Skv; ++j) {
        if (!vis[j]) continue;
        double pij = exp(s[j] - lse);
        const double* vj = om_row(v, p->Hkv, p->Skv, D, b, c, j);
        for (int64_t d = 0; d < D; ++d) Oi[d] += pij * vj[d];
      }
    }
    free(s);
    free(vis);
  }
}

/* Delta_i = <dO_i, O_in_i> for every row of [B,Hq,Sq]. */
void om_delta(const om_problem* p, const double* O_in, const double* dO,
              double* delta) {
  const int64_t n = p->B * p->Hq * p->Sq;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < n; ++r) {
    const int64_t i = r % p->Sq, b = r / (p->Sq * p->Hq);
    delta[r] = i < om_len(p->seqlen_q, b, p->Sq) ? om_dot(dO + r * p->D, O_in + r * p->D, p->D)
                                                  : 0.0;
  }
}

/*
 * dQ for a list of query rows (flat indices into [B,Hq,Sq]).
 * LSE_in and delta are full [B,Hq,Sq] arrays.
 */
void om_dq_rows(const om_problem* p, const double* q, const double* k,
                const double* v, const double* dO, const double* LSE_in,
                const double* delta, int64_t nrows, const int64_t* rows,
                double* dQ_out) {
  const int64_t D = p->D, group = p->Hq / p->Hkv;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t r = 0; r < nrows; ++r) {
    int64_t flat = rows[r];
    int64_t i = flat % p->Sq, h = (flat / p->Sq) % p->Hq,
            b = flat / (p->Sq * p->Hq);
    int64_t c = h / group;
    const double* qi = om_row(q, p->Hq, p->Sq, D, b, h, i);
    const double* dOi = om_row(dO, p->Hq, p->Sq, D, b, h, i);
    double* dQi = dQ_out + r * D;
    for (int64_t d = 0; d < D; ++d) dQi[d] = 0.0;
    for (int64_t j = 0; j < p->Skv; ++j) {
      if (!om_visible(p, b, h, i, j)) continue;
      const double* kj = om_row(k, p->Hkv, p->Skv, D, b, c, j);
      const double* vj = om_row(v, p->Hkv, p->Skv, D, b, c, j);
      double s = p->scale * om_dot(qi, kj, D);
      double P = exp(s - LSE_in[flat]);
      double dP = om_dot(dOi, vj, D);
      double dS = P * (dP - delta[flat]);
      for (int64_t d = 0; d < D; ++d) dQi[d] += p->scale * dS * kj[d];
    }
  }
}

/*
 * dK and dV for a list of key rows (flat indices into [B,Hkv,Skv]).  Each
 * sums over every q-head of its group and every visible query row.
 */
void om_dkdv_cols(const om_problem* p, const double* q, const double* k,
                  const double* v, const double* dO, const double* LSE_in,
                  const double* delta, int64_t ncols, const int64_t* cols,
                  double* dK_out, double* dV_out) {
  const int64_t D = p->D, group = p->Hq / p->Hkv;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t r = 0; r < ncols; ++r) {
    int64_t flat = cols[r];
    int64_t j = flat % p->Skv, c = (flat / p->Skv) % p->Hkv,
            b = flat / (p->Skv * p->Hkv);
    const double* kj = om_row(k, p->Hkv, p->Skv, D, b, c, j);
    const double* vj = om_row(v, p->Hkv, p->Skv, D, b, c, j);
    double* dKj = dK_out + r * D;
    double* dVj = dV_out + r * D;
    for (int64_t d = 0; d < D; ++d) dKj[d] = dVj[d] = 0.0;
    for (int64_t h = c * group; h < (c + 1) * group; ++h) {
      for (int64_t i = 0; i < p->Sq; ++i) {
        if (!om_visible(p, b, h, i, j)) continue;
        int64_t row = (b * p->Hq + h) * p->Sq + i;
        const double* qi = q + row * D;
        const double* dOi = dO + row * D;
        double s = p->scale * om_dot(qi, kj, D);
        double P = exp(s - LSE_in[row]);
        double dP = om_dot(dOi, vj, D);
        double dS = P * (dP - delta[row]);
        for (int64_t d = 0; d < D; ++d) {
          dVj[d] += P * dOi[d];
          dKj[d] += p->scale * dS * qi[d];
        }
      }
    }
  }
}

/* dSink_h = - sum_b sum_i exp(sink_h - LSE_in_i) Delta_i ; zero without sink. */
void om_dsink(const om_problem* p, const double* LSE_in, const double* delta,
              double* dsink) {
  for (int64_t h = 0; h < p->Hq; ++h) {
    double acc = 0.0;
    if (p->sink) {
      for (int64_t b = 0; b < p->B; ++b)
        for (int64_t i = 0; i < om_len(p->seqlen_q, b, p->Sq); ++i) {
          int64_t row = (b * p->Hq + h) * p->Sq + i;
          acc += exp(p->sink[h] - LSE_in[row]) * delta[row];
        }
    }
    dsink[h] = -acc;
  }
}

/* ----------------------------------------------------------------------
 * Block-mask tables (cannbot-knowledge PR #174, BlockSparseAttentionGrad
 * runbook, optimisations 1 and 2: the mask is transposed on the device and
 * compacted into per-row select tables whose entries are stored at the
 * position given by an exclusive prefix count of the kept entries).
 * ---------------------------------------------------------------------- */

/* maskT[b,h,kb,qb] = mask[b,h,qb,kb]. */
void om_mask_transpose(int64_t BH, int64_t nqb, int64_t nkb, const uint8_t* mask,
                       uint8_t* maskT) {
  for (int64_t bh = 0; bh < BH; ++bh)
    for (int64_t qb = 0; qb < nqb; ++qb)
      for (int64_t kb = 0; kb < nkb; ++kb)
        maskT[(bh * nkb + kb) * nqb + qb] = mask[(bh * nqb + qb) * nkb + kb];
}

/* Does any mask block with M=1 overlap query rows [r0,r1) x key cols [c0,c1)? */
static int om_tile_active(const uint8_t* m_bh, int64_t nkb, int64_t bx,
                          int64_t by, int64_t r0, int64_t r1, int64_t c0,
                          int64_t c1) {
  for (int64_t qb = r0 / bx; qb * bx < r1; ++qb)
    for (int64_t kb = c0 / by; kb * by < c1; ++kb)
      if (m_bh[qb * nkb + kb]) return 1;
  return 0;
}

/*
 * Select tables for tile sizes Tq (query rows per tile) and Tk (key rows per
 * tile).  Row kt of sel_k lists, ascending, every query tile qt such that the
 * tile pair (qt, kt) overlaps an active block; unused entries are -1 and
 * cnt_k[b,h,kt] is the count.  sel_q is the same with the roles swapped.
 *   sel_k [B*H, nKT, nQT], cnt_k [B*H, nKT]
 *   sel_q [B*H, nQT, nKT], cnt_q [B*H, nQT]
 * Either pair of output pointers may be NULL to skip it.
 */
void om_select_tables(int64_t BH, int64_t Sq, int64_t Skv, int64_t bx,
                      int64_t by, const uint8_t* mask, int64_t Tq_k,
                      int64_t Tk_k, int32_t* sel_k, int32_t* cnt_k,
                      int64_t Tq_q, int64_t Tk_q, int32_t* sel_q,
                      int32_t* cnt_q) {
  const int64_t nqb = (Sq + bx - 1) / bx, nkb = (Skv + by - 1) / by;
  for (int64_t bh = 0; bh < BH; ++bh) {
    const uint8_t* m = mask + bh * nqb * nkb;
    if (sel_k) {
      int64_t nQT = (Sq + Tq_k - 1) / Tq_k, nKT = (Skv + Tk_k - 1) / Tk_k;
      for (int64_t kt = 0; kt < nKT; ++kt) {
        int32_t* row = sel_k + (bh * nKT + kt) * nQT;
        int32_t n = 0;
        for (int64_t qt = 0; qt < nQT; ++qt) row[qt] = -1;
        for (int64_t qt = 0; qt < nQT; ++qt) {
          int64_t r0 = qt * Tq_k, r1 = r0 + Tq_k < Sq ? r0 + Tq_k : Sq;
          int64_t c0 = kt * Tk_k, c1 = c0 + Tk_k < Skv ? c0 + Tk_k : Skv;
          if (om_tile_active(m, nkb, bx, by, r0, r1, c0, c1)) row[n++] = (int32_t)qt;
        }
        cnt_k[bh * nKT + kt] = n;
      }
    }
    if (sel_q) {
      int64_t nQT = (Sq + Tq_q - 1) / Tq_q, nKT = (Skv + Tk_q - 1) / Tk_q;
      for (int64_t qt = 0; qt < nQT; ++qt) {
        int32_t* row = sel_q + (bh * nQT + qt) * nKT;
        int32_t n = 0;
        for (int64_t kt = 0; kt < nKT; ++kt) row[kt] = -1;
        for (int64_t kt = 0; kt < nKT; ++kt) {
          int64_t r0 = qt * Tq_q, r1 = r0 + Tq_q < Sq ? r0 + Tq_q : Sq;
          int64_t c0 = kt * Tk_q, c1 = c0 + Tk_q < Skv ? c0 + Tk_q : Skv;
          if (om_tile_active(m, nkb, bx, by, r0, r1, c0, c1)) row[n++] = (int32_t)kt;
        }
        cnt_q[bh * nQT + qt] = n;
      }
    }
  }
}

/* Number of visible (b,h,i,j) pairs: the unit the throughput is counted in. */
int64_t om_count_visible(const om_problem* p) {
  int64_t total = 0;
#pragma omp parallel for reduction(+ : total) schedule(dynamic, 1)
  for (int64_t r = 0; r < p->B * p->Hq * p->Sq; ++r) {
    int64_t i = r % p->Sq, h = (r / p->Sq) % p->Hq, b = r / (p->Sq * p->Hq);
    for (int64_t j = 0; j < p->Skv; ++j) total += om_visible(p, b, h, i, j);
  }
  return total;
}

int om_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

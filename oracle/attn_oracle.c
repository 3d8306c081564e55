/*
 * Plain fp64 CPU oracle for scaled-dot-product attention forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file: only the tests, the smoke check and the bench's CPU
 * baseline leg use it.  It shares no code, header, table or constant with
 * the CUDA library.
 *
 * What it computes (one query row at a time, every step in double):
 *
 *   "Flash Attention in CUDA Tile (cuTile)" (NVIDIA blog), section "The
 *   memory bandwidth problem": standard attention materialises the score
 *   row, applies softmax to it, then multiplies by V.  The flash method in
 *   the same page's section "Understanding online softmax" reaches exactly
 *   this result, so the oracle is the plain definition written out:
 *
 *     g     = Hq / Hkv,  kvh = h / g             (section "Grouped-query
 *                                                 attention": query heads
 *                                                 0-7 use K/V head 0, ...)
 *     s_j   = scale * sum_d Q[b,h,i,d] * K[b,kvh,j,d]        j in [0, Skv)
 *     key j is visible iff causal == 0 or j <= input_pos + i
 *                                                (section "Causal attention";
 *                                                 the kernel listing adds
 *                                                 input_pos to the query
 *                                                 offsets and keeps keys with
 *                                                 query offset >= key offset)
 *     and, with a sliding window of W >= 1 keys (causal only),
 *     j > input_pos + i - W                      (the last W positions up to
 *                                                 and including the query's:
 *                                                 "Sliding window attention"
 *                                                 is named as future work on
 *                                                 "Flash Attention from
 *                                                 Scratch", section "What's
 *                                                 Next", without a definition;
 *                                                 this is the reading taken.
 *                                                 W = 0: no window)
 *     M     = max over visible j of s_j
 *     p_j   = exp(s_j - M) if visible else 0      (safe softmax)
 *     L     = sum_j p_j
 *     O[b,h,i,:] = sum_j (p_j / L) * V[b,kvh,j,:]
 *     LSE[b,h,i] = M + ln(L)                      (natural log; the pages
 *                                                 define no LSE output, this
 *                                                 is the reading taken)
 *
 * Layouts: Q, O are [B, Hq, Sq, D]; K, V are [B, Hkv, Skv, D]; LSE is
 * [B, Hq, Sq]; all contiguous, row-major, in double.  Inputs in half or
 * bfloat16 are widened to double exactly by the caller before the call.
 *
 * Parity is pinned by tests that do not use this file's arithmetic: hand
 * derived small cases, the single-key closed form, uniform-score invariants,
 * probability row sums, GQA equivalence with repeated heads, key permutation
 * invariance and a library softmax-attention routine in float64.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Return codes. */
#define ORACLE_OK 0
#define ORACLE_BAD_ARG 1
#define ORACLE_NO_MEMORY 2

static int check_shape(long B, long Hq, long Hkv, long Sq, long Skv, long D,
                       int causal, long input_pos, long window) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || Sq < 0 || Skv <= 0 || D <= 0) return 0;
  if (Hq % Hkv != 0) return 0;
  if (input_pos < 0) return 0;
  if (window < 0 || (window > 0 && !causal)) return 0;
  /* Every row must see a key: the last row's window must reach Skv - 1. */
  if (window > 0 && Sq > 0 && input_pos + (Sq - 1) - window >= Skv - 1)
    return 0;
  return 1;
}

/* Key j is visible to query row i (absolute position input_pos + i). */
static int key_visible(int causal, long input_pos, long window, long i,
                       long j) {
  if (!causal) return 1;
  if (!(j <= input_pos + i)) return 0;              /* no future keys */
  return window <= 0 || j > input_pos + i - window;  /* sliding window */
}

/*
 * One query row (b, h, i).  Fills prob[0..Skv) with the softmax weights
 * p_j / L, out[0..D) with the output row, and *lse with M + ln L.
 * `score` is caller-provided scratch of Skv doubles.
 */
static void oracle_row(const double* Q, const double* K, const double* V,
                       long Hq, long Hkv, long Sq, long Skv, long D,
                       double scale, int causal, long input_pos, long window,
                       long b, long h, long i,
                       double* score, double* prob, double* out, double* lse) {
  const long group = Hq / Hkv;
  const long kvh = h / group;
  const double* q = Q + ((b * Hq + h) * Sq + i) * D;
  const double* k = K + (b * Hkv + kvh) * Skv * D;
  const double* v = V + (b * Hkv + kvh) * Skv * D;

  /* Scores for every key: S = Q K^T * scale, one row of it. */
  for (long j = 0; j < Skv; ++j) {
    double dot = 0.0;
    for (long d = 0; d < D; ++d) dot += q[d] * k[j * D + d];
    score[j] = scale * dot;
  }

  /* Visibility and the row maximum over visible keys. */
  double M = -INFINITY;
  for (long j = 0; j < Skv; ++j) {
    const int visible = key_visible(causal, input_pos, window, i, j);
    if (visible && score[j] > M) M = score[j];
  }

  /* Safe softmax: exponentials shifted by the maximum, then normalised. */
  double L = 0.0;
  for (long j = 0; j < Skv; ++j) {
    const int visible = key_visible(causal, input_pos, window, i, j);
    prob[j] = visible ? exp(score[j] - M) : 0.0;
    L += prob[j];
  }
  for (long j = 0; j < Skv; ++j) prob[j] /= L;

  /* Weighted sum of value rows. */
  for (long d = 0; d < D; ++d) out[d] = 0.0;
  for (long j = 0; j < Skv; ++j) {
    if (prob[j] == 0.0) continue;
    for (long d = 0; d < D; ++d) out[d] += prob[j] * v[j * D + d];
  }
  *lse = M + log(L);
}

/* Full forward pass: every (b, h, i) row.  LSE may be NULL. */
int attn_oracle_fwd(const double* Q, const double* K, const double* V,
                    double* O, double* LSE, long B, long Hq, long Hkv, long Sq,
                    long Skv, long D, double scale, int causal, long input_pos,
                    long window) {
  if (!check_shape(B, Hq, Hkv, Sq, Skv, D, causal, input_pos, window))
    return ORACLE_BAD_ARG;
  const long rows = B * Hq * Sq;
  int failed = 0;
#pragma omp parallel
  {
    double* score = (double*)malloc(sizeof(double) * (size_t)Skv);
    double* prob = (double*)malloc(sizeof(double) * (size_t)Skv);
    if (!score || !prob) {
#pragma omp atomic write
      failed = 1;
    } else {
#pragma omp for schedule(dynamic, 16)
      for (long r = 0; r < rows; ++r) {
        const long b = r / (Hq * Sq);
        const long h = (r / Sq) % Hq;
        const long i = r % Sq;
        double lse;
        oracle_row(Q, K, V, Hq, Hkv, Sq, Skv, D, scale, causal, input_pos,
                   window, b, h, i, score, prob, O + r * D, &lse);
        if (LSE) LSE[r] = lse;
      }
    }
    free(score);
    free(prob);
  }
  return failed ? ORACLE_NO_MEMORY : ORACLE_OK;
}

/*
 * Selected rows only.  rows_bhi holds n triplets (b, h, i); row r of the
 * result goes to O_rows[r*D .. r*D+D) and LSE_rows[r].  Used for parity at
 * sizes where computing every row would take too long.
 */
int attn_oracle_rows(const double* Q, const double* K, const double* V,
                     long B, long Hq, long Hkv, long Sq, long Skv, long D,
                     double scale, int causal, long input_pos, long window,
                     const int64_t* rows_bhi, long n, double* O_rows,
                     double* LSE_rows) {
  if (!check_shape(B, Hq, Hkv, Sq, Skv, D, causal, input_pos, window))
    return ORACLE_BAD_ARG;
  for (long r = 0; r < n; ++r) {
    const int64_t b = rows_bhi[3 * r], h = rows_bhi[3 * r + 1],
                  i = rows_bhi[3 * r + 2];
    if (b < 0 || b >= B || h < 0 || h >= Hq || i < 0 || i >= Sq)
      return ORACLE_BAD_ARG;
  }
  int failed = 0;
#pragma omp parallel
  {
    double* score = (double*)malloc(sizeof(double) * (size_t)Skv);
    double* prob = (double*)malloc(sizeof(double) * (size_t)Skv);
    if (!score || !prob) {
#pragma omp atomic write
      failed = 1;
    } else {
#pragma omp for schedule(dynamic, 4)
      for (long r = 0; r < n; ++r) {
        oracle_row(Q, K, V, Hq, Hkv, Sq, Skv, D, scale, causal, input_pos,
                   window, rows_bhi[3 * r], rows_bhi[3 * r + 1],
                   rows_bhi[3 * r + 2],
                   score, prob, O_rows + r * D, &LSE_rows[r]);
      }
    }
    free(score);
    free(prob);
  }
  return failed ? ORACLE_NO_MEMORY : ORACLE_OK;
}

/* The softmax weight row p_j / L of one query (b, h, i): prob[0..Skv). */
int attn_oracle_prob_row(const double* Q, const double* K, const double* V,
                         long B, long Hq, long Hkv, long Sq, long Skv, long D,
                         double scale, int causal, long input_pos,
                         long window, long b, long h, long i, double* prob) {
  if (!check_shape(B, Hq, Hkv, Sq, Skv, D, causal, input_pos, window))
    return ORACLE_BAD_ARG;
  if (b < 0 || b >= B || h < 0 || h >= Hq || i < 0 || i >= Sq)
    return ORACLE_BAD_ARG;
  double* score = (double*)malloc(sizeof(double) * (size_t)Skv);
  double* out = (double*)malloc(sizeof(double) * (size_t)D);
  if (!score || !out) {
    free(score);
    free(out);
    return ORACLE_NO_MEMORY;
  }
  double lse;
  oracle_row(Q, K, V, Hq, Hkv, Sq, Skv, D, scale, causal, input_pos, window,
             b, h, i, score, prob, out, &lse);
  free(score);
  free(out);
  return ORACLE_OK;
}

/*
 * Backward pass: gradients of the forward output O with respect to Q, K
 * and V for an upstream gradient dO ("Flash Attention from Scratch",
 * section "What's Next", lists the backward pass as future work; no page
 * gives its formulas, so this is the chain rule applied to the definition
 * above, in the order the definition computes):
 *
 *   O_i   = sum_j P_ij V_j                      =>  dV_j += P_ij dO_i
 *   dP_ij = dO_i . V_j
 *   P_ij  = softmax_j(s_ij), s_ij = scale q_i.k_j
 *                     =>  ds_ij = P_ij (dP_ij - sum_k P_ik dP_ik)
 *   dQ_i  = scale sum_j ds_ij K_j,   dK_j += scale ds_ij Q_i
 *
 * Masked keys have P_ij = 0 and get no gradient.  With grouped K/V heads
 * the query heads of a group add into the same dK, dV.  Rows are handled
 * one at a time in double; the parallel loop runs over (b, K/V head) so
 * that every dK / dV row has one writer.  dQ, dK, dV: same layouts as Q,
 * K, V.
 */
int attn_oracle_bwd(const double* Q, const double* K, const double* V,
                    const double* dO, double* dQ, double* dK, double* dV,
                    long B, long Hq, long Hkv, long Sq, long Skv, long D,
                    double scale, int causal, long input_pos, long window) {
  if (!check_shape(B, Hq, Hkv, Sq, Skv, D, causal, input_pos, window))
    return ORACLE_BAD_ARG;
  const long group = Hq / Hkv;
  for (long x = 0; x < B * Hkv * Skv * D; ++x) {
    dK[x] = 0.0;
    dV[x] = 0.0;
  }
  int failed = 0;
#pragma omp parallel
  {
    double* score = (double*)malloc(sizeof(double) * (size_t)Skv);
    double* prob = (double*)malloc(sizeof(double) * (size_t)Skv);
    double* dprob = (double*)malloc(sizeof(double) * (size_t)Skv);
    double* out = (double*)malloc(sizeof(double) * (size_t)D);
    if (!score || !prob || !dprob || !out) {
#pragma omp atomic write
      failed = 1;
    } else {
#pragma omp for schedule(dynamic, 1)
      for (long bk = 0; bk < B * Hkv; ++bk) {
        const long b = bk / Hkv, kvh = bk % Hkv;
        const double* k = K + bk * Skv * D;
        const double* v = V + bk * Skv * D;
        double* dk = dK + bk * Skv * D;
        double* dv = dV + bk * Skv * D;
        for (long h = kvh * group; h < (kvh + 1) * group; ++h) {
          for (long i = 0; i < Sq; ++i) {
            const long r = (b * Hq + h) * Sq + i;
            const double* q = Q + r * D;
            const double* dout = dO + r * D;
            double lse;
            oracle_row(Q, K, V, Hq, Hkv, Sq, Skv, D, scale, causal,
                       input_pos, window, b, h, i, score, prob, out, &lse);
            /* dP_ij = dO_i . V_j and the row sum of P_ij dP_ij. */
            double pdp = 0.0;
            for (long j = 0; j < Skv; ++j) {
              double dot = 0.0;
              for (long d = 0; d < D; ++d) dot += dout[d] * v[j * D + d];
              dprob[j] = dot;
              pdp += prob[j] * dot;
            }
            double* dq = dQ + r * D;
            for (long d = 0; d < D; ++d) dq[d] = 0.0;
            for (long j = 0; j < Skv; ++j) {
              if (prob[j] == 0.0) continue;
              const double ds = prob[j] * (dprob[j] - pdp);
              for (long d = 0; d < D; ++d) {
                dq[d] += scale * ds * k[j * D + d];
                dk[j * D + d] += scale * ds * q[d];
                dv[j * D + d] += prob[j] * dout[d];
              }
            }
          }
        }
      }
    }
    free(score);
    free(prob);
    free(dprob);
    free(out);
  }
  return failed ? ORACLE_NO_MEMORY : ORACLE_OK;
}

/*
 * dQ of selected query rows only (the same chain rule as attn_oracle_bwd,
 * which needs every row for dK and dV; a query row's dQ needs only its own
 * P and dP rows).  rows_bhi holds n triplets (b, h, i); dQ_rows[r*D ..).
 */
int attn_oracle_bwd_dq_rows(const double* Q, const double* K, const double* V,
                            const double* dO, long B, long Hq, long Hkv,
                            long Sq, long Skv, long D, double scale, int causal,
                            long input_pos, long window,
                            const int64_t* rows_bhi, long n, double* dQ_rows) {
  if (!check_shape(B, Hq, Hkv, Sq, Skv, D, causal, input_pos, window))
    return ORACLE_BAD_ARG;
  for (long r = 0; r < n; ++r) {
    const int64_t b = rows_bhi[3 * r], h = rows_bhi[3 * r + 1],
                  i = rows_bhi[3 * r + 2];
    if (b < 0 || b >= B || h < 0 || h >= Hq || i < 0 || i >= Sq)
      return ORACLE_BAD_ARG;
  }
  const long group = Hq / Hkv;
  int failed = 0;
#pragma omp parallel
  {
    double* score = (double*)malloc(sizeof(double) * (size_t)Skv);
    double* prob = (double*)malloc(sizeof(double) * (size_t)Skv);
    double* out = (double*)malloc(sizeof(double) * (size_t)D);
    if (!score || !prob || !out) {
#pragma omp atomic write
      failed = 1;
    } else {
#pragma omp for schedule(dynamic, 4)
      for (long r = 0; r < n; ++r) {
        const long b = rows_bhi[3 * r], h = rows_bhi[3 * r + 1],
                   i = rows_bhi[3 * r + 2];
        const double* k = K + (b * Hkv + h / group) * Skv * D;
        const double* v = V + (b * Hkv + h / group) * Skv * D;
        const double* dout = dO + ((b * Hq + h) * Sq + i) * D;
        double lse;
        oracle_row(Q, K, V, Hq, Hkv, Sq, Skv, D, scale, causal, input_pos,
                   window, b, h, i, score, prob, out, &lse);
        /* score[] is free now: reuse it for dP_ij = dO_i . V_j. */
        double pdp = 0.0;
        for (long j = 0; j < Skv; ++j) {
          double dot = 0.0;
          for (long d = 0; d < D; ++d) dot += dout[d] * v[j * D + d];
          score[j] = dot;
          pdp += prob[j] * dot;
        }
        double* dq = dQ_rows + r * D;
        for (long d = 0; d < D; ++d) dq[d] = 0.0;
        for (long j = 0; j < Skv; ++j) {
          if (prob[j] == 0.0) continue;
          const double ds = prob[j] * (score[j] - pdp);
          for (long d = 0; d < D; ++d) dq[d] += scale * ds * k[j * D + d];
        }
      }
    }
    free(score);
    free(prob);
    free(out);
  }
  return failed ? ORACLE_NO_MEMORY : ORACLE_OK;
}

/*
 * dK and dV of selected key rows only (the same chain rule as
 * attn_oracle_bwd, gathered per key instead of scattered per query row).
 * Key j of K/V head kvh receives from every query row (h, i) of the heads
 * h of its group:
 *   dV_j = sum_{h,i} P_hij dO_hi
 *   dK_j = scale * sum_{h,i} P_hij (dO_hi . V_j - sum_k P_hik dO_hi . V_k) Q_hi
 * The inner sum over k needs the query row's whole probability row, so the
 * query rows of each K/V group that a requested key belongs to are visited
 * once (first pass: that row sum and the row's weights on the requested
 * keys), then every requested key sums over them (second pass).
 * keys_bkj holds n triplets (b, kvh, j); dK_rows[r*D ..), dV_rows[r*D ..).
 */
int attn_oracle_bwd_dkdv_rows(const double* Q, const double* K,
                              const double* V, const double* dO, long B,
                              long Hq, long Hkv, long Sq, long Skv, long D,
                              double scale, int causal, long input_pos,
                              long window, const int64_t* keys_bkj, long n,
                              double* dK_rows, double* dV_rows) {
  if (!check_shape(B, Hq, Hkv, Sq, Skv, D, causal, input_pos, window))
    return ORACLE_BAD_ARG;
  for (long r = 0; r < n; ++r) {
    const int64_t b = keys_bkj[3 * r], kvh = keys_bkj[3 * r + 1],
                  j = keys_bkj[3 * r + 2];
    if (b < 0 || b >= B || kvh < 0 || kvh >= Hkv || j < 0 || j >= Skv)
      return ORACLE_BAD_ARG;
  }
  const long group = Hq / Hkv;
  const long qrows = group * Sq;  /* query rows of one K/V group */
  for (long x = 0; x < n * D; ++x) {
    dK_rows[x] = 0.0;
    dV_rows[x] = 0.0;
  }
  long* sel = (long*)malloc(sizeof(long) * (size_t)(n > 0 ? n : 1));
  double* pdp = (double*)malloc(sizeof(double) * (size_t)qrows);
  double* psel =
      (double*)malloc(sizeof(double) * (size_t)qrows * (size_t)(n > 0 ? n : 1));
  int failed = (!sel || !pdp || !psel);
  /* One K/V group (b, kvh) at a time: the requested keys in it ... */
  for (long first = 0; first < n && !failed; ++first) {
    const int64_t gb = keys_bkj[3 * first], gk = keys_bkj[3 * first + 1];
    int seen = 0;
    for (long r = 0; r < first; ++r)
      if (keys_bkj[3 * r] == gb && keys_bkj[3 * r + 1] == gk) seen = 1;
    if (seen) continue;
    long m = 0;
    for (long r = first; r < n; ++r)
      if (keys_bkj[3 * r] == gb && keys_bkj[3 * r + 1] == gk) sel[m++] = r;
    const double* v = V + (gb * Hkv + gk) * Skv * D;
    /* ... first pass over the group's query rows ... */
#pragma omp parallel
    {
      double* score = (double*)malloc(sizeof(double) * (size_t)Skv);
      double* prob = (double*)malloc(sizeof(double) * (size_t)Skv);
      double* out = (double*)malloc(sizeof(double) * (size_t)D);
      if (!score || !prob || !out) {
#pragma omp atomic write
        failed = 1;
      } else {
#pragma omp for schedule(dynamic, 8)
        for (long rr = 0; rr < qrows; ++rr) {
          const long h = gk * group + rr / Sq, i = rr % Sq;
          const double* dout = dO + ((gb * Hq + h) * Sq + i) * D;
          double lse;
          oracle_row(Q, K, V, Hq, Hkv, Sq, Skv, D, scale, causal, input_pos,
                     window, gb, h, i, score, prob, out, &lse);
          double s_pdp = 0.0;
          for (long jj = 0; jj < Skv; ++jj) {
            if (prob[jj] == 0.0) continue;
            double dot = 0.0;
            for (long d = 0; d < D; ++d) dot += dout[d] * v[jj * D + d];
            s_pdp += prob[jj] * dot;
          }
          pdp[rr] = s_pdp;
          for (long t = 0; t < m; ++t)
            psel[rr * m + t] = prob[keys_bkj[3 * sel[t] + 2]];
        }
      }
      free(score);
      free(prob);
      free(out);
    }
    if (failed) break;
    /* ... second pass: each requested key sums over those rows. */
#pragma omp parallel for schedule(dynamic, 1)
    for (long t = 0; t < m; ++t) {
      const long r = sel[t];
      const long j = keys_bkj[3 * r + 2];
      double* dk = dK_rows + r * D;
      double* dv = dV_rows + r * D;
      for (long rr = 0; rr < qrows; ++rr) {
        const double pj = psel[rr * m + t];
        if (pj == 0.0) continue;
        const long h = gk * group + rr / Sq, i = rr % Sq;
        const double* q = Q + ((gb * Hq + h) * Sq + i) * D;
        const double* dout = dO + ((gb * Hq + h) * Sq + i) * D;
        double dp = 0.0;
        for (long d = 0; d < D; ++d) dp += dout[d] * v[j * D + d];
        const double ds = pj * (dp - pdp[rr]);
        for (long d = 0; d < D; ++d) {
          dk[d] += scale * ds * q[d];
          dv[d] += pj * dout[d];
        }
      }
    }
  }
  free(sel);
  free(pdp);
  free(psel);
  return failed ? ORACLE_NO_MEMORY : ORACLE_OK;
}

/*
 * FP8 inputs.  "Flash Attention from Scratch", section "What's Next", names
 * FP8 tensor cores as future work and defines no format; the reading taken
 * is the 8-bit E4M3 format of the OCP "8-bit Floating Point Specification"
 * (the "e4m3fn" variant the GPU tensor cores consume), with one fp32
 * descale factor per tensor:  Q = q_descale * decode(Q8), and so on.  The
 * attention itself is then the definition above, in double.
 *
 * E4M3 bit fields: sign s (bit 7), exponent e (bits 3-6, bias 7), mantissa
 * m (bits 0-2).
 *   e == 0:            (-1)^s * m * 2^-9            (subnormal, incl. +-0)
 *   e == 15, m == 7:   NaN                          (no infinities)
 *   otherwise:         (-1)^s * (8 + m) * 2^(e-10)   (= 2^(e-7) * (1 + m/8))
 * Every value is exact in double.
 */
double attn_oracle_e4m3_value(unsigned int code) {
  const unsigned int s = (code >> 7) & 1u;
  const unsigned int e = (code >> 3) & 15u;
  const unsigned int m = code & 7u;
  double v;
  if (e == 15u && m == 7u) return NAN;
  if (e == 0u)
    v = ldexp((double)m, -9);
  else
    v = ldexp((double)(8u + m), (int)e - 10);
  return s ? -v : v;
}

/* out[i] = scale * decode(in[i]); the product of a 4-bit significand and
 * an fp32 descale is exact in double. */
int attn_oracle_decode_e4m3(const uint8_t* in, long n, double scale,
                            double* out) {
  if (n < 0 || (n > 0 && (in == NULL || out == NULL))) return ORACLE_BAD_ARG;
  for (long i = 0; i < n; ++i) out[i] = scale * attn_oracle_e4m3_value(in[i]);
  return ORACLE_OK;
}

/* Threads the parallel loops will use. */
int attn_oracle_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/*
 * ssd_oracle.c -- plain, slow, fp64 CPU oracle of one speculative-speculative
 * decoding round (Saguaro) and of tree-masked branch attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file: only the tests, the smoke check and the bench's CPU
 * baseline leg use it.  It shares no code, header, table or constant with the
 * CUDA library; it reads the same input bytes (fp32 or bf16 logits, bf16
 * Q/K/V) and the same uniforms, and computes every quantity in double
 * precision in plain index order, one sequence and one row at a time.
 *
 * Sources (web pages on "Speculative Speculative Decoding", the SSD framework
 * and its Saguaro algorithm):
 *  - 機器之心 article "全球最強推理引擎還快2倍，斯坦福、普林斯頓破解大模型串行魔咒",
 *    section "SSD 如何實現草擬與驗證并行？": the target verifies K draft tokens
 *    in one pass, decides how many to accept and samples one bonus token after
 *    them; the scheme is lossless; the draft predicts the bonus token from its
 *    most likely logits.
 *  - technical summary "超越传统SD：SSD框架全异步解码实现4.7倍平均加速",
 *    section "投机解码的瓶颈与 SSD 的核心机制": acceptance rate alpha; the
 *    speculation cache, read with a single lookup after verification.
 *  - same page, "Saguaro 算法" part 1 "验证结果预测与缓存拓扑优化": outcome space
 *    ~V^K, fan-out F_k per depth under a budget B, optimal F_k a truncated
 *    geometric series.
 *  - same page, part 2 "操纵残差分布": the residual distribution
 *    p_target - p_draft and the sampling scheme sigma_{F,C} that down-weights
 *    the draft's top tokens by C.
 *  - same page, "工程优化与系统表现": all F_k branches decoded in one forward pass
 *    with a custom sparse attention mask.
 * The formulas are missing from the extracted pages; the readings taken here
 * are: alpha = sum_i min(p_i, q'_i); the residual is max(0, p - q') renormalised,
 * q' being the distribution the draft actually sampled from; sigma_{F,C}
 * multiplies the probabilities of the top-F tokens (by draft logit) by C and
 * renormalises; fan-out split r^k weights with the rounding rule of
 * oracle_fanout_split; inverse-CDF draws in vocabulary order; ties broken by
 * (value descending, index ascending).
 *
 * Parity pins (tests/test_oracle_*.py): greedy chain at T = 0, chi-squared
 * losslessness at V = 8, exhaustive enumeration of (accept count, bonus) at
 * V = 8, K = 3 against the closed form prod alpha_j (1 - alpha_{k+1}), the
 * residual identity, sigma_{F,C} invariants, brute-force top-F, the fan-out
 * of the tiny workload, and dense attention with a brute-force mask.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_F32 0
#define OR_BF16 1

/* per-sequence flags, same meaning as the library's status bits */
#define OR_FLAG_BAD_TOKEN 1u
#define OR_FLAG_ZERO_RESIDUAL 2u
#define OR_FLAG_BAD_OUTCOME 8u
#define OR_FLAG_BAD_TREE 16u
#define OR_FLAG_BAD_BLOCK 32u
#define OR_FLAG_BAD_PREFIX 64u

static double load_elem(const void *base, int dtype, int64_t i) {
  if (dtype == OR_F32) return (double)((const float *)base)[i];
  uint32_t bits = ((uint32_t)((const uint16_t *)base)[i]) << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

static void load_row(const void *base, int dtype, int64_t off, int V, double *z) {
  for (int i = 0; i < V; i++) z[i] = load_elem(base, dtype, off + i);
}

/* ---------------------------------------------------------------------- */
/* Fan-out split of a budget over depths 0..K (truncated geometric series). */
/* Weights r^k, k = 0..K; F_k = max(1, floor(budget * w_k / sum w)); a       */
/* shortfall is given back one unit at a time in order of descending        */
/* fractional part (ties: smaller k); an excess is taken from the largest   */
/* F_k > 1 (ties: larger k).  Returns 0, or -1 for invalid arguments.       */
/* ---------------------------------------------------------------------- */
int oracle_fanout_split(int budget, int K, double r, int32_t *F) {
  if (K < 0 || budget < K + 1 || !(r > 0.0) || r > 1.0) return -1;
  double sw = 0.0;
  for (int k = 0; k <= K; k++) sw += pow(r, k);
  double frac[64];
  if (K + 1 > 64) return -1;
  int total = 0;
  for (int k = 0; k <= K; k++) {
    double x = budget * pow(r, k) / sw;
    double fl = floor(x);
    frac[k] = x - fl;
    F[k] = (int32_t)fl;
    if (F[k] < 1) F[k] = 1;
    total += F[k];
  }
  while (total < budget) {
    /* one pass in order of descending fractional part */
    int used[64] = {0};
    for (int t = 0; t <= K && total < budget; t++) {
      int best = -1;
      for (int k = 0; k <= K; k++)
        if (!used[k] && (best < 0 || frac[k] > frac[best])) best = k;
      used[best] = 1;
      F[best] += 1;
      total += 1;
    }
  }
  while (total > budget) {
    int best = -1;
    for (int k = 0; k <= K; k++)
      if (F[k] > 1 && (best < 0 || F[k] >= F[best])) best = k;
    if (best < 0) return -1;
    F[best] -= 1;
    total -= 1;
  }
  return 0;
}

/* ---------------------------------------------------------------------- */
/* Distributions                                                          */
/* ---------------------------------------------------------------------- */

/* Index of the largest value, lowest index on ties. */
static int argmax_lowest(const double *z, int V) {
  int best = 0;
  for (int i = 1; i < V; i++)
    if (z[i] > z[best]) best = i;
  return best;
}

/* p = softmax(z / T) for T > 0; for T == 0 the greedy limit, one-hot at the
 * argmax (lowest index on ties). */
void oracle_softmax(const double *z, int V, double T, double *p) {
  if (T == 0.0) {
    int a = argmax_lowest(z, V);
    for (int i = 0; i < V; i++) p[i] = (i == a) ? 1.0 : 0.0;
    return;
  }
  double m = z[0];
  for (int i = 1; i < V; i++)
    if (z[i] > m) m = z[i];
  double s = 0.0;
  for (int i = 0; i < V; i++) {
    p[i] = exp((z[i] - m) / T);
    s += p[i];
  }
  for (int i = 0; i < V; i++) p[i] /= s;
}

/* the keys of the sort in progress, one per thread (callers may run the
 * oracle on several threads at once) */
static _Thread_local const double *g_sort_keys;
static int cmp_desc_then_index(const void *a, const void *b) {
  int ia = *(const int32_t *)a, ib = *(const int32_t *)b;
  double va = g_sort_keys[ia], vb = g_sort_keys[ib];
  if (va > vb) return -1;
  if (va < vb) return 1;
  return (ia < ib) ? -1 : (ia > ib);
}

/* The F highest-ranked indices of z, ranked by (value descending, index
 * ascending): a full sort of all V indices. */
void oracle_topf(const double *z, int V, int F, int32_t *out) {
  int32_t *idx = (int32_t *)malloc(sizeof(int32_t) * (size_t)V);
  for (int i = 0; i < V; i++) idx[i] = i;
  g_sort_keys = z;
  qsort(idx, (size_t)V, sizeof(int32_t), cmp_desc_then_index);
  for (int i = 0; i < F; i++) out[i] = idx[i];
  free(idx);
}

/* Saguaro sampling distribution sigma_{F,C}(q): the probabilities of the F
 * top-ranked tokens (by raw draft logit) are multiplied by C and the result
 * renormalised:  q'_i = q_i c_i / (1 - (1 - C) sum_{k in S} q_k), c_i = C on S
 * and 1 elsewhere.  q = softmax(z / T).  ``in_s`` (optional, length V) receives
 * the membership of S. */
void oracle_saguaro_dist(const double *z, int V, int F, double C, double T, double *qp,
                         uint8_t *in_s) {
  double *q = (double *)malloc(sizeof(double) * (size_t)V);
  int32_t *S = (int32_t *)malloc(sizeof(int32_t) * (size_t)(F > 0 ? F : 1));
  uint8_t *mem = (uint8_t *)calloc((size_t)V, 1);
  oracle_softmax(z, V, T, q);
  oracle_topf(z, V, F, S);
  double sq = 0.0;
  for (int k = 0; k < F; k++) {
    mem[S[k]] = 1;
    sq += q[S[k]];
  }
  double norm = 1.0 - (1.0 - C) * sq;
  for (int i = 0; i < V; i++) qp[i] = q[i] * (mem[i] ? C : 1.0) / norm;
  if (in_s) memcpy(in_s, mem, (size_t)V);
  free(q);
  free(S);
  free(mem);
}

/* Inverse-CDF draw: the smallest i with sum_{k<=i} w_k > u * sum_k w_k; if
 * rounding leaves no such i, the last index with w > 0.  ``margin`` receives
 * the distance of u * W from the nearer edge of the chosen bin, divided by W
 * (how close the draw came to picking a neighbour). */
int oracle_inv_cdf(const double *w, int V, double u, double *margin) {
  double W = 0.0;
  for (int i = 0; i < V; i++) W += w[i];
  double t = u * W;
  double c = 0.0;
  for (int i = 0; i < V; i++) {
    double prev = c;
    c += w[i];
    if (c > t) {
      if (margin) {
        double lo = t - prev, hi = c - t;
        *margin = (lo < hi ? lo : hi) / W;
      }
      return i;
    }
  }
  int last = -1;
  for (int i = 0; i < V; i++)
    if (w[i] > 0.0) last = i;
  if (margin) *margin = 0.0;
  return last;
}

/* ---------------------------------------------------------------------- */
/* The round                                                               */
/* Logits are [B, K+1, V] with strides seq_stride (between sequences) and */
/* row_stride (between positions), in elements; row r of a sequence holds */
/* position j = r + 1.                                                     */
/* ---------------------------------------------------------------------- */

/* Saguaro draft sampling for positions j = 1..K: d_j ~ sigma_{F_{j-1},C}(q_j),
 * drawn by inverse CDF with u_draft[b, j-1].  qd = q'_j(d_j). */
int oracle_saguaro_sample(const void *draft, int dtype, int64_t seq_stride, int64_t row_stride,
                          int B, int K, int V, const int32_t *F, double C, double T,
                          const float *u_draft, int32_t *d_out, double *qd_out,
                          double *margin_out) {
  double *z = (double *)malloc(sizeof(double) * (size_t)V);
  double *qp = (double *)malloc(sizeof(double) * (size_t)V);
  for (int b = 0; b < B; b++) {
    for (int j = 1; j <= K; j++) {
      load_row(draft, dtype, b * seq_stride + (int64_t)(j - 1) * row_stride, V, z);
      oracle_saguaro_dist(z, V, F[j - 1], C, T, qp, NULL);
      double margin;
      int d = oracle_inv_cdf(qp, V, (double)u_draft[b * K + (j - 1)], &margin);
      d_out[b * K + (j - 1)] = d;
      if (qd_out) qd_out[b * K + (j - 1)] = qp[d];
      if (margin_out) margin_out[b * K + (j - 1)] = (T == 0.0) ? INFINITY : margin;
    }
  }
  free(z);
  free(qp);
  return 0;
}

/* Lossless verification of d_1..d_K per sequence.
 *   p_j = softmax(z^t_j / T), q'_j = sigma_{F_{j-1},C}(softmax(z^d_j / T)).
 *   For j = 1..K: accept d_j iff u_acc_j * q'_j(d_j) < p_j(d_j); stop at the
 *   first rejection; a = number accepted.
 *   a < K: bonus b ~ max(0, p_{a+1} - q'_{a+1}) renormalised (u_bonus); if that
 *          residual has no mass, b ~ p_{a+1} and ZERO_RESIDUAL is flagged.
 *   a = K: bonus b ~ p_{K+1}.
 * Outputs: accept_len[b], out_tokens[b, 0..K] (d_1..d_a, bonus, then -1),
 * bonus[b]; accept_prob[b, j-1] = P(u * q' < p) = min(1, p/q') (1 when q' = 0
 * and p > 0, 0 when both are 0; 0 for an out-of-range d_j); resid_mass[b] = W
 * of the residual used (1 after full acceptance); flags[b]; acc_margin[b, j-1]
 * = |u - p/q'| for the tests actually taken (inf otherwise and at T = 0);
 * bonus_margin[b] as in oracle_inv_cdf (inf at T = 0); alpha[b, j-1] =
 * sum_i min(p_j(i), q'_j(i)). */
int oracle_verify(const void *target, const void *draft, int dtype, int64_t seq_stride,
                  int64_t row_stride, int B, int K, int V, const int32_t *F, double C, double T,
                  const int32_t *d, const float *u_acc, const float *u_bonus,
                  int32_t *accept_len, int32_t *out_tokens, int32_t *bonus, double *accept_prob,
                  double *resid_mass, uint32_t *flags, double *acc_margin, double *bonus_margin,
                  double *alpha) {
  double *zt = (double *)malloc(sizeof(double) * (size_t)V);
  double *zd = (double *)malloc(sizeof(double) * (size_t)V);
  double *p = (double *)malloc(sizeof(double) * (size_t)V);
  double *qp = (double *)malloc(sizeof(double) * (size_t)V);
  double *r = (double *)malloc(sizeof(double) * (size_t)V);
  for (int b = 0; b < B; b++) {
    uint32_t fl = 0;
    int a = 0, rejected = 0;
    for (int j = 1; j <= K; j++) {
      int64_t off = b * seq_stride + (int64_t)(j - 1) * row_stride;
      load_row(target, dtype, off, V, zt);
      load_row(draft, dtype, off, V, zd);
      oracle_softmax(zt, V, T, p);
      oracle_saguaro_dist(zd, V, F[j - 1], C, T, qp, NULL);
      if (alpha) {
        double al = 0.0;
        for (int i = 0; i < V; i++) al += (p[i] < qp[i]) ? p[i] : qp[i];
        alpha[b * K + (j - 1)] = al;
      }
      int dj = d[b * K + (j - 1)];
      double pd = 0.0, qd = 0.0, ap = 0.0;
      int valid = (dj >= 0 && dj < V);
      if (valid) {
        pd = p[dj];
        qd = qp[dj];
        ap = (qd > 0.0) ? ((pd / qd < 1.0) ? pd / qd : 1.0) : (pd > 0.0 ? 1.0 : 0.0);
      } else {
        fl |= OR_FLAG_BAD_TOKEN;
      }
      if (accept_prob) accept_prob[b * K + (j - 1)] = ap;
      if (acc_margin) acc_margin[b * K + (j - 1)] = INFINITY;
      if (!rejected) {
        double u = (double)u_acc[b * K + (j - 1)];
        int acc = valid && (u * qd < pd);
        if (acc_margin && valid && T != 0.0 && qd > 0.0)
          acc_margin[b * K + (j - 1)] = fabs(u - pd / qd);
        if (acc) {
          a += 1;
        } else {
          rejected = 1;
        }
      }
    }
    /* bonus token */
    int bt;
    double W;
    double bm = INFINITY;
    double u = (double)u_bonus[b];
    int64_t off = b * seq_stride + (int64_t)a * row_stride; /* row of position a+1 */
    load_row(target, dtype, off, V, zt);
    oracle_softmax(zt, V, T, p);
    if (a < K) {
      load_row(draft, dtype, off, V, zd);
      oracle_saguaro_dist(zd, V, F[a], C, T, qp, NULL);
      W = 0.0;
      for (int i = 0; i < V; i++) {
        r[i] = (p[i] > qp[i]) ? p[i] - qp[i] : 0.0;
        W += r[i];
      }
      if (W > 0.0) {
        bt = oracle_inv_cdf(r, V, u, &bm);
      } else {
        fl |= OR_FLAG_ZERO_RESIDUAL;
        bt = oracle_inv_cdf(p, V, u, &bm);
      }
    } else {
      W = 1.0;
      bt = oracle_inv_cdf(p, V, u, &bm);
    }
    if (T == 0.0) bm = INFINITY;
    accept_len[b] = a;
    bonus[b] = bt;
    for (int t = 0; t <= K; t++) {
      int32_t v = -1;
      if (t < a) v = d[b * K + t];
      if (t == a) v = bt;
      out_tokens[b * (K + 1) + t] = v;
    }
    if (resid_mass) resid_mass[b] = W;
    if (flags) flags[b] = fl;
    if (bonus_margin) bonus_margin[b] = bm;
  }
  free(zt);
  free(zd);
  free(p);
  free(qp);
  free(r);
  return 0;
}

/* Outcome prediction: for depth k = 0..K the guessed bonus tokens are the
 * top-F_k tokens of draft row k+1 (value descending, index ascending);
 * guess[b, off_k + i], off_k = F_0 + ... + F_{k-1}; guess_q = q_{k+1} of each
 * guess (softmax(z / T), one-hot at T = 0). */
int oracle_predict(const void *draft, int dtype, int64_t seq_stride, int64_t row_stride, int B,
                   int K, int V, const int32_t *F, double T, int32_t *guess, double *guess_q) {
  int sumF = 0;
  for (int k = 0; k <= K; k++) sumF += F[k];
  double *z = (double *)malloc(sizeof(double) * (size_t)V);
  double *q = (double *)malloc(sizeof(double) * (size_t)V);
  for (int b = 0; b < B; b++) {
    int off = 0;
    for (int k = 0; k <= K; k++) {
      load_row(draft, dtype, b * seq_stride + (int64_t)k * row_stride, V, z);
      oracle_topf(z, V, F[k], guess + (int64_t)b * sumF + off);
      if (guess_q) {
        oracle_softmax(z, V, T, q);
        for (int i = 0; i < F[k]; i++)
          guess_q[(int64_t)b * sumF + off + i] = q[guess[(int64_t)b * sumF + off + i]];
      }
      off += F[k];
    }
  }
  free(z);
  free(q);
  return 0;
}

/* Speculation-cache lookup keyed by the outcome (a, b): a hit iff the bonus b
 * is among the F_a guesses of depth a; slot = off_a + its rank there, else -1.
 * next_tokens[b] = payload[b, slot, 0..K-1] on a hit, all -1 on a miss.
 * An accept count outside 0..K is a miss flagged BAD_OUTCOME.  Returns the
 * number of hits. */
int oracle_lookup(const int32_t *guess, const int32_t *payload, int B, int K, const int32_t *F,
                  const int32_t *accept_len, const int32_t *bonus, int32_t *slot,
                  int32_t *next_tokens, uint32_t *flags) {
  int sumF = 0;
  for (int k = 0; k <= K; k++) sumF += F[k];
  int hits = 0;
  for (int b = 0; b < B; b++) {
    int a = accept_len[b];
    int s = -1;
    uint32_t fl = 0;
    if (a < 0 || a > K) {
      fl |= OR_FLAG_BAD_OUTCOME;
    } else {
      int off = 0;
      for (int k = 0; k < a; k++) off += F[k];
      for (int i = 0; i < F[a]; i++)
        if (guess[(int64_t)b * sumF + off + i] == bonus[b]) {
          s = off + i;
          break;
        }
    }
    slot[b] = s;
    if (s >= 0) hits++;
    if (next_tokens)
      for (int t = 0; t < K; t++)
        next_tokens[(int64_t)b * K + t] =
            (s >= 0 && payload) ? payload[((int64_t)b * sumF + s) * K + t] : -1;
    if (flags) flags[b] = fl;
  }
  return hits;
}

/* Exact analytics of one round, before any uniform is drawn (technical
 * summary "超越传统SD：SSD框架全异步解码实现4.7倍平均加速": section "投机解码的瓶颈与
 * SSD 的核心机制" names the acceptance rate alpha; "Saguaro 算法" part 1
 * makes the chance that the bonus token lands among the cached guesses the
 * objective of the fan-out).  With the logit rows fixed, d_j ~ q'_j is
 * accepted with probability sum_i q'_j(i) min(1, p_j(i)/q'_j(i)) =
 * sum_i min(p_j(i), q'_j(i)), so per sequence:
 *   alpha[j-1]  = sum_i min(p_j(i), q'_j(i))                 (j = 1..K)
 *   resid_w[j-1] = W_j = sum_i max(0, p_j(i) - q'_j(i))       (= 1 - alpha_j)
 *   p_accept[k] = P(a = k) = prod_{j<=k} alpha_j * W_{k+1}   (k < K)
 *   p_accept[K] = prod_{j<=K} alpha_j
 *   hit_mass[k] = P(bonus in S_{k+1} | a = k): the bonus is drawn from the
 *                 normalised residual r_{k+1} / W_{k+1} (from p_{k+1} when
 *                 W_{k+1} = 0) for k < K and from p_{K+1} for k = K; S_{k+1}
 *                 is the top-F_k list of draft row k+1 (the depth-k guesses)
 *   hit_rate    = sum_k p_accept[k] hit_mass[k]
 *   exp_tokens  = sum_k p_accept[k] (k + 1)   (tokens emitted per round)
 *   hit_scale[k] = sum_{i in S_{k+1}} (p_{k+1}(i) + q'_{k+1}(i)) / W_{k+1} when
 *                 the residual is used, else hit_mass[k]: the size of the terms
 *                 whose differences make up hit_mass[k] (an error of eps in
 *                 each probability moves hit_mass[k] by at most eps times it). */
int oracle_round_analytics(const void *target, const void *draft, int dtype, int64_t seq_stride,
                           int64_t row_stride, int B, int K, int V, const int32_t *F, double C,
                           double T, double *alpha, double *resid_w, double *p_accept,
                           double *hit_mass, double *hit_rate, double *exp_tokens, double *hit_scale) {
  double *zt = (double *)malloc(sizeof(double) * (size_t)V);
  double *zd = (double *)malloc(sizeof(double) * (size_t)V);
  double *p = (double *)malloc(sizeof(double) * (size_t)V);
  double *qp = (double *)malloc(sizeof(double) * (size_t)V);
  uint8_t *ins = (uint8_t *)malloc((size_t)V);
  for (int b = 0; b < B; b++) {
    double run = 1.0, hit = 0.0, etok = 0.0;
    for (int k = 0; k <= K; k++) {
      int64_t off = b * seq_stride + (int64_t)k * row_stride; /* position k + 1 */
      load_row(target, dtype, off, V, zt);
      load_row(draft, dtype, off, V, zd);
      oracle_softmax(zt, V, T, p);
      /* S_{k+1} and, for k < K, the distribution the draft samples d_{k+1} from */
      oracle_saguaro_dist(zd, V, F[k], C, T, qp, ins);
      double pk, hk = 0.0, hs = 0.0;
      if (k < K) {
        double al = 0.0, w = 0.0;
        for (int i = 0; i < V; i++) {
          al += (p[i] < qp[i]) ? p[i] : qp[i];
          w += (p[i] > qp[i]) ? p[i] - qp[i] : 0.0;
        }
        alpha[b * K + k] = al;
        resid_w[b * K + k] = w;
        for (int i = 0; i < V; i++) {
          if (!ins[i]) continue;
          if (w > 0.0) {
            hk += ((p[i] > qp[i]) ? p[i] - qp[i] : 0.0) / w;
            hs += (p[i] + qp[i]) / w;
          } else {
            hk += p[i];
            hs += p[i];
          }
        }
        pk = run * w;
        run *= al;
      } else {
        for (int i = 0; i < V; i++)
          if (ins[i]) hk += p[i];
        hs = hk;
        pk = run;
      }
      p_accept[b * (K + 1) + k] = pk;
      hit_mass[b * (K + 1) + k] = hk;
      if (hit_scale) hit_scale[b * (K + 1) + k] = hs;
      hit += pk * hk;
      etok += pk * (double)(k + 1);
    }
    hit_rate[b] = hit;
    exp_tokens[b] = etok;
  }
  free(zt);
  free(zd);
  free(p);
  free(qp);
  free(ins);
  return 0;
}

/* ---------------------------------------------------------------------- */
/* Branch attention                                                        */
/* q [B, Nq, Hq, d] bf16; k_cache, v_cache [num_blocks, Hkv, 16, d] bf16;   */
/* block_table [B, maxb]; prefix_len [B]; parent [B, N] (-1 = prefix end).  */
/* Node m of sequence b sits at logical position prefix_len[b] + m; query   */
/* row i is node N - Nq + i.  Row i of head h sees every prefix position    */
/* and the nodes on its ancestor-or-self path; head h reads KV head         */
/* h / (Hq / Hkv).  out = softmax(scale * q k^T over the visible keys) v,   */
/* lse = log sum exp(scale * q k^T) (natural log), both in double.          */
/* A parent outside [-1, m-1] ends the path (BAD_TREE); a block id outside  */
/* [0, num_blocks) hides the keys it would hold (BAD_BLOCK); a negative     */
/* prefix counts as 0 and positions past 16 * maxb are hidden (BAD_PREFIX). */
/* ---------------------------------------------------------------------- */
int oracle_branch_attention(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                            const int32_t *block_table, int maxb, int64_t num_blocks,
                            const int32_t *prefix_len, const int32_t *parent, int B, int N,
                            int Nq, int Hq, int Hkv, int d, double scale, double *out,
                            double *lse, uint32_t *flags) {
  const int page = 16;
  int group = Hq / Hkv;
  for (int b = 0; b < B; b++) {
    uint32_t fl = 0;
    int L = prefix_len[b];
    /* a prefix the block table cannot hold: a negative one counts as 0, and the
     * positions past the table's 16 * maxb are hidden */
    if (L < 0) {
      fl |= OR_FLAG_BAD_PREFIX;
      L = 0;
    }
    if ((int64_t)L + N > (int64_t)maxb * page) fl |= OR_FLAG_BAD_PREFIX;
    int nkeys_max = L + N;
    int32_t *keys = (int32_t *)malloc(sizeof(int32_t) * (size_t)(nkeys_max > 0 ? nkeys_max : 1));
    double *s = (double *)malloc(sizeof(double) * (size_t)(nkeys_max > 0 ? nkeys_max : 1));
    for (int qi = 0; qi < Nq; qi++) {
      int node = N - Nq + qi;
      /* visible logical positions, in increasing order */
      int nk = 0;
      for (int pos = 0; pos < L; pos++) keys[nk++] = pos;
      uint8_t *onpath = (uint8_t *)calloc((size_t)(N > 0 ? N : 1), 1);
      int m = node;
      while (m >= 0) {
        onpath[m] = 1;
        int pm = parent[(int64_t)b * N + m];
        if (pm < -1 || pm >= m) {
          fl |= OR_FLAG_BAD_TREE;
          break;
        }
        m = pm;
      }
      for (int n = 0; n < N; n++)
        if (onpath[n]) keys[nk++] = L + n;
      free(onpath);
      for (int h = 0; h < Hq; h++) {
        int hk = h / group;
        const uint16_t *qrow = q + (((int64_t)b * Nq + qi) * Hq + h) * d;
        double mx = -INFINITY;
        int nvis = 0;
        for (int t = 0; t < nk; t++) {
          int pos = keys[t];
          if (pos / page >= maxb) { /* past the table: hidden */
            s[t] = -INFINITY;
            continue;
          }
          int blk = block_table[(int64_t)b * maxb + pos / page];
          if (blk < 0 || blk >= num_blocks) {
            fl |= OR_FLAG_BAD_BLOCK;
            s[t] = -INFINITY;
            continue;
          }
          const uint16_t *krow = k_cache + (((int64_t)blk * Hkv + hk) * page + pos % page) * d;
          double acc = 0.0;
          for (int e = 0; e < d; e++) acc += load_elem(qrow, OR_BF16, e) * load_elem(krow, OR_BF16, e);
          s[t] = acc * scale;
          if (s[t] > mx) mx = s[t];
          nvis++;
        }
        double *o = out + (((int64_t)b * Nq + qi) * Hq + h) * d;
        for (int e = 0; e < d; e++) o[e] = 0.0;
        double den = 0.0;
        if (nvis > 0) {
          for (int t = 0; t < nk; t++) {
            if (s[t] == -INFINITY) continue;
            double w = exp(s[t] - mx);
            den += w;
            int pos = keys[t];
            int blk = block_table[(int64_t)b * maxb + pos / page];
            const uint16_t *vrow = v_cache + (((int64_t)blk * Hkv + hk) * page + pos % page) * d;
            for (int e = 0; e < d; e++) o[e] += w * load_elem(vrow, OR_BF16, e);
          }
          for (int e = 0; e < d; e++) o[e] /= den;
        }
        if (lse) lse[((int64_t)b * Nq + qi) * Hq + h] = (nvis > 0) ? mx + log(den) : -INFINITY;
      }
    }
    free(keys);
    free(s);
    if (flags) flags[b] = fl;
  }
  return 0;
}

/* ===========================================================================
 * Miss fallback (technical summary "超越传统SD：SSD框架全异步解码实现4.7倍平均加速",
 * "Saguaro 算法" part 3 "大 Batch 下的退避策略", and the speedup statement of
 * "投机解码的瓶颈与 SSD 的核心机制" in p_hit, T_p and T_b).
 * ======================================================================== */

/* A uniform token id from a uniform u in [0, 1) with a 24-bit mantissa:
 * floor(u * V), computed exactly in integers (u * 2^24 is an integer). */
static int32_t uniform_token(float u, int V) {
  const uint64_t m = (uint64_t)((double)u * 16777216.0);
  return (int32_t)((m * (uint64_t)V) >> 24);
}

/* Low-latency backup speculator for the sequences that missed the
 * speculation cache (slot[b] < 0): an n-gram lookup in the sequence's own
 * history.  Reading: with the history h[0..L) (L = hist_len[b]) and its last
 * n tokens s = h[L-n..L), the latest earlier occurrence m (m + n <= L - 1,
 * h[m..m+n) = s, searched from m = L-n-1 down to 0) proposes the K tokens
 * h[m+n], h[m+n+1], ...; positions past L, and every position when s occurs
 * nowhere earlier (or L < n + 1), take the random backup token
 * floor(u_rand[b, t] V).  Hits keep their next_tokens.  match_pos[b] = m,
 * -1 without a match, -2 for a hit. */
int oracle_ngram_backup(const int32_t *hist, int64_t hist_stride, const int32_t *hist_len, int B, int n, int K,
                        int V, const int32_t *slot, const float *u_rand, int32_t *next_tokens,
                        int32_t *match_pos) {
  for (int b = 0; b < B; ++b) {
    if (slot[b] >= 0) {
      match_pos[b] = -2;
      continue;
    }
    const int32_t *h = hist + (int64_t)b * hist_stride;
    const int L = hist_len[b];
    int m = -1;
    if (n >= 1 && L >= n + 1) {
      for (int c = L - n - 1; c >= 0 && m < 0; --c) {
        int eq = 1;
        for (int i = 0; i < n && eq; ++i) eq = (h[c + i] == h[L - n + i]);
        if (eq) m = c;
      }
    }
    match_pos[b] = m;
    for (int t = 0; t < K; ++t) {
      const int p = m + n + t;
      next_tokens[(int64_t)b * K + t] = (m >= 0 && p < L) ? h[p] : uniform_token(u_rand[(int64_t)b * K + t], V);
    }
  }
  return 0;
}

/* The batch-level speedup model and the fallback choice.  Reading (the
 * formula did not survive extraction; restated from the definitions the
 * pages give): the primary speculator drafts for every predicted outcome
 * while the target verifies, so a round whose outcome hits the cache costs
 * max(T_v, T_p); a miss falls back to synchronous speculation with backup o,
 * and one miss stalls the whole batch for T_b[o].  With independent hits of
 * probability p_hit[b]:
 *   time[o]   = max(T_v, T_p) + (1 - prod_b p_hit[b]) T_b[o]
 *   tokens[o] = sum_b (p_hit[b] e_hit[b] + (1 - p_hit[b]) e_miss[o])
 *   throughput[o] = tokens[o] / time[o];
 *   speedup[o] = throughput[o] / (sum_b e_hit[b] / (T_p + T_v)), i.e. against
 *                synchronous speculative decoding with the primary (draft,
 *                then verify, every round);
 *   best = the option of largest throughput (ties: the lower index). */
int oracle_fallback_plan(const float *p_hit, const float *e_hit, int B, double T_v, double T_p, int nopt,
                         const double *T_b, const double *e_miss, double *time, double *tokens,
                         double *throughput, double *speedup) {
  double pall = 1.0, ph = 0.0, ehit = 0.0, pmiss = 0.0;
  for (int b = 0; b < B; ++b) {
    pall *= (double)p_hit[b];
    ph += (double)p_hit[b] * (double)e_hit[b];
    pmiss += 1.0 - (double)p_hit[b];
    ehit += (double)e_hit[b];
  }
  const double base = ehit / (T_p + T_v);
  int best = 0;
  for (int o = 0; o < nopt; ++o) {
    time[o] = (T_v > T_p ? T_v : T_p) + (1.0 - pall) * T_b[o];
    tokens[o] = ph + pmiss * e_miss[o];
    throughput[o] = tokens[o] / time[o];
    speedup[o] = throughput[o] / base;
    if (throughput[o] > throughput[best]) best = o;
  }
  return best;
}

/* ===========================================================================
 * Speculation-cache fill by branch decode (technical summary
 * "超越传统SD：SSD框架全异步解码实现4.7倍平均加速", "投机解码的瓶颈与 SSD 的核心机制":
 * the draft pre-speculates a continuation for every predicted outcome while
 * the target verifies; "工程优化与系统表现": all F_k branches are decoded in one
 * forward pass).  Each decode step feeds one token per branch: its key and
 * value rows are appended to the paged cache at the branch node's position,
 * and the next token of every branch is drawn from the draft's logits with
 * the Saguaro scheme (the draw itself is oracle_saguaro_sample on one row).
 * ======================================================================== */

/* Append the key/value rows of S new tree nodes per sequence to a paged
 * cache [num_blocks, Hkv, 16, d] (bf16 bits): row (b, i, h) goes to logical
 * position pos = prefix_len[b] + node0 + i, i.e. page block_table[b, pos/16],
 * slot pos % 16.  A position past the block table (pos / 16 >= maxb) or a
 * negative prefix writes nothing and sets flag 64 for the sequence; a page id
 * outside [0, num_blocks) writes nothing and sets flag 32. */
int oracle_kv_append(const uint16_t *k_new, const uint16_t *v_new, uint16_t *k_cache, uint16_t *v_cache,
                     const int32_t *block_table, int maxb, int64_t num_blocks, const int32_t *prefix_len,
                     int node0, int B, int S, int Hkv, int d, uint32_t *flags) {
  const int page = 16;
  for (int b = 0; b < B; ++b) {
    uint32_t fl = 0;
    for (int i = 0; i < S; ++i) {
      const int64_t pos = (int64_t)prefix_len[b] + node0 + i;
      if (prefix_len[b] < 0 || pos / page >= maxb) {
        fl |= 64u;
        continue;
      }
      const int64_t blk = block_table[(int64_t)b * maxb + pos / page];
      if (blk < 0 || blk >= num_blocks) {
        fl |= 32u;
        continue;
      }
      for (int h = 0; h < Hkv; ++h) {
        const int64_t src = (((int64_t)b * S + i) * Hkv + h) * d;
        const int64_t dst = ((blk * Hkv + h) * page + pos % page) * d;
        for (int e = 0; e < d; ++e) {
          k_cache[dst + e] = k_new[src + e];
          v_cache[dst + e] = v_new[src + e];
        }
      }
    }
    if (flags) flags[b] = fl;
  }
  return 0;
}

/* ===========================================================================
 * Token-tree verification with several candidates per node (the 機器之心
 * article "全球最強推理引擎還快2倍，斯坦福、普林斯頓破解大模型串行魔咒" names
 * combining SSD with token-tree speculation as future work; the technical
 * summary "超越传统SD：SSD框架全异步解码实现4.7倍平均加速" states the single-chain
 * acceptance rule and the residual p_target - p_draft that this generalises).
 * Reading: the children of a node were drawn independently from the draft's
 * distribution q at that node; they are tested one after another against a
 * target distribution r that starts as p and, after each rejection, becomes
 * the normalised residual max(0, r - q) / sum max(0, r - q), so that the token
 * finally emitted at the node follows p (the multi-draft form of the
 * single-chain rule).
 * ======================================================================== */

/* Logits [B, N+1, V]: row 0 holds the distributions after the prefix (the
 * root), row m+1 those after tree node m.  parent [B, N]: parent[m] in
 * [-1, m-1] (-1 the root); tokens [B, N]; u_acc [B, N] the uniform of node m's
 * test; u_bonus [B].  Per sequence, from the root:
 *   p = softmax(target row / T), q = softmax(draft row / T), r = p;
 *   for each child c of the node in index order (token x):
 *     x outside [0, V): BAD_TOKEN, the child is skipped;
 *     accept iff u_acc[c] * q(x) < r(x) -> the walk moves to c;
 *     else W = sum max(0, r - q); r = max(0, r - q) / W when W > 0, else
 *          ZERO_RESIDUAL and r stays;
 *   no child accepted: bonus ~ r by inverse CDF with u_bonus; stop.
 * A node whose parent lies outside [-1, m-1] is nobody's child (BAD_TREE).
 * T = 0: one-hot p and q at the argmaxes (lowest index on ties).
 * Outputs: accept_len[b] = accepted nodes, path[b, 0..] their indices (-1
 * after), bonus[b]; resid_mass[b] = the W of the last residual taken at the
 * final node (1 when its r is p); acc_margin[b, c] = |u - r(x)/q(x)| for
 * tested children (inf otherwise and at T = 0); bonus_margin as in
 * oracle_inv_cdf (inf at T = 0). */
int oracle_tree_verify(const void *target, const void *draft, int dtype, int64_t seq_stride,
                       int64_t row_stride, int B, int N, int V, double T, const int32_t *parent,
                       const int32_t *tokens, const float *u_acc, const float *u_bonus,
                       int32_t *accept_len, int32_t *path, int32_t *bonus, double *resid_mass,
                       uint32_t *flags, double *acc_margin, double *bonus_margin) {
  double *zt = (double *)malloc(sizeof(double) * (size_t)V);
  double *zd = (double *)malloc(sizeof(double) * (size_t)V);
  double *p = (double *)malloc(sizeof(double) * (size_t)V);
  double *q = (double *)malloc(sizeof(double) * (size_t)V);
  double *r = (double *)malloc(sizeof(double) * (size_t)V);
  for (int b = 0; b < B; b++) {
    const int32_t *par = parent + (int64_t)b * N;
    const int32_t *tok = tokens + (int64_t)b * N;
    uint32_t fl = 0;
    for (int m = 0; m < N; m++) {
      path[(int64_t)b * N + m] = -1;
      if (acc_margin) acc_margin[(int64_t)b * N + m] = INFINITY;
      if (par[m] < -1 || par[m] >= m) fl |= OR_FLAG_BAD_TREE;
    }
    int node = -1, L = 0;
    double Wlast = 1.0;
    for (;;) {
      const int64_t off = b * seq_stride + (int64_t)(node + 1) * row_stride;
      load_row(target, dtype, off, V, zt);
      load_row(draft, dtype, off, V, zd);
      oracle_softmax(zt, V, T, p);
      oracle_softmax(zd, V, T, q);
      memcpy(r, p, sizeof(double) * (size_t)V);
      Wlast = 1.0;
      int next = -1;
      for (int c = node + 1; c < N && next < 0; c++) {
        if (par[c] != node) continue;
        const int x = tok[c];
        if (x < 0 || x >= V) {
          fl |= OR_FLAG_BAD_TOKEN;
          continue;
        }
        const double u = (double)u_acc[(int64_t)b * N + c];
        if (acc_margin && T != 0.0 && q[x] > 0.0) acc_margin[(int64_t)b * N + c] = fabs(u - r[x] / q[x]);
        if (u * q[x] < r[x]) {
          next = c;
          break;
        }
        double W = 0.0;
        for (int i = 0; i < V; i++) W += (r[i] > q[i]) ? r[i] - q[i] : 0.0;
        if (W > 0.0) {
          for (int i = 0; i < V; i++) r[i] = (r[i] > q[i]) ? (r[i] - q[i]) / W : 0.0;
          Wlast = W;
        } else {
          fl |= OR_FLAG_ZERO_RESIDUAL;
        }
      }
      if (next >= 0) {
        path[(int64_t)b * N + L] = next;
        L++;
        node = next;
        continue;
      }
      double bm = INFINITY;
      bonus[b] = oracle_inv_cdf(r, V, (double)u_bonus[b], &bm);
      if (bonus_margin) bonus_margin[b] = (T == 0.0) ? INFINITY : bm;
      break;
    }
    accept_len[b] = L;
    if (resid_mass) resid_mass[b] = Wlast;
    if (flags) flags[b] = fl;
  }
  free(zt);
  free(zd);
  free(p);
  free(q);
  free(r);
  return 0;
}

/*
 * spec_oracle.c -- plain CPU oracle for the draft-then-verify acceptance step.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the test-suite, the smoke check and the benchmark's
 * CPU-baseline / reference leg use it.  It shares no code, header, table or
 * helper with the CUDA library; the two meet only through the seeded inputs.
 *
 * Everything is computed in IEEE double, one sequence at a time, in the order
 * the method states its steps.  OpenMP is used only to run independent
 * sequences on different threads; it does not change any arithmetic.
 *
 * Sources (page title, then section):
 *   [SRS]  "推测性拒绝采样" (Speculative rejection sampling), bmjup.com,
 *          sections "技术原理与步骤" steps 2-4 (parallel verify, ratio test,
 *          first rejection, correction token) and "关键保证：输出分布不变"
 *          (the emitted tokens follow the target distribution exactly).
 *   [SCD]  "논문 리뷰 [Speculative Contrastive Decoding]", minair.tistory.com,
 *          section "Speculative Decoding" (gamma+1-th token when every draft
 *          token is accepted).
 *   [BPD]  "Garden | Blockwise Parallel Decoding", sections 3.2 and 3.5
 *          (greedy verify: longest prefix where draft == argmax(target),
 *          then the target's own token at the first mismatch).
 *   [SR]   "Speculative Rejection" review (AI闲谈), section 4.2 "算法", the
 *          speculative-rejection phase: the cut r_cut is the alpha-quantile
 *          of the partial reward scores and the sequences scoring at least
 *          r_cut go on to the next round.
 *
 * Readings where the pages are silent or garbled (each is listed with its
 * reason in the design notes):
 *   - correction token: drawn from normalize(max(0, p - q)) at the first
 *     rejected position.  [SRS] step 4 literally says "sample from P_large";
 *     that contradicts the exactness guarantee of the same page, so the
 *     literal reading is kept only as variant ORACLE_VARIANT_LITERAL_TARGET,
 *     a negative control that the tests show is NOT exact.
 *   - accept test: accept iff u * q(x) < p(x).  For q > 0 this is
 *     u < min(1, p/q); p >= q always accepts (u < 1); p == 0 always rejects;
 *     q == 0 accepts iff p > 0.
 *   - uniforms: u[0..K-1] drive the K accept tests, u[K] is the one uniform
 *     of the correction / bonus draw, whichever row that is.
 *   - inverse CDF: ascending token id, inclusive running sum C_j, the token
 *     is the smallest j with C_j > u[K] * S.  S == 0 at a rejected row
 *     (p == q there) falls back to p.
 *   - temperature divides both the target and the draft logits.
 *   - greedy: argmax of the raw logit values (bf16 widens exactly), lowest
 *     index on ties.
 *   - contrastive target ([SCD] "Speculative Contrastive Decoding"; the
 *     formula was lost from the page, so contrastive_row follows the plain
 *     reading below, pinned by the tests to its verbal definition built
 *     from library softmaxes, to its two limits and by the verify step's
 *     output law):
 *     contrastive decoding's log p_e - log p_a over the plausible head
 *     { p_e >= alpha * max p_e }, normalised there (contrastive_row); the
 *     amateur supplies the draft distribution q and its row K enters only
 *     P_n,K; replacement and bonus come from P_n as in the plain verify.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Constants of this file.  Their numeric values are stated in the public
 * header of the CUDA library as well; the tests compare behaviour, and the
 * two sides never include each other. */
enum { ORACLE_DTYPE_F32 = 0, ORACLE_DTYPE_BF16 = 1 };
enum { ORACLE_MODE_SAMPLE = 0, ORACLE_MODE_GREEDY = 1 };
enum { ORACLE_OK = 0, ORACLE_ERR_INVALID_ARG = 1, ORACLE_ERR_NOMEM = 6 };
enum {
  ORACLE_VARIANT_EXACT = 0,          /* the method as read above            */
  ORACLE_VARIANT_LITERAL_TARGET = 1  /* negative control: correction ~ p_n   */
};
/* data-error bits, per sequence and OR-ed into *status */
enum {
  ORACLE_DATA_TOKEN = 1,     /* draft token outside [0, V)               */
  ORACLE_DATA_LOGIT = 2,     /* NaN / +inf logit, or a row with no mass  */
  ORACLE_DATA_UNIFORM = 4,   /* uniform outside [0, 1) or NaN            */
  ORACLE_DATA_SCORE = 8      /* NaN / infinite reward score (rejection cut) */
};
/* boundary flags, per sequence (sampling mode only) */
enum {
  ORACLE_FLAG_RATIO = 1,     /* |u_i - min(1, p/q)| < band at an evaluated i */
  ORACLE_FLAG_CDF = 2,       /* |u_K - C_j / S| < band, j = chosen or chosen-1 */
  ORACLE_FLAG_TINY_RESIDUAL = 4 /* 0 < S < band at a rejected row          */
};

static const double kBand = 1e-6;

/* One logit as a double: fp32 widens exactly, bf16 is the top half of an
 * fp32 and widens exactly too. */
static double logit_at(const void* base, int dtype, size_t idx) {
  if (dtype == ORACLE_DTYPE_F32) return (double)((const float*)base)[idx];
  uint32_t bits = ((uint32_t)((const uint16_t*)base)[idx]) << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

/* Temperature softmax of one row, three plain passes:
 *   l_j = x_j / T,  M = max_j l_j,  Z = sum_j exp(l_j - M),  p_j = exp(l_j - M) / Z.
 * (The vocabulary projection ends in a softmax: [BPD] section 3.3; the
 * temperature is part of the sampling setup.)
 * Returns 0 on success, ORACLE_DATA_LOGIT when the row holds NaN or +inf or
 * has no finite entry (then p is left all-zero). */
static int row_softmax(const void* base, int dtype, size_t off, int V, double T,
                       double* p) {
  double M = -INFINITY;
  int bad = 0;
  for (int j = 0; j < V; ++j) {
    double x = logit_at(base, dtype, off + (size_t)j);
    if (isnan(x) || (isinf(x) && x > 0)) bad = 1;
    double l = x / T;
    if (l > M) M = l;
  }
  if (bad || !(M > -INFINITY)) {
    for (int j = 0; j < V; ++j) p[j] = 0.0;
    return ORACLE_DATA_LOGIT;
  }
  double Z = 0.0;
  for (int j = 0; j < V; ++j) {
    double l = logit_at(base, dtype, off + (size_t)j) / T;
    Z += exp(l - M);
  }
  for (int j = 0; j < V; ++j) {
    double l = logit_at(base, dtype, off + (size_t)j) / T;
    p[j] = exp(l - M) / Z;
  }
  return 0;
}

/* Inverse-CDF draw from the unnormalised non-negative weights r[0..V-1]:
 * the smallest j whose inclusive running sum exceeds u * S, S = sum r.
 * *flag gets ORACLE_FLAG_CDF when u lies within kBand of C_{j-1}/S or C_j/S.
 * S must be > 0. */
static int inverse_cdf(const double* r, int V, double u, uint32_t* flag) {
  double S = 0.0;
  for (int j = 0; j < V; ++j) S += r[j];
  double theta = u * S;
  double C = 0.0, C_prev = 0.0;
  int chosen = -1;
  for (int j = 0; j < V; ++j) {
    C_prev = C;
    C += r[j];
    if (C > theta) { chosen = j; break; }
  }
  if (chosen < 0) {
    /* u * S >= S cannot happen for u < 1; kept for a defined answer. */
    for (int j = V - 1; j >= 0; --j)
      if (r[j] > 0) { chosen = j; break; }
    if (chosen < 0) chosen = 0;
    C_prev = C;
  }
  if (fabs(u - C_prev / S) < kBand || fabs(u - C / S) < kBand) *flag |= ORACLE_FLAG_CDF;
  return chosen;
}

/* One sequence in sampling mode ([SRS] steps 2-4, [SCD] "Speculative
 * Decoding").  Rows: target t[b, 0..K], draft d[b, 0..K-1]. */
static int verify_one_sample(const void* target, const void* draft, const int32_t* x,
                             const float* u, int K, int V, int dtype, double T,
                             int variant, size_t b, int32_t* n_out, int32_t* out,
                             double* p_at, double* q_at, uint32_t* flag_out) {
  int status = 0;
  uint32_t flag = 0;
  for (int i = 0; i < K; ++i)
    if (x[i] < 0 || x[i] >= V) status |= ORACLE_DATA_TOKEN;
  for (int i = 0; i <= K; ++i)
    if (!(u[i] >= 0.0f && u[i] < 1.0f)) status |= ORACLE_DATA_UNIFORM;

  double* p = (double*)malloc(sizeof(double) * (size_t)V);
  double* q = (double*)malloc(sizeof(double) * (size_t)V);
  double* r = (double*)malloc(sizeof(double) * (size_t)V);
  double* px = (double*)malloc(sizeof(double) * (size_t)(K + 1));
  double* qx = (double*)malloc(sizeof(double) * (size_t)(K + 1));
  if (!p || !q || !r || !px || !qx) {
    free(p); free(q); free(r); free(px); free(qx);
    return -1;
  }

  /* Every row is read and checked, as the parallel verify step reads all of
   * them ([SRS] step 2); p_i(x_i) and q_i(x_i) are kept for every position. */
  for (int i = 0; i <= K; ++i) {
    size_t off_t = (b * (size_t)(K + 1) + (size_t)i) * (size_t)V;
    status |= row_softmax(target, dtype, off_t, V, T, p);
    if (i == K) break;
    size_t off_d = (b * (size_t)K + (size_t)i) * (size_t)V;
    status |= row_softmax(draft, dtype, off_d, V, T, q);
    int xi = (x[i] >= 0 && x[i] < V) ? x[i] : 0;
    px[i] = p[xi];
    qx[i] = q[xi];
    if (p_at && q_at) {
      p_at[b * (size_t)K + (size_t)i] = px[i];
      q_at[b * (size_t)K + (size_t)i] = qx[i];
    }
  }
  if (status) {
    *n_out = -1;
    for (int i = 0; i <= K; ++i) out[i] = -1;
    *flag_out = 0;
    free(p); free(q); free(r); free(px); free(qx);
    return status;
  }

  /* Ratio test in order; stop at the first rejection ([SRS] step 3). */
  int n = K;
  for (int i = 0; i < K; ++i) {
    double ui = (double)u[i];
    if (qx[i] > 0.0) {
      double ratio = px[i] / qx[i];
      if (ratio > 1.0) ratio = 1.0;
      if (fabs(ui - ratio) < kBand) flag |= ORACLE_FLAG_RATIO;
    }
    int accept = ui * qx[i] < px[i];
    if (!accept) { n = i; break; }
  }

  /* Correction at the first rejection ([SRS] step 4, exactness guarantee),
   * or the extra token from the target when all K were accepted
   * ([SCD] "Speculative Decoding"). */
  int chosen;
  double uK = (double)u[K];
  size_t off_tn = (b * (size_t)(K + 1) + (size_t)n) * (size_t)V;
  row_softmax(target, dtype, off_tn, V, T, p);
  if (n < K) {
    if (variant == ORACLE_VARIANT_LITERAL_TARGET) {
      chosen = inverse_cdf(p, V, uK, &flag);
    } else {
      size_t off_dn = (b * (size_t)K + (size_t)n) * (size_t)V;
      row_softmax(draft, dtype, off_dn, V, T, q);
      double S = 0.0;
      for (int j = 0; j < V; ++j) {
        double d = p[j] - q[j];
        r[j] = d > 0.0 ? d : 0.0;
        S += r[j];
      }
      if (S > 0.0 && S < kBand) flag |= ORACLE_FLAG_TINY_RESIDUAL;
      if (S > 0.0) chosen = inverse_cdf(r, V, uK, &flag);
      else chosen = inverse_cdf(p, V, uK, &flag);
    }
  } else {
    chosen = inverse_cdf(p, V, uK, &flag);
  }

  *n_out = n;
  for (int i = 0; i < n; ++i) out[i] = x[i];
  out[n] = chosen;
  for (int i = n + 1; i <= K; ++i) out[i] = -1;
  *flag_out = flag;
  free(p); free(q); free(r); free(px); free(qx);
  return 0;
}

/* The contrastive target of one position ([SCD] "Speculative Contrastive
 * Decoding": the expert's distribution replaced by the contrastive-decoding
 * distribution P_n of the expert Me and the amateur Ma; the formula itself
 * did not survive on the page, so this is the plain reading of contrastive
 * decoding):
 *   head  = { j : t_j > -inf and t_j >= M + L },  M = max_j t_j,
 *           L = T * ln(alpha)  (p_e(j) >= alpha * max p_e, with p_e =
 *           softmax(t / T); alpha = 0 gives L = -inf: every finite t_j),
 *   P_n(j) = exp((t_j - a_j) / T) / Z  on the head, 0 elsewhere
 *           (log p_e - log p_a up to a constant, normalised over the head).
 * The caller passes L.  Returns ORACLE_DATA_LOGIT (P all-zero) when either
 * row holds NaN or +inf, the target row has no finite entry, or a head token
 * has a_j = -inf (an unbounded contrast). */
static int contrastive_row(const void* target, const void* amateur, int dtype, size_t off,
                           int V, double T, double L, double* P) {
  double M = -INFINITY;
  int bad = 0;
  for (int j = 0; j < V; ++j) {
    const double t = logit_at(target, dtype, off + (size_t)j);
    const double a = logit_at(amateur, dtype, off + (size_t)j);
    if (isnan(t) || (isinf(t) && t > 0) || isnan(a) || (isinf(a) && a > 0)) bad = 1;
    if (t > M) M = t;
  }
  const double thr = M + L;
  double Mc = -INFINITY;
  if (!bad && M > -INFINITY) {
    for (int j = 0; j < V; ++j) {
      const double t = logit_at(target, dtype, off + (size_t)j);
      if (!(t > -INFINITY && t >= thr)) continue;
      const double a = logit_at(amateur, dtype, off + (size_t)j);
      if (!(a > -INFINITY)) { bad = 1; break; }
      const double c = (t - a) / T;
      if (c > Mc) Mc = c;
    }
  }
  if (bad || !(M > -INFINITY)) {
    for (int j = 0; j < V; ++j) P[j] = 0.0;
    return ORACLE_DATA_LOGIT;
  }
  double Z = 0.0;
  for (int j = 0; j < V; ++j) {
    const double t = logit_at(target, dtype, off + (size_t)j);
    if (t > -INFINITY && t >= thr) {
      const double a = logit_at(amateur, dtype, off + (size_t)j);
      P[j] = exp((t - a) / T - Mc);
      Z += P[j];
    } else {
      P[j] = 0.0;
    }
  }
  for (int j = 0; j < V; ++j) P[j] /= Z;
  return 0;
}

/* One sequence of speculative contrastive decoding ([SCD] "Speculative
 * Contrastive Decoding"): speculative sampling with the target p_i replaced
 * by the contrastive P_n,i, including the bonus draw at position K.  The
 * draft tokens come from the amateur, q_i = softmax(a_i / T); its rows are
 * a[b, 0..K] (row K only enters P_n,K).  The steps and flags are those of
 * verify_one_sample. */
static int scd_one(const void* target, const void* amateur, const int32_t* x, const float* u,
                   int K, int V, int dtype, double T, double L, size_t b, int32_t* n_out,
                   int32_t* out, double* p_at, double* q_at, uint32_t* flag_out) {
  int status = 0;
  uint32_t flag = 0;
  for (int i = 0; i < K; ++i)
    if (x[i] < 0 || x[i] >= V) status |= ORACLE_DATA_TOKEN;
  for (int i = 0; i <= K; ++i)
    if (!(u[i] >= 0.0f && u[i] < 1.0f)) status |= ORACLE_DATA_UNIFORM;
  double* p = (double*)malloc(sizeof(double) * (size_t)V);
  double* q = (double*)malloc(sizeof(double) * (size_t)V);
  double* r = (double*)malloc(sizeof(double) * (size_t)V);
  double* px = (double*)malloc(sizeof(double) * (size_t)(K + 1));
  double* qx = (double*)malloc(sizeof(double) * (size_t)(K + 1));
  if (!p || !q || !r || !px || !qx) {
    free(p); free(q); free(r); free(px); free(qx);
    return -1;
  }
  for (int i = 0; i <= K; ++i) {
    const size_t off = (b * (size_t)(K + 1) + (size_t)i) * (size_t)V;
    status |= contrastive_row(target, amateur, dtype, off, V, T, L, p);
    if (i == K) break;
    status |= row_softmax(amateur, dtype, off, V, T, q);
    const int xi = (x[i] >= 0 && x[i] < V) ? x[i] : 0;
    px[i] = p[xi];
    qx[i] = q[xi];
    if (p_at && q_at) {
      p_at[b * (size_t)K + (size_t)i] = px[i];
      q_at[b * (size_t)K + (size_t)i] = qx[i];
    }
  }
  if (status) {
    *n_out = -1;
    for (int i = 0; i <= K; ++i) out[i] = -1;
    *flag_out = 0;
    free(p); free(q); free(r); free(px); free(qx);
    return status;
  }
  int n = K;
  for (int i = 0; i < K; ++i) {
    const double ui = (double)u[i];
    if (qx[i] > 0.0) {
      double ratio = px[i] / qx[i];
      if (ratio > 1.0) ratio = 1.0;
      if (fabs(ui - ratio) < kBand) flag |= ORACLE_FLAG_RATIO;
    }
    if (!(ui * qx[i] < px[i])) { n = i; break; }
  }
  const double uK = (double)u[K];
  const size_t off_n = (b * (size_t)(K + 1) + (size_t)n) * (size_t)V;
  contrastive_row(target, amateur, dtype, off_n, V, T, L, p);
  int chosen;
  if (n < K) {
    row_softmax(amateur, dtype, off_n, V, T, q);
    double S = 0.0;
    for (int j = 0; j < V; ++j) {
      const double d = p[j] - q[j];
      r[j] = d > 0.0 ? d : 0.0;
      S += r[j];
    }
    if (S > 0.0 && S < kBand) flag |= ORACLE_FLAG_TINY_RESIDUAL;
    chosen = S > 0.0 ? inverse_cdf(r, V, uK, &flag) : inverse_cdf(p, V, uK, &flag);
  } else {
    chosen = inverse_cdf(p, V, uK, &flag);
  }
  *n_out = n;
  for (int i = 0; i < n; ++i) out[i] = x[i];
  out[n] = chosen;
  for (int i = n + 1; i <= K; ++i) out[i] = -1;
  *flag_out = flag;
  free(p); free(q); free(r); free(px); free(qx);
  return 0;
}

/* One sequence in greedy mode ([BPD] sections 3.2 "Accept" and 3.5): g_i is
 * the argmax of target row i (lowest index on ties); n is the first i < K
 * with x_i != g_i, else K; emit x_0..x_{n-1} then g_n. */
static int verify_one_greedy(const void* target, const int32_t* x, int K, int V,
                             int dtype, size_t b, int32_t* n_out, int32_t* out) {
  int status = 0;
  for (int i = 0; i < K; ++i)
    if (x[i] < 0 || x[i] >= V) status |= ORACLE_DATA_TOKEN;
  int* g = (int*)malloc(sizeof(int) * (size_t)(K + 1));
  if (!g) return -1;
  for (int i = 0; i <= K; ++i) {
    size_t off = (b * (size_t)(K + 1) + (size_t)i) * (size_t)V;
    double best = logit_at(target, dtype, off);
    int arg = 0;
    for (int j = 0; j < V; ++j) {
      double v = logit_at(target, dtype, off + (size_t)j);
      if (isnan(v) || (isinf(v) && v > 0)) status |= ORACLE_DATA_LOGIT;
      if (v > best) { best = v; arg = j; }
    }
    g[i] = arg;
  }
  if (status) {
    *n_out = -1;
    for (int i = 0; i <= K; ++i) out[i] = -1;
    free(g);
    return status;
  }
  int n = K;
  for (int i = 0; i < K; ++i)
    if (x[i] != g[i]) { n = i; break; }
  *n_out = n;
  for (int i = 0; i < n; ++i) out[i] = x[i];
  out[n] = g[n];
  for (int i = n + 1; i <= K; ++i) out[i] = -1;
  free(g);
  return 0;
}

/*
 * Batched entry point.  Host pointers, row-major contiguous:
 *   target   [B, K+1, V]  fp32 or bf16 (raw uint16 bits)
 *   draft    [B, K,   V]  same dtype; unused (may be NULL) in greedy mode
 *   tokens   [B, K]       int32
 *   uniforms [B, K+1]     fp32; unused (may be NULL) in greedy mode
 * Outputs:
 *   accepted_len [B]      n in [0, K]; -1 for a sequence with a data error
 *   out_tokens   [B, K+1] n+1 tokens then -1
 *   p_at, q_at   [B, K]   p_i(x_i), q_i(x_i) in double (optional, sampling)
 *   flags        [B]      ORACLE_FLAG_* bits (optional, sampling)
 *   status       OR of ORACLE_DATA_* over the batch (optional)
 * Returns ORACLE_OK, ORACLE_ERR_INVALID_ARG or ORACLE_ERR_NOMEM.
 */
int spec_oracle_verify(const void* target, const void* draft, const int32_t* tokens,
                       const float* uniforms, int B, int K, int V, int dtype,
                       double temperature, int mode, int variant,
                       int32_t* accepted_len, int32_t* out_tokens, double* p_at,
                       double* q_at, uint32_t* flags, int32_t* status) {
  if (B < 0 || K < 0 || V < 1) return ORACLE_ERR_INVALID_ARG;
  if (dtype != ORACLE_DTYPE_F32 && dtype != ORACLE_DTYPE_BF16) return ORACLE_ERR_INVALID_ARG;
  if (mode != ORACLE_MODE_SAMPLE && mode != ORACLE_MODE_GREEDY) return ORACLE_ERR_INVALID_ARG;
  if (B == 0) { if (status) *status = 0; return ORACLE_OK; }
  if (!target || (K > 0 && !tokens) || !accepted_len || !out_tokens) return ORACLE_ERR_INVALID_ARG;
  if (mode == ORACLE_MODE_SAMPLE) {
    if ((K > 0 && !draft) || !uniforms) return ORACLE_ERR_INVALID_ARG;
    if (!(temperature > 0.0) || isinf(temperature)) return ORACLE_ERR_INVALID_ARG;
  }
  int total = 0, nomem = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : total) reduction(| : nomem)
  for (long long bb = 0; bb < (long long)B; ++bb) {
    size_t b = (size_t)bb;
    const int32_t* x = tokens ? tokens + b * (size_t)K : NULL;
    int32_t* out = out_tokens + b * (size_t)(K + 1);
    int st;
    if (mode == ORACLE_MODE_GREEDY) {
      st = verify_one_greedy(target, x, K, V, dtype, b, &accepted_len[b], out);
      if (flags) flags[b] = 0;
    } else {
      uint32_t f = 0;
      st = verify_one_sample(target, draft, x, uniforms + b * (size_t)(K + 1), K, V,
                             dtype, temperature, variant, b, &accepted_len[b], out,
                             p_at, q_at, &f);
      if (flags) flags[b] = f;
    }
    if (st < 0) nomem = 1;
    else total |= st;
  }
  if (status) *status = total;
  return nomem ? ORACLE_ERR_NOMEM : ORACLE_OK;
}

/* Speculative contrastive decoding over B sequences (scd_one); target and
 * amateur are both [B, K+1, V]; alpha in [0, 1] is the plausibility cut of
 * the contrastive head.  Outputs and status as spec_oracle_verify. */
int spec_oracle_scd_verify(const void* target, const void* amateur, const int32_t* tokens,
                           const float* uniforms, int B, int K, int V, int dtype,
                           double temperature, double alpha, int32_t* accepted_len,
                           int32_t* out_tokens, double* p_at, double* q_at, uint32_t* flags,
                           int32_t* status) {
  if (B < 0 || K < 0 || V < 1) return ORACLE_ERR_INVALID_ARG;
  if (dtype != ORACLE_DTYPE_F32 && dtype != ORACLE_DTYPE_BF16) return ORACLE_ERR_INVALID_ARG;
  if (!(temperature > 0.0) || isinf(temperature)) return ORACLE_ERR_INVALID_ARG;
  if (!(alpha >= 0.0 && alpha <= 1.0)) return ORACLE_ERR_INVALID_ARG;
  if (B == 0) { if (status) *status = 0; return ORACLE_OK; }
  if (!target || !amateur || (K > 0 && !tokens) || !uniforms || !accepted_len || !out_tokens)
    return ORACLE_ERR_INVALID_ARG;
  const double L = alpha > 0.0 ? temperature * log(alpha) : -INFINITY;
  int total = 0, nomem = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : total) reduction(| : nomem)
  for (long long bb = 0; bb < (long long)B; ++bb) {
    const size_t b = (size_t)bb;
    uint32_t f = 0;
    const int st = scd_one(target, amateur, tokens ? tokens + b * (size_t)K : NULL,
                           uniforms + b * (size_t)(K + 1), K, V, dtype, temperature, L, b,
                           &accepted_len[b], out_tokens + b * (size_t)(K + 1), p_at, q_at, &f);
    if (flags) flags[b] = f;
    if (st < 0) nomem = 1;
    else total |= st;
  }
  if (status) *status = total;
  return nomem ? ORACLE_ERR_NOMEM : ORACLE_OK;
}

/* The drafter's own sampling step, the one before verification ([SRS]
 * 技术原理与步骤 step 1, the draft model proposes its tokens; [SCD]
 * "Speculative Decoding": x_i is sampled from the draft's distribution):
 * for each of R rows, q = softmax(row / T) and x = the inverse-CDF draw of
 * q with u[r] (the same rule as the verifier's draws); q_at[r] = q(x).
 * flags[r] gets ORACLE_FLAG_CDF near a CDF step; a row with NaN / +inf or no
 * finite entry sets ORACLE_DATA_LOGIT in *status (token 0, q_at 0), a
 * uniform outside [0, 1) ORACLE_DATA_UNIFORM. */
int spec_oracle_draft_sample(const void* logits, const float* uniforms, int R, int V, int dtype,
                             double temperature, int32_t* tokens, double* q_at, uint32_t* flags,
                             int32_t* status) {
  if (!logits || !uniforms || !tokens || R < 0 || V < 1 || !(temperature > 0.0))
    return ORACLE_ERR_INVALID_ARG;
  int total = 0, nomem = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : total) reduction(| : nomem)
  for (int r = 0; r < R; ++r) {
    double* p = (double*)malloc(sizeof(double) * (size_t)V);
    if (!p) { nomem = 1; continue; }
    uint32_t fl = 0;
    int tok = 0;
    double qx = 0.0;
    int st = row_softmax(logits, dtype, (size_t)r * (size_t)V, V, temperature, p);
    const double u = (double)uniforms[r];
    if (!(u >= 0.0 && u < 1.0)) st |= ORACLE_DATA_UNIFORM;
    if (!(st & ORACLE_DATA_LOGIT)) {
      tok = inverse_cdf(p, V, u >= 0.0 && u < 1.0 ? u : 0.0, &fl);
      qx = p[tok];
    }
    tokens[r] = tok;
    if (q_at) q_at[r] = qx;
    if (flags) flags[r] = fl;
    total |= st;
    free(p);
  }
  if (status) *status = total;
  return nomem ? ORACLE_ERR_NOMEM : ORACLE_OK;
}

/* Ascending order of doubles for qsort. */
static int cmp_double(const void* a, const void* b) {
  const double x = *(const double*)a, y = *(const double*)b;
  return (x > y) - (x < y);
}

/* Speculative Rejection's cut ([SR] 4.2, the speculative-rejection phase),
 * for G independent prompts of N partial reward scores each (scores [G, N]).
 *
 * Readings: the alpha-quantile is the usual one of sorted samples with
 * linear interpolation between neighbouring order statistics (position
 * h = alpha * (N - 1), 0-based), and a sequence is kept when its score is
 * at least r_cut.  So, per prompt, with s the scores sorted ascending,
 *   j = floor(h), g = h - j, r_cut = s[j] + g * (s[min(j + 1, N - 1)] - s[j])
 * in IEEE double (no fused multiply-add), and accepted[] lists, in ascending
 * order, every index k with scores[k] >= r_cut; the rest of the row is -1.
 * A prompt with a NaN or infinite score sets ORACLE_DATA_SCORE in *status
 * and gets r_cut = NaN, n_accepted = 0 and a row of -1. */
int spec_oracle_rejection_cut(const float* scores, int G, int N, double alpha, double* r_cut,
                              int32_t* n_accepted, int32_t* accepted, int32_t* status) {
  if (G < 0 || N < 0 || !(alpha >= 0.0 && alpha <= 1.0)) return ORACLE_ERR_INVALID_ARG;
  if (G == 0) { if (status) *status = 0; return ORACLE_OK; }
  if (N < 1 || !scores || !r_cut || !n_accepted || !accepted) return ORACLE_ERR_INVALID_ARG;
  const double h = alpha * (double)(N - 1);
  const double jf = floor(h);
  const int j = (int)jf;
  const double g = h - jf;
  int total = 0, nomem = 0;
#pragma omp parallel for schedule(dynamic, 16) reduction(| : total) reduction(| : nomem)
  for (int pr = 0; pr < G; ++pr) {
    const float* row = scores + (size_t)pr * (size_t)N;
    int32_t* out = accepted + (size_t)pr * (size_t)N;
    double* s = (double*)malloc(sizeof(double) * (size_t)N);
    if (!s) { nomem = 1; continue; }
    int bad = 0;
    for (int k = 0; k < N; ++k) {
      s[k] = (double)row[k];
      if (!isfinite(s[k])) bad = 1;
    }
    int n = 0;
    if (bad) {
      r_cut[pr] = NAN;
      total |= ORACLE_DATA_SCORE;
    } else {
      qsort(s, (size_t)N, sizeof(double), cmp_double);
      const double lo = s[j];
      const double hi = s[j + 1 < N ? j + 1 : N - 1];
      const double r = lo + g * (hi - lo);
      r_cut[pr] = r;
      for (int k = 0; k < N; ++k)
        if ((double)row[k] >= r) out[n++] = k;
    }
    n_accepted[pr] = n;
    for (int k = n; k < N; ++k) out[k] = -1;
    free(s);
  }
  if (status) *status = total;
  return nomem ? ORACLE_ERR_NOMEM : ORACLE_OK;
}

/* The temperature softmax of one row, for the tests that pin it against a
 * library softmax.  Returns ORACLE_DATA_LOGIT for a row it refuses. */
int spec_oracle_softmax(const void* row, int V, int dtype, double temperature, double* p) {
  if (!row || !p || V < 1 || !(temperature > 0.0)) return ORACLE_ERR_INVALID_ARG;
  return row_softmax(row, dtype, 0, V, temperature, p);
}

/* Threads the oracle's parallel loop will use (reported as the CPU
 * baseline's core count), and a way to pin it. */
int spec_oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

void spec_oracle_set_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

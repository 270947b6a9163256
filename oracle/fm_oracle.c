/*
 * fm_oracle.c -- plain, slow, fp64 CPU oracle for fixed-m (const-max) attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or load
 * this file; only the tests, the smoke check and the bench's CPU-baseline leg do.
 * It shares no code, header or constant with the CUDA library.
 *
 * Sources (cited by page title and section):
 *   [NKI]    "Kernel reference: ring_attention_const_max_fwd const-max ring attention"
 *            (AWS Neuron docs), sections "What you should know before reading",
 *            "Picking a max that is safe without measuring it",
 *            "A static bound makes the ring reduction pure addition",
 *            "Accumulate, then normalize once", "Adapting this kernel" (key sinks).
 *   [PR477]  "feat(attention): fixed-m splash attention kernel with dynamic bounds and
 *            safety fallbacks" (maxdiffusion PR #477), Summary: "Dynamic eligibility
 *            bounding" equations for C(N), W(N), gate, m_i, U_i and the invariant;
 *            "Virtual K-centering"; "Centering and the Cauchy-Schwarz bound are a
 *            matched pair"; the commit message's V-safety predicate (|V| <= 256,
 *            fp16 rejected).
 *   [PR478]  "feat(attention): 2D Ulysses+Ring attention with Global Virtual
 *            K-Centering" (maxdiffusion PR #478), Summary: key mean over real tokens.
 *
 * What each function computes:
 *   fmo_attention   -- softmax attention by its plain definition.  Fixed-m reaches
 *                      this exactly (up to rounding) because the shift and the
 *                      centering term are per-row constants ([NKI] "softmax shift
 *                      invariance"; [PR477] "Virtual K-centering").  So the oracle
 *                      for the OUTPUT is plain attention, with the textbook max
 *                      subtraction, over the full (concatenated) key sequence.
 *   fmo_constants   -- C(N), W(N), gate from [PR477] Summary.
 *   fmo_bounds      -- norms, key mean, U, m, flag, in the pages' order ([PR477]);
 *                      optionally the key sinks left out of the key max ([NKI]
 *                      "Adapting this kernel").
 *   fmo_attention_bf16p -- the same attention with every numerator weight rounded to
 *                      bf16's 8-bit significand: the "bf16 reference" whose error
 *                      distribution [NKI] "Adapting this kernel" (Validation) tells you to
 *                      compare a kernel's against.  The weight's scale is a per-row shift
 *                      passed in (the fixed-m shift of fmo_bounds, or the row max).
 *   fmo_fixed_m_emulate_f32 -- a sequential fp32 emulation of the fixed-m sum with
 *                      an ARBITRARY shift, flushing subnormal terms to zero.  It
 *                      exists only to show what goes wrong with a wrong gate or an
 *                      unmatched bound ([PR477] "Why the gate is halved", and
 *                      "matched pair"); it is not a model of the CUDA kernels.
 *
 * Parity pins: every function here is pinned by tests that check it against
 * closed forms, invariants, brute force and the values the pages print; none is
 * "parity unpinned" except the single 0.882 mass figure of [PR477], which the page
 * prints without the key set it came from (the gate decision itself is pinned).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define FMO_LOG2E 1.4426950408889634073599246810018921 /* log2(e) */

/* ceil(log2 n) for n >= 1, as the bit length of n-1. */
int fmo_ceil_log2(int64_t n) {
  if (n <= 1) return 0;
  uint64_t x = (uint64_t)(n - 1);
  int b = 0;
  while (x) { b++; x >>= 1; }
  return b;
}

/* [PR477] Summary, "Dynamic eligibility bounding":
 *   C(N) = 127 - ceil(log2 N) - ceil(log2 Vmax),  W(N) = C(N) + 125,  gate = floor(W/2). */
void fmo_constants(int64_t n_total, int64_t vmax, int *C, int *W, int *gate) {
  int c = 127 - fmo_ceil_log2(n_total) - fmo_ceil_log2(vmax);
  int w = c + 125;
  *C = c;
  *W = w;
  /* floor division, correct for negative w too */
  *gate = (w >= 0) ? (w / 2) : -((-w + 1) / 2);
}

/* qsort comparator: descending doubles */
static int fmo_cmp_desc(const void *a, const void *b) {
  double x = *(const double *)a, y = *(const double *)b;
  return (x < y) - (x > y);
}

int fmo_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Plain softmax attention, one independent problem per g (a (batch, head) pair).
 *   q   : [G, R, D]   the query rows to evaluate (any subset of a head's rows)
 *   k,v : [G, N, D]   all keys / values of that head, all chunks concatenated
 *   o   : [G, R, D]   o_i = sum_j exp(s_ij - mu_i) v_j / sum_j exp(s_ij - mu_i)
 *   lse : [G, R] or NULL; natural-log log-sum-exp of the scaled scores
 * with s_ij = scale * q_i . k_j and mu_i = max_j s_ij.  N == 0 gives o = 0 and
 * lse = -inf.  nthreads <= 0 means "all available". */
void fmo_attention(const double *q, const double *k, const double *v, int64_t G, int64_t R,
                   int64_t N, int64_t D, double scale, double *o, double *lse, int nthreads) {
#ifdef _OPENMP
  /* a per-call team size: omp_set_num_threads would stay in force for later calls */
  const int nt = nthreads > 0 ? nthreads : omp_get_max_threads();
#else
  (void)nthreads;
#endif
  int64_t total = G * R;
#pragma omp parallel num_threads(nt)
  {
    double *s = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
#pragma omp for schedule(dynamic, 1)
    for (int64_t gr = 0; gr < total; gr++) {
      int64_t g = gr / R;
      const double *qi = q + gr * D;
      const double *kg = k + g * N * D;
      const double *vg = v + g * N * D;
      double *oi = o + gr * D;
      for (int64_t d = 0; d < D; d++) oi[d] = 0.0;
      if (N == 0) {
        if (lse) lse[gr] = -INFINITY;
        continue;
      }
      double mu = -INFINITY;
      for (int64_t j = 0; j < N; j++) {
        double dot = 0.0;
        for (int64_t d = 0; d < D; d++) dot += qi[d] * kg[j * D + d];
        s[j] = scale * dot;
        if (s[j] > mu) mu = s[j];
      }
      double denom = 0.0;
      for (int64_t j = 0; j < N; j++) {
        double e = exp(s[j] - mu);
        denom += e;
        for (int64_t d = 0; d < D; d++) oi[d] += e * vg[j * D + d];
      }
      for (int64_t d = 0; d < D; d++) oi[d] /= denom;
      if (lse) lse[gr] = mu + log(denom);
    }
    free(s);
  }
}

/* x > 0 rounded to 8 significant bits (bf16's significand: 1 implicit + 7 stored bits),
 * to nearest with ties to even.  Only the significand is rounded, there is no exponent
 * limit: the callers pass values in [1, 2). */
static double fmo_round_sig8(double x) {
  int e;
  const double m = frexp(x, &e); /* x = m * 2^e, m in [0.5, 1) */
  const double t = m * 256.0;    /* [128, 256): the 8 kept bits above the binary point */
  double r = floor(t);
  const double d = t - r;
  if (d > 0.5 || (d == 0.5 && fmod(r, 2.0) != 0.0)) r += 1.0;
  return ldexp(r / 256.0, e);
}

/* Attention with bf16 P: the reference run "in bf16" of [NKI] "Adapting this kernel"
 * (Validation: run exact attention on the CPU in fp32 and in bf16 and compare both error
 * distributions with the kernel's).  Reading: what bf16 changes is the probability weights
 * that multiply V.  Weight j of row i is p_ij = 2^(z_ij - b_i), z_ij = alpha q_i.k_j the
 * base-2 logit (alpha = scale*log2 e) and b_i the row's shift; it enters the numerator
 * rounded to 8 significant bits and the denominator unrounded:
 *   o_i = sum_j bf16(p_ij) v_j / sum_j p_ij.
 * Rounding commutes with a power of two, so bf16(p) = 2^floor(t) * bf16(2^frac(t)) for
 * t = z - b: the rounding depends on frac(z - b) alone, and each weight is formed as
 * 2^(z - mu) times the factor bf16(2^f)/2^f, with mu the row max, so that nothing
 * overflows whatever b is.  Everything else is fp64.
 *   q [G, R, D], k, v [G, N, D], shift [G, R] base-2 shifts or NULL for the row max
 *   o [G, R, D].  N == 0 gives o = 0.                                                    */
void fmo_attention_bf16p(const double *q, const double *k, const double *v, int64_t G, int64_t R,
                         int64_t N, int64_t D, double scale, const double *shift, double *o,
                         int nthreads) {
#ifdef _OPENMP
  const int nt = nthreads > 0 ? nthreads : omp_get_max_threads();
#else
  (void)nthreads;
#endif
  const double alpha = scale * FMO_LOG2E;
  int64_t total = G * R;
#pragma omp parallel num_threads(nt)
  {
    double *z = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
#pragma omp for schedule(dynamic, 1)
    for (int64_t gr = 0; gr < total; gr++) {
      int64_t g = gr / R;
      const double *qi = q + gr * D;
      const double *kg = k + g * N * D;
      const double *vg = v + g * N * D;
      double *oi = o + gr * D;
      for (int64_t d = 0; d < D; d++) oi[d] = 0.0;
      if (N == 0) continue;
      double mu = -INFINITY;
      for (int64_t j = 0; j < N; j++) {
        double dot = 0.0;
        for (int64_t d = 0; d < D; d++) dot += qi[d] * kg[j * D + d];
        z[j] = alpha * dot;
        if (z[j] > mu) mu = z[j];
      }
      const double b = shift ? shift[gr] : mu;
      double denom = 0.0;
      for (int64_t j = 0; j < N; j++) {
        const double p = exp2(z[j] - mu);
        const double t = z[j] - b;
        const double f = t - floor(t);
        const double e2f = exp2(f);
        const double w = p * (fmo_round_sig8(e2f) / e2f);
        denom += p;
        for (int64_t d = 0; d < D; d++) oi[d] += w * vg[j * D + d];
      }
      for (int64_t d = 0; d < D; d++) oi[d] /= denom;
    }
    free(z);
  }
}

/* Bounds in the order of [PR477] (norms -> U -> m, gate -> flag), in fp64.
 * One problem per g (a (batch, head) pair); rows of a problem form Q-blocks of bq rows.
 *   q : [G, Sq, D], k, v : [G, N, D]  (all keys of the head, all chunks)
 *   centering   : 1 = measure keys as k_j - kbar ([PR477] "Virtual K-centering",
 *                 [PR478] key mean over real tokens), 0 = raw keys
 *   dtype_safe  : 1 for bf16/fp32 inputs, 0 for fp16/fp8 ([PR477] commit message)
 *   vmax        : the V bound (256 in the pages)
 * Outputs:
 *   qmax_sq [G, nqb]  max over the block's rows of ||q_i||^2
 *   kbar    [G, D]    mean key (zeros when centering == 0)
 *   kmax_sq [G]       max_j ||k_j - kbar||^2 (or ||k_j||^2)
 *   vmax_sq [1]       max over all elements of v^2 (all problems)
 *   U       [G, nqb]  alpha * sqrt(qmax_sq) * sqrt(kmax_sq), alpha = scale*log2(e):
 *                     the Cauchy-Schwarz bound on the base-2 logit z = alpha q.k
 *   m       [G, nqb]  ceil(U) - C
 *   flag    [G, nqb]  v_ok && U <= gate
 *   qkbar   [G, Sq] or NULL: alpha * q_i . kbar (the per-row centering term)
 *   consts  [4]       C, W, gate, v_ok
 *   U_row, m_row [G, Sq] or NULL: the per-row bound alpha*|q_i|*sqrt(kmax_sq) and its shift
 *   shift   [G, Sq] or NULL: m (per_row ? m_row : the row's Q-block m) + qkbar
 *   n_sink  : 0, or the number of loudest keys per problem left out of the key max
 *   sink_idx [G, n_sink]: those keys' indices, ascending, padded with INT32_MAX
 *   sink_gap [G] or NULL: n_sink-th largest squared key norm minus the (n_sink+1)-th  */
void fmo_bounds(const double *q, const double *k, const double *v, int64_t G, int64_t Sq,
                int64_t N, int64_t D, int64_t bq, double scale, int centering,
                int dtype_safe, int64_t vmax, double *qmax_sq, double *kbar,
                double *kmax_sq, double *vmax_sq, double *U, int32_t *m, uint8_t *flag,
                double *qkbar, int32_t *consts, int per_row, double *U_row, int32_t *m_row,
                double *shift, int64_t n_sink, int32_t *sink_idx, double *sink_gap) {
  const double alpha = scale * FMO_LOG2E;
  int C, W, gate;
  fmo_constants(N, vmax, &C, &W, &gate);
  int64_t nqb = (Sq + bq - 1) / bq;

  /* V magnitude over everything ([PR477] commit message: |V| <= 256). */
  double vm = 0.0;
  for (int64_t i = 0; i < G * N * D; i++) {
    double x = v[i] * v[i];
    if (x > vm) vm = x;
  }
  *vmax_sq = vm;
  int v_ok = dtype_safe && (vm <= (double)vmax * (double)vmax);

  for (int64_t g = 0; g < G; g++) {
    const double *kg = k + g * N * D;
    const double *qg = q + g * Sq * D;
    double *kb = kbar + g * D;
    /* key mean over the real tokens */
    for (int64_t d = 0; d < D; d++) kb[d] = 0.0;
    if (centering && N > 0) {
      for (int64_t j = 0; j < N; j++)
        for (int64_t d = 0; d < D; d++) kb[d] += kg[j * D + d];
      for (int64_t d = 0; d < D; d++) kb[d] /= (double)N;
    }
    /* max key norm, measured on the keys the kernel exponentiates */
    double km = 0.0;
    double *knorm = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
    for (int64_t j = 0; j < N; j++) {
      double ss = 0.0;
      for (int64_t d = 0; d < D; d++) {
        double x = kg[j * D + d] - kb[d];
        ss += x * x;
      }
      knorm[j] = ss;
      if (ss > km) km = ss;
    }
    if (n_sink > 0) {
      /* key sinks ("Kernel reference: ring_attention_const_max_fwd", section "Adapting this
       * kernel": leave the few loudest keys out of the max reduction).  tau = the
       * (n_sink+1)-th largest squared norm, counted with multiplicity (0 with fewer keys);
       * the sinks are the keys strictly above tau, so at most n_sink of them, and the max
       * over every other key is tau itself. */
      double *sorted = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
      memcpy(sorted, knorm, sizeof(double) * (size_t)N);
      qsort(sorted, (size_t)N, sizeof(double), fmo_cmp_desc);
      double tau = (N > n_sink) ? sorted[n_sink] : 0.0;
      int64_t t = 0;
      for (int64_t j = 0; j < N; j++)
        if (knorm[j] > tau) sink_idx[g * n_sink + t++] = (int32_t)j;
      for (; t < n_sink; t++) sink_idx[g * n_sink + t] = INT32_MAX;
      /* how far the n_sink-th largest norm sits above tau: where fp32 norms could pick
       * another set (0 when they tie, +inf with no (n_sink+1)-th key) */
      if (sink_gap) sink_gap[g] = (N > n_sink) ? sorted[n_sink - 1] - tau : INFINITY;
      free(sorted);
      km = tau;
    }
    free(knorm);
    kmax_sq[g] = km;
    /* per-row query norms -> per-block max */
    for (int64_t b = 0; b < nqb; b++) {
      double qm = 0.0;
      for (int64_t i = b * bq; i < Sq && i < (b + 1) * bq; i++) {
        double ss = 0.0;
        for (int64_t d = 0; d < D; d++) ss += qg[i * D + d] * qg[i * D + d];
        if (ss > qm) qm = ss;
      }
      qmax_sq[g * nqb + b] = qm;
      double u = alpha * sqrt(qm) * sqrt(km);
      U[g * nqb + b] = u;
      m[g * nqb + b] = (int32_t)ceil(u) - C;
      flag[g * nqb + b] = (uint8_t)(v_ok && (u <= (double)gate));
    }
    for (int64_t i = 0; i < Sq; i++) {
      double dot = 0.0, ss = 0.0;
      for (int64_t d = 0; d < D; d++) {
        dot += qg[i * D + d] * kb[d];
        ss += qg[i * D + d] * qg[i * D + d];
      }
      /* per-row bound of "Kernel reference: ring_attention_const_max_fwd", sections
       * "Picking a max that is safe without measuring it" and "Best practices" (give each
       * query row its own bound), with the shift of PR #477: m_i = ceil(U_i) - C */
      double ur = alpha * sqrt(ss) * sqrt(km);
      int32_t mr = (int32_t)ceil(ur) - C;
      if (U_row) U_row[g * Sq + i] = ur;
      if (m_row) m_row[g * Sq + i] = mr;
      if (qkbar) qkbar[g * Sq + i] = alpha * dot;
      /* the full base-2 shift of row i: its m (per row, or its Q-block's) plus the
       * centering term alpha*q_i.kbar ("Virtual K-centering") */
      if (shift) shift[g * Sq + i] = (double)(per_row ? mr : m[g * nqb + i / bq]) + alpha * dot;
    }
  }
  consts[0] = C;
  consts[1] = W;
  consts[2] = gate;
  consts[3] = v_ok;
}

/* Sequential fp32 emulation of the fixed-m accumulation with an arbitrary per-row
 * shift m_row (in base-2 units), for ONE problem:
 *   p_j = 2^(z_j - m_row),  z_j = alpha * q . (k_j - kbar)   (kbar may be NULL)
 *   acc_sum += p_j; acc_o += p_j * v_j       -- in fp32, in key order
 * A term whose fp32 value would be subnormal is flushed to zero (as a flush-to-zero
 * exp2 does) and counted in n_flushed[row]; a term that overflows fp32 is counted
 * in n_overflow[row].  The exponent is formed in fp64 so the only fp32 effects are
 * the ones the pages reason about (the range of 2^e and of the sums).
 *   q [R, D], k, v [N, D], acc_o [R, D] (fp32), acc_sum [R] (fp32).            */
void fmo_fixed_m_emulate_f32(const double *q, const double *k, const double *v, int64_t R,
                             int64_t N, int64_t D, double scale, const double *kbar,
                             const double *m_row, float *acc_o, float *acc_sum,
                             int64_t *n_flushed, int64_t *n_overflow) {
  const double alpha = scale * FMO_LOG2E;
  for (int64_t i = 0; i < R; i++) {
    float s = 0.0f;
    float *oi = acc_o + i * D;
    for (int64_t d = 0; d < D; d++) oi[d] = 0.0f;
    int64_t nf = 0, nov = 0;
    for (int64_t j = 0; j < N; j++) {
      double dot = 0.0;
      for (int64_t d = 0; d < D; d++) {
        double kk = k[j * D + d] - (kbar ? kbar[d] : 0.0);
        dot += q[i * D + d] * kk;
      }
      double e = alpha * dot - m_row[i];
      float p;
      if (e < -126.0) { /* 2^e is below the smallest normal fp32 */
        p = 0.0f;
        nf++;
      } else {
        p = (float)exp2(e);
        if (isinf(p)) nov++;
      }
      s += p;
      for (int64_t d = 0; d < D; d++) oi[d] += p * (float)v[j * D + d];
    }
    acc_sum[i] = s;
    n_flushed[i] = nf;
    n_overflow[i] = nov;
  }
}

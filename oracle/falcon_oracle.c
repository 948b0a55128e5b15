/*
 * falcon_oracle.c -- fp64 CPU oracle for the Falcon-1 / Falcon-1A fast-weight
 * recurrences of "Fast Weight Attention for Continual Learning".
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, token-by-token
 * definition of what the GPU library computes.  Only the tests, the smoke
 * check and the benchmark's CPU-baseline leg may load it.  It shares no code,
 * header, table or helper with the CUDA library, and it never calls it.
 *
 * Everything is double precision.  Inputs are the already-rounded values the
 * GPU sees (bf16 or fp32 widened exactly to fp64 by the caller).
 *
 * Passages followed (page hyper.ai/fr/papers/2608.27763 unless noted):
 *   - shifted write stream x_1 = 0, x_t = phi(k_{t-1}): Section 2.2, Eq. (2.3)
 *     and the "Naming and formula summary" at the head of Section 4;
 *   - boundary sentinel eta_1 = 0 (so alpha_1 = 0, gamma_1 = 1): Section 3,
 *     "Indexing and causality conventions";
 *   - NLMS step eta_t = beta_t / (||x_t||^2 + lambda_t + eps), eta := 0 when
 *     the denominator is 0: Section 3.1, Eq. (3.4);
 *   - Falcon-1 update S_t = (1 - eta lambda) S_{t-1} + eta x_t r_t^T with
 *     r_t = v_t - S_{t-1}^T x_t: Section 3.1, Eq. (3.3) and Section 4 summary;
 *   - Falcon-1A update S_t = (1 - eta lambda) S_{t-1} + eta x_t v_t^T with
 *     E_t = ||x_t||^2: Section 4.3, Eq. (4.6) and (4.8);
 *   - positive-decay clamp alpha = min(eta lambda, 1 - eps_gamma),
 *     gamma = 1 - alpha: Section 4.3 "Decay positivity" and Section 4.4
 *     (the clamped recurrence is the implemented one);
 *   - read after write o_t = S_t^T phi(q_t): Section 4 summary;
 *   - one-step pseudocode with the same order of operations: page
 *     rcap.io/posts/fast-weight-attention-for-continual-learning-2026-08-27.
 *
 *   - Falcon-2 (per-column step sizes eta_{j,t} = beta_{j,t} / (||x_t||^2 +
 *     lambda_t + eps), S_t = S_{t-1}(I - lambda_t Diag(eta_t)) +
 *     x_t (eta_t o r_t)^T): Section 3.1, the regression-family display and
 *     the "Per-column NLMS step sizes" paragraph of Section 4.2;
 *   - Falcon-3A (sliding-window inner product, window of B pairs): Section
 *     4.5, the windowed loss, N_bar and E_bar, the step size with E_t^{(B)}
 *     = E_bar, and S_t = (1 - eta_t lambda_t) S_{t-1} + eta_t N_bar_t;
 *   - Falcon-2A (the same with r_t replaced by y_t = v_t, E_t = ||x_t||^2):
 *     Section 4.3, "Falcon-2A: per-column inner-product write" and the
 *     Falcon-1A/Falcon-2A step sizes; the clamp acts per column (the
 *     effective ridge alpha_{j,t} / eta_{j,t} of the same paragraph).
 *
 * Readings where the pages are silent:
 *   - phi is the identity, the l2 normalisation u / max(||u||, 1e-12)
 *     ("QK-l2" in the experiment tables of page juhoplayground.github.io), or
 *     RMSNorm with eps_rms = 1e-6 (the pages name eps_rms without a value);
 *   - a caller that carries state across calls passes x_prev = phi(k_T) of the
 *     previous segment; then step 1 writes with x_1 = x_prev (no sentinel).
 *
 *   - the normalised read (falcon1a_oracle_forward_normalized): Section 2.2,
 *     Eq. (2.1)-(2.3) define o_t = S_t^T phi(q_t) / (z_t^T phi(q_t) + eps_attn)
 *     with an additive normaliser z_t = z_{t-1} + x_t on the shifted stream;
 *     the Falcon-1A version is deferred to an appendix the pages do not
 *     include.  Reading taken: z follows the numerator's update with a
 *     constant unit target, z_t = gamma_t z_{t-1} + eta_t x_t (the same gain
 *     and clamped decay), which is Eq. (2.3) exactly at lambda = 0, eta = 1.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_FALCON1 1  /* regression rule, Eq. (3.3) */
#define ORACLE_FALCON1A 2 /* inner-product rule, Eq. (4.6) */
#define ORACLE_FALCON2 3  /* per-column regression rule (Section 3.1, 4.2) */
#define ORACLE_FALCON2A 4 /* per-column inner-product rule (Section 4.3) */
#define ORACLE_PHI_IDENTITY 0
#define ORACLE_PHI_L2 1
#define ORACLE_PHI_RMS 2 /* RMSNorm, Section 4.1 "Scaled features" */
#define ORACLE_EPS_RMS 1e-6 /* eps_rms: not given by the pages (a reading) */
#define ORACLE_RIDGE_GIVEN 0  /* lambda_t as given */
#define ORACLE_RIDGE_SCALED 1 /* lambda_t = lambda_bar_t * E_t, Section 4.1 */

/* phi applied to one m-vector: identity, the l2 map, or RMSNorm(u) =
 * u / sqrt(||u||^2 / m + eps_rms) (Section 4.1, "Scaled features"). */
static void feature_map(int phi, int m, const double *u, double *out) {
  if (phi == ORACLE_PHI_RMS) {
    double ss = 0.0;
    for (int i = 0; i < m; ++i) ss += u[i] * u[i];
    const double den = sqrt(ss / m + ORACLE_EPS_RMS);
    for (int i = 0; i < m; ++i) out[i] = u[i] / den;
  } else if (phi == ORACLE_PHI_L2) {
    double ss = 0.0;
    for (int i = 0; i < m; ++i) ss += u[i] * u[i];
    double nrm = sqrt(ss);
    if (nrm < 1e-12) nrm = 1e-12;
    for (int i = 0; i < m; ++i) out[i] = u[i] / nrm;
  } else {
    for (int i = 0; i < m; ++i) out[i] = u[i];
  }
}

/* eta_t and gamma_t of one step (Eq. (3.4) and the decay clamp).  With the
 * scale-coupled ridge (Section 4.1) the argument is the base ridge lambda_bar
 * and the recurrence uses lambda_t = lambda_bar * E_t, E_t = ||x_t||^2. */
static void step_scalars(int sentinel, int m, const double *x, double beta,
                         double lambda, int ridge, double eps, double eps_gamma,
                         double *eta_out, double *gamma_out) {
  double eta = 0.0;
  double E = 0.0;
  for (int i = 0; i < m; ++i) E += x[i] * x[i];
  if (ridge == ORACLE_RIDGE_SCALED) lambda *= E;
  if (!sentinel) {
    double den = E + lambda + eps;
    eta = (den > 0.0) ? beta / den : 0.0;
  }
  double alpha = eta * lambda;
  if (alpha > 1.0 - eps_gamma) alpha = 1.0 - eps_gamma;
  *eta_out = eta;
  *gamma_out = 1.0 - alpha;
}

/* One token of the recurrence on one head.  S is m x dv row-major, updated in
 * place.  x is the write feature of this step; qf = phi(q_t).  Writes o_t. */
static void one_token(int rule, int m, int dv, double *S, const double *x,
                      const double *qf, const double *v, double eta,
                      double gamma, double *r /* dv scratch */, double *o) {
  if (rule == ORACLE_FALCON1) {
    /* r_t = v_t - S_{t-1}^T x_t  (prediction from the pre-update state) */
    for (int j = 0; j < dv; ++j) {
      double pred = 0.0;
      for (int i = 0; i < m; ++i) pred += S[(int64_t)i * dv + j] * x[i];
      r[j] = v[j] - pred;
    }
  } else {
    /* Falcon-1A writes the target itself */
    for (int j = 0; j < dv; ++j) r[j] = v[j];
  }
  /* S_t = gamma S_{t-1} + eta x_t r_t^T */
  for (int i = 0; i < m; ++i)
    for (int j = 0; j < dv; ++j)
      S[(int64_t)i * dv + j] = gamma * S[(int64_t)i * dv + j] + eta * x[i] * r[j];
  /* o_t = S_t^T phi(q_t)  (read after write) */
  for (int j = 0; j < dv; ++j) {
    double acc = 0.0;
    for (int i = 0; i < m; ++i) acc += S[(int64_t)i * dv + j] * qf[i];
    o[j] = acc;
  }
}

typedef struct {
  int rule, m, dv, phi, ridge;
  int64_t T;
  double eps, eps_gamma;
  const double *q, *k, *v, *beta, *lambda, *S0, *x_prev;
  double *o, *S_out, *x_last, *S_traj;
} fwd_args;

/* The whole sequence of one head (b, h). */
static void forward_head(const fwd_args *a, int64_t bh) {
  const int m = a->m, dv = a->dv;
  const int64_t T = a->T;
  double *S = (double *)calloc((size_t)m * dv, sizeof(double));
  double *x = (double *)calloc((size_t)m, sizeof(double));
  double *qf = (double *)malloc(sizeof(double) * (size_t)m);
  double *r = (double *)malloc(sizeof(double) * (size_t)dv);
  if (a->S0) memcpy(S, a->S0 + bh * m * dv, sizeof(double) * (size_t)m * dv);
  int sentinel = 1;
  if (a->x_prev) {
    memcpy(x, a->x_prev + bh * m, sizeof(double) * (size_t)m);
    sentinel = 0;
  }
  for (int64_t t = 0; t < T; ++t) {
    const int64_t row = bh * T + t;
    double eta, gamma;
    step_scalars(sentinel && t == 0, m, x, a->beta[row], a->lambda[row], a->ridge,
                 a->eps, a->eps_gamma, &eta, &gamma);
    feature_map(a->phi, m, a->q + row * m, qf);
    one_token(a->rule, m, dv, S, x, qf, a->v + row * dv, eta, gamma, r,
              a->o + row * dv);
    if (a->S_traj)
      memcpy(a->S_traj + row * m * dv, S, sizeof(double) * (size_t)m * dv);
    /* the next step writes under phi(k_t) */
    feature_map(a->phi, m, a->k + row * m, x);
  }
  if (a->S_out) memcpy(a->S_out + bh * m * dv, S, sizeof(double) * (size_t)m * dv);
  if (a->x_last) memcpy(a->x_last + bh * m, x, sizeof(double) * (size_t)m);
  free(S);
  free(x);
  free(qf);
  free(r);
}

typedef struct {
  const fwd_args *a;
  int64_t begin, end;
} fwd_slice;

static void *forward_worker(void *p) {
  const fwd_slice *s = (const fwd_slice *)p;
  for (int64_t bh = s->begin; bh < s->end; ++bh) forward_head(s->a, bh);
  return NULL;
}

/*
 * Whole-sequence forward for all B*H heads.  Layouts (row-major):
 *   q, k: [BH, T, m]   v, o: [BH, T, dv]   beta, lambda: [BH, T]
 *   S0 (nullable => zeros), S_out: [BH, m, dv]
 *   x_prev (nullable => sentinel), x_last (nullable): [BH, m]
 *   S_traj (nullable): [BH, T, m, dv], the state after every token.
 * Heads are independent; they are split over nthreads POSIX threads.
 * Returns 0, or -1 on a bad argument.
 */
int falcon_oracle_forward(int rule, int64_t BH, int64_t T, int m, int dv,
                          int phi, int ridge, double eps, double eps_gamma,
                          const double *q, const double *k, const double *v,
                          const double *beta, const double *lambda,
                          const double *S0, const double *x_prev, double *o,
                          double *S_out, double *x_last, double *S_traj,
                          int nthreads) {
  if (rule != ORACLE_FALCON1 && rule != ORACLE_FALCON1A) return -1;
  if (BH < 0 || T < 0 || m <= 0 || dv <= 0) return -1;
  fwd_args a = {rule, m, dv, phi, ridge, T, eps, eps_gamma, q, k, v, beta, lambda,
                S0, x_prev, o, S_out, x_last, S_traj};
  if (nthreads < 1) nthreads = 1;
  if (nthreads > BH) nthreads = (int)(BH > 0 ? BH : 1);
  pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
  fwd_slice *sl = (fwd_slice *)malloc(sizeof(fwd_slice) * (size_t)nthreads);
  for (int w = 0; w < nthreads; ++w) {
    sl[w].a = &a;
    sl[w].begin = BH * w / nthreads;
    sl[w].end = BH * (w + 1) / nthreads;
  }
  for (int w = 1; w < nthreads; ++w) pthread_create(&tid[w], NULL, forward_worker, &sl[w]);
  forward_worker(&sl[0]);
  for (int w = 1; w < nthreads; ++w) pthread_join(tid[w], NULL);
  free(tid);
  free(sl);
  return 0;
}

/*
 * One recurrent decode step for N independent states (the same token update
 * as above, applied once).  Layouts:
 *   q, k: [N, m]   v, o: [N, dv]   beta, lambda: [N]
 *   S: [N, m, dv], updated in place.
 *   x_prev: [N, m], read as this step's write feature, then overwritten with
 *           phi(k) for the next step.
 *   fresh (nullable): [N] bytes; nonzero marks the first token of a sequence,
 *           where the sentinel applies (x = 0, eta = 0).
 */
int falcon_oracle_decode_step(int rule, int64_t N, int m, int dv, int phi,
                              int ridge, double eps, double eps_gamma, const double *q,
                              const double *k, const double *v,
                              const double *beta, const double *lambda,
                              double *S, double *x_prev,
                              const unsigned char *fresh, double *o) {
  if (rule != ORACLE_FALCON1 && rule != ORACLE_FALCON1A) return -1;
  if (N < 0 || m <= 0 || dv <= 0) return -1;
  double *x = (double *)malloc(sizeof(double) * (size_t)m);
  double *qf = (double *)malloc(sizeof(double) * (size_t)m);
  double *r = (double *)malloc(sizeof(double) * (size_t)dv);
  for (int64_t n = 0; n < N; ++n) {
    const int sentinel = fresh ? (fresh[n] != 0) : 0;
    if (sentinel)
      memset(x, 0, sizeof(double) * (size_t)m);
    else
      memcpy(x, x_prev + n * m, sizeof(double) * (size_t)m);
    double eta, gamma;
    step_scalars(sentinel, m, x, beta[n], lambda[n], ridge, eps, eps_gamma, &eta, &gamma);
    feature_map(phi, m, q + n * m, qf);
    one_token(rule, m, dv, S + n * m * dv, x, qf, v + n * dv, eta, gamma, r,
              o + n * dv);
    feature_map(phi, m, k + n * m, x_prev + n * m);
  }
  free(x);
  free(qf);
  free(r);
  return 0;
}

/*
 * Falcon-2 / Falcon-2A over whole sequences: every column j of S (one value
 * channel) follows its own step size eta_{j,t} and decay gamma_{j,t} =
 * 1 - min(eta_{j,t} lambda_t, 1 - eps_gamma); the write feature x_t, the
 * ridge lambda_t and the read phi(q_t) are shared by the columns.
 * Layouts as falcon_oracle_forward, except beta: [BH, T, dv] (one gain per
 * column and token).  Returns 0, or -1 on a bad argument.
 */
typedef struct {
  int rule, m, dv, phi, ridge;
  int64_t T;
  double eps, eps_gamma;
  const double *q, *k, *v, *beta, *lambda, *S0, *x_prev;
  double *o, *S_out, *x_last;
} fwd2_args;

static void forward2_head(const fwd2_args *a, int64_t bh) {
  const int m = a->m, dv = a->dv;
  const int64_t T = a->T;
  double *S = (double *)calloc((size_t)m * dv, sizeof(double));
  double *x = (double *)calloc((size_t)m, sizeof(double));
  double *qf = (double *)malloc(sizeof(double) * (size_t)m);
  if (a->S0) memcpy(S, a->S0 + bh * m * dv, sizeof(double) * (size_t)m * dv);
  int sentinel = 1;
  if (a->x_prev) {
    memcpy(x, a->x_prev + bh * m, sizeof(double) * (size_t)m);
    sentinel = 0;
  }
  for (int64_t t = 0; t < T; ++t) {
    const int64_t row = bh * T + t;
    double E = 0.0;
    for (int i = 0; i < m; ++i) E += x[i] * x[i];
    const double lambda =
        a->ridge == ORACLE_RIDGE_SCALED ? a->lambda[row] * E : a->lambda[row];
    const double den = E + lambda + a->eps;
    feature_map(a->phi, m, a->q + row * m, qf);
    for (int j = 0; j < dv; ++j) {
      /* column j: its own eta_{j,t}, clamped decay, residual (or target) */
      double eta = 0.0;
      if (!(sentinel && t == 0) && den > 0.0) eta = a->beta[row * dv + j] / den;
      double alpha = eta * lambda;
      if (alpha > 1.0 - a->eps_gamma) alpha = 1.0 - a->eps_gamma;
      const double gamma = 1.0 - alpha;
      double r = a->v[row * dv + j];
      if (a->rule == ORACLE_FALCON2) {
        double pred = 0.0; /* S_{t-1}[:, j]^T x_t, before the update */
        for (int i = 0; i < m; ++i) pred += S[(int64_t)i * dv + j] * x[i];
        r -= pred;
      }
      double acc = 0.0;
      for (int i = 0; i < m; ++i) {
        double *s = &S[(int64_t)i * dv + j];
        *s = gamma * *s + eta * x[i] * r;
        acc += *s * qf[i]; /* read after write */
      }
      a->o[row * dv + j] = acc;
    }
    feature_map(a->phi, m, a->k + row * m, x);
  }
  if (a->S_out) memcpy(a->S_out + bh * m * dv, S, sizeof(double) * (size_t)m * dv);
  if (a->x_last) memcpy(a->x_last + bh * m, x, sizeof(double) * (size_t)m);
  free(S);
  free(x);
  free(qf);
}

typedef struct {
  const fwd2_args *a;
  int64_t begin, end;
} fwd2_slice;

static void *forward2_worker(void *p) {
  const fwd2_slice *s = (const fwd2_slice *)p;
  for (int64_t bh = s->begin; bh < s->end; ++bh) forward2_head(s->a, bh);
  return NULL;
}

int falcon2_oracle_forward(int rule, int64_t BH, int64_t T, int m, int dv, int phi,
                           int ridge, double eps, double eps_gamma, const double *q,
                           const double *k, const double *v, const double *beta,
                           const double *lambda, const double *S0,
                           const double *x_prev, double *o, double *S_out,
                           double *x_last, int nthreads) {
  if (rule != ORACLE_FALCON2 && rule != ORACLE_FALCON2A) return -1;
  if (BH < 0 || T < 0 || m <= 0 || dv <= 0) return -1;
  fwd2_args a = {rule, m, dv, phi, ridge, T, eps, eps_gamma, q, k, v, beta, lambda,
                 S0, x_prev, o, S_out, x_last};
  if (nthreads < 1) nthreads = 1;
  if (nthreads > BH) nthreads = (int)(BH > 0 ? BH : 1);
  pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
  fwd2_slice *sl = (fwd2_slice *)malloc(sizeof(fwd2_slice) * (size_t)nthreads);
  for (int w = 0; w < nthreads; ++w) {
    sl[w].a = &a;
    sl[w].begin = BH * w / nthreads;
    sl[w].end = BH * (w + 1) / nthreads;
  }
  for (int w = 1; w < nthreads; ++w) pthread_create(&tid[w], NULL, forward2_worker, &sl[w]);
  forward2_worker(&sl[0]);
  for (int w = 1; w < nthreads; ++w) pthread_join(tid[w], NULL);
  free(tid);
  free(sl);
  return 0;
}

/*
 * Falcon-3A over whole fresh sequences (Section 4.5): for t >= 2 the window
 * I_t = {max(2, t - B + 1), ..., t} of write pairs (x_j, v_j), B_t = |I_t|,
 *   N_bar_t = (1/B_t) sum_{j in I_t} x_j v_j^T,  E_bar_t = (1/B_t) sum ||x_j||^2,
 *   eta_t = beta_t / (E_bar_t + lambda_t + eps)  (lambda_t = lambda_bar_t *
 *   E_bar_t with the scale-coupled ridge), alpha_t = min(eta_t lambda_t,
 *   1 - eps_gamma), S_t = (1 - alpha_t) S_{t-1} + eta_t N_bar_t;
 * t = 1 is the boundary (no update).  o_t = S_t^T phi(q_t).  The window
 * reaches back only within the call (a fresh sequence: x_1 = 0).
 * Layouts as falcon_oracle_forward (beta, lambda: [BH, T]); no x_prev.
 */
typedef struct {
  int m, dv, phi, ridge, B;
  int64_t T;
  double eps, eps_gamma;
  const double *q, *k, *v, *beta, *lambda, *S0;
  double *o, *S_out, *x_last;
} fwd3_args;

static void forward3a_head(const fwd3_args *a, int64_t bh) {
  const int m = a->m, dv = a->dv;
  const int64_t T = a->T;
  double *S = (double *)calloc((size_t)m * dv, sizeof(double));
  double *X = (double *)calloc((size_t)(T > 0 ? T : 1) * m, sizeof(double)); /* x_t, t = 1..T */
  double *qf = (double *)malloc(sizeof(double) * (size_t)m);
  double *N = (double *)malloc(sizeof(double) * (size_t)m * dv);
  if (a->S0) memcpy(S, a->S0 + bh * m * dv, sizeof(double) * (size_t)m * dv);
  /* write features: x_1 = 0, x_t = phi(k_{t-1}) */
  for (int64_t t = 1; t < T; ++t) feature_map(a->phi, m, a->k + (bh * T + t - 1) * m, X + t * m);
  for (int64_t t = 0; t < T; ++t) { /* t is 0-based: token t + 1 */
    const int64_t row = bh * T + t;
    if (t >= 1) {
      const int64_t j0 = (t - a->B + 1 > 1) ? t - a->B + 1 : 1; /* 0-based window start (>= token 2) */
      const int64_t Bt = t - j0 + 1;
      double Ebar = 0.0;
      memset(N, 0, sizeof(double) * (size_t)m * dv);
      for (int64_t j = j0; j <= t; ++j) {
        const double *xj = X + j * m, *vj = a->v + (bh * T + j) * dv;
        for (int i = 0; i < m; ++i) {
          Ebar += xj[i] * xj[i];
          for (int c = 0; c < dv; ++c) N[(int64_t)i * dv + c] += xj[i] * vj[c];
        }
      }
      Ebar /= (double)Bt;
      double lambda = a->lambda[row];
      if (a->ridge == ORACLE_RIDGE_SCALED) lambda *= Ebar;
      const double den = Ebar + lambda + a->eps;
      const double eta = den > 0.0 ? a->beta[row] / den : 0.0;
      double alpha = eta * lambda;
      if (alpha > 1.0 - a->eps_gamma) alpha = 1.0 - a->eps_gamma;
      for (int64_t e = 0; e < (int64_t)m * dv; ++e)
        S[e] = (1.0 - alpha) * S[e] + eta * N[e] / (double)Bt;
    }
    feature_map(a->phi, m, a->q + row * m, qf);
    for (int c = 0; c < dv; ++c) {
      double acc = 0.0;
      for (int i = 0; i < m; ++i) acc += S[(int64_t)i * dv + c] * qf[i];
      a->o[row * dv + c] = acc;
    }
  }
  if (a->S_out) memcpy(a->S_out + bh * m * dv, S, sizeof(double) * (size_t)m * dv);
  if (a->x_last && T > 0) feature_map(a->phi, m, a->k + (bh * T + T - 1) * m, a->x_last + bh * m);
  free(S);
  free(X);
  free(qf);
  free(N);
}

typedef struct {
  const fwd3_args *a;
  int64_t begin, end;
} fwd3_slice;

static void *forward3a_worker(void *p) {
  const fwd3_slice *s = (const fwd3_slice *)p;
  for (int64_t bh = s->begin; bh < s->end; ++bh) forward3a_head(s->a, bh);
  return NULL;
}

int falcon3a_oracle_forward(int64_t BH, int64_t T, int m, int dv, int phi, int ridge, int B,
                            double eps, double eps_gamma, const double *q, const double *k,
                            const double *v, const double *beta, const double *lambda,
                            const double *S0, double *o, double *S_out, double *x_last,
                            int nthreads) {
  if (BH < 0 || T < 0 || m <= 0 || dv <= 0 || B < 1) return -1;
  fwd3_args a = {m, dv, phi, ridge, B, T, eps, eps_gamma, q, k, v, beta, lambda, S0,
                 o, S_out, x_last};
  if (nthreads < 1) nthreads = 1;
  if (nthreads > BH) nthreads = (int)(BH > 0 ? BH : 1);
  pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
  fwd3_slice *sl = (fwd3_slice *)malloc(sizeof(fwd3_slice) * (size_t)nthreads);
  for (int w = 0; w < nthreads; ++w) {
    sl[w].a = &a;
    sl[w].begin = BH * w / nthreads;
    sl[w].end = BH * (w + 1) / nthreads;
  }
  for (int w = 1; w < nthreads; ++w) pthread_create(&tid[w], NULL, forward3a_worker, &sl[w]);
  forward3a_worker(&sl[0]);
  for (int w = 1; w < nthreads; ++w) pthread_join(tid[w], NULL);
  free(tid);
  free(sl);
  return 0;
}

/* ------------------------------------------------------------------------
 * Backward pass of Falcon-1 / Falcon-1A: reverse-mode differentiation of the
 * token recurrence above, in fp64.
 *
 * The pages state that training differentiates through the update, so that
 * the slow weights producing q, k, v, beta and lambda learn (page
 * hyper.ai/fr/papers/2608.27763, Section 3, "Implicit fast-memory
 * objective"), and that the backward pass differentiates through the
 * log-decay renormalisation and the normalised step size (Section 4.6,
 * "Backward pass"; its appendix is not on the pages).  Nothing else is given,
 * so this is the gradient of the forward function as written above, taken by
 * the chain rule one token at a time, newest token first:
 *
 *   o_t = S_t^T qf_t                 dS_t += qf_t do_t^T,  dqf_t = S_t do_t
 *   S_t = gamma S_{t-1} + eta x r^T  dgamma = <dS_t, S_{t-1}>,
 *                                    deta = x^T dS_t r,  dx = eta dS_t r,
 *                                    dr = eta dS_t^T x,  dS_{t-1} = gamma dS_t
 *   r = v - S_{t-1}^T x (Falcon-1)   dv = dr,  dS_{t-1} -= x dr^T,
 *                                    dx -= S_{t-1} dr
 *   r = v (Falcon-1A)                dv = dr
 *   gamma = 1 - alpha, alpha = min(eta lambda, 1 - eps_gamma):
 *       on the clamped branch alpha is a constant; otherwise
 *       deta += lambda dalpha, dlambda += eta dalpha with dalpha = -dgamma
 *   eta = beta / (E + lambda + eps): dbeta = deta / den,
 *       dE = dlambda_den = -deta eta / den  (eta := 0, a constant, if den <= 0)
 *   lambda_t = lambda_bar E (scaled ridge): dlambda_bar = dlambda E,
 *       dE += dlambda lambda_bar
 *   E = ||x||^2: dx += 2 dE x
 *   x_t = phi(k_{t-1}): dk_{t-1} = J_phi(k_{t-1})^T dx_t; x_1 = x_prev or
 *       the sentinel zero (no gradient); qf_t = phi(q_t): dq_t = J_phi^T dqf_t
 * The sentinel token (eta = 0, gamma = 1) passes no gradient to beta_1,
 * lambda_1.  At the clamp's kink (eta lambda = 1 - eps_gamma exactly) the
 * unclamped branch is taken, as in the forward.
 * ------------------------------------------------------------------------ */

/* J_phi(u)^T g for the feature maps of feature_map(). */
static void feature_map_vjp(int phi, int m, const double *u, const double *g, double *out) {
  if (phi == ORACLE_PHI_RMS) {
    /* phi = u s, s = (||u||^2/m + eps)^(-1/2): d phi_i / d u_j = s delta_ij - s^3 u_i u_j / m */
    double ss = 0.0, ug = 0.0;
    for (int i = 0; i < m; ++i) {
      ss += u[i] * u[i];
      ug += u[i] * g[i];
    }
    const double s = 1.0 / sqrt(ss / m + ORACLE_EPS_RMS);
    for (int i = 0; i < m; ++i) out[i] = s * g[i] - s * s * s * u[i] * ug / m;
  } else if (phi == ORACLE_PHI_L2) {
    /* phi = u / n, n = ||u|| (> 1e-12): d phi_i / d u_j = (delta_ij - phi_i phi_j) / n */
    double ss = 0.0;
    for (int i = 0; i < m; ++i) ss += u[i] * u[i];
    const double n = sqrt(ss);
    if (n < 1e-12) {
      for (int i = 0; i < m; ++i) out[i] = g[i] / 1e-12;
    } else {
      double pg = 0.0;
      for (int i = 0; i < m; ++i) pg += u[i] / n * g[i];
      for (int i = 0; i < m; ++i) out[i] = (g[i] - u[i] / n * pg) / n;
    }
  } else {
    for (int i = 0; i < m; ++i) out[i] = g[i];
  }
}

typedef struct {
  int rule, m, dv, phi, ridge;
  int64_t T;
  double eps, eps_gamma;
  const double *q, *k, *v, *beta, *lambda, *S0, *x_prev;
  const double *dO, *dS_T, *dx_last;
  double *dq, *dk, *dvv, *dbeta, *dlambda, *dS0, *dx_prev;
} bwd_args;

static void backward_head(const bwd_args *a, int64_t bh) {
  const int m = a->m, dv = a->dv;
  const int64_t T = a->T;
  const size_t md = (size_t)m * dv;
  /* forward, keeping every pre-update state S_{t-1} and write feature x_t */
  double *Spre = (double *)malloc(sizeof(double) * md * (size_t)(T > 0 ? T : 1));
  double *X = (double *)calloc((size_t)(T + 1) * m, sizeof(double));
  double *S = (double *)calloc(md, sizeof(double));
  double *qf = (double *)malloc(sizeof(double) * (size_t)m);
  double *r = (double *)malloc(sizeof(double) * (size_t)dv);
  double *o = (double *)malloc(sizeof(double) * (size_t)dv);
  if (a->S0) memcpy(S, a->S0 + bh * md, sizeof(double) * md);
  const int fresh = a->x_prev == NULL;
  if (!fresh) memcpy(X, a->x_prev + bh * m, sizeof(double) * (size_t)m);
  for (int64_t t = 0; t < T; ++t) {
    const int64_t row = bh * T + t;
    double eta, gamma;
    step_scalars(fresh && t == 0, m, X + t * m, a->beta[row], a->lambda[row], a->ridge, a->eps,
                 a->eps_gamma, &eta, &gamma);
    memcpy(Spre + (size_t)t * md, S, sizeof(double) * md);
    feature_map(a->phi, m, a->q + row * m, qf);
    one_token(a->rule, m, dv, S, X + t * m, qf, a->v + row * dv, eta, gamma, r, o);
    feature_map(a->phi, m, a->k + row * m, X + (t + 1) * m);
  }
  /* S now holds S_T; walk back */
  double *dS = (double *)calloc(md, sizeof(double));
  double *Spost = (double *)malloc(sizeof(double) * md);
  double *dx = (double *)malloc(sizeof(double) * (size_t)m);
  double *dxn = (double *)calloc((size_t)m, sizeof(double)); /* d x_{t+1} */
  double *dr = (double *)malloc(sizeof(double) * (size_t)dv);
  double *dqf = (double *)malloc(sizeof(double) * (size_t)m);
  if (a->dS_T) memcpy(dS, a->dS_T + bh * md, sizeof(double) * md);
  if (a->dx_last) memcpy(dxn, a->dx_last + bh * m, sizeof(double) * (size_t)m);
  memcpy(Spost, S, sizeof(double) * md);
  for (int64_t t = T - 1; t >= 0; --t) {
    const int64_t row = bh * T + t;
    const double *x = X + t * m;
    const double *Sp = Spre + (size_t)t * md;
    /* x_{t+1} = phi(k_t) */
    feature_map_vjp(a->phi, m, a->k + row * m, dxn, a->dk + row * m);
    /* scalars of this token, as the forward computed them */
    const int sentinel = fresh && t == 0;
    double E = 0.0;
    for (int i = 0; i < m; ++i) E += x[i] * x[i];
    const double lam_in = a->lambda[row];
    const double lam = (a->ridge == ORACLE_RIDGE_SCALED) ? lam_in * E : lam_in;
    double eta = 0.0, den = E + lam + a->eps;
    if (!sentinel && den > 0.0) eta = a->beta[row] / den;
    const int clamped = eta * lam > 1.0 - a->eps_gamma;
    const double gamma = 1.0 - (clamped ? 1.0 - a->eps_gamma : eta * lam);
    /* r from the pre-update state */
    for (int j = 0; j < dv; ++j) {
      double pred = 0.0;
      if (a->rule == ORACLE_FALCON1)
        for (int i = 0; i < m; ++i) pred += Sp[(size_t)i * dv + j] * x[i];
      r[j] = a->v[row * dv + j] - pred;
    }
    /* read: o_t = S_t^T qf */
    feature_map(a->phi, m, a->q + row * m, qf);
    const double *dot = a->dO + row * dv;
    for (int i = 0; i < m; ++i) {
      double acc = 0.0;
      for (int j = 0; j < dv; ++j) {
        acc += Spost[(size_t)i * dv + j] * dot[j];
        dS[(size_t)i * dv + j] += qf[i] * dot[j];
      }
      dqf[i] = acc;
    }
    feature_map_vjp(a->phi, m, a->q + row * m, dqf, a->dq + row * m);
    /* write: S_t = gamma S_{t-1} + eta x r^T */
    double dgamma = 0.0, deta = 0.0;
    for (int i = 0; i < m; ++i) {
      double dsr = 0.0;
      for (int j = 0; j < dv; ++j) {
        dgamma += dS[(size_t)i * dv + j] * Sp[(size_t)i * dv + j];
        dsr += dS[(size_t)i * dv + j] * r[j];
      }
      deta += x[i] * dsr;
      dx[i] = eta * dsr;
    }
    for (int j = 0; j < dv; ++j) {
      double acc = 0.0;
      for (int i = 0; i < m; ++i) acc += dS[(size_t)i * dv + j] * x[i];
      dr[j] = eta * acc;
      a->dvv[row * dv + j] = dr[j];
    }
    for (size_t e = 0; e < md; ++e) dS[e] *= gamma;
    if (a->rule == ORACLE_FALCON1) {
      for (int i = 0; i < m; ++i) {
        double acc = 0.0;
        for (int j = 0; j < dv; ++j) {
          dS[(size_t)i * dv + j] -= x[i] * dr[j];
          acc += Sp[(size_t)i * dv + j] * dr[j];
        }
        dx[i] -= acc;
      }
    }
    /* step size and decay */
    double dbeta = 0.0, dlam_in = 0.0;
    if (!sentinel && den > 0.0) {
      double dlam = 0.0;
      if (!clamped) {
        const double dalpha = -dgamma;
        deta += lam * dalpha;
        dlam += eta * dalpha;
      }
      dbeta = deta / den;
      const double dden = -deta * eta / den;
      double dE = dden;
      dlam += dden;
      if (a->ridge == ORACLE_RIDGE_SCALED) {
        dlam_in = dlam * E;
        dE += dlam * lam_in;
      } else {
        dlam_in = dlam;
      }
      for (int i = 0; i < m; ++i) dx[i] += 2.0 * dE * x[i];
    }
    a->dbeta[row] = dbeta;
    a->dlambda[row] = dlam_in;
    memcpy(dxn, dx, sizeof(double) * (size_t)m);
    memcpy(Spost, Sp, sizeof(double) * md);
  }
  if (a->dS0) memcpy(a->dS0 + bh * md, dS, sizeof(double) * md);
  if (a->dx_prev) {
    if (fresh)
      memset(a->dx_prev + bh * m, 0, sizeof(double) * (size_t)m);
    else
      memcpy(a->dx_prev + bh * m, dxn, sizeof(double) * (size_t)m);
  }
  free(Spre);
  free(X);
  free(S);
  free(qf);
  free(r);
  free(o);
  free(dS);
  free(Spost);
  free(dx);
  free(dxn);
  free(dr);
  free(dqf);
}

typedef struct {
  const bwd_args *a;
  int64_t begin, end;
} bwd_slice;

static void *backward_worker(void *p) {
  const bwd_slice *s = (const bwd_slice *)p;
  for (int64_t bh = s->begin; bh < s->end; ++bh) backward_head(s->a, bh);
  return NULL;
}

/*
 * Gradients of L = <dO, o> + <dS_T, S_T> + <dx_last, x_last> with respect to
 * every input of falcon_oracle_forward.  Layouts as there; dO [BH, T, dv];
 * dS_T [BH, m, dv] and dx_last [BH, m] nullable (zero cotangents).  Outputs:
 * dq, dk [BH, T, m], dv [BH, T, dv], dbeta, dlambda [BH, T] (dlambda is the
 * gradient with respect to the lambda input: lambda_bar for the scaled
 * ridge), dS0 [BH, m, dv] and dx_prev [BH, m] (nullable; dx_prev is zero for
 * a fresh sequence).  Returns 0, or -1 on a bad argument.
 */
int falcon_oracle_backward(int rule, int64_t BH, int64_t T, int m, int dv, int phi, int ridge,
                           double eps, double eps_gamma, const double *q, const double *k,
                           const double *v, const double *beta, const double *lambda,
                           const double *S0, const double *x_prev, const double *dO,
                           const double *dS_T, const double *dx_last, double *dq, double *dk,
                           double *dvv, double *dbeta, double *dlambda, double *dS0,
                           double *dx_prev, int nthreads) {
  if (rule != ORACLE_FALCON1 && rule != ORACLE_FALCON1A) return -1;
  if (BH < 0 || T < 0 || m <= 0 || dv <= 0) return -1;
  bwd_args a = {rule, m, dv, phi, ridge, T, eps, eps_gamma, q, k, v, beta, lambda, S0, x_prev,
                dO, dS_T, dx_last, dq, dk, dvv, dbeta, dlambda, dS0, dx_prev};
  if (nthreads < 1) nthreads = 1;
  if (nthreads > BH) nthreads = (int)(BH > 0 ? BH : 1);
  pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
  bwd_slice *sl = (bwd_slice *)malloc(sizeof(bwd_slice) * (size_t)nthreads);
  for (int w = 0; w < nthreads; ++w) {
    sl[w].a = &a;
    sl[w].begin = BH * w / nthreads;
    sl[w].end = BH * (w + 1) / nthreads;
  }
  for (int w = 1; w < nthreads; ++w) pthread_create(&tid[w], NULL, backward_worker, &sl[w]);
  backward_worker(&sl[0]);
  for (int w = 1; w < nthreads; ++w) pthread_join(tid[w], NULL);
  free(tid);
  free(sl);
  return 0;
}

/* ---- Falcon-1A with the normalised read -------------------------------- */
typedef struct {
  int m, dv, phi, ridge;
  int64_t T;
  double eps, eps_gamma, eps_attn;
  const double *q, *k, *v, *beta, *lambda, *S0, *z0, *x_prev;
  double *o, *S_out, *z_out, *x_last;
} fwdn_args;

/* One head: the Falcon-1A token loop of forward_head, plus the normaliser
 * z_t = gamma_t z_{t-1} + eta_t x_t and the division of the read. */
static void forward_norm_head(const fwdn_args *a, int64_t bh) {
  const int m = a->m, dv = a->dv;
  const int64_t T = a->T;
  double *S = (double *)calloc((size_t)m * dv, sizeof(double));
  double *z = (double *)calloc((size_t)m, sizeof(double));
  double *x = (double *)calloc((size_t)m, sizeof(double));
  double *qf = (double *)malloc(sizeof(double) * (size_t)m);
  double *r = (double *)malloc(sizeof(double) * (size_t)dv);
  if (a->S0) memcpy(S, a->S0 + bh * m * dv, sizeof(double) * (size_t)m * dv);
  if (a->z0) memcpy(z, a->z0 + bh * m, sizeof(double) * (size_t)m);
  int sentinel = 1;
  if (a->x_prev) {
    memcpy(x, a->x_prev + bh * m, sizeof(double) * (size_t)m);
    sentinel = 0;
  }
  for (int64_t t = 0; t < T; ++t) {
    const int64_t row = bh * T + t;
    double eta, gamma;
    step_scalars(sentinel && t == 0, m, x, a->beta[row], a->lambda[row], a->ridge,
                 a->eps, a->eps_gamma, &eta, &gamma);
    feature_map(a->phi, m, a->q + row * m, qf);
    /* numerator: the Falcon-1A update and read (into o_t) */
    double *o = a->o + row * dv;
    one_token(ORACLE_FALCON1A, m, dv, S, x, qf, a->v + row * dv, eta, gamma, r, o);
    /* normaliser, then the read's denominator */
    double den = 0.0;
    for (int i = 0; i < m; ++i) {
      z[i] = gamma * z[i] + eta * x[i];
      den += z[i] * qf[i];
    }
    den += a->eps_attn;
    for (int j = 0; j < dv; ++j) o[j] /= den;
    feature_map(a->phi, m, a->k + row * m, x);
  }
  if (a->S_out) memcpy(a->S_out + bh * m * dv, S, sizeof(double) * (size_t)m * dv);
  if (a->z_out) memcpy(a->z_out + bh * m, z, sizeof(double) * (size_t)m);
  if (a->x_last) memcpy(a->x_last + bh * m, x, sizeof(double) * (size_t)m);
  free(S);
  free(z);
  free(x);
  free(qf);
  free(r);
}

typedef struct {
  const fwdn_args *a;
  int64_t begin, end;
} fwdn_slice;

static void *forward_norm_worker(void *p) {
  const fwdn_slice *s = (const fwdn_slice *)p;
  for (int64_t bh = s->begin; bh < s->end; ++bh) forward_norm_head(s->a, bh);
  return NULL;
}

/*
 * Falcon-1A with the normalised read o_t = S_t^T phi(q_t) / (z_t^T phi(q_t) +
 * eps_attn), z_t = gamma_t z_{t-1} + eta_t x_t.  Layouts as in
 * falcon_oracle_forward; z0 (nullable => zeros) and z_out (nullable): [BH, m].
 * Returns 0, or -1 on a bad argument.
 */
int falcon1a_oracle_forward_normalized(int64_t BH, int64_t T, int m, int dv, int phi, int ridge,
                                       double eps, double eps_gamma, double eps_attn,
                                       const double *q, const double *k, const double *v,
                                       const double *beta, const double *lambda,
                                       const double *S0, const double *z0, const double *x_prev,
                                       double *o, double *S_out, double *z_out, double *x_last,
                                       int nthreads) {
  if (BH < 0 || T < 0 || m <= 0 || dv <= 0) return -1;
  fwdn_args a = {m, dv, phi, ridge, T, eps, eps_gamma, eps_attn, q, k, v, beta, lambda,
                 S0, z0, x_prev, o, S_out, z_out, x_last};
  if (nthreads < 1) nthreads = 1;
  if (nthreads > BH) nthreads = (int)(BH > 0 ? BH : 1);
  pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
  fwdn_slice *sl = (fwdn_slice *)malloc(sizeof(fwdn_slice) * (size_t)nthreads);
  for (int w = 0; w < nthreads; ++w) {
    sl[w].a = &a;
    sl[w].begin = BH * w / nthreads;
    sl[w].end = BH * (w + 1) / nthreads;
  }
  for (int w = 1; w < nthreads; ++w) pthread_create(&tid[w], NULL, forward_norm_worker, &sl[w]);
  forward_norm_worker(&sl[0]);
  for (int w = 1; w < nthreads; ++w) pthread_join(tid[w], NULL);
  free(tid);
  free(sl);
  return 0;
}

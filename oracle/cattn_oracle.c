/*
 * cattn_oracle.c -- plain, slow, fp64 CPU definition of the pluggable-map
 * attention forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file.  It shares no code, header, table or helper with the CUDA
 * library under softmax_free_attention_gb300/csrc; the two meet only through
 * the seeded inputs that the tests hand to both.
 *
 * Everything is computed in double precision from the inputs exactly as
 * stored (bf16 or fp32 values widened to fp64 by the caller), one query row
 * at a time, in the order the source pages state the steps.  There is no
 * tiling, no fusion and no reordering of the definitions.
 *
 * Sources (page title, section):
 *   - "Softmax-Free Attention in JAX/Flax NNX", section "One module, two
 *     compatibility functions": the softmax branch (scores / sqrt(d_h),
 *     masked to -inf, softmax over the key axis) and the Yat branch
 *     (kappa = (q.k + b)^2 / (max(|q-k|^2, 0) + eps), masked kappa = 0,
 *     mass = sum of kappa over keys, w = kappa / (mass + 1e-9)).
 *   - "The Kernel Between the Roles", sections "What the exponential was
 *     hired to do" and "What each normalizer forgets": the Yat kernel with
 *     per-head b, eps > 0 and the row mass m_i = sum_j kappa_ij kept as a
 *     channel of its own.
 *   - "NNX Scaled Dot-Product Attention", sections "Shapes and the three
 *     steps" and "Mask before softmax": shapes (T_q, d_k), (T_k, d_k),
 *     (T_k, d_v), softmax along the key axis, weights @ v, causal mask blocks
 *     future positions.
 *   - "s^tau: a focal-length knob for attention" (forum.trae.cn topic 15798),
 *     the core-formula paragraph: a_i = phi(s_i)^tau / sum_j phi(s_j)^tau,
 *     phi(s) = softplus(s) + eps, one tau per head.
 *
 * Readings where the pages leave a step open:
 *   - Yat scores are the raw q.k (no 1/sqrt(d) scale); softmax and s^tau use
 *     s = scale * q.k with the caller's scale.
 *   - The squared distance |q-k|^2 is summed directly over the components
 *     here (no norm expansion); the max(., 0) clamp is kept as written.
 *   - s^tau excludes masked keys (zero weight, no contribution to the sum),
 *     as the Yat branch does with zero mass.
 *   - The power phi^tau is taken literally with pow(); a non-finite value is
 *     reported as an error instead of being hidden.
 *   - Causal: key j is allowed for query row t when j <= t.
 *   - GQA: query head i reads key/value head i / (h / hkv); b, eps, tau are
 *     indexed by query head.
 *   - Telemetry per row: Yat row_mass = sum kappa (without the 1e-9),
 *     row_max = max kappa; softmax row_mass = log-sum-exp of the scaled
 *     scores, row_max = max scaled score; s^tau row_mass = log sum phi^tau,
 *     row_max = max scaled score.
 *
 * Yat numerator power ("The Kernel Between the Roles", section "The run":
 * raising the numerator's power, (q.k)^{2m}, sharpens the kernel's peak):
 * kappa = (q.k + b)^{2m} / (max(|q-k|^2, 0) + eps) with an integer m >= 1
 * (m = 1 is the kernel above; b = 0 gives the page's ablation).  Reading:
 * the bias stays inside the power, as in the m = 1 kernel.
 *
 * tau* (same s^tau page, the closed-form paragraph: tau* = Cov(s, log phi(s))
 * / Var(log phi(s)), taken from the score distribution of one forward pass,
 * one value per attention head).  Readings: the scores are the softmax
 * scores s = scale * q.k of every allowed (query row, key) pair of the query
 * head, pooled over the batch; log is the natural log (the slope that makes
 * tau * ln phi(s) + C fit s, which is what the page's equivalence
 * s^tau <-> softmax needs); phi uses the head's s^tau eps.  Covariance and
 * variance are computed in two passes (means first), in fp64.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_SOFTMAX 0
#define ORACLE_YAT 1
#define ORACLE_STAU 2

#define ORACLE_OK 0
#define ORACLE_EBADARG -1
#define ORACLE_ENONFINITE -2
#define ORACLE_ENOMEM -3

typedef struct {
  int variant;
  int B, h, hkv, Tq, Tk, dk, dv;
  int causal;
  double scale;
  const double *q;   /* [B, h,   Tq, dk] */
  const double *k;   /* [B, hkv, Tk, dk] */
  const double *v;   /* [B, hkv, Tk, dv] */
  const double *b;   /* [h] (Yat)   */
  const double *eps; /* [h] (Yat, s^tau) */
  const double *tau; /* [h] (s^tau) */
  const int64_t *rows; /* flat indices into [B, h, Tq]; NULL = every row */
  int64_t nrows;
  double *out;      /* [nrows, dv] */
  double *row_mass; /* [nrows] */
  double *row_max;  /* [nrows] */
  double *weights;  /* optional [nrows, Tk]; NULL = not wanted */
  int yat_m;         /* Yat numerator exponent 2m; 0 is read as m = 1 */
} oracle_problem;

/* softplus(s) = log(1 + exp(s)), in the textbook overflow-free form. */
static double softplus(double s) { return fmax(s, 0.0) + log1p(exp(-fabs(s))); }

static double dot(const double *x, const double *y, int n) {
  double acc = 0.0;
  for (int d = 0; d < n; ++d) acc += x[d] * y[d];
  return acc;
}

static double sqdist(const double *x, const double *y, int n) {
  double acc = 0.0;
  for (int d = 0; d < n; ++d) {
    double diff = x[d] - y[d];
    acc += diff * diff;
  }
  return acc;
}

/* One query row.  `w` is scratch of length Tk that ends up holding the
 * normalised weights (zero for excluded keys). */
static int oracle_row(const oracle_problem *p, int64_t flat, int64_t slot, double *w) {
  const int t = (int)(flat % p->Tq);
  const int64_t bh = flat / p->Tq;
  const int head = (int)(bh % p->h);
  const int bi = (int)(bh / p->h);
  const int group = p->h / p->hkv;
  const int g = head / group;

  const double *qrow = p->q + flat * (int64_t)p->dk;
  const double *kbase = p->k + ((int64_t)bi * p->hkv + g) * (int64_t)p->Tk * p->dk;
  const double *vbase = p->v + ((int64_t)bi * p->hkv + g) * (int64_t)p->Tk * p->dv;

  int nallowed = p->Tk;
  if (p->causal && t + 1 < nallowed) nallowed = t + 1;
  for (int j = nallowed; j < p->Tk; ++j) w[j] = 0.0;

  double row_mass = 0.0, row_max = -INFINITY;

  if (p->variant == ORACLE_SOFTMAX) {
    /* scores = scale * q.k; softmax over the allowed keys. */
    double m = -INFINITY;
    for (int j = 0; j < nallowed; ++j) {
      w[j] = p->scale * dot(qrow, kbase + (int64_t)j * p->dk, p->dk);
      if (w[j] > m) m = w[j];
    }
    double l = 0.0;
    for (int j = 0; j < nallowed; ++j) {
      w[j] = exp(w[j] - m);
      l += w[j];
    }
    for (int j = 0; j < nallowed; ++j) w[j] /= l;
    row_mass = m + log(l);
    row_max = m;
  } else if (p->variant == ORACLE_YAT) {
    /* kappa = (q.k + b)^{2m} / (max(|q-k|^2, 0) + eps); w = kappa / (mass + 1e-9). */
    const double bh_ = p->b[head], eh = p->eps[head];
    const int m = p->yat_m > 1 ? p->yat_m : 1;
    double mass = 0.0, kmax = -INFINITY;
    for (int j = 0; j < nallowed; ++j) {
      const double *krow = kbase + (int64_t)j * p->dk;
      double num = dot(qrow, krow, p->dk) + bh_;
      double d2 = sqdist(qrow, krow, p->dk);
      double kappa = pow(num, 2.0 * m) / (fmax(d2, 0.0) + eh);
      w[j] = kappa;
      mass += kappa;
      if (kappa > kmax) kmax = kappa;
    }
    for (int j = 0; j < nallowed; ++j) w[j] = w[j] / (mass + 1e-9);
    row_mass = mass;
    row_max = kmax;
  } else if (p->variant == ORACLE_STAU) {
    /* a_j = phi(s_j)^tau / sum phi^tau, phi = softplus(s) + eps, s = scale * q.k. */
    const double eh = p->eps[head], th = p->tau[head];
    double smax = -INFINITY, z = 0.0;
    for (int j = 0; j < nallowed; ++j) {
      double s = p->scale * dot(qrow, kbase + (int64_t)j * p->dk, p->dk);
      if (s > smax) smax = s;
      double phi = softplus(s) + eh;
      double u = pow(phi, th);
      if (!isfinite(u)) return ORACLE_ENONFINITE;
      w[j] = u;
      z += u;
    }
    if (!isfinite(z) || !(z > 0.0)) return ORACLE_ENONFINITE;
    for (int j = 0; j < nallowed; ++j) w[j] /= z;
    row_mass = log(z);
    row_max = smax;
  } else {
    return ORACLE_EBADARG;
  }

  /* out = weights @ v */
  double *orow = p->out + slot * (int64_t)p->dv;
  for (int d = 0; d < p->dv; ++d) orow[d] = 0.0;
  for (int j = 0; j < nallowed; ++j) {
    const double *vrow = vbase + (int64_t)j * p->dv;
    for (int d = 0; d < p->dv; ++d) orow[d] += w[j] * vrow[d];
  }
  p->row_mass[slot] = row_mass;
  p->row_max[slot] = row_max;
  if (p->weights) memcpy(p->weights + slot * (int64_t)p->Tk, w, sizeof(double) * (size_t)p->Tk);
  return ORACLE_OK;
}

typedef struct {
  const oracle_problem *p;
  int64_t begin, end;
  int status;
} oracle_job;

static void *oracle_worker(void *arg) {
  oracle_job *job = (oracle_job *)arg;
  const oracle_problem *p = job->p;
  double *w = (double *)malloc(sizeof(double) * (size_t)(p->Tk > 0 ? p->Tk : 1));
  if (!w) {
    job->status = ORACLE_ENOMEM;
    return NULL;
  }
  job->status = ORACLE_OK;
  for (int64_t s = job->begin; s < job->end; ++s) {
    int64_t flat = p->rows ? p->rows[s] : s;
    int rc = oracle_row(p, flat, s, w);
    if (rc != ORACLE_OK) {
      job->status = rc;
      break;
    }
  }
  free(w);
  return NULL;
}

/* Entry point (C ABI, called through ctypes by the tests and by the CPU
 * baseline of the benchmark).  Rows are split evenly over `nthreads` POSIX
 * threads; each row is independent. */
int oracle_forward(const oracle_problem *p, int nthreads) {
  if (!p || !p->q || !p->k || !p->v || !p->out || !p->row_mass || !p->row_max) return ORACLE_EBADARG;
  if (p->B <= 0 || p->h <= 0 || p->hkv <= 0 || p->Tq <= 0 || p->Tk <= 0 || p->dk <= 0 || p->dv <= 0)
    return ORACLE_EBADARG;
  if (p->h % p->hkv != 0) return ORACLE_EBADARG;
  if (p->variant == ORACLE_YAT && (!p->b || !p->eps)) return ORACLE_EBADARG;
  if (p->variant == ORACLE_STAU && (!p->eps || !p->tau)) return ORACLE_EBADARG;
  const int64_t total = (int64_t)p->B * p->h * p->Tq;
  if (p->rows) {
    for (int64_t s = 0; s < p->nrows; ++s)
      if (p->rows[s] < 0 || p->rows[s] >= total) return ORACLE_EBADARG;
  } else if (p->nrows != total) {
    return ORACLE_EBADARG;
  }
  if (nthreads < 1) nthreads = 1;
  if (nthreads > p->nrows) nthreads = (int)(p->nrows > 0 ? p->nrows : 1);

  oracle_job *jobs = (oracle_job *)calloc((size_t)nthreads, sizeof(oracle_job));
  pthread_t *tids = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
  if (!jobs || !tids) {
    free(jobs);
    free(tids);
    return ORACLE_ENOMEM;
  }
  for (int i = 0; i < nthreads; ++i) {
    jobs[i].p = p;
    jobs[i].begin = p->nrows * i / nthreads;
    jobs[i].end = p->nrows * (i + 1) / nthreads;
  }
  int started = 0;
  for (int i = 1; i < nthreads; ++i) {
    if (pthread_create(&tids[i], NULL, oracle_worker, &jobs[i]) != 0) break;
    started = i;
  }
  oracle_worker(&jobs[0]);
  for (int i = 1; i <= started; ++i) pthread_join(tids[i], NULL);
  /* any thread that could not be started runs here */
  for (int i = started + 1; i < nthreads; ++i) oracle_worker(&jobs[i]);
  int rc = ORACLE_OK;
  for (int i = 0; i < nthreads; ++i)
    if (jobs[i].status != ORACLE_OK) rc = jobs[i].status;
  free(jobs);
  free(tids);
  return rc;
}

/* tau* over n scores: the least-squares slope Cov(s, ln phi(s)) / Var(ln phi(s))
 * with phi = softplus + eps.  Two passes: the means, then the centred sums.
 * Returns NaN when there are fewer than two scores or ln phi is constant. */
double oracle_tau_star_scores(const double *s, int64_t n, double eps) {
  if (!s || n < 2) return NAN;
  double ms = 0.0, mg = 0.0;
  for (int64_t i = 0; i < n; ++i) {
    ms += s[i];
    mg += log(softplus(s[i]) + eps);
  }
  ms /= (double)n;
  mg /= (double)n;
  double cov = 0.0, var = 0.0;
  for (int64_t i = 0; i < n; ++i) {
    const double ds = s[i] - ms, dg = log(softplus(s[i]) + eps) - mg;
    cov += ds * dg;
    var += dg * dg;
  }
  if (!(var > 0.0)) return NAN;
  return cov / var;
}

/* tau* of every query head: gathers the allowed scores s = scale * q.k of
 * the head over all batches and rows (causal: key j <= row t), then applies
 * oracle_tau_star_scores with the head's eps.  tau_out: [h].  n_out
 * (optional): [h] counts of allowed pairs. */
int oracle_tau_star(const oracle_problem *p, double *tau_out, double *n_out) {
  if (!p || !p->q || !p->k || !p->eps || !tau_out) return ORACLE_EBADARG;
  if (p->B <= 0 || p->h <= 0 || p->hkv <= 0 || p->Tq <= 0 || p->Tk <= 0 || p->dk <= 0)
    return ORACLE_EBADARG;
  if (p->h % p->hkv != 0) return ORACLE_EBADARG;
  if (p->causal && p->Tq != p->Tk) return ORACLE_EBADARG;
  const int group = p->h / p->hkv;
  double *sc = (double *)malloc(sizeof(double) * (size_t)p->B * p->Tq * p->Tk);
  if (!sc) return ORACLE_ENOMEM;
  for (int i = 0; i < p->h; ++i) {
    int64_t n = 0;
    for (int b = 0; b < p->B; ++b)
      for (int t = 0; t < p->Tq; ++t) {
        const double *qr = p->q + (((int64_t)b * p->h + i) * p->Tq + t) * p->dk;
        for (int j = 0; j < p->Tk; ++j) {
          if (p->causal && j > t) continue;
          const double *kr = p->k + (((int64_t)b * p->hkv + i / group) * p->Tk + j) * p->dk;
          sc[n++] = p->scale * dot(qr, kr, p->dk);
        }
      }
    tau_out[i] = oracle_tau_star_scores(sc, n, p->eps[i]);
    if (n_out) n_out[i] = (double)n;
  }
  free(sc);
  return ORACLE_OK;
}

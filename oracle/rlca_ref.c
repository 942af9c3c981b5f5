/*
 * rlca_ref.c -- plain C, float64, one row at a time: a second,
 * independent CPU reference of the credit-assignment estimators.
 *
 * TEST INFRASTRUCTURE: only the test suite uses it (through oracle/ref_c.py),
 * to check the NumPy reference (oracle/rlca_ref.py) against a separate
 * implementation and to run the same pins on both.  It shares no code with
 * the CUDA path or with the NumPy reference.
 *
 * Source: "rl-triton: High-Performance Triton GPU Kernels for Reinforcement
 * Learning Credit Assignment" (arXiv:2608.17641), §1 Introduction, §3 The
 * Unified Linear Recurrence Framework (§3.2 episode-boundary semantics, §3.3
 * algorithm-specific recurrences), with the estimator definitions of the
 * works it cites (GAE: Schulman et al. 2016; V-Trace: Espeholt et al. 2018;
 * Retrace(lambda): Munos et al. 2016).  Each estimator is its time-step loop
 * over one environment row, never the (alpha, beta) scan form.
 *
 * Layout: env-major [E][T] (per-action [E][T][A]), flags one byte each
 * (nonzero = set), [E] vectors for bootstrap / carry.  Optional arrays may be
 * NULL: terminated / truncated (no flags), bootstrap / carry (zero).
 *
 * Boundary rules (§3.2), with the readings the NumPy reference takes:
 *   terminated at t          -> successor value 0
 *   truncated at t (not term) -> successor value trunc_value[t]
 *   t = T-1 otherwise        -> successor value bootstrap
 *   forward scans restart after a flagged step and on the first step.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>

static int flag_at(const uint8_t *f, int64_t i) { return f != NULL && f[i] != 0; }

/* successor value of step t of a row (offset `o` = row start) when the
 * continuation through step t+1 is `interior` */
static double successor(int64_t o, int64_t t, int64_t T, double interior, const uint8_t *term,
                        const uint8_t *trunc, const double *tv, double boot) {
  if (flag_at(term, o + t)) return 0.0;
  if (flag_at(trunc, o + t)) return tv[o + t];
  if (t == T - 1) return boot;
  return interior;
}

/* does step t's result depend on step t+1's (no edge at t, inside the window) */
static int continues(int64_t o, int64_t t, int64_t T, const uint8_t *term, const uint8_t *trunc) {
  return !flag_at(term, o + t) && !flag_at(trunc, o + t) && t < T - 1;
}

static double boot_of(const double *boot, int64_t e) { return boot != NULL ? boot[e] : 0.0; }

/* A_t = alpha_t + beta_t * A_{t+1} (reverse) or A_{t-1} (forward); the
 * carry (A_T or A_{-1}) is carry[e] or 0. */
void ref_affine_scan(const double *alpha, const double *beta, const double *carry, int64_t E, int64_t T,
                     int reverse, double *out) {
  for (int64_t e = 0; e < E; ++e) {
    const int64_t o = e * T;
    double A = carry != NULL ? carry[e] : 0.0;
    for (int64_t k = 0; k < T; ++k) {
      const int64_t t = reverse ? T - 1 - k : k;
      A = alpha[o + t] + beta[o + t] * A;
      out[o + t] = A;
    }
  }
}

/* GAE: delta_t = r_t + gamma V_next(t) - V_t; A_t = delta_t + gamma lam
 * A_{t+1} while the episode continues inside the window; R_t = A_t + V_t. */
void ref_gae(const double *r, const double *v, const uint8_t *term, const uint8_t *trunc, const double *tv,
             const double *boot, int64_t E, int64_t T, double gamma, double lam, double *adv, double *ret) {
  for (int64_t e = 0; e < E; ++e) {
    const int64_t o = e * T;
    double later = 0.0; /* A_{t+1} */
    for (int64_t t = T - 1; t >= 0; --t) {
      const double v_next = t + 1 < T ? v[o + t + 1] : 0.0;
      const double delta = r[o + t] + gamma * successor(o, t, T, v_next, term, trunc, tv, boot_of(boot, e)) -
                           v[o + t];
      const double a = delta + (continues(o, t, T, term, trunc) ? gamma * lam * later : 0.0);
      adv[o + t] = a;
      if (ret != NULL) ret[o + t] = a + v[o + t];
      later = a;
    }
  }
}

/* G_t = r_t + gamma G_next(t), G_next = G_{t+1} inside an episode. */
void ref_discounted_return(const double *r, const uint8_t *term, const uint8_t *trunc, const double *tv,
                           const double *boot, int64_t E, int64_t T, double gamma, double *out) {
  for (int64_t e = 0; e < E; ++e) {
    const int64_t o = e * T;
    double later = 0.0; /* G_{t+1} */
    for (int64_t t = T - 1; t >= 0; --t) {
      const double g = r[o + t] + gamma * successor(o, t, T, later, term, trunc, tv, boot_of(boot, e));
      out[o + t] = g;
      later = g;
    }
  }
}

/* G_t = r_t + gamma [(1 - lam) V_{t+1} + lam G_{t+1}] inside an episode. */
void ref_td_lambda(const double *r, const double *v, const uint8_t *term, const uint8_t *trunc, const double *tv,
                   const double *boot, int64_t E, int64_t T, double gamma, double lam, double *out) {
  for (int64_t e = 0; e < E; ++e) {
    const int64_t o = e * T;
    double later = 0.0; /* G_{t+1} */
    for (int64_t t = T - 1; t >= 0; --t) {
      const double inner = t + 1 < T ? (1.0 - lam) * v[o + t + 1] + lam * later : 0.0;
      const double g = r[o + t] + gamma * successor(o, t, T, inner, term, trunc, tv, boot_of(boot, e));
      out[o + t] = g;
      later = g;
    }
  }
}

/* V-Trace: ratio = exp(lp_t - lb_t), rho = min(rho_bar, ratio),
 * c = lam min(c_bar, ratio); delta = rho (r + gamma V_next - V);
 * vs - V = delta + gamma c (vs_{t+1} - V_{t+1}) while the episode continues;
 * pg = rho (r + gamma vs_next - V), vs_next = V_next with vs_{t+1}. */
void ref_vtrace(const double *r, const double *v, const double *lp, const double *lb, const uint8_t *term,
                const uint8_t *trunc, const double *tv, const double *boot, int64_t E, int64_t T, double gamma,
                double rho_bar, double c_bar, double lam, double *vs, double *pg) {
  for (int64_t e = 0; e < E; ++e) {
    const int64_t o = e * T;
    const double b = boot_of(boot, e);
    double later_gap = 0.0; /* vs_{t+1} - V_{t+1} */
    double later_vs = 0.0;  /* vs_{t+1} */
    for (int64_t t = T - 1; t >= 0; --t) {
      const double ratio = exp(lp[o + t] - lb[o + t]);
      const double rho = ratio < rho_bar ? ratio : rho_bar;
      const double c = lam * (ratio < c_bar ? ratio : c_bar);
      const double v_next = t + 1 < T ? v[o + t + 1] : 0.0;
      const double delta = rho * (r[o + t] + gamma * successor(o, t, T, v_next, term, trunc, tv, b) - v[o + t]);
      const double gap = delta + (continues(o, t, T, term, trunc) ? gamma * c * later_gap : 0.0);
      const double s = v[o + t] + gap;
      vs[o + t] = s;
      if (pg != NULL)
        pg[o + t] = rho * (r[o + t] + gamma * successor(o, t, T, later_vs, term, trunc, tv, b) - v[o + t]);
      later_gap = gap;
      later_vs = s;
    }
  }
}

/* Retrace(lambda): EV_t = sum_a pi Q, c_t = lam min(1, pi(a_t) / mu(a_t)),
 * G_t = r_t + gamma [EV_{t+1} + c_{t+1} (G_{t+1} - Q(x_{t+1}, a_{t+1}))]
 * inside an episode.  Actions outside [0, A) are clamped (the reading the
 * NumPy reference cannot express: callers pass valid actions). */
static int64_t clamp_action(int32_t a, int64_t A) { return a < 0 ? 0 : (a >= A ? A - 1 : a); }

void ref_retrace(const double *q, const double *pi, const double *mu_a, const int32_t *act, const double *r,
                 const uint8_t *term, const uint8_t *trunc, const double *tv, const double *boot, int64_t E,
                 int64_t T, int64_t A, double gamma, double lam, double *out) {
  for (int64_t e = 0; e < E; ++e) {
    const int64_t o = e * T;
    double later = 0.0; /* G_{t+1} */
    for (int64_t t = T - 1; t >= 0; --t) {
      double inner = 0.0;
      if (t + 1 < T) {
        const int64_t s = o + t + 1;
        const double *qs = q + s * A, *ps = pi + s * A;
        double ev = 0.0;
        for (int64_t a = 0; a < A; ++a) ev += ps[a] * qs[a];
        const int64_t at = clamp_action(act[s], A);
        const double ratio = ps[at] / mu_a[s];
        const double c = lam * (ratio < 1.0 ? ratio : 1.0);
        inner = ev + c * (later - qs[at]);
      }
      const double g = r[o + t] + gamma * successor(o, t, T, inner, term, trunc, tv, boot_of(boot, e));
      out[o + t] = g;
      later = g;
    }
  }
}

/* accumulating trace, forward: e_t = x_t + gamma lam e_{t-1}, restarting on
 * the first step and on every step after a flagged one. */
void ref_eligibility_trace(const double *x, const uint8_t *term, const uint8_t *trunc, int64_t E, int64_t T,
                           double gamma, double lam, double *out) {
  for (int64_t e = 0; e < E; ++e) {
    const int64_t o = e * T;
    double prev = 0.0;
    for (int64_t t = 0; t < T; ++t) {
      const int restart = t == 0 || flag_at(term, o + t - 1) || flag_at(trunc, o + t - 1);
      prev = x[o + t] + (restart ? 0.0 : gamma * lam * prev);
      out[o + t] = prev;
    }
  }
}

/* does step t start a new episode (forward scans) */
static int starts_episode(int64_t o, int64_t t, const uint8_t *term, const uint8_t *trunc, int flag_is_start) {
  if (t == 0) return 1;
  const int64_t i = flag_is_start ? o + t : o + t - 1;
  return flag_at(term, i) || flag_at(trunc, i);
}

/* running sum of x within each episode (inclusive, or exclusive: the steps
 * before t); a flagged step ends its episode, or with flag_is_start begins
 * the next one. */
void ref_prefix_sum_f64(const double *x, const uint8_t *term, const uint8_t *trunc, int64_t E, int64_t T,
                        int exclusive, int flag_is_start, double *out) {
  for (int64_t e = 0; e < E; ++e) {
    const int64_t o = e * T;
    double running = 0.0;
    for (int64_t t = 0; t < T; ++t) {
      const double before = starts_episode(o, t, term, trunc, flag_is_start) ? 0.0 : running;
      running = before + x[o + t];
      out[o + t] = exclusive ? before : running;
    }
  }
}

/* the int32 variant: two's-complement wraparound (summed as uint32) */
void ref_prefix_sum_i32(const int32_t *x, const uint8_t *term, const uint8_t *trunc, int64_t E, int64_t T,
                        int exclusive, int flag_is_start, int32_t *out) {
  for (int64_t e = 0; e < E; ++e) {
    const int64_t o = e * T;
    uint32_t running = 0u;
    for (int64_t t = 0; t < T; ++t) {
      const uint32_t before = starts_episode(o, t, term, trunc, flag_is_start) ? 0u : running;
      running = before + (uint32_t)x[o + t];
      const uint32_t r = exclusive ? before : running;
      out[o + t] = (int32_t)(r <= 0x7fffffffu ? (int64_t)r : (int64_t)r - 4294967296LL);
    }
  }
}

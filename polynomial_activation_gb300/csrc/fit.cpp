// fit.cpp -- host-side constrained fitter (poly_fit).
//
// "Fast Polynomial Transcendentals for LLMs" (arXiv 2610.00049), §3.2:
//   1. for each degree D and fit interval Li, solve the dual endpoint-
//      constrained least-squares problem of eq. 7-8 in FP64 on 2,000
//      Chebyshev nodes;
//   2. round every coefficient to the target format;
//   3. replay the program with target-format rounding at each multiply and
//      add, with the kernel's reduction, clamp, sign restoration and offset;
//   4. score the maximum absolute error on 8,000 points over [0, 12] and
//      reject clamps with Lc > Li + 1 and shape or boundary violations;
//   5. re-score the candidates in the deployed packed-FMA order (one
//      rounding per FMA) and accept the best of those.
// Readings where the paper is silent: first-kind Chebyshev nodes; Li on
// {1, 1.25, ..., 12} and Lc on {1, 1.25, ..., Li + 1}; the score points are
// linspace(0, 12, 8000) rounded to the format; gates = finite outputs, exact
// P(0) = f(0), output range for sigmoid / tanh / sigma' / tanh', and a
// monotone real-arithmetic replay for functions monotone on t >= 0; every
// gated candidate is re-scored in deployed order (exact ties to the smaller
// Table 2 metric, then the smaller Li, then the smaller Lc).
#include <algorithm>
#include <cmath>
#include <cstring>
#include <thread>
#include <vector>

#include "fit_internal.h"
#include "softhalf.h"

namespace polyact {

// ---------------------------------------------------------------- functions

static double sigmoid(double x) {
  if (x >= 0) return 1.0 / (1.0 + std::exp(-x));
  double z = std::exp(x);
  return z / (1.0 + z);
}
static double Phi(double x) { return 0.5 * std::erfc(-x / std::sqrt(2.0)); }
static double phi(double x) { return std::exp(-0.5 * x * x) / std::sqrt(2.0 * M_PI); }

double fn_value(int fn, int dir, double x) {
  if (dir == POLY_FWD) {
    switch (fn) {
      case POLY_SIGMOID: return sigmoid(x);
      case POLY_TANH: return std::tanh(x);
      case POLY_SILU: return x * sigmoid(x);
      default: return x * Phi(x);
    }
  }
  switch (fn) {
    case POLY_SIGMOID: return sigmoid(x) * sigmoid(-x);
    case POLY_TANH: {
      double c = std::cosh(x);
      return 1.0 / (c * c);
    }
    case POLY_SILU: return sigmoid(x) + x * (sigmoid(x) * sigmoid(-x));
    default: return Phi(x) + x * phi(x);
  }
}

int form_of_fn(int fn, int dir) {
  if (dir == POLY_FWD) {
    if (fn == POLY_SIGMOID) return POLY_FORM_CO;
    if (fn == POLY_TANH) return POLY_FORM_O;
    return POLY_FORM_HX;
  }
  if (fn == POLY_SIGMOID || fn == POLY_TANH) return POLY_FORM_E;
  return POLY_FORM_CO;
}

// The half-domain target of the fit (§3.1, §3.3).
static double residual(int fn, int dir, double t) {
  switch (form_of_fn(fn, dir)) {
    case POLY_FORM_CO: return fn_value(fn, dir, t) - 0.5;
    case POLY_FORM_HX: return fn == POLY_SILU ? t * (sigmoid(t) - 0.5) : t * (Phi(t) - 0.5);
    default: return fn_value(fn, dir, t);
  }
}

double residual_at_zero(int fn, int dir) {
  if (form_of_fn(fn, dir) != POLY_FORM_E) return 0.0;
  return fn == POLY_SIGMOID ? 0.25 : 1.0;
}

static bool value_range(int fn, int dir, double *lo, double *hi) {
  if (fn == POLY_SIGMOID) {
    *lo = 0.0;
    *hi = dir == POLY_FWD ? 1.0 : 0.25;
    return true;
  }
  if (fn == POLY_TANH) {
    *lo = dir == POLY_FWD ? -1.0 : 0.0;
    *hi = 1.0;
    return true;
  }
  return false;
}

// +1 rising / -1 falling on t >= 0 / 0 neither (SiLU', GELU' overshoot 1).
static int monotone_on_half(int fn, int dir) {
  if (dir == POLY_FWD) return 1;
  return (fn == POLY_SIGMOID || fn == POLY_TANH) ? -1 : 0;
}

// ------------------------------------------------------------------ replay

uint16_t replay_one(int form, const uint16_t *coef, int degree, uint16_t lc, uint16_t x,
                    int dtype, bool fused) {
  const uint16_t half = dtype == POLY_F16 ? 0x3800 : 0x3F00;
  const uint16_t a = x & 0x7FFF;
  uint16_t t;
  if (is_nan_bits(a, dtype)) {
    t = kQuietNaN;
  } else {
    t = to_double(a, dtype) < to_double(lc, dtype) ? a : lc;
  }
  const int last = form == POLY_FORM_E ? 0 : 1;
  uint16_t v = coef[degree];
  for (int j = degree - 1; j >= last; --j)
    v = fused ? soft_fma(v, t, coef[j], dtype) : soft_add(soft_mul(v, t, dtype), coef[j], dtype);
  const uint16_t sgn = x & 0x8000;
  switch (form) {
    case POLY_FORM_E: return v;
    case POLY_FORM_CO:
      return fused ? soft_fma(v ^ sgn, t, half, dtype)
                   : soft_add(soft_mul(v ^ sgn, t, dtype), half, dtype);
    case POLY_FORM_O: return soft_mul(v ^ sgn, t, dtype);
    default: {
      uint16_t h = soft_mul(x, half, dtype);
      uint16_t y = fused ? soft_fma(v, t, h, dtype) : soft_add(soft_mul(v, t, dtype), h, dtype);
      if (!is_nan_bits(a, dtype) && to_double(a, dtype) > to_double(lc, dtype))
        y = to_double(x, dtype) > 0 ? x : 0;
      return y;
    }
  }
}

double replay_real(int form, const double *c, int degree, double lc, double x) {
  double t = std::min(std::fabs(x), lc);
  const int last = form == POLY_FORM_E ? 0 : 1;
  double v = c[degree];
  for (int j = degree - 1; j >= last; --j) {
    double m = v * t;   // separate multiply and add (host code is built without contraction)
    v = m + c[j];
  }
  if (form == POLY_FORM_E) return v;
  double sv = std::signbit(x) ? -v : v;
  if (form == POLY_FORM_CO) return 0.5 + sv * t;
  if (form == POLY_FORM_O) return sv * t;
  if (std::fabs(x) > lc) return std::max(x, 0.0);
  return 0.5 * x + v * t;
}

// ----------------------------------------------------- least squares (eq. 8)

// Solve min ||A b - y|| (A: m x k, column-major) by Householder QR.
static void householder_lstsq(std::vector<double> &A, int m, int k, std::vector<double> &y,
                              double *b) {
  for (int j = 0; j < k; ++j) {
    double *col = &A[(size_t)j * m];
    double norm = 0;
    for (int i = j; i < m; ++i) norm += col[i] * col[i];
    norm = std::sqrt(norm);
    double alpha = col[j] > 0 ? -norm : norm;
    // v = col[j:] - alpha e1, stored in place
    col[j] -= alpha;
    double vnorm2 = 0;
    for (int i = j; i < m; ++i) vnorm2 += col[i] * col[i];
    if (vnorm2 == 0) continue;
    for (int jj = j + 1; jj < k; ++jj) {
      double *c2 = &A[(size_t)jj * m];
      double s = 0;
      for (int i = j; i < m; ++i) s += col[i] * c2[i];
      s = 2 * s / vnorm2;
      for (int i = j; i < m; ++i) c2[i] -= s * col[i];
    }
    double s = 0;
    for (int i = j; i < m; ++i) s += col[i] * y[i];
    s = 2 * s / vnorm2;
    for (int i = j; i < m; ++i) y[i] -= s * col[i];
    // the diagonal of R is alpha; keep it where back substitution finds it
    col[j] = alpha;
    for (int i = j + 1; i < m; ++i) col[i] = 0;   // v no longer needed
  }
  for (int j = k - 1; j >= 0; --j) {
    double s = y[j];
    for (int jj = j + 1; jj < k; ++jj) s -= A[(size_t)jj * m + j] * b[jj];
    b[j] = s / A[(size_t)j * m + j];
  }
}

void fit_coefficients(int fn, int dir, int degree, double li, int n_nodes, double *c) {
  const double f0 = residual_at_zero(fn, dir);
  const double fl = residual(fn, dir, li);
  const double slope = (fl - f0) / li;
  const int k = degree - 1;
  std::vector<double> A((size_t)n_nodes * k), y(n_nodes);
  for (int i = 0; i < n_nodes; ++i) {
    double x = 0.5 * li * (1.0 + std::cos((2.0 * i + 1.0) * M_PI / (2.0 * n_nodes)));
    double u = x / li;   // normalised coordinate: basis u^j - u (Fig. 2a)
    double uj = u;
    for (int j = 2; j <= degree; ++j) {
      uj *= u;
      A[(size_t)(j - 2) * n_nodes + i] = uj - u;
    }
    y[i] = residual(fn, dir, x) - (f0 + x * slope);
  }
  double b[POLY_MAX_DEGREE + 1] = {0};
  householder_lstsq(A, n_nodes, k, y, b);
  // a_j (x^j - x Li^(j-1)) = b_j (u^j - u)  =>  a_j = b_j / Li^j
  c[0] = f0;
  c[1] = slope;
  for (int j = 2; j <= degree; ++j) {
    double aj = b[j - 2] / std::pow(li, j);
    c[j] = aj;
    c[1] -= aj * std::pow(li, j - 1);
  }
}

// ------------------------------------------------------------------ search

namespace {
struct Cand {
  double score;
  double li, lc;
  uint16_t coef[POLY_MAX_DEGREE + 1];
};
}  // namespace

static bool gates(int fn, int dir, int dtype, int form, int degree, const uint16_t *cb,
                  double lc, const std::vector<uint16_t> &grid, const std::vector<uint16_t> &y) {
  for (uint16_t v : y) {
    double d = to_double(v, dtype);
    if (!std::isfinite(d)) return false;
  }
  if (cb[0] != from_double(residual_at_zero(fn, dir), dtype)) return false;
  double lo, hi;
  if (value_range(fn, dir, &lo, &hi)) {
    for (uint16_t v : y) {
      double d = to_double(v, dtype);
      if (d < lo || d > hi) return false;
    }
  }
  int mono = monotone_on_half(fn, dir);
  if (mono != 0) {
    double cv[POLY_MAX_DEGREE + 1];
    for (int j = 0; j <= degree; ++j) cv[j] = to_double(cb[j], dtype);
    double prev = replay_real(form, cv, degree, lc, to_double(grid[0], dtype));
    for (size_t i = 1; i < grid.size(); ++i) {
      double cur = replay_real(form, cv, degree, lc, to_double(grid[i], dtype));
      if ((cur - prev) * mono < 0) return false;
      prev = cur;
    }
  }
  return true;
}

static double table2_metric(int fn, int dir, int dtype, int form, int degree, const uint16_t *cb,
                            double lc) {
  double cv[POLY_MAX_DEGREE + 1];
  for (int j = 0; j <= degree; ++j) cv[j] = to_double(cb[j], dtype);
  const int n = 20001;
  const double step = (2 * lc) / (n - 1);
  double worst = 0;
  for (int i = 0; i < n; ++i) {
    double x = i == n - 1 ? lc : -lc + i * step;
    double e = std::fabs(replay_real(form, cv, degree, lc, x) - fn_value(fn, dir, x));
    worst = std::max(worst, e);
  }
  return worst;
}

// Differentiated-polynomial backward (§3.3): an odd / centred-odd program
// y = [1/2 +] sign(x) (c_1 t + ... + c_D t^D) has, on |x| < Lc, the even
// derivative c_1 + 2 c_2 t + ... + D c_D t^(D-1); each coefficient is formed
// exactly in FP64 and rounded once.  Same clamp; degree D - 1.
int derive_program(const poly_program &f, poly_program *out) {
  poly_program d;
  std::memset(&d, 0, sizeof(d));
  d.fn = f.fn;
  d.dir = POLY_BWD;
  d.dtype = f.dtype;
  d.form = POLY_FORM_E;
  d.degree = f.degree - 1;
  for (int j = 0; j < f.degree; ++j)
    d.coef[j] = from_double((j + 1) * to_double(f.coef[j + 1], f.dtype), f.dtype);
  d.lc_bits = f.lc_bits;
  d.li = f.li;
  d.lc = f.lc;
  d.search_score = -1;       // not searched: derived from a searched program
  d.deployed_score = -1;
  d.rank = -1;
  d.version = POLY_PROGRAM_VERSION;
  double bound = 0;
  for (uint32_t b = 0; b < 65536; ++b) {
    const uint16_t x = (uint16_t)b;
    const double xv = to_double(x, d.dtype);
    if (!std::isfinite(xv)) continue;
    const uint16_t yy = replay_one(d.form, d.coef, d.degree, d.lc_bits, x, d.dtype, true);
    bound = std::max(bound, std::fabs(to_double(yy, d.dtype) - fn_value(d.fn, POLY_BWD, xv)));
  }
  d.stated_max_abs_err = bound;
  d.table2 = table2_metric(d.fn, POLY_BWD, d.dtype, d.form, d.degree, d.coef, d.lc);
  *out = d;
  return POLY_OK;
}

// Paired sine / cosine programs for RoPE (Appendix B.2: packed FP16 D5 sine
// and D6 cosine sharing the squared input), on the folded half-turn
// coordinate u in [0, 1/2]: sin(pi u) ~ s1 u + s3 u^3 + s5 u^5 and
// cos(pi u) ~ 1 + c2 u^2 + c4 u^4 + c6 u^6, least squares on 2,000 Chebyshev
// nodes with the end value exact (sin = 1, cos = 0 at u = 1/2), the last
// coefficient eliminated through that constraint (the eq. 7-8 construction).
static void constrained_fit3(bool sine, double *coef) {
  const int m = 2000;
  const double xe = 0.5;
  const int p[3] = {sine ? 1 : 2, sine ? 3 : 4, sine ? 5 : 6};
  const double fixed_end = sine ? 0.0 : 1.0, end_value = sine ? 1.0 : 0.0;
  const double r = end_value - fixed_end;
  const double pe = std::pow(xe, p[2]);
  std::vector<double> A((size_t)m * 2), y(m);
  for (int i = 0; i < m; ++i) {
    const double x = 0.5 * xe * (1.0 + std::cos((2.0 * i + 1.0) * M_PI / (2.0 * m)));
    const double f = sine ? std::sin(M_PI * x) : std::cos(M_PI * x) - 1.0;
    const double xl = std::pow(x, p[2]);
    for (int k = 0; k < 2; ++k) A[(size_t)k * m + i] = std::pow(x, p[k]) - xl * (std::pow(xe, p[k]) / pe);
    y[i] = f - xl * (r / pe);
  }
  double a[2];
  householder_lstsq(A, m, 2, y, a);
  coef[0] = a[0];
  coef[1] = a[1];
  coef[2] = (r - a[0] * std::pow(xe, p[0]) - a[1] * std::pow(xe, p[1])) / pe;
}

void fit_sincos(uint16_t *s, uint16_t *c) {
  double sv[3], cv[3];
  constrained_fit3(true, sv);
  constrained_fit3(false, cv);
  for (int j = 0; j < 3; ++j) {
    s[j] = from_double(sv[j], POLY_F16);
    c[j] = from_double(cv[j], POLY_F16);
  }
}

int fit_program(int fn, int dir, int dtype, int degree, const poly_fit_opts &o,
                poly_program *out) {
  const int form = form_of_fn(fn, dir);
  // score grid: linspace(0, hi, n) rounded to the format; duplicates after
  // rounding change neither the maximum nor the monotonicity test
  std::vector<uint16_t> grid;
  {
    const double step = o.score_hi / (o.n_score - 1);
    uint16_t prev = 0xFFFF;
    for (int i = 0; i < o.n_score; ++i) {
      double x = i == o.n_score - 1 ? o.score_hi : i * step;
      uint16_t b = from_double(x, dtype);
      if (b != prev) grid.push_back(b);
      prev = b;
    }
  }
  std::vector<double> truth(grid.size());
  for (size_t i = 0; i < grid.size(); ++i) truth[i] = fn_value(fn, dir, to_double(grid[i], dtype));

  // one task per fit interval Li; tasks are independent and the candidates
  // are merged and sorted afterwards, so the result does not depend on the
  // number of threads
  std::vector<double> lis;
  for (int li_k = 0;; ++li_k) {
    const double li = o.li_min + li_k * o.li_step;
    if (li > o.li_max + 1e-9) break;
    lis.push_back(li);
  }
  std::vector<std::vector<Cand>> per_li(lis.size());
  auto work = [&](size_t first, size_t stride) {
    std::vector<uint16_t> yy(grid.size());
    for (size_t t = first; t < lis.size(); t += stride) {
      const double li = lis[t];
      double c[POLY_MAX_DEGREE + 1];
      fit_coefficients(fn, dir, degree, li, o.n_nodes, c);
      Cand cd{};
      for (int j = 0; j <= degree; ++j) cd.coef[j] = from_double(c[j], dtype);
      cd.li = li;
      for (int lc_k = 0;; ++lc_k) {
        const double lc = o.lc_min + lc_k * o.lc_step;
        if (lc > li + 1.0 + 1e-9) break;                  // Lc <= Li + 1
        const uint16_t lcb = from_double(lc, dtype);
        double worst = 0;
        for (size_t i = 0; i < grid.size(); ++i) {
          yy[i] = replay_one(form, cd.coef, degree, lcb, grid[i], dtype, false);
          worst = std::max(worst, std::fabs(to_double(yy[i], dtype) - truth[i]));
        }
        if (!gates(fn, dir, dtype, form, degree, cd.coef, lc, grid, yy)) continue;
        cd.score = worst;
        cd.lc = lc;
        per_li[t].push_back(cd);
      }
    }
  };
  unsigned nth = std::thread::hardware_concurrency();
  if (nth == 0) nth = 1;
  if (nth > lis.size()) nth = (unsigned)lis.size();
  if (nth <= 1) {
    work(0, 1);
  } else {
    std::vector<std::thread> pool;
    for (unsigned t = 0; t < nth; ++t) pool.emplace_back(work, (size_t)t, (size_t)nth);
    for (auto &th : pool) th.join();
  }
  std::vector<Cand> cands;
  for (auto &v : per_li) cands.insert(cands.end(), v.begin(), v.end());
  if (cands.empty()) return POLY_ENOFIT;
  std::stable_sort(cands.begin(), cands.end(), [](const Cand &a, const Cand &b) {
    if (a.score != b.score) return a.score < b.score;
    if (a.li != b.li) return a.li < b.li;
    return a.lc < b.lc;
  });
  // deployed-order replay of the finalists (all gated candidates when top_k
  // is 0), each clamp also moved by 1..lc_refine_ulps format ulps either way
  const int k = o.top_k > 0 ? std::min<int>(o.top_k, (int)cands.size()) : (int)cands.size();
  std::vector<int> offsets{0};
  for (int j = 1; j <= o.lc_refine_ulps; ++j) {
    offsets.push_back(-j);
    offsets.push_back(j);
  }
  const uint32_t inf_bits = dtype == POLY_F16 ? 0x7C00u : 0x7F80u;
  struct Trial {
    int rank;
    uint16_t lcb;
    double lc, err;
    bool ok;
  };
  std::vector<Trial> trials;
  for (int r = 0; r < k; ++r) {
    const int lcb0 = from_double(cands[r].lc, dtype);
    for (size_t oi = 0; oi < offsets.size(); ++oi) {
      const int b = lcb0 + offsets[oi];
      if (b <= 0 || (uint32_t)b >= inf_bits) continue;
      const double lc = to_double((uint16_t)b, dtype);
      if (!(lc > 0.0 && lc <= cands[r].li + 1.0)) continue;
      trials.push_back(Trial{r, (uint16_t)b, lc, 0.0, false});
    }
  }
  auto deployed = [&](size_t first, size_t stride) {
    std::vector<uint16_t> y(grid.size());
    for (size_t t = first; t < trials.size(); t += stride) {
      Trial &tr = trials[t];
      const Cand &c = cands[tr.rank];
      double worst = 0;
      for (size_t i = 0; i < grid.size(); ++i) {
        y[i] = replay_one(form, c.coef, degree, tr.lcb, grid[i], dtype, true);
        worst = std::max(worst, std::fabs(to_double(y[i], dtype) - truth[i]));
      }
      tr.err = worst;
      tr.ok = gates(fn, dir, dtype, form, degree, c.coef, tr.lc, grid, y);
    }
  };
  unsigned nth2 = std::thread::hardware_concurrency();
  if (nth2 == 0) nth2 = 1;
  if (nth2 > trials.size()) nth2 = (unsigned)trials.size();
  if (nth2 <= 1) {
    deployed(0, 1);
  } else {
    std::vector<std::thread> pool;
    for (unsigned t = 0; t < nth2; ++t) pool.emplace_back(deployed, (size_t)t, (size_t)nth2);
    for (auto &th : pool) th.join();
  }
  // smallest deployed-order error; exact ties go to the smaller Table 2
  // metric (real arithmetic over [-Lc, Lc]), then the smaller Li, then Lc
  int bt = -1;
  for (int t = 0; t < (int)trials.size(); ++t)
    if (trials[t].ok && (bt < 0 || trials[t].err < trials[bt].err)) bt = t;
  if (bt >= 0) {
    std::vector<int> tied;
    for (int t = 0; t < (int)trials.size(); ++t)
      if (trials[t].ok && trials[t].err == trials[bt].err) tied.push_back(t);
    if (tied.size() > 1) {
      double bt2 = 0;
      bt = -1;
      for (int t : tied) {
        const Cand &c = cands[trials[t].rank];
        const double t2 = table2_metric(fn, dir, dtype, form, degree, c.coef, trials[t].lc);
        if (bt < 0 || t2 < bt2 ||
            (t2 == bt2 && (c.li < cands[trials[bt].rank].li ||
                           (c.li == cands[trials[bt].rank].li && trials[t].lc < trials[bt].lc)))) {
          bt = t;
          bt2 = t2;
        }
      }
    }
  }
  const int best = bt < 0 ? -1 : trials[bt].rank;
  const double best_err = bt < 0 ? 0.0 : trials[bt].err;
  if (best < 0) return POLY_ENOFIT;
  const Cand &w = cands[best];
  poly_program p;
  std::memset(&p, 0, sizeof(p));
  p.fn = fn;
  p.dir = dir;
  p.dtype = dtype;
  p.form = form;
  p.degree = degree;
  for (int j = 0; j <= degree; ++j) p.coef[j] = w.coef[j];
  p.lc_bits = trials[bt].lcb;
  p.li = w.li;
  p.lc = trials[bt].lc;
  p.search_score = w.score;
  p.deployed_score = best_err;
  p.rank = best;
  p.version = POLY_PROGRAM_VERSION;
  // stated bound: every finite input, deployed order, against FP64
  double bound = 0;
  for (uint32_t b = 0; b < 65536; ++b) {
    const uint16_t x = (uint16_t)b;
    const double xv = to_double(x, dtype);
    if (!std::isfinite(xv)) continue;
    const uint16_t yy = replay_one(form, p.coef, degree, p.lc_bits, x, dtype, true);
    bound = std::max(bound, std::fabs(to_double(yy, dtype) - fn_value(fn, dir, xv)));
  }
  p.stated_max_abs_err = bound;
  p.table2 = table2_metric(fn, dir, dtype, form, degree, p.coef, p.lc);
  *out = p;
  return POLY_OK;
}

}  // namespace polyact

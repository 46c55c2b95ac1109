// moment_fit.cu -- host-side Chebyshev fits of the Gaussian partial moments
// J_ν(t) = E[(t + Z)_+^ν], Z ~ N(0, 1), that the Gaussian selector needs at an
// entmax order other than α ∈ {1.5, 2} (EntmaxKV, gist.science technical
// summary §2B.2: the normalisation equation F(τ) = Σ_p n_p·E[(Z_p − τ)_+^β] = 1
// and its τ-derivatives, of orders β, β − 1 and β − 2).
//
// Values come from tanh-sinh quadrature of the defining integrals in double:
//   left  (t = −x ≤ 0):  J_ν(−x)/φ(x) = ∫_0^12 y^ν·e^{−y²/2 − xy} dy (fitted
//                        times u^{−(ν+1)}, u = 1/(1 + x/3))
//   right (t ≥ 0):       J_ν(t) = ∫_0^{t+14} y^ν·φ(y − t) dy (fitted as
//                        J_ν(t)/(1 + t)^ν for ν < 1, as its log2 for ν ≥ 1,
//                        where the ratio spans orders of magnitude)
// (past the upper limits the integrands are below e^{−70} of their peak). The
// tanh-sinh rule absorbs the y^ν end point; the mass below its first node,
// ∫_0^{y0} y^ν f(y) dy ≈ f(0)·y0^{ν+1}/(ν+1), is added in closed form. Each fit
// interpolates at the kFitN Chebyshev points and is checked in float against
// fresh quadrature at 200 points per side and on the large-t series; a β whose
// fits miss 1e-6 relative is refused. Fits are cached per β.
#include <cmath>
#include <cstring>
#include <mutex>

#include "common.cuh"

namespace ekv {
namespace {

// ∫_0^Y y^ν f(y) dy by the tanh-sinh rule, y = Y/(1 + e^{−2a}), a = (π/2)·sinh u.
template <class Fn>
double tanh_sinh(const Fn& f, double Y, double nu) {
  const double h = 1.0 / 64.0;
  double sum = 0.0, y0 = Y;
  for (int i = -256; i <= 256; ++i) {
    const double u = i * h;
    const double e = exp(-M_PI * sinh(u));  // e^{−2a}
    const double y = Y / (1.0 + e);
    if (!(y > 0.0) || !(y < Y)) continue;
    const double w = Y * e * M_PI * cosh(u) / ((1.0 + e) * (1.0 + e));  // dy/du
    sum += w * pow(y, nu) * f(y);
    y0 = fmin(y0, y);
  }
  return sum * h + f(0.0) * pow(y0, nu + 1.0) / (nu + 1.0);
}

double j_left_ratio(double x, double nu) {  // J_ν(−x)/φ(x), x ≥ 0
  return tanh_sinh([x](double y) { return exp(-0.5 * y * y - x * y); }, 12.0, nu);
}

double j_right(double t, double nu) {  // J_ν(t), t ≥ 0
  const double c = 1.0 / sqrt(2.0 * M_PI);
  return tanh_sinh([t, c](double y) { return c * exp(-0.5 * (y - t) * (y - t)); }, t + 14.0, nu);
}

double binom(double nu, int n) {  // C(ν, n)
  double r = 1.0;
  for (int i = 0; i < n; ++i) r *= (nu - i) / (i + 1);
  return r;
}

// Chebyshev interpolation of g on [−1, 1] at the kFitN Chebyshev points.
template <class Fn>
void cheb_fit(const Fn& g, float* c) {
  double fv[kFitN];
  for (int j = 0; j < kFitN; ++j) fv[j] = g(cos(M_PI * (j + 0.5) / kFitN));
  for (int k = 0; k < kFitN; ++k) {
    double s = 0.0;
    for (int j = 0; j < kFitN; ++j) s += fv[j] * cos(M_PI * k * (j + 0.5) / kFitN);
    c[k] = (float)(s * (k == 0 ? 1.0 : 2.0) / kFitN);
  }
}

float clenshaw_host(const float* c, float x) {  // the device's float Clenshaw
  const float x2 = 2.0f * x;
  float b1 = 0.0f, b2 = 0.0f;
  for (int k = kFitN - 1; k >= 1; --k) {
    const float b = fmaf(x2, b1, c[k] - b2);
    b2 = b1;
    b1 = b;
  }
  return fmaf(x, b1, c[0] - b2);
}

// The fit of order k (ν = β − k) into F; false when it misses its check.
bool build_order(double beta, int k, MomentFit& F) {
  const double nu = beta - k;
  F.nu[k] = (float)nu;
  // left: w ↦ u = (w + 1.5)/2.5 ↦ x = 3(1/u − 1); fit J_ν(−x)/φ(x)·u^{−(ν+1)}
  auto gl = [nu](double w) {
    const double u = (w + 1.5) / 2.5, x = 3.0 * (1.0 / u - 1.0);
    return j_left_ratio(x, nu) * pow(u, -(nu + 1.0));
  };
  // right: z ↦ t = 8(z + 1); fit J_ν(t)/(1 + t)^ν, or its log2 for ν ≥ 1
  // (there the ratio spans orders of magnitude; for ν near −1 the log has
  // complex singularities close to the axis and the ratio itself is tame)
  const bool lg = nu >= 1.0;
  F.rlog[k] = lg;
  auto gr = [nu, lg](double z) {
    const double t = 8.0 * (z + 1.0);
    return lg ? log2(j_right(t, nu)) - nu * log2(1.0 + t) : j_right(t, nu) * pow(1.0 + t, -nu);
  };
  cheb_fit(gl, F.cl[k]);
  cheb_fit(gr, F.cr[k]);
  double dfact = 1.0;
  for (int m = 1; m <= 5; ++m) {
    dfact *= 2 * m - 1;
    F.ca[k][m - 1] = (float)(binom(nu, 2 * m) * dfact);
  }
  // checks, in the float arithmetic the kernels use for the fitted factors
  for (int i = 0; i <= 200; ++i) {
    const double v = -1.0 + 2.0 * i / 200.0;
    const double rl = gl(v), rr = gr(v);
    if (!(fabs(clenshaw_host(F.cl[k], (float)v) - rl) <= 1e-6 * fabs(rl))) return false;
    const double er = fabs(clenshaw_host(F.cr[k], (float)v) - rr);
    if (!(lg ? er <= 1e-6 / M_LN2 : er <= 1e-6 * fabs(rr))) return false;
  }
  for (double t = 16.0; t <= 64.0; t += 4.0) {
    const double it2 = 1.0 / (t * t);
    double s = 1.0, p = 1.0;
    for (int m = 0; m < 5; ++m) s += F.ca[k][m] * (p *= it2);
    const double ref = j_right(t, nu);
    if (!(fabs(pow(t, nu) * s - ref) <= 1e-6 * fabs(ref))) return false;
  }
  return true;
}

// Orders β and β − 1 must pass. Order β − 2 only feeds the τ̂ solve's Halley
// correction: where it fails (β just above 1, ν near −1, where J_ν is nearly
// singular) the solve takes Newton steps instead, as for β ≤ 1.
bool build(double beta, MomentFit& F) {
  memset(&F, 0, sizeof(F));
  if (!build_order(beta, 0, F) || !build_order(beta, 1, F)) return false;
  F.orders = (beta > 1.0 && build_order(beta, 2, F)) ? 3 : 2;
  return true;
}

struct Entry {
  float beta;
  bool ok;
  unsigned long long used;  // last use (a counter): the least recently used entry is replaced
  MomentFit fit;
};
constexpr int kCacheSlots = 8;
std::mutex g_mu;
Entry g_cache[kCacheSlots];
int g_used = 0;
unsigned long long g_clock = 0;

}  // namespace

// The fits of order β from the cache of the kCacheSlots most recently used
// orders; a miss builds them (0.1-0.4 s of host quadrature) without holding
// the lock, so decodes with cached orders on other threads do not wait, then
// inserts them over the least recently used entry. A caller that cycles
// through more than kCacheSlots orders rebuilds on every miss.
int moment_fit_for(float beta, MomentFit* out) {
  {
    std::lock_guard<std::mutex> lock(g_mu);
    for (int i = 0; i < g_used; ++i)
      if (g_cache[i].beta == beta) {
        g_cache[i].used = ++g_clock;
        if (g_cache[i].ok) *out = g_cache[i].fit;
        return g_cache[i].ok ? 0 : 1;
      }
  }
  Entry e;
  e.beta = beta;
  e.ok = beta > 0.0f && std::isfinite(beta) && build((double)beta, e.fit);
  {
    std::lock_guard<std::mutex> lock(g_mu);
    int slot = -1;
    for (int i = 0; i < g_used; ++i)
      if (g_cache[i].beta == beta) slot = i;  // built meanwhile by another thread
    if (slot < 0 && g_used < kCacheSlots) slot = g_used++;
    if (slot < 0) {
      slot = 0;
      for (int i = 1; i < kCacheSlots; ++i)
        if (g_cache[i].used < g_cache[slot].used) slot = i;
    }
    e.used = ++g_clock;
    g_cache[slot] = e;
  }
  if (e.ok) *out = e.fit;
  return e.ok ? 0 : 1;
}

}  // namespace ekv

// ---------------------------------------------------------------------------
// C ABI: support query and the host evaluation of the fits.

namespace {

float beta_of(float alpha) { return (float)(1.0 / ((double)alpha - 1.0)); }

// The kernels' evaluation (jfit, then 2^E·M), in host float arithmetic.
float jfit_host(const ekv::MomentFit& F, int k, float t) {
  const float nu = F.nu[k];
  float E, M;
  if (t <= 0.0f) {
    const float x = -t, xc = fminf(x, 12.0f);
    const float u = 1.0f / (1.0f + xc * 0.33333334f);
    E = fmaf(-0.72134752f, x * x, (nu + 1.0f) * log2f(u));
    M = 0.3989422804f * ekv::clenshaw_host(F.cl[k], fmaf(2.5f, u, -1.5f));
  } else if (t <= 16.0f) {
    const float c = ekv::clenshaw_host(F.cr[k], fmaf(t, 0.125f, -1.0f));
    const float l2 = log2f(1.0f + t);
    E = F.rlog[k] ? fmaf(nu, l2, c) : nu * l2;
    M = F.rlog[k] ? 1.0f : c;
  } else {
    const float it2 = 1.0f / (t * t);
    M = fmaf(it2, fmaf(it2, fmaf(it2, fmaf(it2, fmaf(it2, F.ca[k][4], F.ca[k][3]), F.ca[k][2]),
                                 F.ca[k][1]), F.ca[k][0]), 1.0f);
    E = nu * log2f(t);
  }
  return M != 0.0f ? exp2f(E) * M : 0.0f;
}

}  // namespace

extern "C" int32_t entmaxkv_gaussian_alpha_supported(float alpha) {
  if (!(alpha > 1.0f) || !std::isfinite(alpha)) return 0;
  if (alpha == 1.5f || alpha == 2.0f) return 1;
  ekv::MomentFit F;
  return ekv::moment_fit_for(beta_of(alpha), &F) == 0 ? 1 : 0;
}

extern "C" int32_t entmaxkv_moment_fit_eval(float alpha, int32_t order, const float* t, int32_t n, float* out) {
  if (n < 0 || (n > 0 && (!t || !out)) || order < 0 || order > 2) return ENTMAXKV_ERR_INVALID_ARG;
  if (!(alpha > 1.0f) || !std::isfinite(alpha)) return ENTMAXKV_ERR_INVALID_ARG;
  if (alpha == 1.5f || alpha == 2.0f) return ENTMAXKV_ERR_UNSUPPORTED;
  ekv::MomentFit F;
  if (ekv::moment_fit_for(beta_of(alpha), &F)) return ENTMAXKV_ERR_UNSUPPORTED;
  if (order >= F.orders) return ENTMAXKV_ERR_INVALID_ARG;
  for (int i = 0; i < n; ++i) out[i] = jfit_host(F, order, t[i]);
  return ENTMAXKV_OK;
}

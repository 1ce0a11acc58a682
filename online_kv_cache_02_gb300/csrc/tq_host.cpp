// Host-side construction of the method's fixed tables: the random rotation
// Pi, the QJL projection S and the Lloyd-Max codebooks (for N(0,1), or for the
// exact density of a rotated coordinate, [P4] §4.2's Beta distribution).
//
// [P4] riverfrot.github.io "TurboQuant란 무엇이며…", §4.1: multiply every KV
// vector by one data-oblivious random orthogonal matrix; §4.2: a Lloyd-Max
// codebook per bit-width, computed once and only looked up at run time;
// §4.3: QJL keeps the signs of a random Gaussian projection of the residual.
//
// Random source (the pages fix none): SplitMix64 (Steele, Lea & Flood 2014)
// in counter form, stream s of seed: out(i) = mix64(seed + s*2^40 +
// (i+1)*0x9E3779B97F4A7C15); uniform = ((out >> 11) + 0.5) * 2^-53;
// Box-Muller on consecutive pairs (cos for the even index, sin for the odd).
// Stream 1 -> the Gaussian matrix G (d x d, row-major), stream 2 -> S.

#include "tq_internal.h"

#include <cmath>
#include <cstring>
#include <vector>

namespace tq {

static inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

static inline double uniform01(uint64_t seed, uint64_t stream, uint64_t i) {
  uint64_t state = seed + (stream << 40) + (i + 1) * 0x9E3779B97F4A7C15ULL;
  return (static_cast<double>(mix64(state) >> 11) + 0.5) * 0x1.0p-53;
}

void gaussian_fill(uint64_t seed, uint64_t stream, size_t n, double* out) {
  const double two_pi = 6.283185307179586476925286766559;
  for (size_t j = 0; 2 * j < n; ++j) {
    double u1 = uniform01(seed, stream, 2 * j);
    double u2 = uniform01(seed, stream, 2 * j + 1);
    double r = std::sqrt(-2.0 * std::log(u1));
    double t = two_pi * u2;
    out[2 * j] = r * std::cos(t);
    if (2 * j + 1 < n) out[2 * j + 1] = r * std::sin(t);
  }
}

// Pi = Q diag(sign(R_kk)) for G = QR by Householder reflections; equivalently
// the orthogonal factor whose R has a positive diagonal (unique for full-rank G).
void rotation_fill(int d, uint64_t seed, double* pi) {
  std::vector<double> a(static_cast<size_t>(d) * d);
  gaussian_fill(seed, 1, a.size(), a.data());
  std::vector<double> vs(static_cast<size_t>(d) * d, 0.0);  // reflector k in row k (entries k..d-1)
  std::vector<double> rdiag(d);
  for (int k = 0; k < d; ++k) {
    double nrm2 = 0.0;
    for (int i = k; i < d; ++i) nrm2 += a[i * d + k] * a[i * d + k];
    double nrm = std::sqrt(nrm2);
    double x0 = a[k * d + k];
    double alpha = (x0 >= 0.0) ? -nrm : nrm;         // reflect onto -sign(x0) e_k
    double* v = &vs[static_cast<size_t>(k) * d];
    for (int i = k; i < d; ++i) v[i] = a[i * d + k];
    v[k] -= alpha;
    double vn2 = 0.0;
    for (int i = k; i < d; ++i) vn2 += v[i] * v[i];
    rdiag[k] = alpha;
    if (vn2 == 0.0) continue;                         // column already reduced
    double vn = std::sqrt(vn2);
    for (int i = k; i < d; ++i) v[i] /= vn;
    for (int j = k; j < d; ++j) {                     // A <- (I - 2 v v^T) A
      double dot = 0.0;
      for (int i = k; i < d; ++i) dot += v[i] * a[i * d + j];
      for (int i = k; i < d; ++i) a[i * d + j] -= 2.0 * v[i] * dot;
    }
  }
  // Q = H_0 H_1 ... H_{d-1}: apply the reflectors to I from the last one.
  std::vector<double> q(static_cast<size_t>(d) * d, 0.0);
  for (int i = 0; i < d; ++i) q[i * d + i] = 1.0;
  for (int k = d - 1; k >= 0; --k) {
    const double* v = &vs[static_cast<size_t>(k) * d];
    for (int j = 0; j < d; ++j) {
      double dot = 0.0;
      for (int i = k; i < d; ++i) dot += v[i] * q[i * d + j];
      for (int i = k; i < d; ++i) q[i * d + j] -= 2.0 * v[i] * dot;
    }
  }
  for (int i = 0; i < d; ++i)
    for (int j = 0; j < d; ++j) pi[i * d + j] = q[i * d + j] * (rdiag[j] < 0.0 ? -1.0 : 1.0);
}

void qjl_fill(int m, int d, uint64_t seed, double* s) {
  gaussian_fill(seed, 2, static_cast<size_t>(m) * d, s);
}

// Lloyd-Max for N(0,1) with 2^bits levels.  The density is symmetric, so the
// positive half is iterated (cells [t_k, t_{k+1}), t_0 = 0, last cell open)
// and mirrored.  Centroid of a cell = conditional mean
// (phi(lo) - phi(hi)) / (Q(lo) - Q(hi)), Q the upper tail; boundary =
// midpoint of neighbouring centroids.  Stops when no centroid moves by more
// than 1e-15 (or after 200000 sweeps).
void codebook_fill(int bits, double* centroids, double* boundaries) {
  const int h = 1 << (bits - 1);
  const double inv_sqrt2 = 0.70710678118654752440084436210485;
  const double inv_sqrt2pi = 0.39894228040143267793994605993438;
  std::vector<double> a(h), lo(h), nx(h);
  for (int k = 0; k < h; ++k) a[k] = (k + 0.5) * 3.0 / h;
  for (int it = 0; it < 200000; ++it) {
    lo[0] = 0.0;
    for (int k = 1; k < h; ++k) lo[k] = 0.5 * (a[k - 1] + a[k]);
    double delta = 0.0;
    for (int k = 0; k < h; ++k) {
      double l = lo[k];
      bool open = (k == h - 1);
      double hi = open ? 0.0 : lo[k + 1];
      double num = std::exp(-0.5 * l * l) - (open ? 0.0 : std::exp(-0.5 * hi * hi));
      double den = 0.5 * (std::erfc(l * inv_sqrt2) - (open ? 0.0 : std::erfc(hi * inv_sqrt2)));
      nx[k] = num * inv_sqrt2pi / den;
      delta = std::fmax(delta, std::fabs(nx[k] - a[k]));
    }
    a.swap(nx);
    if (delta <= 1e-15) break;
  }
  for (int k = 0; k < h; ++k) {
    centroids[h + k] = a[k];
    centroids[h - 1 - k] = -a[k];
  }
  boundaries[h - 1] = 0.0;
  for (int k = 1; k < h; ++k) {
    double t = 0.5 * (a[k - 1] + a[k]);
    boundaries[h - 1 + k] = t;
    boundaries[h - 1 - k] = -t;
  }
}

// Regularized incomplete beta I_x(a, b): the continued fraction of
// Abramowitz & Stegun 26.5.8 evaluated by the modified Lentz method, used
// directly below x = (a+1)/(a+b+2) and through I_x(a,b) = 1 - I_{1-x}(b,a)
// above it (where the fraction converges fast).
static double beta_cf(double a, double b, double x) {
  const double tiny = 1e-300;
  double c = 1.0, dd = 1.0 - (a + b) * x / (a + 1.0);
  if (std::fabs(dd) < tiny) dd = tiny;
  dd = 1.0 / dd;
  double f = dd;
  for (int m = 1; m <= 100000; ++m) {
    const double m2 = 2.0 * m;
    double num = m * (b - m) * x / ((a + m2 - 1.0) * (a + m2));      // d_{2m}
    dd = 1.0 + num * dd;
    if (std::fabs(dd) < tiny) dd = tiny;
    dd = 1.0 / dd;
    c = 1.0 + num / c;
    if (std::fabs(c) < tiny) c = tiny;
    f *= dd * c;
    num = -(a + m) * (a + b + m) * x / ((a + m2) * (a + m2 + 1.0));   // d_{2m+1}
    dd = 1.0 + num * dd;
    if (std::fabs(dd) < tiny) dd = tiny;
    dd = 1.0 / dd;
    c = 1.0 + num / c;
    if (std::fabs(c) < tiny) c = tiny;
    const double del = dd * c;
    f *= del;
    if (std::fabs(del - 1.0) < 4e-16) break;             // a couple of ulps of 1
  }
  return f;
}
static double reg_inc_beta(double a, double b, double x) {
  if (x <= 0.0) return 0.0;
  if (x >= 1.0) return 1.0;
  const double front =
      std::exp(std::lgamma(a + b) - std::lgamma(a) - std::lgamma(b) + a * std::log(x) + b * std::log1p(-x));
  if (x < (a + 1.0) / (a + b + 2.0)) return front * beta_cf(a, b, x) / a;
  return 1.0 - front * beta_cf(b, a, 1.0 - x) / b;
}

// Lloyd-Max for the density of u = sqrt(d) x_1, x uniform on the unit sphere
// of R^d (the coordinate of a randomly rotated vector in unit-variance units):
// f(u) proportional to (1 - u^2/d)^((d-3)/2) on |u| < sqrt(d).  Same sweep as
// the Gaussian case on the positive half: with z = u/sqrt(d), the upper tail
// P(Z >= z) = I_{1-z^2}((d-1)/2, 1/2) / 2 and the partial first moment
// E[Z; Z >= z] = C (1 - z^2)^((d-1)/2) / (d-1), C = Gamma(d/2) /
// (sqrt(pi) Gamma((d-1)/2)), so a cell's conditional mean is closed form.
void codebook_fill_sphere(int bits, int d, double* centroids, double* boundaries) {
  const int h = 1 << (bits - 1);
  const double rd = std::sqrt(static_cast<double>(d));
  const double ca = 0.5 * (d - 1), cb = 0.5;
  const double cmom = std::exp(std::lgamma(0.5 * d) - std::lgamma(0.5 * (d - 1))) / std::sqrt(M_PI) / (d - 1);
  auto tail = [&](double u) {                 // P(U >= u), u >= 0
    const double z = u / rd;
    return z >= 1.0 ? 0.0 : 0.5 * reg_inc_beta(ca, cb, 1.0 - z * z);
  };
  auto moment = [&](double u) {               // E[Z; Z >= z], z = u/sqrt(d) (times sqrt(d): E[U; U >= u])
    const double z = u / rd;
    return z >= 1.0 ? 0.0 : cmom * std::pow(1.0 - z * z, 0.5 * (d - 1));
  };
  std::vector<double> a(h), lo(h), nx(h);
  // start inside (0, sqrt(d)): a centroid at or beyond the support's end
  // would leave its cell empty (0/0)
  for (int k = 0; k < h; ++k) a[k] = (k + 0.5) * std::fmin(3.0, rd) / h;
  for (int it = 0; it < 200000; ++it) {
    lo[0] = 0.0;
    for (int k = 1; k < h; ++k) lo[k] = 0.5 * (a[k - 1] + a[k]);
    double delta = 0.0;
    for (int k = 0; k < h; ++k) {
      const bool open = (k == h - 1);
      const double l = lo[k], hi = open ? rd : lo[k + 1];
      const double num = rd * (moment(l) - (open ? 0.0 : moment(hi)));
      const double den = tail(l) - (open ? 0.0 : tail(hi));
      nx[k] = num / den;
      delta = std::fmax(delta, std::fabs(nx[k] - a[k]));
    }
    a.swap(nx);
    // the incomplete beta's rounding (about 1e-13 near its slow region) keeps
    // the sweep from settling below ~1e-12 at 4 bits: accept that after 2000
    if (delta <= 4e-15 || (it >= 2000 && delta < 1e-12)) break;
  }
  for (int k = 0; k < h; ++k) {
    centroids[h + k] = a[k];
    centroids[h - 1 - k] = -a[k];
  }
  boundaries[h - 1] = 0.0;
  for (int k = 1; k < h; ++k) {
    const double t = 0.5 * (a[k - 1] + a[k]);
    boundaries[h - 1 + k] = t;
    boundaries[h - 1 - k] = -t;
  }
}

}  // namespace tq

extern "C" tq_status tq_host_rotation(int d, uint64_t seed, double* pi) {
  if (!pi || d < 2 || d > 4096) return TQ_ERR_INVALID_ARG;
  tq::rotation_fill(d, seed, pi);
  return TQ_OK;
}

extern "C" tq_status tq_host_qjl(int m, int d, uint64_t seed, double* s) {
  if (!s || m < 1 || d < 1) return TQ_ERR_INVALID_ARG;
  tq::qjl_fill(m, d, seed, s);
  return TQ_OK;
}

extern "C" tq_status tq_host_codebook(int bits, double* centroids, double* boundaries) {
  if (!centroids || !boundaries || bits < 1 || bits > 8) return TQ_ERR_INVALID_ARG;
  tq::codebook_fill(bits, centroids, boundaries);
  return TQ_OK;
}

extern "C" tq_status tq_host_codebook_ex(int bits, int d, int density, double* centroids, double* boundaries) {
  if (!centroids || !boundaries || bits < 1 || bits > 8) return TQ_ERR_INVALID_ARG;
  if (density == TQ_CODEBOOK_GAUSSIAN) {
    tq::codebook_fill(bits, centroids, boundaries);
    return TQ_OK;
  }
  if (density != TQ_CODEBOOK_SPHERE || d < 4) return TQ_ERR_INVALID_ARG;
  tq::codebook_fill_sphere(bits, d, centroids, boundaries);
  return TQ_OK;
}

// Host-side construction of the method's fixed tables: the random rotation
// Pi, the QJL projection S and the Gaussian Lloyd-Max codebooks.
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

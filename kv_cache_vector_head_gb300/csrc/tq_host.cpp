// Host-side setup of the TurboQuant hot path: the Lloyd-Max codebook and the
// seeded random transforms.  Plain C++17, double precision, runs once per
// layer at initialisation.
//
// Codebook ([Reconstruction] §5 Steps 2-4): Lloyd-Max on the density of one
// coordinate of a uniformly rotated unit vector in R^d,
//     f(x) = C_d (1 - x^2)^e,  e = (d - 3) / 2,  C_d = G(d/2) / (sqrt(pi) G((d-1)/2)).
// The cell mass uses J_e(b) = int_0^b (1 - x^2)^e dx, evaluated by the
// integration-by-parts recurrence
//     J_e(b) = ( b (1 - b^2)^e + 2 e J_{e-1}(b) ) / (2 e + 1),
// started from J_0(b) = b (odd d) or J_{-1/2}(b) = asin(b) (even d); the
// coefficient 2e / (2e + 1) < 1 keeps the upward recurrence stable.  The first
// moment has the closed form int_a^b x f = C_d / (2 (e + 1)) ((1-a^2)^(e+1) -
// (1-b^2)^(e+1)).
//
// Transforms ([Reconstruction] §5 Step 2, §6, §9, §13; [Design study]
// §Dense and structured transform comparison): SplitMix64 (Steele, Lea,
// Flood 2014), Box-Muller normals, Householder QR with the column signs of Q
// fixed by sign(R_jj) so the rotation is Haar distributed.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

#include "tq_internal.h"

namespace tq {
namespace {

// ---------------------------------------------------------------- codebook
struct SphereMarginal {
  int d;
  double e;      // (d - 3) / 2
  double cd;     // density constant
  explicit SphereMarginal(int d_) : d(d_), e((d_ - 3) / 2.0) {
    cd = std::exp(std::lgamma(d_ / 2.0) - 0.5 * std::log(M_PI) - std::lgamma((d_ - 1) / 2.0));
  }
  // J_e(b) by the upward recurrence.
  double J(double b) const {
    const double s = 1.0 - b * b;
    double ee, val;
    if ((d & 1) == 1) {  // e integer: start at e = 0
      ee = 0.0;
      val = b;
    } else {             // e half-integer: start at e = -1/2
      ee = -0.5;
      val = std::asin(b);
    }
    while (ee < e - 0.25) {
      ee += 1.0;
      val = (b * std::pow(s, ee) + 2.0 * ee * val) / (2.0 * ee + 1.0);
    }
    return val;
  }
  double mass(double a, double b) const { return cd * (J(b) - J(a)); }
  double first_moment(double a, double b) const {
    const double p = e + 1.0;
    return cd / (2.0 * p) * (std::pow(1.0 - a * a, p) - std::pow(1.0 - b * b, p));
  }
};

// ---------------------------------------------------------------- generator
struct SplitMix64 {
  uint64_t s;
  explicit SplitMix64(uint64_t st) : s(st) {}
  static uint64_t mix(uint64_t z) {
    z += 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
  }
  uint64_t next() {
    s += 0x9E3779B97F4A7C15ull;
    uint64_t z = s;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
  }
  double uniform() { return (double)(next() >> 11) * 0x1.0p-53; }
};

uint64_t stream_state(uint64_t seed, int layer, int head, int role) {
  const uint64_t key = ((uint64_t)layer << 24) | ((uint64_t)head << 8) | (uint64_t)role;
  return seed ^ SplitMix64::mix(key);
}

void gaussian_fill(SplitMix64& g, double* out, size_t n) {
  for (size_t i = 0; i < n; i += 2) {
    const double u1 = g.uniform(), u2 = g.uniform();
    const double r = std::sqrt(-2.0 * std::log(1.0 - u1));
    out[i] = r * std::cos(2.0 * M_PI * u2);
    if (i + 1 < n) out[i + 1] = r * std::sin(2.0 * M_PI * u2);
  }
}

// Haar rotation: Householder QR of A (row-major d x d, destroyed); writes
// Q diag(sign(R_jj)) row-major into q.
void haar_from_gaussian(int d, std::vector<double>& A, std::vector<double>& q) {
  std::vector<std::vector<double>> vs;
  std::vector<double> rdiag(d);
  vs.reserve(d);
  for (int k = 0; k < d; ++k) {
    const int m = d - k;
    std::vector<double> v(m);
    double nrm2 = 0;
    for (int i = 0; i < m; ++i) {
      v[i] = A[(size_t)(k + i) * d + k];
      nrm2 += v[i] * v[i];
    }
    const double nrm = std::sqrt(nrm2);
    if (k == d - 1 || nrm == 0.0) {
      rdiag[k] = v[0];
      vs.emplace_back();  // identity reflector
      continue;
    }
    const double alpha = v[0] >= 0 ? -nrm : nrm;  // R_kk
    rdiag[k] = alpha;
    v[0] -= alpha;
    double vn2 = 0;
    for (int i = 0; i < m; ++i) vn2 += v[i] * v[i];
    const double vn = std::sqrt(vn2);
    for (int i = 0; i < m; ++i) v[i] /= vn;
    // A[k:, k:] -= 2 v (v^T A[k:, k:])
    for (int j = k; j < d; ++j) {
      double dot = 0;
      for (int i = 0; i < m; ++i) dot += v[i] * A[(size_t)(k + i) * d + j];
      for (int i = 0; i < m; ++i) A[(size_t)(k + i) * d + j] -= 2.0 * v[i] * dot;
    }
    vs.push_back(std::move(v));
  }
  // Q = H_0 H_1 ... H_{d-1}: apply the reflectors in reverse to the identity.
  q.assign((size_t)d * d, 0.0);
  for (int i = 0; i < d; ++i) q[(size_t)i * d + i] = 1.0;
  for (int k = d - 1; k >= 0; --k) {
    const std::vector<double>& v = vs[k];
    if (v.empty()) continue;
    const int m = d - k;
    for (int j = 0; j < d; ++j) {
      double dot = 0;
      for (int i = 0; i < m; ++i) dot += v[i] * q[(size_t)(k + i) * d + j];
      for (int i = 0; i < m; ++i) q[(size_t)(k + i) * d + j] -= 2.0 * v[i] * dot;
    }
  }
  for (int j = 0; j < d; ++j) {
    if (rdiag[j] < 0) {
      for (int i = 0; i < d; ++i) q[(size_t)i * d + j] = -q[(size_t)i * d + j];
    }
  }
}

}  // namespace
}  // namespace tq

extern "C" tq_status tq_build_codebook(int d, int bits, float* centroids, float* boundaries,
                                       double* mse_unit) {
  using namespace tq;
  if (d < 4 || d > 4096) return fail(TQ_ERR_INVALID_ARG, "tq_build_codebook: d must be in [4, 4096]");
  if (bits < 1 || bits > TQ_MAX_BITS) return fail(TQ_ERR_UNSUPPORTED, "tq_build_codebook: bits must be 1..4");
  if (!centroids || !boundaries) return fail(TQ_ERR_INVALID_ARG, "tq_build_codebook: null output");
  const SphereMarginal f(d);
  const int half = 1 << (bits - 1);
  const double sd = std::sqrt((double)d);
  std::vector<double> mu(half), edges(half + 1), nw(half);
  // any increasing start inside (0, 1) converges; spread it over ~3 sigma
  for (int k = 0; k < half; ++k) mu[k] = std::fmin(0.9, 3.0 * (k + 0.5) / half / sd);
  bool converged = false;
  for (int it = 0; it < 100000; ++it) {
    edges[0] = 0.0;
    edges[half] = 1.0;
    for (int k = 1; k < half; ++k) edges[k] = 0.5 * (mu[k - 1] + mu[k]);
    double delta = 0;
    for (int k = 0; k < half; ++k) {
      nw[k] = f.first_moment(edges[k], edges[k + 1]) / f.mass(edges[k], edges[k + 1]);
      delta = std::fmax(delta, std::fabs(nw[k] - mu[k]) * sd);
    }
    mu = nw;
    if (delta < 1e-13) {
      converged = true;
      break;
    }
  }
  if (!converged) return fail(TQ_ERR_NO_CONVERGENCE, "tq_build_codebook: Lloyd-Max did not converge");
  for (int k = 1; k < half; ++k) edges[k] = 0.5 * (mu[k - 1] + mu[k]);
  const int L = 2 * half;
  for (int k = 0; k < half; ++k) {
    const float c = (float)(mu[k] * sd);
    centroids[half + k] = c;
    centroids[half - 1 - k] = -c;
  }
  for (int j = 0; j + 1 < L; ++j) boundaries[j] = (centroids[j] + centroids[j + 1]) * 0.5f;
  if (mse_unit) {
    double s = 0;
    for (int k = 0; k < half; ++k) s += f.mass(edges[k], edges[k + 1]) * mu[k] * mu[k];
    *mse_unit = 1.0 - d * 2.0 * s;
  }
  return ok();
}

extern "C" tq_status tq_build_transform(tq_transform_kind kind, int d, uint64_t seed, int layer, int head,
                                        int role, float* out) {
  using namespace tq;
  if (!out) return fail(TQ_ERR_INVALID_ARG, "tq_build_transform: null output");
  if (d < 2 || d > 4096) return fail(TQ_ERR_INVALID_ARG, "tq_build_transform: d must be in [2, 4096]");
  if (layer < 0 || layer >= (1 << 20) || head < 0 || head >= (1 << 16) || role < 0 || role > 3)
    return fail(TQ_ERR_INVALID_ARG, "tq_build_transform: layer/head/role out of range");
  if (kind != TQ_DENSE && kind != TQ_FWHT) return fail(TQ_ERR_INVALID_ARG, "tq_build_transform: bad kind");
  if (kind == TQ_FWHT && (d & (d - 1)))
    return fail(TQ_ERR_UNSUPPORTED, "tq_build_transform: FWHT needs a power-of-two d");
  SplitMix64 g(stream_state(seed, layer, head, role));
  if (role == TQ_ROLE_QJL) {
    std::vector<double> s((size_t)d * d);
    gaussian_fill(g, s.data(), s.size());
    for (size_t i = 0; i < s.size(); ++i) out[i] = (float)s[i];
    return ok();
  }
  if (kind == TQ_FWHT || role == TQ_ROLE_QJL_SIGNS) {
    if (d & (d - 1)) return fail(TQ_ERR_UNSUPPORTED, "tq_build_transform: sign vectors need a power-of-two d");
    for (int i = 0; i < d; ++i) out[i] = (g.next() & 1ull) ? -1.0f : 1.0f;
    return ok();
  }
  std::vector<double> a((size_t)d * d), q;
  gaussian_fill(g, a.data(), a.size());
  haar_from_gaussian(d, a, q);
  for (size_t i = 0; i < q.size(); ++i) out[i] = (float)q[i];
  return ok();
}

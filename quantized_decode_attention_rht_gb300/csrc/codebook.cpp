// Host-side codebooks for the rotated unit-norm coordinates (computed once at start-up).
//
// VeloxQuant-MLX page ("I Ported a Google Research Paper to Apple Silicon"), section
// "Stage 2: Lloyd-Max Scalar Quantization": the Lloyd-Max quantiser of N(0,1) alternates
// two conditions -- boundaries at centroid midpoints, centroids at the conditional mean of
// the density over their cell -- until it settles, and the tables are reused for every
// token.  Here the conditional mean is evaluated in closed form,
//   E[X | a < X < b] = (phi(a) - phi(b)) / (Phi(b) - Phi(a)),
// with the outer cells ending at +-8, and the iteration runs until the centroids move by
// less than 1e-15.  The uniform codebook takes the symmetric step that minimises the
// N(0,1) mean squared error (the fixed point of its stationarity condition).
#include <cmath>
#include <vector>

#include "../../include/kvq.h"

namespace {

constexpr double kSupport = 8.0;
constexpr double kInvSqrt2 = 0.70710678118654752440;
constexpr double kInvSqrt2Pi = 0.39894228040143267794;

double pdf(double x) { return kInvSqrt2Pi * std::exp(-0.5 * x * x); }

// Probability mass of N(0,1) on [a, b], written so that tails keep their precision.
double mass(double a, double b) {
  if (a >= 0.0) return 0.5 * (std::erfc(a * kInvSqrt2) - std::erfc(b * kInvSqrt2));
  if (b <= 0.0) return 0.5 * (std::erfc(-b * kInvSqrt2) - std::erfc(-a * kInvSqrt2));
  return 1.0 - 0.5 * std::erfc(b * kInvSqrt2) - 0.5 * std::erfc(-a * kInvSqrt2);
}

}  // namespace

extern "C" KVQ_API kvq_status kvq_lloyd_max_codebook(int32_t bits, double* centroids,
                                                     double* bounds) {
  if (bits < 1 || bits > 6) return KVQ_ERR_UNSUPPORTED;
  if (!centroids || !bounds) return KVQ_ERR_INVALID_ARGUMENT;
  const int n = 1 << bits;
  std::vector<double> c(n), e(n + 1);
  for (int i = 0; i < n; ++i) c[i] = -kSupport + 2.0 * kSupport * i / (n - 1);
  for (int it = 0; it < 2000000; ++it) {
    e[0] = -kSupport;
    e[n] = kSupport;
    for (int i = 1; i < n; ++i) e[i] = 0.5 * (c[i - 1] + c[i]);
    double moved = 0.0;
    for (int i = 0; i < n; ++i) {
      const double nc = (pdf(e[i]) - pdf(e[i + 1])) / mass(e[i], e[i + 1]);
      moved = std::fmax(moved, std::fabs(nc - c[i]));
      c[i] = nc;
    }
    if (moved < 1e-15) break;
  }
  // The fixed point of a symmetric start is symmetric; remove rounding asymmetry.
  for (int i = 0; i < n / 2; ++i) {
    const double m = 0.5 * (c[n - 1 - i] - c[i]);
    c[i] = -m;
    c[n - 1 - i] = m;
  }
  for (int i = 0; i < n; ++i) centroids[i] = c[i];
  for (int i = 0; i + 1 < n; ++i) bounds[i] = 0.5 * (c[i] + c[i + 1]);
  return KVQ_OK;
}

extern "C" KVQ_API kvq_status kvq_uniform_codebook(int32_t bits, double* centroids,
                                                   double* bounds) {
  if (bits < 1 || bits > 8) return KVQ_ERR_UNSUPPORTED;
  if (!centroids || !bounds) return KVQ_ERR_INVALID_ARGUMENT;
  const int n = 1 << bits;
  // Stationarity of the MSE in the step delta (the boundary terms cancel at midpoints):
  //   sum_i k_i [phi(a_i) - phi(b_i)] = delta * sum_i k_i^2 [Phi(b_i) - Phi(a_i)],
  // with level k_i * delta on cell [a_i, b_i]; iterated as a fixed point in delta.
  double delta = 1.0;
  for (int it = 0; it < 1000000; ++it) {
    double num = 0.0, den = 0.0;
    for (int i = 0; i < n; ++i) {
      const double k = i - 0.5 * (n - 1);
      const double a = i == 0 ? -INFINITY : (k - 0.5) * delta;
      const double b = i == n - 1 ? INFINITY : (k + 0.5) * delta;
      num += k * ((std::isfinite(a) ? pdf(a) : 0.0) - (std::isfinite(b) ? pdf(b) : 0.0));
      den += k * k * mass(a, b);
    }
    const double next = num / den;
    const bool done = std::fabs(next - delta) <= 4e-16 * next;
    delta = next;
    if (done) break;
  }
  for (int i = 0; i < n; ++i) centroids[i] = (i - 0.5 * (n - 1)) * delta;
  for (int i = 0; i + 1 < n; ++i) bounds[i] = 0.5 * (centroids[i] + centroids[i + 1]);
  return KVQ_OK;
}

extern "C" KVQ_API kvq_status kvq_codebook_tables(int32_t bits, const double* centroids,
                                                  float* centroids32, float* bounds32) {
  if (bits < 1 || bits > 8) return KVQ_ERR_UNSUPPORTED;
  if (!centroids || !centroids32 || !bounds32) return KVQ_ERR_INVALID_ARGUMENT;
  const int n = 1 << bits;
  for (int i = 0; i < n; ++i) centroids32[i] = static_cast<float>(centroids[i]);
  for (int i = 0; i + 1 < n; ++i) {
    if (!(centroids32[i] < centroids32[i + 1])) return KVQ_ERR_INVALID_ARGUMENT;
    bounds32[i] = static_cast<float>(
        (static_cast<double>(centroids32[i]) + static_cast<double>(centroids32[i + 1])) * 0.5);
  }
  return KVQ_OK;
}

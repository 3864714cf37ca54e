// Host-built tables of the library: the RoPE cos/sin table, the TurboQuant
// sign diagonal and the Beta(a, a) Lloyd-Max codebooks.
#include <cmath>
#include <cstdint>
#include <vector>

#include "kvq_internal.h"

namespace kvq {

// Vanilla RoPE (posttrainllm "StreamingLLM + KIVI", section "RoPE caveat"):
// half-split pairs (i, i + D/2), theta_i = base^(-2i/D), angle = pos theta_i,
// cos/sin evaluated in double and rounded once to float.
void build_rope_table(float* out, int64_t max_pos, int D, double base) {
  const int half = D / 2;
  for (int i = 0; i < half; ++i) {
    const double inv = std::pow(base, -(2.0 * i) / D);
    for (int64_t p = 0; p < max_pos; ++p) {
      const double ang = static_cast<double>(p) * inv;
      out[(p * half + i) * 2 + 0] = static_cast<float>(std::cos(ang));
      out[(p * half + i) * 2 + 1] = static_cast<float>(std::sin(ang));
    }
  }
}

// SplitMix64 (Vigna): state += golden gamma, then two xor-shift-multiply
// rounds and a final xor-shift. Sign j is -1 when output j has its top bit set
// (Foundry "TurboQuant" spec, "Step 1": a diagonal of random +-1 signs
// generated from the seed).
void build_signs(float* out, int D, uint64_t seed) {
  uint64_t state = seed;
  for (int j = 0; j < D; ++j) {
    state += 0x9E3779B97F4A7C15ull;
    uint64_t z = state;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    z ^= z >> 31;
    out[j] = (z >> 63) ? -1.0f : 1.0f;
  }
}

namespace {

// Nodes and weights of n-point Gauss-Legendre quadrature on [-1, 1]: roots
// of P_n by Newton's method from the Chebyshev-like start, P_n and P_n'
// from the three-term recurrence.
void gauss_legendre(int n, std::vector<double>* x, std::vector<double>* w) {
  x->assign(n, 0.0);
  w->assign(n, 0.0);
  const double pi = 3.14159265358979323846;
  for (int i = 0; i < (n + 1) / 2; ++i) {
    double z = std::cos(pi * (i + 0.75) / (n + 0.5));
    double dp = 1.0;
    for (int it = 0; it < 100; ++it) {
      double p0 = 1.0, p1 = z;
      for (int k = 2; k <= n; ++k) {
        const double p2 = ((2.0 * k - 1.0) * z * p1 - (k - 1.0) * p0) / k;
        p0 = p1;
        p1 = p2;
      }
      dp = n * (z * p1 - p0) / (z * z - 1.0);
      const double dz = p1 / dp;
      z -= dz;
      if (std::fabs(dz) < 1e-16) break;
    }
    (*x)[i] = -z;
    (*x)[n - 1 - i] = z;
    (*w)[i] = (*w)[n - 1 - i] = 2.0 / ((1.0 - z * z) * dp * dp);
  }
}

struct BetaCells {
  double a, log_peak;
  std::vector<double> gx, gw;
  static constexpr int kPanels = 16;

  // Unnormalised Beta(a, a) density scaled to 1 at x = 1/2.
  double density(double x) const {
    if (x <= 0.0 || x >= 1.0) return 0.0;
    return std::exp((a - 1.0) * (std::log(x) + std::log1p(-x)) - log_peak);
  }
  // Integrals of f and x f over [lo, hi] by composite Gauss-Legendre.
  void moments(double lo, double hi, double* m0, double* m1) const {
    double s0 = 0.0, s1 = 0.0;
    const double h = (hi - lo) / kPanels;
    for (int p = 0; p < kPanels; ++p) {
      const double c = lo + (p + 0.5) * h, r = 0.5 * h;
      for (size_t i = 0; i < gx.size(); ++i) {
        const double xx = c + r * gx[i];
        const double f = density(xx) * gw[i] * r;
        s0 += f;
        s1 += f * xx;
      }
    }
    *m0 = s0;
    *m1 = s1;
  }
};

}  // namespace

// Lloyd-Max for Beta(a, a) (Foundry "TurboQuant" spec, "Codebook
// Generation"): uniform boundaries on [0, 1] to start; centroid of each cell
// = its conditional mean; boundaries = midpoints of adjacent centroids;
// repeated until no boundary moves by more than 1e-14. An empty cell keeps its
// midpoint as centroid.
void build_beta_codebook(double a, int bits, double* boundaries, double* centroids) {
  const int L = 1 << bits;
  BetaCells bc;
  bc.a = a;
  bc.log_peak = (a - 1.0) * 2.0 * std::log(0.5);
  gauss_legendre(32, &bc.gx, &bc.gw);
  std::vector<double> b(L + 1), c(L);
  for (int i = 0; i <= L; ++i) b[i] = static_cast<double>(i) / L;
  auto centroids_of = [&](void) {
    for (int i = 0; i < L; ++i) {
      double m0, m1;
      bc.moments(b[i], b[i + 1], &m0, &m1);
      c[i] = (m0 > 0.0) ? m1 / m0 : 0.5 * (b[i] + b[i + 1]);
    }
  };
  centroids_of();
  for (int it = 0; it < 200000; ++it) {
    double moved = 0.0;
    for (int i = 1; i < L; ++i) {
      const double nb = 0.5 * (c[i - 1] + c[i]);
      moved = std::fmax(moved, std::fabs(nb - b[i]));
      b[i] = nb;
    }
    centroids_of();
    if (moved < 1e-14) break;
  }
  for (int i = 0; i < L - 1; ++i) boundaries[i] = b[i + 1];
  for (int i = 0; i < L; ++i) centroids[i] = c[i];
}

}  // namespace kvq

// Host-side setup of libturboquant: random rotation, Lloyd-Max codebook and
// QJL matrix, all in float64.  Runs once per shape and is not on the hot path
// (the yeyulingfeng article: the codebook is computed once and reused for any
// model, with no calibration data).
//
// Random numbers: SplitMix64 (Steele, Lea & Flood 2014) in counter form,
// output i of stream `seed` = mix64(seed + (i+1)·0x9E3779B97F4A7C15);
// uniforms ((z >> 11) + 0.5)·2^-53; Box-Muller pairs (sqrt(-2 ln u1)·cos 2πu2,
// sqrt(-2 ln u1)·sin 2πu2) filled in order.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

#include "../../include/turboquant.h"

namespace {

constexpr uint64_t kGolden = 0x9E3779B97F4A7C15ull;

inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

inline double uniform01(uint64_t seed, uint64_t i) {
  return (static_cast<double>(mix64(seed + (i + 1) * kGolden) >> 11) + 0.5) * 0x1.0p-53;
}

// count normals, row-major, from stream `seed`
void fill_normals(uint64_t seed, size_t count, double* out) {
  const double two_pi = 6.283185307179586;
  for (size_t k = 0; 2 * k < count; ++k) {
    double u1 = uniform01(seed, 2 * k), u2 = uniform01(seed, 2 * k + 1);
    double r = std::sqrt(-2.0 * std::log(u1));
    double t = two_pi * u2;
    out[2 * k] = r * std::cos(t);
    if (2 * k + 1 < count) out[2 * k + 1] = r * std::sin(t);
  }
}

// Householder QR of a d x d matrix; returns Q with R's diagonal made positive
// (Q ← Q·diag(sign diag R)), i.e. the unique QR factor with positive diagonal.
// a: column-major copy of G (overwritten).  q: row-major d x d output.
void householder_q_positive(int d, std::vector<double>& a, double* q) {
  auto A = [&](int r, int c) -> double& { return a[static_cast<size_t>(c) * d + r]; };
  std::vector<double> vs(static_cast<size_t>(d) * d, 0.0);  // reflectors, column k = v_k
  std::vector<double> rdiag(d);
  for (int k = 0; k < d; ++k) {
    double nrm = 0.0;
    for (int r = k; r < d; ++r) nrm += A(r, k) * A(r, k);
    nrm = std::sqrt(nrm);
    double x0 = A(k, k);
    double alpha = (x0 >= 0.0) ? -nrm : nrm;  // R_kk = alpha, v = x - alpha e1
    double* v = &vs[static_cast<size_t>(k) * d];
    for (int r = k; r < d; ++r) v[r] = A(r, k);
    v[k] -= alpha;
    double vn2 = 0.0;
    for (int r = k; r < d; ++r) vn2 += v[r] * v[r];
    rdiag[k] = alpha;
    if (vn2 == 0.0) continue;  // column already reduced: H_k = I
    double inv = 2.0 / vn2;
    for (int c = k + 1; c < d; ++c) {
      double* col = &a[static_cast<size_t>(c) * d];
      double s = 0.0;
      for (int r = k; r < d; ++r) s += v[r] * col[r];
      s *= inv;
      for (int r = k; r < d; ++r) col[r] -= s * v[r];
    }
  }
  // Q = H_0 H_1 ... H_{d-1}: apply reflectors right-to-left to the identity.
  std::vector<double> qc(static_cast<size_t>(d) * d, 0.0);  // column-major
  for (int i = 0; i < d; ++i) qc[static_cast<size_t>(i) * d + i] = 1.0;
  for (int k = d - 1; k >= 0; --k) {
    const double* v = &vs[static_cast<size_t>(k) * d];
    double vn2 = 0.0;
    for (int r = k; r < d; ++r) vn2 += v[r] * v[r];
    if (vn2 == 0.0) continue;
    double inv = 2.0 / vn2;
    for (int c = 0; c < d; ++c) {
      double* col = &qc[static_cast<size_t>(c) * d];
      double s = 0.0;
      for (int r = k; r < d; ++r) s += v[r] * col[r];
      s *= inv;
      for (int r = k; r < d; ++r) col[r] -= s * v[r];
    }
  }
  for (int r = 0; r < d; ++r)
    for (int c = 0; c < d; ++c) {
      double sg = (rdiag[c] < 0.0) ? -1.0 : 1.0;
      q[static_cast<size_t>(r) * d + c] = qc[static_cast<size_t>(c) * d + r] * sg;
    }
}

// ---- Lloyd-Max on f_d(x) ∝ (1-x²)^((d-3)/2) by composite Gauss-Legendre ----

struct GaussLegendre {
  std::vector<double> x, w;
  explicit GaussLegendre(int n) : x(n), w(n) {
    for (int i = 0; i < n; ++i) {  // Newton on P_n from the Chebyshev guess
      double z = std::cos(M_PI * (i + 0.75) / (n + 0.5)), pp = 0.0;
      for (int it = 0; it < 100; ++it) {
        double p1 = 1.0, p2 = 0.0;
        for (int j = 1; j <= n; ++j) {
          double p3 = p2;
          p2 = p1;
          p1 = ((2.0 * j - 1.0) * z * p2 - (j - 1.0) * p3) / j;
        }
        pp = n * (z * p1 - p2) / (z * z - 1.0);
        double dz = p1 / pp;
        z -= dz;
        if (std::fabs(dz) < 1e-17) break;
      }
      x[i] = z;
      w[i] = 2.0 / ((1.0 - z * z) * pp * pp);
    }
  }
};

// ∫_a^b x^k (1-x²)^e dx for k = 0, 1 (unnormalised), a, b in [0, 1]
void cell_moments(const GaussLegendre& gl, double e, double a, double b, double lim, double* m0, double* m1) {
  *m0 = 0.0;
  *m1 = 0.0;
  if (b > lim) b = lim;  // beyond lim the density is below 1e-300 of its peak
  if (b <= a) return;
  const int panels = 64;
  double h = (b - a) / panels;
  for (int p = 0; p < panels; ++p) {
    double lo = a + p * h, mid = lo + 0.5 * h;
    for (size_t i = 0; i < gl.x.size(); ++i) {
      double xx = mid + 0.5 * h * gl.x[i];
      // exp(e log1p(-x²)) keeps full relative accuracy where pow(1 - x², e)
      // would multiply the rounding error of 1 - x² by e
      double f = std::exp(e * std::log1p(-xx * xx)) * gl.w[i] * 0.5 * h;
      *m0 += f;
      *m1 += f * xx;
    }
  }
}

}  // namespace

extern "C" tq_status tq_make_rotation(int d, uint64_t seed, double* pi) {
  if (d < 2 || d > 4096 || pi == nullptr) return TQ_ERR_ARG;
  std::vector<double> g(static_cast<size_t>(d) * d);
  fill_normals(seed, g.size(), g.data());  // row-major G
  std::vector<double> a(g.size());
  for (int r = 0; r < d; ++r)
    for (int c = 0; c < d; ++c) a[static_cast<size_t>(c) * d + r] = g[static_cast<size_t>(r) * d + c];
  householder_q_positive(d, a, pi);
  return TQ_OK;
}

extern "C" tq_status tq_make_codebook(int d, int w, double* centroids, double* bounds, double* mse_per_coord) {
  if (d < 3 || w < 1 || w > 4 || centroids == nullptr || bounds == nullptr) return TQ_ERR_ARG;
  const int L = 1 << w, half = L / 2;
  const double e = 0.5 * (d - 3);
  const double sd = 1.0 / std::sqrt(static_cast<double>(d));
  // (1-x²)^e < 1e-300 beyond x² > 1 - 1e-300^(1/e); cap the range at 60 sd
  double lim = std::fmin(1.0, 60.0 * sd);
  static const GaussLegendre gl(24);
  double tot0, tot1;
  cell_moments(gl, e, 0.0, 1.0, lim, &tot0, &tot1);  // half of the normaliser
  std::vector<double> c(half), t(half + 1), cn(half);
  for (int k = 0; k < half; ++k) c[k] = (k + 0.5) * 2.0 * sd / half;  // spread over ~2 sd
  double best = 1e300;
  int since_best = 0;
  bool ok = false;
  for (int it = 0; it < 100000; ++it) {
    t[0] = 0.0;
    for (int k = 1; k < half; ++k) t[k] = 0.5 * (c[k - 1] + c[k]);
    t[half] = 1.0;
    double delta = 0.0;
    for (int k = 0; k < half; ++k) {
      double m0, m1;
      cell_moments(gl, e, t[k], t[k + 1], lim, &m0, &m1);
      cn[k] = m1 / m0;
      delta = std::fmax(delta, std::fabs(cn[k] - c[k]));
    }
    c = cn;
    if (delta <= 1e-14 * c[half - 1]) { ok = true; break; }
    if (delta < best) { best = delta; since_best = 0; }
    else if (++since_best >= 100 && best <= 1e-12 * c[half - 1]) { ok = true; break; }
  }
  if (!ok) return TQ_ERR_NUMERIC;
  t[0] = 0.0;
  for (int k = 1; k < half; ++k) t[k] = 0.5 * (c[k - 1] + c[k]);
  t[half] = 1.0;
  double sum_pc2 = 0.0;
  for (int k = 0; k < half; ++k) {
    double m0, m1;
    cell_moments(gl, e, t[k], t[k + 1], lim, &m0, &m1);
    sum_pc2 += (m0 / tot0) * 0.5 * c[k] * c[k];  // mass of the cell = m0 / (2 tot0)
  }
  for (int k = 0; k < half; ++k) {
    centroids[half + k] = c[k];
    centroids[half - 1 - k] = -c[k];
  }
  for (int k = 1; k < half; ++k) {
    bounds[half - 1 + k] = t[k];
    bounds[half - 1 - k] = -t[k];
  }
  bounds[half - 1] = 0.0;
  if (mse_per_coord) *mse_per_coord = 1.0 / d - 2.0 * sum_pc2;
  return TQ_OK;
}

extern "C" tq_status tq_make_qjl(int m, int d, uint64_t seed, const double* pi, double* S, double* s_rot) {
  if (m < 1 || d < 1 || m > 65536 || d > 4096 || S == nullptr) return TQ_ERR_ARG;
  fill_normals(seed, static_cast<size_t>(m) * d, S);
  if (pi != nullptr && s_rot != nullptr) {
    // s_rot[i][j] = Σ_k S[i][k] Π[j][k]
    for (int i = 0; i < m; ++i)
      for (int j = 0; j < d; ++j) {
        double s = 0.0;
        const double* sr = S + static_cast<size_t>(i) * d;
        const double* pr = pi + static_cast<size_t>(j) * d;
        for (int k = 0; k < d; ++k) s += sr[k] * pr[k];
        s_rot[static_cast<size_t>(i) * d + j] = s;
      }
  }
  return TQ_OK;
}

extern "C" const char* tq_status_str(tq_status s) {
  switch (s) {
    case TQ_OK: return "ok";
    case TQ_ERR_ARG: return "invalid argument";
    case TQ_ERR_UNSUPPORTED: return "unsupported configuration";
    case TQ_ERR_CUDA: return "CUDA error";
    case TQ_ERR_WORKSPACE: return "workspace too small";
    case TQ_ERR_NUMERIC: return "setup iteration did not converge";
  }
  return "unknown status";
}

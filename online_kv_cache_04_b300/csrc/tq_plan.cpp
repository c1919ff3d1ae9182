// Device plan: fp32 / bf16 copies of the setup tables in one caller-owned
// buffer.  Host-side conversion, then plain cudaMemcpyAsync uploads.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <thread>
#include <vector>

#include "tq_internal.h"

namespace {

constexpr size_t kAlign = 256;
inline size_t up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

struct Layout {
  size_t pi, pi_t, s_rot, s_rot_t, cent, bnd, walsh, pi_bf, s_bf, pi_fr, s_fr, s_x, total;
  bool frag;  // warp-MMA operand copies present (d a multiple of 128)
  bool sx;    // bf16 pieces of S itself present (d a multiple of 256, m = d)
};

Layout layout(int d, int m, int w) {
  Layout l{};
  size_t o = 0;
  const size_t L = size_t(1) << w;
  l.pi = o;      o += up(sizeof(float) * d * d);
  l.pi_t = o;    o += up(sizeof(float) * d * d);
  l.s_rot = o;   o += up(sizeof(float) * size_t(m) * d);
  l.s_rot_t = o; o += up(sizeof(float) * size_t(m) * d);
  l.cent = o;    o += up(sizeof(float) * L);
  l.bnd = o;     o += up(sizeof(float) * L);
  l.walsh = o;   o += up(sizeof(float) * L);
  l.pi_bf = o;   o += up(sizeof(uint16_t) * 2 * d * d);
  l.s_bf = o;    o += up(sizeof(uint16_t) * 2 * size_t(m) * d);
  l.frag = d % 128 == 0;
  l.pi_fr = o;   o += l.frag ? up(sizeof(uint16_t) * 2 * size_t(d) * d) : 0;
  l.s_fr = o;    o += l.frag ? up(sizeof(uint16_t) * 2 * size_t(m) * d) : 0;
  l.sx = d % 256 == 0 && m == d;
  l.s_x = o;     o += l.sx ? up(sizeof(uint16_t) * 2 * size_t(m) * d) : 0;
  l.total = o;
  return l;
}

// round-to-nearest-even float -> bf16 bits (inputs are finite)
uint16_t bf16_rne(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return static_cast<uint16_t>(u >> 16);
}
double bf16_value(uint16_t h) {
  uint32_t u = uint32_t(h) << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

// S = (S Πᵀ) Π (m x d, float64), rows split over host threads.
std::vector<double> unrotate_qjl(const double* s_rot, const double* pi, int m, int d) {
  std::vector<double> S(size_t(m) * d, 0.0);
  auto rows = [&](int i0, int i1) {
    for (int i = i0; i < i1; ++i) {
      double* out = S.data() + size_t(i) * d;
      for (int k = 0; k < d; ++k) {
        const double a = s_rot[size_t(i) * d + k];
        const double* p = pi + size_t(k) * d;
        for (int j = 0; j < d; ++j) out[j] += a * p[j];
      }
    }
  };
  const int nt = std::max(1, std::min<int>(16, static_cast<int>(std::thread::hardware_concurrency())));
  std::vector<std::thread> pool;
  const int per = (m + nt - 1) / nt;
  for (int t = 0; t < nt; ++t) {
    const int i0 = t * per, i1 = std::min(m, i0 + per);
    if (i0 < i1) pool.emplace_back(rows, i0, i1);
  }
  for (auto& th : pool) th.join();
  return S;
}

}  // namespace

extern "C" size_t tq_plan_bytes(int d, int m, int w) {
  if (!tq::valid_shape(d, m, w)) return 0;
  return layout(d, m, w).total;
}

extern "C" tq_status tq_plan_init(tq_plan* plan, int d, int m, int w, const double* pi, const double* s_rot,
                                  const double* centroids, const double* bounds, void* dev, size_t bytes,
                                  tq_stream stream) {
  if (!plan || !pi || (m > 0 && !s_rot) || !centroids || !bounds || !dev || !tq::valid_shape(d, m, w))
    return TQ_ERR_ARG;
  const Layout l = layout(d, m, w);
  if (bytes < l.total || (reinterpret_cast<uintptr_t>(dev) % kAlign) != 0) return TQ_ERR_ARG;
  const int L = 1 << w;
  std::vector<unsigned char> host(l.total, 0);
  auto F = [&](size_t off) { return reinterpret_cast<float*>(host.data() + off); };
  auto H = [&](size_t off) { return reinterpret_cast<uint16_t*>(host.data() + off); };
  for (int i = 0; i < d; ++i)
    for (int j = 0; j < d; ++j) {
      double v = pi[size_t(i) * d + j];
      F(l.pi)[size_t(i) * d + j] = static_cast<float>(v);
      F(l.pi_t)[size_t(j) * d + i] = static_cast<float>(v);
      uint16_t hi = bf16_rne(static_cast<float>(v));
      uint16_t lo = bf16_rne(static_cast<float>(v - bf16_value(hi)));
      H(l.pi_bf)[size_t(i) * d + j] = hi;
      H(l.pi_bf)[size_t(d) * d + size_t(i) * d + j] = lo;
    }
  for (int i = 0; i < m; ++i)
    for (int j = 0; j < d; ++j) {
      double v = s_rot[size_t(i) * d + j];
      F(l.s_rot)[size_t(i) * d + j] = static_cast<float>(v);
      F(l.s_rot_t)[size_t(j) * m + i] = static_cast<float>(v);
      uint16_t hi = bf16_rne(static_cast<float>(v));
      uint16_t lo = bf16_rne(static_cast<float>(v - bf16_value(hi)));
      H(l.s_bf)[size_t(i) * d + j] = hi;
      H(l.s_bf)[size_t(m) * d + size_t(i) * d + j] = lo;
    }
  // bf16 pieces of S = (S Πᵀ) Π for the wide tensor-core quantizer's sign stage
  if (l.sx) {
    const std::vector<double> S = unrotate_qjl(s_rot, pi, m, d);
    for (size_t e = 0; e < size_t(m) * d; ++e) {
      const uint16_t hi = bf16_rne(static_cast<float>(S[e]));
      H(l.s_x)[e] = hi;
      H(l.s_x)[size_t(m) * d + e] = bf16_rne(static_cast<float>(S[e] - bf16_value(hi)));
    }
  }
  // warp-MMA operand order of the pieces (see tq_plan.pi_frag)
  if (l.frag) {
    auto frag = [&](size_t off, const uint16_t* src, int rows) {
      const size_t ks_n = d / 16, fr_n = rows / 8;
      for (int p = 0; p < 2; ++p)
        for (size_t ks = 0; ks < ks_n; ++ks)
          for (size_t f = 0; f < fr_n; ++f)
            for (int lane = 0; lane < 32; ++lane) {
              const int g = lane >> 2, t = lane & 3;
              const size_t r = 8 * f + g, c = 16 * ks + 2 * t;
              uint16_t* dst = H(off) + (((p * ks_n + ks) * fr_n + f) * 32 + lane) * 4;
              const uint16_t* row = src + size_t(p) * rows * d + r * d;
              dst[0] = row[c];
              dst[1] = row[c + 1];
              dst[2] = row[c + 8];
              dst[3] = row[c + 9];
            }
    };
    frag(l.pi_fr, H(l.pi_bf), d);
    frag(l.s_fr, H(l.s_bf), m);
  }
  for (int k = 0; k < L; ++k) F(l.cent)[k] = static_cast<float>(centroids[k]);
  for (int k = 0; k < L - 1; ++k) F(l.bnd)[k] = static_cast<float>(bounds[k]);
  // Walsh coefficients: walsh[mask] = 2^-w Σ_idx c[idx] Π_{p in mask} (2 bit_p(idx) - 1)
  for (int mask = 0; mask < L; ++mask) {
    double s = 0.0;
    for (int idx = 0; idx < L; ++idx) {
      double sign = 1.0;
      for (int p = 0; p < w; ++p)
        if (mask >> p & 1) sign *= ((idx >> p) & 1) ? 1.0 : -1.0;
      s += centroids[idx] * sign;
    }
    F(l.walsh)[mask] = static_cast<float>(s / L);
  }
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(dev, host.data(), l.total, cudaMemcpyHostToDevice, st) != cudaSuccess) return TQ_ERR_CUDA;
  // pageable source: the copy has been staged when the call returns, so `host` may go
  if (cudaStreamSynchronize(st) != cudaSuccess) return TQ_ERR_CUDA;
  unsigned char* base = static_cast<unsigned char*>(dev);
  plan->d = d;
  plan->m = m;
  plan->w = w;
  plan->qjl_alpha = m > 0 ? static_cast<float>(std::sqrt(M_PI / 2.0) / m) : 0.0f;
  plan->pi = reinterpret_cast<const float*>(base + l.pi);
  plan->pi_t = reinterpret_cast<const float*>(base + l.pi_t);
  plan->s_rot = reinterpret_cast<const float*>(base + l.s_rot);
  plan->s_rot_t = reinterpret_cast<const float*>(base + l.s_rot_t);
  plan->centroids = reinterpret_cast<const float*>(base + l.cent);
  plan->bounds = reinterpret_cast<const float*>(base + l.bnd);
  plan->walsh = reinterpret_cast<const float*>(base + l.walsh);
  plan->pi_bf16 = reinterpret_cast<const uint16_t*>(base + l.pi_bf);
  plan->s_bf16 = reinterpret_cast<const uint16_t*>(base + l.s_bf);
  plan->pi_frag = l.frag ? reinterpret_cast<const uint16_t*>(base + l.pi_fr) : nullptr;
  plan->s_frag = l.frag && m > 0 ? reinterpret_cast<const uint16_t*>(base + l.s_fr) : nullptr;
  plan->s_x_bf16 = l.sx ? reinterpret_cast<const uint16_t*>(base + l.s_x) : nullptr;
  return TQ_OK;
}

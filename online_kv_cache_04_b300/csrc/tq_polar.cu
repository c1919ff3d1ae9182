// PolarQuant's recursive polar stage as an alternative first stage, followed
// by the same 1-bit QJL stage on the residual ("TurboQuant 与 AI 效率革命" §二
// "突破：极坐标" and §四; "TurboQuant压缩效果": the first level at 4 bits,
// later levels at 2).
//
// Transform of a rotated vector u = Π x (d a power of two): level 1 pairs
// (u_2i, u_2i+1) into a radius and an angle atan2(u_2i+1, u_2i) in [0, 2π);
// level ℓ ≥ 2 pairs the level ℓ-1 radii (a, b) into √(a² + b²) and
// atan2(b, a) in [0, π/2]; one radius (‖x‖) and d - 1 angles remain.  Level 1
// angles are uniform, so their codebook is 2^b1 equal cells with midpoint
// centroids; a level-ℓ angle follows the page's law ∝ sin^(k-1)(2ψ) with
// k = 2^(ℓ-1) coordinates under each radius, and takes the Lloyd-Max codebook
// of that law at b bits.  Reconstruction runs the tree back down from the
// stored norm with the centroids' cosines and sines; the residual
// r = x - Πᵀũ goes through QJL (σ = sign(S r), ‖r‖) as in tq_quantize.
//
// Records (TQ_LAYOUT_ROWS): tq_polar_index_words(d, b1, b) words per vector,
// the d/2 level-1 codes of b1 bits packed 32/b1 to a word (code i at bits
// b1·(i mod 32/b1) of word i / (32/b1); "TurboQuant压缩效果": eight 4-bit
// numbers in one 32-bit word), then from the next word the codes of levels 2,
// 3, ... in that order, b bits each, packed the same way; norm = ‖x‖ (fp32),
// signs and residual norm as for tq_quantize.
//
// Decode: the general path's query prep (Π q, S q) and log-sum-exp combine,
// with a split kernel that rebuilds each key's and value's rotated vector
// from its angle codes in shared memory (one token per thread) and then
// scores and accumulates as the general kernel does.
#include <cuda_bf16.h>

#include <algorithm>
#include <cmath>
#include <vector>

#include "tq_internal.h"

namespace {

constexpr int kMaxLevels = 8;   // d <= 256
constexpr int kTab = 16;        // entries per table row (b1, b <= 4)
constexpr int kThreads = 128;
constexpr int kMaxG = 8;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kTwoPi = 6.283185307179586f;

int levels_of(int d) {
  int L = 0;
  while ((1 << L) < d) ++L;
  return (1 << L) == d ? L : -1;
}

bool valid_bits(int bits) { return bits == 1 || bits == 2 || bits == 4; }

bool valid_polar_shape(int d, int m, int b1, int b) {
  const int L = levels_of(d);
  return L >= 2 && L <= kMaxLevels && m >= 32 && m <= 256 && m % 32 == 0 && valid_bits(b1) && valid_bits(b);
}

__host__ __device__ inline int words1(int d, int b1) { return ((d / 2) * b1 + 31) / 32; }
int index_words(int d, int b1, int b) { return words1(d, b1) + ((d / 2 - 1) * b + 31) / 32; }

// ---------------------------------------------------------------- host codebooks
struct GL {
  std::vector<double> x, w;
  explicit GL(int n) : x(n), w(n) {
    for (int i = 0; i < n; ++i) {  // Newton on P_n from the Chebyshev guess
      double z = std::cos(M_PI * (i + 0.75) / (n + 0.5)), pp = 0.0;
      for (int it = 0; it < 100; ++it) {
        double p1 = 1.0, p2 = 0.0;
        for (int j = 1; j <= n; ++j) {
          const double p3 = p2;
          p2 = p1;
          p1 = ((2.0 * j - 1.0) * z * p2 - (j - 1.0) * p3) / j;
        }
        pp = n * (z * p1 - p2) / (z * z - 1.0);
        const double dz = p1 / pp;
        z -= dz;
        if (std::fabs(dz) < 1e-17) break;
      }
      x[i] = z;
      w[i] = 2.0 / ((1.0 - z * z) * pp * pp);
    }
  }
};

// ∫_a^b v^j cos^(k-1)(2v) dv for j = 0, 1 (unnormalised, v = ψ - π/4 >= 0)
void angle_moments(const GL& gl, int k, double a, double b, double lim, double* m0, double* m1) {
  *m0 = 0.0;
  *m1 = 0.0;
  if (b > lim) b = lim;
  if (b <= a) return;
  const int panels = 64;
  const double h = (b - a) / panels;
  for (int p = 0; p < panels; ++p) {
    const double mid = a + (p + 0.5) * h;
    for (size_t i = 0; i < gl.x.size(); ++i) {
      const double v = mid + 0.5 * h * gl.x[i];
      const double c = std::cos(2.0 * v);
      const double f = c > 0.0 ? std::exp((k - 1) * std::log(c)) * gl.w[i] * 0.5 * h : 0.0;
      *m0 += f;
      *m1 += f * v;
    }
  }
}

// Lloyd-Max codebook with n = 2^bits levels of the law ∝ sin^(k-1)(2ψ) on
// [0, π/2], symmetric about π/4: iterate on the upper half in v = ψ - π/4.
bool lloyd_max_angle(int k, int bits, double* cent, double* bnd) {
  const int n = 1 << bits, half = n / 2;
  static const GL gl(24);
  const double sd = 0.5 / std::sqrt(std::max(1.0, k - 1.0));
  const double lim = std::min(M_PI / 4.0, 40.0 * sd);
  std::vector<double> c(half), t(half + 1), cn(half);
  for (int j = 0; j < half; ++j) c[j] = std::min(lim, (j + 0.5) * 2.0 * sd / half);
  bool ok = false;
  for (int it = 0; it < 100000; ++it) {
    t[0] = 0.0;
    for (int j = 1; j < half; ++j) t[j] = 0.5 * (c[j - 1] + c[j]);
    t[half] = M_PI / 4.0;
    double delta = 0.0;
    for (int j = 0; j < half; ++j) {
      double m0, m1;
      angle_moments(gl, k, t[j], t[j + 1], lim, &m0, &m1);
      cn[j] = m0 > 0.0 ? m1 / m0 : 0.5 * (t[j] + t[j + 1]);
      delta = std::max(delta, std::fabs(cn[j] - c[j]));
    }
    c = cn;
    if (delta <= 1e-15) { ok = true; break; }
  }
  if (!ok) return false;
  for (int j = 0; j < half; ++j) {
    cent[half + j] = M_PI / 4.0 + c[j];
    cent[half - 1 - j] = M_PI / 4.0 - c[j];
  }
  for (int j = 0; j < n - 1; ++j) bnd[j] = 0.5 * (cent[j] + cent[j + 1]);
  return true;
}

// ---------------------------------------------------------------- plan layout
constexpr size_t kAlign = 256;
inline size_t up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }
struct PLayout {
  size_t pi, pi_t, s_rot, s_rot_t, tab, total;
};
PLayout playout(int d, int m) {
  PLayout l{};
  size_t o = 0;
  l.pi = o;      o += up(sizeof(float) * d * d);
  l.pi_t = o;    o += up(sizeof(float) * d * d);
  l.s_rot = o;   o += up(sizeof(float) * size_t(m) * d);
  l.s_rot_t = o; o += up(sizeof(float) * size_t(m) * d);
  l.tab = o;     o += up(sizeof(float) * kMaxLevels * 3 * kTab);
  l.total = o;
  return l;
}

// ---------------------------------------------------------------- device helpers
// code of level `lev` (1-based) angle i from one vector's index words
__device__ __forceinline__ int angle_code(const uint32_t* words, int d, int b1, int b, int lev, int i) {
  if (lev == 1) {
    const int per = 32 / b1;
    return (words[i / per] >> (b1 * (i % per))) & ((1 << b1) - 1);
  }
  const int off = d / 2 - (d >> (lev - 1)) + i;  // codes of levels 2 .. lev-1 come first
  const int per = 32 / b, base = ((d / 2) * b1 + 31) / 32;
  return (words[base + off / per] >> (b * (off % per))) & ((1 << b) - 1);
}

// ũ (rotated domain) of one record, built top-down in place in buf[0 .. d):
// buf[0] = radius; at each level the n radii at buf[0 .. n) become 2n values,
// highest index first so that nothing unread is overwritten.  tab: [level][3][16]
// (cos, sin, bounds) in shared memory.
__device__ __forceinline__ void rebuild(const uint32_t* words, float radius, int d, int L, int b1, int b,
                                        const float* tab, float* buf, int stride) {
  buf[0] = radius;
  for (int lev = L; lev >= 1; --lev) {
    const int n = d >> lev;
    const float* ct = tab + (lev - 1) * 3 * kTab;
    for (int i = n - 1; i >= 0; --i) {
      const int c = angle_code(words, d, b1, b, lev, i);
      const float r = buf[i * stride];
      buf[(2 * i) * stride] = r * ct[c];
      buf[(2 * i + 1) * stride] = r * ct[kTab + c];
    }
  }
}

struct PolarQArgs {
  const void* x;
  int64_t n, ld;
  int d, m, L, b1, b, nw;
  const float* pi_t;     // [d][d]
  const float* s_rot_t;  // [d][m]
  const float* tables;   // [L][3][16]
  uint32_t* idx;         // rows already offset, nw words per row
  uint32_t* sgn;
  float* norm;
  float* rnorm;
};

template <typename T>
__device__ __forceinline__ float load_x(const T* p);
template <>
__device__ __forceinline__ float load_x<float>(const float* p) { return *p; }
template <>
__device__ __forceinline__ float load_x<__nv_bfloat16>(const __nv_bfloat16* p) { return __bfloat162float(*p); }

// One CTA per tile of TV vectors: rotate (thread = coordinate), then one warp per
// vector runs the transform, bucketizes every angle, packs the codes and
// rebuilds ũ; the residual's QJL signs come last (thread = JL row).
template <int TV, typename T>
__global__ void __launch_bounds__(kThreads) quantize_polar_kernel(PolarQArgs a) {
  extern __shared__ float sm[];
  const int d = a.d, m = a.m, L = a.L;
  float* xs = sm;                  // [TV][d] input, then the residual Πx - ũ
  float* us = xs + TV * d;         // [TV][d] Π x
  float* ra = us + TV * d;         // [TV][d] radii ping-pong (two halves of d/2)
  float* rb = ra + TV * d;         // [TV][d] rebuild buffer
  float* nrm = rb + TV * d;        // [TV]
  float* rsq = nrm + TV;           // [TV]
  float* tab = rsq + TV;           // [L][3][16]
  uint32_t* codes = reinterpret_cast<uint32_t*>(tab + kMaxLevels * 3 * kTab);  // [TV][nw] packed words
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int e = tid; e < L * 3 * kTab; e += kThreads) tab[e] = a.tables[e];
  const T* x = static_cast<const T*>(a.x);
  const int64_t ntiles = (a.n + TV - 1) / TV;
  for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
    const int64_t v0 = tile * TV;
    for (int e = tid; e < TV * d; e += kThreads) {
      const int v = e / d, i = e - v * d;
      xs[e] = v0 + v < a.n ? load_x<T>(x + (v0 + v) * a.ld + i) : 0.f;
    }
    for (int e = tid; e < TV * a.nw; e += kThreads) codes[e] = 0u;
    __syncthreads();
    for (int v = warp; v < TV; v += kThreads / 32) {
      float s = 0.f;
      for (int i = lane; i < d; i += 32) s = fmaf(xs[v * d + i], xs[v * d + i], s);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
      if (lane == 0) nrm[v] = sqrtf(s);
    }
    for (int j = tid; j < d; j += kThreads) {
      float acc[TV];
#pragma unroll
      for (int v = 0; v < TV; ++v) acc[v] = 0.f;
      for (int i = 0; i < d; ++i) {
        const float p = __ldg(a.pi_t + (size_t)i * d + j);
#pragma unroll
        for (int v = 0; v < TV; ++v) acc[v] = fmaf(p, xs[v * d + i], acc[v]);
      }
#pragma unroll
      for (int v = 0; v < TV; ++v) us[v * d + j] = acc[v];
    }
    __syncthreads();
    for (int v = warp; v < TV; v += kThreads / 32) {
      const float* u = us + v * d;
      float* r0 = ra + v * d;           // level radii: even levels in r0, odd in r1
      float* r1 = r0 + d / 2;
      uint32_t* cw = codes + v * a.nw;
      const int per1 = 32 / a.b1, per = 32 / a.b, base = words1(d, a.b1);
      for (int i = lane; i < d / 2; i += 32) {
        const float xx = u[2 * i], yy = u[2 * i + 1];
        float psi = atan2f(yy, xx);
        if (psi < 0.f) psi += kTwoPi;
        int c = 0;
        for (int k = 0; k < (1 << a.b1) - 1; ++k) c += tab[2 * kTab + k] < psi ? 1 : 0;
        atomicOr(cw + i / per1, (uint32_t)c << (a.b1 * (i % per1)));
        r0[i] = sqrtf(xx * xx + yy * yy);
      }
      __syncwarp();
      int off = 0;
      for (int lev = 2; lev <= L; ++lev) {
        const int n = d >> lev;
        const float* src = (lev & 1) ? r1 : r0;
        float* dst = (lev & 1) ? r0 : r1;
        const float* bt = tab + ((lev - 1) * 3 + 2) * kTab;
        for (int i = lane; i < n; i += 32) {
          const float aa = src[2 * i], bb = src[2 * i + 1];
          const float psi = atan2f(bb, aa);
          int c = 0;
          for (int k = 0; k < (1 << a.b) - 1; ++k) c += bt[k] < psi ? 1 : 0;
          atomicOr(cw + base + (off + i) / per, (uint32_t)c << (a.b * ((off + i) % per)));
          dst[i] = sqrtf(aa * aa + bb * bb);
        }
        off += n;
        __syncwarp();
      }
      // ũ from the codes, radius ‖x‖ (one lane: the tree is sequential per vector)
      if (lane == 0) rebuild(cw, nrm[v], d, L, a.b1, a.b, tab, rb + v * d, 1);
      __syncwarp();
      float s2 = 0.f;
      for (int j = lane; j < d; j += 32) {
        const float rr = u[j] - rb[v * d + j];
        xs[v * d + j] = rr;
        s2 = fmaf(rr, rr, s2);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) s2 += __shfl_xor_sync(0xffffffffu, s2, o);
      if (lane == 0) rsq[v] = s2;
      __syncwarp();
      const int64_t row = v0 + v;
      for (int k = lane; k < a.nw; k += 32)
        if (row < a.n) a.idx[row * a.nw + k] = cw[k];
    }
    __syncthreads();
    // σ = sign(S r) = sign(S̃ (Π x - ũ))
    for (int jj = tid; jj < m; jj += kThreads) {
      float acc[TV];
#pragma unroll
      for (int v = 0; v < TV; ++v) acc[v] = 0.f;
      for (int i = 0; i < d; ++i) {
        const float sij = __ldg(a.s_rot_t + (size_t)i * m + jj);
#pragma unroll
        for (int v = 0; v < TV; ++v) acc[v] = fmaf(sij, xs[v * d + i], acc[v]);
      }
#pragma unroll
      for (int v = 0; v < TV; ++v) {
        const uint32_t word = __ballot_sync(0xffffffffu, acc[v] >= 0.f);
        if (lane == 0 && v0 + v < a.n) a.sgn[(v0 + v) * (m / 32) + jj / 32] = word;
      }
    }
    if (tid < TV && v0 + tid < a.n) {
      a.norm[v0 + tid] = nrm[tid];
      a.rnorm[v0 + tid] = sqrtf(rsq[tid]);
    }
    __syncthreads();
  }
}

struct PolarSplitArgs {
  int B, Hq, Hkv, G, d, m, L, b1, b, nw;
  int64_t ctx_stride, tokens_per_split;
  int nsplit;
  const uint32_t *kidx, *ksgn, *vidx, *vsgn;
  const float *knorm, *krnorm, *vnorm, *vrnorm;
  const int32_t* ctx_len;
  const float* qt;   // [B*Hq][d]
  const float* st;   // [B*Hq][m]
  const float* tables;
  float scale, alpha;
  float* part;       // [B*Hq][nsplit][2 + d + m]
};

// One context slice of one kv head for its G query heads, 128 tokens per chunk:
// thread t rebuilds token t's key (then value) into row t of a shared buffer.
__global__ void __launch_bounds__(kThreads) polar_split_kernel(PolarSplitArgs a) {
  extern __shared__ float sm[];
  const int d = a.d, m = a.m, G = a.G, ws = m / 32, ds = d + 1;  // row stride ds avoids bank conflicts
  float* qts = sm;                     // [G][d]
  float* sts = qts + G * d;            // [G][m]
  float* tab = sts + G * m;            // [L][3][16]
  float* buf = tab + kMaxLevels * 3 * kTab;  // [kThreads][d + 1] rebuilt vectors
  float* pn = buf + kThreads * ds;     // [G][kThreads] p (values carry their norm in ũ)
  float* pr = pn + G * kThreads;       // [G][kThreads] p·‖r_v‖
  float* red = pr + G * kThreads;      // [4][kMaxG]
  float* runm = red + 4 * kMaxG;       // [kMaxG]
  float* corr = runm + kMaxG;          // [kMaxG]
  uint32_t* vs = reinterpret_cast<uint32_t*>(corr + kMaxG);  // [kThreads][ws] value sign words
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int bh = blockIdx.y, b = bh / a.Hkv, h = bh - b * a.Hkv, split = blockIdx.x;
  const int64_t L = min((int64_t)max(__ldg(a.ctx_len + b), 0), a.ctx_stride);
  const int64_t t0 = split * a.tokens_per_split, t1 = min(t0 + a.tokens_per_split, L);
  const int head0 = b * a.Hq + h * G;
  for (int e = tid; e < G * d; e += kThreads) qts[e] = a.qt[(size_t)head0 * d + e];
  for (int e = tid; e < G * m; e += kThreads) sts[e] = a.st[(size_t)head0 * m + e];
  for (int e = tid; e < a.L * 3 * kTab; e += kThreads) tab[e] = a.tables[e];
  if (tid < kMaxG) runm[tid] = -INFINITY;
  __syncthreads();
  const int64_t rowbase = (int64_t)bh * a.ctx_stride;
  float acc_r[2][kMaxG], acc_s[2][kMaxG], lsum[kMaxG];
#pragma unroll
  for (int k = 0; k < 2; ++k)
#pragma unroll
    for (int g = 0; g < kMaxG; ++g) acc_r[k][g] = acc_s[k][g] = 0.f;
#pragma unroll
  for (int g = 0; g < kMaxG; ++g) lsum[g] = 0.f;
  uint32_t words[64];
  for (int64_t c0 = t0; c0 < t1; c0 += kThreads) {
    const int64_t t = c0 + tid;
    const bool valid = t < t1;
    const int cnt = (int)min((int64_t)kThreads, t1 - c0);
    float sc[kMaxG];
#pragma unroll
    for (int g = 0; g < kMaxG; ++g) sc[g] = -INFINITY;
    float* row = buf + tid * ds;
    if (valid) {
      const int64_t r = rowbase + t;
      for (int k = 0; k < a.nw; ++k) words[k] = __ldg(a.kidx + r * a.nw + k);
      rebuild(words, __ldg(a.knorm + r), d, a.L, a.b1, a.b, tab, row, 1);
      float d1[kMaxG], d2[kMaxG];
#pragma unroll
      for (int g = 0; g < kMaxG; ++g) d1[g] = d2[g] = 0.f;
      for (int j = 0; j < d; ++j) {
        const float uj = row[j];
#pragma unroll
        for (int g = 0; g < kMaxG; ++g)
          if (g < G) d1[g] = fmaf(qts[g * d + j], uj, d1[g]);
      }
      for (int k = 0; k < ws; ++k) {
        const uint32_t word = __ldg(a.ksgn + r * ws + k);
        for (int bb = 0; bb < 32; ++bb) {
          const float sg = ((word >> bb) & 1) ? 1.f : -1.f;
#pragma unroll
          for (int g = 0; g < kMaxG; ++g)
            if (g < G) d2[g] = fmaf(sts[g * m + k * 32 + bb], sg, d2[g]);
        }
      }
      const float rk = __ldg(a.krnorm + r);
#pragma unroll
      for (int g = 0; g < kMaxG; ++g)
        if (g < G) sc[g] = a.scale * (d1[g] + a.alpha * rk * d2[g]) * kLog2e;
      // the value record of the same token replaces the key in row t
      for (int k = 0; k < a.nw; ++k) words[k] = __ldg(a.vidx + r * a.nw + k);
      rebuild(words, __ldg(a.vnorm + r), d, a.L, a.b1, a.b, tab, row, 1);
      for (int k = 0; k < ws; ++k) vs[tid * ws + k] = __ldg(a.vsgn + r * ws + k);
    }
#pragma unroll
    for (int g = 0; g < kMaxG; ++g) {
      float v = sc[g];
      for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
      if (lane == 0 && g < G) red[warp * kMaxG + g] = v;
    }
    __syncthreads();
    if (tid < G) {
      const float cm = fmaxf(fmaxf(red[tid], red[kMaxG + tid]), fmaxf(red[2 * kMaxG + tid], red[3 * kMaxG + tid]));
      const float nm = fmaxf(runm[tid], cm);
      corr[tid] = exp2f(runm[tid] - nm);
      runm[tid] = nm;
    }
    __syncthreads();
    const float rv = valid ? __ldg(a.vrnorm + rowbase + t) : 0.f;
    for (int g = 0; g < G; ++g) {
      const float p = valid ? exp2f(sc[g] - runm[g]) : 0.f;
      pn[g * kThreads + tid] = p;
      pr[g * kThreads + tid] = p * rv;
      float ps = p;
      for (int o = 16; o > 0; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
      if (lane == 0) red[warp * kMaxG + g] = ps;
    }
    __syncthreads();
#pragma unroll
    for (int g = 0; g < kMaxG; ++g)
      if (g < G) lsum[g] = lsum[g] * corr[g] + (red[g] + red[kMaxG + g] + red[2 * kMaxG + g] + red[3 * kMaxG + g]);
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int j = tid + k * kThreads;
#pragma unroll
      for (int g = 0; g < kMaxG; ++g) {
        acc_r[k][g] *= corr[g < G ? g : 0];
        acc_s[k][g] *= corr[g < G ? g : 0];
      }
      if (j < d)
        for (int tt = 0; tt < cnt; ++tt) {
          const float uj = buf[tt * ds + j];
#pragma unroll
          for (int g = 0; g < kMaxG; ++g)
            if (g < G) acc_r[k][g] = fmaf(pn[g * kThreads + tt], uj, acc_r[k][g]);
        }
      if (j < m)
        for (int tt = 0; tt < cnt; ++tt) {
          const float sg = ((vs[tt * ws + (j >> 5)] >> (j & 31)) & 1) ? 1.f : -1.f;
#pragma unroll
          for (int g = 0; g < kMaxG; ++g)
            if (g < G) acc_s[k][g] = fmaf(pr[g * kThreads + tt], sg, acc_s[k][g]);
        }
    }
    __syncthreads();
  }
  const int stride = 2 + d + m;
  for (int g = 0; g < G; ++g) {
    float* pp = a.part + ((size_t)(head0 + g) * a.nsplit + split) * stride;
    if (tid == 0) {
      pp[0] = runm[g];
      pp[1] = lsum[g];
    }
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int j = tid + k * kThreads;
      if (j < d) pp[2 + j] = acc_r[k][g];
      if (j < m) pp[2 + d + j] = acc_s[k][g];
    }
  }
}

bool valid_polar_plan(const tq_polar_plan* p) {
  return p && valid_polar_shape(p->d, p->m, p->b1, p->b) && p->pi && p->pi_t && p->s_rot && p->s_rot_t && p->tables;
}

bool valid_polar_records(const tq_records* r, int64_t rows) {
  return r && r->idx && r->sgn && r->norm && r->rnorm && r->layout == TQ_LAYOUT_ROWS && r->capacity >= rows &&
         tq::aligned16(r->idx) && tq::aligned16(r->sgn) && tq::aligned16(r->norm) && tq::aligned16(r->rnorm);
}

struct PolarShape {
  int nsplit;
  int64_t tps;
};
PolarShape polar_shape(int B, int Hkv, int64_t ctx_stride) {
  const int64_t units = int64_t(B) * Hkv;
  const int64_t want = tq::cdiv(2 * int64_t(tq::sm_count()), units);
  const int64_t maxs = std::max<int64_t>(1, tq::cdiv(ctx_stride, 2 * kThreads));
  PolarShape s;
  s.nsplit = (int)std::max<int64_t>(1, std::min(want, maxs));
  s.tps = tq::cdiv(tq::cdiv(ctx_stride, s.nsplit), kThreads) * kThreads;
  return s;
}

size_t polar_ws_floats(const tq_polar_plan* p, int B, int Hq, int Hkv, int64_t ctx_stride) {
  const size_t heads = size_t(B) * Hq;
  return heads * (p->d + p->m) + heads * polar_shape(B, Hkv, ctx_stride).nsplit * (2 + p->d + p->m);
}

}  // namespace

extern "C" int tq_polar_index_words(int d, int b1, int b) {
  if (!valid_polar_shape(d, 32, b1, b)) return 0;
  return index_words(d, b1, b);
}

extern "C" tq_status tq_make_polar_codebooks(int d, int b1, int b, double* centroids, double* bounds) {
  if (!valid_polar_shape(d, 32, b1, b) || !centroids || !bounds) return TQ_ERR_ARG;
  const int L = levels_of(d), n1 = 1 << b1, n = 1 << b;
  for (int j = 0; j < n1; ++j) centroids[j] = 2.0 * M_PI * (j + 0.5) / n1;
  for (int j = 0; j < n1 - 1; ++j) bounds[j] = 2.0 * M_PI * (j + 1) / n1;
  for (int lev = 2; lev <= L; ++lev)
    if (!lloyd_max_angle(1 << (lev - 1), b, centroids + n1 + (lev - 2) * n, bounds + (n1 - 1) + (lev - 2) * (n - 1)))
      return TQ_ERR_NUMERIC;
  return TQ_OK;
}

extern "C" size_t tq_polar_plan_bytes(int d, int m, int b1, int b) {
  return valid_polar_shape(d, m, b1, b) ? playout(d, m).total : 0;
}

extern "C" tq_status tq_polar_plan_init(tq_polar_plan* plan, int d, int m, int b1, int b, const double* pi,
                                        const double* s_rot, const double* centroids, const double* bounds,
                                        void* dev, size_t bytes, tq_stream stream) {
  if (!plan || !valid_polar_shape(d, m, b1, b) || !pi || !s_rot || !centroids || !bounds || !dev ||
      !tq::aligned16(dev))
    return TQ_ERR_ARG;
  const PLayout l = playout(d, m);
  if (bytes < l.total) return TQ_ERR_ARG;
  std::vector<unsigned char> host(l.total, 0);
  auto F = [&](size_t off) { return reinterpret_cast<float*>(host.data() + off); };
  for (int r = 0; r < d; ++r)
    for (int c = 0; c < d; ++c) {
      F(l.pi)[r * d + c] = static_cast<float>(pi[r * d + c]);
      F(l.pi_t)[c * d + r] = static_cast<float>(pi[r * d + c]);
    }
  for (int i = 0; i < m; ++i)
    for (int j = 0; j < d; ++j) {
      F(l.s_rot)[i * d + j] = static_cast<float>(s_rot[i * d + j]);
      F(l.s_rot_t)[j * m + i] = static_cast<float>(s_rot[i * d + j]);
    }
  const int L = levels_of(d), n1 = 1 << b1, n = 1 << b;
  float* tab = F(l.tab);
  for (int lev = 1; lev <= L; ++lev) {
    const int cnt = lev == 1 ? n1 : n;
    const double* c = lev == 1 ? centroids : centroids + n1 + (lev - 2) * n;
    const double* bd = lev == 1 ? bounds : bounds + (n1 - 1) + (lev - 2) * (n - 1);
    float* row = tab + (lev - 1) * 3 * kTab;
    for (int j = 0; j < kTab; ++j) {
      row[j] = j < cnt ? static_cast<float>(std::cos(c[j])) : 0.f;
      row[kTab + j] = j < cnt ? static_cast<float>(std::sin(c[j])) : 0.f;
      row[2 * kTab + j] = j < cnt - 1 ? static_cast<float>(bd[j]) : INFINITY;
    }
  }
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(dev, host.data(), l.total, cudaMemcpyHostToDevice, st) != cudaSuccess) return TQ_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return TQ_ERR_CUDA;
  unsigned char* base = static_cast<unsigned char*>(dev);
  plan->d = d;
  plan->m = m;
  plan->b1 = b1;
  plan->b = b;
  plan->qjl_alpha = static_cast<float>(std::sqrt(M_PI / 2.0) / m);
  plan->pi = reinterpret_cast<const float*>(base + l.pi);
  plan->pi_t = reinterpret_cast<const float*>(base + l.pi_t);
  plan->s_rot = reinterpret_cast<const float*>(base + l.s_rot);
  plan->s_rot_t = reinterpret_cast<const float*>(base + l.s_rot_t);
  plan->tables = reinterpret_cast<const float*>(base + l.tab);
  return TQ_OK;
}

extern "C" tq_status tq_quantize_polar(const tq_polar_plan* plan, const void* x, tq_dtype dtype, int64_t n,
                                       int64_t ld_x, const tq_records* out, int64_t out_offset, tq_stream stream) {
  if (!valid_polar_plan(plan) || n < 0 || out_offset < 0 || (dtype != TQ_F32 && dtype != TQ_BF16)) return TQ_ERR_ARG;
  if (!valid_polar_records(out, 0)) return TQ_ERR_ARG;
  if (n == 0) return TQ_OK;
  if (!x || !tq::aligned16(x) || ld_x < plan->d || ld_x % 8 != 0) return TQ_ERR_ARG;
  if (out_offset > out->capacity || n > out->capacity - out_offset) return TQ_ERR_ARG;
  constexpr int TV = 8;
  PolarQArgs a{};
  a.x = x;
  a.n = n;
  a.ld = ld_x;
  a.d = plan->d;
  a.m = plan->m;
  a.L = levels_of(plan->d);
  a.b1 = plan->b1;
  a.b = plan->b;
  a.nw = index_words(plan->d, plan->b1, plan->b);
  a.pi_t = plan->pi_t;
  a.s_rot_t = plan->s_rot_t;
  a.tables = plan->tables;
  a.idx = out->idx + out_offset * a.nw;
  a.sgn = out->sgn + out_offset * (plan->m / 32);
  a.norm = out->norm + out_offset;
  a.rnorm = out->rnorm + out_offset;
  const size_t smem = sizeof(float) * (4 * TV * plan->d + 2 * TV + kMaxLevels * 3 * kTab) +
                      sizeof(uint32_t) * TV * a.nw;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int64_t grid = std::min<int64_t>((n + TV - 1) / TV, int64_t(tq::sm_count()) * 8);
  auto launch = [&](auto kern) -> tq_status {
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return TQ_ERR_CUDA;
    kern<<<(unsigned)grid, kThreads, smem, st>>>(a);
    return tq::launch_status();
  };
  return dtype == TQ_F32 ? launch(quantize_polar_kernel<TV, float>) : launch(quantize_polar_kernel<TV, __nv_bfloat16>);
}

extern "C" tq_status tq_decode_polar_workspace_size(const tq_polar_plan* plan, int B, int Hq, int Hkv,
                                                    int64_t ctx_stride, size_t* bytes) {
  if (!bytes || !valid_polar_plan(plan) || B < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv || Hq / Hkv > kMaxG ||
      ctx_stride < 1)
    return TQ_ERR_ARG;
  *bytes = sizeof(float) * polar_ws_floats(plan, B, Hq, Hkv, ctx_stride);
  return TQ_OK;
}

extern "C" tq_status tq_decode_attention_polar(const tq_polar_plan* plan, const void* q, tq_dtype q_dtype, int B,
                                               int Hq, int Hkv, const tq_records* K, const tq_records* V,
                                               const int32_t* ctx_len, int64_t ctx_stride, float scale, float* out,
                                               void* workspace, size_t ws_bytes, tq_stream stream) {
  size_t need = 0;
  tq_status rc = tq_decode_polar_workspace_size(plan, B, Hq, Hkv, ctx_stride, &need);
  if (rc != TQ_OK) return rc;
  if (!q || !ctx_len || !tq::aligned16(q) || (q_dtype != TQ_F32 && q_dtype != TQ_BF16)) return TQ_ERR_ARG;
  const int64_t rows = int64_t(B) * Hkv * ctx_stride;
  if (!valid_polar_records(K, rows) || !valid_polar_records(V, rows)) return TQ_ERR_ARG;
  if (!out || !tq::aligned16(out) || !workspace || !tq::aligned16(workspace)) return TQ_ERR_ARG;
  if (ws_bytes < need) return TQ_ERR_WORKSPACE;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  const int d = plan->d, m = plan->m;
  float* qt = static_cast<float*>(workspace);
  float* st = qt + size_t(B) * Hq * d;
  float* part = st + size_t(B) * Hq * m;
  tq_plan qp{};  // the query prep reads only the shape and the two matrices
  qp.d = d;
  qp.m = m;
  qp.pi = plan->pi;
  qp.s_rot = plan->s_rot;
  if ((rc = tq::launch_query_prep(&qp, q, q_dtype, B * Hq, qt, st, cs)) != TQ_OK) return rc;
  const PolarShape ps = polar_shape(B, Hkv, ctx_stride);
  PolarSplitArgs a{};
  a.B = B; a.Hq = Hq; a.Hkv = Hkv; a.G = Hq / Hkv; a.d = d; a.m = m;
  a.L = levels_of(d); a.b1 = plan->b1; a.b = plan->b; a.nw = index_words(d, plan->b1, plan->b);
  a.ctx_stride = ctx_stride;
  a.tokens_per_split = ps.tps;
  a.nsplit = ps.nsplit;
  a.kidx = K->idx; a.ksgn = K->sgn; a.knorm = K->norm; a.krnorm = K->rnorm;
  a.vidx = V->idx; a.vsgn = V->sgn; a.vnorm = V->norm; a.vrnorm = V->rnorm;
  a.ctx_len = ctx_len;
  a.qt = qt;
  a.st = st;
  a.tables = plan->tables;
  a.scale = scale > 0.f ? scale : 1.f / sqrtf((float)d);
  a.alpha = plan->qjl_alpha;
  a.part = part;
  const size_t smem = sizeof(float) * (a.G * (d + m) + kMaxLevels * 3 * kTab + kThreads * (d + 1) +
                                       2 * a.G * kThreads + 6 * kMaxG) +
                      sizeof(uint32_t) * kThreads * (m / 32);
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(polar_split_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return TQ_ERR_CUDA;
  polar_split_kernel<<<dim3(ps.nsplit, B * Hkv), kThreads, smem, cs>>>(a);
  if ((rc = tq::launch_status()) != TQ_OK) return rc;
  return tq::launch_decode_combine(part, B, Hq, ps.nsplit, d, m, plan->pi_t, plan->s_rot_t, plan->qjl_alpha, out, cs);
}

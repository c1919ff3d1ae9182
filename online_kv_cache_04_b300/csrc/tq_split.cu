// Outlier-channel split precision: quantize and decode attention over two
// TurboQuant instances that share one head ("TurboQuant压缩效果", the 2.5 and
// 3.5-bit settings: the 128 channels split, the few outlier channels one bit
// higher than the rest, the label being the average).
//
// A permutation of the d channels names the outlier channels perm[0 .. d_o)
// and the regular ones perm[d_o .. d); keys and values have their own (their
// outlier channels differ), the query is split like the keys.  Each side is a complete
// instance with its own plan (its rotation of dimension d_o or d - d_o, its
// codebook, its QJL rows) and its own records, so a key's score is the sum
// of the two estimators
//   s = scale · Σ_side (‖k_side‖⟨Π_side q_side, c_side[idx]⟩
//                       + √(π/2)/m_side ‖r_side‖⟨S_side q_side, σ_side⟩),
// and the output carries each side's Π_sideᵀ(acc_rot + α S̃ᵀ acc_sgn)/l at its
// own channels.  The kernels follow the general decode path (query prep,
// context splits, log-sum-exp combine) with both sides handled in the same
// pass over the tokens: one softmax over the summed scores.
#include <cuda_bf16.h>

#include <algorithm>

#include "tq_internal.h"

namespace {

constexpr int kThreads = 128;   // tokens per chunk == threads per CTA
constexpr int kMaxG = 8;
constexpr int kMaxWordsSide = 16;  // index + sign words of one side's record
constexpr float kLog2e = 1.4426950408889634f;

struct Side {
  int d, m, w;
  const float* pi;       // [d][d]
  const float* s_rot;    // [m][d]
  const float* pi_t;     // [d][d]
  const float* s_rot_t;  // [d][m]
  const float* centroids;
  float alpha;
  const int32_t* cols;   // device: this side's channels of the head
};

struct Shape2 {
  int B, Hq, Hkv, G;
  int64_t ctx_stride;
  int nsplit;
  int64_t tokens_per_split;
  int dt, mt;            // d_o + d_r, m_o + m_r
};

int choose_splits(int B, int Hkv, int64_t ctx_stride) {
  const int64_t units = int64_t(B) * Hkv;
  const int64_t want = tq::cdiv(2 * int64_t(tq::sm_count()), units);
  const int64_t maxs = std::max<int64_t>(1, tq::cdiv(ctx_stride, 2 * kThreads));
  return (int)std::max<int64_t>(1, std::min(want, maxs));
}

// ---------------------------------------------------------------- prep
// q̃_side = Π_side q[cols_side], s̃_side = S̃_side q̃_side for one query head per
// CTA; one warp per output row at a time, lanes across the row.
template <typename T>
__global__ void __launch_bounds__(256) prep2_kernel(const T* __restrict__ q, int d, Side o, Side r, float* qt,
                                                    float* st) {
  extern __shared__ float sm[];
  const int head = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  const int dt = o.d + r.d, mt = o.m + r.m;
  float* qs = sm;          // [dt] gathered query, side o then side r
  float* qr = qs + dt;     // [dt] rotated
  for (int j = threadIdx.x; j < dt; j += blockDim.x) {
    const int c = j < o.d ? o.cols[j] : r.cols[j - o.d];
    if constexpr (sizeof(T) == 2) qs[j] = __bfloat162float(q[(size_t)head * d + c]);
    else qs[j] = q[(size_t)head * d + c];
  }
  __syncthreads();
  auto rows = [&](const float* A, int n, int k, const float* x, float* out) {
    for (int row = warp; row < n; row += nw) {
      float s = 0.f;
      for (int c = lane; c < k; c += 32) s = fmaf(__ldg(A + (size_t)row * k + c), x[c], s);
#pragma unroll
      for (int sh = 16; sh > 0; sh >>= 1) s += __shfl_xor_sync(0xffffffffu, s, sh);
      if (lane == 0) out[row] = s;
    }
  };
  rows(o.pi, o.d, o.d, qs, qr);
  rows(r.pi, r.d, r.d, qs + o.d, qr + o.d);
  __syncthreads();
  for (int j = threadIdx.x; j < dt; j += blockDim.x) qt[(size_t)head * dt + j] = qr[j];
  float* sv = st + (size_t)head * mt;
  rows(o.s_rot, o.m, o.d, qr, sv);
  rows(r.s_rot, r.m, r.d, qr + o.d, sv + o.m);
}

struct Split2Args {
  Shape2 s;
  Side side[2];
  const uint32_t* kidx[2]; const uint32_t* ksgn[2]; const float* knorm[2]; const float* krnorm[2];
  const uint32_t* vidx[2]; const uint32_t* vsgn[2]; const float* vnorm[2]; const float* vrnorm[2];
  const int32_t* ctx_len;
  const float* qt; const float* st;   // [B*Hq][dt], [B*Hq][mt]
  float scale;
  float* part;                         // [B*Hq][nsplit][2 + dt + mt]
};

// index of coordinate j of side p from a record's words (bit-planes of 32-coordinate words)
__device__ __forceinline__ int index_of(const uint32_t* words, int w, int d, int j) {
  int idx = 0;
  for (int p = 0; p < w; ++p) idx |= ((words[p * (d / 32) + (j >> 5)] >> (j & 31)) & 1) << p;
  return idx;
}

__global__ void __launch_bounds__(kThreads) split2_kernel(Split2Args a) {
  extern __shared__ float sm[];
  const Shape2& s = a.s;
  const int G = s.G, dt = s.dt, mt = s.mt;
  const Side& so = a.side[0];
  const Side& sr = a.side[1];
  const int wr[2] = {(so.w * so.d + so.m) / 32, (sr.w * sr.d + sr.m) / 32};
  float* qts = sm;                     // [G][dt]
  float* sts = qts + G * dt;           // [G][mt]
  float* cent = sts + G * mt;          // [2][8]
  float* pw = cent + 16;               // [4][G][kThreads]: p·‖v_o‖, p·‖r_vo‖, p·‖v_r‖, p·‖r_vr‖
  float* red = pw + 4 * G * kThreads;  // [4][kMaxG]
  float* runm = red + 4 * kMaxG;       // [kMaxG]
  float* corr = runm + kMaxG;          // [kMaxG]
  uint32_t* vw = reinterpret_cast<uint32_t*>(corr + kMaxG);  // [kThreads][wr0 + wr1]

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int bh = blockIdx.y, b = bh / s.Hkv, h = bh - b * s.Hkv, split = blockIdx.x;
  const int64_t L = min((int64_t)max(__ldg(a.ctx_len + b), 0), s.ctx_stride);
  const int64_t t0 = split * s.tokens_per_split;
  const int64_t t1 = min(t0 + s.tokens_per_split, L);
  const int head0 = b * s.Hq + h * G;
  for (int e = tid; e < G * dt; e += kThreads) qts[e] = a.qt[(size_t)head0 * dt + e];
  for (int e = tid; e < G * mt; e += kThreads) sts[e] = a.st[(size_t)head0 * mt + e];
  if (tid < 16) {
    const Side& sd = tid < 8 ? so : sr;
    cent[tid] = (tid & 7) < (1 << sd.w) ? sd.centroids[tid & 7] : 0.f;
  }
  if (tid < kMaxG) runm[tid] = -INFINITY;
  __syncthreads();

  const int64_t rowbase = (int64_t)bh * s.ctx_stride;
  float acc_r[2][kMaxG], acc_s[2][kMaxG], lsum[kMaxG];
#pragma unroll
  for (int k = 0; k < 2; ++k)
#pragma unroll
    for (int g = 0; g < kMaxG; ++g) acc_r[k][g] = acc_s[k][g] = 0.f;
#pragma unroll
  for (int g = 0; g < kMaxG; ++g) lsum[g] = 0.f;

  for (int64_t c0 = t0; c0 < t1; c0 += kThreads) {
    const int64_t t = c0 + tid;
    const bool valid = t < t1;
    const int cnt = (int)min((int64_t)kThreads, t1 - c0);
    float sc[kMaxG];
#pragma unroll
    for (int g = 0; g < kMaxG; ++g) sc[g] = valid ? 0.f : -INFINITY;
    if (valid) {
      const int64_t row = rowbase + t;
      for (int p = 0; p < 2; ++p) {
        const Side& sd = a.side[p];
        const int wi = sd.w * sd.d / 32, ws = sd.m / 32;
        uint32_t words[kMaxWordsSide];
#pragma unroll
        for (int k = 0; k < kMaxWordsSide; ++k)
          if (k < wi) words[k] = __ldg(a.kidx[p] + row * wi + k);
        float d1[kMaxG], d2[kMaxG];
#pragma unroll
        for (int g = 0; g < kMaxG; ++g) d1[g] = d2[g] = 0.f;
        const int qoff = p == 0 ? 0 : so.d, soff = p == 0 ? 0 : so.m;
        for (int j = 0; j < sd.d; ++j) {
          const float c = cent[8 * p + index_of(words, sd.w, sd.d, j)];
#pragma unroll
          for (int g = 0; g < kMaxG; ++g)
            if (g < G) d1[g] = fmaf(qts[g * dt + qoff + j], c, d1[g]);
        }
        for (int k = 0; k < ws; ++k) {
          const uint32_t word = __ldg(a.ksgn[p] + row * ws + k);
          for (int bb = 0; bb < 32; ++bb) {
            const float sg = ((word >> bb) & 1) ? 1.f : -1.f;
#pragma unroll
            for (int g = 0; g < kMaxG; ++g)
              if (g < G) d2[g] = fmaf(sts[g * mt + soff + k * 32 + bb], sg, d2[g]);
          }
        }
        const float nk = __ldg(a.knorm[p] + row), rk = __ldg(a.krnorm[p] + row);
#pragma unroll
        for (int g = 0; g < kMaxG; ++g)
          if (g < G) sc[g] = fmaf(a.scale, nk * d1[g] + sd.alpha * rk * d2[g], sc[g]);
      }
    }
    // chunk max per head, log2 domain
#pragma unroll
    for (int g = 0; g < kMaxG; ++g) {
      float v = sc[g] * kLog2e;
      sc[g] = v;
      for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
      if (lane == 0 && g < G) red[warp * kMaxG + g] = v;
    }
    // this chunk's value records: token tid's words of side 0 then side 1
    if (valid) {
      const int64_t row = rowbase + t;
      int off = 0;
      for (int p = 0; p < 2; ++p) {
        const Side& sd = a.side[p];
        const int wi = sd.w * sd.d / 32, ws = sd.m / 32;
        for (int k = 0; k < wi; ++k) vw[tid * (wr[0] + wr[1]) + off + k] = __ldg(a.vidx[p] + row * wi + k);
        for (int k = 0; k < ws; ++k) vw[tid * (wr[0] + wr[1]) + off + wi + k] = __ldg(a.vsgn[p] + row * ws + k);
        off += wi + ws;
      }
    }
    __syncthreads();
    if (tid < G) {
      const float cm = fmaxf(fmaxf(red[tid], red[kMaxG + tid]), fmaxf(red[2 * kMaxG + tid], red[3 * kMaxG + tid]));
      const float nm = fmaxf(runm[tid], cm);
      corr[tid] = nm == -INFINITY ? 1.f : exp2f(runm[tid] - nm);  // runm = -inf on the first chunk -> 0
      runm[tid] = nm;
    }
    __syncthreads();
    float nv[4];
    for (int p = 0; p < 2; ++p) {
      nv[2 * p] = valid ? __ldg(a.vnorm[p] + rowbase + t) : 0.f;
      nv[2 * p + 1] = valid ? __ldg(a.vrnorm[p] + rowbase + t) : 0.f;
    }
    for (int g = 0; g < G; ++g) {
      const float pg = valid && runm[g] != -INFINITY ? exp2f(sc[g] - runm[g]) : 0.f;
#pragma unroll
      for (int k = 0; k < 4; ++k) pw[(k * G + g) * kThreads + tid] = pg * nv[k];
      float ps = pg;
      for (int o = 16; o > 0; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
      if (lane == 0) red[warp * kMaxG + g] = ps;
    }
    __syncthreads();
#pragma unroll
    for (int g = 0; g < kMaxG; ++g)
      if (g < G) lsum[g] = lsum[g] * corr[g] + (red[g] + red[kMaxG + g] + red[2 * kMaxG + g] + red[3 * kMaxG + g]);
    // value accumulation: thread owns rotated coordinates j = tid, tid + 128 of
    // side 0 then side 1, and sign coordinates likewise
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int j = tid + k * kThreads;
#pragma unroll
      for (int g = 0; g < kMaxG; ++g) {
        acc_r[k][g] *= corr[g < G ? g : 0];
        acc_s[k][g] *= corr[g < G ? g : 0];
      }
      if (j < dt) {
        const int p = j < so.d ? 0 : 1;
        const Side& sd = a.side[p];
        const int jl = p == 0 ? j : j - so.d, off = p == 0 ? 0 : wr[0];
        for (int tt = 0; tt < cnt; ++tt) {
          const float c = cent[8 * p + index_of(vw + tt * (wr[0] + wr[1]) + off, sd.w, sd.d, jl)];
#pragma unroll
          for (int g = 0; g < kMaxG; ++g)
            if (g < G) acc_r[k][g] = fmaf(pw[(2 * p * G + g) * kThreads + tt], c, acc_r[k][g]);
        }
      }
      if (j < mt) {
        const int p = j < so.m ? 0 : 1;
        const Side& sd = a.side[p];
        const int jl = p == 0 ? j : j - so.m;
        const int off = (p == 0 ? 0 : wr[0]) + sd.w * sd.d / 32;
        for (int tt = 0; tt < cnt; ++tt) {
          const uint32_t sw = vw[tt * (wr[0] + wr[1]) + off + (jl >> 5)] >> (jl & 31);
          const float sg = (sw & 1) ? 1.f : -1.f;
#pragma unroll
          for (int g = 0; g < kMaxG; ++g)
            if (g < G) acc_s[k][g] = fmaf(pw[((2 * p + 1) * G + g) * kThreads + tt], sg, acc_s[k][g]);
        }
      }
    }
    __syncthreads();
  }
  const int stride = 2 + dt + mt;
  for (int g = 0; g < G; ++g) {
    float* pp = a.part + ((size_t)(head0 + g) * s.nsplit + split) * stride;
    if (tid == 0) {
      pp[0] = runm[g];
      pp[1] = lsum[g];
    }
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int j = tid + k * kThreads;
      if (j < dt) pp[2 + j] = acc_r[k][g];
      if (j < mt) pp[2 + dt + j] = acc_s[k][g];
    }
  }
}

// Log-sum-exp merge of the splits of one query head, then each side's
// o_side = Π_sideᵀ(acc_rot + α_side S̃_sideᵀ acc_sgn) / l, written at the
// side's channels.
__global__ void __launch_bounds__(256) combine2_kernel(Shape2 s, Side so, Side sr, const float* part, int d,
                                                       float* out) {
  extern __shared__ float sm[];
  const int dt = s.dt, mt = s.mt, stride = 2 + dt + mt, ns = s.nsplit;
  const int head = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  float* acc = sm;            // [dt + mt]
  float* y = acc + dt + mt;   // [dt]
  float* wgt = y + dt;        // [ns]
  __shared__ float lsum;
  const float* pp = part + (size_t)head * ns * stride;
  if (threadIdx.x < 32) {
    float mx = -INFINITY;
    for (int k = lane; k < ns; k += 32) mx = fmaxf(mx, pp[(size_t)k * stride]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float l = 0.f;
    for (int k = lane; k < ns; k += 32) {
      const float mk = pp[(size_t)k * stride];
      const float wk = mk == -INFINITY ? 0.f : exp2f(mk - mx);
      wgt[k] = wk;
      l = fmaf(wk, pp[(size_t)k * stride + 1], l);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
    if (lane == 0) lsum = l;
  }
  __syncthreads();
  for (int j = threadIdx.x; j < dt + mt; j += blockDim.x) {
    float v = 0.f;
    for (int k = 0; k < ns; ++k) v = wgt[k] != 0.f ? fmaf(wgt[k], pp[(size_t)k * stride + 2 + j], v) : v;
    acc[j] = v;
  }
  __syncthreads();
  // y_side[j] = acc_rot_side[j] + α_side Σ_i S̃_sideᵀ[j][i] acc_sgn_side[i]
  for (int p = 0; p < 2; ++p) {
    const Side& sd = p == 0 ? so : sr;
    const int roff = p == 0 ? 0 : so.d, soff = dt + (p == 0 ? 0 : so.m);
    for (int row = warp; row < sd.d; row += nw) {
      float v = 0.f;
      for (int c = lane; c < sd.m; c += 32) v = fmaf(__ldg(sd.s_rot_t + (size_t)row * sd.m + c), acc[soff + c], v);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0) y[roff + row] = fmaf(sd.alpha, v, acc[roff + row]);
    }
  }
  __syncthreads();
  const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
  for (int p = 0; p < 2; ++p) {
    const Side& sd = p == 0 ? so : sr;
    const int roff = p == 0 ? 0 : so.d;
    for (int row = warp; row < sd.d; row += nw) {
      float v = 0.f;
      for (int c = lane; c < sd.d; c += 32) v = fmaf(__ldg(sd.pi_t + (size_t)row * sd.d + c), y[roff + c], v);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0) out[(size_t)head * d + sd.cols[row]] = v * inv;
    }
  }
}

Side side_of(const tq_plan* p, const int32_t* cols) {
  Side s{};
  s.d = p->d; s.m = p->m; s.w = p->w;
  s.pi = p->pi; s.s_rot = p->s_rot; s.pi_t = p->pi_t; s.s_rot_t = p->s_rot_t;
  s.centroids = p->centroids;
  s.alpha = p->qjl_alpha;
  s.cols = cols;
  return s;
}

// The two plans of one split: both with QJL rows, each side at most 128
// channels wide, the widths adding up to d <= 256.
bool valid_pair(const tq_plan* po, const tq_plan* pr) {
  return tq::valid_plan(po) && tq::valid_plan(pr) && po->m > 0 && pr->m > 0 && po->d <= 128 && pr->d <= 128 &&
         po->m <= 128 && pr->m <= 128 && (po->w * po->d + po->m) / 32 <= kMaxWordsSide &&
         (pr->w * pr->d + pr->m) / 32 <= kMaxWordsSide;
}

bool fill_shape2(const tq_plan* po, const tq_plan* pr, int B, int Hq, int Hkv, int64_t ctx_stride, Shape2* s) {
  if (!valid_pair(po, pr) || B < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || Hq / Hkv > kMaxG || ctx_stride < 1)
    return false;
  s->B = B; s->Hq = Hq; s->Hkv = Hkv; s->G = Hq / Hkv;
  s->ctx_stride = ctx_stride;
  s->nsplit = choose_splits(B, Hkv, ctx_stride);
  s->tokens_per_split = tq::cdiv(tq::cdiv(ctx_stride, s->nsplit), kThreads) * kThreads;
  s->dt = po->d + pr->d;
  s->mt = po->m + pr->m;
  return true;
}

size_t ws_floats2(const Shape2& s) {
  const size_t heads = size_t(s.B) * s.Hq;
  return heads * (s.dt + s.mt) + heads * s.nsplit * (2 + s.dt + s.mt);
}

bool rows_records(const tq_records* r, const tq_plan* p, int64_t rows) {
  return tq::valid_records(r, p) && r->layout == TQ_LAYOUT_ROWS && r->capacity >= rows;
}

}  // namespace

extern "C" tq_status tq_quantize_split(const tq_plan* plan_o, const tq_plan* plan_r, const int32_t* perm,
                                       const void* x, tq_dtype dtype, int64_t n, int64_t ld_x,
                                       const tq_records* out_o, const tq_records* out_r, int64_t out_offset,
                                       tq_stream stream) {
  if (!valid_pair(plan_o, plan_r) || !perm || n < 0 || out_offset < 0) return TQ_ERR_ARG;
  if (dtype != TQ_F32 && dtype != TQ_BF16) return TQ_ERR_ARG;
  if (!rows_records(out_o, plan_o, 0) || !rows_records(out_r, plan_r, 0)) return TQ_ERR_ARG;
  if (n == 0) return TQ_OK;
  const int d = plan_o->d + plan_r->d;
  if (x == nullptr || !tq::aligned16(x) || ld_x < d || ld_x % 8 != 0) return TQ_ERR_ARG;
  for (const tq_records* o : {out_o, out_r})
    if (out_offset > o->capacity || n > o->capacity - out_offset) return TQ_ERR_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  tq_status s = tq::quantize_simt_cols(plan_o, x, dtype, n, ld_x, perm, out_o, out_offset, st);
  if (s != TQ_OK) return s;
  return tq::quantize_simt_cols(plan_r, x, dtype, n, ld_x, perm + plan_o->d, out_r, out_offset, st);
}

extern "C" tq_status tq_decode_split_workspace_size(const tq_plan* plan_o, const tq_plan* plan_r, int B, int Hq,
                                                    int Hkv, int64_t ctx_stride, size_t* bytes) {
  Shape2 s;
  if (!bytes || !fill_shape2(plan_o, plan_r, B, Hq, Hkv, ctx_stride, &s)) return TQ_ERR_ARG;
  *bytes = sizeof(float) * ws_floats2(s);
  return TQ_OK;
}

extern "C" tq_status tq_decode_attention_split(const tq_plan* plan_o, const tq_plan* plan_r, const int32_t* perm_k,
                                               const int32_t* perm_v, const void* q, tq_dtype q_dtype, int B, int Hq, int Hkv,
                                               const tq_records* K_o, const tq_records* K_r, const tq_records* V_o,
                                               const tq_records* V_r, const int32_t* ctx_len, int64_t ctx_stride,
                                               float scale, float* out, void* workspace, size_t ws_bytes,
                                               tq_stream stream) {
  Shape2 s;
  if (!fill_shape2(plan_o, plan_r, B, Hq, Hkv, ctx_stride, &s)) return TQ_ERR_ARG;
  if (!perm_k || !perm_v || !q || !ctx_len || !tq::aligned16(q) || (q_dtype != TQ_F32 && q_dtype != TQ_BF16))
    return TQ_ERR_ARG;
  const int64_t rows = int64_t(B) * Hkv * ctx_stride;
  if (!rows_records(K_o, plan_o, rows) || !rows_records(V_o, plan_o, rows) || !rows_records(K_r, plan_r, rows) ||
      !rows_records(V_r, plan_r, rows))
    return TQ_ERR_ARG;
  if (!out || !tq::aligned16(out) || !workspace || !tq::aligned16(workspace)) return TQ_ERR_ARG;
  if (ws_bytes < sizeof(float) * ws_floats2(s)) return TQ_ERR_WORKSPACE;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  const int d = s.dt;
  // the query is split like the keys, the output is assembled like the values
  const Side so = side_of(plan_o, perm_k), sr = side_of(plan_r, perm_k + plan_o->d);
  const Side vo = side_of(plan_o, perm_v), vr = side_of(plan_r, perm_v + plan_o->d);
  float* qt = static_cast<float*>(workspace);
  float* st = qt + size_t(B) * Hq * s.dt;
  float* part = st + size_t(B) * Hq * s.mt;
  const size_t psmem = sizeof(float) * 2 * s.dt;
  if (q_dtype == TQ_F32)
    prep2_kernel<float><<<B * Hq, 256, psmem, cs>>>(static_cast<const float*>(q), d, so, sr, qt, st);
  else
    prep2_kernel<__nv_bfloat16><<<B * Hq, 256, psmem, cs>>>(static_cast<const __nv_bfloat16*>(q), d, so, sr, qt, st);
  tq_status rc = tq::launch_status();
  if (rc != TQ_OK) return rc;
  Split2Args a{};
  a.s = s;
  a.side[0] = so;
  a.side[1] = sr;
  const tq_records* Ks[2] = {K_o, K_r};
  const tq_records* Vs[2] = {V_o, V_r};
  for (int p = 0; p < 2; ++p) {
    a.kidx[p] = Ks[p]->idx; a.ksgn[p] = Ks[p]->sgn; a.knorm[p] = Ks[p]->norm; a.krnorm[p] = Ks[p]->rnorm;
    a.vidx[p] = Vs[p]->idx; a.vsgn[p] = Vs[p]->sgn; a.vnorm[p] = Vs[p]->norm; a.vrnorm[p] = Vs[p]->rnorm;
  }
  a.ctx_len = ctx_len;
  a.qt = qt;
  a.st = st;
  a.scale = scale > 0.f ? scale : 1.f / sqrtf((float)d);
  a.part = part;
  const int wr = (plan_o->w * plan_o->d + plan_o->m + plan_r->w * plan_r->d + plan_r->m) / 32;
  const size_t smem = sizeof(float) * (s.G * (s.dt + s.mt) + 16 + 4 * s.G * kThreads + 6 * kMaxG) +
                      sizeof(uint32_t) * kThreads * wr;
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(split2_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return TQ_ERR_CUDA;
  split2_kernel<<<dim3(s.nsplit, B * Hkv), kThreads, smem, cs>>>(a);
  if ((rc = tq::launch_status()) != TQ_OK) return rc;
  combine2_kernel<<<B * Hq, 256, sizeof(float) * (2 * s.dt + s.mt + s.nsplit), cs>>>(s, vo, vr, part, d, out);
  return tq::launch_status();
}

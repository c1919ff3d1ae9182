// tq_decode_attention / tq_decode_scores: one GQA decode step over the
// compressed cache, computed directly on the packed records.
//
// Score of key t for query head g ("TurboQuant 与 AI 效率革命" §三, the
// asymmetric QJL estimator, applied to the residual as in
// "谷歌TurboQuant如何绕过内存墙？" §2 stage 2):
//   s = scale · ( ||k|| <q̃, c[idx]> + √(π/2)/m ||r|| <s̃, σ> ),  q̃ = Π q, s̃ = S q.
// Softmax is online (running max and sum per head); the value side is
// accumulated in the rotated domain, acc_rot = Σ p ||v|| c[idx] and
// acc_sgn = Σ p ||r_v|| σ, and one final Πᵀ (S Πᵀ)ᵀ fold gives
// o = Πᵀ (acc_rot + √(π/2)/m (S Πᵀ)ᵀ acc_sgn) / l.  No dequantized K or V is
// ever written ("TurboQuant压缩效果": decode in registers while reading).
//
// Kernels of the general path (any d, m; the d = m = 128 value-block case runs
// as one launch of the tensor-core kernel in tq_decode_tc.cu instead):
//   prep     q̃ = Π q and s̃ = (S Πᵀ) q̃ per query head -> workspace
//   split    grid (splits, B*Hkv): streams one context slice of one kv head
//            for its G query heads, writes (max, sum, acc) partials
//   combine  grid (B*Hq): log-sum-exp merge of the splits, fold, unrotate
#include <cuda_bf16.h>

#include <algorithm>

#include "tq_internal.h"

namespace {

constexpr int kThreads = 128;     // tokens per chunk == threads per CTA
constexpr int kMaxG = 8;          // query heads per kv head
constexpr int kMaxWords = 32;     // index + sign words of one record (d, m <= 256)
constexpr float kLog2e = 1.4426950408889634f;

struct DecodeShape {
  int B, Hq, Hkv, G, d, m, w;
  int64_t ctx_stride;
  int nsplit;
  int64_t tokens_per_split;
};

int choose_splits(int B, int Hkv, int64_t ctx_stride) {
  const int64_t units = int64_t(B) * Hkv;
  const int64_t want = tq::cdiv(2 * int64_t(tq::sm_count()), units);
  const int64_t maxs = std::max<int64_t>(1, tq::cdiv(ctx_stride, 2 * kThreads));
  return (int)std::max<int64_t>(1, std::min(want, maxs));
}

// Partial slots per head of the tensor-core path (0 when it cannot apply).
int tc_slots(const DecodeShape& s) {
  if (s.d != 128 || (s.m != 128 && s.m != 0) || s.G > kMaxG || s.ctx_stride % 128 != 0) return 0;
  const int64_t units = int64_t(s.B) * s.Hkv, tpu = tq::decode_tc_tpu(s.ctx_stride);
  return tq::decode_tc_slots(units, tpu, tq::decode_tc_ctas(units, tpu, s.G));
}

// Workspace of the tensor-core path: the per-unit query tables, then the
// partials (byte offsets, 256-byte aligned).
struct TcLayout {
  size_t tables, part, bytes;
};
TcLayout tc_layout(const DecodeShape& s) {
  auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
  const size_t units = size_t(s.B) * s.Hkv, heads = size_t(s.B) * s.Hq;
  TcLayout l;
  l.tables = 0;
  l.part = up(l.tables + units * tq::decode_tc_table_bytes(s.w, s.G, s.m));
  l.bytes = l.part + sizeof(float) * heads * tc_slots(s) * (2 + 2 * s.d);  // reference, sum, acc_rot, acc_sgn
  return l;
}

// Workspace: the general path's q̃ and s̃ per query head and split partials,
// or the tensor-core path's layout, whichever is larger.
size_t ws_floats(const DecodeShape& s) {
  const size_t heads = size_t(s.B) * s.Hq;
  const size_t general = heads * (s.d + s.m) + heads * s.nsplit * (2 + s.d + s.m);
  return tc_slots(s) > 0 ? std::max(general, (tc_layout(s).bytes + 3) / 4) : general;
}

bool fill_shape(const tq_plan* plan, int B, int Hq, int Hkv, int64_t ctx_stride, DecodeShape* s) {
  if (!tq::valid_plan(plan) || B < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || ctx_stride < 1) return false;
  s->B = B;
  s->Hq = Hq;
  s->Hkv = Hkv;
  s->G = Hq / Hkv;
  s->d = plan->d;
  s->m = plan->m;
  s->w = plan->w;
  s->ctx_stride = ctx_stride;
  s->nsplit = choose_splits(B, Hkv, ctx_stride);
  s->tokens_per_split = tq::cdiv(tq::cdiv(ctx_stride, s->nsplit), kThreads) * kThreads;
  return true;
}

bool supported(const DecodeShape& s) {
  return s.G <= kMaxG && s.d <= 256 && s.m <= 256 && (s.w * s.d + s.m) / 32 <= kMaxWords;
}

// ---------------------------------------------------------------- prep
// out[r] = Σ_{c<k} A[r·lda + c]·x[c] for r < n (A row-major, rows contiguous),
// by all warps of the block: a warp takes 16 rows at once, each lane reads
// 4 consecutive columns of each row with one 128-bit load (all 16 loads in
// flight together), and the 16 dot products are reduced across the warp.
// x and out live in shared memory, 16-byte aligned; k is a multiple of 4 and
// lda of 4.  Ends with the block synchronised.
__device__ __forceinline__ void block_rowdot(const float* __restrict__ A, int lda, int n, int k, const float* x,
                                             float* out) {
  constexpr int R = 16;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  for (int r0 = warp * R; r0 < n; r0 += nw * R) {
    float acc[R];
#pragma unroll
    for (int q = 0; q < R; ++q) acc[q] = 0.f;
    for (int c = 4 * lane; c < k; c += 128) {
      const float4 xv = *reinterpret_cast<const float4*>(x + c);
#pragma unroll
      for (int q = 0; q < R; ++q) {
        if (r0 + q < n) {
          const float4 av = __ldg(reinterpret_cast<const float4*>(A + (size_t)(r0 + q) * lda + c));
          acc[q] = fmaf(av.x, xv.x, fmaf(av.y, xv.y, fmaf(av.z, xv.z, fmaf(av.w, xv.w, acc[q]))));
        }
      }
    }
#pragma unroll
    for (int q = 0; q < R; ++q) {
      float v = acc[q];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0 && r0 + q < n) out[r0 + q] = v;
    }
  }
  __syncthreads();
}

template <typename T>
__global__ void __launch_bounds__(256) prep_kernel(const T* __restrict__ q, const float* __restrict__ pi,
                                                   const float* __restrict__ s_rot, int d, int m,
                                                   float* __restrict__ qt, float* __restrict__ st) {
  extern __shared__ float sm[];
  float* qs = sm;           // [d]
  float* qr = qs + d;       // [d]   Π q
  float* sr = qr + d;       // [m]   S q = (S Πᵀ) Π q
  const int head = blockIdx.x;
  for (int i = threadIdx.x; i < d; i += blockDim.x) {
    if constexpr (sizeof(T) == 2) qs[i] = __bfloat162float(q[(size_t)head * d + i]);
    else qs[i] = q[(size_t)head * d + i];
  }
  __syncthreads();
  block_rowdot(pi, d, d, d, qs, qr);  // row j of Π
  for (int j = threadIdx.x; j < d; j += blockDim.x) qt[(size_t)head * d + j] = qr[j];
  block_rowdot(s_rot, d, m, d, qr, sr);  // row i of S Πᵀ
  for (int j = threadIdx.x; j < m; j += blockDim.x) st[(size_t)head * m + j] = sr[j];
}

struct SplitArgs {
  DecodeShape s;
  int v_layout;                        // tq_layout of the value records
  const uint32_t* kidx; const uint32_t* ksgn; const float* knorm; const float* krnorm;
  const uint32_t* vidx; const uint32_t* vsgn; const float* vnorm; const float* vrnorm;
  const int32_t* ctx_len;
  const float* qt; const float* st;   // [B*Hq][d], [B*Hq][m]
  const float* centroids;
  float scale, alpha;
  float* part;                         // [B*Hq][nsplit][2 + d + m]
  float* scores;                       // scores-only mode: [B*Hq][ctx_stride]
  const int32_t* pages;                // paged caches: [B*Hkv][max_pages] (NULL: contiguous rows)
  int64_t max_pages, npages;           // pages per unit; pages the record arrays hold
  unsigned* fault;
};

constexpr int kPage = 256;             // tokens per page of a paged cache
constexpr unsigned kFaultPage = 16u;   // a page-table entry outside the record arrays

// Record row of token t of unit bh: contiguous units, or through the page table
// (an entry outside the record arrays reads page 0 and raises kFaultPage).
__device__ __forceinline__ int64_t row_of(const SplitArgs& a, int64_t bh, int64_t t) {
  if (a.pages == nullptr) return bh * a.s.ctx_stride + t;
  int64_t pg = __ldg(a.pages + bh * a.max_pages + t / kPage);
  if (pg < 0 || pg >= a.npages) {
    atomicOr(a.fault, kFaultPage);
    pg = 0;
  }
  return pg * kPage + t % kPage;
}

// score of one token for all G heads (thread-private record in registers)
__device__ __forceinline__ void score_token(const SplitArgs& a, int64_t row, const float* qts, const float* sts,
                                            const float* cent, int G, float* out) {
  const int d = a.s.d, m = a.s.m, w = a.s.w, wi = w * d / 32, ws = m / 32;
  uint32_t words[kMaxWords];
  const uint32_t* ip = a.kidx + row * wi;
#pragma unroll
  for (int k = 0; k < kMaxWords; ++k)
    if (k < wi) words[k] = __ldg(ip + k);
  float d1[kMaxG], d2[kMaxG];
#pragma unroll
  for (int g = 0; g < kMaxG; ++g) d1[g] = d2[g] = 0.0f;
  for (int j = 0; j < d; ++j) {
    int idx = 0;
    for (int p = 0; p < w; ++p) idx |= ((words[p * (d / 32) + (j >> 5)] >> (j & 31)) & 1) << p;
    const float c = cent[idx];
#pragma unroll
    for (int g = 0; g < kMaxG; ++g)
      if (g < G) d1[g] = fmaf(qts[g * d + j], c, d1[g]);
  }
  const uint32_t* sp = a.ksgn + row * ws;
  for (int k = 0; k < ws; ++k) {
    const uint32_t word = __ldg(sp + k);
    for (int b = 0; b < 32; ++b) {
      const float sg = ((word >> b) & 1) ? 1.0f : -1.0f;
#pragma unroll
      for (int g = 0; g < kMaxG; ++g)
        if (g < G) d2[g] = fmaf(sts[g * m + k * 32 + b], sg, d2[g]);
    }
  }
  const float nk = __ldg(a.knorm + row), rk = m > 0 ? __ldg(a.krnorm + row) : 0.0f;
#pragma unroll
  for (int g = 0; g < kMaxG; ++g)
    if (g < G) out[g] = a.scale * (nk * d1[g] + a.alpha * rk * d2[g]);
}

template <bool kScoresOnly>
__global__ void __launch_bounds__(kThreads) split_kernel(SplitArgs a) {
  extern __shared__ float sm[];
  const DecodeShape& s = a.s;
  const int d = s.d, m = s.m, w = s.w, G = s.G;
  const int wi = w * d / 32, ws = m / 32, wr = wi + ws;
  float* qts = sm;                     // [G][d]
  float* sts = qts + G * d;            // [G][m]
  float* cent = sts + G * m;           // [8]
  float* pn = cent + 8;                // [G][kThreads]  p·||v||
  float* pr = pn + G * kThreads;       // [G][kThreads]  p·||r_v||
  float* red = pr + G * kThreads;      // [4][G] warp partials
  float* runm = red + 4 * kMaxG;       // [G] running max (log2 domain)
  float* corr = runm + kMaxG;          // [G] rescale of the previous accumulators
  uint32_t* vw = reinterpret_cast<uint32_t*>(corr + kMaxG);  // [kThreads][wr]

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int bh = blockIdx.y, b = bh / s.Hkv, h = bh - b * s.Hkv, split = blockIdx.x;
  const int64_t L = min((int64_t)__ldg(a.ctx_len + b), s.ctx_stride);
  const int64_t t0 = split * s.tokens_per_split;
  const int64_t t1 = min(t0 + s.tokens_per_split, L);
  const int head0 = b * s.Hq + h * G;
  for (int e = tid; e < G * d; e += kThreads) qts[e] = a.qt[(size_t)head0 * d + e];
  for (int e = tid; e < G * m; e += kThreads) sts[e] = a.st[(size_t)head0 * m + e];
  if (tid < 8) cent[tid] = tid < (1 << w) ? a.centroids[tid] : 0.0f;
  if (tid < kMaxG) runm[tid] = -INFINITY;
  __syncthreads();

  float acc_r[2][kMaxG], acc_s[2][kMaxG], lsum[kMaxG];
#pragma unroll
  for (int k = 0; k < 2; ++k)
#pragma unroll
    for (int g = 0; g < kMaxG; ++g) acc_r[k][g] = acc_s[k][g] = 0.0f;
#pragma unroll
  for (int g = 0; g < kMaxG; ++g) lsum[g] = 0.0f;

  for (int64_t c0 = t0; c0 < t1; c0 += kThreads) {
    const int64_t t = c0 + tid;
    const bool valid = t < t1;
    const int cnt = (int)min((int64_t)kThreads, t1 - c0);
    float sc[kMaxG];
#pragma unroll
    for (int g = 0; g < kMaxG; ++g) sc[g] = -INFINITY;
    const int64_t row = valid ? row_of(a, bh, t) : 0;
    if (valid) score_token(a, row, qts, sts, cent, G, sc);
    if constexpr (kScoresOnly) {
      if (valid)
        for (int g = 0; g < G; ++g) a.scores[(size_t)(head0 + g) * s.ctx_stride + t] = sc[g];
      continue;
    } else {
      // chunk max per head, in the log2 domain
#pragma unroll
      for (int g = 0; g < kMaxG; ++g) {
        float v = sc[g] * kLog2e;
        sc[g] = v;
        for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
        if (lane == 0 && g < G) red[warp * kMaxG + g] = v;
      }
      // stage this chunk's value records.  Rows layout: token tid's words at
      // vw[tid*wr ...].  Block layout (c0 is a multiple of 32 and so is the
      // row base): block kb of the chunk at vw[kb*(w*d+m) ...], plane-major
      // index words then sign words, one coordinate per word.
      if (a.v_layout == TQ_LAYOUT_ROWS) {
        if (valid) {
          const uint32_t* ip = a.vidx + row * wi;
          const uint32_t* sp = a.vsgn + row * ws;
          for (int k = 0; k < wi; ++k) vw[tid * wr + k] = __ldg(ip + k);
          for (int k = 0; k < ws; ++k) vw[tid * wr + wi + k] = __ldg(sp + k);
        }
      } else {
        const int nb = (cnt + 31) >> 5, bw = w * d + m;
        const int64_t blk = row_of(a, bh, c0) >> 5;  // a chunk never straddles a page
        for (int e = tid; e < nb * bw; e += kThreads) {
          const int kb = e / bw, o = e - kb * bw;
          vw[e] = o < w * d ? __ldg(a.vidx + (blk + kb) * (int64_t)(w * d) + o)
                            : __ldg(a.vsgn + (blk + kb) * (int64_t)m + (o - w * d));
        }
      }
      __syncthreads();
      if (tid < G) {
        const float cm = fmaxf(fmaxf(red[tid], red[kMaxG + tid]), fmaxf(red[2 * kMaxG + tid], red[3 * kMaxG + tid]));
        const float nm = fmaxf(runm[tid], cm);
        corr[tid] = exp2f(runm[tid] - nm);  // runm = -inf on the first chunk -> 0
        runm[tid] = nm;
      }
      __syncthreads();
      const float nv = valid ? __ldg(a.vnorm + row) : 0.0f;
      const float rv = valid && m > 0 ? __ldg(a.vrnorm + row) : 0.0f;
      for (int g = 0; g < G; ++g) {
        const float p = valid ? exp2f(sc[g] - runm[g]) : 0.0f;
        pn[g * kThreads + tid] = p * nv;
        pr[g * kThreads + tid] = p * rv;
        float ps = p;
        for (int o = 16; o > 0; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
        if (lane == 0) red[warp * kMaxG + g] = ps;
      }
      __syncthreads();
#pragma unroll
      for (int g = 0; g < kMaxG; ++g)
        if (g < G) lsum[g] = lsum[g] * corr[g] + (red[g] + red[kMaxG + g] + red[2 * kMaxG + g] + red[3 * kMaxG + g]);
      // value accumulation: thread owns coordinates j = tid, tid + 128
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int j = tid + k * kThreads;
#pragma unroll
        for (int g = 0; g < kMaxG; ++g) {
          acc_r[k][g] *= corr[g < G ? g : 0];
          acc_s[k][g] *= corr[g < G ? g : 0];
        }
        const bool vrows = a.v_layout == TQ_LAYOUT_ROWS;
        const int bw = w * d + m;
        if (j < d) {
          for (int tt = 0; tt < cnt; ++tt) {
            int idx = 0;
            if (vrows)
              for (int p = 0; p < w; ++p) idx |= ((vw[tt * wr + p * (d / 32) + (j >> 5)] >> (j & 31)) & 1) << p;
            else
              for (int p = 0; p < w; ++p)
                idx |= ((vw[(tt >> 5) * bw + p * d + j] >> tq::block32_bit(tt & 31)) & 1) << p;
            const float c = cent[idx];
#pragma unroll
            for (int g = 0; g < kMaxG; ++g)
              if (g < G) acc_r[k][g] = fmaf(pn[g * kThreads + tt], c, acc_r[k][g]);
          }
        }
        if (j < m) {
          for (int tt = 0; tt < cnt; ++tt) {
            const uint32_t sw = vrows ? vw[tt * wr + wi + (j >> 5)] >> (j & 31)
                                      : vw[(tt >> 5) * bw + w * d + j] >> tq::block32_bit(tt & 31);
            const float sg = (sw & 1) ? 1.0f : -1.0f;
#pragma unroll
            for (int g = 0; g < kMaxG; ++g)
              if (g < G) acc_s[k][g] = fmaf(pr[g * kThreads + tt], sg, acc_s[k][g]);
          }
        }
      }
      __syncthreads();
    }
  }
  if constexpr (!kScoresOnly) {
    const int stride = 2 + d + m;
    for (int g = 0; g < G; ++g) {
      float* pp = a.part + ((size_t)(head0 + g) * s.nsplit + split) * stride;
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
}

struct CombineArgs {
  DecodeShape s;
  const float* part;
  const float* pi_t;      // [d][d] Πᵀ
  const float* s_rot_t;   // [d][m] (S Πᵀ)ᵀ
  float alpha;
  float* out;             // [B*Hq][d]
};

__global__ void __launch_bounds__(256) combine_kernel(CombineArgs a) {
  extern __shared__ float sm[];
  const int d = a.s.d, m = a.s.m, stride = 2 + d + m;
  const int head = blockIdx.x;
  const int ns = a.s.nsplit, pitch = a.s.nsplit;
  float* acc = sm;              // [d + m]
  float* y = acc + d + m;       // [d]
  float* o = y + d;             // [d]
  float* wgt = o + d;           // [ns]
  __shared__ float lsum;
  const float* pp = a.part + (size_t)head * pitch * stride;
  if (threadIdx.x < 32) {
    // slot weights 2^(m_k - max) and l = Σ_k w_k l_k, one slot per lane
    const int lane = threadIdx.x;
    float mx = -INFINITY;
    for (int k = lane; k < ns; k += 32) mx = fmaxf(mx, pp[(size_t)k * stride]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float l = 0.0f;
    for (int k = lane; k < ns; k += 32) {
      const float mk = pp[(size_t)k * stride];
      const float wk = (mk == -INFINITY) ? 0.0f : exp2f(mk - mx);
      wgt[k] = wk;
      l = fmaf(wk, pp[(size_t)k * stride + 1], l);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
    if (lane == 0) lsum = l;
  }
  __syncthreads();
  for (int j = threadIdx.x; j < d + m; j += blockDim.x) {
    float v0 = 0.0f, v1 = 0.0f, v2 = 0.0f, v3 = 0.0f;
    int k = 0;
    // a slot of weight 0 (no token) contributes nothing, whatever it holds
    auto term = [&](int kk, float v) {
      const float x = pp[(size_t)kk * stride + 2 + j];
      return wgt[kk] != 0.0f ? fmaf(wgt[kk], x, v) : v;
    };
    for (; k + 4 <= ns; k += 4) {
      v0 = term(k, v0);
      v1 = term(k + 1, v1);
      v2 = term(k + 2, v2);
      v3 = term(k + 3, v3);
    }
    for (; k < ns; ++k) v0 = term(k, v0);
    acc[j] = (v0 + v1) + (v2 + v3);
  }
  __syncthreads();
  // y = acc_rot + α (S Πᵀ)ᵀ acc_sgn
  block_rowdot(a.s_rot_t, m, d, m, acc + d, y);  // row j of (S Πᵀ)ᵀ
  for (int j = threadIdx.x; j < d; j += blockDim.x) y[j] = fmaf(a.alpha, y[j], acc[j]);
  __syncthreads();
  // o = Πᵀ y / l
  block_rowdot(a.pi_t, d, d, d, y, o);  // row i of Πᵀ
  const float inv = lsum > 0.0f ? 1.0f / lsum : 0.0f;
  for (int i = threadIdx.x; i < d; i += blockDim.x) a.out[(size_t)head * d + i] = o[i] * inv;
}

tq_status check_common(const tq_plan* plan, const void* q, tq_dtype qd, const tq_records* K, const int32_t* ctx_len,
                       const DecodeShape& s) {
  if (!q || !ctx_len || !tq::aligned16(q) || (qd != TQ_F32 && qd != TQ_BF16)) return TQ_ERR_ARG;
  if (!tq::valid_records(K, plan)) return TQ_ERR_ARG;
  if (K->layout != TQ_LAYOUT_ROWS) return TQ_ERR_UNSUPPORTED;
  if (K->capacity / s.ctx_stride < int64_t(s.B) * s.Hkv) return TQ_ERR_ARG;
  if (!supported(s)) return TQ_ERR_UNSUPPORTED;
  (void)plan;
  return TQ_OK;
}

tq_status launch_prep(const tq_plan* plan, const void* q, tq_dtype qd, const DecodeShape& s, float* qt, float* st,
                      cudaStream_t stream) {
  return tq::launch_query_prep(plan, q, qd, s.B * s.Hq, qt, st, stream);
}

size_t split_smem(const DecodeShape& s) {
  const int wr = (s.w * s.d + s.m) / 32;  // words per record: 128 records == 4 blocks of 32
  return sizeof(float) * (s.G * (s.d + s.m) + 8 + 2 * s.G * kThreads + 4 * kMaxG + 2 * kMaxG) +
         sizeof(uint32_t) * kThreads * wr;
}

}  // namespace

tq_status tq::launch_query_prep(const tq_plan* plan, const void* q, tq_dtype qd, int nheads, float* qt, float* st,
                                cudaStream_t stream) {
  const size_t smem = sizeof(float) * (2 * plan->d + plan->m);
  if (qd == TQ_F32)
    prep_kernel<float><<<nheads, 256, smem, stream>>>(static_cast<const float*>(q), plan->pi, plan->s_rot,
                                                      plan->d, plan->m, qt, st);
  else
    prep_kernel<__nv_bfloat16><<<nheads, 256, smem, stream>>>(static_cast<const __nv_bfloat16*>(q), plan->pi,
                                                              plan->s_rot, plan->d, plan->m, qt, st);
  return tq::launch_status();
}

tq_status tq::launch_decode_combine(const float* part, int B, int Hq, int nsplit, int d, int m, const float* pi_t,
                                   const float* s_rot_t, float alpha, float* out, cudaStream_t stream) {
  CombineArgs c{};
  c.s.B = B;
  c.s.Hq = Hq;
  c.s.d = d;
  c.s.m = m;
  c.s.nsplit = nsplit;
  c.part = part;
  c.pi_t = pi_t;
  c.s_rot_t = s_rot_t;
  c.alpha = alpha;
  c.out = out;
  combine_kernel<<<B * Hq, 256, sizeof(float) * (3 * d + m + nsplit), stream>>>(c);
  return tq::launch_status();
}

extern "C" tq_status tq_decode_workspace_size(const tq_plan* plan, int B, int Hq, int Hkv, int64_t ctx_stride,
                                              size_t* bytes) {
  DecodeShape s;
  if (!bytes || !fill_shape(plan, B, Hq, Hkv, ctx_stride, &s)) return TQ_ERR_ARG;
  *bytes = sizeof(float) * ws_floats(s);
  return TQ_OK;
}

namespace {

// app: the fused append of tq_decode_attention_append (NULL: none).  The
// tensor-core path quantizes the new rows inside its launch sequence; the
// general path runs tq_append_kv's launches first.
tq_status decode_impl(const tq_plan* plan, const void* q, tq_dtype q_dtype, int B, int Hq, int Hkv,
                      const tq_records* K, const tq_records* V, const int32_t* ctx_len, int64_t ctx_stride,
                      float scale, float* out, void* workspace, size_t ws_bytes, tq_stream stream,
                      const int32_t* pages, const tq::TcAppend* app = nullptr) {
  DecodeShape s;
  if (!fill_shape(plan, B, Hq, Hkv, ctx_stride, &s)) return TQ_ERR_ARG;
  tq_status st = TQ_OK;
  if (pages == nullptr) {
    if ((st = check_common(plan, q, q_dtype, K, ctx_len, s)) != TQ_OK) return st;
    if (!tq::valid_records(V, plan) || V->capacity / s.ctx_stride < int64_t(B) * Hkv) return TQ_ERR_ARG;
  } else {  // a paged cache: any number of whole pages; the page table names them
    if (!q || !ctx_len || !tq::aligned16(q) || (q_dtype != TQ_F32 && q_dtype != TQ_BF16)) return TQ_ERR_ARG;
    if (!tq::valid_records(K, plan) || !tq::valid_records(V, plan) || K->capacity < kPage || V->capacity < kPage)
      return TQ_ERR_ARG;
    if (K->layout != TQ_LAYOUT_ROWS) return TQ_ERR_UNSUPPORTED;
    if (!supported(s)) return TQ_ERR_UNSUPPORTED;
  }
  if (V->layout == TQ_LAYOUT_BLOCK32 && ctx_stride % 32 != 0) return TQ_ERR_ARG;
  if (!out || !tq::aligned16(out) || !workspace || !tq::aligned16(workspace)) return TQ_ERR_ARG;
  if (ws_bytes < sizeof(float) * ws_floats(s)) return TQ_ERR_WORKSPACE;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  float* qt = static_cast<float*>(workspace);
  float* stv = qt + size_t(B) * Hq * s.d;
  float* part = stv + size_t(B) * Hq * s.m;
  const float sc = scale > 0.0f ? scale : 1.0f / sqrtf((float)s.d);
  if (tq::decode_tc_supported(plan, s.G, V, ctx_stride)) {
    const TcLayout l = tc_layout(s);
    uint8_t* ws8 = static_cast<uint8_t*>(workspace);
    return tq::launch_decode_tc(plan, q, q_dtype, K, V, ctx_len, B, Hq, Hkv, ctx_stride, sc,
                                reinterpret_cast<float*>(ws8 + l.part), tc_slots(s), ws8 + l.tables, out, cs,
                                pages, app);
  }
  if (app != nullptr &&
      (st = tq::append_kv(plan, app->k_new, app->v_new, app->bf16 ? TQ_BF16 : TQ_F32, B, Hkv, K, V, app->ctx_len,
                          ctx_stride, cs, pages)) != TQ_OK)
    return st;
  if ((st = launch_prep(plan, q, q_dtype, s, qt, stv, cs)) != TQ_OK) return st;
  SplitArgs a{};
  a.s = s;
  a.kidx = K->idx; a.ksgn = K->sgn; a.knorm = K->norm; a.krnorm = K->rnorm;
  a.vidx = V->idx; a.vsgn = V->sgn; a.vnorm = V->norm; a.vrnorm = V->rnorm;
  a.v_layout = V->layout;
  a.ctx_len = ctx_len;
  a.qt = qt; a.st = stv;
  a.centroids = plan->centroids;
  a.scale = scale > 0.0f ? scale : 1.0f / sqrtf((float)s.d);
  a.alpha = plan->qjl_alpha;
  a.part = part;
  a.pages = pages;
  a.max_pages = ctx_stride / kPage;
  a.npages = std::min(K->capacity, V->capacity) / kPage;
  a.fault = tq::fault_word();
  if (!a.fault) return TQ_ERR_CUDA;
  const size_t smem = split_smem(s);
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(split_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return TQ_ERR_CUDA;
  split_kernel<false><<<dim3(s.nsplit, B * Hkv), kThreads, smem, cs>>>(a);
  if ((st = tq::launch_status()) != TQ_OK) return st;
  CombineArgs c{};
  c.s = s;
  c.part = part;
  c.pi_t = plan->pi_t;
  c.s_rot_t = plan->s_rot_t;
  c.alpha = plan->qjl_alpha;
  c.out = out;
  combine_kernel<<<B * Hq, 256, sizeof(float) * (3 * s.d + s.m + s.nsplit), cs>>>(c);
  return tq::launch_status();
}

}  // namespace

extern "C" tq_status tq_decode_attention(const tq_plan* plan, const void* q, tq_dtype q_dtype, int B, int Hq, int Hkv,
                                         const tq_records* K, const tq_records* V, const int32_t* ctx_len,
                                         int64_t ctx_stride, float scale, float* out, void* workspace,
                                         size_t ws_bytes, tq_stream stream) {
  return decode_impl(plan, q, q_dtype, B, Hq, Hkv, K, V, ctx_len, ctx_stride, scale, out, workspace, ws_bytes, stream,
                     nullptr);
}

extern "C" tq_status tq_decode_attention_paged(const tq_plan* plan, const void* q, tq_dtype q_dtype, int B, int Hq,
                                               int Hkv, const tq_records* K, const tq_records* V,
                                               const int32_t* ctx_len, const int32_t* pages, int max_pages,
                                               float scale, float* out, void* workspace, size_t ws_bytes,
                                               tq_stream stream) {
  if (pages == nullptr || !tq::aligned16(pages) || max_pages < 1) return TQ_ERR_ARG;
  return decode_impl(plan, q, q_dtype, B, Hq, Hkv, K, V, ctx_len, int64_t(max_pages) * kPage, scale, out, workspace,
                     ws_bytes, stream, pages);
}

extern "C" tq_status tq_decode_attention_append(const tq_plan* plan, const void* q, tq_dtype q_dtype,
                                                const void* k_new, const void* v_new, tq_dtype kv_dtype, int B,
                                                int Hq, int Hkv, const tq_records* K, const tq_records* V,
                                                int32_t* ctx_len, int64_t ctx_stride, const int32_t* pages,
                                                float scale, float* out, void* workspace, size_t ws_bytes,
                                                tq_stream stream) {
  if (!k_new || !v_new || !tq::aligned16(k_new) || !tq::aligned16(v_new) || (kv_dtype != TQ_F32 && kv_dtype != TQ_BF16))
    return TQ_ERR_ARG;
  if (!K || !V || K->idx == V->idx || (K->sgn && K->sgn == V->sgn) || K->norm == V->norm) return TQ_ERR_ARG;
  if (pages != nullptr && (!tq::aligned16(pages) || ctx_stride % kPage != 0)) return TQ_ERR_ARG;
  const tq::TcAppend app{k_new, v_new, kv_dtype == TQ_BF16, ctx_len};
  return decode_impl(plan, q, q_dtype, B, Hq, Hkv, K, V, ctx_len, ctx_stride, scale, out, workspace, ws_bytes, stream,
                     pages, &app);
}

extern "C" tq_status tq_decode_scores(const tq_plan* plan, const void* q, tq_dtype q_dtype, int B, int Hq, int Hkv,
                                      const tq_records* K, const int32_t* ctx_len, int64_t ctx_stride, float scale,
                                      float* scores, void* workspace, size_t ws_bytes, tq_stream stream) {
  DecodeShape s;
  if (!fill_shape(plan, B, Hq, Hkv, ctx_stride, &s)) return TQ_ERR_ARG;
  tq_status st = check_common(plan, q, q_dtype, K, ctx_len, s);
  if (st != TQ_OK) return st;
  if (!scores || !tq::aligned16(scores) || !workspace || !tq::aligned16(workspace)) return TQ_ERR_ARG;
  if (ws_bytes < sizeof(float) * ws_floats(s)) return TQ_ERR_WORKSPACE;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  float* qt = static_cast<float*>(workspace);
  float* stv = qt + size_t(B) * Hq * s.d;
  if ((st = launch_prep(plan, q, q_dtype, s, qt, stv, cs)) != TQ_OK) return st;
  SplitArgs a{};
  a.s = s;
  a.kidx = K->idx; a.ksgn = K->sgn; a.knorm = K->norm; a.krnorm = K->rnorm;
  a.ctx_len = ctx_len;
  a.qt = qt; a.st = stv;
  a.centroids = plan->centroids;
  a.scale = scale > 0.0f ? scale : 1.0f / sqrtf((float)s.d);
  a.alpha = plan->qjl_alpha;
  a.scores = scores;
  const size_t smem = split_smem(s);
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(split_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return TQ_ERR_CUDA;
  split_kernel<true><<<dim3(s.nsplit, B * Hkv), kThreads, smem, cs>>>(a);
  return tq::launch_status();
}

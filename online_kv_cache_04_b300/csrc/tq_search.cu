// tq_search_topk: inner-product top-k over compressed vectors.
//
// The quantizer also serves vector search engines ("TurboQuant压缩效果";
// "谷歌TurboQuant如何绕过内存墙？" §2).  The score of stored vector i for a
// query q is the same unbiased estimator as in attention, without a scale:
//   score_i = ||x_i|| <Π q, c[idx_i]> + √(π/2)/m ||r_i|| <S q, σ_i>.
// The k best are returned in descending order; equal scores go to the lower
// index (the order (score desc, index asc) is total, so selection is exact).
//
// Kernels: query prep (shared with decode); for d a multiple of 256 (m = d or
// 0) and k <= 16, the tcgen05 kernel of tq_search_wide.cu; otherwise, when d
// and m are multiples of 128, the warp-MMA kernel of tq_search_tc.cu.  Both
// keep each query's k best per CTA as they go, and a merge of those candidate
// lists follows.  Otherwise the SIMT score kernel below writes the nq x n
// score matrix to the workspace and two selection passes follow (per chunk of
// vectors, then a merge of the per-chunk candidates).
#include <cuda_bf16.h>

#include <algorithm>

#include "tq_internal.h"

namespace {

constexpr int kQB = 8;          // queries per score CTA
constexpr int kVB = 128;        // vectors per score CTA (one per thread)
constexpr int kSel = 256;       // threads per selection CTA
constexpr int64_t kChunk = 4096;

struct SearchLayout {
  size_t qt, st, table, scores, cand_idx, cand_sc, total;
  int64_t nchunks;
};

// Workspace: q̃, s̃, then the tensor-core path's query table and candidate
// lists, or the general path's score matrix and per-chunk candidates.
SearchLayout layout(const tq_plan* plan, int nq, int64_t n, int k) {
  const int d = plan->d, m = plan->m;
  const bool wide = tq::search_wide_supported(plan, k);
  const bool tc = wide || (d % 128 == 0 && m % 128 == 0);
  SearchLayout l{};
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  l.nchunks = wide ? tq::search_wide_lists(nq) : tc ? tq::search_tc_vchunks(n, nq) : tq::cdiv(n, kChunk);
  size_t o = 0;
  l.qt = o; o += up(sizeof(float) * size_t(nq) * d);
  l.st = o; o += up(sizeof(float) * size_t(nq) * m);
  l.table = o;
  if (tc) o += up(wide ? tq::search_wide_table_bytes(plan, nq) : tq::search_tc_table_bytes(plan, nq));
  l.scores = o;
  if (!tc) o += up(sizeof(float) * size_t(nq) * size_t(n));
  l.cand_idx = o; o += up(sizeof(int32_t) * size_t(nq) * l.nchunks * k);
  l.cand_sc = o; o += up(sizeof(float) * size_t(nq) * l.nchunks * k);
  l.total = o;
  return l;
}

struct ScoreArgs {
  const uint32_t* idx; const uint32_t* sgn; const float* norm; const float* rnorm;
  int64_t n;
  int nq, d, m, w;
  const float* qt; const float* st; const float* centroids;
  float alpha;
  float* scores;  // [nq][n]
};

__global__ void __launch_bounds__(kVB) score_kernel(ScoreArgs a) {
  extern __shared__ float sm[];
  const int d = a.d, m = a.m, w = a.w, wi = w * d / 32, ws = m / 32;
  const int q0 = blockIdx.y * kQB, nqb = min(kQB, a.nq - q0);
  float* qts = sm;               // [kQB][d]
  float* sts = qts + kQB * d;    // [kQB][m]
  float* cent = sts + kQB * m;   // [8]
  for (int e = threadIdx.x; e < kQB * d; e += kVB) qts[e] = (e / d) < nqb ? a.qt[(size_t)q0 * d + e] : 0.0f;
  for (int e = threadIdx.x; e < kQB * m; e += kVB) sts[e] = (e / m) < nqb ? a.st[(size_t)q0 * m + e] : 0.0f;
  if (threadIdx.x < 8) cent[threadIdx.x] = threadIdx.x < (1 << w) ? a.centroids[threadIdx.x] : 0.0f;
  __syncthreads();
  const int64_t i = int64_t(blockIdx.x) * kVB + threadIdx.x;
  if (i >= a.n) return;
  float d1[kQB], d2[kQB];
#pragma unroll
  for (int q = 0; q < kQB; ++q) d1[q] = d2[q] = 0.0f;
  const uint32_t* ip = a.idx + i * wi;
  for (int kw = 0; kw < d / 32; ++kw) {
    uint32_t pw[3] = {0u, 0u, 0u};
    for (int p = 0; p < w; ++p) pw[p] = __ldg(ip + p * (d / 32) + kw);
    for (int bit = 0; bit < 32; ++bit) {
      int idx = 0;
      for (int p = 0; p < w; ++p) idx |= ((pw[p] >> bit) & 1) << p;
      const float c = cent[idx];
      const int j = kw * 32 + bit;
#pragma unroll
      for (int q = 0; q < kQB; ++q) d1[q] = fmaf(qts[q * d + j], c, d1[q]);
    }
  }
  const uint32_t* sp = a.sgn + i * ws;
  for (int kw = 0; kw < ws; ++kw) {
    const uint32_t word = __ldg(sp + kw);
    for (int bit = 0; bit < 32; ++bit) {
      const float sg = ((word >> bit) & 1) ? 1.0f : -1.0f;
      const int j = kw * 32 + bit;
#pragma unroll
      for (int q = 0; q < kQB; ++q) d2[q] = fmaf(sts[q * m + j], sg, d2[q]);
    }
  }
  const float nv = __ldg(a.norm + i), rv = m > 0 ? __ldg(a.rnorm + i) : 0.0f;
  for (int q = 0; q < nqb; ++q) a.scores[(size_t)(q0 + q) * a.n + i] = nv * d1[q] + a.alpha * rv * d2[q];
}

// (s1, i1) ranks before (s2, i2): higher score, then lower index
__device__ __forceinline__ bool before(float s1, int64_t i1, float s2, int64_t i2) {
  return s1 > s2 || (s1 == s2 && i1 < i2);
}

// k rounds of "best element ranked after the previous winner" over one list.
// ids == nullptr: the element's id is its position + id0.
__device__ void select_topk(const float* sc, const int32_t* ids, int64_t count, int64_t id0, int k, int32_t* out_idx,
                            float* out_sc) {
  __shared__ float rs[kSel / 32];
  __shared__ int64_t ri[kSel / 32];
  __shared__ float prev_s;
  __shared__ int64_t prev_i;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    prev_s = INFINITY;
    prev_i = -1;
  }
  __syncthreads();
  for (int r = 0; r < k; ++r) {
    const float ps = prev_s;
    const int64_t pi = prev_i;
    float bs = -INFINITY;
    int64_t bi = INT64_MAX;
    for (int64_t e = threadIdx.x; e < count; e += kSel) {
      const float s = sc[e];
      const int64_t id = ids ? (int64_t)ids[e] : id0 + e;
      if (id < 0) continue;
      if (before(ps, pi, s, id) && before(s, id, bs, bi)) {
        bs = s;
        bi = id;
      }
    }
    for (int o = 16; o > 0; o >>= 1) {
      const float os = __shfl_xor_sync(0xffffffffu, bs, o);
      const int64_t oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (before(os, oi, bs, bi)) {
        bs = os;
        bi = oi;
      }
    }
    if (lane == 0) {
      rs[warp] = bs;
      ri[warp] = bi;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      for (int v = 1; v < kSel / 32; ++v)
        if (before(rs[v], ri[v], bs, bi)) {
          bs = rs[v];
          bi = ri[v];
        }
      const bool found = bi != INT64_MAX;
      out_idx[r] = found ? (int32_t)bi : -1;
      out_sc[r] = found ? bs : -INFINITY;
      prev_s = bs;
      prev_i = found ? bi : INT64_MAX;
    }
    __syncthreads();
  }
}

__global__ void __launch_bounds__(kSel) select_chunks_kernel(const float* scores, int64_t n, int64_t nchunks, int k,
                                                             int32_t* cand_idx, float* cand_sc) {
  const int64_t chunk = blockIdx.x, q = blockIdx.y;
  const int64_t e0 = chunk * kChunk, cnt = min(kChunk, n - e0);
  const size_t o = ((size_t)q * nchunks + chunk) * k;
  select_topk(scores + (size_t)q * n + e0, nullptr, cnt, e0, k, cand_idx + o, cand_sc + o);
}

__global__ void __launch_bounds__(kSel) merge_kernel(const int32_t* cand_idx, const float* cand_sc, int64_t nchunks,
                                                     int k, int32_t* idx_out, float* score_out) {
  const int64_t q = blockIdx.x;
  const size_t o = (size_t)q * nchunks * k;
  select_topk(cand_sc + o, cand_idx + o, nchunks * k, 0, k, idx_out + (size_t)q * k, score_out + (size_t)q * k);
}

}  // namespace

extern "C" tq_status tq_search_workspace_size(const tq_plan* plan, int nq, int64_t n, int k, size_t* bytes) {
  if (!tq::valid_plan(plan) || !bytes || nq < 1 || n < 1 || n > INT32_MAX || k < 1 || k > 64) return TQ_ERR_ARG;
  *bytes = layout(plan, nq, n, k).total;
  return TQ_OK;
}

extern "C" tq_status tq_search_topk(const tq_plan* plan, const void* q, tq_dtype q_dtype, int nq,
                                    const tq_records* recs, int64_t n, int k, int32_t* idx_out, float* score_out,
                                    void* workspace, size_t ws_bytes, tq_stream stream) {
  if (!tq::valid_plan(plan) || !tq::valid_records(recs, plan) || !q || !tq::aligned16(q) || nq < 1 || n < 1 ||
      n > recs->capacity || n > INT32_MAX || k < 1 || k > 64 || !idx_out || !score_out || !workspace ||
      !tq::aligned16(workspace) || (q_dtype != TQ_F32 && q_dtype != TQ_BF16))
    return TQ_ERR_ARG;
  if (recs->layout != TQ_LAYOUT_ROWS) return TQ_ERR_UNSUPPORTED;
  const SearchLayout l = layout(plan, nq, n, k);
  if (ws_bytes < l.total) return TQ_ERR_WORKSPACE;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  float* qt = reinterpret_cast<float*>(ws + l.qt);
  float* st = reinterpret_cast<float*>(ws + l.st);
  float* scores = reinterpret_cast<float*>(ws + l.scores);
  int32_t* cand_idx = reinterpret_cast<int32_t*>(ws + l.cand_idx);
  float* cand_sc = reinterpret_cast<float*>(ws + l.cand_sc);
  tq_status s = tq::launch_query_prep(plan, q, q_dtype, nq, qt, st, cs);
  if (s != TQ_OK) return s;
  const bool wide = tq::search_wide_supported(plan, k);
  if (wide || tq::search_tc_supported(plan, recs)) {
    s = wide ? tq::launch_search_wide(plan, recs, n, nq, qt, st, ws + l.table, k, cand_idx, cand_sc, cs)
             : tq::launch_search_tc(plan, recs, n, nq, qt, st, ws + l.table, k, cand_idx, cand_sc, cs);
    if (s != TQ_OK) return s;
    merge_kernel<<<nq, kSel, 0, cs>>>(cand_idx, cand_sc, l.nchunks, k, idx_out, score_out);
    return tq::launch_status();
  } else {
    ScoreArgs a{recs->idx, recs->sgn, recs->norm, recs->rnorm, n, nq, plan->d, plan->m, plan->w, qt, st,
                plan->centroids, plan->qjl_alpha, scores};
    const size_t smem = sizeof(float) * (kQB * (plan->d + plan->m) + 8);
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(score_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return TQ_ERR_CUDA;
    score_kernel<<<dim3((unsigned)tq::cdiv(n, kVB), (unsigned)tq::cdiv(nq, kQB)), kVB, smem, cs>>>(a);
    if ((s = tq::launch_status()) != TQ_OK) return s;
  }
  select_chunks_kernel<<<dim3((unsigned)l.nchunks, nq), kSel, 0, cs>>>(scores, n, l.nchunks, k, cand_idx, cand_sc);
  if ((s = tq::launch_status()) != TQ_OK) return s;
  merge_kernel<<<nq, kSel, 0, cs>>>(cand_idx, cand_sc, l.nchunks, k, idx_out, score_out);
  return tq::launch_status();
}

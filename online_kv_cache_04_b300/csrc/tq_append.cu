// tq_append_kv: the online step of a decode loop -- quantize the new key and
// value of every (batch row, kv head) and store them at the next free token
// of their caches, then advance the context lengths.
//
// Each new vector goes through the same two stages as tq_quantize
// ("谷歌TurboQuant如何绕过内存墙？" §2, stages 1 and 2; "TurboQuant 与 AI
// 效率革命" §四, three-step pipeline): n = ||x||, u = Π x / n, bucket index
// against the Lloyd-Max bounds, ρ = u - c[idx], ||r|| = n ||ρ||, σ =
// sign(S Πᵀ ρ) with sign(0) = +1, and the zero vector stored as u = 0, r = 0,
// all σ = +1.  A decode step appends B·Hkv keys and as many values: one CTA
// per vector, fp32 FMAs against the transposed matrices (Πᵀ and (S Πᵀ)ᵀ, so
// that consecutive threads read consecutive words).  Each column's sum is cut
// into kParts runs held by kParts threads, which bounds the chain of
// dependent loads a thread waits for (the vectors are few: the step is
// latency-bound); the first 128 threads add the runs in order and finish
// coordinates j0 + tid, so that a warp ballot forms one packed word.
//
// The token position of batch row b is ctx_len[b]; the second launch adds one
// to every ctx_len[b] whose row was written, after every CTA of the first has
// read it (stream order).  Rows of a full cache (ctx_len[b] >= ctx_stride) or
// with a negative length are left alone and raise fault bit kFaultAppend.
#include <cuda_bf16.h>

#include <algorithm>

#include "tq_internal.h"

namespace {

constexpr int kCols = 128;               // output columns per pass
constexpr int kParts = 8;                // each column's sum is cut into kParts runs of i
constexpr int kThreads = kCols * kParts;
constexpr int kMaxD = 1024;
constexpr unsigned kFaultAppend = 8u;

struct AppendArgs {
  const void* x[2];        // new keys, new values: [B][Hkv][d]
  tq_records rec[2];       // key cache, value cache
  const int32_t* ctx_len;  // [B]
  int64_t ctx_stride;
  int Hkv, d, m, w;
  const float* pi_t;       // [d][d]  Πᵀ
  const float* s_rot_t;    // [d][m]  (S Πᵀ)ᵀ
  const float* centroids;
  const float* bounds;
  unsigned* fault;
  const int32_t* pages;    // paged caches: [B*Hkv][ctx_stride / 256] (NULL: contiguous rows)
  int64_t npages;          // pages the record arrays hold
};

constexpr int kPage = 256;             // tokens per page of a paged cache
constexpr unsigned kFaultPage = 16u;   // a page-table entry outside the record arrays

template <typename T>
__device__ __forceinline__ float load_elem(const T* p);
template <>
__device__ __forceinline__ float load_elem<float>(const float* p) { return *p; }
template <>
__device__ __forceinline__ float load_elem<__nv_bfloat16>(const __nv_bfloat16* p) { return __bfloat162float(*p); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Σ_{i0 <= i < i1} M[i][j] v[i] in increasing i.
__device__ __forceinline__ float column_run(const float* __restrict__ M, int ld, int j, const float* v, int i0,
                                           int i1) {
  float acc = 0.0f;
#pragma unroll 4
  for (int i = i0; i < i1; ++i) acc = fmaf(__ldg(M + (size_t)i * ld + j), v[i], acc);
  return acc;
}

// Column sums of M (rows i < d, leading dimension ld) against v for columns
// [j0, j0 + kCols): thread (part, col) sums rows [part·d/kParts, (part+1)·d/kParts)
// of column j0 + col into runs[part][col]; each thread then waits for d/kParts
// loads, not d.  Ends with a barrier; the caller adds the runs in part order.
__device__ __forceinline__ void column_runs(const float* __restrict__ M, int ld, int ncols, int j0, const float* v,
                                            int d, float (*runs)[kCols]) {
  const int col = threadIdx.x % kCols, part = threadIdx.x / kCols;
  const int len = d / kParts;  // d % 32 == 0, so len is a whole number
  if (j0 + col < ncols) runs[part][col] = column_run(M, ld, j0 + col, v, part * len, (part + 1) * len);
  __syncthreads();
}

__device__ __forceinline__ float sum_runs(const float (*runs)[kCols], int col) {
  float acc = runs[0][col];
#pragma unroll
  for (int p = 1; p < kParts; ++p) acc += runs[p][col];
  return acc;
}

// Set (or clear) bit `bit` of one word that no other thread of the launch writes.
__device__ __forceinline__ void put_bit(uint32_t* word, uint32_t bit, bool set) {
  const uint32_t v = *word;
  *word = set ? (v | bit) : (v & ~bit);
}

// grid (B·Hkv, 2): x = (batch row, kv head) unit, y = 0 keys / 1 values.
template <typename T>
__global__ void __launch_bounds__(kThreads) append_kernel(AppendArgs a) {
  __shared__ float xs[kMaxD];   // the new vector, fp32
  __shared__ float rs[kMaxD];   // ρ, unit-norm domain
  __shared__ float cent[8], bnd[8];
  __shared__ float nrm, rsq;
  __shared__ float runs[kParts][kCols];
  const int unit = blockIdx.x, which = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int d = a.d, m = a.m, w = a.w, L = 1 << w;
  const int64_t t = a.ctx_len[unit / a.Hkv];
  if (t < 0 || t >= a.ctx_stride) {  // the whole CTA leaves together
    if (tid == 0) atomicOr(a.fault, kFaultAppend);
    return;
  }
  // fields picked one by one: a runtime index into the parameter arrays would go through local memory
  uint32_t* const ridx = which ? a.rec[1].idx : a.rec[0].idx;
  uint32_t* const rsgn = which ? a.rec[1].sgn : a.rec[0].sgn;
  float* const rnrm = which ? a.rec[1].norm : a.rec[0].norm;
  float* const rrn = which ? a.rec[1].rnorm : a.rec[0].rnorm;
  const bool rows = (which ? a.rec[1].layout : a.rec[0].layout) == TQ_LAYOUT_ROWS;
  int64_t row = (int64_t)unit * a.ctx_stride + t;
  if (a.pages != nullptr) {  // the page holding token t
    const int64_t pg = a.pages[(int64_t)unit * (a.ctx_stride / kPage) + t / kPage];
    if (pg < 0 || pg >= a.npages) {
      if (tid == 0) atomicOr(a.fault, kFaultPage);
      return;
    }
    row = pg * kPage + t % kPage;
  }
  const T* x = static_cast<const T*>(which ? a.x[1] : a.x[0]) + (size_t)unit * d;
  if (tid < L) cent[tid] = a.centroids[tid];
  if (tid < L - 1) bnd[tid] = a.bounds[tid];
  for (int i = tid; i < d; i += kThreads) xs[i] = load_elem<T>(x + i);
  __syncthreads();
  if (warp == 0) {
    float s = 0.0f;
    for (int i = lane; i < d; i += 32) s = fmaf(xs[i], xs[i], s);
    s = warp_sum(s);
    if (lane == 0) nrm = sqrtf(s);
  }
  __syncthreads();

  // stage 1: rotate, bucketize, residual, index bits.  Threads tid < kCols
  // finish column j0 + tid (d % 32 == 0: a warp is either wholly inside
  // [0, d) or wholly outside).
  const float n = nrm;
  const int64_t blk = row >> 5;
  const uint32_t bbit = 1u << tq::block32_bit((int)(row & 31));
  for (int j0 = 0; j0 < d; j0 += kCols) {
    column_runs(a.pi_t, d, d, j0, xs, d, runs);
    const int j = j0 + tid;
    if (tid < kCols && j < d) {
      const float acc = sum_runs(runs, tid);
      const float u = n > 0.0f ? acc / n : 0.0f;
      int idx = 0;
      for (int k = 0; k < L - 1; ++k) idx += (bnd[k] < u) ? 1 : 0;
      rs[j] = n > 0.0f ? u - cent[idx] : 0.0f;
      if (rows) {
        for (int p = 0; p < w; ++p) {
          const uint32_t word = __ballot_sync(0xffffffffu, (idx >> p) & 1);
          if (lane == 0) ridx[row * (w * d / 32) + p * (d / 32) + j / 32] = word;
        }
      } else {
        for (int p = 0; p < w; ++p) put_bit(ridx + blk * (int64_t)(w * d) + p * d + j, bbit, (idx >> p) & 1);
      }
    }
    __syncthreads();  // runs[] is refilled by the next pass; rs[] complete after the last
  }

  if (m > 0) {
    if (warp == 0) {
      float s2 = 0.0f;
      for (int i = lane; i < d; i += 32) s2 = fmaf(rs[i], rs[i], s2);
      s2 = warp_sum(s2);
      if (lane == 0) rsq = s2;
    }
    // stage 2: σ = sign(S Πᵀ ρ), sign(0) = +1
    for (int j0 = 0; j0 < m; j0 += kCols) {
      column_runs(a.s_rot_t, m, m, j0, rs, d, runs);
      const int jj = j0 + tid;
      if (tid < kCols && jj < m) {
        const float acc = sum_runs(runs, tid);
        if (rows) {
          const uint32_t word = __ballot_sync(0xffffffffu, acc >= 0.0f);
          if (lane == 0) rsgn[row * (m / 32) + jj / 32] = word;
        } else {
          put_bit(rsgn + blk * (int64_t)m + jj, bbit, acc >= 0.0f);
        }
      }
      __syncthreads();
    }
  }
  if (tid == 0) {
    rnrm[row] = n;
    if (m > 0) rrn[row] = n * sqrtf(rsq);
  }
}

__global__ void advance_kernel(int32_t* ctx_len, int B, int64_t ctx_stride) {
  for (int b = threadIdx.x; b < B; b += blockDim.x) {
    const int32_t t = ctx_len[b];
    if (t >= 0 && t < ctx_stride) ctx_len[b] = t + 1;
  }
}

}  // namespace

namespace {

tq_status append_impl(const tq_plan* plan, const void* k_new, const void* v_new, tq_dtype dtype, int B, int Hkv,
                      const tq_records* K, const tq_records* V, int32_t* ctx_len, int64_t ctx_stride,
                      tq_stream stream, const int32_t* pages) {
  if (!tq::valid_plan(plan) || !tq::valid_records(K, plan) || !tq::valid_records(V, plan) || !k_new || !v_new ||
      !tq::aligned16(k_new) || !tq::aligned16(v_new) || !ctx_len || B < 1 || Hkv < 1 || ctx_stride < 1 ||
      ctx_stride > INT32_MAX || (dtype != TQ_F32 && dtype != TQ_BF16))
    return TQ_ERR_ARG;
  // keys and values of one step land on the same rows: one cache for both would race
  if (K->idx == V->idx || (K->sgn && K->sgn == V->sgn) || K->norm == V->norm) return TQ_ERR_ARG;
  const int64_t units = (int64_t)B * Hkv;
  if (units > INT32_MAX) return TQ_ERR_ARG;
  if (pages == nullptr && (units * ctx_stride > K->capacity || units * ctx_stride > V->capacity)) return TQ_ERR_ARG;
  if (pages != nullptr && (K->capacity < kPage || V->capacity < kPage)) return TQ_ERR_ARG;
  // a block-layout cache keeps whole 32-row blocks per (batch row, kv head)
  if ((K->layout == TQ_LAYOUT_BLOCK32 || V->layout == TQ_LAYOUT_BLOCK32) && ctx_stride % 32 != 0) return TQ_ERR_ARG;
  unsigned* fault = tq::fault_word();
  if (!fault) return TQ_ERR_CUDA;
  AppendArgs a{{k_new, v_new}, {*K, *V}, ctx_len, ctx_stride, Hkv, plan->d, plan->m, plan->w, plan->pi_t,
               plan->s_rot_t, plan->centroids, plan->bounds, fault, pages,
               std::min(K->capacity, V->capacity) / kPage};
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  const dim3 grid((unsigned)units, 2);
  if (dtype == TQ_F32)
    append_kernel<float><<<grid, kThreads, 0, cs>>>(a);
  else
    append_kernel<__nv_bfloat16><<<grid, kThreads, 0, cs>>>(a);
  tq_status s = tq::launch_status();
  if (s != TQ_OK) return s;
  advance_kernel<<<1, 256, 0, cs>>>(ctx_len, B, ctx_stride);
  return tq::launch_status();
}

}  // namespace

tq_status tq::append_kv(const tq_plan* plan, const void* k_new, const void* v_new, tq_dtype dtype, int B, int Hkv,
                        const tq_records* K, const tq_records* V, int32_t* ctx_len, int64_t ctx_stride,
                        cudaStream_t stream, const int32_t* pages) {
  return append_impl(plan, k_new, v_new, dtype, B, Hkv, K, V, ctx_len, ctx_stride,
                     reinterpret_cast<tq_stream>(stream), pages);
}

extern "C" tq_status tq_append_kv(const tq_plan* plan, const void* k_new, const void* v_new, tq_dtype dtype, int B,
                                  int Hkv, const tq_records* K, const tq_records* V, int32_t* ctx_len,
                                  int64_t ctx_stride, tq_stream stream) {
  return append_impl(plan, k_new, v_new, dtype, B, Hkv, K, V, ctx_len, ctx_stride, stream, nullptr);
}

extern "C" tq_status tq_append_kv_paged(const tq_plan* plan, const void* k_new, const void* v_new, tq_dtype dtype,
                                        int B, int Hkv, const tq_records* K, const tq_records* V, int32_t* ctx_len,
                                        const int32_t* pages, int max_pages, tq_stream stream) {
  if (pages == nullptr || !tq::aligned16(pages) || max_pages < 1) return TQ_ERR_ARG;
  return append_impl(plan, k_new, v_new, dtype, B, Hkv, K, V, ctx_len, int64_t(max_pages) * kPage, stream, pages);
}

// tq_quantize: online two-stage quantization of KV vectors.
//
// Steps per vector ("谷歌TurboQuant如何绕过内存墙？" §2, stages 1 and 2;
// "TurboQuant 与 AI 效率革命" §四, three-step pipeline):
//   n = ||x||;  u = Π x / n;  idx_j = #{k : β_k < u_j};  ρ = u - c[idx]
//   (= Π r / n);  ||r|| = n ||ρ||;  σ = sign(S r) = sign(S Πᵀ ρ), sign(0) = +1.
// Indices are stored as w bit-planes of 32-coordinate words and the signs as
// m/32 words ("TurboQuant压缩效果": several codes per 32-bit word).
//
// This file holds the portable SIMT path (fp32 FMA, any d, m multiple of 32
// up to 1024).  A tile of TV vectors is staged in shared memory; each thread
// owns coordinates j ≡ tid (mod 128), so every warp holds 32 consecutive
// coordinates and one warp ballot forms one packed word.
#include <cuda_bf16.h>

#include <algorithm>

#include "tq_internal.h"

namespace {

struct QuantArgs {
  const void* x;
  int64_t n, ld;
  int d, m, w;
  const float* pi_t;     // [d][d]  Πᵀ  (pi_t[i*d + j] = Π[j][i])
  const float* s_rot_t;  // [d][m]  (S Πᵀ)ᵀ
  const float* centroids;
  const float* bounds;
  uint32_t* idx;         // layout 0: rows already offset; layout 1: base of the cache
  uint32_t* sgn;
  float* norm;           // rows already offset
  float* rnorm;
  int64_t row0;          // cache row of x's row 0 (layout 1 addressing)
  const int32_t* cols;   // optional [d] device column list: element j of a row is x[row][cols[j]]
};

// Layout 1: merge the bits of the tile's rows into the 32-row block words.
// Rows [r_lo, r_lo + TV) span at most two blocks; `bits[k]` / `mask[k]` hold
// the rows of block (r_lo >> 5) + k.  Each bit has one writer per call, so
// and-then-or on disjoint masks is race-free across CTAs.
__device__ __forceinline__ void merge_block_word(uint32_t* w0, uint32_t* w1, const uint32_t (&bits)[2],
                                                 const uint32_t (&mask)[2]) {
  if (mask[0]) {
    atomicAnd(w0, ~mask[0]);
    atomicOr(w0, bits[0] & mask[0]);
  }
  if (mask[1]) {
    atomicAnd(w1, ~mask[1]);
    atomicOr(w1, bits[1] & mask[1]);
  }
}

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

constexpr int kThreads = 128;

template <int TV, typename T, int LAYOUT>
__global__ void __launch_bounds__(kThreads) quantize_simt_kernel(QuantArgs a) {
  static_assert(TV <= 32 && 32 % TV == 0, "a tile spans at most two 32-row blocks");
  extern __shared__ float sm[];
  const int d = a.d, m = a.m, w = a.w, L = 1 << w;
  float* xs = sm;              // [TV][d] input tile, fp32
  float* rs = xs + TV * d;     // [TV][d] residual ρ (unit-norm domain)
  float* nrm = rs + TV * d;    // [TV]
  float* rsq = nrm + TV;       // [TV]   ||ρ||²
  float* cent = rsq + TV;      // [L]
  float* bnd = cent + 8;       // [L-1]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid < L) cent[tid] = a.centroids[tid];
  if (tid < L - 1) bnd[tid] = a.bounds[tid];
  const int64_t ntiles = (a.n + TV - 1) / TV;
  const int words_idx = w * d / 32, words_sgn = m / 32;
  const T* x = static_cast<const T*>(a.x);

  for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
    const int64_t v0 = tile * TV;
    for (int e = tid; e < TV * d; e += kThreads) {
      const int v = e / d, i = e - v * d;
      const int64_t row = v0 + v;
      const int64_t col = a.cols ? __ldg(a.cols + i) : i;
      xs[e] = row < a.n ? load_elem<T>(x + row * a.ld + col) : 0.0f;
    }
    __syncthreads();
    for (int v = warp; v < TV; v += kThreads / 32) {
      float s = 0.0f;
      for (int i = lane; i < d; i += 32) s = fmaf(xs[v * d + i], xs[v * d + i], s);
      s = warp_sum(s);
      if (lane == 0) nrm[v] = sqrtf(s);
    }
    __syncthreads();

    // stage 1: u = Π x / n, bucketize, residual, index bit-planes
    const int64_t blk0 = (a.row0 + v0) & ~int64_t(31);  // first block row of this tile
    for (int j = tid; j < d; j += kThreads) {
      uint32_t mask[2] = {0u, 0u}, pbits[3][2] = {{0u, 0u}, {0u, 0u}, {0u, 0u}};
      (void)mask;
      (void)pbits;
      float acc[TV];
#pragma unroll
      for (int v = 0; v < TV; ++v) acc[v] = 0.0f;
      for (int i = 0; i < d; ++i) {
        const float pij = __ldg(a.pi_t + (size_t)i * d + j);
#pragma unroll
        for (int v = 0; v < TV; ++v) acc[v] = fmaf(pij, xs[v * d + i], acc[v]);
      }
#pragma unroll
      for (int v = 0; v < TV; ++v) {
        const float n = nrm[v];
        const float u = n > 0.0f ? acc[v] / n : 0.0f;
        int idx = 0;
        for (int k = 0; k < L - 1; ++k) idx += (bnd[k] < u) ? 1 : 0;
        const float rho = n > 0.0f ? u - cent[idx] : 0.0f;
        rs[v * d + j] = rho;
        const int64_t row = v0 + v;
        if constexpr (LAYOUT == TQ_LAYOUT_ROWS) {
          for (int p = 0; p < w; ++p) {
            const uint32_t word = __ballot_sync(0xffffffffu, (idx >> p) & 1);
            if (lane == 0 && row < a.n) a.idx[row * words_idx + p * (d / 32) + j / 32] = word;
          }
        } else {
          const int64_t r = a.row0 + row;
          const int k = (int)((r >> 5) - (blk0 >> 5));
          const uint32_t bit = row < a.n ? 1u << tq::block32_bit((int)(r & 31)) : 0u;
          mask[k] |= bit;
#pragma unroll
          for (int p = 0; p < 3; ++p)
            if (p < w && ((idx >> p) & 1)) pbits[p][k] |= bit;
        }
      }
      if constexpr (LAYOUT == TQ_LAYOUT_BLOCK32) {
        for (int p = 0; p < w; ++p) {
          uint32_t* w0 = a.idx + (blk0 >> 5) * (int64_t)(w * d) + p * d + j;
          merge_block_word(w0, w0 + w * d, pbits[p], mask);
        }
      }
    }
    __syncthreads();
    // ||ρ||² per vector in a fixed order (the records do not depend on scheduling)
    for (int v = warp; v < TV; v += kThreads / 32) {
      float s2 = 0.0f;
      for (int i = lane; i < d; i += 32) s2 = fmaf(rs[v * d + i], rs[v * d + i], s2);
      s2 = warp_sum(s2);
      if (lane == 0) rsq[v] = s2;
    }
    __syncthreads();

    // stage 2: σ = sign(S Πᵀ ρ)
    for (int jj = tid; jj < m; jj += kThreads) {
      float acc[TV];
#pragma unroll
      for (int v = 0; v < TV; ++v) acc[v] = 0.0f;
      for (int i = 0; i < d; ++i) {
        const float sij = __ldg(a.s_rot_t + (size_t)i * m + jj);
#pragma unroll
        for (int v = 0; v < TV; ++v) acc[v] = fmaf(sij, rs[v * d + i], acc[v]);
      }
      if constexpr (LAYOUT == TQ_LAYOUT_ROWS) {
#pragma unroll
        for (int v = 0; v < TV; ++v) {
          const uint32_t word = __ballot_sync(0xffffffffu, acc[v] >= 0.0f);
          const int64_t row = v0 + v;
          if (lane == 0 && row < a.n) a.sgn[row * words_sgn + jj / 32] = word;
        }
      } else {
        uint32_t mask[2] = {0u, 0u}, sbits[2] = {0u, 0u};
#pragma unroll
        for (int v = 0; v < TV; ++v) {
          const int64_t row = v0 + v, r = a.row0 + row;
          const int k = (int)((r >> 5) - (blk0 >> 5));
          const uint32_t bit = row < a.n ? 1u << tq::block32_bit((int)(r & 31)) : 0u;
          mask[k] |= bit;
          if (acc[v] >= 0.0f) sbits[k] |= bit;
        }
        uint32_t* w0 = a.sgn + (blk0 >> 5) * (int64_t)m + jj;
        merge_block_word(w0, w0 + m, sbits, mask);
      }
    }
    if (tid < TV && v0 + tid < a.n) {
      a.norm[v0 + tid] = nrm[tid];
      if (m > 0) a.rnorm[v0 + tid] = nrm[tid] * sqrtf(rsq[tid]);
    }
    __syncthreads();
  }
}

template <int TV, typename T, int LAYOUT>
tq_status launch_simt(const QuantArgs& a, cudaStream_t st) {
  const size_t smem = sizeof(float) * (2 * TV * a.d + 2 * TV + 16);
  auto kern = quantize_simt_kernel<TV, T, LAYOUT>;
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return TQ_ERR_CUDA;
  const int64_t ntiles = (a.n + TV - 1) / TV;
  const int64_t grid = std::min<int64_t>(ntiles, int64_t(tq::sm_count()) * 8);
  kern<<<(unsigned)grid, kThreads, smem, st>>>(a);
  return tq::launch_status();
}

template <int LAYOUT>
tq_status launch_simt_any(const QuantArgs& a, tq_dtype dtype, cudaStream_t st) {
  if (a.d <= 256)
    return dtype == TQ_F32 ? launch_simt<16, float, LAYOUT>(a, st) : launch_simt<16, __nv_bfloat16, LAYOUT>(a, st);
  return dtype == TQ_F32 ? launch_simt<8, float, LAYOUT>(a, st) : launch_simt<8, __nv_bfloat16, LAYOUT>(a, st);
}

}  // namespace

tq_status tq::quantize_simt_cols(const tq_plan* plan, const void* x, tq_dtype dtype, int64_t n, int64_t ld_x,
                                 const int32_t* cols, const tq_records* out, int64_t out_offset, cudaStream_t st) {
  QuantArgs a{};
  a.x = x;
  a.n = n;
  a.ld = ld_x;
  a.d = plan->d;
  a.m = plan->m;
  a.w = plan->w;
  a.pi_t = plan->pi_t;
  a.s_rot_t = plan->s_rot_t;
  a.centroids = plan->centroids;
  a.bounds = plan->bounds;
  a.idx = out->idx + out_offset * (plan->w * plan->d / 32);
  a.sgn = plan->m > 0 ? out->sgn + out_offset * (plan->m / 32) : nullptr;
  a.norm = out->norm + out_offset;
  a.rnorm = plan->m > 0 ? out->rnorm + out_offset : nullptr;
  a.row0 = out_offset;
  a.cols = cols;
  return launch_simt_any<TQ_LAYOUT_ROWS>(a, dtype, st);
}

extern "C" tq_status tq_quantize(const tq_plan* plan, const void* x, tq_dtype dtype, int64_t n, int64_t ld_x,
                                 const tq_records* out, int64_t out_offset, tq_stream stream) {
  if (!tq::valid_plan(plan) || !tq::valid_records(out, plan) || n < 0 || out_offset < 0) return TQ_ERR_ARG;
  if (dtype != TQ_F32 && dtype != TQ_BF16) return TQ_ERR_ARG;
  if (n == 0) return TQ_OK;
  if (x == nullptr || !tq::aligned16(x) || ld_x < plan->d || ld_x % 8 != 0) return TQ_ERR_ARG;
  if (out_offset > out->capacity || n > out->capacity - out_offset) return TQ_ERR_ARG;
  const bool rows = out->layout == TQ_LAYOUT_ROWS;
  QuantArgs a{};
  a.x = x;
  a.n = n;
  a.ld = ld_x;
  a.d = plan->d;
  a.m = plan->m;
  a.w = plan->w;
  a.pi_t = plan->pi_t;
  a.s_rot_t = plan->s_rot_t;
  a.centroids = plan->centroids;
  a.bounds = plan->bounds;
  a.idx = rows ? out->idx + out_offset * (plan->w * plan->d / 32) : out->idx;
  a.sgn = rows ? out->sgn + out_offset * (plan->m / 32) : out->sgn;
  a.norm = out->norm + out_offset;
  a.rnorm = out->rnorm + out_offset;
  a.row0 = out_offset;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (rows) {
    if (tq::quantize_tc_supported(plan, dtype, n))
      return tq::quantize_tc(plan, x, nullptr, n, ld_x, out, nullptr, out_offset, st);
    if (tq::quantize_wide_supported(plan, out)) return tq::quantize_wide(plan, x, dtype, n, ld_x, out, out_offset, st);
    if (tq::quantize_mma_supported(plan, out)) return tq::quantize_mma(plan, x, dtype, n, ld_x, out, out_offset, st);
    return launch_simt_any<TQ_LAYOUT_ROWS>(a, dtype, st);
  }
  // 32-row blocks: rows up to the first block boundary go through the SIMT
  // kernel (it merges into a partly written block); the aligned rest may take
  // the tensor-core kernel, which owns whole blocks.
  const int64_t head = std::min<int64_t>(n, (32 - out_offset % 32) % 32);
  if (head > 0) {
    QuantArgs h = a;
    h.n = head;
    tq_status s = launch_simt_any<TQ_LAYOUT_BLOCK32>(h, dtype, st);
    if (s != TQ_OK || head == n) return s;
  }
  const int64_t rest = n - head;
  const size_t esz = dtype == TQ_F32 ? 4 : 2;
  const void* xr = static_cast<const char*>(x) + head * ld_x * esz;
  if (tq::quantize_tc_supported(plan, dtype, rest))
    return tq::quantize_tc(plan, xr, nullptr, rest, ld_x, out, nullptr, out_offset + head, st);
  QuantArgs r = a;
  r.x = xr;
  r.n = rest;
  r.norm += head;
  r.rnorm += head;
  r.row0 = out_offset + head;
  return launch_simt_any<TQ_LAYOUT_BLOCK32>(r, dtype, st);
}

extern "C" tq_status tq_quantize_pair(const tq_plan* plan, const void* x0, const void* x1, tq_dtype dtype, int64_t n,
                                      int64_t ld_x, const tq_records* out0, const tq_records* out1,
                                      int64_t out_offset, tq_stream stream) {
  // the same checks as tq_quantize, for both pairs, before anything is launched
  if (!tq::valid_plan(plan) || !tq::valid_records(out0, plan) || !tq::valid_records(out1, plan) || n < 0 ||
      out_offset < 0)
    return TQ_ERR_ARG;
  if (dtype != TQ_F32 && dtype != TQ_BF16) return TQ_ERR_ARG;
  if (n == 0) return TQ_OK;
  for (const void* x : {x0, x1})
    if (x == nullptr || !tq::aligned16(x) || ld_x < plan->d || ld_x % 8 != 0) return TQ_ERR_ARG;
  for (const tq_records* o : {out0, out1})
    if (out_offset > o->capacity || n > o->capacity - out_offset) return TQ_ERR_ARG;
  const bool aligned = out_offset % 32 == 0 ||
                       (out0->layout == TQ_LAYOUT_ROWS && out1->layout == TQ_LAYOUT_ROWS);
  if (tq::quantize_tc_supported(plan, dtype, n) && aligned)
    return tq::quantize_tc(plan, x0, x1, n, ld_x, out0, out1, out_offset, reinterpret_cast<cudaStream_t>(stream));
  const tq_status s = tq_quantize(plan, x0, dtype, n, ld_x, out0, out_offset, stream);
  return s != TQ_OK ? s : tq_quantize(plan, x1, dtype, n, ld_x, out1, out_offset, stream);
}

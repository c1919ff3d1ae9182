// tq_quantize on the warp tensor-core path: d a multiple of 128 up to 1024,
// m = d or m = 0, fp32 or bf16 input, records in TQ_LAYOUT_ROWS.  (d = m = 128
// bf16 takes the tcgen05 quantizer.)
//
// What is computed is the two-stage quantizer of tq_quantize.cu
// ("谷歌TurboQuant如何绕过内存墙？" §2 stages 1 and 2; "TurboQuant 与 AI
// 效率革命" §四): n = ||x||, u = Π x / n, idx = #{k : β_k < u}, ρ = u - c[idx],
// ||r|| = n ||ρ||, σ = sign(S Πᵀ ρ).
//
// Both products are dense contractions over many vectors, run as mma.sync
// m16n8k16 bf16 with fp32 accumulation in split precision: x = x_hi + x_lo
// and Π = Π_hi + Π_lo as bf16 pairs, U = x_hi Π_hiᵀ + x_hi Π_loᵀ + x_lo Π_hiᵀ
// (the dropped x_lo Π_lo and the rest of x beyond 16 bits are ~2^-16
// relative), and the same for P = ρ (S Πᵀ)ᵀ.  A CTA takes 16 vectors: their
// bf16 pieces sit in shared memory (rows padded against bank conflicts), the
// matrix pieces are read as B fragments straight from the plan's copies in
// operand order, and each warp owns max(d/8, 32) output coordinates rounded
// up to whole 32-bit words, so that every index word fills in one warp (at
// d = 128 four warps own 32 each and the other four only stage and wait; at
// d = 384 six own 64 each).  After the first product the warps
// bucketize in registers, pack the index planes with quad shuffles, and write
// ρ's bf16 pieces over x's for the second product.
#include <cuda_bf16.h>

#include <algorithm>

#include "tq_internal.h"

namespace {

constexpr int kWarps = 8, kThreads = 32 * kWarps;
constexpr int kTV = 16;       // vectors per CTA (one MMA row block)
constexpr int kMaxNF = 16;    // n-fragments of 8 columns per warp (d/64 at d = 1024)
constexpr int kPad = 8;       // bf16 pad per shared row: rows land on different banks

struct MmaArgs {
  const void* x;
  int64_t n, ld;
  int d, m;
  const uint2* pi_fr;      // Π hi, lo in warp-MMA operand order (tq_plan.pi_frag)
  const uint2* s_fr;       // S Πᵀ hi, lo likewise
  const float* centroids;
  const float* bounds;
  uint32_t* idx;           // rows already offset
  uint32_t* sgn;
  float* norm;
  float* rnorm;
};

__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// bf16 pair (lo element first) of two floats, round to nearest even
__device__ __forceinline__ uint32_t bf2(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

template <typename T>
__device__ __forceinline__ float ld_elem(const T* p);
template <>
__device__ __forceinline__ float ld_elem<float>(const float* p) { return __ldg(p); }
template <>
__device__ __forceinline__ float ld_elem<__nv_bfloat16>(const __nv_bfloat16* p) { return __bfloat162float(*p); }

// acc[f] += A[16 x K] · B for the warp's n-fragments f < nf, B[k][col] = M[col][k]
// for a matrix M of `rows` rows whose bf16 pieces (hi at mh, lo at ml) are in
// warp-MMA operand order: one 8-byte load per lane and fragment, 256 contiguous
// bytes per warp.  Columns col0 + 8f + (0..7).  A's pieces (hi, lo) are rows of
// stride `lda` bf16 in shared memory.
__device__ __forceinline__ void gemm_split(float (&acc)[kMaxNF][4], const uint16_t* ah, const uint16_t* al,
                                           int lda, const uint2* __restrict__ mh, const uint2* __restrict__ ml,
                                           int K, int rows, int col0, int nf, int lane) {
  const int gq = lane >> 2, tig = lane & 3;
  const int frs = rows / 8;  // row groups of M
#pragma unroll 1
  for (int k0 = 0; k0 < K; k0 += 16) {
    const int c0 = k0 + 2 * tig;
    const uint32_t xh0 = *reinterpret_cast<const uint32_t*>(ah + gq * lda + c0);
    const uint32_t xh1 = *reinterpret_cast<const uint32_t*>(ah + (gq + 8) * lda + c0);
    const uint32_t xh2 = *reinterpret_cast<const uint32_t*>(ah + gq * lda + c0 + 8);
    const uint32_t xh3 = *reinterpret_cast<const uint32_t*>(ah + (gq + 8) * lda + c0 + 8);
    const uint32_t xl0 = *reinterpret_cast<const uint32_t*>(al + gq * lda + c0);
    const uint32_t xl1 = *reinterpret_cast<const uint32_t*>(al + (gq + 8) * lda + c0);
    const uint32_t xl2 = *reinterpret_cast<const uint32_t*>(al + gq * lda + c0 + 8);
    const uint32_t xl3 = *reinterpret_cast<const uint32_t*>(al + (gq + 8) * lda + c0 + 8);
    const size_t kbase = (size_t)(k0 / 16) * frs + col0 / 8;
#pragma unroll
    for (int f = 0; f < kMaxNF; ++f) {
      if (f < nf) {
        const uint2 bh = __ldg(mh + (kbase + f) * 32 + lane);
        const uint2 bl = __ldg(ml + (kbase + f) * 32 + lane);
        mma_bf16(acc[f], xh0, xh1, xh2, xh3, bh.x, bh.y);
        mma_bf16(acc[f], xh0, xh1, xh2, xh3, bl.x, bl.y);
        mma_bf16(acc[f], xl0, xl1, xl2, xl3, bh.x, bh.y);
      }
    }
  }
}

// OR of a 32-bit word over the four lanes of a quad (lanes 4g .. 4g + 3)
__device__ __forceinline__ uint32_t quad_or(uint32_t v) {
  v |= __shfl_xor_sync(0xffffffffu, v, 1);
  v |= __shfl_xor_sync(0xffffffffu, v, 2);
  return v;
}

// Output coordinates per warp: d/8, at least 32, rounded up to whole 32-bit words.
__device__ __forceinline__ int words_per_warp(int d) { return (max(d / 8, 32) + 31) / 32 * 32; }

__device__ __forceinline__ float warp_total(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

template <typename T, int W>
__global__ void __launch_bounds__(kThreads) quantize_mma_kernel(MmaArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int d = a.d, m = a.m, lda = d + kPad;
  uint16_t* ah = reinterpret_cast<uint16_t*>(smem);      // [16][lda] bf16 hi: x, then ρ
  uint16_t* al = ah + kTV * lda;                          // [16][lda] bf16 lo
  float* nrm = reinterpret_cast<float*>(al + kTV * lda);  // [16] ||x||
  float* rsq = nrm + kTV;                                 // [8 warps][16] partial ||ρ||²
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gq = lane >> 2, tig = lane & 3;
  const int64_t v0 = (int64_t)blockIdx.x * kTV;
  const T* x = static_cast<const T*>(a.x);

  // ---- x as bf16 pieces, and the norms (warp w: rows 2w and 2w + 1)
  for (int rr = 0; rr < 2; ++rr) {
    const int r = 2 * warp + rr;
    const int64_t v = v0 + r;
    float ss = 0.f;
    for (int i = 2 * lane; i < d; i += 64) {
      float e0 = 0.f, e1 = 0.f;
      if (v < a.n) {
        e0 = ld_elem<T>(x + v * a.ld + i);
        e1 = ld_elem<T>(x + v * a.ld + i + 1);
      }
      ss = fmaf(e0, e0, fmaf(e1, e1, ss));
      const uint32_t h = bf2(e0, e1);
      const float2 hf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&h));
      *reinterpret_cast<uint32_t*>(ah + r * lda + i) = h;
      *reinterpret_cast<uint32_t*>(al + r * lda + i) = bf2(e0 - hf.x, e1 - hf.y);
    }
    ss = warp_total(ss);
    if (lane == 0) nrm[r] = sqrtf(ss);
  }
  __syncthreads();

  // ---- U = x Πᵀ; warp w owns output coordinates [w d/8, (w + 1) d/8)
  float acc[kMaxNF][4];
#pragma unroll
  for (int f = 0; f < kMaxNF; ++f)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[f][e] = 0.f;
  // a warp's block of output coordinates is a whole number of 32-bit words
  // (d/8 rounded up to one; at d = 384, say, six warps own 64 each)
  const int cw1 = words_per_warp(d), col1 = warp * cw1, nf1 = col1 < d ? min(cw1, d - col1) / 8 : 0;
  gemm_split(acc, ah, al, lda, a.pi_fr, a.pi_fr + (size_t)d * d / 4, d, d, col1, nf1, lane);

  // ---- stage 1 in registers: u = U / n, idx, ρ (kept in acc), ||ρ||², index words
  constexpr int L = 1 << W;
  float cent[L], bnd[L - 1];
#pragma unroll
  for (int k = 0; k < L; ++k) cent[k] = __ldg(a.centroids + k);
#pragma unroll
  for (int k = 0; k < L - 1; ++k) bnd[k] = __ldg(a.bounds + k);
  const float n0 = nrm[gq], n1 = nrm[gq + 8];
  const float inv0 = n0 > 0.f ? 1.0f / n0 : 0.f, inv1 = n1 > 0.f ? 1.0f / n1 : 0.f;
  const int64_t vr0 = v0 + gq, vr1 = vr0 + 8;
  const int wi = W * d / 32;
  float rs0 = 0.f, rs1 = 0.f;
  uint32_t wb[2][W];
#pragma unroll
  for (int p = 0; p < W; ++p) wb[0][p] = wb[1][p] = 0u;
#pragma unroll
  for (int f = 0; f < kMaxNF; ++f) {
    if (f < nf1) {
#pragma unroll
      for (int e2 = 0; e2 < 4; ++e2) {
        const int row = e2 >> 1, e = e2 & 1;
        const float nr = row ? n1 : n0;
        const float u = acc[f][e2] * (row ? inv1 : inv0);
        int idx = 0;
#pragma unroll
        for (int k = 0; k < L - 1; ++k) idx += bnd[k] < u ? 1 : 0;
        float cv = cent[0];
#pragma unroll
        for (int k = 1; k < L; ++k) cv = idx == k ? cent[k] : cv;
        const float rho = nr > 0.f ? u - cv : 0.f;  // u - c[idx], and 0 for a zero vector
        acc[f][e2] = rho;
        if (row) rs1 = fmaf(rho, rho, rs1);
        else rs0 = fmaf(rho, rho, rs0);
        const uint32_t bit = 1u << ((f & 3) * 8 + 2 * tig + e);
#pragma unroll
        for (int p = 0; p < W; ++p)
          if ((idx >> p) & 1) wb[row][p] |= bit;
      }
      if ((f & 3) == 3) {  // a 32-coordinate word is complete for both rows
        const int word = col1 / 32 + f / 4;
#pragma unroll
        for (int p = 0; p < W; ++p) {
          const uint32_t w0 = quad_or(wb[0][p]), w1 = quad_or(wb[1][p]);
          if (tig == 0) {
            if (vr0 < a.n) a.idx[vr0 * wi + p * (d / 32) + word] = w0;
            if (vr1 < a.n) a.idx[vr1 * wi + p * (d / 32) + word] = w1;
          }
          wb[0][p] = wb[1][p] = 0u;
        }
      }
    }
  }
  rs0 += __shfl_xor_sync(0xffffffffu, rs0, 1);
  rs0 += __shfl_xor_sync(0xffffffffu, rs0, 2);
  rs1 += __shfl_xor_sync(0xffffffffu, rs1, 1);
  rs1 += __shfl_xor_sync(0xffffffffu, rs1, 2);
  if (tig == 0) {
    rsq[warp * kTV + gq] = rs0;
    rsq[warp * kTV + gq + 8] = rs1;
  }
  __syncthreads();  // every warp is done reading x's pieces
  // ---- ρ as bf16 pieces over x's
#pragma unroll
  for (int f = 0; f < kMaxNF; ++f) {
    if (f < nf1) {
      const int col = col1 + 8 * f + 2 * tig;
#pragma unroll
      for (int row = 0; row < 2; ++row) {
        const float r0 = acc[f][2 * row], r1 = acc[f][2 * row + 1];
        const uint32_t h = bf2(r0, r1);
        const float2 hf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&h));
        *reinterpret_cast<uint32_t*>(ah + (gq + 8 * row) * lda + col) = h;
        *reinterpret_cast<uint32_t*>(al + (gq + 8 * row) * lda + col) = bf2(r0 - hf.x, r1 - hf.y);
      }
    }
  }
  __syncthreads();

  if (m > 0) {
    // ---- P = ρ (S Πᵀ)ᵀ (= S r / n); σ = [P >= 0]
#pragma unroll
    for (int f = 0; f < kMaxNF; ++f)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[f][e] = 0.f;
    const int cw2 = words_per_warp(m), col2 = warp * cw2, nf2 = col2 < m ? min(cw2, m - col2) / 8 : 0;
    gemm_split(acc, ah, al, lda, a.s_fr, a.s_fr + (size_t)m * d / 4, d, m, col2, nf2, lane);
    uint32_t sb0 = 0u, sb1 = 0u;
#pragma unroll
    for (int f = 0; f < kMaxNF; ++f) {
      if (f < nf2) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const uint32_t bit = 1u << ((f & 3) * 8 + 2 * tig + e);
          if (acc[f][e] >= 0.f) sb0 |= bit;
          if (acc[f][2 + e] >= 0.f) sb1 |= bit;
        }
        if ((f & 3) == 3) {
          const int word = col2 / 32 + f / 4;
          const uint32_t w0 = quad_or(sb0), w1 = quad_or(sb1);
          if (tig == 0) {
            if (vr0 < a.n) a.sgn[vr0 * (m / 32) + word] = w0;
            if (vr1 < a.n) a.sgn[vr1 * (m / 32) + word] = w1;
          }
          sb0 = sb1 = 0u;
        }
      }
    }
  }
  // ---- norms
  if (threadIdx.x < kTV) {
    const int r = threadIdx.x;
    const int64_t v = v0 + r;
    if (v < a.n) {
      a.norm[v] = nrm[r];
      if (m > 0) {
        float s = 0.f;
        for (int q = 0; q < kWarps; ++q) s += rsq[q * kTV + r];
        a.rnorm[v] = nrm[r] * sqrtf(s);
      }
    }
  }
}

template <typename T, int W>
tq_status launch_mma(const MmaArgs& a, cudaStream_t st) {
  auto kern = quantize_mma_kernel<T, W>;
  const int smem = 2 * kTV * (a.d + kPad) * 2 + (kTV + kWarps * kTV) * 4;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return TQ_ERR_CUDA;
  kern<<<(unsigned)((a.n + kTV - 1) / kTV), kThreads, smem, st>>>(a);
  return tq::launch_status();
}

}  // namespace

bool tq::quantize_mma_supported(const tq_plan* plan, const tq_records* out) {
  return plan->d % 128 == 0 && plan->d <= 1024 && (plan->m == plan->d || plan->m == 0) &&
         out->layout == TQ_LAYOUT_ROWS && plan->pi_frag != nullptr && (plan->m == 0 || plan->s_frag != nullptr);
}

tq_status tq::quantize_mma(const tq_plan* plan, const void* x, tq_dtype dtype, int64_t n, int64_t ld_x,
                           const tq_records* out, int64_t row0, cudaStream_t st) {
  MmaArgs a{};
  a.x = x;
  a.n = n;
  a.ld = ld_x;
  a.d = plan->d;
  a.m = plan->m;
  a.pi_fr = reinterpret_cast<const uint2*>(plan->pi_frag);
  a.s_fr = reinterpret_cast<const uint2*>(plan->s_frag);
  a.centroids = plan->centroids;
  a.bounds = plan->bounds;
  a.idx = out->idx + row0 * (plan->w * plan->d / 32);
  a.sgn = plan->m > 0 ? out->sgn + row0 * (plan->m / 32) : nullptr;
  a.norm = out->norm + row0;
  a.rnorm = plan->m > 0 ? out->rnorm + row0 : nullptr;
  const bool f32 = dtype == TQ_F32;
  switch (plan->w) {
    case 1: return f32 ? launch_mma<float, 1>(a, st) : launch_mma<__nv_bfloat16, 1>(a, st);
    case 2: return f32 ? launch_mma<float, 2>(a, st) : launch_mma<__nv_bfloat16, 2>(a, st);
    default: return f32 ? launch_mma<float, 3>(a, st) : launch_mma<__nv_bfloat16, 3>(a, st);
  }
}

// tq_search_topk on the 5th-generation tensor cores (tcgen05) for wide
// records: d a multiple of 256 up to 1024, m = d or m = 0, w in 1..3,
// records in TQ_LAYOUT_ROWS, k <= 16.
//
// The score of stored vector i for query q ("TurboQuant压缩效果": vector
// search engines; the estimator of "TurboQuant 与 AI 效率革命" §三 applied to
// the residual as in "谷歌TurboQuant如何绕过内存墙？" §2 stage 2) is
//   score = ‖x_i‖ ⟨Π q, c[idx_i]⟩ + √(π/2)/m ‖r_i‖ ⟨S q, σ_i⟩.
// Over many queries and stored vectors both inner products are dense
// contractions.  Per unit of 128 queries (MMA M, one per TMEM lane) and 256
// stored vectors (MMA N):
//   A  [Π q | S q]·2^-E_q split into f16 hi + lo, one row per query (a table
//      built once per call, read by TMA in 128 x 64 boxes)
//   B  the centroid values c[idx] (f16 hi + lo, looked up per coordinate
//      pair in a 64-entry table) and the signs σ (exact ±1), expanded from
//      the record bits by producer warps into 256 x 64 operand stages
//   C  = A_hi·c_hi + A_lo·c_hi + A_hi·c_lo over the d coordinates, and
//   S  = A_hi·σ + A_lo·σ over the m sign coordinates, fp32 in TMEM
//   score = 2^E_q (‖x_i‖ C + α ‖r_i‖ S).
// A CTA keeps one block of 128 queries and walks every G-th unit of stored
// vectors; each epilogue thread owns one query and one half of the unit's
// columns and keeps its 16 best (score desc, index asc) in registers.  At the end the lists go to the
// workspace as candidates, which the merge kernel of tq_search.cu reduces to
// the k best: the nq x n score matrix is never formed.
//
// Warp roles (832 threads): warps 0-7 epilogue (warp % 4 = TMEM lane quadrant,
// warp / 4 = column half), 8-23 B producers, warp 24 TMA for A, warp 25 MMA
// issue and TMEM owner.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include <algorithm>

#include "tq_internal.h"
#include "tq_sm100.cuh"

namespace {

using namespace tq::sm100;

constexpr int kQ = 128;                        // queries per CTA (MMA M)
constexpr int kN = 256;                        // stored vectors per unit (MMA N)
constexpr int kKc = 64;                        // K columns per stage (one 128-byte swizzle atom)
constexpr int kPieceA = kQ * kKc * 2;          // 16 KB: one f16 piece of an A stage
constexpr int kSlotA = 2 * kPieceA;            // hi | lo
constexpr int kPieceB = kN * kKc * 2;          // 32 KB: one f16 piece of a B stage
constexpr int kSlotB = 2 * kPieceB;            // hi | lo (a sign stage uses the first piece)
constexpr int kNA = 3, kNB = 2;                // ring depths
constexpr int kOffA = 0, kOffB = kNA * kSlotA, kOffAux = kOffB + kNB * kSlotB;
constexpr int kOffBar = kOffAux;               // Bars (256 B)
constexpr int kOffPair = kOffBar + 256;        // [64] uint2: c of a coordinate pair, f16 hi pair and lo pair
constexpr int kSmemBytes = kOffPair + 64 * 8 + 1024;  // + alignment slack
constexpr int kEpiWarps = 8;                   // epilogue: two per TMEM lane quadrant
constexpr int kProdWarp0 = 8, kProdWarps = 16;  // B producers: warps 8 .. 23
constexpr int kTmaWarp = 24, kMmaWarp = 25, kThreads = 32 * 26;
constexpr int kList = 16;                      // list entries per query (k <= kList)
constexpr uint32_t kTmemCols = 512;            // C: columns 0..255, S: 256..511
constexpr unsigned kFaultSearch = 4u;          // fault bit: a pipeline wait ran out of its bound

static_assert(kSmemBytes <= 232448, "shared memory beyond the per-CTA limit");

struct Bars {
  uint64_t a_full[kNA], a_empty[kNA], b_full[kNB], b_empty[kNB];
  uint64_t acc_full, acc_empty;
  uint64_t drain;
  uint32_t tmem_base;
};
static_assert(sizeof(Bars) <= 256, "barriers must fit their shared-memory region");

struct SearchWideArgs {
  const uint32_t* idx; const uint32_t* sgn; const float* norm; const float* rnorm;
  int64_t n;
  int nq, d, m;
  float alpha;
  const float* centroids;  // [2^w]
  const float* qscale;     // [nq padded]: 2^E_q
  int qtiles, groups;      // query blocks; CTAs per query block (two candidate lists per query each)
  int64_t units;           // blocks of kN stored vectors
  int k;
  int32_t* cand_idx;       // [nq][2 groups][k]
  float* cand_sc;
  unsigned* fault;
};

__device__ __forceinline__ uint32_t h2(float lo, float hi) {
  const __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

// Byte offset of 16-byte chunk c (0..7) of row r in a 128-byte-swizzled
// K-major tile of 128-byte rows (8-row groups of 1024 bytes).
__device__ __forceinline__ uint32_t sw128(int r, int c) { return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4)); }

// Instruction descriptor, kind::f16: f16 x f16 -> f32, both K-major.
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N) {
  return (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// Eight signs (bit j = σ_j ≥ 0 of coordinate j) as f16 ±1.0, pairs (2t, 2t+1):
// bit set -> +1.0.
__device__ __forceinline__ uint4 signs8(uint32_t bits) {
  uint32_t r[4];
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const uint32_t b0 = (bits >> (2 * t)) & 1u, b1 = (bits >> (2 * t + 1)) & 1u;
    // 0x3C00 is +1.0; a clear bit sets the sign (0x8000)
    r[t] = 0x3C003C00u | ((b0 ^ 1u) << 15) | ((b1 ^ 1u) << 31);
  }
  return make_uint4(r[0], r[1], r[2], r[3]);
}

// One row per query: [Π q | S q]·2^-E_q as f16 hi pieces, then the lo pieces
// (rows past nq are zeros); qscale = 2^E_q, E_q the exponent that brings the
// row's largest magnitude into [0.5, 1).
__global__ void __launch_bounds__(256) search_wide_table_kernel(const float* qt, const float* st, int nq, int d, int m,
                                                                __half* table, float* qscale) {
  __shared__ float red[8];
  const int q = blockIdx.x, K = d + m;
  float mx = 0.f;
  if (q < nq)
    for (int j = threadIdx.x; j < K; j += blockDim.x)
      mx = fmaxf(mx, fabsf(j < d ? qt[(size_t)q * d + j] : st[(size_t)q * m + (j - d)]));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
  __syncthreads();
  mx = 0.f;
#pragma unroll
  for (int w = 0; w < 8; ++w) mx = fmaxf(mx, red[w]);
  int e = 0;
  if (mx > 0.f) frexpf(mx, &e);  // mx = f·2^e, f in [0.5, 1)
  const float sc = ldexpf(1.f, -e);
  __half* row = table + (size_t)q * 2 * K;
  for (int j = threadIdx.x; j < K; j += blockDim.x) {
    const float v = q < nq ? (j < d ? qt[(size_t)q * d + j] : st[(size_t)q * m + (j - d)]) * sc : 0.f;
    const __half hi = __float2half_rn(v);
    row[j] = hi;
    row[K + j] = __float2half_rn(v - __half2float(hi));
  }
  if (threadIdx.x == 0) qscale[q] = ldexpf(1.f, e);
}

template <int W, bool Q>
__global__ void __launch_bounds__(kThreads, 1)
    search_wide_kernel(const __grid_constant__ CUtensorMap tm_q, const SearchWideArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t base = smem_u32(smem);
  Bars* bars = reinterpret_cast<Bars*>(smem + kOffBar);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int d = a.d, m = a.m, K = d + m;
  const int KC = d / kKc, nst = KC + (Q ? m / kKc : 0);  // centroid stages, then sign stages
  const int qt = (int)(blockIdx.x % a.qtiles), g = (int)(blockIdx.x / a.qtiles);

  if (threadIdx.x == 0) {
    for (int i = 0; i < kNA; ++i) {
      mbar_init(smem_u32(&bars->a_full[i]), 1);
      mbar_init(smem_u32(&bars->a_empty[i]), 1);
    }
    for (int i = 0; i < kNB; ++i) {
      mbar_init(smem_u32(&bars->b_full[i]), kProdWarps);  // one arrival per producer warp
      mbar_init(smem_u32(&bars->b_empty[i]), 1);
    }
    mbar_init(smem_u32(&bars->acc_full), 1);
    mbar_init(smem_u32(&bars->acc_empty), kEpiWarps);
    mbar_init(smem_u32(&bars->drain), 1);
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(&bars->tmem_base), kTmemCols);
    tmem_relinquish();
  }
  if (warp == kTmaWarp && lane == 0) tma_prefetch_desc(&tm_q);
  // c over a pair of coordinates: entry bits (plane 0 of s, of s + 1, plane 1
  // of s, of s + 1, plane 2 of s, of s + 1), value (f16 hi pair, f16 lo pair)
  if (threadIdx.x >= 32 * kProdWarp0 && threadIdx.x < 32 * kProdWarp0 + 64) {
    const int e = threadIdx.x - 32 * kProdWarp0, L = 1 << W;
    const int i0 = ((e & 1) | ((e >> 2) & 1) << 1 | ((e >> 4) & 1) << 2) & (L - 1);
    const int i1 = (((e >> 1) & 1) | ((e >> 3) & 1) << 1 | ((e >> 5) & 1) << 2) & (L - 1);
    const float c0 = __ldg(a.centroids + i0), c1 = __ldg(a.centroids + i1);
    const uint32_t hi = h2(c0, c1);
    const __half2 hv = *reinterpret_cast<const __half2*>(&hi);
    reinterpret_cast<uint2*>(smem + kOffPair)[e] =
        make_uint2(hi, h2(c0 - __low2float(hv), c1 - __high2float(hv)));
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp == kTmaWarp) {
    if (lane == 0) {
      // the block's query rows: stage st reads columns 64·st of the hi pieces and of the lo pieces
      int64_t as = 0;
      bool ok = true;
      for (int64_t u = g; ok && u < a.units; u += a.groups) {
        for (int st = 0; st < nst; ++st) {
          const int s = (int)(as % kNA);
          if (!mbar_wait(smem_u32(&bars->a_empty[s]), ((uint32_t)(as / kNA) & 1u) ^ 1u, a.fault, kFaultSearch)) {
            ok = false;
            break;
          }
          const uint32_t full = smem_u32(&bars->a_full[s]), dst = base + kOffA + s * kSlotA;
          mbar_arrive_expect_tx(full, kSlotA);
          tma_load_2d(dst, &tm_q, st * kKc, qt * kQ, full);
          tma_load_2d(dst + kPieceA, &tm_q, K + st * kKc, qt * kQ, full);
          ++as;
        }
      }
      // no copy of this CTA may still be in flight when it exits
      for (int64_t j = as > kNA ? as - kNA : 0; j < as; ++j)
        mbar_wait(smem_u32(&bars->a_full[j % kNA]), (uint32_t)(j / kNA) & 1u, a.fault, kFaultSearch);
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16_f32(kQ, kN);
      int64_t as = 0, bs = 0;
      uint32_t uses = 0;
      bool ok = true;
      for (int64_t u = g; ok && u < a.units; u += a.groups, ++uses) {
        if (!mbar_wait(smem_u32(&bars->acc_empty), (uses & 1u) ^ 1u, a.fault, kFaultSearch)) break;
        tc_fence_after();
        for (int st = 0; st < nst; ++st) {
          const int sa = (int)(as % kNA), sb = (int)(bs % kNB);
          if (!mbar_wait(smem_u32(&bars->a_full[sa]), (uint32_t)(as / kNA) & 1u, a.fault, kFaultSearch) ||
              !mbar_wait(smem_u32(&bars->b_full[sb]), (uint32_t)(bs / kNB) & 1u, a.fault, kFaultSearch)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ah = desc_sw128(base + kOffA + sa * kSlotA), al = desc_sw128(base + kOffA + sa * kSlotA + kPieceA);
          const uint64_t bh = desc_sw128(base + kOffB + sb * kSlotB), bl = desc_sw128(base + kOffB + sb * kSlotB + kPieceB);
          // K-step ks: the start addresses advance 32 bytes (2 in 16-byte units)
          if (st < KC) {  // centroid values into C: a_hi c_hi + a_lo c_hi + a_hi c_lo
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) mma_ss(tmem, ah + 2 * ks, bh + 2 * ks, idesc, (st | ks) != 0);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) mma_ss(tmem, al + 2 * ks, bh + 2 * ks, idesc, 1u);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) mma_ss(tmem, ah + 2 * ks, bl + 2 * ks, idesc, 1u);
          } else {  // signs (exact ±1) into S: a_hi σ + a_lo σ
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) mma_ss(tmem + kN, ah + 2 * ks, bh + 2 * ks, idesc, ((st - KC) | ks) != 0);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) mma_ss(tmem + kN, al + 2 * ks, bh + 2 * ks, idesc, 1u);
          }
          mma_commit(smem_u32(&bars->b_empty[sb]));
          mma_commit(smem_u32(&bars->a_empty[sa]));
          ++as;
          ++bs;
        }
        if (!ok) break;
        mma_commit(smem_u32(&bars->acc_full));
      }
      // TMEM is released only once every product issued here has completed
      mma_commit(smem_u32(&bars->drain));
      mbar_wait(smem_u32(&bars->drain), 0u, a.fault, kFaultSearch);
    }
  } else if (warp >= kProdWarp0 && warp < kProdWarp0 + kProdWarps) {
    // B operands.  Warp pw fills rows r0 = 8pw + lane % 8 and r0 + 128 of a
    // stage, 16-byte chunks (8 coordinates) cc = lane / 8 and cc + 4 of each:
    // in every 8-lane phase the rows differ, so the swizzled writes meet no
    // bank conflicts.  The record words of a stage are loaded one stage ahead.
    const int pw = warp - kProdWarp0, cc = lane >> 3;
    const int r0 = 8 * pw + (lane & 7);
    const int wi = W * d / 32;
    const uint32_t pair_s = base + kOffPair;
    int64_t bs = 0;
    uint2 wn[2][W];  // the next stage's words (2kc, 2kc + 1) of rows r0, r0 + 128: planes, or signs in [h][0]
    auto load = [&](int64_t u, int st) {
      const int64_t v0 = u * kN;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int64_t v = v0 + r0 + 128 * h;
        const bool ok_v = v < a.n;
        if (st < KC) {
#pragma unroll
          for (int pl = 0; pl < W; ++pl)
            wn[h][pl] = ok_v ? __ldg(reinterpret_cast<const uint2*>(a.idx + v * wi + pl * (d / 32) + 2 * st))
                             : make_uint2(0u, 0u);
        } else {
          wn[h][0] = ok_v ? __ldg(reinterpret_cast<const uint2*>(a.sgn + v * (m / 32) + 2 * (st - KC)))
                          : make_uint2(0u, 0u);
        }
      }
    };
    // The next unit's record words are brought into L2 while this one is
    // expanded, so the loads above meet L2 rather than DRAM latency (one lane
    // of warp 0 issues the bulk prefetches, 16 KiB at a time, when the arrays
    // are 16-byte aligned as bulk copies require).
    const bool pf = pw == 0 && lane == 0 && (reinterpret_cast<uintptr_t>(a.idx) & 15) == 0 &&
                    (!Q || (reinterpret_cast<uintptr_t>(a.sgn) & 15) == 0);
    auto prefetch_unit = [&](int64_t uu) {
      if (!pf || uu >= a.units) return;
      const int64_t v0 = uu * kN, nv = a.n - v0 < kN ? a.n - v0 : kN;
      const char* pi = reinterpret_cast<const char*>(a.idx + v0 * wi);
      const int64_t bi = nv * wi * 4;  // rows of W·d/8 bytes: a multiple of 16
      for (int64_t o = 0; o < bi; o += 16384) bulk_prefetch_l2(pi + o, (uint32_t)(bi - o < 16384 ? bi - o : 16384));
      if (Q) {
        const char* ps = reinterpret_cast<const char*>(a.sgn + v0 * (m / 32));
        const int64_t bs = nv * (m / 8);
        for (int64_t o = 0; o < bs; o += 16384) bulk_prefetch_l2(ps + o, (uint32_t)(bs - o < 16384 ? bs - o : 16384));
      }
    };
    bool ok = true;
    int64_t u = g;
    int st = 0;
    if (u < a.units) load(u, st);
    prefetch_unit(u + a.groups);
    while (ok && u < a.units) {
      uint2 cw[2][W];
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int pl = 0; pl < W; ++pl) cw[h][pl] = wn[h][pl];
      const int cst = st;
      if (++st == nst) {
        st = 0;
        u += a.groups;
        prefetch_unit(u + a.groups);
      }
      if (u < a.units) load(u, st);
      const int sb = (int)(bs % kNB);
      if (!mbar_wait(smem_u32(&bars->b_empty[sb]), ((uint32_t)(bs / kNB) & 1u) ^ 1u, a.fault, kFaultSearch)) break;
      const uint32_t bh = base + kOffB + sb * kSlotB, bl = bh + kPieceB;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int r = r0 + 128 * h;
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const int c = cc + 4 * q;
          if (cst < KC) {
            uint32_t vb = 0u;  // byte pl: plane pl's bits of the chunk's 8 coordinates
#pragma unroll
            for (int pl = 0; pl < W; ++pl) vb |= ((q ? cw[h][pl].y : cw[h][pl].x) >> (8 * cc) & 0xFFu) << (8 * pl);
            uint32_t hv[4], lv[4];
#pragma unroll
            for (int t = 0; t < 4; ++t) {  // coordinates 2t, 2t + 1
              const uint32_t gb = (vb >> (2 * t)) & 0x030303u;
              const uint2 e = lds64(pair_s + 8 * ((gb | (gb >> 6) | (gb >> 12)) & 0x3Fu));
              hv[t] = e.x;
              lv[t] = e.y;
            }
            sts128(bh + sw128(r, c), make_uint4(hv[0], hv[1], hv[2], hv[3]));
            sts128(bl + sw128(r, c), make_uint4(lv[0], lv[1], lv[2], lv[3]));
          } else {
            sts128(bh + sw128(r, c), signs8((q ? cw[h][0].y : cw[h][0].x) >> (8 * cc) & 0xFFu));
          }
        }
      }
      // generic-proxy stores -> visible to the tensor core's reads
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bars->b_full[sb]));
      ++bs;
    }
  } else if (warp < kEpiWarps) {
    // Epilogue: thread = query 32·(warp % 4) + lane of the block (its TMEM
    // lane), columns 128·(warp / 4) .. + 127 of each unit.
    const int qd = warp & 3, hh = warp >> 2;
    const int qi = 32 * qd + lane;
    const int64_t qg = (int64_t)qt * kQ + qi;
    const uint32_t lane_base = static_cast<uint32_t>(32 * qd) << 16;
    float ls[kList];
    int32_t li[kList];
#pragma unroll
    for (int j = 0; j < kList; ++j) {
      ls[j] = -INFINITY;
      li[j] = -1;
    }
    uint32_t uses = 0;
    for (int64_t u = g; u < a.units; u += a.groups, ++uses) {
      // the norms of 32 columns at a time, lane l holding column 32J + l
      // (broadcast below by shuffles), loaded one block ahead
      const int64_t v0 = u * kN + 128 * hh;
      auto norms = [&](int J, float& nn, float& an) {
        const int64_t v = v0 + lane + 32 * J;
        nn = v < a.n ? __ldg(a.norm + v) : 0.f;
        an = Q && v < a.n ? a.alpha * __ldg(a.rnorm + v) : 0.f;
      };
      float nNext, aNext;
      norms(0, nNext, aNext);
      const int nv = a.n - v0 < 128 ? (int)(a.n - v0) : 128;  // stored vectors of this half (may be <= 0)
      if (!mbar_wait(smem_u32(&bars->acc_full), uses & 1u, a.fault, kFaultSearch)) break;
      tc_fence_after();
#pragma unroll 1
      for (int J = 0; J < 4; ++J) {
        const float nJ = nNext, aJ = aNext;
        if (J < 3) norms(J + 1, nNext, aNext);
#pragma unroll
        for (int jb = 0; jb < 8; ++jb) {
          const int c0 = 32 * J + 4 * jb;  // first column of these four, within the half
          uint32_t cv[4], sv[4];
          tmem_ld4(tmem + lane_base + 128 * hh + c0, cv);
          if (Q) tmem_ld4(tmem + lane_base + kN + 128 * hh + c0, sv);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float nrm = __shfl_sync(0xffffffffu, nJ, 4 * jb + j);
            float sc = nrm * __uint_as_float(cv[j]);
            if (Q) sc = fmaf(__shfl_sync(0xffffffffu, aJ, 4 * jb + j), __uint_as_float(sv[j]), sc);
            if (c0 + j < nv && sc > ls[kList - 1]) {
              // insertion: an equal score stays behind the earlier (lower) index
              float cs = sc;
              int32_t ci = (int32_t)(v0 + c0 + j);
#pragma unroll
              for (int e = 0; e < kList; ++e) {
                const bool sw = cs > ls[e];
                const float ts = ls[e];
                const int32_t ti = li[e];
                ls[e] = sw ? cs : ts;
                li[e] = sw ? ci : ti;
                cs = sw ? ts : cs;
                ci = sw ? ti : ci;
              }
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bars->acc_empty));
    }
    if (qg < a.nq) {
      const float qs = a.qscale[qg];
      const size_t o = ((size_t)qg * 2 * a.groups + 2 * g + hh) * a.k;
#pragma unroll
      for (int j = 0; j < kList; ++j) {
        if (j < a.k) {
          a.cand_idx[o + j] = li[j];
          a.cand_sc[o + j] = li[j] >= 0 ? ls[j] * qs : -INFINITY;
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int W, bool Q>
tq_status launch_wide(const CUtensorMap& mq, const SearchWideArgs& a, cudaStream_t st) {
  auto kern = search_wide_kernel<W, Q>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) != cudaSuccess)
    return TQ_ERR_CUDA;
  kern<<<a.qtiles * a.groups, kThreads, kSmemBytes, st>>>(mq, a);
  return tq::launch_status();
}

int qtiles_of(int nq) { return (nq + kQ - 1) / kQ; }
int groups_of(int nq) { return std::max(1, tq::sm_count() / qtiles_of(nq)); }

}  // namespace

bool tq::search_wide_supported(const tq_plan* plan, int k) {
  return plan->d % 256 == 0 && plan->d <= 1024 && (plan->m == 0 || plan->m == plan->d) && plan->w >= 1 &&
         plan->w <= 3 && k <= kList && tq::tensor_map_encoder() != nullptr;
}

int tq::search_wide_lists(int nq) { return 2 * groups_of(nq); }

size_t tq::search_wide_table_bytes(const tq_plan* plan, int nq) {
  const size_t rows = (size_t)qtiles_of(nq) * kQ;
  return (rows * 2 * (plan->d + plan->m) * sizeof(__half) + 255) / 256 * 256 + rows * sizeof(float);
}

tq_status tq::launch_search_wide(const tq_plan* plan, const tq_records* recs, int64_t n, int nq, const float* qt,
                                 const float* st, void* table, int k, int32_t* cand_idx, float* cand_sc,
                                 cudaStream_t stream) {
  const int d = plan->d, m = plan->m, qtiles = qtiles_of(nq);
  const size_t rows = (size_t)qtiles * kQ;
  __half* tab = static_cast<__half*>(table);
  float* qscale = reinterpret_cast<float*>(static_cast<char*>(table) +
                                           (rows * 2 * (d + m) * sizeof(__half) + 255) / 256 * 256);
  search_wide_table_kernel<<<(unsigned)rows, 256, 0, stream>>>(qt, st, nq, d, m, tab, qscale);
  tq_status s = tq::launch_status();
  if (s != TQ_OK) return s;
  CUtensorMap mq;
  if (!tq::map_bf16_tiles(&mq, tab, rows, 2 * (uint64_t)(d + m), 2 * (uint64_t)(d + m), kQ)) return TQ_ERR_CUDA;
  SearchWideArgs a{};
  a.idx = recs->idx;
  a.sgn = recs->sgn;
  a.norm = recs->norm;
  a.rnorm = recs->rnorm;
  a.n = n;
  a.nq = nq;
  a.d = d;
  a.m = m;
  a.alpha = plan->qjl_alpha;
  a.centroids = plan->centroids;
  a.qscale = qscale;
  a.qtiles = qtiles;
  a.groups = groups_of(nq);
  a.units = (n + kN - 1) / kN;
  a.k = k;
  a.cand_idx = cand_idx;
  a.cand_sc = cand_sc;
  a.fault = tq::fault_word();
  if (!a.fault) return TQ_ERR_CUDA;
  const bool q = m > 0;
  switch (plan->w) {
    case 1: return q ? launch_wide<1, true>(mq, a, stream) : launch_wide<1, false>(mq, a, stream);
    case 2: return q ? launch_wide<2, true>(mq, a, stream) : launch_wide<2, false>(mq, a, stream);
    default: return q ? launch_wide<3, true>(mq, a, stream) : launch_wide<3, false>(mq, a, stream);
  }
}

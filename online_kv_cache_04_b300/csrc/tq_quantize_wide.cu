// tq_quantize on the 5th-generation tensor cores (tcgen05) for wide vectors:
// d a multiple of 256 up to 1024, m = d or m = 0, fp32 or bf16 input, records
// in TQ_LAYOUT_ROWS.
//
// What is computed is the two-stage quantizer ("谷歌TurboQuant如何绕过内存墙？"
// §2 stages 1 and 2; "TurboQuant 与 AI 效率革命" §四 three-step pipeline):
// n = ||x||, u = Π x / n, idx = #{k : β_k < u}, ρ = u - c[idx],
// ||r|| = n ||ρ||, σ = [S r >= 0] with r = n Πᵀ ρ.
//
// At these widths the residual of a 128-vector tile (128 x d fp32, 512 KB at
// d = 1024) fits neither in shared memory nor in TMEM, and an MMA needs 128
// vectors on M to run at full rate.  So the sign stage does not read ρ: with
// S = (S Πᵀ) Π,
//     S r / n = S x / n - (S Πᵀ) c[idx],
// a contraction of the input (streamed again) and of the centroid values of
// the index planes just written, accumulated in one TMEM slot.  Its rounding
// error is that of the products at the scale ||x / n|| = 1, the same order as
// the error U = x Πᵀ already passes on to ρ.
//
// Every product runs in bf16 pieces with fp32 accumulation: a = a_hi + a_lo
// and M = M_hi + M_lo, a·Mᵀ ≈ a_hi M_hiᵀ + a_lo M_hiᵀ + a_hi M_loᵀ (the
// dropped a_lo M_loᵀ and the rest beyond 16 bits are ~2^-17 relative; bf16
// input is exact in a_hi, so its first contraction has no a_lo term).
//
// A CTA owns 128-vector tiles (persistent).  Per tile, d/256 passes of 256
// columns of U = x Πᵀ, then m/256 passes of 256 columns of
// P = (x/n)·Sᵀ + (-c[idx])·(S Πᵀ)ᵀ (K = 2d: the input's columns, then the
// centroid values'), each pass into one of two 256-column TMEM slots so that
// the epilogue of one pass overlaps the products of the next.  Warp roles
// (864 threads):
//   warps 0-3   epilogue of the U passes (warp = TMEM lane quadrant = 32
//               vectors): u = U / n, binary-search bucketize into index
//               planes, ||ρ||², ||r||
//   warps 4-7   epilogue of the P passes: sign words (idle when m = 0)
//   warps 8-23  A operands, 128 rows x 64 columns per stage, 128-byte
//               swizzled K-major: x (or x / n) split into bf16 hi and lo, or
//               the centroid values -c[idx] (hi, lo) looked up per pair of
//               coordinates in a 64-entry table; the first U pass reads
//               every column of the tile once, so it also yields ||x||
//   warp 24     B operands by TMA: 256 rows x 64 columns of Π, S or S Πᵀ,
//               hi or lo, per stage
//   warp 25     MMA issue (one thread), TMEM owner
//   warp 26     the input's columns by TMA into a raw ring, and the next
//               tile's rows into L2 during the last pass
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <algorithm>

#include "tq_internal.h"
#include "tq_sm100.cuh"

namespace {

using namespace tq::sm100;

constexpr int kTile = 128;                        // vectors per tile (MMA M)
constexpr int kCols = 256;                        // output columns per pass (MMA N)
constexpr int kKc = 64;                           // K columns per stage (one 128-byte swizzle atom)
constexpr int kPieceA = kTile * kKc * 2;          // 16 KB: one bf16 piece of an A stage
constexpr int kSlotA = 2 * kPieceA;               // hi | lo
constexpr int kSlotR = kTile * kKc * 4;           // 32 KB: the raw input of a stage (fp32 at most)
constexpr int kSlotB = kCols * kKc * 2;           // 32 KB: one bf16 piece of a B stage
constexpr int kNA = 2, kNR = 2, kNB = 3;          // ring depths
constexpr int kOffA = 0, kOffR = kNA * kSlotA, kOffB = kOffR + kNR * kSlotR, kOffAux = kOffB + kNB * kSlotB;
constexpr int kOffBar = kOffAux;                  // Bars (256 B)
constexpr int kOffNrm = kOffBar + 256;            // [tile parity 2][128] ||x||
constexpr int kOffCtab = kOffNrm + 2 * kTile * 4; // [64] uint2: -c of a coordinate pair, bf16 hi and lo
constexpr int kSmemBytes = kOffCtab + 64 * 8 + 1024;  // + alignment slack
constexpr int kProdWarp0 = 8, kProdWarps = 16;  // A-operand producers: warps 8 .. 23
constexpr int kTmaWarp = 24, kMmaWarp = 25, kRawWarp = 26, kThreads = 32 * 27;
constexpr uint32_t kTmemCols = 512;               // two 256-column accumulator slots
constexpr unsigned kFaultWait = 1u;               // fault bit: a pipeline wait ran out of its bound

static_assert(kSmemBytes <= 232448, "shared memory beyond the per-CTA limit");

// A slot is filled by U passes and P passes in turn, so each epilogue group
// has its own "full" barrier per slot (a parity wait is only exact one phase
// ahead); "empty" takes the arrivals of whichever group read the slot, in
// pass order.
struct Bars {
  uint64_t a_full[kNA], a_empty[kNA], r_full[kNR], r_empty[kNR], b_full[kNB], b_empty[kNB];
  uint64_t u_full[2], p_full[2], acc_empty[2];
  uint64_t norm_ready;  // the tile's norms are in shared memory
  uint64_t idx_ready;   // the tile's index planes are in global memory
  uint64_t drain;       // every MMA of this CTA has completed
  uint32_t tmem_base;
};
static_assert(sizeof(Bars) <= 256, "barriers must fit their shared-memory region");

struct WideArgs {
  const void* x;
  int64_t n, ld, ntiles;
  int d, m;
  const float* centroids;  // device [2^w]
  const float* bounds;     // device [2^w - 1]
  uint32_t* idx;           // rows already offset
  uint32_t* sgn;
  float* norm;
  float* rnorm;
  unsigned* fault;
};

// The stage sequence of a tile, shared by the four roles: pass p < P1 is a U
// pass (K = d, the input), pass p >= P1 a P pass (K = 2d: the input scaled by
// 1/n, then the centroid values).
struct Sched {
  int P1, P2, KC;  // U passes, P passes, K stages of d columns
  __device__ int passes() const { return P1 + P2; }
  __device__ int stages(int p) const { return p < P1 ? KC : 2 * KC; }
};

__device__ __forceinline__ uint32_t bf2(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Eight floats -> their bf16 hi pieces and the bf16 pieces of the remainders.
__device__ __forceinline__ void split8(const float (&f)[8], uint4& hi, uint4& lo) {
  uint32_t h[4], l[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    h[j] = bf2(f[2 * j], f[2 * j + 1]);
    const float h0 = __uint_as_float(h[j] << 16), h1 = __uint_as_float(h[j] & 0xFFFF0000u);
    l[j] = bf2(f[2 * j] - h0, f[2 * j + 1] - h1);
  }
  hi = make_uint4(h[0], h[1], h[2], h[3]);
  lo = make_uint4(l[0], l[1], l[2], l[3]);
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}
__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

// Byte offset of 16-byte chunk c (0..7) of row r in a 128-byte-swizzled
// K-major tile of 128-byte rows (8-row groups of 1024 bytes).
__device__ __forceinline__ uint32_t sw128(int r, int c) { return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4)); }

template <typename T, int W, bool Q>
__global__ void __launch_bounds__(kThreads, 1)
    quantize_wide_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_pi,
                         const __grid_constant__ CUtensorMap tm_s, const __grid_constant__ CUtensorMap tm_sr,
                         const WideArgs a) {
  constexpr bool kBf16 = sizeof(T) == 2;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t base = smem_u32(smem);
  Bars* bars = reinterpret_cast<Bars*>(smem + kOffBar);
  float* nrm_s = reinterpret_cast<float*>(smem + kOffNrm);
  uint2* ctab = reinterpret_cast<uint2*>(smem + kOffCtab);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int d = a.d, m = a.m;
  const Sched sc{d / kCols, Q ? m / kCols : 0, d / kKc};

  if (threadIdx.x == 0) {
    for (int i = 0; i < kNA; ++i) {
      mbar_init(smem_u32(&bars->a_full[i]), kProdWarps);  // one arrival per producer warp
      mbar_init(smem_u32(&bars->a_empty[i]), 1);
    }
    for (int i = 0; i < kNR; ++i) {
      mbar_init(smem_u32(&bars->r_full[i]), 1);
      mbar_init(smem_u32(&bars->r_empty[i]), kProdWarps);  // one arrival per producer warp
    }
    for (int i = 0; i < kNB; ++i) {
      mbar_init(smem_u32(&bars->b_full[i]), 1);
      mbar_init(smem_u32(&bars->b_empty[i]), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&bars->u_full[s]), 1);
      mbar_init(smem_u32(&bars->p_full[s]), 1);
      mbar_init(smem_u32(&bars->acc_empty[s]), 4);  // the four warps of the pass's epilogue group
    }
    mbar_init(smem_u32(&bars->norm_ready), kProdWarps);
    mbar_init(smem_u32(&bars->idx_ready), 4);
    mbar_init(smem_u32(&bars->drain), 1);
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(&bars->tmem_base), kTmemCols);
    tmem_relinquish();
  }
  if (warp == kTmaWarp && lane == 0) {
    tma_prefetch_desc(&tm_pi);
    if (Q) {
      tma_prefetch_desc(&tm_s);
      tma_prefetch_desc(&tm_sr);
    }
  }
  if (warp == kRawWarp && lane == 0) tma_prefetch_desc(&tm_x);
  // -c over a pair of coordinates: entry bits (plane 0 of s, of s + 1, plane 1
  // of s, of s + 1, plane 2 of s, of s + 1), value (bf16 hi pair, bf16 lo pair)
  if (Q && threadIdx.x >= 32 * kProdWarp0 && threadIdx.x < 32 * kProdWarp0 + 64) {
    const int e = threadIdx.x - 32 * kProdWarp0, L = 1 << W;
    const int i0 = ((e & 1) | ((e >> 2) & 1) << 1 | ((e >> 4) & 1) << 2) & (L - 1);
    const int i1 = (((e >> 1) & 1) | ((e >> 3) & 1) << 1 | ((e >> 5) & 1) << 2) & (L - 1);
    const float c0 = -__ldg(a.centroids + i0), c1 = -__ldg(a.centroids + i1);
    const uint32_t h = bf2(c0, c1);
    ctab[e] = make_uint2(h, bf2(c0 - __uint_as_float(h << 16), c1 - __uint_as_float(h & 0xFFFF0000u)));
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp == kTmaWarp) {
    if (lane == 0) {
      int64_t bs = 0;  // B stages issued
      bool ok = true;
      for (int64_t tile = blockIdx.x; ok && tile < a.ntiles; tile += gridDim.x) {
        for (int p = 0; ok && p < sc.passes(); ++p) {
          const bool u = p < sc.P1;
          const int pp = u ? p : p - sc.P1, rows = u ? d : m;
          for (int k = 0; ok && k < sc.stages(p); ++k) {
            // Π for U; S for the input columns of P, S Πᵀ for its centroid columns
            const CUtensorMap* tm = u ? &tm_pi : (k < sc.KC ? &tm_s : &tm_sr);
            const int kc = k < sc.KC ? k : k - sc.KC;
            for (int piece = 0; piece < 2; ++piece) {
              const int s = (int)(bs % kNB);
              if (!mbar_wait(smem_u32(&bars->b_empty[s]), ((uint32_t)(bs / kNB) & 1u) ^ 1u, a.fault, kFaultWait)) {
                ok = false;
                break;
              }
              const uint32_t full = smem_u32(&bars->b_full[s]);
              mbar_arrive_expect_tx(full, kSlotB);
              tma_load_2d(base + kOffB + s * kSlotB, tm, kc * kKc, piece * rows + pp * kCols, full);
              ++bs;
            }
          }
        }
      }
      // no copy of this CTA may still be in flight when it exits
      for (int64_t j = bs > kNB ? bs - kNB : 0; j < bs; ++j)
        mbar_wait(smem_u32(&bars->b_full[j % kNB]), (uint32_t)(j / kNB) & 1u, a.fault, kFaultWait);
    }
  } else if (warp == kRawWarp) {
    if (lane == 0) {
      // The input's columns of every stage that reads them, by TMA (rows past
      // n read as zeros), and the next tile's rows into L2 ahead of its first
      // pass: once its input columns are all issued, in the last pass.
      const T* x = static_cast<const T*>(a.x);
      auto prefetch_tile = [&](int64_t tile) {
        for (int r = 0; r < kTile; ++r) {
          const int64_t v = tile * kTile + r;
          if (v < a.n) bulk_prefetch_l2(x + v * a.ld, (uint32_t)(d * sizeof(T)));
        }
      };
      if (blockIdx.x < a.ntiles) prefetch_tile(blockIdx.x);
      int64_t rs = 0;  // raw stages issued
      bool ok = true;
      for (int64_t tile = blockIdx.x; ok && tile < a.ntiles; tile += gridDim.x) {
        for (int p = 0; ok && p < sc.passes(); ++p) {
          for (int k = 0; ok && k < sc.KC; ++k) {
            const int s = (int)(rs % kNR);
            if (!mbar_wait(smem_u32(&bars->r_empty[s]), ((uint32_t)(rs / kNR) & 1u) ^ 1u, a.fault, kFaultWait)) {
              ok = false;
              break;
            }
            const uint32_t full = smem_u32(&bars->r_full[s]);
            mbar_arrive_expect_tx(full, kTile * kKc * (uint32_t)sizeof(T));
            // 128-byte rows: fp32 in two 32-column halves, bf16 in one box
            for (int h = 0; h < (int)sizeof(T) / 2; ++h)
              tma_load_2d(base + kOffR + s * kSlotR + h * (kSlotR / 2), &tm_x, k * kKc + h * 32,
                          (int32_t)(tile * kTile), full);
            ++rs;
            const bool last = p == sc.passes() - 1;
            if (last && k == (Q ? sc.KC - 1 : sc.KC / 2) && tile + gridDim.x < a.ntiles)
              prefetch_tile(tile + gridDim.x);
          }
        }
      }
      for (int64_t j = rs > kNR ? rs - kNR : 0; j < rs; ++j)
        mbar_wait(smem_u32(&bars->r_full[j % kNR]), (uint32_t)(j / kNR) & 1u, a.fault, kFaultWait);
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(kTile, kCols);
      int64_t as = 0, bs = 0, gp = 0;  // A stages, B stages, passes consumed
      bool ok = true;
      for (int64_t tile = blockIdx.x; ok && tile < a.ntiles; tile += gridDim.x) {
        for (int p = 0; ok && p < sc.passes(); ++p, ++gp) {
          const int slot = (int)(gp & 1);
          if (!mbar_wait(smem_u32(&bars->acc_empty[slot]), ((uint32_t)(gp >> 1) & 1u) ^ 1u, a.fault, kFaultWait)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t acc = tmem + kCols * slot;
          const bool lo_terms = !(kBf16 && p < sc.P1);  // bf16 input is exact in its hi piece
          for (int k = 0; ok && k < sc.stages(p); ++k) {
            const int sa = (int)(as % kNA);
            if (!mbar_wait(smem_u32(&bars->a_full[sa]), (uint32_t)(as / kNA) & 1u, a.fault, kFaultWait)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t ah = desc_sw128(base + kOffA + sa * kSlotA);
            const uint64_t al = desc_sw128(base + kOffA + sa * kSlotA + kPieceA);
            for (int piece = 0; piece < 2; ++piece) {
              const int sb = (int)(bs % kNB);
              if (!mbar_wait(smem_u32(&bars->b_full[sb]), (uint32_t)(bs / kNB) & 1u, a.fault, kFaultWait)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint64_t bd = desc_sw128(base + kOffB + sb * kSlotB);
              // K-step ks: the start address advances 32 bytes (2 in 16-byte units)
              if (piece == 0) {  // M_hi: a_hi and a_lo
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) mma_ss(acc, ah + 2 * ks, bd + 2 * ks, idesc, (k | ks) != 0);
                if (lo_terms) {
#pragma unroll
                  for (int ks = 0; ks < 4; ++ks) mma_ss(acc, al + 2 * ks, bd + 2 * ks, idesc, 1u);
                }
              } else {  // M_lo: a_hi
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) mma_ss(acc, ah + 2 * ks, bd + 2 * ks, idesc, 1u);
              }
              mma_commit(smem_u32(&bars->b_empty[sb]));
              ++bs;
            }
            if (!ok) break;
            mma_commit(smem_u32(&bars->a_empty[sa]));
            ++as;
          }
          if (!ok) break;
          mma_commit(smem_u32(p < sc.P1 ? &bars->u_full[slot] : &bars->p_full[slot]));
        }
      }
      // TMEM is released only once every product issued here has completed
      mma_commit(smem_u32(&bars->drain));
      mbar_wait(smem_u32(&bars->drain), 0u, a.fault, kFaultWait);
    }
  } else if (warp >= kProdWarp0 && warp < kProdWarp0 + kProdWarps) {
    // A operands.  Warp pw fills row r = 8pw + lane % 8, 16-byte chunks (8
    // columns) cc = lane / 8 and cc + 4: in every 8-lane phase the rows
    // differ, so the 128-byte-swizzled reads and writes meet no bank conflicts.  The input's columns arrive in the raw ring by
    // TMA (128-byte swizzled rows: fp32 as two 32-column halves, bf16 as one
    // box); the index-plane words of a centroid stage are loaded one stage
    // ahead.
    const int pw = warp - kProdWarp0, cc = lane >> 3;
    const int r = 8 * pw + (lane & 7);
    const int wi = W * d / 32;
    const int ust = sc.P1 * sc.KC, nst = ust + sc.P2 * 2 * sc.KC;  // A stages per tile
    int64_t as = 0, rs = 0;  // A stages filled, raw stages consumed
    float ss = 0.f, inv = 0.f;
    uint2 wn[W];             // plane words (2kc, 2kc + 1) of row r for the next centroid stage
#pragma unroll
    for (int pl = 0; pl < W; ++pl) wn[pl] = make_uint2(0u, 0u);
    const uint32_t ctab_s = smem_u32(ctab);
    auto stage_pk = [&](int st, int& p, int& k) {
      if (st < ust) {
        p = st / sc.KC;
        k = st - p * sc.KC;
      } else {
        const int s2 = st - ust;
        p = sc.P1 + s2 / (2 * sc.KC);
        k = s2 - (p - sc.P1) * 2 * sc.KC;
      }
    };
    bool ok = true;
    int it = 0;
    int pending_r = -1;  // raw slot read by the stage just published
    for (int64_t tile = blockIdx.x; ok && tile < a.ntiles; tile += gridDim.x, ++it) {
      const int64_t v0 = tile * kTile;  // row r of the tile is vector v0 + r
      for (int st = 0; st < nst; ++st) {
        int p, k;
        stage_pk(st, p, k);
        const bool u = p < sc.P1;
        // items q: chunk cc + 4q of row r
        float f[2][8];
        if (k < sc.KC) {  // input columns k·64 .. from the raw ring
          const int rsl = (int)(rs % kNR);
          if (!mbar_wait(smem_u32(&bars->r_full[rsl]), (uint32_t)(rs / kNR) & 1u, a.fault, kFaultWait)) {
            ok = false;
            break;
          }
          const uint32_t raw = base + kOffR + rsl * kSlotR;
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const int c = cc + 4 * q;
            if constexpr (kBf16) {
              const uint4 w4 = lds128(raw + sw128(r, c));
              const uint32_t wv[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                f[q][2 * j] = __uint_as_float(wv[j] << 16);
                f[q][2 * j + 1] = __uint_as_float(wv[j] & 0xFFFF0000u);
              }
            } else {  // columns 8c .. 8c + 7: half c / 4, chunks 2(c % 4) and 2(c % 4) + 1 of its row
              const uint32_t hb = raw + (c >> 2) * (kSlotR / 2);
              const uint4 w0 = lds128(hb + sw128(r, 2 * (c & 3))), w1 = lds128(hb + sw128(r, 2 * (c & 3) + 1));
              f[q][0] = __uint_as_float(w0.x); f[q][1] = __uint_as_float(w0.y);
              f[q][2] = __uint_as_float(w0.z); f[q][3] = __uint_as_float(w0.w);
              f[q][4] = __uint_as_float(w1.x); f[q][5] = __uint_as_float(w1.y);
              f[q][6] = __uint_as_float(w1.z); f[q][7] = __uint_as_float(w1.w);
            }
          }
          pending_r = rsl;
          ++rs;
          if (p == 0) {  // the first U pass sees every column once: ||x||² on the way
            if (k == 0) ss = 0.f;
#pragma unroll
            for (int q = 0; q < 2; ++q) {
              float s8 = 0.f;
#pragma unroll
              for (int j = 0; j < 8; ++j) s8 = fmaf(f[q][j], f[q][j], s8);
              ss += s8;
            }
          }
          if (!u) {
#pragma unroll
            for (int q = 0; q < 2; ++q)
#pragma unroll
              for (int j = 0; j < 8; ++j) f[q][j] *= inv;
          }
        }
        const int sa = (int)(as % kNA);
        if (!mbar_wait(smem_u32(&bars->a_empty[sa]), ((uint32_t)(as / kNA) & 1u) ^ 1u, a.fault, kFaultWait)) {
          ok = false;
          break;
        }
        const uint32_t hi = base + kOffA + sa * kSlotA, lo = hi + kPieceA;
        if (k < sc.KC) {  // x for U, x / n for P, split into bf16 hi and lo
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const int c = cc + 4 * q;
            uint4 h4, l4;
            split8(f[q], h4, l4);
            sts128(hi + sw128(r, c), h4);
            if (!(kBf16 && u)) sts128(lo + sw128(r, c), l4);
          }
        } else {  // centroid columns (k - KC)·64 ..: -c[idx] from the index planes
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const int c = cc + 4 * q;
            uint32_t vb = 0u;  // byte pl: plane pl's bits of the chunk's 8 coordinates
#pragma unroll
            for (int pl = 0; pl < W; ++pl) vb |= ((q ? wn[pl].y : wn[pl].x) >> (8 * cc) & 0xFFu) << (8 * pl);
            uint32_t h[4], l[4];
#pragma unroll
            for (int t = 0; t < 4; ++t) {  // coordinates 2t, 2t + 1
              const uint32_t g = (vb >> (2 * t)) & 0x030303u;
              const uint2 e = lds64(ctab_s + 8 * ((g | (g >> 6) | (g >> 12)) & 0x3Fu));
              h[t] = e.x;
              l[t] = e.y;
            }
            sts128(hi + sw128(r, c), make_uint4(h[0], h[1], h[2], h[3]));
            sts128(lo + sw128(r, c), make_uint4(l[0], l[1], l[2], l[3]));
          }
        }
        // One proxy fence orders this stage's generic-proxy accesses before the
        // async proxy's: the A stores before the tensor core reads them, and
        // the raw reads before the next TMA write into that raw slot.
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(smem_u32(&bars->a_full[sa]));
          if (pending_r >= 0) mbar_arrive(smem_u32(&bars->r_empty[pending_r]));
        }
        pending_r = -1;
        ++as;
        if (Q && st + 1 < nst) {  // the next stage's index words, when it is a centroid stage
          int p1, k1;
          stage_pk(st + 1, p1, k1);
          if (k1 >= sc.KC) {
            if (p1 == sc.P1 && k1 == sc.KC &&  // the tile's planes must be written first
                !mbar_wait(smem_u32(&bars->idx_ready), (uint32_t)it & 1u, a.fault, kFaultWait)) {
              ok = false;
              break;
            }
            const int kc = k1 - sc.KC;
            const int64_t v = v0 + r;
#pragma unroll
            for (int pl = 0; pl < W; ++pl)
              wn[pl] = v < a.n ? __ldcg(reinterpret_cast<const uint2*>(a.idx + v * wi + pl * (d / 32) + 2 * kc))
                               : make_uint2(0u, 0u);
          }
        }
        if (p == 0 && k == sc.KC - 1) {
          // the four lanes of a row (cc = 0..3) hold its eight column chunks: the norms
          float* nrm = nrm_s + (it & 1) * kTile;
          float t = ss;
          t += __shfl_xor_sync(0xffffffffu, t, 8);
          t += __shfl_xor_sync(0xffffffffu, t, 16);
          const float nn = sqrtf(t);
          inv = nn > 0.f ? 1.0f / nn : 0.f;
          if (cc == 0) {
            nrm[r] = nn;
            if (v0 + r < a.n) a.norm[v0 + r] = nn;
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&bars->norm_ready));
        }
      }
    }
  } else {
    // Epilogues.  Warps 0-3 take the U passes, 4-7 the P passes; warp % 4 is
    // the TMEM lane quadrant, thread = one vector, all 256 columns of a pass.
    const int q = warp & 3, r = 32 * q + lane;
    const bool sign_group = warp >= 4;
    const int wi = W * d / 32;
    float cent[8], bnd[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      cent[k] = k < (1 << W) ? __ldg(a.centroids + k) : 0.f;
      bnd[k] = k < (1 << W) - 1 ? __ldg(a.bounds + k) : 0.f;
    }
    const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
    int64_t gp = 0;          // passes seen (both groups count all of them: slot = gp % 2)
    uint32_t uses[2] = {0u, 0u};  // this group's passes so far in each slot
    int it = 0;
    if (!sign_group || Q) {
      for (int64_t tile = blockIdx.x; tile < a.ntiles; tile += gridDim.x, ++it) {
        const int64_t v = tile * kTile + r;
        const bool valid = v < a.n;
        if (!mbar_wait(smem_u32(&bars->norm_ready), (uint32_t)it & 1u, a.fault, kFaultWait)) break;
        const float n = nrm_s[(it & 1) * kTile + r];
        bool ok = true;
        if (!sign_group) {
          const float inv = n > 0.f ? 1.0f / n : 0.f, nlive = n > 0.f ? -1.f : 0.f;
          const uint64_t inv2 = f2_pack(inv, inv), nlive2 = f2_pack(nlive, nlive);
          uint64_t rsq2 = 0ull;
          for (int p = 0; p < sc.P1; ++p, ++gp) {
            const int slot = (int)(gp & 1);
            if (!mbar_wait(smem_u32(&bars->u_full[slot]), uses[slot]++ & 1u, a.fault, kFaultWait)) {
              ok = false;
              break;
            }
            tc_fence_after();
            uint32_t* oidx = a.idx + v * wi + p * 8;  // word j of plane pl at pl·(d/32) + j
#pragma unroll 1
            for (int j = 0; j < 8; ++j) {
              uint32_t pw[W];
#pragma unroll
              for (int pl = 0; pl < W; ++pl) pw[pl] = 0u;
#pragma unroll
              for (int half = 0; half < 2; ++half) {  // 16 columns per TMEM load
              uint32_t uv[16];
              tmem_ld16(tmem + lane_base + kCols * slot + 32 * j + 16 * half, uv);
              tmem_ld_wait();
#pragma unroll
              for (int jj = 8 * half; jj < 8 * half + 8; ++jj) {
                const uint64_t u2 = f2_mul(f2_pack(__uint_as_float(uv[2 * jj - 16 * half]),
                                                   __uint_as_float(uv[2 * jj + 1 - 16 * half])), inv2);
                const float2 uu = f2_unpack(u2);
                float cv[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                  const float uo = e ? uu.y : uu.x;
                  // idx = #{k : bound_k < u} by binary search over the sorted
                  // bounds; the branch taken at level l is bit W-1-l of idx
                  const uint32_t bit = 1u << (2 * jj + e);
                  if constexpr (W == 1) {
                    const bool p0 = uo > bnd[0];
                    cv[e] = p0 ? cent[1] : cent[0];
                    if (p0) pw[0] |= bit;
                  } else if constexpr (W == 2) {
                    const bool p1 = uo > bnd[1];
                    const bool p0 = uo > (p1 ? bnd[2] : bnd[0]);
                    const float chi = p1 ? cent[3] : cent[1], clo = p1 ? cent[2] : cent[0];
                    cv[e] = p0 ? chi : clo;
                    if (p1) pw[1] |= bit;
                    if (p0) pw[0] |= bit;
                  } else {
                    const bool p2 = uo > bnd[3];
                    const bool p1 = uo > (p2 ? bnd[5] : bnd[1]);
                    const bool p0 = uo > (p2 ? (p1 ? bnd[6] : bnd[4]) : (p1 ? bnd[2] : bnd[0]));
                    const float codd = p2 ? (p1 ? cent[7] : cent[5]) : (p1 ? cent[3] : cent[1]);
                    const float cevn = p2 ? (p1 ? cent[6] : cent[4]) : (p1 ? cent[2] : cent[0]);
                    cv[e] = p0 ? codd : cevn;
                    if (p2) pw[2] |= bit;
                    if (p1) pw[1] |= bit;
                    if (p0) pw[0] |= bit;
                  }
                }
                if (Q) {
                  const uint64_t rho2 = f2_fma(f2_pack(cv[0], cv[1]), nlive2, u2);  // u - c[idx]; 0 for a zero vector
                  rsq2 = f2_fma(rho2, rho2, rsq2);
                }
              }
              }
              if (valid) {
#pragma unroll
                for (int pl = 0; pl < W; ++pl) oidx[pl * (d / 32) + j] = pw[pl];
              }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bars->acc_empty[slot]));
          }
          if (!ok) break;
          gp += sc.P2;
          if (Q) {
            // the P passes' centroid columns read these planes back
            __threadfence_block();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bars->idx_ready));
            const float2 rs = f2_unpack(rsq2);
            if (valid) a.rnorm[v] = n * sqrtf(rs.x + rs.y);
          }
        } else {
          gp += sc.P1;
          for (int p = 0; p < sc.P2; ++p, ++gp) {
            const int slot = (int)(gp & 1);
            if (!mbar_wait(smem_u32(&bars->p_full[slot]), uses[slot]++ & 1u, a.fault, kFaultWait)) {
              ok = false;
              break;
            }
            tc_fence_after();
            uint32_t* osgn = a.sgn + v * (m / 32) + p * 8;
#pragma unroll 1
            for (int j = 0; j < 8; ++j) {
              uint32_t pv[32];
              tmem_ld32(tmem + lane_base + kCols * slot + 32 * j, pv);
              tmem_ld_wait();
              // bit i = [P_i >= 0]: the sign bits shifted in from the top row
              // down, then inverted; a zero vector (P = 0) takes all ones
              uint32_t neg = 0u;
#pragma unroll
              for (int i = 31; i >= 0; --i) neg = __funnelshift_l(pv[i], neg, 1);
              if (valid) osgn[j] = n > 0.f ? ~neg : 0xFFFFFFFFu;
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bars->acc_empty[slot]));
          }
          if (!ok) break;
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

struct WideMaps {
  CUtensorMap x, pi, s, sr;
};

template <typename T, int W, bool Q>
tq_status launch_wide(const WideMaps& mp, const WideArgs& a, cudaStream_t st) {
  auto kern = quantize_wide_kernel<T, W, Q>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) != cudaSuccess)
    return TQ_ERR_CUDA;
  const int grid = (int)std::min<int64_t>(a.ntiles, tq::sm_count());
  kern<<<grid, kThreads, kSmemBytes, st>>>(mp.x, mp.pi, mp.s, mp.sr, a);
  return tq::launch_status();
}

template <typename T>
tq_status launch_wide_t(int w, bool q, const WideMaps& mp, const WideArgs& a, cudaStream_t st) {
  switch (w) {
    case 1: return q ? launch_wide<T, 1, true>(mp, a, st) : launch_wide<T, 1, false>(mp, a, st);
    case 2: return q ? launch_wide<T, 2, true>(mp, a, st) : launch_wide<T, 2, false>(mp, a, st);
    default: return q ? launch_wide<T, 3, true>(mp, a, st) : launch_wide<T, 3, false>(mp, a, st);
  }
}

// Input rows by TMA: n x d elements of row stride ld, boxes of 128-byte rows
// (32 fp32 or 64 bf16 columns) x 128 rows, 128-byte swizzle (rows past n read
// as zeros).
bool map_input(CUtensorMap* map, const void* x, tq_dtype dtype, int64_t n, int d, int64_t ld) {
  auto fn = tq::tensor_map_encoder();
  if (!fn) return false;
  const size_t esz = dtype == TQ_F32 ? 4 : 2;
  cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)n};
  cuuint64_t strides[1] = {(cuuint64_t)ld * esz};
  cuuint32_t box[2] = {(cuuint32_t)(128 / esz), (cuuint32_t)kTile};
  cuuint32_t es[2] = {1, 1};
  return fn(map, dtype == TQ_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
            const_cast<void*>(x), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool tq::quantize_wide_supported(const tq_plan* plan, const tq_records* out) {
  return plan->d % 256 == 0 && plan->d >= 256 && plan->d <= 1024 && tq::tensor_map_encoder() != nullptr &&
         (plan->m == 0 || (plan->m == plan->d && plan->s_x_bf16 != nullptr)) && out->layout == TQ_LAYOUT_ROWS;
}

tq_status tq::quantize_wide(const tq_plan* plan, const void* x, tq_dtype dtype, int64_t n, int64_t ld_x,
                            const tq_records* out, int64_t row0, cudaStream_t st) {
  const int d = plan->d, m = plan->m, w = plan->w;
  const bool q = m > 0;
  if (n >= (int64_t(1) << 31)) return TQ_ERR_ARG;  // TMA row coordinates are 32-bit
  WideMaps mp;
  // (m = 0: the two S maps go unused)
  if (!map_input(&mp.x, x, dtype, n, d, ld_x) ||
      !tq::map_bf16_tiles(&mp.pi, plan->pi_bf16, 2 * (uint64_t)d, d, d, kCols) ||
      !tq::map_bf16_tiles(&mp.s, q ? plan->s_x_bf16 : plan->pi_bf16, 2 * (uint64_t)(q ? m : d), d, d, kCols) ||
      !tq::map_bf16_tiles(&mp.sr, q ? plan->s_bf16 : plan->pi_bf16, 2 * (uint64_t)(q ? m : d), d, d, kCols))
    return TQ_ERR_CUDA;
  WideArgs a{};
  a.x = x;
  a.n = n;
  a.ld = ld_x;
  a.ntiles = (n + kTile - 1) / kTile;
  a.d = d;
  a.m = m;
  a.centroids = plan->centroids;
  a.bounds = plan->bounds;
  a.idx = out->idx + row0 * (w * d / 32);
  a.sgn = q ? out->sgn + row0 * (m / 32) : nullptr;
  a.norm = out->norm + row0;
  a.rnorm = q ? out->rnorm + row0 : nullptr;
  a.fault = tq::fault_word();
  if (!a.fault) return TQ_ERR_CUDA;
  return dtype == TQ_F32 ? launch_wide_t<float>(w, q, mp, a, st) : launch_wide_t<__nv_bfloat16>(w, q, mp, a, st);
}

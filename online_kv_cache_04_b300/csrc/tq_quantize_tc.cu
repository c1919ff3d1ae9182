// tq_quantize on the 5th-generation tensor cores (tcgen05), for bf16 input
// with d = m = 128: the head-dim-128 KV-cache case.
//
// Per tile of 128 vectors (one CTA per SM, persistent over tiles):
//   TMA        x tile (bf16, 128-byte swizzle) -> shared memory, 2 stages
//   GEMM1      U = x Πᵀ as x·Π_hiᵀ + x·Π_loᵀ (Π split into two bf16 terms;
//              bf16 x is exact): two N = 128 products per K-step into one
//              fp32 accumulator of 128 columns
//   norms      n = ||x|| of the tile's vectors from the staged tile, by one
//              warp of its own (the epilogue warps never read x)
//   epilogue 1 u = U / n, bucketize against
//              the Lloyd-Max bounds (binary search) -> index bit-planes,
//              ρ = u - c[idx], ||ρ||², ρ split into bf16 hi + lo written back
//              to TMEM over the columns of U just read; coordinate pairs in
//              packed fp32x2 arithmetic
//   GEMM2      P = ρ (S Πᵀ)ᵀ as ρ_hi·S_hi + ρ_hi·S_lo + ρ_lo·S_hi, with ρ
//              read from TMEM as the A operand
//   epilogue 2 σ = [P >= 0] packed into words, ||r|| = n ||ρ||, stores
// ("谷歌TurboQuant如何绕过内存墙？" §2 stages 1 and 2; "TurboQuant 与 AI 效率革命"
// §四 three-step pipeline; "TurboQuant压缩效果": codes packed into 32-bit words.)
//
// One launch covers one input or two (tq_quantize_pair: the keys and values
// of the same tokens, each with its own output layout) as one sequence of
// tiles, so the pipeline fills and drains once.  It is a programmatic
// dependent launch: the prologue overlaps the previous kernel, and the input
// loads and record stores wait for it.
//
// TMEM holds four regions of 128 columns.  Tile i keeps U (then ρ) in region
// i mod 4 and writes P into region (i - 1) mod 4, the one that held tile
// i - 1's residual: GEMM1 of tile i waits only for the sign epilogue of tile
// i - 3, so the tensor core has the products of three tiles to choose from
// while the epilogues of the others run (with two slots of U | P, GEMM1 of
// tile i waited for the sign epilogue of tile i - 2).  Two epilogue
// warpgroups take alternate tiles.  Warp roles (640 threads):
// warps 0-7 epilogue of even tiles, 8-15 of odd tiles (warp % 4 = TMEM lane
// quadrant; the two warps of a quadrant split the 128 coordinates of its 32
// vectors and meet through shared memory for ||r||), warp 16 issues GEMM1
// and owns TMEM, warp 17 issues TMA loads, warp 18 issues GEMM2, warp 19
// forms the norms.  A
// tcgen05.mma costs its issuing thread far more cycles than the tensor core
// needs for an N = 128 product, so the two GEMMs have an issuer each.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <algorithm>

#include "tq_internal.h"
#include "tq_sm100.cuh"

namespace {

using namespace tq::sm100;

constexpr int kTile = 128;                       // vectors per tile (MMA M)
constexpr int kBoxBytes = 64 * 128 * 2;          // TMA box: 64 bf16 columns x 128 rows
constexpr int kMatBytes = 2 * kBoxBytes;         // one 128 x 128 bf16 operand
// Π_hi and Π_lo per 64-column box ([box][hi, lo] x 128 rows)
constexpr int kOffPi = 0, kOffSHi = 2 * kMatBytes, kOffSLo = 3 * kMatBytes;
constexpr int kOffX = 4 * kMatBytes;             // two x stages
constexpr int kOffBar = kOffX + 2 * kMatBytes;
constexpr int kOffRsq = kOffBar + 256;           // [slot 2][tile parity 2][128] partial ||ρ||² of the upper half
constexpr int kOffNrm = kOffRsq + 2 * 2 * 128 * 4;  // [tile parity 2][128] ||x|| of the tile's vectors
// [slot 2][tile parity 2][word 8][128]: the upper half's index and sign words of
// a row-layout tile (words 2p, 2p + 1: plane p; 6, 7: signs), which the lower
// half stores together with its own as whole 16-byte pieces of each record
constexpr int kOffXch = kOffNrm + 2 * 128 * 4;
constexpr int kSmemBytes = kOffXch + 2 * 2 * 8 * 128 * 4 + 1024;  // + alignment slack
constexpr int kThreads = 640, kMmaWarp = 16, kTmaWarp = 17, kMma2Warp = 18, kNormWarp = 19;
constexpr uint32_t kTmemCols = 512;              // four regions of 128 columns: U, then ρ K-steps [hi 8 | lo 8]; or P

constexpr unsigned kFaultWait = 1u;              // fault bit: a pipeline wait ran out of its bound

struct Bars {
  uint64_t b_full;
  uint64_t x_full[2], x_empty[2], rho_full[2], p_full[2];
  // indexed by tile mod 4: a barrier completes at most once per four tiles,
  // so no waiter can see it complete twice (the epilogue warpgroups and the
  // issuers run up to three tiles apart)
  uint64_t u_full[4], acc_empty[4];
  uint64_t norm_full[2], norm_empty[2];  // the norms of the tile's vectors are in / have been read
  uint64_t rsq_full[2];   // the upper coordinate half's ||ρ||² partials are in
  uint64_t rsq_empty[2];  // the lower half has read them (the halves run apart otherwise)
  uint32_t tmem_base;
};

static_assert(sizeof(Bars) <= 256, "barriers must fit their shared-memory region");

// One output of a launch: the records of `n` input rows.
struct TcOut {
  uint32_t* idx;           // TQ_LAYOUT_ROWS: row 0 of this call; TQ_LAYOUT_BLOCK32: block of row 0
  uint32_t* sgn;
  float* norm;             // row 0 of this call
  float* rnorm;
  int64_t n;
  int layout;              // tq_layout
};

// A launch quantizes one or two inputs of 128-row tiles: tiles [0, ntiles0) are
// input 0's, the rest input 1's (the keys and values of the same tokens, say),
// so that one persistent grid fills and drains its pipeline once for both.
struct TcArgs {
  TcOut out0, out1;
  int64_t ntiles0, ntiles;
  const float* centroids;  // device [2^w]
  const float* bounds;     // device [2^w - 1]
  unsigned* fault;
};

__device__ unsigned g_fault_word;

// 32 x 32 bit transpose across a warp into the block layout's bit order.  On
// entry lane r holds row r (bit c = element (r, c)).  The butterfly runs with
// every lane index rotated left by one bit (lane L plays position
// t/2 + 16·(t%2) of row t = L), so on exit lane L holds column
// L/2 + 16·(L%2) with row t at bit t/2 + 16·(t%2): the block layout's word,
// with no separate bit permutation.
__device__ __forceinline__ uint32_t warp_transpose32_block(uint32_t x, int lane) {
  const uint32_t masks[5] = {0x0000FFFFu, 0x00FF00FFu, 0x0F0F0F0Fu, 0x33333333u, 0x55555555u};
#pragma unroll
  for (int k = 0; k < 5; ++k) {
    const int sh = 16 >> k;                             // bit distance within the word
    const int ls = ((sh << 1) & 31) | (sh >> 4);        // lane distance: sh rotated left by one
    const uint32_t m = masks[k];
    const uint32_t y = __shfl_xor_sync(0xffffffffu, x, ls);
    x = (lane & ls) ? ((x & ~m) | ((y >> sh) & m)) : ((x & m) | ((y & m) << sh));
  }
  return x;
}

// Even bits to the low half-word, odd bits to the high half (bit t -> t/2 + 16(t%2)).
__device__ __forceinline__ uint32_t unshuffle32(uint32_t x) {
  uint32_t t;
  t = (x ^ (x >> 1)) & 0x22222222u; x = x ^ t ^ (t << 1);
  t = (x ^ (x >> 2)) & 0x0C0C0C0Cu; x = x ^ t ^ (t << 2);
  t = (x ^ (x >> 4)) & 0x00F000F0u; x = x ^ t ^ (t << 4);
  t = (x ^ (x >> 8)) & 0x0000FF00u; x = x ^ t ^ (t << 8);
  return x;
}

// TQ_LAYOUT_BLOCK32 store of one warp's 32 rows (one block): `words[c]` is
// this lane's row word for coordinates 32c..32c+31 (counted from `blk`);
// `valid` has bit L set for valid row L.  Lane L writes the block word of
// coordinate 32c + L/2 + 16·(L%2) (the warp's 32 stores still cover 128
// contiguous bytes), merging with the stored bits of rows that this call does
// not write.
template <int NW>
__device__ __forceinline__ void store_block32(uint32_t* blk, const uint32_t (&words)[NW], uint32_t valid, int lane) {
  const uint32_t vm = unshuffle32(valid);
  const int colw = (lane >> 1) | ((lane & 1) << 4);
#pragma unroll
  for (int c = 0; c < NW; ++c) {
    const uint32_t col = warp_transpose32_block(words[c], lane);
    uint32_t* dst = blk + 32 * c + colw;
    if (vm == 0xFFFFFFFFu) *dst = col;
    else if (vm != 0u) *dst = (*dst & ~vm) | (col & vm);
  }
}

// Q: the QJL stage is on (m = 128); without it (m = 0, stage 1 alone) there is
// no GEMM2, no residual in TMEM and no sign epilogue: the TMEM slot is free once
// epilogue 1 has read U.
template <int W, bool Q>
__global__ void __launch_bounds__(kThreads, 1)
    quantize_tc_kernel(const __grid_constant__ CUtensorMap tm_x0, const __grid_constant__ CUtensorMap tm_x1,
                       const __grid_constant__ CUtensorMap tm_pi,
                       const __grid_constant__ CUtensorMap tm_s, const TcArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t base = smem_u32(smem);
  Bars* bars = reinterpret_cast<Bars*>(smem + kOffBar);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t ntiles = a.ntiles;

  // the next launch in the stream may be scheduled now (it waits for this grid
  // before it reads anything this grid writes)
  asm volatile("griddepcontrol.launch_dependents;");
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bars->b_full), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&bars->x_full[s]), 1);
      mbar_init(smem_u32(&bars->x_empty[s]), 2);  // GEMM1 done, norms read
      mbar_init(smem_u32(&bars->norm_full[s]), 1);
      mbar_init(smem_u32(&bars->norm_empty[s]), 8);
      mbar_init(smem_u32(&bars->rho_full[s]), 8);
      mbar_init(smem_u32(&bars->p_full[s]), 1);
      mbar_init(smem_u32(&bars->rsq_full[s]), 4);
      mbar_init(smem_u32(&bars->rsq_empty[s]), 4);
    }
    for (int i = 0; i < 4; ++i) {
      mbar_init(smem_u32(&bars->u_full[i]), 1);
      mbar_init(smem_u32(&bars->acc_empty[i]), 8);
    }
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(&bars->tmem_base), kTmemCols);
    tmem_relinquish();
  }
  if (warp == kTmaWarp && lane == 0) {
    tma_prefetch_desc(&tm_x0);
    if (a.ntiles > a.ntiles0) tma_prefetch_desc(&tm_x1);
    tma_prefetch_desc(&tm_pi);
    tma_prefetch_desc(&tm_s);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp == kTmaWarp) {
    if (lane == 0) {
      const uint32_t bfull = smem_u32(&bars->b_full);
      mbar_arrive_expect_tx(bfull, 4 * kMatBytes);
      for (int mat = 0; mat < 2; ++mat)
        for (int h = 0; h < 2; ++h) {
          tma_load_2d(base + kOffPi + (2 * h + mat) * kBoxBytes, &tm_pi, h * 64, mat * 128, bfull);
          tma_load_2d(base + kOffSHi + mat * kMatBytes + h * kBoxBytes, &tm_s, h * 64, mat * 128, bfull);
        }
      // the inputs may come from the previous launch in the stream: read them
      // only once it has completed (the plan tables above are not written by it)
      asm volatile("griddepcontrol.wait;" ::: "memory");
      int it = 0, last_k[2] = {-1, -1};
      for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++it) {
        const int s = it & 1, k = it >> 1;
        if (!mbar_wait(smem_u32(&bars->x_empty[s]), (k & 1) ^ 1, a.fault, kFaultWait)) break;
        const uint32_t xf = smem_u32(&bars->x_full[s]);
        mbar_arrive_expect_tx(xf, kMatBytes);
        const uint32_t dst = base + kOffX + s * kMatBytes;
        const bool second = tile >= a.ntiles0;
        const CUtensorMap* tm = second ? &tm_x1 : &tm_x0;
        const int32_t y = (int32_t)((tile - (second ? a.ntiles0 : 0)) * kTile);
        tma_load_2d(dst, tm, 0, y, xf);
        tma_load_2d(dst + kBoxBytes, tm, 64, y, xf);
        last_k[s] = k;
      }
      // no copy of this CTA may still be in flight when it exits
      mbar_wait(bfull, 0, a.fault, kFaultWait);
      for (int s = 0; s < 2; ++s)
        if (last_k[s] >= 0) mbar_wait(smem_u32(&bars->x_full[s]), last_k[s] & 1, a.fault, kFaultWait);
    }
  } else if (warp == kMmaWarp) {
    // GEMM1 of every tile (U into region it mod 4; it mod 2 without QJL)
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, 128);
      bool ok = mbar_wait(smem_u32(&bars->b_full), 0, a.fault, kFaultWait);
      tc_fence_after();
      const uint64_t pd = desc_sw128(base + kOffPi);
      int it = 0;
      for (int64_t tile = blockIdx.x; ok && tile < ntiles; tile += gridDim.x, ++it) {
        const int s = it & 1, k = it >> 1;
        if (!mbar_wait(smem_u32(&bars->x_full[s]), k & 1, a.fault, kFaultWait)) break;
        // the region this tile's U goes into: with QJL, tile it - 3 held its P
        // there (released by that tile's sign epilogue, after GEMM2 of tiles up
        // to it - 3 completed); without, tile it - 2 held its U in region it mod 2
        // (released once epilogue 1 read it)
        if (Q ? (it >= 3 && !mbar_wait(smem_u32(&bars->acc_empty[(it - 3) & 3]), ((it - 3) >> 2) & 1, a.fault,
                                       kFaultWait))
              : (it >= 2 && !mbar_wait(smem_u32(&bars->acc_empty[(it - 2) & 3]), ((it - 2) >> 2) & 1, a.fault,
                                       kFaultWait)))
          break;
        tc_fence_after();
        const uint32_t acc = tmem + 128 * (Q ? (it & 3) : s);
        const uint64_t xd = desc_sw128(base + kOffX + s * kMatBytes);
        // U = x·Π_hiᵀ + x·Π_loᵀ: both products of a K-step into the same 128 columns
#pragma unroll 1
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t offa = ((kk >> 2) * kBoxBytes + (kk & 3) * 32) >> 4;
          const uint32_t offb = ((kk >> 2) * 2 * kBoxBytes + (kk & 3) * 32) >> 4;
          mma_ss(acc, xd + offa, pd + offb, idesc, kk != 0);
          mma_ss(acc, xd + offa, pd + offb + (kBoxBytes >> 4), idesc, 1u);
        }
        mma_commit(smem_u32(&bars->u_full[it & 3]));
        mma_commit(smem_u32(&bars->x_empty[s]));
      }
    }
  } else if (warp == kMma2Warp) {
    // GEMM2 of every tile j, issued by a thread of its own so that its products
    // queue beside GEMM1's: A = ρ from region j mod 4, P into region (j - 1) mod 4
    if (Q && lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, 128);
      bool ok = mbar_wait(smem_u32(&bars->b_full), 0, a.fault, kFaultWait);
      const uint64_t shd = desc_sw128(base + kOffSHi), sld = desc_sw128(base + kOffSLo);
      int j = 0;
      for (int64_t tile = blockIdx.x; ok && tile < ntiles; tile += gridDim.x, ++j) {
        const int s = j & 1, k = j >> 1;
        if (!mbar_wait(smem_u32(&bars->rho_full[s]), k & 1, a.fault, kFaultWait)) break;
        // region (j - 1) mod 4 held tile j - 1's residual: its GEMM2 must have read it
        if (j >= 1 && !mbar_wait(smem_u32(&bars->p_full[s ^ 1]), ((j - 1) >> 1) & 1, a.fault, kFaultWait)) break;
        tc_fence_after();
        const uint32_t acc = tmem + 128 * ((j + 3) & 3), rreg = tmem + 128 * (j & 3);
        // terms (ρ_hi, S_hi), (ρ_hi, S_lo), (ρ_lo, S_hi); K-step kk: ρ pieces of
        // coordinates 16kk.. sit in [hi 8 | lo 8] at 16kk, and the B start
        // address advances in 16-byte units
#pragma unroll 1
        for (int t = 0; t < 3; ++t) {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t boff = ((kk >> 2) * kBoxBytes + (kk & 3) * 32) >> 4;
            mma_ts(acc, rreg + 16 * kk + (t == 2 ? 8 : 0), (t == 1 ? sld : shd) + boff, idesc, (t | kk) != 0);
          }
        }
        mma_commit(smem_u32(&bars->p_full[s]));
      }
    }
  } else if (warp == kNormWarp) {
    // ||x|| of every vector of the tile from the staged tile (row r, 128-byte
    // swizzle): each 64-coordinate box in two packed pairs of partial sums,
    // lower box + upper box; lane l takes rows l, l + 32, l + 64, l + 96
    int it = 0;
    for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++it) {
      const int s = it & 1, k = it >> 1;
      if (!mbar_wait(smem_u32(&bars->x_full[s]), k & 1, a.fault, kFaultWait)) break;
      // the slot's previous norms (tile it - 2) have been read by its epilogue
      if (!mbar_wait(smem_u32(&bars->norm_empty[s]), (k & 1) ^ 1, a.fault, kFaultWait)) break;
      float* nrm = reinterpret_cast<float*>(smem + kOffNrm) + s * 128;
#pragma unroll 1
      for (int i = 0; i < 4; ++i) {
        const int r = lane + 32 * i;
        float part0 = 0.f, part1 = 0.f;
#pragma unroll 1
        for (int hb = 0; hb < 2; ++hb) {
          uint64_t ssa = 0ull, ssb = 0ull;
          const uint8_t* row = smem + kOffX + s * kMatBytes + hb * kBoxBytes + (r >> 3) * 1024 + (r & 7) * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint4 v = *reinterpret_cast<const uint4*>(row + ((c ^ (r & 7)) << 4));
            const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const uint64_t x2 = f2_pack(__uint_as_float(wv[e] << 16), __uint_as_float(wv[e] & 0xFFFF0000u));
              if (e & 1) ssb = f2_fma(x2, x2, ssb);
              else ssa = f2_fma(x2, x2, ssa);
            }
          }
          const float2 pa = f2_unpack(ssa), pb = f2_unpack(ssb);
          const float ps = (pa.x + pa.y) + (pb.x + pb.y);
          if (hb == 0) part0 = ps;
          else part1 = ps;
        }
        nrm[r] = sqrtf(part0 + part1);
      }
      // the next TMA write into this stage (async proxy) follows these generic reads
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_u32(&bars->x_empty[s]));
        mbar_arrive(smem_u32(&bars->norm_full[s]));
      }
    }
  } else {
    // the previous launch in the stream may still read the records written here
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // epilogue: warpgroup g = warp / 4 handles tiles it ≡ g (mod 2); thread = one vector (TMEM lane)
    float cent[8], bnd[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      cent[k] = k < (1 << W) ? __ldg(a.centroids + k) : 0.f;
      bnd[k] = k < (1 << W) - 1 ? __ldg(a.bounds + k) : 0.f;
    }
    // Warps 0-7 take the even tiles (TMEM slot 0), 8-15 the odd ones (slot 1).
    // Warp % 4 is the TMEM lane quadrant (32 vectors); the two warps of a
    // quadrant split the coordinates: half h takes 64h .. 64h + 63.
    const int g = warp >> 3, h = (warp >> 2) & 1, q = warp & 3, r = q * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    const int s = g;
    float* rsq_s = reinterpret_cast<float*>(smem + kOffRsq) + (s * 2) * 128;
    int it = g;
    for (int64_t tile = blockIdx.x + (int64_t)g * gridDim.x; tile < ntiles; tile += 2 * (int64_t)gridDim.x, it += 2) {
      const int ph = (it >> 1) & 1;
      // n = ||x|| from the norm warp
      if (!mbar_wait(smem_u32(&bars->norm_full[s]), ph, a.fault, kFaultWait)) break;
      const float n = reinterpret_cast<const float*>(smem + kOffNrm)[s * 128 + r];
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bars->norm_empty[s]));
      // U (then ρ) in region it mod 4 (it mod 2 without QJL), P in region (it - 1) mod 4
      const uint32_t uacc = tmem + lane_base + 128 * (Q ? (it & 3) : s);
      const uint32_t pacc = tmem + lane_base + 128 * ((it + 3) & 3);
      if (!mbar_wait(smem_u32(&bars->u_full[it & 3]), (it >> 2) & 1, a.fault, kFaultWait)) break;
      tc_fence_after();
      const float inv = n > 0.f ? 1.0f / n : 0.f, nlive = n > 0.f ? -1.f : 0.f;
      const uint64_t inv2 = f2_pack(inv, inv), nlive2 = f2_pack(nlive, nlive);
      uint32_t planes[W][2];
      uint64_t rsq2 = 0ull;
      // 16 coordinates per TMEM load: chunks 4h .. 4h + 3 (two per plane word)
#pragma unroll
      for (int p = 0; p < W; ++p) planes[p][0] = planes[p][1] = 0u;
#pragma unroll 1
      for (int cc = 0; cc < 4; ++cc) {
        const int c = 4 * h + cc;
        uint32_t v[16];
        tmem_ld16(uacc + 16 * c, v);
        tmem_ld_wait();
        uint32_t pw[W], hi[8], lo[8];
#pragma unroll
        for (int p = 0; p < W; ++p) pw[p] = 0u;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          // u = U / n for coordinates 2j, 2j + 1 of the chunk
          const uint64_t u2 = f2_mul(f2_pack(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1])), inv2);
          const float2 uu = f2_unpack(u2);
          float cv[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const float u = e ? uu.y : uu.x;
            // idx = #{k : bound_k < u} by binary search over the sorted bounds;
            // the branch taken at level l is bit W-1-l of idx (plane W-1-l)
            const uint32_t bit = 1u << (2 * j + e);
            if constexpr (W == 1) {
              const bool p0 = u > bnd[0];
              cv[e] = p0 ? cent[1] : cent[0];
              if (p0) pw[0] |= bit;
            } else if constexpr (W == 2) {
              const bool p1 = u > bnd[1];
              const bool p0 = u > (p1 ? bnd[2] : bnd[0]);
              const float chi = p1 ? cent[3] : cent[1], clo = p1 ? cent[2] : cent[0];
              cv[e] = p0 ? chi : clo;
              if (p1) pw[1] |= bit;
              if (p0) pw[0] |= bit;
            } else {
              const bool p2 = u > bnd[3];
              const bool p1 = u > (p2 ? bnd[5] : bnd[1]);
              const bool p0 = u > (p2 ? (p1 ? bnd[6] : bnd[4]) : (p1 ? bnd[2] : bnd[0]));
              const float codd = p2 ? (p1 ? cent[7] : cent[5]) : (p1 ? cent[3] : cent[1]);
              const float cevn = p2 ? (p1 ? cent[6] : cent[4]) : (p1 ? cent[2] : cent[0]);
              cv[e] = p0 ? codd : cevn;
              if (p2) pw[2] |= bit;
              if (p1) pw[1] |= bit;
              if (p0) pw[0] |= bit;
            }
          }
          const uint64_t rho2 = f2_fma(f2_pack(cv[0], cv[1]), nlive2, u2);  // u - c[idx], 0 for a zero vector
          rsq2 = f2_fma(rho2, rho2, rsq2);
          if (Q) {
            const float2 rr = f2_unpack(rho2);
            const __nv_bfloat162 hv = __floats2bfloat162_rn(rr.x, rr.y);
            const float2 hf = __bfloat1622float2(hv);
            const float2 lf = f2_unpack(f2_add(rho2, f2_pack(-hf.x, -hf.y)));
            const __nv_bfloat162 l = __floats2bfloat162_rn(lf.x, lf.y);
            hi[j] = *reinterpret_cast<const uint32_t*>(&hv);
            lo[j] = *reinterpret_cast<const uint32_t*>(&l);
          }
        }
        if (Q) {  // over the columns of U just read: K-step c = [hi 8 | lo 8]
          tmem_st8(uacc + 16 * c, hi);
          tmem_st8(uacc + 16 * c + 8, lo);
        }
        // chunk c holds bits 16·(c & 1).. of plane word c / 2 (word (c >> 1) - 2h here)
#pragma unroll
        for (int p = 0; p < W; ++p) {
          const uint32_t x = (cc & 1) ? pw[p] << 16 : pw[p];
          if (cc >> 1) planes[p][1] |= x;
          else planes[p][0] |= x;
        }
      }
      const float2 rs = f2_unpack(rsq2);
      const float rsq = rs.x + rs.y;
      if (Q) tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      // with QJL, GEMM2 reads the residual next; without, the slot is free
      if (lane == 0) mbar_arrive(smem_u32(Q ? &bars->rho_full[s] : &bars->acc_empty[it & 3]));
      // this tile's output (fields picked one by one: no dynamic index into the parameters)
      const bool second = tile >= a.ntiles0;
      const int64_t lt = tile - (second ? a.ntiles0 : 0), on = second ? a.out1.n : a.out0.n;
      const bool rows_layout = (second ? a.out1.layout : a.out0.layout) == TQ_LAYOUT_ROWS;
      uint32_t* const oidx = second ? a.out1.idx : a.out0.idx;
      const int64_t row = lt * kTile + r;
      const int64_t blk_row = lt * kTile + q * 32;  // this warp's block (block layout)
      const uint32_t valid = __ballot_sync(0xffffffffu, row < on);
      // At w = 3 with QJL the lower half stores whole rows of a row-layout tile
      // after the sign epilogue (the upper half's words through shared memory):
      // the index planes then need no registers across the sign epilogue, which
      // is what the w = 3 epilogue was short of.  At w <= 2 each half stores its
      // own words as soon as they are known.
      constexpr bool kStageRows = Q && W == 3;
      if (rows_layout) {
        if (!kStageRows && row < on) {
#pragma unroll
          for (int p = 0; p < W; ++p)
            *reinterpret_cast<uint2*>(oidx + row * (4 * W) + p * 4 + 2 * h) = make_uint2(planes[p][0], planes[p][1]);
        }
      } else {
        if (valid != 0u) {
#pragma unroll
          for (int p = 0; p < W; ++p)
            store_block32<2>(oidx + (blk_row >> 5) * (W * 128) + p * 128 + 64 * h, planes[p], valid, lane);
        }
      }
      if (!Q) {  // stage 1 alone: the norm is the record's last field
        if (h == 0 && row < on) (second ? a.out1.norm : a.out0.norm)[row] = n;
        continue;
      }
      if (!mbar_wait(smem_u32(&bars->p_full[s]), ph, a.fault, kFaultWait)) break;
      tc_fence_after();
      uint32_t sg[2];
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        // bit j = [P_j >= 0]: the sign bits shifted in from the top coordinate
        // down (upper 16 columns first), then inverted; a zero vector (P = 0 of
        // either sign) takes all ones
        uint32_t neg = 0u;
#pragma unroll
        for (int hc = 1; hc >= 0; --hc) {
          uint32_t v[16];
          tmem_ld16(pacc + 32 * (2 * h + cc) + 16 * hc, v);
          tmem_ld_wait();
#pragma unroll
          for (int j = 15; j >= 0; --j) neg = __funnelshift_l(v[j], neg, 1);
        }
        sg[cc] = n > 0.f ? ~neg : 0xFFFFFFFFu;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bars->acc_empty[it & 3]));
      uint32_t* const osgn = second ? a.out1.sgn : a.out0.sgn;
      if (rows_layout) {
        if (!kStageRows && row < on) *reinterpret_cast<uint2*>(osgn + row * 4 + 2 * h) = make_uint2(sg[0], sg[1]);
      } else {
        if (valid != 0u) store_block32<2>(osgn + (blk_row >> 5) * 128 + 64 * h, sg, valid, lane);
      }
      // The halves meet once per tile: the upper half hands its ||ρ||² partial
      // (and, when staged, its index and sign words) to the lower half, which
      // writes ||x||, ||r|| (and the whole records).
      float* const rs_slot = rsq_s + (it >> 1 & 1) * 128;
      uint32_t* const xw = reinterpret_cast<uint32_t*>(smem + kOffXch) + (s * 2 + (it >> 1 & 1)) * 8 * 128 + r;
      if (h == 1) {
        // once the lower half has read this slot's words of the group's previous tile
        if (!mbar_wait(smem_u32(&bars->rsq_empty[s]), ph ^ 1, a.fault, kFaultWait)) break;
        rs_slot[r] = rsq;
        if (kStageRows && rows_layout) {
#pragma unroll
          for (int p = 0; p < W; ++p) xw[(2 * p) * 128] = planes[p][0], xw[(2 * p + 1) * 128] = planes[p][1];
          xw[6 * 128] = sg[0];
          xw[7 * 128] = sg[1];
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bars->rsq_full[s]));
      } else {
        if (!mbar_wait(smem_u32(&bars->rsq_full[s]), ph, a.fault, kFaultWait)) break;
        if (row < on) {
          (second ? a.out1.norm : a.out0.norm)[row] = n;
          (second ? a.out1.rnorm : a.out0.rnorm)[row] = n * sqrtf(rsq + rs_slot[r]);
          if (kStageRows && rows_layout) {
#pragma unroll
            for (int p = 0; p < W; ++p)
              *reinterpret_cast<uint4*>(oidx + row * (4 * W) + p * 4) =
                  make_uint4(planes[p][0], planes[p][1], xw[(2 * p) * 128], xw[(2 * p + 1) * 128]);
            *reinterpret_cast<uint4*>(osgn + row * 4) = make_uint4(sg[0], sg[1], xw[6 * 128], xw[7 * 128]);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bars->rsq_empty[s]));
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

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// rows x cols bf16 matrix with row stride ld elements; 64 x 128 boxes, 128-byte swizzle
bool map_bf16(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols, uint64_t ld) {
  return tq::map_bf16_tiles(m, ptr, rows, cols, ld, 128);
}

template <int W, bool Q>
tq_status launch_w(const CUtensorMap& mx0, const CUtensorMap& mx1, const CUtensorMap& mp, const CUtensorMap& ms,
                   const TcArgs& a, cudaStream_t st) {
  auto kern = quantize_tc_kernel<W, Q>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) != cudaSuccess)
    return TQ_ERR_CUDA;
  cudaFuncAttributes fa;
  if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess || fa.maxThreadsPerBlock < kThreads) return TQ_ERR_CUDA;
  const int grid = (int)std::min<int64_t>(a.ntiles, tq::sm_count());
  // programmatic dependent launch: the prologue (barriers, TMEM, the plan
  // operands) overlaps the previous kernel; inputs and outputs wait for it
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, mx0, mx1, mp, ms, a) != cudaSuccess) return TQ_ERR_CUDA;
  return tq::launch_status();
}

}  // namespace

bool tq::map_bf16_tiles(CUtensorMap* map, const void* ptr, uint64_t rows, uint64_t cols, uint64_t ld,
                        uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {ld * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

tq::TensorMapEncoder tq::tensor_map_encoder() { return encode_fn(); }

unsigned* tq::fault_word() {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_fault_word) != cudaSuccess) return nullptr;
  return static_cast<unsigned*>(p);
}

bool tq::quantize_tc_supported(const tq_plan* plan, tq_dtype dtype, int64_t n) {
  return plan->d == 128 && (plan->m == 128 || plan->m == 0) && dtype == TQ_BF16 && n < (int64_t(1) << 31) &&
         encode_fn() != nullptr;
}

// Output fields of rows [row0, row0 + n) of `out`.
static TcOut tc_out(const tq_records* out, int64_t n, int64_t row0, int w) {
  const bool rows = out->layout == TQ_LAYOUT_ROWS;
  TcOut o;
  o.idx = rows ? out->idx + row0 * (w * 4) : out->idx + (row0 / 32) * (w * 128);
  o.sgn = out->sgn == nullptr ? nullptr : rows ? out->sgn + row0 * 4 : out->sgn + (row0 / 32) * 128;
  o.norm = out->norm + row0;
  o.rnorm = out->rnorm == nullptr ? nullptr : out->rnorm + row0;
  o.n = n;
  o.layout = out->layout;
  return o;
}

tq_status tq::quantize_tc(const tq_plan* plan, const void* x0, const void* x1, int64_t n, int64_t ld_x,
                          const tq_records* out0, const tq_records* out1, int64_t row0, cudaStream_t st) {
  for (const tq_records* o : {out0, out1})
    if (o != nullptr && o->layout != TQ_LAYOUT_ROWS && row0 % 32 != 0) return TQ_ERR_ARG;
  const bool pair = x1 != nullptr && out1 != nullptr;
  CUtensorMap mx0, mx1, mp, ms;
  if (!map_bf16(&mx0, x0, (uint64_t)n, 128, (uint64_t)ld_x) ||
      !map_bf16(&mx1, pair ? x1 : x0, (uint64_t)n, 128, (uint64_t)ld_x) ||
      !map_bf16(&mp, plan->pi_bf16, 256, 128, 128) ||
      !map_bf16(&ms, plan->m > 0 ? plan->s_bf16 : plan->pi_bf16, 256, 128, 128))  // (m = 0: the S map goes unused)
    return TQ_ERR_CUDA;
  const int w = plan->w;
  TcArgs a{};
  a.out0 = tc_out(out0, n, row0, w);
  a.out1 = pair ? tc_out(out1, n, row0, w) : a.out0;
  a.ntiles0 = (n + kTile - 1) / kTile;
  a.ntiles = pair ? 2 * a.ntiles0 : a.ntiles0;
  a.centroids = plan->centroids;
  a.bounds = plan->bounds;
  a.fault = tq::fault_word();
  if (!a.fault) return TQ_ERR_CUDA;
  const bool q = plan->m > 0;
  switch (w) {
    case 1: return q ? launch_w<1, true>(mx0, mx1, mp, ms, a, st) : launch_w<1, false>(mx0, mx1, mp, ms, a, st);
    case 2: return q ? launch_w<2, true>(mx0, mx1, mp, ms, a, st) : launch_w<2, false>(mx0, mx1, mp, ms, a, st);
    default: return q ? launch_w<3, true>(mx0, mx1, mp, ms, a, st) : launch_w<3, false>(mx0, mx1, mp, ms, a, st);
  }
}

extern "C" tq_status tq_fault_flags(uint32_t* flags, int reset) {
  if (flags == nullptr) return TQ_ERR_ARG;
  unsigned v = 0;
  if (cudaMemcpyFromSymbol(&v, g_fault_word, sizeof(v)) != cudaSuccess) return TQ_ERR_CUDA;
  *flags = v;
  if (reset) {
    const unsigned z = 0;
    if (cudaMemcpyToSymbol(g_fault_word, &z, sizeof(z)) != cudaSuccess) return TQ_ERR_CUDA;
  }
  return TQ_OK;
}

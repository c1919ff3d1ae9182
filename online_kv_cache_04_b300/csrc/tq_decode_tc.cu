// Decode attention over the compressed cache on the tensor cores, for
// d = m = 128 and up to 8 query heads per kv head.
//
// What is computed is the same as the general kernel in tq_decode.cu
// ("TurboQuant 与 AI 效率革命" §三, the asymmetric estimator applied to the
// residual as in "谷歌TurboQuant如何绕过内存墙？" §2 stage 2):
//   s_t = scale·(‖k_t‖⟨Πq, c[idx_t]⟩ + √(π/2)/m·‖r_t‖⟨Sq, σ_t⟩),
//   o   = Πᵀ Σ_t p_t (‖v_t‖ c[idx_t] + √(π/2)/m·‖r_v,t‖ S̃ᵀσ_t) / Σ_t p_t.
// Packed words are read once and turned into tensor-core operands in
// registers; no dequantized key or value is ever written to memory
// ("TurboQuant压缩效果": decode in registers while reading).
//
// Bits as exact operands.  A symmetric Lloyd-Max codebook is a sum of ±1
// bit-planes, c[idx] = Σ_P coef_P·s_P with s = 2·bit − 1 (Walsh expansion;
// w = 1: one plane, w = 2: two, w = 3: three plus their product).  The QJL
// signs are one more ±1 plane.  An f16 operand register holds bits L and
// 16 + L of a plane word (one per half): a multiply by a power of two moves
// them, and one and-or with a constant places each either in the sign of
// 1.0 (operand ±1, exactly −s) or in exponent bit 1 of 0.125 (operand 0.125
// or 0.5, an affine image of s whose offset is folded into a per-(batch,
// kv head) constant).  Keys use both kinds, values only the sign kind, so
// the long sums over the context carry no offset to cancel.
//
//   scores: mma.sync m16n8k16 f16, rows = 16 tokens, K = 16 coordinates of
//           one plane, B = the query weights (registers, per unit).
//   values: the same instruction with rows = 16 coordinates and K = 16
//           tokens of one 32-row block word (TQ_LAYOUT_BLOCK32), B = the
//           attention weights p·‖v‖ and p·‖r_v‖; fp32 accumulators stay in
//           registers over the whole context.
// Each weight enters as two f16 columns, hi = f16(x) and lo = f16(x − hi)
// (22 significant bits): an 8-column operand tile holds 4 heads x (hi, lo),
// and 5 to 8 heads take a second tile over the same expanded bits.
// Why f16 warp MMAs: decode has one query per head, so every product here
// is at most 8 columns wide.  A tcgen05.mma costs its issuing thread over a
// hundred cycles whatever its width, and an e4m3 or int8 mma.sync runs far
// below the f16 one.
//
// Work split.  A persistent grid of one CTA per SM takes contiguous ranges of
// 256-token tiles over all (batch, kv head) units (the last tile of a unit
// may hold 128); the partials of a unit (two per CTA that touches it) are
// merged by the combine kernel of tq_decode.cu.  Sixteen warps do the same
// work: warp w scores 16 tokens of each tile (half w & 1 of block w / 2) and
// accumulates values for 16 coordinates (rows w % 8) over half of the blocks
// (w / 8).  Warps 0-7 thus only touch tokens 0-127 of a tile and warps 8-15
// tokens 128-255, and the two halves run as independent pipelines: each has
// its own softmax reference, running sum, named barriers and partial.  The
// weights of a tile go through shared memory, already laid out as the value
// operand.  Per tile and half there are two named barriers: the first
// publishes the weights of tile i − 1; between the two, the value products of
// tile i − 1, the score products of tile i and its softmax run as one block
// the compiler can interleave; the second carries the vote of the lazy
// softmax.  One thread starts the bulk copies of later tiles into a ring
// stage once both halves have handed it back (a two-arrival mbarrier).
//
// Softmax is online with a lazy reference: the running reference M (of
// log2(p·max(‖v‖, ‖r_v‖)), clamped at 2^-32) moves only when a tile exceeds
// it by more than 2^6; the accumulators are then rescaled.  Every mbarrier
// wait is bounded; on timeout the kernel sets a fault bit (tq_fault_flags),
// skips the remaining waits and runs to its end.
#include <cuda_fp16.h>

#include <algorithm>

#include "tq_internal.h"
#include "tq_sm100.cuh"

namespace {

using namespace tq::sm100;

constexpr int kNW = 16;                                // warps
constexpr int kBlocks = 8;                             // 32-row blocks per tile
constexpr int kTile = 32 * kBlocks;                    // tokens per tile
constexpr int kHalfTile = 128;                         // the last tile of a unit may hold this many
constexpr int kD = 128;
constexpr int kStages = 4;                             // power of two
constexpr int kThreads = 32 * kNW;
constexpr float kTau = 6.0f;                           // lazy-rescale threshold (log2 units)
constexpr float kLog2e = 1.4426950408889634f;
constexpr unsigned kFaultDecode = 2u;

// f16 operand kinds: sign of 1.0 (bit set -> -1) and exponent bit 1 of 0.125
// (bit clear -> 0.125, set -> 0.5).
constexpr uint32_t kSignMask = 0x80008000u, kSignBase = 0x3C003C00u;
constexpr uint32_t kExpMask = 0x08000800u, kExpBase = 0x30003000u;
constexpr float kExpDelta = 0.375f, kExpMean = 0.3125f;  // C' - C, (C + C')/2

// Per quad index q: 2^(3-q) times 1, 2^4, 2^8, 2^12.  Read from constant
// memory so that the moves stay integer multiplies (FMA pipe) instead of
// shifts on the busier integer pipe.
__constant__ uint32_t c_mul[4][4] = {{8u, 128u, 2048u, 32768u},
                                     {4u, 64u, 1024u, 16384u},
                                     {2u, 32u, 512u, 8192u},
                                     {1u, 16u, 256u, 4096u}};

// The masks and bases live in registers loaded from constant memory: with
// both in registers each operand is a single three-input logic op.
__constant__ uint32_t c_ops[4] = {kSignMask, kSignBase, kExpMask, kExpBase};
struct OperandKinds {
  uint32_t sm, sb, em, eb;
  __device__ __forceinline__ OperandKinds() : sm(c_ops[0]), sb(c_ops[1]), em(c_ops[2]), eb(c_ops[3]) {}
  __device__ __forceinline__ static uint32_t andor(uint32_t t, uint32_t m, uint32_t b) {
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(t), "r"(m), "r"(b));  // (t & m) | b
    return r;
  }
  __device__ __forceinline__ uint32_t sign(uint32_t t) const { return andor(t, sm, sb); }
  __device__ __forceinline__ uint32_t expo(uint32_t t) const { return andor(t, em, eb); }
};

__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t f16x2_of(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint32_t word_of(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// Named barriers: all warps (id 3), and the warps of one half h (id 1 + h),
// plain or with an OR vote.
__device__ __forceinline__ void cta_sync() { asm volatile("bar.sync 3, %0;" ::"n"(kThreads) : "memory"); }
__device__ __forceinline__ void half_sync(int h) {
  asm volatile("bar.sync %0, %1;" ::"r"(1 + h), "n"(kThreads / 2) : "memory");
}
__device__ __forceinline__ bool half_any(int h, bool p) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred q, o;\n setp.ne.u32 q, %1, 0;\n bar.red.or.pred o, %2, %3, q;\n selp.u32 %0, 1, 0, o;\n}"
      : "=r"(r)
      : "r"((uint32_t)p), "r"(1 + h), "n"(kThreads / 2)
      : "memory");
  return r != 0;
}

struct TcArgs {
  const uint32_t *kidx, *ksgn, *vidx, *vsgn;
  const float *knorm, *krnorm, *vnorm, *vrnorm;
  const int32_t* ctx_len;
  int64_t ctx_stride;
  int B, Hq, Hkv, G;
  const float* qt;   // [B*Hq][128]  Π q
  const float* st;   // [B*Hq][128]  S q
  const float* walsh;
  float scale, alpha;
  float* part;       // [B*Hq][smax][2 + 2*128]
  int smax;
  int64_t tpu;       // tiles per unit = ceil(ctx_stride / 256)
  int64_t total;     // units * tpu
  unsigned* fault;
};

// CTA that owns flat tile f when `total` tiles are cut into `ctas` even ranges.
__host__ __device__ inline int64_t owner(int64_t f, int64_t total, int64_t ctas) {
  return ((f + 1) * ctas - 1) / total;
}

// Operand columns: head g sits in head tile g / 4, columns 2·(g % 4) (hi)
// and 2·(g % 4) + 1 (lo), so the thread with quad index q ends with both
// pieces of heads q and 4 + q.

template <int W, int GP>
struct Shape {
  static constexpr int NPM = W == 3 ? 4 : W;   // ±1 planes of the codebook
  static constexpr int NP = NPM + 1;           // plus the QJL sign plane
  static constexpr int NKS = 8 * NP;           // score K-steps of 16 coordinates
  static constexpr int GH = GP / 4;            // head tiles = heads per thread
  // ring stage of one full tile; a short tile fills the first half of each region
  static constexpr int kIdxBytes = kTile * 4 * W * 4;
  static constexpr int kSgnBytes = kTile * 16, kNormBytes = kTile * 4;
  static constexpr int kStage = 2 * kIdxBytes + 2 * kSgnBytes + 4 * kNormBytes;
  static constexpr int kOffKIdx = 0, kOffKSgn = kIdxBytes, kOffKNorm = kOffKSgn + kSgnBytes,
                       kOffKRn = kOffKNorm + kNormBytes;
  static constexpr int kOffVIdx = kOffKRn + kNormBytes, kOffVSgn = kOffVIdx + kIdxBytes,
                       kOffVNorm = kOffVSgn + kSgnBytes, kOffVRn = kOffVNorm + kNormBytes;
  // shared memory plan
  // [ks][head tile][n 8][quad 4][b0, b1][half] f16 query weights, one 64-bit fragment per lane
  static constexpr int kBKBytes = NKS * GH * 8 * 16 * 2;
  // [part][head tile][block 8][K half 2][n 8][quad 4][b0, b1] f16x2 attention weights
  static constexpr int kBVBuf = 2 * GH * kBlocks * 2 * 8 * 4 * 8;
  static constexpr int kOffRing = 0;
  static constexpr int kOffBK = kOffRing + kStages * kStage;
  static constexpr int kOffBV = kOffBK + kBKBytes;
  static constexpr int kOffMisc = kOffBV + 2 * kBVBuf;
};

struct Misc {
  uint64_t ld_full[kStages], ld_empty[kStages];  // empty: one arrival per half
  int abort;
  float red[kNW][8];          // per-warp tile maxima (reference moves only)
  float amax[2][8];           // per-unit query weight maxima (as non-negative float bits)
  float O[2][8];              // per-unit score offsets per (part, head)
  float lred[2][kNW][8];      // per segment parity, per warp: Σ p per head
};
constexpr int kMiscBytes = 2048;
static_assert(sizeof(Misc) <= kMiscBytes, "barriers and per-head state must fit their region");

template <int W>
constexpr int smem_bytes() {
  return 1024 + Shape<W, 8>::kOffMisc + kMiscBytes;
}
static_assert(smem_bytes<3>() <= 227 * 1024, "shared memory plan exceeds a CTA's limit");

// Segment of this CTA's tile range that falls in one unit.
struct Seg {
  int64_t u;          // unit = b*Hkv + h
  int64_t t0;         // first tile (in the unit)
  int n;              // tiles with tokens below ctx_len
  int slot;           // partial slot of this CTA for the unit
  int L;              // context length of the unit's batch row
};

__device__ __forceinline__ Seg segment_at(const TcArgs& a, int64_t f, int64_t f1, int64_t* next) {
  Seg s;
  s.u = f / a.tpu;
  s.t0 = f - s.u * a.tpu;
  const int64_t fe = min(f1, (s.u + 1) * a.tpu);
  *next = fe;
  const int b = (int)(s.u / a.Hkv);
  s.L = (int)min((int64_t)max(__ldg(a.ctx_len + b), 0), a.ctx_stride);
  const int64_t nvalid = (s.L + kTile - 1) / kTile;
  const int64_t tend = s.t0 + (fe - f);
  s.n = (int)max((int64_t)0, min(tend, nvalid) - s.t0);
  s.slot = (int)(blockIdx.x - owner(s.u * a.tpu, a.total, gridDim.x));
  return s;
}

template <int W, int GP>
__global__ void __launch_bounds__(kThreads, 1) decode_tc_kernel(const TcArgs a) {
  using Sh = Shape<W, GP>;
  constexpr int NPM = Sh::NPM, NP = Sh::NP, GH = Sh::GH;
  constexpr float kWS = 256.f;  // attention weights carry 2^8: up to 2^14 in f16
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Misc* ms = reinterpret_cast<Misc*>(smem + Sh::kOffMisc);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gq = lane >> 2, tig = lane & 3;  // mma fragment coordinates
  const int64_t C = gridDim.x;
  const int64_t f0 = (int64_t)blockIdx.x * a.total / C, f1 = ((int64_t)blockIdx.x + 1) * a.total / C;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&ms->ld_full[s]), 1);
      mbar_init(smem_u32(&ms->ld_empty[s]), 2);
    }
    ms->abort = 0;
    fence_mbar_init();
  }
  // weight operands start at zero (columns of absent heads are never written)
  for (int e = threadIdx.x; e < 2 * Sh::kBVBuf / 16; e += kThreads)
    reinterpret_cast<uint4*>(smem + Sh::kOffBV)[e] = make_uint4(0u, 0u, 0u, 0u);
  __syncthreads();
  volatile int* abort_flag = &ms->abort;
  auto wait = [&](uint64_t* bar, uint32_t parity) {
    mbar_wait_abortable(smem_u32(bar), parity, a.fault, kFaultDecode, abort_flag);
  };
  // Bulk copies, issued by thread 0: tile `issued` of this CTA's sequence of
  // valid tiles goes to stage issued % kStages once `done` tiles have been
  // consumed and issued < done + kStages.  The cursor (cur, cu, ct, cL) walks
  // flat tiles: unit cu, tile ct in it, context length cL of the unit.
  int64_t issued = 0, cur = f0, cu = f0 / a.tpu, ct = f0 - cu * a.tpu;
  int cL = (int)min((int64_t)max(__ldg(a.ctx_len + cu / a.Hkv), 0), a.ctx_stride);
  auto issue_upto = [&](int64_t done) {
    const uint32_t sbase = smem_u32(smem);
    while (issued < done + kStages && cur < f1 && !*abort_flag) {
      if (ct >= a.tpu || ct * kTile >= cL) {  // next unit (the rest of this one is past its context)
        cur += a.tpu - ct;
        ++cu;
        ct = 0;
        if (cur < f1) cL = (int)min((int64_t)max(__ldg(a.ctx_len + cu / a.Hkv), 0), a.ctx_stride);
        continue;
      }
      const int64_t row0 = cu * a.ctx_stride + ct * kTile;
      const int ntok = (int)min((int64_t)kTile, a.ctx_stride - ct * kTile);  // 256, or 128 at a unit's end
      ++cur;
      ++ct;
      const int s = (int)(issued & (kStages - 1));
      // the other half may still be reading the stage's previous tile
      if (issued >= kStages)
        wait(&ms->ld_empty[s], (uint32_t)(((issued - kStages) / kStages) & 1));
      ++issued;
      const uint32_t bar = smem_u32(&ms->ld_full[s]);
      const uint32_t dst = sbase + Sh::kOffRing + s * Sh::kStage;
      const int idxb = ntok * 16 * W, sgnb = ntok * 16, nrmb = ntok * 4;
      mbar_arrive_expect_tx(bar, 2 * idxb + 2 * sgnb + 4 * nrmb);
      bulk_load(dst + Sh::kOffKIdx, a.kidx + row0 * (4 * W), idxb, bar);
      bulk_load(dst + Sh::kOffKSgn, a.ksgn + row0 * 4, sgnb, bar);
      bulk_load(dst + Sh::kOffKNorm, a.knorm + row0, nrmb, bar);
      bulk_load(dst + Sh::kOffKRn, a.krnorm + row0, nrmb, bar);
      bulk_load(dst + Sh::kOffVIdx, a.vidx + (row0 >> 5) * (W * kD), idxb, bar);
      bulk_load(dst + Sh::kOffVSgn, a.vsgn + (row0 >> 5) * kD, sgnb, bar);
      bulk_load(dst + Sh::kOffVNorm, a.vnorm + row0, nrmb, bar);
      bulk_load(dst + Sh::kOffVRn, a.vrnorm + row0, nrmb, bar);
    }
  };
  if (threadIdx.x == 0) issue_upto(0);

  const int w = warp, kbk = w >> 1, g2 = w & 1, vrow = w & 7, hf = w >> 3;
  // Score rows gq, gq + 8 <-> tokens tok, tok + 1 of the tile (block kbk).
  // Their value bits are bits L and 16 + L of the block words, L = 8·g2 + gq,
  // i.e. one f16x2 operand register: this thread writes whole registers of
  // the value weights.
  const int tok = 32 * kbk + 16 * g2 + 2 * gq;
  const int crd = 16 * vrow + 2 * gq;  // value rows gq, gq + 8 <-> coordinates crd, crd + 1
  // multipliers moving bits tig, 4+tig, 8+tig, 12+tig of each half to bits
  // 3, 7, 11, 15 (mul), and each of those to bit 15 (mul·2^12 .. mul)
  const uint32_t mul = c_mul[tig][0], mul4 = c_mul[tig][1], mul8 = c_mul[tig][2], mul12 = c_mul[tig][3];
  const OperandKinds op;
  uint8_t* BK = smem + Sh::kOffBK;
  float vacc[NP][GH][4];
  float M[GH], lsum[GH], pend[GH], A0[GH], B0[GH], A1[GH], B1[GH];
  int64_t gi = 0;
  int segc = 0;
  for (int64_t f = f0; f < f1; ++segc) {
    int64_t next;
    const Seg sg = segment_at(a, f, f1, &next);
    f = next;
    const int b = (int)(sg.u / a.Hkv), h = (int)(sg.u - (int64_t)b * a.Hkv);
    const int head0 = b * a.Hq + h * a.G;
#pragma unroll
    for (int P = 0; P < NP; ++P)
#pragma unroll
      for (int ht = 0; ht < GH; ++ht)
#pragma unroll
        for (int e = 0; e < 4; ++e) vacc[P][ht][e] = 0.f;
#pragma unroll
    for (int hh = 0; hh < GH; ++hh) M[hh] = -INFINITY, lsum[hh] = 0.f, pend[hh] = 1.f;
    if (sg.n > 0) {
      // ---- query weights of this unit (f16 hi + lo, scale E per part and head) and offsets O;
      // both halves must be done with the previous unit's table first
      cta_sync();
      for (int e = threadIdx.x; e < Sh::kBKBytes / 16; e += kThreads)
        reinterpret_cast<uint4*>(BK)[e] = make_uint4(0, 0, 0, 0);
      if (threadIdx.x < 16) {
        ms->amax[threadIdx.x >> 3][threadIdx.x & 7] = 0.f;
        ms->O[threadIdx.x >> 3][threadIdx.x & 7] = 0.f;
      }
      cta_sync();
      // coordinate j: word kw, bit x = 16e + L; L = 8·ks2 + 4·hi + q -> K index 8·hi + 2q + e
      const int j = threadIdx.x & (kD - 1);
      const bool setup = threadIdx.x < kD;
      const int kw = j >> 5, e16 = (j >> 4) & 1, L = j & 15, ks2 = L >> 3, hi = (L >> 2) & 1, q4 = L & 3;
      const int kk = 8 * hi + 2 * q4 + e16;
      // exponent-kind operand (hi = 0): s = (F - mean)·2/δ; sign kind: s = -F
      const float wsc = hi ? -1.f : 2.f / kExpDelta;
      float qv[GP], sv[GP], cf[NPM];
#pragma unroll
      for (int P = 0; P < NPM; ++P) cf[P] = __ldg(a.walsh + (P < W ? (1 << P) : 7));
      if (setup) {
#pragma unroll
        for (int g = 0; g < GP; ++g) {
          qv[g] = g < a.G ? __ldg(a.qt + (size_t)(head0 + g) * kD + j) : 0.f;
          sv[g] = g < a.G ? __ldg(a.st + (size_t)(head0 + g) * kD + j) : 0.f;
          float am = 0.f;
#pragma unroll
          for (int P = 0; P < NPM; ++P) am = fmaxf(am, fabsf(wsc * cf[P] * qv[g]));
          float aq = fabsf(wsc * sv[g]);
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
            aq = fmaxf(aq, __shfl_xor_sync(0xffffffffu, aq, o));
          }
          if (lane == 0) {
            atomicMax(reinterpret_cast<int*>(&ms->amax[0][g]), __float_as_int(am));
            atomicMax(reinterpret_cast<int*>(&ms->amax[1][g]), __float_as_int(aq));
          }
        }
      }
      cta_sync();
      auto escale = [&](int p, int g) {  // power of two taking the part's largest weight below 2^12
        const float am = ms->amax[p][g];
        int ex;
        frexpf(am, &ex);
        return am > 0.f ? ldexpf(1.f, ex - 12) : 1.f;
      };
      if (setup) {
        __half* bk = reinterpret_cast<__half*>(BK);
#pragma unroll
        for (int P = 0; P < NP; ++P) {
          const int part = P < NPM ? 0 : 1;
          const int ks = (P * 4 + kw) * 2 + ks2;
#pragma unroll
          for (int g = 0; g < GP; ++g) {
            const float E = escale(part, g);
            const float x = wsc * (part == 0 ? cf[P < NPM ? P : 0] * qv[g] : sv[g]) / E;
            const __half xh = __float2half_rn(x), xl = __float2half_rn(x - __half2float(xh));
            // (k, n) sits in lane (n, k % 8 / 2), fragment k / 8, half k % 2
            const int base = ((((ks * GH + (g >> 2)) * 8 + 2 * (g & 3)) * 4 + ((kk & 7) >> 1)) * 2 + (kk >> 3)) * 2 +
                             (kk & 1);
            bk[base] = xh;
            bk[base + 16] = xl;
            float o = hi ? 0.f : (__half2float(xh) + __half2float(xl)) * E * kExpMean;
#pragma unroll
            for (int sh = 16; sh > 0; sh >>= 1) o += __shfl_xor_sync(0xffffffffu, o, sh);
            if (lane == 0) atomicAdd(&ms->O[part][g], o);
          }
        }
      }
      cta_sync();
      {
        const float c = a.scale * kLog2e;
#pragma unroll
        for (int hh = 0; hh < GH; ++hh) {
          const int g = 4 * hh + tig;
          A0[hh] = c * escale(0, g);
          B0[hh] = -c * ms->O[0][g];
          A1[hh] = c * a.alpha * escale(1, g);
          B1[hh] = -c * a.alpha * ms->O[1][g];
        }
      }
      auto bfrag = [&](int ks, int ht) -> uint2 {
        return reinterpret_cast<const uint2*>(BK)[((ks * GH + ht) * 8 + gq) * 4 + tig];
      };
      // ---- tiles.  Per tile k: weights of tile k-1 | barrier | values of tile
      // k-1 and scores of tile k (one straight block) | barrier + vote.
      float s2p[GH][2], vnp[2], vrp[2];  // tile k-1: scores (log2 units), cleaned value norms
      float s2c[GH][2], vnc[2], vrc[2], mx[GH];

      // attention weights of the previous tile -> value operand registers (hi, lo)
      auto weights_step = [&](int kp) {
        uint32_t* bv = reinterpret_cast<uint32_t*>(smem + Sh::kOffBV + (kp & 1) * Sh::kBVBuf);
#pragma unroll
        for (int hh = 0; hh < GH; ++hh) {
          float p[2];
#pragma unroll
          for (int r = 0; r < 2; ++r) p[r] = s2p[hh][r] == -INFINITY ? 0.f : exp2f(s2p[hh][r] - M[hh]);
          lsum[hh] += p[0] + p[1];
#pragma unroll
          for (int part = 0; part < 2; ++part) {
            const float x0 = p[0] * (part == 0 ? vnp[0] : vrp[0]) * kWS;
            const float x1 = p[1] * (part == 0 ? vnp[1] : vrp[1]) * kWS;
            const uint32_t whi = f16x2_of(x0, x1);
            const float2 back = __half22float2(*reinterpret_cast<const __half2*>(&whi));
            const uint32_t wlo = f16x2_of(x0 - back.x, x1 - back.y);
            const int base =
                ((((part * GH + hh) * kBlocks + kbk) * 2 + g2) * 8 + 2 * tig) * 8 + (gq & 3) * 2 + (gq >> 2);
            bv[base] = whi;
            bv[base + 8] = wlo;
          }
        }
      };

      // values of tile kv (CTA tile index gv): 16 coordinates of every plane over
      // blocks 4·hf .. 4·hf + 3.  A short tile's upper blocks hold stale
      // words with zero weights.
      auto values_step = [&](int kv, int64_t gv) {
        const uint8_t* stg = smem + Sh::kOffRing + (int)(gv & (kStages - 1)) * Sh::kStage;
        const uint32_t* vi = reinterpret_cast<const uint32_t*>(stg + Sh::kOffVIdx);
        const uint32_t* vsg = reinterpret_cast<const uint32_t*>(stg + Sh::kOffVSgn);
        const uint32_t* bv = reinterpret_cast<const uint32_t*>(smem + Sh::kOffBV + (kv & 1) * Sh::kBVBuf);
        // the reference moved at tile kv: bring the earlier tiles to it (factor 1 otherwise)
#pragma unroll
        for (int P = 0; P < NP; ++P)
#pragma unroll
          for (int ht = 0; ht < GH; ++ht)
#pragma unroll
            for (int e = 0; e < 4; ++e) vacc[P][ht][e] *= pend[ht];
#pragma unroll
        for (int i = 0; i < kBlocks / 2; ++i) {
          const int kb = (kBlocks / 2) * hf + i;
          uint2 bb[2][GH][2];  // [part][head tile][K half]
#pragma unroll
          for (int part = 0; part < 2; ++part)
#pragma unroll
            for (int ht = 0; ht < GH; ++ht)
#pragma unroll
              for (int s2i = 0; s2i < 2; ++s2i)
                bb[part][ht][s2i] = *reinterpret_cast<const uint2*>(
                    bv + (((((part * GH + ht) * kBlocks + kb) * 2 + s2i) * 8 + gq) * 4 + tig) * 2);
#pragma unroll
          for (int P = 0; P < NP; ++P) {
            uint2 ww;
            if (P < W) {
              ww = *reinterpret_cast<const uint2*>(vi + (kb * W + P) * kD + crd);
            } else if (P < NPM) {  // product plane
              const uint2 x0 = *reinterpret_cast<const uint2*>(vi + (kb * W) * kD + crd);
              const uint2 x1 = *reinterpret_cast<const uint2*>(vi + (kb * W + 1 % W) * kD + crd);
              const uint2 x2 = *reinterpret_cast<const uint2*>(vi + (kb * W + 2 % W) * kD + crd);
              ww = make_uint2(x0.x ^ x1.x ^ x2.x, x0.y ^ x1.y ^ x2.y);
            } else {
              ww = *reinterpret_cast<const uint2*>(vsg + kb * kD + crd);
            }
            const int part = P < NPM ? 0 : 1;
            // every layer as a sign operand: bit 15 of the word times mul·(4096, 256, 16, 1)
            const uint32_t a00 = op.sign(ww.x * mul12), a01 = op.sign(ww.y * mul12);
            const uint32_t a02 = op.sign(ww.x * mul8), a03 = op.sign(ww.y * mul8);
            const uint32_t a10 = op.sign(ww.x * mul4), a11 = op.sign(ww.y * mul4);
            const uint32_t a12 = op.sign(ww.x * mul), a13 = op.sign(ww.y * mul);
#pragma unroll
            for (int ht = 0; ht < GH; ++ht) {
              mma_f16(vacc[P][ht], a00, a01, a02, a03, bb[part][ht][0].x, bb[part][ht][0].y);
              mma_f16(vacc[P][ht], a10, a11, a12, a13, bb[part][ht][1].x, bb[part][ht][1].y);
            }
          }
        }
      };

      // scores of tile kc (CTA tile index gc, stage already landed): 16 tokens
      // -> s2c, cleaned norms, and the tile maximum
      auto scores_step = [&](int kc, int64_t gc) {
        const uint8_t* stg = smem + Sh::kOffRing + (int)(gc & (kStages - 1)) * Sh::kStage;
        const uint4* kq = reinterpret_cast<const uint4*>(stg + Sh::kOffKIdx);  // token t, plane P: kq[t·W + P]
        const uint4* sq = reinterpret_cast<const uint4*>(stg + Sh::kOffKSgn);  // token t: sq[t]
        float acc[2][GH][4];  // [part][head tile][fragment]
#pragma unroll
        for (int pt = 0; pt < 2; ++pt)
#pragma unroll
          for (int ht = 0; ht < GH; ++ht)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[pt][ht][e] = 0.f;
#pragma unroll
        for (int P = 0; P < NP; ++P) {
          const int part = P < NPM ? 0 : 1;
          uint4 wd[2];  // [row]
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            const int t = tok + r;
            if (P < W) {
              wd[r] = kq[t * W + P];
            } else if (P < NPM) {  // product plane b0 ^ b1 ^ b2
              const uint4 x0 = kq[t * W], x1 = kq[t * W + 1 % W], x2 = kq[t * W + 2 % W];
              wd[r] = make_uint4(x0.x ^ x1.x ^ x2.x, x0.y ^ x1.y ^ x2.y, x0.z ^ x1.z ^ x2.z, x0.w ^ x1.w ^ x2.w);
            } else {
              wd[r] = sq[t];
            }
          }
#pragma unroll
          for (int kw = 0; kw < 4; ++kw) {
            const int ks = (P * 4 + kw) * 2;
            const uint32_t x0 = word_of(wd[0], kw), x1 = word_of(wd[1], kw);
            const uint32_t t0 = x0 * mul, t1 = x1 * mul;    // layers 8+q, 12+q at bits 11, 15
            const uint32_t u0 = x0 * mul8, u1 = x1 * mul8;  // layers q, 4+q at bits 11, 15
#pragma unroll
            for (int ht = 0; ht < GH; ++ht) {
              const uint2 b0 = bfrag(ks, ht), b1 = bfrag(ks + 1, ht);
              mma_f16(acc[part][ht], op.expo(u0), op.expo(u1), op.sign(u0), op.sign(u1), b0.x, b0.y);
              mma_f16(acc[part][ht], op.expo(t0), op.expo(t1), op.sign(t0), op.sign(t1), b1.x, b1.y);
            }
          }
        }
        const float* kn = reinterpret_cast<const float*>(stg + Sh::kOffKNorm);
        const float* kr = reinterpret_cast<const float*>(stg + Sh::kOffKRn);
        const float* vn = reinterpret_cast<const float*>(stg + Sh::kOffVNorm);
        const float* vr = reinterpret_cast<const float*>(stg + Sh::kOffVRn);
        const int64_t tb = (sg.t0 + kc) * kTile;
        const float2 kn2 = *reinterpret_cast<const float2*>(kn + tok), kr2 = *reinterpret_cast<const float2*>(kr + tok);
        const float2 vn2 = *reinterpret_cast<const float2*>(vn + tok), vr2 = *reinterpret_cast<const float2*>(vr + tok);
#pragma unroll
        for (int hh = 0; hh < GH; ++hh) mx[hh] = -INFINITY;
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const bool valid = tb + tok + r < sg.L;
          vnc[r] = valid ? (r ? vn2.y : vn2.x) : 0.f;
          vrc[r] = valid ? (r ? vr2.y : vr2.x) : 0.f;
          const float knr = r ? kn2.y : kn2.x, krr = r ? kr2.y : kr2.x;
          const float lv = __log2f(fmaxf(fmaxf(vnc[r], vrc[r]), 0x1p-32f));
#pragma unroll
          for (int hh = 0; hh < GH; ++hh) {
            const float dm = acc[0][hh][2 * r] + acc[0][hh][2 * r + 1];
            const float dq = acc[1][hh][2 * r] + acc[1][hh][2 * r + 1];
            const float sc = fmaf(knr, fmaf(A0[hh], dm, B0[hh]), krr * fmaf(A1[hh], dq, B1[hh]));
            s2c[hh][r] = (valid && 4 * hh + tig < a.G) ? sc : -INFINITY;
            mx[hh] = fmaxf(mx[hh], s2c[hh][r] + lv);
          }
        }
#pragma unroll
        for (int hh = 0; hh < GH; ++hh)
#pragma unroll
          for (int o = 4; o < 32; o <<= 1) mx[hh] = fmaxf(mx[hh], __shfl_xor_sync(0xffffffffu, mx[hh], o));
      };

      // Second barrier of a tile (this half's warps): the vote of the lazy
      // reference on the scores just computed.  With have_values, this half is
      // through tile done - 1, whose stage it hands back; thread 0 refills
      // stages.  The scores and norms move to the "previous tile" slots.
      auto vote_step = [&](bool have_scores, bool have_values, int64_t done) {
        bool exceed = false;
        if (have_scores) {
#pragma unroll
          for (int hh = 0; hh < GH; ++hh)
            exceed |= M[hh] == -INFINITY ? mx[hh] > -INFINITY : mx[hh] > M[hh] + kTau;
        }
        const bool bump = half_any(hf, exceed);
        if (have_values && (threadIdx.x & (kThreads / 2 - 1)) == 0)
          mbar_arrive(smem_u32(&ms->ld_empty[(done - 1) & (kStages - 1)]));
        if (threadIdx.x == 0) issue_upto(done);
        float fac[GH];
#pragma unroll
        for (int hh = 0; hh < GH; ++hh) fac[hh] = 1.f;
        if (bump) {
          if (gq == 0) {
#pragma unroll
            for (int hh = 0; hh < GH; ++hh) ms->red[w][4 * hh + tig] = mx[hh];
          }
          half_sync(hf);
#pragma unroll
          for (int hh = 0; hh < GH; ++hh) {
            float tm = ms->red[8 * hf][4 * hh + tig];
#pragma unroll
            for (int q = 1; q < kNW / 2; ++q) tm = fmaxf(tm, ms->red[8 * hf + q][4 * hh + tig]);
            float nm = M[hh];
            if (M[hh] == -INFINITY || tm > M[hh] + kTau) nm = tm;
            fac[hh] = nm == M[hh] ? 1.f : exp2f(M[hh] - nm);
            M[hh] = nm;
            lsum[hh] *= fac[hh];
          }
        }
#pragma unroll
        for (int hh = 0; hh < GH; ++hh) pend[hh] = fac[hh], s2p[hh][0] = s2c[hh][0], s2p[hh][1] = s2c[hh][1];
#pragma unroll
        for (int r = 0; r < 2; ++r) vnp[r] = vnc[r], vrp[r] = vrc[r];
      };

      // prologue: scores of the first tile
      wait(&ms->ld_full[gi & (kStages - 1)], (uint32_t)((gi / kStages) & 1));
      scores_step(0, gi);
      vote_step(true, false, gi);
      // steady state: the wait comes first so that values and scores form one block
      for (int k = 1; k < sg.n; ++k) {
        const int64_t g = gi + k;
        weights_step(k - 1);
        half_sync(hf);
        wait(&ms->ld_full[g & (kStages - 1)], (uint32_t)((g / kStages) & 1));
        values_step(k - 1, g - 1);
        scores_step(k, g);
        vote_step(true, true, g);
      }
      // epilogue: weights and values of the last tile
      weights_step(sg.n - 1);
      half_sync(hf);
      values_step(sg.n - 1, gi + sg.n - 1);
      vote_step(false, true, gi + sg.n);
      gi += sg.n;
    }
    // ---- partials of this CTA for the unit: one per half (slot 2·slot + half),
    // each over its own tokens with its own reference
    const int sp = segc & 1;
#pragma unroll
    for (int hh = 0; hh < GH; ++hh) {
      float l = lsum[hh];
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
      if (gq == 0) ms->lred[sp][w][4 * hh + tig] = l;
    }
    half_sync(hf);
    float cf[NPM];
#pragma unroll
    for (int P = 0; P < NPM; ++P) cf[P] = __ldg(a.walsh + (P < W ? (1 << P) : 7));
#pragma unroll
    for (int hh = 0; hh < GH; ++hh) {
      const int head = 4 * hh + tig;
      if (head < a.G) {
        float* pp = a.part + ((size_t)(head0 + head) * a.smax + 2 * sg.slot + hf) * (2 + 2 * kD);
        // fragment e = 2·row + piece; the value operand is -s, so sums enter negated
        float rot[2], sgn[2];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          float x = 0.f;
#pragma unroll
          for (int P = 0; P < NPM; ++P) x = fmaf(cf[P], vacc[P][hh][2 * r] + vacc[P][hh][2 * r + 1], x);
          rot[r] = -x * (1.f / kWS);
          sgn[r] = -(vacc[NPM][hh][2 * r] + vacc[NPM][hh][2 * r + 1]) * (1.f / kWS);
        }
        *reinterpret_cast<float2*>(pp + 2 + crd) = make_float2(rot[0], rot[1]);
        *reinterpret_cast<float2*>(pp + 2 + kD + crd) = make_float2(sgn[0], sgn[1]);
        if (vrow == 0 && gq == 0) {
          float l = 0.f;
#pragma unroll
          for (int q = 0; q < kNW / 2; ++q) l += ms->lred[sp][8 * hf + q][head];
          pp[0] = M[hh];
          pp[1] = l;
        }
      }
    }
  }
  // no copy of this CTA may be in flight when it exits
  if (threadIdx.x == 0)
    for (int64_t g = max((int64_t)0, issued - kStages); g < issued; ++g)
      mbar_wait(smem_u32(&ms->ld_full[g & (kStages - 1)]), (uint32_t)((g / kStages) & 1), a.fault, kFaultDecode);
  __syncthreads();
}

}  // namespace

namespace tq {

int64_t decode_tc_tpu(int64_t ctx_stride) { return (ctx_stride + kTile - 1) / kTile; }

// Partial slots per unit for a grid of `ctas` CTAs over units * tpu tiles: two
// per CTA that touches the unit (one per half of its warps).
int decode_tc_slots(int64_t units, int64_t tpu, int64_t ctas) {
  const int64_t total = units * tpu;
  int64_t smax = 1;
  for (int64_t u = 0; u < units; ++u) {
    const int64_t s = owner((u + 1) * tpu - 1, total, ctas) - owner(u * tpu, total, ctas) + 1;
    smax = std::max(smax, s);
  }
  return 2 * (int)smax;  // one partial per half of each CTA
}

int decode_tc_ctas(int64_t units, int64_t tpu) { return (int)std::min<int64_t>(units * tpu, sm_count()); }

bool decode_tc_supported(const tq_plan* plan, int G, const tq_records* V, int64_t ctx_stride) {
  return plan->d == 128 && plan->m == 128 && G >= 1 && G <= 8 && V->layout == TQ_LAYOUT_BLOCK32 &&
         ctx_stride % kHalfTile == 0;
}

tq_status launch_decode_tc(const tq_plan* plan, const tq_records* K, const tq_records* V, const int32_t* ctx_len,
                           int B, int Hq, int Hkv, int64_t ctx_stride, float scale, const float* qt, const float* st,
                           float* part, int smax, cudaStream_t stream) {
  TcArgs a{};
  a.kidx = K->idx; a.ksgn = K->sgn; a.knorm = K->norm; a.krnorm = K->rnorm;
  a.vidx = V->idx; a.vsgn = V->sgn; a.vnorm = V->norm; a.vrnorm = V->rnorm;
  a.ctx_len = ctx_len;
  a.ctx_stride = ctx_stride;
  a.B = B; a.Hq = Hq; a.Hkv = Hkv; a.G = Hq / Hkv;
  a.qt = qt; a.st = st;
  a.walsh = plan->walsh;
  a.scale = scale;
  a.alpha = plan->qjl_alpha;
  a.part = part;
  a.smax = smax;
  a.tpu = decode_tc_tpu(ctx_stride);
  a.total = (int64_t)B * Hkv * a.tpu;
  a.fault = fault_word();
  if (!a.fault) return TQ_ERR_CUDA;
  const int grid = decode_tc_ctas((int64_t)B * Hkv, a.tpu);
  auto go = [&](auto kern, int smem) -> tq_status {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return TQ_ERR_CUDA;
    kern<<<grid, kThreads, smem, stream>>>(a);
    return launch_status();
  };
  const bool g8 = a.G > 4;
  switch (plan->w) {
    case 1: return g8 ? go(decode_tc_kernel<1, 8>, smem_bytes<1>()) : go(decode_tc_kernel<1, 4>, smem_bytes<1>());
    case 2: return g8 ? go(decode_tc_kernel<2, 8>, smem_bytes<2>()) : go(decode_tc_kernel<2, 4>, smem_bytes<2>());
    default: return g8 ? go(decode_tc_kernel<3, 8>, smem_bytes<3>()) : go(decode_tc_kernel<3, 4>, smem_bytes<3>());
  }
}

}  // namespace tq

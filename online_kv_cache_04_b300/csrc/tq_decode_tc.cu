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
// signs are one more ±1 plane.
//   keys:   one and-or keeps bit i of every byte of a plane word over a
//           constant e4m3 byte C_i (layer i), giving per element one of two
//           exact values C_i, C'_i; the map back to ±1 is folded into the
//           query weights (2x/(C' − C)) and a per-(batch, kv head) offset.
//   values: a shift and an and-or move bit i of every byte to the sign of
//           1.0, so the operand is exactly −s; no offset is needed, which
//           keeps the long sums over the context free of cancellation.
//
//   scores: mma.sync m16n8k32 e4m3, rows = 16 tokens, K = the 32 coordinates
//           of one plane word, B = the query weights in three e4m3 pieces
//           (each the next 4 bits; one power-of-two scale per head and part).
//   values: the same instruction with rows = 16 coordinates and K = the 32
//           tokens of one block word (TQ_LAYOUT_BLOCK32), B = the attention
//           weights p·‖v‖ and p·‖r_v‖ rounded to f16 and split exactly into
//           three e4m3 pieces; fp32 accumulators stay in registers over the
//           whole context.
// Warp-level mma.sync rather than tcgen05.mma: decode has one query per
// head, so every product here is at most 32 columns wide, and a tcgen05.mma
// costs its issuing thread over a hundred cycles whatever its width.
//
// Work split.  A persistent grid of one CTA per SM takes contiguous ranges of
// 128-token tiles over all (batch, kv head) units; a unit cut between CTAs
// leaves one partial per CTA, merged by the combine kernel of tq_decode.cu.
// Eight warps do the same work: warp w scores 16 tokens of each tile and
// accumulates values for 16 coordinates.  The weights of a tile go through
// shared memory, already laid out as the value operand, and the warps
// pipeline one tile deep (scores of tile i, then values of tile i − 1), so
// one named barrier per tile orders everything: it publishes the weights, it
// frees the ring stage of tile i − 2, into which one thread then starts the
// bulk copies of a later tile, and it carries the vote of the lazy softmax.
//
// Softmax is online with a lazy reference: the running reference M (of
// log2(p·max(‖v‖, ‖r_v‖)), clamped at 2^-32) moves only when a tile exceeds
// it by more than 2^6; the workers then rescale their accumulators.  Every
// mbarrier wait is bounded; on timeout the kernel sets a fault bit
// (tq_fault_flags), skips the remaining waits and runs to its end.
#include <cuda_fp16.h>

#include <algorithm>

#include "tq_internal.h"
#include "tq_sm100.cuh"

namespace {

using namespace tq::sm100;

constexpr int kNW = 8;                                 // worker warps
constexpr int kTile = 16 * kNW;                        // tokens per tile
constexpr int kD = 128;
constexpr int kStages = 6;
constexpr int kWorkers = 32 * kNW;
constexpr int kThreads = kWorkers;
constexpr float kTau = 6.0f;                           // lazy-rescale threshold (log2 units)
constexpr float kLog2e = 1.4426950408889634f;
constexpr unsigned kFaultDecode = 2u;

// key operand: layer i = bit i of each byte over the e4m3 byte C_i
__constant__ uint32_t c_base[8] = {0x38383838u, 0x38383838u, 0x38383838u, 0x30303030u,
                                   0x28282828u, 0x18181818u, 0x00000000u, 0x38383838u};
__constant__ float c_delta[8] = {0.125f, 0.25f, 0.5f, 0.5f, 0.75f, 0.9375f, 2.0f, -2.0f};     // C' - C
__constant__ float c_mean[8] = {1.0625f, 1.125f, 1.25f, 0.75f, 0.625f, 0.53125f, 1.0f, 0.0f};  // (C + C')/2

// A-operand register of layer q (lo) or 4 + q (hi) of a key plane word.
struct Layers {
  uint32_t mlo, mhi, blo, bhi;
  __device__ __forceinline__ explicit Layers(int q)
      : mlo(0x01010101u << q), mhi(0x10101010u << q), blo(c_base[q]), bhi(c_base[4 + q]) {}
  __device__ __forceinline__ uint32_t lo(uint32_t w) const { return (w & mlo) | blo; }
  __device__ __forceinline__ uint32_t hi(uint32_t w) const { return (w & mhi) | bhi; }
};

// Value operand: bit 7 - sh of every byte of w as the sign of 1.0 (set -> -1).
__device__ __forceinline__ uint32_t sign_layer(uint32_t w, int sh) { return ((w << sh) & 0x80808080u) | 0x38383838u; }

__device__ __forceinline__ void mma_e4m3(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ---- packed conversions (low half <-> low byte)
__device__ __forceinline__ uint32_t f16x2_of(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ uint16_t e4m3x2_of(uint32_t h) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(r) : "r"(h));
  return r;
}
__device__ __forceinline__ uint32_t f16x2_of_e4m3x2(uint16_t b) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(b));
  return r;
}
__device__ __forceinline__ uint32_t residual16(uint32_t y, uint32_t v) {  // (y - v)·16, exact
  uint32_t r;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(y), "r"(v));
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(r), "r"(0x4C004C00u));
  return r;
}

// Two weights rounded to f16 and split into three e4m3 pieces each (piece k
// = the next 4 bits, weight = p0 + p1/16 + p2/256 exactly): e4m3 pairs.
__device__ __forceinline__ void pieces_pair(float lo, float hi, uint16_t (&p)[3]) {
  uint32_t y = f16x2_of(lo, hi);
#pragma unroll
  for (int k = 0; k < 3; ++k) {
    p[k] = e4m3x2_of(y);
    if (k < 2) y = residual16(y, f16x2_of_e4m3x2(p[k]));
  }
}

// Three e4m3 pieces of one float (query weights, once per unit).
__device__ __forceinline__ float pieces3(float x, uint8_t (&p)[3]) {
  float rep = 0.f, sc = 1.f;
#pragma unroll
  for (int k = 0; k < 3; ++k) {
    const uint16_t b = e4m3x2_of(f16x2_of(x, 0.f)) & 0xFFu;  // x in f16 first: exact split of its 11 bits
    const float v = __half2float(__ushort_as_half((uint16_t)(f16x2_of_e4m3x2(b) & 0xFFFFu)));
    p[k] = (uint8_t)b;
    rep = fmaf(v, sc, rep);
    x = (x - v) * 16.f;
    sc *= 0.0625f;
  }
  return rep;
}

// Named barrier of the worker warps, and the same barrier with an OR vote.
__device__ __forceinline__ void workers_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kWorkers) : "memory"); }
__device__ __forceinline__ bool workers_any(bool p) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred q, o;\n setp.ne.u32 q, %1, 0;\n bar.red.or.pred o, 1, %2, q;\n selp.u32 %0, 1, 0, o;\n}"
      : "=r"(r)
      : "r"((uint32_t)p), "n"(kWorkers)
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
  int64_t tpu;       // tiles per unit = ctx_stride / 128
  int64_t total;     // units * tpu
  unsigned* fault;
};

// CTA that owns flat tile f when `total` tiles are cut into `ctas` even ranges.
__host__ __device__ inline int64_t owner(int64_t f, int64_t total, int64_t ctas) {
  return ((f + 1) * ctas - 1) / total;
}

// Column of piece k (0..2) of head g in the score and weight operands.  The
// thread with quad index q holds columns 2q, 2q+1 | 8+2q, 9+2q | 16+2q, 17+2q
// of the n-tiles; head q takes the first three, head 4 + q the last three.
__host__ __device__ constexpr int col_of(int k, int g) {
  return g < 4 ? (k < 2 ? 2 * g + k : 8 + 2 * g) : (k == 0 ? 9 + 2 * (g - 4) : 16 + 2 * (g - 4) + (k - 1));
}

// p0 + p1/16 + p2/256 of head slot hh (head q or 4 + q), row j, from one
// accumulator set [n-tile][fragment].
template <int NT>
__device__ __forceinline__ float combine3(const float (&c)[NT][4], int hh, int j) {
  if constexpr (NT >= 3) {
    if (hh == 1) return fmaf(c[2][2 * j + 1], 1.f / 256.f, fmaf(c[2][2 * j], 1.f / 16.f, c[1][2 * j + 1]));
  }
  return fmaf(c[1][2 * j], 1.f / 256.f, fmaf(c[0][2 * j + 1], 1.f / 16.f, c[0][2 * j]));
}

template <int W, int GP>
struct Shape {
  static constexpr int NPM = W == 3 ? 4 : W;   // ±1 planes of the codebook
  static constexpr int NP = NPM + 1;           // plus the QJL sign plane
  static constexpr int NKS = 4 * NP;           // score K-steps: 4 words of 32 coordinates per plane
  static constexpr int NT = GP == 8 ? 3 : 2;   // n-tiles of 8 columns (3 pieces x GP heads)
  static constexpr int GH = GP / 4;            // heads per thread
  static constexpr bool kBRegs = NKS * NT * 2 <= 48;  // query-weight fragments held in registers
  static constexpr int kIdxBytes = kTile * 4 * W * 4;
  static constexpr int kSgnBytes = kTile * 16, kNormBytes = kTile * 4;
  static constexpr int kStage = 2 * kIdxBytes + 2 * kSgnBytes + 4 * kNormBytes;
  static constexpr int kOffKIdx = 0, kOffKSgn = kIdxBytes, kOffKNorm = kOffKSgn + kSgnBytes,
                       kOffKRn = kOffKNorm + kNormBytes;
  static constexpr int kOffVIdx = kOffKRn + kNormBytes, kOffVSgn = kOffVIdx + kIdxBytes,
                       kOffVNorm = kOffVSgn + kSgnBytes, kOffVRn = kOffVNorm + kNormBytes;
  // shared memory plan
  static constexpr int kBKBytes = NKS * NT * 256;     // [ks][nt][n 8][k 32] query weight bytes
  static constexpr int kBVBuf = 2 * 4 * NT * 256;     // [part][block][nt][n 8][quad 4][b0, b1] weight words
  static constexpr int kOffRing = 0;
  static constexpr int kOffBK = kOffRing + kStages * kStage;
  static constexpr int kOffBV = kOffBK + kBKBytes;
  static constexpr int kOffMisc = kOffBV + 2 * kBVBuf;
};

struct Misc {
  uint64_t ld_full[kStages];
  int abort;
  int rescale[2];             // per weight buffer: the reference moved for this tile
  float fac[2][8];            // per weight buffer: accumulator rescale factor per head
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
  constexpr int NPM = Sh::NPM, NP = Sh::NP, NKS = Sh::NKS, NT = Sh::NT, GH = Sh::GH;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Misc* ms = reinterpret_cast<Misc*>(smem + Sh::kOffMisc);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gq = lane >> 2, tig = lane & 3;  // mma fragment coordinates
  const int64_t C = gridDim.x;
  const int64_t f0 = (int64_t)blockIdx.x * a.total / C, f1 = ((int64_t)blockIdx.x + 1) * a.total / C;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(smem_u32(&ms->ld_full[s]), 1);
    ms->abort = 0;
    fence_mbar_init();
  }
  // weight operands start at zero (padding columns are never written)
  for (int e = threadIdx.x; e < 2 * Sh::kBVBuf / 16; e += kThreads)
    reinterpret_cast<uint4*>(smem + Sh::kOffBV)[e] = make_uint4(0u, 0u, 0u, 0u);
  __syncthreads();
  volatile int* abort_flag = &ms->abort;
  auto wait = [&](uint64_t* bar, uint32_t parity) {
    mbar_wait_abortable(smem_u32(bar), parity, a.fault, kFaultDecode, abort_flag);
  };
  // Bulk copies, issued by thread 0: tile `issued` of this CTA's sequence of
  // valid tiles goes to stage issued % kStages once the tile kStages earlier
  // has been consumed (`done` tiles are).
  int64_t issued = 0, cur = f0;
  auto issue_upto = [&](int64_t done) {
    const uint32_t sbase = smem_u32(smem);
    while (issued < done + kStages && cur < f1 && !*abort_flag) {
      const int64_t u = cur / a.tpu, t = cur - u * a.tpu;
      const int L = (int)min((int64_t)max(__ldg(a.ctx_len + u / a.Hkv), 0), a.ctx_stride);
      if (t * kTile >= L) {  // rest of the unit is past its context length
        cur = (u + 1) * a.tpu;
        continue;
      }
      ++cur;
      const int s = (int)(issued % kStages);
      ++issued;
      const int64_t row0 = u * a.ctx_stride + t * kTile;
      const uint32_t bar = smem_u32(&ms->ld_full[s]);
      const uint32_t dst = sbase + Sh::kOffRing + s * Sh::kStage;
      mbar_arrive_expect_tx(bar, Sh::kStage);
      bulk_load(dst + Sh::kOffKIdx, a.kidx + row0 * (4 * W), Sh::kIdxBytes, bar);
      bulk_load(dst + Sh::kOffKSgn, a.ksgn + row0 * 4, Sh::kSgnBytes, bar);
      bulk_load(dst + Sh::kOffKNorm, a.knorm + row0, Sh::kNormBytes, bar);
      bulk_load(dst + Sh::kOffKRn, a.krnorm + row0, Sh::kNormBytes, bar);
      bulk_load(dst + Sh::kOffVIdx, a.vidx + (row0 >> 5) * (W * kD), Sh::kIdxBytes, bar);
      bulk_load(dst + Sh::kOffVSgn, a.vsgn + (row0 >> 5) * kD, Sh::kSgnBytes, bar);
      bulk_load(dst + Sh::kOffVNorm, a.vnorm + row0, Sh::kNormBytes, bar);
      bulk_load(dst + Sh::kOffVRn, a.vrnorm + row0, Sh::kNormBytes, bar);
    }
  };
  if (threadIdx.x == 0) issue_upto(0);
  {
    const int w = warp, kbw = w >> 1, hf = w & 1;
    // score rows gq, gq + 8 <-> tokens tok[0], tok[1] of the tile: their bits sit
    // in byte (2·hf + j) of layer gq of block word kbw, which is what lets this
    // thread write whole operand half-words of the value weights
    const int tok[2] = {32 * kbw + 2 * gq + hf, 32 * kbw + 16 + 2 * gq + hf};
    const int crd = 16 * w + 2 * gq;  // value rows gq, gq + 8 <-> coordinates crd, crd + 1
    const int shl = 7 - tig, shh = 3 - tig;
    const Layers ly(tig);
    uint8_t* BK = smem + Sh::kOffBK;
    uint32_t bf[Sh::kBRegs ? NKS : 1][NT][2];
    float vacc[NP][NT][4];
    float M[GH], lsum[GH], A0[GH], B0[GH], A1[GH], B1[GH];
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
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) vacc[P][nt][e] = 0.f;
#pragma unroll
      for (int hh = 0; hh < GH; ++hh) M[hh] = -INFINITY, lsum[hh] = 0.f;
      if (sg.n > 0) {
        // ---- query weights of this unit: piece scales E, pieces in BK, offsets O
        for (int e = threadIdx.x; e < Sh::kBKBytes / 16; e += kWorkers)
          reinterpret_cast<uint4*>(BK)[e] = make_uint4(0, 0, 0, 0);
        if (threadIdx.x < 16) {
          ms->amax[threadIdx.x >> 3][threadIdx.x & 7] = 0.f;
          ms->O[threadIdx.x >> 3][threadIdx.x & 7] = 0.f;
        }
        workers_sync();
        const int j = threadIdx.x & (kD - 1);  // coordinate: word j / 32, bit x = j % 32 -> layer x % 8, byte x / 8
        const bool setup = threadIdx.x < kD;
        const int jl = j & 7, jk = 4 * jl + ((j & 31) >> 3), jw = j >> 5;
        const float dl = c_delta[jl], mean = c_mean[jl];
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
            for (int P = 0; P < NPM; ++P) am = fmaxf(am, fabsf(2.f * cf[P] * qv[g] / dl));
            float aq = fabsf(2.f * sv[g] / dl);
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
        workers_sync();
        auto escale = [&](int p, int g) {
          const float am = ms->amax[p][g];
          int e;
          frexpf(am, &e);
          return am > 0.f ? ldexpf(1.f, e - 8) : 1.f;
        };
        if (setup) {
#pragma unroll
          for (int P = 0; P < NP; ++P) {
            const int part = P < NPM ? 0 : 1;
#pragma unroll
            for (int g = 0; g < GP; ++g) {
              const float E = escale(part, g);
              const float x = (part == 0 ? 2.f * cf[P < NPM ? P : 0] * qv[g] : 2.f * sv[g]) / dl;
              uint8_t pc[3];
              const float rep = pieces3(x / E, pc);
#pragma unroll
              for (int k = 0; k < 3; ++k) {
                const int c = col_of(k, g);
                BK[(((P * 4 + jw) * NT + (c >> 3)) * 8 + (c & 7)) * 32 + jk] = pc[k];
              }
              float o = rep * E * mean;
#pragma unroll
              for (int s = 16; s > 0; s >>= 1) o += __shfl_xor_sync(0xffffffffu, o, s);
              if (lane == 0) atomicAdd(&ms->O[part][g], o);
            }
          }
        }
        workers_sync();
        {
          const float c = a.scale * kLog2e;
#pragma unroll
          for (int hh = 0; hh < GH; ++hh) {
            const int g = tig + 4 * hh;
            A0[hh] = c * escale(0, g);
            B0[hh] = -c * ms->O[0][g];
            A1[hh] = c * a.alpha * escale(1, g);
            B1[hh] = -c * a.alpha * ms->O[1][g];
          }
        }
        if constexpr (Sh::kBRegs) {
#pragma unroll
          for (int ks = 0; ks < NKS; ++ks)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              const uint32_t* row = reinterpret_cast<const uint32_t*>(BK + ((ks * NT + nt) * 8 + gq) * 32);
              bf[ks][nt][0] = row[tig];
              bf[ks][nt][1] = row[4 + tig];
            }
        }

        // ---- tiles: scores of tile k, then values of tile k - 1
        for (int k = 0; k <= sg.n; ++k) {
          const int64_t g = gi + k;
          const bool keys = k < sg.n;
          float s2[GH][2], mx[GH], vnc[2], vrc[2];
          bool exceed = false;
          if (keys) {
            const int s = (int)(g % kStages);
            wait(&ms->ld_full[s], (uint32_t)((g / kStages) & 1));
            const uint8_t* stg = smem + Sh::kOffRing + s * Sh::kStage;
            const uint4* kq = reinterpret_cast<const uint4*>(stg + Sh::kOffKIdx);  // token t, plane P: kq[t·W + P]
            const uint4* sq = reinterpret_cast<const uint4*>(stg + Sh::kOffKSgn);  // token t: sq[t]
            uint4 wd[2][NP];
#pragma unroll
            for (int r = 0; r < 2; ++r) {
#pragma unroll
              for (int P = 0; P < W; ++P) wd[r][P] = kq[tok[r] * W + P];
              if constexpr (W == 3) {  // product plane b0 ^ b1 ^ b2
                wd[r][3].x = wd[r][0].x ^ wd[r][1].x ^ wd[r][2].x;
                wd[r][3].y = wd[r][0].y ^ wd[r][1].y ^ wd[r][2].y;
                wd[r][3].z = wd[r][0].z ^ wd[r][1].z ^ wd[r][2].z;
                wd[r][3].w = wd[r][0].w ^ wd[r][1].w ^ wd[r][2].w;
              }
              wd[r][NPM] = sq[tok[r]];
            }
            float acc[NP][NT][4];
#pragma unroll
            for (int P = 0; P < NP; ++P)
#pragma unroll
              for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[P][nt][e] = 0.f;
#pragma unroll
            for (int kw = 0; kw < 4; ++kw)
#pragma unroll
              for (int P = 0; P < NP; ++P) {
                const int ks = 4 * P + kw;
                const uint32_t xa = kw == 0 ? wd[0][P].x : kw == 1 ? wd[0][P].y : kw == 2 ? wd[0][P].z : wd[0][P].w;
                const uint32_t xb = kw == 0 ? wd[1][P].x : kw == 1 ? wd[1][P].y : kw == 2 ? wd[1][P].z : wd[1][P].w;
                const uint32_t a0 = ly.lo(xa), a1 = ly.lo(xb), a2 = ly.hi(xa), a3 = ly.hi(xb);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                  uint32_t b0, b1;
                  if constexpr (Sh::kBRegs) {
                    b0 = bf[ks][nt][0];
                    b1 = bf[ks][nt][1];
                  } else {
                    const uint32_t* row = reinterpret_cast<const uint32_t*>(BK + ((ks * NT + nt) * 8 + gq) * 32);
                    b0 = row[tig];
                    b1 = row[4 + tig];
                  }
                  mma_e4m3(acc[P][nt], a0, a1, a2, a3, b0, b1);
                }
              }
#pragma unroll
            for (int P = 1; P < NPM; ++P)
#pragma unroll
              for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[0][nt][e] += acc[P][nt][e];
            const float* kn = reinterpret_cast<const float*>(stg + Sh::kOffKNorm);
            const float* kr = reinterpret_cast<const float*>(stg + Sh::kOffKRn);
            const float* vn = reinterpret_cast<const float*>(stg + Sh::kOffVNorm);
            const float* vr = reinterpret_cast<const float*>(stg + Sh::kOffVRn);
            const int tb = (int)(sg.t0 + k) * kTile;
#pragma unroll
            for (int hh = 0; hh < GH; ++hh) mx[hh] = -INFINITY;
#pragma unroll
            for (int r = 0; r < 2; ++r) {
              const bool valid = tb + tok[r] < sg.L;
              vnc[r] = valid ? vn[tok[r]] : 0.f;
              vrc[r] = valid ? vr[tok[r]] : 0.f;
              const float knr = kn[tok[r]], krr = kr[tok[r]];
              const float lv = __log2f(fmaxf(fmaxf(vnc[r], vrc[r]), 0x1p-32f));
#pragma unroll
              for (int hh = 0; hh < GH; ++hh) {
                const float dm = combine3<NT>(acc[0], hh, r), dq = combine3<NT>(acc[NPM], hh, r);
                const float sc = fmaf(knr, fmaf(A0[hh], dm, B0[hh]), krr * fmaf(A1[hh], dq, B1[hh]));
                s2[hh][r] = (valid && tig + 4 * hh < a.G) ? sc : -INFINITY;
                mx[hh] = fmaxf(mx[hh], s2[hh][r] + lv);
              }
            }
#pragma unroll
            for (int hh = 0; hh < GH; ++hh) {
#pragma unroll
              for (int o = 4; o < 32; o <<= 1) mx[hh] = fmaxf(mx[hh], __shfl_xor_sync(0xffffffffu, mx[hh], o));
              exceed |= M[hh] == -INFINITY ? mx[hh] > -INFINITY : mx[hh] > M[hh] + kTau;
            }
          }
          // one barrier per tile: weights of tile k - 1 are complete, and the vote
          const bool bump = workers_any(exceed);
          if (threadIdx.x == 0) issue_upto(gi + max(k - 1, 0));
          if (bump) {
            if (gq == 0) {
#pragma unroll
              for (int hh = 0; hh < GH; ++hh) ms->red[w][tig + 4 * hh] = mx[hh];
            }
            workers_sync();
#pragma unroll
            for (int hh = 0; hh < GH; ++hh) {
              float tm = ms->red[0][tig + 4 * hh];
#pragma unroll
              for (int q = 1; q < kNW; ++q) tm = fmaxf(tm, ms->red[q][tig + 4 * hh]);
              float nm = M[hh];
              if (M[hh] == -INFINITY || tm > M[hh] + kTau) nm = tm;
              const float fac = nm == M[hh] ? 1.f : exp2f(M[hh] - nm);
              M[hh] = nm;
              lsum[hh] *= fac;
              if (w == 0 && gq == 0) ms->fac[k & 1][tig + 4 * hh] = fac;
            }
          }
          if (keys && threadIdx.x == 0) ms->rescale[k & 1] = bump;
          if (k > 0) {
            // ---- values of tile k - 1: 16 coordinates of every plane
            const int64_t gv = g - 1;
            const int s = (int)(gv % kStages), buf = (k - 1) & 1;
            const uint8_t* stg = smem + Sh::kOffRing + s * Sh::kStage;
            const uint32_t* vi = reinterpret_cast<const uint32_t*>(stg + Sh::kOffVIdx);
            const uint32_t* vsg = reinterpret_cast<const uint32_t*>(stg + Sh::kOffVSgn);
            const uint8_t* bv = smem + Sh::kOffBV + buf * Sh::kBVBuf;
            if (ms->rescale[buf]) {
              float fh[GH];
#pragma unroll
              for (int hh = 0; hh < GH; ++hh) fh[hh] = ms->fac[buf][tig + 4 * hh];
#pragma unroll
              for (int P = 0; P < NP; ++P)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                  for (int e = 0; e < 4; ++e) {
                    // columns (nt, e & 1): (0,0) (0,1) (1,0) head slot 0; (1,1) (2,0) (2,1) head slot 1
                    const int hs = (nt * 2 + (e & 1)) < 3 ? 0 : 1;
                    vacc[P][nt][e] *= fh[hs < GH ? hs : 0];
                  }
            }
#pragma unroll
            for (int kb = 0; kb < 4; ++kb) {
              uint2 bb[2][NT];
#pragma unroll
              for (int part = 0; part < 2; ++part)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
                  bb[part][nt] = *reinterpret_cast<const uint2*>(
                      bv + (((((part * 4 + kb) * NT + nt) * 8 + gq) * 4 + tig) * 2) * 4);
              uint2 ww[NP];
#pragma unroll
              for (int P = 0; P < W; ++P) ww[P] = *reinterpret_cast<const uint2*>(vi + (kb * W + P) * kD + crd);
              if constexpr (W == 3) {
                ww[3].x = ww[0].x ^ ww[1].x ^ ww[2].x;
                ww[3].y = ww[0].y ^ ww[1].y ^ ww[2].y;
              }
              ww[NPM] = *reinterpret_cast<const uint2*>(vsg + kb * kD + crd);
#pragma unroll
              for (int P = 0; P < NP; ++P) {
                const int part = P < NPM ? 0 : 1;
                const uint32_t a0 = sign_layer(ww[P].x, shl), a1 = sign_layer(ww[P].y, shl);
                const uint32_t a2 = sign_layer(ww[P].x, shh), a3 = sign_layer(ww[P].y, shh);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
                  mma_e4m3(vacc[P][nt], a0, a1, a2, a3, bb[part][nt].x, bb[part][nt].y);
              }
            }
          }
          if (keys) {
            // ---- attention weights of tile k -> value operand half-words
            uint8_t* bv = smem + Sh::kOffBV + (k & 1) * Sh::kBVBuf;
#pragma unroll
            for (int hh = 0; hh < GH; ++hh) {
              float p[2];
#pragma unroll
              for (int r = 0; r < 2; ++r) p[r] = s2[hh][r] == -INFINITY ? 0.f : exp2f(s2[hh][r] - M[hh]);
              lsum[hh] += p[0] + p[1];
              uint16_t pm[3], pq[3];
              pieces_pair(p[0] * vnc[0], p[1] * vnc[1], pm);
              pieces_pair(p[0] * vrc[0], p[1] * vrc[1], pq);
#pragma unroll
              for (int kk = 0; kk < 3; ++kk) {
                const int c = col_of(kk, tig + 4 * hh), nt = c >> 3, n8 = c & 7;
                const int wm = (((((0 * 4 + kbw) * NT + nt) * 8 + n8) * 4 + (gq & 3)) * 2 + (gq >> 2));
                const int wq = (((((1 * 4 + kbw) * NT + nt) * 8 + n8) * 4 + (gq & 3)) * 2 + (gq >> 2));
                *reinterpret_cast<uint16_t*>(bv + wm * 4 + 2 * hf) = pm[kk];
                *reinterpret_cast<uint16_t*>(bv + wq * 4 + 2 * hf) = pq[kk];
              }
            }
          }
        }
        gi += sg.n;
      }
      // ---- partial of this CTA for the unit
      const int sp = segc & 1;
#pragma unroll
      for (int hh = 0; hh < GH; ++hh) {
        float l = lsum[hh];
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
        if (gq == 0) ms->lred[sp][w][tig + 4 * hh] = l;
      }
      workers_sync();
      float cf[NPM];
#pragma unroll
      for (int P = 0; P < NPM; ++P) cf[P] = __ldg(a.walsh + (P < W ? (1 << P) : 7));
#pragma unroll
      for (int hh = 0; hh < GH; ++hh) {
        const int g = tig + 4 * hh;
        if (g < a.G) {
          float* pp = a.part + ((size_t)(head0 + g) * a.smax + sg.slot) * (2 + 2 * kD);
          float rot[2], sgn[2];
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            // the value operand is -s, so every sum enters negated
            float x = 0.f;
#pragma unroll
            for (int P = 0; P < NPM; ++P) x = fmaf(cf[P], combine3<NT>(vacc[P], hh, r), x);
            rot[r] = -x;
            sgn[r] = -combine3<NT>(vacc[NPM], hh, r);
          }
          *reinterpret_cast<float2*>(pp + 2 + crd) = make_float2(rot[0], rot[1]);
          *reinterpret_cast<float2*>(pp + 2 + kD + crd) = make_float2(sgn[0], sgn[1]);
          if (w == 0 && gq == 0) {
            float l = 0.f;
#pragma unroll
            for (int q = 0; q < kNW; ++q) l += ms->lred[sp][q][g];
            pp[0] = M[hh];
            pp[1] = l;
          }
        }
      }
    }
  }
  // no copy of this CTA may be in flight when it exits
  if (threadIdx.x == 0)
    for (int64_t g = max((int64_t)0, issued - kStages); g < issued; ++g)
      mbar_wait(smem_u32(&ms->ld_full[g % kStages]), (uint32_t)((g / kStages) & 1), a.fault, kFaultDecode);
  __syncthreads();
}

}  // namespace

namespace tq {

// Partial slots per unit for a grid of `ctas` CTAs over units * tpu tiles.
int decode_tc_slots(int64_t units, int64_t tpu, int64_t ctas) {
  const int64_t total = units * tpu;
  int64_t smax = 1;
  for (int64_t u = 0; u < units; ++u) {
    const int64_t s = owner((u + 1) * tpu - 1, total, ctas) - owner(u * tpu, total, ctas) + 1;
    smax = std::max(smax, s);
  }
  return (int)smax;
}

int decode_tc_ctas(int64_t units, int64_t tpu) { return (int)std::min<int64_t>(units * tpu, sm_count()); }

bool decode_tc_supported(const tq_plan* plan, int G, const tq_records* V, int64_t ctx_stride) {
  return plan->d == 128 && plan->m == 128 && G >= 1 && G <= 8 && V->layout == TQ_LAYOUT_BLOCK32 &&
         ctx_stride % kTile == 0;
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
  a.tpu = ctx_stride / kTile;
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

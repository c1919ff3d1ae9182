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
// Launches.  unit_table_kernel (one CTA per (batch, kv head) unit) computes
// Π q and S q for the unit's heads and writes the query operand table and the
// score constants, once per unit; every decode CTA that works on the unit
// fetches that table with one bulk copy.  Both kernels are programmatic
// dependent launches (each waits for its predecessor before reading what the
// predecessor wrote).
//
// Work split.  A persistent grid of one CTA per SM takes contiguous ranges of
// 256-token tiles over all (batch, kv head) units (the last tile of a unit
// may hold 128).  At the end of its part of a unit a CTA merges its two
// halves on chip into one partial, then counts itself in on the unit's
// arrival counter; the CTA that arrives last merges the unit's partials and
// applies the unrotation, so there is no combine launch.  Sixteen warps do the same
// work: warp w scores 16 tokens of each tile (half w & 1 of block w / 2) and
// accumulates values for 16 coordinates (rows w % 8) over half of the blocks
// (w / 8).  Warps 0-7 thus only touch tokens 0-127 of a tile and warps 8-15
// tokens 128-255, and the two halves run as independent pipelines: each has
// its own softmax reference, running sum and named barriers.  The
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
#include <cuda_bf16.h>
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
  const void* q;     // [B*Hq][128] queries, bf16 (q_bf16) or fp32
  int q_bf16;
  const float *pi, *pi_t, *s_rot, *s_rot_t;  // Π, Πᵀ, S̃ = S Πᵀ, S̃ᵀ (128 x 128, row-major)
  const float* walsh;
  float scale, alpha;
  float* part;       // [B*Hq][smax][2 + 2*128]
  int smax;
  int64_t tpu;       // tiles per unit = ceil(ctx_stride / 256)
  int64_t total;     // units * tpu
  uint8_t* tables;     // [B*Hkv] per-unit query tables (unit_table_kernel)
  unsigned* arrivals;  // [B*Hkv] CTAs of each unit done with their partials (zeroed by unit_table_kernel)
  float* out;        // [B*Hq][128]
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
  alignas(16) float consts[4][8];  // this unit's A0, B0, A1, B1 per head (bulk copy of its table's tail)
  uint64_t ld_full[kStages], ld_empty[kStages];  // empty: one arrival per half
  uint64_t tab_full;          // the unit's query table has landed
  int abort;
  float red[kNW][8];          // per-warp tile maxima (reference moves only)
  float lred[2][kNW][8];      // per segment parity, per warp: Σ p per head
  float Mh[2][8];             // per half: softmax reference per head at the end of a segment
  float cf[4];                // Walsh coefficients of the codebook planes
  int last;                   // this CTA is the last of its unit to hand in its partial
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

// Scratch of the per-unit query transform, half merge and unit merge: the
// query-weight table and the value-weight buffers, both dead between units (the
// ring may already hold copies of the next unit and is not touched).  Global
// loads on these one-off paths are issued in as few dependent rounds as the
// registers allow: a round trip to L2 costs over a microsecond here.
constexpr int kMaxCtas = 160;                          // grid limit: bounds the slots per unit
template <int GP>
struct Scratch {
  static constexpr int kPrep = 7 * GP * kD;                                // q, 4 partial sums, Πq, Sq
  static constexpr int kHalf = GP * 2 * kD;                                // one half's acc_rot | acc_sgn
  static constexpr int kMerge = GP * (2 + kMaxCtas + 2 * kD + 4 * kD + kD);  // see unit_merge
};

// Column c = threadIdx % 128 of rows 32·grp .. 32·grp + 31 (grp = threadIdx / 128)
// of a 128 x 128 row-major matrix: consecutive threads read whole rows.
__device__ __forceinline__ void load_cols(const float* __restrict__ A, float (&v)[32]) {
  const int grp = threadIdx.x >> 7, c = threadIdx.x & (kD - 1);
#pragma unroll
  for (int t = 0; t < 32; ++t) v[t] = __ldg(A + (32 * grp + t) * kD + c);
}

// red[grp][g][c] = Σ_t v[t] · x[g][32·grp + t]: this thread's share of
// (Aᵀ x_g)_c for GP vectors x_g of stride xs in shared memory.
template <int GP>
__device__ __forceinline__ void cols_times(const float (&v)[32], const float* x, int xs, float* red) {
  const int grp = threadIdx.x >> 7, c = threadIdx.x & (kD - 1);
  float acc[GP];
#pragma unroll
  for (int g = 0; g < GP; ++g) acc[g] = 0.f;
#pragma unroll
  for (int t = 0; t < 32; ++t)
#pragma unroll
    for (int g = 0; g < GP; ++g) acc[g] = fmaf(v[t], x[g * xs + 32 * grp + t], acc[g]);
#pragma unroll
  for (int g = 0; g < GP; ++g) red[(grp * GP + g) * kD + c] = acc[g];
}

__device__ __forceinline__ float sum4(const float* red, int e, int stride) {
  return (red[e] + red[stride + e]) + (red[2 * stride + e] + red[3 * stride + e]);
}

// Query transform of the unit's heads head0 .. head0 + G - 1 ("TurboQuant 与 AI
// 效率革命" §三: the estimator takes Π q and S q): on return qr[g][j] = (Π q_g)_j
// and sr[g][i] = (S̃ Π q_g)_i = (S q_g)_i, zero for g >= G.  All threads; one
// round of global loads (q and both matrices).
template <int GP>
__device__ __noinline__ void unit_query_prep(const TcArgs& a, int head0, float* scr, float** qr_out,
                                             float** sr_out) {
  float* qs = scr;
  float* red = qs + GP * kD;
  float* qr = red + 4 * GP * kD;
  float* sr = qr + GP * kD;
  constexpr int QP = GP * kD / kThreads;  // query elements per thread
  float qv[QP];
#pragma unroll
  for (int i = 0; i < QP; ++i) {
    const int e = threadIdx.x + kThreads * i;
    const size_t off = (size_t)head0 * kD + e;
    qv[i] = (e >> 7) >= a.G ? 0.f
            : a.q_bf16      ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(a.q)[off])
                            : reinterpret_cast<const float*>(a.q)[off];
  }
  float v1[32], v2[32];
  load_cols(a.pi_t, v1);     // (Π q)_j = Σ_c Πᵀ[c][j] q_c
  load_cols(a.s_rot_t, v2);  // (S̃ q̃)_i = Σ_j S̃ᵀ[j][i] q̃_j
  // The query and the workspace belong to the stream's earlier launches: wait
  // for them (programmatic dependent launch).  Only then may the decode kernel
  // start, since its first copies read the records those launches wrote.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  // bring Π and S̃ (row-major), which the unit's merge reads, into L2 meanwhile
  for (int e = threadIdx.x; e < 2 * kD * kD / 32; e += kThreads) {
    const float* line = e < kD * kD / 32 ? a.pi + 32 * e : a.s_rot + 32 * (e - kD * kD / 32);
    asm volatile("prefetch.global.L2 [%0];" ::"l"(line));
  }
#pragma unroll
  for (int i = 0; i < QP; ++i) qs[threadIdx.x + kThreads * i] = qv[i];
  cta_sync();
  cols_times<GP>(v1, qs, kD, red);
  cta_sync();
  for (int e = threadIdx.x; e < GP * kD; e += kThreads) qr[e] = sum4(red, e, GP * kD);
  cta_sync();
  cols_times<GP>(v2, qr, kD, red);
  cta_sync();
  for (int e = threadIdx.x; e < GP * kD; e += kThreads) sr[e] = sum4(red, e, GP * kD);
  cta_sync();
  *qr_out = qr;
  *sr_out = sr;
}

// Merge of the ns partials (one per CTA) of each head of the unit, log-sum-exp
// over their references, and the output o = Πᵀ(acc_rot + α S̃ᵀ acc_sgn) / l, by
// the last CTA of the unit to hand in its partial.  All threads; partials
// written by other CTAs are read past L1.  Two rounds of global loads when ns
// fits one chunk: (references, sums, partial values), then both matrices.
template <int GP>
__device__ __noinline__ void unit_merge(const TcArgs& a, int head0, int ns, float* scr) {
  constexpr int kStride = 2 + 2 * kD;
  float* ml = scr;                      // [GP][2] reference max, Σ w·l
  float* wgt = ml + 2 * GP;             // [GP][kMaxCtas] slot weights
  float* acc = wgt + GP * kMaxCtas;     // [GP][256] merged acc_rot | acc_sgn
  float* red = acc + GP * 2 * kD;       // [4][GP][128]
  float* y = red + 4 * GP * kD;         // [GP][128]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // outputs o = threadIdx.x + 512·r (head o / 256, element o % 256), U slots per chunk
  constexpr int R = GP * 2 * kD / kThreads, U = 48 / R;
  const float* pp[R];
  const float* wg[R];
  float v[R], x[R][U];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int o = threadIdx.x + kThreads * r, g = o >> 8, j = o & (2 * kD - 1);
    pp[r] = a.part + (size_t)(head0 + min(g, a.G - 1)) * a.smax * kStride + 2 + j;
    wg[r] = wgt + g * kMaxCtas;
    v[r] = 0.f;
#pragma unroll
    for (int t = 0; t < U; ++t) x[r][t] = t < ns ? __ldcg(pp[r] + (size_t)t * kStride) : 0.f;
  }
  constexpr int kPerLane = kMaxCtas / 32;
  if (warp < GP) {
    const float* pm = a.part + (size_t)(head0 + warp) * a.smax * kStride;
    float mk[kPerLane], lk[kPerLane];
#pragma unroll
    for (int t = 0; t < kPerLane; ++t) {
      const int k = lane + 32 * t;
      const bool in = warp < a.G && k < ns;
      mk[t] = in ? __ldcg(pm + (size_t)k * kStride) : -INFINITY;
      lk[t] = in ? __ldcg(pm + (size_t)k * kStride + 1) : 0.f;
    }
    float mx = -INFINITY, l = 0.f;
#pragma unroll
    for (int t = 0; t < kPerLane; ++t) mx = fmaxf(mx, mk[t]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
#pragma unroll
    for (int t = 0; t < kPerLane; ++t) {
      const float wk = mk[t] == -INFINITY ? 0.f : exp2f(mk[t] - mx);
      wgt[warp * kMaxCtas + lane + 32 * t] = wk;
      l = fmaf(wk, lk[t], l);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
    if (lane == 0) ml[2 * warp] = mx, ml[2 * warp + 1] = l;
  }
  cta_sync();
  // acc[g][j] = Σ_k w_k part_k[j]; a slot of weight 0 (no token, or past ns) adds
  // nothing, whatever it holds
  for (int k0 = 0; k0 < ns; k0 += U) {
    if (k0 > 0) {
#pragma unroll
      for (int r = 0; r < R; ++r)
#pragma unroll
        for (int t = 0; t < U; ++t) x[r][t] = k0 + t < ns ? __ldcg(pp[r] + (size_t)(k0 + t) * kStride) : 0.f;
    }
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int t = 0; t < U; ++t) {
        const float wk = k0 + t < ns ? wg[r][k0 + t] : 0.f;
        v[r] = wk != 0.f ? fmaf(wk, x[r][t], v[r]) : v[r];
      }
  }
#pragma unroll
  for (int r = 0; r < R; ++r) acc[threadIdx.x + kThreads * r] = v[r];
  float v1[32], v2[32];
  load_cols(a.s_rot, v1);  // (S̃ᵀ acc_sgn)_j = Σ_i S̃[i][j] acc_sgn_i
  load_cols(a.pi, v2);     // (Πᵀ y)_i = Σ_j Π[j][i] y_j
  cta_sync();
  cols_times<GP>(v1, acc + kD, 2 * kD, red);
  cta_sync();
  for (int e = threadIdx.x; e < GP * kD; e += kThreads)
    y[e] = fmaf(a.alpha, sum4(red, e, GP * kD), acc[(e >> 7) * 2 * kD + (e & (kD - 1))]);
  cta_sync();
  cols_times<GP>(v2, y, kD, red);
  cta_sync();
  for (int e = threadIdx.x; e < a.G * kD; e += kThreads) {
    const float l = ml[2 * (e >> 7) + 1];
    a.out[(size_t)head0 * kD + e] = sum4(red, e, GP * kD) * (l > 0.f ? 1.f / l : 0.f);
  }
  cta_sync();
}

// Per-unit query table, built once per (batch, kv head) unit by
// unit_table_kernel and bulk-copied by every decode CTA that works on the unit:
// the query operand of the score products (the shared-memory image: f16 hi + lo
// per head and K index, stored divided by a power of two E per part and head)
// followed by the constants A0, B0, A1, B1 of each head's affine map from the
// products to scores in log2 units.
template <int W, int GP>
struct Table {
  static constexpr int kConstBytes = 4 * 8 * 4;
  static constexpr int kBytes = Shape<W, GP>::kBKBytes + kConstBytes;
};
struct TableState {
  float amax[2][8];  // per part and head: largest |weight| (as non-negative float bits)
  float O[2][8];     // per part and head: score offset of the exponent-kind operands
  float cf[4];       // Walsh coefficients of the codebook planes
};
template <int W, int GP>
constexpr int table_smem_bytes() {
  return 1024 + Shape<W, GP>::kBKBytes + Scratch<GP>::kPrep * 4 + (int)sizeof(TableState);
}

// One CTA per unit: q̃ = Π q and s̃ = S q of its G heads, then the table.  The
// key operand bits are exact ±1 (sign kind) or 0.125 / 0.5 (exponent kind) per
// f16 lane, so a head's weight x enters as x·s (sign kind, s = -F) or as
// x·(F - mean)·2/δ (exponent kind), the mean folded into the offset O.  Also
// zeroes the unit's arrival counter for the decode kernel that follows.
template <int W, int GP>
__global__ void __launch_bounds__(kThreads) unit_table_kernel(const TcArgs a) {
  using Sh = Shape<W, GP>;
  constexpr int NPM = Sh::NPM, NP = Sh::NP, GH = Sh::GH;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* BK = smem;
  float* scr = reinterpret_cast<float*>(smem + Sh::kBKBytes);
  TableState* ts = reinterpret_cast<TableState*>(smem + Sh::kBKBytes + Scratch<GP>::kPrep * 4);
  const int u = blockIdx.x, lane = threadIdx.x & 31;
  const int b = u / a.Hkv, h = u - b * a.Hkv, head0 = b * a.Hq + h * a.G;
  if (threadIdx.x < NPM) ts->cf[threadIdx.x] = __ldg(a.walsh + (threadIdx.x < W ? (1 << threadIdx.x) : 7));
  if (threadIdx.x < 16) {
    ts->amax[threadIdx.x >> 3][threadIdx.x & 7] = 0.f;
    ts->O[threadIdx.x >> 3][threadIdx.x & 7] = 0.f;
  }
  for (int e = threadIdx.x; e < Sh::kBKBytes / 16; e += kThreads)
    reinterpret_cast<uint4*>(BK)[e] = make_uint4(0, 0, 0, 0);
  float *qr, *sr;
  unit_query_prep<GP>(a, head0, scr, &qr, &sr);  // its first barrier publishes the lines above
  // (past the grid dependency wait inside unit_query_prep: the workspace is ours)
  if (threadIdx.x == 0) a.arrivals[u] = 0u;
  // thread group grp = threadIdx / 128 takes heads grp and grp + 4; thread j its coordinate
  // j: word kw, bit x = 16e + L; L = 8·ks2 + 4·hi + q -> K index 8·hi + 2q + e
  constexpr int HG = GP / 4;  // heads per thread group
  const int grp = threadIdx.x >> 7, j = threadIdx.x & (kD - 1);
  const int kw = j >> 5, e16 = (j >> 4) & 1, L = j & 15, ks2 = L >> 3, hi = (L >> 2) & 1, q4 = L & 3;
  const int kk = 8 * hi + 2 * q4 + e16;
  // exponent-kind operand (hi = 0): s = (F - mean)·2/δ; sign kind: s = -F
  const float wsc = hi ? -1.f : 2.f / kExpDelta;
  float qv[HG], sv[HG], cf[NPM];
#pragma unroll
  for (int i = 0; i < HG; ++i) qv[i] = qr[(grp + 4 * i) * kD + j], sv[i] = sr[(grp + 4 * i) * kD + j];
#pragma unroll
  for (int P = 0; P < NPM; ++P) cf[P] = ts->cf[P];
#pragma unroll
  for (int i = 0; i < HG; ++i) {
    const int g = grp + 4 * i;
    float am = 0.f;
#pragma unroll
    for (int P = 0; P < NPM; ++P) am = fmaxf(am, fabsf(wsc * cf[P] * qv[i]));
    float aq = fabsf(wsc * sv[i]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
      aq = fmaxf(aq, __shfl_xor_sync(0xffffffffu, aq, o));
    }
    if (lane == 0) {
      atomicMax(reinterpret_cast<int*>(&ts->amax[0][g]), __float_as_int(am));
      atomicMax(reinterpret_cast<int*>(&ts->amax[1][g]), __float_as_int(aq));
    }
  }
  cta_sync();
  // E: the power of two taking a part's largest weight below 2^12 (weights are
  // stored divided by E, exactly)
  auto escale = [&](int p, int g, bool inverse) {
    const float am = ts->amax[p][g];
    int ex;
    frexpf(am, &ex);
    return am > 0.f ? ldexpf(1.f, inverse ? 12 - ex : ex - 12) : 1.f;
  };
  {
    __half* bk = reinterpret_cast<__half*>(BK);
#pragma unroll
    for (int i = 0; i < HG; ++i) {
      const int g = grp + 4 * i;
      const float inv0 = escale(0, g, true), inv1 = escale(1, g, true);
      float osum0 = 0.f, osum1 = 0.f;
#pragma unroll
      for (int P = 0; P < NP; ++P) {
        const int part = P < NPM ? 0 : 1;
        const int ks = (P * 4 + kw) * 2 + ks2;
        const float x = part == 0 ? wsc * cf[P < NPM ? P : 0] * qv[i] * inv0 : wsc * sv[i] * inv1;
        const __half xh = __float2half_rn(x), xl = __float2half_rn(x - __half2float(xh));
        // (k, n) sits in lane (n, k % 8 / 2), fragment k / 8, half k % 2
        const int base =
            ((((ks * GH + (g >> 2)) * 8 + 2 * (g & 3)) * 4 + ((kk & 7) >> 1)) * 2 + (kk >> 3)) * 2 + (kk & 1);
        bk[base] = xh;
        bk[base + 16] = xl;
        if (!hi) (part == 0 ? osum0 : osum1) += __half2float(xh) + __half2float(xl);
      }
      // offsets O[part][g] = mean · E · Σ (stored exponent-kind weights)
#pragma unroll
      for (int sh = 16; sh > 0; sh >>= 1) {
        osum0 += __shfl_xor_sync(0xffffffffu, osum0, sh);
        osum1 += __shfl_xor_sync(0xffffffffu, osum1, sh);
      }
      if (lane == 0) {
        atomicAdd(&ts->O[0][g], osum0 * escale(0, g, false) * kExpMean);
        atomicAdd(&ts->O[1][g], osum1 * escale(1, g, false) * kExpMean);
      }
    }
  }
  cta_sync();
  uint8_t* dst = a.tables + (size_t)u * Table<W, GP>::kBytes;
  for (int e = threadIdx.x; e < Sh::kBKBytes / 16; e += kThreads)
    reinterpret_cast<uint4*>(dst)[e] = reinterpret_cast<const uint4*>(BK)[e];
  if (threadIdx.x < 8) {
    const int g = threadIdx.x;
    const float c = a.scale * kLog2e;
    float* cs = reinterpret_cast<float*>(dst + Sh::kBKBytes);
    cs[g] = c * escale(0, g, false);
    cs[8 + g] = -c * ts->O[0][g];
    cs[16 + g] = c * a.alpha * escale(1, g, false);
    cs[24 + g] = -c * a.alpha * ts->O[1][g];
  }
}

template <int W, int GP>
__global__ void __launch_bounds__(kThreads, 1) decode_tc_kernel(const TcArgs a) {
  using Sh = Shape<W, GP>;
  constexpr int NPM = Sh::NPM, NP = Sh::NP, GH = Sh::GH;
  static_assert(Scratch<GP>::kPrep * 4 <= 2 * Sh::kBVBuf && Scratch<GP>::kHalf * 4 <= 2 * Sh::kBVBuf,
                "query transform or half-merge scratch exceeds the value-weight buffers");
  static_assert(Scratch<GP>::kMerge * 4 <= Sh::kOffMisc - Sh::kOffBK, "merge scratch exceeds the weight tables");
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
    mbar_init(smem_u32(&ms->tab_full), 1);
    ms->abort = 0;
    fence_mbar_init();
  }
  // (every tile rewrites the whole value-weight buffer it uses, zeros for absent
  // heads and tokens, so the buffers need no initial value)
  // The codebook coefficients stay in flight in a register until each segment
  // publishes them; the two matrices of the unit merge are brought into L2.
  const float cf_ld = threadIdx.x < NPM ? __ldg(a.walsh + (threadIdx.x < W ? (1 << threadIdx.x) : 7)) : 0.f;
  for (int e = threadIdx.x; e < 2 * kD * kD / 32; e += kThreads) {
    const float* line = e < kD * kD / 32 ? a.pi + 32 * e : a.s_rot + 32 * (e - kD * kD / 32);
    asm volatile("prefetch.global.L2 [%0];" ::"l"(line));
  }
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
  // the query tables and arrival counters come from unit_table_kernel, which may
  // still be running (programmatic dependent launch): wait for it to complete
  asm volatile("griddepcontrol.wait;" ::: "memory");

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
  uint32_t tab_phase = 0u;
  for (int64_t f = f0; f < f1; ++segc) {
    int64_t next;
    const Seg sg = segment_at(a, f, f1, &next);
    f = next;
    const int b = (int)(sg.u / a.Hkv), h = (int)(sg.u - (int64_t)b * a.Hkv);
    const int head0 = b * a.Hq + h * a.G;
    if (threadIdx.x < NPM) ms->cf[threadIdx.x] = cf_ld;  // read after the next CTA barrier
#pragma unroll
    for (int P = 0; P < NP; ++P)
#pragma unroll
      for (int ht = 0; ht < GH; ++ht)
#pragma unroll
        for (int e = 0; e < 4; ++e) vacc[P][ht][e] = 0.f;
#pragma unroll
    for (int hh = 0; hh < GH; ++hh) M[hh] = -INFINITY, lsum[hh] = 0.f, pend[hh] = 1.f;
    if (sg.n > 0) {
      // ---- this unit's query table (unit_table_kernel): one bulk copy once both
      // halves are done with the previous unit's table (the unit merge also
      // writes the region through the generic proxy)
      cta_sync();
      if (threadIdx.x == 0) {
        fence_proxy_async_smem();
        const uint32_t bar = smem_u32(&ms->tab_full);
        const uint8_t* src = a.tables + (size_t)sg.u * Table<W, GP>::kBytes;
        mbar_arrive_expect_tx(bar, Table<W, GP>::kBytes);
        bulk_load(smem_u32(BK), src, Sh::kBKBytes, bar);
        bulk_load(smem_u32(&ms->consts[0][0]), src + Sh::kBKBytes, Table<W, GP>::kConstBytes, bar);
      }
      wait(&ms->tab_full, tab_phase);
      tab_phase ^= 1u;
#pragma unroll
      for (int hh = 0; hh < GH; ++hh) {
        const int g = 4 * hh + tig;
        A0[hh] = ms->consts[0][g];
        B0[hh] = ms->consts[1][g];
        A1[hh] = ms->consts[2][g];
        B1[hh] = ms->consts[3][g];
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
    // ---- the partial of this CTA for the unit: the two halves, each over its
    // own tokens with its own reference, merged on chip (half 1 hands its share
    // to half 0 through the value-weight buffers)
    const int sp = segc & 1;
#pragma unroll
    for (int hh = 0; hh < GH; ++hh) {
      float l = lsum[hh];
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
      if (gq == 0) ms->lred[sp][w][4 * hh + tig] = l;
      if (vrow == 0 && gq == 0) ms->Mh[hf][4 * hh + tig] = M[hh];
    }
    cta_sync();
    {
      float cf[NPM];
#pragma unroll
      for (int P = 0; P < NPM; ++P) cf[P] = ms->cf[P];
      float* hs = reinterpret_cast<float*>(smem + Sh::kOffBV);  // [GP][acc_rot 128 | acc_sgn 128]
      float rot[GH][2], sgn[GH][2], Mx[GH], f0[GH], f1[GH];
#pragma unroll
      for (int hh = 0; hh < GH; ++hh) {
        const int head = 4 * hh + tig;
        const float M0 = ms->Mh[0][head], M1 = ms->Mh[1][head];
        Mx[hh] = fmaxf(M0, M1);
        f0[hh] = M0 == -INFINITY ? 0.f : exp2f(M0 - Mx[hh]);
        f1[hh] = M1 == -INFINITY ? 0.f : exp2f(M1 - Mx[hh]);
        // fragment e = 2·row + piece; the value operand is -s, so sums enter negated
        const float fs = -(hf ? f1[hh] : f0[hh]) * (1.f / kWS);
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          float x = 0.f;
#pragma unroll
          for (int P = 0; P < NPM; ++P) x = fmaf(cf[P], vacc[P][hh][2 * r] + vacc[P][hh][2 * r + 1], x);
          rot[hh][r] = x * fs;
          sgn[hh][r] = (vacc[NPM][hh][2 * r] + vacc[NPM][hh][2 * r + 1]) * fs;
        }
        if (hf == 1) {
          *reinterpret_cast<float2*>(hs + head * 2 * kD + crd) = make_float2(rot[hh][0], rot[hh][1]);
          *reinterpret_cast<float2*>(hs + head * 2 * kD + kD + crd) = make_float2(sgn[hh][0], sgn[hh][1]);
        }
      }
      cta_sync();
      if (hf == 0) {
#pragma unroll
        for (int hh = 0; hh < GH; ++hh) {
          const int head = 4 * hh + tig;
          if (head < a.G) {
            float* pp = a.part + ((size_t)(head0 + head) * a.smax + sg.slot) * (2 + 2 * kD);
            const float2 hr = *reinterpret_cast<const float2*>(hs + head * 2 * kD + crd);
            const float2 hq = *reinterpret_cast<const float2*>(hs + head * 2 * kD + kD + crd);
            *reinterpret_cast<float2*>(pp + 2 + crd) = make_float2(rot[hh][0] + hr.x, rot[hh][1] + hr.y);
            *reinterpret_cast<float2*>(pp + 2 + kD + crd) = make_float2(sgn[hh][0] + hq.x, sgn[hh][1] + hq.y);
            if (vrow == 0 && gq == 0) {
              float l0 = 0.f, l1 = 0.f;
#pragma unroll
              for (int q = 0; q < kNW / 2; ++q) l0 += ms->lred[sp][q][head], l1 += ms->lred[sp][8 + q][head];
              pp[0] = Mx[hh];
              pp[1] = fmaf(f0[hh], l0, f1[hh] * l1);
            }
          }
        }
      }
    }
    // ---- the last CTA of the unit to hand in its partial merges them all
    __threadfence();
    cta_sync();
    if (threadIdx.x == 0) {
      const int64_t nct = owner((sg.u + 1) * a.tpu - 1, a.total, C) - owner(sg.u * a.tpu, a.total, C) + 1;
      ms->last = atomicAdd(a.arrivals + sg.u, 1u) == (unsigned)(nct - 1);
      if (ms->last) __threadfence();
    }
    cta_sync();
    if (ms->last) {
      const int ns = (int)(owner((sg.u + 1) * a.tpu - 1, a.total, C) - owner(sg.u * a.tpu, a.total, C) + 1);
      unit_merge<GP>(a, head0, ns, reinterpret_cast<float*>(smem + Sh::kOffBK));
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

// Partial slots per unit for a grid of `ctas` CTAs over units * tpu tiles: one
// per CTA that touches the unit.
int decode_tc_slots(int64_t units, int64_t tpu, int64_t ctas) {
  const int64_t total = units * tpu;
  int64_t smax = 1;
  for (int64_t u = 0; u < units; ++u) {
    const int64_t s = owner((u + 1) * tpu - 1, total, ctas) - owner(u * tpu, total, ctas) + 1;
    smax = std::max(smax, s);
  }
  return (int)smax;  // one partial per CTA
}

int decode_tc_ctas(int64_t units, int64_t tpu) {
  return (int)std::min<int64_t>(units * tpu, std::min(sm_count(), kMaxCtas));
}

bool decode_tc_supported(const tq_plan* plan, int G, const tq_records* V, int64_t ctx_stride) {
  return plan->d == 128 && plan->m == 128 && G >= 1 && G <= 8 && V->layout == TQ_LAYOUT_BLOCK32 &&
         ctx_stride % kHalfTile == 0;
}

size_t decode_tc_table_bytes(int w, int G) {
  const bool g8 = G > 4;
  switch (w) {
    case 1: return g8 ? Table<1, 8>::kBytes : Table<1, 4>::kBytes;
    case 2: return g8 ? Table<2, 8>::kBytes : Table<2, 4>::kBytes;
    default: return g8 ? Table<3, 8>::kBytes : Table<3, 4>::kBytes;
  }
}

tq_status launch_decode_tc(const tq_plan* plan, const void* q, tq_dtype q_dtype, const tq_records* K,
                           const tq_records* V, const int32_t* ctx_len, int B, int Hq, int Hkv, int64_t ctx_stride,
                           float scale, float* part, int smax, uint8_t* tables, unsigned* arrivals, float* out,
                           cudaStream_t stream) {
  TcArgs a{};
  a.kidx = K->idx; a.ksgn = K->sgn; a.knorm = K->norm; a.krnorm = K->rnorm;
  a.vidx = V->idx; a.vsgn = V->sgn; a.vnorm = V->norm; a.vrnorm = V->rnorm;
  a.ctx_len = ctx_len;
  a.ctx_stride = ctx_stride;
  a.B = B; a.Hq = Hq; a.Hkv = Hkv; a.G = Hq / Hkv;
  a.q = q;
  a.q_bf16 = q_dtype == TQ_BF16;
  a.pi = plan->pi; a.pi_t = plan->pi_t; a.s_rot = plan->s_rot; a.s_rot_t = plan->s_rot_t;
  a.tables = tables;
  a.arrivals = arrivals;
  a.out = out;
  a.walsh = plan->walsh;
  a.scale = scale;
  a.alpha = plan->qjl_alpha;
  a.part = part;
  a.smax = smax;
  a.tpu = decode_tc_tpu(ctx_stride);
  a.total = (int64_t)B * Hkv * a.tpu;
  a.fault = fault_word();
  if (!a.fault) return TQ_ERR_CUDA;
  const int units = B * Hkv;
  const int grid = decode_tc_ctas(units, a.tpu);
  // the per-unit query tables (and zeroed arrival counters), then the decode
  auto go = [&](auto table_kern, int table_smem, auto kern, int smem) -> tq_status {
    if (cudaFuncSetAttribute(table_kern, cudaFuncAttributeMaxDynamicSharedMemorySize, table_smem) != cudaSuccess ||
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return TQ_ERR_CUDA;
    // both as programmatic dependent launches: the table kernel's matrix loads
    // overlap the previous kernel, the decode kernel's prologue and first copies
    // overlap the table kernel (each waits for its predecessor before it reads
    // what that one wrote)
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg{};
    cfg.blockDim = dim3(kThreads);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.gridDim = dim3(units);
    cfg.dynamicSmemBytes = table_smem;
    if (cudaLaunchKernelEx(&cfg, table_kern, a) != cudaSuccess) return TQ_ERR_CUDA;
    cfg.gridDim = dim3(grid);
    cfg.dynamicSmemBytes = smem;
    if (cudaLaunchKernelEx(&cfg, kern, a) != cudaSuccess) return TQ_ERR_CUDA;
    return launch_status();
  };
#define TQ_DECODE_TC_GO(W_, GP_) \
  go(unit_table_kernel<W_, GP_>, table_smem_bytes<W_, GP_>(), decode_tc_kernel<W_, GP_>, smem_bytes<W_>())
  const bool g8 = a.G > 4;
  switch (plan->w) {
    case 1: return g8 ? TQ_DECODE_TC_GO(1, 8) : TQ_DECODE_TC_GO(1, 4);
    case 2: return g8 ? TQ_DECODE_TC_GO(2, 8) : TQ_DECODE_TC_GO(2, 4);
    default: return g8 ? TQ_DECODE_TC_GO(3, 8) : TQ_DECODE_TC_GO(3, 4);
  }
#undef TQ_DECODE_TC_GO
}

}  // namespace tq

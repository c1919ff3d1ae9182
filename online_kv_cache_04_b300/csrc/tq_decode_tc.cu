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
// signs are one more ±1 plane.  An f16x2 operand register holds bits L and
// 16 + L of a plane word, one per half.
//   keys:   thread t of an mma quad uses bits L = 4t .. 4t + 3 of every word.
//           One multiply by 2^(12 − 4t) moves them to bits 12..15 (and
//           28..31), and one logic op per register keeps one of them: bit 12,
//           13 or 14 alone is the f16 value 2^-11, 2^-7 or 2 (an exponent bit
//           over a zero base: {0, x}, an affine image of s whose offset is
//           folded into a per-(batch, kv head) constant), bit 15 over 1.0 is
//           ±1 (exactly −s).  The query weight of each coordinate is scaled by
//           the inverse of its kind.
//   values: every register is of the ±1 kind (a multiply per register moves
//           its bit to 15), so the long sums over the context carry no offset.
//
//   scores: mma.sync m16n8k16 f16, rows = 16 tokens, K = 16 coordinates of
//           one plane, B = the query weights (shared memory, per unit).
//   values: the same instruction with rows = 16 coordinates and K = 16
//           tokens of one 32-row block word (TQ_LAYOUT_BLOCK32), B = the
//           attention weights p·‖v‖·coef_P and p·‖r_v‖ (registers); fp32
//           accumulators stay in registers over the whole context.  With the
//           codebook coefficient in the weight, every index plane adds into
//           one accumulator, the value of c[idx] itself.
// A query weight enters as two f16 columns, hi = f16(x) and lo = f16(x − hi)
// (22 significant bits): up to 4 heads x (hi, lo) fill an 8-column score
// tile, and 5 to 8 heads take a second tile over the same expanded bits.
// Value weights: with up to 4 heads the same (hi, lo) columns; with 5 to 8,
// one f16 column per head (the error of a rounded value weight averages out
// over the tokens, unlike that of a query weight).
// Why f16 warp MMAs: decode has one query per head, so every product here is
// at most 8 columns wide; a tcgen05.mma costs its issuing thread over a
// hundred cycles whatever its width, and an e4m3 or int8 mma.sync runs far
// below the f16 one.
//
// Launches.  unit_table_kernel (one CTA per (batch, kv head) unit) computes
// Π q and S q for the unit's heads and writes the query operand table and the
// score constants, once per unit (and, for tq_decode_attention_append, also
// quantizes the unit's new key and value into the caches); every decode CTA
// that works on the unit fetches that table with one bulk copy.
// unit_combine_kernel (one CTA per unit) then merges the unit's partials and
// unrotates.  All three are programmatic dependent launches (each waits for
// its predecessor before reading what the predecessor wrote).
//
// Work split.  A persistent grid of 4-warp CTAs, three per SM (two when a kv
// head serves more than four query heads), takes contiguous ranges of
// 128-token tiles over all (batch, kv head) units.  The kernel is bound by
// instruction issue, so the 12 warps a SM are what hides the latency of each
// warp's dependent chains.  Each warp owns one 32-token block of every tile
// and does everything for it: the scores of its 32 tokens (two 16-row tiles),
// its own online softmax, and the values of those tokens for all 128
// coordinates.  The attention weights go from the score fragments to the
// value operands by shuffles inside the warp, so warps never wait for one
// another within a unit; the only shared state is the ring of bulk-copied
// tiles (a stage is refilled once all four warps have arrived on its
// stage-empty mbarrier).  Within a warp the values of tile k − 1 and the
// scores of tile k form one straight block.  At the end of its part of a
// unit a CTA merges its warps on chip into one partial (reference, Σ p and
// the two value sums per head) for unit_combine_kernel.
//
// Softmax is online with a lazy reference per warp: the running reference M
// (of log2(p·max(‖v‖, ‖r_v‖)), clamped at 2^-32) moves only when a tile
// exceeds it by more than 2^6; the warp's accumulators are then rescaled.
// Every mbarrier wait is bounded; on timeout the kernel sets a fault bit
// (tq_fault_flags), skips the remaining waits and runs to its end.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>

#include "tq_internal.h"
#include "tq_sm100.cuh"

namespace {

using namespace tq::sm100;

constexpr int kNW = 4;                                 // decode warps (one 32-token block each)
constexpr int kBlocks = 4;                             // 32-row blocks per tile
constexpr int kTile = 32 * kBlocks;                    // tokens per tile
constexpr int kPage = 256;                             // tokens per page of a paged cache: two tiles
constexpr int kD = 128;
constexpr int kStages = 2;                             // power of two
constexpr int kThreads = 32 * kNW;                     // decode kernel
// decode CTAs resident per SM: 12 warps at up to 4 heads per kv head; with 8
// the value accumulators of both parts stay apart and take more registers
constexpr int ctas_per_sm(int GP) { return GP == 4 ? 3 : 2; }
constexpr int kCombThreads = 256;                      // unit merge kernel
constexpr int kTableThreads = 512;                     // query-table kernel
constexpr float kTau = 6.0f;                           // lazy-rescale threshold (log2 units)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kWS = 256.f;                           // attention weights carry 2^8 (up to 2^14 in f16)
constexpr int kBMaxExp = 15;                           // query operand entries stay below 2^15
constexpr unsigned kFaultDecode = 2u;
constexpr unsigned kFaultPage = 16u;                   // a page-table entry outside the record arrays
constexpr unsigned kFaultAppend = 8u;                  // fused append: a full cache or a negative length

// Key operand kinds after the move to bits 12..15: exponent bits over a zero
// base (values 2^-11, 2^-7, 2 when set, 0 when clear), and the sign of 1.0.
constexpr uint32_t kK12 = 0x10001000u, kK13 = 0x20002000u, kK14 = 0x40004000u;
constexpr uint32_t kSignMask = 0x80008000u, kSignBase = 0x3C003C00u;

// The sign kind's mask and base in registers (loaded from constant memory):
// with both in registers the operand is a single three-input logic op.
__constant__ uint32_t c_ops[2] = {kSignMask, kSignBase};
// per quad index t: the key multiplier 2^(12-4t) and the value multipliers
// 2^(15-4t-j), read from constant memory so that the moves stay integer
// multiplies (FMA pipe) rather than shifts on the busier integer pipe
__constant__ uint32_t c_kmul[4] = {4096u, 256u, 16u, 1u};
__constant__ uint32_t c_vmul[4][4] = {{32768u, 16384u, 8192u, 4096u},
                                      {2048u, 1024u, 512u, 256u},
                                      {128u, 64u, 32u, 16u},
                                      {8u, 4u, 2u, 1u}};
struct SignKind {
  uint32_t m, b;
  __device__ __forceinline__ SignKind() : m(c_ops[0]), b(c_ops[1]) {}
  __device__ __forceinline__ uint32_t operator()(uint32_t t) const {
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(t), "r"(m), "r"(b));  // (t & m) | b
    return r;
  }
};

__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
  asm(
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

// Barrier over all threads of a CTA of NT threads (named barrier 3).
template <int NT>
__device__ __forceinline__ void cta_sync_n() {
  asm volatile("bar.sync 3, %0;" ::"n"(NT) : "memory");
}

struct TcArgs {
  uint32_t *kidx, *ksgn, *vidx, *vsgn;  // written only by the fused append
  float *knorm, *krnorm, *vnorm, *vrnorm;
  const int32_t* ctx_len;
  int64_t ctx_stride;
  const int32_t* pages;  // paged caches: [B*Hkv][max_pages] page of each 256 tokens (NULL: contiguous rows)
  int64_t max_pages, npages;  // pages per unit; pages the record arrays hold
  int B, Hq, Hkv, G;
  const void* q;     // [B*Hq][128] queries, bf16 (q_bf16) or fp32
  int q_bf16;
  const float *pi, *pi_t, *s_rot, *s_rot_t;  // Π, Πᵀ, S̃ = S Πᵀ, S̃ᵀ (128 x 128, row-major)
  const float* walsh;
  // Fused append (append != 0): the step's new key and value of every unit
  // ([B*Hkv][128], bf16 or fp32) go to token ctx_len[b] of the caches, written
  // by unit_table_kernel before the decode reads them; the decode attends over
  // ctx_len[b] + 1 tokens and unit_combine_kernel advances ctx_len[b].  A row
  // with a full cache or a negative length is left alone (kFaultAppend).
  int append, new_bf16;
  const void *k_new, *v_new;
  int32_t* ctx_len_mut;      // the same array as ctx_len
  const float *centroids, *bounds;
  float scale, alpha;
  float* part;       // [B*Hq][smax][2 + 2*128]
  int smax;
  int64_t tpu;       // tiles per unit = ceil(ctx_stride / kTile)
  int64_t total;     // units * tpu
  uint8_t* tables;     // [B*Hkv] per-unit query tables (unit_table_kernel)
  float* out;        // [B*Hq][128]
  unsigned* fault;
};

// CTA that owns flat tile f when `total` tiles are cut into `ctas` even ranges.
__host__ __device__ inline int64_t owner(int64_t f, int64_t total, int64_t ctas) {
  return ((f + 1) * ctas - 1) / total;
}

// Token count of batch row b that this launch attends over: ctx_len[b] (0 if
// negative, at most ctx_stride), plus the appended token when there is one.
__device__ __forceinline__ int ctx_of(const TcArgs& a, int b) {
  const int L = __ldg(a.ctx_len + b);
  const bool app = a.append && L >= 0 && L < a.ctx_stride;
  return (int)min((int64_t)max(L, 0) + (app ? 1 : 0), a.ctx_stride);
}

// Score columns: head g sits in head tile g / 4, columns 2·(g % 4) (hi) and
// 2·(g % 4) + 1 (lo), so the thread with quad index q ends with both pieces
// of heads q and 4 + q.  Value columns: with GP = 4, column 2q + piece is
// head q; with GP = 8, column 2q is head q and 2q + 1 head 4 + q (hi only),
// so the thread with quad index q again holds heads q and 4 + q.
//
// Score rows: in 16-row tile s of a warp's block, row r (r < 8) is token 2Q
// and row r + 8 token 2Q + 1 of the block, Q = 4·(r / 2) + 2s + r % 2: the
// tokens of score tile s are exactly those of value K-step s (below), and
// each score thread holds one pair of consecutive tokens, the pair an f16x2
// value weight register carries.
//
// Key K-step ks = (P·4 + kw)·2 + sub of plane P, word kw: k-slot 2t + e is
// coordinate 32·kw + 4t + 2·sub + 16e, k-slot 8 + 2t + e is coordinate
// 32·kw + 4t + 2·sub + 1 + 16e (kinds: sub 0 -> bits 12 and 13, sub 1 ->
// bit 14 and the sign).  Value K-step sub of a block word: k-slot 2t + e is
// token 8t + 4·sub + e, k-slot 8 + 2t + e token 8t + 4·sub + 2 + e (word bits
// L = 4t + 2·sub (+1) and 16 + L).

template <int W, int GP, bool Q>
struct Shape {
  static constexpr int NPM = W == 3 ? 4 : W;   // ±1 planes of the codebook
  static constexpr int NP = NPM + (Q ? 1 : 0);  // plus the QJL sign plane (none for stage 1 alone)
  static constexpr int NKS = 8 * NP;           // score K-steps of 16 coordinates
  static constexpr int GH = GP / 4;            // score head tiles = heads per thread
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
  // per-warp shares of the CTA partial, one group of 4 heads at a time: [warp][32 values][lane]
  static constexpr int kRedBytes = kNW * 32 * 32 * 4;
  static constexpr int kOffRing = 0;
  static constexpr int kOffBK = kOffRing + kStages * kStage;
  static constexpr int kOffRed = kOffBK + kBKBytes;
  static constexpr int kOffMisc = kOffRed + kRedBytes;
};

struct Misc {
  alignas(16) float consts[4][8];  // this unit's A0, B0, A1, B1 per head (bulk copy of its table's tail)
  uint64_t ld_full[kStages], ld_empty[kStages];  // empty: one arrival per warp
  uint64_t tab_full;          // the unit's query table has landed
  int abort;
  float mw[kNW][8];           // per warp: softmax reference per head at the end of a segment
  float lw[kNW][8];           // per warp: Σ p per head
  float cf[4];                // Walsh coefficients of the codebook planes
};
constexpr int kMiscBytes = 2048;
static_assert(sizeof(Misc) <= kMiscBytes, "barriers and per-head state must fit their region");

template <int W, int GP, bool Q>
constexpr int smem_bytes() {
  return 1024 + Shape<W, GP, Q>::kOffMisc + kMiscBytes;
}
// ctas_per_sm(GP) CTAs, each with the 1 KiB the system reserves per CTA, in an SM's 228 KiB
static_assert(ctas_per_sm(4) * (smem_bytes<3, 4, true>() + 1024) <= 228 * 1024 &&
                  ctas_per_sm(8) * (smem_bytes<3, 8, true>() + 1024) <= 228 * 1024,
              "shared memory plan exceeds a CTA's share of an SM");

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
  s.L = ctx_of(a, b);
  const int64_t nvalid = (s.L + kTile - 1) / kTile;
  const int64_t tend = s.t0 + (fe - f);
  s.n = (int)max((int64_t)0, min(tend, nvalid) - s.t0);
  s.slot = (int)(blockIdx.x - owner(s.u * a.tpu, a.total, gridDim.x));
  return s;
}

// Scratch of the per-unit query transform and of the unit merge.  Global loads
// on these one-off paths are issued in as few dependent rounds as the
// registers allow: a round trip to L2 costs over a microsecond here.
constexpr int kMaxCtas = 448;                          // grid limit: bounds the slots per unit
template <int GP, int NT>
struct Scratch {
  static constexpr int NG = NT / 128;                                        // thread groups
  static constexpr int kPrep = (3 + NG) * GP * kD;                           // q, NG partial sums, Πq, Sq
  static constexpr int kAppend = 2 * kD + NG * 2 * kD + 16;                  // see append_step
  static constexpr int kMerge = GP * (2 + kMaxCtas + 2 * kD + NG * kD + kD);  // see unit_combine_kernel
};

// Column c = threadIdx % 128 of rows R·grp .. R·grp + R - 1 (grp = threadIdx / 128,
// R = 128 / (NT / 128)) of a 128 x 128 row-major matrix: consecutive threads
// read whole rows.
template <int NT>
__device__ __forceinline__ void load_cols(const float* __restrict__ A, float (&v)[128 * 128 / NT]) {
  constexpr int R = 128 * 128 / NT;
  const int grp = threadIdx.x >> 7, c = threadIdx.x & (kD - 1);
#pragma unroll
  for (int t = 0; t < R; ++t) v[t] = __ldg(A + (R * grp + t) * kD + c);
}

// red[grp][g][c] = Σ_t v[t] · x[g][R·grp + t]: this thread's share of
// (Aᵀ x_g)_c for GP vectors x_g of stride xs in shared memory.
template <int GP, int NT>
__device__ __forceinline__ void cols_times(const float (&v)[128 * 128 / NT], const float* x, int xs, float* red) {
  constexpr int R = 128 * 128 / NT;
  const int grp = threadIdx.x >> 7, c = threadIdx.x & (kD - 1);
  float acc[GP];
#pragma unroll
  for (int g = 0; g < GP; ++g) acc[g] = 0.f;
#pragma unroll
  for (int t = 0; t < R; ++t)
#pragma unroll
    for (int g = 0; g < GP; ++g) acc[g] = fmaf(v[t], x[g * xs + R * grp + t], acc[g]);
#pragma unroll
  for (int g = 0; g < GP; ++g) red[(grp * GP + g) * kD + c] = acc[g];
}

// Σ over the NG thread groups' partial sums of element e.
template <int NG>
__device__ __forceinline__ float sum_groups(const float* red, int e, int stride) {
  float s = red[e];
#pragma unroll
  for (int k = 1; k < NG; ++k) s += red[k * stride + e];
  return s;
}

// Fused append of unit u: its new key (into K, row layout) and new value (into
// V, 32-row blocks) quantized at token L = ctx_len[b] by the two stages of
// "谷歌TurboQuant如何绕过内存墙？" §2 -- n = ||x||, u = Π x / n, the bucket
// index against the Lloyd-Max bounds, ρ = u - c[idx], σ = sign(S Πᵀ ρ) with
// sign(0) = +1, ||r|| = n ||ρ||, the zero vector stored as u = 0, r = 0 --
// with the columns of Πᵀ (v1) and S̃ᵀ (v2) this thread already holds.  All NT
// threads; thread t < 256 finishes coordinate t % 128 of vector t / 128, so a
// warp ballot forms one packed row word.  `scr`: Scratch::kAppend floats.
template <int W, int NT, bool Q>
__device__ __forceinline__ void append_step(const TcArgs& a, int u, const float (&v1)[128 * 128 / NT],
                                            const float (&v2)[128 * 128 / NT], float* scr) {
  constexpr int NG = NT / 128;
  const int b = u / a.Hkv;
  const int L = __ldg(a.ctx_len + b);
  if (L < 0 || L >= a.ctx_stride) {  // uniform over the CTA
    if (threadIdx.x == 0) atomicOr(a.fault, kFaultAppend);
    return;
  }
  int64_t row = (int64_t)u * a.ctx_stride + L;
  if (a.pages != nullptr) {  // the page holding token L
    const int64_t pg = __ldg(a.pages + (int64_t)u * a.max_pages + L / kPage);
    if (pg < 0 || pg >= a.npages) {
      if (threadIdx.x == 0) atomicOr(a.fault, kFaultPage);
      return;
    }
    row = pg * kPage + L % kPage;
  }
  float* xs = scr;                 // [2][128] the new vectors, then ρ
  float* red = xs + 2 * kD;        // [NG][2][128] partial sums
  float* wsum = red + NG * 2 * kD; // [2 vectors][4 warps] partial ||x||², then ||ρ||²
  const int t = threadIdx.x, vec = t >> 7, j = t & (kD - 1), lane = t & 31, wv = (t >> 5) & 3;
  const bool mine = t < 2 * kD;
  float x = 0.f;
  if (mine) {
    const size_t off = (size_t)u * kD + j;
    const void* src = vec ? a.v_new : a.k_new;
    x = a.new_bf16 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(src)[off])
                   : reinterpret_cast<const float*>(src)[off];
    xs[t] = x;
    float s2 = x * x;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s2 += __shfl_xor_sync(0xffffffffu, s2, o);
    if (lane == 0) wsum[vec * 4 + wv] = s2;
  }
  cta_sync_n<NT>();
  cols_times<2, NT>(v1, xs, kD, red);  // (Π x)_j
  cta_sync_n<NT>();
  float n = 0.f, rho = 0.f;
  int idx = 0;
  if (mine) {
    n = sqrtf((wsum[vec * 4] + wsum[vec * 4 + 1]) + (wsum[vec * 4 + 2] + wsum[vec * 4 + 3]));
    const float uj = n > 0.f ? sum_groups<NG>(red, t, 2 * kD) / n : 0.f;
#pragma unroll
    for (int k = 0; k < (1 << W) - 1; ++k) idx += __ldg(a.bounds + k) < uj ? 1 : 0;
    rho = n > 0.f ? uj - __ldg(a.centroids + idx) : 0.f;
  }
  cta_sync_n<NT>();  // everyone is through with xs and wsum
  if (mine) {
    xs[t] = rho;
    float r2 = rho * rho;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) r2 += __shfl_xor_sync(0xffffffffu, r2, o);
    if (lane == 0) wsum[vec * 4 + wv] = r2;
    const uint32_t bbit = 1u << tq::block32_bit((int)(row & 31));
#pragma unroll
    for (int p = 0; p < W; ++p) {
      const bool bit = (idx >> p) & 1;
      const uint32_t word = __ballot_sync(0xffffffffu, bit);
      if (vec == 0) {
        if (lane == 0) a.kidx[row * (4 * W) + p * 4 + (j >> 5)] = word;
      } else {
        uint32_t* wp = a.vidx + (row >> 5) * (W * kD) + p * kD + j;
        *wp = bit ? (*wp | bbit) : (*wp & ~bbit);
      }
    }
    if (j == 0) (vec ? a.vnorm : a.knorm)[row] = n;
  }
  if constexpr (Q) {
    cta_sync_n<NT>();
    cols_times<2, NT>(v2, xs, kD, red);  // (S̃ ρ)_i
    cta_sync_n<NT>();
    if (mine) {
      const bool pos = sum_groups<NG>(red, t, 2 * kD) >= 0.f;
      const uint32_t bbit = 1u << tq::block32_bit((int)(row & 31));
      const uint32_t word = __ballot_sync(0xffffffffu, pos);
      if (vec == 0) {
        if (lane == 0) a.ksgn[row * 4 + (j >> 5)] = word;
      } else {
        uint32_t* wp = a.vsgn + (row >> 5) * kD + j;
        *wp = pos ? (*wp | bbit) : (*wp & ~bbit);
      }
      if (j == 0) {
        const float r2 = (wsum[vec * 4] + wsum[vec * 4 + 1]) + (wsum[vec * 4 + 2] + wsum[vec * 4 + 3]);
        (vec ? a.vrnorm : a.krnorm)[row] = n * sqrtf(r2);
      }
    }
  }
  cta_sync_n<NT>();
}

// Query transform of the unit's heads head0 .. head0 + G - 1 ("TurboQuant 与 AI
// 效率革命" §三: the estimator takes Π q and S q): on return qr[g][j] = (Π q_g)_j
// and sr[g][i] = (S̃ Π q_g)_i = (S q_g)_i, zero for g >= G.  All NT threads; one
// round of global loads (q and both matrices).
template <int W, int GP, int NT, bool Q>
__device__ __noinline__ void unit_query_prep(const TcArgs& a, int u, int head0, float* scr, float** qr_out,
                                             float** sr_out) {
  constexpr int NG = NT / 128, R = 128 * 128 / NT;
  float* qs = scr;
  float* red = qs + GP * kD;
  float* qr = red + NG * GP * kD;
  float* sr = qr + GP * kD;
  constexpr int QP = GP * kD / NT;  // query elements per thread
  float qv[QP];
#pragma unroll
  for (int i = 0; i < QP; ++i) {
    const int e = threadIdx.x + NT * i;
    const size_t off = (size_t)head0 * kD + e;
    qv[i] = (e >> 7) >= a.G ? 0.f
            : a.q_bf16      ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(a.q)[off])
                            : reinterpret_cast<const float*>(a.q)[off];
  }
  float v1[R], v2[R];
  load_cols<NT>(a.pi_t, v1);                  // (Π q)_j = Σ_c Πᵀ[c][j] q_c
  if constexpr (Q) load_cols<NT>(a.s_rot_t, v2);  // (S̃ q̃)_i = Σ_j S̃ᵀ[j][i] q̃_j
  // The query and the workspace belong to the stream's earlier launches: wait
  // for them (programmatic dependent launch).  Only then may the decode kernel
  // start, since its first copies read the records those launches wrote.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  // bring Π and S̃ (row-major), which the unit's merge reads, into L2 meanwhile
  for (int e = threadIdx.x; e < (Q ? 2 : 1) * kD * kD / 32; e += NT) {
    const float* line = e < kD * kD / 32 ? a.pi + 32 * e : a.s_rot + 32 * (e - kD * kD / 32);
    asm volatile("prefetch.global.L2 [%0];" ::"l"(line));
  }
#pragma unroll
  for (int i = 0; i < QP; ++i) qs[threadIdx.x + NT * i] = qv[i];
  cta_sync_n<NT>();
  cols_times<GP, NT>(v1, qs, kD, red);
  cta_sync_n<NT>();
  for (int e = threadIdx.x; e < GP * kD; e += NT) qr[e] = sum_groups<NG>(red, e, GP * kD);
  cta_sync_n<NT>();
  if constexpr (Q) {
    cols_times<GP, NT>(v2, qr, kD, red);
    cta_sync_n<NT>();
    for (int e = threadIdx.x; e < GP * kD; e += NT) sr[e] = sum_groups<NG>(red, e, GP * kD);
  } else {
    for (int e = threadIdx.x; e < GP * kD; e += NT) sr[e] = 0.f;
  }
  cta_sync_n<NT>();
  // the fused append reuses the matrix columns this thread holds
  if (a.append) append_step<W, NT, Q>(a, u, v1, v2, sr + GP * kD);
  *qr_out = qr;
  *sr_out = sr;
}

// Merge of the ns partials (one per decode CTA) of each head of a unit,
// log-sum-exp over their references, and the output o = Πᵀ(acc_rot + α S̃ᵀ
// acc_sgn) / l: one CTA per unit (HEAD = false), or, when the heads are few
// enough for one wave, one CTA per query head (HEAD = true, GP = 1: a
// quarter of the partial loads and products per CTA, all slots in one round);
// a programmatic dependent launch after the decode kernel.  The matrix columns (the plan's, not written by the decode)
// are loaded before the wait for the decode grid, so they overlap its tail;
// after the wait the partials come in one round of global loads when ns fits
// one chunk.
template <int GP, bool Q, bool HEAD>
__global__ void __launch_bounds__(kCombThreads, 1) unit_combine_kernel(const TcArgs a, int ctas) {
  static_assert(!HEAD || GP == 1, "one head per CTA");
  constexpr int NT = kCombThreads;
  constexpr int NG = NT / 128, RR = 128 * 128 / NT;
  constexpr int kStride = 2 + 2 * kD;
  extern __shared__ uint8_t smem_raw[];
  float* scr = reinterpret_cast<float*>((reinterpret_cast<uintptr_t>(smem_raw) + 15) & ~uintptr_t(15));
  // this CTA's heads head0 .. head0 + G - 1, of unit u = (b, h)
  int b, h, head0, G;
  if (HEAD) {
    head0 = blockIdx.x;
    b = head0 / a.Hq;
    h = (head0 - b * a.Hq) / a.G;
    G = 1;
  } else {
    b = (int)(blockIdx.x / a.Hkv);
    h = (int)(blockIdx.x - b * a.Hkv);
    head0 = b * a.Hq + h * a.G;
    G = a.G;
  }
  const int64_t u = (int64_t)b * a.Hkv + h;
  // the decode CTAs that own tiles of the unit: one partial slot each
  const int ns = (int)(owner((u + 1) * a.tpu - 1, a.total, ctas) - owner(u * a.tpu, a.total, ctas) + 1);
  float v1[RR], v2[RR];
  if constexpr (Q) load_cols<NT>(a.s_rot, v1);  // (S̃ᵀ acc_sgn)_j = Σ_i S̃[i][j] acc_sgn_i
  load_cols<NT>(a.pi, v2);                     // (Πᵀ y)_i = Σ_j Π[j][i] y_j
  // the partials are the decode kernel's: wait for it to complete
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  // fused append: every read of ctx_len[b] is done; the row's first CTA advances it
  if (a.append && threadIdx.x == 0 && (HEAD ? head0 == b * a.Hq : h == 0)) {
    const int L = a.ctx_len_mut[b];
    if (L >= 0 && L < a.ctx_stride) a.ctx_len_mut[b] = L + 1;
  }
  float* ml = scr;                      // [GP][2] reference max, Σ w·l
  float* wgt = ml + 2 * GP;             // [GP][kMaxCtas] slot weights
  float* acc = wgt + GP * kMaxCtas;     // [GP][256] merged acc_rot | acc_sgn
  float* red = acc + GP * 2 * kD;       // [NG][GP][128]
  float* y = red + NG * GP * kD;        // [GP][128]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // outputs o = threadIdx.x + NT·r (head o / 256, element o % 256), U slots per chunk
  constexpr int R = GP * 2 * kD / NT, U = 48 / R;
  const float* pp[R];
  const float* wg[R];
  float v[R], x[R][U];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int o = threadIdx.x + NT * r, g = o >> 8, j = o & (2 * kD - 1);
    pp[r] = a.part + (size_t)(head0 + min(g, G - 1)) * a.smax * kStride + 2 + j;
    wg[r] = wgt + g * kMaxCtas;
    v[r] = 0.f;
#pragma unroll
    for (int t = 0; t < U; ++t) x[r][t] = t < ns ? __ldcg(pp[r] + (size_t)t * kStride) : 0.f;
  }
  static_assert(GP <= NT / 32, "one warp per head weighs the slots");
  constexpr int kPerLane = kMaxCtas / 32;
  if (warp < GP) {
    const float* pm = a.part + (size_t)(head0 + warp) * a.smax * kStride;
    float mk[kPerLane], lk[kPerLane];
#pragma unroll
    for (int t = 0; t < kPerLane; ++t) {
      const int k = lane + 32 * t;
      const bool in = warp < G && k < ns;
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
  cta_sync_n<NT>();
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
  for (int r = 0; r < R; ++r) acc[threadIdx.x + NT * r] = v[r];
  cta_sync_n<NT>();
  if constexpr (Q) {
    cols_times<GP, NT>(v1, acc + kD, 2 * kD, red);
    cta_sync_n<NT>();
  }
  for (int e = threadIdx.x; e < GP * kD; e += NT)
    y[e] = Q ? fmaf(a.alpha, sum_groups<NG>(red, e, GP * kD), acc[(e >> 7) * 2 * kD + (e & (kD - 1))])
             : acc[(e >> 7) * 2 * kD + (e & (kD - 1))];
  cta_sync_n<NT>();
  cols_times<GP, NT>(v2, y, kD, red);
  cta_sync_n<NT>();
  for (int e = threadIdx.x; e < G * kD; e += NT) {
    const float l = ml[2 * (e >> 7) + 1];
    a.out[(size_t)head0 * kD + e] = sum_groups<NG>(red, e, GP * kD) * (l > 0.f ? 1.f / l : 0.f);
  }
}

// Per-unit query table, built once per (batch, kv head) unit by
// unit_table_kernel and bulk-copied by every decode CTA that works on the unit:
// the query operand of the score products (the shared-memory image: f16 hi + lo
// per head and K index, stored divided by a power of two E per part and head)
// followed by the constants A0, B0, A1, B1 of each head's affine map from the
// products to scores in log2 units.
template <int W, int GP, bool Q>
struct Table {
  static constexpr int kConstBytes = 4 * 8 * 4;
  static constexpr int kBytes = Shape<W, GP, Q>::kBKBytes + kConstBytes;
};
struct TableState {
  float amax[2][8];     // per part and head: largest |entry| (as non-negative float bits)
  float osum[16][2][2]; // per warp, part, head of the warp's thread group: Σ of the {0, x} kinds' offsets
  float cf[4];          // Walsh coefficients of the codebook planes
};
template <int W, int GP, bool Q>
constexpr int table_smem_bytes() {
  return 1024 + Shape<W, GP, Q>::kBKBytes + (Scratch<GP, kTableThreads>::kPrep + Scratch<GP, kTableThreads>::kAppend) * 4 +
         (int)sizeof(TableState);
}

// One CTA per unit: q̃ = Π q and s̃ = S q of its G heads, then the table.  A key
// operand bit is a {0, x} value (coordinates at word bits 4t, 4t+1, 4t+2 and
// 16 more: x = 2^-11, 2^-7, 2) or ±1 (word bits 4t+3, 4t+19: exactly −s).  A
// head's weight w enters as 2w/x (then the product is w·(1 + s), and the
// offset Σ w over those coordinates goes into the score constant) or as −w.
// Every sum has a fixed order, so the table is the same on every call.
template <int W, int GP, bool Q>
__global__ void __launch_bounds__(kTableThreads) unit_table_kernel(const TcArgs a) {
  using Sh = Shape<W, GP, Q>;
  constexpr int NT = kTableThreads;
  constexpr int NPM = Sh::NPM, NP = Sh::NP, GH = Sh::GH;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* BK = smem;
  float* scr = reinterpret_cast<float*>(smem + Sh::kBKBytes);
  TableState* ts = reinterpret_cast<TableState*>(smem + Sh::kBKBytes +
                                                 (Scratch<GP, NT>::kPrep + Scratch<GP, NT>::kAppend) * 4);
  const int u = blockIdx.x, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int b = u / a.Hkv, h = u - b * a.Hkv, head0 = b * a.Hq + h * a.G;
  if (threadIdx.x < NPM) ts->cf[threadIdx.x] = __ldg(a.walsh + (threadIdx.x < W ? (1 << threadIdx.x) : 7));
  if (threadIdx.x < 16) ts->amax[threadIdx.x >> 3][threadIdx.x & 7] = 0.f;
  for (int e = threadIdx.x; e < Sh::kBKBytes / 16; e += NT) reinterpret_cast<uint4*>(BK)[e] = make_uint4(0, 0, 0, 0);
  float *qr, *sr;
  unit_query_prep<W, GP, NT, Q>(a, u, head0, scr, &qr, &sr);  // its first barrier publishes the lines above
  // (past the grid dependency wait inside unit_query_prep: the workspace is ours)
  // thread group grp = threadIdx / 128 takes heads grp and grp + 4; thread j its coordinate j:
  // word kw, half e16, bit L = 4·tq + jj of the half -> K-step (P·4 + kw)·2 + jj / 2,
  // k-slot 8·(jj % 2) + 2·tq + e16
  constexpr int HG = GP / 4;  // heads per thread group
  const int grp = threadIdx.x >> 7, j = threadIdx.x & (kD - 1);
  const int kw = j >> 5, e16 = (j >> 4) & 1, L = j & 15, tq = L >> 2, jj = L & 3;
  const int sub = jj >> 1, a2 = jj & 1;
  const int kk = 8 * a2 + 2 * tq + e16;
  // kind of this coordinate's operand: weight scale 2/x for {0, x}, -1 for ±1 (= -s)
  const float wsc = jj == 0 ? 4096.f : jj == 1 ? 256.f : jj == 2 ? 1.f : -1.f;
  const float xhalf = jj == 0 ? 0x1p-12f : jj == 1 ? 0x1p-8f : jj == 2 ? 1.f : 0.f;  // x / 2
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
    float aq = Q ? fabsf(wsc * sv[i]) : 0.f;
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
  cta_sync_n<NT>();
  // E: the power of two taking a part's largest entry below 2^15 (entries are
  // stored divided by E, exactly)
  auto escale = [&](int p, int g, bool inverse) {
    const float am = ts->amax[p][g];
    int ex;
    frexpf(am, &ex);
    return am > 0.f ? ldexpf(1.f, inverse ? kBMaxExp - ex : ex - kBMaxExp) : 1.f;
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
        const int ks = (P * 4 + kw) * 2 + sub;
        const float x = part == 0 ? wsc * cf[P < NPM ? P : 0] * qv[i] * inv0 : wsc * sv[i] * inv1;
        const __half xh = __float2half_rn(x), xl = __float2half_rn(x - __half2float(xh));
        // (k, n) sits in lane (n, k % 8 / 2), fragment k / 8, half k % 2
        const int base =
            ((((ks * GH + (g >> 2)) * 8 + 2 * (g & 3)) * 4 + ((kk & 7) >> 1)) * 2 + (kk >> 3)) * 2 + (kk & 1);
        bk[base] = xh;
        bk[base + 16] = xl;
        (part == 0 ? osum0 : osum1) += xhalf * (__half2float(xh) + __half2float(xl));
      }
      // per-warp offset sums, added in a fixed order below
#pragma unroll
      for (int sh = 16; sh > 0; sh >>= 1) {
        osum0 += __shfl_xor_sync(0xffffffffu, osum0, sh);
        osum1 += __shfl_xor_sync(0xffffffffu, osum1, sh);
      }
      if (lane == 0) ts->osum[warp][0][i] = osum0, ts->osum[warp][1][i] = osum1;
    }
  }
  cta_sync_n<NT>();
  uint8_t* dst = a.tables + (size_t)u * Table<W, GP, Q>::kBytes;
  for (int e = threadIdx.x; e < Sh::kBKBytes / 16; e += NT)
    reinterpret_cast<uint4*>(dst)[e] = reinterpret_cast<const uint4*>(BK)[e];
  if (threadIdx.x < 8) {
    const int g = threadIdx.x, gg = g & 3, i = g >> 2;  // head g: thread group gg, slot i
    float o0 = 0.f, o1 = 0.f;
    if (i < HG) {
#pragma unroll
      for (int q = 0; q < 4; ++q) o0 += ts->osum[4 * gg + q][0][i], o1 += ts->osum[4 * gg + q][1][i];
    }
    const float c = a.scale * kLog2e;
    float* cs = reinterpret_cast<float*>(dst + Sh::kBKBytes);
    cs[g] = c * escale(0, g, false);
    cs[8 + g] = -c * escale(0, g, false) * o0;
    cs[16 + g] = c * a.alpha * escale(1, g, false);
    cs[24 + g] = -c * a.alpha * escale(1, g, false) * o1;
  }
}

template <int W, int GP, bool Q>
__global__ void __launch_bounds__(kThreads, ctas_per_sm(GP)) decode_tc_kernel(const TcArgs a) {
  using Sh = Shape<W, GP, Q>;
  constexpr int NPM = Sh::NPM, NP = Sh::NP, GH = Sh::GH;
  constexpr int NT = kThreads;
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
      mbar_init(smem_u32(&ms->ld_empty[s]), kNW);
    }
    mbar_init(smem_u32(&ms->tab_full), 1);
    ms->abort = 0;
    fence_mbar_init();
  }
  if (threadIdx.x < NPM) ms->cf[threadIdx.x] = __ldg(a.walsh + (threadIdx.x < W ? (1 << threadIdx.x) : 7));
  // the two matrices of the unit merge are brought into L2
  for (int e = threadIdx.x; e < 2 * kD * kD / 32; e += NT) {
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
  // consumed by warp 0 and issued < done + kStages.  The cursor (cur, cu, ct,
  // cL) walks flat tiles: unit cu, tile ct in it, context length cL of the unit.
  int64_t issued = 0, cur = f0, cu = f0 / a.tpu, ct = f0 - cu * a.tpu;
  int cL = ctx_of(a, (int)(cu / a.Hkv));
  auto issue_upto = [&](int64_t done) {
    const uint32_t sbase = smem_u32(smem);
    while (issued < done + kStages && cur < f1 && !*abort_flag) {
      if (ct >= a.tpu || ct * kTile >= cL) {  // next unit (the rest of this one is past its context)
        cur += a.tpu - ct;
        ++cu;
        ct = 0;
        if (cur < f1) cL = ctx_of(a, (int)(cu / a.Hkv));
        continue;
      }
      int64_t row0 = cu * a.ctx_stride + ct * kTile;
      if (a.pages != nullptr) {  // paged cache: the tile is one half of a page
        int64_t pg = __ldg(a.pages + cu * a.max_pages + ct / (kPage / kTile));
        if (pg < 0 || pg >= a.npages) {
          atomicOr(a.fault, kFaultPage);
          pg = 0;
        }
        row0 = pg * kPage + (ct % (kPage / kTile)) * kTile;
      }
      const int ntok = kTile;
      ++cur;
      ++ct;
      const int s = (int)(issued & (kStages - 1));
      // other warps may still be reading the stage's previous tile
      if (issued >= kStages)
        wait(&ms->ld_empty[s], (uint32_t)(((issued - kStages) / kStages) & 1));
      ++issued;
      const uint32_t bar = smem_u32(&ms->ld_full[s]);
      const uint32_t dst = sbase + Sh::kOffRing + s * Sh::kStage;
      const int idxb = ntok * 16 * W, sgnb = ntok * 16, nrmb = ntok * 4;
      mbar_arrive_expect_tx(bar, Q ? 2 * idxb + 2 * sgnb + 4 * nrmb : 2 * idxb + 2 * nrmb);
      bulk_load(dst + Sh::kOffKIdx, a.kidx + row0 * (4 * W), idxb, bar);
      bulk_load(dst + Sh::kOffKNorm, a.knorm + row0, nrmb, bar);
      bulk_load(dst + Sh::kOffVIdx, a.vidx + (row0 >> 5) * (W * kD), idxb, bar);
      bulk_load(dst + Sh::kOffVNorm, a.vnorm + row0, nrmb, bar);
      if constexpr (Q) {  // stage 1 alone stores no signs and no residual norms
        bulk_load(dst + Sh::kOffKSgn, a.ksgn + row0 * 4, sgnb, bar);
        bulk_load(dst + Sh::kOffKRn, a.krnorm + row0, nrmb, bar);
        bulk_load(dst + Sh::kOffVSgn, a.vsgn + (row0 >> 5) * kD, sgnb, bar);
        bulk_load(dst + Sh::kOffVRn, a.vrnorm + row0, nrmb, bar);
      }
    }
  };
  // the first copies overlap unit_table_kernel, unless it appends to the caches
  if (threadIdx.x == 0 && !a.append) issue_upto(0);
  // the query tables come from unit_table_kernel, which may still be running
  // (programmatic dependent launch): wait for it to complete
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (threadIdx.x == 0 && a.append) issue_upto(0);
  // unit_combine_kernel may be scheduled now: its CTAs take an SM as decode CTAs
  // leave, load their matrices and wait for this grid to complete
  asm volatile("griddepcontrol.launch_dependents;");

  // key words: one multiply moves bits 4·tig .. 4·tig + 3 (and 16 more) to 12..15
  const uint32_t kmul = c_kmul[tig];
  // value words: bit 4·tig + jv (and 16 more) to bit 15 (and 31)
  const uint32_t vm0 = c_vmul[tig][0], vm1 = c_vmul[tig][1], vm2 = c_vmul[tig][2], vm3 = c_vmul[tig][3];
  const SignKind sk;
  const uint8_t* BK = smem + Sh::kOffBK;
  float cf[NPM];
#pragma unroll
  for (int P = 0; P < NPM; ++P) cf[P] = ms->cf[P];
  // this thread's score rows in the warp's block: pair Qs of score tile s = tokens 2Qs, 2Qs + 1
  const int pr0 = 4 * (gq >> 1) + (gq & 1);  // Q of tile 0; tile 1 adds 2
  // [part][row tile][fragment]: c[idx] sums (part 0), σ sums (part 1).  With at
  // most 4 heads (GP = 4) both parts share one accumulator: value column 2·tig
  // holds head tig's c[idx] sums and column 2·tig + 1 its σ sums (the B
  // fragment of a plane is zero in the other part's columns); with GP = 8 the
  // columns are heads tig and tig + 4, one accumulator per part.
  constexpr int NPART = GP == 4 ? 1 : 2;
  float vacc[NPART][8][4];
  float M[GH], lsum[GH], A0[GH], B0[GH], A1[GH], B1[GH];
  uint32_t bv[NP][2][2];  // value B fragments of the previous tile: [plane][K-step][b0, b1]
  int64_t gi = 0;
  int segc = 0;
  uint32_t tab_phase = 0u;
  for (int64_t f = f0; f < f1; ++segc) {
    int64_t next;
    const Seg sg = segment_at(a, f, f1, &next);
    f = next;
    const int b = (int)(sg.u / a.Hkv), h = (int)(sg.u - (int64_t)b * a.Hkv);
    const int head0 = b * a.Hq + h * a.G;
#pragma unroll
    for (int p = 0; p < NPART; ++p)
#pragma unroll
      for (int rt = 0; rt < 8; ++rt)
#pragma unroll
        for (int e = 0; e < 4; ++e) vacc[p][rt][e] = 0.f;
#pragma unroll
    for (int hh = 0; hh < GH; ++hh) M[hh] = -INFINITY, lsum[hh] = 0.f;
    if (sg.n > 0) {
      // ---- this unit's query table (unit_table_kernel): one bulk copy once every
      // warp is done with the previous unit's table (the merges also write the
      // region through the generic proxy)
      fence_proxy_async_smem();
      cta_sync_n<NT>();
      if (threadIdx.x == 0) {
        const uint32_t bar = smem_u32(&ms->tab_full);
        const uint8_t* src = a.tables + (size_t)sg.u * Table<W, GP, Q>::kBytes;
        mbar_arrive_expect_tx(bar, Table<W, GP, Q>::kBytes);
        bulk_load(smem_u32(BK), src, Sh::kBKBytes, bar);
        bulk_load(smem_u32(&ms->consts[0][0]), src + Sh::kBKBytes, Table<W, GP, Q>::kConstBytes, bar);
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

      // scores of CTA tile gc (tile kc of the segment): s2[tile][head tile][row]
      // in log2 units (-inf outside the context), the cleaned value norms of
      // the thread's tokens, and the warp's tile maximum of s2 + log2(norm)
      float s2[2][GH][2], vnc[2][2], vrc[2][2], mx[GH];
      auto scores_step = [&](int kc, int64_t gc) {
        const uint8_t* stg = smem + Sh::kOffRing + (int)(gc & (kStages - 1)) * Sh::kStage;
        const uint4* kq = reinterpret_cast<const uint4*>(stg + Sh::kOffKIdx);  // token t, plane P: kq[t·W + P]
        const uint4* sq = reinterpret_cast<const uint4*>(stg + Sh::kOffKSgn);  // token t: sq[t]
        // [score tile][part][head tile][fragment]: one chain per K-substep at
        // GP = 8 and at w = 3; otherwise (12 warps a SM hide the chain's latency,
        // and the registers are short) one chain, acc2 staying zero
        constexpr bool kTwoChains = GP == 8 || W == 3;
        float acc[2][2][GH][4], acc2[2][2][GH][4];
#pragma unroll
        for (int st = 0; st < 2; ++st)
#pragma unroll
          for (int pt = 0; pt < 2; ++pt)
#pragma unroll
            for (int ht = 0; ht < GH; ++ht)
#pragma unroll
              for (int e = 0; e < 4; ++e) acc[st][pt][ht][e] = acc2[st][pt][ht][e] = 0.f;
#pragma unroll
        for (int P = 0; P < NP; ++P) {
          const int part = P < NPM ? 0 : 1;
          uint4 wd[2][2];  // [score tile][row]
#pragma unroll
          for (int st = 0; st < 2; ++st)
#pragma unroll
            for (int r = 0; r < 2; ++r) {
              const int t = 32 * warp + 2 * (pr0 + 2 * st) + r;
              if (P < W) {
                wd[st][r] = kq[t * W + P];
              } else if (P < NPM) {  // product plane b0 ^ b1 ^ b2
                const uint4 x0 = kq[t * W], x1 = kq[t * W + 1 % W], x2 = kq[t * W + 2 % W];
                wd[st][r] =
                    make_uint4(x0.x ^ x1.x ^ x2.x, x0.y ^ x1.y ^ x2.y, x0.z ^ x1.z ^ x2.z, x0.w ^ x1.w ^ x2.w);
              } else {
                wd[st][r] = sq[t];
              }
            }
#pragma unroll
          for (int kw = 0; kw < 4; ++kw) {
            const int ks = (P * 4 + kw) * 2;
            uint32_t u[2][2];
#pragma unroll
            for (int st = 0; st < 2; ++st)
#pragma unroll
              for (int r = 0; r < 2; ++r) u[st][r] = word_of(wd[st][r], kw) * kmul;
#pragma unroll
            for (int ht = 0; ht < GH; ++ht) {
              const uint2 b0 = bfrag(ks, ht), b1 = bfrag(ks + 1, ht);
#pragma unroll
              for (int st = 0; st < 2; ++st) {
                const uint32_t u0 = u[st][0], u1 = u[st][1];
                mma_f16(acc[st][part][ht], u0 & kK12, u1 & kK12, u0 & kK13, u1 & kK13, b0.x, b0.y);
                if constexpr (kTwoChains)
                  mma_f16(acc2[st][part][ht], u0 & kK14, u1 & kK14, sk(u0), sk(u1), b1.x, b1.y);
                else
                  mma_f16(acc[st][part][ht], u0 & kK14, u1 & kK14, sk(u0), sk(u1), b1.x, b1.y);
              }
            }
          }
        }
        const float* kn = reinterpret_cast<const float*>(stg + Sh::kOffKNorm);
        const float* kr = reinterpret_cast<const float*>(stg + Sh::kOffKRn);
        const float* vn = reinterpret_cast<const float*>(stg + Sh::kOffVNorm);
        const float* vr = reinterpret_cast<const float*>(stg + Sh::kOffVRn);
        const int64_t tb = (sg.t0 + kc) * kTile;
#pragma unroll
        for (int hh = 0; hh < GH; ++hh) mx[hh] = -INFINITY;
#pragma unroll
        for (int st = 0; st < 2; ++st) {
          const int t = 32 * warp + 2 * (pr0 + 2 * st);
          const float2 kn2 = *reinterpret_cast<const float2*>(kn + t), vn2 = *reinterpret_cast<const float2*>(vn + t);
          const float2 kr2 = Q ? *reinterpret_cast<const float2*>(kr + t) : make_float2(0.f, 0.f);
          const float2 vr2 = Q ? *reinterpret_cast<const float2*>(vr + t) : make_float2(0.f, 0.f);
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            const bool valid = tb + t + r < sg.L;
            vnc[st][r] = valid ? (r ? vn2.y : vn2.x) : 0.f;
            vrc[st][r] = valid ? (r ? vr2.y : vr2.x) : 0.f;
            const float knr = r ? kn2.y : kn2.x, krr = r ? kr2.y : kr2.x;
            const float lv = __log2f(fmaxf(fmaxf(vnc[st][r], vrc[st][r]), 0x1p-32f));
#pragma unroll
            for (int hh = 0; hh < GH; ++hh) {
              const float dm = (acc[st][0][hh][2 * r] + acc[st][0][hh][2 * r + 1]) +
                               (acc2[st][0][hh][2 * r] + acc2[st][0][hh][2 * r + 1]);
              const float dq = (acc[st][1][hh][2 * r] + acc[st][1][hh][2 * r + 1]) +
                               (acc2[st][1][hh][2 * r] + acc2[st][1][hh][2 * r + 1]);
              const float sc = Q ? fmaf(knr, fmaf(A0[hh], dm, B0[hh]), krr * fmaf(A1[hh], dq, B1[hh]))
                                 : knr * fmaf(A0[hh], dm, B0[hh]);
              s2[st][hh][r] = (valid && 4 * hh + tig < a.G) ? sc : -INFINITY;
              mx[hh] = fmaxf(mx[hh], s2[st][hh][r] + lv);
            }
          }
        }
#pragma unroll
        for (int hh = 0; hh < GH; ++hh)
#pragma unroll
          for (int o = 4; o < 32; o <<= 1) mx[hh] = fmaxf(mx[hh], __shfl_xor_sync(0xffffffffu, mx[hh], o));
      };

      // softmax step of the tile just scored (the warp's lazy reference may move:
      // the accumulators, which hold the earlier tiles, are rescaled), then its
      // attention weights -> the value B fragments bv
      auto weights_step = [&]() {
        bool exceed = false;
#pragma unroll
        for (int hh = 0; hh < GH; ++hh) exceed |= M[hh] == -INFINITY ? mx[hh] > -INFINITY : mx[hh] > M[hh] + kTau;
        if (__any_sync(0xffffffffu, exceed)) {
          float fac[GH];
#pragma unroll
          for (int hh = 0; hh < GH; ++hh) {
            float nm = M[hh];
            if (M[hh] == -INFINITY || mx[hh] > M[hh] + kTau) nm = mx[hh];
            fac[hh] = nm == M[hh] ? 1.f : exp2f(M[hh] - nm);
            M[hh] = nm;
            lsum[hh] *= fac[hh];
          }
          // value column 2·tig + c holds head tig (GP = 4, both columns) or head
          // tig + 4c (GP = 8)
#pragma unroll
          for (int p = 0; p < NPART; ++p)
#pragma unroll
            for (int rt = 0; rt < 8; ++rt)
#pragma unroll
              for (int e = 0; e < 4; ++e) vacc[p][rt][e] *= fac[GH == 1 ? 0 : (e & 1)];
        }
        // this thread's weights, one f16x2 register per (score tile, head tile, plane,
        // piece): the pair of tokens 2Q, 2Q + 1, times -coef_P (index planes) or -1
        // (sign plane) since the value operand is -s
        uint32_t hv[2][GH][NP];  // f16 alone: a value weight's rounding averages out over tokens
#pragma unroll
        for (int st = 0; st < 2; ++st)
#pragma unroll
          for (int hh = 0; hh < GH; ++hh) {
            float p[2];
#pragma unroll
            for (int r = 0; r < 2; ++r) p[r] = s2[st][hh][r] == -INFINITY ? 0.f : exp2f(s2[st][hh][r] - M[hh]);
            lsum[hh] += p[0] + p[1];
#pragma unroll
            for (int P = 0; P < NP; ++P) {
              const float c = P < NPM ? -cf[P] * kWS : -kWS;
              const float x0 = p[0] * (P < NPM ? vnc[st][0] : vrc[st][0]) * c;
              const float x1 = p[1] * (P < NPM ? vnc[st][1] : vrc[st][1]) * c;
              hv[st][hh][P] = f16x2_of(x0, x1);
            }
          }
        // B fragment of K-step st for lane (gq, tig): b0 = pair 4·tig + 2·st, b1 =
        // pair 4·tig + 2·st + 1, column gq: from the score thread (2·tig + b, gq / 2)
        // of score tile st; with GP = 4 column gq takes plane P's weights when its
        // part (gq % 2: c[idx] or σ) is P's and zero otherwise, with GP = 8 head
        // tile gq % 2
#pragma unroll
        for (int st = 0; st < 2; ++st)
#pragma unroll
          for (int bb = 0; bb < 2; ++bb) {
            const int src = 4 * (2 * tig + bb) + (gq >> 1);
#pragma unroll
            for (int P = 0; P < NP; ++P) {
              if (GP == 4) {
                const uint32_t x0 = __shfl_sync(0xffffffffu, hv[st][0][P], src);
                bv[P][st][bb] = (gq & 1) == (P < NPM ? 0 : 1) ? x0 : 0u;
              } else {
                const uint32_t x0 = __shfl_sync(0xffffffffu, hv[st][0][P], src);
                const uint32_t x1 = __shfl_sync(0xffffffffu, hv[st][GH - 1][P], src);
                bv[P][st][bb] = (gq & 1) ? x1 : x0;
              }
            }
          }
      };

      // values of CTA tile gv: the warp's block, 8 row tiles of 16 coordinates,
      // every plane, two K-steps of 16 tokens
      auto values_step = [&](int64_t gv) {
        const uint8_t* stg = smem + Sh::kOffRing + (int)(gv & (kStages - 1)) * Sh::kStage;
        const uint32_t* vi = reinterpret_cast<const uint32_t*>(stg + Sh::kOffVIdx) + warp * W * kD;
        const uint32_t* vsg = reinterpret_cast<const uint32_t*>(stg + Sh::kOffVSgn) + warp * kD;
#pragma unroll
        for (int rt = 0; rt < 8; ++rt) {
          const int crd = 16 * rt + 2 * gq;  // rows gq, gq + 8 <-> coordinates crd, crd + 1
#pragma unroll
          for (int P = 0; P < NP; ++P) {
            uint2 ww;
            if (P < W) {
              ww = *reinterpret_cast<const uint2*>(vi + P * kD + crd);
            } else if (P < NPM) {  // product plane
              const uint2 x0 = *reinterpret_cast<const uint2*>(vi + crd);
              const uint2 x1 = *reinterpret_cast<const uint2*>(vi + (1 % W) * kD + crd);
              const uint2 x2 = *reinterpret_cast<const uint2*>(vi + (2 % W) * kD + crd);
              ww = make_uint2(x0.x ^ x1.x ^ x2.x, x0.y ^ x1.y ^ x2.y);
            } else {
              ww = *reinterpret_cast<const uint2*>(vsg + crd);
            }
            const int part = GP == 4 || P < NPM ? 0 : 1;
            mma_f16(vacc[part][rt], sk(ww.x * vm0), sk(ww.y * vm0), sk(ww.x * vm1), sk(ww.y * vm1), bv[P][0][0],
                    bv[P][0][1]);
            mma_f16(vacc[part][rt], sk(ww.x * vm2), sk(ww.y * vm2), sk(ww.x * vm3), sk(ww.y * vm3), bv[P][1][0],
                    bv[P][1][1]);
          }
        }
      };

      // this warp is through CTA tile g: hand its stage back; thread 0 refills
      auto release = [&](int64_t g, int64_t done) {
        fence_proxy_async_smem();  // these generic reads before the refilling bulk copy
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&ms->ld_empty[g & (kStages - 1)]));
        if (threadIdx.x == 0) issue_upto(done);
      };

      if constexpr (W < 3 && GP == 4) {
        // each tile whole: scores, weights, values, then its stage goes back, so
        // the refill of a two-stage ring has a whole tile's work to land
        for (int k = 0; k < sg.n; ++k) {
          const int64_t g = gi + k;
          wait(&ms->ld_full[g & (kStages - 1)], (uint32_t)((g / kStages) & 1));
          scores_step(k, g);
          weights_step();
          values_step(g);
          release(g, g + 1);
        }
      } else {
        // w = 3 or 8 heads (more registers): the values of tile k - 1 and the
        // scores of tile k form one block, which spills less; tile k - 1's stage
        // goes back as soon as its values are done
        wait(&ms->ld_full[gi & (kStages - 1)], (uint32_t)((gi / kStages) & 1));
        scores_step(0, gi);
        weights_step();
        for (int k = 1; k < sg.n; ++k) {
          const int64_t g = gi + k;
          wait(&ms->ld_full[g & (kStages - 1)], (uint32_t)((g / kStages) & 1));
          values_step(g - 1);
          release(g - 1, g);
          scores_step(k, g);
          weights_step();
        }
        values_step(gi + sg.n - 1);
        release(gi + sg.n - 1, gi + sg.n);
      }
      gi += sg.n;
    }
    // ---- the partial of this CTA for the unit: its warps, each over its
    // own tokens with its own reference, merged on chip
#pragma unroll
    for (int hh = 0; hh < GH; ++hh) {
      float l = lsum[hh];
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
      if (gq == 0) ms->mw[warp][4 * hh + tig] = M[hh], ms->lw[warp][4 * hh + tig] = l;
    }
    cta_sync_n<NT>();
    float* red = reinterpret_cast<float*>(smem + Sh::kOffRed);  // [warp][value 32][lane]
    float* pbase = a.part + ((size_t)head0 * a.smax + sg.slot) * (2 + 2 * kD);
    const size_t hstride = (size_t)a.smax * (2 + 2 * kD);
    if (threadIdx.x < GP) {
      const int g = threadIdx.x;
      float mc = -INFINITY, l = 0.f;
#pragma unroll
      for (int w = 0; w < kNW; ++w) mc = fmaxf(mc, ms->mw[w][g]);
#pragma unroll
      for (int w = 0; w < kNW; ++w) l += ms->mw[w][g] == -INFINITY ? 0.f : exp2f(ms->mw[w][g] - mc) * ms->lw[w][g];
      if (g < a.G) pbase[g * hstride] = mc, pbase[g * hstride + 1] = l;
    }
#pragma unroll
    for (int hp = 0; hp < GH; ++hp) {  // heads tig + 4·hp
      const int g = tig + 4 * hp;
      float mc = -INFINITY;
#pragma unroll
      for (int w = 0; w < kNW; ++w) mc = fmaxf(mc, ms->mw[w][g]);
      const float mine = ms->mw[warp][g];
      const float fs = (mine == -INFINITY ? 0.f : exp2f(mine - mc)) * (1.f / kWS);
      // value v = part·16 + rt·2 + rp: coordinate 16·rt + 2·gq + rp
#pragma unroll
      for (int p = 0; p < 2; ++p)
#pragma unroll
        for (int rt = 0; rt < 8; ++rt)
#pragma unroll
          for (int rp = 0; rp < 2; ++rp) {
            const float x = GP == 4 ? vacc[0][rt][2 * rp + p] : vacc[p][rt][2 * rp + hp];
            red[(warp * 32 + p * 16 + rt * 2 + rp) * 32 + lane] = x * fs;
          }
      cta_sync_n<NT>();
      {
        // thread (value group vg = warp, lane): values VPW·vg .. VPW·vg + VPW - 1 of
        // lane, summed over warps
        constexpr int VPW = 32 / kNW;
        const int ln = lane, lg = ln >> 2, lt = ln & 3, gh = lt + 4 * hp;
#pragma unroll
        for (int i = 0; i < VPW; ++i) {
          const int v = VPW * warp + i, p = v >> 4, rt = (v >> 1) & 7, rp = v & 1;
          float s = 0.f;
#pragma unroll
          for (int w = 0; w < kNW; ++w) s += red[(w * 32 + v) * 32 + ln];
          if (gh < a.G) pbase[gh * hstride + 2 + p * kD + 16 * rt + 2 * lg + rp] = s;
        }
      }
      cta_sync_n<NT>();
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

int decode_tc_ctas(int64_t units, int64_t tpu, int G) {
  return (int)std::min<int64_t>(units * tpu, std::min(ctas_per_sm(G > 4 ? 8 : 4) * sm_count(), kMaxCtas));
}

bool decode_tc_supported(const tq_plan* plan, int G, const tq_records* V, int64_t ctx_stride) {
  return plan->d == 128 && (plan->m == 128 || plan->m == 0) && G >= 1 && G <= 8 && V->layout == TQ_LAYOUT_BLOCK32 &&
         ctx_stride % kTile == 0;
}

size_t decode_tc_table_bytes(int w, int G, int m) {
  const bool g8 = G > 4, q = m > 0;
  switch (w) {
    case 1: return q ? (g8 ? Table<1, 8, true>::kBytes : Table<1, 4, true>::kBytes)
                     : (g8 ? Table<1, 8, false>::kBytes : Table<1, 4, false>::kBytes);
    case 2: return q ? (g8 ? Table<2, 8, true>::kBytes : Table<2, 4, true>::kBytes)
                     : (g8 ? Table<2, 8, false>::kBytes : Table<2, 4, false>::kBytes);
    default: return q ? (g8 ? Table<3, 8, true>::kBytes : Table<3, 4, true>::kBytes)
                      : (g8 ? Table<3, 8, false>::kBytes : Table<3, 4, false>::kBytes);
  }
}

tq_status launch_decode_tc(const tq_plan* plan, const void* q, tq_dtype q_dtype, const tq_records* K,
                           const tq_records* V, const int32_t* ctx_len, int B, int Hq, int Hkv, int64_t ctx_stride,
                           float scale, float* part, int smax, uint8_t* tables, float* out, cudaStream_t stream,
                           const int32_t* pages, const TcAppend* app) {
  TcArgs a{};
  if (app != nullptr) {
    a.append = 1;
    a.k_new = app->k_new;
    a.v_new = app->v_new;
    a.new_bf16 = app->bf16;
    a.ctx_len_mut = app->ctx_len;
    a.centroids = plan->centroids;
    a.bounds = plan->bounds;
  }
  a.pages = pages;
  a.max_pages = ctx_stride / kPage;
  a.npages = std::min(K->capacity, V->capacity) / kPage;
  a.kidx = K->idx; a.ksgn = K->sgn; a.knorm = K->norm; a.krnorm = K->rnorm;
  a.vidx = V->idx; a.vsgn = V->sgn; a.vnorm = V->norm; a.vrnorm = V->rnorm;
  a.ctx_len = ctx_len;
  a.ctx_stride = ctx_stride;
  a.B = B; a.Hq = Hq; a.Hkv = Hkv; a.G = Hq / Hkv;
  a.q = q;
  a.q_bf16 = q_dtype == TQ_BF16;
  a.pi = plan->pi; a.pi_t = plan->pi_t; a.s_rot = plan->s_rot; a.s_rot_t = plan->s_rot_t;
  a.tables = tables;
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
  const int grid = decode_tc_ctas(units, a.tpu, a.G);
  // the per-unit query tables, the decode, then the per-unit merge
  // the merge: one CTA per query head when those fit one wave, else one per unit
  const bool per_head = (int64_t)B * Hq <= sm_count();
  auto go = [&](auto table_kern, int table_smem, auto kern, int smem, auto comb_unit, int comb_unit_smem,
                auto comb_head, int comb_head_smem) -> tq_status {
    void (*comb_kern)(const TcArgs, int) = per_head ? comb_head : comb_unit;
    const int comb_smem = per_head ? comb_head_smem : comb_unit_smem;
    if (cudaFuncSetAttribute(table_kern, cudaFuncAttributeMaxDynamicSharedMemorySize, table_smem) != cudaSuccess ||
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess ||
        cudaFuncSetAttribute(comb_kern, cudaFuncAttributeMaxDynamicSharedMemorySize, comb_smem) != cudaSuccess)
      return TQ_ERR_CUDA;
    // all three as programmatic dependent launches: the table kernel's matrix
    // loads overlap the previous kernel, the decode kernel's prologue and first
    // copies overlap the table kernel, the merge's matrix loads overlap the
    // decode's tail (each waits for its predecessor before it reads what that
    // one wrote)
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg{};
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.blockDim = dim3(kTableThreads);
    cfg.gridDim = dim3(units);
    cfg.dynamicSmemBytes = table_smem;
    if (cudaLaunchKernelEx(&cfg, table_kern, a) != cudaSuccess) return TQ_ERR_CUDA;
    cfg.blockDim = dim3(kThreads);
    cfg.gridDim = dim3(grid);
    cfg.dynamicSmemBytes = smem;
    if (cudaLaunchKernelEx(&cfg, kern, a) != cudaSuccess) return TQ_ERR_CUDA;
    cfg.blockDim = dim3(kCombThreads);
    cfg.gridDim = dim3(per_head ? B * Hq : units);
    cfg.dynamicSmemBytes = comb_smem;
    if (cudaLaunchKernelEx(&cfg, comb_kern, a, grid) != cudaSuccess) return TQ_ERR_CUDA;
    return launch_status();
  };
#define TQ_DECODE_TC_GO(W_, GP_, Q_)                                                                \
  go(unit_table_kernel<W_, GP_, Q_>, table_smem_bytes<W_, GP_, Q_>(), decode_tc_kernel<W_, GP_, Q_>, \
     smem_bytes<W_, GP_, Q_>(), unit_combine_kernel<GP_, Q_, false>, 16 + Scratch<GP_, kCombThreads>::kMerge * 4, \
     unit_combine_kernel<1, Q_, true>, 16 + Scratch<1, kCombThreads>::kMerge * 4)
  const bool g8 = a.G > 4;
  if (plan->m > 0) {
    switch (plan->w) {
      case 1: return g8 ? TQ_DECODE_TC_GO(1, 8, true) : TQ_DECODE_TC_GO(1, 4, true);
      case 2: return g8 ? TQ_DECODE_TC_GO(2, 8, true) : TQ_DECODE_TC_GO(2, 4, true);
      default: return g8 ? TQ_DECODE_TC_GO(3, 8, true) : TQ_DECODE_TC_GO(3, 4, true);
    }
  }
  switch (plan->w) {  // stage 1 alone
    case 1: return g8 ? TQ_DECODE_TC_GO(1, 8, false) : TQ_DECODE_TC_GO(1, 4, false);
    case 2: return g8 ? TQ_DECODE_TC_GO(2, 8, false) : TQ_DECODE_TC_GO(2, 4, false);
    default: return g8 ? TQ_DECODE_TC_GO(3, 8, false) : TQ_DECODE_TC_GO(3, 4, false);
  }
#undef TQ_DECODE_TC_GO
}

}  // namespace tq

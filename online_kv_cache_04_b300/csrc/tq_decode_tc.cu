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
// signs are one more ±1 plane.  One and-or turns a 32-bit plane word into
// an e4m3 operand register: it keeps bit i of every byte (layer i) over a
// constant byte C_i, giving per element one of two exact values C_i, C'_i.
// The affine map back to ±1, s = 2(F − (C + C')/2)/(C' − C), is folded into
// the other operand (weights 2x/(C' − C)) and an offset Σ w·(C + C')/2.
//
//   scores: mma.sync m16n8k32 e4m3, rows = 16 tokens, K = 32 coordinates
//           of one plane word, B = the query weights in three e4m3 pieces
//           (each the next 4 bits; one power-of-two scale per head and
//           part), held in registers for the whole (batch, kv head) unit.
//   values: mma.sync m16n8k32 e4m3, rows = 16 coordinates of one plane,
//           K = 32 tokens (one 32-row block word of TQ_LAYOUT_BLOCK32),
//           B = attention weights p·‖v‖ / p·‖r_v‖ in three e4m3 pieces;
//           fp32 accumulators stay in registers over the whole context,
//           and each tile's operand offset is subtracted after the tile.
// Warp-level mma.sync is used instead of tcgen05.mma: decode has one query
// per head, so every MMA here is 8 columns wide, and a tcgen05.mma costs its
// issuing thread ~110-160 cycles whatever its width, while register-operand
// mma.sync lets every warp drive the tensor pipe on its own.
//
// Softmax is online with a lazy reference: the running reference M (of
// log2(p·‖v‖), clamped at ‖v‖ ≥ 2^-32) moves only when a tile exceeds it
// by more than 2^6; the value warps then rescale their accumulators.
//
// Work split: a persistent grid of one CTA per SM takes contiguous ranges of
// 128-token tiles over all (batch, kv head) units; a unit cut between CTAs
// leaves one partial per CTA, merged by the combine kernel of tq_decode.cu.
// Warp roles (288 threads, so that 3 warps per scheduler may use 168
// registers): 0-3 keys (32 tokens each: scores, softmax, weights), 4-7 values
// (32 coordinates of every plane each, as two 16-row MMA tiles), 8 bulk-copy
// loader.  Every wait is bounded; on timeout the kernel sets a fault bit
// (tq_fault_flags) and unwinds.
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <algorithm>

#include "tq_internal.h"
#include "tq_sm100.cuh"

namespace {

using namespace tq::sm100;

constexpr int kTile = 128;
constexpr int kD = 128;
constexpr int kStages = 4;
constexpr int kKW = 4, kVW = 4;                        // key warps, value warps (32 coordinates each)
constexpr int kLoadWarp = kKW + kVW;
constexpr int kThreads = 32 * (kKW + kVW + 1);
constexpr float kTau = 6.0f;                           // lazy-rescale threshold (log2 units)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kVScale = 0.125f;                      // value weights carry 2/δ·2^-3 (below 2^7)
constexpr unsigned kFaultDecode = 2u;

// e4m3 operand, layer i = bit i of each byte: value C_i (bit clear) or C'_i (bit set)
__constant__ uint32_t c_base[8] = {0x38383838u, 0x38383838u, 0x38383838u, 0x30303030u,
                                   0x28282828u, 0x18181818u, 0x00000000u, 0x38383838u};
__constant__ float c_delta[8] = {0.125f, 0.25f, 0.5f, 0.5f, 0.75f, 0.9375f, 2.0f, -2.0f};     // C' - C
__constant__ float c_mean[8] = {1.0625f, 1.125f, 1.25f, 0.75f, 0.625f, 0.53125f, 1.0f, 0.0f};  // (C + C')/2

// A-operand register of layer tig (lo) or 4 + tig (hi) of plane word w: one and-or.
struct Layers {
  uint32_t mlo, mhi, blo, bhi;
  __device__ __forceinline__ explicit Layers(int tig)
      : mlo(0x01010101u << tig), mhi(0x10101010u << tig), blo(c_base[tig]), bhi(c_base[4 + tig]) {}
  __device__ __forceinline__ uint32_t lo(uint32_t w) const { return (w & mlo) | blo; }
  __device__ __forceinline__ uint32_t hi(uint32_t w) const { return (w & mhi) | bhi; }
};

__device__ __forceinline__ void mma_e4m3(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float e4m3_value(uint8_t b) {
  return __half2float(__half(__nv_cvt_fp8_to_halfraw(b, __NV_E4M3)));
}

// Three e4m3 pieces of x (each the next 4 bits): x ≈ v0 + v1/16 + v2/256.
// Writes the bytes and returns the represented value.
__device__ __forceinline__ float pieces3(float x, uint8_t (&p)[3]) {
  float rep = 0.f, sc = 1.f;
#pragma unroll
  for (int k = 0; k < 3; ++k) {
    const __nv_fp8_storage_t b = __nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3);
    const float v = e4m3_value(b);
    p[k] = b;
    rep = fmaf(v, sc, rep);
    x = (x - v) * 16.f;
    sc *= 0.0625f;
  }
  return rep;
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

template <int W, int GP>
struct Shape {
  static constexpr int NPM = W == 3 ? 4 : W;   // ±1 planes of the codebook
  static constexpr int NP = NPM + 1;           // plus the QJL sign plane
  static constexpr int NKS = 4 * NP;           // score K-steps: 4 words of 32 coordinates per plane
  static constexpr int NC = 3 * GP;            // columns of one part: 3 pieces x GP heads
  static constexpr int NCP = NC <= 16 ? 16 : 32;  // NC rounded up to a power of two
  static constexpr int NT = (NC + 7) / 8;      // n-tiles of 8 columns
  static constexpr bool kBRegs = NKS * NT * 2 <= 80;  // query-weight fragments held in registers
  static constexpr int kIdxBytes = kTile * 4 * W * 4;
  static constexpr int kStage = 2 * kIdxBytes + 2 * 2048 + 4 * 512;
  static constexpr int kOffKIdx = 0, kOffKSgn = kIdxBytes, kOffKNorm = kOffKSgn + 2048, kOffKRn = kOffKNorm + 512;
  static constexpr int kOffVIdx = kOffKRn + 512, kOffVSgn = kOffVIdx + kIdxBytes, kOffVNorm = kOffVSgn + 2048,
                       kOffVRn = kOffVNorm + 512;
  // shared memory plan
  static constexpr int kBKBytes = NKS * NT * 256;           // [ks][nt][n 8][k 32] query weight bytes
  static constexpr int SP = 2 * NT * 8 + 1;                // score row pitch in floats (odd: no bank conflicts)
  static constexpr int kSBytes = (kTile * SP * 4 + 15) / 16 * 16;  // raw score pieces [token][part][col]
  static constexpr int kBVBytes = 2 * 4 * NT * 256;         // [part][block][nt][n][k] weight bytes
  static constexpr int kScratch = 32 * NT * 8 * 4;          // per value warp, one plane
  static constexpr int kOffRing = 0;
  static constexpr int kOffBK = kOffRing + kStages * kStage;
  static constexpr int kOffS = kOffBK + kBKBytes;
  static constexpr int kOffBV = kOffS + kSBytes;
  static constexpr int kOffScr = kOffBV + 2 * kBVBytes;
  static constexpr int kOffMisc = kOffScr + kVW * kScratch;
};

struct Misc {
  uint64_t ld_full[kStages], ld_empty[kStages];
  uint64_t p_full[2], p_empty[2], kgroup, st_full[2], st_empty[2];
  int abort;
  float red[2][kKW][8];       // per-tile warp maxima [parity][warp][head]
  float amax[2][8];           // per-unit weight maxima (as non-negative float bits)
  float O[2][8];              // per-unit score offsets per (part, head)
  float coef[4];
  float fac[2][8];            // per weight buffer: accumulator rescale factor per head
  float off[2][kKW][2][24];   // per weight buffer, per key warp: value operand offsets per (part, col)
  float stat_m[2][8];         // per segment parity: reference M per head
  float stat_l[2][kKW][8];    // per segment parity, per key warp: Σ p
};
constexpr int kMiscBytes = 4096;
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

__device__ __forceinline__ bool kgroup_sync(Misc* ms, uint32_t* count, unsigned* fault) {
  __syncwarp();
  const uint32_t bar = smem_u32(&ms->kgroup);
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
  const bool ok = mbar_wait_abortable(bar, (*count) & 1, fault, kFaultDecode, &ms->abort);
  ++*count;
  return ok;
}

// Sum (or max) of N values over the 32 lanes of a warp, N a power of two <= 32,
// by halving; lane L ends with the result for index lane_index<N>(L).
template <int N, bool MAX>
__device__ __forceinline__ float warp_reduce_many(float (&v)[N], int lane) {
#pragma unroll
  for (int n = N, sh = 16; n > 1; n >>= 1, sh >>= 1) {
    const bool upper = lane & sh;
#pragma unroll
    for (int i = 0; i < n / 2; ++i) {
      const float send = upper ? v[i] : v[i + n / 2];
      const float keep = upper ? v[i + n / 2] : v[i];
      const float got = __shfl_xor_sync(0xffffffffu, send, sh);
      v[i] = MAX ? fmaxf(keep, got) : keep + got;
    }
  }
  float x = v[0];
#pragma unroll
  for (int sh = 32 / N / 2; sh > 0; sh >>= 1) {
    const float got = __shfl_xor_sync(0xffffffffu, x, sh);
    x = MAX ? fmaxf(x, got) : x + got;
  }
  return x;
}
template <int N>
__device__ __forceinline__ int lane_index(int lane) {
  int idx = 0;
#pragma unroll
  for (int n = N, sh = 16, bit = N / 2; n > 1; n >>= 1, sh >>= 1, bit >>= 1)
    if (lane & sh) idx += bit;
  return idx;
}

template <int W, int GP>
__global__ void __launch_bounds__(kThreads, 1) decode_tc_kernel(const TcArgs a) {
  using Sh = Shape<W, GP>;
  constexpr int NPM = Sh::NPM, NP = Sh::NP, NKS = Sh::NKS, NC = Sh::NC, NCP = Sh::NCP, NT = Sh::NT;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Misc* ms = reinterpret_cast<Misc*>(smem + Sh::kOffMisc);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gq = lane >> 2, tig = lane & 3;  // mma fragment coordinates
  const Layers ly(tig);
  const int64_t C = gridDim.x;
  const int64_t f0 = (int64_t)blockIdx.x * a.total / C, f1 = ((int64_t)blockIdx.x + 1) * a.total / C;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&ms->ld_full[s]), 1);
      mbar_init(smem_u32(&ms->ld_empty[s]), kKW + kVW);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&ms->p_full[s]), kKW);
      mbar_init(smem_u32(&ms->p_empty[s]), kVW);
      mbar_init(smem_u32(&ms->st_full[s]), kKW);
      mbar_init(smem_u32(&ms->st_empty[s]), kVW);
    }
    mbar_init(smem_u32(&ms->kgroup), kKW);
    ms->abort = 0;
    fence_mbar_init();
  }
  // weight operands start at zero (columns of absent heads stay zero)
  for (int e = threadIdx.x; e < 2 * Sh::kBVBytes / 16; e += kThreads)
    reinterpret_cast<uint4*>(smem + Sh::kOffBV)[e] = make_uint4(0u, 0u, 0u, 0u);
  __syncthreads();
  volatile int* abort_flag = &ms->abort;
  auto wait = [&](uint64_t* bar, uint32_t parity) {
    return mbar_wait_abortable(smem_u32(bar), parity, a.fault, kFaultDecode, abort_flag);
  };

  if (warp == kLoadWarp) {
    // ------------------------------------------------------------ loader
    if (lane == 0) {
      const uint32_t sbase = smem_u32(smem);
      int64_t gi = 0;
      bool ok = true;
      for (int64_t f = f0; ok && f < f1;) {
        int64_t next;
        const Seg sg = segment_at(a, f, f1, &next);
        for (int k = 0; ok && k < sg.n; ++k, ++gi) {
          const int s = (int)(gi % kStages);
          if (gi >= kStages && !(ok = wait(&ms->ld_empty[s], (uint32_t)((gi / kStages - 1) & 1)))) break;
          const int64_t row0 = sg.u * a.ctx_stride + (sg.t0 + k) * kTile;
          const uint32_t bar = smem_u32(&ms->ld_full[s]);
          const uint32_t dst = sbase + Sh::kOffRing + s * Sh::kStage;
          mbar_arrive_expect_tx(bar, Sh::kStage);
          bulk_load(dst + Sh::kOffKIdx, a.kidx + row0 * (4 * W), Sh::kIdxBytes, bar);
          bulk_load(dst + Sh::kOffKSgn, a.ksgn + row0 * 4, 2048, bar);
          bulk_load(dst + Sh::kOffKNorm, a.knorm + row0, 512, bar);
          bulk_load(dst + Sh::kOffKRn, a.krnorm + row0, 512, bar);
          bulk_load(dst + Sh::kOffVIdx, a.vidx + (row0 >> 5) * (W * kD), Sh::kIdxBytes, bar);
          bulk_load(dst + Sh::kOffVSgn, a.vsgn + (row0 >> 5) * kD, 2048, bar);
          bulk_load(dst + Sh::kOffVNorm, a.vnorm + row0, 512, bar);
          bulk_load(dst + Sh::kOffVRn, a.vrnorm + row0, 512, bar);
        }
        f = next;
      }
      // no copy of this CTA may be in flight when it exits
      for (int64_t g = max((int64_t)0, gi - kStages); g < gi; ++g)
        mbar_wait(smem_u32(&ms->ld_full[g % kStages]), (uint32_t)((g / kStages) & 1), a.fault, kFaultDecode);
    }
  } else if (warp < kKW) {
    // ------------------------------------------------------------ keys
    const int r = threadIdx.x;  // token of the tile in the softmax phase; coordinate in the weight set-up
    uint32_t kgc = 0;
    int64_t gi = 0;
    int segc = 0;
    bool ok = true;
    float M[GP], lsum[GP], E[2][GP], O[2][GP];
    uint32_t bf[Sh::kBRegs ? NKS : 1][NT][2];
    // bit position of this token in a 32-row block word: its e4m3 layer and K-element
    const int xb = tq::block32_bit(r & 31), vlay = xb & 7, vk = 4 * (xb & 7) + (xb >> 3);
    const float vw2 = 2.0f * kVScale / c_delta[vlay], vmean = c_mean[vlay];
    float* S = reinterpret_cast<float*>(smem + Sh::kOffS);
    uint8_t* BK = smem + Sh::kOffBK;
    for (int64_t f = f0; ok && f < f1;) {
      int64_t next;
      const Seg sg = segment_at(a, f, f1, &next);
      f = next;
      const int b = (int)(sg.u / a.Hkv), h = (int)(sg.u - (int64_t)b * a.Hkv);
      const int head0 = b * a.Hq + h * a.G;
#pragma unroll
      for (int g = 0; g < GP; ++g) M[g] = -INFINITY, lsum[g] = 0.f;
      if (sg.n > 0) {
        // ---- query weights of this unit: piece scales E, pieces in BK, offsets O
        for (int e = r; e < Sh::kBKBytes / 16; e += 32 * kKW) reinterpret_cast<uint4*>(BK)[e] = make_uint4(0, 0, 0, 0);
        if (r < 16) {
          ms->amax[r >> 3][r & 7] = 0.f;
          ms->O[r >> 3][r & 7] = 0.f;
        }
        if (r < NPM) ms->coef[r] = __ldg(a.walsh + (r < W ? (1 << r) : 7));
        if (!(ok = kgroup_sync(ms, &kgc, a.fault))) break;
        const int j = r;  // coordinate: word j / 32, bit x = j % 32 -> layer x % 8, byte x / 8
        const int jl = j & 7, jk = 4 * jl + ((j & 31) >> 3), jw = j >> 5;
        const float dl = c_delta[jl], mean = c_mean[jl];
        float qv[GP], sv[GP], cf[NPM];
#pragma unroll
        for (int g = 0; g < GP; ++g) {
          qv[g] = g < a.G ? __ldg(a.qt + (size_t)(head0 + g) * kD + j) : 0.f;
          sv[g] = g < a.G ? __ldg(a.st + (size_t)(head0 + g) * kD + j) : 0.f;
        }
#pragma unroll
        for (int P = 0; P < NPM; ++P) cf[P] = ms->coef[P];
#pragma unroll
        for (int g = 0; g < GP; ++g) {
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
        if (!(ok = kgroup_sync(ms, &kgc, a.fault))) break;
#pragma unroll
        for (int p = 0; p < 2; ++p)
#pragma unroll
          for (int g = 0; g < GP; ++g) {
            int e;
            frexpf(ms->amax[p][g], &e);
            E[p][g] = ms->amax[p][g] > 0.f ? ldexpf(1.f, e - 8) : 1.f;
          }
#pragma unroll
        for (int P = 0; P < NP; ++P) {
          const int part = P < NPM ? 0 : 1;
#pragma unroll
          for (int g = 0; g < GP; ++g) {
            const float w = (part == 0 ? 2.f * cf[P < NPM ? P : 0] * qv[g] : 2.f * sv[g]) / dl;
            uint8_t pc[3];
            const float rep = pieces3(w / E[part][g], pc);
#pragma unroll
            for (int k = 0; k < 3; ++k) {
              const int c = k * GP + g;
              BK[(((P * 4 + jw) * NT + (c >> 3)) * 8 + (c & 7)) * 32 + jk] = pc[k];
            }
            float o = rep * E[part][g] * mean;
#pragma unroll
            for (int s = 16; s > 0; s >>= 1) o += __shfl_xor_sync(0xffffffffu, o, s);
            if (lane == 0) atomicAdd(&ms->O[part][g], o);
          }
        }
        if (!(ok = kgroup_sync(ms, &kgc, a.fault))) break;
#pragma unroll
        for (int g = 0; g < GP; ++g) O[0][g] = ms->O[0][g], O[1][g] = ms->O[1][g];
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

        for (int k = 0; ok && k < sg.n; ++k) {
          const int64_t g = gi + k;
          const int s = (int)(g % kStages), buf = (int)(g & 1);
          if (!(ok = wait(&ms->ld_full[s], (uint32_t)((g / kStages) & 1)))) break;
          const uint8_t* stg = smem + Sh::kOffRing + s * Sh::kStage;
          const uint32_t* kiw = reinterpret_cast<const uint32_t*>(stg + Sh::kOffKIdx);
          const uint32_t* ksw = reinterpret_cast<const uint32_t*>(stg + Sh::kOffKSgn);
          // ---- scores: 2 groups of 16 tokens, rows gq and gq + 8 of each; pieces -> S[token][part][col]
#pragma unroll 1
          for (int gr = 0; gr < 2; ++gr) {
            const int tA = 32 * warp + 16 * gr + gq, tB = tA + 8;
            float acc[2][NT][4];
#pragma unroll
            for (int p = 0; p < 2; ++p)
#pragma unroll
              for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[p][nt][e] = 0.f;
#pragma unroll
            for (int ks = 0; ks < NKS; ++ks) {
              const int P = ks >> 2, kw = ks & 3, part = P < NPM ? 0 : 1;
              uint32_t wA, wB;
              if (P < W) {
                wA = kiw[tA * 4 * W + P * 4 + kw];
                wB = kiw[tB * 4 * W + P * 4 + kw];
              } else if (P < NPM) {  // w = 3 product plane: b0 ^ b1 ^ b2
                wA = kiw[tA * 4 * W + kw] ^ kiw[tA * 4 * W + (4 + kw) % (4 * W)] ^ kiw[tA * 4 * W + (8 + kw) % (4 * W)];
                wB = kiw[tB * 4 * W + kw] ^ kiw[tB * 4 * W + (4 + kw) % (4 * W)] ^ kiw[tB * 4 * W + (8 + kw) % (4 * W)];
              } else {
                wA = ksw[tA * 4 + kw];
                wB = ksw[tB * 4 + kw];
              }
              const uint32_t a0 = ly.lo(wA), a1 = ly.lo(wB), a2 = ly.hi(wA), a3 = ly.hi(wB);
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
                mma_e4m3(acc[part][nt], a0, a1, a2, a3, b0, b1);
              }
            }
#pragma unroll
            for (int p = 0; p < 2; ++p)
#pragma unroll
              for (int nt = 0; nt < NT; ++nt) {
                const int c = p * NT * 8 + 8 * nt + 2 * tig;
                S[tA * Sh::SP + c] = acc[p][nt][0];
                S[tA * Sh::SP + c + 1] = acc[p][nt][1];
                S[tB * Sh::SP + c] = acc[p][nt][2];
                S[tB * Sh::SP + c + 1] = acc[p][nt][3];
              }
          }
          __syncwarp();
          const float* Sr = S + r * Sh::SP;
          const float kn = reinterpret_cast<const float*>(stg + Sh::kOffKNorm)[r];
          const float kr = reinterpret_cast<const float*>(stg + Sh::kOffKRn)[r];
          const float vn = reinterpret_cast<const float*>(stg + Sh::kOffVNorm)[r];
          const float vr = reinterpret_cast<const float*>(stg + Sh::kOffVRn)[r];
          const bool valid = (sg.t0 + k) * kTile + r < sg.L;
          const float lvn = log2f(vn);
          float s2[GP], av[GP];
#pragma unroll
          for (int hh = 0; hh < GP; ++hh) {
            const float dm = (Sr[hh] + Sr[GP + hh] * 0.0625f) + Sr[2 * GP + hh] * 0.00390625f;
            const float dq = (Sr[NT * 8 + hh] + Sr[NT * 8 + GP + hh] * 0.0625f) + Sr[NT * 8 + 2 * GP + hh] * 0.00390625f;
            const float mse = fmaf(E[0][hh], dm, -O[0][hh]);
            const float qjl = fmaf(E[1][hh], dq, -O[1][hh]);
            const float sc = a.scale * fmaf(kn, mse, a.alpha * kr * qjl);
            s2[hh] = (valid && hh < a.G) ? sc * kLog2e : -INFINITY;
            av[hh] = s2[hh] + fmaxf(lvn, -32.f);
          }
          // tile maximum of log2(p·‖v‖) per head across the key warps
          {
            float x[GP];
#pragma unroll
            for (int hh = 0; hh < GP; ++hh) x[hh] = av[hh];
            const float mx = warp_reduce_many<GP, true>(x, lane);
            if ((lane & (32 / GP - 1)) == 0) ms->red[g & 1][warp][lane_index<GP>(lane)] = mx;
          }
          if (!(ok = kgroup_sync(ms, &kgc, a.fault))) break;
          float fac[GP];
#pragma unroll
          for (int hh = 0; hh < GP; ++hh) {
            float tm = ms->red[g & 1][0][hh];
#pragma unroll
            for (int q = 1; q < kKW; ++q) tm = fmaxf(tm, ms->red[g & 1][q][hh]);
            float nm = M[hh];
            if (M[hh] == -INFINITY) nm = tm;
            else if (tm > M[hh] + kTau) nm = tm;
            fac[hh] = (M[hh] != -INFINITY && nm != M[hh]) ? exp2f(M[hh] - nm) : 1.f;
            M[hh] = nm;
            lsum[hh] *= fac[hh];
          }
          // ---- attention weights of this tile -> value operands (three e4m3 pieces)
          if (g >= 2 && !(ok = wait(&ms->p_empty[buf], (uint32_t)(((g >> 1) - 1) & 1)))) break;
          uint8_t* bv = smem + Sh::kOffBV + buf * Sh::kBVBytes;
          float offv[2][NCP];
#pragma unroll
          for (int p = 0; p < 2; ++p)
#pragma unroll
            for (int c = 0; c < NCP; ++c) offv[p][c] = 0.f;
#pragma unroll
          for (int hh = 0; hh < GP; ++hh) {
            const bool live = valid && hh < a.G && M[hh] != -INFINITY;
            const float p = live ? exp2f(s2[hh] - M[hh]) : 0.f;
            const float wm = live ? exp2f(s2[hh] + lvn - M[hh]) : 0.f;
            lsum[hh] += p;
#pragma unroll
            for (int part = 0; part < 2; ++part) {
              uint8_t pc[3];
              pieces3((part == 0 ? wm : p * vr) * vw2, pc);
#pragma unroll
              for (int q = 0; q < 3; ++q) {
                const int c = q * GP + hh;
                bv[(((part * 4 + warp) * NT + (c >> 3)) * 8 + (c & 7)) * 32 + vk] = pc[q];
                offv[part][c] = e4m3_value(pc[q]) * vmean;
              }
            }
          }
          // this warp's operand offsets per (part, column)
#pragma unroll
          for (int part = 0; part < 2; ++part) {
            const float o = warp_reduce_many<NCP, false>(offv[part], lane);
            const int c = lane_index<NCP>(lane);
            if ((lane & (32 / NCP - 1)) == 0 && c < NC) ms->off[buf][warp][part][c] = o;
          }
          if (lane < GP) ms->fac[buf][lane] = fac[lane];
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(smem_u32(&ms->p_full[buf]));
            mbar_arrive(smem_u32(&ms->ld_empty[s]));
          }
        }
        gi += sg.n;
      }
      if (!ok) break;
      // ---- segment statistics for the value warps (slot by segment parity)
      const int sp = segc & 1;
      if (segc >= 2 && !(ok = wait(&ms->st_empty[sp], (uint32_t)(((segc >> 1) - 1) & 1)))) break;
#pragma unroll
      for (int hh = 0; hh < GP; ++hh) {
        float l = lsum[hh];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
        if (lane == 0) {
          ms->stat_l[sp][warp][hh] = l;
          if (warp == 0) ms->stat_m[sp][hh] = M[hh];
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&ms->st_full[sp]));
      ++segc;
    }
  } else {
    // ------------------------------------------------------------ values: 32 coordinates of every plane
    const int vwarp = warp - kKW;
    float* scr = reinterpret_cast<float*>(smem + Sh::kOffScr + vwarp * Sh::kScratch);
    float vacc[NP][2][NT][4];  // [plane][row tile: coordinates 32v + 16mt + (gq, gq + 8)][n-tile][fragment]
#pragma unroll
    for (int P = 0; P < NP; ++P)
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) vacc[P][mt][nt][e] = 0.f;
    int64_t gi = 0;
    int segc = 0;
    bool ok = true;
    for (int64_t f = f0; ok && f < f1;) {
      int64_t next;
      const Seg sg = segment_at(a, f, f1, &next);
      f = next;
      for (int k = 0; ok && k < sg.n; ++k) {
        const int64_t g = gi + k;
        const int s = (int)(g % kStages), buf = (int)(g & 1);
        if (!(ok = wait(&ms->ld_full[s], (uint32_t)((g / kStages) & 1)))) break;
        if (!(ok = wait(&ms->p_full[buf], (uint32_t)((g >> 1) & 1)))) break;
        const uint8_t* stg = smem + Sh::kOffRing + s * Sh::kStage;
        const uint32_t* vi = reinterpret_cast<const uint32_t*>(stg + Sh::kOffVIdx);
        const uint32_t* vsg = reinterpret_cast<const uint32_t*>(stg + Sh::kOffVSgn);
        const uint8_t* bv = smem + Sh::kOffBV + buf * Sh::kBVBytes;
        // lazy rescale of the accumulators (the head of column c is c % GP)
        {
          float fh[GP];
          bool any = false;
#pragma unroll
          for (int hh = 0; hh < GP; ++hh) {
            fh[hh] = ms->fac[buf][hh];
            any |= fh[hh] != 1.f;
          }
          if (any) {
#pragma unroll
            for (int P = 0; P < NP; ++P)
#pragma unroll
              for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                  for (int e = 0; e < 2; ++e) {
                    const int c = 8 * nt + 2 * tig + e;
                    const float x = c < NC ? fh[c % GP] : 1.f;
                    vacc[P][mt][nt][e] *= x;
                    vacc[P][mt][nt][2 + e] *= x;
                  }
          }
        }
#pragma unroll
        for (int kb = 0; kb < 4; ++kb) {
          uint32_t b0[2][NT], b1[2][NT];
#pragma unroll
          for (int part = 0; part < 2; ++part)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              const uint32_t* row = reinterpret_cast<const uint32_t*>(bv + (((part * 4 + kb) * NT + nt) * 8 + gq) * 32);
              b0[part][nt] = row[tig];
              b1[part][nt] = row[4 + tig];
            }
#pragma unroll
          for (int P = 0; P < NP; ++P) {
            const int part = P < NPM ? 0 : 1;
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
              const int jA = 32 * vwarp + 16 * mt + gq, jB = jA + 8;
              uint32_t wA, wB;
              if (P < W) {
                wA = vi[(kb * W + P) * kD + jA];
                wB = vi[(kb * W + P) * kD + jB];
              } else if (P < NPM) {  // w = 3 product plane
                wA = vi[(kb * W) * kD + jA] ^ vi[(kb * W + 1 % W) * kD + jA] ^ vi[(kb * W + 2 % W) * kD + jA];
                wB = vi[(kb * W) * kD + jB] ^ vi[(kb * W + 1 % W) * kD + jB] ^ vi[(kb * W + 2 % W) * kD + jB];
              } else {
                wA = vsg[kb * kD + jA];
                wB = vsg[kb * kD + jB];
              }
              const uint32_t a0 = ly.lo(wA), a1 = ly.lo(wB), a2 = ly.hi(wA), a3 = ly.hi(wB);
#pragma unroll
              for (int nt = 0; nt < NT; ++nt) mma_e4m3(vacc[P][mt][nt], a0, a1, a2, a3, b0[part][nt], b1[part][nt]);
            }
          }
        }
        // minus this tile's operand offsets Σ w·(C + C')/2 per column
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int c = 8 * nt + 2 * tig + e;
            float om = 0.f, oq = 0.f;
            if (c < NC) {
#pragma unroll
              for (int q = 0; q < kKW; ++q) om += ms->off[buf][q][0][c], oq += ms->off[buf][q][1][c];
            }
#pragma unroll
            for (int P = 0; P < NP; ++P)
#pragma unroll
              for (int mt = 0; mt < 2; ++mt) {
                const float o = P < NPM ? om : oq;
                vacc[P][mt][nt][e] -= o;
                vacc[P][mt][nt][2 + e] -= o;
              }
          }
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(smem_u32(&ms->p_empty[buf]));
          mbar_arrive(smem_u32(&ms->ld_empty[s]));
        }
      }
      if (!ok) break;
      // ---- partial of this CTA for the unit
      const int sp = segc & 1;
      if (!(ok = wait(&ms->st_full[sp], (uint32_t)((segc >> 1) & 1)))) break;
      const int b = (int)(sg.u / a.Hkv), h = (int)(sg.u - (int64_t)b * a.Hkv);
      const int head0 = b * a.Hq + h * a.G;
      constexpr int NO = 32 * GP / 32;  // outputs (coordinate, head) per lane
      float rot[NO], sgn[NO];
#pragma unroll
      for (int o = 0; o < NO; ++o) rot[o] = sgn[o] = 0.f;
      if (sg.n > 0) {
#pragma unroll
        for (int P = 0; P < NP; ++P) {
          const float cf = P < NPM ? __ldg(a.walsh + (P < W ? (1 << P) : 7)) : 1.f;
#pragma unroll
          for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              const int c = 8 * nt + 2 * tig, rA = 16 * mt + gq;
              *reinterpret_cast<float2*>(scr + rA * NT * 8 + c) = make_float2(vacc[P][mt][nt][0], vacc[P][mt][nt][1]);
              *reinterpret_cast<float2*>(scr + (rA + 8) * NT * 8 + c) =
                  make_float2(vacc[P][mt][nt][2], vacc[P][mt][nt][3]);
            }
          __syncwarp();
#pragma unroll
          for (int o = 0; o < NO; ++o) {
            const int cj = lane, hh = o;  // coordinate 32v + lane, head o
            const float* row = scr + cj * NT * 8;
            // Σ_t W_t s_t = (Σ_t w_t (F_t - mean_t)) / kVScale, w in three pieces
            const float v = ((row[hh] + row[GP + hh] * 0.0625f) + row[2 * GP + hh] * 0.00390625f) * (1.f / kVScale);
            if (P < NPM) rot[o] = fmaf(cf, v, rot[o]);
            else sgn[o] = v;
          }
          __syncwarp();
        }
      }
#pragma unroll
      for (int o = 0; o < NO; ++o) {
        const int hh = o;
        if (hh < a.G) {
          float* pp = a.part + ((size_t)(head0 + hh) * a.smax + sg.slot) * (2 + 2 * kD);
          pp[2 + 32 * vwarp + lane] = rot[o];
          pp[2 + kD + 32 * vwarp + lane] = sgn[o];
          if (vwarp == 0 && lane == 0) {
            float l = 0.f;
#pragma unroll
            for (int q = 0; q < kKW; ++q) l += ms->stat_l[sp][q][hh];
            pp[0] = ms->stat_m[sp][hh];
            pp[1] = l;
          }
        }
      }
#pragma unroll
      for (int P = 0; P < NP; ++P)
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) vacc[P][mt][nt][e] = 0.f;
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&ms->st_empty[sp]));
      gi += sg.n;
      ++segc;
    }
  }
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

// Decode attention over the compressed cache on the 5th-generation tensor
// cores (tcgen05), for d = m = 128 and up to 8 query heads per kv head.
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
// Bits as exact tensor-core operands.  A symmetric Lloyd-Max codebook is a
// sum of ±1 bit-planes, c[idx] = Σ_P coef_P·s_P with s = 2·bit − 1 (Walsh
// expansion; w = 1: one plane, w = 2: two, w = 3: three plus their product).
// The QJL signs are one more ±1 plane.  A plane word is expanded with one
// and-or per output register: bit i of every byte (e4m3 operand) or bit p of
// every half-word (f16 operand) is placed over a constant, giving one of two
// exactly representable values C or C' per element.  The affine map back to
// ±1 (s = 2(F − (C + C')/2)/(C' − C)) is folded into the other operand and a
// per-column correction.
//
//   keys:   A = expanded key planes (e4m3) in TMEM, lane = token;
//           B = query weights 2·coef·q̃_j/δ split into four e4m3 pieces
//           (each carries the next 4 bits), kind::f8f6f4.
//   values: A = expanded value planes (f16) in TMEM, lane = coordinate,
//           which needs the 32-row block layout (one coordinate of 32 tokens
//           per word); B = attention weights p·‖v‖ and p·‖r_v‖ (f16),
//           kind::f16, accumulated over the whole context in TMEM.
// Softmax is online with a lazy reference: the running reference M moves
// only when a tile exceeds it by more than 2^8, and then the value
// accumulators in TMEM are rescaled once.  M tracks log2(p·‖v‖) so that the
// f16 weights stay in range for any value norm.
//
// Work split: a persistent grid of one CTA per SM takes contiguous ranges of
// 128-token tiles over all (batch, kv head) units; a unit cut between CTAs
// leaves one partial per CTA, merged by the combine kernel of tq_decode.cu.
//
// Warp roles (320 threads): 0-3 keys (thread = token), 4-7 values (thread =
// coordinate), 8 MMA issue + TMEM owner, 9 bulk-copy loader.  Every wait is
// bounded; on timeout the kernel sets a fault bit (tq_fault_flags) and
// unwinds.
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
constexpr int kThreads = 352, kMmaWarp = 8, kLoadWarp = 9, kVMmaWarp = 10;
constexpr float kTau = 6.0f;                  // lazy-rescale threshold (log2 units)
constexpr float kLog2e = 1.4426950408889634f;
constexpr unsigned kFaultDecode = 2u;
constexpr uint32_t kTmemCols = 512;

// e4m3 key operand, layer i = bit i of each byte: value C (bit clear) or C' (bit set)
__constant__ uint32_t c_k_base[8] = {0x38383838u, 0x38383838u, 0x38383838u, 0x30303030u,
                                     0x28282828u, 0x18181818u, 0x00000000u, 0x38383838u};
__constant__ float c_k_delta[8] = {0.125f, 0.25f, 0.5f, 0.5f, 0.75f, 0.9375f, 2.0f, -2.0f};  // C' - C
__constant__ float c_k_mean[8] = {1.0625f, 1.125f, 1.25f, 0.75f, 0.625f, 0.53125f, 1.0f, 0.0f};  // (C + C')/2
// f16 value operand, bit position p in 10..15 of each half-word
__constant__ uint32_t c_v_base[6] = {0x38003800u, 0x34003400u, 0x2C002C00u, 0x1C001C00u, 0x00000000u, 0x3C003C00u};
__constant__ float c_v_delta[6] = {0.5f, 0.75f, 0.9375f, 0.99609375f, 2.0f, -2.0f};
__constant__ float c_v_mean[6] = {0.75f, 0.625f, 0.53125f, 0.501953125f, 1.0f, 0.0f};

// Token pair i (tokens 2i, 2i+1 of a 32-row block sit at bits i, i+16) is
// shifted left so that it lands on position vpos(i) in 10..15.
__host__ __device__ constexpr int vpos(int i) { return i >= 10 ? i : (i >= 4 ? i + 6 : i + 12); }

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

// Per-instantiation sizes.  TMEM columns: key ring (KR slots of one plane,
// 32 columns = 128 e4m3), value ring (VR slots of half a plane, 32 columns =
// 64 tokens of f16), score accumulators (2 buffers x MSE|QJL x NH), value
// accumulators (NP x 16), one constant -1 operand column group (8).
template <int W, int GP>
struct Shape {
  static constexpr int NPM = W == 3 ? 4 : W;  // ±1 planes of the codebook
  static constexpr int NP = NPM + 1;          // plus the QJL sign plane
  static constexpr int NH = 4 * GP;           // 4 pieces x GP heads
  static constexpr int kRing = (512 - 4 * NH - 16 * NP - 8) / 32;  // key + value slots that fit
  static constexpr int KR = (kRing + 1) / 2 < 2 * NP ? (kRing + 1) / 2 : 2 * NP;
  static constexpr int VR = kRing - KR < 4 * NP ? kRing - KR : 4 * NP;
  static constexpr uint32_t kColK = 0, kColV = 32 * KR, kColS = kColV + 32 * VR, kColVD = kColS + 4 * NH,
                            kColOne = kColVD + 16 * NP;
  static_assert(kColOne + 8 <= kTmemCols, "TMEM plan exceeds 512 columns");
  static_assert(KR >= NP && VR >= 2, "rings too small for one tile");
  static_assert(VR <= 4 * NP, "value ring deeper than two tiles breaks the end-of-segment wait");
  static constexpr int kIdxBytes = kTile * 4 * W * 4;
  static constexpr int kStage = 2 * kIdxBytes + 2 * 2048 + 4 * 512;
  static constexpr int kOffKIdx = 0, kOffKSgn = kIdxBytes, kOffKNorm = kOffKSgn + 2048, kOffKRn = kOffKNorm + 512;
  static constexpr int kOffVIdx = kOffKRn + 512, kOffVSgn = kOffVIdx + kIdxBytes, kOffVNorm = kOffVSgn + 2048,
                       kOffVRn = kOffVNorm + 512;
};

constexpr int kOffBK = 0;                  // NP planes x 4 KB (NH <= 32 rows of 128 bytes)
constexpr int kOffBV = 5 * 4096;           // 2 buffers x 3 SW128 atoms of 2 KB (tokens 0-63, 64-127, offsets)
constexpr int kBVBytes = 3 * 2048;
constexpr int kOffRing = kOffBV + 2 * kBVBytes;
constexpr int kMiscBytes = 4096;
constexpr int kMaxRing = 16;

struct Misc {
  uint64_t ld_full[kStages], ld_empty[kStages];
  uint64_t ka_full[kMaxRing], ka_empty[kMaxRing], va_full[kMaxRing], va_empty[kMaxRing];
  uint64_t s_full[2], s_empty[2], p_full[2], p_empty[2];
  uint64_t bk_full, vd_free, kgroup, st_full[2], st_empty[2];
  uint32_t tmem_base;
  int abort;
  float red[2][4][8];       // per-tile warp maxima [parity][warp][head]
  float amax[2][8];         // per-unit weight maxima (as non-negative float bits)
  float O[2][8];            // per-unit offset per (part, head)
  float coef[4];
  float stat_m[2][8];       // per segment parity: reference M per head
  float stat_l[2][4][8];    // per segment parity, per key warp: Σ p
};
static_assert(sizeof(Misc) <= kMiscBytes, "barriers and per-head state must fit their region");

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

__device__ __forceinline__ uint32_t kgroup_sync(Misc* ms, uint32_t* count, unsigned* fault) {
  __syncwarp();
  const uint32_t bar = smem_u32(&ms->kgroup);
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
  const bool ok = mbar_wait_abortable(bar, (*count) & 1, fault, kFaultDecode, &ms->abort);
  ++*count;
  return ok;
}

// SW128 K-major offset of element (row n, byte e) in a tile of 128-byte rows.
__device__ __forceinline__ uint32_t sw128(int n, int e) {
  return (n >> 3) * 1024 + (n & 7) * 128 + ((((e >> 4) ^ (n & 7))) << 4) + (e & 15);
}

// Offset of f16 element (row n, token t) in a 16 x 128 attention-weight tile:
// two SW128 atoms of 64 tokens (128 bytes per row), 2 KB apart.
__device__ __forceinline__ uint32_t bv_off(int n, int t) { return (t >> 6) * 2048 + sw128(n, (t & 63) * 2); }

// Sum (or max) of N values over the 32 lanes of a warp, N a power of two <= 32,
// by halving: afterwards lane L holds the result for index bits (L >> (5 -
// log2 N)) ... of v (see lane_index), written to v[0].
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
// Index of the value that warp_reduce_many<N> leaves in lane L.
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
  constexpr int NPM = Sh::NPM, NP = Sh::NP, NH = Sh::NH, KR = Sh::KR, VR = Sh::VR;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  Misc* ms = reinterpret_cast<Misc*>(smem + kOffRing + kStages * Sh::kStage);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t C = gridDim.x;
  const int64_t f0 = (int64_t)blockIdx.x * a.total / C, f1 = ((int64_t)blockIdx.x + 1) * a.total / C;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&ms->ld_full[s]), 1);
      mbar_init(smem_u32(&ms->ld_empty[s]), 8);
    }
    for (int s = 0; s < KR; ++s) {
      mbar_init(smem_u32(&ms->ka_full[s]), 4);
      mbar_init(smem_u32(&ms->ka_empty[s]), 1);
    }
    for (int s = 0; s < VR; ++s) {
      mbar_init(smem_u32(&ms->va_full[s]), 4);
      mbar_init(smem_u32(&ms->va_empty[s]), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&ms->s_full[s]), 1);
      mbar_init(smem_u32(&ms->s_empty[s]), 4);
      mbar_init(smem_u32(&ms->p_full[s]), 4);
      mbar_init(smem_u32(&ms->p_empty[s]), 1);
      mbar_init(smem_u32(&ms->st_full[s]), 4);
      mbar_init(smem_u32(&ms->st_empty[s]), 4);
    }
    mbar_init(smem_u32(&ms->bk_full), 4);
    mbar_init(smem_u32(&ms->vd_free), 4);
    mbar_init(smem_u32(&ms->kgroup), 4);
    ms->abort = 0;
    fence_mbar_init();
  }
  // attention-weight operands start at zero (rows of absent heads stay zero)
  for (int e = threadIdx.x; e < 2 * kBVBytes / 16; e += kThreads)
    reinterpret_cast<uint4*>(smem + kOffBV)[e] = make_uint4(0u, 0u, 0u, 0u);
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(&ms->tmem_base), kTmemCols);
    tmem_relinquish();
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ms->tmem_base;
  volatile int* abort_flag = &ms->abort;
  auto wait = [&](uint64_t* bar, uint32_t parity) {
    return mbar_wait_abortable(smem_u32(bar), parity, a.fault, kFaultDecode, abort_flag);
  };

  if (warp == kLoadWarp) {
    // ------------------------------------------------------------ loader
    if (lane == 0) {
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
          const uint32_t dst = sbase + kOffRing + s * Sh::kStage;
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
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ key MMAs (scores)
    if (lane == 0) {
      constexpr uint32_t idk = idesc_e4m3_f32(128, NH);
      int64_t gi = 0, kc = 0;
      int nseg = 0;
      bool ok = true;
      for (int64_t f = f0; ok && f < f1;) {
        int64_t next;
        const Seg sg = segment_at(a, f, f1, &next);
        f = next;
        if (sg.n == 0) continue;
        if (!(ok = wait(&ms->bk_full, (uint32_t)(nseg & 1)))) break;
        tc_fence_after();
        for (int k = 0; ok && k < sg.n; ++k) {
          const int64_t g = gi + k;
          const int sb = (int)(g & 1);
          if (g >= 2 && !(ok = wait(&ms->s_empty[sb], (uint32_t)(((g >> 1) - 1) & 1)))) break;
#pragma unroll 1
          for (int P = 0; P < NP; ++P, ++kc) {
            const int slot = (int)(kc % KR);
            if (!(ok = wait(&ms->ka_full[slot], (uint32_t)((kc / KR) & 1)))) break;
            tc_fence_after();
            const uint32_t d = tmem + Sh::kColS + sb * 2 * NH + (P < NPM ? 0 : NH);
            const uint64_t bd = desc_sw128(sbase + kOffBK + P * 4096);
#pragma unroll 1
            for (int kk = 0; kk < 4; ++kk) {
              const uint32_t acc = (P < NPM) ? ((P > 0 || kk > 0) ? 1u : 0u) : (kk > 0 ? 1u : 0u);
              mma_ts_f8(d, tmem + Sh::kColK + slot * 32 + kk * 8, bd + ((kk * 32) >> 4), idk, acc);
            }
            mma_commit(smem_u32(&ms->ka_empty[slot]));
          }
          if (!ok) break;
          mma_commit(smem_u32(&ms->s_full[sb]));
        }
        gi += sg.n;
        ++nseg;
      }
    }
  } else if (warp == kVMmaWarp) {
    // ------------------------------------------------------------ value MMAs (weights x values)
    if (lane == 0) {
      constexpr uint32_t idv = idesc_f16_f32(128, 16);
      int64_t gi = 0, vc = 0;
      int nseg = 0;
      bool ok = true;
      for (int64_t f = f0; ok && f < f1;) {
        int64_t next;
        const Seg sg = segment_at(a, f, f1, &next);
        f = next;
        if (sg.n == 0) continue;
        for (int k = 0; ok && k < sg.n; ++k) {
          const int64_t g = gi + k;
          const int sb = (int)(g & 1);
          const bool first = k == 0;
          if (!(ok = wait(&ms->p_full[sb], (uint32_t)((g >> 1) & 1)))) break;
          if (first && nseg >= 1 && !(ok = wait(&ms->vd_free, (uint32_t)((nseg - 1) & 1)))) break;
          tc_fence_after();
          const uint32_t bv = sbase + kOffBV + sb * kBVBytes;
#pragma unroll 1
          for (int P = 0; ok && P < NP; ++P) {
#pragma unroll 1
            for (int half = 0; half < 2; ++half, ++vc) {
              const int slot = (int)(vc % VR);
              if (!(ok = wait(&ms->va_full[slot], (uint32_t)((vc / VR) & 1)))) break;
              tc_fence_after();
              const uint32_t d = tmem + Sh::kColVD + 16 * P;
#pragma unroll 1
              for (int kk = 0; kk < 4; ++kk) {
                const uint64_t bd = desc_sw128(bv + half * 2048) + ((kk * 32) >> 4);
                mma_ts(d, tmem + Sh::kColV + slot * 32 + kk * 8, bd, idv, (first && half == 0 && kk == 0) ? 0u : 1u);
              }
              // minus this tile's operand offsets Σ w·(C + C')/2 (per key warp, f16 hi + lo)
              if (half == 1) mma_ts(d, tmem + Sh::kColOne, desc_sw128(bv + 2 * 2048), idv, 1u);
              mma_commit(smem_u32(&ms->va_empty[slot]));
            }
          }
          if (!ok) break;
          mma_commit(smem_u32(&ms->p_empty[sb]));
        }
        gi += sg.n;
        ++nseg;
      }
    }
  } else if (warp < 4) {
    // ------------------------------------------------------------ keys: thread = token
    const int r = threadIdx.x;  // token of the tile, TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    uint32_t kgc = 0;           // kgroup phases used
    int64_t gi = 0, kc = 0;
    int segc = 0;
    bool ok = true;
    float M[GP], lsum[GP], E_m[GP], E_q[GP], O_m[GP], O_q[GP];
    const int vp = vpos((r & 31) >> 1) - 10;
    const float two_over_delta = 2.0f / c_v_delta[vp], vmean = c_v_mean[vp];
    // expand tile g (stage g % kStages) into the NP key planes of the TMEM ring
    auto expand = [&](int64_t g) {
      const int s = (int)(g % kStages);
      if (!wait(&ms->ld_full[s], (uint32_t)((g / kStages) & 1))) return false;
      const uint8_t* st = smem + kOffRing + s * Sh::kStage;
      uint32_t iw[4 * W], sw[4], tw[4];
#pragma unroll
      for (int p = 0; p < W; ++p) {
        const uint4 v = reinterpret_cast<const uint4*>(st + Sh::kOffKIdx + r * 16 * W)[p];
        iw[4 * p] = v.x; iw[4 * p + 1] = v.y; iw[4 * p + 2] = v.z; iw[4 * p + 3] = v.w;
      }
      {
        const uint4 v = reinterpret_cast<const uint4*>(st + Sh::kOffKSgn)[r];
        sw[0] = v.x; sw[1] = v.y; sw[2] = v.z; sw[3] = v.w;
      }
#pragma unroll
      for (int k = 0; k < 4; ++k)  // w = 3: the product plane s0·s1·s2 has bit b0 ^ b1 ^ b2
        tw[k] = W == 3 ? iw[k] ^ iw[(4 + k) % (4 * W)] ^ iw[(8 + k) % (4 * W)] : 0u;
      // all planes of the tile are stored, then one wait for the stores, then
      // every slot is released to the MMA warp
#pragma unroll
      for (int P = 0; P < NP; ++P) {
        uint32_t pw[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) pw[k] = P < W ? iw[(4 * P + k) % (4 * W)] : (P < NPM ? tw[k] : sw[k]);
        const int64_t c = kc + P;
        const int slot = (int)(c % KR);
        if (c >= KR && !wait(&ms->ka_empty[slot], (uint32_t)((c / KR - 1) & 1))) return false;
        uint32_t vals[32];
#pragma unroll
        for (int k = 0; k < 4; ++k)
#pragma unroll
          for (int i = 0; i < 8; ++i) vals[8 * k + i] = (pw[k] & (0x01010101u << i)) | c_k_base[i];
        tmem_st32(tmem + lane_base + Sh::kColK + slot * 32, vals);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0)
        for (int P = 0; P < NP; ++P) mbar_arrive(smem_u32(&ms->ka_full[(kc + P) % KR]));
      kc += NP;
      return true;
    };
    for (int64_t f = f0; ok && f < f1;) {
      int64_t next;
      const Seg sg = segment_at(a, f, f1, &next);
      f = next;
      const int b = (int)(sg.u / a.Hkv), h = (int)(sg.u - (int64_t)b * a.Hkv);
      const int head0 = b * a.Hq + h * a.G;
#pragma unroll
      for (int g = 0; g < GP; ++g) M[g] = -INFINITY, lsum[g] = 0.f;
      if (sg.n > 0) {
        // ---- query weights for this unit: B_K planes, piece scales E, offsets O
        if (r < 16) {
          ms->amax[r >> 3][r & 7] = 0.f;
          ms->O[r >> 3][r & 7] = 0.f;
        }
        if (r < NPM) ms->coef[r] = __ldg(a.walsh + (r < W ? (1 << r) : 7));
        if (!(ok = kgroup_sync(ms, &kgc, a.fault))) break;
        const int j = r;  // coordinate handled by this thread
        const float dl = c_k_delta[j & 7], mean = c_k_mean[j & 7];
        float qv[GP], sv[GP];
#pragma unroll
        for (int g = 0; g < GP; ++g) {
          qv[g] = g < a.G ? __ldg(a.qt + (size_t)(head0 + g) * kD + j) : 0.f;
          sv[g] = g < a.G ? __ldg(a.st + (size_t)(head0 + g) * kD + j) : 0.f;
        }
        float cf[NPM];
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
        for (int g = 0; g < GP; ++g) {
          int e;
          frexpf(ms->amax[0][g], &e);
          E_m[g] = ms->amax[0][g] > 0.f ? ldexpf(1.f, e - 8) : 1.f;
          frexpf(ms->amax[1][g], &e);
          E_q[g] = ms->amax[1][g] > 0.f ? ldexpf(1.f, e - 8) : 1.f;
        }
        // element position of coordinate j in a 128-element key plane row
        const int eidx = 4 * (8 * (j >> 5) + (j & 7)) + ((j & 31) >> 3);
#pragma unroll
        for (int P = 0; P < NP; ++P) {
#pragma unroll
          for (int g = 0; g < GP; ++g) {
            const bool mse = P < NPM;
            const float E = mse ? E_m[g] : E_q[g];
            float x = (mse ? 2.f * cf[P < NPM ? P : 0] * qv[g] : 2.f * sv[g]) / dl / E;
            float rep = 0.f, sc = 1.f;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const __nv_fp8_storage_t p8 = __nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3);
              const float pv = __half2float(__half(__nv_cvt_fp8_to_halfraw(p8, __NV_E4M3)));
              smem[kOffBK + P * 4096 + sw128(k * GP + g, eidx)] = p8;
              rep += pv * sc;
              x = (x - pv) * 16.f;
              sc *= 0.0625f;
            }
            float o = rep * E * mean;
#pragma unroll
            for (int s = 16; s > 0; s >>= 1) o += __shfl_xor_sync(0xffffffffu, o, s);
            if (lane == 0) atomicAdd(&ms->O[mse ? 0 : 1][g], o);
          }
        }
        fence_proxy_async_smem();
        if (!(ok = kgroup_sync(ms, &kgc, a.fault))) break;
#pragma unroll
        for (int g = 0; g < GP; ++g) O_m[g] = ms->O[0][g], O_q[g] = ms->O[1][g];
        if (lane == 0) mbar_arrive(smem_u32(&ms->bk_full));

        // ---- tiles: expand the next tile's keys, then score / weigh this one
        if (!(ok = expand(gi))) break;
        for (int k = 0; ok && k < sg.n; ++k) {
          const int64_t g = gi + k;
          if (k + 1 < sg.n && !(ok = expand(g + 1))) break;
          const int sb = (int)(g & 1), s = (int)(g % kStages);
          if (!(ok = wait(&ms->s_full[sb], (uint32_t)((g >> 1) & 1)))) break;
          tc_fence_after();
          float dv[2 * NH];
          {
            uint32_t v[32];
#pragma unroll
            for (int c = 0; c < 2 * NH / 32; ++c) {
              tmem_ld32(tmem + lane_base + Sh::kColS + sb * 2 * NH + 32 * c, v);
              tmem_ld_wait();
#pragma unroll
              for (int e = 0; e < 32; ++e) dv[32 * c + e] = __uint_as_float(v[e]);
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&ms->s_empty[sb]));
          const uint8_t* stg = smem + kOffRing + s * Sh::kStage;
          const float kn = reinterpret_cast<const float*>(stg + Sh::kOffKNorm)[r];
          const float kr = reinterpret_cast<const float*>(stg + Sh::kOffKRn)[r];
          const float vn = reinterpret_cast<const float*>(stg + Sh::kOffVNorm)[r];
          const float vr = reinterpret_cast<const float*>(stg + Sh::kOffVRn)[r];
          const bool valid = (sg.t0 + k) * kTile + r < sg.L;
          const float lvn = log2f(vn);
          float s2[GP], av[GP];
#pragma unroll
          for (int hh = 0; hh < GP; ++hh) {
            const float dm = ((dv[hh] + dv[GP + hh] * 0.0625f) + dv[2 * GP + hh] * 0.00390625f) +
                             dv[3 * GP + hh] * 0.000244140625f;
            const float dq = ((dv[NH + hh] + dv[NH + GP + hh] * 0.0625f) + dv[NH + 2 * GP + hh] * 0.00390625f) +
                             dv[NH + 3 * GP + hh] * 0.000244140625f;
            const float mse = fmaf(E_m[hh], dm, -O_m[hh]);
            const float qjl = fmaf(E_q[hh], dq, -O_q[hh]);
            const float sc = a.scale * fmaf(kn, mse, a.alpha * kr * qjl);
            s2[hh] = (valid && hh < a.G) ? sc * kLog2e : -INFINITY;
            av[hh] = s2[hh] + fmaxf(lvn, -32.f);
          }
          // tile maximum of log2(p·‖v‖) per head, across the four key warps
          {
            float x[GP];
#pragma unroll
            for (int hh = 0; hh < GP; ++hh) x[hh] = av[hh];
            const float mx = warp_reduce_many<GP, true>(x, lane);
            if ((lane & (32 / GP - 1)) == 0) ms->red[g & 1][warp][lane_index<GP>(lane)] = mx;
          }
          if (!(ok = kgroup_sync(ms, &kgc, a.fault))) break;
          float fac[GP];
          bool rescale = false;
#pragma unroll
          for (int hh = 0; hh < GP; ++hh) {
            const float tm = fmaxf(fmaxf(ms->red[g & 1][0][hh], ms->red[g & 1][1][hh]),
                                   fmaxf(ms->red[g & 1][2][hh], ms->red[g & 1][3][hh]));
            float nm = M[hh];
            if (M[hh] == -INFINITY) nm = tm;
            else if (tm > M[hh] + kTau) nm = tm;
            fac[hh] = (M[hh] != -INFINITY && nm != M[hh]) ? exp2f(M[hh] - nm) : 1.f;
            rescale |= fac[hh] != 1.f;
            M[hh] = nm;
          }
          if (rescale) {
            // value accumulators of the tiles so far: wait for their MMAs (tile g-1's
            // weight buffer release; its phase is at most one behind, since tile g-3's
            // release was awaited before tile g-1's weights were written), scale in place
            if (!(ok = wait(&ms->p_empty[(g - 1) & 1], (uint32_t)(((g - 1) >> 1) & 1)))) break;
            tc_fence_after();
#pragma unroll
            for (int P = 0; P < NP; ++P) {
              uint32_t v[16];
              tmem_ld16(tmem + lane_base + Sh::kColVD + 16 * P, v);
              tmem_ld_wait();
#pragma unroll
              for (int c = 0; c < 16; ++c) {
                const int hh = c & 7;
                if (hh < GP) v[c] = __float_as_uint(__uint_as_float(v[c]) * fac[hh]);
              }
              uint32_t v8a[8], v8b[8];
#pragma unroll
              for (int c = 0; c < 8; ++c) v8a[c] = v[c], v8b[c] = v[8 + c];
              tmem_st8(tmem + lane_base + Sh::kColVD + 16 * P, v8a);
              tmem_st8(tmem + lane_base + Sh::kColVD + 16 * P + 8, v8b);
            }
            tmem_st_wait();
            tc_fence_before();
#pragma unroll
            for (int hh = 0; hh < GP; ++hh) lsum[hh] *= fac[hh];
          }
          // attention weights of this tile -> f16 B operand of the value MMA
          if (g >= 2 && !(ok = wait(&ms->p_empty[sb], (uint32_t)(((g >> 1) - 1) & 1)))) break;
          uint8_t* bv = smem + kOffBV + sb * kBVBytes;
          float off[2 * GP];
#pragma unroll
          for (int hh = 0; hh < GP; ++hh) {
            off[hh] = off[GP + hh] = 0.f;
            if (hh >= a.G) continue;
            const bool live = valid && M[hh] != -INFINITY;
            const float p = live ? exp2f(s2[hh] - M[hh]) : 0.f;
            const float wm = live ? exp2f(s2[hh] + lvn - M[hh]) : 0.f;
            const float wq = p * vr;
            lsum[hh] += p;
            const __half hm = __float2half_rn(wm * two_over_delta);
            const __half hq = __float2half_rn(wq * two_over_delta);
            *reinterpret_cast<__half*>(bv + bv_off(hh, r)) = hm;
            *reinterpret_cast<__half*>(bv + bv_off(8 + hh, r)) = hq;
            off[hh] = __half2float(hm) * vmean;
            off[GP + hh] = __half2float(hq) * vmean;
          }
          // this warp's operand offsets for every weight row, as f16 hi + lo at
          // elements 2·warp, 2·warp + 1 of the offset row (A there is -1)
          {
            const float o = warp_reduce_many<2 * GP, false>(off, lane);
            const int c = lane_index<2 * GP>(lane);
            if ((lane & (16 / GP - 1)) == 0 && (c % GP) < a.G) {
              const __half hi = __float2half_rn(o), lo = __float2half_rn(o - __half2float(hi));
              const int n = c < GP ? c : 8 + (c - GP);
              *reinterpret_cast<__half2*>(bv + 2 * 2048 + sw128(n, 4 * warp)) = __halves2half2(hi, lo);
            }
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(smem_u32(&ms->p_full[sb]));
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
    // ------------------------------------------------------------ values: thread = coordinate
    const int j = threadIdx.x - 128;
    const uint32_t lane_base = static_cast<uint32_t>((warp - 4) * 32) << 16;
    {
      const uint32_t one[8] = {0xBC00BC00u, 0xBC00BC00u, 0xBC00BC00u, 0xBC00BC00u, 0u, 0u, 0u, 0u};
      tmem_st8(tmem + lane_base + Sh::kColOne, one);
      tmem_st_wait();
      tc_fence_before();
    }
    int64_t gi = 0, vc = 0;
    int segc = 0;
    bool ok = true;
    for (int64_t f = f0; ok && f < f1;) {
      int64_t next;
      const Seg sg = segment_at(a, f, f1, &next);
      f = next;
      for (int k = 0; ok && k < sg.n; ++k) {
        const int64_t g = gi + k;
        const int s = (int)(g % kStages);
        if (!(ok = wait(&ms->ld_full[s], (uint32_t)((g / kStages) & 1)))) break;
        const uint32_t* vi = reinterpret_cast<const uint32_t*>(smem + kOffRing + s * Sh::kStage + Sh::kOffVIdx);
        const uint32_t* vsg = reinterpret_cast<const uint32_t*>(smem + kOffRing + s * Sh::kStage + Sh::kOffVSgn);
        // half-planes are stored in groups of up to VR, one store wait per group
        int pending = 0;
        auto release = [&]() {
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0)
            for (int e = 0; e < pending; ++e) mbar_arrive(smem_u32(&ms->va_full[(vc - pending + e) % VR]));
          pending = 0;
        };
#pragma unroll 1
        for (int P = 0; ok && P < NP; ++P) {
          uint32_t bw[4];
#pragma unroll
          for (int kb = 0; kb < 4; ++kb) {
            if (P < W) bw[kb] = vi[(kb * W + P) * kD + j];
            else if (P < NPM)  // w = 3 product plane
              bw[kb] = vi[(kb * W) * kD + j] ^ vi[(kb * W + 1 % W) * kD + j] ^ vi[(kb * W + 2 % W) * kD + j];
            else bw[kb] = vsg[kb * kD + j];
          }
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            const int slot = (int)(vc % VR);
            if (pending == VR) release();
            if (vc >= VR && !(ok = wait(&ms->va_empty[slot], (uint32_t)((vc / VR - 1) & 1)))) break;
            uint32_t vals[32];
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
              const uint32_t wd = bw[2 * half + kk];
              const uint32_t x0 = wd, x1 = wd << 6, x2 = wd << 12;
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const int p = vpos(i);
                const uint32_t src = i >= 10 ? x0 : (i >= 4 ? x1 : x2);
                vals[16 * kk + i] = (src & ((1u << p) | (1u << (p + 16)))) | c_v_base[p - 10];
              }
            }
            tmem_st32(tmem + lane_base + Sh::kColV + slot * 32, vals);
            ++vc;
            ++pending;
          }
        }
        if (!ok) break;
        if (pending > 0) release();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&ms->ld_empty[s]));
      }
      if (!ok) break;
      // ---- partial of this CTA for the unit
      const int sp = segc & 1;
      if (!(ok = wait(&ms->st_full[sp], (uint32_t)((segc >> 1) & 1)))) break;
      float d[NP][16];
      if (sg.n > 0) {
        // all value MMAs of the segment: the last tile's weight-buffer release.
        // Its phase is at most one behind: expanding the last tile needed ring
        // slots freed by the value MMAs of two tiles earlier (the ring holds at
        // most two tiles), and those MMAs released the same buffer one phase ago.
        const int64_t last = gi + sg.n - 1;
        if (!(ok = wait(&ms->p_empty[last & 1], (uint32_t)((last >> 1) & 1)))) break;
        tc_fence_after();
#pragma unroll
        for (int P = 0; P < NP; ++P) {
          uint32_t v[16];
          tmem_ld16(tmem + lane_base + Sh::kColVD + 16 * P, v);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 16; ++c) d[P][c] = __uint_as_float(v[c]);
        }
        tc_fence_before();
      }
      const int b = (int)(sg.u / a.Hkv), h = (int)(sg.u - (int64_t)b * a.Hkv);
      const int head0 = b * a.Hq + h * a.G;
      float cf[NPM];
#pragma unroll
      for (int P = 0; P < NPM; ++P) cf[P] = __ldg(a.walsh + (P < W ? (1 << P) : 7));
      for (int hh = 0; hh < a.G && hh < GP; ++hh) {
        float ar = 0.f, as = 0.f;
        if (sg.n > 0) {
#pragma unroll
          for (int P = 0; P < NPM; ++P) ar = fmaf(cf[P], d[P][hh], ar);
          as = d[NPM][8 + hh];
        }
        float* pp = a.part + ((size_t)(head0 + hh) * a.smax + sg.slot) * (2 + 2 * kD);
        pp[2 + j] = ar;
        pp[2 + kD + j] = as;
        if (j == 0) {
          pp[0] = ms->stat_m[sp][hh];
          pp[1] = (ms->stat_l[sp][0][hh] + ms->stat_l[sp][1][hh]) + (ms->stat_l[sp][2][hh] + ms->stat_l[sp][3][hh]);
        }
      }
      __syncwarp();
      if (lane == 0) {
        if (sg.n > 0) mbar_arrive(smem_u32(&ms->vd_free));
        mbar_arrive(smem_u32(&ms->st_empty[sp]));
      }
      gi += sg.n;
      ++segc;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int W>
constexpr int smem_bytes() {
  return 1024 + kOffRing + kStages * Shape<W, 4>::kStage + kMiscBytes;
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
    const int bytes = std::max(smem, 120 * 1024);  // one CTA per SM: it owns all of TMEM
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
      return TQ_ERR_CUDA;
    kern<<<grid, kThreads, bytes, stream>>>(a);
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

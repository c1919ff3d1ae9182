// Search scores on the tensor cores: for d and m multiples of 128 (m may be
// 0), w in 1..3, records in TQ_LAYOUT_ROWS.
//
// The score of stored vector i for query q ("TurboQuant压缩效果": vector
// search engines; the estimator of "TurboQuant 与 AI 效率革命" §三 applied to
// the residual as in "谷歌TurboQuant如何绕过内存墙？" §2 stage 2) is
//   score = ‖x_i‖ Σ_P coef_P ⟨Π q, s_P,i⟩ + √(π/2)/m ‖r_i‖ ⟨S q, σ_i⟩,
// where c[idx] = Σ_P coef_P s_P is the Walsh expansion of the symmetric
// codebook into ±1 bit-planes (w = 3 adds the product plane b0 ^ b1 ^ b2) and
// σ is one more ±1 plane.  Over many queries this is a dense contraction:
// rows = stored vectors, K = planes x coordinates, columns = queries.
//
// search_table_kernel: per group of four queries, the column operand of
//   every K-step, laid out as the mma.sync B fragments (f16 hi + lo pairs of
//   -coef_P (Π q)_j / E0 and -(S q)_j / E1, E a power of two per query and
//   part), and the per-query constants E0 and α·E1.
// search_score_kernel: a CTA scores blocks of 128 vectors against 32 queries
//   with mma.sync m16n8k16 f16, block after block (vector blocks blockIdx.x,
//   + gridDim.x, ...).  The bits of a record word become exact ±1 f16
//   operands in registers: one integer multiply moves bits L and 16 + L to the
//   sign positions of an f16x2 register and one logic op fills in 1.0, so the
//   operand is -s.  The query operand streams through shared memory in
//   16 KiB chunks (bulk copies, two buffers); fp32 accumulators per part
//   stay in registers.  The epilogue scales by the record's norms and keeps,
//   per query, the k best (score desc, index asc) of every vector the CTA has
//   seen: warp w owns the shared-memory lists of the CTA's queries 4w .. 4w + 3
//   and merges each block's scores into them.  At the end the lists go to the workspace as candidates, which
//   the merge kernel of tq_search.cu reduces to the k best: the nq x n score
//   matrix is never written.
#include <cuda_fp16.h>

#include <algorithm>
#include <type_traits>

#include "tq_internal.h"
#include "tq_sm100.cuh"

namespace {

using namespace tq::sm100;

constexpr int kWarps = 8, kThreads = 32 * kWarps;
constexpr int kRows = 16 * kWarps;         // vectors per CTA
constexpr int kTilesPerCta = 8;            // groups of four queries per CTA: 32 queries
constexpr int kChunkWords = 4;             // one chunk: 4 words (128 coordinates) of one plane = 8 K-steps
constexpr int kChunkSteps = 2 * kChunkWords;
constexpr int kFragBytes = 256;            // one (K-step, query group) B operand: 32 lanes x uint2
constexpr int kChunkBytes = kChunkSteps * kTilesPerCta * kFragBytes;
constexpr unsigned kFaultSearch = 4u;
constexpr int kMaxK = 64;                  // list entries a warp keeps per query (two per lane)
constexpr int kStagePitch = kRows + 1;     // floats per query row of the score staging area

// Per lane q: 2^(3-q), 2^(7-q), 2^(11-q), 2^(15-q) (multiplier from constant
// memory: the move stays an integer multiply on the FMA pipe).
__constant__ uint32_t c_smul[4][4] = {{8u, 128u, 2048u, 32768u},
                                      {4u, 64u, 1024u, 16384u},
                                      {2u, 32u, 512u, 8192u},
                                      {1u, 16u, 256u, 4096u}};

struct SearchTcArgs {
  const uint32_t* idx; const uint32_t* sgn; const float* norm; const float* rnorm;
  int64_t n;
  int nq, d, m, w, npm;     // npm: codebook planes (w, or 4 with the product plane)
  // deq (w = 3): the codebook part contracts the centroid values themselves,
  // c[idx] as f16 hi + lo looked up from the index bits, against one block of
  // Π q (npm_t = 1 table block instead of npm planes)
  int deq, npm_t;
  const float* centroids;   // [2^w]
  uint32_t* ctab;           // deq: [8] bytes of f16 c_hi[0..7] (lo bytes, hi bytes), then of c_lo[0..7]
  int groups;               // query groups of four
  int64_t ksteps;           // 2 (npm d + m) / 32
  const float* qt; const float* st;   // [nq][d] Π q, [nq][m] S q
  const float* walsh;
  float alpha;
  __half* table;            // [ksteps][groups][8 n][4 quad][2 reg][2 half]
  float* consts;            // [nq][2]: E0, α E1
  int k;                    // list length (1 .. kMaxK)
  int vchunks;              // gridDim.x: CTAs along the vectors = candidate lists per query
  int32_t* cand_idx;        // [nq][vchunks][k]
  float* cand_sc;
  unsigned* fault;
};

__device__ __forceinline__ uint32_t sign_operand(uint32_t t) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(t), "r"(0x80008000u), "r"(0x3C003C00u));
  return r;
}

__device__ __forceinline__ uint32_t prmt(uint32_t lo, uint32_t hi, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(lo), "r"(hi), "r"(sel));
  return r;
}

// Bucket indices of four coordinates, as the four selector nibbles of a byte
// permute: bits 0, 1, 8, 9 of each plane word t_p (already shifted) are the
// coordinates' bit p; nibble k of the result = Σ_p bit_p << p of coordinate k
// (bits 0, 1, 8, 9 -> nibbles 0, 1, 2, 3).  (t & 0x303)·9 copies bits 0, 1, 8, 9
// to 3, 4, 11, 12 without overlap, so the mask keeps bits 0, 4, 8, 12.
__device__ __forceinline__ uint32_t index_nibbles(uint32_t t0, uint32_t t1, uint32_t t2) {
  return (((t0 & 0x303u) * 9u) & 0x1111u) | (((t1 & 0x303u) * 18u) & 0x2222u) | (((t2 & 0x303u) * 36u) & 0x4444u);
}

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Query column operand.  Coordinate j of a plane sits in word j / 32 at bit
// x = 16e + L (e: f16 half of the operand register, L = 0..15); K-step
// 2·(word) + L / 8 of the plane; inside it K index 8·((L / 4) % 2) + 2·(L % 4) + e.
__global__ void __launch_bounds__(kThreads) search_table_kernel(SearchTcArgs a) {
  __shared__ float amax[2][4];
  const int grp = blockIdx.x, lane = threadIdx.x & 31;
  if (threadIdx.x < 8) amax[threadIdx.x >> 2][threadIdx.x & 3] = 0.f;
  __syncthreads();
  float cmax = 0.f;
  for (int P = 0; P < a.npm; ++P) cmax = fmaxf(cmax, fabsf(__ldg(a.walsh + (P < a.w ? (1 << P) : 7))));
  if (a.deq) cmax = 1.f;  // the weights are Π q itself
  for (int g = 0; g < 4; ++g) {
    const int q = 4 * grp + g;
    float m0 = 0.f, m1 = 0.f;
    if (q < a.nq) {
      for (int j = threadIdx.x; j < a.d; j += kThreads) m0 = fmaxf(m0, fabsf(a.qt[(size_t)q * a.d + j]) * cmax);
      for (int j = threadIdx.x; j < a.m; j += kThreads) m1 = fmaxf(m1, fabsf(a.st[(size_t)q * a.m + j]));
    }
    for (int o = 16; o > 0; o >>= 1) {
      m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, o));
      m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, o));
    }
    if (lane == 0) {
      atomicMax(reinterpret_cast<int*>(&amax[0][g]), __float_as_int(m0));
      atomicMax(reinterpret_cast<int*>(&amax[1][g]), __float_as_int(m1));
    }
  }
  __syncthreads();
  // E: the power of two taking the part's largest weight below 2^12; weights are stored divided by E
  auto escale = [&](int p, int g) {
    int ex;
    frexpf(amax[p][g], &ex);
    return amax[p][g] > 0.f ? ldexpf(1.f, ex - 12) : 1.f;
  };
  if (a.deq && grp == 0 && threadIdx.x == 0) {
    // the centroids as f16 hi + lo pairs, byte-sliced for byte permutes: word
    // 2s + h (s: 0 lo bytes, 1 hi bytes; h: entries 4h .. 4h + 3) of piece pc
    uint32_t words[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
    for (int i = 0; i < 8; ++i) {
      const float c = __ldg(a.centroids + i);
      const __half ch = __float2half_rn(c), cl = __float2half_rn(c - __half2float(ch));
      const uint32_t bits[2] = {__half_as_ushort(ch), __half_as_ushort(cl)};
      for (int pc = 0; pc < 2; ++pc) {
        words[4 * pc + (i >> 2)] |= (bits[pc] & 0xFFu) << (8 * (i & 3));
        words[4 * pc + 2 + (i >> 2)] |= (bits[pc] >> 8) << (8 * (i & 3));
      }
    }
    for (int i = 0; i < 8; ++i) a.ctab[i] = words[i];
  }
  if (threadIdx.x < 4 && 4 * grp + (int)threadIdx.x < a.nq) {
    const int g = threadIdx.x;
    a.consts[(size_t)(4 * grp + g) * 2] = escale(0, g);
    a.consts[(size_t)(4 * grp + g) * 2 + 1] = a.alpha * escale(1, g);
  }
  const int words_d = a.d / 32;
  const int np = a.npm_t;
  const int64_t total = (int64_t)np * a.d + a.m;  // plane coordinates, codebook planes first
  for (int64_t e = threadIdx.x; e < total; e += kThreads) {
    const bool qjl = e >= (int64_t)np * a.d;
    const int P = qjl ? np : (int)(e / a.d);
    const int j = qjl ? (int)(e - (int64_t)np * a.d) : (int)(e - (int64_t)P * a.d);
    const int x = j & 31, eh = x >> 4, L = x & 15;
    int64_t ks = 2 * ((int64_t)P * words_d + (j >> 5)) + (L >> 3);
    int kk = 8 * ((L >> 2) & 1) + 2 * (L & 3) + eh;
    if (a.deq && !qjl) {  // centroid values: coordinate j at K-step j / 16, K index j % 16
      ks = j >> 4;
      kk = j & 15;
    }
    // the ±1 planes' operand is -s, so their weight is negated; centroids carry their sign
    const float coef = qjl ? 0.f : a.deq ? -1.f : __ldg(a.walsh + (P < a.w ? (1 << P) : 7));
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const int q = 4 * grp + g;
      float xv = 0.f;
      if (q < a.nq) {
        xv = qjl ? -a.st[(size_t)q * a.m + j] / escale(1, g) : -coef * a.qt[(size_t)q * a.d + j] / escale(0, g);
      }
      const __half xh = __float2half_rn(xv), xl = __float2half_rn(xv - __half2float(xh));
      // [n][quad][reg][half]: column 2g holds hi, 2g + 1 lo
      const size_t base = ((((size_t)ks * a.groups + grp) * 8 + 2 * g) * 4 + ((kk & 7) >> 1)) * 4 +
                          (kk >> 3) * 2 + (kk & 1);
      a.table[base] = xh;
      a.table[base + 16] = xl;
    }
  }
}

// CTA (vector chunk bx, query block by): vector blocks bx, bx + gridDim.x, ...
// of 128 rows each (rows v0 .. v0 + 127), query groups 8·by .. 8·by + 7.  Warp
// wp takes rows v0 + 16 wp + (0..15): fragment row gq is vector v0 + 16 wp +
// gq, row gq + 8 the vector eight further.
template <bool DEQ>
__global__ void __launch_bounds__(kThreads, 2) search_score_kernel(SearchTcArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* buf = smem;  // [2][kChunkSteps][kTilesPerCta][256 B]
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + 2 * kChunkBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gq = lane >> 2, tig = lane & 3;
  const int g0 = blockIdx.y * kTilesPerCta, ntl = min(kTilesPerCta, a.groups - g0);
  const int words_d = a.d / 32, words_m = a.m / 32;
  const int nchunks = (a.npm_t * words_d + words_m) / kChunkWords;
  float* stage = reinterpret_cast<float*>(smem + 2 * kChunkBytes + 64);  // [32 queries][kStagePitch]
  float* lsc = stage + 32 * kStagePitch;                                   // [32 queries][kMaxK] list scores
  int32_t* lid = reinterpret_cast<int32_t*>(lsc + 32 * kMaxK);              // [32 queries][kMaxK] list indices
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&full[0]), 1);
    mbar_init(smem_u32(&full[1]), 1);
    fence_mbar_init();
  }
  __syncthreads();
  const int64_t nblocks = (a.n + kRows - 1) / kRows;
  const int64_t myblocks = blockIdx.x < nblocks ? (nblocks - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  const int64_t total_chunks = myblocks * nchunks;  // over all of this CTA's vector blocks
  // global chunk gc = (block iteration)·nchunks + c covers K-steps 8c .. 8c + 7;
  // its operand for groups g0 .. g0 + ntl - 1 is ntl contiguous 256-byte
  // fragments per K-step in the table
  auto issue = [&](int64_t gc) {
    const int c = (int)(gc % nchunks);
    const uint32_t bar = smem_u32(&full[gc & 1]);
    mbar_arrive_expect_tx(bar, (uint32_t)(kChunkSteps * ntl * kFragBytes));
    const uint32_t dst = smem_u32(buf + (gc & 1) * kChunkBytes);
    for (int s = 0; s < kChunkSteps; ++s) {
      const int64_t ks = (int64_t)kChunkSteps * c + s;
      bulk_load(dst + s * kTilesPerCta * kFragBytes, a.table + (ks * a.groups + g0) * (kFragBytes / 2),
                ntl * kFragBytes, bar);
    }
  };
  if (threadIdx.x == 0) {
    if (total_chunks > 0) issue(0);
    if (total_chunks > 1) issue(1);
  }
  const int wi = a.w * words_d;  // index words per record
  const uint32_t m15 = c_smul[tig][3], m11 = c_smul[tig][2], m7 = c_smul[tig][1], m3 = c_smul[tig][0];
  bool alive = true;
  int64_t nissued = total_chunks > 1 ? 2 : total_chunks;  // thread 0: chunks whose copies were started
  int64_t ndone = 0;                                      // chunks whose copies this thread has seen land
  // the k-best lists, in rank order; empty entries rank last
  for (int e = threadIdx.x; e < 32 * kMaxK; e += kThreads) lsc[e] = -INFINITY, lid[e] = INT32_MAX;
  float acc[2][kTilesPerCta][4];
  int64_t r0 = 0, r1 = 0;
  bool ok0 = false, ok1 = false;
  int64_t gbase = 0;  // global chunk number of this block's chunk 0
  // deq: the byte tables of f16 c_hi and c_lo (lo bytes of entries 0..7, then hi bytes)
  uint32_t ct[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) ct[i] = DEQ ? __ldg(a.ctab + i) : 0u;
  // one chunk of centroid values (deq): 128 coordinates of every index plane;
  // K-step sl covers coordinates 16·sl .. 16·sl + 15 of the chunk in order
  auto chunk_deq = [&](int c) {
    const int kw0 = c * kChunkWords;
    uint4 x[2][3];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int64_t row = r ? r1 : r0;
#pragma unroll
      for (int p = 0; p < 3; ++p)
        x[r][p] = (r ? ok1 : ok0) ? __ldg(reinterpret_cast<const uint4*>(a.idx + row * wi + p * words_d + kw0))
                                  : make_uint4(0u, 0u, 0u, 0u);
    }
    const int64_t gc = gbase + c;
    if (alive) {
      alive = mbar_wait(smem_u32(&full[gc & 1]), (uint32_t)((gc >> 1) & 1), a.fault, kFaultSearch);
      ndone += alive ? 1 : 0;
    }
    const uint2* bfr = reinterpret_cast<const uint2*>(buf + (gc & 1) * kChunkBytes);
#pragma unroll
    for (int kw = 0; kw < kChunkWords; ++kw) {
#pragma unroll
      for (int sh = 0; sh < 2; ++sh) {
        // this lane's coordinates 2·tig, 2·tig + 1, 8 + 2·tig, 9 + 2·tig of K-step 2·kw + sh
        const int off = 16 * sh + 2 * tig;
        uint32_t hi[2][2], lo[2][2];  // [row][k-slot pair 2tig | 8 + 2tig]
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const uint4* xr = x[r];
          auto word = [&](int p) {
            return kw == 0 ? xr[p].x : kw == 1 ? xr[p].y : kw == 2 ? xr[p].z : xr[p].w;
          };
          const uint32_t sel = index_nibbles(word(0) >> off, word(1) >> off, word(2) >> off);
          const uint32_t hl = prmt(ct[0], ct[1], sel), hh = prmt(ct[2], ct[3], sel);
          const uint32_t ll = prmt(ct[4], ct[5], sel), lh = prmt(ct[6], ct[7], sel);
          hi[r][0] = prmt(hl, hh, 0x5140u);
          hi[r][1] = prmt(hl, hh, 0x7362u);
          lo[r][0] = prmt(ll, lh, 0x5140u);
          lo[r][1] = prmt(ll, lh, 0x7362u);
        }
        const int sl = 2 * kw + sh;
#pragma unroll
        for (int t = 0; t < kTilesPerCta; ++t) {
          const uint2 b = bfr[(sl * kTilesPerCta + t) * 32 + lane];
          mma16816(acc[0][t], hi[0][0], hi[1][0], hi[0][1], hi[1][1], b.x, b.y);
          mma16816(acc[0][t], lo[0][0], lo[1][0], lo[0][1], lo[1][1], b.x, b.y);
        }
      }
    }
    // every warp is done with this buffer; its generic-proxy reads are ordered
    // before the bulk copy (async proxy) that refills it
    fence_proxy_async_smem();
    __syncthreads();
    if (threadIdx.x == 0 && gc + 2 < total_chunks && alive) {
      issue(gc + 2);
      nissued = gc + 3;
    }
  };
  // one chunk into the accumulators of part PART (0: codebook planes, 1: QJL plane)
  auto chunk = [&](int c, auto part_tag) {
    constexpr int PART = decltype(part_tag)::value;
    const int wpos = c * kChunkWords;  // word position over all planes
    const int P = PART ? a.npm_t : wpos / words_d;
    const int kw0 = PART ? wpos - a.npm_t * words_d : wpos - P * words_d;
    uint4 x[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int64_t row = r ? r1 : r0;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (r ? ok1 : ok0) {
        if (PART) {
          v = __ldg(reinterpret_cast<const uint4*>(a.sgn + row * words_m + kw0));
        } else if (P < a.w) {
          v = __ldg(reinterpret_cast<const uint4*>(a.idx + row * wi + P * words_d + kw0));
        } else {  // product plane b0 ^ b1 ^ b2
          const uint4 p0 = __ldg(reinterpret_cast<const uint4*>(a.idx + row * wi + kw0));
          const uint4 p1 = __ldg(reinterpret_cast<const uint4*>(a.idx + row * wi + words_d + kw0));
          const uint4 p2 = __ldg(reinterpret_cast<const uint4*>(a.idx + row * wi + 2 * words_d + kw0));
          v = make_uint4(p0.x ^ p1.x ^ p2.x, p0.y ^ p1.y ^ p2.y, p0.z ^ p1.z ^ p2.z, p0.w ^ p1.w ^ p2.w);
        }
      }
      x[r] = v;
    }
    const int64_t gc = gbase + c;
    if (alive) {
      alive = mbar_wait(smem_u32(&full[gc & 1]), (uint32_t)((gc >> 1) & 1), a.fault, kFaultSearch);
      ndone += alive ? 1 : 0;
    }
    const uint2* bfr = reinterpret_cast<const uint2*>(buf + (gc & 1) * kChunkBytes);
#pragma unroll
    for (int kw = 0; kw < kChunkWords; ++kw) {
      const uint32_t w0 = kw == 0 ? x[0].x : kw == 1 ? x[0].y : kw == 2 ? x[0].z : x[0].w;
      const uint32_t w1 = kw == 0 ? x[1].x : kw == 1 ? x[1].y : kw == 2 ? x[1].z : x[1].w;
#pragma unroll
      for (int s = 0; s < 2; ++s) {
        // layers q + 8s (K 2q + e) and 4 + q + 8s (K 8 + 2q + e) to the sign bits
        const uint32_t mlo = s ? m7 : m15, mhi = s ? m3 : m11;
        const uint32_t a0 = sign_operand(w0 * mlo), a1 = sign_operand(w1 * mlo);
        const uint32_t a2 = sign_operand(w0 * mhi), a3 = sign_operand(w1 * mhi);
        const int sl = 2 * kw + s;
#pragma unroll
        for (int t = 0; t < kTilesPerCta; ++t) {
          const uint2 b = bfr[(sl * kTilesPerCta + t) * 32 + lane];
          mma16816(acc[PART][t], a0, a1, a2, a3, b.x, b.y);
        }
      }
    }
    // every warp is done with this buffer; its generic-proxy reads are ordered
    // before the bulk copy (async proxy) that refills it
    fence_proxy_async_smem();
    __syncthreads();
    if (threadIdx.x == 0 && gc + 2 < total_chunks && alive) {
      issue(gc + 2);
      nissued = gc + 3;
    }
  };
  const int ncb = a.npm_t * words_d / kChunkWords;  // codebook chunks; the QJL plane's follow
  const int k = a.k;
#pragma unroll 1
  for (int64_t it = 0; it < myblocks; ++it) {
    const int64_t v0 = ((int64_t)blockIdx.x + it * gridDim.x) * kRows;
    gbase = it * nchunks;
    r0 = v0 + 16 * warp + gq;
    r1 = r0 + 8;
    ok0 = r0 < a.n;
    ok1 = r1 < a.n;
#pragma unroll
    for (int p = 0; p < 2; ++p)
#pragma unroll
      for (int t = 0; t < kTilesPerCta; ++t)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[p][t][e] = 0.f;
    if constexpr (DEQ) {
#pragma unroll 1
      for (int c = 0; c < ncb; ++c) chunk_deq(c);
    } else {
#pragma unroll 1
      for (int c = 0; c < ncb; ++c) chunk(c, std::integral_constant<int, 0>{});
    }
#pragma unroll 1
    for (int c = ncb; c < nchunks; ++c) chunk(c, std::integral_constant<int, 1>{});
    // scores of the block: column pair (hi, lo) 2·tig of tile t is query
    // 4 (g0 + t) + tig, staged as [4t + tig][vector - v0] (-inf past n)
    const float nv0 = ok0 ? __ldg(a.norm + r0) : 0.f, nv1 = ok1 ? __ldg(a.norm + r1) : 0.f;
    const float rv0 = ok0 && a.m > 0 ? __ldg(a.rnorm + r0) : 0.f, rv1 = ok1 && a.m > 0 ? __ldg(a.rnorm + r1) : 0.f;
#pragma unroll
    for (int t = 0; t < kTilesPerCta; ++t) {
      const int q = 4 * (g0 + t) + tig;
      const bool live = t < ntl && q < a.nq;
      const float e0 = live ? a.consts[(size_t)q * 2] : 0.f, e1 = live ? a.consts[(size_t)q * 2 + 1] : 0.f;
      float* row = stage + (4 * t + tig) * kStagePitch + 16 * warp + gq;
      row[0] = ok0 ? fmaf(nv0 * e0, acc[0][t][0] + acc[0][t][1], rv0 * e1 * (acc[1][t][0] + acc[1][t][1]))
                   : -INFINITY;
      row[8] = ok1 ? fmaf(nv1 * e0, acc[0][t][2] + acc[0][t][3], rv1 * e1 * (acc[1][t][2] + acc[1][t][3]))
                   : -INFINITY;
    }
    __syncthreads();
    // merge into the lists: candidates in increasing vector order, each inserted
    // at its rank (entries ranking after it move down one, the last falls off)
#pragma unroll 1
    for (int j = 0; j < 4; ++j) {
      const float* row = stage + (4 * warp + j) * kStagePitch;
      float* qs = lsc + (4 * warp + j) * kMaxK;
      int32_t* qi = lid + (4 * warp + j) * kMaxK;
#pragma unroll 1
      for (int part = 0; part < kRows / 32; ++part) {
        const float sv = row[32 * part + lane];
        const int32_t iv = (int32_t)(v0 + 32 * part + lane);
        const float ks = qs[k - 1];  // the list's last entry
        const int32_t ki = qi[k - 1];
        uint32_t want = __ballot_sync(0xffffffffu, sv > -INFINITY && (sv > ks || (sv == ks && iv < ki)));
        while (want != 0u) {
          const int src = __ffs(want) - 1;
          want &= want - 1;
          const float cs = __shfl_sync(0xffffffffu, sv, src);
          const int32_t ci = __shfl_sync(0xffffffffu, iv, src);
          // rank = entries that rank before (cs, ci); lane l looks at entries l and l + 32
          const float s0 = qs[lane], s1 = qs[lane + 32];
          const int32_t i0 = qi[lane], i1 = qi[lane + 32];
          const bool b0 = s0 > cs || (s0 == cs && i0 < ci);
          const bool b1 = s1 > cs || (s1 == cs && i1 < ci);
          const int pos = __popc(__ballot_sync(0xffffffffu, b0)) + __popc(__ballot_sync(0xffffffffu, b1));
          if (pos >= k) continue;  // no longer makes the list (it grew better meanwhile)
          // entries pos .. k - 2 move down one, the candidate takes pos
          const float t0 = lane > 0 ? qs[lane - 1] : 0.f, t1 = qs[lane + 31];
          const int32_t u0 = lane > 0 ? qi[lane - 1] : 0, u1 = qi[lane + 31];
          __syncwarp();
          if (lane > pos && lane < k) qs[lane] = t0, qi[lane] = u0;
          else if (lane == pos) qs[lane] = cs, qi[lane] = ci;
          if (lane + 32 > pos && lane + 32 < k) qs[lane + 32] = t1, qi[lane + 32] = u1;
          else if (lane + 32 == pos) qs[lane + 32] = cs, qi[lane + 32] = ci;
          __syncwarp();
        }
      }
    }
    __syncthreads();  // the staging area is rewritten by the next block
  }
  // no copy of this CTA may be in flight when it exits: after a wait ran out,
  // thread 0 waits (bounded again) for every copy it started
  if (threadIdx.x == 0 && !alive)
    for (int64_t c = ndone; c < nissued; ++c)
      mbar_wait(smem_u32(&full[c & 1]), (uint32_t)((c >> 1) & 1), a.fault, kFaultSearch);
  // the lists as candidates: [q][blockIdx.x][k], empty entries as index -1
  for (int j = 0; j < 4; ++j) {
    const int ql = 4 * warp + j, q = 4 * g0 + ql;
    if (ql < 4 * ntl && q < a.nq) {
      const size_t o = ((size_t)q * a.vchunks + blockIdx.x) * k;
      for (int e = lane; e < k; e += 32) {
        a.cand_sc[o + e] = lsc[ql * kMaxK + e];
        const int32_t id = lid[ql * kMaxK + e];
        a.cand_idx[o + e] = id == INT32_MAX ? -1 : id;
      }
    }
  }
}

}  // namespace

bool tq::search_tc_supported(const tq_plan* plan, const tq_records* recs) {
  return plan->d % 128 == 0 && plan->m % 128 == 0 && recs->layout == TQ_LAYOUT_ROWS;
}

namespace {
// Codebook planes of the query table: w ±1 planes (4 with the product plane at
// w = 3), or, at w = 3, one block of centroid values.
int table_planes(const tq_plan* plan) { return plan->w == 3 ? 1 : plan->w; }
}  // namespace

size_t tq::search_tc_table_bytes(const tq_plan* plan, int nq) {
  const size_t ksteps = 2 * (size_t(table_planes(plan)) * plan->d + plan->m) / 32;
  return ksteps * size_t((nq + 3) / 4) * kFragBytes + sizeof(float) * 2 * size_t(nq) + 8 * sizeof(uint32_t);
}

int tq::search_tc_vchunks(int64_t n, int nq) {
  // as many CTAs as one wave of two per SM of a B300 (148 SMs) holds, over the
  // query blocks: every CTA then gets the same number of vector blocks, give or take one
  const int64_t qblocks = ((nq + 3) / 4 + kTilesPerCta - 1) / kTilesPerCta;
  const int64_t nblocks = (n + kRows - 1) / kRows;
  return (int)std::max<int64_t>(1, std::min<int64_t>(nblocks, 2 * 148 / qblocks));
}

tq_status tq::launch_search_tc(const tq_plan* plan, const tq_records* recs, int64_t n, int nq, const float* qt,
                               const float* st, void* table, int k, int32_t* cand_idx, float* cand_sc,
                               cudaStream_t stream) {
  if (k < 1 || k > kMaxK) return TQ_ERR_ARG;
  SearchTcArgs a{};
  a.idx = recs->idx; a.sgn = recs->sgn; a.norm = recs->norm; a.rnorm = recs->rnorm;
  a.n = n;
  a.nq = nq;
  a.d = plan->d; a.m = plan->m; a.w = plan->w;
  a.npm = plan->w == 3 ? 4 : plan->w;
  a.deq = plan->w == 3;
  a.npm_t = table_planes(plan);
  a.groups = (nq + 3) / 4;
  a.ksteps = 2 * (int64_t(a.npm_t) * a.d + a.m) / 32;
  a.centroids = plan->centroids;
  a.qt = qt; a.st = st;
  a.walsh = plan->walsh;
  a.alpha = plan->qjl_alpha;
  a.table = static_cast<__half*>(table);
  a.consts = reinterpret_cast<float*>(static_cast<uint8_t*>(table) + size_t(a.ksteps) * a.groups * kFragBytes);
  a.ctab = reinterpret_cast<uint32_t*>(a.consts + 2 * size_t(nq));
  a.k = k;
  a.vchunks = search_tc_vchunks(n, nq);
  a.cand_idx = cand_idx;
  a.cand_sc = cand_sc;
  a.fault = tq::fault_word();
  if (!a.fault) return TQ_ERR_CUDA;
  search_table_kernel<<<a.groups, kThreads, 0, stream>>>(a);
  if (launch_status() != TQ_OK) return TQ_ERR_CUDA;
  const int smem = 2 * kChunkBytes + 64 + 32 * kStagePitch * 4 + 32 * kMaxK * 8;
  auto kern = a.deq ? search_score_kernel<true> : search_score_kernel<false>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return TQ_ERR_CUDA;
  const dim3 grid((unsigned)a.vchunks, (unsigned)((a.groups + kTilesPerCta - 1) / kTilesPerCta));
  kern<<<grid, kThreads, smem, stream>>>(a);
  return launch_status();
}

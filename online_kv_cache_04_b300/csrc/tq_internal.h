// Internal helpers shared by the libturboquant translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "../../include/turboquant.h"

namespace tq {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// m = 0: stage 1 alone (no QJL rows, records without signs or residual norms)
inline bool valid_shape(int d, int m, int w) {
  return d >= 32 && d <= 1024 && d % 32 == 0 && (m == 0 || (m >= 32 && m <= 1024 && m % 32 == 0)) && w >= 1 &&
         w <= 3;
}

inline bool valid_plan(const tq_plan* p) {
  return p != nullptr && valid_shape(p->d, p->m, p->w) && p->pi && p->pi_t && p->centroids && p->bounds &&
         p->walsh && p->pi_bf16 && (p->m == 0 || (p->s_rot && p->s_rot_t && p->s_bf16));
}

// Records of a plan; without QJL rows (plan m = 0) sgn and rnorm may be NULL.
inline bool valid_records(const tq_records* r, const tq_plan* plan) {
  const bool qjl = plan->m > 0;
  if (r == nullptr || !r->idx || !r->norm || r->capacity < 0) return false;
  if (qjl && (!r->sgn || !r->rnorm)) return false;
  if (!aligned16(r->idx) || !aligned16(r->sgn) || !aligned16(r->norm) || !aligned16(r->rnorm)) return false;
  if (r->layout == TQ_LAYOUT_ROWS) return true;
  return r->layout == TQ_LAYOUT_BLOCK32 && r->capacity % 32 == 0;
}

// Bit of row t (0..31) inside a 32-row block word of TQ_LAYOUT_BLOCK32.
__host__ __device__ inline int block32_bit(int t) { return (t >> 1) + ((t & 1) << 4); }

// Status of the most recent launch on this thread.
inline tq_status launch_status() { return cudaGetLastError() == cudaSuccess ? TQ_OK : TQ_ERR_CUDA; }

inline int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
  return n;
}

// q̃ = Π q and s̃ = (S Πᵀ) q̃ for nheads query vectors of length d (tq_decode.cu).
tq_status launch_query_prep(const tq_plan* plan, const void* q, tq_dtype qd, int nheads, float* qt, float* st,
                            cudaStream_t stream);

// Log-sum-exp merge of nsplit partials [B*Hq][nsplit][2 + d + m] (reference,
// sum, acc_rot[d], acc_sgn[m]) per query head and the output
// o = Πᵀ(acc_rot + alpha·S̃ᵀ acc_sgn)/l (tq_decode.cu).
tq_status launch_decode_combine(const float* part, int B, int Hq, int nsplit, int d, int m, const float* pi_t,
                                const float* s_rot_t, float alpha, float* out, cudaStream_t stream);

// Device word of fault bits set by bounded waits (tq_quantize_tc.cu).
unsigned* fault_word();

// tcgen05 quantizer (bf16 input, d = m = 128); rows already offset.
bool quantize_tc_supported(const tq_plan* plan, tq_dtype dtype, int64_t n);
// x0 -> rows [row0, row0 + n) of out0 and, when x1 and out1 are given, x1 ->
// the same rows of out1, in one launch; for a TQ_LAYOUT_BLOCK32 output,
// row0 % 32 == 0.
tq_status quantize_tc(const tq_plan* plan, const void* x0, const void* x1, int64_t n, int64_t ld_x,
                      const tq_records* out0, const tq_records* out1, int64_t row0, cudaStream_t st);

// Tensor-core decode (tq_decode_tc.cu): d = 128, m = 128 or 0, G <= 8, values in
// TQ_LAYOUT_BLOCK32, ctx_stride % 128 == 0.  Three launches: one CTA per
// (batch, kv head) unit builds its query table (decode_tc_table_bytes(w, G, m)
// bytes, 16-byte aligned); the decode kernel does the scores, softmax and
// values and writes one partial per CTA and head ([B*Hq][smax][2 + 256]); one
// CTA per unit merges the unit's partials into out.  Each unit is cut into
// decode_tc_tpu(ctx_stride) tiles.
int64_t decode_tc_tpu(int64_t ctx_stride);
bool decode_tc_supported(const tq_plan* plan, int G, const tq_records* V, int64_t ctx_stride);
int decode_tc_ctas(int64_t units, int64_t tpu, int G);
int decode_tc_slots(int64_t units, int64_t tpu, int64_t ctas);
size_t decode_tc_table_bytes(int w, int G, int m);
// pages: NULL for contiguous units, else the page table of a paged cache
// ([B*Hkv][ctx_stride / 256] page of each 256-token tile; ctx_stride % 256 == 0).
// Fused append of the step's new keys and values (tq_decode_attention_append):
// [B*Hkv][d] each, bf16 (bf16 != 0) or fp32; ctx_len is the decode's length
// array, advanced on the device by the launch.
struct TcAppend {
  const void* k_new;
  const void* v_new;
  int bf16;
  int32_t* ctx_len;
};
tq_status launch_decode_tc(const tq_plan* plan, const void* q, tq_dtype q_dtype, const tq_records* K,
                           const tq_records* V, const int32_t* ctx_len, int B, int Hq, int Hkv, int64_t ctx_stride,
                           float scale, float* part, int smax, uint8_t* tables, float* out, cudaStream_t stream,
                           const int32_t* pages = nullptr, const TcAppend* app = nullptr);
// tq_append_kv's two launches (tq_append.cu), for caches the fused path does not take.
tq_status append_kv(const tq_plan* plan, const void* k_new, const void* v_new, tq_dtype dtype, int B, int Hkv,
                    const tq_records* K, const tq_records* V, int32_t* ctx_len, int64_t ctx_stride,
                    cudaStream_t stream, const int32_t* pages);

// SIMT quantizer over a column subset (tq_quantize.cu): element j of row r is
// x[r][cols[j]] for j < plan->d (cols: device int32); rows [out_offset,
// out_offset + n) of `out`, TQ_LAYOUT_ROWS.  Arguments already checked.
tq_status quantize_simt_cols(const tq_plan* plan, const void* x, tq_dtype dtype, int64_t n, int64_t ld_x,
                             const int32_t* cols, const tq_records* out, int64_t out_offset, cudaStream_t st);

// tcgen05 quantizer for wide vectors (tq_quantize_wide.cu): d a multiple of
// 256 up to 1024, m = d (with the plan's pieces of S) or 0, fp32 or bf16 input,
// TQ_LAYOUT_ROWS output; rows [row0, row0 + n) of `out`.
bool quantize_wide_supported(const tq_plan* plan, const tq_records* out);
tq_status quantize_wide(const tq_plan* plan, const void* x, tq_dtype dtype, int64_t n, int64_t ld_x,
                        const tq_records* out, int64_t row0, cudaStream_t st);

// 2-D tensor map over a rows x cols bf16 matrix of row stride ld elements:
// boxes of 64 columns x box_rows rows, 128-byte swizzle (tq_quantize_tc.cu).
// False if the driver's encoder is unavailable or rejects the map.
bool map_bf16_tiles(CUtensorMap* map, const void* ptr, uint64_t rows, uint64_t cols, uint64_t ld,
                    uint32_t box_rows);
// The driver's tensor-map encoder (NULL if unavailable).
typedef CUresult (*TensorMapEncoder)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                     const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                     CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
TensorMapEncoder tensor_map_encoder();

// Warp tensor-core quantizer (tq_quantize_mma.cu): d a multiple of 128 up to
// 1024, m = d or 0, fp32 or bf16 input, TQ_LAYOUT_ROWS output; rows
// [row0, row0 + n) of `out`.
bool quantize_mma_supported(const tq_plan* plan, const tq_records* out);
tq_status quantize_mma(const tq_plan* plan, const void* x, tq_dtype dtype, int64_t n, int64_t ld_x,
                       const tq_records* out, int64_t row0, cudaStream_t st);

// tcgen05 search for wide records (tq_search_wide.cu): d a multiple of 256 up to
// 1024, m = d or 0, k <= 16, records in TQ_LAYOUT_ROWS (the entry point's
// requirement for every path).  `table`:
// search_wide_table_bytes(plan, nq) bytes, 256-byte aligned.  Writes, per query,
// search_wide_lists(nq) lists of the k best (score desc, index asc; index -1
// for an empty entry) to cand_idx / cand_sc [nq][lists][k].
bool search_wide_supported(const tq_plan* plan, int k);
int search_wide_lists(int nq);
size_t search_wide_table_bytes(const tq_plan* plan, int nq);
tq_status launch_search_wide(const tq_plan* plan, const tq_records* recs, int64_t n, int nq, const float* qt,
                             const float* st, void* table, int k, int32_t* cand_idx, float* cand_sc,
                             cudaStream_t stream);

// Tensor-core search with the selection fused in (tq_search_tc.cu): d and m
// multiples of 128 (m may be 0), records in TQ_LAYOUT_ROWS, k <= 64.
// `table`: search_tc_table_bytes(plan, nq) bytes, 16-byte aligned.  Writes,
// per query, search_tc_vchunks(n, nq) lists of the k best (score desc, index
// asc; index -1 for an empty entry) to cand_idx / cand_sc [nq][vchunks][k].
bool search_tc_supported(const tq_plan* plan, const tq_records* recs);
size_t search_tc_table_bytes(const tq_plan* plan, int nq);
int search_tc_vchunks(int64_t n, int nq);
tq_status launch_search_tc(const tq_plan* plan, const tq_records* recs, int64_t n, int nq, const float* qt,
                           const float* st, void* table, int k, int32_t* cand_idx, float* cand_sc,
                           cudaStream_t stream);

}  // namespace tq

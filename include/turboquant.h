/*
 * libturboquant -- TurboQuant's online KV-vector quantizer and decode
 * attention over the compressed cache, for NVIDIA B300 (sm_103a).
 *
 * Plain C ABI: pointers and sizes only.  Sources of each operation are cited
 * by page title and section:
 *   [memory-wall]  "谷歌TurboQuant如何绕过内存墙？重新审视它的技术突破"
 *                  (youleyou), §2 "TurboQuant到底做了什么？", stage 1 and
 *                  stage 2.
 *   [efficiency]   "TurboQuant 与 AI 效率革命：当旧数学遇到新智能"
 *                  (mini-blog), §三 (JL transform, asymmetric estimator, bit
 *                  accounting) and §四 (three-step pipeline, H100 timings).
 *   [video]        "TurboQuant压缩效果" (douyin transcripts): fused operators
 *                  that read packed 32-bit words and decode in registers.
 *   [yeyu]         yeyulingfeng article: codebook computed once, no
 *                  calibration data.
 *
 * Conventions shared by every call
 *   - Ownership: the caller owns every buffer.  The library never allocates
 *     or frees memory and may be called concurrently on different streams
 *     with disjoint outputs.  Its state is one device word of fault bits
 *     (see tq_fault_flags) and the fixed scratch array of
 *     tq_decode_attention_noalloc, with that array's per-device address.
 *   - Device calls are asynchronous on the given stream (NULL = legacy
 *     default stream).  Argument errors are detected on the host and
 *     returned before anything is launched; a failed launch returns
 *     TQ_ERR_CUDA.  Device pointers must be 16-byte aligned.
 *   - Shapes: d (head dim) and m (QJL rows) are multiples of 32 in
 *     [32, 1024]; w = b - 1 index bits per coordinate, w in {1, 2, 3}
 *     (b = 2, 3, 4 total bits).
 *   - Stored record of one vector (SoA, see tq_records): w*d/32 index words
 *     (bit-planes: word p*(d/32)+k holds bit p of idx[32k+i] at bit i),
 *     m/32 sign words (bit i of word k = 1 <-> sign(S r)[32k+i] = +1), the
 *     fp32 norm ||x|| and the fp32 residual norm ||r||.
 */
#ifndef TURBOQUANT_H
#define TURBOQUANT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  TQ_OK = 0,
  TQ_ERR_ARG = -1,          /* invalid argument (size, pointer, alignment)   */
  TQ_ERR_UNSUPPORTED = -2,  /* valid but not supported by this build         */
  TQ_ERR_CUDA = -3,         /* a CUDA runtime call or launch failed          */
  TQ_ERR_WORKSPACE = -4,    /* workspace smaller than the size query says    */
  TQ_ERR_NUMERIC = -5       /* setup iteration failed to converge            */
} tq_status;

typedef enum { TQ_F32 = 0, TQ_BF16 = 1 } tq_dtype;

/* Same object as cudaStream_t, without including the CUDA headers. */
typedef struct CUstream_st* tq_stream;

/* ------------------------------------------------------------------ setup
 * Host-only, float64, deterministic, not timed.  Run once per shape; the
 * outputs are reused for any model ([yeyu]: computed once, no calibration).
 */

/* Random rotation Π, [memory-wall] §2 stage 1 / [efficiency] §四 Step 1.
 * G = d x d iid N(0,1) from SplitMix64(seed) + Box-Muller, row-major fill;
 * G = QR (Householder); Π = Q diag(sign diag R) (Haar).  Convention u = Π x.
 * pi: host, d*d doubles, row-major, written.  Errors: TQ_ERR_ARG if d is not
 * in [2, 4096] or pi is NULL. */
tq_status tq_make_rotation(int d, uint64_t seed, double* pi);

/* Lloyd-Max codebook with 2^w levels for the post-rotation coordinate law
 * f_d(x) ∝ (1-x²)^((d-3)/2) on [-1, 1], [memory-wall] §2 stage 1.
 * centroids: host, 2^w doubles ascending; bounds: host, 2^w-1 doubles
 * ascending (midpoints); mse_per_coord: host, 1 double, may be NULL.
 * Errors: TQ_ERR_ARG (d < 3, w not in [1, 4], NULL outputs),
 * TQ_ERR_NUMERIC (no convergence). */
tq_status tq_make_codebook(int d, int w, double* centroids, double* bounds, double* mse_per_coord);

/* QJL matrix, [efficiency] §三 "JL 变换" and §四 Step 3: S = m x d iid
 * N(0,1) from SplitMix64(seed), row-major.  If pi and s_rot are both
 * non-NULL, also writes s_rot = S Πᵀ (m x d), so that S r = s_rot (Π r).
 * S: host m*d doubles, written.  Errors: TQ_ERR_ARG. */
tq_status tq_make_qjl(int m, int d, uint64_t seed, const double* pi, double* S, double* s_rot);

/* ------------------------------------------------------------------ plan
 * Device copies of the setup tables, laid out for the kernels.  All
 * pointers live inside one caller-owned device buffer of tq_plan_bytes().
 */
typedef struct tq_plan {
  int d, m, w;
  float qjl_alpha;          /* √(π/2)/m                                     */
  const float* pi;          /* [d][d]  Π, row-major (u = Π x)               */
  const float* pi_t;        /* [d][d]  Πᵀ                                   */
  const float* s_rot;       /* [m][d]  S Πᵀ                                 */
  const float* s_rot_t;     /* [d][m]  (S Πᵀ)ᵀ                               */
  const float* centroids;   /* [2^w]                                        */
  const float* bounds;      /* [2^w - 1]                                    */
  const float* walsh;       /* [2^w] Walsh coefficients of the codebook    */
  const uint16_t* pi_bf16;  /* [2][d][d] bf16 hi/lo split of Π              */
  const uint16_t* s_bf16;   /* [2][m][d] bf16 hi/lo split of S Πᵀ           */
  /* The same bf16 pieces in warp-MMA operand order, for d a multiple of 128
   * (NULL otherwise): piece p, K-step k (16 columns), row group f (8 rows), lane
   * l = 4g + t hold M[8f + g][16k + 2t + {0, 1, 8, 9}] at 4 consecutive
   * halves ((p·(K/16) + k)·(rows/8) + f)·32 + l, for M = Π and M = S Πᵀ. */
  const uint16_t* pi_frag;  /* [2][d/16][d/8][32][4]                        */
  const uint16_t* s_frag;   /* [2][d/16][m/8][32][4]                        */
  /* bf16 hi/lo split of S itself (= (S Πᵀ) Π), for d a multiple of 256 with
   * m = d (NULL otherwise): the wide tensor-core quantizer forms the signs as
   * S x / n - (S Πᵀ) c[idx] = S r / n without holding the residual. */
  const uint16_t* s_x_bf16; /* [2][m][d]                                    */
} tq_plan;

/* Device bytes needed by tq_plan_init for (d, m, w); 0 if unsupported.
 * m = 0 selects stage 1 alone ([memory-wall] §2 stage 1: the rotation and
 * the MSE-optimal codebook with all w bits, no QJL rows): records then hold
 * only indices and norms (their sgn and rnorm may be NULL), scores are
 * ||k|| <Π q, c[idx]> and values ||v|| Πᵀ c[idx].  At d = 128 such plans run
 * on the tensor-core quantizer and decode like the two-stage ones. */
size_t tq_plan_bytes(int d, int m, int w);

/* Fill `plan` and the device buffer `dev` (bytes >= tq_plan_bytes) from the
 * host float64 tables of tq_make_rotation / tq_make_qjl / tq_make_codebook
 * (s_rot may be NULL when m = 0).
 * Copies are issued on `stream`; the host tables may be released once the
 * stream has passed this call.  walsh[mask] holds the coefficients of the
 * expansion c[idx] = Σ_mask walsh[mask] · Π_{p in mask} (2·bit_p(idx) - 1)
 * (exact; only odd-size masks are non-zero for a symmetric codebook), which
 * lets the decode kernels score ±1 bit-planes directly.
 * Errors: TQ_ERR_ARG (shape, NULL, bytes too small), TQ_ERR_CUDA. */
tq_status tq_plan_init(tq_plan* plan, int d, int m, int w, const double* pi, const double* s_rot,
                       const double* centroids, const double* bounds, void* dev, size_t bytes,
                       tq_stream stream);

/* ------------------------------------------------------------------ records
 * Compressed vectors, structure of arrays in device memory.  KV caches use
 * row (b*Hkv + h)*ctx_stride + t.  norm[i] and rnorm[i] belong to row i in
 * both layouts; the bit words are laid out by `layout`:
 *
 * TQ_LAYOUT_ROWS (0, any capacity): row i owns idx[i*(w*d/32) ...] and
 *   sgn[i*(m/32) ...], with the bit-plane words described at the top.
 *   Keys, search sets, and any cache read by vector.
 * TQ_LAYOUT_BLOCK32 (1, capacity a multiple of 32): rows are grouped in
 *   blocks of 32 (block r/32).  Block k owns idx[k*w*d ...], where word
 *   p*d + j holds bit p of idx[j] of the block's 32 rows, and sgn[k*m ...],
 *   where word j holds σ[j] of the 32 rows.  Row t of the block sits at bit
 *   t/2 + 16*(t%2) (even rows in the low half-word, odd rows in the high
 *   half).  The same bytes as layout 0, transposed so that one word carries
 *   one coordinate of 32 consecutive tokens: the layout the value cache
 *   needs for the tensor-core attention-times-values contraction, which sums
 *   over tokens.  Writers of one block (tq_quantize appends) merge into it,
 *   so calls that write the same block must be ordered on one stream.
 */
typedef enum { TQ_LAYOUT_ROWS = 0, TQ_LAYOUT_BLOCK32 = 1 } tq_layout;

typedef struct tq_records {
  uint32_t* idx;
  uint32_t* sgn;
  float* norm;
  float* rnorm;
  int64_t capacity;
  int32_t layout;  /* tq_layout */
} tq_records;

/* ------------------------------------------------------------------ quantize
 * Online quantization of n vectors, [memory-wall] §2 (stages 1 and 2) and
 * [efficiency] §四 (three-step pipeline): n = ||x||, u = Π x / n,
 * idx_j = #{k: bounds_k < u_j}, ρ = u - c[idx] (= Π r / n), ||r|| = n ||ρ||,
 * σ = sign(S r) = sign(s_rot ρ) with sign(0) = +1; packed as described
 * above.  A zero vector gives u = 0, ||r|| = 0 and all σ = +1.
 * x: device, n rows of d elements of `dtype`, row stride ld_x elements
 * (>= d, multiple of 8).  Writes rows [out_offset, out_offset + n) of
 * `out` (online append into a preallocated cache).  n = 0 is a no-op.
 * Errors: TQ_ERR_ARG (n < 0, rows beyond capacity, NULL, misaligned),
 * TQ_ERR_CUDA. */
tq_status tq_quantize(const tq_plan* plan, const void* x, tq_dtype dtype, int64_t n, int64_t ld_x,
                      const tq_records* out, int64_t out_offset, tq_stream stream);

/* tq_quantize of two inputs of the same shape -- the key and value rows of
 * the same tokens -- in one call: x0 -> rows [out_offset, out_offset + n) of
 * out0 and x1 -> the same rows of out1 (each output in its own layout).
 * Results are those of the two tq_quantize calls; where the tensor-core
 * quantizer applies (bf16, d = m = 128, and out_offset % 32 == 0 for a block
 * layout output) both run in one launch, which starts and drains its
 * pipeline once.  Same arguments, ownership and errors as tq_quantize, for
 * each of the two; out0 and out1 must not overlap. */
tq_status tq_quantize_pair(const tq_plan* plan, const void* x0, const void* x1, tq_dtype dtype, int64_t n,
                           int64_t ld_x, const tq_records* out0, const tq_records* out1, int64_t out_offset,
                           tq_stream stream);

/* The online step of a decode loop ([efficiency] §四: quantize every new
 * vector as it arrives; [memory-wall] §2): quantize the new key and value of
 * every (batch row b, kv head h) exactly as tq_quantize does and store them
 * at token t = ctx_len[b] of their caches (row (b*Hkv + h)*ctx_stride + t,
 * merged into its 32-row block in TQ_LAYOUT_BLOCK32), then add one to
 * ctx_len[b] on the device, stream-ordered after every read of it.
 * k_new, v_new: device [B][Hkv][d] of dtype, rows contiguous.  K, V: distinct
 * caches (sharing a word array is TQ_ERR_ARG) of B*Hkv*ctx_stride rows or more (ctx_stride a multiple of 32 when
 * either is in TQ_LAYOUT_BLOCK32).  ctx_len: device int32 [B], read and
 * advanced.  A batch row whose cache is full (ctx_len[b] >= ctx_stride) or
 * whose length is negative is neither written nor advanced, and fault bit 3
 * is set.  Two launches.
 * Errors: TQ_ERR_ARG (shapes, capacity, NULL, misaligned), TQ_ERR_CUDA. */
tq_status tq_append_kv(const tq_plan* plan, const void* k_new, const void* v_new, tq_dtype dtype, int B, int Hkv,
                       const tq_records* K, const tq_records* V, int32_t* ctx_len, int64_t ctx_stride,
                       tq_stream stream);

/* ------------------------------------------------------------------ decode
 * One decode step of GQA softmax attention over compressed K/V caches.
 * Per query head g (kv head h = g / (Hq/Hkv)) and token t < ctx_len[b]:
 *   s_{g,t} = scale * ( ||k_t|| <Π q_g, c[idx_t]>
 *                       + √(π/2)/m ||r_t|| <S q_g, σ_t> )
 * ([efficiency] §三 asymmetric estimator on the residual, [memory-wall] §2
 * stage 2); p = softmax_t(s); the value side is accumulated in the rotated
 * domain, acc = Σ_t p_t (||v_t|| c[idx_t] + √(π/2)/m ||r_t|| s_rotᵀ σ_t),
 * and o_g = Πᵀ acc -- a single unrotation, with no dequantized copy
 * written anywhere ([video]: decode in registers while reading).
 * q: device [B][Hq][d] of q_dtype.  ctx_len: device int32 [B], each in
 * [0, ctx_stride] (a row with ctx_len 0 outputs zeros).  scale <= 0 means
 * 1/√d.  out: device fp32 [B][Hq][d].  workspace: device, at least
 * tq_decode_workspace_size() bytes for the same (B, Hq, Hkv, ctx_stride).
 * Errors: TQ_ERR_ARG (Hq % Hkv, sizes, capacity < B*Hkv*ctx_stride, NULL),
 * TQ_ERR_WORKSPACE, TQ_ERR_CUDA. */
tq_status tq_decode_workspace_size(const tq_plan* plan, int B, int Hq, int Hkv, int64_t ctx_stride,
                                   size_t* bytes);
tq_status tq_decode_attention(const tq_plan* plan, const void* q, tq_dtype q_dtype, int B, int Hq, int Hkv,
                              const tq_records* K, const tq_records* V, const int32_t* ctx_len,
                              int64_t ctx_stride, float scale, float* out, void* workspace,
                              size_t ws_bytes, tq_stream stream);

/* Decode attention without a caller workspace, for callers that cannot
 * allocate device memory (graph captures that forbid allocation, embedded
 * runtimes with memory fixed at start-up, plugins whose host owns the
 * allocator).  The sources describe no counterpart: this is a deployment variant of
 * tq_decode_attention, with the same arguments minus the workspace and the
 * same results.
 * Scratch: one array of TQ_NOALLOC_SCRATCH_BYTES (8 MiB) compiled into the
 * library, resident on every GPU that loads it until the process exits.  The
 * first call on a device looks up the array's device address (make that first
 * call before any stream capture) and later calls reuse it for the life of
 * the process; a cudaDeviceReset of that device invalidates it, so do not
 * call this entry point on a device after resetting it.  No call allocates
 * or frees memory.  All
 * calls share the array: calls whose GPU work overlaps race on it, so order
 * them on one stream.  Nothing in the array needs clearing between calls.
 * Errors: as tq_decode_attention; TQ_ERR_WORKSPACE when the shape needs more
 * scratch than TQ_NOALLOC_SCRATCH_BYTES (tq_decode_workspace_size tells). */
#define TQ_NOALLOC_SCRATCH_BYTES ((size_t)8 << 20)
tq_status tq_decode_attention_noalloc(const tq_plan* plan, const void* q, tq_dtype q_dtype, int B, int Hq, int Hkv,
                                      const tq_records* K, const tq_records* V, const int32_t* ctx_len,
                                      int64_t ctx_stride, float scale, float* out, tq_stream stream);

/* Paged caches (a decode loop whose sequences grow by pages instead of each
 * owning one contiguous stretch of ctx_stride rows; "谷歌TurboQuant如何绕过
 * 内存墙？" §2: the quantizer is online, one vector at a time).  Token t of
 * (batch row b, kv head h) lives at record row pages[(b*Hkv + h)*max_pages +
 * t/256]*256 + t%256: a page is 256 consecutive rows (eight 32-row blocks of
 * TQ_LAYOUT_BLOCK32) starting at a multiple of 256, and each sequence holds
 * up to max_pages of them, in any order.  pages: device int32
 * [B*Hkv][max_pages], 16-byte aligned; an entry must lie in
 * [0, capacity/256) of both caches -- an entry outside is read as page 0 and
 * sets fault bit 4 (the outputs of that call are then undefined).
 * Decode: as tq_decode_attention with ctx_stride = 256*max_pages (workspace
 * from tq_decode_workspace_size with that ctx_stride); results equal those of
 * the contiguous call on the same tokens.  Append: as tq_append_kv, the new
 * token at position ctx_len[b] of its sequence. */
tq_status tq_decode_attention_paged(const tq_plan* plan, const void* q, tq_dtype q_dtype, int B, int Hq, int Hkv,
                                    const tq_records* K, const tq_records* V, const int32_t* ctx_len,
                                    const int32_t* pages, int max_pages, float scale, float* out, void* workspace,
                                    size_t ws_bytes, tq_stream stream);
tq_status tq_append_kv_paged(const tq_plan* plan, const void* k_new, const void* v_new, tq_dtype dtype, int B,
                             int Hkv, const tq_records* K, const tq_records* V, int32_t* ctx_len,
                             const int32_t* pages, int max_pages, tq_stream stream);

/* A whole decode step with the online append fused in ([memory-wall] §2:
 * the quantizer runs per vector as tokens arrive; [efficiency] §四): the new
 * key and value of every (b, h) are quantized exactly as tq_append_kv does
 * and stored at token ctx_len[b], attention then runs over ctx_len[b] + 1
 * tokens as tq_decode_attention does, and ctx_len[b] is advanced on the
 * device.  On the tensor-core path (as tq_decode_attention's) the append
 * happens inside the decode's own launches -- the per-(b, h) table kernel
 * writes the new rows before the decode kernel copies any tile and the merge
 * kernel advances ctx_len -- so a step is one call and no extra launch;
 * other caches run tq_append_kv's two launches first.  Arguments as
 * tq_append_kv (k_new, v_new, kv_dtype, ctx_len, read and advanced) and
 * tq_decode_attention (q, out, workspace of tq_decode_workspace_size with
 * this ctx_stride); pages: NULL for contiguous caches, else the page table of
 * tq_decode_attention_paged ([B*Hkv][ctx_stride / 256], ctx_stride a multiple
 * of 256).  A row whose cache is full or whose length is negative is neither
 * written nor advanced (fault bit 3) and attends over its ctx_len[b] tokens.
 * Errors: those of tq_append_kv and tq_decode_attention. */
tq_status tq_decode_attention_append(const tq_plan* plan, const void* q, tq_dtype q_dtype, const void* k_new,
                                     const void* v_new, tq_dtype kv_dtype, int B, int Hq, int Hkv,
                                     const tq_records* K, const tq_records* V, int32_t* ctx_len, int64_t ctx_stride,
                                     const int32_t* pages, float scale, float* out, void* workspace,
                                     size_t ws_bytes, tq_stream stream);

/* Attention logits alone (the quantity the H100 timings of [efficiency] §四
 * and [memory-wall] §2 measure): scores[b][g][t] = s_{g,t} as above for
 * t < ctx_len[b]; entries t >= ctx_len[b] are left untouched.
 * scores: device fp32 [B][Hq][ctx_stride].  workspace as for
 * tq_decode_attention.  Errors as above. */
tq_status tq_decode_scores(const tq_plan* plan, const void* q, tq_dtype q_dtype, int B, int Hq, int Hkv,
                           const tq_records* K, const int32_t* ctx_len, int64_t ctx_stride, float scale,
                           float* scores, void* workspace, size_t ws_bytes, tq_stream stream);

/* ------------------------------------------------------------------ split
 * Outlier-channel split precision ("TurboQuant压缩效果": the 128 channels of a
 * head split, the few outlier channels quantized one bit higher than the
 * rest -- the 2.5- and 3.5-bit settings, the label being the average over
 * the channels).  perm: device int32 [d], a permutation of the head's d
 * channels: perm[0 .. d_o) are the outlier channels, perm[d_o .. d) the
 * regular ones (fixed per head, chosen by the caller, e.g. the channels of
 * largest mean square).  Each side is its own instance with its own plan:
 * plan_o with d = d_o channels and w = b bits of MSE indices (b + 1 total
 * bits), plan_r with d = d - d_o and w = b - 1 (b total bits), both with
 * QJL rows (m > 0), each side at most 128 channels.  Records of each side are
 * TQ_LAYOUT_ROWS, one row per vector as for tq_quantize.  Bits per
 * coordinate (indices and signs): b + d_o/d, e.g. 2.5 for b = 2, d_o = d/2.
 */

/* Quantize n vectors of d = plan_o->d + plan_r->d channels: the channels
 * perm[0 .. d_o) of each row through plan_o into out_o, the rest through
 * plan_r into out_r, rows [out_offset, out_offset + n) of both.  x: device,
 * row stride ld_x elements (>= d, multiple of 8).  Two launches.
 * Errors: TQ_ERR_ARG (shapes, capacity, NULL, misaligned, a record set not in
 * TQ_LAYOUT_ROWS), TQ_ERR_CUDA. */
tq_status tq_quantize_split(const tq_plan* plan_o, const tq_plan* plan_r, const int32_t* perm, const void* x,
                            tq_dtype dtype, int64_t n, int64_t ld_x, const tq_records* out_o,
                            const tq_records* out_r, int64_t out_offset, tq_stream stream);

/* Decode attention over split records: the score of a key is the sum of the
 * two sides' estimators (the inner product splits over the channel sets; the
 * query is split by perm_k, the keys' permutation), one softmax over those
 * sums, and the output carries each side's unrotated value sum at its own
 * channels of perm_v (the values' permutation: the outlier channels of keys
 * and values differ).  Other arguments as tq_decode_attention (q: device
 * [B][Hq][d], out: device fp32 [B][Hq][d], scale <= 0 means 1/√d), with both
 * sides' key and value records (row (b*Hkv + h)*ctx_stride + t in each), at
 * most 8 query heads per kv head.  Three launches (query prep, context
 * splits, combine).
 * Errors: TQ_ERR_ARG, TQ_ERR_WORKSPACE, TQ_ERR_CUDA. */
tq_status tq_decode_split_workspace_size(const tq_plan* plan_o, const tq_plan* plan_r, int B, int Hq, int Hkv,
                                         int64_t ctx_stride, size_t* bytes);
tq_status tq_decode_attention_split(const tq_plan* plan_o, const tq_plan* plan_r, const int32_t* perm_k,
                                    const int32_t* perm_v, const void* q,
                                    tq_dtype q_dtype, int B, int Hq, int Hkv, const tq_records* K_o,
                                    const tq_records* K_r, const tq_records* V_o, const tq_records* V_r,
                                    const int32_t* ctx_len, int64_t ctx_stride, float scale, float* out,
                                    void* workspace, size_t ws_bytes, tq_stream stream);

/* ------------------------------------------------------------------ polar
 * PolarQuant's recursive polar stage as an alternative first stage, then the
 * same 1-bit QJL stage on the residual ("TurboQuant 与 AI 效率革命" §二
 * "突破：极坐标" and §四; "TurboQuant压缩效果": 4 bits at the first level,
 * 2 at later ones).  A rotated vector u = Π x (d a power of two) becomes one
 * radius and d - 1 angles: level 1 pairs (u_2i, u_2i+1) into a radius and
 * atan2(u_2i+1, u_2i) in [0, 2π); level l >= 2 pairs the level l-1 radii
 * (a, b) into sqrt(a² + b²) and atan2(b, a) in [0, π/2].  Level-1 angles are
 * uniform and take 2^b1 equal cells with midpoint centroids; a level-l angle
 * follows the law ∝ sin^(k-1)(2ψ), k = 2^(l-1), with mean π/4 ("TurboQuant 与
 * AI 效率革命" §二) and takes the Lloyd-Max codebook of that law at b bits.
 * Shapes: d a power of two in [4, 256], m a multiple of 32 in [32, 256],
 * b1 and b in {1, 2, 4}.
 */

/* Angle codebooks, float64, host.  centroids: 2^b1 level-1 values, then
 * 2^b per level for levels 2 .. log2(d); bounds: 2^b1 - 1, then 2^b - 1 per
 * level (ascending within each level).  Errors: TQ_ERR_ARG, TQ_ERR_NUMERIC. */
tq_status tq_make_polar_codebooks(int d, int b1, int b, double* centroids, double* bounds);

/* 32-bit index words of one polar record: the d/2 level-1 codes (b1 bits)
 * packed 32/b1 to a word, code i at bits b1·(i mod 32/b1) of word
 * i / (32/b1) ("TurboQuant压缩效果": eight 4-bit numbers in one 32-bit word),
 * then from the next word the codes of levels 2, 3, ... in that order, b bits
 * each, packed the same way.  0 for an unsupported shape. */
int tq_polar_index_words(int d, int b1, int b);

typedef struct tq_polar_plan {
  int d, m, b1, b;
  float qjl_alpha;          /* √(π/2)/m                                     */
  const float* pi;          /* [d][d]  Π                                    */
  const float* pi_t;        /* [d][d]  Πᵀ                                   */
  const float* s_rot;       /* [m][d]  S Πᵀ                                 */
  const float* s_rot_t;     /* [d][m]                                       */
  const float* tables;      /* [levels][3][16]: cos, sin of the centroids, bounds */
} tq_polar_plan;

/* Device bytes of a polar plan (0 if unsupported), and its initialisation
 * from tq_make_rotation, tq_make_qjl (s_rot) and tq_make_polar_codebooks
 * (one caller-owned device buffer; the copy completes before the call
 * returns).  Errors: TQ_ERR_ARG, TQ_ERR_CUDA. */
size_t tq_polar_plan_bytes(int d, int m, int b1, int b);
tq_status tq_polar_plan_init(tq_polar_plan* plan, int d, int m, int b1, int b, const double* pi,
                             const double* s_rot, const double* centroids, const double* bounds, void* dev,
                             size_t bytes, tq_stream stream);

/* Quantize n vectors: rotate, transform, bucketize every angle with its
 * level's codebook (a tie goes to the lower cell), rebuild ũ from the
 * centroids and the norm, and take σ = sign(S r), ||r|| for r = x - Πᵀũ.
 * out: TQ_LAYOUT_ROWS records with tq_polar_index_words(d, b1, b) index words
 * per row, m/32 sign words, norm = ||x|| and rnorm = ||r||, rows
 * [out_offset, out_offset + n).  x: device, row stride ld_x (>= d, multiple
 * of 8).  Errors: TQ_ERR_ARG, TQ_ERR_CUDA. */
tq_status tq_quantize_polar(const tq_polar_plan* plan, const void* x, tq_dtype dtype, int64_t n, int64_t ld_x,
                            const tq_records* out, int64_t out_offset, tq_stream stream);

/* Decode attention over polar records, as tq_decode_attention: score of key
 * t = scale·(⟨Π q, ũ_t⟩ + √(π/2)/m ||r_t|| ⟨S q, σ_t⟩), softmax, values
 * accumulated in the rotated domain, one unrotation.  At most 8 query heads
 * per kv head.  Three launches (query prep, context splits, combine).
 * Errors: TQ_ERR_ARG, TQ_ERR_WORKSPACE, TQ_ERR_CUDA. */
tq_status tq_decode_polar_workspace_size(const tq_polar_plan* plan, int B, int Hq, int Hkv, int64_t ctx_stride,
                                         size_t* bytes);
tq_status tq_decode_attention_polar(const tq_polar_plan* plan, const void* q, tq_dtype q_dtype, int B, int Hq,
                                    int Hkv, const tq_records* K, const tq_records* V, const int32_t* ctx_len,
                                    int64_t ctx_stride, float scale, float* out, void* workspace, size_t ws_bytes,
                                    tq_stream stream);

/* ------------------------------------------------------------------ search
 * Inner-product top-k over n compressed vectors ([video] / [memory-wall]:
 * vector search engines): score_i = ||x_i|| <Π q, c[idx_i]> + √(π/2)/m
 * ||r_i|| <S q, σ_i>, k largest in descending order, equal scores -> lower
 * index.  q: device [nq][d] of q_dtype; idx_out: device int32 [nq][k];
 * score_out: device fp32 [nq][k]; 1 <= k <= 64.  When k > n, ranks n .. k-1
 * hold index -1 and score -inf.
 * Errors: TQ_ERR_ARG, TQ_ERR_WORKSPACE, TQ_ERR_CUDA. */
tq_status tq_search_workspace_size(const tq_plan* plan, int nq, int64_t n, int k, size_t* bytes);
tq_status tq_search_topk(const tq_plan* plan, const void* q, tq_dtype q_dtype, int nq, const tq_records* recs,
                         int64_t n, int k, int32_t* idx_out, float* score_out, void* workspace,
                         size_t ws_bytes, tq_stream stream);

/* Fault bits set on the device by kernels whose pipeline waits are bounded
 * (bit 0: a tensor-core quantize wait ran out of its bound, a few seconds;
 * bit 1: a tensor-core decode wait; bit 2: a tensor-core search wait; the
 * outputs of that launch are then undefined.  Bit 3: tq_append_kv met a
 * full cache or a negative length and skipped that batch row; bit 4: a
 * page-table entry outside the record arrays).  Kernels
 * never spin forever: they set the bit and finish.  Copies the word to *flags (synchronous) and clears it
 * when reset != 0.  Errors: TQ_ERR_ARG (NULL), TQ_ERR_CUDA. */
tq_status tq_fault_flags(uint32_t* flags, int reset);

/* Human-readable name of a status code (static string). */
const char* tq_status_str(tq_status s);

#ifdef __cplusplus
}
#endif

#endif /* TURBOQUANT_H */

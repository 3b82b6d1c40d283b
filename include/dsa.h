/*
 * dsa.h - C ABI of the GB300 (sm_103a) DSA attention layer group with
 * IndexShare.
 *
 * The method (GLM-5.2 pages):
 *  - "GLM-5.2 / 总览", config table (@tbl-glm52-config): 64 MLA heads, QK head
 *    dim 256 (NoPE 192 + RoPE 64), per-token per-layer KV = 512-d latent plus
 *    64-d RoPE key (1152 B in bf16); IndexShare indexer 32 heads x 128 dims,
 *    top-K = 2048, shared every 4 layers.  Sub-doc index row 02: indexer with
 *    ReLU and an "FP8 per-block + Hadamard" variant.
 *  - "GLM-5.2 架构深度拆解" CH 2.2: an F (full) layer scores every earlier token
 *    and keeps the top 2048 as the sparse set of its attention; an S (shared)
 *    layer skips the indexer and reuses the nearest F layer's indices; CH 2.4:
 *    the indices are written at F and read at S through an outer buffer.
 *  - "GLM-5 -> 5.1 -> 5.2" section 10: indexer once per layer group, shared
 *    indices written to a buffer reused within the group, each layer gathers
 *    the selected entries from its own K/V cache, then sparse attention.
 *  - Beyond the layer group itself: paged caches (CH 4.4, PagedAttention over
 *    the compressed MLA KV), FP8 KV latent rows (config table and glossary
 *    "KV8 / KV FP8"), the indexer cache append with interleaved RoPE (CH 7.1)
 *    and a hot/cold KV with a GPU hot buffer in front of a host store
 *    (glossary "HiSparse").
 *
 * Conventions for every entry point:
 *  - Pointers named d_* and every tensor argument are DEVICE pointers owned by
 *    the caller; the library allocates and frees nothing.  Host structs
 *    (dsa_batch_t, dsa_group_t, dsa_hot_t, dsa_hot_group_t) are read during
 *    the call only; a hot/cold cold store is page-locked HOST memory.
 *  - Calls are asynchronous on `stream`: they validate their host-side
 *    arguments, enqueue kernels and return.  Argument errors are reported
 *    synchronously before anything is enqueued.  Errors only a kernel can see
 *    (an index outside [-1, q_pos], inconsistent batch arrays, a bounded wait
 *    that ran out, a hot buffer without room for a step's misses) are OR-ed
 *    into the status word at the head of the workspace; dsa_status_fetch()
 *    reads and clears it.
 *  - Nothing falls back: an unsupported shape or dtype returns
 *    DSA_ERR_UNSUPPORTED.  No exception crosses the ABI.
 *  - bf16 tensors are IEEE bfloat16 bit patterns; fp8 tensors are OCP E4M3
 *    codes.  All layouts are row-major and densely packed.
 */
#ifndef DSA_H_
#define DSA_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define DSA_API __attribute__((visibility("default")))
#else
#define DSA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* dsa_stream_t; /* a cudaStream_t; NULL = legacy default stream */

typedef enum {
  DSA_OK = 0,
  DSA_ERR_INVALID_ARG = 1, /* null pointer, bad size, misaligned pointer, bad layer string */
  DSA_ERR_UNSUPPORTED = 2, /* a shape / dtype outside what the kernels implement */
  DSA_ERR_WORKSPACE = 3,   /* workspace null or smaller than the matching *_workspace_size */
  DSA_ERR_CUDA = 4,        /* a CUDA runtime call failed (see dsa_last_error_string) */
  DSA_ERR_TIMEOUT = 5,     /* device: a bounded wait inside a kernel ran out */
  DSA_ERR_DEVICE_INDEX = 6, /* device: an index outside [-1, q_pos], or bad batch arrays */
  DSA_ERR_HOT_OVERFLOW = 7  /* device: a sequence selected more distinct positions than its
                               hot buffer has slots free at this step */
} dsa_status_t;

typedef enum { DSA_BF16 = 0, DSA_FP8_E4M3 = 1 } dsa_dtype_t;

/* Fixed widths of the method (config table of "GLM-5.2 / 总览"). */
enum {
  DSA_INDEX_HEADS = 32, /* indexer heads */
  DSA_INDEX_DIM = 128,  /* indexer width; one shared 128-d key per position */
  DSA_LATENT = 512,     /* MLA KV latent */
  DSA_ROPE = 64,        /* MLA RoPE key */
  DSA_KV_ROW = 576,     /* latent + RoPE key, one cache row */
  DSA_KV_ROW_BYTES = 1152,     /* bytes of a bf16 KV row */
  DSA_KV_ROW_BYTES_FP8 = 656,  /* bytes of an FP8 KV row (dsa_kv_fp8_quantize) */
  DSA_HOT_MAX_SLOTS = 16384    /* largest hot buffer per sequence (dsa_hot_t) */
};

/*
 * Batch layout shared by every call.  Queries are rows 0..num_q-1; the rows
 * of sequence b are [q_start[b], q_start[b+1]).  Query t sits at absolute
 * position q_pos[t] of its sequence and sees positions 0..q_pos[t] (causal,
 * itself included).  Every per-layer cache (indexer keys, KV latent) stores
 * position s of sequence b at row seq_row0[b] + s (contiguous layout), or,
 * when block_table is not NULL (paged layout: caches allocated in blocks of
 * block_rows rows, a sequence's blocks anywhere in the cache), at row
 *   block_table[b * blocks_per_seq + s / block_rows] * block_rows + s % block_rows.
 * The paged layout is the block-table cache of PagedAttention, which pages
 * the compressed 512-d MLA KV ("GLM-5.2 架构深度拆解" CH 4.4); the pages fix no
 * block format, and this is its plainest form.
 *   num_seqs  >= 1
 *   num_q     >= 0 (0 is a no-op)
 *   max_q     >= the largest query count of one sequence
 *   max_len   capacity of a score row: a multiple of 128 and > every q_pos
 *   q_start   device int32 [num_seqs + 1], non-decreasing, q_start[0] = 0,
 *             q_start[num_seqs] = num_q
 *   q_pos     device int32 [num_q]
 *   seq_row0  device int64 [num_seqs] (contiguous layout; NULL allowed when paged)
 *   block_table     device int32 [num_seqs * blocks_per_seq] block ids, or NULL
 *   block_rows      paged layout: rows per block, a power of two >= 128 (so
 *                   that a 128-position key tile never straddles blocks)
 *   blocks_per_seq  paged layout: table row stride; blocks_per_seq * block_rows
 *                   must cover max_len
 * A kernel that finds q_start / q_pos inconsistent with these sizes, or a
 * negative block id for a visible position, skips the affected rows and
 * raises DSA_ERR_DEVICE_INDEX in the status word.
 */
typedef struct {
  int32_t num_seqs;
  int32_t num_q;
  int32_t max_q;
  int32_t max_len;
  const int32_t* q_start;
  const int32_t* q_pos;
  const int64_t* seq_row0;
  const int32_t* block_table;
  int32_t block_rows;
  int32_t blocks_per_seq;
} dsa_batch_t;

/* ------------------------------------------------------------------ status */

/* Text of the last host-side error of the calling thread ("" if none). */
DSA_API const char* dsa_last_error_string(void);

/* Bytes of the status block at the head of every workspace (256). */
DSA_API size_t dsa_status_bytes(void);

/* Zero the status block of `d_ws` on `stream` (once before first use). */
DSA_API dsa_status_t dsa_workspace_init(void* d_ws, size_t ws_bytes, dsa_stream_t stream);

/* Synchronise `stream`, return the device status accumulated in `d_ws` as a
 * dsa_status_t (DSA_OK if clean; otherwise the most severe recorded error,
 * DSA_ERR_TIMEOUT before DSA_ERR_DEVICE_INDEX before DSA_ERR_HOT_OVERFLOW)
 * and clear it.  *raw_bits, if non-null, receives the raw error bits (1
 * timeout, 2 index, 4 batch arrays, 8 hot-buffer overflow). */
DSA_API dsa_status_t dsa_status_fetch(void* d_ws, dsa_stream_t stream, int32_t* raw_bits);

/* Per-kernel launch counters kept by the host side of the library (for
 * tests and benchmarks): counts[0] indexer, [1] top-K, [2] sparse MLA,
 * [3] split combine, [4] FP8 quantisers, [5] indexer cache append, [6] hot
 * buffer plan, [7] hot buffer swap-in, [8] other.  `n` is the length of
 * `counts`; returns how many counters exist. */
DSA_API int dsa_launch_counts(uint64_t* counts, int n);
DSA_API void dsa_launch_counts_reset(void);

/* Per-launch timing for benchmarks: while enabled, the library records a
 * CUDA event pair on the launching stream around every kernel it launches.
 * dsa_profile_collect() waits for the recorded events, adds the elapsed
 * milliseconds and launch counts per kind (same order as dsa_launch_counts)
 * into ms[0..n) / launches[0..n) (zeroed by the call), and clears the record.
 * Returns how many kinds exist, or -1 on a CUDA error. */
DSA_API void dsa_profile_enable(int on);
DSA_API int dsa_profile_collect(double* ms, uint64_t* launches, int n);

/* Upper bound in nanoseconds on every spin-wait inside the kernels launched
 * after this call (default 2e9).  Exposed so that tests can shorten it. */
DSA_API void dsa_set_wait_timeout_ns(uint64_t ns);

/* Kernel choice for sparse attention over many tokens (at least twice as many
 * as the GPU has SMs) with 64 heads on bf16 rows of contiguous or paged
 * caches of at most 96 MB, which L2 holds (dsa_sparse_mla_attn and the group
 * calls): with `on` (the default) one
 * persistent CTA per SM walks a list of tokens, overlapping each token's
 * output and the next token's query and first gather with the current
 * token's products; with 0, one CTA per token.  Both compute the same
 * results bit for bit; the switch exists for tests and measurements.  Takes
 * effect for launches after the call; not synchronised with launches on
 * other host threads. */
DSA_API void dsa_set_mla_persistent(int on);

/* Test aid for the failure path: launch one CTA that waits on an mbarrier
 * nothing ever arrives on, bounded by the current wait limit, records
 * DSA_ERR_TIMEOUT in the status block of `d_ws` and exits cleanly. */
DSA_API dsa_status_t dsa_selftest_wait_timeout(void* d_ws, size_t ws_bytes, dsa_stream_t stream);

/* ------------------------------------------------------------------ step a1 */

/*
 * Lightning-indexer scores (the candidate-scoring step of an F layer):
 *   scores[t, s] = sum_{j<32} w[t,j] * ReLU(q_idx[t,j,:] . k_idx[row(s),:])
 * for 0 <= s <= q_pos[t], and -inf for q_pos[t] < s < max_len.
 *   dt = DSA_BF16:     q_idx bf16 [num_q, 32, 128], k_idx bf16 [k_rows, 128];
 *                      q_scale and k_scale are ignored (may be NULL).
 *   dt = DSA_FP8_E4M3: q_idx E4M3 [num_q, 32, 128] with q_scale fp32
 *                      [num_q, 32]; k_idx E4M3 [k_rows, 128] with k_scale
 *                      fp32 [k_rows]; an element's value is code * scale, and
 *                      scales must be > 0 (as dsa_fp8_quantize writes them).
 *   w       fp32 [num_q, 32]
 *   scores  fp32 [num_q, max_len] (written in full)
 * Pointers to q_idx / k_idx must be 16-byte aligned.  The reduction over
 * heads and the products are fp32 (tensor-core accumulation of the dots).
 * ws: status block only (dsa_indexer_workspace_size).
 */
DSA_API size_t dsa_indexer_workspace_size(const dsa_batch_t* b);
DSA_API dsa_status_t dsa_indexer_scores(const void* q_idx, const float* q_scale, const float* w,
                                const void* k_idx, const float* k_scale, int64_t k_rows,
                                dsa_dtype_t dt, const dsa_batch_t* b, float* scores, void* ws,
                                size_t ws_bytes, dsa_stream_t stream);

/* ------------------------------------------------------------------ step a2 */

/*
 * Top-K selection ("keep the top 2048 as the sparse set", CH 2.2 of
 * "GLM-5.2 架构深度拆解"): for each query t, the k positions s in
 * [0, q_pos[t]] with the largest scores[t, s]; equal scores go to the lower
 * position.  idx[t, :] receives them in ascending position order; if
 * q_pos[t] + 1 < k every visible position is taken and the remaining slots
 * are -1.  scores is fp32 [num_q, max_len] (only s <= q_pos[t] is read), idx
 * int32 [num_q, k].  1 <= k <= 4096.  Scores compare as fp32 values:
 * -0.0 equals +0.0 (a tie, so the lower position wins); a NaN whose sign bit
 * is clear ranks above +inf and one whose sign bit is set below -inf.
 * ws: dsa_topk_workspace_size (the status
 * block, plus about 128 KB of scratch per row for batches of fewer than 80
 * rows longer than 16K positions).
 */
DSA_API size_t dsa_topk_workspace_size(const dsa_batch_t* b, int32_t k);
DSA_API dsa_status_t dsa_topk(const float* scores, const dsa_batch_t* b, int32_t k, int32_t* idx,
                      void* ws, size_t ws_bytes, dsa_stream_t stream);

/* ------------------------------------------------------------------ steps a4-a5 */

/*
 * Absorbed-MLA sparse attention over the selected positions of one layer
 * (gather from this layer's own cache, then attention):
 *   z_s = scale * (q_lat[t,h,:] . kv[row(s), :512] + q_rope[t,h,:] . kv[row(s), 512:])
 *   out[t,h,:] = sum_s softmax(z)_s kv[row(s), :512],  lse[t,h] = ln sum_s exp(z_s)
 * over s in idx[t, :] (k entries; -1 = empty slot).  Valid entries must be
 * distinct positions in [0, q_pos[t]] and occupy the first slots of the row
 * (dsa_topk output does); slots from index min(k, q_pos[t]+1) on are not
 * read.  An entry outside [-1, q_pos[t]] is skipped and raises
 * DSA_ERR_DEVICE_INDEX.  A row with no valid entry gives out = 0,
 * lse = -inf.
 *   q_lat  bf16 [num_q, heads, 512], q_rope bf16 [num_q, heads, 64]
 *   kv     bf16 [kv_rows, 576] (latent then RoPE key), 16-byte aligned
 *   out    bf16 [num_q, heads, 512]; lse fp32 [num_q, heads] or NULL
 *   heads in {16, 64}; 1 <= k <= 4096 (slots are processed in blocks of 128,
 *   the last one masked).  Softmax statistics are fp32; P is
 *   rounded to bf16 for the P.V product (fp32 accumulation).
 * ws: dsa_sparse_mla_workspace_size: the status block, plus, when there are
 * few enough queries for each to be split over 4 or more CTAs (decode), their
 * fp32 partial results (num_q * split * heads * 514 * 4 bytes: 4.2 MB for 4
 * queries of 64 heads split 16 ways).
 */
DSA_API size_t dsa_sparse_mla_workspace_size(const dsa_batch_t* b, int32_t heads, int32_t k);
DSA_API dsa_status_t dsa_sparse_mla_attn(const void* q_lat, const void* q_rope, const void* kv,
                                 int64_t kv_rows, const int32_t* idx, int32_t k, int32_t heads,
                                 float scale, const dsa_batch_t* b, void* out, float* lse,
                                 void* ws, size_t ws_bytes, dsa_stream_t stream);

/* ------------------------------------------------------------------ step a6 */

/*
 * One layer group with IndexShare.  layer_types is a string over {F, S}
 * ("FSSS", "FSSSFSSS", or "FFFF" for the every-layer-indexer ablation) whose
 * first letter is F.  Per layer l (arrays of num_layers host-side pointers to
 * device tensors):
 *   F layer: dsa_indexer_scores(q_idx[l], w[l], k_idx[l]) -> dsa_topk -> idx_buf
 *   every layer: dsa_sparse_mla_attn(q_lat[l], q_rope[l], kv[l], idx_buf) -> out[l]
 * so the indexer runs exactly once per F layer and every S layer reads the
 * index buffer its F layer wrote.  q_idx/w/k_idx/q_scale/k_scale entries of S
 * layers are ignored (may be NULL).  lse[l] may be NULL.
 * idx_buf: int32 [num_q, k], caller-owned; after the call it holds the
 * indices of the last F layer.  The workspace holds the status block and the
 * fp32 score matrix with the top-K scratch, whose space the attention's
 * partial results reuse afterwards; size from dsa_group_workspace_size.
 * For a prefill (some sequence with more than one query) whose rows exceed
 * 16K positions (up to 2M), an F layer selects without writing the score
 * matrix ("GLM-5.2 架构深度拆解" CH 2.2, the top-2048, and CH 4.4; "GLM-5 ->
 * 5.1 -> 5.2" section 10, the fused operator steps): the indexer keeps only the keys at or
 * above a cutoff taken from a sample of each row, and the top-K is resolved
 * from those; a row for which that cannot be shown exact is scored into the
 * workspace's matrix and selected there.  The indices are the same as
 * dsa_indexer_scores + dsa_topk would give (ties to the lower position).
 */
typedef struct {
  const char* layer_types;
  int32_t heads;
  int32_t k;
  float scale;
  dsa_dtype_t idx_dtype;
  int64_t kv_rows;  /* rows of every kv[l] */
  int64_t k_rows;   /* rows of every k_idx[l] */
  const void* const* q_lat;
  const void* const* q_rope;
  const void* const* kv;
  void* const* out;
  float* const* lse;
  const void* const* q_idx;
  const float* const* q_scale;
  const float* const* w;
  const void* const* k_idx;
  const float* const* k_scale;
  dsa_dtype_t kv_dtype; /* DSA_BF16: kv[l] bf16 [kv_rows, 576]; DSA_FP8_E4M3: FP8 rows
                           uint8 [kv_rows, 656] (see dsa_kv_fp8_quantize; heads 64) */
} dsa_group_t;

DSA_API size_t dsa_group_workspace_size(const dsa_group_t* g, const dsa_batch_t* b);
DSA_API dsa_status_t indexshare_group_forward(const dsa_group_t* g, const dsa_batch_t* b,
                                      int32_t* idx_buf, void* ws, size_t ws_bytes,
                                      dsa_stream_t stream);

/* ------------------------------------------------------------------ step a7 */

/*
 * FP8 per-block quantiser of the indexer ("FP8 per-block + Hadamard",
 * sub-doc index row 02 of "GLM-5.2 / 总览"): each 128-element row of x (bf16
 * [rows, 128]) is rotated by the normalised 128-point Hadamard matrix
 * (Sylvester order, 1/sqrt(128)), its scale is amax/448 (1 for an all-zero
 * row) and each element becomes the E4M3 code of x/scale (round to nearest
 * even, saturating).  codes uint8 [rows, 128], scale fp32 [rows].  The same
 * call quantises indexer keys (rows = cache rows) and queries
 * (rows = num_q * 32).  Every step is one IEEE fp32 operation in a fixed
 * order, so results are reproducible bit for bit.
 */
DSA_API dsa_status_t dsa_fp8_quantize(const void* x, int64_t rows, uint8_t* codes, float* scale,
                              dsa_stream_t stream);

/* ------------------------------------------------------------------ FP8 KV latent */

/*
 * FP8 KV cache rows ("GLM-5.2 / 总览" config table: per-token per-layer KV
 * cache BF16 = 1152 bytes, FP8 ~656 bytes per-group): 656 bytes per position,
 *   [0, 512)    the 512-d latent as E4M3 codes, in four groups of 128 dims
 *   [512, 528)  the four groups' fp32 scales, amax/448 (1 for an all-zero group)
 *   [528, 656)  the 64-d RoPE key, bf16 as given
 * Codes are E4M3(x / scale), computed in fp32, round to nearest even,
 * saturating.  dsa_kv_fp8_quantize writes such rows from bf16 rows
 * kv [rows, 576] (out uint8 [rows, 656]; both 16-byte aligned).
 *
 * dsa_sparse_mla_attn_fp8kv: dsa_sparse_mla_attn over an FP8 cache
 * (kv8 uint8 [kv_rows, 656], heads = 64); each gathered latent value is
 * the fp32 product code * scale (round to nearest even) narrowed to bf16
 * (round to nearest even), then the attention is the bf16 one.
 * The group call takes such caches with dsa_group_t.kv_dtype = DSA_FP8_E4M3.
 */
DSA_API dsa_status_t dsa_kv_fp8_quantize(const void* kv, int64_t rows, uint8_t* out,
                                 dsa_stream_t stream);
DSA_API dsa_status_t dsa_sparse_mla_attn_fp8kv(const void* q_lat, const void* q_rope,
                                       const void* kv8, int64_t kv_rows, const int32_t* idx,
                                       int32_t k, int32_t heads, float scale,
                                       const dsa_batch_t* b, void* out, float* lse, void* ws,
                                       size_t ws_bytes, dsa_stream_t stream);

/* ------------------------------------------------------------------ indexer cache append */

/*
 * The step just before a1 for new tokens: interleaved RoPE of the indexer
 * vectors ("GLM-5.2 架构深度拆解" CH 7.1: indexer 32 heads x 128 with
 * indexer_rope_interleave; partial RoPE on a 64-d subspace, interleaved;
 * CH 1.1: rope_theta 8,000,000), then, for the FP8 indexer, the quantiser of
 * dsa_fp8_quantize.  Entries (2i, 2i+1), i < 32, of a 128-vector at position
 * p are rotated by the angle p * inv_freq[i]:
 *   y[2i] = x[2i] cos a - x[2i+1] sin a,  y[2i+1] = x[2i] sin a + x[2i+1] cos a
 * computed in fp64 on the bf16 inputs and rounded once to bf16 (nearest,
 * ties to even); entries 64..127 are copied.  inv_freq: 32 host doubles,
 * theta^(-2i/64) for the model's base theta (passed in so that every
 * implementation rotates by the same angles).
 *
 * dsa_indexer_append_keys: n new keys, k_new bf16 [n, 128]; key i belongs to
 * sequence k_seq[i] at position k_pos[i] (device int32 [n]) and is written at
 * that position's cache row in the batch layout (contiguous or paged):
 * k_cache bf16 [k_rows, 128], or E4M3 codes uint8 [k_rows, 128] with
 * k_scale fp32 [k_rows] for dt = FP8.  A key whose row is outside
 * [0, k_rows) (or unmapped) is skipped and raises DSA_ERR_DEVICE_INDEX.
 *
 * dsa_indexer_prepare_queries: q_new bf16 [num_q, 32, 128], every head of
 * query t rotated at q_pos[t]; q_out bf16 [num_q, 32, 128], or E4M3 codes
 * with q_scale fp32 [num_q, 32].
 *
 * Inputs and outputs must not overlap; pointers to vectors 16-byte aligned.
 * ws: the status block (dsa_status_bytes()).
 */
DSA_API dsa_status_t dsa_indexer_append_keys(const void* k_new, const int32_t* k_seq,
                                     const int32_t* k_pos, int32_t n, const dsa_batch_t* b,
                                     dsa_dtype_t dt, const double* inv_freq, void* k_cache,
                                     float* k_scale, int64_t k_rows, void* ws, size_t ws_bytes,
                                     dsa_stream_t stream);
DSA_API dsa_status_t dsa_indexer_prepare_queries(const void* q_new, const dsa_batch_t* b,
                                         dsa_dtype_t dt, const double* inv_freq, void* q_out,
                                         float* q_scale, void* ws, size_t ws_bytes,
                                         dsa_stream_t stream);

/* ------------------------------------------------------------------ hot / cold KV */

/*
 * A GPU "hot" buffer of KV rows in front of the full cache kept in host
 * memory ("GLM-5.2 / 总览" glossary entry HiSparse: 6144 hot KV slots on the
 * GPU, the full KV in CPU pinned memory, rows swapped in on demand after the
 * DSA top-K; config table: a 1M-token context's KV held by a GPU hot buffer
 * plus a CPU cold store).  One state per index span (an F layer and the S
 * layers that read its index buffer: they select the same positions, so one
 * plan serves every layer of the span).  All arrays are device int32,
 * caller-owned:
 *   slot_pos    [num_seqs, hot_slots]  position held by each slot, -1 empty
 *   slot_stamp  [num_seqs, hot_slots]  last step that used the slot, -1 never
 *   pos_slot    [num_seqs, max_pos]    slot holding each position, -1 none
 *   fetch_pos, fetch_slot [num_seqs, hot_slots], fetch_count [num_seqs]:
 *               the last plan's swap-in list, per sequence
 * Initialise slot_pos, slot_stamp and pos_slot to -1 (every byte 0xFF).
 * max_pos >= the batch's max_len; 1 <= hot_slots <= DSA_HOT_MAX_SLOTS;
 * num_seqs * hot_slots < 2^31.  The hot KV of a layer is a device array of
 * num_seqs * hot_slots rows (bf16 [.., 576] or FP8 [.., 656]); position s of
 * sequence b, once resident in slot j, is hot row b * hot_slots + j.
 */
typedef struct {
  int32_t hot_slots;
  int32_t max_pos;
  int32_t* slot_pos;
  int32_t* slot_stamp;
  int32_t* pos_slot;
  int32_t* fetch_pos;
  int32_t* fetch_slot;
  int32_t* fetch_count;
} dsa_hot_t;

/*
 * dsa_hot_plan: one step of the hot buffer for the index buffer idx
 * (int32 [num_q, k], positions, -1 padding).  Per sequence, over the valid
 * entries (0 <= s <= q_pos[t]) of its queries, query by query and slot by
 * slot: a resident position is a hit and its slot's stamp becomes `step`;
 * the other positions are misses, in order of first appearance; the misses
 * take the least recently used slots among those not used at this step
 * (smallest stamp, then lowest slot index), handed out in increasing slot
 * index; each chosen slot drops its old position and records (position,
 * slot) on the fetch list.  rows (int32 [num_q, k], device) receives the
 * hot row of every valid entry and -1 elsewhere.  `step` >= 0 must exceed
 * every step used before with this state.  A sequence with more misses than
 * unused slots changes no slot, gets rows -1 and raises
 * DSA_ERR_HOT_OVERFLOW; an entry outside [-1, q_pos] is skipped and raises
 * DSA_ERR_DEVICE_INDEX (both in the workspace's status word).
 *
 * dsa_hot_fetch: the swap-in of the last plan's fetch lists for `layers`
 * layers: hot_kv[l][b * hot_slots + slot] = cold_kv[l][row of (b, position)]
 * with the batch's cache layout (seq_row0 or block table) addressing the cold
 * caches of cold_rows rows; each hot_kv[l] has hot_rows rows, at least
 * num_seqs * hot_slots (DSA_ERR_INVALID_ARG otherwise).  cold_kv[l] is host memory the device can read
 * (page-locked: cudaHostAlloc / cudaMallocHost, or cudaHostRegister'ed;
 * device memory is accepted too); pageable memory returns
 * DSA_ERR_INVALID_ARG.  The kernel reads it directly (NVLink-C2C on Grace),
 * no staging copies.  Rows are 1152 bytes (kv_dtype DSA_BF16) or 656
 * (DSA_FP8_E4M3); all pointers 16-byte aligned.
 *
 * dsa_sparse_mla_attn_rows: dsa_sparse_mla_attn (or _fp8kv, by kv_dtype)
 * whose index entries are absolute rows of kv (e.g. the hot rows of
 * dsa_hot_plan) instead of positions: entry r >= 0 reads kv row r, -1 is
 * padding; rows outside [0, kv_rows) are skipped and raise
 * DSA_ERR_DEVICE_INDEX.  The batch supplies the query rows and positions.
 */
DSA_API dsa_status_t dsa_hot_plan(const int32_t* idx, int32_t k, const dsa_batch_t* b,
                                  const dsa_hot_t* h, int32_t step, int32_t* rows, void* ws,
                                  size_t ws_bytes, dsa_stream_t stream);
DSA_API dsa_status_t dsa_hot_fetch(const dsa_hot_t* h, const dsa_batch_t* b, int32_t layers,
                                   const void* const* cold_kv, int64_t cold_rows,
                                   void* const* hot_kv, int64_t hot_rows, dsa_dtype_t kv_dtype,
                                   void* ws, size_t ws_bytes, dsa_stream_t stream);
/*
 * dsa_hot_touch: one read every `stride` bytes (a multiple of 16; the host
 * page size, e.g. 65536 on Grace) of each of `layers` cold caches of
 * cold_bytes bytes (a multiple of 16), so that the device's translations of their host pages
 * exist before the first swap-in: measured on GB300, a swap-in whose rows
 * lie on host pages the GPU has never read runs 6-30x slower than one over
 * pages it has read before.  Call once after a cold cache is allocated (or
 * grown); it changes no memory.  cold_kv as for dsa_hot_fetch.
 */
DSA_API dsa_status_t dsa_hot_touch(int32_t layers, const void* const* cold_kv, int64_t cold_bytes,
                                   int64_t stride, dsa_stream_t stream);
DSA_API dsa_status_t dsa_sparse_mla_attn_rows(const void* q_lat, const void* q_rope,
                                              const void* kv, int64_t kv_rows,
                                              dsa_dtype_t kv_dtype, const int32_t* rows,
                                              int32_t k, int32_t heads, float scale,
                                              const dsa_batch_t* b, void* out, float* lse,
                                              void* ws, size_t ws_bytes, dsa_stream_t stream);

/*
 * indexshare_group_forward_hot: indexshare_group_forward over hot buffers.
 * g->kv[l] are the layers' HOT KV arrays (kv_rows = num_seqs * hot_slots of
 * every span), hot->cold_kv[l] their full caches in host memory.  Each F
 * layer scores and selects as usual into idx_buf, then plans its span
 * (hot->spans[i] for the i-th F layer of layer_types, hot->n_spans of them),
 * swaps in the span's missing rows for all of its layers at once and every
 * layer of the span attends over its hot rows (hot->rows: device int32
 * [num_q, k] scratch).  Errors as for the calls above.
 */
typedef struct {
  const dsa_hot_t* spans;
  int32_t n_spans;
  const void* const* cold_kv;
  int64_t cold_rows;
  int32_t step;
  int32_t* rows;
} dsa_hot_group_t;

DSA_API dsa_status_t indexshare_group_forward_hot(const dsa_group_t* g, const dsa_batch_t* b,
                                                  const dsa_hot_group_t* hot, int32_t* idx_buf,
                                                  void* ws, size_t ws_bytes, dsa_stream_t stream);

/* ------------------------------------------------------------------ no workspace */

/*
 * dsa_indexer_scores followed by dsa_topk, with no caller workspace.  This
 * entry point has no counterpart in the method's description; it exists for
 * callers that cannot allocate device memory: a host framework that owns all
 * of the device memory and gives its plugins no allocator, or a serving loop
 * that must not call cudaMalloc / cudaFree because those calls can
 * synchronise the device and stall every stream.
 *
 * The fp32 score matrix and the device status word live in a file-scope
 * device array of 64 MiB that every GPU loading this library holds until the
 * process exits.  Limit: num_q * max_len * 4 bytes must not exceed 48 MiB
 * minus 256 bytes (12,582,848 scores, e.g. 64 decode rows of 128K positions
 * or 4 rows of 1M; the last 16 MiB hold top-K scratch); larger batches return
 * DSA_ERR_WORKSPACE before anything is enqueued.  Arguments, layouts and results are those of
 * dsa_indexer_scores and dsa_topk; idx is int32 [num_q, k].
 *
 * The first call on a device looks up the array's device address with that
 * device current (and again after the device's context has changed, e.g.
 * after cudaDeviceReset); make that first call before any stream capture.
 * Every call clears the status word, then enqueues both kernels on `stream`;
 * if d_status_out (a device int32) is non-NULL the call's device status bits
 * are copied there at the end (0 = clean).  d_status_out is written only
 * when the call returns DSA_OK; on an error return the steps before the
 * failing one may already be enqueued, and dsa_last_error_string names the
 * step that failed.  All calls share the array and it keeps the last call's
 * contents, so calls whose kernels overlap on the GPU (other streams, other
 * host threads on the same device) race on it.  Nothing is allocated or
 * freed by this call.
 */
DSA_API dsa_status_t dsa_indexer_topk_noalloc(const void* q_idx, const float* q_scale,
                                              const float* w, const void* k_idx,
                                              const float* k_scale, int64_t k_rows,
                                              dsa_dtype_t dt, const dsa_batch_t* b, int32_t k,
                                              int32_t* idx, int32_t* d_status_out,
                                              dsa_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* DSA_H_ */

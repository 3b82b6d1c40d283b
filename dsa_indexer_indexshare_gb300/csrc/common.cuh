// Internal declarations shared by the kernels and the host launchers.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "../../include/dsa.h"
#include "ptx.cuh"

namespace dsa {

constexpr size_t kStatusBytes = 256;

// Device view of dsa_batch_t (plain values, passed by value to kernels).
struct BatchArgs {
  int32_t num_seqs, num_q, max_q, max_len;
  const int32_t* q_start;
  const int32_t* q_pos;
  const int64_t* seq_row0;
  const int32_t* block_table;  // paged layout when not null
  int32_t block_rows, blocks_per_seq;
};

inline BatchArgs to_args(const dsa_batch_t& b) {
  return BatchArgs{b.num_seqs, b.num_q, b.max_q, b.max_len, b.q_start, b.q_pos, b.seq_row0,
                   b.block_table, b.block_rows, b.blocks_per_seq};
}

// First cache row of sequence `seq` in the contiguous layout (0 when paged).
__device__ __forceinline__ int64_t seq_base_row(const BatchArgs& b, int seq) {
  return b.block_table ? 0 : b.seq_row0[seq];
}

// Cache row of position s (>= 0) of sequence `seq`; base = seq_base_row(b, seq).
// Paged layout: the row inside the block the table names, or -1 for a
// negative block id or a block beyond the table.
__device__ __forceinline__ int64_t cache_row(const BatchArgs& b, int seq, int64_t base, int s) {
  if (!b.block_table) return base + s;
  const int blk = s / b.block_rows;
  if (blk >= b.blocks_per_seq) return -1;
  const int32_t id = b.block_table[static_cast<int64_t>(seq) * b.blocks_per_seq + blk];
  return id < 0 ? -1 : static_cast<int64_t>(id) * b.block_rows + (s - blk * b.block_rows);
}

// Rows [qs, qe) of sequence `seq`, validated against the batch sizes.  On
// inconsistency records DSA_DEVERR_BATCH and returns an empty range.
__device__ __forceinline__ void seq_rows(const BatchArgs& b, int seq, int* status, int& qs,
                                         int& qe) {
  qs = b.q_start[seq];
  qe = b.q_start[seq + 1];
  if (qs < 0 || qe < qs || qe > b.num_q) {
    if (threadIdx.x == 0) atomicOr(status, DSA_DEVERR_BATCH);
    qs = qe = 0;
  }
}

// Position of query t, or -1 (with DSA_DEVERR_BATCH) when outside [0, max_len).
__device__ __forceinline__ int query_pos(const BatchArgs& b, int t, int* status) {
  int p = b.q_pos[t];
  if (p < 0 || p >= b.max_len) {
    if (status) atomicOr(status, DSA_DEVERR_BATCH);
    return -1;
  }
  return p;
}

// Programmatic dependent launch.  The library's kernels on the indexer /
// top-K / attention path are launched with programmatic stream
// serialization (launch_chained): such a kernel may be scheduled while the
// previous kernel of its stream is still running, so each of them calls
// chain_wait() before its first access to global memory (it returns once
// every earlier kernel of the stream has completed and its writes are
// visible) and then chain_release(), which lets the next kernel be
// scheduled.  Both are no-ops in a kernel launched without the attribute.
__device__ __forceinline__ void chain_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void chain_release() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// cudaLaunchKernelEx with programmatic stream serialization and, for
// cluster > 1, that many CTAs per cluster along x.
template <typename... KArgs, typename... Args>
cudaError_t launch_chained(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                           cudaStream_t stream, unsigned cluster, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  unsigned n = 0;
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (cluster > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

// Order-preserving image of an fp32 score: a > b as floats iff key(a) >
// key(b) as unsigned integers.  -0.0 is first replaced by +0.0 so that the
// two zeros are one value (equal scores, ties to the lower position); a NaN
// with the sign bit clear ranks above +inf, one with it set below -inf.
__device__ __forceinline__ uint32_t order_key(float x) {
  uint32_t u = __float_as_uint(x);
  u = (u == 0x80000000u) ? 0u : u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// ------------------------------------------------------------- host helpers
// Implemented in api.cu.
// Record a message for dsa_last_error_string and return s.
dsa_status_t fail(dsa_status_t s, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
// DSA_OK for cudaSuccess, else DSA_ERR_CUDA with the error's name and `where`.
dsa_status_t cuda_status(cudaError_t e, const char* where);
// Argument checks shared by the entry points (each records its message).
dsa_status_t check_batch(const dsa_batch_t* b);
dsa_status_t check_indexer_args(const void* q_idx, const float* q_scale, const float* w,
                                const void* k_idx, const float* k_scale, int64_t k_rows,
                                dsa_dtype_t dt);
dsa_status_t check_topk_k(int32_t k);
bool make_tmap_2d(CUtensorMap* map, const void* base, CUtensorMapDataType dt, int esize,
                  uint64_t inner, uint64_t rows, uint32_t box_inner, uint32_t box_rows);
void count_launch(int which);
// Event pair around a launch when profiling is enabled (no-ops otherwise).
void prof_begin(cudaStream_t stream);
void prof_end(int which, cudaStream_t stream);
uint64_t wait_timeout_ns();

enum LaunchKind { kLaunchIndexer = 0, kLaunchTopk, kLaunchMla, kLaunchCombine, kLaunchQuant,
                  kLaunchAppend, kLaunchHot, kLaunchFetch, kLaunchOther, kNumLaunchKinds };

// Launchers (return a CUDA error code; argument checks are done by api.cu).
cudaError_t launch_indexer(const void* q_idx, const float* q_scale, const float* w,
                           const void* k_idx, const float* k_scale, int64_t k_rows, bool fp8,
                           const dsa_batch_t& b, float* scores, bool fill_tail, int* status,
                           cudaStream_t stream);
// Select-only F layer for rows longer than 16K positions: the indexer's
// epilogue keeps, per query row, only the (key, position) pairs at or above
// a cutoff taken from a sample of the row's scores, and the top-K is resolved
// from those lists, so that no score matrix is written (rows whose sample
// misled fall back to the score matrix and the exact top-K).
constexpr int kTopkCnt = 8;          // per-row words: 0 key chunks of the capture, 1 captured,
                                     // 2 dropped, 3 cutoff (fp32 bits), 4 T, 5 pstar, 6 fallback,
                                     // 7 sampled positions
constexpr int kTopkCandCap = 16384;  // captured keys kept per row
constexpr int kSampleTilesMax = 64;  // 128-key tiles sampled per row at most
constexpr int kSegMax = 256;         // key chunks of a row at most (its list is split evenly,
                                     // each chunk's segment again in 4 quarters)
constexpr int kSampleChunk = 8;      // sampled tiles per CTA of the sample pass
struct TopkLists {
  int* cnt;        // [num_q][kTopkCnt]
  uint32_t* ckey;  // [num_q][kTopkCandCap] captured order keys: quarter q of segment c of a
                   // row (the keys of key chunk c in TMEM lane quarter q) at
                   // (4c + q) * (kTopkCandCap / (4 chunks))
  int32_t* cpos;   // [num_q][kTopkCandCap] their positions
  int* segcnt;     // [num_q][kSegMax][4] keys each quarter found at or above the cutoff
  float* sample;   // [num_q][kSampleTilesMax * 128] sampled scores
};
enum IndexerMode { kIdxScores = 0, kIdxSample = 1, kIdxCapture = 2 };
bool use_select_only(const dsa_batch_t& b, int k);
size_t select_only_bytes(const dsa_batch_t& b);
TopkLists select_only_lists(const dsa_batch_t& b, void* base);
// mode kIdxScores: scores (rows of blocks holding a row flagged in `only`
// when only != nullptr); kIdxSample / kIdxCapture: the lists' sample / capture
cudaError_t launch_indexer_mode(const void* q_idx, const float* q_scale, const float* w,
                                const void* k_idx, const float* k_scale, int64_t k_rows, bool fp8,
                                const dsa_batch_t& b, int mode, float* scores, const int* only,
                                const TopkLists& lists, int* status, cudaStream_t stream);
// the whole select-only F layer: sample, cutoff, capture, resolve and write,
// then the fallback rows through the score matrix (scores: [num_q][max_len])
cudaError_t launch_indexer_topk_select(const void* q_idx, const float* q_scale, const float* w,
                                       const void* k_idx, const float* k_scale, int64_t k_rows,
                                       bool fp8, const dsa_batch_t& b, int k, int32_t* idx,
                                       float* scores, void* lists_base, int* status,
                                       cudaStream_t stream);
size_t topk_scratch_bytes(const dsa_batch_t& b, int k);
cudaError_t launch_topk(const float* scores, const dsa_batch_t& b, int k, int32_t* idx,
                        int* status, void* scratch, size_t scratch_bytes, cudaStream_t stream);
// Prefill-sized attention launches on a persistent grid (default on).
void set_mla_persistent(bool on);
size_t mla_workspace_bytes(const dsa_batch_t& b, int heads, int k);
cudaError_t launch_sparse_mla(const void* q_lat, const void* q_rope, const void* kv,
                              int64_t kv_rows, const int32_t* idx, int k, int heads, float scale,
                              const dsa_batch_t& b, void* out, float* lse, void* ws_extra,
                              size_t ws_extra_bytes, int* status, cudaStream_t stream,
                              bool kv_fp8 = false, bool direct_rows = false,
                              bool after_own_kernel = false, bool after_attention = false);
// Hot / cold KV: the plan of one step (one CTA per sequence) and the swap-in
// of its fetch lists for `layers` layers from host-resident cold caches.
cudaError_t launch_hot_plan(const int32_t* idx, int k, const dsa_batch_t& b, const dsa_hot_t& h,
                            int step, int32_t* rows, int* status, cudaStream_t stream);
cudaError_t launch_hot_fetch(const dsa_hot_t& h, const dsa_batch_t& b, int layers,
                             const void* const* cold, int64_t cold_rows, void* const* hot,
                             int row_bytes, int* status, cudaStream_t stream);
// RoPE (+ Hadamard + FP8) of n indexer vectors; vector v at position
// pos_of[v / group], written to the cache row of (seq_of[v / group], pos)
// (seq_of set) or to row v.  inv_freq: 32 host doubles.
cudaError_t launch_rope_append(const void* x, int64_t n, int group, const int32_t* pos_of,
                               const int32_t* seq_of, const dsa_batch_t& b, const double* inv_freq,
                               bool fp8, void* out, float* out_scale, int64_t out_rows, int* status,
                               cudaStream_t stream);
cudaError_t launch_kv_fp8_quantize(const void* kv, int64_t rows, uint8_t* out,
                                   cudaStream_t stream);
cudaError_t launch_quantize(const void* x, int64_t rows, uint8_t* codes, float* scale,
                            cudaStream_t stream);
cudaError_t launch_selftest_wait(int* status, cudaStream_t stream);

}  // namespace dsa

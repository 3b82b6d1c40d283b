// Allocation-free form of the F-layer step (indexer scores, then top-K).
//
// Some callers cannot provide a workspace: a host framework that owns all of
// the device memory and hands its plugins no allocator, or a serving loop
// that must never call cudaMalloc / cudaFree because those calls can
// synchronise the whole device and stall every stream.  For them,
// dsa_indexer_topk_noalloc keeps the score matrix and the status word in a
// file-scope device array of fixed size instead of a caller workspace.
//
// Every GPU that loads this library holds the array (64 MiB) until the
// process exits.  All calls share it and it keeps the last call's contents,
// so calls whose kernels overlap on the GPU (different streams, or different
// host threads on one device) race on it.
#include <mutex>

#include "common.cuh"

namespace dsa {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;
// the last 16 MiB hold the top-K scratch of decode-sized batches
constexpr size_t kNoAllocTopkBytes = size_t(16) << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the array on the current device (looked up once per
// device, with that device current).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace dsa

using namespace dsa;

extern "C" DSA_API dsa_status_t dsa_indexer_topk_noalloc(
    const void* q_idx, const float* q_scale, const float* w, const void* k_idx,
    const float* k_scale, int64_t k_rows, dsa_dtype_t dt, const dsa_batch_t* b, int32_t k,
    int32_t* idx, int32_t* d_status_out, dsa_stream_t stream) {
  // Argument checks mirror dsa_indexer_scores + dsa_topk.
  if (!b || !q_idx || !w || !k_idx || !idx) return DSA_ERR_INVALID_ARG;
  if (b->num_seqs < 1 || b->num_q < 0 || b->max_q < 0 || b->max_q > b->num_q ||
      b->max_len < 128 || b->max_len % 128 != 0 || !b->q_start || !b->q_pos ||
      (!b->block_table && !b->seq_row0) || (b->num_q > 0 && b->max_q < 1))
    return DSA_ERR_INVALID_ARG;
  if (b->block_table &&
      (b->block_rows < 128 || (b->block_rows & (b->block_rows - 1)) != 0 || b->blocks_per_seq < 1 ||
       static_cast<int64_t>(b->blocks_per_seq) * b->block_rows < b->max_len))
    return DSA_ERR_INVALID_ARG;
  if (b->num_seqs > 65535) return DSA_ERR_UNSUPPORTED;
  if (dt != DSA_BF16 && dt != DSA_FP8_E4M3) return DSA_ERR_UNSUPPORTED;
  if (dt == DSA_FP8_E4M3 && (!q_scale || !k_scale)) return DSA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(q_idx) & 15u) || (reinterpret_cast<uintptr_t>(k_idx) & 15u))
    return DSA_ERR_INVALID_ARG;
  if (k_rows < 1 || k_rows > (int64_t(1) << 31) - 1) return DSA_ERR_INVALID_ARG;
  if (k < 1 || k > 4096) return DSA_ERR_UNSUPPORTED;
  // The score matrix must fit the fixed array after the status block, and
  // the top-K scratch its reserved tail.
  const size_t need = static_cast<size_t>(b->num_q) * static_cast<size_t>(b->max_len) * 4;
  if (need > kNoAllocScratchBytes - kNoAllocTopkBytes - kStatusBytes) return DSA_ERR_WORKSPACE;
  if (topk_scratch_bytes(*b, k) > kNoAllocTopkBytes) return DSA_ERR_WORKSPACE;
  void* base = nullptr;
  if (scratch_address(&base) != cudaSuccess) return DSA_ERR_CUDA;
  int* status = static_cast<int*>(base);
  float* scores = reinterpret_cast<float*>(static_cast<unsigned char*>(base) + kStatusBytes);
  // the status word must start at zero; the scores need no clearing (top-K
  // reads only positions the indexer writes)
  if (cudaMemsetAsync(status, 0, sizeof(int), stream) != cudaSuccess) return DSA_ERR_CUDA;
  if (b->num_q > 0) {
    if (launch_indexer(q_idx, q_scale, w, k_idx, k_scale, k_rows, dt == DSA_FP8_E4M3, *b, scores,
                       false, status, stream) != cudaSuccess)
      return DSA_ERR_CUDA;
    unsigned char* topk_scratch =
        static_cast<unsigned char*>(base) + kNoAllocScratchBytes - kNoAllocTopkBytes;
    if (launch_topk(scores, *b, k, idx, status, topk_scratch, kNoAllocTopkBytes, stream) !=
        cudaSuccess)
      return DSA_ERR_CUDA;
  }
  if (d_status_out &&
      cudaMemcpyAsync(d_status_out, status, sizeof(int), cudaMemcpyDeviceToDevice, stream) !=
          cudaSuccess)
    return DSA_ERR_CUDA;
  return DSA_OK;
}

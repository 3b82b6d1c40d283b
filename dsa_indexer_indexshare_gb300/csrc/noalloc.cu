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

// The array's device address, looked up per device with that device current
// and kept with the context it belongs to: after cudaDeviceReset the device's
// primary context is a new one, in which the module (and the array) is
// loaded again at another address, so a cached address is used only while
// the current context is the one it was taken in.
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
CtxGetCurrentFn g_ctx_get = nullptr;
void* g_noalloc_ptr[kMaxDevices] = {};
CUcontext g_noalloc_ctx[kMaxDevices] = {};

cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_ctx_get) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    e = cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess) return e;
    if (q != cudaDriverEntryPointSuccess || !fn) return cudaErrorNotSupported;
    g_ctx_get = reinterpret_cast<CtxGetCurrentFn>(fn);
  }
  CUcontext ctx = nullptr;
  if (g_ctx_get(&ctx) != CUDA_SUCCESS) return cudaErrorInvalidDevice;
  if (!ctx || !g_noalloc_ptr[dev] || g_noalloc_ctx[dev] != ctx) {
    // (the lookup also makes the device's primary context current when no
    // context is yet)
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    if (g_ctx_get(&ctx) != CUDA_SUCCESS || !ctx) return cudaErrorInvalidDevice;
    g_noalloc_ptr[dev] = p;
    g_noalloc_ctx[dev] = ctx;
  }
  *out = g_noalloc_ptr[dev];
  return cudaSuccess;
}

// A CUDA failure of this entry point: its message recorded, and the
// runtime's sticky last error cleared so that a later call does not report
// it as its own.
dsa_status_t noalloc_cuda_fail(cudaError_t e, const char* where) {
  cudaGetLastError();
  return cuda_status(e, where);
}

}  // namespace
}  // namespace dsa

using namespace dsa;

extern "C" DSA_API dsa_status_t dsa_indexer_topk_noalloc(
    const void* q_idx, const float* q_scale, const float* w, const void* k_idx,
    const float* k_scale, int64_t k_rows, dsa_dtype_t dt, const dsa_batch_t* b, int32_t k,
    int32_t* idx, int32_t* d_status_out, dsa_stream_t stream) {
  // the checks (and codes, and messages) of dsa_indexer_scores + dsa_topk
  if (dsa_status_t s = check_batch(b)) return s;
  if (dsa_status_t s = check_indexer_args(q_idx, q_scale, w, k_idx, k_scale, k_rows, dt)) return s;
  if (dsa_status_t s = check_topk_k(k)) return s;
  if (!idx) return fail(DSA_ERR_INVALID_ARG, "idx is required");
  // The score matrix must fit the fixed array after the status block, and
  // the top-K scratch its reserved tail.
  const size_t need = static_cast<size_t>(b->num_q) * static_cast<size_t>(b->max_len) * 4;
  const size_t have = kNoAllocScratchBytes - kNoAllocTopkBytes - kStatusBytes;
  if (need > have)
    return fail(DSA_ERR_WORKSPACE, "num_q * max_len * 4 = %zu bytes exceeds the fixed %zu-byte array",
                need, have);
  if (topk_scratch_bytes(*b, k) > kNoAllocTopkBytes)
    return fail(DSA_ERR_WORKSPACE, "top-K scratch of %zu bytes exceeds the fixed %zu bytes",
                topk_scratch_bytes(*b, k), kNoAllocTopkBytes);
  void* base = nullptr;
  if (cudaError_t e = scratch_address(&base)) return noalloc_cuda_fail(e, "scratch address");
  int* status = static_cast<int*>(base);
  float* scores = reinterpret_cast<float*>(static_cast<unsigned char*>(base) + kStatusBytes);
  // the status word must start at zero; the scores need no clearing (top-K
  // reads only positions the indexer writes)
  if (cudaError_t e = cudaMemsetAsync(status, 0, sizeof(int), stream))
    return noalloc_cuda_fail(e, "status clear");
  if (b->num_q > 0) {
    if (cudaError_t e = launch_indexer(q_idx, q_scale, w, k_idx, k_scale, k_rows,
                                       dt == DSA_FP8_E4M3, *b, scores, false, status, stream))
      return noalloc_cuda_fail(e, "indexer launch");
    unsigned char* topk_scratch =
        static_cast<unsigned char*>(base) + kNoAllocScratchBytes - kNoAllocTopkBytes;
    if (cudaError_t e = launch_topk(scores, *b, k, idx, status, topk_scratch, kNoAllocTopkBytes,
                                    stream))
      return noalloc_cuda_fail(e, "top-K launch");
  }
  if (d_status_out)
    if (cudaError_t e = cudaMemcpyAsync(d_status_out, status, sizeof(int), cudaMemcpyDeviceToDevice,
                                        stream))
      return noalloc_cuda_fail(e, "status copy");
  return DSA_OK;
}

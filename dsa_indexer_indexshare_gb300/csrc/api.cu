// C ABI of the library: argument validation, workspace layout, status
// handling, tensor-map construction and the IndexShare group loop.  Every
// compute step is one of the kernels in indexer.cu, topk.cu, sparse_mla.cu
// and quant.cu; nothing here computes on the host.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "common.cuh"

namespace dsa {

namespace {
thread_local std::string g_last_error;
}  // namespace

dsa_status_t fail(dsa_status_t s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

dsa_status_t cuda_status(cudaError_t e, const char* where) {
  if (e == cudaSuccess) return DSA_OK;
  return fail(DSA_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

namespace {
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
}  // namespace

dsa_status_t check_batch(const dsa_batch_t* b) {
  if (!b) return fail(DSA_ERR_INVALID_ARG, "batch is NULL");
  if (b->num_seqs < 1 || b->num_q < 0 || b->max_q < 0 || b->max_len < 128 ||
      b->max_len % 128 != 0)
    return fail(DSA_ERR_INVALID_ARG,
                "batch sizes: num_seqs=%d num_q=%d max_q=%d max_len=%d (max_len must be a "
                "positive multiple of 128)",
                b->num_seqs, b->num_q, b->max_q, b->max_len);
  if (b->num_q > 0 && b->max_q < 1)
    return fail(DSA_ERR_INVALID_ARG, "max_q must be >= 1 when num_q > 0");
  if (b->max_q > b->num_q) return fail(DSA_ERR_INVALID_ARG, "max_q > num_q");
  if (b->num_seqs > 65535) return fail(DSA_ERR_UNSUPPORTED, "num_seqs > 65535");
  const bool paged = b->block_table != nullptr;
  if (!b->q_start || !b->q_pos || (!paged && !b->seq_row0))
    return fail(DSA_ERR_INVALID_ARG, "batch arrays must be non-NULL device pointers");
  if (paged) {
    if (b->block_rows < 128 || (b->block_rows & (b->block_rows - 1)) != 0)
      return fail(DSA_ERR_INVALID_ARG, "block_rows=%d must be a power of two >= 128",
                  b->block_rows);
    if (b->blocks_per_seq < 1 ||
        static_cast<int64_t>(b->blocks_per_seq) * b->block_rows < b->max_len)
      return fail(DSA_ERR_INVALID_ARG, "blocks_per_seq=%d x block_rows=%d does not cover max_len=%d",
                  b->blocks_per_seq, b->block_rows, b->max_len);
  }
  return DSA_OK;
}

dsa_status_t check_indexer_args(const void* q_idx, const float* q_scale, const float* w,
                                const void* k_idx, const float* k_scale, int64_t k_rows,
                                dsa_dtype_t dt) {
  if (dt != DSA_BF16 && dt != DSA_FP8_E4M3) return fail(DSA_ERR_UNSUPPORTED, "indexer dtype %d", dt);
  if (!q_idx || !w || !k_idx) return fail(DSA_ERR_INVALID_ARG, "q_idx, w and k_idx are required");
  if (dt == DSA_FP8_E4M3 && (!q_scale || !k_scale))
    return fail(DSA_ERR_INVALID_ARG, "FP8 indexer needs q_scale and k_scale");
  if (!aligned16(q_idx) || !aligned16(k_idx))
    return fail(DSA_ERR_INVALID_ARG, "q_idx and k_idx must be 16-byte aligned");
  if (k_rows < 1) return fail(DSA_ERR_INVALID_ARG, "k_rows must be >= 1");
  if (k_rows > (int64_t(1) << 31) - 1) return fail(DSA_ERR_UNSUPPORTED, "k_rows >= 2^31");
  return DSA_OK;
}

dsa_status_t check_topk_k(int32_t k) {
  if (k < 1 || k > 4096) return fail(DSA_ERR_UNSUPPORTED, "k=%d (supported: 1..4096)", k);
  return DSA_OK;
}

namespace {
std::atomic<uint64_t> g_launches[kNumLaunchKinds];
std::atomic<uint64_t> g_timeout_ns{2000000000ull};

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

dsa_status_t check_ws(void* ws, size_t have, size_t need) {
  if (!ws) return fail(DSA_ERR_WORKSPACE, "workspace is NULL");
  if (reinterpret_cast<uintptr_t>(ws) & 255u)
    return fail(DSA_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  if (have < need)
    return fail(DSA_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", have, need);
  return DSA_OK;
}

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

dsa_status_t check_mla_args(const void* q_lat, const void* q_rope, const void* kv, int64_t kv_rows,
                            const int32_t* idx, int32_t k, int32_t heads, float scale,
                            const dsa_batch_t* b, const void* out) {
  if (heads != 16 && heads != 64)
    return fail(DSA_ERR_UNSUPPORTED, "heads=%d (supported: 16, 64)", heads);
  if (k < 1 || k > 4096) return fail(DSA_ERR_UNSUPPORTED, "k=%d (supported: 1..4096)", k);
  if (!q_lat || !q_rope || !kv || !idx || !out)
    return fail(DSA_ERR_INVALID_ARG, "q_lat, q_rope, kv, idx and out are required");
  if (!aligned16(q_lat) || !aligned16(q_rope) || !aligned16(kv) || !aligned16(out))
    return fail(DSA_ERR_INVALID_ARG, "q_lat, q_rope, kv and out must be 16-byte aligned");
  if (kv_rows < 1 || kv_rows > (int64_t(1) << 31) - 1)
    return fail(DSA_ERR_INVALID_ARG, "kv_rows=%lld", static_cast<long long>(kv_rows));
  if (!(scale == scale)) return fail(DSA_ERR_INVALID_ARG, "scale is NaN");
  if (static_cast<int64_t>(b->num_q) * heads > (int64_t(1) << 31) - 1)
    return fail(DSA_ERR_UNSUPPORTED, "num_q * heads >= 2^31");
  return DSA_OK;
}

dsa_status_t launch_status(cudaError_t e, const char* where) { return cuda_status(e, where); }

dsa_status_t check_hot(const dsa_hot_t* h, const dsa_batch_t* b) {
  if (!h) return fail(DSA_ERR_INVALID_ARG, "hot state is NULL");
  if (h->hot_slots < 1 || h->hot_slots > DSA_HOT_MAX_SLOTS)
    return fail(DSA_ERR_UNSUPPORTED, "hot_slots=%d (supported: 1..%d)", h->hot_slots,
                static_cast<int>(DSA_HOT_MAX_SLOTS));
  if (h->max_pos < b->max_len)
    return fail(DSA_ERR_INVALID_ARG, "hot state max_pos=%d < batch max_len=%d", h->max_pos, b->max_len);
  if (static_cast<int64_t>(b->num_seqs) * h->hot_slots > (int64_t(1) << 31) - 1)
    return fail(DSA_ERR_UNSUPPORTED, "num_seqs * hot_slots >= 2^31");
  if (!h->slot_pos || !h->slot_stamp || !h->pos_slot || !h->fetch_pos || !h->fetch_slot ||
      !h->fetch_count)
    return fail(DSA_ERR_INVALID_ARG, "hot state arrays must be non-NULL device pointers");
  return DSA_OK;
}

// The layer string and every layer's arguments of a group call (the batch is
// checked by the caller).
dsa_status_t check_group(const dsa_group_t* g, const dsa_batch_t* b, const int32_t* idx_buf) {
  if (!g->layer_types || g->layer_types[0] != 'F')
    return fail(DSA_ERR_INVALID_ARG, "layer_types must start with F");
  const int nl = static_cast<int>(strlen(g->layer_types));
  if (nl > 4096) return fail(DSA_ERR_INVALID_ARG, "layer_types too long");
  for (int l = 0; l < nl; ++l)
    if (g->layer_types[l] != 'F' && g->layer_types[l] != 'S')
      return fail(DSA_ERR_INVALID_ARG, "layer_types[%d] = '%c' (want F or S)", l, g->layer_types[l]);
  if (!g->q_lat || !g->q_rope || !g->kv || !g->out || !idx_buf)
    return fail(DSA_ERR_INVALID_ARG, "q_lat, q_rope, kv, out arrays and idx_buf are required");
  for (int l = 0; l < nl; ++l) {
    if (dsa_status_t s = check_mla_args(g->q_lat[l], g->q_rope[l], g->kv[l], g->kv_rows, idx_buf,
                                        g->k, g->heads, g->scale, b, g->out[l]))
      return s;
    if (g->layer_types[l] == 'F') {
      if (!g->q_idx || !g->w || !g->k_idx ||
          (g->idx_dtype == DSA_FP8_E4M3 && (!g->q_scale || !g->k_scale)))
        return fail(DSA_ERR_INVALID_ARG, "F layer %d: indexer arrays missing", l);
      if (dsa_status_t s = check_indexer_args(g->q_idx[l], g->q_scale ? g->q_scale[l] : nullptr,
                                              g->w[l], g->k_idx[l],
                                              g->k_scale ? g->k_scale[l] : nullptr, g->k_rows,
                                              g->idx_dtype))
        return s;
    }
  }
  if (g->kv_dtype != DSA_BF16 && g->kv_dtype != DSA_FP8_E4M3)
    return fail(DSA_ERR_UNSUPPORTED, "kv_dtype %d", g->kv_dtype);
  if (g->kv_dtype == DSA_FP8_E4M3 && g->heads != 64)
    return fail(DSA_ERR_UNSUPPORTED, "FP8 KV rows: heads must be 64");
  return DSA_OK;
}

// The parts of a group workspace: status block, fp32 score matrix, top-K scratch.
struct GroupWs {
  int* status;
  float* scores;
  uint8_t* topk_scratch;
  size_t topk_bytes;
  uint8_t* mla_extra;  // after the status block (the MLA's own scratch)
  size_t mla_extra_bytes;
};

// Top-K scratch of a group's F layers: the capture lists and samples of the
// select-only path (rows beyond 16K positions), else the top-K's own.
size_t group_topk_bytes(const dsa_group_t* g, const dsa_batch_t* b) {
  return round256(use_select_only(*b, g->k) ? select_only_bytes(*b) : topk_scratch_bytes(*b, g->k));
}

GroupWs group_ws(const dsa_group_t* g, const dsa_batch_t* b, void* ws, size_t need) {
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  const size_t score_bytes = round256(static_cast<size_t>(b->num_q) * static_cast<size_t>(b->max_len) * 4);
  return GroupWs{static_cast<int*>(ws), reinterpret_cast<float*>(wsb + kStatusBytes),
                 wsb + kStatusBytes + score_bytes, group_topk_bytes(g, b),
                 wsb + kStatusBytes, need - kStatusBytes};
}

// F layer l of a group: candidate scoring, then top-K into the shared index buffer.
dsa_status_t run_f_layer(const dsa_group_t* g, const dsa_batch_t* b, int l, int32_t* idx_buf,
                         const GroupWs& w, cudaStream_t stream) {
  const bool fp8 = g->idx_dtype == DSA_FP8_E4M3;
  // rows beyond 16K positions: select-only (no score matrix unless a row's
  // sample misleads), else scores then top-K
  if (use_select_only(*b, g->k))
    return launch_status(
        launch_indexer_topk_select(g->q_idx[l], fp8 ? g->q_scale[l] : nullptr, g->w[l], g->k_idx[l],
                                   fp8 ? g->k_scale[l] : nullptr, g->k_rows, fp8, *b, g->k, idx_buf,
                                   w.scores, w.topk_scratch, w.status, stream),
        "select-only indexer / top-K launch");
  if (dsa_status_t s = launch_status(
          launch_indexer(g->q_idx[l], fp8 ? g->q_scale[l] : nullptr, g->w[l], g->k_idx[l],
                         fp8 ? g->k_scale[l] : nullptr, g->k_rows, fp8, *b, w.scores, false, w.status,
                         stream),
          "indexer launch"))
    return s;
  return launch_status(launch_topk(w.scores, *b, g->k, idx_buf, w.status, w.topk_scratch, w.topk_bytes,
                                   stream),
                       "top-K launch");
}

// A pointer the device can dereference: device, managed or page-locked host
// memory (its device address returned); pageable host memory is refused.
dsa_status_t device_view(const void* p, const char* what, int l, const void** dev) {
  if (!p) return fail(DSA_ERR_INVALID_ARG, "%s[%d] is NULL", what, l);
  if (!aligned16(p)) return fail(DSA_ERR_INVALID_ARG, "%s[%d] must be 16-byte aligned", what, l);
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return fail(DSA_ERR_INVALID_ARG, "%s[%d]: not memory CUDA knows", what, l);
  }
  if ((a.type != cudaMemoryTypeHost && a.type != cudaMemoryTypeDevice &&
       a.type != cudaMemoryTypeManaged) || !a.devicePointer)
    return fail(DSA_ERR_INVALID_ARG, "%s[%d]: pageable host memory (page-lock it first)", what, l);
  *dev = a.devicePointer;
  return DSA_OK;
}

}  // namespace

// ------------------------------------------------------------- host helpers
bool make_tmap_2d(CUtensorMap* map, const void* base, CUtensorMapDataType dt, int esize,
                  uint64_t inner, uint64_t rows, uint32_t box_inner, uint32_t box_rows) {
  if (!g_encode) {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn) {
      g_last_error = "cuTensorMapEncodeTiled unavailable";
      return false;
    }
    g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  }
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * static_cast<uint64_t>(esize)};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t es[2] = {1, 1};
  CUresult r = g_encode(map, dt, 2, const_cast<void*>(base), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    char buf[160];
    snprintf(buf, sizeof buf, "cuTensorMapEncodeTiled failed (%d) for [%llu x %llu]", static_cast<int>(r),
             static_cast<unsigned long long>(rows), static_cast<unsigned long long>(inner));
    g_last_error = buf;
    return false;
  }
  return true;
}

void count_launch(int which) { g_launches[which].fetch_add(1, std::memory_order_relaxed); }

namespace {
struct ProfRec {
  cudaEvent_t start, stop;
  int kind;
};
std::mutex g_prof_mu;
std::atomic<int> g_prof_on{0};
std::vector<ProfRec> g_prof_recs;      // recorded, not yet collected
std::vector<cudaEvent_t> g_prof_free;  // reusable events
thread_local cudaEvent_t g_prof_pending = nullptr;

cudaEvent_t prof_event() {
  if (!g_prof_free.empty()) {
    cudaEvent_t e = g_prof_free.back();
    g_prof_free.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}
}  // namespace

void prof_begin(cudaStream_t stream) {
  if (!g_prof_on.load(std::memory_order_relaxed)) return;
  std::lock_guard<std::mutex> lk(g_prof_mu);
  g_prof_pending = prof_event();
  if (g_prof_pending) cudaEventRecord(g_prof_pending, stream);
}

void prof_end(int which, cudaStream_t stream) {
  if (!g_prof_on.load(std::memory_order_relaxed) || !g_prof_pending) return;
  std::lock_guard<std::mutex> lk(g_prof_mu);
  cudaEvent_t stop = prof_event();
  if (!stop) return;
  cudaEventRecord(stop, stream);
  g_prof_recs.push_back(ProfRec{g_prof_pending, stop, which});
  g_prof_pending = nullptr;
}
uint64_t wait_timeout_ns() { return g_timeout_ns.load(std::memory_order_relaxed); }

}  // namespace dsa

using namespace dsa;

extern "C" {

const char* dsa_last_error_string(void) { return g_last_error.c_str(); }

size_t dsa_status_bytes(void) { return kStatusBytes; }

dsa_status_t dsa_workspace_init(void* d_ws, size_t ws_bytes, dsa_stream_t stream) {
  if (dsa_status_t s = check_ws(d_ws, ws_bytes, kStatusBytes)) return s;
  return cuda_status(cudaMemsetAsync(d_ws, 0, kStatusBytes, stream), "cudaMemsetAsync");
}

dsa_status_t dsa_status_fetch(void* d_ws, dsa_stream_t stream, int32_t* raw_bits) {
  if (!d_ws) return fail(DSA_ERR_WORKSPACE, "workspace is NULL");
  int32_t bits = 0;
  if (dsa_status_t s = cuda_status(cudaMemcpyAsync(&bits, d_ws, 4, cudaMemcpyDeviceToHost, stream),
                                   "cudaMemcpyAsync"))
    return s;
  if (dsa_status_t s = cuda_status(cudaStreamSynchronize(stream), "cudaStreamSynchronize")) return s;
  if (bits) {
    if (dsa_status_t s = cuda_status(cudaMemsetAsync(d_ws, 0, 4, stream), "cudaMemsetAsync")) return s;
  }
  if (raw_bits) *raw_bits = bits;
  if (bits & DSA_DEVERR_TIMEOUT) return fail(DSA_ERR_TIMEOUT, "a bounded wait in a kernel ran out");
  if (bits & (DSA_DEVERR_INDEX | DSA_DEVERR_BATCH))
    return fail(DSA_ERR_DEVICE_INDEX, "a kernel found an index or batch entry out of range (bits %d)", bits);
  if (bits & DSA_DEVERR_HOT_OVERFLOW)
    return fail(DSA_ERR_HOT_OVERFLOW, "a sequence selected more positions than its hot buffer has free slots");
  return DSA_OK;
}

int dsa_launch_counts(uint64_t* counts, int n) {
  for (int i = 0; i < n && i < kNumLaunchKinds; ++i) counts[i] = g_launches[i].load();
  return kNumLaunchKinds;
}
void dsa_launch_counts_reset(void) {
  for (auto& c : g_launches) c.store(0);
}

void dsa_set_wait_timeout_ns(uint64_t ns) { g_timeout_ns.store(ns); }

void dsa_set_mla_persistent(int on) { set_mla_persistent(on != 0); }

void dsa_profile_enable(int on) { g_prof_on.store(on ? 1 : 0); }

int dsa_profile_collect(double* ms, uint64_t* launches, int n) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  for (int i = 0; i < n; ++i) {
    ms[i] = 0.0;
    launches[i] = 0;
  }
  int rc = kNumLaunchKinds;
  for (const ProfRec& r : g_prof_recs) {
    float t = 0.f;
    if (cudaEventSynchronize(r.stop) != cudaSuccess ||
        cudaEventElapsedTime(&t, r.start, r.stop) != cudaSuccess)
      rc = -1;
    if (r.kind < n) {
      ms[r.kind] += t;
      launches[r.kind] += 1;
    }
    g_prof_free.push_back(r.start);
    g_prof_free.push_back(r.stop);
  }
  g_prof_recs.clear();
  return rc;
}

dsa_status_t dsa_selftest_wait_timeout(void* d_ws, size_t ws_bytes, dsa_stream_t stream) {
  if (dsa_status_t s = check_ws(d_ws, ws_bytes, kStatusBytes)) return s;
  return launch_status(launch_selftest_wait(static_cast<int*>(d_ws), stream), "selftest launch");
}

// ------------------------------------------------------------- a1: scores
size_t dsa_indexer_workspace_size(const dsa_batch_t*) { return kStatusBytes; }

dsa_status_t dsa_indexer_scores(const void* q_idx, const float* q_scale, const float* w,
                                const void* k_idx, const float* k_scale, int64_t k_rows,
                                dsa_dtype_t dt, const dsa_batch_t* b, float* scores, void* ws,
                                size_t ws_bytes, dsa_stream_t stream) {
  if (dsa_status_t s = check_batch(b)) return s;
  if (dsa_status_t s = check_indexer_args(q_idx, q_scale, w, k_idx, k_scale, k_rows, dt)) return s;
  if (!scores || !aligned16(scores)) return fail(DSA_ERR_INVALID_ARG, "scores must be 16-byte aligned");
  if (dsa_status_t s = check_ws(ws, ws_bytes, kStatusBytes)) return s;
  return launch_status(launch_indexer(q_idx, q_scale, w, k_idx, k_scale, k_rows,
                                      dt == DSA_FP8_E4M3, *b, scores, true,
                                      static_cast<int*>(ws), stream),
                       "indexer launch");
}

// ------------------------------------------------------------- a2: top-K
size_t dsa_topk_workspace_size(const dsa_batch_t* b, int32_t k) {
  if (!b) return kStatusBytes;
  return kStatusBytes + round256(topk_scratch_bytes(*b, k));
}

dsa_status_t dsa_topk(const float* scores, const dsa_batch_t* b, int32_t k, int32_t* idx, void* ws,
                      size_t ws_bytes, dsa_stream_t stream) {
  if (dsa_status_t s = check_batch(b)) return s;
  if (dsa_status_t s = check_topk_k(k)) return s;
  if (!scores || !idx) return fail(DSA_ERR_INVALID_ARG, "scores and idx are required");
  if (!aligned16(scores)) return fail(DSA_ERR_INVALID_ARG, "scores must be 16-byte aligned");
  const size_t need = dsa_topk_workspace_size(b, k);
  if (dsa_status_t s = check_ws(ws, ws_bytes, need)) return s;
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  return launch_status(launch_topk(scores, *b, k, idx, static_cast<int*>(ws), wsb + kStatusBytes,
                                   need - kStatusBytes, stream),
                       "top-K launch");
}

// ------------------------------------------------------------- a4-a5: sparse MLA
size_t dsa_sparse_mla_workspace_size(const dsa_batch_t* b, int32_t heads, int32_t k) {
  if (!b) return kStatusBytes;
  return kStatusBytes + round256(mla_workspace_bytes(*b, heads, k));
}

dsa_status_t dsa_sparse_mla_attn(const void* q_lat, const void* q_rope, const void* kv,
                                 int64_t kv_rows, const int32_t* idx, int32_t k, int32_t heads,
                                 float scale, const dsa_batch_t* b, void* out, float* lse, void* ws,
                                 size_t ws_bytes, dsa_stream_t stream) {
  if (dsa_status_t s = check_batch(b)) return s;
  if (dsa_status_t s = check_mla_args(q_lat, q_rope, kv, kv_rows, idx, k, heads, scale, b, out)) return s;
  const size_t need = dsa_sparse_mla_workspace_size(b, heads, k);
  if (dsa_status_t s = check_ws(ws, ws_bytes, need)) return s;
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  return launch_status(launch_sparse_mla(q_lat, q_rope, kv, kv_rows, idx, k, heads, scale, *b, out,
                                         lse, wsb + kStatusBytes, need - kStatusBytes,
                                         static_cast<int*>(ws), stream),
                       "sparse MLA launch");
}

dsa_status_t dsa_sparse_mla_attn_fp8kv(const void* q_lat, const void* q_rope, const void* kv8,
                                       int64_t kv_rows, const int32_t* idx, int32_t k,
                                       int32_t heads, float scale, const dsa_batch_t* b, void* out,
                                       float* lse, void* ws, size_t ws_bytes, dsa_stream_t stream) {
  if (dsa_status_t s = check_batch(b)) return s;
  if (dsa_status_t s = check_mla_args(q_lat, q_rope, kv8, kv_rows, idx, k, heads, scale, b, out)) return s;
  if (heads != 64) return fail(DSA_ERR_UNSUPPORTED, "FP8 KV rows: heads must be 64");
  const size_t need = dsa_sparse_mla_workspace_size(b, heads, k);
  if (dsa_status_t s = check_ws(ws, ws_bytes, need)) return s;
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  return launch_status(launch_sparse_mla(q_lat, q_rope, kv8, kv_rows, idx, k, heads, scale, *b,
                                         out, lse, wsb + kStatusBytes, need - kStatusBytes,
                                         static_cast<int*>(ws), stream, true),
                       "sparse MLA (FP8 KV) launch");
}

// ------------------------------------------------------------- a6: group
size_t dsa_group_workspace_size(const dsa_group_t* g, const dsa_batch_t* b) {
  if (!g || !b) return kStatusBytes;
  const size_t scores = round256(static_cast<size_t>(b->num_q) * static_cast<size_t>(b->max_len) * 4) +
                        group_topk_bytes(g, b);
  const size_t mla = round256(mla_workspace_bytes(*b, g->heads, g->k));
  return kStatusBytes + (scores > mla ? scores : mla);
}

dsa_status_t indexshare_group_forward(const dsa_group_t* g, const dsa_batch_t* b, int32_t* idx_buf,
                                      void* ws, size_t ws_bytes, dsa_stream_t stream) {
  if (!g) return fail(DSA_ERR_INVALID_ARG, "group is NULL");
  if (dsa_status_t s = check_batch(b)) return s;
  if (dsa_status_t s = check_group(g, b, idx_buf)) return s;
  const int nl = static_cast<int>(strlen(g->layer_types));
  const size_t need = dsa_group_workspace_size(g, b);
  if (dsa_status_t s = check_ws(ws, ws_bytes, need)) return s;
  const GroupWs w = group_ws(g, b, ws, need);
  const bool kv_fp8 = g->kv_dtype == DSA_FP8_E4M3;
  for (int l = 0; l < nl; ++l) {
    if (g->layer_types[l] == 'F')
      if (dsa_status_t s = run_f_layer(g, b, l, idx_buf, w, stream)) return s;
    // every layer: gather from its own cache + sparse attention over idx_buf
    if (dsa_status_t s = launch_status(
            launch_sparse_mla(g->q_lat[l], g->q_rope[l], g->kv[l], g->kv_rows, idx_buf, g->k,
                              g->heads, g->scale, *b, g->out[l], g->lse ? g->lse[l] : nullptr,
                              w.mla_extra, w.mla_extra_bytes, w.status, stream, kv_fp8, false,
                              true,  // after the group's own F-layer or attention kernels
                              g->layer_types[l] == 'S'),  // right after the previous layer's
            "sparse MLA launch"))
      return s;
  }
  return DSA_OK;
}

// ------------------------------------------------------------- hot / cold KV
dsa_status_t dsa_hot_plan(const int32_t* idx, int32_t k, const dsa_batch_t* b, const dsa_hot_t* h,
                          int32_t step, int32_t* rows, void* ws, size_t ws_bytes,
                          dsa_stream_t stream) {
  if (dsa_status_t s = check_batch(b)) return s;
  if (dsa_status_t s = check_hot(h, b)) return s;
  if (k < 1 || k > 4096) return fail(DSA_ERR_UNSUPPORTED, "k=%d (supported: 1..4096)", k);
  if (step < 0) return fail(DSA_ERR_INVALID_ARG, "step < 0");
  if (b->num_q > 0 && (!idx || !rows)) return fail(DSA_ERR_INVALID_ARG, "idx and rows are required");
  if (static_cast<int64_t>(b->num_q) * k > (int64_t(1) << 31) - 4)
    return fail(DSA_ERR_UNSUPPORTED, "num_q * k >= 2^31");
  if (dsa_status_t s = check_ws(ws, ws_bytes, kStatusBytes)) return s;
  return launch_status(launch_hot_plan(idx, k, *b, *h, step, rows, static_cast<int*>(ws), stream),
                       "hot plan launch");
}

namespace {
dsa_status_t hot_fetch_impl(const dsa_hot_t* h, const dsa_batch_t* b, int32_t layers,
                            const void* const* cold_kv, int64_t cold_rows, void* const* hot_kv,
                            dsa_dtype_t kv_dtype, int* status, cudaStream_t stream) {
  if (kv_dtype != DSA_BF16 && kv_dtype != DSA_FP8_E4M3) return fail(DSA_ERR_UNSUPPORTED, "kv_dtype");
  if (layers < 0 || layers > 4096) return fail(DSA_ERR_INVALID_ARG, "layers=%d", layers);
  if (layers == 0) return DSA_OK;
  if (!cold_kv || !hot_kv) return fail(DSA_ERR_INVALID_ARG, "cold_kv and hot_kv are required");
  if (cold_rows < 1) return fail(DSA_ERR_INVALID_ARG, "cold_rows < 1");
  std::vector<const void*> cold(static_cast<size_t>(layers));
  for (int l = 0; l < layers; ++l) {
    if (dsa_status_t s = device_view(cold_kv[l], "cold_kv", l, &cold[l])) return s;
    if (!hot_kv[l] || !aligned16(hot_kv[l]))
      return fail(DSA_ERR_INVALID_ARG, "hot_kv[%d] must be a 16-byte aligned device pointer", l);
  }
  const int row_bytes = kv_dtype == DSA_FP8_E4M3 ? DSA_KV_ROW_BYTES_FP8 : DSA_KV_ROW_BYTES;
  return launch_status(launch_hot_fetch(*h, *b, layers, cold.data(), cold_rows, hot_kv, row_bytes,
                                        status, stream),
                       "hot fetch launch");
}
}  // namespace

dsa_status_t dsa_hot_fetch(const dsa_hot_t* h, const dsa_batch_t* b, int32_t layers,
                           const void* const* cold_kv, int64_t cold_rows, void* const* hot_kv,
                           int64_t hot_rows, dsa_dtype_t kv_dtype, void* ws, size_t ws_bytes,
                           dsa_stream_t stream) {
  if (dsa_status_t s = check_batch(b)) return s;
  if (dsa_status_t s = check_hot(h, b)) return s;
  if (hot_rows < static_cast<int64_t>(b->num_seqs) * h->hot_slots)
    return fail(DSA_ERR_INVALID_ARG, "hot_rows=%lld < num_seqs * hot_slots",
                static_cast<long long>(hot_rows));
  if (dsa_status_t s = check_ws(ws, ws_bytes, kStatusBytes)) return s;
  return hot_fetch_impl(h, b, layers, cold_kv, cold_rows, hot_kv, kv_dtype, static_cast<int*>(ws),
                        stream);
}

}  // extern "C"

namespace dsa {
// hot.cu: one device read per `stride` bytes of each cold cache
cudaError_t launch_hot_touch(int layers, const void* const* cold, int64_t bytes, int64_t stride,
                             cudaStream_t stream);
}  // namespace dsa

extern "C" {

dsa_status_t dsa_hot_touch(int32_t layers, const void* const* cold_kv, int64_t cold_bytes,
                           int64_t stride, dsa_stream_t stream) {
  if (layers < 0 || layers > 4096) return fail(DSA_ERR_INVALID_ARG, "layers=%d", layers);
  if (layers == 0) return DSA_OK;
  if (!cold_kv) return fail(DSA_ERR_INVALID_ARG, "cold_kv is required");
  if (cold_bytes < 16 || cold_bytes % 16 != 0)
    return fail(DSA_ERR_INVALID_ARG, "cold_bytes must be a positive multiple of 16");
  if (stride < 16 || stride % 16 != 0) return fail(DSA_ERR_INVALID_ARG, "stride must be a multiple of 16");
  std::vector<const void*> cold(static_cast<size_t>(layers));
  for (int l = 0; l < layers; ++l)
    if (dsa_status_t s = device_view(cold_kv[l], "cold_kv", l, &cold[l])) return s;
  return launch_status(launch_hot_touch(layers, cold.data(), cold_bytes, stride, stream),
                       "hot touch launch");
}

dsa_status_t dsa_sparse_mla_attn_rows(const void* q_lat, const void* q_rope, const void* kv,
                                      int64_t kv_rows, dsa_dtype_t kv_dtype, const int32_t* rows,
                                      int32_t k, int32_t heads, float scale, const dsa_batch_t* b,
                                      void* out, float* lse, void* ws, size_t ws_bytes,
                                      dsa_stream_t stream) {
  if (dsa_status_t s = check_batch(b)) return s;
  if (dsa_status_t s = check_mla_args(q_lat, q_rope, kv, kv_rows, rows, k, heads, scale, b, out)) return s;
  if (kv_dtype != DSA_BF16 && kv_dtype != DSA_FP8_E4M3) return fail(DSA_ERR_UNSUPPORTED, "kv_dtype");
  const bool kv_fp8 = kv_dtype == DSA_FP8_E4M3;
  if (kv_fp8 && heads != 64) return fail(DSA_ERR_UNSUPPORTED, "FP8 KV rows: heads must be 64");
  const size_t need = dsa_sparse_mla_workspace_size(b, heads, k);
  if (dsa_status_t s = check_ws(ws, ws_bytes, need)) return s;
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  return launch_status(launch_sparse_mla(q_lat, q_rope, kv, kv_rows, rows, k, heads, scale, *b, out,
                                         lse, wsb + kStatusBytes, need - kStatusBytes,
                                         static_cast<int*>(ws), stream, kv_fp8, true),
                       "sparse MLA (rows) launch");
}

dsa_status_t indexshare_group_forward_hot(const dsa_group_t* g, const dsa_batch_t* b,
                                          const dsa_hot_group_t* hot, int32_t* idx_buf, void* ws,
                                          size_t ws_bytes, dsa_stream_t stream) {
  if (!g) return fail(DSA_ERR_INVALID_ARG, "group is NULL");
  if (!hot) return fail(DSA_ERR_INVALID_ARG, "hot group is NULL");
  if (dsa_status_t s = check_batch(b)) return s;
  if (dsa_status_t s = check_group(g, b, idx_buf)) return s;
  const int nl = static_cast<int>(strlen(g->layer_types));
  int nf = 0;
  for (int l = 0; l < nl; ++l) nf += g->layer_types[l] == 'F';
  if (hot->n_spans != nf || !hot->spans)
    return fail(DSA_ERR_INVALID_ARG, "hot->n_spans=%d, layer_types has %d F layers", hot->n_spans, nf);
  if (!hot->rows || !hot->cold_kv) return fail(DSA_ERR_INVALID_ARG, "hot->rows and hot->cold_kv are required");
  if (hot->step < 0) return fail(DSA_ERR_INVALID_ARG, "hot->step < 0");
  for (int i = 0; i < nf; ++i) {
    if (dsa_status_t s = check_hot(&hot->spans[i], b)) return s;
    if (g->kv_rows < static_cast<int64_t>(b->num_seqs) * hot->spans[i].hot_slots)
      return fail(DSA_ERR_INVALID_ARG, "kv_rows=%lld < num_seqs * hot_slots of span %d",
                  static_cast<long long>(g->kv_rows), i);
  }
  if (static_cast<int64_t>(b->num_q) * g->k > (int64_t(1) << 31) - 4)
    return fail(DSA_ERR_UNSUPPORTED, "num_q * k >= 2^31");
  const size_t need = dsa_group_workspace_size(g, b);
  if (dsa_status_t s = check_ws(ws, ws_bytes, need)) return s;
  const GroupWs w = group_ws(g, b, ws, need);
  const bool kv_fp8 = g->kv_dtype == DSA_FP8_E4M3;
  int span = -1;
  for (int l = 0; l < nl; ++l) {
    if (g->layer_types[l] == 'F') {
      ++span;
      if (dsa_status_t s = run_f_layer(g, b, l, idx_buf, w, stream)) return s;
      // one plan for the span, then the span's missing rows for all of its layers
      const dsa_hot_t& h = hot->spans[span];
      if (dsa_status_t s = launch_status(
              launch_hot_plan(idx_buf, g->k, *b, h, hot->step, hot->rows, w.status, stream),
              "hot plan launch"))
        return s;
      int l1 = l + 1;
      while (l1 < nl && g->layer_types[l1] == 'S') ++l1;
      if (dsa_status_t s = hot_fetch_impl(&h, b, l1 - l, hot->cold_kv + l, hot->cold_rows,
                                          const_cast<void* const*>(g->kv + l), g->kv_dtype, w.status,
                                          stream))
        return s;
    }
    if (dsa_status_t s = launch_status(
            launch_sparse_mla(g->q_lat[l], g->q_rope[l], g->kv[l], g->kv_rows, hot->rows, g->k,
                              g->heads, g->scale, *b, g->out[l], g->lse ? g->lse[l] : nullptr,
                              w.mla_extra, w.mla_extra_bytes, w.status, stream, kv_fp8, true,
                              true, g->layer_types[l] == 'S'),
            "sparse MLA launch"))
      return s;
  }
  return DSA_OK;
}

// ------------------------------------------------------------- a7: FP8 quantiser
dsa_status_t dsa_fp8_quantize(const void* x, int64_t rows, uint8_t* codes, float* scale,
                              dsa_stream_t stream) {
  if (rows < 0) return fail(DSA_ERR_INVALID_ARG, "rows < 0");
  if (rows > 0 && (!x || !codes || !scale))
    return fail(DSA_ERR_INVALID_ARG, "x, codes and scale are required");
  if (rows > 0 && (!aligned16(x) || !aligned16(codes)))
    return fail(DSA_ERR_INVALID_ARG, "x and codes must be 16-byte aligned");
  if (rows > (int64_t(1) << 34)) return fail(DSA_ERR_UNSUPPORTED, "rows too large");
  return launch_status(launch_quantize(x, rows, codes, scale, stream), "quantiser launch");
}

// ------------------------------------------------------------- FP8 KV rows
dsa_status_t dsa_kv_fp8_quantize(const void* kv, int64_t rows, uint8_t* out, dsa_stream_t stream) {
  if (rows < 0) return fail(DSA_ERR_INVALID_ARG, "rows < 0");
  if (rows > 0 && (!kv || !out)) return fail(DSA_ERR_INVALID_ARG, "kv and out are required");
  if (rows > 0 && (!aligned16(kv) || !aligned16(out)))
    return fail(DSA_ERR_INVALID_ARG, "kv and out must be 16-byte aligned");
  if (rows > (int64_t(1) << 33)) return fail(DSA_ERR_UNSUPPORTED, "rows too large");
  return launch_status(launch_kv_fp8_quantize(kv, rows, out, stream), "KV quantiser launch");
}

// ------------------------------------------------------------- indexer cache append
dsa_status_t dsa_indexer_append_keys(const void* k_new, const int32_t* k_seq,
                                     const int32_t* k_pos, int32_t n, const dsa_batch_t* b,
                                     dsa_dtype_t dt, const double* inv_freq, void* k_cache,
                                     float* k_scale, int64_t k_rows, void* ws, size_t ws_bytes,
                                     dsa_stream_t stream) {
  if (dsa_status_t s = check_batch(b)) return s;
  if (n < 0) return fail(DSA_ERR_INVALID_ARG, "n < 0");
  if (dt != DSA_BF16 && dt != DSA_FP8_E4M3) return fail(DSA_ERR_UNSUPPORTED, "dtype");
  if (!inv_freq) return fail(DSA_ERR_INVALID_ARG, "inv_freq (32 host doubles) is required");
  if (n > 0 && (!k_new || !k_seq || !k_pos || !k_cache || (dt == DSA_FP8_E4M3 && !k_scale)))
    return fail(DSA_ERR_INVALID_ARG, "k_new, k_seq, k_pos, k_cache (and k_scale for FP8) are required");
  if (n > 0 && (!aligned16(k_new) || !aligned16(k_cache)))
    return fail(DSA_ERR_INVALID_ARG, "k_new and k_cache must be 16-byte aligned");
  if (k_rows < 1) return fail(DSA_ERR_INVALID_ARG, "k_rows < 1");
  if (dsa_status_t s = check_ws(ws, ws_bytes, kStatusBytes)) return s;
  return launch_status(launch_rope_append(k_new, n, 1, k_pos, k_seq, *b, inv_freq,
                                          dt == DSA_FP8_E4M3, k_cache, k_scale, k_rows,
                                          static_cast<int*>(ws), stream),
                       "append launch");
}

dsa_status_t dsa_indexer_prepare_queries(const void* q_new, const dsa_batch_t* b, dsa_dtype_t dt,
                                         const double* inv_freq, void* q_out, float* q_scale,
                                         void* ws, size_t ws_bytes, dsa_stream_t stream) {
  if (dsa_status_t s = check_batch(b)) return s;
  if (dt != DSA_BF16 && dt != DSA_FP8_E4M3) return fail(DSA_ERR_UNSUPPORTED, "dtype");
  if (!inv_freq) return fail(DSA_ERR_INVALID_ARG, "inv_freq (32 host doubles) is required");
  if (b->num_q > 0 && (!q_new || !q_out || (dt == DSA_FP8_E4M3 && !q_scale)))
    return fail(DSA_ERR_INVALID_ARG, "q_new, q_out (and q_scale for FP8) are required");
  if (b->num_q > 0 && (!aligned16(q_new) || !aligned16(q_out)))
    return fail(DSA_ERR_INVALID_ARG, "q_new and q_out must be 16-byte aligned");
  if (dsa_status_t s = check_ws(ws, ws_bytes, kStatusBytes)) return s;
  const int64_t nv = static_cast<int64_t>(b->num_q) * DSA_INDEX_HEADS;
  return launch_status(launch_rope_append(q_new, nv, DSA_INDEX_HEADS, b->q_pos, nullptr, *b,
                                          inv_freq, dt == DSA_FP8_E4M3, q_out, q_scale, nv,
                                          static_cast<int*>(ws), stream),
                       "query preparation launch");
}

}  // extern "C"

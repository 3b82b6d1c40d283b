// Hot/cold KV: a GPU "hot" buffer of a few thousand KV rows per sequence in
// front of the full cache held in host memory; after the top-K the selected
// rows missing from the hot buffer are swapped in, then the attention reads
// hot rows ("GLM-5.2 / 总览" glossary, HiSparse: 6144 hot slots on the GPU,
// the full KV in CPU pinned memory, on-demand swap-in after the DSA top-K;
// config table: the 1M-context cache held by a GPU hot buffer plus a CPU cold
// store).
//
// Policy, per sequence and step: hits refresh their slot's stamp; misses, in
// order of first appearance in the index buffer, take the least recently used
// slots not used at this step (smallest stamp, then lowest slot), handed out
// in increasing slot order.
//
// GB300 design.  The plan is one CTA per sequence: claims through atomicMin
// on the position -> slot map find the first appearance of every miss, block
// scans give the misses their order, a radix select over the slot stamps finds
// the LRU cut and a scan in slot order hands the chosen slots out.  The
// swap-in reads the cold rows straight from pinned host memory over
// NVLink-C2C (16-byte loads from the mapped address, one warp per row, every
// layer of the index span in one launch) and writes them into the hot rows;
// no host round trip is needed to learn which rows miss.
#include "common.cuh"

namespace dsa {
namespace {

constexpr int kPlanBS = 1024;
constexpr int kFetchBS = 256;
constexpr int kFetchLayers = 16;

struct HotArgs {
  int32_t hot_slots;
  int32_t max_pos;  // row stride of pos_slot (>= max_len)
  int32_t* slot_pos;
  int32_t* slot_stamp;
  int32_t* pos_slot;
  int32_t* fetch_pos;
  int32_t* fetch_slot;
  int32_t* fetch_count;
};

// Exclusive prefix sum of v over the CTA (thread order); *total = the sum.
// `sums` is shared scratch of kPlanBS / 32 ints.
__device__ __forceinline__ int block_excl_scan(int v, int* total, int* sums) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = sums[lane];  // kPlanBS / 32 == 32 warps
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    sums[lane] = w;
  }
  __syncthreads();
  const int before = warp ? sums[warp - 1] : 0;
  *total = sums[kPlanBS / 32 - 1];
  __syncthreads();  // sums is reused by the next scan
  return before + x - v;
}

__global__ void __launch_bounds__(kPlanBS) hot_plan_kernel(const int32_t* idx, int K,
                                                           const BatchArgs b, const HotArgs h,
                                                           int step, int32_t* rows, int* status) {
  static_assert(kPlanBS == 1024, "the scans assume 32 warps");
  extern __shared__ int32_t vict[];  // [hot_slots]: the chosen slots in slot order
  __shared__ int sums[kPlanBS / 32];
  __shared__ int hist[256];
  __shared__ int sel[2];
  const int seq = blockIdx.x, tid = threadIdx.x;
  const int H = h.hot_slots;
  int qs, qe;
  seq_rows(b, seq, status, qs, qe);
  const int64_t nent = static_cast<int64_t>(qe - qs) * K;
  int32_t* ps = h.pos_slot + static_cast<int64_t>(seq) * h.max_pos;
  int32_t* sp = h.slot_pos + static_cast<int64_t>(seq) * H;
  int32_t* ss = h.slot_stamp + static_cast<int64_t>(seq) * H;
  int32_t* fpos = h.fetch_pos + static_cast<int64_t>(seq) * H;
  int32_t* fslot = h.fetch_slot + static_cast<int64_t>(seq) * H;
  // a claim on position e by entry f; smaller f gives a smaller (winning) value, all < -1
  auto claim = [&](int64_t f) { return static_cast<int32_t>(-2 - (nent - f)); };
  // entry f = (query qs + f / K, slot f % K): its position if valid, else -1
  auto entry = [&](int64_t f, bool report) -> int {
    const int t = qs + static_cast<int>(f / K);
    const int e = idx[static_cast<int64_t>(t) * K + f % K];
    if (e == -1) return -1;
    const int pos = b.q_pos[t];
    if (e < 0 || e > pos || e >= b.max_len) {
      if (report) atomicOr(status, DSA_DEVERR_INDEX);
      return -1;
    }
    return e;
  };
  // State arrays are read with ld.global.cg (L2): other threads of this CTA
  // update them between the phases, and L1 is not coherent with their atomics.

  // ---- phase A: hits refresh their stamp, misses claim their position
  for (int64_t f = tid; f < nent; f += kPlanBS) {
    const int e = entry(f, true);
    if (e < 0) continue;
    const int v = __ldcg(&ps[e]);
    if (v >= H) {  // a state this plan did not write: leave it alone
      atomicOr(status, DSA_DEVERR_INDEX);
    } else if (v >= 0) {
      ss[v] = step;
    } else {
      atomicMin(&ps[e], claim(f));
    }
  }
  __syncthreads();

  // ---- phase B: first appearances in entry order -> the miss list
  int m = 0;
  for (int64_t c0 = 0; c0 < nent; c0 += kPlanBS) {
    const int64_t f = c0 + tid;
    int e = -1;
    bool own = false;
    if (f < nent) {
      e = entry(f, false);
      own = e >= 0 && __ldcg(&ps[e]) == claim(f);
    }
    int total;
    const int r = m + block_excl_scan(own ? 1 : 0, &total, sums);
    if (own && r < H) fpos[r] = e;
    m += total;
  }

  // ---- phase C: enough unused slots?  (stamps of this step's hits are final)
  int nfree_local = 0;
  for (int s = tid; s < H; s += kPlanBS) nfree_local += __ldcg(&ss[s]) < step ? 1 : 0;
  int nfree;
  block_excl_scan(nfree_local, &nfree, sums);
  if (m > nfree) {  // overflow: no slot changes, the claims are withdrawn
    if (tid == 0) {
      atomicOr(status, DSA_DEVERR_HOT_OVERFLOW);
      h.fetch_count[seq] = 0;
    }
    for (int64_t f = tid; f < nent; f += kPlanBS) {
      const int t = qs + static_cast<int>(f / K);
      rows[static_cast<int64_t>(t) * K + f % K] = -1;
      const int e = entry(f, false);
      if (e >= 0 && __ldcg(&ps[e]) < -1) ps[e] = -1;
    }
    return;
  }

  // ---- the m least recently used unused slots: radix select of the m-th
  // smallest key stamp + 1 (>= 0) among them, then the ties by slot index
  uint32_t pv = 0;
  int need = m;
  if (m > 0) {
    for (int shift = 24; shift >= 0; shift -= 8) {
      for (int i = tid; i < 256; i += kPlanBS) hist[i] = 0;
      __syncthreads();
      for (int s = tid; s < H; s += kPlanBS) {
        const int st = __ldcg(&ss[s]);
        if (st >= step) continue;
        const uint32_t key = static_cast<uint32_t>(st + 1);
        if ((static_cast<uint64_t>(key) >> (shift + 8)) != pv) continue;
        atomicAdd(&hist[(key >> shift) & 255u], 1);
      }
      __syncthreads();
      if (tid < 32) {
        int c[8], sum = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          c[j] = hist[tid * 8 + j];
          sum += c[j];
        }
        int incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, o);
          if (tid >= o) incl += y;
        }
        int acc = incl - sum;
        if (acc < need && need <= incl) {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            if (acc < need && need <= acc + c[j]) {
              sel[0] = tid * 8 + j;
              sel[1] = need - acc;
            }
            acc += c[j];
          }
        }
      }
      __syncthreads();
      pv = (pv << 8) | static_cast<uint32_t>(sel[0]);
      need = sel[1];
      __syncthreads();
    }
  }
  const uint32_t cut = pv;  // the m-th smallest key; `need` of its slots are taken
  // chosen slots in slot order: thread tid owns slots [lo, hi)
  const int per = (H + kPlanBS - 1) / kPlanBS;  // <= 16
  const int lo = min(tid * per, H), hi = min(lo + per, H);
  int eq_local = 0;
  if (m > 0)
    for (int s = lo; s < hi; ++s) {
      const int st = __ldcg(&ss[s]);
      eq_local += (st < step && static_cast<uint32_t>(st + 1) == cut) ? 1 : 0;
    }
  int tmp;
  int eq_rank = block_excl_scan(eq_local, &tmp, sums);
  uint32_t mine = 0;
  int nv_local = 0;
  if (m > 0)
    for (int s = lo; s < hi; ++s) {
      const int st = __ldcg(&ss[s]);
      if (st >= step) continue;
      const uint32_t key = static_cast<uint32_t>(st + 1);
      bool take = key < cut;
      if (key == cut) take = eq_rank++ < need;
      if (take) {
        mine |= 1u << (s - lo);
        ++nv_local;
      }
    }
  int nv;
  int vbase = block_excl_scan(nv_local, &nv, sums);
  for (int s = lo; s < hi; ++s)
    if (mine >> (s - lo) & 1u) vict[vbase++] = s;
  __syncthreads();

  // ---- phase D: evict, then install the misses
  for (int r = tid; r < m; r += kPlanBS) {
    const int s = vict[r];
    const int old = __ldcg(&sp[s]);
    if (old >= 0 && old < h.max_pos) ps[old] = -1;
    fslot[r] = s;
  }
  __syncthreads();
  for (int r = tid; r < m; r += kPlanBS) {
    const int s = vict[r];
    const int e = __ldcg(&fpos[r]);
    ps[e] = s;
    sp[s] = e;
    ss[s] = step;
  }
  if (tid == 0) h.fetch_count[seq] = m;
  __syncthreads();

  // ---- phase E: hot rows of every entry
  for (int64_t f = tid; f < nent; f += kPlanBS) {
    const int t = qs + static_cast<int>(f / K);
    const int e = entry(f, false);
    const int v = e >= 0 ? __ldcg(&ps[e]) : -1;
    rows[static_cast<int64_t>(t) * K + f % K] = (v >= 0 && v < H) ? seq * H + v : -1;
  }
}

struct FetchLayers {
  const uint8_t* cold[kFetchLayers];
  uint8_t* hot[kFetchLayers];
  int n;
};

// Swap-in: warp w of CTA (x, seq) copies fetch entries r = x * 8 + w, + 8 *
// gridDim.x, ... of the sequence, every layer, 16 bytes per lane per load.
template <int ROWB>
__global__ void __launch_bounds__(kFetchBS) hot_fetch_kernel(const HotArgs h, const BatchArgs b,
                                                             const FetchLayers L,
                                                             int64_t cold_rows, int* status) {
  constexpr int NCH = ROWB / 16, PER = (NCH + 31) / 32;
  static_assert(ROWB % 16 == 0, "rows are moved in 16-byte pieces");
  constexpr int WPB = kFetchBS / 32;
  const int seq = blockIdx.y;
  const int H = h.hot_slots;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m = min(__ldcg(&h.fetch_count[seq]), H);
  const int64_t base = seq_base_row(b, seq);
  for (int r = blockIdx.x * WPB + warp; r < m; r += gridDim.x * WPB) {
    const int e = __ldcg(&h.fetch_pos[static_cast<int64_t>(seq) * H + r]);
    const int s = __ldcg(&h.fetch_slot[static_cast<int64_t>(seq) * H + r]);
    const int64_t src = (e >= 0 && e < b.max_len) ? cache_row(b, seq, base, e) : -1;
    if (src < 0 || src >= cold_rows || s < 0 || s >= H) {
      if (lane == 0) atomicOr(status, DSA_DEVERR_INDEX);
      continue;
    }
    const int64_t dst = static_cast<int64_t>(seq) * H + s;
    // the rows of up to four layers are all in flight before any is stored
    // (a host read is a long round trip; stores could alias the loads, so the
    // compiler would not hoist them on its own)
    for (int l0 = 0; l0 < L.n; l0 += 4) {
      uint4 v[4][PER];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if (l0 + q >= L.n) break;
        const uint4* from = reinterpret_cast<const uint4*>(L.cold[l0 + q] + src * ROWB);
#pragma unroll
        for (int j = 0; j < PER; ++j)
          if (lane + 32 * j < NCH) v[q][j] = from[lane + 32 * j];
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if (l0 + q >= L.n) break;
        uint4* to = reinterpret_cast<uint4*>(L.hot[l0 + q] + dst * ROWB);
#pragma unroll
        for (int j = 0; j < PER; ++j)
          if (lane + 32 * j < NCH) to[lane + 32 * j] = v[q][j];
      }
    }
  }
}

// One read every `stride` bytes of each cold cache, so that the device-side
// translations of its host pages exist before the first swap-in (a first
// access to a host page costs far more than a later one).  The loads are
// volatile, so they are issued although nothing uses their values.
__global__ void __launch_bounds__(256) hot_touch_kernel(const FetchLayers L, int64_t bytes,
                                                        int64_t stride) {
  const int64_t per = (bytes + stride - 1) / stride;
  const int64_t total = per * L.n;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int l = static_cast<int>(i / per);
    const int64_t off = (i % per) * stride;
    asm volatile("{\n\t.reg .u32 t;\n\tld.volatile.global.u32 t, [%0];\n\t}" ::"l"(L.cold[l] + off) : "memory");
  }
}

HotArgs to_hot(const dsa_hot_t& h) {
  return HotArgs{h.hot_slots, h.max_pos, h.slot_pos, h.slot_stamp, h.pos_slot,
                 h.fetch_pos, h.fetch_slot, h.fetch_count};
}

}  // namespace

cudaError_t launch_hot_plan(const int32_t* idx, int k, const dsa_batch_t& b, const dsa_hot_t& h,
                            int step, int32_t* rows, int* status, cudaStream_t stream) {
  const size_t smem = static_cast<size_t>(h.hot_slots) * 4;
  static int configured_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device != dev) {
    cudaError_t e = cudaFuncSetAttribute(hot_plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(DSA_HOT_MAX_SLOTS * 4));
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  prof_begin(stream);
  hot_plan_kernel<<<static_cast<unsigned>(b.num_seqs), kPlanBS, smem, stream>>>(
      idx, k, to_args(b), to_hot(h), step, rows, status);
  prof_end(kLaunchHot, stream);
  count_launch(kLaunchHot);
  return cudaGetLastError();
}

cudaError_t launch_hot_fetch(const dsa_hot_t& h, const dsa_batch_t& b, int layers,
                             const void* const* cold, int64_t cold_rows, void* const* hot,
                             int row_bytes, int* status, cudaStream_t stream) {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  // about eight CTAs per SM over the whole batch, at most one warp per slot
  const int per_seq_max = (h.hot_slots + kFetchBS / 32 - 1) / (kFetchBS / 32);
  int gx = (8 * sms + b.num_seqs - 1) / b.num_seqs;
  gx = gx < 1 ? 1 : (gx > per_seq_max ? per_seq_max : gx);
  for (int l0 = 0; l0 < layers; l0 += kFetchLayers) {
    FetchLayers L{};
    L.n = layers - l0 < kFetchLayers ? layers - l0 : kFetchLayers;
    for (int i = 0; i < L.n; ++i) {
      L.cold[i] = static_cast<const uint8_t*>(cold[l0 + i]);
      L.hot[i] = static_cast<uint8_t*>(hot[l0 + i]);
    }
    const dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(b.num_seqs));
    prof_begin(stream);
    if (row_bytes == DSA_KV_ROW_BYTES_FP8)
      hot_fetch_kernel<DSA_KV_ROW_BYTES_FP8><<<grid, kFetchBS, 0, stream>>>(to_hot(h), to_args(b), L,
                                                                            cold_rows, status);
    else
      hot_fetch_kernel<DSA_KV_ROW_BYTES><<<grid, kFetchBS, 0, stream>>>(to_hot(h), to_args(b), L,
                                                                        cold_rows, status);
    prof_end(kLaunchFetch, stream);
    count_launch(kLaunchFetch);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_hot_touch(int layers, const void* const* cold, int64_t bytes, int64_t stride,
                             cudaStream_t stream) {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  for (int l0 = 0; l0 < layers; l0 += kFetchLayers) {
    FetchLayers L{};
    L.n = layers - l0 < kFetchLayers ? layers - l0 : kFetchLayers;
    for (int i = 0; i < L.n; ++i) L.cold[i] = static_cast<const uint8_t*>(cold[l0 + i]);
    hot_touch_kernel<<<static_cast<unsigned>(8 * sms), 256, 0, stream>>>(L, bytes, stride);
    count_launch(kLaunchOther);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace dsa

// Top-K selection of the indexer scores ("GLM-5.2 架构深度拆解" CH 2.2: keep
// the top 2048 positions as the sparse set; "GLM-5 -> 5.1 -> 5.2" section 10:
// the shared indices are written once into the group's buffer).
//
// For each query row t (length len = q_pos[t] + 1) the k largest scores are
// found by an exact three-pass radix select on the order-preserving 32-bit
// image of the fp32 score (11 + 11 + 10 bits), then written by an ordered
// compaction: position s goes to slot (#greater before s) + min(#equal
// before s, need), which yields every position above the threshold plus the
// `need` lowest positions equal to it, in ascending order, independent of
// thread scheduling.
//
// A row is handled by one CTA, or by a cluster of CL CTAs each owning a
// contiguous slice that it may stage in shared memory once;
// per-pass histograms and slice counts are merged through distributed
// shared memory, so long rows (128K..1M) spread over several SMs without any
// global atomics or spin-waits.
#include "common.cuh"

namespace dsa {
namespace {

constexpr int kStageMax = 18432;                 // positions staged per CTA
constexpr int kStageBytesMax = kStageMax * 4;    // 72 KB of shared memory

__device__ __forceinline__ uint32_t order_key(float x) {
  const uint32_t u = __float_as_uint(x);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive prefix sum over the CTA in thread order; *total gets the sum.
template <int BS>
__device__ __forceinline__ int block_excl_scan(int v, int* warp_sums, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < BS / 32 ? warp_sums[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    warp_sums[lane] = w;  // inclusive
  }
  __syncthreads();
  const int before = warp > 0 ? warp_sums[warp - 1] : 0;
  *total = warp_sums[BS / 32 - 1];
  __syncthreads();
  return before + x - v;
}

// STAGE: the CTA's slice of the row is read from global memory once, as
// order keys into shared memory, and every pass runs from there; otherwise
// each pass re-reads the slice from global memory (L2).
template <int CL, int BS, bool STAGE>
__global__ void __launch_bounds__(BS) topk_kernel(const float* __restrict__ scores, BatchArgs b,
                                                  int K, int32_t* __restrict__ idx, int* status) {
  extern __shared__ uint32_t skeys[];
  __shared__ int hist[2048];
  __shared__ int tot[CL > 1 ? 2048 : 1];
  __shared__ int warp_sums[32];
  __shared__ int s_digit, s_above;
  __shared__ int s_cnt[2];
  const int tid = threadIdx.x;
  const int t = blockIdx.x / CL;
  const int rank = CL > 1 ? static_cast<int>(cluster_ctarank()) : 0;
  const int pos = query_pos(b, t, (rank == 0 && tid == 0) ? status : nullptr);
  const int len = pos + 1;
  int32_t* out = idx + static_cast<int64_t>(t) * K;
  if (len <= K) {  // every visible position, then -1 padding (uniform over the cluster)
    for (int j = rank * BS + tid; j < K; j += CL * BS) out[j] = j < len ? j : -1;
    return;
  }
  const float* row = scores + static_cast<int64_t>(t) * b.max_len;
  const int chunk = (((len + CL - 1) / CL) + 3) & ~3;
  const int lo = min(rank * chunk, len);
  const int hi = min(lo + chunk, len);
  const int hi4 = lo + ((hi - lo) & ~3);
  if constexpr (STAGE) {
    for (int s = lo + tid * 4; s < hi4; s += BS * 4) {
      const float4 v = *reinterpret_cast<const float4*>(row + s);
      *reinterpret_cast<uint4*>(skeys + (s - lo)) =
          make_uint4(order_key(v.x), order_key(v.y), order_key(v.z), order_key(v.w));
    }
    for (int s = hi4 + tid; s < hi; s += BS) skeys[s - lo] = order_key(row[s]);
    __syncthreads();
  }
  // order key of position s of this CTA's slice
  auto key_at = [&](int s) -> uint32_t {
    if constexpr (STAGE) return skeys[s - lo];
    else return order_key(row[s]);
  };

  uint32_t prefix = 0;
  int need = K;
#pragma unroll 1
  for (int pass = 0; pass < 3; ++pass) {
    const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
    const int bits = pass == 2 ? 10 : 11;
    const int nbins = 1 << bits;
    for (int i = tid; i < nbins; i += BS) hist[i] = 0;
    __syncthreads();
    auto add = [&](uint32_t k) {
      if (pass == 0 || (k >> (shift + bits)) == prefix)
        atomicAdd(&hist[(k >> shift) & (nbins - 1)], 1);
    };
    for (int s = lo + tid * 4; s < hi4; s += BS * 4) {
      uint4 k4;
      if constexpr (STAGE) {
        k4 = *reinterpret_cast<const uint4*>(skeys + (s - lo));
      } else {
        const float4 v = *reinterpret_cast<const float4*>(row + s);
        k4 = make_uint4(order_key(v.x), order_key(v.y), order_key(v.z), order_key(v.w));
      }
      add(k4.x);
      add(k4.y);
      add(k4.z);
      add(k4.w);
    }
    for (int s = hi4 + tid; s < hi; s += BS) add(key_at(s));
    __syncthreads();
    const int* cnt = hist;
    if constexpr (CL > 1) {
      cluster_sync();
      for (int i = tid; i < nbins; i += BS) {
        const uint32_t a = smem_u32(&hist[i]);
        int sum = 0;
#pragma unroll
        for (int r = 0; r < CL; ++r) sum += static_cast<int>(ld_dsmem_u32(mapa_shared(a, r)));
        tot[i] = sum;
      }
      cluster_sync();
      cnt = tot;
    }
    // digit d with count(bins above d) < need <= count(bins >= d); bins are
    // walked from the top, each thread owning `per` consecutive bins
    const int per = (nbins + BS - 1) / BS;
    int local = 0;
    for (int k = 0; k < per; ++k) {
      const int bb = nbins - 1 - (tid * per + k);
      if (bb >= 0) local += cnt[bb];
    }
    int total;
    int running = block_excl_scan<BS>(local, warp_sums, &total);
    for (int k = 0; k < per; ++k) {
      const int bb = nbins - 1 - (tid * per + k);
      if (bb < 0) break;
      const int c = cnt[bb];
      if (running < need && running + c >= need) {
        s_digit = bb;
        s_above = running;
      }
      running += c;
    }
    __syncthreads();
    need -= s_above;
    prefix = (prefix << bits) | static_cast<uint32_t>(s_digit);
    __syncthreads();
  }
  const uint32_t thr = prefix;  // the k-th largest key; take `need` of the keys equal to it

  // ---- slice counts, cluster prefix
  int cg = 0, ce = 0;
  for (int s = lo + tid; s < hi; s += BS) {
    const uint32_t k = key_at(s);
    cg += k > thr;
    ce += k == thr;
  }
  int tot_g, tot_e;
  block_excl_scan<BS>(cg, warp_sums, &tot_g);
  block_excl_scan<BS>(ce, warp_sums, &tot_e);
  int gt_base = 0, eq_base = 0;
  if constexpr (CL > 1) {
    if (tid == 0) {
      s_cnt[0] = tot_g;
      s_cnt[1] = tot_e;
    }
    cluster_sync();
    for (int r = 0; r < rank; ++r) {
      gt_base += static_cast<int>(ld_dsmem_u32(mapa_shared(smem_u32(&s_cnt[0]), r)));
      eq_base += static_cast<int>(ld_dsmem_u32(mapa_shared(smem_u32(&s_cnt[1]), r)));
    }
  }

  // ---- ordered compaction in tiles of 4 * BS positions
  int run_g = gt_base, run_e = eq_base;
#pragma unroll 1
  for (int base = lo; base < hi; base += 4 * BS) {
    const int s0 = base + tid * 4;
    uint32_t k4[4];
    int ng = 0, ne = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      k4[q] = (s0 + q < hi) ? key_at(s0 + q) : 0u;
      const bool in = s0 + q < hi;
      ng += in && k4[q] > thr;
      ne += in && k4[q] == thr;
    }
    int tile_tot;
    const int ex = block_excl_scan<BS>(ng | (ne << 16), warp_sums, &tile_tot);
    int g = run_g + (ex & 0xFFFF);
    int e = run_e + (ex >> 16);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (s0 + q >= hi) break;
      if (k4[q] > thr) {
        const int slot = g + min(e, need);
        if (slot < K) out[slot] = s0 + q;
        ++g;
      } else if (k4[q] == thr) {
        if (e < need && g + e < K) out[g + e] = s0 + q;
        ++e;
      }
    }
    run_g += tile_tot & 0xFFFF;
    run_e += tile_tot >> 16;
  }
  if constexpr (CL > 1) cluster_sync();  // keep s_cnt alive until every rank has read it
}

template <int CL, int BS, bool STAGE>
cudaError_t launch_cl(const float* scores, const dsa_batch_t& b, int k, int32_t* idx, int* status,
                      size_t smem, cudaStream_t stream) {
  auto* kern = topk_kernel<CL, BS, STAGE>;
  if (STAGE) {
    static int configured_device = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_device != dev) {
      cudaError_t e =
          cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kStageBytesMax);
      if (e != cudaSuccess) return e;
      configured_device = dev;
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(CL) * static_cast<unsigned>(b.num_q));
  cfg.blockDim = dim3(BS);
  cfg.dynamicSmemBytes = STAGE ? smem : 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  prof_begin(stream);
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, scores, to_args(b), k, idx, status);
  prof_end(kLaunchTopk, stream);
  count_launch(kLaunchTopk);
  return e;
}

}  // namespace

cudaError_t launch_topk(const float* scores, const dsa_batch_t& b, int k, int32_t* idx,
                        int* status, cudaStream_t stream) {
  if (b.num_q == 0) return cudaSuccess;
  // Many rows (prefill, chunked prefill): one CTA per row, its row re-read
  // from L2 per pass (rows up to 16K positions use 256 threads, longer ones
  // 1024).  Few rows (decode): a cluster of 8 CTAs per row, each staging its
  // slice in shared memory once; 1M-position rows, whose slices exceed the
  // staging buffer, make their passes over L2.
  if (static_cast<int64_t>(b.num_q) >= 2 * 152) {
    return b.max_len <= 16384 ? launch_cl<1, 256, false>(scores, b, k, idx, status, 0, stream)
                              : launch_cl<1, 1024, false>(scores, b, k, idx, status, 0, stream);
  }
  const int64_t slice = ((b.max_len + 7) / 8 + 3) & ~3;
  if (slice > kStageMax) return launch_cl<8, 1024, false>(scores, b, k, idx, status, 0, stream);
  return launch_cl<8, 1024, true>(scores, b, k, idx, status, static_cast<size_t>(slice) * 4, stream);
}

}  // namespace dsa

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
// Rows of up to 16K positions are handled by one CTA each (many rows) or by
// a cluster of CL CTAs each owning a contiguous slice that it stages in
// shared memory once (few rows), per-pass histograms and slice counts merged
// through distributed shared memory.  Longer rows go to a persistent
// one-CTA-per-SM kernel that reads each row once (32 rows or more) or, for
// fewer, to a three-launch path that spreads each row over many CTAs; see
// the sections below.
#include <algorithm>

#include "common.cuh"

namespace dsa {
namespace {

constexpr int kStageMax = 18432;                 // positions staged per CTA
constexpr int kStageBytesMax = kStageMax * 4;    // 72 KB of shared memory

// Order-preserving image of an fp32 score: a > b as floats iff key(a) >
// key(b) as unsigned integers.  -0.0 is first replaced by +0.0 so that the
// two zeros are one value (equal scores, ties to the lower position); a NaN
// with the sign bit clear ranks above +inf, one with it set below -inf.
__device__ __forceinline__ uint32_t order_key(float x) {
  uint32_t u = __float_as_uint(x);
  u = (u == 0x80000000u) ? 0u : u;
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


// ------------------------------------------------------------------ long rows
// Few long rows (decode): three launches, no inter-CTA waits.
//  1. hist:   each CTA adds a 12-bit histogram of its slice of a row into the
//             row's global histogram.
//  2. select: every CTA of the row finds the threshold bin b1 (the bin that
//             holds the k-th largest key) from that histogram, writes every
//             position of a higher bin straight to the output row and
//             appends the positions of bin b1 (the candidates) to a per-row
//             list of up to kCandCap entries.
//  3. finish: one CTA per row selects the remaining `need` positions among
//             the candidates (radix on the low 20 key bits, ties to the lower
//             position), then sorts the row's k positions ascending.  A row
//             whose candidate list overflowed rescans its scores instead.
constexpr int kHBits = 12;
constexpr int kHBins = 1 << kHBits;   // 4096 bins over key bits [31:20]
constexpr int kCandCap = 8192;        // candidates kept per row
constexpr int kLongBS = 512;
constexpr int kFinBS = 512;
constexpr int kFinDynBytes = 2 * kCandCap * 4;  // candidate keys + positions (64 KB)
constexpr int kLocalCand = 2048;                 // candidates buffered per select CTA

struct LongScratch {
  uint32_t* hist;  // [num_q][kHBins]
  int* cnt;        // [num_q][4]: written-above, candidates, b1, above-count
  int32_t* cand;   // [num_q][kCandCap]
};

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Slice [lo, hi) of a row of length len for CTA c of `split`.
__device__ __forceinline__ void slice_of(int len, int split, int c, int& lo, int& hi) {
  const int chunk = (((len + split - 1) / split) + 3) & ~3;
  lo = min(c * chunk, len);
  hi = min(lo + chunk, len);
}

__global__ void __launch_bounds__(kLongBS) topk_hist_kernel(const float* __restrict__ scores,
                                                            BatchArgs b, int K, int split,
                                                            LongScratch ws) {
  __shared__ uint32_t h[kHBins];
  const int t = blockIdx.y, tid = threadIdx.x;
  const int pos = query_pos(b, t, nullptr);
  if (pos + 1 <= K) return;
  int lo, hi;
  slice_of(pos + 1, split, blockIdx.x, lo, hi);
  if (lo >= hi) return;
  for (int i = tid; i < kHBins; i += kLongBS) h[i] = 0;
  __syncthreads();
  const float* row = scores + static_cast<int64_t>(t) * b.max_len;
  const int hi4 = lo + ((hi - lo) & ~3);
  for (int s = lo + tid * 4; s < hi4; s += kLongBS * 4) {
    const float4 v = *reinterpret_cast<const float4*>(row + s);
    atomicAdd(&h[order_key(v.x) >> 20], 1u);
    atomicAdd(&h[order_key(v.y) >> 20], 1u);
    atomicAdd(&h[order_key(v.z) >> 20], 1u);
    atomicAdd(&h[order_key(v.w) >> 20], 1u);
  }
  for (int s = hi4 + tid; s < hi; s += kLongBS) atomicAdd(&h[order_key(row[s]) >> 20], 1u);
  __syncthreads();
  uint32_t* g = ws.hist + static_cast<int64_t>(t) * kHBins;
  for (int i = tid; i < kHBins; i += kLongBS)
    if (h[i]) atomicAdd(&g[i], h[i]);
}

// Threshold bin of a row from its histogram: the bin d with
// count(bins > d) < K <= count(bins >= d).  Result in *d, *above.
template <int BS>
__device__ void threshold_bin(const uint32_t* hist, int K, int* warp_sums, int* s_d, int* s_above) {
  constexpr int per = kHBins / BS;
  const int tid = threadIdx.x;
  int local = 0;
#pragma unroll
  for (int k = 0; k < per; ++k) local += static_cast<int>(hist[kHBins - 1 - (tid * per + k)]);
  int total;
  int running = block_excl_scan<BS>(local, warp_sums, &total);
#pragma unroll
  for (int k = 0; k < per; ++k) {
    const int bb = kHBins - 1 - (tid * per + k);
    const int c = static_cast<int>(hist[bb]);
    if (running < K && running + c >= K) {
      *s_d = bb;
      *s_above = running;
    }
    running += c;
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kLongBS) topk_select_kernel(const float* __restrict__ scores,
                                                              BatchArgs b, int K, int split,
                                                              LongScratch ws, int32_t* idx) {
  __shared__ uint32_t h[kHBins];
  __shared__ int warp_sums[32];
  __shared__ int s_b1, s_above;
  const int t = blockIdx.y, tid = threadIdx.x;
  const int pos = query_pos(b, t, nullptr);
  if (pos + 1 <= K) return;
  int lo, hi;
  slice_of(pos + 1, split, blockIdx.x, lo, hi);
  if (lo >= hi) return;
  const uint32_t* g = ws.hist + static_cast<int64_t>(t) * kHBins;
  for (int i = tid; i < kHBins; i += kLongBS) h[i] = g[i];
  __syncthreads();
  threshold_bin<kLongBS>(h, K, warp_sums, &s_b1, &s_above);
  const uint32_t b1 = static_cast<uint32_t>(s_b1);
  int* cnt = ws.cnt + static_cast<int64_t>(t) * 4;
  if (tid == 0 && blockIdx.x == 0) {
    cnt[2] = s_b1;
    cnt[3] = s_above;
  }
  const float* row = scores + static_cast<int64_t>(t) * b.max_len;
  // positions of this slice above the threshold bin (fewer than K in all) and
  // in it (the candidates) are buffered in shared memory, then appended to
  // the row's lists with one global atomic each
  __shared__ int32_t sgt[4096];
  __shared__ int32_t scand[kLocalCand];
  __shared__ int s_ng, s_nc, s_bg, s_bc;
  if (tid == 0) {
    s_ng = 0;
    s_nc = 0;
  }
  __syncthreads();
  const int hi4 = lo + ((hi - lo) & ~3);
  auto visit = [&](int s, uint32_t key) {
    const uint32_t bin = key >> 20;
    if (bin > b1) {
      const int i = atomicAdd(&s_ng, 1);
      if (i < 4096) sgt[i] = s;
    } else if (bin == b1) {
      const int i = atomicAdd(&s_nc, 1);
      if (i < kLocalCand) scand[i] = s;
    }
  };
  for (int s = lo + tid * 4; s < hi4; s += kLongBS * 4) {
    const float4 v = *reinterpret_cast<const float4*>(row + s);
    visit(s, order_key(v.x));
    visit(s + 1, order_key(v.y));
    visit(s + 2, order_key(v.z));
    visit(s + 3, order_key(v.w));
  }
  for (int s = hi4 + tid; s < hi; s += kLongBS) visit(s, order_key(row[s]));
  __syncthreads();
  if (tid == 0) {
    s_bg = atomicAdd(&cnt[0], s_ng);
    // a slice with more candidates than its buffer marks the row as overflowed
    s_bc = atomicAdd(&cnt[1], s_nc <= kLocalCand ? s_nc : kCandCap + 1);
  }
  __syncthreads();
  int32_t* out = idx + static_cast<int64_t>(t) * K;
  int32_t* cand = ws.cand + static_cast<int64_t>(t) * kCandCap;
  const int ng = min(s_ng, 4096), nc = s_nc <= kLocalCand ? s_nc : 0;
  for (int i = tid; i < ng; i += kLongBS)
    if (s_bg + i < K) out[s_bg + i] = sgt[i];
  for (int i = tid; i < nc; i += kLongBS)
    if (s_bc + i < kCandCap) cand[s_bc + i] = scand[i];
}

// Radix select inside the finish kernel: among n items (key, position),
// all with key >> 20 == b1, find the key T of the need-th largest and how
// many items equal to T are taken (ties to the lower position are resolved
// afterwards).  get(i) returns the key of item i (or ~0u for a non-member).
template <int BS, typename Get>
__device__ void select_low_bits(int n, int need, Get get, uint32_t b1, int* hist2, int* warp_sums,
                                int* s_d, int* s_above, uint32_t* T, int* need_out) {
  const int tid = threadIdx.x;
  uint32_t prefix = b1;
  int rem = need;
#pragma unroll 1
  for (int pass = 0; pass < 2; ++pass) {
    const int shift = pass == 0 ? 10 : 0;
    for (int i = tid; i < 1024; i += BS) hist2[i] = 0;
    __syncthreads();
    for (int i = tid; i < n; i += BS) {
      const uint32_t k = get(i);
      if (k != ~0u && (k >> (shift + 10)) == prefix) atomicAdd(&hist2[(k >> shift) & 1023], 1);
    }
    __syncthreads();
    // digit d with count(digits above d) < rem <= count(digits >= d); thread
    // tid owns digits 1023 - tid*per - k, k < per (top first)
    constexpr int per = 1024 / BS;
    int c[per];
    int local = 0;
#pragma unroll
    for (int k = 0; k < per; ++k) {
      c[k] = hist2[1023 - (tid * per + k)];
      local += c[k];
    }
    int total;
    int run = block_excl_scan<BS>(local, warp_sums, &total);
#pragma unroll
    for (int k = 0; k < per; ++k) {
      if (run < rem && run + c[k] >= rem) {
        *s_d = 1023 - (tid * per + k);
        *s_above = run;
      }
      run += c[k];
    }
    __syncthreads();
    rem -= *s_above;
    prefix = (prefix << 10) | static_cast<uint32_t>(*s_d);
    __syncthreads();
  }
  *T = prefix;
  *need_out = rem;
}

// Items whose key equals T: the position of the need-th lowest of them (radix
// over position bits [30:20], [19:10], [9:0]), or 0x7fffffff when every tied
// item is taken.  Ends with a CTA barrier.
template <int BS, typename GetK, typename GetP>
__device__ int tied_position_cut(int n, int need, uint32_t T, GetK get_key, GetP get_pos,
                                 int* hist2, int* warp_sums, int* s_d, int* s_above, int* s_n) {
  const int tid = threadIdx.x;
  if (tid == 0) *s_n = 0;
  __syncthreads();
  int my_eq = 0;
  for (int i = tid; i < n; i += BS) my_eq += get_key(i) == T;
  atomicAdd(s_n, my_eq);
  __syncthreads();
  const bool all_ties = *s_n == need;
  __syncthreads();
  uint32_t pprefix = all_ties ? 0x7fffffffu : 0u;
  int rem = need;
#pragma unroll 1
  for (int pass = 0; pass < (all_ties ? 0 : 3); ++pass) {
    const int shift = pass == 0 ? 20 : (pass == 1 ? 10 : 0);
    const int nb = pass == 0 ? 2048 : 1024;
    for (int i = tid; i < nb; i += BS) hist2[i] = 0;
    __syncthreads();
    for (int i = tid; i < n; i += BS) {
      if (get_key(i) != T) continue;
      const uint32_t p = static_cast<uint32_t>(get_pos(i));
      if (pass == 0 || (p >> (shift + 10)) == pprefix) atomicAdd(&hist2[(p >> shift) & (nb - 1)], 1);
    }
    __syncthreads();
    // smallest digit e with count(digits below e) < rem <= count(digits <= e);
    // thread tid owns digits [tid * per, tid * per + per)
    const int per = (nb + BS - 1) / BS;  // at most 4
    int c[4] = {0, 0, 0, 0};
    int local = 0;
    for (int k = 0; k < per; ++k) {
      const int d = tid * per + k;
      c[k] = d < nb ? hist2[d] : 0;
      local += c[k];
    }
    int total;
    const int below = block_excl_scan<BS>(local, warp_sums, &total);
    int run = below;
    for (int k = 0; k < per; ++k) {
      if (run < rem && run + c[k] >= rem) {
        *s_d = tid * per + k;
        *s_above = run;
      }
      run += c[k];
    }
    __syncthreads();
    rem -= *s_above;
    pprefix = (pprefix << (pass == 0 ? 0 : 10)) | static_cast<uint32_t>(*s_d);
    __syncthreads();
  }
  return static_cast<int>(pprefix);
}

// Ascending bitonic sort of buf[0, K) in shared memory (buf holds P >= K
// entries, P the next power of two).  Ends with a CTA barrier.
template <int BS>
__device__ void sort_positions(int32_t* buf, int K) {
  const int tid = threadIdx.x;
  int P = 1;
  while (P < K) P <<= 1;
  for (int i = K + tid; i < P; i += BS) buf[i] = 0x7fffffff;
  __syncthreads();
  for (int size = 2; size <= P; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = tid; i < P; i += BS) {
        const int j = i ^ stride;
        if (j > i) {
          const bool up = (i & size) == 0;
          const int a = buf[i], c = buf[j];
          if ((a > c) == up) {
            buf[i] = c;
            buf[j] = a;
          }
        }
      }
      __syncthreads();
    }
  }
}

// Write the positions marked in bits[0, nwords) to out[0, K) in ascending
// order.  Each warp owns a contiguous segment of words and reads it 32
// consecutive words at a time (no bank conflicts), a warp prefix sum placing
// each lane's positions; warp segments are ordered by a scan of their counts.
// Flags DSA_DEVERR_BATCH when the bitmap does not hold exactly K positions.
// Ends with a CTA barrier.
template <int BS>
__device__ void bitmap_compact(const uint32_t* bits, int nwords, int K, int32_t* out,
                               int* warp_sums, int* status) {
  constexpr int NW = BS / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int per = (nwords + NW - 1) / NW;
  const int w0 = min(warp * per, nwords), w1 = min(w0 + per, nwords);
  int cnt = 0;
  for (int w = w0 + lane; w < w1; w += 32) cnt += __popc(bits[w]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
  __syncthreads();  // warp_sums may still be read by the caller's last scan
  if (lane == 0) warp_sums[warp] = cnt;
  __syncthreads();
  int base = 0, total = 0;
  for (int i = 0; i < NW; ++i) {
    const int v = warp_sums[i];
    base += i < warp ? v : 0;
    total += v;
  }
  if (threadIdx.x == 0 && total != K) atomicOr(status, DSA_DEVERR_BATCH);
  for (int c0 = w0; c0 < w1; c0 += 32) {
    const int w = c0 + lane;
    uint32_t m = w < w1 ? bits[w] : 0u;
    const int n = __popc(m);
    int incl = n;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    int slot = base + incl - n;
    while (m) {
      const int bit = __ffs(m) - 1;
      m &= m - 1;
      if (slot < K) out[slot] = w * 32 + bit;
      ++slot;
    }
    base += __shfl_sync(0xffffffffu, incl, 31);
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kFinBS, 1) topk_finish_kernel(const float* __restrict__ scores,
                                                             BatchArgs b, int K, LongScratch ws,
                                                             int32_t* idx, int* status,
                                                             int dyn_words) {
  __shared__ int hist2[2048];
  __shared__ int warp_sums[32];
  __shared__ int s_d, s_above, s_n;
  extern __shared__ uint32_t fin_dyn[];  // kFinDynBytes
  uint32_t* ckey = fin_dyn;                                        // [kCandCap]
  int32_t* cpos = reinterpret_cast<int32_t*>(fin_dyn + kCandCap);  // [kCandCap]
  int32_t* sorted = reinterpret_cast<int32_t*>(fin_dyn);           // [4096], after ckey is done
  const int t = blockIdx.x, tid = threadIdx.x;
  const int pos = query_pos(b, t, tid == 0 ? status : nullptr);
  const int len = pos + 1;
  int32_t* out = idx + static_cast<int64_t>(t) * K;
  if (len <= K) {
    for (int j = tid; j < K; j += kFinBS) out[j] = j < len ? j : -1;
    return;
  }
  const int* cnt = ws.cnt + static_cast<int64_t>(t) * 4;
  const int nabove = cnt[3];            // positions in bins above b1 (already written)
  const uint32_t b1 = static_cast<uint32_t>(cnt[2]);
  const int nc = cnt[1];
  const int need1 = K - nabove;
  if (tid == 0 && cnt[0] != nabove) atomicOr(status, DSA_DEVERR_BATCH);
  const float* row = scores + static_cast<int64_t>(t) * b.max_len;
  const bool fits = nc <= kCandCap;
  const int n = fits ? nc : len;  // overflow: scan the whole row, members are bin b1
  if (fits) {
    const int32_t* cand = ws.cand + static_cast<int64_t>(t) * kCandCap;
    for (int i = tid; i < nc; i += kFinBS) {
      const int32_t p = cand[i];
      cpos[i] = p;
      ckey[i] = order_key(row[p]);
    }
  }
  __syncthreads();
  auto get_key = [&](int i) -> uint32_t {
    if (fits) return ckey[i];
    const uint32_t k = order_key(row[i]);
    return (k >> 20) == b1 ? k : ~0u;
  };
  auto get_pos = [&](int i) -> int { return fits ? cpos[i] : i; };
  uint32_t T;
  int need;
  select_low_bits<kFinBS>(n, need1, get_key, b1, hist2, warp_sums, &s_d, &s_above, &T, &need);
  const int pstar = tied_position_cut<kFinBS>(n, need, T, get_key, get_pos, hist2, warp_sums, &s_d,
                                              &s_above, &s_n);
  if (tid == 0) s_n = nabove;
  __syncthreads();
  for (int i = tid; i < n; i += kFinBS) {
    const uint32_t k = get_key(i);
    if (k == ~0u) continue;
    if (k > T || (k == T && get_pos(i) <= pstar)) {
      const int slot = atomicAdd(&s_n, 1);
      if (slot < K) out[slot] = get_pos(i);
    }
  }
  __syncthreads();
  // ascending order: the K positions marked in a bitmap over the row (in the
  // candidate arrays' space, no longer needed) and compacted in order by one
  // prefix scan; rows beyond the bitmap's reach are sorted instead
  const int nwords = (len + 31) >> 5;
  if (nwords <= dyn_words) {
    uint32_t* bits = fin_dyn;
    for (int i = tid; i < nwords; i += kFinBS) bits[i] = 0;
    __syncthreads();
    for (int i = tid; i < K; i += kFinBS) {
      const int p = out[i];
      if (p >= 0 && p < len) atomicOr(&bits[p >> 5], 1u << (p & 31));
    }
    __syncthreads();
    bitmap_compact<kFinBS>(bits, nwords, K, out, warp_sums, status);
  } else {
    for (int i = tid; i < K; i += kFinBS) sorted[i] = out[i];
    sort_positions<kFinBS>(sorted, K);
    for (int i = tid; i < K; i += kFinBS) out[i] = sorted[i];
  }
}

// ------------------------------------------------------------------ many long rows
// Many long rows (chunked prefill: thousands of rows of 128K+ positions).
// One CTA per SM loops over rows and normally reads each row from HBM once:
//  1. a 12-bit histogram of the order keys of kPrefix positions sampled in
//     16 runs spread over the row gives a cutoff bin that leaves about 1.5
//     times the sample's share of K above it;
//  2. one pass over the row keeps every key in a bin >= the cutoff, with its
//     position, in shared memory.  With at least K keys kept (and none
//     dropped) the k-th largest key is >= the cutoff, so every key the
//     selection needs is kept, and the threshold bin (the one holding the
//     k-th largest key) follows from a histogram of the kept keys;
//  3. otherwise (an unrepresentative sample, or a buffer overflow from many
//     equal keys) the whole row is histogrammed and a second pass collects
//     the positions above the threshold bin and its members.
// The threshold bin's members are resolved as in the finish kernel above,
// the selected positions are marked in a bitmap over the row and written out
// in ascending order by one prefix scan (rows beyond the bitmap's reach use a
// sort instead).
// The scores of a row fall into few bins of the key's top 12 bits, so the
// histogram is kept in 8 copies (lane & 7 picks one; copies start 4 banks
// apart) to spread the shared-memory atomics on those bins, then summed.
constexpr int kRowBS = 1024;
constexpr int kRowWarps = kRowBS / 32;
constexpr int kHCopies = 8;
constexpr int kHStride = kHBins + 4;                      // words between histogram copies
constexpr int kRegionA = kHCopies * kHStride;             // words: copies, later hist + bitmap
constexpr int kBitWords = 28672;                          // bitmap: rows up to 917,504 positions
constexpr int kSeg = 352;                                 // buffered keys per warp
constexpr int kRowCand = kRowWarps * kSeg;                // buffer slots (warp segments)
constexpr int kPrefix = 16384;      // sampled positions whose histogram sets the capture cutoff
constexpr int kPrefixSlack = 64;
constexpr int kRowDynBytes = (kRegionA + 2 * kRowCand) * 4;  // 221,312 B: one CTA per SM
static_assert(kHBins + kBitWords <= kRegionA, "merged histogram + bitmap fit the copies' space");

// Visit positions [0, hi) of a row: f(s, order key, valid) for every
// position of warp-uniform tiles (valid false past hi), so f may use warp
// votes.  Lane l of warp w takes the float4 at w * 128 + l * 4 of every
// 4 * BS positions, UNR float4 loads issued before any is used (enough bytes
// in flight to keep HBM busy with one CTA per SM).  A float4 read up to the
// next multiple of 4 stays inside the row, whose capacity is a multiple of
// 128.
template <int BS, int UNR, typename F>
__device__ __forceinline__ void scan_row(const float* __restrict__ row, int hi, F f) {
  const int lane = threadIdx.x & 31;
  for (int wbase = (threadIdx.x >> 5) * 128; wbase < hi; wbase += BS * 4 * UNR) {
    float4 v[UNR];
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const int s = wbase + u * BS * 4 + lane * 4;
      v[u] = s < hi ? __ldg(reinterpret_cast<const float4*>(row + s))
                    : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const int s = wbase + u * BS * 4 + lane * 4;
      f(s, v[u].x, s < hi);
      f(s + 1, v[u].y, s + 1 < hi);
      f(s + 2, v[u].z, s + 2 < hi);
      f(s + 3, v[u].w, s + 3 < hi);
    }
  }
}

__global__ void __launch_bounds__(kRowBS, 1) topk_rows_kernel(const float* __restrict__ scores,
                                                             BatchArgs b, int K, int32_t* idx,
                                                             int* status) {
  extern __shared__ uint32_t row_dyn[];
  uint32_t* hcopies = row_dyn;                                  // [kHCopies][kHStride], pass 1
  uint32_t* hist = row_dyn;                                     // [kHBins], summed copies
  int* hist2 = reinterpret_cast<int*>(row_dyn);                 // after the threshold bin
  uint32_t* bits = row_dyn + kHBins;                            // [kBitWords], after the sum
  int32_t* sel = reinterpret_cast<int32_t*>(bits);              // [4096], rows beyond the bitmap
  uint32_t* ckey = row_dyn + kRegionA;                          // [kRowWarps][kSeg]
  int32_t* cpos = reinterpret_cast<int32_t*>(ckey + kRowCand);  // [kRowWarps][kSeg]
  __shared__ int warp_sums[32];
  __shared__ int s_wcnt[kRowWarps];
  __shared__ int s_d, s_above, s_n, s_b1, s_nabove, s_ns, s_cut;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t lt = lanemask_lt();
  uint32_t* hmine = hcopies + (lane & 7) * kHStride;
  uint32_t* wkey = ckey + warp * kSeg;
  int32_t* wpos = cpos + warp * kSeg;
  // sum the copies into copy 0's bins (each bin read and written by one thread)
  auto sum_copies = [&]() {
    for (int i = tid; i < kHBins; i += kRowBS) {
      uint32_t sum = 0;
#pragma unroll
      for (int c = 0; c < kHCopies; ++c) sum += hcopies[c * kHStride + i];
      hist[i] = sum;
    }
  };
  // warp-segmented buffer: slot i holds an entry when i % kSeg < its warp's count
  auto buf_key = [&](int i) -> uint32_t {
    return (i % kSeg) < s_wcnt[i / kSeg] ? ckey[i] : ~0u;
  };
#pragma unroll 1
  for (int t = blockIdx.x; t < b.num_q; t += gridDim.x) {
    const int pos = query_pos(b, t, tid == 0 ? status : nullptr);
    const int len = pos + 1;
    int32_t* out = idx + static_cast<int64_t>(t) * K;
    if (len <= K) {
      for (int j = tid; j < K; j += kRowBS) out[j] = j < len ? j : -1;
      continue;
    }
    const float* row = scores + static_cast<int64_t>(t) * b.max_len;
    const bool use_bits = len <= kBitWords * 32;
    const int nwords = (len + 31) >> 5;
    for (int i = tid; i < kRegionA; i += kRowBS) hcopies[i] = 0;
    if (tid == 0) {
      s_ns = 0;
      s_cut = 0;  // no bin found below: keep everything (overflows, second pass)
    }
    __syncthreads();
    // ---- pass 1a: histogram of a sample of kPrefix positions, 16 runs of
    // kPrefix/16 spread evenly over the row (the whole row when shorter), so
    // that scores that drift with position are sampled everywhere; a cutoff
    // bin leaving about 1.5 times the sample's share of K above it follows
    const int P0 = min(len, kPrefix);
    {
      constexpr int kRun = kPrefix / 16;
      const bool whole = len <= kPrefix;
      const int stride = (len / 16) & ~3;  // run starts stay float4-aligned
#pragma unroll 4
      for (int v = tid * 4; v < P0; v += kRowBS * 4) {
        const int s = whole ? v : (v / kRun) * stride + (v % kRun);
        const float4 x = *reinterpret_cast<const float4*>(row + s);
        atomicAdd(&hmine[order_key(x.x) >> 20], 1u);
        if (s + 1 < len) atomicAdd(&hmine[order_key(x.y) >> 20], 1u);
        if (s + 2 < len) atomicAdd(&hmine[order_key(x.z) >> 20], 1u);
        if (s + 3 < len) atomicAdd(&hmine[order_key(x.w) >> 20], 1u);
      }
    }
    auto count = [&](int, float x, bool valid) {
      if (valid) atomicAdd(&hmine[order_key(x) >> 20], 1u);
    };
    __syncthreads();
    sum_copies();
    __syncthreads();
    const int need_p =
        static_cast<int>(3 * static_cast<int64_t>(K) * P0 / (2 * static_cast<int64_t>(len))) +
        kPrefixSlack;
    threshold_bin<kRowBS>(hist, need_p, warp_sums, &s_cut, &s_d);
    const uint32_t cut = static_cast<uint32_t>(s_cut);
    // ---- pass 1b: every key of the row in a bin >= cut into this warp's
    // segment.  Compared as floats with the smallest value of bin `cut` (NaN
    // and, at a cutoff of +0, -0 are kept too: a superset is harmless).
    {
      const uint32_t k0 = cut << 20;
      const float cf = cut == 0 ? -INFINITY
                                : __uint_as_float((k0 & 0x80000000u) ? (k0 & 0x7fffffffu) : ~k0);
      int wcount = 0;  // warp-uniform
      auto capture = [&](int s, float x, bool valid) {
        const bool p = valid && !(x < cf);
        const uint32_t m = __ballot_sync(0xffffffffu, p);
        if (m) {
          if (p) {
            const int i = wcount + __popc(m & lt);
            if (i < kSeg) {
              wkey[i] = order_key(x);
              wpos[i] = s;
            }
          }
          wcount += __popc(m);
        }
      };
      scan_row<kRowBS, 8>(row, len, capture);
      if (lane == 0) s_wcnt[warp] = wcount;
    }
    for (int i = tid; i < kRegionA; i += kRowBS) hcopies[i] = 0;
    if (tid == 0) s_b1 = -1;
    __syncthreads();
    // When the threshold bin of the buffered keys (the bin of their k-th
    // largest) is >= the cutoff and no segment overflowed, at least K keys of
    // the row are in bins >= the cutoff, all of them buffered: the buffer
    // holds every key the selection needs.  Otherwise the whole row is
    // histogrammed and a second pass collects what is needed.
    bool captured = true;
    int nbuf = 0;
    for (int w = 0; w < kRowWarps; ++w) {
      captured = captured && s_wcnt[w] <= kSeg;
      nbuf += s_wcnt[w];
    }
    captured = captured && nbuf >= K;
    if (captured) {
      for (int i = tid; i < kRowCand; i += kRowBS) {
        const uint32_t k = buf_key(i);
        if (k != ~0u) atomicAdd(&hmine[k >> 20], 1u);
      }
      __syncthreads();
      sum_copies();
      __syncthreads();
      threshold_bin<kRowBS>(hist, K, warp_sums, &s_b1, &s_nabove);
      captured = s_b1 >= static_cast<int>(cut);
      if (!captured) {
        for (int i = tid; i < kRegionA; i += kRowBS) hcopies[i] = 0;
        __syncthreads();
      }
    }
    if (!captured) {
      scan_row<kRowBS, 8>(row, len, count);
      __syncthreads();
      sum_copies();
      __syncthreads();
      threshold_bin<kRowBS>(hist, K, warp_sums, &s_b1, &s_nabove);
    }
    if (use_bits)
      for (int i = tid; i < nwords; i += kRowBS) bits[i] = 0;
    __syncthreads();
    const uint32_t b1 = static_cast<uint32_t>(s_b1);
    const int nabove = s_nabove;
    auto take = [&](int s) {
      if (use_bits) {
        atomicOr(&bits[s >> 5], 1u << (s & 31));
      } else {
        const int i = atomicAdd(&s_ns, 1);
        if (i < K) sel[i] = s;
      }
    };
    if (captured) {
      for (int i = tid; i < kRowCand; i += kRowBS) {
        const uint32_t k = buf_key(i);
        if (k != ~0u && (k >> 20) > b1) take(cpos[i]);
      }
    } else {
      // ---- pass 2: positions above the threshold bin, members of it
      int wcount = 0;
      auto visit = [&](int s, float x, bool valid) {
        const uint32_t key = order_key(x);
        const uint32_t bin = key >> 20;
        if (valid && bin > b1) take(s);
        const bool p = valid && bin == b1;
        const uint32_t m = __ballot_sync(0xffffffffu, p);
        if (m) {
          if (p) {
            const int i = wcount + __popc(m & lt);
            if (i < kSeg) {
              wkey[i] = key;
              wpos[i] = s;
            }
          }
          wcount += __popc(m);
        }
      };
      scan_row<kRowBS, 8>(row, len, visit);
      __syncthreads();  // every thread has read the previous counts
      if (lane == 0) s_wcnt[warp] = wcount;
      __syncthreads();
    }
    // the threshold bin's members: from the buffer, or from the row itself
    // when a segment overflowed
    bool fits = true;
    for (int w = 0; w < kRowWarps; ++w) fits = fits && s_wcnt[w] <= kSeg;
    const int n = fits ? kRowCand : len;
    auto get_key = [&](int i) -> uint32_t {
      const uint32_t k = fits ? buf_key(i) : order_key(row[i]);
      return (k != ~0u && (k >> 20) == b1) ? k : ~0u;
    };
    auto get_pos = [&](int i) -> int { return fits ? cpos[i] : i; };
    uint32_t T;
    int need;
    select_low_bits<kRowBS>(n, K - nabove, get_key, b1, hist2, warp_sums, &s_d, &s_above, &T,
                            &need);
    const int pstar = tied_position_cut<kRowBS>(n, need, T, get_key, get_pos, hist2, warp_sums,
                                                &s_d, &s_above, &s_n);
    for (int i = tid; i < n; i += kRowBS) {
      const uint32_t k = get_key(i);
      if (k == ~0u) continue;
      if (k > T || (k == T && get_pos(i) <= pstar)) take(get_pos(i));
    }
    __syncthreads();
    if (use_bits) {
      bitmap_compact<kRowBS>(bits, nwords, K, out, warp_sums, status);
    } else {
      if (tid == 0 && s_ns != K) atomicOr(status, DSA_DEVERR_BATCH);
      sort_positions<kRowBS>(sel, K);
      for (int i = tid; i < K; i += kRowBS) out[i] = sel[i];
    }
    __syncthreads();  // the next row reuses the shared buffers
  }
}

// Rows beyond 16K positions: fewer than kRowsMin of them are spread over
// several CTAs each (the three launches above); more get a CTA each.
constexpr int kRowsMin = 32;

bool use_long_path(const dsa_batch_t& b) {
  return b.num_q < kRowsMin && b.max_len > 16384;
}

size_t round256z(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

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

cudaError_t launch_rows(const float* scores, const dsa_batch_t& b, int k, int32_t* idx, int* status,
                        cudaStream_t stream) {
  static int configured_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device != dev) {
    cudaError_t e = cudaFuncSetAttribute(topk_rows_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kRowDynBytes);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  int sms = 152;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int grid = static_cast<int>(std::min<int64_t>(b.num_q, sms));
  prof_begin(stream);
  topk_rows_kernel<<<grid, kRowBS, kRowDynBytes, stream>>>(scores, to_args(b), k, idx, status);
  prof_end(kLaunchTopk, stream);
  count_launch(kLaunchTopk);
  return cudaGetLastError();
}

}  // namespace

size_t topk_scratch_bytes(const dsa_batch_t& b, int) {
  if (b.num_q == 0 || !use_long_path(b)) return 0;
  const size_t q = static_cast<size_t>(b.num_q);
  return round256z(q * kHBins * 4) + round256z(q * 16) + round256z(q * kCandCap * 4);
}

cudaError_t launch_topk(const float* scores, const dsa_batch_t& b, int k, int32_t* idx,
                        int* status, void* scratch, size_t scratch_bytes, cudaStream_t stream) {
  if (b.num_q == 0) return cudaSuccess;
  if (use_long_path(b)) {
    if (!scratch || scratch_bytes < topk_scratch_bytes(b, k)) return cudaErrorInvalidValue;
    const size_t q = static_cast<size_t>(b.num_q);
    uint8_t* base = static_cast<uint8_t*>(scratch);
    LongScratch ws;
    ws.hist = reinterpret_cast<uint32_t*>(base);
    ws.cnt = reinterpret_cast<int*>(base + round256z(q * kHBins * 4));
    ws.cand = reinterpret_cast<int32_t*>(base + round256z(q * kHBins * 4) + round256z(q * 16));
    cudaError_t e = cudaMemsetAsync(base, 0, round256z(q * kHBins * 4) + round256z(q * 16), stream);
    if (e != cudaSuccess) return e;
    // CTAs per row: about 4 waves of 152 SMs in all, at least 8K positions each
    int split = static_cast<int>((4 * 152 + b.num_q - 1) / b.num_q);
    split = max(1, min(split, (b.max_len + 8191) / 8192));
    const dim3 grid(static_cast<unsigned>(split), static_cast<unsigned>(b.num_q));
    const BatchArgs a = to_args(b);
    prof_begin(stream);
    topk_hist_kernel<<<grid, kLongBS, 0, stream>>>(scores, a, k, split, ws);
    topk_select_kernel<<<grid, kLongBS, 0, stream>>>(scores, a, k, split, ws, idx);
    // dynamic shared memory: the candidate arrays, or the row's position
    // bitmap when larger (up to 200 KB: with the static 8 KB, inside 227 KB)
    const size_t bitmap_bytes = ((static_cast<size_t>(b.max_len) + 31) / 32) * 4;
    const size_t fin_bytes = std::max<size_t>(kFinDynBytes, std::min<size_t>(bitmap_bytes, 200 << 10));
    {
      static int configured_device = -1;
      int dev = 0;
      cudaGetDevice(&dev);
      if (configured_device != dev) {
        e = cudaFuncSetAttribute(topk_finish_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 200 << 10);
        if (e != cudaSuccess) return e;
        configured_device = dev;
      }
    }
    topk_finish_kernel<<<b.num_q, kFinBS, fin_bytes, stream>>>(scores, a, k, ws, idx, status,
                                                                static_cast<int>(fin_bytes / 4));
    prof_end(kLaunchTopk, stream);
    count_launch(kLaunchTopk);
    count_launch(kLaunchTopk);
    count_launch(kLaunchTopk);
    return cudaGetLastError();
  }
  // Rows beyond 16K positions (kRowsMin or more of them): one persistent CTA
  // per SM, a row at a time.  Many short rows (prefill): one CTA of 256
  // threads per row, its row re-read from L2 per pass.  Few short rows: a
  // cluster of 8 CTAs per row, each staging its slice in shared memory once.
  if (b.max_len > 16384) return launch_rows(scores, b, k, idx, status, stream);
  if (static_cast<int64_t>(b.num_q) >= 2 * 152)
    return launch_cl<1, 256, false>(scores, b, k, idx, status, 0, stream);
  const int64_t slice = ((b.max_len + 7) / 8 + 3) & ~3;
  return launch_cl<8, 1024, true>(scores, b, k, idx, status, static_cast<size_t>(slice) * 4, stream);
}

}  // namespace dsa

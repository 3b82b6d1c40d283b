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
  chain_wait();     // the previous kernel of the stream has completed
  chain_release();  // the next one may be scheduled
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
// Few long rows (decode of a few sequences): a row is cut into `split` slices of
// consecutive positions; three launches without inter-CTA waits, and a
// fallback launch for rows whose sample misled:
//  0. cutoff:  one CTA per row histograms a sample of the row (kPrefix
//              positions in 16 runs spread over it) and picks a cutoff bin
//              that leaves about 1.5 times the sample's share of K above it.
//  1. capture: every CTA of a row appends every key of its slice at or
//              above the cutoff (float compare, warp ballots, no atomics per
//              position) with its position to the row's capture list.
//  2. resolve and write: one CTA per row.  With at least K keys captured
//              (and none dropped) the k-th largest key is at or above the
//              cutoff, so every key the selection takes is in the list: the
//              threshold key T and the cut position pstar among keys equal
//              to T follow from radix passes over the list, and the taken
//              positions (key > T, or key == T at a position up to pstar)
//              are written in ascending order from the list alone.  A row
//              without that guarantee is marked for the fallback.
//  3. fallback: the many-rows kernel below, on the marked rows only (each
//              read in full, histogrammed, resolved exactly).
constexpr int kHBits = 12;
constexpr int kHBins = 1 << kHBits;   // 4096 bins over key bits [31:20]
constexpr int kCandCap = kTopkCandCap;  // captured keys kept per row
constexpr int kLongSlack = 16;        // sampled keys added to the cutoff's 1.5x share of K
constexpr int kLongBS = 512;
constexpr int kFinBS = 512;
constexpr int kCapSeg = 192;          // captured keys buffered per warp of a capture CTA
constexpr int kCnt = kTopkCnt;  // per-row words: 1 captured, 2 dropped, 3 cutoff, 4 T, 5 pstar, 6 fallback

struct LongScratch {
  int* cnt;          // [num_q][kCnt]
  uint32_t* ckey;    // [num_q][kCandCap] captured keys
  int32_t* cpos;     // [num_q][kCandCap] their positions
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

// Radix select of a row's threshold-bin members: among n items (key, position),
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

// Ascending bitonic sort of the positions buf[0, K), written to out[0, K).
// Thread t holds the E consecutive entries t*E .. t*E+E-1 in registers
// (P = BS*E >= K entries, the tail padded with INT_MAX): the compare-exchange
// steps of stride < E stay inside a thread, those of stride < 32*E go
// between the lanes of a warp by shuffles, and only the larger strides pass
// through shared memory (buf must hold P entries).  Ends with a CTA barrier.
template <int BS, int E>
__device__ void sort_positions_e(int32_t* buf, int K, int32_t* out) {
  constexpr int P = BS * E;
  const int tid = threadIdx.x, lane = tid & 31;
  int v[E];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int i = tid * E + e;
    v[e] = i < K ? buf[i] : 0x7fffffff;
  }
  for (int size = 2; size <= P; size <<= 1) {
    int stride = size >> 1;
    if (stride >= 32 * E) {  // across warps, through shared memory
      __syncthreads();       // every thread has read buf
#pragma unroll
      for (int e = 0; e < E; ++e) buf[tid * E + e] = v[e];
      __syncthreads();
      for (; stride >= 32 * E; stride >>= 1) {
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
#pragma unroll
      for (int e = 0; e < E; ++e) v[e] = buf[tid * E + e];
    }
    for (; stride >= E; stride >>= 1) {  // between the lanes of a warp
      const int lm = stride / E;
      const bool lower = (lane & lm) == 0;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const bool up = ((tid * E + e) & size) == 0;
        const int o = __shfl_xor_sync(0xffffffffu, v[e], lm);
        v[e] = (lower == up) ? min(v[e], o) : max(v[e], o);
      }
    }
#pragma unroll
    for (int st = E / 2; st > 0; st >>= 1) {  // inside a thread
      if (st < size) {
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const int f = e ^ st;
          if (f > e) {
            const bool up = ((tid * E + e) & size) == 0;
            const int a = v[e], c = v[f];
            if ((a > c) == up) {
              v[e] = c;
              v[f] = a;
            }
          }
        }
      }
    }
  }
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int i = tid * E + e;
    if (i < K) out[i] = v[e];
  }
  __syncthreads();
}

// The sort above for K <= 8*BS positions; buf holds max(BS, the next power
// of two >= K) entries.
template <int BS>
__device__ void sort_positions(int32_t* buf, int K, int32_t* out) {
  if (K <= BS)
    sort_positions_e<BS, 1>(buf, K, out);
  else if (K <= 2 * BS)
    sort_positions_e<BS, 2>(buf, K, out);
  else if (K <= 4 * BS)
    sort_positions_e<BS, 4>(buf, K, out);
  else
    sort_positions_e<BS, 8>(buf, K, out);
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
                                                             int* status, const int* only) {
  chain_wait();     // the previous kernel of the stream has completed
  chain_release();  // the next one may be scheduled
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
    // `only` (the long path's per-row words): rows it marks for the fallback
    if (only && only[static_cast<int64_t>(t) * kCnt + 6] == 0) continue;
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
      sort_positions<kRowBS>(sel, K, out);
    }
    __syncthreads();  // the next row reuses the shared buffers
  }
}

// Long path, launch 0: the row's cutoff from the same sample as the
// many-rows kernel (the bin leaving about 1.5 times the sample's share of K
// above it, plus kLongSlack), stored as the smallest fp32 value of that bin
// (-inf for bin 0).  The sample is histogrammed in 4 copies (lane & 3) to
// spread the shared atomics on the few bins the scores fall into.
constexpr int kCutCopies = 4;
constexpr int kCutDynBytes = kCutCopies * kHBins * 4;
__global__ void __launch_bounds__(kLongBS) topk_cutoff_kernel(const float* __restrict__ scores,
                                                              BatchArgs b, int K, LongScratch ws) {
  chain_wait();     // the previous kernel of the stream has completed
  chain_release();  // the next one may be scheduled
  extern __shared__ uint32_t cut_dyn[];  // [kCutCopies][kHBins]
  __shared__ int warp_sums[32];
  __shared__ int s_cut, s_tmp;
  const int t = blockIdx.x, tid = threadIdx.x;
  // the row's words start at zero: the later launches count into 1 and 2
  // and mark 6 (every row, short ones included: the fallback reads word 6)
  if (tid < kCnt) ws.cnt[static_cast<int64_t>(t) * kCnt + tid] = 0;
  const int pos = query_pos(b, t, nullptr);
  const int len = pos + 1;
  if (len <= K) return;
  const float* row = scores + static_cast<int64_t>(t) * b.max_len;
  for (int i = tid; i < kCutCopies * kHBins; i += kLongBS) cut_dyn[i] = 0;
  if (tid == 0) s_cut = 0;
  __syncthreads();
  uint32_t* h = cut_dyn + (tid & (kCutCopies - 1)) * kHBins;
  const int P0 = min(len, kPrefix);
  constexpr int kRun = kPrefix / 16;
  const bool whole = len <= kPrefix;
  const int stride = (len / 16) & ~3;  // run starts stay float4-aligned
  auto at = [&](int v) { return whole ? v : (v / kRun) * stride + (v % kRun); };
  // every sampled float4 of this thread is requested before any is counted
  // (one round trip to L2 instead of one per float4)
  constexpr int kCutLoads = kPrefix / (kLongBS * 4);
  static_assert(kPrefix % (kLongBS * 4) == 0, "whole float4 loads per thread");
  float4 xs[kCutLoads];
#pragma unroll
  for (int u = 0; u < kCutLoads; ++u) {
    const int v = (tid + u * kLongBS) * 4;
    xs[u] = v < P0 ? *reinterpret_cast<const float4*>(row + at(v)) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int u = 0; u < kCutLoads; ++u) {
    const int v = (tid + u * kLongBS) * 4;
    if (v >= P0) break;
    const int s = at(v);
    const float4 x = xs[u];
    atomicAdd(&h[order_key(x.x) >> 20], 1u);
    if (s + 1 < len) atomicAdd(&h[order_key(x.y) >> 20], 1u);
    if (s + 2 < len) atomicAdd(&h[order_key(x.z) >> 20], 1u);
    if (s + 3 < len) atomicAdd(&h[order_key(x.w) >> 20], 1u);
  }
  __syncthreads();
  for (int i = tid; i < kHBins; i += kLongBS) {
    uint32_t sum = 0;
#pragma unroll
    for (int c = 0; c < kCutCopies; ++c) sum += cut_dyn[c * kHBins + i];
    cut_dyn[i] = sum;
  }
  __syncthreads();
  const int need_p =
      static_cast<int>(3 * static_cast<int64_t>(K) * P0 / (2 * static_cast<int64_t>(len))) +
      kLongSlack;
  threshold_bin<kLongBS>(cut_dyn, need_p, warp_sums, &s_cut, &s_tmp);
  if (tid == 0) {
    const uint32_t k0 = static_cast<uint32_t>(s_cut) << 20;
    const float cf = s_cut == 0 ? -INFINITY
                                : __uint_as_float((k0 & 0x80000000u) ? (k0 & 0x7fffffffu) : ~k0);
    ws.cnt[static_cast<int64_t>(t) * kCnt + 3] = __float_as_int(cf);
  }
}

// Long path, launch 1: the slice's keys at or above the row's cutoff.
__global__ void __launch_bounds__(kLongBS) topk_capture_kernel(const float* __restrict__ scores,
                                                               BatchArgs b, int K, int split,
                                                               LongScratch ws) {
  chain_wait();     // the previous kernel of the stream has completed
  chain_release();  // the next one may be scheduled
  __shared__ uint32_t skey[(kLongBS / 32) * kCapSeg];
  __shared__ int32_t spos[(kLongBS / 32) * kCapSeg];
  __shared__ int s_wcnt[kLongBS / 32];
  __shared__ int s_base;
  const int t = blockIdx.y, c = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int pos = query_pos(b, t, nullptr);
  const int len = pos + 1;
  if (len <= K) return;
  int lo, hi;
  slice_of(len, split, c, lo, hi);
  if (lo >= hi) return;
  const float* row = scores + static_cast<int64_t>(t) * b.max_len;
  const float cf = __int_as_float(ws.cnt[static_cast<int64_t>(t) * kCnt + 3]);
  // keys >= cf (float compare: NaN kept too, a superset is harmless), per
  // warp in its own segment of the shared buffer, in warp-uniform tiles; a
  // slice of 8K positions is requested in one batch of float4 loads
  const uint32_t lt = lanemask_lt();
  int wcount = 0;  // warp-uniform
  auto capture = [&](int s, float x, bool valid) {
    const bool p = valid && !(x < cf);
    const uint32_t m = __ballot_sync(0xffffffffu, p);
    if (m) {
      if (p) {
        const int i = wcount + __popc(m & lt);
        if (i < kCapSeg) {
          skey[warp * kCapSeg + i] = order_key(x);
          spos[warp * kCapSeg + i] = lo + s;
        }
      }
      wcount += __popc(m);
    }
  };
  scan_row<kLongBS, 4>(row + lo, hi - lo, capture);  // lo is a multiple of 4
  if (lane == 0) s_wcnt[warp] = wcount;
  __syncthreads();
  int* cnt = ws.cnt + static_cast<int64_t>(t) * kCnt;
  if (tid == 0) {
    int total = 0, dropped = 0;
    for (int w = 0; w < kLongBS / 32; ++w) {
      total += min(s_wcnt[w], kCapSeg);
      dropped += s_wcnt[w] > kCapSeg;
    }
    s_base = atomicAdd(&cnt[1], total);
    if (dropped || s_base + total > kCandCap) atomicOr(&cnt[2], 1);
  }
  __syncthreads();
  // copy this CTA's entries to the row's list (warp w's segment after the
  // segments of warps < w)
  int off = s_base;
  for (int w = 0; w < warp; ++w) off += min(s_wcnt[w], kCapSeg);
  const int n = min(s_wcnt[warp], kCapSeg);
  for (int i = lane; i < n; i += 32)
    if (off + i < kCandCap) {
      ws.ckey[static_cast<int64_t>(t) * kCandCap + off + i] = skey[warp * kCapSeg + i];
      ws.cpos[static_cast<int64_t>(t) * kCandCap + off + i] = spos[warp * kCapSeg + i];
    }
}

// The taken entries of a capture list (key > T, or key == T at a position up
// to pstar) appended to taken[0, K), one shared counter update per warp.
// Ends with a CTA barrier.
__device__ __forceinline__ void take_listed(int n, int K, uint32_t T, int pstar, const uint32_t* ckey,
                                            const int32_t* cpos, int32_t* taken, int* s_taken) {
  const int lane = threadIdx.x & 31;
  for (int i0 = 0; i0 < n; i0 += blockDim.x) {  // n is the same in every thread
    const int i = i0 + static_cast<int>(threadIdx.x);
    bool tk = false;
    int p = 0;
    if (i < n) {
      const uint32_t k = ckey[i];
      p = cpos[i];
      tk = k > T || (k == T && p <= pstar);
    }
    const uint32_t m = __ballot_sync(0xffffffffu, tk);
    int base = 0;
    if (lane == 0 && m) base = atomicAdd(s_taken, __popc(m));
    base = __shfl_sync(0xffffffffu, base, 0);
    if (tk) {
      const int j = base + __popc(m & lanemask_lt());
      if (j < K) taken[j] = p;
    }
  }
  __syncthreads();
}

// The K taken positions taken[0, K) of a row of len positions written to
// out in ascending order: through a bitmap over the row in `area` (free
// shared memory of kBitmapLen / 32 words) for rows up to kBitmapLen
// positions, else by the sort.  Flags DSA_DEVERR_BATCH unless exactly K were
// taken.  Ends with a CTA barrier.
constexpr int kBitmapLen = 262144;  // measured: the sort's fixed cost wins beyond this
template <int BS>
__device__ void write_taken(int len, int K, int32_t* taken, int n_taken, uint32_t* area, int32_t* out,
                            int* warp_sums, int* status) {
  if (len <= kBitmapLen) {
    const int nwords = (len + 31) >> 5;
    for (int i = threadIdx.x; i < nwords; i += BS) area[i] = 0;
    __syncthreads();
    for (int j = threadIdx.x; j < min(n_taken, K); j += BS)
      atomicOr(&area[taken[j] >> 5], 1u << (taken[j] & 31));
    __syncthreads();
    bitmap_compact<BS>(area, nwords, K, out, warp_sums, status);
  } else {
    if (threadIdx.x == 0 && n_taken != K) atomicOr(status, DSA_DEVERR_BATCH);
    sort_positions<BS>(taken, K, out);
  }
}

// Long path, launch 2: the threshold key and tie cut of a row from its
// capture list, then the taken positions (key > T, or key == T at a position
// up to pstar: exactly K of them) in ascending order.  A row without the
// guarantee (too few keys captured, or any dropped) is marked for the
// fallback (word 6).
__global__ void __launch_bounds__(kFinBS, 1) topk_resolve_write_kernel(BatchArgs b, int K,
                                                                       LongScratch ws, int32_t* idx,
                                                                       int* status) {
  chain_wait();     // the previous kernel of the stream has completed
  chain_release();  // the next one may be scheduled
  __shared__ int hist2[2048];
  __shared__ uint32_t h[kHBins];
  __shared__ int warp_sums[32];
  __shared__ int s_d, s_above, s_n, s_b1, s_nabove, s_taken;
  extern __shared__ uint32_t res_dyn[];  // captured keys and positions, then the taken positions
  uint32_t* ckey = res_dyn;
  int32_t* cpos = reinterpret_cast<int32_t*>(res_dyn + kCandCap);
  int32_t* taken = reinterpret_cast<int32_t*>(res_dyn + 2 * kCandCap);
  const int t = blockIdx.x, tid = threadIdx.x;
  const int pos = query_pos(b, t, tid == 0 ? status : nullptr);
  const int len = pos + 1;
  int32_t* out = idx + static_cast<int64_t>(t) * K;
  if (len <= K) {  // every visible position, then -1 padding
    for (int j = tid; j < K; j += kFinBS) out[j] = j < len ? j : -1;
    return;
  }
  int* cnt = ws.cnt + static_cast<int64_t>(t) * kCnt;
  const int n = cnt[1];
  if (cnt[2] != 0 || n < K || n > kCandCap) {  // no guarantee: the fallback takes the row
    if (tid == 0) cnt[6] = 1;
    return;
  }
  // the list into shared memory, 8 entries per thread requested before any is stored
  for (int i0 = tid; i0 < n; i0 += 8 * kFinBS) {
    uint32_t kk[8];
    int32_t pp[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = i0 + u * kFinBS;
      if (i < n) {
        kk[u] = ws.ckey[static_cast<int64_t>(t) * kCandCap + i];
        pp[u] = ws.cpos[static_cast<int64_t>(t) * kCandCap + i];
      }
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = i0 + u * kFinBS;
      if (i < n) {
        ckey[i] = kk[u];
        cpos[i] = pp[u];
      }
    }
  }
  for (int i = tid; i < kHBins; i += kFinBS) h[i] = 0;
  if (tid == 0) s_taken = 0;
  __syncthreads();
  for (int i = tid; i < n; i += kFinBS) atomicAdd(&h[ckey[i] >> 20], 1u);
  __syncthreads();
  threshold_bin<kFinBS>(h, K, warp_sums, &s_b1, &s_nabove);
  const uint32_t b1 = static_cast<uint32_t>(s_b1);
  auto get_key = [&](int i) -> uint32_t { return (ckey[i] >> 20) == b1 ? ckey[i] : ~0u; };
  auto get_pos = [&](int i) -> int { return cpos[i]; };
  uint32_t T;
  int need;
  select_low_bits<kFinBS>(n, K - s_nabove, get_key, b1, hist2, warp_sums, &s_d, &s_above, &T,
                          &need);
  const int pstar = tied_position_cut<kFinBS>(n, need, T, get_key, get_pos, hist2, warp_sums, &s_d,
                                              &s_above, &s_n);
  take_listed(n, K, T, pstar, ckey, cpos, taken, &s_taken);
  write_taken<kFinBS>(len, K, taken, s_taken, res_dyn, out, warp_sums, status);
}

// Rows beyond 16K positions: fewer than kRowsFew of them are spread over
// several CTAs each (the launches above); more get a persistent CTA per SM,
// a row at a time.  Measured on GB300 with K = 2048 (top-K alone, chained
// launches): 64 rows of ~115K positions take 34 us sliced against 37 us in
// the persistent kernel, 96 rows 39 against 38, 128 rows 44 against 38
// (where one pass of the persistent kernel covers them); 4 rows of 1M take
// 31 us sliced.
constexpr int kRowsFew = 80;

bool use_long_path(const dsa_batch_t& b) {
  return b.num_q < kRowsFew && b.max_len > 16384;
}

// Slices (CTAs) per row of the long path: about 4 waves of 152 SMs in all,
// at least 8K positions each.
int long_split(const dsa_batch_t& b) {
  int split = static_cast<int>((4 * 152 + b.num_q - 1) / b.num_q);
  return std::max(1, std::min(split, (b.max_len + 8191) / 8192));
}

size_t round256z(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Layout of the long path's scratch (its per-row words are cleared by the
// cutoff launch).
LongScratch long_scratch(const dsa_batch_t& b, void* base_v, size_t* total) {
  const size_t q = static_cast<size_t>(b.num_q);
  uint8_t* base = static_cast<uint8_t*>(base_v);
  LongScratch ws;
  size_t off = 0;
  ws.cnt = reinterpret_cast<int*>(base + off);
  off += round256z(q * kCnt * 4);
  ws.ckey = reinterpret_cast<uint32_t*>(base + off);
  off += round256z(q * kCandCap * 4);
  ws.cpos = reinterpret_cast<int32_t*>(base + off);
  off += round256z(q * kCandCap * 4);
  if (total) *total = off;
  return ws;
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
  prof_begin(stream);
  cudaError_t e = launch_chained(kern, dim3(static_cast<unsigned>(CL) * static_cast<unsigned>(b.num_q)),
                                 dim3(BS), STAGE ? smem : 0, stream, CL, scores, to_args(b), k, idx,
                                 status);
  prof_end(kLaunchTopk, stream);
  count_launch(kLaunchTopk);
  return e;
}

cudaError_t launch_rows(const float* scores, const dsa_batch_t& b, int k, int32_t* idx, int* status,
                        cudaStream_t stream, const int* only = nullptr) {
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
  if (!only) prof_begin(stream);
  cudaError_t e = launch_chained(topk_rows_kernel, dim3(grid), dim3(kRowBS), kRowDynBytes, stream, 1,
                                 scores, to_args(b), k, idx, status, only);
  if (!only) prof_end(kLaunchTopk, stream);
  count_launch(kLaunchTopk);
  return e != cudaSuccess ? e : cudaGetLastError();
}

// ------------------------------------------------------------------ select-only F layer
// The indexer's sample mode leaves, per row, the scores of up to
// kSampleTilesMax 128-key tiles spread over the row (-inf at positions
// beyond the row) and their count in word 7.  The cutoff is the exact value
// of the need-th largest sample, need about 1.5 times the sample's share of
// K (plus kLongSlack): a 12-bit histogram gives its bin, two 10-bit passes
// over that bin's members the rest of its key (a bin edge would keep up to
// a bin's width more keys).  +inf for rows that keep every position, -inf
// when the sample holds fewer than need values.
__global__ void __launch_bounds__(kLongBS) topk_sample_cutoff_kernel(BatchArgs b, int K,
                                                                     TopkLists ls) {
  chain_wait();     // the previous kernel of the stream has completed
  chain_release();  // the next one may be scheduled
  extern __shared__ uint32_t cut_dyn[];  // [kCutCopies][kHBins]
  __shared__ int hist2[1024];
  __shared__ int warp_sums[32];
  __shared__ int s_cut, s_tmp, s_valid, s_d, s_above;
  const int t = blockIdx.x, tid = threadIdx.x;
  const int pos = query_pos(b, t, nullptr);
  const int len = pos + 1;
  int* cnt = ls.cnt + static_cast<int64_t>(t) * kTopkCnt;
  if (len <= K) {
    if (tid == 0) cnt[3] = __float_as_int(INFINITY);
    return;
  }
  for (int i = tid; i < kCutCopies * kHBins; i += kLongBS) cut_dyn[i] = 0;
  if (tid == 0) {
    s_cut = 0;
    s_valid = 0;
  }
  __syncthreads();
  uint32_t* h = cut_dyn + (tid & (kCutCopies - 1)) * kHBins;
  const float* row = ls.sample + static_cast<int64_t>(t) * (kSampleTilesMax * 128);
  const int ns = min(cnt[7], kSampleTilesMax * 128);
  // order key of sample i, ~0 for a sampled position beyond the row (-inf)
  auto get = [&](int i) -> uint32_t {
    const float x = row[i];
    return x == -INFINITY ? ~0u : order_key(x);
  };
  int mine = 0;
  for (int v = tid; v < ns; v += kLongBS) {
    const uint32_t k = get(v);
    if (k != ~0u) {
      atomicAdd(&h[k >> 20], 1u);
      ++mine;
    }
  }
  atomicAdd(&s_valid, mine);
  __syncthreads();
  for (int i = tid; i < kHBins; i += kLongBS) {
    uint32_t sum = 0;
#pragma unroll
    for (int c = 0; c < kCutCopies; ++c) sum += cut_dyn[c * kHBins + i];
    cut_dyn[i] = sum;
  }
  __syncthreads();
  const int need_p =
      static_cast<int>(3 * static_cast<int64_t>(K) * s_valid / (2 * static_cast<int64_t>(len))) +
      kLongSlack;
  if (need_p > s_valid) {  // too few samples: keep everything (the fallback resolves the row)
    if (tid == 0) cnt[3] = __float_as_int(-INFINITY);
    return;
  }
  threshold_bin<kLongBS>(cut_dyn, need_p, warp_sums, &s_cut, &s_tmp);
  uint32_t T;
  int rest;
  select_low_bits<kLongBS>(ns, need_p - s_tmp, get, static_cast<uint32_t>(s_cut), hist2, warp_sums,
                           &s_d, &s_above, &T, &rest);
  if (tid == 0) {
    // the float of key T (the inverse of order_key)
    const float cf = __uint_as_float((T & 0x80000000u) ? (T & 0x7fffffffu) : ~T);
    cnt[3] = __float_as_int(cf);
  }
}

// One CTA per row: the row's capture list gathered from its key chunks'
// segments, the threshold key T and tie cut pstar from it (as the long
// path's resolve), then the taken positions (key > T, or key == T at a
// position up to pstar: exactly K of them) written in ascending order.
// A row without the guarantee (too few keys captured, or a chunk with more
// keys than its segment or the list more than kResCap) is marked for the
// fallback (word 6).
constexpr int kResCap = 8192;
static_assert(kBitmapLen / 32 <= 2 * kResCap && kBitmapLen / 32 <= 2 * kCandCap,
              "the bitmap fits in the lists' space of both resolve-and-write kernels");
__global__ void __launch_bounds__(kFinBS) topk_list_resolve_write_kernel(BatchArgs b, int K,
                                                                         TopkLists ls,
                                                                         int32_t* idx,
                                                                         int* status) {
  chain_wait();     // the previous kernel of the stream has completed
  chain_release();  // the next one may be scheduled
  __shared__ int hist2[2048];
  __shared__ uint32_t h[kHBins];
  __shared__ int warp_sums[32];
  __shared__ int s_d, s_above, s_n, s_b1, s_nabove, s_taken, s_over;
  __shared__ int s_segoff[4 * kSegMax];
  extern __shared__ uint32_t res_dyn[];  // gathered keys and positions, then the taken positions
  uint32_t* ckey = res_dyn;
  int32_t* cpos = reinterpret_cast<int32_t*>(res_dyn + kResCap);
  int32_t* taken = reinterpret_cast<int32_t*>(res_dyn + 2 * kResCap);
  const int t = blockIdx.x, tid = threadIdx.x;
  const int pos = query_pos(b, t, tid == 0 ? status : nullptr);
  const int len = pos + 1;
  int32_t* out = idx + static_cast<int64_t>(t) * K;
  if (len <= K) {  // every visible position, then -1 padding
    for (int j = tid; j < K; j += kFinBS) out[j] = j < len ? j : -1;
    return;
  }
  int* cnt = ls.cnt + static_cast<int64_t>(t) * kTopkCnt;
  const int nkc = cnt[0];
  const int ncell = 4 * nkc;  // (key chunk, TMEM lane quarter) cells of the list
  const int segq = nkc > 0 ? kTopkCandCap / ncell : 0;
  const int* segcnt = ls.segcnt + static_cast<int64_t>(t) * kSegMax * 4;
  // cell offsets in the gathered list (thread tid owns cells tid*per ..)
  if (tid == 0) s_over = (nkc <= 0 || nkc > kSegMax) ? 1 : 0;
  __syncthreads();
  constexpr int per = 4 * kSegMax / kFinBS;
  int c_[per];
  int local = 0;
#pragma unroll
  for (int k2 = 0; k2 < per; ++k2) {
    const int c = tid * per + k2;
    const int v = c < ncell ? segcnt[c] : 0;
    if (v > segq) s_over = 1;
    c_[k2] = min(v, segq);
    local += c_[k2];
  }
  int n;
  int run = block_excl_scan<kFinBS>(local, warp_sums, &n);
#pragma unroll
  for (int k2 = 0; k2 < per; ++k2) {
    s_segoff[tid * per + k2] = run;
    run += c_[k2];
  }
  __syncthreads();
  if (s_over || n < K || n > kResCap) {  // no guarantee: the fallback takes the row
    if (tid == 0) cnt[6] = 1;
    return;
  }
  // gather: entry o of the gathered list lies in the last cell c with
  // s_segoff[c] <= o (a binary search; empty cells share their successor's
  // offset), at position o - s_segoff[c] of that cell's segment; 8 entries
  // per thread are requested before any is stored
  for (int o0 = tid; o0 < n; o0 += 8 * kFinBS) {
    uint32_t kk[8];
    int32_t pp[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int o = o0 + u * kFinBS;
      if (o < n) {
        int lo = 0, hi = ncell - 1;  // s_segoff[lo] <= o
        while (lo < hi) {
          const int mid = (lo + hi + 1) >> 1;
          if (s_segoff[mid] <= o) lo = mid;
          else hi = mid - 1;
        }
        const int64_t src = static_cast<int64_t>(t) * kTopkCandCap + static_cast<int64_t>(lo) * segq +
                            (o - s_segoff[lo]);
        kk[u] = ls.ckey[src];
        pp[u] = ls.cpos[src];
      }
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int o = o0 + u * kFinBS;
      if (o < n) {
        ckey[o] = kk[u];
        cpos[o] = pp[u];
      }
    }
  }
  for (int i = tid; i < kHBins; i += kFinBS) h[i] = 0;
  if (tid == 0) s_taken = 0;
  __syncthreads();
  for (int i = tid; i < n; i += kFinBS) atomicAdd(&h[ckey[i] >> 20], 1u);
  __syncthreads();
  threshold_bin<kFinBS>(h, K, warp_sums, &s_b1, &s_nabove);
  const uint32_t b1 = static_cast<uint32_t>(s_b1);
  auto get_key = [&](int i) -> uint32_t { return (ckey[i] >> 20) == b1 ? ckey[i] : ~0u; };
  auto get_pos = [&](int i) -> int { return cpos[i]; };
  uint32_t T;
  int need;
  select_low_bits<kFinBS>(n, K - s_nabove, get_key, b1, hist2, warp_sums, &s_d, &s_above, &T,
                          &need);
  const int pstar = tied_position_cut<kFinBS>(n, need, T, get_key, get_pos, hist2, warp_sums, &s_d,
                                              &s_above, &s_n);
  take_listed(n, K, T, pstar, ckey, cpos, taken, &s_taken);
  write_taken<kFinBS>(len, K, taken, s_taken, res_dyn, out, warp_sums, status);
}

}  // namespace

// Rows beyond 16K positions (and at most 2M, so that a row has at most
// kSegMax key chunks of the capture), prefill and chunked prefill only: for
// a decode batch (one query per sequence) the sample, cutoff and resolve
// launches cost more than the top-K over the score matrix they replace.
bool use_select_only(const dsa_batch_t& b, int) {
  return b.num_q > 0 && b.max_q > 1 && b.max_len > 16384 && b.max_len <= kSegMax * 64 * 128;
}
static_assert(kSegMax * 64 * 128 <= (1 << 21), "rows of the select-only path: at most 2M positions");

size_t select_only_bytes(const dsa_batch_t& b) {
  const size_t q = static_cast<size_t>(b.num_q);
  return round256z(q * kTopkCnt * 4) + 2 * round256z(q * kTopkCandCap * 4) +
         round256z(q * kSegMax * 4 * 4) + round256z(q * kSampleTilesMax * 128 * 4);
}

TopkLists select_only_lists(const dsa_batch_t& b, void* base_v) {
  const size_t q = static_cast<size_t>(b.num_q);
  uint8_t* base = static_cast<uint8_t*>(base_v);
  TopkLists ls;
  size_t off = 0;
  ls.cnt = reinterpret_cast<int*>(base + off);
  off += round256z(q * kTopkCnt * 4);
  ls.ckey = reinterpret_cast<uint32_t*>(base + off);
  off += round256z(q * kTopkCandCap * 4);
  ls.cpos = reinterpret_cast<int32_t*>(base + off);
  off += round256z(q * kTopkCandCap * 4);
  ls.segcnt = reinterpret_cast<int*>(base + off);
  off += round256z(q * kSegMax * 4 * 4);
  ls.sample = reinterpret_cast<float*>(base + off);
  return ls;
}

cudaError_t launch_indexer_topk_select(const void* q_idx, const float* q_scale, const float* w,
                                       const void* k_idx, const float* k_scale, int64_t k_rows,
                                       bool fp8, const dsa_batch_t& b, int k, int32_t* idx,
                                       float* scores, void* lists_base, int* status,
                                       cudaStream_t stream) {
  if (b.num_q == 0) return cudaSuccess;
  const TopkLists ls = select_only_lists(b, lists_base);
  cudaError_t e = cudaMemsetAsync(ls.cnt, 0, static_cast<size_t>(b.num_q) * kTopkCnt * 4, stream);
  if (e != cudaSuccess) return e;
  static int configured_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device != dev) {
    e = cudaFuncSetAttribute(topk_sample_cutoff_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kCutDynBytes);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(topk_list_resolve_write_kernel,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (2 * kResCap + 4096) * 4);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  const BatchArgs a = to_args(b);
  // 1. sampled scores, 2. the rows' cutoffs, 3. the capture lists
  e = launch_indexer_mode(q_idx, q_scale, w, k_idx, k_scale, k_rows, fp8, b, kIdxSample, nullptr,
                          nullptr, ls, status, stream);
  if (e != cudaSuccess) return e;
  prof_begin(stream);
  e = launch_chained(topk_sample_cutoff_kernel, dim3(b.num_q), dim3(kLongBS), kCutDynBytes, stream, 1, a,
                     k, ls);
  if (e != cudaSuccess) return e;
  prof_end(kLaunchTopk, stream);
  count_launch(kLaunchTopk);
  e = cudaMemsetAsync(ls.segcnt, 0, static_cast<size_t>(b.num_q) * kSegMax * 4 * 4, stream);
  if (e != cudaSuccess) return e;
  e = launch_indexer_mode(q_idx, q_scale, w, k_idx, k_scale, k_rows, fp8, b, kIdxCapture, nullptr,
                          nullptr, ls, status, stream);
  if (e != cudaSuccess) return e;
  // 4. exact selection from the lists, written in ascending order
  int pw = kFinBS;  // the sort's area: max(kFinBS, the next power of two >= k)
  while (pw < k) pw <<= 1;
  prof_begin(stream);
  e = launch_chained(topk_list_resolve_write_kernel, dim3(b.num_q), dim3(kFinBS),
                     (2 * static_cast<size_t>(kResCap) + pw) * 4, stream, 1, a, k, ls, idx, status);
  if (e != cudaSuccess) return e;
  prof_end(kLaunchTopk, stream);
  count_launch(kLaunchTopk);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // 5. rows marked for the fallback (normally none): their scores, then the
  // exact many-long-rows top-K on those rows only
  e = launch_indexer_mode(q_idx, q_scale, w, k_idx, k_scale, k_rows, fp8, b, kIdxScores, scores,
                          ls.cnt, ls, status, stream);
  if (e != cudaSuccess) return e;
  return launch_rows(scores, b, k, idx, status, stream, ls.cnt);
}

size_t topk_scratch_bytes(const dsa_batch_t& b, int) {
  if (b.num_q == 0 || !use_long_path(b)) return 0;
  size_t total = 0;
  long_scratch(b, nullptr, &total);
  return total;
}

cudaError_t launch_topk(const float* scores, const dsa_batch_t& b, int k, int32_t* idx,
                        int* status, void* scratch, size_t scratch_bytes, cudaStream_t stream) {
  if (b.num_q == 0) return cudaSuccess;
  if (use_long_path(b)) {
    if (!scratch || scratch_bytes < topk_scratch_bytes(b, k)) return cudaErrorInvalidValue;
    const LongScratch ws = long_scratch(b, scratch, nullptr);
    cudaError_t e = cudaSuccess;
    const int split = long_split(b);
    const dim3 grid(static_cast<unsigned>(split), static_cast<unsigned>(b.num_q));
    const BatchArgs a = to_args(b);
    // resolve and write: the captured keys and positions, then the taken
    // positions (padded to a power of two for the sort)
    int pw = kFinBS;
    while (pw < k) pw <<= 1;
    const size_t res_bytes = (2 * static_cast<size_t>(kCandCap) + pw) * 4;
    {
      static int configured_device = -1;
      int dev = 0;
      cudaGetDevice(&dev);
      if (configured_device != dev) {
        e = cudaFuncSetAttribute(topk_resolve_write_kernel,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (2 * kCandCap + 4096) * 4);
        if (e != cudaSuccess) return e;
        configured_device = dev;
      }
    }
    {
      static int configured_device = -1;
      int dev = 0;
      cudaGetDevice(&dev);
      if (configured_device != dev) {
        e = cudaFuncSetAttribute(topk_cutoff_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kCutDynBytes);
        if (e != cudaSuccess) return e;
        configured_device = dev;
      }
    }
    prof_begin(stream);
    e = launch_chained(topk_cutoff_kernel, dim3(b.num_q), dim3(kLongBS), kCutDynBytes, stream, 1,
                       scores, a, k, ws);
    if (e == cudaSuccess)
      e = launch_chained(topk_capture_kernel, grid, dim3(kLongBS), 0, stream, 1, scores, a, k, split, ws);
    if (e == cudaSuccess)
      e = launch_chained(topk_resolve_write_kernel, dim3(b.num_q), dim3(kFinBS), res_bytes, stream, 1, a,
                         k, ws, idx, status);
    if (e == cudaSuccess) e = launch_rows(scores, b, k, idx, status, stream, ws.cnt);  // marked rows only
    prof_end(kLaunchTopk, stream);
    for (int i = 0; i < 3; ++i) count_launch(kLaunchTopk);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
  }
  // Rows beyond 16K positions (kRowsFew or more of them): one persistent CTA
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

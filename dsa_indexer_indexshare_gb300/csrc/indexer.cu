// Lightning-indexer scoring on the tcgen05 tensor cores.
//
//   scores[t, s] = sum_{j<32} w[t,j] * ReLU(q_idx[t,j,:] . k_idx[s,:])
//
// ("GLM-5.2 / 总览" config table: 32 heads x 128 dims; sub-doc index row 02:
// ReLU, FP8 per-block + Hadamard variant; "GLM-5.2 架构深度拆解" CH 2.2.)
//
// The contraction runs with the KEYS on the MMA M dimension (128 keys per
// tile) and the (token, head) pairs of a block of NTOK queries on N, so that
// TMEM lane i holds every head's dot product for key i.  The epilogue then
// reduces over heads with ReLU and the head weights thread-locally (no
// shuffles) and writes a coalesced row segment of scores per token.
//
// Warp roles: epilogue warps first (thread = TMEM lane = key; 8 warps, two
// per lane quarter splitting the tokens, when a tile holds 8 tokens; 4 for
// decode), then one TMA producer warp and one MMA issuer warp (TMEM owner).  The key tiles
// stream through a STAGES-deep shared-memory ring; the accumulator is double
// buffered in TMEM so the epilogue of tile i overlaps the MMAs of tile i+1.
#include <algorithm>
#include <cstdint>

#include "common.cuh"

namespace dsa {
namespace {

template <int NTOK, bool FP8, int STAGES, int MODE>
struct IdxCfg {
  static constexpr int N = NTOK * 32;                // MMA N: (token, head) pairs
  // epilogue warps: two per TMEM lane quarter (each takes half of the tokens)
  // when a tile holds several tokens, one per quarter otherwise
  static constexpr int NEPI = NTOK >= 2 ? 8 : 4;
  static constexpr int TOK_PER_WARP = NTOK * 4 / NEPI;
  static constexpr int NT = NEPI * 32 + 64;          // + TMA producer warp + MMA warp
  static constexpr int KSUB = FP8 ? 1 : 2;           // 128-byte swizzle atoms per 128-d row
  static constexpr int Q_SUB = N * 128;              // bytes of one Q sub-tile
  static constexpr int Q_BYTES = KSUB * Q_SUB;
  static constexpr int K_SUB = 128 * 128;            // bytes of one K sub-tile (128 keys)
  static constexpr int K_BYTES = KSUB * K_SUB;
  static constexpr int KSTEPS = FP8 ? 4 : 8;         // MMA K-steps of 32 bytes each
  static constexpr int TMEM_COLS = 2 * N < 32 ? 32 : 2 * N;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + Q_BYTES;
  static constexpr int OFF_W = OFF_K + STAGES * K_BYTES;
  static constexpr int OFF_BAR = OFF_W + N * 4;
  static constexpr int NBAR = 1 + 2 * STAGES + 4 + 1;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_MISC + 64 + 1024;  // + slack for 1024-byte alignment
  static_assert(STAGES >= 2, "need a ring");
  static_assert(SMEM <= 232448, "shared memory");
};

struct IndexerParams {
  BatchArgs b;
  const float* w;
  const float* q_scale;
  const float* k_scale;
  int64_t k_rows;
  float* scores;
  int* status;
  int kc_blocks;   // 128-key blocks per CTA
  int num_kc;      // key chunks per query block
  int num_qb;      // query blocks per sequence
  int fill_tail;   // write -inf beyond the computed blocks
  uint64_t timeout_ns;
  const int* only;  // scores mode: only blocks holding a row flagged here (word 6 of kTopkCnt)
  int whole_rows;   // one CTA per query block over all its keys
  TopkLists lists;  // sample / capture modes
};

// Wait until the tcgen05.ld results in v are valid; the asm takes v as
// in/out operands so that no use of v can be scheduled before the wait.
__device__ __forceinline__ void tmem_wait_ld_dep(float (&v)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+f"(v[0]), "+f"(v[1]), "+f"(v[2]), "+f"(v[3]), "+f"(v[4]), "+f"(v[5]),
                 "+f"(v[6]), "+f"(v[7]), "+f"(v[8]), "+f"(v[9]), "+f"(v[10]), "+f"(v[11]),
                 "+f"(v[12]), "+f"(v[13]), "+f"(v[14]), "+f"(v[15]), "+f"(v[16]), "+f"(v[17]),
                 "+f"(v[18]), "+f"(v[19]), "+f"(v[20]), "+f"(v[21]), "+f"(v[22]), "+f"(v[23]),
                 "+f"(v[24]), "+f"(v[25]), "+f"(v[26]), "+f"(v[27]), "+f"(v[28]), "+f"(v[29]),
                 "+f"(v[30]), "+f"(v[31])
               :
               : "memory");
}

template <int NTOK, bool FP8, int STAGES, int MODE>
__global__ void __launch_bounds__(IdxCfg<NTOK, FP8, STAGES, MODE>::NT, 1)
    indexer_kernel(const __grid_constant__ CUtensorMap qmap,
                   const __grid_constant__ CUtensorMap kmap, const IndexerParams p) {
  chain_wait();     // the previous kernel of the stream has completed
  chain_release();  // the next one may be scheduled
  using C = IdxCfg<NTOK, FP8, STAGES, MODE>;
  constexpr int W_PROD = C::NEPI, W_MMA = C::NEPI + 1, NEPT = C::NEPI * 32;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ---- work unit: (sequence, query block, key chunk); heavy query blocks first
  const int seq = blockIdx.y;
  const int kc = blockIdx.x % p.num_kc;
  const int qb = p.num_qb - 1 - static_cast<int>(blockIdx.x / p.num_kc);
  int qs, qe;
  seq_rows(p.b, seq, p.status, qs, qe);
  const int q0 = qs + qb * NTOK;
  if (q0 >= qe) return;
  const int nq = min(NTOK, qe - q0);
  int pos[NTOK];
  int pmax = -1;
#pragma unroll
  for (int n = 0; n < NTOK; ++n) {
    pos[n] = n < nq ? query_pos(p.b, q0 + n, tid == 0 ? p.status : nullptr) : -1;
    pmax = max(pmax, pos[n]);
  }
  if constexpr (MODE == kIdxScores) {
    if (p.only) {  // the fallback rows of a select-only F layer
      bool any = false;
      for (int n = 0; n < nq; ++n) any |= p.only[static_cast<int64_t>(q0 + n) * kTopkCnt + 6] != 0;
      if (!any) return;
    }
  }
  // key tiles: the chunk's consecutive tiles, or (sample mode) ns tiles
  // spread evenly over the T tiles that cover [0, pmax], all of them when
  // T <= ns
  // (sample mode: CTA kc takes sampled tiles kc * kSampleChunk ..)
  const int s_begin = MODE == kIdxSample ? 0 : kc * p.kc_blocks * 128;
  if (s_begin >= p.b.max_len) return;
  const int s_stop = min(s_begin + p.kc_blocks * 128, p.b.max_len);
  const int T = pmax < 0 ? 0 : pmax / 128 + 1;
  const int ns = min(max(32, T / 64), kSampleTilesMax);
  const int i0 = MODE == kIdxSample ? kc * kSampleChunk : 0;  // first sampled tile of this CTA
  int nkb;
  if constexpr (MODE == kIdxSample) {
    const int total = min(T, ns);
    if (kc == 0 && tid < nq) p.lists.cnt[static_cast<int64_t>(q0 + tid) * kTopkCnt + 7] = total * 128;
    nkb = max(0, min(kSampleChunk, total - i0));
  } else {
    nkb = pmax < s_begin ? 0 : min(p.kc_blocks, (pmax - s_begin) / 128 + 1);
  }
  auto tile_start = [&](int i) -> int {
    if constexpr (MODE == kIdxSample) {
      const int g = i0 + i;
      return (T <= ns ? g : static_cast<int>(static_cast<int64_t>(g) * T / ns)) * 128;
    } else {
      return s_begin + i * 128;
    }
  };
  if (MODE == kIdxScores && p.fill_tail) {
    const int f0 = s_begin + nkb * 128;
    const float4 ninf = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    for (int n = 0; n < nq; ++n) {
      float* row = p.scores + static_cast<int64_t>(q0 + n) * p.b.max_len;
      for (int s = f0 + tid * 4; s < s_stop; s += C::NT * 4)
        *reinterpret_cast<float4*>(row + s) = ninf;
    }
  }
  if (nkb == 0) return;
  const int64_t row0 = seq_base_row(p.b, seq);

  // ---- shared memory, barriers, TMEM
  const uint32_t sQ = smem_u32(sm + C::OFF_Q);
  const uint32_t sK = smem_u32(sm + C::OFF_K);
  float* sW = reinterpret_cast<float*>(sm + C::OFF_W);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::OFF_BAR);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + C::OFF_MISC);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + C::OFF_MISC + 8);
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  const int B_QFULL = 0, B_KFULL = 1, B_KEMPTY = 1 + STAGES, B_ACCF = 1 + 2 * STAGES,
            B_ACCE = 3 + 2 * STAGES, B_DONE = 5 + 2 * STAGES;

  if (tid == 0) {
    *abort_flag = 0;
    mbar_init(bar(B_QFULL), 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar(B_KFULL + s), 1);
      mbar_init(bar(B_KEMPTY + s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(bar(B_ACCF + a), 1);
      mbar_init(bar(B_ACCE + a), NEPT);
    }
    mbar_init(bar(B_DONE), 1);
    fence_mbar_init();
  }
  if (warp == W_MMA) {
    tmem_alloc(smem_u32(tslot), C::TMEM_COLS);
    tmem_relinquish();
  }
  if (tid < NEPT) {
    for (int i = tid; i < C::N; i += NEPT) {
      const int n = i >> 5, j = i & 31;
      float v = 0.f;
      if (n < nq) {
        v = p.w[static_cast<int64_t>(q0 + n) * 32 + j];
        if (FP8) v *= p.q_scale[static_cast<int64_t>(q0 + n) * 32 + j];
      }
      sW[i] = v;
    }
  }
  if (warp == W_PROD && lane == 0) {
    tma_prefetch_desc(&qmap);
    tma_prefetch_desc(&kmap);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;
  const uint64_t to = p.timeout_ns;
  volatile int no_abort = 0;

  if (warp == W_PROD) {
    // ------------------------------------------------ TMA producer
    if (lane == 0) {
      mbar_arrive_expect_tx(bar(B_QFULL), C::Q_BYTES);
#pragma unroll
      for (int ks = 0; ks < C::KSUB; ++ks)
        tma_load_2d(sQ + ks * C::Q_SUB, &qmap, ks * 64, q0 * 32, bar(B_QFULL));
      int issued = 0;
      for (int i = 0; i < nkb; ++i) {
        const int st = i % STAGES;
        if (i >= STAGES &&
            !mbar_wait(bar(B_KEMPTY + st), ((i / STAGES) - 1) & 1, abort_flag, p.status, to))
          break;
        mbar_arrive_expect_tx(bar(B_KFULL + st), C::K_BYTES);
        // first cache row of the tile (a tile never straddles a cache block);
        // an unmapped block loads as zeros (tile fully outside the map)
        const int64_t ty = cache_row(p.b, seq, row0, tile_start(i));
        if (ty < 0) atomicOr(p.status, DSA_DEVERR_INDEX);
        const int y = ty < 0 ? -128 : static_cast<int>(ty);
#pragma unroll
        for (int ks = 0; ks < C::KSUB; ++ks)
          tma_load_2d(sK + st * C::K_BYTES + ks * C::K_SUB, &kmap, ks * 64, y, bar(B_KFULL + st));
        issued = i + 1;
      }
      // let every copy this CTA started land before it can exit
      mbar_wait(bar(B_QFULL), 0, &no_abort, nullptr, to);
      for (int i = max(0, issued - STAGES); i < issued; ++i)
        mbar_wait(bar(B_KFULL + i % STAGES), (i / STAGES) & 1, &no_abort, nullptr, to);
    }
    __syncwarp();
  } else if (warp == W_MMA) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = FP8 ? idesc_e4m3(128, C::N) : idesc_bf16(128, C::N, false, false);
      bool ok = mbar_wait(bar(B_QFULL), 0, abort_flag, p.status, to);
      for (int i = 0; ok && i < nkb; ++i) {
        const int st = i % STAGES, acc = i & 1;
        if (!mbar_wait(bar(B_KFULL + st), (i / STAGES) & 1, abort_flag, p.status, to)) break;
        if (i >= 2 && !mbar_wait(bar(B_ACCE + acc), ((i >> 1) - 1) & 1, abort_flag, p.status, to))
          break;
        tc_fence_after();
        const uint32_t d = tbase + acc * C::N;
#pragma unroll
        for (int kk = 0; kk < C::KSTEPS; ++kk) {
          const uint32_t off = FP8 ? kk * 32 : (kk >> 2) * C::K_SUB + (kk & 3) * 32;
          const uint32_t qoff = FP8 ? kk * 32 : (kk >> 2) * C::Q_SUB + (kk & 3) * 32;
          const uint64_t ad = sdesc_sw128(sK + st * C::K_BYTES + off, 0, 1024);
          const uint64_t bd = sdesc_sw128(sQ + qoff, 0, 1024);
          if (FP8)
            umma_f8(d, ad, bd, idesc, kk > 0);
          else
            umma_bf16(d, ad, bd, idesc, kk > 0);
        }
        umma_commit(bar(B_KEMPTY + st));
        umma_commit(bar(B_ACCF + acc));
      }
      umma_commit(bar(B_DONE));
      mbar_wait(bar(B_DONE), 0, &no_abort, nullptr, to);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ epilogue: ReLU . w over heads
    // warp w reads TMEM lane quarter (w & 3), i.e. keys 32*(w & 3) + lane of
    // the tile, for tokens [(w >> 2) * TOK_PER_WARP, +TOK_PER_WARP)
    const int quarter = warp & 3;
    const int n0 = (warp >> 2) * C::TOK_PER_WARP;
    const uint32_t lane_base = tbase + (static_cast<uint32_t>(quarter * 32) << 16);
    // FP8: this thread's key scale, loaded one tile ahead so that its memory
    // latency overlaps the previous tile instead of following the MMA
    auto load_kscale = [&](int i) -> float {
      if (!FP8 || i >= nkb) return 1.f;
      const int64_t kr = cache_row(p.b, seq, row0, tile_start(i) + quarter * 32 + lane);
      return (kr >= 0 && kr < p.k_rows) ? __ldg(&p.k_scale[kr]) : 0.f;
    };
    // capture mode: the rows' cutoffs; this CTA (key chunk kc) owns segment
    // kc of each row's list, and this warp (TMEM lane quarter q) quarter q
    // of it, placing its keys with a warp-uniform count (no atomics)
    const int segq = kTopkCandCap / (4 * p.num_kc);
    float cf[C::TOK_PER_WARP];
    int wc[C::TOK_PER_WARP];
    uint32_t* ck[C::TOK_PER_WARP];  // this warp's quarter segment of each token's list
    int32_t* cp[C::TOK_PER_WARP];
#pragma unroll
    for (int nn = 0; nn < C::TOK_PER_WARP; ++nn) {
      const int n = n0 + nn;
      cf[nn] = (MODE == kIdxCapture && n < nq)
                   ? __int_as_float(p.lists.cnt[static_cast<int64_t>(q0 + n) * kTopkCnt + 3])
                   : INFINITY;
      wc[nn] = 0;
      const int64_t base = static_cast<int64_t>(q0 + n) * kTopkCandCap + (4 * kc + quarter) * segq;
      ck[nn] = p.lists.ckey + base;
      cp[nn] = p.lists.cpos + base;
    }
    const uint32_t lt = (1u << lane) - 1u;
    float kscale_next = load_kscale(0);
    for (int i = 0; i < nkb; ++i) {
      const int acc = i & 1;
      if (!mbar_wait(bar(B_ACCF + acc), (i >> 1) & 1, abort_flag, p.status, to)) break;
      tc_fence_after();
      const int s = tile_start(i) + quarter * 32 + lane;
      const float kscale = kscale_next;
      kscale_next = load_kscale(i + 1);
#pragma unroll
      for (int nn = 0; nn < C::TOK_PER_WARP; ++nn) {
        const int n = n0 + nn;
        int pn = -1;  // pos[n] without dynamic indexing (keeps pos[] in registers)
#pragma unroll
        for (int k = 0; k < NTOK; ++k)
          if (k == n) pn = pos[k];
        float v[32];
        tmem_ld32(lane_base + acc * C::N + n * 32, v);
        tmem_wait_ld_dep(v);
        if (n < nq) {
          const float4* wv = reinterpret_cast<const float4*>(sW + n * 32);
          // four running sums (heads j = 0, 1, 2, 3 mod 4), two per packed
          // f32x2 fma: each lane rounds exactly as a scalar fma would
          float2 a01 = make_float2(0.f, 0.f), a23 = make_float2(0.f, 0.f);
#pragma unroll
          for (int j4 = 0; j4 < 8; ++j4) {
            const float4 ww = wv[j4];
            a01 = __ffma2_rn(make_float2(ww.x, ww.y),
                             make_float2(fmaxf(v[4 * j4 + 0], 0.f), fmaxf(v[4 * j4 + 1], 0.f)), a01);
            a23 = __ffma2_rn(make_float2(ww.z, ww.w),
                             make_float2(fmaxf(v[4 * j4 + 2], 0.f), fmaxf(v[4 * j4 + 3], 0.f)), a23);
          }
          float sc = (a01.x + a01.y) + (a23.x + a23.y);
          if (FP8) sc *= kscale;
          if constexpr (MODE == kIdxScores) {
            if (s > pn) sc = -INFINITY;
            p.scores[static_cast<int64_t>(q0 + n) * p.b.max_len + s] = sc;
          } else if constexpr (MODE == kIdxSample) {
            if (s > pn) sc = -INFINITY;
            p.lists.sample[static_cast<int64_t>(q0 + n) * (kSampleTilesMax * 128) + (i0 + i) * 128 +
                           quarter * 32 + lane] = sc;
          } else {
            // keys at or above the row's cutoff (a float compare: NaN kept
            // too; a superset is harmless)
            const bool take = s <= pn && !(sc < cf[nn]);
            const uint32_t m = __ballot_sync(0xffffffffu, take);
            const int j = wc[nn] + __popc(m & lt);
            if (take && j < segq) {
              ck[nn][j] = order_key(sc);
              cp[nn][j] = s;
            }
            wc[nn] += __popc(m);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(bar(B_ACCE + acc));
    }
    if constexpr (MODE == kIdxCapture) {
      // this quarter's counts (a count above the quarter segment sends the
      // row to the fallback)
#pragma unroll
      for (int nn = 0; nn < C::TOK_PER_WARP; ++nn) {
        const int n = n0 + nn;
        if (lane == 0 && n < nq) {
          const int64_t r = q0 + n;
          p.lists.segcnt[(r * kSegMax + kc) * 4 + quarter] = wc[nn];
          if (kc == 0 && quarter == 0) p.lists.cnt[r * kTopkCnt + 0] = p.num_kc;
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == W_MMA) {
    tc_fence_after();
    tmem_dealloc(tbase, C::TMEM_COLS);
  }
}

template <int NTOK, bool FP8, int STAGES, int MODE>
cudaError_t launch_one(const CUtensorMap& qmap, const CUtensorMap& kmap, IndexerParams p,
                       cudaStream_t stream) {
  using C = IdxCfg<NTOK, FP8, STAGES, MODE>;
  auto* kern = indexer_kernel<NTOK, FP8, STAGES, MODE>;
  static int configured_device = -1;  // attribute is per device
  static int slots = 0;               // resident CTAs on the whole GPU
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device != dev) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    int sms = 0, per_sm = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, C::NT, C::SMEM);
    if (e != cudaSuccess) return e;
    slots = sms * (per_sm > 0 ? per_sm : 1);
    configured_device = dev;
  }
  if (p.whole_rows) {
    p.kc_blocks = (p.b.max_len + 127) / 128;
  } else if (NTOK == 1) {
    // decode: tiles per CTA chosen so that the CTAs fill whole waves of the
    // resident slots, weighing each CTA's start (barriers, TMEM, Q, first
    // tile) as about four tiles of streaming: min over kc of
    // ceil(CTAs(kc) / slots) * (kc + 4)
    const int64_t tiles = (p.b.max_len + 127) / 128;
    int best = 32;
    int64_t best_cost = INT64_MAX;
    // (at most kSegMax chunks per row: the capture splits a row's list by chunk)
    for (int kc = std::max<int64_t>(16, (tiles + kSegMax - 1) / kSegMax); kc <= 128; ++kc) {
      const int64_t ctas = static_cast<int64_t>(p.b.num_seqs) * ((tiles + kc - 1) / kc);
      const int64_t cost = ((ctas + slots - 1) / slots) * (kc + 4);
      if (cost < best_cost || (cost == best_cost && kc == 32)) {
        best_cost = cost;
        best = kc;
      }
    }
    p.kc_blocks = best;
  }
  p.num_qb = (p.b.max_q + NTOK - 1) / NTOK;
  if (MODE == kIdxSample) {
    // sampled tiles of the longest row (the same rule as in the kernel)
    const int tiles = (p.b.max_len + 127) / 128;
    const int ns = std::min(std::max(32, tiles / 64), kSampleTilesMax);
    p.num_kc = (std::min(tiles, ns) + kSampleChunk - 1) / kSampleChunk;
  } else {
    p.num_kc = (p.b.max_len + p.kc_blocks * 128 - 1) / (p.kc_blocks * 128);
  }
  dim3 grid(static_cast<unsigned>(p.num_qb) * static_cast<unsigned>(p.num_kc),
            static_cast<unsigned>(p.b.num_seqs));
  prof_begin(stream);
  cudaError_t e = launch_chained(kern, grid, dim3(C::NT), C::SMEM, stream, 1, qmap, kmap, p);
  prof_end(kLaunchIndexer, stream);
  count_launch(kLaunchIndexer);
  return e != cudaSuccess ? e : cudaGetLastError();
}

template <int MODE>
cudaError_t launch_mode(const CUtensorMap& qmap, const CUtensorMap& kmap, const IndexerParams& p,
                        bool decode, bool fp8, cudaStream_t stream) {
  if (decode)
    return fp8 ? launch_one<1, true, 6, MODE>(qmap, kmap, p, stream)
               : launch_one<1, false, 3, MODE>(qmap, kmap, p, stream);
  return fp8 ? launch_one<8, true, 6, MODE>(qmap, kmap, p, stream)
             : launch_one<8, false, 4, MODE>(qmap, kmap, p, stream);
}

}  // namespace

cudaError_t launch_indexer_mode(const void* q_idx, const float* q_scale, const float* w,
                                const void* k_idx, const float* k_scale, int64_t k_rows, bool fp8,
                                const dsa_batch_t& b, int mode, float* scores, const int* only,
                                const TopkLists& lists, int* status, cudaStream_t stream) {
  if (b.num_q == 0) return cudaSuccess;
  const bool decode = b.max_q <= 1;
  const int ntok = decode ? 1 : 8;
  const auto dt = fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const int es = fp8 ? 1 : 2;
  const uint32_t box_inner = fp8 ? 128 : 64;
  CUtensorMap qmap, kmap;
  if (!make_tmap_2d(&qmap, q_idx, dt, es, 128, static_cast<uint64_t>(b.num_q) * 32, box_inner,
                    ntok * 32))
    return cudaErrorInvalidValue;
  if (!make_tmap_2d(&kmap, k_idx, dt, es, 128, static_cast<uint64_t>(k_rows), box_inner, 128))
    return cudaErrorInvalidValue;
  IndexerParams p{};
  p.b = to_args(b);
  p.w = w;
  p.q_scale = q_scale;
  p.k_scale = k_scale;
  p.k_rows = k_rows;
  p.scores = scores;
  p.status = status;
  p.kc_blocks = 64;  // 128-key tiles per CTA (one Q load per 8K keys); decode: see launch_one
  p.fill_tail = 0;
  p.timeout_ns = wait_timeout_ns();
  p.only = only;
  p.whole_rows = only ? 1 : 0;  // the fallback: few rows, normally none
  p.lists = lists;
  if (mode == kIdxSample) return launch_mode<kIdxSample>(qmap, kmap, p, decode, fp8, stream);
  if (mode == kIdxCapture) return launch_mode<kIdxCapture>(qmap, kmap, p, decode, fp8, stream);
  return launch_mode<kIdxScores>(qmap, kmap, p, decode, fp8, stream);
}

cudaError_t launch_indexer(const void* q_idx, const float* q_scale, const float* w,
                           const void* k_idx, const float* k_scale, int64_t k_rows, bool fp8,
                           const dsa_batch_t& b, float* scores, bool fill_tail, int* status,
                           cudaStream_t stream) {
  if (b.num_q == 0) return cudaSuccess;
  const bool decode = b.max_q <= 1;
  const int ntok = decode ? 1 : 8;
  const auto dt = fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const int es = fp8 ? 1 : 2;
  const uint32_t box_inner = fp8 ? 128 : 64;
  CUtensorMap qmap, kmap;
  if (!make_tmap_2d(&qmap, q_idx, dt, es, 128, static_cast<uint64_t>(b.num_q) * 32, box_inner,
                    ntok * 32))
    return cudaErrorInvalidValue;
  if (!make_tmap_2d(&kmap, k_idx, dt, es, 128, static_cast<uint64_t>(k_rows), box_inner, 128))
    return cudaErrorInvalidValue;
  IndexerParams p{};
  p.b = to_args(b);
  p.w = w;
  p.q_scale = q_scale;
  p.k_scale = k_scale;
  p.k_rows = k_rows;
  p.scores = scores;
  p.status = status;
  p.kc_blocks = 64;  // 128-key tiles per CTA (one Q load per 8K keys); decode: see launch_one
  p.fill_tail = fill_tail ? 1 : 0;
  p.timeout_ns = wait_timeout_ns();
  return launch_mode<kIdxScores>(qmap, kmap, p, decode, fp8, stream);
}

}  // namespace dsa

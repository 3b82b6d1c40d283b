// Absorbed-MLA sparse attention over the selected positions of one layer.
//
//   z_s = scale * (q_lat[t,h] . C[s,:512] + q_rope[t,h] . C[s,512:])
//   out[t,h] = sum_s softmax(z)_s C[s,:512]
//
// ("GLM-5.2 / 总览" config table: the 512-d latent is both key and value, the
// 64-d RoPE key enters only the score, QK head dim 256 -> scale 1/16;
// "GLM-5 -> 5.1 -> 5.2" section 10: each layer gathers the selected entries
// of its own cache, then runs sparse attention.)
//
// GB300 design.  One CTA (or a cluster of NSPLIT CTAs, for decode) per query
// token.  Both products run on tcgen05 with the 128 gathered KEYS on the MMA
// M dimension:
//   S^T[128 keys, H]   = C[128, 576] . Q[H, 576]^T         (A = C, K-major)
//   O^T[512 dims, H]  += C[128, :512]^T . P^T[H, 128]^T     (A = C^T, MN-major)
// so both contractions use the full 128-row datapath even with H = 64 (or
// 16) heads.  The selected rows are gathered with 16-byte cp.async straight
// into the 128-byte-swizzled MMA operand layout, in four groups of 64-column
// sub-tiles (completion tracked on one mbarrier per group), and each group is
// refilled for the next block as soon as the P.V chunk that reads it
// completes.  (TMA gather4 of 128-byte row segments sustains only about
// 2 TB/s over the whole chip; cp.async sustains several times that.)  P^T
// reuses the RoPE sub-tile, which is free once S^T is computed.
//
// Softmax: the thread of TMEM lane i owns key i of the block; at H = 64 two
// warps share each lane quarter, one per half of the heads.  The running
// maximum per head is only raised when a block exceeds it by more than 2^8
// (then O^T and the partial sums are rescaled in place); row sums are kept
// per thread and reduced once at the end.
//
// Warp roles: softmax / gather / epilogue warps (8 at H = 64, 4 at H = 16;
// idle during the products, so they also issue the next block's gathers),
// then the QK issuer warp (also loads Q by TMA) and the P.V issuer warp
// (also the TMEM owner).  Issuing the two products from different warps
// matters: an mbarrier wait in an issuing thread stalls until that thread's
// queued MMAs have drained, so one issuer waiting for gathered data would
// empty the tensor pipe every time.
#include <cuda_bf16.h>

#include <algorithm>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "common.cuh"

namespace dsa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

template <int H>
struct MlaCfg {
  static constexpr int QSUB = H * 128;       // one 64-dim sub-tile of Q: H rows x 128 B
  static constexpr int Q_BYTES = 9 * QSUB;
  static constexpr int CSUB = 128 * 128;     // one 64-dim sub-tile of 128 gathered rows
  static constexpr int PSUB = H * 128;       // P^T sub-tile (H = 16): H rows x 64 keys
  // At H = 64, P is stored MN-major: one 128-byte row of 64 heads per key.
  static constexpr bool P_MN = H == 64;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_C = OFF_Q + Q_BYTES;
  static constexpr int OFF_P = OFF_C + 8 * CSUB;  // the RoPE sub-tile
  static constexpr int OFF_SCR = OFF_C + 9 * CSUB;
  // scratch (floats): m_used[H], red[4][H], lsum[H], fac[16][H]; flags[NSW]
  static constexpr int SCR_FLOATS = H + 4 * H + H + 16 * H;
  static constexpr int OFF_FLAGS = OFF_SCR + SCR_FLOATS * 4;
  static constexpr int OFF_BAR = (OFF_FLAGS + 4 * 8 + 7) & ~7;
  static constexpr int NBAR = 1 + 4 + 4 + 4;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  // the sequence's block-table row (paged caches), when it has <= TAB_MAX entries
  static constexpr int TAB_MAX = 512;
  static constexpr int OFF_TAB = (OFF_MISC + 64 + 15) & ~15;
  // FP8 KV rows: the block's 128 x 4 fp32 group scales (16-byte cp.async targets)
  static constexpr int OFF_KSC = OFF_TAB + TAB_MAX * 4;
  static constexpr int SMEM = OFF_KSC + 128 * 16 + 1024;
  static_assert(OFF_KSC % 16 == 0, "cp.async destinations need 16-byte alignment");
  static constexpr int HW = H > 32 ? 32 : H;       // heads per softmax warp
  static constexpr int NSW = 4 * (H / HW);           // softmax warps (two per lane quarter at H=64)
  static constexpr int NT = NSW * 32 + 64;           // + the QK and the P.V issuer warps
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t TM_S = 0;        // S^T: H columns
  static constexpr uint32_t TM_O = 256;      // O^T chunk c: columns 256 + c*H
  static_assert(OFF_C % 1024 == 0 && OFF_P % 1024 == 0, "swizzled tiles need 1024-B alignment");
  static_assert(PSUB * 2 <= CSUB, "P^T must fit in the RoPE sub-tile");
  static_assert(H * 512 * 4 <= 9 * CSUB, "O staging must fit in the C tile");
  static_assert(SMEM <= 232448, "shared memory");
};

struct MlaParams {
  BatchArgs b;
  const uint16_t* kv;  // [kv_rows, 576] bf16
  const uint8_t* kv8;  // or FP8 rows [kv_rows, 656]: 512 E4M3, 4 fp32 group scales, 64 bf16
  int64_t kv_rows;
  int direct;  // index entries are absolute kv rows (no causal test), not positions
  int l2_prefetch;  // prefetch the block after next into L2 (caches larger than L2)
  const int32_t* idx;
  int K;
  float scale_log2;
  uint16_t* out;
  float* lse;
  // tokens split over 4, 8 or 16 CTAs: partial results of CTA r of token t at
  // part + (t * NSPLIT + r) * (H * 512 + 2 * H): O^T as [h][512], then the
  // running maxima and the row sums of the H heads
  float* part;
  int* status;
  uint64_t timeout_ns;
  // launched right after another of the library's kernels of the group call
  // (none of which writes the batch metadata): the token's metadata and the
  // barrier and TMEM set-up run before the wait for that kernel; the query
  // load (in a model the kernel just before would produce the queries), the
  // indices, the cache rows and every write after it.  This kernel lets the
  // next one be scheduled only after its own wait, so a kernel launched after
  // it finds every kernel two or more places back in the stream complete.
  int early_inputs;
  // (with early_inputs, bf16 rows) launched right after another attention
  // launch, whose predecessor wrote the indices and the cache rows if
  // anything did: the first block's indices, and its rows of positions before
  // the sequence's first query of the call, are gathered before the wait too
  // (in a model those exist before the layer starts; the call's own new rows
  // come from the layer's projection just before it and follow the wait)
  int early_gather;
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Per-head reduction over the 32 keys (lanes) of a warp, N heads per lane, as
// a transposing butterfly: at distance 16 each lane keeps half of its heads
// and trades the other half with its partner, then the same at distance 8 on
// the half it kept, down to distance 1: 31 shuffles for 32 heads instead of
// 5 per head.  Each level combines the same two partial results as the plain
// xor butterfly, so sums come out bit for bit the same.  On return v[0] holds
// the result for head lane (N = 32) or lane / 2 (N = 16).
template <int N, int OFF, bool MAX>
__device__ __forceinline__ void head_reduce(float* v, int lane) {
  if constexpr (OFF >= 1) {
    if constexpr (N > 1) {
      constexpr int HF = N / 2;
      const bool up = (lane & OFF) != 0;
#pragma unroll
      for (int i = 0; i < HF; ++i) {
        const float keep = up ? v[i + HF] : v[i];
        const float give = up ? v[i] : v[i + HF];
        const float got = __shfl_xor_sync(0xffffffffu, give, OFF);
        v[i] = MAX ? fmaxf(keep, got) : keep + got;
      }
      head_reduce<HF, OFF / 2, MAX>(v, lane);
    } else {
      const float got = __shfl_xor_sync(0xffffffffu, v[0], OFF);
      v[0] = MAX ? fmaxf(v[0], got) : v[0] + got;
      head_reduce<1, OFF / 2, MAX>(v, lane);
    }
  }
}

template <int NV>
__device__ __forceinline__ void wait_ld_dep(float (&v)[NV]) {
  static_assert(NV == 16 || NV == 32, "");
  if constexpr (NV == 32) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+f"(v[0]), "+f"(v[1]), "+f"(v[2]), "+f"(v[3]), "+f"(v[4]), "+f"(v[5]),
                   "+f"(v[6]), "+f"(v[7]), "+f"(v[8]), "+f"(v[9]), "+f"(v[10]), "+f"(v[11]),
                   "+f"(v[12]), "+f"(v[13]), "+f"(v[14]), "+f"(v[15]), "+f"(v[16]), "+f"(v[17]),
                   "+f"(v[18]), "+f"(v[19]), "+f"(v[20]), "+f"(v[21]), "+f"(v[22]), "+f"(v[23]),
                   "+f"(v[24]), "+f"(v[25]), "+f"(v[26]), "+f"(v[27]), "+f"(v[28]), "+f"(v[29]),
                   "+f"(v[30]), "+f"(v[31])
                 :
                 : "memory");
  } else {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+f"(v[0]), "+f"(v[1]), "+f"(v[2]), "+f"(v[3]), "+f"(v[4]), "+f"(v[5]),
                   "+f"(v[6]), "+f"(v[7]), "+f"(v[8]), "+f"(v[9]), "+f"(v[10]), "+f"(v[11]),
                   "+f"(v[12]), "+f"(v[13]), "+f"(v[14]), "+f"(v[15])
                 :
                 : "memory");
  }
}

// Load / store NV consecutive fp32 TMEM columns of this thread's lane.
template <int NV>
__device__ __forceinline__ void tmem_cols_load(uint32_t taddr, float (&v)[NV]) {
  if constexpr (NV == 16)
    tmem_ld16(taddr, v);
  else
    tmem_ld32(taddr, v);
  wait_ld_dep(v);
}
template <int NV>
__device__ __forceinline__ void tmem_cols_store(uint32_t taddr, const float (&v)[NV]) {
  if constexpr (NV == 16)
    tmem_st16(taddr, v);
  else
    tmem_st32(taddr, v);
}

// MMA issue.  One thread issues every product of a block, and the tensor
// pipe takes an M128 N64 K16 bf16 MMA every ~49 cycles; computing each
// operand descriptor from a run-time sub-tile or chunk index cost the issuing
// thread more than that (measured: ~72 cycles per QK and ~66 per P.V MMA with
// those loops, ~49 fully unrolled).  So the issuers take a descriptor of each
// tile's base once and step through the tile with compile-time offsets: the
// start-address field holds (address >> 4) in its low 14 bits and every tile
// ends below 256 KB of shared memory, so adding offset >> 4 to the 64-bit
// descriptor never carries out of the field.
__device__ __forceinline__ uint64_t sdesc_at(uint64_t base, uint32_t byte_off) {
  // only the low word changes: one add per descriptor
  return (base & 0xFFFFFFFF00000000ull) | (static_cast<uint32_t>(base) + (byte_off >> 4));
}

// S^T (+)= C_s . Q_s^T for the sub-tiles s of dims group G (0-2: two latent
// sub-tiles; 3: the last two latent sub-tiles and the RoPE sub-tile).
template <int G, class C>
__device__ __forceinline__ void issue_qk_group(uint32_t d_s, uint64_t dc, uint64_t dq,
                                               uint32_t idesc) {
  // the bases are opaque here, so the descriptors are formed as they are
  // issued rather than all kept in registers across the block loop
  asm volatile("" : "+l"(dc), "+l"(dq));
  constexpr int s_end = G == 3 ? 9 : 2 * G + 2;
#pragma unroll
  for (int s = 2 * G; s < s_end; ++s)
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
      umma_bf16(d_s, sdesc_at(dc, s * C::CSUB + kk * 32), sdesc_at(dq, s * C::QSUB + kk * 32),
                idesc, (s | kk) != 0);
}

// O^T chunk c (+)= C^T . P over the block's 128 keys (K = 16 per MMA); the
// first MMA of a token's first block overwrites the accumulator.
template <int c, class C>
__device__ __forceinline__ void issue_pv_chunk(uint32_t d_o, uint64_t dcv, uint64_t dp,
                                               uint32_t idesc, bool first) {
  asm volatile("" : "+l"(dcv), "+l"(dp));
#pragma unroll
  for (int kk = 0; kk < 8; ++kk)
    umma_bf16(d_o, sdesc_at(dcv, 2 * c * C::CSUB + kk * 2048),
              sdesc_at(dp, C::P_MN ? kk * 2048 : (kk >> 2) * C::PSUB + (kk & 3) * 32), idesc,
              (kk > 0 || !first) ? 1u : 0u);
}

// bf16 bits of four E4M3 codes (one 32-bit word, lowest byte first) times
// their group scale: the codes widen exactly to fp16 then fp32, the fp32
// products round to nearest even (two lanes per packed multiply), and each
// narrows to bf16 with round to nearest even.
__device__ __forceinline__ uint2 scaled_e4m3x4_to_bf16x4(uint32_t w, float2 sc2) {
  const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w & 0xFFFFu), __NV_E4M3);
  const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w >> 16), __NV_E4M3);
  const __nv_bfloat162 a = __float22bfloat162_rn(__fmul2_rn(__half22float2(__half2(lo)), sc2));
  const __nv_bfloat162 b = __float22bfloat162_rn(__fmul2_rn(__half22float2(__half2(hi)), sc2));
  return make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b));
}

template <int H, int NSPLIT, bool PAGED, bool KV8>
__global__ void __launch_bounds__(MlaCfg<H>::NT, 1)
    sparse_mla_kernel(const __grid_constant__ CUtensorMap qlat_map,
                      const __grid_constant__ CUtensorMap qrope_map, const MlaParams p) {
  if (!p.early_inputs) {
    chain_wait();     // the previous kernel of the stream has completed
    chain_release();  // the next one may be scheduled
  }
  using C = MlaCfg<H>;
  constexpr int HW = C::HW, NSW = C::NSW, NT = C::NT, NST = NSW * 32;
  // split tokens combine their partial results through L2 for 4 to 16 CTAs
  // (each CTA would read 128 KB through the cluster, at ~35 GB/s per SM),
  // through distributed shared memory for 2 (half of it local)
  constexpr bool kMergeL2 = NSPLIT >= 4;
  // Two issuer warps: an mbarrier wait in the issuing thread stalls until its
  // own queued MMAs have drained, so the QK products (which wait for each
  // gathered group) and the P.V products (which wait for P) come from
  // different warps and the tensor pipe keeps the other stream's work.
  constexpr int W_QK = NSW, W_PV = NSW + 1;
  // gathering: thread g of the softmax warps copies 16-byte chunk (g & 7) of
  // rows (g >> 3) + GROW * c, c < RPT, of every 64-column sub-tile
  constexpr int GROW = NST / 8, RPT = 128 / GROW;
  static_assert(GROW % 8 == 0, "rows of one thread must share the swizzle phase");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rank = NSPLIT > 1 ? static_cast<int>(cluster_ctarank()) : 0;

  // ---- token of this CTA (cluster): heaviest (latest) tokens first
  const int seq = blockIdx.y;
  const int qi = p.b.max_q - 1 - static_cast<int>(blockIdx.x / NSPLIT);
  int qs, qe;
  seq_rows(p.b, seq, p.status, qs, qe);
  const int t = qs + qi;
  if (t >= qe) return;  // uniform over the cluster
  const int pos = query_pos(p.b, t, (tid == 0 && rank == 0) ? p.status : nullptr);
  const int nvalid = pos < 0 ? 0 : min(p.K, pos + 1);
  // first position this call adds to the sequence (its first query's)
  const int first_new = p.early_gather ? (t == qs ? pos : query_pos(p.b, qs, nullptr)) : 0;
  const int nb = (nvalid + 127) / 128;
  const int j0 = rank * nb / NSPLIT, j1 = (rank + 1) * nb / NSPLIT;  // this CTA's blocks
  const int64_t row0 = p.direct ? 0 : seq_base_row(p.b, seq);
  const int32_t* idx_row = p.idx + static_cast<int64_t>(t) * p.K;
  if (nb == 0) {  // nothing visible: zero output, lse = -inf
    if (p.early_inputs) {
      chain_wait();
      chain_release();
    }
    constexpr int DS = 512 / NSPLIT;
    for (int i = tid; i < H * DS; i += NT) {
      const int h = i / DS, d = rank * DS + i % DS;
      p.out[(static_cast<int64_t>(t) * H + h) * 512 + d] = 0;
    }
    if (rank == 0 && p.lse && tid < H) p.lse[static_cast<int64_t>(t) * H + tid] = -INFINITY;
    return;
  }

  const uint32_t sQ = smem_u32(sm + C::OFF_Q);
  const uint32_t sC = smem_u32(sm + C::OFF_C);
  const uint32_t sP = smem_u32(sm + C::OFF_P);
  float* m_used = reinterpret_cast<float*>(sm + C::OFF_SCR);
  float* red = m_used + H;
  float* lsum = red + 4 * H;
  float* fac = lsum + H;
  int* flags = reinterpret_cast<int*>(sm + C::OFF_FLAGS);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::OFF_BAR);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + C::OFF_MISC);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + C::OFF_MISC + 8);
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  // CFULL(g) / CFREE(g): gathered group g landed / P.V chunk g done reading it.
  // Group g = sub-tiles 2g, 2g+1 (group 3 also the RoPE sub-tile 8).
  const int B_Q = 0, B_CFULL = 1, B_CFREE = 5, B_S = 9, B_P = 10, B_O = 11, B_QD = 12;

  if (tid == 0) {
    *abort_flag = 0;
    mbar_init(bar(B_Q), 1);
    for (int i = 0; i < 4; ++i) mbar_init(bar(B_CFULL + i), NST);
    for (int i = 0; i < 4; ++i) mbar_init(bar(B_CFREE + i), 1);
    mbar_init(bar(B_S), 1);
    mbar_init(bar(B_P), NST);
    mbar_init(bar(B_O), 1);
    mbar_init(bar(B_QD), 1);
    fence_mbar_init();
  }
  if (tid < H) m_used[tid] = -INFINITY;
  // Paged caches: the sequence's block-table row is staged in shared memory
  // (when short enough) so that the per-key row lookups of the gather and
  // of the softmax's validity test stay off global memory.
  int32_t* stab = reinterpret_cast<int32_t*>(sm + C::OFF_TAB);
  const int bps = p.b.blocks_per_seq;
  const bool tab_smem = PAGED && bps <= C::TAB_MAX;
  if (tab_smem)
    for (int i = tid; i < bps; i += NT) stab[i] = p.b.block_table[static_cast<int64_t>(seq) * bps + i];
  const int rshift = PAGED ? __ffs(p.b.block_rows) - 1 : 0;  // block_rows is a power of two
  auto row_of = [&](int e) -> int64_t {  // cache row of selected position e >= 0, -1 if unmapped
    if constexpr (!PAGED) {
      return row0 + e;
    } else {
      const int blk = e >> rshift;
      if (blk >= bps) return -1;
      const int32_t id =
          tab_smem ? stab[blk] : p.b.block_table[static_cast<int64_t>(seq) * bps + blk];
      return id < 0 ? -1
                    : (static_cast<int64_t>(id) << rshift) + (e & (p.b.block_rows - 1));
    }
  };
  if (warp == W_PV) {
    tmem_alloc(smem_u32(tslot), C::TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == W_QK && lane == 0) {
    tma_prefetch_desc(&qlat_map);
    tma_prefetch_desc(&qrope_map);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;
  const uint64_t to = p.timeout_ns;
  volatile int no_abort = 0;
  if (warp == W_QK && lane == 0) {  // Q of the token, once, by TMA
    if (p.early_inputs) chain_wait();
    mbar_arrive_expect_tx(bar(B_Q), C::Q_BYTES);
    for (int c = 0; c < 8; ++c) tma_load_2d(sQ + c * C::QSUB, &qlat_map, 64 * c, t * H, bar(B_Q));
    tma_load_2d(sQ + 8 * C::QSUB, &qrope_map, 0, t * H, bar(B_Q));
  }
  if (p.early_inputs && !p.early_gather) {  // before the indices, the cache rows and any write
    chain_wait();
    chain_release();
  }

  if (warp == W_QK) {
    // ------------------------------------------------ QK issuer: S^T = C . Q^T per block
    if (lane == 0) {
      constexpr uint32_t id_qk = idesc_bf16(128, H, false, false);
      const uint64_t dc = sdesc_sw128(sC, 0, 1024), dq = sdesc_sw128(sQ, 0, 1024);
      const uint32_t d_s = tbase + C::TM_S;
      bool ok = mbar_wait(bar(B_Q), 0, abort_flag, p.status, to);
      for (int j = j0; ok && j < j1; ++j) {
        const int u = j - j0;
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          ok = mbar_wait(bar(B_CFULL + g), u & 1, abort_flag, p.status, to);
          if (!ok) break;
          fence_proxy_async_smem();  // cp.async (generic proxy) writes -> tcgen05.mma reads
          tc_fence_after();
          if (g == 0)
            issue_qk_group<0, C>(d_s, dc, dq, id_qk);
          else if (g == 1)
            issue_qk_group<1, C>(d_s, dc, dq, id_qk);
          else if (g == 2)
            issue_qk_group<2, C>(d_s, dc, dq, id_qk);
          else
            issue_qk_group<3, C>(d_s, dc, dq, id_qk);
        }
        if (!ok) break;
        umma_commit(bar(B_S));
      }
      umma_commit(bar(B_QD));  // drain this warp's products before exit
      mbar_wait(bar(B_QD), 0, &no_abort, nullptr, to);
      mbar_wait(bar(B_Q), 0, &no_abort, nullptr, to);  // the Q copy has landed before exit
    }
    __syncwarp();
  } else if (warp == W_PV) {
    // ------------------------------------------------ P.V issuer: O^T += C^T . P per block
    if (lane == 0) {
      constexpr uint32_t id_pv = idesc_bf16(128, H, true, C::P_MN);
      const uint64_t dcv = sdesc_sw128(sC, C::CSUB, 1024);
      const uint64_t dp = C::P_MN ? sdesc_sw128(sP, 8192, 1024) : sdesc_sw128(sP, 0, 1024);
      const uint32_t d_o = tbase + C::TM_O;
      bool ok = true;
      for (int j = j0; ok && j < j1; ++j) {
        const int u = j - j0;
        ok = mbar_wait(bar(B_P), u & 1, abort_flag, p.status, to);
        if (!ok) break;
        tc_fence_after();
        issue_pv_chunk<0, C>(d_o, dcv, dp, id_pv, u == 0);
        umma_commit(bar(B_CFREE + 0));
        issue_pv_chunk<1, C>(d_o + H, dcv, dp, id_pv, u == 0);
        umma_commit(bar(B_CFREE + 1));
        issue_pv_chunk<2, C>(d_o + 2 * H, dcv, dp, id_pv, u == 0);
        umma_commit(bar(B_CFREE + 2));
        issue_pv_chunk<3, C>(d_o + 3 * H, dcv, dp, id_pv, u == 0);
        umma_commit(bar(B_CFREE + 3));
      }
      umma_commit(bar(B_O));
      mbar_wait(bar(B_O), 0, &no_abort, nullptr, to);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ softmax: key = TMEM lane, HW heads
    const int quarter = warp & 3;              // TMEM lane quarter this warp may access
    const int h0 = (warp >> 2) * HW;           // first head of this warp
    const int key = quarter * 32 + lane;       // key of the block (= TMEM lane)
    const uint32_t lane_base = tbase + (static_cast<uint32_t>(quarter * 32) << 16);
    const float sl2 = p.scale_log2;
    float lpart[HW];  // this thread's share of the softmax denominators
    // minus the running maxima (log2 units, +inf before any key): in registers
    // for unsplit tokens, read from shared memory where they are used in the
    // split instances (registers for them made those spill; the unsplit ones
    // measured 1.7 % (bf16) and 2.3 % (FP8 rows) slower with the shared-memory
    // reads)
    constexpr bool kMaxRegs = NSPLIT == 1;
    float mneg[kMaxRegs ? HW : 1];
#pragma unroll
    for (int h = 0; h < HW; ++h) {
      lpart[h] = 0.f;
      if constexpr (kMaxRegs) mneg[h] = INFINITY;
    }
    auto neg_max = [&](int h) -> float {
      if constexpr (kMaxRegs)
        return mneg[h];
      else
        return -m_used[h0 + h];
    };
    // ---- gathering role: the selected rows of the next block are copied
    // with 16-byte cp.async into the 128-byte-swizzled K-major layout the
    // MMA reads, each sub-tile as soon as the P.V chunk reading it is done.
    // (Spread over all softmax warps: a warp's cp.async and its mbarrier
    // waits share one queue, so few gathering warps issue slowly.)
    const int kch = tid & 7, rb = tid >> 3;
    const uint32_t gdst0 = sC + rb * 128 + ((kch ^ (rb & 7)) << 4);
    const uint16_t* kvk = p.kv + kch * 8;
    int gsel[RPT];  // selected positions of this thread's rows in the block being gathered
    auto fetch_sel = [&](int jj) {
#pragma unroll
      for (int c = 0; c < RPT; ++c) {
        const int sl = jj * 128 + rb + GROW * c;
        gsel[c] = sl < nvalid ? idx_row[sl] : -1;
      }
    };
    int grow[RPT];  // cache rows (< kv_rows < 2^31) of those positions; row 0 for padding
    auto resolve_rows = [&]() {
#pragma unroll
      for (int c = 0; c < RPT; ++c) {
        const int e = gsel[c];
        const int64_t rr = e >= 0 ? row_of(e) : -1;
        const bool ok = e >= 0 && (p.direct || e <= pos) && rr >= 0 && rr < p.kv_rows;
        if (!ok && e != -1 && kch == 0) atomicOr(p.status, DSA_DEVERR_INDEX);
        grow[c] = ok ? static_cast<int>(rr) : 0;
      }
    };
    // rows rb + GROW * c of sub-tile i for the c set in `rows`
    auto issue_rows = [&](int i, uint32_t rows) {
      const uint32_t dst = gdst0 + i * C::CSUB;
#pragma unroll
      for (int c = 0; c < RPT; ++c)
        if ((rows >> c) & 1u)
          asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst + c * GROW * 128),
                       "l"(kvk + static_cast<int64_t>(grow[c]) * 576 + 64 * i)
                       : "memory");
    };
    auto issue = [&](int i) { issue_rows(i, (1u << RPT) - 1u); };
    // ---- FP8 KV rows: a group's codes (128 keys x 128 dims, 16 KB) are staged
    // unswizzled in its second sub-tile, its rows' scales in a 2 KB area,
    // then the threads that copied them expand them in place to the swizzled
    // bf16 operand layout (the 8 threads of a row share a warp, so warp
    // barriers order the reads of the codes before the writes over them).
    const uint32_t sKsc = smem_u32(sm + C::OFF_KSC);
    auto issue8 = [&](int g) {
      const uint32_t dst = sC + (2 * g + 1) * C::CSUB + rb * 128 + kch * 16;
#pragma unroll
      for (int c = 0; c < RPT; ++c)
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst + c * GROW * 128),
                     "l"(p.kv8 + static_cast<int64_t>(grow[c]) * 656 + 128 * g + kch * 16)
                     : "memory");
      if (g == 0 && kch == 0) {
#pragma unroll
        for (int c = 0; c < RPT; ++c)
          asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sKsc + (rb + GROW * c) * 16),
                       "l"(p.kv8 + static_cast<int64_t>(grow[c]) * 656 + 512)
                       : "memory");
      }
      if (g == 3) {  // the RoPE key, bf16 as stored, into its swizzled sub-tile
        const uint32_t rdst = gdst0 + 8 * C::CSUB;
#pragma unroll
        for (int c = 0; c < RPT; ++c)
          asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(rdst + c * GROW * 128),
                       "l"(p.kv8 + static_cast<int64_t>(grow[c]) * 656 + 528 + kch * 16)
                       : "memory");
      }
      asm volatile("cp.async.commit_group;" ::: "memory");
    };
    auto convert8 = [&](int g, int pending) {  // pending: younger copy groups still allowed
      if (pending == 0)
        asm volatile("cp.async.wait_group 0;" ::: "memory");
      else if (pending == 1)
        asm volatile("cp.async.wait_group 1;" ::: "memory");
      else if (pending == 2)
        asm volatile("cp.async.wait_group 2;" ::: "memory");
      else
        asm volatile("cp.async.wait_group 3;" ::: "memory");
#pragma unroll 1
      for (int c = 0; c < RPT; ++c) {
        const int r = rb + GROW * c;
        // every code of row r is read (by its 8 threads, one warp) before any
        // of them writes over it; rows of other c are disjoint
        __syncwarp();
        const uint4 cv = *reinterpret_cast<const uint4*>(sm + C::OFF_C + (2 * g + 1) * C::CSUB +
                                                         r * 128 + kch * 16);
        const float sc = *reinterpret_cast<const float*>(sm + C::OFF_KSC + r * 16 + 4 * g);
        __syncwarp();
        const float2 s2 = make_float2(sc, sc);
        const uint2 o01 = scaled_e4m3x4_to_bf16x4(cv.x, s2), o23 = scaled_e4m3x4_to_bf16x4(cv.y, s2);
        const uint2 o45 = scaled_e4m3x4_to_bf16x4(cv.z, s2), o67 = scaled_e4m3x4_to_bf16x4(cv.w, s2);
        // dims 128g + 16kch .. +15: sub-tile 2g + kch/4, 16-byte chunks 2(kch%4), 2(kch%4)+1
        uint8_t* tile = sm + C::OFF_C + (2 * g + (kch >> 2)) * C::CSUB + r * 128;
        const int ch = 2 * (kch & 3);
        *reinterpret_cast<uint4*>(tile + ((ch ^ (r & 7)) << 4)) = make_uint4(o01.x, o01.y, o23.x, o23.y);
        *reinterpret_cast<uint4*>(tile + (((ch + 1) ^ (r & 7)) << 4)) =
            make_uint4(o45.x, o45.y, o67.x, o67.y);
      }
      fence_proxy_async_smem();
      mbar_arrive(bar(B_CFULL + g));
    };
    // CFULL(g) completes once every copy this thread issued so far has landed
    auto signal = [&](int g) {
      asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar(B_CFULL + g))
                   : "memory");
    };
    // ---- the rows of the block after next are prefetched into L2 (bulk, no
    // completion) while this block runs, so that the refill gathers hit L2
    // rather than HBM; the 8 threads of a row share it, thread kch == 0 issues
    int psel[RPT];
    auto fetch_pf = [&](int jj) {
      if (kch == 0 && p.l2_prefetch)
#pragma unroll
        for (int c = 0; c < RPT; ++c) {
          const int sl = jj * 128 + rb + GROW * c;
          psel[c] = (jj < j1 && sl < nvalid) ? idx_row[sl] : -1;
        }
    };
    auto prefetch_rows = [&]() {
      if (kch == 0 && p.l2_prefetch)
#pragma unroll
        for (int c = 0; c < RPT; ++c) {
          const int e = psel[c];
          if (e < 0 || (!p.direct && e > pos)) continue;
          const int64_t rr = row_of(e);
          if (rr < 0 || rr >= p.kv_rows) continue;
          if constexpr (KV8)
            bulk_prefetch_l2(p.kv8 + rr * 656, 656);
          else
            bulk_prefetch_l2(p.kv + rr * 576, 1152);
        }
    };
    if (j0 < j1) {
      fetch_pf(j0 + 1);
      fetch_sel(j0);
      resolve_rows();
      if constexpr (KV8) {
#pragma unroll 1
        for (int g = 0; g < 4; ++g) issue8(g);
#pragma unroll 1
        for (int g = 0; g < 4; ++g) convert8(g, 3 - g);
      } else {
        // rows of this call's new positions (at or after the sequence's first
        // query) wait for the previous kernel when gathering early
        uint32_t late = 0;
        if (p.early_gather)
#pragma unroll
          for (int c = 0; c < RPT; ++c)
            if (gsel[c] >= first_new) late |= 1u << c;
        const uint32_t early = ((1u << RPT) - 1u) & ~late;
#pragma unroll 1
        for (int g = 0; g < 4; ++g) {
          issue_rows(2 * g, early);
          issue_rows(2 * g + 1, early);
          if (g == 3) issue_rows(8, early);
        }
        if (p.early_gather) {
          chain_wait();
          chain_release();
        }
#pragma unroll 1
        for (int g = 0; g < 4; ++g) {
          issue_rows(2 * g, late);
          issue_rows(2 * g + 1, late);
          if (g == 3) issue_rows(8, late);
          signal(g);
        }
      }
    }
    if (p.early_gather && j0 >= j1) {
      chain_wait();
      chain_release();
    }

    int e_next = (j0 * 128 + key < nvalid && j0 < j1) ? idx_row[j0 * 128 + key] : -1;
    for (int j = j0; j < j1; ++j) {
      const int u = j - j0;
      const bool more = j + 1 < j1;
      const int e = e_next;  // index of this thread's key, loaded one block ahead
      {
        const int sn = (j + 1) * 128 + key;
        e_next = (more && sn < nvalid) ? idx_row[sn] : -1;
      }
      if (more) fetch_sel(j + 1);  // consumed after P of this block
      if (j == j0) prefetch_rows();  // block j0 + 1
      if (j + 2 < j1) fetch_pf(j + 2);  // prefetched after this block's refill
      // the gather's test on this thread's key, before the wait (which hides a
      // paged cache's table lookup)
      bool valid = e >= 0 && (p.direct || e <= pos);
      if (valid) {
        const int64_t rr = row_of(e);
        valid = rr >= 0 && rr < p.kv_rows;
      }
      if (!mbar_wait(bar(B_S), u & 1, abort_flag, p.status, to)) break;
      tc_fence_after();
      // d = scale*log2(e)*s - m: the exponent of P and the rescale test in one FFMA
      float d[HW];
      tmem_cols_load<HW>(lane_base + C::TM_S + h0, d);
      // the first block sets the running maximum; a later one raises it only
      // when one of its scores exceeds it by more than the threshold
      int resc = 1;
      if (u > 0) {
        float dmax = -INFINITY;
#pragma unroll
        for (int h = 0; h < HW; ++h) {
          d[h] = fmaf(d[h], sl2, neg_max(h));
          dmax = fmaxf(dmax, d[h]);
        }
        const bool exceed = valid && dmax > kRescaleThreshold;
        const unsigned any = __any_sync(0xffffffffu, exceed);
        if (lane == 0) flags[warp] = any ? 1 : 0;
        named_bar_sync(1, NST);
        resc = 0;
#pragma unroll
        for (int w = 0; w < NSW; ++w) resc |= flags[w];
        if (resc) tmem_cols_load<HW>(lane_base + C::TM_S + h0, d);  // raw scores again
      }
      if (resc) {
        // raise the running maximum to this block's maximum (rare after the
        // first block): exact per-head maximum over the valid keys
#pragma unroll
        for (int h = 0; h < HW; ++h) d[h] = valid ? d[h] * sl2 : -INFINITY;
        head_reduce<HW, 16, true>(d, lane);
        if (HW == 32 || (lane & 1) == 0) red[quarter * H + h0 + (HW == 32 ? lane : lane >> 1)] = d[0];
        named_bar_sync(1, NST);
        if (tid < H) {
          const float mo = m_used[tid];
          const float mb = fmaxf(fmaxf(red[tid], red[H + tid]), fmaxf(red[2 * H + tid], red[3 * H + tid]));
          const float mn = fmaxf(mo, mb);
          fac[tid] = (mn == -INFINITY) ? 1.f : ex2(mo - mn);
          m_used[tid] = mn;
        }
        named_bar_sync(1, NST);
        tmem_cols_load<HW>(lane_base + C::TM_S + h0, d);  // and once more for the exponents
#pragma unroll
        for (int h = 0; h < HW; ++h) {
          if constexpr (kMaxRegs) mneg[h] = -m_used[h0 + h];
          lpart[h] *= fac[h0 + h];
          d[h] = fmaf(d[h], sl2, neg_max(h));
        }
        if (u > 0) {  // O^T rows of this thread: dims 128c + key, 16 heads at a time
#pragma unroll 1
          for (int c = 0; c < 4 * (HW / 16); ++c) {
            const int hh = (c % (HW / 16)) * 16;
            const uint32_t col = C::TM_O + (c / (HW / 16)) * H + h0 + hh;
            float o[16];
            tmem_cols_load<16>(lane_base + col, o);
#pragma unroll
            for (int h = 0; h < 16; ++h) o[h] *= fac[h0 + hh + h];
            tmem_cols_store<16>(lane_base + col, o);
          }
          tmem_wait_st();
        }
      }
      if constexpr (C::P_MN) {
        // P[key][h] = bf16(2^d): one 128-byte swizzled row per key (heads
        // contiguous), written as 16-byte vectors of eight heads
        uint8_t* prow = sm + C::OFF_P + key * 128;
#pragma unroll
        for (int q = 0; q < HW / 8; ++q) {
          uint32_t wv[4];
#pragma unroll
          for (int k2 = 0; k2 < 4; ++k2) {
            const int h = q * 8 + k2 * 2;
            const float p0 = valid ? ex2(d[h]) : 0.f;
            const float p1 = valid ? ex2(d[h + 1]) : 0.f;
            lpart[h] += p0;
            lpart[h + 1] += p1;
            __nv_bfloat162 b2 = __floats2bfloat162_rn(p0, p1);
            wv[k2] = *reinterpret_cast<uint32_t*>(&b2);
          }
          const int chunk = ((h0 >> 3) + q) ^ (key & 7);
          *reinterpret_cast<uint4*>(prow + (chunk << 4)) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
        }
      } else {
        // P^T[h][key]: K-major rows of 64 keys per head (H = 16)
        uint8_t* pbase = sm + C::OFF_P + (key >> 6) * C::PSUB;
        const int kb = (key & 63) * 2;
#pragma unroll
        for (int h = 0; h < HW; ++h) {
          const int hg = h0 + h;
          const float pv = valid ? ex2(d[h]) : 0.f;
          lpart[h] += pv;
          const int off = hg * 128 + ((((kb >> 4) ^ (hg & 7)) << 4) | (kb & 15));
          *reinterpret_cast<__nv_bfloat16*>(pbase + off) = __float2bfloat16_rn(pv);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar(B_P));
      if (more) {
        // refill for block j+1: chunk c of P.V frees sub-tiles 2c, 2c+1 (the
        // last one also the RoPE sub-tile holding P)
        resolve_rows();
        bool alive = true;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          const bool freed = mbar_wait(bar(B_CFREE + c), u & 1, abort_flag, p.status, to);
          if (!(KV8 ? __all_sync(0xffffffffu, freed) : freed)) {
            alive = false;
            break;
          }
          if constexpr (KV8) {
            issue8(c);
            if (c > 0) convert8(c - 1, 1);
          } else {
            issue(2 * c);
            issue(2 * c + 1);
            if (c == 3) issue(8);
            signal(c);
          }
        }
        if (!alive) break;
        if constexpr (KV8) convert8(3, 0);
        if (j + 2 < j1) prefetch_rows();
      }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    // row sums over the 128 keys
    head_reduce<HW, 16, false>(lpart, lane);
    if (HW == 32 || (lane & 1) == 0) red[quarter * H + h0 + (HW == 32 ? lane : lane >> 1)] = lpart[0];
    named_bar_sync(1, NST);
    if (tid < H) lsum[tid] = (red[tid] + red[H + tid]) + (red[2 * H + tid] + red[3 * H + tid]);
    // the unnormalised O^T of this CTA as [h][512]: staged in shared memory,
    // or for a token split over 4 to 16 CTAs written with the running maxima
    // and the row sums to the token's partial results in global memory
    // (zeros for a CTA without blocks), which the cluster combines through L2
    const bool have = j1 > j0 && mbar_wait(bar(B_O), 0, abort_flag, p.status, to);
    tc_fence_after();
    float* Od = kMergeL2 ? p.part + (static_cast<int64_t>(t) * NSPLIT + rank) * (H * 512 + 2 * H)
                         : reinterpret_cast<float*>(sm + C::OFF_C);
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
      float o[HW];
      if (have) {
        tmem_cols_load<HW>(lane_base + C::TM_O + c * H + h0, o);
      } else {
#pragma unroll
        for (int h = 0; h < HW; ++h) o[h] = 0.f;
      }
#pragma unroll
      for (int h = 0; h < HW; ++h) Od[(h0 + h) * 512 + c * 128 + key] = o[h];
    }
    if (kMergeL2 && tid < H) {
      Od[H * 512 + tid] = m_used[tid];
      Od[H * 512 + H + tid] = lsum[tid];
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == W_PV) {
    tc_fence_after();
    tmem_dealloc(tbase, C::TMEM_COLS);
  }

  // ---- combine the NSPLIT partial results and write bf16 out (+ lse)
  float* Os = reinterpret_cast<float*>(sm + C::OFF_C);
  if constexpr (NSPLIT > 1) {
    // every rank's partial results are complete before any is read: in
    // global memory (L2, read at L2: the other SMs' writes are not in this
    // L1), or in each rank's shared memory (read through the cluster)
    if (kMergeL2) __threadfence();
    cluster_sync();
    const float* part_t = p.part + static_cast<int64_t>(t) * NSPLIT * (H * 512 + 2 * H);
    auto part4 = [&](int r, int h, int d) -> float4 {
      if constexpr (kMergeL2)
        return __ldcg(reinterpret_cast<const float4*>(part_t + r * (H * 512 + 2 * H) + h * 512 + d));
      else
        return ld_dsmem_f4(mapa_shared(smem_u32(&Os[h * 512 + d]), r));
    };
    if (tid < H) {
      float mr[NSPLIT], lr[NSPLIT];
      float M = -INFINITY;
#pragma unroll
      for (int r = 0; r < NSPLIT; ++r) {
        if constexpr (kMergeL2) {
          const float* pr = part_t + r * (H * 512 + 2 * H) + H * 512;
          mr[r] = __ldcg(pr + tid);
          lr[r] = __ldcg(pr + H + tid);
        } else {
          mr[r] = __uint_as_float(ld_dsmem_u32(mapa_shared(smem_u32(&m_used[tid]), r)));
          lr[r] = __uint_as_float(ld_dsmem_u32(mapa_shared(smem_u32(&lsum[tid]), r)));
        }
        M = fmaxf(M, mr[r]);
      }
      float L = 0.f;
#pragma unroll
      for (int r = 0; r < NSPLIT; ++r) L += (mr[r] == -INFINITY) ? 0.f : lr[r] * ex2(mr[r] - M);
#pragma unroll
      for (int r = 0; r < NSPLIT; ++r)
        fac[r * H + tid] = (L > 0.f && mr[r] != -INFINITY) ? ex2(mr[r] - M) / L : 0.f;
      if (rank == 0 && p.lse)
        p.lse[static_cast<int64_t>(t) * H + tid] = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
    }
    __syncthreads();
    // this rank's DS dims of every head: each thread takes U float4 outputs
    // per pass and requests all their U * NSPLIT vectors before summing any
    constexpr int DS = 512 / NSPLIT, ITEMS = H * DS / 4, U = 16 / NSPLIT;
    for (int i0 = tid; i0 < ITEMS; i0 += U * NT) {
      float4 v[U][NSPLIT];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i = i0 + u * NT;
        if (i < ITEMS) {
          const int h = i / (DS / 4), d = rank * DS + (i % (DS / 4)) * 4;
#pragma unroll
          for (int r = 0; r < NSPLIT; ++r) v[u][r] = part4(r, h, d);
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i = i0 + u * NT;
        if (i >= ITEMS) break;
        const int h = i / (DS / 4), d = rank * DS + (i % (DS / 4)) * 4;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int r = 0; r < NSPLIT; ++r) {
          const float f = fac[r * H + h];
          acc.x = fmaf(f, v[u][r].x, acc.x);
          acc.y = fmaf(f, v[u][r].y, acc.y);
          acc.z = fmaf(f, v[u][r].z, acc.z);
          acc.w = fmaf(f, v[u][r].w, acc.w);
        }
        __nv_bfloat162 lo2 = __floats2bfloat162_rn(acc.x, acc.y);
        __nv_bfloat162 hi2 = __floats2bfloat162_rn(acc.z, acc.w);
        uint2 pk;
        pk.x = *reinterpret_cast<uint32_t*>(&lo2);
        pk.y = *reinterpret_cast<uint32_t*>(&hi2);
        *reinterpret_cast<uint2*>(p.out + (static_cast<int64_t>(t) * H + h) * 512 + d) = pk;
      }
    }
    if (!kMergeL2) cluster_sync();  // this CTA's shared memory stays until every rank has read it
  } else {
    if (tid < H) {
      const float L = lsum[tid];
      fac[tid] = L > 0.f ? 1.f / L : 0.f;
      if (p.lse)
        p.lse[static_cast<int64_t>(t) * H + tid] =
            L > 0.f ? (m_used[tid] + log2f(L)) * kLn2 : -INFINITY;
    }
    __syncthreads();
    for (int i = tid; i < H * 128; i += NT) {
      const int h = i >> 7, d = (i & 127) * 4;
      const float f = fac[h];
      const float4 v = *reinterpret_cast<const float4*>(&Os[h * 512 + d]);
      __nv_bfloat162 lo2 = __floats2bfloat162_rn(v.x * f, v.y * f);
      __nv_bfloat162 hi2 = __floats2bfloat162_rn(v.z * f, v.w * f);
      uint2 pk;
      pk.x = *reinterpret_cast<uint32_t*>(&lo2);
      pk.y = *reinterpret_cast<uint32_t*>(&hi2);
      *reinterpret_cast<uint2*>(p.out + (static_cast<int64_t>(t) * H + h) * 512 + d) = pk;
    }
  }
}

// ---------------------------------------------------------------------------
// Prefill-sized launches (many tokens, 64 heads, bf16 rows of contiguous or
// paged caches that L2 holds, one CTA per token): a persistent grid, one CTA
// per SM, each walking a list of tokens.  A CTA per token pays, besides its blocks,
// about 9.5 us of start-up and tail on GB300 (barrier and TMEM set-up,
// metadata, the query and first gather, the pipeline fill, the output
// written after the last product): about a sixth of an 8K prefill's
// attention.  Here the next token's first block is gathered in the refill
// slot of the current token's last block, its query is loaded by TMA as soon
// as the current token's last QK product is done, and the current token's
// output goes from TMEM straight to global memory (the C tile already holds
// the next token's rows) while that token's first QK product runs.  The next
// token's first P.V product, which overwrites O^T, waits for that token's
// P, which the softmax warps give only after reading the previous O^T.
// Per block the work is that of the kernel above, operation for operation,
// so both give bit-identical results.
constexpr int kMlaPersistMaxTokens = 256;  // tokens per CTA (one per softmax thread)

template <int H, bool PAGED>
__global__ void __launch_bounds__(MlaCfg<H>::NT + 64, 1)
    sparse_mla_persistent_kernel(const __grid_constant__ CUtensorMap qlat_map,
                                 const __grid_constant__ CUtensorMap qrope_map, const MlaParams p) {
  using C = MlaCfg<H>;
  static_assert(H == 64, "the persistent variant covers the 64-head model");
  constexpr int HW = C::HW, NSW = C::NSW, NST = NSW * 32;
  constexpr int W_QK = NSW, W_PV = NSW + 1;
  constexpr int GROW = NST / 8, RPT = 128 / GROW;
  static_assert(NST == kMlaPersistMaxTokens, "one list entry per softmax thread");
  // the token list {t, pos, first cache row (lo, hi)} -- {t, pos, sequence, 0}
  // for paged caches -- reuses the block-table and FP8-scale areas, which
  // this variant does not use (it reads a paged cache's block table through
  // L1)
  static_assert(C::OFF_KSC + 128 * 16 - C::OFF_TAB >= kMlaPersistMaxTokens * 16, "token list");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t sQ = smem_u32(sm + C::OFF_Q);
  const uint32_t sC = smem_u32(sm + C::OFF_C);
  float* m_used = reinterpret_cast<float*>(sm + C::OFF_SCR);
  float* red = m_used + H;
  float* fac = red + 4 * H + H;
  int* flags = reinterpret_cast<int*>(sm + C::OFF_FLAGS);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::OFF_BAR);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + C::OFF_MISC);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + C::OFF_MISC + 8);
  int* wcnt = reinterpret_cast<int*>(sm + C::OFF_MISC + 16);  // list entries per softmax warp
  int4* toks = reinterpret_cast<int4*>(sm + C::OFF_TAB);
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  const int B_Q = 0, B_CFULL = 1, B_CFREE = 5, B_S = 9, B_P = 10, B_O = 11, B_QD = 12;

  if (tid == 0) {
    *abort_flag = 0;
    mbar_init(bar(B_Q), 1);
    for (int i = 0; i < 4; ++i) mbar_init(bar(B_CFULL + i), NST);
    for (int i = 0; i < 4; ++i) mbar_init(bar(B_CFREE + i), 1);
    mbar_init(bar(B_S), 1);
    mbar_init(bar(B_P), NST);
    mbar_init(bar(B_O), 1);
    mbar_init(bar(B_QD), 1);
    fence_mbar_init();
  }
  if (tid < H) m_used[tid] = -INFINITY;
  if (warp == W_PV) {
    tmem_alloc(smem_u32(tslot), C::TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == W_QK && lane == 0) {
    tma_prefetch_desc(&qlat_map);
    tma_prefetch_desc(&qrope_map);
  }
  chain_wait();     // the previous kernel of the stream has completed
  chain_release();  // the next one may be scheduled

  // ---- this CTA's tokens, heaviest first: the work items are dealt out in
  // rounds of gridDim.x, to the CTAs in order in even rounds and in reverse
  // order in odd ones, which evens out the falling weights (8K causal
  // prefill: the most loaded CTA 0.1 % above the average, against 1 % when
  // every round is dealt in order).
  // Item w is the (w / num_seqs)-th latest query of sequence w % num_seqs;
  // items past a sequence's end are skipped, a query at an invalid position
  // gets a zero output and lse = -inf (and DSA_DEVERR_BATCH).
  if (tid < NST) {
    bool mine = false;
    int4 tk = make_int4(0, 0, 0, 0);
    const int64_t w = static_cast<int64_t>(tid) * gridDim.x +
                      ((tid & 1) ? gridDim.x - 1 - blockIdx.x : blockIdx.x);
    if (w < static_cast<int64_t>(p.b.max_q) * p.b.num_seqs) {
      const int seq = static_cast<int>(w % p.b.num_seqs);
      const int qi = p.b.max_q - 1 - static_cast<int>(w / p.b.num_seqs);
      const int qs = p.b.q_start[seq], qe = p.b.q_start[seq + 1];
      if (qs < 0 || qe < qs || qe > p.b.num_q) {
        atomicOr(p.status, DSA_DEVERR_BATCH);
      } else if (qs + qi < qe) {
        const int t = qs + qi;
        const int pos = query_pos(p.b, t, p.status);
        if (pos >= 0) {
          const int64_t r0 = PAGED ? seq : seq_base_row(p.b, seq);
          mine = true;
          tk = make_int4(t, pos, static_cast<int>(static_cast<uint32_t>(r0)),
                         static_cast<int>(static_cast<uint64_t>(r0) >> 32));
        } else {
          uint4* o = reinterpret_cast<uint4*>(p.out + static_cast<int64_t>(t) * H * 512);
          for (int i = 0; i < H * 512 / 8; ++i) o[i] = make_uint4(0, 0, 0, 0);
          if (p.lse)
            for (int h = 0; h < H; ++h) p.lse[static_cast<int64_t>(t) * H + h] = -INFINITY;
        }
      }
    }
    const unsigned bal = __ballot_sync(0xffffffffu, mine);
    if (lane == 0) wcnt[warp] = __popc(bal);
    named_bar_sync(1, NST);
    int off = 0;
    for (int w2 = 0; w2 < warp; ++w2) off += wcnt[w2];
    if (mine) toks[off + __popc(bal & ((1u << lane) - 1u))] = tk;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  int ntok = 0;
#pragma unroll
  for (int w2 = 0; w2 < NSW; ++w2) ntok += wcnt[w2];
  const uint32_t tbase = *tslot;
  const uint64_t to = p.timeout_ns;
  volatile int no_abort = 0;
  auto tok_nb = [&](const int4& tk) { return (min(p.K, tk.y + 1) + 127) / 128; };

  // Register split: the QK and P.V issuer warps and two idle ones form the
  // third warpgroup and give up registers to the eight softmax warps.  At
  // launch every thread has 168 (three warps share a sub-partition's 16K);
  // 128 x 88 + 256 x 208 = 384 x 168, so the increase always completes.
  // Each branch runs under its own limit up to the common tail.
  if (warp >= NSW) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 88;" ::: "memory");
    if (warp == W_QK) {
      // ------------------------------------------------ QK issuer, and the query of each token
      if (lane == 0) {
        constexpr uint32_t id_qk = idesc_bf16(128, H, false, false);
        const uint64_t dc = sdesc_sw128(sC, 0, 1024), dq = sdesc_sw128(sQ, 0, 1024);
        const uint32_t d_s = tbase + C::TM_S;
        bool ok = true;
        uint32_t gu = 0;   // blocks of this CTA so far (barrier phases)
        int nqd = 0, nq = 0;  // commits to B_QD, query loads issued
        for (int i = 0; ok && i < ntok; ++i) {
          const int4 tk = toks[i];
          const int nb = tok_nb(tk);
          if (i > 0) {  // the previous token's products have read the query tile
            umma_commit(bar(B_QD));
            ok = mbar_wait(bar(B_QD), nqd & 1, abort_flag, p.status, to);
            ++nqd;
            if (!ok) break;
          }
          mbar_arrive_expect_tx(bar(B_Q), C::Q_BYTES);
          for (int c = 0; c < 8; ++c) tma_load_2d(sQ + c * C::QSUB, &qlat_map, 64 * c, tk.x * H, bar(B_Q));
          tma_load_2d(sQ + 8 * C::QSUB, &qrope_map, 0, tk.x * H, bar(B_Q));
          if (i + 1 < ntok) {  // the next token's query into L2 (read from HBM it takes ~2.5 us)
            const int tn = toks[i + 1].x;
            for (int c = 0; c < 8; ++c) tma_prefetch_l2_2d(&qlat_map, 64 * c, tn * H);
            tma_prefetch_l2_2d(&qrope_map, 0, tn * H);
          }
          ok = mbar_wait(bar(B_Q), nq & 1, abort_flag, p.status, to);
          ++nq;
          for (int j = 0; ok && j < nb; ++j, ++gu) {
  #pragma unroll
            for (int g = 0; g < 4; ++g) {
              ok = mbar_wait(bar(B_CFULL + g), gu & 1, abort_flag, p.status, to);
              if (!ok) break;
              fence_proxy_async_smem();  // cp.async (generic proxy) writes -> tcgen05.mma reads
              tc_fence_after();
              if (g == 0)
                issue_qk_group<0, C>(d_s, dc, dq, id_qk);
              else if (g == 1)
                issue_qk_group<1, C>(d_s, dc, dq, id_qk);
              else if (g == 2)
                issue_qk_group<2, C>(d_s, dc, dq, id_qk);
              else
                issue_qk_group<3, C>(d_s, dc, dq, id_qk);
            }
            if (!ok) break;
            umma_commit(bar(B_S));
          }
        }
        umma_commit(bar(B_QD));  // drain this warp's products before exit
        mbar_wait(bar(B_QD), nqd & 1, &no_abort, nullptr, to);
        if (nq > 0) mbar_wait(bar(B_Q), (nq - 1) & 1, &no_abort, nullptr, to);  // the last copy landed
      }
      __syncwarp();
    } else if (warp == W_PV) {
      // ------------------------------------------------ P.V issuer: O^T (+)= C^T . P per block
      if (lane == 0) {
        constexpr uint32_t id_pv = idesc_bf16(128, H, true, C::P_MN);
        static_assert(C::P_MN, "the persistent grid keeps P MN-major");
        const uint64_t dcv = sdesc_sw128(sC, C::CSUB, 1024);
        const uint64_t dp = sdesc_sw128(smem_u32(sm + C::OFF_P), 8192, 1024);
        const uint32_t d_o = tbase + C::TM_O;
        bool ok = true;
        uint32_t gu = 0;
        int no = 0;  // commits to B_O (one per token)
        for (int i = 0; ok && i < ntok; ++i) {
          const int nb = tok_nb(toks[i]);
          // the first product of a token overwrites O^T: its P arrives only
          // after the softmax warps have read the previous token's O^T
          for (int u = 0; u < nb; ++u, ++gu) {
            ok = mbar_wait(bar(B_P), gu & 1, abort_flag, p.status, to);
            if (!ok) break;
            tc_fence_after();
            issue_pv_chunk<0, C>(d_o, dcv, dp, id_pv, u == 0);
            umma_commit(bar(B_CFREE + 0));
            issue_pv_chunk<1, C>(d_o + H, dcv, dp, id_pv, u == 0);
            umma_commit(bar(B_CFREE + 1));
            issue_pv_chunk<2, C>(d_o + 2 * H, dcv, dp, id_pv, u == 0);
            umma_commit(bar(B_CFREE + 2));
            issue_pv_chunk<3, C>(d_o + 3 * H, dcv, dp, id_pv, u == 0);
            umma_commit(bar(B_CFREE + 3));
          }
          if (!ok) break;
          umma_commit(bar(B_O));
          ++no;
        }
        // drain: the last token's commit, or one more when none completed
        // (after an abort nothing waits for B_O's phases any more)
        if (no == 0 || !ok) {
          umma_commit(bar(B_O));
          ++no;
        }
        mbar_wait(bar(B_O), (no - 1) & 1, &no_abort, nullptr, to);
      }
      __syncwarp();
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 208;" ::: "memory");
    // ------------------------------------------------ softmax / gather / output warps
    const int quarter = warp & 3;
    const int h0 = (warp >> 2) * HW;
    const int key = quarter * 32 + lane;
    const uint32_t lane_base = tbase + (static_cast<uint32_t>(quarter * 32) << 16);
    const float sl2 = p.scale_log2;
    float lpart[HW];  // this thread's share of the softmax denominators
    // (the running maxima are read from shared memory where they are used:
    // registers for them made this kernel spill)
    const int kch = tid & 7, rb = tid >> 3;
    const uint32_t gdst0 = sC + rb * 128 + ((kch ^ (rb & 7)) << 4);
    const uint16_t* kvk = p.kv + kch * 8;
    // cache row of position e >= 0 of a listed token's sequence, -1 if unmapped
    const int bps = p.b.blocks_per_seq;
    const int rshift = PAGED ? __ffs(p.b.block_rows) - 1 : 0;  // block_rows is a power of two
    auto row_of = [&](const int4& tk, int e) -> int64_t {
      if constexpr (!PAGED) {
        return static_cast<int64_t>((static_cast<uint64_t>(static_cast<uint32_t>(tk.w)) << 32) |
                                    static_cast<uint32_t>(tk.z)) + e;
      } else {
        const int blk = e >> rshift;
        if (blk >= bps) return -1;
        const int32_t id = ld_keep_i32(p.b.block_table + static_cast<int64_t>(tk.z) * bps + blk);
        return id < 0 ? -1 : (static_cast<int64_t>(id) << rshift) + (e & (p.b.block_rows - 1));
      }
    };
    int gsel[RPT];
    auto fetch_sel = [&](const int32_t* irow, int nv, int jj) {
#pragma unroll
      for (int c = 0; c < RPT; ++c) {
        const int sl = jj * 128 + rb + GROW * c;
        gsel[c] = sl < nv ? ld_stream_i32(irow + sl) : -1;
      }
    };
    int grow[RPT];
    auto resolve_rows = [&](const int4& gtk) {
#pragma unroll
      for (int c = 0; c < RPT; ++c) {
        const int e = gsel[c];
        const int64_t rr = e >= 0 ? row_of(gtk, e) : -1;
        const bool ok = e >= 0 && e <= gtk.y && rr >= 0 && rr < p.kv_rows;
        if (!ok && e != -1 && kch == 0) atomicOr(p.status, DSA_DEVERR_INDEX);
        grow[c] = ok ? static_cast<int>(rr) : 0;
      }
    };
    auto issue = [&](int i) {
      const uint32_t dst = gdst0 + i * C::CSUB;
#pragma unroll
      for (int c = 0; c < RPT; ++c)
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst + c * GROW * 128),
                     "l"(kvk + static_cast<int64_t>(grow[c]) * 576 + 64 * i)
                     : "memory");
    };
    auto signal = [&](int g) {
      asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar(B_CFULL + g))
                   : "memory");
    };
    uint32_t gu = 0;  // blocks of this CTA so far (barrier phases)
    int e_next = -1;  // this thread's key in the next block
    if (ntok > 0) {   // the first token's first block
      const int4 tk = toks[0];
      const int nv = min(p.K, tk.y + 1);
      const int32_t* irow = p.idx + static_cast<int64_t>(tk.x) * p.K;
      fetch_sel(irow, nv, 0);
      resolve_rows(tk);
#pragma unroll 1
      for (int g = 0; g < 4; ++g) {
        issue(2 * g);
        issue(2 * g + 1);
        if (g == 3) issue(8);
        signal(g);
      }
      e_next = key < nv ? ld_stream_i32(irow + key) : -1;
    }
    bool alive = true;
#pragma unroll 1
    for (int i = 0; alive && i < ntok; ++i) {
      const int4 tk = toks[i];  // (its token index is read again where it is used)
      const int pos = tk.y;
      const int nvalid = min(p.K, pos + 1), nb = (nvalid + 127) / 128;
      const bool has_next = i + 1 < ntok;  // the next token's entry is read where it is used
#pragma unroll
      for (int h = 0; h < HW; ++h) lpart[h] = 0.f;
#pragma unroll 1
      for (int j = 0; j < nb; ++j, ++gu) {
        const int u = j;
        const bool more = j + 1 < nb;
        const int e = e_next;
        if (more) {
          const int32_t* idx_row = p.idx + static_cast<int64_t>(toks[i].x) * p.K;
          const int sn = (j + 1) * 128 + key;
          e_next = sn < nvalid ? ld_stream_i32(idx_row + sn) : -1;
          fetch_sel(idx_row, nvalid, j + 1);
        } else if (has_next) {  // the next token's first block
          const int4 tn = toks[i + 1];
          const int nvalid_n = min(p.K, tn.y + 1);
          const int32_t* idx_row_n = p.idx + static_cast<int64_t>(tn.x) * p.K;
          e_next = key < nvalid_n ? ld_stream_i32(idx_row_n + key) : -1;
          fetch_sel(idx_row_n, nvalid_n, 0);
        }
        // this thread's key (a mapped row of a visible position?) and, for a
        // paged cache, the refill's rows: their block-table lookups come
        // before the wait, which hides their latency
        bool valid = e >= 0 && e <= pos;
        if (valid) {
          const int64_t rr = row_of(tk, e);
          valid = rr >= 0 && rr < p.kv_rows;
        }
        if constexpr (PAGED) {
          if (more)
            resolve_rows(tk);
          else if (has_next)
            resolve_rows(toks[i + 1]);
        }
        if (!mbar_wait(bar(B_S), gu & 1, abort_flag, p.status, to)) {
          alive = false;
          break;
        }
        tc_fence_after();
        float d[HW];
        tmem_cols_load<HW>(lane_base + C::TM_S + h0, d);
        // the first block sets the running maximum; a later one raises it only
        // when one of its scores exceeds it by more than the threshold
        int resc = 1;
        if (u > 0) {
          float dmax = -INFINITY;
#pragma unroll
          for (int h = 0; h < HW; ++h) {
            d[h] = fmaf(d[h], sl2, -m_used[h0 + h]);
            dmax = fmaxf(dmax, d[h]);
          }
          const bool exceed = valid && dmax > kRescaleThreshold;
          const unsigned any = __any_sync(0xffffffffu, exceed);
          if (lane == 0) flags[warp] = any ? 1 : 0;
          named_bar_sync(1, NST);
          resc = 0;
#pragma unroll
          for (int w = 0; w < NSW; ++w) resc |= flags[w];
          if (resc) tmem_cols_load<HW>(lane_base + C::TM_S + h0, d);  // raw scores again
        }
        if (resc) {
#pragma unroll
          for (int h = 0; h < HW; ++h) d[h] = valid ? d[h] * sl2 : -INFINITY;
          head_reduce<HW, 16, true>(d, lane);
          red[quarter * H + h0 + lane] = d[0];
          named_bar_sync(1, NST);
          if (tid < H) {
            const float mo = m_used[tid];
            const float mb = fmaxf(fmaxf(red[tid], red[H + tid]), fmaxf(red[2 * H + tid], red[3 * H + tid]));
            const float mn = fmaxf(mo, mb);
            fac[tid] = (mn == -INFINITY) ? 1.f : ex2(mo - mn);
            m_used[tid] = mn;
          }
          named_bar_sync(1, NST);
          tmem_cols_load<HW>(lane_base + C::TM_S + h0, d);
#pragma unroll
          for (int h = 0; h < HW; ++h) {
            lpart[h] *= fac[h0 + h];
            d[h] = fmaf(d[h], sl2, -m_used[h0 + h]);
          }
          if (u > 0) {
#pragma unroll 1
            for (int c = 0; c < 4 * (HW / 16); ++c) {
              const int hh = (c % (HW / 16)) * 16;
              const uint32_t col = C::TM_O + (c / (HW / 16)) * H + h0 + hh;
              float o[16];
              tmem_cols_load<16>(lane_base + col, o);
#pragma unroll
              for (int h = 0; h < 16; ++h) o[h] *= fac[h0 + hh + h];
              tmem_cols_store<16>(lane_base + col, o);
            }
            tmem_wait_st();
          }
        }
        {  // P[key][h] = bf16(2^d), one 128-byte swizzled row per key
          uint8_t* prow = sm + C::OFF_P + key * 128;
#pragma unroll
          for (int q = 0; q < HW / 8; ++q) {
            uint32_t wv[4];
#pragma unroll
            for (int k2 = 0; k2 < 4; ++k2) {
              const int h = q * 8 + k2 * 2;
              const float p0 = valid ? ex2(d[h]) : 0.f;
              const float p1 = valid ? ex2(d[h + 1]) : 0.f;
              lpart[h] += p0;
              lpart[h + 1] += p1;
              __nv_bfloat162 b2 = __floats2bfloat162_rn(p0, p1);
              wv[k2] = *reinterpret_cast<uint32_t*>(&b2);
            }
            const int chunk = ((h0 >> 3) + q) ^ (key & 7);
            *reinterpret_cast<uint4*>(prow + (chunk << 4)) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(bar(B_P));
        if (more || has_next) {
          // refill: block j+1, or the next token's first block
          if constexpr (!PAGED) {
            if (more)
              resolve_rows(tk);
            else
              resolve_rows(toks[i + 1]);
          }
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            if (!mbar_wait(bar(B_CFREE + c), gu & 1, abort_flag, p.status, to)) {
              alive = false;
              break;
            }
            issue(2 * c);
            issue(2 * c + 1);
            if (c == 3) issue(8);
            signal(c);
          }
          if (!alive) break;
        }
      }
      if (!alive) break;
      // ---- the token's output: row sums, then O^T / L from TMEM to global memory
      head_reduce<HW, 16, false>(lpart, lane);
      red[quarter * H + h0 + lane] = lpart[0];
      named_bar_sync(1, NST);
      if (tid < H) {
        const float L = (red[tid] + red[H + tid]) + (red[2 * H + tid] + red[3 * H + tid]);
        fac[tid] = L > 0.f ? 1.f / L : 0.f;
        if (p.lse)
          p.lse[static_cast<int64_t>(toks[i].x) * H + tid] = L > 0.f ? (m_used[tid] + log2f(L)) * kLn2 : -INFINITY;
        m_used[tid] = -INFINITY;  // the next token's running maximum
      }
      named_bar_sync(1, NST);
      if (!mbar_wait(bar(B_O), i & 1, abort_flag, p.status, to)) {
        alive = false;
        break;
      }
      tc_fence_after();
      // dims 128c + key of this thread's 32 heads: lanes 2m and 2m+1 swap one
      // value of each head pair, so that each writes one head's two dims
      const bool odd = lane & 1;
      uint16_t* orow = p.out + static_cast<int64_t>(toks[i].x) * H * 512 + (key & ~1);
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        float o[HW];
        tmem_cols_load<HW>(lane_base + C::TM_O + c * H + h0, o);
#pragma unroll
        for (int hp = 0; hp < HW / 2; ++hp) {
          const float mine = odd ? o[2 * hp + 1] : o[2 * hp];
          const float other = __shfl_xor_sync(0xffffffffu, odd ? o[2 * hp] : o[2 * hp + 1], 1);
          const int h = h0 + 2 * hp + (odd ? 1 : 0);
          const float f = fac[h];
          const __nv_bfloat162 b2 = odd ? __floats2bfloat162_rn(other * f, mine * f)
                                        : __floats2bfloat162_rn(mine * f, other * f);
          *reinterpret_cast<uint32_t*>(orow + h * 512 + c * 128) = *reinterpret_cast<const uint32_t*>(&b2);
        }
      }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  if (warp == W_PV) {
    tc_fence_after();
    tmem_dealloc(tbase, C::TMEM_COLS);
  }
}

template <int H, int NSPLIT, bool PAGED, bool KV8>
cudaError_t launch_mla(const CUtensorMap& ql, const CUtensorMap& qr, const MlaParams& p,
                       cudaStream_t stream) {
  using C = MlaCfg<H>;
  auto* kern = sparse_mla_kernel<H, NSPLIT, PAGED, KV8>;
  static int configured_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device != dev) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e == cudaSuccess && NSPLIT > 8)  // 16 CTAs per cluster: beyond the portable size
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  const dim3 grid(static_cast<unsigned>(p.b.max_q) * NSPLIT, static_cast<unsigned>(p.b.num_seqs));
  prof_begin(stream);
  cudaError_t e = launch_chained(kern, grid, dim3(C::NT), C::SMEM, stream, NSPLIT, ql, qr, p);
  prof_end(kLaunchMla, stream);
  count_launch(kLaunchMla);
  return e;
}

template <int H, bool PAGED>
cudaError_t launch_mla_persistent(const CUtensorMap& ql, const CUtensorMap& qr, const MlaParams& p,
                                  int grid, cudaStream_t stream) {
  using C = MlaCfg<H>;
  auto* kern = sparse_mla_persistent_kernel<H, PAGED>;
  static int configured_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device != dev) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  prof_begin(stream);
  // the softmax warps, the QK and P.V issuers and two idle warps (the issuers' warpgroup)
  cudaError_t e = launch_chained(kern, dim3(static_cast<unsigned>(grid)), dim3(C::NT + 64), C::SMEM,
                                 stream, 1, ql, qr, p);
  prof_end(kLaunchMla, stream);
  count_launch(kLaunchMla);
  return e;
}

int g_mla_persistent = 1;

template <int H, bool KV8>
cudaError_t launch_h(const CUtensorMap& ql, const CUtensorMap& qr, const MlaParams& p, int nsplit,
                     bool paged, cudaStream_t stream) {
  switch (nsplit) {
    case 1: return paged ? launch_mla<H, 1, true, KV8>(ql, qr, p, stream)
                         : launch_mla<H, 1, false, KV8>(ql, qr, p, stream);
    case 2: return paged ? launch_mla<H, 2, true, KV8>(ql, qr, p, stream)
                         : launch_mla<H, 2, false, KV8>(ql, qr, p, stream);
    case 4: return paged ? launch_mla<H, 4, true, KV8>(ql, qr, p, stream)
                         : launch_mla<H, 4, false, KV8>(ql, qr, p, stream);
    case 8: return paged ? launch_mla<H, 8, true, KV8>(ql, qr, p, stream)
                         : launch_mla<H, 8, false, KV8>(ql, qr, p, stream);
    default: return paged ? launch_mla<H, 16, true, KV8>(ql, qr, p, stream)
                          : launch_mla<H, 16, false, KV8>(ql, qr, p, stream);
  }
}

}  // namespace

void set_mla_persistent(bool on) { g_mla_persistent = on ? 1 : 0; }

// CTAs per token (one cluster): a token's key blocks are split over several
// CTAs when there are too few tokens to cover the SMs (decode).
int mla_nsplit(const dsa_batch_t& b, int k) {
  const int nblk = (k + 127) / 128;
  int nsplit = 1;
  while (nsplit < 8 && nsplit * 2 <= nblk && static_cast<int64_t>(b.num_q) * nsplit * 2 <= 152)
    nsplit *= 2;
  // 16 CTAs per token while the launch is at most four such clusters, all
  // resident at once (measured, K = 2048: 4 tokens 23.0 -> 21.2 us per layer;
  // 8 tokens' eight 16-CTA clusters did not fit together: 24.7 -> 37.0 us)
  if (nsplit == 8 && 16 <= nblk && static_cast<int64_t>(b.num_q) * 16 <= 64) nsplit = 16;
  return nsplit;
}

// The partial results of tokens split over 4 to 16 CTAs (pairs combine
// through distributed shared memory).
size_t mla_workspace_bytes(const dsa_batch_t& b, int heads, int k) {
  const int nsplit = mla_nsplit(b, k);
  if (nsplit < 4) return 0;
  return static_cast<size_t>(b.num_q) * nsplit * (static_cast<size_t>(heads) * 512 + 2 * heads) * 4;
}

cudaError_t launch_sparse_mla(const void* q_lat, const void* q_rope, const void* kv,
                              int64_t kv_rows, const int32_t* idx, int k, int heads, float scale,
                              const dsa_batch_t& b, void* out, float* lse, void* ws, size_t ws_bytes,
                              int* status, cudaStream_t stream, bool kv_fp8, bool direct_rows,
                              bool after_own_kernel, bool after_attention) {
  if (b.num_q == 0) return cudaSuccess;
  CUtensorMap ql, qr;
  const uint64_t qrows = static_cast<uint64_t>(b.num_q) * heads;
  if (!make_tmap_2d(&ql, q_lat, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 512, qrows, 64, heads) ||
      !make_tmap_2d(&qr, q_rope, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 64, qrows, 64, heads))
    return cudaErrorInvalidValue;
  MlaParams p{};
  p.b = to_args(b);
  p.kv = kv_fp8 ? nullptr : static_cast<const uint16_t*>(kv);
  p.kv8 = kv_fp8 ? static_cast<const uint8_t*>(kv) : nullptr;
  p.kv_rows = kv_rows;
  p.direct = direct_rows ? 1 : 0;
  // A cache that L2 holds (short prefills) is read from L2 anyway; larger ones
  // (decode, long prefixes) get the next rows prefetched from HBM.
  p.l2_prefetch = kv_rows * (kv_fp8 ? 656 : 1152) > (int64_t(96) << 20) ? 1 : 0;
  p.idx = idx;
  p.K = k;
  p.scale_log2 = scale * kLog2e;
  p.out = static_cast<uint16_t*>(out);
  p.lse = lse;
  p.status = status;
  p.timeout_ns = wait_timeout_ns();
  p.early_inputs = after_own_kernel ? 1 : 0;
  p.early_gather = after_own_kernel && after_attention && !kv_fp8 ? 1 : 0;
  const int nsplit = mla_nsplit(b, k);
  if (nsplit >= 4) {  // the partial results go through the workspace
    if (!ws || ws_bytes < mla_workspace_bytes(b, heads, k)) return cudaErrorInvalidValue;
    p.part = static_cast<float*>(ws);
  }
  const bool paged = b.block_table != nullptr && !direct_rows;
  // prefill-sized launches of the 64-head model over bf16 rows of caches
  // that L2 holds (contiguous or paged): a persistent grid of one CTA per SM
  // (at most 256 tokens each)
  // (HBM-resident caches keep the CTA-per-token kernel, whose CTAs the
  // hardware hands out as SMs free up: with rows from HBM the time per token
  // varies, and the static token lists measured 4 % slower)
  if (g_mla_persistent && nsplit == 1 && heads == 64 && !kv_fp8 && !direct_rows &&
      !p.l2_prefetch) {
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms > 0 && b.num_q >= 2 * static_cast<int64_t>(sms)) {
      const int64_t items = static_cast<int64_t>(b.max_q) * b.num_seqs;
      const int64_t grid =
          std::max<int64_t>(sms, (items + kMlaPersistMaxTokens - 1) / kMlaPersistMaxTokens);
      return paged ? launch_mla_persistent<64, true>(ql, qr, p, static_cast<int>(grid), stream)
                   : launch_mla_persistent<64, false>(ql, qr, p, static_cast<int>(grid), stream);
    }
  }
  if (kv_fp8) {  // FP8 KV rows: the model's 64 heads only
    if (heads != 64) return cudaErrorNotSupported;
    return launch_h<64, true>(ql, qr, p, nsplit, paged, stream);
  }
  return heads == 16 ? launch_h<16, false>(ql, qr, p, nsplit, paged, stream)
                     : launch_h<64, false>(ql, qr, p, nsplit, paged, stream);
}

}  // namespace dsa

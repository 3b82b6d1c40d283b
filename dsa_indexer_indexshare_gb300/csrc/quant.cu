// FP8 per-block quantiser of the indexer ("GLM-5.2 / 总览" sub-doc index row
// 02: "FP8 per-block + Hadamard"): rotate each 128-vector by the normalised
// Sylvester Hadamard matrix, scale the block by amax / 448 and encode every
// element as E4M3 (round to nearest even, saturating).
//
// One warp per row, four consecutive elements per lane.  The butterfly runs
// in the fixed order h = 1, 2, ..., 64 (pairs (j, j+h) -> (a+b, a-b)); the
// first two stages stay inside a lane, the other five pair lane l with lane
// l ^ (h/4).  Every operation is a single IEEE fp32 add, subtract, multiply
// or divide with explicit round-to-nearest, so the codes are reproducible bit
// for bit by any implementation that performs the same steps.
#include <cuda_fp8.h>

#include "common.cuh"

namespace dsa {
namespace {

__device__ __forceinline__ float bf16_bits_to_float(uint16_t h) {
  return __uint_as_float(static_cast<uint32_t>(h) << 16);
}

// Hadamard rotation + FP8 quantisation of one 128-vector held by a warp
// (lane l: elements 4l .. 4l+3), codes and scale stored at the given row.
__device__ __forceinline__ void hadamard_quant_store(float (&v)[4], int lane, uint8_t* codes_row,
                                                     float* scale_slot) {
  // h = 1: (0,1), (2,3)
  {
    const float a0 = v[0], b0 = v[1], a1 = v[2], b1 = v[3];
    v[0] = __fadd_rn(a0, b0);
    v[1] = __fsub_rn(a0, b0);
    v[2] = __fadd_rn(a1, b1);
    v[3] = __fsub_rn(a1, b1);
  }
  // h = 2: (0,2), (1,3)
  {
    const float a0 = v[0], b0 = v[2], a1 = v[1], b1 = v[3];
    v[0] = __fadd_rn(a0, b0);
    v[2] = __fsub_rn(a0, b0);
    v[1] = __fadd_rn(a1, b1);
    v[3] = __fsub_rn(a1, b1);
  }
  // h = 4 .. 64: partner lane l ^ (h / 4)
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    const bool upper = (lane & m) != 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float y = __shfl_xor_sync(0xffffffffu, v[k], m);
      v[k] = upper ? __fsub_rn(y, v[k]) : __fadd_rn(v[k], y);
    }
  }
  const float inv_sqrt128 = 0.08838834764831845f;
  float amax = 0.f;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    v[k] = __fmul_rn(v[k], inv_sqrt128);
    amax = fmaxf(amax, fabsf(v[k]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float sc = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
  uint32_t packed = 0;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const __nv_fp8_storage_t c = __nv_cvt_float_to_fp8(__fdiv_rn(v[k], sc), __NV_SATFINITE, __NV_E4M3);
    packed |= static_cast<uint32_t>(c) << (8 * k);
  }
  *reinterpret_cast<uint32_t*>(codes_row + lane * 4) = packed;
  if (lane == 0) *scale_slot = sc;
}

__global__ void __launch_bounds__(256) fp8_quant_kernel(const uint16_t* __restrict__ x,
                                                        int64_t rows, uint8_t* __restrict__ codes,
                                                        float* __restrict__ scale) {
  const int lane = threadIdx.x & 31;
  const int64_t r = static_cast<int64_t>(blockIdx.x) * (blockDim.x / 32) + (threadIdx.x >> 5);
  if (r >= rows) return;
  const uint2 raw = *reinterpret_cast<const uint2*>(x + r * 128 + lane * 4);
  float v[4] = {bf16_bits_to_float(raw.x & 0xFFFF), bf16_bits_to_float(raw.x >> 16),
                bf16_bits_to_float(raw.y & 0xFFFF), bf16_bits_to_float(raw.y >> 16)};
  hadamard_quant_store(v, lane, codes + r * 128, scale + r);
}

// fp64 -> bf16 bits, one rounding to nearest (ties to even).  The double is
// first narrowed to fp32 with round-to-odd (toward zero, then the lowest bit
// set when anything was dropped), then the fp32 value is rounded to bf16
// with ties to even; because fp32 keeps 16 more bits than bf16, this double
// rounding equals the single correct rounding (the round-to-odd argument).
__device__ __forceinline__ uint16_t f64_to_bf16_bits(double x) {
  if (x != x) return 0x7FC0;
  const float fz = __double2float_rz(x);
  uint32_t u = __float_as_uint(fz);
  if (static_cast<double>(fz) != x) u |= 1u;  // sticky: inexact narrowing
  if ((u & 0x7F800000u) == 0x7F800000u) return static_cast<uint16_t>(u >> 16);  // +-inf
  u += 0x7FFFu + ((u >> 16) & 1u);
  return static_cast<uint16_t>(u >> 16);
}

struct RopeFreq {
  double f[32];  // theta^(-2i/64), the rotary frequencies of the first 64 dims
};

// sin and cos of an fp64 angle a (|a| < 2^30) in fp64, without a library
// call: a is reduced to r = a - k pi/2, |r| <= pi/4 (a little more when
// a * 2/pi rounds off), quadrant k mod 4, with pi/2 split as P1 + P2, P1
// truncated to 22 significant bits so that k * P1 is exact for |k| < 2^31
// and a - k * P1 is exact (error of r below |k| * 1.1e-23 + 2^-53: at most
// 2^-44 at the largest angles allowed); then the Taylor series of sin to
// r^13 and of cos to r^14 (truncation errors r^15/15! < 2^-45 and
// r^16/16! < 2^-49 on |r| <= 0.8).
constexpr double kTwoOverPi = 0.6366197723675814;
constexpr double kHalfPiHi = 1.570796012878418;      // 22 significant bits of pi/2
constexpr double kHalfPiLo = 3.139164786504813e-07;  // pi/2 - kHalfPiHi, rounded
constexpr double kMaxReducedAngle = 1073741824.0;    // 2^30

__device__ __forceinline__ void taylor_sincos(double a, double& s, double& c) {
  const double k = rint(a * kTwoOverPi);
  const double r = fma(-k, kHalfPiLo, fma(-k, kHalfPiHi, a));
  const double r2 = r * r;
  // +-1/n!
  double ps = 1.6059043836821613e-10;                 // 1/13!
  ps = fma(ps, r2, -2.505210838544172e-08);           // -1/11!
  ps = fma(ps, r2, 2.7557319223985893e-06);           // 1/9!
  ps = fma(ps, r2, -0.0001984126984126984);           // -1/7!
  ps = fma(ps, r2, 0.008333333333333333);             // 1/5!
  ps = fma(ps, r2, -0.16666666666666666);             // -1/3!
  const double sr = fma(ps * r2, r, r);
  double pc = -1.1470745597729725e-11;                // -1/14!
  pc = fma(pc, r2, 2.08767569878681e-09);             // 1/12!
  pc = fma(pc, r2, -2.755731922398589e-07);           // -1/10!
  pc = fma(pc, r2, 2.48015873015873e-05);             // 1/8!
  pc = fma(pc, r2, -0.001388888888888889);            // -1/6!
  pc = fma(pc, r2, 0.041666666666666664);             // 1/4!
  pc = fma(pc, r2, -0.5);                             // -1/2!
  const double cr = fma(pc, r2, 1.0);
  switch (static_cast<int>(static_cast<long long>(k) & 3)) {
    case 0: s = sr; c = cr; break;
    case 1: s = cr; c = -sr; break;
    case 2: s = -sr; c = -cr; break;
    default: s = -cr; c = sr; break;
  }
}

// x0 * ch + x0 * cl - (x1 * sh + x1 * sl) as an unevaluated fp32 pair
// (hi, lo), |lo| <= ulp(hi) / 2, for fp32 x0, x1 and double-float (ch, cl),
// (sh, sl): the products with the high parts are split exactly by fma, the
// difference of their high parts by TwoSum, and the remaining small terms
// are added in fp32 (error below 2^-45 (|x0| + |x1|) besides the error of
// the double-float cos / sin themselves).
__device__ __forceinline__ void df_dot2(float x0, float ch, float cl, float x1, float sh, float sl,
                                        float& hi, float& lo) {
  const float p = __fmul_rn(x0, ch), pe = __fmaf_rn(x0, ch, -p);
  const float q = __fmul_rn(x1, sh), qe = __fmaf_rn(x1, sh, -q);
  const float t = __fsub_rn(p, q);
  const float z = __fsub_rn(t, p);
  const float te = __fadd_rn(__fsub_rn(p, __fsub_rn(t, z)), __fsub_rn(-q, z));
  const float small = __fadd_rn(__fadd_rn(te, __fsub_rn(pe, qe)),
                                __fsub_rn(__fmul_rn(x0, cl), __fmul_rn(x1, sl)));
  hi = __fadd_rn(t, small);
  const float z2 = __fsub_rn(hi, t);
  lo = __fadd_rn(__fsub_rn(t, __fsub_rn(hi, z2)), __fsub_rn(small, z2));
}

// bf16 bits of hi + lo (|lo| <= ulp(hi) / 2, hi finite and nonzero when lo
// is nonzero), round to nearest even: hi is narrowed toward zero by the
// sign of lo and marked inexact (round to odd), then rounded to bf16; fp32
// keeps 16 more bits than bf16, so this equals one rounding of hi + lo.
__device__ __forceinline__ uint16_t df_to_bf16_bits(float hi, float lo) {
  uint32_t u = __float_as_uint(hi);
  if (lo != 0.f) {
    if ((lo < 0.f) != (hi < 0.f)) u -= 1u;  // |hi + lo| < |hi|: one unit toward zero
    u |= 1u;
  }
  u += 0x7FFFu + ((u >> 16) & 1u);
  return static_cast<uint16_t>(u >> 16);
}

// Distance of hi + lo from the midpoint between the two bf16 values around
// hi exceeds e (so that any value within e of hi + lo rounds to the same
// bf16).  hi - m is exact (m lies in hi's binade, within a factor of two).
__device__ __forceinline__ bool df_clear_of_bf16_midpoint(float hi, float lo, float e) {
  const float m = __uint_as_float((__float_as_uint(hi) & 0xFFFF0000u) | 0x8000u);
  return fabsf(__fadd_rn(__fsub_rn(hi, m), lo)) > e;
}

// The exact path of one pair: fp64 rotation by the library's fp64 sin / cos
// of the fp64 angle a, each result rounded once to bf16 (kept out of line:
// it runs for about one pair in 10^9).
__device__ __noinline__ uint32_t rotate_pair_f64(double a, float x0, float x1) {
  double sd, cd;
  sincos(a, &sd, &cd);
  const double d0 = x0, d1 = x1;
  const uint32_t lo = f64_to_bf16_bits(__dsub_rn(__dmul_rn(d0, cd), __dmul_rn(d1, sd)));
  const uint32_t hi = f64_to_bf16_bits(__dadd_rn(__dmul_rn(d0, sd), __dmul_rn(d1, cd)));
  return lo | (hi << 16);
}

// Indexer cache append / query preparation ("GLM-5.2 架构深度拆解" CH 7.1:
// interleaved RoPE of the indexer vectors; then the FP8 per-block quantiser
// above).  Warp w takes the `group` vectors w*group .. w*group+group-1 (of
// the 32 heads of a query, or one key), all at position pos_of[w / split]
// (`split` warps share a position), so the fp64 sin/cos of the 32 angles
// pos * f[i] are computed once per warp.  The pairs (2i, 2i+1) of the first 64 entries are
// rotated in fp64 and rounded once to bf16 (lanes 0..15 hold them), entries
// 64.. are copied; the result is stored as bf16 or, FP8, Hadamard-rotated and
// quantised.  Destination row: the cache row of (seq_of[w], pos) in the batch
// layout when seq_of is set (keys), else the vector's index (queries).
template <bool FP8>
__global__ void __launch_bounds__(256) rope_append_kernel(
    const uint16_t* __restrict__ x, int64_t npos, int group, int split,
    const int32_t* __restrict__ pos_of,
    const int32_t* __restrict__ seq_of, BatchArgs b, RopeFreq rf, uint16_t* __restrict__ out_bf16,
    uint8_t* __restrict__ out_codes, float* __restrict__ out_scale, int64_t out_rows, int* status) {
  const int lane = threadIdx.x & 31;
  const int64_t w = static_cast<int64_t>(blockIdx.x) * (blockDim.x / 32) + (threadIdx.x >> 5);
  if (w >= npos) return;
  const int pos = pos_of[w / split];
  int64_t row0 = w * group;
  if (seq_of) {
    const int seq = seq_of[w / split];
    row0 = (seq >= 0 && seq < b.num_seqs && pos >= 0)
               ? cache_row(b, seq, seq_base_row(b, seq), pos)
               : -1;
  }
  if (pos < 0 || row0 < 0 || row0 + group > out_rows) {  // uniform over the warp
    if (lane == 0) atomicOr(status, DSA_DEVERR_INDEX);
    return;
  }
  // cos / sin of the 32 angles pos * f[i], one per lane, in fp64 (Taylor
  // series after an fp64 reduction), as double-float fp32 pairs; lanes 0..15
  // (which hold the 64 rotated entries) then fetch those of their two pairs
  float ch, cl, sh, sl;
  bool fast;
  {
    const double a = static_cast<double>(pos) * rf.f[lane];
    fast = fabs(a) < kMaxReducedAngle;
    double sd = 0.0, cd = 1.0;
    if (fast) taylor_sincos(a, sd, cd);
    ch = static_cast<float>(cd);
    cl = static_cast<float>(cd - static_cast<double>(ch));
    sh = static_cast<float>(sd);
    sl = static_cast<float>(sd - static_cast<double>(sh));
  }
  float CH[2], CL[2], SH[2], SL[2];
  bool FAST[2];
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const int src = (2 * lane + q) & 31;
    CH[q] = __shfl_sync(0xffffffffu, ch, src);
    CL[q] = __shfl_sync(0xffffffffu, cl, src);
    SH[q] = __shfl_sync(0xffffffffu, sh, src);
    SL[q] = __shfl_sync(0xffffffffu, sl, src);
    FAST[q] = __shfl_sync(0xffffffffu, fast ? 1 : 0, src) != 0;
  }
  // four vectors' loads in flight before any is used
#pragma unroll 1
  for (int k0 = 0; k0 < group; k0 += 4) {
    uint2 raw[4];
#pragma unroll
    for (int u = 0; u < 4; ++u)
      raw[u] = k0 + u < group
                   ? *reinterpret_cast<const uint2*>(x + (w * group + k0 + u) * 128 + lane * 4)
                   : make_uint2(0u, 0u);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (k0 + u >= group) break;
      const int64_t row = row0 + k0 + u;
      uint16_t h[4] = {static_cast<uint16_t>(raw[u].x & 0xFFFF), static_cast<uint16_t>(raw[u].x >> 16),
                       static_cast<uint16_t>(raw[u].y & 0xFFFF), static_cast<uint16_t>(raw[u].y >> 16)};
      if (lane < 16) {
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const float x0 = bf16_bits_to_float(h[2 * q]), x1 = bf16_bits_to_float(h[2 * q + 1]);
          // y0 = x0 cos - x1 sin, y1 = x0 sin + x1 cos in double-float: error
          // below 2^-43 (|x0| + |x1|) in all (reduction, series, the fp32
          // splits and sums); their bf16 rounding is the exact one unless a
          // value lies within that of a bf16 midpoint
          float y0h, y0l, y1h, y1l;
          df_dot2(x0, CH[q], CL[q], x1, SH[q], SL[q], y0h, y0l);
          df_dot2(x0, SH[q], SL[q], -x1, CH[q], CL[q], y1h, y1l);
          const float mag = fabsf(x0) + fabsf(x1);
          const float e = mag * 9.094947017729282e-13f;  // 2^-40: a margin of 8x
          const bool ok = FAST[q] && mag >= 7.888609052210118e-31f  // 2^-100: no subnormal steps
                          && fabsf(y0h) < 3.0e38f && fabsf(y1h) < 3.0e38f &&
                          df_clear_of_bf16_midpoint(y0h, y0l, e) &&
                          df_clear_of_bf16_midpoint(y1h, y1l, e);
          if (ok) {
            h[2 * q] = df_to_bf16_bits(y0h, y0l);
            h[2 * q + 1] = df_to_bf16_bits(y1h, y1l);
          } else {
            // within 2^-40 of a bf16 midpoint or outside the fast path
            const uint32_t r =
                rotate_pair_f64(static_cast<double>(pos) * rf.f[2 * lane + q], x0, x1);
            h[2 * q] = static_cast<uint16_t>(r & 0xFFFF);
            h[2 * q + 1] = static_cast<uint16_t>(r >> 16);
          }
        }
      }
      if constexpr (!FP8) {
        uint2 o;
        o.x = static_cast<uint32_t>(h[0]) | (static_cast<uint32_t>(h[1]) << 16);
        o.y = static_cast<uint32_t>(h[2]) | (static_cast<uint32_t>(h[3]) << 16);
        *reinterpret_cast<uint2*>(out_bf16 + row * 128 + lane * 4) = o;
      } else {
        float vv[4] = {bf16_bits_to_float(h[0]), bf16_bits_to_float(h[1]),
                       bf16_bits_to_float(h[2]), bf16_bits_to_float(h[3])};
        hadamard_quant_store(vv, lane, out_codes + row * 128, out_scale + row);
      }
    }
  }
}

// E4M3 code of the exact quotient x / sc (nearest, ties to even,
// saturating) for an fp32 x and a positive fp32 scale.  Both are first
// scaled by the same power of two so that sc lies in [1, 2) (exact; an x
// that underflows there has a quotient far below the smallest E4M3
// subnormal).  The quotient is rounded toward zero to fp32 and its lowest
// bit set when the division was inexact (the fma gives the exact remainder's
// sign, and with sc in [1, 2) a nonzero remainder cannot underflow): fp32
// keeps 20 more bits than E4M3, so rounding this round-to-odd value to
// nearest equals one rounding of the exact quotient.
__device__ __forceinline__ __nv_fp8_storage_t e4m3_of_quotient(float x, float sc) {
  int e;
  frexpf(sc, &e);
  const float s1 = ldexpf(sc, 1 - e), x1 = ldexpf(x, 1 - e);
  const float qz = __fdiv_rz(x1, s1);
  uint32_t u = __float_as_uint(qz);
  if (fmaf(-qz, s1, x1) != 0.f) u |= 1u;
  return __nv_cvt_float_to_fp8(__uint_as_float(u), __NV_SATFINITE, __NV_E4M3);
}

// FP8 KV latent rows ("GLM-5.2 / 总览" config table: FP8 KV ~656 B per token
// and layer, per-group): warp r quantises bf16 row r [576] into 656 bytes,
// the 512 latent dims as E4M3 codes in four groups of 128 (lane l: dims
// 16l .. 16l+15, group l / 8), each group scaled by amax/448 (the fp32
// division of the exact amax, i.e. its nearest fp32; 1 for an all-zero
// group) and every code the nearest E4M3 to the exact quotient x / scale,
// then the four fp32 scales, then the 64 bf16 RoPE dims.
__global__ void __launch_bounds__(256) kv_fp8_quant_kernel(const uint16_t* __restrict__ kv,
                                                           int64_t rows,
                                                           uint8_t* __restrict__ out) {
  const int lane = threadIdx.x & 31;
  const int64_t r = static_cast<int64_t>(blockIdx.x) * (blockDim.x / 32) + (threadIdx.x >> 5);
  if (r >= rows) return;
  const uint16_t* x = kv + r * 576;
  uint8_t* o = out + r * 656;
  const uint4 a = *reinterpret_cast<const uint4*>(x + lane * 16);
  const uint4 b2 = *reinterpret_cast<const uint4*>(x + lane * 16 + 8);
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b2.x, b2.y, b2.z, b2.w};
  float v[16];
  float amax = 0.f;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    v[2 * k] = bf16_bits_to_float(static_cast<uint16_t>(w[k] & 0xFFFF));
    v[2 * k + 1] = bf16_bits_to_float(static_cast<uint16_t>(w[k] >> 16));
    amax = fmaxf(amax, fmaxf(fabsf(v[2 * k]), fabsf(v[2 * k + 1])));
  }
#pragma unroll
  for (int m = 1; m < 8; m <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, m));
  const float sc = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
  uint32_t packed[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    uint32_t pk = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      pk |= static_cast<uint32_t>(e4m3_of_quotient(v[4 * k + j], sc)) << (8 * j);
    }
    packed[k] = pk;
  }
  *reinterpret_cast<uint4*>(o + lane * 16) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
  if ((lane & 7) == 0) *reinterpret_cast<float*>(o + 512 + 4 * (lane >> 3)) = sc;
  if (lane < 8)
    *reinterpret_cast<uint4*>(o + 528 + lane * 16) =
        *reinterpret_cast<const uint4*>(x + 512 + lane * 8);
}

// One CTA waits on an mbarrier that nothing arrives on; the bounded wait
// gives up, records the timeout and the kernel returns normally.
__global__ void selftest_wait_kernel(int* status, uint64_t timeout_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(smem_u32(&bar), 0, &abort_flag, status, timeout_ns);
  __syncthreads();
}

}  // namespace

cudaError_t launch_quantize(const void* x, int64_t rows, uint8_t* codes, float* scale,
                            cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  const int64_t blocks = (rows + 7) / 8;
  prof_begin(stream);
  fp8_quant_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
      static_cast<const uint16_t*>(x), rows, codes, scale);
  prof_end(kLaunchQuant, stream);
  count_launch(kLaunchQuant);
  return cudaGetLastError();
}

cudaError_t launch_rope_append(const void* x, int64_t n, int group, const int32_t* pos_of,
                               const int32_t* seq_of, const dsa_batch_t& b, const double* inv_freq,
                               bool fp8, void* out, float* out_scale, int64_t out_rows, int* status,
                               cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  RopeFreq rf;
  for (int i = 0; i < 32; ++i) rf.f[i] = inv_freq[i];
  // few positions (decode): split a position's vectors over up to 8 warps
  // (each recomputes the 32 sin/cos), so that more warps are in flight
  int split = 1;
  while (split < 8 && group % (split * 2) == 0 && (n / group) * split * 2 <= 8 * 152) split *= 2;
  group /= split;
  const int64_t npos = n / group;
  const int64_t blocks = (npos + 7) / 8;
  prof_begin(stream);
  if (fp8)
    rope_append_kernel<true><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        static_cast<const uint16_t*>(x), npos, group, split, pos_of, seq_of, to_args(b), rf, nullptr,
        static_cast<uint8_t*>(out), out_scale, out_rows, status);
  else
    rope_append_kernel<false><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        static_cast<const uint16_t*>(x), npos, group, split, pos_of, seq_of, to_args(b), rf,
        static_cast<uint16_t*>(out), nullptr, nullptr, out_rows, status);
  prof_end(kLaunchAppend, stream);
  count_launch(kLaunchAppend);
  return cudaGetLastError();
}

cudaError_t launch_kv_fp8_quantize(const void* kv, int64_t rows, uint8_t* out,
                                   cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  const int64_t blocks = (rows + 7) / 8;
  prof_begin(stream);
  kv_fp8_quant_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
      static_cast<const uint16_t*>(kv), rows, out);
  prof_end(kLaunchQuant, stream);
  count_launch(kLaunchQuant);
  return cudaGetLastError();
}

cudaError_t launch_selftest_wait(int* status, cudaStream_t stream) {
  selftest_wait_kernel<<<1, 32, 0, stream>>>(status, wait_timeout_ns());
  count_launch(kLaunchOther);
  return cudaGetLastError();
}

}  // namespace dsa

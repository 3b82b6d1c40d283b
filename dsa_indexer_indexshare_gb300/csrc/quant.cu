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
#include <cuda_bf16.h>
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

// The same for a vector held as lane l: elements 2l, 2l+1, 64+2l, 65+2l
// (the layout of the RoPE kernel below).  Index bits 0 and 6 are inside a
// lane, bits 1..5 are lane bits 0..4; the seven butterfly stages give the
// same transform in any order (only the fp32 roundings differ).
__device__ __forceinline__ void hadamard_quant_store_split(float (&v)[4], int lane,
                                                           uint8_t* codes_row, float* scale_slot) {
  {  // h = 1: (2l, 2l+1) and (64+2l, 65+2l)
    const float a0 = v[0], b0 = v[1], a1 = v[2], b1 = v[3];
    v[0] = __fadd_rn(a0, b0);
    v[1] = __fsub_rn(a0, b0);
    v[2] = __fadd_rn(a1, b1);
    v[3] = __fsub_rn(a1, b1);
  }
  // h = 2 .. 32: partner lane l ^ (h / 2)
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    const bool upper = (lane & m) != 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float y = __shfl_xor_sync(0xffffffffu, v[k], m);
      v[k] = upper ? __fsub_rn(y, v[k]) : __fadd_rn(v[k], y);
    }
  }
  {  // h = 64: (2l + b, 64 + 2l + b)
    const float a0 = v[0], b0 = v[2], a1 = v[1], b1 = v[3];
    v[0] = __fadd_rn(a0, b0);
    v[2] = __fsub_rn(a0, b0);
    v[1] = __fadd_rn(a1, b1);
    v[3] = __fsub_rn(a1, b1);
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
  uint32_t c[4];
#pragma unroll
  for (int k = 0; k < 4; ++k)
    c[k] = __nv_cvt_float_to_fp8(__fdiv_rn(v[k], sc), __NV_SATFINITE, __NV_E4M3);
  *reinterpret_cast<uint16_t*>(codes_row + 2 * lane) = static_cast<uint16_t>(c[0] | (c[1] << 8));
  *reinterpret_cast<uint16_t*>(codes_row + 64 + 2 * lane) = static_cast<uint16_t>(c[2] | (c[3] << 8));
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

// sin and cos of an fp64 angle a (|a| < 2^30) as double-float fp32 pairs
// (hi + lo), without a library call.  a is reduced in fp64 to r = a - k pi/2,
// |r| <= pi/4 (a little more when a * 2/pi rounds off), quadrant k mod 4,
// with pi/2 split as P1 + P2, P1 truncated to 22 significant bits so that
// k * P1 is exact for |k| < 2^31 and a - k * P1 is exact (error of r below
// |k| * 1.1e-23 + 2^-53: at most 2^-44 at the largest angles allowed).
// The Taylor series of sin to r^15 and of cos to r^14 (truncation errors
// below 2^-54 and 2^-50 on |r| <= 0.8) are then evaluated in double-float
// arithmetic (Knuth's TwoSum, the fma-based exact product), the terms below
// 2^-24 (from r^10 on) in plain fp32: about 2^-46 of rounding error each,
// and the only fp64 work left is the reduction (GB300's fp64 pipe issues
// about 2 operations per cycle per SM, its fp32 pipe 128).
constexpr double kTwoOverPi = 0.6366197723675814;
constexpr double kHalfPiHi = 1.570796012878418;      // 22 significant bits of pi/2
constexpr double kHalfPiLo = 3.139164786504813e-07;  // pi/2 - kHalfPiHi, rounded

struct DF {
  float h, l;  // the value h + l, |l| <= ulp(h) / 2
};
// a + b as a pair, for |a| >= |b| (or a == 0)
__device__ __forceinline__ DF df_fast_two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  return {s, __fsub_rn(b, __fsub_rn(s, a))};
}
// c + t * q for pairs t, q and a constant c = (ch, cl)
__device__ __forceinline__ DF df_mul_add(DF t, DF q, float ch, float cl) {
  const float p = __fmul_rn(t.h, q.h);
  float pe = __fmaf_rn(t.h, q.h, -p);                      // exact error of p
  pe = __fmaf_rn(t.h, q.l, __fmaf_rn(t.l, q.h, pe));       // + the cross terms
  const float s = __fadd_rn(ch, p);                        // TwoSum(ch, p) = s + se
  const float bv = __fsub_rn(s, ch);
  const float se = __fadd_rn(__fsub_rn(ch, __fsub_rn(s, bv)), __fsub_rn(p, bv));
  return df_fast_two_sum(s, __fadd_rn(se, __fadd_rn(cl, pe)));
}
// a constant as a pair
struct DFC {
  float h, l;
};
constexpr DFC dfc(double x) {
  return {static_cast<float>(x), static_cast<float>(x - static_cast<double>(static_cast<float>(x)))};
}
// +-1/n!
constexpr DFC kC2 = dfc(-1.0 / 2), kC4 = dfc(1.0 / 24), kC6 = dfc(-1.0 / 720),
              kC8 = dfc(1.0 / 40320);
constexpr DFC kS3 = dfc(-1.0 / 6), kS5 = dfc(1.0 / 120), kS7 = dfc(-1.0 / 5040),
              kS9 = dfc(1.0 / 362880);
constexpr float kC10 = static_cast<float>(-1.0 / 3628800), kC12 = static_cast<float>(1.0 / 479001600),
                kC14 = static_cast<float>(-1.0 / 87178291200.0);
constexpr float kS11 = static_cast<float>(-1.0 / 39916800), kS13 = static_cast<float>(1.0 / 6227020800.0),
                kS15 = static_cast<float>(-1.0 / 1307674368000.0);

// The fp32 value of the finite double d truncated toward zero to 24
// significant bits, with integer operations only (0 when |d| < 2^-126);
// and the exact widening of such a value back to fp64.  (fp64 <-> fp32
// conversions issue on GB300's narrow fp64 pipe; these do not.)
__device__ __forceinline__ float f64_trunc_f32(double d) {
  const uint64_t u = static_cast<uint64_t>(__double_as_longlong(d));
  const uint32_t hi = static_cast<uint32_t>(u >> 32), lo = static_cast<uint32_t>(u);
  const int e = static_cast<int>((hi >> 20) & 0x7FFu) - 1023;
  if (e < -126) return 0.f;
  return __uint_as_float((hi & 0x80000000u) | (static_cast<uint32_t>(e + 127) << 23) |
                         ((hi & 0xFFFFFu) << 3) | (lo >> 29));
}
__device__ __forceinline__ double f32_widen_f64(float f) {  // f normal or zero
  const uint32_t b = __float_as_uint(f);
  if ((b & 0x7FFFFFFFu) == 0) return 0.0;
  const uint64_t e = ((b >> 23) & 0xFFu) - 127 + 1023;
  return __longlong_as_double(static_cast<long long>((static_cast<uint64_t>(b & 0x80000000u) << 32) |
                                                     (e << 52) |
                                                     (static_cast<uint64_t>(b & 0x7FFFFFu) << 29)));
}

// sin and cos of the fp64 angle a = pos * f (pos >= 0, f > 0), the product
// rounded once in fp64 as the definition has it.  Returns false (and
// leaves s, c) when a >= 2^30.  The fp64 work is six add / multiply / fma
// operations and no conversion: pos enters through its bits (2^52 + pos
// is exact), k = rint(a * 2/pi) through the 1.5 * 2^52 rounding constant
// (any integer within one of a * 2/pi reduces as well; k mod 4 is the low
// bits of that sum), and r is split into fp32 head and tail by truncation.
__device__ __forceinline__ bool df_sincos_pos(int pos, double f, DF& s, DF& c) {
  const double pd = __dsub_rn(__longlong_as_double(static_cast<long long>(0x4330000000000000ull |
                                                                           static_cast<uint32_t>(pos))),
                              4503599627370496.0);  // 2^52
  const double a = __dmul_rn(pd, f);
  if ((static_cast<uint32_t>(__double_as_longlong(a) >> 32) & 0x7FFFFFFFu) >= 0x41D00000u)
    return false;  // a >= 2^30
  const double tk = __fma_rn(a, kTwoOverPi, 6755399441055744.0);  // 1.5 * 2^52 + k
  const int kq = static_cast<int>(static_cast<uint32_t>(__double_as_longlong(tk)) & 3u);
  const double k = __dsub_rn(tk, 6755399441055744.0);
  const double r = __fma_rn(-k, kHalfPiLo, __fma_rn(-k, kHalfPiHi, a));
  const float rh = f64_trunc_f32(r);
  const float rl = f64_trunc_f32(__dsub_rn(r, f32_widen_f64(rh)));  // r - rh exact
  // t = r^2 as a pair
  const float th = __fmul_rn(rh, rh);
  const DF t = df_fast_two_sum(th, __fmaf_rn(2.f * rh, rl, __fmaf_rn(rh, rh, -th)));
  // cos r = 1 + t (-1/2 + t (1/4! + t (-1/6! + t (1/8! + t (fp32 tail)))))
  const float ec = __fmaf_rn(__fmaf_rn(kC14, th, kC12), th, kC10);
  DF q = df_mul_add(t, DF{ec, 0.f}, kC8.h, kC8.l);
  q = df_mul_add(t, q, kC6.h, kC6.l);
  q = df_mul_add(t, q, kC4.h, kC4.l);
  q = df_mul_add(t, q, kC2.h, kC2.l);
  const DF cr = df_mul_add(t, q, 1.f, 0.f);
  // sin r = r (1 + t (-1/3! + t (1/5! + t (-1/7! + t (1/9! + t (fp32 tail))))))
  const float es = __fmaf_rn(__fmaf_rn(kS15, th, kS13), th, kS11);
  q = df_mul_add(t, DF{es, 0.f}, kS9.h, kS9.l);
  q = df_mul_add(t, q, kS7.h, kS7.l);
  q = df_mul_add(t, q, kS5.h, kS5.l);
  q = df_mul_add(t, q, kS3.h, kS3.l);
  q = df_mul_add(t, q, 1.f, 0.f);
  DF sr;
  {
    const float p = __fmul_rn(rh, q.h);
    const float pe = __fmaf_rn(rh, q.l, __fmaf_rn(rl, q.h, __fmaf_rn(rh, q.h, -p)));
    sr = df_fast_two_sum(p, pe);
  }
  const DF nsr{-sr.h, -sr.l}, ncr{-cr.h, -cr.l};
  switch (kq) {
    case 0: s = sr; c = cr; break;
    case 1: s = cr; c = nsr; break;
    case 2: s = nsr; c = ncr; break;
    default: s = ncr; c = sr; break;
  }
  return true;
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

// The double-float path of one pair (for the rare pair the fp32 path cannot
// decide): y0 = x0 cos - x1 sin, y1 = x0 sin + x1 cos in double-float, error
// below 2^-43 (|x0| + |x1|) in all (reduction, series, the fp32 sums); their
// bf16 rounding is the exact one unless a value lies within that of a bf16
// midpoint, where the exact fp64 path decides.
__device__ __noinline__ uint32_t rotate_pair_df(int pos, double f, bool fast, DF cs, DF sn,
                                                float x0, float x1) {
  float y0h, y0l, y1h, y1l;
  df_dot2(x0, cs.h, cs.l, x1, sn.h, sn.l, y0h, y0l);
  df_dot2(x0, sn.h, sn.l, -x1, cs.h, cs.l, y1h, y1l);
  const float mag = fabsf(x0) + fabsf(x1);
  const float e = mag * 9.094947017729282e-13f;  // 2^-40: a margin of 8x
  const bool ok = fast && mag >= 7.888609052210118e-31f  // 2^-100: no subnormal steps
                  && fabsf(y0h) < 3.0e38f && fabsf(y1h) < 3.0e38f &&
                  df_clear_of_bf16_midpoint(y0h, y0l, e) && df_clear_of_bf16_midpoint(y1h, y1l, e);
  if (ok)
    return static_cast<uint32_t>(df_to_bf16_bits(y0h, y0l)) |
           (static_cast<uint32_t>(df_to_bf16_bits(y1h, y1l)) << 16);
  return rotate_pair_f64(static_cast<double>(pos) * f, x0, x1);
}

// Distance of the fp32 value y from the midpoint between the two bf16 values
// around it exceeds e (y - m is exact: both lie in one binade).
__device__ __forceinline__ bool clear_of_bf16_midpoint(float y, float e) {
  const float m = __uint_as_float((__float_as_uint(y) & 0xFFFF0000u) | 0x8000u);
  return fabsf(__fsub_rn(y, m)) > e;
}

// One rotated pair (lane l: the pair (2l, 2l+1)) as bf16 bits, low half the
// first entry: the fp32 path when it decides, else the double-float one.
__device__ __forceinline__ uint32_t rope_pair_bits(int pos, double f, bool fast, DF cs, DF sn,
                                                   float x0, float x1) {
  const float mag = fabsf(x0) + fabsf(x1);
  const float y0 = __fmaf_rn(x0, cs.h, -__fmul_rn(x1, sn.h));
  const float y1 = __fmaf_rn(x0, sn.h, __fmul_rn(x1, cs.h));
  const float e = mag * 2.384185791015625e-07f;  // 2^-22
  const bool ok = fast && mag >= 7.888609052210118e-31f && fabsf(y0) < 3.0e38f &&
                  fabsf(y1) < 3.0e38f && clear_of_bf16_midpoint(y0, e) && clear_of_bf16_midpoint(y1, e);
  if (ok) {
    const __nv_bfloat162 r2 = __floats2bfloat162_rn(y0, y1);
    return *reinterpret_cast<const uint32_t*>(&r2);
  }
  return rotate_pair_df(pos, f, fast, cs, sn, x0, x1);
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
  // lane l rotates the pair (2l, 2l+1) by the angle pos * f[l] and copies
  // entries 64 + 2l, 65 + 2l; cos / sin of its angle as double-float pairs
  DF sn{0.f, 0.f}, cs{1.f, 0.f};
  const double fq = rf.f[lane];
  const bool fast = df_sincos_pos(pos, fq, sn, cs);
  // eight vectors' loads in flight before any is used
#pragma unroll 1
  for (int k0 = 0; k0 < group; k0 += 8) {
    uint2 raw[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const uint16_t* src = x + (w * group + k0 + u) * 128 + 2 * lane;
      raw[u] = k0 + u < group ? make_uint2(*reinterpret_cast<const uint32_t*>(src),
                                           *reinterpret_cast<const uint32_t*>(src + 64))
                              : make_uint2(0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if (k0 + u >= group) break;
      const int64_t row = row0 + k0 + u;
      const float x0 = bf16_bits_to_float(static_cast<uint16_t>(raw[u].x & 0xFFFF));
      const float x1 = bf16_bits_to_float(static_cast<uint16_t>(raw[u].x >> 16));
      // fp32 first: y0 = fl(x0 ch - fl(x1 sh)), y1 = fl(x0 sh + fl(x1 ch)) with
      // (ch, sh) the fp32 heads of the double-float cos / sin.  Each differs
      // from the exact rotation of the fp64 angle by less than
      // 3.1 * 2^-24 (|x0| + |x1|) (two roundings of at most 2^-24 |y| and
      // 2^-24 |x1|, cos and sin rounded to fp32, the series' 2^-46), so
      // where y lies more than 2^-22 (|x0| + |x1|) from the midpoint between
      // its two bf16 neighbours, y and the exact value round to the same
      // bf16 (about 1 pair in 2000 is closer and takes the double-float path)
      const uint32_t rot = rope_pair_bits(pos, fq, fast, cs, sn, x0, x1);
      if constexpr (!FP8) {
        uint16_t* dst = out_bf16 + row * 128 + 2 * lane;
        *reinterpret_cast<uint32_t*>(dst) = rot;
        *reinterpret_cast<uint32_t*>(dst + 64) = raw[u].y;
      } else {
        float vv[4] = {bf16_bits_to_float(static_cast<uint16_t>(rot & 0xFFFF)),
                       bf16_bits_to_float(static_cast<uint16_t>(rot >> 16)),
                       bf16_bits_to_float(static_cast<uint16_t>(raw[u].y & 0xFFFF)),
                       bf16_bits_to_float(static_cast<uint16_t>(raw[u].y >> 16))};
        hadamard_quant_store_split(vv, lane, out_codes + row * 128, out_scale + row);
      }
    }
  }
}

// New keys (one vector per position): each warp takes kKeysPerWarp keys, so
// that their independent chains (index loads, cache row, angle reduction and
// series, vector load) overlap and every warp of a prefill's keys is resident
// at once.  Same arithmetic and layout as rope_append_kernel.
constexpr int kKeysPerWarp = 2;
template <bool FP8>
__global__ void __launch_bounds__(256) rope_keys_kernel(
    const uint16_t* __restrict__ x, int64_t n, const int32_t* __restrict__ pos_of,
    const int32_t* __restrict__ seq_of, BatchArgs b, RopeFreq rf, uint16_t* __restrict__ out_bf16,
    uint8_t* __restrict__ out_codes, float* __restrict__ out_scale, int64_t out_rows, int* status) {
  const int lane = threadIdx.x & 31;
  const int64_t w0 =
      (static_cast<int64_t>(blockIdx.x) * (blockDim.x / 32) + (threadIdx.x >> 5)) * kKeysPerWarp;
  if (w0 >= n) return;
  int pos[kKeysPerWarp], seq[kKeysPerWarp];
  bool in[kKeysPerWarp];
#pragma unroll
  for (int u = 0; u < kKeysPerWarp; ++u) {
    in[u] = w0 + u < n;
    pos[u] = in[u] ? pos_of[w0 + u] : 0;
    seq[u] = in[u] ? seq_of[w0 + u] : -1;
  }
  int64_t row[kKeysPerWarp];
  uint2 raw[kKeysPerWarp];
#pragma unroll
  for (int u = 0; u < kKeysPerWarp; ++u) {
    const int sq = seq[u];
    row[u] = (sq >= 0 && sq < b.num_seqs && pos[u] >= 0) ? cache_row(b, sq, seq_base_row(b, sq), pos[u])
                                                         : -1;
    const uint16_t* src = x + (w0 + u) * 128 + 2 * lane;
    raw[u] = in[u] ? make_uint2(*reinterpret_cast<const uint32_t*>(src),
                                   *reinterpret_cast<const uint32_t*>(src + 64))
                      : make_uint2(0u, 0u);
  }
  DF sn[kKeysPerWarp], cs[kKeysPerWarp];
  bool fast[kKeysPerWarp];
  const double fq = rf.f[lane];
#pragma unroll
  for (int u = 0; u < kKeysPerWarp; ++u) {
    sn[u] = DF{0.f, 0.f};
    cs[u] = DF{1.f, 0.f};
    fast[u] = pos[u] >= 0 && df_sincos_pos(pos[u], fq, sn[u], cs[u]);
  }
#pragma unroll
  for (int u = 0; u < kKeysPerWarp; ++u) {
    if (!in[u]) break;  // past the last key (uniform over the warp)
    if (pos[u] < 0 || row[u] < 0 || row[u] + 1 > out_rows) {
      if (lane == 0) atomicOr(status, DSA_DEVERR_INDEX);
      continue;
    }
    const uint32_t rot = rope_pair_bits(pos[u], fq, fast[u], cs[u], sn[u],
                                        bf16_bits_to_float(static_cast<uint16_t>(raw[u].x & 0xFFFF)),
                                        bf16_bits_to_float(static_cast<uint16_t>(raw[u].x >> 16)));
    if constexpr (!FP8) {
      uint16_t* dst = out_bf16 + row[u] * 128 + 2 * lane;
      *reinterpret_cast<uint32_t*>(dst) = rot;
      *reinterpret_cast<uint32_t*>(dst + 64) = raw[u].y;
    } else {
      float vv[4] = {bf16_bits_to_float(static_cast<uint16_t>(rot & 0xFFFF)),
                     bf16_bits_to_float(static_cast<uint16_t>(rot >> 16)),
                     bf16_bits_to_float(static_cast<uint16_t>(raw[u].y & 0xFFFF)),
                     bf16_bits_to_float(static_cast<uint16_t>(raw[u].y >> 16))};
      hadamard_quant_store_split(vv, lane, out_codes + row[u] * 128, out_scale + row[u]);
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
  if (seq_of && group == 1 && split == 1) {  // new keys
    const int64_t kb = (n + 8 * kKeysPerWarp - 1) / (8 * kKeysPerWarp);
    if (fp8)
      rope_keys_kernel<true><<<static_cast<unsigned>(kb), 256, 0, stream>>>(
          static_cast<const uint16_t*>(x), n, pos_of, seq_of, to_args(b), rf, nullptr,
          static_cast<uint8_t*>(out), out_scale, out_rows, status);
    else
      rope_keys_kernel<false><<<static_cast<unsigned>(kb), 256, 0, stream>>>(
          static_cast<const uint16_t*>(x), n, pos_of, seq_of, to_args(b), rf,
          static_cast<uint16_t*>(out), nullptr, nullptr, out_rows, status);
  } else if (fp8)
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

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
  double sn[2] = {0.0, 0.0}, cs[2] = {1.0, 1.0};
  if (lane < 16) {
#pragma unroll
    for (int q = 0; q < 2; ++q) sincos(static_cast<double>(pos) * rf.f[2 * lane + q], &sn[q], &cs[q]);
  }
#pragma unroll 1
  for (int k = 0; k < group; ++k) {
    const int64_t v = w * group + k, row = row0 + k;
    const uint2 raw = *reinterpret_cast<const uint2*>(x + v * 128 + lane * 4);
    uint16_t h[4] = {static_cast<uint16_t>(raw.x & 0xFFFF), static_cast<uint16_t>(raw.x >> 16),
                     static_cast<uint16_t>(raw.y & 0xFFFF), static_cast<uint16_t>(raw.y >> 16)};
    if (lane < 16) {
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const double x0 = bf16_bits_to_float(h[2 * q]), x1 = bf16_bits_to_float(h[2 * q + 1]);
        h[2 * q] = f64_to_bf16_bits(__dsub_rn(__dmul_rn(x0, cs[q]), __dmul_rn(x1, sn[q])));
        h[2 * q + 1] = f64_to_bf16_bits(__dadd_rn(__dmul_rn(x0, sn[q]), __dmul_rn(x1, cs[q])));
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

// FP8 KV latent rows ("GLM-5.2 / 总览" config table: FP8 KV ~656 B per token
// and layer, per-group): warp r quantises bf16 row r [576] into 656 bytes,
// the 512 latent dims as E4M3 codes in four groups of 128 (lane l: dims
// 16l .. 16l+15, group l / 8), each group scaled by amax/448 (fp32; 1 for
// an all-zero group), then the four fp32 scales, then the 64 bf16 RoPE dims.
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
      const __nv_fp8_storage_t c =
          __nv_cvt_float_to_fp8(__fdiv_rn(v[4 * k + j], sc), __NV_SATFINITE, __NV_E4M3);
      pk |= static_cast<uint32_t>(c) << (8 * j);
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

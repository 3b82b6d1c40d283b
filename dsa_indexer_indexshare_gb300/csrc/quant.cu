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

__global__ void __launch_bounds__(256) fp8_quant_kernel(const uint16_t* __restrict__ x,
                                                        int64_t rows, uint8_t* __restrict__ codes,
                                                        float* __restrict__ scale) {
  const int lane = threadIdx.x & 31;
  const int64_t r = static_cast<int64_t>(blockIdx.x) * (blockDim.x / 32) + (threadIdx.x >> 5);
  if (r >= rows) return;
  const uint2 raw = *reinterpret_cast<const uint2*>(x + r * 128 + lane * 4);
  float v[4] = {bf16_bits_to_float(raw.x & 0xFFFF), bf16_bits_to_float(raw.x >> 16),
                bf16_bits_to_float(raw.y & 0xFFFF), bf16_bits_to_float(raw.y >> 16)};
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
  *reinterpret_cast<uint32_t*>(codes + r * 128 + lane * 4) = packed;
  if (lane == 0) scale[r] = sc;
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

cudaError_t launch_selftest_wait(int* status, cudaStream_t stream) {
  selftest_wait_kernel<<<1, 32, 0, stream>>>(status, wait_timeout_ns());
  count_launch(kLaunchOther);
  return cudaGetLastError();
}

}  // namespace dsa

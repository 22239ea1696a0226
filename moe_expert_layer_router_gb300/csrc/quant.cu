// fp8 e4m3 quantisation: 128x128 weight blocks and 1x128 activation groups.
// Scale s = amax / 448 in fp32 (1 for an all-zero block); code =
// cvt.rn.satfinite.e4m3(x / s) with the quotient rounded to fp32.
#include <cuda_fp8.h>

#include "moe_internal.h"

namespace moe {
namespace {

__device__ __forceinline__ uint8_t to_e4m3(float v) {
  return static_cast<uint8_t>(__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3));
}

// One block per 128x128 block: 256 threads, each 64 elements (two rows of 32).
__global__ void __launch_bounds__(256)
    quant_weight_kernel(const float* __restrict__ w, int64_t N, int64_t K, uint8_t* __restrict__ q,
                        float* __restrict__ scales) {
  __shared__ float red[8];
  const int64_t bn = blockIdx.y, bk = blockIdx.x;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 32 x 8 threads
  float amax = 0.0f;
  for (int rr = ty; rr < 128; rr += 8) {
    const float* row = w + (bn * 128 + rr) * K + bk * 128;
#pragma unroll
    for (int c = 0; c < 4; ++c) amax = fmaxf(amax, fabsf(row[tx + 32 * c]));
  }
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, d));
  if (tx == 0) red[ty] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) amax = fmaxf(amax, red[i]);
  const float s = amax == 0.0f ? 1.0f : __fdiv_rn(amax, 448.0f);
  if (threadIdx.x == 0) scales[bn * (K / 128) + bk] = s;
  for (int rr = ty; rr < 128; rr += 8) {
    const float* row = w + (bn * 128 + rr) * K + bk * 128;
    uint8_t* qr = q + (bn * 128 + rr) * K + bk * 128;
#pragma unroll
    for (int c = 0; c < 4; ++c) qr[tx + 32 * c] = to_e4m3(__fdiv_rn(row[tx + 32 * c], s));
  }
}

// One half-warp per (row, 128-group): 16 lanes x 8 bf16.
__global__ void __launch_bounds__(256)
    quant_act_kernel(const __nv_bfloat16* __restrict__ x, int64_t M, int64_t K,
                     uint8_t* __restrict__ q, float* __restrict__ scales) {
  const int64_t groups = M * (K / 128);
  const int64_t hw = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 4;
  const int l = threadIdx.x & 15;
  const bool on = hw < groups;
  const int64_t row = on ? hw / (K / 128) : 0, g = on ? hw % (K / 128) : 0;
  float f[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  if (on) {
    const uint4 v = *reinterpret_cast<const uint4*>(x + row * K + g * 128 + l * 8);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
#pragma unroll
  for (int d = 8; d >= 1; d >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, d));
  if (!on) return;
  const float s = amax == 0.0f ? 1.0f : __fdiv_rn(amax, 448.0f);
  uint8_t b[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) b[i] = to_e4m3(__fdiv_rn(f[i], s));
  uint2 out;
  out.x = b[0] | (uint32_t(b[1]) << 8) | (uint32_t(b[2]) << 16) | (uint32_t(b[3]) << 24);
  out.y = b[4] | (uint32_t(b[5]) << 8) | (uint32_t(b[6]) << 16) | (uint32_t(b[7]) << 24);
  *reinterpret_cast<uint2*>(q + row * K + g * 128 + l * 8) = out;
  if (l == 0) scales[row * (K / 128) + g] = s;
}

}  // namespace

cudaError_t launch_quant_weight_fp8(const float* w, int64_t N, int64_t K, uint8_t* q,
                                    float* scales, cudaStream_t stream) {
  dim3 grid(static_cast<unsigned>(K / 128), static_cast<unsigned>(N / 128));
  quant_weight_kernel<<<grid, 256, 0, stream>>>(w, N, K, q, scales);
  return cudaGetLastError();
}

cudaError_t launch_quant_act_fp8(const void* x, int64_t M, int64_t K, uint8_t* q, float* scales,
                                 cudaStream_t stream) {
  const int64_t threads = M * (K / 128) * 16;
  const unsigned blocks = static_cast<unsigned>((threads + 255) / 256);
  quant_act_kernel<<<blocks, 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(x), M, K, q,
                                                scales);
  return cudaGetLastError();
}

}  // namespace moe

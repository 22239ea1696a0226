// fp8 e4m3 quantisation: 128x128 weight blocks and 1x128 activation groups.
// Scale s = amax / 448 in fp32 (1 for an all-zero block); code =
// cvt.rn.satfinite.e4m3(x / s) with the quotient rounded to fp32.
// NVFP4 quantisation (nvfp4.cuh): weights with the tensor scale amax / 2688,
// activations with a given static tensor scale.
#include <cuda_fp8.h>

#include "moe_internal.h"
#include "nvfp4.cuh"

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

// ---------------------------------------------------------------- NVFP4
__device__ __forceinline__ void bf16x16(const __nv_bfloat16* p, float (&f)[16]) {
  const uint4 a = *reinterpret_cast<const uint4*>(p);
  const uint4 b = *reinterpret_cast<const uint4*>(p + 8);
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

// amax of one or two bf16 matrices (n8 16-byte chunks each) into *amax_bits:
// non-negative floats order like their bit patterns.
__global__ void __launch_bounds__(256)
    nvfp4_amax_kernel(const __nv_bfloat16* __restrict__ w, const __nv_bfloat16* __restrict__ w2,
                      int64_t n8, uint32_t* amax_bits) {
  float a = 0.0f;
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int src = 0; src < (w2 ? 2 : 1); ++src) {
    const uint4* p = reinterpret_cast<const uint4*>(src ? w2 : w);
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n8; i += stride) {
      const uint4 v = p[i];
      const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 4; ++j)
        a = fmaxf(a, fmaxf(fabsf(__uint_as_float(u[j] << 16)),
                           fabsf(__uint_as_float(u[j] & 0xffff0000u))));
    }
  }
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, d));
  if ((threadIdx.x & 31) == 0) atomicMax(amax_bits, __float_as_uint(a));
}

__device__ __forceinline__ float weight_tensor_scale(uint32_t amax_bits) {
  const float amax = __uint_as_float(amax_bits);
  return amax == 0.0f ? 1.0f : __fdiv_rn(amax, nvfp4::kTensorDiv);
}

// One thread per (output row, 16-element block).  With w2, output row v is row
// 128 (v / 256) + v % 128 of w (v % 256 < 128) or of w2 (otherwise).
__global__ void __launch_bounds__(256)
    nvfp4_quant_weight_kernel(const __nv_bfloat16* __restrict__ w,
                              const __nv_bfloat16* __restrict__ w2, int64_t N, int64_t K,
                              const uint32_t* __restrict__ amax_bits, uint8_t* __restrict__ codes,
                              uint8_t* __restrict__ sf) {
  const int64_t nb = K / nvfp4::kBlock;
  const int64_t rows = w2 ? 2 * N : N;
  const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= rows * nb) return;
  const int64_t v = i / nb;
  const int kb = static_cast<int>(i - v * nb);
  const __nv_bfloat16* src;
  if (w2) {
    const int64_t r = (v >> 8) * 128 + (v & 127);
    src = ((v & 255) < 128 ? w : w2) + r * K;
  } else {
    src = w + v * K;
  }
  float f[16];
  bf16x16(src + kb * nvfp4::kBlock, f);
  uint2 q;
  const uint32_t sc = nvfp4::quantize16(f, weight_tensor_scale(*amax_bits), q);
  *reinterpret_cast<uint2*>(codes + v * (K / 2) + kb * 8) = q;
  sf[nvfp4::sf_offset(v, kb, static_cast<int>(K))] = static_cast<uint8_t>(sc);
}

__global__ void nvfp4_finish_kernel(float* tensor_scale) {
  const uint32_t bits = *reinterpret_cast<const uint32_t*>(tensor_scale);
  *tensor_scale = weight_tensor_scale(bits);
}

// One thread per (row, 16-element block); row-major e4m3 scale codes.
__global__ void __launch_bounds__(256)
    nvfp4_quant_act_kernel(const __nv_bfloat16* __restrict__ x, int64_t M, int64_t K, float g,
                           uint8_t* __restrict__ codes, uint8_t* __restrict__ sf) {
  const int64_t nb = K / nvfp4::kBlock;
  const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= M * nb) return;
  const int64_t row = i / nb;
  const int64_t kb = i - row * nb;
  float f[16];
  bf16x16(x + row * K + kb * nvfp4::kBlock, f);
  uint2 q;
  sf[i] = static_cast<uint8_t>(nvfp4::quantize16(f, g, q));
  *reinterpret_cast<uint2*>(codes + row * (K / 2) + kb * 8) = q;
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

cudaError_t launch_quant_weight_nvfp4(const void* w, const void* w2, int64_t N, int64_t K,
                                      uint8_t* codes, uint8_t* sf, float* tensor_scale,
                                      cudaStream_t stream) {
  cudaError_t e = cudaMemsetAsync(tensor_scale, 0, sizeof(float), stream);
  if (e != cudaSuccess) return e;
  const int64_t n8 = N * K / 8;
  int64_t blocks = (n8 + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  nvfp4_amax_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(w), static_cast<const __nv_bfloat16*>(w2), n8,
      reinterpret_cast<uint32_t*>(tensor_scale));
  const int64_t threads = (w2 ? 2 * N : N) * (K / nvfp4::kBlock);
  nvfp4_quant_weight_kernel<<<static_cast<unsigned>((threads + 255) / 256), 256, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(w), static_cast<const __nv_bfloat16*>(w2), N, K,
      reinterpret_cast<const uint32_t*>(tensor_scale), codes, sf);
  nvfp4_finish_kernel<<<1, 1, 0, stream>>>(tensor_scale);
  return cudaGetLastError();
}

cudaError_t launch_quant_act_nvfp4(const void* x, int64_t M, int64_t K, float g, uint8_t* codes,
                                   uint8_t* sf, cudaStream_t stream) {
  const int64_t threads = M * (K / nvfp4::kBlock);
  nvfp4_quant_act_kernel<<<static_cast<unsigned>((threads + 255) / 256), 256, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(x), M, K, g, codes, sf);
  return cudaGetLastError();
}

}  // namespace moe

// Combine: out[t] = sum_j y_perm[inv_row[t, j]] (+ shared_out[t]) -- the
// expert results of each token gathered back to token order and summed in
// fp32, slot order j = 0..k-1 then the shared expert, rounded once to bf16.
// y_perm and shared_out are fp32 rows (the grouped down projection writes
// them unrounded), or, in the layer forward, fp16 rows with a power-of-two
// scale per 32 columns.  One block per token; each thread owns 8-column chunks and
// issues the k row loads of a chunk back to back so they are in flight together.
#include <cuda_fp16.h>

#include "moe_internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kThreads = 128;
constexpr int kMaxK = 16;

__device__ __forceinline__ uint32_t pack2(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ void add4(float (&acc)[8], int o, const float4& v) {
  acc[o] += v.x;
  acc[o + 1] += v.y;
  acc[o + 2] += v.z;
  acc[o + 3] += v.w;
}

// 128 threads, up to 8 blocks (32 warps) per SM: enough loads in flight to
// keep HBM busy without holding all k rows in registers at once.
__global__ void __launch_bounds__(kThreads, 8)
    combine_kernel(const float4* __restrict__ y, const int32_t* __restrict__ inv_row,
                   const float4* __restrict__ sh, uint4* __restrict__ out, int k, int H, int64_t R,
                   uint32_t* err) {
  __shared__ int64_t rows[kMaxK];
  const int64_t t = blockIdx.x;
  const int nch = H / 8;  // 8 columns: two float4 in, one uint4 of bf16 out
  if (threadIdx.x < k) {
    const int32_t r = inv_row[t * k + threadIdx.x];
    int64_t rr = r;
    if (r < 0 || r >= R) {
      atomicOr(err, kErrBounds);
      rr = -1;
    }
    rows[threadIdx.x] = rr;
  }
  __syncthreads();
  for (int c = threadIdx.x; c < nch; c += kThreads) {
    float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    // slots in order j = 0..k-1, four rows' loads in flight at a time
    for (int j0 = 0; j0 < k; j0 += 4) {
      float4 v[4][2];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int j = j0 + u;
        if (j < k && rows[j] >= 0) {
          const float4* src = y + rows[j] * (2 * nch) + 2 * c;
          v[u][0] = __ldcs(src);
          v[u][1] = __ldcs(src + 1);
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int j = j0 + u;
        if (j < k && rows[j] >= 0) {
          add4(acc, 0, v[u][0]);
          add4(acc, 4, v[u][1]);
        }
      }
    }
    if (sh) {
      const float4* src = sh + t * (2 * nch) + 2 * c;
      add4(acc, 0, __ldcs(src));
      add4(acc, 4, __ldcs(src + 1));
    }
    out[t * nch + c] = make_uint4(pack2(acc[0], acc[1]), pack2(acc[2], acc[3]),
                                  pack2(acc[4], acc[5]), pack2(acc[6], acc[7]));
  }
}

// acc[0..7] += 8 fp16 values (one uint4) times their power-of-two scale s.
__device__ __forceinline__ void add8h(float (&acc)[8], const uint4& v, float s) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
    acc[2 * i] += f.x * s;
    acc[2 * i + 1] += f.y * s;
  }
}

// The same combine over fp16 rows with one power-of-two scale per 32 columns
// ([rows][H/32]): each value is widened exactly, y = h * s, then summed in
// fp32 in slot order, the shared row last.  One uint4 (8 columns) of every
// row per chunk.
__global__ void __launch_bounds__(kThreads, 8)
    combine_half_kernel(const uint4* __restrict__ y, const float* __restrict__ ysc,
                        const int32_t* __restrict__ inv_row, const uint4* __restrict__ sh,
                        const float* __restrict__ shsc, uint4* __restrict__ out, int k, int H,
                        int64_t R, uint32_t* err) {
  __shared__ int64_t rows[kMaxK];
  const int64_t t = blockIdx.x;
  const int nch = H / 8;
  const int nsc = H / 32;
  if (threadIdx.x < k) {
    const int32_t r = inv_row[t * k + threadIdx.x];
    int64_t rr = r;
    if (r < 0 || r >= R) {
      atomicOr(err, kErrBounds);
      rr = -1;
    }
    rows[threadIdx.x] = rr;
  }
  __syncthreads();
  for (int c = threadIdx.x; c < nch; c += kThreads) {
    float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    for (int j0 = 0; j0 < k; j0 += 4) {
      uint4 v[4];
      float sc[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int j = j0 + u;
        if (j < k && rows[j] >= 0) {
          v[u] = __ldcs(y + rows[j] * nch + c);
          sc[u] = __ldg(ysc + rows[j] * nsc + (c >> 2));
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int j = j0 + u;
        if (j < k && rows[j] >= 0) add8h(acc, v[u], sc[u]);
      }
    }
    if (sh) add8h(acc, __ldcs(sh + t * nch + c), __ldg(shsc + t * nsc + (c >> 2)));
    out[t * nch + c] = make_uint4(pack2(acc[0], acc[1]), pack2(acc[2], acc[3]),
                                  pack2(acc[4], acc[5]), pack2(acc[6], acc[7]));
  }
}

// fp16 rows with a power-of-two scale per 32 columns widened to fp32 rows:
// each value is h * s exactly (the step interface of NVFP4 layers hands fp32
// expert rows to the combine).  One thread per 8 columns, grid-stride.
__global__ void __launch_bounds__(256)
    widen_half_kernel(const uint4* __restrict__ y, const float* __restrict__ ysc,
                      float4* __restrict__ out, int64_t rows, int H) {
  const int nch = H / 8;
  const int nsc = H / 32;
  const int64_t n = rows * nch;
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n;
       i += int64_t(gridDim.x) * blockDim.x) {
    const int64_t r = i / nch;
    const int c = static_cast<int>(i - r * nch);
    const uint4 v = __ldcs(y + i);
    const float s = __ldg(ysc + r * nsc + (c >> 2));
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float f[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 h = __half22float2(*reinterpret_cast<const __half2*>(&w[j]));
      f[2 * j] = h.x * s;
      f[2 * j + 1] = h.y * s;
    }
    out[2 * i] = make_float4(f[0], f[1], f[2], f[3]);
    out[2 * i + 1] = make_float4(f[4], f[5], f[6], f[7]);
  }
}

}  // namespace

cudaError_t launch_combine_half(const void* y, const float* y_scales, const int32_t* inv_row,
                                const void* shared, const float* shared_scales, void* out,
                                int64_t T, int k, int H, int64_t R, uint32_t* err,
                                cudaStream_t stream) {
  combine_half_kernel<<<static_cast<unsigned>(T), kThreads, 0, stream>>>(
      static_cast<const uint4*>(y), y_scales, inv_row, static_cast<const uint4*>(shared),
      shared_scales, static_cast<uint4*>(out), k, H, R, err);
  return cudaGetLastError();
}

cudaError_t launch_combine(const void* y_perm, const int32_t* inv_row, const void* shared_out,
                           void* out, int64_t T, int k, int H, int64_t R, uint32_t* err,
                           cudaStream_t stream) {
  combine_kernel<<<static_cast<unsigned>(T), kThreads, 0, stream>>>(
      static_cast<const float4*>(y_perm), inv_row, static_cast<const float4*>(shared_out),
      static_cast<uint4*>(out), k, H, R, err);
  return cudaGetLastError();
}

cudaError_t launch_widen_half(const void* y, const float* scales, float* out, int64_t rows, int H,
                              cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t n = rows * (H / 8);
  int64_t grid = (n + 255) / 256;
  const int64_t cap = int64_t(sms > 0 ? sms : 1) * 8;
  if (grid > cap) grid = cap;
  widen_half_kernel<<<static_cast<unsigned>(grid), 256, 0, stream>>>(
      static_cast<const uint4*>(y), scales, reinterpret_cast<float4*>(out), rows, H);
  return cudaGetLastError();
}

}  // namespace moe

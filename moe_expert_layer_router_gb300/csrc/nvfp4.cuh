// NVFP4 arithmetic shared by the quantisers, the scatter and the grouped GEMM
// epilogue: E2M1 elements (OCP Microscaling v1.0 FP4; magnitudes 0, 0.5, 1,
// 1.5, 2, 3, 4, 6), one UE4M3 scale per 16 consecutive elements along K and a
// float32 tensor scale g; value = e2m1 * e4m3 * g.  For a block x[0..15]:
//   s = e4m3_rn_satfinite(amax / (6 g)),  q_i = e2m1_rn(x_i / (s g))
// every step rounded to float32 (q = 0 when s g == 0); E2M1 rounds to nearest,
// ties to the even code, saturates at 6 and writes zero as +0.
#pragma once

#include <cuda_fp8.h>

#include <cstdint>

namespace moe {
namespace nvfp4 {

constexpr int kBlock = 16;           // elements per scale
constexpr float kE2M1Max = 6.0f;
constexpr float kTensorDiv = 2688.0f;  // 6 * 448: weight tensor scale g = amax / 2688

// E2M1 code of r: the magnitude code is the number of rounding thresholds at or
// below |r| (ties to the even code: 0.25 -> 0, 0.75 -> 1.0, 1.25 -> 1.0,
// 1.75 -> 2, 2.5 -> 2, 3.5 -> 4, 5 -> 4), saturating at 6 (code 7).
__device__ __forceinline__ uint32_t e2m1(float r) {
  const float a = fabsf(r);
  const uint32_t m = uint32_t(a > 0.25f) + uint32_t(a >= 0.75f) + uint32_t(a > 1.25f) +
                     uint32_t(a >= 1.75f) + uint32_t(a > 2.5f) + uint32_t(a >= 3.5f) +
                     uint32_t(a > 5.0f);
  return (r < 0.0f && m != 0u) ? (m | 8u) : m;
}

// Value of a non-negative e4m3 code (bias 7, 3 mantissa bits).
__device__ __forceinline__ float e4m3_value(uint32_t c) {
  const uint32_t e = (c >> 3) & 15u, m = c & 7u;
  return e ? __uint_as_float(((e + 120u) << 23) | (m << 20)) : float(m) * 0.001953125f;
}

// Quantises 16 values with tensor scale g: returns the e4m3 scale code and the
// 16 codes packed into 8 bytes (element 2i in the low nibble of byte i).
__device__ __forceinline__ uint32_t quantize16(const float (&v)[16], float g, uint2& packed) {
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
  const float d = __fmul_rn(kE2M1Max, g);
  const uint32_t sc = static_cast<uint32_t>(
      __nv_cvt_float_to_fp8(__fdiv_rn(amax, d), __NV_SATFINITE, __NV_E4M3));
  const float den = __fmul_rn(e4m3_value(sc), g);
  uint32_t lo = 0u, hi = 0u;
  if (den != 0.0f) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      lo |= e2m1(__fdiv_rn(v[i], den)) << (4 * i);
      hi |= e2m1(__fdiv_rn(v[i + 8], den)) << (4 * i);
    }
  }
  packed = make_uint2(lo, hi);
  return sc;
}

// Byte offset of the scale of (row, 16-element block kb) in the MMA scale
// layout of a matrix with K columns (rows a multiple of 128, K of 64): 512-byte
// atoms of 128 rows x 4 blocks, atom (row / 128, kb / 4) at
// ((row / 128) * (K / 64) + kb / 4) * 512, holding byte
// (row % 32) * 16 + ((row % 128) / 32) * 4 + kb % 4.  One atom is what one
// tcgen05.cp of 32 x 128 bits carries into TMEM for one MMA (K = 64).
__host__ __device__ __forceinline__ int64_t sf_offset(int64_t row, int kb, int K) {
  return ((row >> 7) * (K >> 6) + (kb >> 2)) * 512 + (row & 31) * 16 + ((row & 127) >> 5) * 4 +
         (kb & 3);
}

}  // namespace nvfp4
}  // namespace moe

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

// Eight values -> their E2M1 codes packed into 32 bits (value 2i in the low
// nibble of byte i, 2i + 1 in the high one), by the hardware conversion
// cvt.rn.satfinite.e2m1x2.f32: round to nearest, ties to the even code
// (0.25 -> 0, 0.75 -> 1.0, 1.25 -> 1.0, 1.75 -> 2, 2.5 -> 2, 3.5 -> 4,
// 5 -> 4), saturating at 6.  It keeps the sign of a value that rounds to zero;
// those codes are cleared to +0.
__device__ __forceinline__ uint32_t e2m1x8(const float* r) {
  uint32_t w;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(w)
      : "f"(r[0]), "f"(r[1]), "f"(r[2]), "f"(r[3]), "f"(r[4]), "f"(r[5]), "f"(r[6]), "f"(r[7]));
  const uint32_t nonzero = (w | (w >> 1) | (w >> 2)) & 0x11111111u;  // bit 0 of each nibble
  return (w & 0x77777777u) | (w & (nonzero << 3));
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
    float r[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) r[i] = __fdiv_rn(v[i], den);
    lo = e2m1x8(r);
    hi = e2m1x8(r + 8);
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

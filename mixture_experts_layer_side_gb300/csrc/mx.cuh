// MXFP8 element helpers shared by the quantiser and the GEMM epilogues that
// quantise their outputs (OCP MX v1.0 rule: X = floor(log2 amax) - 8, clamped
// to [-127, 127], all-zero block -127; elements RNE to E4M3, saturating).
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace mok {

__device__ __forceinline__ int mx_block_exponent(float amax) {
  const int ef = (__float_as_int(amax) >> 23) & 0xFF;
  if (ef == 0) return -127;
  const int x = ef - 127 - 8;
  return x < -127 ? -127 : (x > 127 ? 127 : x);
}

__device__ __forceinline__ float mx_exp2_int(int e) {  // 2^e for e in [-126, 127]
  return __int_as_float((e + 127) << 23);
}

// Two floats -> two E4M3 codes (lo in the low byte), RNE, saturate to finite.
__device__ __forceinline__ uint16_t mx_cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// One 32-element block: E4M3 codes (8 words, element i in byte i) and the
// E8M0 scale code.
__device__ __forceinline__ uint8_t mx_quant32(const float (&v)[32], uint32_t (&codes)[8]) {
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
  const int X = mx_block_exponent(amax);
  const float inv = mx_exp2_int(-X);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint16_t a = mx_cvt_e4m3x2(v[4 * i] * inv, v[4 * i + 1] * inv);
    const uint16_t b = mx_cvt_e4m3x2(v[4 * i + 2] * inv, v[4 * i + 3] * inv);
    codes[i] = (uint32_t)a | ((uint32_t)b << 16);
  }
  return (uint8_t)(X + 127);
}

// Offset of scale (mn, kb) inside a 512-byte block of 128 rows (or columns) x
// 4 K-blocks -- the layout tcgen05.cp .32x128b.warpx4 replicates into the
// four TMEM lane quarters: byte (mn % 32) * 16 + (mn / 32) * 4 + kb.
__device__ __forceinline__ int mx_sf_offset(int mn, int kb) { return (mn & 31) * 16 + (mn >> 5) * 4 + kb; }

}  // namespace mok

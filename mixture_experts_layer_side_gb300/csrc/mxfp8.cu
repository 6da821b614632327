// MXFP8 block quantisation: E4M3 elements, one E8M0 scale per 32 elements.
//
// The pages name the mode and say weights are pre-quantised with
// ops.mxfp8_quantize ("Mixture-of-Kittens (MoK)", "Core concepts" table,
// MXFP8 row; "Limitations / considerations").  Format and rule are the OCP
// Microscaling v1.0 MXFP8 conversion:
//   X = floor(log2(amax)) - 8, clamped to [-127, 127] (all-zero block: -127)
//   q = RNE(v * 2^-X) to E4M3, saturating at +-448
// floor(log2(amax)) is read from the float32 exponent field of amax (exact);
// a zero or subnormal amax gives X = -127 after the clamp.  v * 2^-X is an
// exact power-of-two scaling, and the conversion is the hardware's
// round-to-nearest-even, saturate-to-finite cvt.
#include "mok_internal.cuh"

namespace mok {

namespace {

__device__ __forceinline__ int block_exponent(float amax) {
  const int ef = (__float_as_int(amax) >> 23) & 0xFF;
  if (ef == 0) return -127;
  int x = ef - 127 - 8;
  return x < -127 ? -127 : (x > 127 ? 127 : x);
}

__device__ __forceinline__ float exp2_int(int e) {  // 2^e for e in [-126, 127]
  return __int_as_float((e + 127) << 23);
}

// Two floats -> two E4M3 codes (lo in the low byte).
__device__ __forceinline__ uint16_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Blocks along the contiguous axis: one thread per 32-element block.
__global__ void quant_rowblocks(const __nv_bfloat16* __restrict__ src, long nblocks, uint8_t* __restrict__ q,
                                uint8_t* __restrict__ sf) {
  for (long b = blockIdx.x * (long)blockDim.x + threadIdx.x; b < nblocks; b += (long)gridDim.x * blockDim.x) {
    const uint4* s = reinterpret_cast<const uint4*>(src + b * 32);
    float v[32];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 w = s[i];
      const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ww[j]));
        v[8 * i + 2 * j] = f.x;
        v[8 * i + 2 * j + 1] = f.y;
      }
    }
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
    const int X = block_exponent(amax);
    const float inv = exp2_int(-X);
    uint32_t out[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint16_t a = cvt_e4m3x2(v[4 * i] * inv, v[4 * i + 1] * inv);
      const uint16_t c = cvt_e4m3x2(v[4 * i + 2] * inv, v[4 * i + 3] * inv);
      out[i] = (uint32_t)a | ((uint32_t)c << 16);
    }
    uint4* d = reinterpret_cast<uint4*>(q + b * 32);
    d[0] = make_uint4(out[0], out[1], out[2], out[3]);
    d[1] = make_uint4(out[4], out[5], out[6], out[7]);
    sf[b] = (uint8_t)(X + 127);
  }
}

// Blocks along the row axis of [batch, rows, cols]: one thread per
// (batch, row block, column); consecutive threads take consecutive columns.
__global__ void quant_colblocks(const __nv_bfloat16* __restrict__ src, int batch, int rows, int cols,
                                uint8_t* __restrict__ q, uint8_t* __restrict__ sf) {
  const long rb_per = rows / 32;
  const long n = (long)batch * rb_per * cols;
  for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < n; i += (long)gridDim.x * blockDim.x) {
    const int c = (int)(i % cols);
    const long br = i / cols;  // batch * rb_per + rb
    const long bidx = br / rb_per;
    const long rb = br % rb_per;
    const long base = (bidx * rows + rb * 32) * (long)cols + c;
    float v[32];
    float amax = 0.0f;
#pragma unroll
    for (int r = 0; r < 32; ++r) {
      v[r] = __bfloat162float(src[base + (long)r * cols]);
      amax = fmaxf(amax, fabsf(v[r]));
    }
    const int X = block_exponent(amax);
    const float inv = exp2_int(-X);
#pragma unroll
    for (int r = 0; r < 32; r += 2) {
      const uint16_t pr = cvt_e4m3x2(v[r] * inv, v[r + 1] * inv);
      q[base + (long)r * cols] = (uint8_t)(pr & 0xFF);
      q[base + (long)(r + 1) * cols] = (uint8_t)(pr >> 8);
    }
    sf[br * cols + c] = (uint8_t)(X + 127);
  }
}

}  // namespace

cudaError_t launch_mxfp8_quantize(const __nv_bfloat16* src, int batch, int rows, int cols, int block_axis,
                                  uint8_t* q, uint8_t* sf, cudaStream_t st) {
  const int sms = device_sm_count();
  if (block_axis == 1) {
    const long nblocks = (long)batch * rows * (cols / 32);
    long grid = (nblocks + 255) / 256;
    if (grid > (long)sms * 32) grid = (long)sms * 32;
    quant_rowblocks<<<(int)(grid < 1 ? 1 : grid), 256, 0, st>>>(src, nblocks, q, sf);
  } else {
    const long n = (long)batch * (rows / 32) * cols;
    long grid = (n + 255) / 256;
    if (grid > (long)sms * 32) grid = (long)sms * 32;
    quant_colblocks<<<(int)(grid < 1 ? 1 : grid), 256, 0, st>>>(src, batch, rows, cols, q, sf);
  }
  return cudaGetLastError();
}

}  // namespace mok

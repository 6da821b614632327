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
#include "mx.cuh"

namespace mok {

namespace {

__device__ __forceinline__ int block_exponent(float amax) { return mx_block_exponent(amax); }
__device__ __forceinline__ float exp2_int(int e) { return mx_exp2_int(e); }
__device__ __forceinline__ uint16_t cvt_e4m3x2(float lo, float hi) { return mx_cvt_e4m3x2(lo, hi); }

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

__device__ __forceinline__ int sf_block_offset(int mn, int kb) { return mx_sf_offset(mn, kb); }

// Tiled scale layout of a weight: 512-byte blocks, one per 128 N x 128 K
// tile, grouped so that one bulk load brings what one stage of a GEMM tile
// needs: [batch][N / (128 g)][K/128][s blocks], the block of N block nb at
// slot `slot + nb % g` of its group.  g = s = 1: one block per group; g = s
// = 2: the two 128-wide N blocks of a 256-wide N tile side by side; g = 1,
// s = 2, slot 0 / 1: two weights' blocks interleaved (W1 | W3).
__device__ __forceinline__ long tiled_block(long b, int nb, int kg, int n_blocks, int kg_count, int g, int s,
                                            int slot) {
  return (((b * (n_blocks / g) + nb / g) * kg_count + kg) * s + slot + nb % g) * 512;
}

// Plain scales of a K-major operand [batch][N][K/32] (blocks along each
// row) -> the same tiled layout: the four scale bytes of (n, 128-wide K
// group) are contiguous in the source.
__global__ void tile_scales_rows_kernel(const uint8_t* __restrict__ sf, int batch, int N, int kb_count,
                                        uint8_t* __restrict__ out, int g, int s, int slot) {
  const int kg_count = kb_count / 4;
  const long n_words = (long)batch * N * kg_count;
  for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < n_words; i += (long)gridDim.x * blockDim.x) {
    const int kg = (int)(i % kg_count);
    const long bn = i / kg_count;
    const int n = (int)(bn % N);
    const long b = bn / N;
    const uint32_t w = *reinterpret_cast<const uint32_t*>(sf + bn * kb_count + (long)kg * 4);
    uint8_t* blk = out + tiled_block(b, n / 128, kg, N / 128, kg_count, g, s, slot);
    *reinterpret_cast<uint32_t*>(blk + sf_block_offset(n & 127, 0)) = w;
  }
}

// The tilings with coalesced reads and writes: a CTA builds whole 512-byte
// blocks in shared memory and writes them out in 16-byte pieces (one word
// per thread, as tile_scales_rows_kernel does, scatters 4-byte stores over
// each block; it stays for runs too long for shared memory).
//   tile_scales_blocks_kernel: plain scales [batch][K/32][N] (blocks along
//   K = rows); one CTA of 128 threads per block (b, 128 N, K group); thread
//   n reads its four scale bytes from four rows of 128 contiguous bytes.
__global__ void __launch_bounds__(128) tile_scales_blocks_kernel(const uint8_t* __restrict__ sf, int batch,
                                                                 int kb_count, int N, uint8_t* __restrict__ out,
                                                                 int g, int s, int slot) {
  __shared__ uint32_t blk[128];
  const int kg_count = kb_count / 4, nbs = N / 128;
  const long nblocks = (long)batch * nbs * kg_count;
  const int n = threadIdx.x;
  for (long bi = blockIdx.x; bi < nblocks; bi += gridDim.x) {
    const int kg = (int)(bi % kg_count);
    const long bn = bi / kg_count;
    const int nb = (int)(bn % nbs);
    const long b = bn / nbs;
    const uint8_t* src = sf + (b * kb_count + (long)kg * 4) * N + (long)nb * 128 + n;
    const uint32_t w = (uint32_t)src[0] | ((uint32_t)src[N] << 8) | ((uint32_t)src[2L * N] << 16) |
                       ((uint32_t)src[3L * N] << 24);
    __syncthreads();  // the previous block is written out
    blk[sf_block_offset(n, 0) / 4] = w;
    __syncthreads();
    if (n < 32)
      reinterpret_cast<uint4*>(out + tiled_block(b, nb, kg, nbs, kg_count, g, s, slot))[n] =
          reinterpret_cast<const uint4*>(blk)[n];
  }
}

//   tile_scales_run_kernel: the same for one CTA of 256 threads per (b,
//   128 N) and every K group of it (all of its blocks in shared memory), so
//   each thread has many independent loads in flight.  A thread takes four
//   N columns of one K group: one 32-bit load from each of the group's four
//   scale rows (a warp reads 128 contiguous bytes of a row), then a 4 x 4
//   byte transpose in registers gives the four columns' words.
__global__ void __launch_bounds__(256) tile_scales_run_kernel(const uint8_t* __restrict__ sf, int batch,
                                                              int kb_count, int N, uint8_t* __restrict__ out, int g,
                                                              int s, int slot) {
  extern __shared__ __align__(16) uint32_t blks[];  // [kg_count][128 words]
  const int kg_count = kb_count / 4, nbs = N / 128;
  const long nrun = (long)batch * nbs;
  for (long bi = blockIdx.x; bi < nrun; bi += gridDim.x) {
    const int nb = (int)(bi % nbs);
    const long b = bi / nbs;
    const uint8_t* src0 = sf + b * kb_count * (long)N + (long)nb * 128;
    __syncthreads();  // the previous run is written out
#pragma unroll 2
    for (int i = threadIdx.x; i < kg_count * 32; i += blockDim.x) {
      const int kg = i >> 5, n4 = (i & 31) * 4;
      const uint8_t* src = src0 + (long)kg * 4 * N + n4;
      const uint32_t r0 = *reinterpret_cast<const uint32_t*>(src);
      const uint32_t r1 = *reinterpret_cast<const uint32_t*>(src + N);
      const uint32_t r2 = *reinterpret_cast<const uint32_t*>(src + 2L * N);
      const uint32_t r3 = *reinterpret_cast<const uint32_t*>(src + 3L * N);
      // column n4 + t: byte t of each row, K block j in byte j
      const uint32_t lo01 = __byte_perm(r0, r1, 0x5140), hi01 = __byte_perm(r0, r1, 0x7362);
      const uint32_t lo23 = __byte_perm(r2, r3, 0x5140), hi23 = __byte_perm(r2, r3, 0x7362);
      uint32_t* blk = blks + kg * 128;
      blk[sf_block_offset(n4 + 0, 0) / 4] = __byte_perm(lo01, lo23, 0x5410);
      blk[sf_block_offset(n4 + 1, 0) / 4] = __byte_perm(lo01, lo23, 0x7632);
      blk[sf_block_offset(n4 + 2, 0) / 4] = __byte_perm(hi01, hi23, 0x5410);
      blk[sf_block_offset(n4 + 3, 0) / 4] = __byte_perm(hi01, hi23, 0x7632);
    }
    __syncthreads();
    for (int i = threadIdx.x; i < kg_count * 32; i += blockDim.x) {
      const int kg = i >> 5, l = i & 31;
      reinterpret_cast<uint4*>(out + tiled_block(b, nb, kg, nbs, kg_count, g, s, slot))[l] =
          reinterpret_cast<const uint4*>(blks + kg * 128)[l];
    }
  }
}

//   tile_scales_rows_blocks_kernel: one CTA of 256 threads per (b, 128 N):
//   the 128 rows' kb_count scale bytes are one contiguous run (16-byte
//   copies into shared memory), then every K group's block is written out.
__global__ void __launch_bounds__(256) tile_scales_rows_blocks_kernel(const uint8_t* __restrict__ sf, int batch,
                                                                      int N, int kb_count, uint8_t* __restrict__ out,
                                                                      int g, int s, int slot) {
  extern __shared__ __align__(16) uint8_t rows_s[];  // [128][kb_count]
  const int kg_count = kb_count / 4, nbs = N / 128;
  const long nrun = (long)batch * nbs;
  const int run16 = 128 * kb_count / 16;
  for (long bi = blockIdx.x; bi < nrun; bi += gridDim.x) {
    const int nb = (int)(bi % nbs);
    const long b = bi / nbs;
    const uint4* src = reinterpret_cast<const uint4*>(sf + (b * N + (long)nb * 128) * kb_count);
    __syncthreads();  // the previous run is written out
    for (int i = threadIdx.x; i < run16; i += blockDim.x) reinterpret_cast<uint4*>(rows_s)[i] = src[i];
    __syncthreads();
    // piece l of K group kg: the words of rows l, l + 32, l + 64, l + 96
    for (int i = threadIdx.x; i < kg_count * 32; i += blockDim.x) {
      const int kg = i / 32, l = i % 32;
      uint4 v;
      v.x = *reinterpret_cast<const uint32_t*>(rows_s + (l)*kb_count + kg * 4);
      v.y = *reinterpret_cast<const uint32_t*>(rows_s + (l + 32) * kb_count + kg * 4);
      v.z = *reinterpret_cast<const uint32_t*>(rows_s + (l + 64) * kb_count + kg * 4);
      v.w = *reinterpret_cast<const uint32_t*>(rows_s + (l + 96) * kb_count + kg * 4);
      reinterpret_cast<uint4*>(out + tiled_block(b, nb, kg, nbs, kg_count, g, s, slot))[l] = v;
    }
  }
}

// Scales of a K-major activation operand, in padded-row order, tiled like
// the weights': padded row p takes the scales of row src(p) of `sf`
// [rows][kb_count] (the token of p when `pad_perm` is given, else p itself;
// a padding row gets scale code 0, its codes being zero), into
// [used rows / 128][kb_count / 4][512 B] for the rows in use.
__global__ void tile_row_scales_kernel(const uint8_t* __restrict__ sf, int kb_count,
                                       const int32_t* __restrict__ pad_perm, int k,
                                       const int32_t* __restrict__ rows_used, uint8_t* __restrict__ out) {
  const int kg_count = kb_count / 4;
  const long n_words = (long)(*rows_used) * kg_count;
  for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < n_words; i += (long)gridDim.x * blockDim.x) {
    const int kg = (int)(i % kg_count);
    const long p = i / kg_count;
    long src = p;
    if (pad_perm) {
      const int f = pad_perm[p];
      src = f >= 0 ? f / k : -1;
    }
    const uint32_t w = src >= 0 ? *reinterpret_cast<const uint32_t*>(sf + src * kb_count + (long)kg * 4) : 0u;
    uint8_t* blk = out + ((p / 128) * kg_count + kg) * 512;
    *reinterpret_cast<uint32_t*>(blk + sf_block_offset((int)(p & 127), 0)) = w;
  }
}

// Quantise bf16 [rows_cap, C] along the rows (blocks of 32 rows) for the rows
// in use (header word), codes [rows, C] and tiled scales
// [rows/128][C/128][512 B] (scale of (row block, column) at
// sf_block_offset(column % 128, (row / 32) % 4)).
__global__ void quant_rows_tiled_kernel(const __nv_bfloat16* __restrict__ src, const int32_t* __restrict__ rows_used,
                                        int C, uint8_t* __restrict__ q, uint8_t* __restrict__ sf) {
  // two columns a thread: four-byte loads, a warp reads 128 bytes of a row
  const int rows = *rows_used;
  const int C2 = C / 2;
  const long n = (long)(rows / 32) * C2;
  for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < n; i += (long)gridDim.x * blockDim.x) {
    const int c = 2 * (int)(i % C2);
    const int rb = (int)(i / C2);
    const long base = (long)rb * 32 * C + c;
    float v0[32], v1[32];
    float a0 = 0.0f, a1 = 0.0f;
#pragma unroll
    for (int r = 0; r < 32; ++r) {
      const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(src + base + (long)r * C));
      v0[r] = x.x;
      v1[r] = x.y;
      a0 = fmaxf(a0, fabsf(x.x));
      a1 = fmaxf(a1, fabsf(x.y));
    }
    const int X0 = block_exponent(a0), X1 = block_exponent(a1);
    const float i0 = exp2_int(-X0), i1 = exp2_int(-X1);
#pragma unroll
    for (int r = 0; r < 32; ++r)
      *reinterpret_cast<uint16_t*>(q + base + (long)r * C) = cvt_e4m3x2(v0[r] * i0, v1[r] * i1);
    uint8_t* blk = sf + ((long)(rb / 4) * (C / 128) + c / 128) * 512;
    blk[sf_block_offset(c & 127, rb & 3)] = (uint8_t)(X0 + 127);
    blk[sf_block_offset((c + 1) & 127, rb & 3)] = (uint8_t)(X1 + 127);
  }
}

// The same quantisation of token rows gathered in padded-row order: padded
// row p is row pad_perm[p] / k of src [T, C] (zeros for a padding row).  A
// CTA of 256 threads takes a tile of 32 padded rows x 512 columns, two
// columns a thread: the 32 source row offsets go to shared memory first,
// then each thread issues the 32 four-byte loads of its column pair at once
// (a padding row reads row 0 and is zeroed), so each source row is read in
// 1 KB runs and the token-sorted bf16 rows are never stored.
__global__ void __launch_bounds__(256) quant_rows_gather_kernel(const __nv_bfloat16* __restrict__ src,
                                                                const int32_t* __restrict__ rows_used, int C,
                                                                const int32_t* __restrict__ pad_perm, int k,
                                                                uint8_t* __restrict__ q, uint8_t* __restrict__ sf) {
  __shared__ long off[32];
  const int rbs = *rows_used / 32;
  const int cch = (C + 511) / 512;
  const long ntiles = (long)rbs * cch;
  for (long t = blockIdx.x; t < ntiles; t += gridDim.x) {
    const int rb = (int)(t / cch);
    const int c = (int)(t % cch) * 512 + 2 * threadIdx.x;
    __syncthreads();  // the previous tile is done with off[]
    if (threadIdx.x < 32) {
      const int f = pad_perm[(long)rb * 32 + threadIdx.x];
      off[threadIdx.x] = f >= 0 ? (long)(f / k) * C : -1;
    }
    __syncthreads();
    if (c >= C) continue;
    float v0[32], v1[32];
#pragma unroll
    for (int r = 0; r < 32; ++r) {
      const long o = off[r];
      const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(src + (o < 0 ? 0 : o) + c));
      v0[r] = o < 0 ? 0.0f : x.x;
      v1[r] = o < 0 ? 0.0f : x.y;
    }
    float a0 = 0.0f, a1 = 0.0f;
#pragma unroll
    for (int r = 0; r < 32; ++r) {
      a0 = fmaxf(a0, fabsf(v0[r]));
      a1 = fmaxf(a1, fabsf(v1[r]));
    }
    const int X0 = block_exponent(a0), X1 = block_exponent(a1);
    const float i0 = exp2_int(-X0), i1 = exp2_int(-X1);
    const long base = (long)rb * 32 * C + c;
#pragma unroll
    for (int r = 0; r < 32; ++r) {
      const uint16_t pr = cvt_e4m3x2(v0[r] * i0, v1[r] * i1);
      *reinterpret_cast<uint16_t*>(q + base + (long)r * C) = pr;
    }
    uint8_t* blk = sf + ((long)(rb / 4) * (C / 128) + c / 128) * 512;
    blk[sf_block_offset(c & 127, rb & 3)] = (uint8_t)(X0 + 127);
    blk[sf_block_offset((c + 1) & 127, rb & 3)] = (uint8_t)(X1 + 127);
  }
}

}  // namespace

cudaError_t launch_tile_scales(const uint8_t* sf, int batch, int kb_count, int N, uint8_t* out, cudaStream_t st,
                               int g, int s, int slot) {
  if (g < 1 || s < g || slot + g > s || (N / 128) % g) return cudaErrorInvalidValue;
  const size_t run = (size_t)(kb_count / 4) * 512;
  if (run <= 48 * 1024 && (reinterpret_cast<uintptr_t>(sf) & 3) == 0) {
    long grid = (long)batch * (N / 128);
    const long cap = (long)device_sm_count() * 8;
    if (grid > cap) grid = cap;
    tile_scales_run_kernel<<<(int)(grid < 1 ? 1 : grid), 256, run, st>>>(sf, batch, kb_count, N, out, g, s, slot);
    return cudaGetLastError();
  }
  const long blocks = (long)batch * (N / 128) * (kb_count / 4);
  long grid = blocks;
  const long cap = (long)device_sm_count() * 16;
  if (grid > cap) grid = cap;
  tile_scales_blocks_kernel<<<(int)(grid < 1 ? 1 : grid), 128, 0, st>>>(sf, batch, kb_count, N, out, g, s, slot);
  return cudaGetLastError();
}

cudaError_t launch_tile_scales_rows(const uint8_t* sf, int batch, int N, int kb_count, uint8_t* out,
                                    cudaStream_t st, int g, int s, int slot) {
  if (g < 1 || s < g || slot + g > s || (N / 128) % g) return cudaErrorInvalidValue;
  const size_t run = (size_t)128 * kb_count;
  if (run <= 48 * 1024 && (reinterpret_cast<uintptr_t>(sf) & 15) == 0) {
    long grid = (long)batch * (N / 128);
    const long cap = (long)device_sm_count() * 8;
    if (grid > cap) grid = cap;
    tile_scales_rows_blocks_kernel<<<(int)(grid < 1 ? 1 : grid), 256, run, st>>>(sf, batch, N, kb_count, out, g, s,
                                                                               slot);
    return cudaGetLastError();
  }
  const long words = (long)batch * N * (kb_count / 4);
  long grid = (words + 255) / 256;
  const long cap = (long)device_sm_count() * 32;
  if (grid > cap) grid = cap;
  tile_scales_rows_kernel<<<(int)(grid < 1 ? 1 : grid), 256, 0, st>>>(sf, batch, N, kb_count, out, g, s, slot);
  return cudaGetLastError();
}

cudaError_t launch_tile_row_scales(const uint8_t* sf, int kb_count, const int32_t* pad_perm, int k,
                                   const int32_t* rows_used, long rows_cap, uint8_t* out, cudaStream_t st) {
  const long words = rows_cap * (kb_count / 4);
  long grid = (words + 255) / 256;
  const long cap = (long)device_sm_count() * 32;
  if (grid > cap) grid = cap;
  tile_row_scales_kernel<<<(int)(grid < 1 ? 1 : grid), 256, 0, st>>>(sf, kb_count, pad_perm, k, rows_used, out);
  return cudaGetLastError();
}

cudaError_t launch_quant_rows_gather(const __nv_bfloat16* src, const int32_t* rows_used, long rows_cap, int C,
                                     const int32_t* pad_perm, int k, uint8_t* q, uint8_t* sf, cudaStream_t st) {
  const long tiles = (rows_cap / 32) * ((C + 511) / 512);
  long grid = tiles;
  const long cap = (long)device_sm_count() * 8;
  if (grid > cap) grid = cap;
  quant_rows_gather_kernel<<<(int)(grid < 1 ? 1 : grid), 256, 0, st>>>(src, rows_used, C, pad_perm, k, q, sf);
  return cudaGetLastError();
}

cudaError_t launch_quant_rows_tiled(const __nv_bfloat16* src, const int32_t* rows_used, long rows_cap, int C,
                                    uint8_t* q, uint8_t* sf, cudaStream_t st) {
  const long n = (rows_cap / 32) * (C / 2);
  long grid = (n + 255) / 256;
  const long cap = (long)device_sm_count() * 32;
  if (grid > cap) grid = cap;
  quant_rows_tiled_kernel<<<(int)(grid < 1 ? 1 : grid), 256, 0, st>>>(src, rows_used, C, q, sf);
  return cudaGetLastError();
}

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

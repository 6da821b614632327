// HBM-bound kernels around the grouped GEMMs:
//   combine     out[t] = sum_j s[t,j] * y[t*k+j]   (f32, increasing j, one rounding)
//               -- the forward combine, and with s = 1 the backward's dX combine
//               ("Cursor Open-Sources Mixture-of-Kittens (MoK)", "Three design
//               decisions that matter", communication-direction paragraph:
//               push combine / push reverse-dispatch; deterministic fixed
//               order per the paragraph after that list)
//   ds_reduce   dL/ds[f] = sum over the N tiles of the SwiGLU-backward epilogue's
//               per-tile partial dot products, in increasing tile order
//   gather_rows standalone dispatch copy xg[padded row] = x[token]
//   replay_copy bounded-memory backward: the forward context's last ring
//               slots of [h|u] back to their routed rows
// Each thread moves 16-byte vectors; consecutive threads take consecutive
// vectors of a row, so every warp access is coalesced.
#include <algorithm>

#include "mok_internal.cuh"

namespace mok {

namespace {

__device__ __forceinline__ void unpack8(const uint4& v, float (&o)[8]) {
  const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(p[i]);
    o[2 * i] = f.x;
    o[2 * i + 1] = f.y;
  }
}

__device__ __forceinline__ uint4 pack8(const float (&a)[8]) {
  uint4 v;
  uint32_t* w = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat162 p = __floats2bfloat162_rn(a[2 * i], a[2 * i + 1]);
    w[i] = *reinterpret_cast<uint32_t*>(&p);
  }
  return v;
}

template <int KMAX>
__global__ void __launch_bounds__(256) combine_kernel(int T, int H, int k, const int32_t* __restrict__ pad_inv,
                                                      const __nv_bfloat16* __restrict__ yk,
                                                      const float* __restrict__ scores,
                                                      __nv_bfloat16* __restrict__ out) {
  const int hv = H / 8;
  const long n = (long)T * hv;
  for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < n; i += (long)gridDim.x * blockDim.x) {
    const int t = (int)(i / hv);
    const int c = (int)(i - (long)t * hv);
    uint4 v[KMAX];
    float w[KMAX];
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      if (j < k) {
        const long f = (long)t * k + j;
        const bool ok = pad_inv[f] >= 0;
        w[j] = ok ? (scores ? scores[f] : 1.0f) : 0.0f;
        v[j] = ok ? __ldcs(reinterpret_cast<const uint4*>(yk + f * H) + c) : make_uint4(0, 0, 0, 0);
      }
    }
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.0f;
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      if (j < k) {
        float y[8];
        unpack8(v[j], y);
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = fmaf(w[j], y[e], acc[e]);
      }
    }
    reinterpret_cast<uint4*>(out + (long)t * H)[c] = pack8(acc);
  }
}

__global__ void ds_reduce_kernel(int R, int nparts, const int32_t* __restrict__ pad_inv,
                                 const float* __restrict__ dsp, float* __restrict__ ds) {
  const int f = blockIdx.x * blockDim.x + threadIdx.x;
  if (f >= R) return;
  const int p = pad_inv[f];
  float acc = 0.0f;
  if (p >= 0)
    for (int n = 0; n < nparts; ++n) acc += dsp[(long)p * nparts + n];
  ds[f] = acc;
}

__global__ void __launch_bounds__(256) gather_rows_kernel(int T, int H, int k, const int32_t* __restrict__ hdr,
                                                          const int32_t* __restrict__ pad_perm,
                                                          const __nv_bfloat16* __restrict__ x,
                                                          __nv_bfloat16* __restrict__ xg,
                                                          const int32_t* __restrict__ skip) {
  if (skip && *skip) return;  // the copy is already there
  const int rows = hdr[kHdrPaddedRows];
  const int hv = H / 8;
  const long n = (long)rows * hv;
  for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < n; i += (long)gridDim.x * blockDim.x) {
    const int p = (int)(i / hv);
    const int c = (int)(i - (long)p * hv);
    const int f = pad_perm[p];
    uint4 v = make_uint4(0, 0, 0, 0);
    if (f >= 0) v = __ldg(reinterpret_cast<const uint4*>(x + (long)(f / k) * H) + c);
    __stcs(reinterpret_cast<uint4*>(xg + (long)p * H) + c, v);
  }
}

// Token-sorted copy of E4M3 code rows (MXFP8 x or dout quantised along H):
// dst[padded row] = codes[token] (zeros for padding rows), 16 bytes a thread.
__global__ void __launch_bounds__(256) gather_code_rows_kernel(int H, int k, const int32_t* __restrict__ hdr,
                                                               const int32_t* __restrict__ pad_perm,
                                                               const uint8_t* __restrict__ codes,
                                                               uint8_t* __restrict__ dst) {
  const int rows = hdr[kHdrPaddedRows];
  const int hv = H / 16;
  const long n = (long)rows * hv;
  for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < n; i += (long)gridDim.x * blockDim.x) {
    const int p = (int)(i / hv);
    const int c = (int)(i - (long)p * hv);
    const int f = pad_perm[p];
    uint4 v = make_uint4(0, 0, 0, 0);
    if (f >= 0) v = __ldg(reinterpret_cast<const uint4*>(codes + (long)(f / k) * H) + c);
    __stcs(reinterpret_cast<uint4*>(dst + (long)p * H) + c, v);
  }
}

// Bounded-memory backward: the [h|u] rows of the last `slots` minibatches,
// kept by the forward in ring-slot order, copied to their routed-row places
// in dh|du (the dA' epilogue then reads and overwrites them in place).
__global__ void __launch_bounds__(256) replay_copy_kernel(int I, int M, int slots, const int32_t* __restrict__ hdr,
                                                          const __nv_bfloat16* __restrict__ ctx_ring,
                                                          __nv_bfloat16* __restrict__ dhu) {
  const int used = hdr[kHdrPaddedRows];
  const int nb = (used + M - 1) / M;
  const long row0 = (long)max(nb - slots, 0) * M;
  const int vec = 2 * I / 8;
  const long n = (used - row0) * vec;
  for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < n; i += (long)gridDim.x * blockDim.x) {
    const long r = row0 + i / vec;
    const int c = (int)(i % vec);
    const long mb = r / M;
    const long src = (mb % slots) * M + (r - mb * M);
    reinterpret_cast<uint4*>(dhu + r * 2 * I)[c] = reinterpret_cast<const uint4*>(ctx_ring + src * 2 * I)[c];
  }
}

int grid_for(long items, int threads) {
  const int sms = device_sm_count();
  long blocks = (items + threads - 1) / threads;
  const long cap = (long)sms * 16;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return (int)blocks;
}

}  // namespace

cudaError_t launch_replay_copy(const mok_shape& s, const WsLayout& L, const uint8_t* ws,
                               const __nv_bfloat16* ctx_ring, __nv_bfloat16* dhu, cudaStream_t st) {
  const long items = (long)std::min<int64_t>((int64_t)L.ring_slots * L.minibatch_rows, L.pad_capacity) * (2 * s.I / 8);
  replay_copy_kernel<<<grid_for(items, 256), 256, 0, st>>>(s.I, L.minibatch_rows, L.ring_slots,
                                                           reinterpret_cast<const int32_t*>(ws + L.header), ctx_ring,
                                                           dhu);
  return cudaGetLastError();
}

cudaError_t launch_combine(const mok_shape& s, const WsLayout& L, const uint8_t* ws, const __nv_bfloat16* yk,
                           const float* scores, __nv_bfloat16* out, cudaStream_t st) {
  const int32_t* pad_inv = reinterpret_cast<const int32_t*>(ws + L.pad_inv);
  const long items = (long)s.T * (s.H / 8);
  const int grid = grid_for(items, 256);
  if (s.k <= 2)
    combine_kernel<2><<<grid, 256, 0, st>>>(s.T, s.H, s.k, pad_inv, yk, scores, out);
  else if (s.k <= 4)
    combine_kernel<4><<<grid, 256, 0, st>>>(s.T, s.H, s.k, pad_inv, yk, scores, out);
  else if (s.k <= 8)
    combine_kernel<8><<<grid, 256, 0, st>>>(s.T, s.H, s.k, pad_inv, yk, scores, out);
  else if (s.k <= 16)
    combine_kernel<16><<<grid, 256, 0, st>>>(s.T, s.H, s.k, pad_inv, yk, scores, out);
  else
    combine_kernel<32><<<grid, 256, 0, st>>>(s.T, s.H, s.k, pad_inv, yk, scores, out);
  return cudaGetLastError();
}

cudaError_t launch_ds_reduce(const mok_shape& s, const WsLayout& L, const uint8_t* ws, float* ds, int n_parts,
                             cudaStream_t st) {
  const int R = s.T * s.k;
  ds_reduce_kernel<<<(R + 255) / 256, 256, 0, st>>>(R, n_parts, reinterpret_cast<const int32_t*>(ws + L.pad_inv),
                                                   reinterpret_cast<const float*>(ws + L.dsp), ds);
  return cudaGetLastError();
}

cudaError_t launch_gather_rows(const mok_shape& s, const WsLayout& L, const uint8_t* ws, const __nv_bfloat16* x,
                               __nv_bfloat16* xg, cudaStream_t st, const int32_t* skip) {
  const long items = L.pad_capacity * (s.H / 8);
  gather_rows_kernel<<<grid_for(items, 256), 256, 0, st>>>(
      s.T, s.H, s.k, reinterpret_cast<const int32_t*>(ws + L.header),
      reinterpret_cast<const int32_t*>(ws + L.pad_perm), x, xg, skip);
  return cudaGetLastError();
}

cudaError_t launch_gather_code_rows(const mok_shape& s, const WsLayout& L, const uint8_t* ws, const uint8_t* codes,
                                    uint8_t* dst, cudaStream_t st) {
  const long items = L.pad_capacity * (s.H / 16);
  gather_code_rows_kernel<<<grid_for(items, 256), 256, 0, st>>>(
      s.H, s.k, reinterpret_cast<const int32_t*>(ws + L.header), reinterpret_cast<const int32_t*>(ws + L.pad_perm),
      codes, dst);
  return cudaGetLastError();
}

}  // namespace mok

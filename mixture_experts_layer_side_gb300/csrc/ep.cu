// Expert parallelism (EP): the layer's experts split over G ranks, tokens
// split by data parallelism, one exchange of routed rows each way per pass
// ("Cursor Open-Sources Mixture-of-Kittens (MoK)", "Three design decisions
// that matter", communication-direction paragraph: dispatch, combine and
// their two reverse directions all driven by the one schedule table;
// "Results": the layer measured at EP 64).
//
// What this file holds:
//   * the expert partition (contiguous blocks of experts per rank);
//   * the exchange plan, on the host: from each source rank's per-expert
//     counts (the schedule's histogram, exchanged between ranks) the rows each
//     rank sends to and receives from every other rank, and the local expert
//     of every received row in arrival order -- the per-(source rank,
//     destination expert) histogram and its scans;
//   * three source-side kernels around the exchange: pack the routed rows in
//     the schedule's expert-sorted order (which is destination-major, since
//     experts are partitioned in contiguous blocks), combine the returned
//     expert outputs back to token order through the inverse permutation, and
//     scatter the returned per-row score gradients back to [T, k].
//
// The receiving rank runs the ordinary layer calls on its received rows with
// k = 1, each row routed to its local expert with score 1 (forward) or its
// score (backward).  Received rows arrive source-major and, within a source,
// in the source's sorted order; the receiver's stable schedule therefore
// orders each expert's rows by (source rank, source flat index), which is
// ascending global flat index when token t of rank g is global token
// g*T + t -- the order one GPU holding every token would use.  Expert
// outputs, weight gradients and score gradients are then bitwise those of
// the single-GPU layer.
#include <string.h>

#include "mok_internal.cuh"

namespace mok {
namespace {

__device__ __forceinline__ void unpack8f(const uint4& v, float (&o)[8]) {
  const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(p[i]);
    o[2 * i] = f.x;
    o[2 * i + 1] = f.y;
  }
}

__device__ __forceinline__ uint4 pack8f(const float (&a)[8]) {
  uint4 v;
  uint32_t* w = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat162 p = __floats2bfloat162_rn(a[2 * i], a[2 * i + 1]);
    w[i] = *reinterpret_cast<uint32_t*>(&p);
  }
  return v;
}

// rows[r] = x[perm[r] / k] for the routed rows r < offsets[E] (rows past it,
// the ids outside [0, E), are not written); s_rows[r] = s[perm[r]].
__global__ void __launch_bounds__(256) ep_pack_kernel(int H, int k, int E, const int32_t* __restrict__ offsets,
                                                      const int32_t* __restrict__ perm,
                                                      const __nv_bfloat16* __restrict__ x,
                                                      const float* __restrict__ s, __nv_bfloat16* __restrict__ rows,
                                                      float* __restrict__ s_rows) {
  const int n_rows = offsets[E];
  const int hv = H / 8;
  const long n = (long)n_rows * hv;
  for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < n; i += (long)gridDim.x * blockDim.x) {
    const int r = (int)(i / hv);
    const int c = (int)(i - (long)r * hv);
    const int f = perm[r];
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(x + (long)(f / k) * H) + c);
    __stcs(reinterpret_cast<uint4*>(rows + (long)r * H) + c, v);
    if (s_rows && c == 0) s_rows[r] = s[f];
  }
}

// out[t] = sum_j w[t,j] * rows[inv_perm[t*k+j]] in f32, increasing j, one
// rounding (w = scores, or 1 with no scores); a row routed nowhere adds 0.
// The same fused multiply-adds in the same order as the layer's combine.
template <int KMAX>
__global__ void __launch_bounds__(256) ep_combine_kernel(int T, int H, int k, const int32_t* __restrict__ inv_perm,
                                                         const __nv_bfloat16* __restrict__ rows,
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
        const int r = inv_perm[f];
        w[j] = r >= 0 ? (scores ? scores[f] : 1.0f) : 0.0f;
        v[j] = r >= 0 ? __ldcs(reinterpret_cast<const uint4*>(rows + (long)r * H) + c) : make_uint4(0, 0, 0, 0);
      }
    }
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.0f;
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      if (j < k) {
        float y[8];
        unpack8f(v[j], y);
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = fmaf(w[j], y[e], acc[e]);
      }
    }
    reinterpret_cast<uint4*>(out + (long)t * H)[c] = pack8f(acc);
  }
}

// out[f] = vals[inv_perm[f]], or 0 for a row routed nowhere.
__global__ void ep_unsort_kernel(int R, const int32_t* __restrict__ inv_perm, const float* __restrict__ vals,
                                 float* __restrict__ out) {
  const int f = blockIdx.x * blockDim.x + threadIdx.x;
  if (f >= R) return;
  const int r = inv_perm[f];
  out[f] = r >= 0 ? vals[r] : 0.0f;
}

int ep_grid(long items) {
  const int sms = device_sm_count();
  long blocks = (items + 255) / 256;
  const long cap = (long)(sms > 0 ? sms : 1) * 16;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return (int)blocks;
}

}  // namespace

cudaError_t launch_ep_pack(const mok_shape& s, const WsLayout& L, const uint8_t* ws, const __nv_bfloat16* x,
                           const float* scores, __nv_bfloat16* rows, float* s_rows, cudaStream_t st) {
  const long items = (long)s.T * s.k * (s.H / 8);
  ep_pack_kernel<<<ep_grid(items), 256, 0, st>>>(s.H, s.k, s.E, reinterpret_cast<const int32_t*>(ws + L.offsets),
                                                 reinterpret_cast<const int32_t*>(ws + L.perm), x, scores, rows,
                                                 s_rows);
  return cudaGetLastError();
}

cudaError_t launch_ep_combine(const mok_shape& s, const WsLayout& L, const uint8_t* ws, const __nv_bfloat16* rows,
                              const float* scores, __nv_bfloat16* out, cudaStream_t st) {
  const int32_t* inv = reinterpret_cast<const int32_t*>(ws + L.inv_perm);
  const int grid = ep_grid((long)s.T * (s.H / 8));
  if (s.k <= 2)
    ep_combine_kernel<2><<<grid, 256, 0, st>>>(s.T, s.H, s.k, inv, rows, scores, out);
  else if (s.k <= 4)
    ep_combine_kernel<4><<<grid, 256, 0, st>>>(s.T, s.H, s.k, inv, rows, scores, out);
  else if (s.k <= 8)
    ep_combine_kernel<8><<<grid, 256, 0, st>>>(s.T, s.H, s.k, inv, rows, scores, out);
  else if (s.k <= 16)
    ep_combine_kernel<16><<<grid, 256, 0, st>>>(s.T, s.H, s.k, inv, rows, scores, out);
  else
    ep_combine_kernel<32><<<grid, 256, 0, st>>>(s.T, s.H, s.k, inv, rows, scores, out);
  return cudaGetLastError();
}

cudaError_t launch_ep_unsort(const mok_shape& s, const WsLayout& L, const uint8_t* ws, const float* vals, float* out,
                             cudaStream_t st) {
  const int R = s.T * s.k;
  ep_unsort_kernel<<<(R + 255) / 256, 256, 0, st>>>(R, reinterpret_cast<const int32_t*>(ws + L.inv_perm), vals, out);
  return cudaGetLastError();
}

}  // namespace mok

// ---------------------------------------------------------------------------
// Host-only part of the exchange plan (no device work; callable without a GPU)
// ---------------------------------------------------------------------------
extern "C" int32_t mok_ep_first_expert(int32_t E, int32_t G, int32_t g) {
  if (E < 1 || G < 1 || G > E || g < 0 || g > G) return -1;
  const int32_t base = E / G, rem = E % G;
  return g * base + (g < rem ? g : rem);
}

extern "C" mok_status mok_ep_plan(int32_t E, int32_t G, int32_t rank, const int32_t* local_counts,
                                  const int32_t* recv_counts, int64_t* send_rows, int64_t* recv_rows,
                                  int32_t* recv_expert, int64_t recv_capacity, int64_t* n_recv) {
  if (E < 1 || G < 1 || G > E || rank < 0 || rank >= G) return MOK_ERR_INVALID_ARG;
  if (!local_counts || !recv_counts || !send_rows || !recv_rows || !n_recv) return MOK_ERR_INVALID_ARG;
  if (recv_capacity < 0) return MOK_ERR_INVALID_ARG;
  for (int32_t e = 0; e < E; ++e)
    if (local_counts[e] < 0) return MOK_ERR_INVALID_ARG;
  // rows this rank sends: its sorted rows are contiguous per destination
  for (int32_t g = 0; g < G; ++g) {
    int64_t n = 0;
    for (int32_t e = mok_ep_first_expert(E, G, g); e < mok_ep_first_expert(E, G, g + 1); ++e) n += local_counts[e];
    send_rows[g] = n;
  }
  // rows it receives: the [G, E_rank] histogram of (source rank, local expert)
  const int32_t El = mok_ep_first_expert(E, G, rank + 1) - mok_ep_first_expert(E, G, rank);
  int64_t total = 0;
  for (int32_t src = 0; src < G; ++src) {
    int64_t n = 0;
    for (int32_t e = 0; e < El; ++e) {
      const int32_t c = recv_counts[(int64_t)src * El + e];
      if (c < 0) return MOK_ERR_INVALID_ARG;
      n += c;
    }
    recv_rows[src] = n;
    total += n;
  }
  *n_recv = total;
  if (!recv_expert) return MOK_OK;
  if (total > recv_capacity) return MOK_ERR_UNSUPPORTED;
  // local expert of each received row, in arrival order: source-major, and
  // within a source in its expert-sorted order
  int64_t pos = 0;
  for (int32_t src = 0; src < G; ++src)
    for (int32_t e = 0; e < El; ++e)
      for (int32_t i = 0; i < recv_counts[(int64_t)src * El + e]; ++i) recv_expert[pos++] = e;
  return MOK_OK;
}

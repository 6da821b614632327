// Device-side schedule: expert histogram, exclusive scan, stable counting-sort
// permutation, 128-row padded offsets, tile table and inverse permutations.
//
// One schedule table serves forward dispatch/combine and the backward's
// reverse combine/dispatch ("Cursor Open-Sources Mixture-of-Kittens (MoK)",
// "Three design decisions that matter", communication-direction paragraph),
// and it is built on the GPU without any host readback (same section,
// ring-token-buffer paragraph: the CPU is taken out of the loop).
//
// Three kernels, all integer work, so the result is exact and independent
// of scheduling:
//   1. sched_count: per chunk of 1024 routed rows, a per-expert histogram.
//   2. sched_scan : one block; per expert an exclusive scan over chunks (the
//                   chunk's base position), then the exclusive scans of the
//                   counts and of the 128-padded counts, the tile table and
//                   the -1 markers of padding rows.
//   3. sched_place: per chunk, one warp walks its rows in increasing f,
//                   32 at a time; __match_any_sync groups equal experts and
//                   the rank inside the group is the count of lower lanes,
//                   so positions are assigned in increasing f (stable).
#include "mok_internal.cuh"

namespace mok {

namespace {

constexpr int kCountThreads = 256;

__global__ void sched_count(const int32_t* __restrict__ idx, int R, int E, int32_t* __restrict__ chunk_hist,
                            int32_t* __restrict__ hdr) {
  extern __shared__ int32_t hist[];
  const int chunk = blockIdx.x;
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  const int f0 = chunk * kSchedChunk;
  const int f1 = min(f0 + kSchedChunk, R);
  bool bad = false;
  for (int f = f0 + threadIdx.x; f < f1; f += blockDim.x) {
    const int e = idx[f];
    if (e >= 0 && e < E)
      atomicAdd(&hist[e], 1);
    else
      bad = true;
  }
  if (bad) atomicOr(&hdr[kHdrError], MOK_ERRBIT_BAD_INDEX);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) chunk_hist[(size_t)chunk * E + e] = hist[e];
}

// Exclusive block scan of one value per thread (blockDim.x == 1024).
__device__ int block_exclusive_scan(int v, int* warp_tot, int* total_out) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += n;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = warp_tot[lane];
    int wi = w;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, wi, d);
      if (lane >= d) wi += n;
    }
    warp_tot[lane] = wi - w;  // exclusive prefix of warp totals
    if (lane == 31) *total_out = wi;
  }
  __syncthreads();
  const int r = warp_tot[warp] + incl - v;
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(1024) sched_scan(int E, int nchunks, const int32_t* __restrict__ chunk_hist,
                                                   int32_t* __restrict__ chunk_base, int32_t* __restrict__ counts,
                                                   int32_t* __restrict__ offsets, int32_t* __restrict__ poff,
                                                   int32_t* __restrict__ tile_expert, int32_t* __restrict__ pad_perm,
                                                   int32_t* __restrict__ hdr) {
  __shared__ int warp_tot[32];
  __shared__ int tot0, tot1;
  const int e = threadIdx.x;
  int cnt = 0;
  if (e < E) {
    // running sum over chunks; loads are independent of the sum, so unroll
    int c = 0;
    for (; c + 8 <= nchunks; c += 8) {
      int v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) v[u] = chunk_hist[(size_t)(c + u) * E + e];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        chunk_base[(size_t)(c + u) * E + e] = cnt;
        cnt += v[u];
      }
    }
    for (; c < nchunks; ++c) {
      const int v = chunk_hist[(size_t)c * E + e];
      chunk_base[(size_t)c * E + e] = cnt;
      cnt += v;
    }
  }
  const int padded = (cnt + kTileRows - 1) / kTileRows * kTileRows;
  const int off = block_exclusive_scan(e < E ? cnt : 0, warp_tot, &tot0);
  const int poffe = block_exclusive_scan(e < E ? padded : 0, warp_tot, &tot1);
  if (e < E) {
    counts[e] = cnt;
    offsets[e] = off;
    poff[e] = poffe;
    for (int t = poffe / kTileRows; t < (poffe + padded) / kTileRows; ++t) tile_expert[t] = e;
    for (int r = poffe + cnt; r < poffe + padded; ++r) pad_perm[r] = -1;
  }
  if (e == 0) {
    offsets[E] = tot0;
    poff[E] = tot1;
    hdr[kHdrPaddedRows] = tot1;
    hdr[kHdrTiles] = tot1 / kTileRows;
  }
}

// Each warp handles one chunk of kSchedChunk routed rows.
constexpr int kPlaceWarps = 4;

__global__ void __launch_bounds__(kPlaceWarps * 32)
    sched_place(const int32_t* __restrict__ idx, int R, int E, int nchunks, const int32_t* __restrict__ chunk_base,
                const int32_t* __restrict__ offsets, const int32_t* __restrict__ poff, int32_t* __restrict__ perm,
                int32_t* __restrict__ inv_perm, int32_t* __restrict__ pad_perm, int32_t* __restrict__ pad_inv) {
  extern __shared__ int32_t cursor_all[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int chunk = blockIdx.x * kPlaceWarps + warp;
  int32_t* cursor = cursor_all + warp * E;
  if (chunk < nchunks)
    for (int e = lane; e < E; e += 32) cursor[e] = chunk_base[(size_t)chunk * E + e];
  __syncwarp();
  if (chunk >= nchunks) return;
  const unsigned lt_mask = (1u << lane) - 1u;
  const int f0 = chunk * kSchedChunk;
  for (int it = 0; it < kSchedChunk / 32; ++it) {
    const int f = f0 + it * 32 + lane;
    int e = -1;
    if (f < R) {
      e = idx[f];
      if (e < 0 || e >= E) e = -1;
    }
    const unsigned grp = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(grp & lt_mask);
    int pos = 0;
    if (e >= 0) pos = cursor[e] + rank;
    __syncwarp();
    if (e >= 0 && rank == 0) cursor[e] += __popc(grp);
    __syncwarp();
    if (f < R) {
      if (e >= 0) {
        const int r = offsets[e] + pos;
        const int prow = poff[e] + pos;
        perm[r] = f;
        inv_perm[f] = r;
        pad_perm[prow] = f;
        pad_inv[f] = prow;
      } else {
        inv_perm[f] = -1;
        pad_inv[f] = -1;
      }
    }
  }
}

// Split of the row tiles (forward ring, dA', dX) between a CTA-pair launch
// and a single-CTA launch, every expert wholly in one of them (its weights
// then stream from DRAM in one launch only).  An expert with t >= min_pair
// padded tiles goes to the pairs, taken two at a time from its first tile
// (an odd last tile is a solo pair: one idle CTA for one tile in t + 1);
// the others run on single CTAs.  pair_m0[j] = 2 * (first tile of unit j)
// + solo, single_list[q] = tile, both in increasing tile order.  One block;
// integer work, exact.
__global__ void __launch_bounds__(1024) split_table_kernel(const int32_t* __restrict__ tile_expert,
                                                           const int32_t* __restrict__ poff, int32_t* __restrict__ hdr,
                                                           int32_t* __restrict__ pair_m0,
                                                           int32_t* __restrict__ single_list, int min_pair) {
  __shared__ int warp_tot[32];
  __shared__ int tot;
  const int U = hdr[kHdrTiles];
  int carry_p = 0, carry_s = 0;
  for (int base = 0; base < U; base += 1024) {
    const int m = base + threadIdx.x;
    int head = 0, solo = 0, single = 0;
    if (m < U) {
      const int e = tile_expert[m];
      const int first = poff[e] / kTileRows;
      const int t = (poff[e + 1] - poff[e]) / kTileRows;
      const int j = m - first;
      const bool paired = t >= min_pair;
      head = paired && !(j & 1);
      solo = head && j == t - 1;
      single = !paired;
    }
    const int pp = carry_p + block_exclusive_scan(head, warp_tot, &tot);
    const int np = tot;
    const int ps = carry_s + block_exclusive_scan(single, warp_tot, &tot);
    if (head) pair_m0[pp] = 2 * m + solo;
    if (single) single_list[ps] = m;
    carry_p += np;
    carry_s += tot;
  }
  if (threadIdx.x == 0) {
    hdr[kHdrPairs] = carry_p;
    hdr[kHdrSingles] = carry_s;
  }
}

}  // namespace

cudaError_t launch_schedule(const mok_shape& s, const WsLayout& L, uint8_t* ws, const int32_t* idx,
                            cudaStream_t st) {
  const int R = s.T * s.k, E = s.E;
  const int nchunks = (int)L.nchunks;
  int32_t* hdr = reinterpret_cast<int32_t*>(ws + L.header);
  auto P = [&](size_t off) { return reinterpret_cast<int32_t*>(ws + off); };
  cudaError_t err = cudaMemsetAsync(hdr, 0, kHeaderWords * sizeof(int32_t), st);
  if (err != cudaSuccess) return err;
  sched_count<<<nchunks, kCountThreads, E * sizeof(int32_t), st>>>(idx, R, E, P(L.chunk_hist), hdr);
  sched_scan<<<1, 1024, 0, st>>>(E, nchunks, P(L.chunk_hist), P(L.chunk_base), P(L.counts), P(L.offsets),
                                 P(L.padded_offsets), P(L.tile_expert), P(L.pad_perm), hdr);
  const int blocks = (nchunks + kPlaceWarps - 1) / kPlaceWarps;
  const size_t smem = (size_t)kPlaceWarps * E * sizeof(int32_t);
  sched_place<<<blocks, kPlaceWarps * 32, smem, st>>>(idx, R, E, nchunks, P(L.chunk_base), P(L.offsets),
                                                      P(L.padded_offsets), P(L.perm), P(L.inv_perm),
                                                      P(L.pad_perm), P(L.pad_inv));
  return cudaGetLastError();
}

cudaError_t launch_split_table(const WsLayout& L, uint8_t* ws, int min_pair_tiles, cudaStream_t st) {
  auto P = [&](size_t off) { return reinterpret_cast<int32_t*>(ws + off); };
  split_table_kernel<<<1, 1024, 0, st>>>(P(L.tile_expert), P(L.padded_offsets), P(L.header), P(L.pair_m0),
                                         P(L.pair_mb), min_pair_tiles);
  return cudaGetLastError();
}

}  // namespace mok

// ---------------------------------------------------------------------------
// Schedule without device allocation: the same three kernels, with their
// scratch (per-chunk histograms and their scans) in a static device array
// instead of the caller's workspace.  For callers that cannot allocate
// device memory (see mok_build_schedule_noalloc in mok.h).
// ---------------------------------------------------------------------------
#include <mutex>

namespace {

constexpr size_t kNoallocScratchBytes = MOK_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kNoallocMaxDevices = 64;
std::mutex g_noalloc_mu;
struct NoallocSlot {
  unsigned long long ctx_id;  // unique id of the context the address belongs to (0: none yet)
  void* addr;
};
NoallocSlot g_noalloc_slot[kNoallocMaxDevices] = {};

// Unique id of the current context (driver calls reached through the runtime,
// so the library needs no link to libcuda).  A context made after a
// cudaDeviceReset gets a new id, so a cached address of the old one is never
// reused.
typedef int (*CtxGetCurrentFn)(void**);
typedef int (*CtxGetIdFn)(void*, unsigned long long*);
bool current_context_id(unsigned long long* id) {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  void* ctx = nullptr;
  if (!get_current || !get_id || get_current(&ctx) != 0 || !ctx) return false;
  return get_id(ctx, id) == 0;
}

// Device address of the static scratch on the current device.  It is looked
// up with cudaGetSymbolAddress once per device and context, with that device
// current, and cached; host code must not use the symbol itself, which on
// the host only names a stand-in.
void* noalloc_scratch_address(int dev, cudaError_t* err) {
  *err = cudaSuccess;
  if (dev < 0 || dev >= kNoallocMaxDevices) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  // cudaSetDevice makes (or re-makes, after a reset) the device's primary
  // context current, so its id can be read
  *err = cudaSetDevice(dev);
  if (*err != cudaSuccess) return nullptr;
  unsigned long long id = 0;
  if (!current_context_id(&id)) {
    *err = cudaErrorDeviceUninitialized;
    return nullptr;
  }
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  NoallocSlot& slot = g_noalloc_slot[dev];
  if (slot.ctx_id != id || !slot.addr) {
    void* ptr = nullptr;
    *err = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (*err != cudaSuccess) return nullptr;
    slot.addr = ptr;
    slot.ctx_id = id;
  }
  return slot.addr;
}

template <typename... Params, typename... Args>
cudaError_t launch_on(cudaStream_t st, int grid, int block, size_t smem, void (*kernel)(Params...),
                      Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

}  // namespace

extern "C" mok_status mok_build_schedule_noalloc(const mok_shape* shape, const int32_t* topk_idx,
                                                 const mok_schedule_buffers* out, void* stream) {
  using namespace mok;
  if (!shape || !topk_idx || !out) return MOK_ERR_INVALID_ARG;
  if (!out->header || !out->counts || !out->offsets || !out->padded_offsets || !out->perm || !out->inv_perm ||
      !out->pad_perm || !out->pad_inv || !out->tile_expert)
    return MOK_ERR_INVALID_ARG;
  const mok_shape& s = *shape;
  if (s.T < 1 || s.k < 1 || s.E < 1) return MOK_ERR_INVALID_ARG;
  if (s.E > 1024 || s.k > 32 || (int64_t)s.T * s.k > (1 << 24)) return MOK_ERR_UNSUPPORTED;
  const int R = s.T * s.k, E = s.E;
  const int64_t nchunks = (R + kSchedChunk - 1) / kSchedChunk;
  const size_t need = 2 * (size_t)nchunks * E * sizeof(int32_t);
  if (need > kNoallocScratchBytes) return MOK_ERR_UNSUPPORTED;  // beyond the static scratch
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOK_ERR_CUDA;
  if (st) {  // the kernels use the current device's array: the stream must be on that device
    int sdev = -1;
    if (cudaStreamGetDevice(st, &sdev) != cudaSuccess) return MOK_ERR_CUDA;
    if (sdev != dev) return MOK_ERR_INVALID_ARG;
  }
  cudaError_t err = cudaSuccess;
  uint8_t* scratch = static_cast<uint8_t*>(noalloc_scratch_address(dev, &err));
  if (!scratch) return MOK_ERR_CUDA;
  int32_t* chunk_hist = reinterpret_cast<int32_t*>(scratch);
  int32_t* chunk_base = chunk_hist + nchunks * E;
  // the header starts at zero; the two scratch arrays are fully rewritten.
  // Each call reports its own launches' status (not an earlier, unrelated
  // error left in the runtime's last-error slot).
  if (cudaMemsetAsync(out->header, 0, kHeaderWords * sizeof(int32_t), st) != cudaSuccess) return MOK_ERR_CUDA;
  if (launch_on(st, (int)nchunks, kCountThreads, E * sizeof(int32_t), sched_count, topk_idx, R, E, chunk_hist,
                out->header) != cudaSuccess)
    return MOK_ERR_CUDA;
  if (launch_on(st, 1, 1024, 0, sched_scan, E, (int)nchunks, chunk_hist, chunk_base, out->counts, out->offsets,
                out->padded_offsets, out->tile_expert, out->pad_perm, out->header) != cudaSuccess)
    return MOK_ERR_CUDA;
  const int blocks = (int)((nchunks + kPlaceWarps - 1) / kPlaceWarps);
  if (launch_on(st, blocks, kPlaceWarps * 32, (size_t)kPlaceWarps * E * sizeof(int32_t), sched_place, topk_idx, R,
                E, (int)nchunks, chunk_base, out->offsets, out->padded_offsets, out->perm, out->inv_perm,
                out->pad_perm, out->pad_inv) != cudaSuccess)
    return MOK_ERR_CUDA;
  return MOK_OK;
}

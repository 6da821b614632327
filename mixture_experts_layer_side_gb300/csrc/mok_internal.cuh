// Definitions shared by the library's translation units (not part of the ABI).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/mok.h"

// Device error bits of the workspace error word (header word 0).
#define MOK_ERRBIT_BAD_INDEX 1
#define MOK_ERRBIT_TIMEOUT 2

namespace mok {

constexpr int kTileRows = 128;      // padded expert segments and GEMM M tile
constexpr int kSchedChunk = 1024;   // routed rows per schedule warp
constexpr int kHeaderWords = 64;    // int32 words of the workspace header
// header word indices
constexpr int kHdrError = 0;
constexpr int kHdrPaddedRows = 1;
constexpr int kHdrTiles = 2;
constexpr int kHdrAbort = 3;       // launch-wide abort word (cleared per call)
constexpr int kHdrPairs = 4;       // CTA-pair units of the split table (see launch_split_table)
constexpr int kHdrSingles = 11;    // single tiles of the split table (see launch_split_table)
// single-launch forward: completed schedule items (count, scan, place) and
// GEMM2 epilogue warps that stored their rows of y
constexpr int kHdrCountDone = 5;
constexpr int kHdrScanDone = 6;
constexpr int kHdrPlaceDone = 7;
constexpr int kHdrG2Done = 8;
constexpr int kHdrCombineNext = 9;  // next token of the single-launch forward's combine
// nonzero while the sorted buffer holds the token-sorted x of the last
// BF16 forward on this schedule (its backward then skips sorting x again);
// cleared by every schedule build and by forwards that do not sort x.  Past
// the words each call's counter reset clears ([kHdrAbort, kHdrCounters +
// kNumCounters)), so it lives from the forward to the backward.
constexpr int kHdrSortedX = 56;
constexpr int kHdrCounters = 16;    // [16, 48): per-launch dynamic tile counters
constexpr int kNumCounters = 32;
static_assert(kHdrSortedX >= kHdrCounters + kNumCounters && kHdrSortedX < kHeaderWords, "flag outside the reset words");

struct WsLayout {
  // schedule
  size_t header, counts, offsets, padded_offsets, perm, inv_perm, pad_perm, pad_inv, tile_expert;
  size_t chunk_hist, chunk_base;
  // forward
  size_t ring_flags;  // uint32 [4 * tile_capacity]: GEMM1 / GEMM2 tiles done per walk position
  size_t ring;        // bf16 [ring_slots * minibatch_rows, I]  (MXFP8: e4m3 codes)
  size_t ring_sf;     // MXFP8: u8 scales of the ring rows, tiled [ring rows/128][I/128][512 B]
  size_t ring_flags2, ring2;  // BF16: the flags and ring of the single-CTA ring launch that runs
                              // beside the CTA-pair one (same sizes as ring_flags, ring)
  size_t yk;          // bf16 [R, H]: expert outputs (forward), dX parts (backward)
  // backward
  size_t dhu;         // bf16 [pad_capacity, 2I]
  size_t as;          // bf16 [pad_capacity, I]  s * a
  size_t dsp;         // f32  [pad_capacity, I/128] router-gradient partial sums
  size_t sorted;      // BF16: [pad_capacity, H] token-sorted x (the forward ring reads it; then dW1|dW3)
  size_t sorted2;     // bf16 [pad_capacity, H]: BF16 token-sorted dout (dA', dW2)
  size_t pair_m0;     // int32 [tile_capacity]: CTA-pair units of dA' / dX / the ring (first M tile * 2 + solo)
  size_t pair_mb;     // int32 [tile_capacity + 2]: the list of tiles those launches run on single CTAs
  // MXFP8 operand copies
  size_t xq, xsf;     // x (forward) or dout (backward) along H: u8 [T, H], [T, H/32]
  size_t xq_sorted;   // those codes in padded-row order (GEMM1 / dA' A operand): u8 [pad_capacity, H]
  size_t sfa_rows_t;  // the A operand's scales in padded-row order, tiled: [pad/128][max(H,2I)/128][512]
  size_t wsf1, wsf3, wsf2;  // weight scales tiled for the GEMMs; wsf3 = wsf1 + one weight's scales, so
                            // [wsf1, wsf3 end) holds W1's and W3's blocks interleaved (GEMM1)
  size_t dhuq, dhusf; // dh|du quantised along I: u8 [pad, 2I], [pad, 2I/32]
  size_t wqa, wsfa;   // weight gradients: sorted x / dout along rows, [pad, H] + tiled scales
  size_t wqb, wsfb;   // weight gradients: dh|du / s*a along rows, [pad, 2I] + tiled scales
  size_t total;
  int64_t pad_capacity, tile_capacity, nchunks;
  int minibatch_rows, ring_slots;
};

// Host: layout of the workspace (offsets are 256-byte aligned).
WsLayout ws_layout(const mok_shape& s, const mok_config& c, mok_precision prec, int num_sms);
int effective_minibatch_rows(const mok_shape& s, const mok_config& c, int num_sms);
int device_sm_count();

// Host: tensor maps (driver entry point resolved once).
bool make_tmap(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* ptr, const uint64_t* dims,
               const uint64_t* strides_bytes /* rank-1 */, const uint32_t* box, bool swizzle128);

// Launchers (return a CUDA error code).
cudaError_t launch_schedule(const mok_shape& s, const WsLayout& L, uint8_t* ws, const int32_t* idx,
                            cudaStream_t st);
// the row tiles' split (forward ring, dA', dX): CTA-pair units (pair_m0,
// header word kHdrPairs) and single tiles (pair_mb as the list, word kHdrSingles)
cudaError_t launch_split_table(const WsLayout& L, uint8_t* ws, int min_pair_tiles, cudaStream_t st);
cudaError_t launch_combine(const mok_shape& s, const WsLayout& L, const uint8_t* ws, const __nv_bfloat16* yk,
                           const float* scores, __nv_bfloat16* out, cudaStream_t st);
cudaError_t launch_ds_reduce(const mok_shape& s, const WsLayout& L, const uint8_t* ws, float* ds, int n_parts,
                             cudaStream_t st);
// MXFP8: token-sorted copy of E4M3 code rows [T, H] -> [pad_capacity, H]
cudaError_t launch_gather_code_rows(const mok_shape& s, const WsLayout& L, const uint8_t* ws, const uint8_t* codes,
                                    uint8_t* dst, cudaStream_t st);
// skip (device, optional): the launch does nothing while *skip != 0
cudaError_t launch_gather_rows(const mok_shape& s, const WsLayout& L, const uint8_t* ws, const __nv_bfloat16* x,
                               __nv_bfloat16* xg, cudaStream_t st, const int32_t* skip = nullptr);
// MXFP8 weight scales tiled for the GEMMs' bulk loads (see mxfp8.cu):
// [batch][N / (128 g)][K/128][s x 512 B], N block nb at slot slot + nb % g.
// From plain scales blocked along K = rows ([batch][K/32][N]) or along each
// row of a K-major operand ([batch][N][K/32]).
cudaError_t launch_tile_scales(const uint8_t* sf, int batch, int kb_count, int N, uint8_t* out, cudaStream_t st,
                               int g = 1, int s = 1, int slot = 0);
cudaError_t launch_tile_scales_rows(const uint8_t* sf, int batch, int N, int kb_count, uint8_t* out,
                                    cudaStream_t st, int g = 1, int s = 1, int slot = 0);
cudaError_t launch_tile_row_scales(const uint8_t* sf, int kb_count, const int32_t* pad_perm, int k,
                                   const int32_t* rows_used, long rows_cap, uint8_t* out, cudaStream_t st);
cudaError_t launch_replay_copy(const mok_shape& s, const WsLayout& L, const uint8_t* ws,
                               const __nv_bfloat16* ctx_ring, __nv_bfloat16* dhu, cudaStream_t st);
// Router (router.cu)
cudaError_t launch_router_pad_weights(int H, int E, int Epad, const __nv_bfloat16* w, __nv_bfloat16* wp,
                                      cudaStream_t st);
cudaError_t launch_router_topk(int T, int E, int Epad, int k, const float* logits, const float* bias, int32_t* idx,
                               float* scores, cudaStream_t st);
cudaError_t launch_router_logit_grad(int T, int Tpad, int E, int Epad, int k, const int32_t* idx, const float* s,
                                     const float* ds, __nv_bfloat16* dl, cudaStream_t st);
cudaError_t launch_router_take_cols(int rows, int E, int Epad, const float* src, float* dst, cudaStream_t st);
cudaError_t launch_quant_rows_tiled(const __nv_bfloat16* src, const int32_t* rows_used, long rows_cap, int C,
                                    uint8_t* q, uint8_t* sf, cudaStream_t st);
// The same codes and scales for the token rows pad_perm[p] / k of src [T, C]
// in padded-row order (zeros for padding rows), without a sorted bf16 copy.
cudaError_t launch_quant_rows_gather(const __nv_bfloat16* src, const int32_t* rows_used, long rows_cap, int C,
                                     const int32_t* pad_perm, int k, uint8_t* q, uint8_t* sf, cudaStream_t st);
// Expert parallelism (ep.cu): source-side pack / combine / un-sort around the exchange
cudaError_t launch_ep_pack(const mok_shape& s, const WsLayout& L, const uint8_t* ws, const __nv_bfloat16* x,
                           const float* scores, __nv_bfloat16* rows, float* s_rows, cudaStream_t st);
cudaError_t launch_ep_combine(const mok_shape& s, const WsLayout& L, const uint8_t* ws, const __nv_bfloat16* rows,
                              const float* scores, __nv_bfloat16* out, cudaStream_t st);
cudaError_t launch_ep_unsort(const mok_shape& s, const WsLayout& L, const uint8_t* ws, const float* vals, float* out,
                             cudaStream_t st);
cudaError_t launch_mxfp8_quantize(const __nv_bfloat16* src, int batch, int rows, int cols, int block_axis,
                                  uint8_t* q, uint8_t* sf, cudaStream_t st);

}  // namespace mok

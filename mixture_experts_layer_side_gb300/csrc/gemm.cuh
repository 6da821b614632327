// Expert-grouped GEMM kernel family (tcgen05 + TMEM + TMA), shared declarations.
#pragma once

#include "mok_internal.cuh"

namespace mok {

// What one launch of the grouped GEMM computes.
enum GemmMode : int {
  GM_DENSE = 0,   // C[M,N] f32 = A * B, A [M,K] or [K,M], B [N,K] or [K,N] (diagnostic)
  GM_FWD1 = 1,    // [h|u] = gather(x) * [W1|W3];  epilogue SwiGLU -> ring (a), ctx (h, u)
  GM_FWD2 = 2,    // y = ring(a) * W2;             epilogue scatter y -> Yk[f]
  GM_BWD_DA = 3,  // dA' = gather(dout) * W2^T;    epilogue SwiGLU backward, s*a, ds partials
  GM_BWD_DX = 4,  // dx = [dh|du] * [W1|W3]^T;     epilogue scatter -> dXk[f]
  GM_WG13 = 5,    // [dW1|dW3]_e = gather(x)_e^T * [dh|du]_e
  GM_WG2 = 6,     // dW2_e = (s a)_e^T * gather(dout)_e
  GM_FWD_RING = 7, // GM_FWD1 and GM_FWD2 interleaved through the minibatch ring in one launch
  GM_FWD_FUSED = 8 // the whole forward in one launch: schedule items, the ring's items, a combine phase
};

constexpr int kStages = 4;
constexpr int kPairStages = 6;      // CTA-pair launches: 16 KB of A + 16 KB of B per stage
constexpr int kMaxStages = 6;
constexpr int kAStage = 128 * 128;  // 128 rows x 128 bytes
constexpr int kBStage = 256 * 128;  // up to 256 rows x 128 bytes
constexpr int kQueue = 4;           // depth of the work-item queue in smem
constexpr int kGemmThreads = 320;   // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue, warps 6-9 gather
constexpr int kMaxExperts = 1024;


constexpr int kMaxMaps = 6;
constexpr int kOutStage = 32 * 64 * 2;  // one epilogue warp's 32 x 64 bf16 output chunk
constexpr int kSfStage = 512 + 1024;    // MXFP8 scale blocks of one stage: A (128 rows), B (256)
struct TmapSet {
  CUtensorMap m[kMaxMaps];
};

struct GemmParams {
  int bn;         // N tile (128 or 256)
  int n_tiles;    // N tiles per M tile
  int k_iters;    // K iterations of 128 bytes (row-tiled and dense modes)
  int m_tiles;    // dense: M/128; weight-gradient modes: M/128 per expert
  int m_tile_begin, m_tile_end;  // row-tiled modes: range of 128-row tiles
  int T, H, I, E, k;
  int32_t* hdr;   // workspace header: error word, used rows/tiles, counters
  int counter;    // index of this launch's dynamic tile counter
  const int32_t* tile_expert;
  const int32_t* pad_perm;
  const int32_t* padded_offsets;
  const int32_t* counts;   // routed rows per expert
  // epilogue operands
  float* out_f32;
  long ld_out;
  __nv_bfloat16* out_bf16;  // dense: bf16 output instead, of the first m_valid rows
  long m_valid;
  __nv_bfloat16* ctx_hu;   // [pad, 2I]
  int ctx_ring;            // GEMM1: [h|u] rows in ring-slot order (bounded-memory forward)
  int replay_keep;         // GEMM1 launch: stop before the last replay_keep minibatches
  __nv_bfloat16* ring;     // [ring_slots * ring_rows, I]
  int ring_rows, ring_slots;
  uint32_t* ring_flags;    // [4 * tile_capacity]
  __nv_bfloat16* yk;       // [R, H]
  __nv_bfloat16* dhu;      // [pad, 2I]
  __nv_bfloat16* as;       // [pad, I]
  float* dsp;              // [pad, n_tiles]
  const float* scores;     // [R]
  const __nv_bfloat16* gather_src;  // x (GEMM1, dW1|dW3) or dout (dA', dW2): [T, H]
  __nv_bfloat16* dW1;      // weight-gradient outputs: dW1, dW3 (GM_WG13)
  __nv_bfloat16* dW3;
  __nv_bfloat16* dW2;      // dW2 (GM_WG2)
  // weight-gradient launches: the experts whose padded rows lie in
  // [wg_rows_min, wg_rows_max) are this launch's items; the launch with
  // wg_rows_min = 0 also writes the empty experts' zero gradients
  int wg_rows_min, wg_rows_max;
  int a_mn, b_mn;          // dense: operand major-ness (1 = M/N-major)
  int g1_tiles;            // ring: GEMM1 N tiles per M tile
  int debug_flags;
  int nmaps;               // tensor maps in use (prefetched at start)
  int wg_sorted;           // weight gradients read token-sorted copies (plain TMA)
  int rows_sorted;         // dA' reads a token-sorted copy of dout (plain TMA)
  // CTA-pair launches of dA' / dX / the forward ring: the pair table (first
  // M tile * 2 + solo)
  const int32_t* pair_m0;
  // ring launches: the units they walk, counted by header word
  // ring_count_word -- all tiles (kHdrTiles, ring_list null), the tiles of
  // ring_list (kHdrSingles), or the pairs of pair_m0 (kHdrPairs, CTA pairs);
  // a tile's ring rows and flags follow its position in that walk
  const int32_t* ring_list;
  int ring_count_word;
  int fwd_sorted;          // GEMM1 reads a token-sorted copy of x (plain TMA) instead of gathering
  // Overlapped launches (programmatic dependent launch, one stream): a
  // memory-bound launch on a few SMs sets pdl_trigger, so the next launch
  // (pdl_launch: launched with programmatic stream serialisation, reading
  // nothing the first one writes) starts on the other SMs at once and takes
  // each SM the first one leaves; pdl_wait_end makes that second launch wait
  // for the first before it exits, so the stream's later launches see both.
  int pdl_trigger;
  int pdl_wait_end;
  int pdl_launch;          // host side: the launch attribute
  // single-CTA ring launch beside a pair launch: CTAs at or above this index
  // leave at once (0: none leave; -1: the share of the grid that matches
  // this launch's tiles, hdr[kHdrSingles], against the pair launch's,
  // 2 * hdr[kHdrPairs], each pair tile counted at 4/5 of a single one)
  int active_ctas;
  // single-launch forward (GM_FWD_FUSED): the schedule's input and arrays
  // (written by its schedule items), and the combine's output
  const int32_t* topk_idx;
  int nchunks;             // routed-row chunks of kSchedChunk rows
  int32_t* chunk_hist;     // [nchunks, E]
  int32_t* chunk_base;     // [nchunks, E]
  int32_t* s_counts;       // [E]
  int32_t* s_offsets;      // [E + 1]
  int32_t* s_poff;         // [E + 1]
  int32_t* s_perm;         // [R]
  int32_t* s_inv_perm;     // [R]
  int32_t* s_pad_perm;     // [pad]
  int32_t* s_pad_inv;      // [R]
  int32_t* s_tile_expert;  // [tile_capacity]
  __nv_bfloat16* out;      // [T, H]
  // ---- MXFP8 (E4M3 codes, E8M0 scales per 32 K-elements)
  // K-major operands: scales [rows][K/32], four bytes per row per stage,
  // copied by the gather threads; rows of A are gathered by token when A is.
  const uint8_t* sfa_rows;    // A scales (x, dout, ring or dh|du)
  long sfa_ld;                // bytes per row of sfa_rows
  const uint8_t* sfb_rows0;   // B scales (W2 along H; W1 along I)
  const uint8_t* sfb_rows1;   // B scales, second weight (W3 along I)
  long sfb_ld;
  // Scales pre-tiled into 512-byte blocks per 128 M/N x 128 K (see
  // mxfp8.cu), loaded by the TMA producer one bulk load per operand per
  // stage: weights' blocks grouped per bn-wide N tile (GEMM1: W1's and W3's
  // interleaved in sfb_tiled0), activations' per 128 rows.
  const uint8_t* sfa_tiled;
  const uint8_t* sfb_tiled0;
  const uint8_t* sfb_tiled1;  // dX: W3 (W1 in tiled0)
  const uint8_t* sfb_tiled2;  // W2 in the ring launch (W1 | W3 in tiled0)
  const uint8_t* gq_src;      // gathered E4M3 rows (x or dout codes) [T, H]
  uint8_t* ring_sf;           // GEMM1 epilogue: scales of a, tiled [ring rows/128][I/128][512 B]
  uint8_t* dhu_q;             // dA' epilogue: dh|du codes [pad, 2I] ...
  uint8_t* dhu_sf;            // ... and scales [pad, 2I/32]
  // Ring launch: m_tiles holds twice the tile capacity (the walk positions'
  // bound); ring_flags[q] counts the epilogue warps (4 per column tile) that
  // published GEMM1 rows of walk position q, ring_flags[m_tiles + q] the
  // GEMM2 column tiles that consumed them.
};

size_t gemm_smem_bytes();
// CTAs of the pair launches the device holds at once (0: no cluster of two fits).
int gemm_pair_capacity();
cudaError_t launch_gemm(int mode, const TmapSet& maps, const GemmParams& p, int grid, cudaStream_t st);
cudaError_t launch_gemm_mx(int mode, const TmapSet& maps, const GemmParams& p, int grid, cudaStream_t st);
// BF16 launches on clusters of two CTAs that share each 256 x 256 tile
// through one cta_group::2 MMA: the weight-gradient GEMMs (GM_WG13 / GM_WG2,
// token-sorted operands, an even number of 128-row M tiles, bn = 256), the
// row-tiled backward GEMMs (GM_BWD_DA with token-sorted dout, GM_BWD_DX;
// bn = 256, the pair units of launch_split_table, weight maps with 128-row
// boxes) and the forward ring (GM_FWD_RING with a token-sorted copy of x,
// bn = 256, over the pairs of launch_split_table, an even number of tiles per
// minibatch).  Returns cudaErrorNotSupported when the device cannot hold a
// cluster of two.
cudaError_t launch_gemm_pair(int mode, const TmapSet& maps, const GemmParams& p, int grid, cudaStream_t st);

}  // namespace mok

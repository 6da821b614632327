// Expert-grouped GEMMs of the MoE layer on sm_103a tensor cores.
//
// One persistent, warp-specialised kernel family:
//   warp 0      TMA producer for the operands that are plain tiles (weights,
//               sorted-row activations): cp.async.bulk.tensor.
//   warps 6..9  gather producers: the dispatch gather (sorted row -> token
//               row of x or dout) is fused into the load path as 16-byte
//               cp.async copies written straight into the 128-byte-swizzled
//               operand layout, completing on the stage's mbarrier
//               (cp.async.mbarrier.arrive.noinc).  (TMA tile::gather4 moved
//               a third of the bytes per SM-cycle of these copies at the
//               same depth, so the gathered operands do not use it.)
//   warp 1      MMA issuer: tcgen05.mma (BF16 kind::f16, or MXFP8
//               kind::mxf8f6f4.block_scale with the stage scales copied to
//               TMEM by tcgen05.cp), FP32 accumulate in TMEM, 128 x N tiles,
//               N = 128 or 256; TMEM holds two accumulators (BF16) so the
//               epilogue of one tile overlaps the main loop of the next.
//   warps 2..5  epilogue: tcgen05.ld of the accumulator, then the fused
//               per-mode work (SwiGLU, scatter to token order, SwiGLU
//               backward with the router-score partial sums, weight-gradient
//               stores).  MXFP8 has one accumulator: its epilogues park what
//               they still need in free TMEM columns and hand it back early;
//               in the MXFP8 ring the otherwise idle warps 6..9 take half of
//               each tile row.  In the dense MXFP8 core warps 6..9 move the
//               stage scales into TMEM instead (tcgen05.st).
// Weight-gradient launches read token-sorted operands with plain TMA (the
// gather warps write the empty experts' zero gradients instead) and come in
// two forms: single CTAs, and clusters of two CTAs sharing a 256 x 256 tile
// through one cta_group::2 MMA (launch_gemm_pair) for long-K experts.  dX,
// and dA' on token-sorted dout, also run on such clusters, two 128-row
// tiles of one expert per 256 x 256 tile.  GM_FWD_FUSED adds the
// schedule's and the combine's work to the forward ring launch.
// Work items (output tiles) are taken from a device counter in increasing
// order, so a CTA only ever waits on items taken before its own; the
// numerics of a tile never depend on which CTA computes it (fixed K order,
// no split-K, no atomics on data), which keeps every output bitwise
// reproducible.
//
// Pages: expert-grouped GEMM and SwiGLU ("Cursor Open-Sources
// Mixture-of-Kittens (MoK)", "Three design decisions that matter",
// overlap-granularity paragraph, and the paragraph after that list);
// pull dispatch / push combine mapped to gather-in-load and
// scatter-in-epilogue (same section, communication-direction paragraph);
// the ring token buffer consumed per minibatch (ring-token-buffer paragraph);
// router gradient fused into the SwiGLU backward (paragraph after the list).
#include <climits>

#include "gemm.cuh"
#include "mx.cuh"
#include "tc.cuh"

namespace mok {

namespace {

struct Ctl {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t sfready[kMaxStages];  // dense MXFP8 core: the stage's scales are in TMEM (written by the gather warps)
  uint64_t sffull[kMaxStages];   // dense MXFP8 core: the stage's scale blocks are in smem
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t qfull[kQueue];
  uint64_t qempty[kQueue];
  int q[kQueue];
  uint32_t tmem_base;
  int abort;
  int po[kMaxExperts + 1];  // padded expert offsets (weight-gradient modes)
  // weight-gradient modes: experts by descending padded rows, each entry
  // e | (K iterations << 10); the n_nonempty experts with routed rows first
  int order[kMaxExperts];
  int n_nonempty;
  int n_skip;  // experts ahead of this launch's row range in that order
  int n_sel;   // experts in this launch's row range (its items)
  int pair_rank;  // CTA-pair launches: 0 for the leader (issues the MMAs), 1 for the other
  int combine_go;  // single-launch forward: 1 once every GEMM2 row of y is stored, 2 on a wait that gave up
};

// A decoded work item.
struct Item {
  int type;     // effective mode of this item (GM_FWD1 / GM_FWD2 inside the ring kernel)
  int m;        // 128-row tile index (row-tiled modes) or M tile inside the expert (wgrad)
  int n;        // N tile
  int e;        // expert
  int row0;     // first padded row of the tile (row-tiled) or of the expert (wgrad)
  int k_iters;  // K iterations of 128 bytes
  int idle;     // CTA pairs: the second CTA of a solo pair (loads, stores nothing)
  int rp;       // ring launches: the tile's position in the launch's walk (ring rows, flags)
};

__device__ __forceinline__ int used_tiles(const GemmParams& p) { return p.hdr[kHdrTiles]; }

// The ring launch, alone or inside the single-launch forward.
template <int MODE>
__device__ __forceinline__ constexpr bool is_ring() { return MODE == GM_FWD_RING || MODE == GM_FWD_FUSED; }

// Single-launch forward: items [0, nch) histogram one chunk of routed rows
// each, item nch scans, items [nch + 1, 2 nch + 1) place one chunk each,
// then come the ring's items; every item waits only on items before it.
// A CTA that draws past the last item runs the combine phase (its warps
// take tokens from a second counter) and stops.
constexpr int kItemCount = 16, kItemScan = 17, kItemPlace = 18, kItemCombine = 19;
__device__ __forceinline__ int fused_ring_base(const GemmParams& p) { return 2 * p.nchunks + 1; }
// (valid once the scan item has published the tile count)
__device__ __forceinline__ int fused_total(const GemmParams& p) {
  return fused_ring_base(p) + used_tiles(p) * (p.g1_tiles + p.n_tiles);
}

// Number of work items of a launch (device-side: depends on the schedule).
template <int MODE>
__device__ int count_items(const GemmParams& p) {
  if constexpr (MODE == GM_DENSE) {
    return p.m_tiles * p.n_tiles;
  } else if constexpr (MODE == GM_WG13 || MODE == GM_WG2) {
    return 0;  // known only inside the kernel (experts with routed rows)
  } else if constexpr (MODE == GM_FWD_RING) {
    return p.hdr[p.ring_count_word] * (p.g1_tiles + p.n_tiles);
  } else {
    // a launch over a tile list (the single tiles of a split)
    if (p.ring_list) return p.hdr[p.ring_count_word] * p.n_tiles;
    int end = min(p.m_tile_end, used_tiles(p));
    if (p.replay_keep > 0) {
      // GEMM1 recomputed in the backward: every minibatch but the last
      // replay_keep, whose [h|u] the bounded forward context still holds
      const int Mt = p.ring_rows / kTileRows;
      const int nb = (used_tiles(p) + Mt - 1) / Mt;
      end = min(end, max(nb - p.replay_keep, 0) * Mt);
    }
    return max(end - p.m_tile_begin, 0) * p.n_tiles;
  }
}

// Work items of a row-tiled launch on CTA pairs: pair tiles x N tiles.
__device__ __forceinline__ int count_pair_items(const GemmParams& p) { return p.hdr[kHdrPairs] * p.n_tiles; }

// Ring kernel: item w -> (type, tile, n).  Sequence of steps: step 0 is
// GEMM1 of minibatch 0; step s >= 1 is GEMM1 of minibatch s followed by
// GEMM2 of minibatch s-1; the last step is GEMM2 of the last minibatch.
// Inside a step the items run N-tile-major over the minibatch's M tiles,
// so the M tiles of one expert, which share a weight slice, run together
// (1.8% faster on the DeepSeek-V3-shaped forward than M-tile-major).
// Generic form: `tiles` units (tiles, or pairs of tiles), Mt units per
// minibatch.
__device__ void decode_ring_n(const GemmParams& p, int w, int tiles, int Mt, int& type, int& m, int& n) {
  const int nb = (tiles + Mt - 1) / Mt;
  const int g1 = p.g1_tiles, g2 = p.n_tiles;
  auto mt_of = [&](int b) { return min(Mt, tiles - b * Mt); };
  auto emit = [&](int t, int b, int r, int nt) {
    type = t;
    const int mb = mt_of(b);
    m = b * Mt + r % mb;
    n = r / mb;
  };
  // step 0
  const int s10 = mt_of(0) * g1;
  if (w < s10) return emit(GM_FWD1, 0, w, g1);
  w -= s10;
  const int full_steps = max(nb - 2, 0);
  const int F = Mt * (g1 + g2);
  if (w < full_steps * F) {
    const int s = 1 + w / F;
    const int r = w % F;
    if (r < Mt * g1) return emit(GM_FWD1, s, r, g1);
    return emit(GM_FWD2, s - 1, r - Mt * g1, g2);
  }
  w -= full_steps * F;
  if (nb >= 2) {
    const int a = mt_of(nb - 1) * g1;
    if (w < a) return emit(GM_FWD1, nb - 1, w, g1);
    w -= a;
    const int b2 = Mt * g2;
    if (w < b2) return emit(GM_FWD2, nb - 2, w, g2);
    w -= b2;
  }
  return emit(GM_FWD2, nb - 1, w, g2);
}

__device__ __forceinline__ void decode_ring(const GemmParams& p, int w, int& type, int& m, int& n) {
  decode_ring_n(p, w, used_tiles(p), p.ring_rows / kTileRows, type, m, n);
}

__device__ __forceinline__ int row_k_iters(const GemmParams& p, int type, int el) {
  return (type == GM_FWD1 || type == GM_BWD_DA) ? p.H / el
         : (type == GM_FWD2)                   ? p.I / el
                                               : 2 * p.I / el;  // GM_BWD_DX
}

template <int MODE, bool MX = false, bool PAIR = false>
__device__ Item decode(const GemmParams& p, const Ctl* ctl, int w) {
  constexpr int kEl = MX ? 128 : 64;  // K elements per stage (128 bytes)
  const int* po = ctl->po;
  Item it;
  it.idle = 0;
  it.rp = 0;
  if constexpr (MODE == GM_DENSE) {
    it.type = MODE;
    it.m = w / p.n_tiles;
    it.n = w % p.n_tiles;
    it.e = 0;
    it.row0 = it.m * kTileRows;
    it.k_iters = p.k_iters;
  } else if constexpr (MODE == GM_WG13 || MODE == GM_WG2) {
    // Items are the tiles of the experts that have routed rows, experts
    // sorted by descending K; fetches alternate between the two ends of that
    // list, so a CTA pairs a long-K tile (MMA-bound) with a short one (store-
    // bound epilogue) and the two overlap through the double-buffered TMEM.
    // (Empty experts' zero gradients are written outside the item list.)
    // CTA pairs take the M tiles two at a time: the leader the even one
    const int per_e = (PAIR ? p.m_tiles / 2 : p.m_tiles) * p.n_tiles;
    const int total = ctl->n_sel * per_e;
    const int pos = (w & 1) ? total - 1 - (w >> 1) : (w >> 1);
    const int rank = pos / per_e;
    const int oe = ctl->order[ctl->n_skip + rank];
    it.type = MODE;
    it.e = oe & 1023;
    const int r = pos - rank * per_e;
    it.m = PAIR ? 2 * (r / p.n_tiles) + ctl->pair_rank : r / p.n_tiles;
    it.n = r % p.n_tiles;
    it.row0 = po[it.e];
    it.k_iters = oe >> 10;
  } else if constexpr (MODE == GM_FWD_FUSED) {
    const int nch = p.nchunks, a0 = fused_ring_base(p);
    it.n = 0;
    it.e = 0;
    it.row0 = 0;
    it.k_iters = 0;
    if (w < a0) {
      it.type = w < nch ? kItemCount : w == nch ? kItemScan : kItemPlace;
      it.m = w < nch ? w : w == nch ? 0 : w - nch - 1;
    } else {
      const int ring_items = used_tiles(p) * (p.g1_tiles + p.n_tiles);
      if (w - a0 >= ring_items) {
        it.type = kItemCombine;
        it.m = 0;
      } else {
        int type, m, n;
        decode_ring(p, w - a0, type, m, n);
        it.type = type;
        it.m = m;
        it.rp = m;
        it.n = n;
        it.e = p.tile_expert[m];
        it.row0 = m * kTileRows;
        it.k_iters = row_k_iters(p, type, kEl);
      }
    }
  } else if constexpr (PAIR && MODE == GM_FWD_RING) {
    // the ring on CTA pairs: its units are the pairs of the split table (two
    // tiles of one expert, or an expert's odd last tile as a solo pair),
    // ring_rows / 256 of them per minibatch; the leader takes the unit's
    // first tile, the other CTA the second (idle in a solo pair), and unit
    // u's tiles sit at walk positions 2u and 2u + 1
    int type, u, n;
    decode_ring_n(p, w, p.hdr[kHdrPairs], p.ring_rows / (2 * kTileRows), type, u, n);
    const int code = p.pair_m0[u];
    it.idle = (code & 1) && ctl->pair_rank == 1;
    const int r = it.idle ? 0 : ctl->pair_rank;
    const int m = (code >> 1) + r;
    it.type = type;
    it.m = m;
    it.rp = 2 * u + r;
    it.n = n;
    it.e = p.tile_expert[m];
    it.row0 = m * kTileRows;
    it.k_iters = row_k_iters(p, type, kEl);
  } else if constexpr (PAIR) {
    // dA' / dX on CTA pairs: the leader takes the pair's first tile, the
    // other CTA the second (or, in a solo pair, the first again, idle)
    const int code = p.pair_m0[w / p.n_tiles];
    it.idle = (code & 1) && ctl->pair_rank == 1;
    const int m = (code >> 1) + (it.idle ? 0 : ctl->pair_rank);
    it.type = MODE;
    it.m = m;
    it.rp = m;
    it.n = w % p.n_tiles;
    it.e = p.tile_expert[m];
    it.row0 = m * kTileRows;
    it.k_iters = row_k_iters(p, MODE, kEl);
  } else {
    int type = MODE, m, n, rp;
    if constexpr (MODE == GM_FWD_RING) {
      // walk position -> tile: the position itself, or the tile a list holds there
      decode_ring_n(p, w, p.hdr[p.ring_count_word], p.ring_rows / kTileRows, type, rp, n);
      m = p.ring_list ? p.ring_list[rp] : rp;
    } else {
      m = p.ring_list ? p.ring_list[w / p.n_tiles] : p.m_tile_begin + w / p.n_tiles;
      n = w % p.n_tiles;
      rp = m;
    }
    it.type = type;
    it.m = m;
    it.rp = rp;
    it.n = n;
    it.e = p.tile_expert[m];
    it.row0 = m * kTileRows;
    it.k_iters = row_k_iters(p, type, kEl);
  }
  return it;
}

__device__ __forceinline__ int item_bn(const GemmParams& p, int type) { return type == GM_FWD1 ? 256 : p.bn; }

__device__ __forceinline__ int ring_row(const GemmParams& p, int prow) {
  const int mb = prow / p.ring_rows;
  return (mb % p.ring_slots) * p.ring_rows + (prow - mb * p.ring_rows);
}

// ------------------------------------------------------------------ producers
// Which operand of an item is gathered by token (0 none, 1 A, 2 B).
// With p.wg_sorted the weight-gradient GEMMs, and with p.rows_sorted dA',
// read a token-sorted copy of x / dout (rows in padded schedule order) with
// plain TMA instead.
__device__ __forceinline__ int gathered_operand(const GemmParams& p, int type) {
  if (p.wg_sorted && (type == GM_WG13 || type == GM_WG2)) return 0;
  if (p.fwd_sorted && type == GM_FWD1) return 0;
  if (p.rows_sorted && type == GM_BWD_DA) return 0;
  return (type == GM_FWD1 || type == GM_BWD_DA || type == GM_WG13) ? 1 : (type == GM_WG2 ? 2 : 0);
}

template <int MODE>
__device__ __forceinline__ constexpr bool mode_gathers() {
  return MODE == GM_FWD1 || MODE == GM_BWD_DA || MODE == GM_WG13 || MODE == GM_WG2 || is_ring<MODE>();
}

// Bytes the TMA producer brings into one stage (gathered operands excluded).
__device__ __forceinline__ uint32_t tma_stage_bytes(const GemmParams& p, int type, int bn) {
  const int g = gathered_operand(p, type);
  return (g == 1 ? 0u : (uint32_t)kAStage) + (g == 2 ? 0u : (uint32_t)bn * 128u);
}

// TMA producer (lane 0 of warp 0) for one K stage of the plain operands.
template <int MODE>
__device__ __forceinline__ void tma_loads(const TmapSet& mp, const GemmParams& p, const Item& it, int kk, uint8_t* a,
                                          uint8_t* b, uint64_t* bar) {
  const int type = it.type;
  if (MODE == GM_DENSE) {
    if (p.a_mn) {
      for (int c = 0; c < 2; ++c) tma_load_2d(a + c * 8192, &mp.m[0], bar, it.m * 128 + c * 64, kk * 64);
    } else {
      tma_load_2d(a, &mp.m[0], bar, kk * 64, it.m * 128);
    }
    if (p.b_mn) {
      for (int c = 0; c < p.bn / 64; ++c) tma_load_2d(b + c * 8192, &mp.m[1], bar, it.n * p.bn + c * 64, kk * 64);
    } else {
      tma_load_2d(b, &mp.m[1], bar, kk * 64, it.n * p.bn);
    }
  } else if (type == GM_FWD1) {
    // A: the token-sorted copy of x, when GEMM1 does not gather
    if (p.fwd_sorted) tma_load_2d(a, &mp.m[0], bar, kk * 64, it.row0);
    // B: W1 and W3 column blocks (N-major); 128 h columns then 128 u columns
    for (int c = 0; c < 2; ++c) tma_load_3d(b + c * 8192, &mp.m[1], bar, it.n * 128 + c * 64, kk * 64, it.e);
    for (int c = 0; c < 2; ++c) tma_load_3d(b + (2 + c) * 8192, &mp.m[2], bar, it.n * 128 + c * 64, kk * 64, it.e);
  } else if (type == GM_FWD2) {
    const int mslot = is_ring<MODE>() ? 3 : 0;
    const int wmap = is_ring<MODE>() ? 4 : 1;
    tma_load_2d(a, &mp.m[mslot], bar, kk * 64, ring_row(p, it.rp * kTileRows));
    for (int c = 0; c < p.bn / 64; ++c) tma_load_3d(b + c * 8192, &mp.m[wmap], bar, it.n * p.bn + c * 64, kk * 64, it.e);
  } else if (type == GM_BWD_DA) {
    if (p.rows_sorted) tma_load_2d(a, &mp.m[0], bar, kk * 64, it.row0);
    tma_load_3d(b, &mp.m[1], bar, kk * 64, it.n * p.bn, it.e);
  } else if (type == GM_BWD_DX) {
    tma_load_2d(a, &mp.m[0], bar, kk * 64, it.row0);
    const int ki = p.I / 64;
    if (kk < ki)
      tma_load_3d(b, &mp.m[1], bar, kk * 64, it.n * p.bn, it.e);
    else
      tma_load_3d(b, &mp.m[2], bar, (kk - ki) * 64, it.n * p.bn, it.e);
  } else if (type == GM_WG13) {
    // B = [dh|du] rows of the expert (N = 2I, MN-major)
    for (int cc = 0; cc < p.bn / 64; ++cc)
      tma_load_2d(b + cc * 8192, &mp.m[1], bar, it.n * p.bn + cc * 64, it.row0 + kk * 64);
    // A = token-sorted x rows (M = H, MN-major), when not gathered
    if (p.wg_sorted)
      for (int ca = 0; ca < 2; ++ca) tma_load_2d(a + ca * 8192, &mp.m[0], bar, it.m * 128 + ca * 64, it.row0 + kk * 64);
  } else if (type == GM_WG2) {
    // A = (s a) rows of the expert (M = I, MN-major)
    for (int ca = 0; ca < 2; ++ca) tma_load_2d(a + ca * 8192, &mp.m[0], bar, it.m * 128 + ca * 64, it.row0 + kk * 64);
    // B = token-sorted dout rows (N = H, MN-major), when not gathered
    if (p.wg_sorted)
      for (int cc = 0; cc < p.bn / 64; ++cc)
        tma_load_2d(b + cc * 8192, &mp.m[1], bar, it.n * p.bn + cc * 64, it.row0 + kk * 64);
  }
}

// CTA-pair stage: this CTA's A tile (its own 128 M rows) and its half of
// the 256-column B tile, completing on the leader's barrier.
template <int MODE>
__device__ __forceinline__ void tma_loads_pair(const TmapSet& mp, const GemmParams& p, const Item& it, int kk,
                                               int rank, uint8_t* a, uint8_t* b, uint32_t bar) {
  const int bcol = it.n * 256 + rank * 128;
  if constexpr (MODE == GM_FWD_RING) {
    if (it.type == GM_FWD1) {
      // A: token-sorted x rows; B: the leader's half is the W1 column block
      // (h), the other CTA's the W3 block (u) of intermediate columns n*128..
      tma_load_2d_pair(a, &mp.m[0], bar, kk * 64, it.row0);
      for (int c = 0; c < 2; ++c)
        tma_load_3d_pair(b + c * 8192, &mp.m[rank ? 2 : 1], bar, it.n * 128 + c * 64, kk * 64, it.e);
    } else {
      // A: this tile's ring rows; B: this CTA's 128 columns of the W2 block
      tma_load_2d_pair(a, &mp.m[3], bar, kk * 64, ring_row(p, it.rp * kTileRows));
      for (int c = 0; c < 2; ++c) tma_load_3d_pair(b + c * 8192, &mp.m[4], bar, bcol + c * 64, kk * 64, it.e);
    }
  } else if constexpr (MODE == GM_WG13 || MODE == GM_WG2) {
    const int krow = it.row0 + kk * 64;
    for (int c = 0; c < 2; ++c) tma_load_2d_pair(a + c * 8192, &mp.m[0], bar, it.m * 128 + c * 64, krow);
    for (int c = 0; c < 2; ++c) tma_load_2d_pair(b + c * 8192, &mp.m[1], bar, bcol + c * 64, krow);
  } else if (MODE == GM_BWD_DA) {  // A: token-sorted dout rows
    tma_load_2d_pair(a, &mp.m[0], bar, kk * 64, it.row0);
    tma_load_3d_pair(b, &mp.m[1], bar, kk * 64, bcol, it.e);
  } else {  // GM_BWD_DX: K runs over dh (W1) and then du (W3)
    tma_load_2d_pair(a, &mp.m[0], bar, kk * 64, it.row0);
    const int ki = p.I / 64;
    tma_load_3d_pair(b, &mp.m[kk < ki ? 1 : 2], bar, (kk < ki ? kk : kk - ki) * 64, bcol, it.e);
  }
}

__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}

__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ int token_or_neg(const GemmParams& p, int prow) {
  const int f = p.pad_perm[prow];
  return f >= 0 ? f / p.k : -1;
}

// Gathered operand of one K stage, by the 128 gather threads (gt = 0..127).
// K-major (A of GEMM1 / dA'): 128 token rows x 128 bytes; thread gt copies
//   16-byte chunk (gt & 7) of rows (gt >> 3) + 16 j.  tok[] holds them.
// M/N-major (A of dW1|dW3, B of dW2): 64 routed rows (the K dimension) x
//   cpr 16-byte chunks; chunk c = gt + 128 j is row c / cpr, column chunk
//   c % cpr, stored in 64-column blocks of 8192 bytes.  tok[] holds the
//   tokens of those rows for this stage.
// Rows with no token (padding) are zero-filled.  Every thread's copies
// complete on the stage's full barrier (one no-increment arrival each).
__device__ __forceinline__ void gather_kmajor(uint8_t* dst, const __nv_bfloat16* src, int ld, int col0, int gt,
                                              const int (&tok)[8], uint64_t* full) {
  const int ch = gt & 7;
  const int sw = (ch ^ ((gt >> 3) & 7)) << 4;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int row = (gt >> 3) + 16 * j;
    const int t = tok[j];
    cp_async_16(smem_u32(dst + row * 128 + sw), src + (long)max(t, 0) * ld + col0 + ch * 8, t >= 0 ? 16u : 0u);
  }
  cp_async_arrive_noinc(full);
}

template <int CPR>  // 16-byte chunks per routed row: 16 (128 columns) or 32 (256 columns)
__device__ __forceinline__ void gather_mnmajor(uint8_t* dst, const __nv_bfloat16* src, int ld, int col0, int gt,
                                               const int (&tok)[64 / (128 / CPR)], uint64_t* full) {
  constexpr int kRowsPerPass = 128 / CPR;
  constexpr int kPasses = 64 / kRowsPerPass;
  const int cc = gt % CPR;
  const int blk = cc >> 3, ch = cc & 7;
#pragma unroll
  for (int j = 0; j < kPasses; ++j) {
    const int krow = gt / CPR + kRowsPerPass * j;
    const int t = tok[j];
    cp_async_16(smem_u32(dst + blk * 8192 + krow * 128 + ((ch ^ (krow & 7)) << 4)),
                src + (long)max(t, 0) * ld + col0 + blk * 64 + ch * 8, t >= 0 ? 16u : 0u);
  }
  cp_async_arrive_noinc(full);
}

// Tokens a gather thread needs for K stage kk of an M/N-major item.
template <int CPR>
__device__ __forceinline__ void mn_tokens(const GemmParams& p, const Item& it, int kk, int gt,
                                          int (&tok)[64 / (128 / CPR)]) {
  constexpr int kRowsPerPass = 128 / CPR;
  constexpr int kPasses = 64 / kRowsPerPass;
#pragma unroll
  for (int j = 0; j < kPasses; ++j) tok[j] = token_or_neg(p, it.row0 + kk * 64 + gt / CPR + kRowsPerPass * j);
}

// ---------------------------------------------------------------- MXFP8 producers
// Stage layout in MXFP8 mode: A and B codes fill the same 128-byte rows as
// bf16 (128 K-elements per stage); an M/N-major operand is one 16 KB
// 128-column chunk per 128 M/N (128 K-rows x 128 bytes).  Scales of a stage:
// sfa 512 bytes (128 A rows x 4 K-blocks), sfb 512 bytes per 128 B columns,
// in the tcgen05.cp .32x128b.warpx4 block layout.

// Bytes the TMA producer brings into one MXFP8 stage.
template <int MODE>
__device__ __forceinline__ uint32_t mx_stage_bytes(const GemmParams& p, int type, int bn) {
  const uint32_t bchunks = (uint32_t)bn / 128;
  switch (MODE == GM_DENSE ? GM_DENSE : type) {
    case GM_DENSE: return kAStage + bn * 128 + 512u + 512u * bchunks;
    case GM_FWD1: return 2u * 16384u + 1024u + 512u + (p.fwd_sorted ? (uint32_t)kAStage : 0u);
    case GM_FWD2: return kAStage + bn * 128 + 512u + 512u * bchunks;
    case GM_BWD_DA: return bn * 128 + 512u * bchunks + 512u + (p.rows_sorted ? (uint32_t)kAStage : 0u);
    case GM_BWD_DX: return kAStage + bn * 128 + 512u * bchunks + 512u;
    default: return kAStage + bn * 128 + 512u + 512u * bchunks;  // GM_WG13, GM_WG2
  }
}

// MXFP8 scale bytes of one stage: A's block (512 B) and B's blocks (512 B
// per 128 columns of the tile)
__device__ __forceinline__ uint32_t mx_sf_bytes(int bn) { return 512u * (1u + (uint32_t)bn / 128u); }

template <int MODE>
__device__ __forceinline__ void tma_loads_mx(const TmapSet& mp, const GemmParams& p, const Item& it, int kk, uint8_t* a,
                                             uint8_t* b, uint8_t* sfa, uint8_t* sfb, uint64_t* bar,
                                             uint64_t* sfbar) {
  const int type = it.type;
  const int bn = item_bn(p, type);
  if (MODE == GM_DENSE) {
    // both operands' scales come pre-tiled ([MN/128][K/128][512 B])
    const int kgroups = p.k_iters;
    if (p.a_mn)
      tma_load_2d(a, &mp.m[0], bar, it.m * 128, kk * 128);
    else
      tma_load_2d(a, &mp.m[0], bar, kk * 128, it.m * 128);
    bulk_load(sfa, p.sfa_tiled + ((long)it.m * kgroups + kk) * 512, 512, sfbar);
    if (p.b_mn) {
      for (int c = 0; c < bn / 128; ++c) tma_load_2d(b + c * 16384, &mp.m[1], bar, it.n * bn + c * 128, kk * 128);
    } else {
      tma_load_2d(b, &mp.m[1], bar, kk * 128, it.n * bn);
    }
    // B's scales grouped per bn-wide N tile: one load
    bulk_load(sfb, p.sfb_tiled0 + ((long)it.n * kgroups + kk) * (bn / 128) * 512, (bn / 128) * 512, sfbar);
  } else if (type == GM_FWD1) {
    const int hg = p.H / 128;
    // A: x's codes in padded-row order, when GEMM1 does not gather them
    if (p.fwd_sorted) tma_load_2d(a, &mp.m[0], bar, kk * 128, it.row0);
    tma_load_3d(b, &mp.m[1], bar, it.n * 128, kk * 128, it.e);
    tma_load_3d(b + 16384, &mp.m[2], bar, it.n * 128, kk * 128, it.e);
    // W1's and W3's scale blocks interleaved: one load
    const long blk = ((long)it.e * (p.I / 128) + it.n) * hg + kk;
    bulk_load(sfb, p.sfb_tiled0 + blk * 1024, 1024, sfbar);
    // A (gathered x rows): its scales pre-tiled in padded-row order
    bulk_load(sfa, p.sfa_tiled + ((long)it.m * hg + kk) * 512, 512, sfbar);
  } else if (type == GM_FWD2) {
    const int mslot = is_ring<MODE>() ? 3 : 0;
    const int wmap = is_ring<MODE>() ? 4 : 1;
    tma_load_2d(a, &mp.m[mslot], bar, kk * 128, ring_row(p, it.rp * kTileRows));
    // a's scales, tiled by the GEMM1 epilogue next to the ring codes
    bulk_load(sfa, p.ring_sf + ((long)(ring_row(p, it.rp * kTileRows) >> 7) * (p.I / 128) + kk) * 512, 512, sfbar);
    for (int c = 0; c < bn / 128; ++c) tma_load_3d(b + c * 16384, &mp.m[wmap], bar, it.n * bn + c * 128, kk * 128, it.e);
    // W2's scales grouped per bn-wide N tile: one load
    const long blk = ((long)it.e * (p.H / bn) + it.n) * (p.I / 128) + kk;
    bulk_load(sfb, (is_ring<MODE>() ? p.sfb_tiled2 : p.sfb_tiled0) + blk * (bn / 128) * 512, (bn / 128) * 512,
              sfbar);
  } else if (type == GM_BWD_DA) {
    // A: dout's codes in padded-row order, when dA' does not gather them;
    // B = W2 along H (K-major); its scales, and those of the dout rows,
    // pre-tiled per 128 rows x 128 K
    if (p.rows_sorted) tma_load_2d(a, &mp.m[0], bar, kk * 128, it.row0);
    tma_load_3d(b, &mp.m[1], bar, kk * 128, it.n * bn, it.e);
    bulk_load(sfa, p.sfa_tiled + ((long)it.m * (p.H / 128) + kk) * 512, 512, sfbar);
    const long blk = ((long)it.e * (p.I / bn) + it.n) * (p.H / 128) + kk;
    bulk_load(sfb, p.sfb_tiled0 + blk * (bn / 128) * 512, (bn / 128) * 512, sfbar);
  } else if (type == GM_BWD_DX) {
    // B = W1 then W3 along I (K-major); scales pre-tiled likewise
    tma_load_2d(a, &mp.m[0], bar, kk * 128, it.row0);
    bulk_load(sfa, p.sfa_tiled + ((long)it.m * (2 * p.I / 128) + kk) * 512, 512, sfbar);
    const int ki = p.I / 128;
    const int kb = kk < ki ? kk : kk - ki;
    tma_load_3d(b, &mp.m[kk < ki ? 1 : 2], bar, kb * 128, it.n * bn, it.e);
    const long blk = ((long)it.e * (p.H / bn) + it.n) * ki + kb;
    bulk_load(sfb, (kk < ki ? p.sfb_tiled0 : p.sfb_tiled1) + blk * (bn / 128) * 512, (bn / 128) * 512, sfbar);
  } else if (type == GM_WG13 || type == GM_WG2) {
    // token-sorted operands quantised along the routed rows (K), M/N-major
    const int cols_a = (type == GM_WG13) ? p.H : p.I;
    const int cols_b = (type == GM_WG13) ? 2 * p.I : p.H;
    const int rb = it.row0 / 128 + kk;
    tma_load_2d(a, &mp.m[0], bar, it.m * 128, it.row0 + kk * 128);
    bulk_load(sfa, p.sfa_tiled + ((long)rb * (cols_a / 128) + it.m) * 512, 512, sfbar);
    for (int c = 0; c < bn / 128; ++c) tma_load_2d(b + c * 16384, &mp.m[1], bar, it.n * bn + c * 128, it.row0 + kk * 128);
    // the bn / 128 column blocks of B's scales are adjacent: one load
    bulk_load(sfb, p.sfb_tiled0 + ((long)rb * (cols_b / 128) + it.n * (bn / 128)) * 512, (bn / 128) * 512, sfbar);
  }
}

// Gather threads, one MXFP8 stage: gathered E4M3 rows of A (GEMM1, dA') and
// the scales of K-major operands, four bytes per row (zero for padding
// rows), all completing on the stage barrier.
template <int MODE>
__device__ __forceinline__ void gather_stage_mx(const GemmParams& p, const Item& it, int kk, uint8_t* a, uint8_t* sfa,
                                                uint8_t* sfb, int gt, const int (&tok)[8], int tok_row,
                                                uint64_t* full) {
  const int type = it.type;
  const int bn = item_bn(p, type);
  const bool gather_a = (MODE != GM_DENSE) && (type == GM_FWD1 || type == GM_BWD_DA);
  if (gather_a) {
    const int ch = gt & 7;
    const int sw = (ch ^ ((gt >> 3) & 7)) << 4;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int row = (gt >> 3) + 16 * j;
      const int t = tok[j];
      cp_async_16(smem_u32(a + row * 128 + sw), p.gq_src + (long)max(t, 0) * p.H + kk * 128 + ch * 16,
                  t >= 0 ? 16u : 0u);
    }
  }
  // scales of A, row gt of the tile (GEMM1's, dA''s and dX's come pre-tiled
  // with the TMA loads)
  const uint8_t* sa = nullptr;
  if (MODE == GM_DENSE) {
    if (!p.a_mn) sa = p.sfa_rows + ((long)it.m * 128 + gt) * p.sfa_ld + kk * 4;
  }
  if (sa) cp_async_4(smem_u32(sfa + mx_sf_offset(gt, 0)), sa, 4u);
  // scales of K-major B, rows gt and gt + 128 of the N tile (dense launches;
  // the weights' scales of dA' and dX come pre-tiled with the TMA loads)
  const uint8_t* sb = nullptr;
  long brow0 = 0;
  const int kb = kk;
  if (MODE == GM_DENSE) {
    if (!p.b_mn) { sb = p.sfb_rows0; brow0 = (long)it.n * bn; }
  }
  if (sb) {
    for (int nl = gt; nl < bn; nl += 128)
      cp_async_4(smem_u32(sfb + (nl >> 7) * 512 + mx_sf_offset(nl & 127, 0)), sb + (brow0 + nl) * p.sfb_ld + kb * 4,
                 4u);
  }
  cp_async_arrive_noinc(full);
}

template <int MODE>
__device__ __forceinline__ bool a_mn_major(const GemmParams& p, int type) {
  if (MODE == GM_DENSE) return p.a_mn != 0;
  return type == GM_WG13 || type == GM_WG2;
}

template <int MODE>
__device__ __forceinline__ bool b_mn_major(const GemmParams& p, int type) {
  if (MODE == GM_DENSE) return p.b_mn != 0;
  return type == GM_FWD1 || type == GM_FWD2 || type == GM_WG13 || type == GM_WG2;
}

// ------------------------------------------------------------------ epilogues
__device__ __forceinline__ void store32_bf16(__nv_bfloat16* dst, const uint32_t (&w)[16]) {
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int i = 0; i < 4; ++i) d[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
}

__device__ __forceinline__ float sigmoidf_(float h) { return 1.0f / (1.0f + __expf(-h)); }

// GEMM1: columns [0,128) of the tile are h, [128,256) are u, for
// intermediate columns [n*128, n*128+128).  a = silu(h) * u from the bf16
// values that are saved for the backward.
__device__ void epi_fwd1(const GemmParams& p, const Item& it, uint32_t tbase, int row) {
  const long prow = (long)it.row0 + row;
  const int i0 = it.n * 128;
  const long crow = p.ctx_ring ? (long)ring_row(p, (int)prow) : prow;
  __nv_bfloat16* hrow = p.ctx_hu + crow * 2 * p.I + i0;
  __nv_bfloat16* urow = hrow + p.I;
  __nv_bfloat16* arow = p.ring + (long)ring_row(p, it.rp * kTileRows + row) * p.I + i0;
#pragma unroll 1
  for (int c = 0; c < 128; c += 32) {
    float h[32], u[32];
    tmem_ld32(tbase + c, h);
    tmem_ld32(tbase + 128 + c, u);
    uint32_t hw[16], uw[16], aw[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float h0 = bf16_round(h[2 * i]), h1 = bf16_round(h[2 * i + 1]);
      const float u0 = bf16_round(u[2 * i]), u1 = bf16_round(u[2 * i + 1]);
      hw[i] = pack_bf16x2(h0, h1);
      uw[i] = pack_bf16x2(u0, u1);
      aw[i] = pack_bf16x2(h0 * sigmoidf_(h0) * u0, h1 * sigmoidf_(h1) * u1);
    }
    store32_bf16(hrow + c, hw);
    store32_bf16(urow + c, uw);
    store32_bf16(arow + c, aw);
  }
}

// 64 accumulator columns of this lane's row (two 32-column TMEM loads, one
// wait) as 32 packed bf16 pairs (round to nearest even, low half first).
__device__ __forceinline__ void acc_load64_bf16(uint32_t taddr, uint32_t (&w)[32]) {
  uint32_t ra[32], rb[32];
  tmem_ld32_issue(taddr, ra);
  tmem_ld32_issue(taddr + 32, rb);
  tmem_wait_ld();
  tmem_regs_ready(ra);
  tmem_regs_ready(rb);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    w[i] = pack_bf16x2(__uint_as_float(ra[2 * i]), __uint_as_float(ra[2 * i + 1]));
    w[16 + i] = pack_bf16x2(__uint_as_float(rb[2 * i]), __uint_as_float(rb[2 * i + 1]));
  }
}

// A lane's 32 packed words parked in (and read back from) its own 128-byte
// row of the warp's staging buffer, 16-byte chunks XOR-swizzled by lane.
__device__ __forceinline__ void park64(uint8_t* stage, int lane, const uint32_t (&w)[32]) {
#pragma unroll
  for (int i = 0; i < 8; ++i)
    *reinterpret_cast<uint4*>(stage + lane * 128 + ((i ^ (lane & 7)) << 4)) =
        make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
}

__device__ __forceinline__ uint4 unpark16(const uint8_t* stage, int lane, int i) {
  return *reinterpret_cast<const uint4*>(stage + lane * 128 + ((i ^ (lane & 7)) << 4));
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// MXFP8 launches keep one accumulator (TMEM columns 0..255) and the stage
// scales (256..319); the epilogues park accumulator values in the columns
// past those, so they can hand the accumulator back early.
constexpr uint32_t kParkCol = 320;  // past the accumulator (0..255) and the stage scales (256..319)
static_assert(256 + kStages * 16 <= kParkCol && kParkCol + 192 <= 512, "parked columns overlap or leave TMEM");

// MXFP8 GEMM1 epilogue: as epi_fwd1, but a goes to the ring as E4M3 codes
// with one scale per 32 intermediate columns (the K blocks of GEMM2).  The
// row's h and u are first read as the bf16 values the backward keeps (h
// columns 0..63 into the staging buffer, the other 192 columns packed into
// parked TMEM columns), the accumulator is handed back (`release`), and
// only then is a formed, quantised and stored: the same values, with the
// next tile's main loop already running.
template <typename Release>
// With split epilogues (hm 1 / 2: two warps per lane quarter, each taking
// half of the row) the first warp takes h and u columns 0..63 (c = 0, 1),
// the second 64..127 (c = 2, 3), which it parks without the staging
// buffer; hm 0: one warp takes the whole row.
__device__ void epi_fwd1_mx(const GemmParams& p, const Item& it, uint32_t tbase, int row, int lane, uint8_t* stage,
                            Release&& release, int hm = 0) {
  const long prow = (long)it.row0 + row;
  const int i0 = it.n * 128;
  const long crow = p.ctx_ring ? (long)ring_row(p, (int)prow) : prow;
  const bool lo = hm != 2, hi = hm != 1;  // this warp's halves
  // packed bf16 words parked from kParkCol: h 64..127 at +0, u 0..127 at +32
  const uint32_t park = tbase + kParkCol;
  if (lo) {
    uint32_t hw0[32];
    acc_load64_bf16(tbase, hw0);
    park64(stage, lane, hw0);
  }
#pragma unroll 1
  for (int g = 1; g < 4; ++g) {
    // g = 1: h 64..127, g = 2: u 0..63, g = 3: u 64..127
    if (g == 2 ? !lo : !hi) continue;
    uint32_t w[32];
    acc_load64_bf16(tbase + 64 * g, w);
    tmem_st32(park + 32 * (g - 1), w);
  }
  tmem_wait_st();
  release();
  __nv_bfloat16* hrow = p.ctx_hu + crow * 2 * p.I + i0;
  __nv_bfloat16* urow = hrow + p.I;
  const long rr = ring_row(p, it.rp * kTileRows + row);
  uint8_t* qrow = reinterpret_cast<uint8_t*>(p.ring) + rr * p.I + i0;
  // the row's four scales of this 128-column group go out as one word, in
  // the tiled layout GEMM2's TMA thread bulk-loads ([ring rows / 128]
  // [I / 128][512 B], see mx_sf_offset)
  uint32_t* sword = reinterpret_cast<uint32_t*>(p.ring_sf + ((rr >> 7) * (p.I / 128) + it.n) * 512 +
                                                mx_sf_offset((int)(rr & 127), 0));
  uint32_t scales = 0;
#pragma unroll 1
  for (int c = 0; c < 4; ++c) {
    if (c < 2 ? !lo : !hi) continue;
    // 32 columns = 16 packed words each of h and u
    uint32_t h[16], u[16];
    tmem_ld16_issue(park + 32 + 16 * c, u);
    if (c >= 2) tmem_ld16_issue(park + 16 * (c - 2), h);
    tmem_wait_ld();
    tmem_regs_ready16(u);
    if (c >= 2) {
      tmem_regs_ready16(h);
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint4 v = unpark16(stage, lane, c * 4 + i);
        h[4 * i] = v.x; h[4 * i + 1] = v.y; h[4 * i + 2] = v.z; h[4 * i + 3] = v.w;
      }
    }
    uint4* dh = reinterpret_cast<uint4*>(hrow + c * 32);
    uint4* du = reinterpret_cast<uint4*>(urow + c * 32);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      dh[i] = make_uint4(h[4 * i], h[4 * i + 1], h[4 * i + 2], h[4 * i + 3]);
      du[i] = make_uint4(u[4 * i], u[4 * i + 1], u[4 * i + 2], u[4 * i + 3]);
    }
    // a = silu(h) u of the 32-column block, quantised as mx_quant32 does:
    // its amax first, then a formed again (the same values) as it is converted
    auto act = [&](int e) {
      const uint32_t hv = h[e >> 1], uv = u[e >> 1];
      const float hh = (e & 1) ? bf16_hi(hv) : bf16_lo(hv);
      const float uu = (e & 1) ? bf16_hi(uv) : bf16_lo(uv);
      return hh * sigmoidf_(hh) * uu;
    };
    float amax = 0.0f;
#pragma unroll
    for (int e = 0; e < 32; ++e) amax = fmaxf(amax, fabsf(act(e)));
    const int X = mx_block_exponent(amax);
    const float inv = mx_exp2_int(-X);
    uint32_t q[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint16_t lo = mx_cvt_e4m3x2(act(4 * i) * inv, act(4 * i + 1) * inv);
      const uint16_t hi = mx_cvt_e4m3x2(act(4 * i + 2) * inv, act(4 * i + 3) * inv);
      q[i] = (uint32_t)lo | ((uint32_t)hi << 16);
    }
    scales |= (uint32_t)(X + 127) << (8 * c);
    uint4* d = reinterpret_cast<uint4*>(qrow + c * 32);
    d[0] = make_uint4(q[0], q[1], q[2], q[3]);
    d[1] = make_uint4(q[4], q[5], q[6], q[7]);
  }
  if (hm == 0)
    *sword = scales;
  else if (hm == 1)
    reinterpret_cast<uint16_t*>(sword)[0] = (uint16_t)scales;
  else
    reinterpret_cast<uint16_t*>(sword)[1] = (uint16_t)(scales >> 16);
}

// MXFP8 scatter (single-buffered accumulator): the whole row is read as
// packed bf16 first (columns 0..63 parked in the staging buffer, the rest
// in parked TMEM columns), the accumulator handed back, then the row
// stored (padding rows load with the warp, store nothing).
// (hm 1 / 2: the first or the second half of the row's 64-column groups,
// the staged group 0 in the first; hm 0: the whole row)
template <int BN, typename Release>
__device__ void epi_scatter_mx_n(const GemmParams& p, const Item& it, uint32_t tbase, int row, int lane,
                                 uint8_t* stage, Release&& release, int hm) {
  constexpr int bn = BN;
  constexpr int kG = bn / 64;
  const int g0 = hm == 2 ? kG / 2 : 0, g1 = hm == 1 ? kG / 2 : kG;
  const int prow = it.row0 + row;
  const int f = p.pad_perm[prow];
  const uint32_t park = tbase + kParkCol;
  if (g0 == 0) {
    uint32_t w0[32];
    acc_load64_bf16(tbase, w0);
    park64(stage, lane, w0);
  }
#pragma unroll 1
  for (int g = g0 > 1 ? g0 : 1; g < g1; ++g) {
    uint32_t w[32];
    acc_load64_bf16(tbase + 64 * g, w);
    tmem_st32(park + 32 * (g - 1), w);
  }
  tmem_wait_st();
  release();
  __nv_bfloat16* dst = p.yk + (long)(f < 0 ? 0 : f) * p.H + it.n * bn;
  if (f >= 0 && g0 == 0) {
    uint4* d0 = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int i = 0; i < 8; ++i) d0[i] = unpark16(stage, lane, i);
  }
#pragma unroll 1
  for (int g = g0 > 1 ? g0 : 1; g < g1; ++g) {
    uint32_t w[32];
    tmem_ld32_issue(park + 32 * (g - 1), w);
    tmem_wait_ld();
    tmem_regs_ready(w);
    if (f >= 0) {
      uint4* d = reinterpret_cast<uint4*>(dst + 64 * g);
#pragma unroll
      for (int i = 0; i < 8; ++i) d[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
    }
  }
}

template <typename Release>
__device__ void epi_scatter_mx(const GemmParams& p, const Item& it, uint32_t tbase, int row, int bn, int lane,
                               uint8_t* stage, Release&& release, int hm = 0) {
  if (bn == 256)
    epi_scatter_mx_n<256>(p, it, tbase, row, lane, stage, release, hm);
  else
    epi_scatter_mx_n<128>(p, it, tbase, row, lane, stage, release, hm);
}

// Scatter a tile row to token order: row f of dst (skipped for padding rows;
// every lane still takes part in the warp-collective TMEM loads).
__device__ void epi_scatter(const GemmParams& p, const Item& it, uint32_t tbase, int row, int bn) {
  const int prow = it.row0 + row;
  const int f = p.pad_perm[prow];
  __nv_bfloat16* dst = p.yk + (long)max(f, 0) * p.H + it.n * bn;
#pragma unroll 1
  for (int c = 0; c < bn; c += 32) {
    float v[32];
    tmem_ld32(tbase + c, v);
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) w[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
    if (f >= 0) store32_bf16(dst + c, w);
  }
}

// SwiGLU backward.  Accumulator = dA' = dout_t W2_e^T for intermediate
// columns [n*bn, n*bn+bn).  With s the row's router score:
//   ds partial = sum_i dA'_i a_i          (router-score gradient)
//   dA = s dA',  dh = dA u sig(h) (1 + h (1 - sig(h))),  du = dA silu(h)
//   A_s = s a  (the left operand of dW2)
// MXFP8 keeps one accumulator, so this epilogue would hold up the next
// tile's MMAs for all of its work: it first parks accumulator columns
// [64, bn) unchanged (f32) in the TMEM columns no MMA or scale uses
// (kParkCol.., 192 of them), works through columns [0, 64), hands the
// accumulator back, and takes the rest from the parked copy while the next
// tile's main loop runs.  The values are the same f32 bits either way.

// MXFP8 dA': the accumulator goes back to the MMA thread once this many
// columns are worked through (the rest parked in TMEM first).  Earlier
// hand-backs measured slower: the epilogue's loads and stores beside the
// next tile's MMAs slow those more than the accumulator wait costs.
constexpr int kDaHandBack = 64;

template <bool MX, typename Release>
__device__ void epi_bwd_da(const GemmParams& p, const Item& it, uint32_t tbase, int row, Release&& release) {
  const uint32_t park = tbase + kParkCol;  // MXFP8: single accumulator at column 0
  if constexpr (MX) {
#pragma unroll 1
    for (int c = kDaHandBack; c < p.bn; c += 32) {
      uint32_t r[32];
      tmem_ld32_issue(tbase + c, r);
      tmem_wait_ld();
      tmem_regs_ready(r);
      tmem_st32(park + (c - kDaHandBack), r);
    }
    tmem_wait_st();
  }
  const long prow = (long)it.row0 + row;
  const int f = p.pad_perm[prow];
  const float s = f >= 0 ? p.scores[f] : 0.0f;
  const int bn = p.bn;
  const __nv_bfloat16* hrow = p.ctx_hu + prow * 2 * p.I + it.n * bn;
  const __nv_bfloat16* urow = hrow + p.I;
  __nv_bfloat16* dhrow = p.dhu + prow * 2 * p.I + it.n * bn;
  __nv_bfloat16* durow = dhrow + p.I;
  __nv_bfloat16* asrow = p.as + prow * p.I + it.n * bn;
  float dsum = 0.0f;
  // h and u of the next 32 columns are in flight while this chunk's TMEM
  // load and arithmetic run (each row's loads are dependent on nothing but
  // the address, so their latency need not add to every chunk)
  uint4 hn[4], un[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    hn[i] = reinterpret_cast<const uint4*>(hrow)[i];
    un[i] = reinterpret_cast<const uint4*>(urow)[i];
  }
#pragma unroll 1
  for (int c = 0; c < bn; c += 32) {
    uint32_t hc[16], uc[16];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      hc[4 * i] = hn[i].x, hc[4 * i + 1] = hn[i].y, hc[4 * i + 2] = hn[i].z, hc[4 * i + 3] = hn[i].w;
      uc[4 * i] = un[i].x, uc[4 * i + 1] = un[i].y, uc[4 * i + 2] = un[i].z, uc[4 * i + 3] = un[i].w;
    }
    if (c + 32 < bn) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        hn[i] = reinterpret_cast<const uint4*>(hrow + c + 32)[i];
        un[i] = reinterpret_cast<const uint4*>(urow + c + 32)[i];
      }
    }
    float g[32];
    tmem_ld32((MX && c >= kDaHandBack) ? park + (c - kDaHandBack) : tbase + c, g);
    // columns [0, kDaHandBack) are read: the rest is parked
    if (MX && c == kDaHandBack - 32) release();
    uint32_t dhw[16], duw[16], asw[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float2 h2 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&hc[i]));
      const float2 u2 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&uc[i]));
      const float hp[2] = {h2.x, h2.y}, up[2] = {u2.x, u2.y};
      float r[2][3];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const float hh = hp[j], uu = up[j], gg = g[2 * i + j];
        const float sg = sigmoidf_(hh);
        const float sl = hh * sg;
        const float a = sl * uu;
        dsum = fmaf(gg, a, dsum);
        const float dA = s * gg;
        r[j][0] = dA * uu * sg * (1.0f + hh * (1.0f - sg));
        r[j][1] = dA * sl;
        r[j][2] = s * a;
      }
      dhw[i] = pack_bf16x2(r[0][0], r[1][0]);
      duw[i] = pack_bf16x2(r[0][1], r[1][1]);
      asw[i] = pack_bf16x2(r[0][2], r[1][2]);
    }
    store32_bf16(dhrow + c, dhw);
    store32_bf16(durow + c, duw);
    store32_bf16(asrow + c, asw);
    if constexpr (MX) {
      // dh|du quantised along I for the dX GEMM (32 columns per scale)
      const int col = it.n * bn + c;
      float v[32];
      uint32_t q[8];
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const uint32_t(&src)[16] = half == 0 ? dhw : duw;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&src[i]));
          v[2 * i] = f.x;
          v[2 * i + 1] = f.y;
        }
        const long qc = (long)half * p.I + col;
        p.dhu_sf[prow * (2 * p.I / 32) + qc / 32] = mx_quant32(v, q);
        uint4* d = reinterpret_cast<uint4*>(p.dhu_q + prow * 2 * p.I + qc);
        d[0] = make_uint4(q[0], q[1], q[2], q[3]);
        d[1] = make_uint4(q[4], q[5], q[6], q[7]);
      }
    }
  }
  p.dsp[prow * p.n_tiles + it.n] = dsum;
}

// A warp's 32 x 64 bf16 chunk (lane = row, w[] = its 64 values as bf16
// pairs) leaves as full 128-byte row segments: staged in a 4 KB smem buffer
// (16-byte chunks XOR-swizzled by row), read back with 8 lanes per row and
// stored 4 rows x 128 bytes per instruction -- four whole cache lines each.
__device__ __forceinline__ void stage_chunk64(uint8_t* stage, int lane, const uint32_t (&w)[32]);
template <typename RowPtr>
__device__ __forceinline__ void flush_chunk64(uint8_t* stage, int lane, RowPtr row_ptr);

template <typename RowPtr>
__device__ __forceinline__ void store_chunk64_coalesced(uint8_t* stage, int lane, const uint32_t (&w)[32],
                                                        RowPtr row_ptr) {
  stage_chunk64(stage, lane, w);
  flush_chunk64(stage, lane, row_ptr);
}

// The two halves of store_chunk64_coalesced: a lane's row into the staging
// buffer, then the buffer out as whole row segments.
__device__ __forceinline__ void stage_chunk64(uint8_t* stage, int lane, const uint32_t (&w)[32]) {
  const int sw = lane & 7;
#pragma unroll
  for (int i = 0; i < 8; ++i)
    *reinterpret_cast<uint4*>(stage + lane * 128 + ((i ^ sw) << 4)) =
        make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
  __syncwarp();
}

template <typename RowPtr>
__device__ __forceinline__ void flush_chunk64(uint8_t* stage, int lane, RowPtr row_ptr) {
  const int ch = lane & 7;
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    const int rr = 4 * s + (lane >> 3);
    const uint4 v = *reinterpret_cast<const uint4*>(stage + rr * 128 + ((ch ^ (rr & 7)) << 4));
    __nv_bfloat16* dst = row_ptr(rr);
    if (dst) *reinterpret_cast<uint4*>(dst + ch * 8) = v;
  }
  __syncwarp();
}

// Weight gradients: tile rows are rows of dW (H rows of dW1/dW3, I rows of
// dW2), columns are its columns.  An expert with no routed rows has no
// accumulation and gets exact zeros.  A weight-gradient item has a short K
// loop (the expert's rows), so the 64 KB output tile must leave fast:
// coalesced stores through the warp's staging buffer.
// 64 columns of accumulator (two 32-column TMEM loads) -> bf16 -> dW rows.
// First dW element of rows r0.. at column col of the item's output, and the
// row pitch.  I is a multiple of 128, so a 64-column chunk never straddles
// dW1 | dW3.
__device__ __forceinline__ __nv_bfloat16* wgrad_base(const GemmParams& p, const Item& it, int r0, int col, long& ld) {
  if (it.type == GM_WG13) {
    ld = p.I;
    return (col < p.I) ? p.dW1 + ((long)it.e * p.H + r0) * p.I + col
                       : p.dW3 + ((long)it.e * p.H + r0) * p.I + (col - p.I);
  }
  ld = p.H;
  return p.dW2 + ((long)it.e * p.I + r0) * p.H + col;
}

// 64 columns at a time: two TMEM loads, one wait, then the coalesced store.
// With PARKED (MXFP8: one accumulator, so this epilogue would otherwise hold
// up the next tile's MMAs) the row is first rounded to bf16 64 columns at a
// time -- the first 64 into the staging buffer, the rest packed into the
// TMEM columns past the accumulator and the stage scales (kParkCol..) --
// then `release` hands the accumulator back and the stores run from the
// staging buffer and the parked copy while the next tile's main loop runs
// (the same bf16 values either way).  Otherwise the caller releases the
// accumulator after the stores.
template <int BN, bool PARKED, typename Release>
__device__ __forceinline__ void epi_wgrad_n(const GemmParams& p, const Item& it, uint32_t tbase, int q, int lane,
                                            uint8_t* stage, Release&& release) {
  constexpr int kGroups = BN / 64;
  const int r0 = it.m * 128 + q * 32;  // first dW row of this warp
  const int col0 = it.n * BN;
  if constexpr (!PARKED) {
#pragma unroll
    for (int g = 0; g < kGroups; ++g) {
      uint32_t w[32];
      acc_load64_bf16(tbase + 64 * g, w);
      long ld;
      __nv_bfloat16* base = wgrad_base(p, it, r0, col0 + 64 * g, ld);
      store_chunk64_coalesced(stage, lane, w, [&](int rr) { return base + rr * ld; });
    }
    return;
  }
  const uint32_t park = tbase + kParkCol;  // single accumulator at column 0
  {
    uint32_t w0[32];
    acc_load64_bf16(tbase, w0);
    stage_chunk64(stage, lane, w0);
  }
#pragma unroll 1
  for (int g = 1; g < kGroups; ++g) {
    uint32_t w[32];
    acc_load64_bf16(tbase + 64 * g, w);
    tmem_st32(park + 32 * (g - 1), w);
  }
  tmem_wait_st();
  release();
  long ld;
  __nv_bfloat16* base = wgrad_base(p, it, r0, col0, ld);
  flush_chunk64(stage, lane, [&](int rr) { return base + rr * ld; });
#pragma unroll 1
  for (int g = 1; g < kGroups; ++g) {
    uint32_t w[32];
    tmem_ld32_issue(park + 32 * (g - 1), w);
    tmem_wait_ld();
    tmem_regs_ready(w);
    base = wgrad_base(p, it, r0, col0 + 64 * g, ld);
    store_chunk64_coalesced(stage, lane, w, [&](int rr) { return base + rr * ld; });
  }
}

template <bool PARKED, typename Release>
__device__ void epi_wgrad(const GemmParams& p, const Item& it, uint32_t tbase, int q, int lane, uint8_t* stage,
                          Release&& release) {
  if (p.bn == 256)
    epi_wgrad_n<256, PARKED>(p, it, tbase, q, lane, stage, release);
  else
    epi_wgrad_n<128, PARKED>(p, it, tbase, q, lane, stage, release);
}

__device__ void epi_dense(const GemmParams& p, const Item& it, uint32_t tbase, int row) {
  const long grow = (long)it.m * 128 + row;
  if (p.out_bf16) {
    // bf16 output of the first m_valid rows only (the TMEM loads are
    // warp-wide, so every lane takes part in them)
    __nv_bfloat16* dst = p.out_bf16 + grow * p.ld_out + it.n * p.bn;
#pragma unroll 1
    for (int c = 0; c < p.bn; c += 32) {
      float v[32];
      tmem_ld32(tbase + c, v);
      if (grow < p.m_valid) {
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) w[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
        uint4* d = reinterpret_cast<uint4*>(dst + c);
#pragma unroll
        for (int i = 0; i < 4; ++i) d[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
      }
    }
    return;
  }
  float* dst = p.out_f32 + grow * p.ld_out + it.n * p.bn;
#pragma unroll 1
  for (int c = 0; c < p.bn; c += 32) {
    float v[32];
    tmem_ld32(tbase + c, v);
    float4* d = reinterpret_cast<float4*>(dst + c);
#pragma unroll
    for (int i = 0; i < 8; ++i) d[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
  }
}

// All K stages of one item's M/N-major gathered operand (weight-gradient
// GEMMs, where K is the expert's routed rows).  Row -> token lookups are
// dependent loads, so they run kPrefetch stages ahead in a register ring.
template <int CPR, int NST>
__device__ bool gather_item_mn(const GemmParams& p, const Item& it, uint8_t* op_base, int op_stride, int col0,
                               Ctl* ctl, uint32_t& stage, uint32_t& phase, int gt, const WaitCtx& wc) {
  constexpr int kTok = 64 / (128 / CPR);
  constexpr int kPrefetch = 4;
  int ring[kPrefetch][kTok];
#pragma unroll
  for (int d = 0; d < kPrefetch; ++d)
    if (d < it.k_iters) mn_tokens<CPR>(p, it, d, gt, ring[d]);
  for (int kk0 = 0; kk0 < it.k_iters; kk0 += kPrefetch) {
#pragma unroll
    for (int u = 0; u < kPrefetch; ++u) {
      const int kk = kk0 + u;
      if (kk < it.k_iters) {
        if (!mbar_wait(&ctl->empty[stage], phase ^ 1, wc)) return false;
        gather_mnmajor<CPR>(op_base + stage * op_stride, p.gather_src, p.H, col0, gt, ring[u], &ctl->full[stage]);
        if (kk + kPrefetch < it.k_iters) mn_tokens<CPR>(p, it, kk + kPrefetch, gt, ring[u]);
        if (++stage == NST) { stage = 0; phase ^= 1; }
      }
    }
  }
  return true;
}

// All K stages of one item whose gathered operand is K-major (GEMM1, dA'):
// the 128 token rows are fixed for the item.  Items with nothing to gather
// (GEMM2 inside the ring launch) only keep the stage barriers' phase count.
template <int NST>
__device__ bool gather_item_k(const GemmParams& p, const Item& it, uint8_t* sA, Ctl* ctl, uint32_t& stage,
                              uint32_t& phase, int gt, const WaitCtx& wc) {
  const bool gather = gathered_operand(p, it.type) == 1;
  int tok[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) tok[j] = gather ? token_or_neg(p, it.row0 + (gt >> 3) + 16 * j) : -1;
  for (int kk = 0; kk < it.k_iters; ++kk) {
    if (!mbar_wait(&ctl->empty[stage], phase ^ 1, wc)) return false;
    if (gather)
      gather_kmajor(sA + stage * kAStage, p.gather_src, p.H, kk * 64, gt, tok, &ctl->full[stage]);
    else
      mbar_arrive(&ctl->full[stage]);
    if (++stage == NST) { stage = 0; phase ^= 1; }
  }
  return true;
}

// Weight gradients of the experts without routed rows are exact zeros: the
// four gather warps of every CTA write them in 32 KB chunks (one 512-byte
// warp store per step), dealt round-robin over all CTAs' gather warps.  In
// launches whose operands are TMA-loaded these warps have no other work, so
// the zero stores overlap the MMA-bound tiles of the item list.
template <int MODE>
__device__ void zero_empty_experts(const GemmParams& p, const Ctl* ctl, int gw, int lane) {
  constexpr long kChunk = 16384;  // bf16 elements per chunk
  const int n_empty = p.E - ctl->n_nonempty;
  const long slab = (long)p.H * p.I;  // dW1_e, dW3_e: [H, I]; dW2_e: [I, H]
  const int per_expert = (MODE == GM_WG13) ? 2 : 1;
  const long chunks_per_slab = slab / kChunk;  // H and I are multiples of 128
  const long total = (long)n_empty * per_expert * chunks_per_slab;
  const uint4 z = make_uint4(0u, 0u, 0u, 0u);
  for (long c = (long)blockIdx.x * 4 + gw; c < total; c += (long)gridDim.x * 4) {
    const long sl = c / chunks_per_slab;
    const int e = ctl->order[ctl->n_nonempty + (int)(sl / per_expert)] & 1023;
    __nv_bfloat16* base = (MODE == GM_WG2) ? p.dW2 : (sl % per_expert) ? p.dW3 : p.dW1;
    uint4* dst = reinterpret_cast<uint4*>(base + (long)e * slab + (c - sl * chunks_per_slab) * kChunk);
#pragma unroll 8
    for (int i = 0; i < (int)(kChunk * 2 / 16 / 32); ++i) __stcs(dst + i * 32 + lane, z);
  }
}

// ---------------------------------------------------------------- single-launch forward
// The schedule items and the combine phase of GM_FWD_FUSED.  The four
// gather warps (128 threads, named barrier 1) run the schedule items; they
// and the four epilogue warps run the combine phase.  Each item publishes
// its completion with a release add on a header counter, and every item
// that reads another's output acquires that counter first (bounded waits).
// The arithmetic is the schedule kernels' and the combine kernel's, so the
// arrays and the output are bitwise those of the separate launches.
__device__ __forceinline__ void gather_warps_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

__device__ __forceinline__ uint32_t* hdr_word(const GemmParams& p, int i) {
  return reinterpret_cast<uint32_t*>(&p.hdr[i]);
}

// Expert histogram of routed-row chunk c (ids outside [0, E) set the error bit).
__device__ void fused_count(const GemmParams& p, int c, int* hist, int gt) {
  const int E = p.E, R = p.T * p.k;
  for (int e = gt; e < E; e += 128) hist[e] = 0;
  gather_warps_sync();
  const int f0 = c * kSchedChunk, f1 = min(f0 + kSchedChunk, R);
  bool bad = false;
  for (int f = f0 + gt; f < f1; f += 128) {
    const int e = p.topk_idx[f];
    if (e >= 0 && e < E)
      atomicAdd(&hist[e], 1);
    else
      bad = true;
  }
  if (bad) atomicOr(&p.hdr[kHdrError], MOK_ERRBIT_BAD_INDEX);
  gather_warps_sync();
  for (int e = gt; e < E; e += 128) p.chunk_hist[(size_t)c * E + e] = hist[e];
  __threadfence();
  gather_warps_sync();
  if (gt == 0) red_release_gpu_add(hdr_word(p, kHdrCountDone), 1u);
}

// Per expert the running base of every chunk, then the exclusive scans of
// the counts and of the 128-padded counts (thread gt owns the contiguous
// experts [gt * per, gt * per + per)), the tile table and the padding rows'
// -1 markers.  tot: 8 ints of shared memory.
__device__ void fused_scan(const GemmParams& p, int* tot, int gt) {
  const int E = p.E, nch = p.nchunks, per = (E + 127) / 128;
  const int lane = gt & 31, wg = gt >> 5;
  int cnt[8];
  int tc = 0, tp = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    cnt[i] = 0;
    const int e = gt * per + i;
    if (i < per && e < E) {
      // loads independent of the running sum: eight in flight at a time
      int run = 0, c = 0;
      for (; c + 8 <= nch; c += 8) {
        int v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) v[u] = p.chunk_hist[(size_t)(c + u) * E + e];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          p.chunk_base[(size_t)(c + u) * E + e] = run;
          run += v[u];
        }
      }
      for (; c < nch; ++c) {
        const int v = p.chunk_hist[(size_t)c * E + e];
        p.chunk_base[(size_t)c * E + e] = run;
        run += v;
      }
      cnt[i] = run;
      tc += run;
      tp += (run + kTileRows - 1) / kTileRows * kTileRows;
    }
  }
  int ic = tc, ip = tp;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int a = __shfl_up_sync(0xffffffffu, ic, d), b = __shfl_up_sync(0xffffffffu, ip, d);
    if (lane >= d) {
      ic += a;
      ip += b;
    }
  }
  if (lane == 31) {
    tot[wg] = ic;
    tot[4 + wg] = ip;
  }
  gather_warps_sync();
  int bc = ic - tc, bp = ip - tp;
  for (int v = 0; v < wg; ++v) {
    bc += tot[v];
    bp += tot[4 + v];
  }
  const int total_c = tot[0] + tot[1] + tot[2] + tot[3];
  const int total_p = tot[4] + tot[5] + tot[6] + tot[7];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = gt * per + i;
    if (i < per && e < E) {
      const int padded = (cnt[i] + kTileRows - 1) / kTileRows * kTileRows;
      p.s_counts[e] = cnt[i];
      p.s_offsets[e] = bc;
      p.s_poff[e] = bp;
      for (int t = bp / kTileRows; t < (bp + padded) / kTileRows; ++t) p.s_tile_expert[t] = e;
      for (int r = bp + cnt[i]; r < bp + padded; ++r) p.s_pad_perm[r] = -1;
      bc += cnt[i];
      bp += padded;
    }
  }
  if (gt == 0) {
    p.s_offsets[E] = total_c;
    p.s_poff[E] = total_p;
    p.hdr[kHdrPaddedRows] = total_p;
    p.hdr[kHdrTiles] = total_p / kTileRows;
  }
  __threadfence();
  gather_warps_sync();
  if (gt == 0) red_release_gpu_add(hdr_word(p, kHdrScanDone), 1u);
}

// Places chunk c's rows (one warp; cursor: E ints of shared memory): rows of
// one expert in increasing f, after the chunk's base.  MXFP8: also the row's
// x scales (token f / k of sfa_rows, H / 32 bytes) into the tiled A-scale
// layout GEMM1's TMA thread loads, [padded rows / 128][H / 128][512 B]
// (padding rows keep the zeros the caller cleared them to).
template <bool MX>
__device__ void fused_place(const GemmParams& p, int c, int* cursor, int lane) {
  const int E = p.E, R = p.T * p.k;
  for (int e = lane; e < E; e += 32) cursor[e] = p.chunk_base[(size_t)c * E + e];
  __syncwarp();
  const unsigned lt = (1u << lane) - 1u;
  const int f0 = c * kSchedChunk;
  for (int i = 0; i < kSchedChunk / 32; ++i) {
    const int f = f0 + i * 32 + lane;
    int e = -1;
    if (f < R) {
      e = p.topk_idx[f];
      if (e < 0 || e >= E) e = -1;
    }
    const unsigned grp = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(grp & lt);
    int pos = 0;
    if (e >= 0) pos = cursor[e] + rank;
    __syncwarp();
    if (e >= 0 && rank == 0) cursor[e] += __popc(grp);
    __syncwarp();
    if (f < R) {
      if (e >= 0) {
        const int r = p.s_offsets[e] + pos, prow = p.s_poff[e] + pos;
        p.s_perm[r] = f;
        p.s_inv_perm[f] = r;
        p.s_pad_perm[prow] = f;
        p.s_pad_inv[f] = prow;
        if constexpr (MX) {
          const uint8_t* src = p.sfa_rows + (long)(f / p.k) * p.sfa_ld;
          uint8_t* dst = const_cast<uint8_t*>(p.sfa_tiled) + (long)(prow / kTileRows) * (p.H / 128) * 512 +
                         mx_sf_offset(prow % kTileRows, 0);
          for (int kg = 0; kg < p.H / 128; ++kg)
            *reinterpret_cast<uint32_t*>(dst + (long)kg * 512) = *reinterpret_cast<const uint32_t*>(src + kg * 4);
        }
      } else {
        p.s_inv_perm[f] = -1;
        p.s_pad_inv[f] = -1;
      }
    }
  }
  // (MXFP8: the tiled scales are read by TMA, the async proxy)
  if constexpr (MX) fence_proxy_async_global();
  __threadfence();
  __syncwarp();
  if (lane == 0) red_release_gpu_add(hdr_word(p, kHdrPlaceDone), 1u);
}

__device__ __forceinline__ void unpack8_bf16(const uint4& v, float (&o)[8]) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(h[i]);
    o[2 * i] = f.x;
    o[2 * i + 1] = f.y;
  }
}

// out[t] = sum_j s[t,j] y[t*k+j] for one token, by one warp: f32,
// increasing j, one rounding.  The warp stages four 16-byte column chunks
// per lane of eight rows at a time in its 16 KB of the (then idle) stage
// buffers with cp.async, so 32 copies per lane are in flight without
// holding registers; rows of no expert are zero-filled with weight 0, as
// in the combine kernel.
__device__ void combine_token(const GemmParams& p, int t, int lane, uint8_t* buf) {
  const int hv = p.H / 8, k = p.k;
  const long fb = (long)t * k;
  const uint32_t sb = smem_u32(buf);
  for (int cb = 0; cb < hv; cb += 128) {
    float acc[4][8];
#pragma unroll
    for (int q = 0; q < 4; ++q)
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[q][e] = 0.0f;
    for (int j0 = 0; j0 < k; j0 += 8) {
      float wgt[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const bool ok = j0 + j < k && p.s_pad_inv[fb + j0 + j] >= 0;
        wgt[j] = ok ? p.scores[fb + j0 + j] : 0.0f;
        const __nv_bfloat16* row = p.yk + (fb + min(j0 + j, k - 1)) * p.H;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int c = cb + lane + 32 * q;
          const bool in = ok && c < hv;
          cp_async_16(sb + ((q * 8 + j) * 32 + lane) * 16, row + (in ? c : 0) * 8, in ? 16u : 0u);
        }
      }
      asm volatile("cp.async.wait_all;" ::: "memory");
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (j0 + j < k) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            float y[8];
            unpack8_bf16(*reinterpret_cast<const uint4*>(buf + ((q * 8 + j) * 32 + lane) * 16), y);
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[q][e] = fmaf(wgt[j], y[e], acc[q][e]);
          }
        }
      }
    }
    uint4* orow = reinterpret_cast<uint4*>(p.out + (long)t * p.H);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int c = cb + lane + 32 * q;
      if (c < hv)
        orow[c] = make_uint4(pack_bf16x2(acc[q][0], acc[q][1]), pack_bf16x2(acc[q][2], acc[q][3]),
                             pack_bf16x2(acc[q][4], acc[q][5]), pack_bf16x2(acc[q][6], acc[q][7]));
    }
  }
}

// The combine phase, by each of the four gather warps and four epilogue
// warps: wait until the epilogue warps of every GEMM2 item have published
// their rows of y (one thread per CTA polls the global count, the other
// warps its outcome in shared memory), then take tokens from a device
// counter until none is left.  False: a bounded wait gave up.
__device__ bool fused_combine_phase(const GemmParams& p, Ctl* ctl, uint8_t* stages, int warp, int lane,
                                    const WaitCtx& wc) {
  volatile int* go = &ctl->combine_go;
  int state = 0;
  if (lane == 0) {
    if (warp == 6) {
      state = wait_flag_geq(hdr_word(p, kHdrG2Done), 4u * (uint32_t)(used_tiles(p) * p.n_tiles), wc) ? 1 : 2;
      __threadfence_block();
      *go = state;
    } else {
      const uint64_t t0 = globaltimer();
      for (uint32_t it = 1; (state = *go) == 0; ++it) {
        __nanosleep(128);
        if ((it & 15u) == 0 && (wait_aborted(wc) || globaltimer() - t0 > kWaitLimitNs)) {
          state = 2;
          break;
        }
      }
      __threadfence_block();
    }
  }
  state = __shfl_sync(0xffffffffu, state, 0);
  __syncwarp();  // the other lanes' loads of y after lane 0's acquire
  if (state != 1) return false;
  while (true) {
    int t = 0;
    if (lane == 0) t = atomicAdd(reinterpret_cast<int*>(hdr_word(p, kHdrCombineNext)), 1);
    t = __shfl_sync(0xffffffffu, t, 0);
    if (t >= p.T) break;
    // 16 KB of the stage buffers per warp: gather warps 6-9 slots 0-3,
    // epilogue warps 2-5 slots 4-7 (every GEMM2 item, hence every MMA
    // read of those buffers, is complete)
    combine_token(p, t, lane, stages + (warp >= 6 ? warp - 6 : warp + 2) * 16384);
  }
  return true;
}

// The gather warps' part of a schedule item or of the combine phase
// (false: a bounded wait gave up).
template <bool MX>
__device__ bool fused_aux_gather(const GemmParams& p, Ctl* ctl, uint8_t* stages, const Item& it, int gt,
                                 const WaitCtx& wc) {
  const int lane = gt & 31;
  bool ok = true;
  if (it.type == kItemCount) {
    fused_count(p, it.m, ctl->po, gt);
  } else if (it.type == kItemScan) {
    // thread 0 acquires the count items' completions and hands the outcome
    // to all 128 threads through shared memory, so that either all or none
    // of them enter the scan's barriers
    volatile int* go = ctl->order + 16;
    if (gt == 0) *go = wait_flag_geq(hdr_word(p, kHdrCountDone), (uint32_t)p.nchunks, wc) ? 1 : 0;
    gather_warps_sync();
    ok = *go != 0;
    if (ok) fused_scan(p, ctl->order, gt);
  } else if (it.type == kItemPlace) {
    // (one warp; the other three go on to the next item)
    if (gt < 32) {
      if (lane == 0) ok = wait_flag_geq(hdr_word(p, kHdrScanDone), 1u, wc);
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (ok) fused_place<MX>(p, it.m, ctl->po, lane);
    }
  } else {
    ok = fused_combine_phase(p, ctl, stages, 6 + (gt >> 5), lane, wc);
  }
  return ok;
}

// At exit, how long a CTA waits for copies still in flight after an abort.
constexpr uint64_t kDrainNs = 20000000ull;  // 20 ms

// ------------------------------------------------------------------ kernel
template <int MODE, bool MX, bool PAIR>
__global__ void __launch_bounds__(kGemmThreads, 1) gemm_kernel(const __grid_constant__ TmapSet maps,
                                                                const GemmParams p) {
  // CTA-pair launches: 6 stages of 16 KB A + 16 KB B (this CTA's half of a
  // 256-column B tile); otherwise 4 stages of 16 KB A + 32 KB B.  Both fill
  // the same 192 KB.
  constexpr int kSt = PAIR ? kPairStages : kStages;
  constexpr int kBSt = PAIR ? kAStage : kBStage;
  static_assert(kSt * (kAStage + kBSt) == kStages * (kAStage + kBStage), "stage layouts differ in size");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = base;
  uint8_t* sB = base + kSt * kAStage;
  Ctl* ctl = reinterpret_cast<Ctl*>(sB + kSt * kBSt);
  // per epilogue warp, one 4 KB output staging buffer (128-byte aligned)
  uint8_t* sOut = sB + kSt * kBSt + ((sizeof(Ctl) + 127) / 128) * 128;
  // MXFP8: per stage, the scale blocks of A (512 B) and B (1024 B)
  uint8_t* sSF = sOut + 4 * kOutStage;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const WaitCtx wc{&ctl->abort, &p.hdr[kHdrAbort], &p.hdr[kHdrError]};
  // MXFP8 launches always use the gather threads (scales of K-major operands)
  constexpr bool kGather = mode_gathers<MODE>() || MX;
  // MXFP8 keeps one accumulator (TMEM columns 256.. hold the stage scales)
  constexpr uint32_t kAccBufs = MX ? 1u : 2u;
  constexpr bool kWgrad = (MODE == GM_WG13 || MODE == GM_WG2);

  // Weight-gradient launches whose operands are all TMA-loaded (token-sorted
  // copies) take the gather warps out of the stage pipeline; those warps
  // write the empty experts' zero gradients instead.
  const bool gather_in_pipe = kGather && !PAIR && !(MODE == GM_DENSE && MX) && !(kWgrad && (MX || p.wg_sorted)) &&
                              !(MODE == GM_BWD_DA && p.rows_sorted) && !(MX && MODE == GM_BWD_DX) &&
                              !((MODE == GM_FWD_RING || MODE == GM_FWD1) && p.fwd_sorted);
  // The dense MXFP8 core's gather warps, which copy nothing, move each
  // stage's scale blocks from shared memory into TMEM with tcgen05.st
  // (replicated over the four lane quarters, the layout tcgen05.cp
  // .32x128b.warpx4 makes), so its MMA thread issues only MMAs; the blocks
  // complete on a barrier of their own (sffull) and a per-stage barrier
  // (sfready) tells the MMA thread the scales are in place (dense core
  // 2,004 -> 2,254 TFLOP/s at 8192^3).  The layer's GEMMs keep the copies
  // in the MMA thread: with the hand-off their k-steps were slower (Kimi-
  // shaped dA' 2.67 against 2.47 ms, dX 3.63 against 3.51).
  const bool sf_writer = MX && MODE == GM_DENSE && !gather_in_pipe;
  // MXFP8 ring launches whose gather warps copy nothing split each tile's
  // epilogue: warps 2-5 take the first half of every row's columns, warps
  // 6-9 (the same lane quarters) the second, so the single accumulator goes
  // back to the MMA thread in about half the time.  (dX's long K loop hides
  // its light epilogue already; dA''s, bound by its global loads and stores,
  // measured slower split.)
  const bool epi_split = MX && !PAIR && !gather_in_pipe && !sf_writer && MODE == GM_FWD_RING;
  // epilogue warps per tile (each ring GEMM1 tile's warps publish its rows)
  const uint32_t epi_warps = epi_split ? 8u : 4u;
  // CTA pairs: the leader's queue is read by its MMA and epilogue warps and
  // by the other CTA's TMA producer and epilogue warps (pair launches have
  // no gathered operand)
  const uint32_t queue_consumers = PAIR ? 10u : (gather_in_pipe || sf_writer || epi_split) ? 9u : 5u;
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  if (p.pdl_trigger) griddep_launch_dependents();
  if constexpr (MODE == GM_FWD_RING && !PAIR) {
    if (p.active_ctas != 0) {
      int n = p.active_ctas;
      if (n < 0) {
        const long a = p.hdr[kHdrSingles], b = 2l * p.hdr[kHdrPairs];
        n = b == 0 ? (int)gridDim.x : (int)((5 * a * gridDim.x + 5 * a + 4 * b - 1) / (5 * a + 4 * b));
      }
      if ((int)blockIdx.x >= (n > 0 ? n : 1)) return;  // before any barrier or TMEM use
    }
  }

  if (threadIdx.x == 0) {
    for (int i = 0; i < kSt; ++i) {
      // TMA producer's arrive.expect_tx, plus one no-increment arrival per
      // gather thread when the gather warps take part
      mbar_init(&ctl->full[i], gather_in_pipe ? 129u : 1u);
      mbar_init(&ctl->empty[i], 1);
      mbar_init(&ctl->sfready[i], 4);  // the four gather warps
      mbar_init(&ctl->sffull[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ctl->tfull[i], 1);
      // the epilogue warps that read the accumulator (both CTAs of a pair)
      mbar_init(&ctl->tempty[i], PAIR ? 8u : epi_warps);
    }
    for (int i = 0; i < kQueue; ++i) {
      mbar_init(&ctl->qfull[i], 1);
      mbar_init(&ctl->qempty[i], queue_consumers);
    }
    ctl->abort = 0;
    ctl->n_nonempty = 0;
    ctl->n_skip = 0;
    ctl->n_sel = 0;
    ctl->pair_rank = (int)rank;
    ctl->combine_go = 0;
    ctl->tmem_base = 0;  // a 512-column allocation always starts at column 0
    fence_mbar_init();
  }
  if (kWgrad) {
    for (int e = threadIdx.x; e <= p.E; e += blockDim.x) ctl->po[e] = p.padded_offsets[e];
    __syncthreads();
    // rank of each expert by descending padded rows (ties by expert id): the
    // same order in every CTA, a function of the schedule only.  An expert's
    // K loop covers its routed rows rounded up to one stage (64 rows; MXFP8:
    // 128, its padding); the rows past the count are zero in both operands.
    for (int e = threadIdx.x; e < p.E; e += blockDim.x) {
      const int ke = ctl->po[e + 1] - ctl->po[e];
      int pos = 0;
      for (int o = 0; o < p.E; ++o) {
        const int ko = ctl->po[o + 1] - ctl->po[o];
        pos += (ko > ke) || (ko == ke && o < e);
      }
      const int kit = MX ? ke / 128 : (p.counts[e] + 63) / 64;
      ctl->order[pos] = e | (kit << 10);
      if (ke > 0) atomicAdd(&ctl->n_nonempty, 1);
      if (ke >= p.wg_rows_max) atomicAdd(&ctl->n_skip, 1);
      if (ke > 0 && ke >= p.wg_rows_min && ke < p.wg_rows_max) atomicAdd(&ctl->n_sel, 1);
    }
  }
  if (warp == 0 && lane == 0)
    for (int i = 0; i < p.nmaps; ++i) tma_prefetch_desc(&maps.m[i]);
  if (warp == 1) {
    if constexpr (PAIR) {
      tmem_alloc_pair(&ctl->tmem_base, 512);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(&ctl->tmem_base, 512);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  // CTA pairs: both CTAs' barriers are initialised before either signals
  // the other's
  if constexpr (PAIR) cluster_sync();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  // (single-launch forward: known once the schedule items are done)
  int num_items = kWgrad ? ctl->n_sel * (PAIR ? p.m_tiles / 2 : p.m_tiles) * p.n_tiles
                  : (PAIR && MODE == GM_FWD_RING) ? p.hdr[kHdrPairs] * (p.g1_tiles + p.n_tiles)
                  : PAIR ? count_pair_items(p)
                  : MODE == GM_FWD_FUSED ? INT_MAX
                                         : count_items<MODE>(p);

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer + work fetch
    if (lane == 0) {
      uint32_t stage = 0, phase = 0, qs = 0, qp = 0, issued = 0;
      if (PAIR && rank != 0) {
        // the other CTA of a pair: take the leader's items from the queue it
        // fills, load this CTA's operand halves, and complete their bytes on
        // the leader's stage barrier
        while (true) {
          if (!mbar_wait_cluster(&ctl->qfull[qs], qp, wc)) break;
          const int w = ctl->q[qs];
          mbar_arrive_cluster(mapa_shared(&ctl->qempty[qs], 0));
          if (++qs == kQueue) { qs = 0; qp ^= 1; }
          if (w < 0) break;
          const Item it = decode<MODE, MX, PAIR>(p, ctl, w);
          bool ok = true;
          if (is_ring<MODE>() && it.type == GM_FWD2) {
            // this CTA loads the ring rows of its own tile: acquire their
            // GEMM1 completion itself, then order the async-proxy loads after it
            ok = wait_flag_geq(&p.ring_flags[it.rp], epi_warps * (uint32_t)p.g1_tiles, wc);
            fence_proxy_async_global();
            if (!ok) break;
          }
          for (int kk = 0; kk < it.k_iters; ++kk) {
            if (!mbar_wait(&ctl->empty[stage], phase ^ 1, wc)) { ok = false; break; }
            tma_loads_pair<MODE>(maps, p, it, kk, 1, sA + stage * kAStage, sB + stage * kBSt,
                                 mapa_shared(&ctl->full[stage], 0));
            ++issued;
            if (++stage == kSt) { stage = 0; phase ^= 1; }
          }
          if (!ok) break;
        }
        // the leader's MMAs read these stages: wait for their release (which
        // also means the copies landed) before the CTA may leave
        const uint64_t t0 = globaltimer();
        for (uint32_t j = 0; j < kSt; ++j) {
          const uint64_t spent = globaltimer() - t0;
          if (spent < kDrainNs) mbar_drain(&ctl->empty[stage], phase ^ 1, kDrainNs - spent);
          if (++stage == kSt) { stage = 0; phase ^= 1; }
        }
      } else {
        uint32_t* counter = reinterpret_cast<uint32_t*>(&p.hdr[kHdrCounters + p.counter]);
        // Weight-gradient launches take two consecutive counter values per
        // fetch -- one item from each end of the descending-K list (see
        // decode), so every CTA runs a long tile and a short one back to
        // back -- and keep two such pairs in flight, so a run of short items
        // does not pay an atomic round trip each.  Launches with long items
        // fetch one ahead (holding more would cost tail balance and, in the
        // ring launch, delay the GEMM2 tiles other CTAs wait on).
        int w = (int)atomicAdd(counter, kWgrad ? 2u : 1u);
        int f1 = 0, f2 = 0, f3 = 0;
        if (kWgrad) {
          f1 = w + 1;
          f2 = (int)atomicAdd(counter, 2u);
          f3 = f2 + 1;
        }
        bool ok = true;
        bool sched_ready = false, combine_sent = false;
        while (ok) {
          if (MODE == GM_FWD_FUSED && !sched_ready && w >= fused_ring_base(p)) {
            // the ring's and the combine's items read the whole schedule:
            // acquire the place items' completions before publishing them
            sched_ready = true;
            if (wait_flag_geq(hdr_word(p, kHdrPlaceDone), (uint32_t)p.nchunks, wc)) {
              num_items = fused_total(p);
              // (MXFP8: this thread's TMA then reads the place items' tiled scales)
              if constexpr (MX) fence_proxy_async_global();
            } else {
              w = -1;
            }
          }
          if (MODE == GM_FWD_FUSED && w >= num_items && num_items != INT_MAX && !combine_sent) {
            // past the last item: this CTA's combine phase, then the end
            w = num_items;
            combine_sent = true;
          } else if (w >= num_items) {
            w = -1;
          }
          ok = PAIR ? mbar_wait_cluster(&ctl->qempty[qs], qp ^ 1, wc) : mbar_wait(&ctl->qempty[qs], qp ^ 1, wc);
          const int wq = ok ? w : -1;
          ctl->q[qs] = wq;
          if constexpr (PAIR) {
            // the same item for the other CTA of the pair
            st_cluster_u32(mapa_shared(&ctl->q[qs], 1), (uint32_t)wq);
            mbar_arrive_cluster(mapa_shared(&ctl->qfull[qs], 1));
          }
          mbar_arrive(&ctl->qfull[qs]);
          if (++qs == kQueue) { qs = 0; qp ^= 1; }
          if (!ok || w < 0) break;
          int w_next;
          if (kWgrad) {
            w_next = f1;
            f1 = f2;
            f2 = f3;
            f3 = (f2 & 1) ? (int)atomicAdd(counter, 2u) : f2 + 1;
          } else {
            w_next = (int)atomicAdd(counter, 1u);
          }
          const Item it = decode<MODE, MX, PAIR>(p, ctl, w);
          if (is_ring<MODE>() && it.type == GM_FWD2) {
            // GEMM2 of a tile reads the ring rows GEMM1 wrote: wait until all
            // of its GEMM1 column tiles are published, then order the
            // async-proxy loads after the acquire
            ok = wait_flag_geq(&p.ring_flags[it.rp], epi_warps * (uint32_t)p.g1_tiles, wc);
            fence_proxy_async_global();
            if (!ok) break;
          }
          // CTA pairs: this CTA's 32 KB and the other CTA's 32 KB
          const uint32_t bytes = PAIR ? 4u * kAStage
                                 : MX ? mx_stage_bytes<MODE>(p, it.type, item_bn(p, it.type))
                                      : tma_stage_bytes(p, it.type, item_bn(p, it.type));
          for (int kk = 0; kk < it.k_iters; ++kk) {
            if (!mbar_wait(&ctl->empty[stage], phase ^ 1, wc)) { ok = false; break; }
            if (MX && sf_writer) {
              // the scale blocks complete on a barrier of their own, so the
              // gather warps move them into TMEM while the operands land
              const uint32_t sfb = mx_sf_bytes(item_bn(p, it.type));
              mbar_arrive_expect_tx(&ctl->full[stage], bytes - sfb);
              mbar_arrive_expect_tx(&ctl->sffull[stage], sfb);
            } else {
              mbar_arrive_expect_tx(&ctl->full[stage], bytes);
            }
            if constexpr (PAIR)
              tma_loads_pair<MODE>(maps, p, it, kk, 0, sA + stage * kAStage, sB + stage * kBSt,
                                   mapa_shared(&ctl->full[stage], 0));
            else if constexpr (MX)
              tma_loads_mx<MODE>(maps, p, it, kk, sA + stage * kAStage, sB + stage * kBSt, sSF + stage * kSfStage,
                                 sSF + stage * kSfStage + 512, &ctl->full[stage],
                                 sf_writer ? &ctl->sffull[stage] : &ctl->full[stage]);
            else
              tma_loads<MODE>(maps, p, it, kk, sA + stage * kAStage, sB + stage * kBSt, &ctl->full[stage]);
            ++issued;
            if (++stage == kSt) { stage = 0; phase ^= 1; }
          }
          w = w_next;
        }
        // let the copies in flight land before the CTA may leave (after an
        // abort the MMA warp may not have waited for them): the last fills
        // of each stage, newest first
        const uint64_t t0 = globaltimer();
        const uint32_t last = issued < (uint32_t)kSt ? issued : (uint32_t)kSt;
        for (uint32_t j = 1; j <= last; ++j) {
          const uint32_t f = issued - j;
          const uint64_t spent = globaltimer() - t0;
          if (spent < kDrainNs) mbar_drain(&ctl->full[f % kSt], (f / kSt) & 1u, kDrainNs - spent);
          if (MX && sf_writer) {
            const uint64_t spent2 = globaltimer() - t0;
            if (spent2 < kDrainNs) mbar_drain(&ctl->sffull[f % kSt], (f / kSt) & 1u, kDrainNs - spent2);
          }
        }
      }
    }
    // lanes 1-31 skipped the producer loop: the warp reaches the final
    // barrier converged
    __syncwarp();
  } else if (warp >= 6 && !epi_split) {
    // ---------------------------------------------------------------- gather producers
    if (gather_in_pipe) {
      const int gt = threadIdx.x - 192;
      uint32_t stage = 0, phase = 0, qs = 0, qp = 0;
      while (true) {
        if (!mbar_wait(&ctl->qfull[qs], qp, wc)) break;
        const int w = ctl->q[qs];
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->qempty[qs]);
        if (++qs == kQueue) { qs = 0; qp ^= 1; }
        if (w < 0) break;
        const Item it = decode<MODE, MX, PAIR>(p, ctl, w);
        bool ok = true;
        if constexpr (MODE == GM_FWD_FUSED) {
          if (it.type >= kItemCount) {
            if (!fused_aux_gather<MX>(p, ctl, sA, it, gt, wc)) break;
            continue;
          }
        }
        if constexpr (MX) {
          int tok[8];
          int tok_row = -1;
          const bool ga = (MODE != GM_DENSE) && (it.type == GM_FWD1 || it.type == GM_BWD_DA);
#pragma unroll
          for (int j = 0; j < 8; ++j) tok[j] = ga ? token_or_neg(p, it.row0 + (gt >> 3) + 16 * j) : -1;
          if (ga) tok_row = token_or_neg(p, it.row0 + gt);
          const bool copies = (MODE == GM_DENSE) || !(it.type == GM_WG13 || it.type == GM_WG2);
          for (int kk = 0; kk < it.k_iters; ++kk) {
            if (!mbar_wait(&ctl->empty[stage], phase ^ 1, wc)) { ok = false; break; }
            if (copies)
              gather_stage_mx<MODE>(p, it, kk, sA + stage * kAStage, sSF + stage * kSfStage,
                                    sSF + stage * kSfStage + 512, gt, tok, tok_row, &ctl->full[stage]);
            else
              mbar_arrive(&ctl->full[stage]);
            if (++stage == kStages) { stage = 0; phase ^= 1; }
          }
        } else if (gathered_operand(p, it.type) == 0)
          ok = gather_item_k<kSt>(p, it, sA, ctl, stage, phase, gt, wc);
        else if (it.type == GM_WG13)
          ok = gather_item_mn<16, kSt>(p, it, sA, kAStage, it.m * 128, ctl, stage, phase, gt, wc);
        else if (it.type == GM_WG2 && p.bn == 256)
          ok = gather_item_mn<32, kSt>(p, it, sB, kBSt, it.n * p.bn, ctl, stage, phase, gt, wc);
        else if (it.type == GM_WG2)
          ok = gather_item_mn<16, kSt>(p, it, sB, kBSt, it.n * p.bn, ctl, stage, phase, gt, wc);
        else
          ok = gather_item_k<kSt>(p, it, sA, ctl, stage, phase, gt, wc);
        if (!ok) break;
      }
      // let this thread's copies land before the CTA can exit
      asm volatile("cp.async.wait_all;" ::: "memory");
    } else if (sf_writer) {
      // each lane writes, in its warp's lane quarter, the 16 bytes at
      // lane * 16 of each 512-byte scale block: 4 columns (A), then 4 per
      // 128 columns of the B tile
      const uint32_t lanes = (uint32_t)((warp & 3) * 32) << 16;
      uint32_t stage = 0, phase = 0, qs = 0, qp = 0;
      while (true) {
        if (!mbar_wait(&ctl->qfull[qs], qp, wc)) break;
        const int w = ctl->q[qs];
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->qempty[qs]);
        if (++qs == kQueue) { qs = 0; qp ^= 1; }
        if (w < 0) break;
        const Item it = decode<MODE, MX, PAIR>(p, ctl, w);
        const int bchunks = item_bn(p, it.type) / 128;
        bool ok = true;
        for (int kk = 0; kk < it.k_iters; ++kk) {
          if (!mbar_wait(&ctl->sffull[stage], phase, wc)) { ok = false; break; }
          const uint8_t* sfs = sSF + stage * kSfStage + lane * 16;
          const uint32_t col = tmem + lanes + 256u + (uint32_t)stage * 16u;
          tmem_st4(col, *reinterpret_cast<const uint4*>(sfs));
          for (int c = 0; c < bchunks; ++c)
            tmem_st4(col + 4u + 4u * (uint32_t)c, *reinterpret_cast<const uint4*>(sfs + 512 + c * 512));
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&ctl->sfready[stage]);
          if (++stage == kStages) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
      }
    }
    if (kWgrad && p.wg_rows_min == 0) zero_empty_experts<MODE>(p, ctl, warp - 6, lane);
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    // (CTA pairs: the leader issues the pair's MMAs; the other CTA's MMA
    // warp only takes part in the TMEM allocation)
    uint32_t stage = 0, phase = 0, qs = 0, qp = 0, tcount = 0;
    while (!PAIR || rank == 0) {
      if (!mbar_wait(&ctl->qfull[qs], qp, wc)) break;
      const int w = ctl->q[qs];
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->qempty[qs]);
      if (++qs == kQueue) { qs = 0; qp ^= 1; }
      if (w < 0) break;
      const Item it = decode<MODE, MX, PAIR>(p, ctl, w);
      if (MODE == GM_FWD_FUSED && it.type >= kItemCount) continue;  // no MMA
      const uint32_t buf = tcount % kAccBufs, tph = (tcount / kAccBufs) & 1;
      // (CTA pairs: released by both CTAs' epilogue warps)
      if (!(PAIR ? mbar_wait_cluster(&ctl->tempty[buf], tph ^ 1, wc) : mbar_wait(&ctl->tempty[buf], tph ^ 1, wc)))
        break;
      tc_fence_after();
      const int bn = item_bn(p, it.type);
      const bool amn = a_mn_major<MODE>(p, it.type), bmn = b_mn_major<MODE>(p, it.type);
      const uint32_t idesc = PAIR ? idesc_bf16(256, 256, amn ? 1 : 0, bmn ? 1 : 0)
                                  : idesc_bf16(128, bn, amn ? 1 : 0, bmn ? 1 : 0);
      const uint32_t d = tmem + buf * 256;
      const bool gathered = gathered_operand(p, it.type) != 0;
      bool ok = true;
      for (int kk = 0; kk < it.k_iters; ++kk) {
        if (!mbar_wait(&ctl->full[stage], phase, wc)) { ok = false; break; }
        if (MX && sf_writer && !mbar_wait(&ctl->sfready[stage], phase, wc)) { ok = false; break; }
        tc_fence_after();
        if (lane == 0) {
          // the gather threads wrote part of this stage with cp.async: order
          // those writes before the tensor core's (async-proxy) reads
          if (gathered || (MX && gather_in_pipe)) fence_proxy_async_shared();
          const uint32_t a0 = smem_u32(sA + stage * kAStage), b0 = smem_u32(sB + stage * kBSt);
          if constexpr (MX) {
            // stage scales into TMEM (columns 256 + 16 * stage): A at +0
            // (4 columns), B at +4 (4 columns per 128 N)
            const uint32_t sf_t = tmem + 256 + stage * 16;
            if (!sf_writer) {
              const uint32_t sfa_s = smem_u32(sSF + stage * kSfStage);
              tmem_cp_32x128b_warpx4(sf_t, sdesc_plain(sfa_s, 16, 128));
              for (int c = 0; c < bn / 128; ++c)
                tmem_cp_32x128b_warpx4(sf_t + 4 + 4 * c, sdesc_plain(sfa_s + 512 + c * 512, 16, 128));
            }
#pragma unroll
            for (int k32 = 0; k32 < 4; ++k32) {
              const uint64_t ad = amn ? sdesc_sw128(a0 + k32 * 4096, 16384, 1024) : sdesc_sw128(a0 + k32 * 32, 16, 1024);
              const uint64_t bd = bmn ? sdesc_sw128(b0 + k32 * 4096, 16384, 1024) : sdesc_sw128(b0 + k32 * 32, 16, 1024);
              mma_mxf8(d, ad, bd, idesc_mxf8(128, bn, amn ? 1 : 0, bmn ? 1 : 0, k32, k32), sf_t, sf_t + 4,
                       (kk | k32) != 0 ? 1u : 0u);
            }
          } else {
#pragma unroll
            for (int k16 = 0; k16 < 4; ++k16) {
              const uint64_t ad = amn ? sdesc_sw128(a0 + k16 * 2048, 8192, 1024) : sdesc_sw128(a0 + k16 * 32, 16, 1024);
              const uint64_t bd = bmn ? sdesc_sw128(b0 + k16 * 2048, 8192, 1024) : sdesc_sw128(b0 + k16 * 32, 16, 1024);
              if constexpr (PAIR)
                mma_bf16_pair(d, ad, bd, idesc, (kk | k16) != 0 ? 1u : 0u);
              else
                mma_bf16(d, ad, bd, idesc, (kk | k16) != 0 ? 1u : 0u);
            }
          }
          // CTA pairs: releases the stage in both CTAs
          if constexpr (PAIR)
            mma_commit_pair(&ctl->empty[stage]);
          else
            mma_commit(&ctl->empty[stage]);
        }
        __syncwarp();
        if (++stage == kSt) { stage = 0; phase ^= 1; }
      }
      if (!ok) break;
      if (lane == 0) {
        if constexpr (PAIR)
          mma_commit_pair(&ctl->tfull[buf]);
        else
          mma_commit(&ctl->tfull[buf]);
      }
      __syncwarp();
      ++tcount;
    }
  } else {
    // ---------------------------------------------------------------- epilogue (warps 2..5)
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int row = q * 32 + lane;
    // split epilogues: warps 2-5 the first half of each row (hm 1), warps
    // 6-9 the second (hm 2, no staging buffer); otherwise the whole row (0)
    const int hm = epi_split ? (warp >= 6 ? 2 : 1) : 0;
    uint8_t* stage_out = warp < 6 ? sOut + (warp - 2) * kOutStage : nullptr;
    uint32_t qs = 0, qp = 0, tcount = 0;
    while (true) {
      if (!(PAIR ? mbar_wait_cluster(&ctl->qfull[qs], qp, wc) : mbar_wait(&ctl->qfull[qs], qp, wc))) break;
      const int w = ctl->q[qs];
      __syncwarp();
      if (lane == 0) {
        // CTA pairs: every consumer releases the leader's queue slot
        if constexpr (PAIR)
          mbar_arrive_cluster(mapa_shared(&ctl->qempty[qs], 0));
        else
          mbar_arrive(&ctl->qempty[qs]);
      }
      if (++qs == kQueue) { qs = 0; qp ^= 1; }
      if (w < 0) break;
      const Item it = decode<MODE, MX, PAIR>(p, ctl, w);
      if (MODE == GM_FWD_FUSED && it.type >= kItemCount) {
        // schedule items are the gather warps'; the combine phase is shared
        if (it.type == kItemCombine && !fused_combine_phase(p, ctl, sA, warp, lane, wc)) break;
        continue;
      }
      const uint32_t buf = tcount % kAccBufs, tph = (tcount / kAccBufs) & 1;
      if (!mbar_wait(&ctl->tfull[buf], tph, wc)) break;
      tc_fence_after();
      const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + buf * 256;
      // hands the accumulator back to the MMA warp, once per tile
      bool released = false;
      auto release_acc = [&]() {
        if (released) return;
        released = true;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          // CTA pairs: the leader's MMA warp waits for both CTAs' epilogues
          if constexpr (PAIR)
            mbar_arrive_cluster(mapa_shared(&ctl->tempty[buf], 0));
          else
            mbar_arrive(&ctl->tempty[buf]);
        }
      };
      if (is_ring<MODE>() && it.type == GM_FWD2 && warp == 2 && lane == 0) {
        // the accumulator is complete, so every load of this tile's ring
        // rows has landed: release the rows for reuse.  The idle CTA of a
        // solo pair releases its own walk position, 2u + 1 (its item names
        // the leader's, 2u): no tile writes or reads that position's rows,
        // but the GEMM1 that reuses its slot a ring later waits on it.
        red_release_gpu_add(&p.ring_flags[p.m_tiles + it.rp + (it.idle ? 1 : 0)], 1u);
      }
      bool ok = true;
      if (is_ring<MODE>() && it.type == GM_FWD1 && !it.idle) {
        // the ring slot rows this tile writes were last read by GEMM2 of the
        // tile ring_slots minibatches back; each warp waits on its own (no
        // CTA-level barrier on a path that a bounded wait can abandon)
        const int back = it.rp - p.ring_slots * (p.ring_rows / kTileRows);
        if (back >= 0) {
          if (lane == 0) ok = wait_flag_geq(&p.ring_flags[p.m_tiles + back], (uint32_t)p.n_tiles, wc);
          ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        }
      }
      if (!ok) break;
      // (the idle CTA of a solo pair only hands the accumulator back)
      switch (it.idle ? -1 : it.type) {
        case -1: break;
        case GM_DENSE: epi_dense(p, it, tbase, row); break;
        case GM_FWD1:
          if constexpr (MX) epi_fwd1_mx(p, it, tbase, row, lane, stage_out, release_acc, hm);
          else epi_fwd1(p, it, tbase, row);
          break;
        case GM_FWD2:
        case GM_BWD_DX:
          if constexpr (MX) epi_scatter_mx(p, it, tbase, row, p.bn, lane, stage_out, release_acc, hm);
          else epi_scatter(p, it, tbase, row, p.bn);
          break;
        case GM_BWD_DA: epi_bwd_da<MX>(p, it, tbase, row, release_acc); break;
        default: epi_wgrad<MX>(p, it, tbase, q, lane, stage_out, release_acc); break;
      }
      release_acc();
      if (MODE == GM_FWD_FUSED && it.type == GM_FWD2) {
        // this warp's 32 rows of y are stored: count them for the combine
        // phase, which waits on every GEMM2 item (all drawn before it)
        __syncwarp();
        if (lane == 0) {
          __threadfence();
          red_release_gpu_add(hdr_word(p, kHdrG2Done), 1u);
        }
      }
      if (is_ring<MODE>() && it.type == GM_FWD1 && !it.idle) {
        // publish this warp's 32 ring rows of the tile to GEMM2 (another CTA,
        // read by TMA): each epilogue warp adds 1, so a tile is complete when
        // its counter reaches (epilogue warps per tile) * (GEMM1 column tiles)
        fence_proxy_async_global();
        __syncwarp();
        if (lane == 0) {
          const bool skip = (p.debug_flags & MOK_DEBUG_SKIP_RING_SIGNAL) && it.m == 0 && it.n == 0 && warp == 2;
          __threadfence();
          if (!skip) red_release_gpu_add(&p.ring_flags[it.rp], 1u);
        }
      }
      ++tcount;
    }
  }

  tc_fence_before();
  // (the non-aligned barrier form, defined for warps that arrive diverged;
  // the aligned __syncthreads form is not)
  asm volatile("barrier.sync 0;" ::: "memory");
  // CTA pairs: neither CTA leaves (nor frees TMEM) while the other may
  // still signal its barriers or run MMAs on its smem and TMEM
  if constexpr (PAIR) cluster_sync();
  tc_fence_after();
  if (warp == 1) {
    if constexpr (PAIR)
      tmem_dealloc_pair(tmem, 512);
    else
      tmem_dealloc(tmem, 512);
  }
  if (p.pdl_wait_end) griddep_wait();
}

template <int MODE, bool MX>
cudaError_t launch_mode(const TmapSet& maps, const GemmParams& p, int grid, cudaStream_t st) {
  const size_t smem = gemm_smem_bytes();
  static int configured_device = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_device != dev) {
    e = cudaFuncSetAttribute(gemm_kernel<MODE, MX, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  if (!p.pdl_launch) {
    gemm_kernel<MODE, MX, false><<<grid, kGemmThreads, smem, st>>>(maps, p);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3(kGemmThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, gemm_kernel<MODE, MX, false>, maps, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// Clusters of two CTAs.  The grid is the number of such clusters the device
// holds at once (each CTA needs a whole SM's shared memory), so the
// persistent CTAs are all resident.
template <int MODE>
cudaError_t launch_pair_mode(const TmapSet& maps, const GemmParams& p, int grid, cudaStream_t st) {
  const size_t smem = gemm_smem_bytes();
  static int configured_device = -1;
  static int pair_grid = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.blockDim = dim3(kGemmThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (configured_device != dev) {
    e = cudaFuncSetAttribute(gemm_kernel<MODE, false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3((unsigned)(grid & ~1), 1, 1);
    int clusters = 0;
    e = cudaOccupancyMaxActiveClusters(&clusters, gemm_kernel<MODE, false, true>, &cfg);
    if (e != cudaSuccess) return e;
    pair_grid = 2 * clusters;
    configured_device = dev;
  }
  const int g = (grid & ~1) < pair_grid ? (grid & ~1) : pair_grid;
  if (g < 2) return cudaErrorNotSupported;
  cfg.gridDim = dim3((unsigned)g, 1, 1);
  cfg.numAttrs = p.pdl_launch ? 2 : 1;
  e = cudaLaunchKernelEx(&cfg, gemm_kernel<MODE, false, true>, maps, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

int gemm_pair_capacity() {
  const size_t smem = gemm_smem_bytes();
  if (cudaFuncSetAttribute(gemm_kernel<GM_FWD_RING, false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess)
    return 0;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(kGemmThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, gemm_kernel<GM_FWD_RING, false, true>, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  return 2 * clusters;
}

size_t gemm_smem_bytes() {
  return 1024 + kStages * (kAStage + kBStage) + ((sizeof(Ctl) + 127) / 128) * 128 + 4 * kOutStage +
         kStages * kSfStage;
}

cudaError_t launch_gemm(int mode, const TmapSet& maps, const GemmParams& p, int grid, cudaStream_t st) {
  switch (mode) {
    case GM_DENSE: return launch_mode<GM_DENSE, false>(maps, p, grid, st);
    case GM_FWD1: return launch_mode<GM_FWD1, false>(maps, p, grid, st);
    case GM_FWD2: return launch_mode<GM_FWD2, false>(maps, p, grid, st);
    case GM_BWD_DA: return launch_mode<GM_BWD_DA, false>(maps, p, grid, st);
    case GM_BWD_DX: return launch_mode<GM_BWD_DX, false>(maps, p, grid, st);
    case GM_WG13: return launch_mode<GM_WG13, false>(maps, p, grid, st);
    case GM_WG2: return launch_mode<GM_WG2, false>(maps, p, grid, st);
    case GM_FWD_RING: return launch_mode<GM_FWD_RING, false>(maps, p, grid, st);
    case GM_FWD_FUSED: return launch_mode<GM_FWD_FUSED, false>(maps, p, grid, st);
    default: return cudaErrorInvalidValue;
  }
}

// MXFP8 (block-scaled E4M3) launches of the same kernel family.
cudaError_t launch_gemm_mx(int mode, const TmapSet& maps, const GemmParams& p, int grid, cudaStream_t st) {
  switch (mode) {
    case GM_DENSE: return launch_mode<GM_DENSE, true>(maps, p, grid, st);
    case GM_FWD1: return launch_mode<GM_FWD1, true>(maps, p, grid, st);
    case GM_BWD_DA: return launch_mode<GM_BWD_DA, true>(maps, p, grid, st);
    case GM_BWD_DX: return launch_mode<GM_BWD_DX, true>(maps, p, grid, st);
    case GM_WG13: return launch_mode<GM_WG13, true>(maps, p, grid, st);
    case GM_WG2: return launch_mode<GM_WG2, true>(maps, p, grid, st);
    case GM_FWD_RING: return launch_mode<GM_FWD_RING, true>(maps, p, grid, st);
    case GM_FWD_FUSED: return launch_mode<GM_FWD_FUSED, true>(maps, p, grid, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_gemm_pair(int mode, const TmapSet& maps, const GemmParams& p, int grid, cudaStream_t st) {
  if (p.bn != 256) return cudaErrorInvalidValue;
  if (mode == GM_WG13 || mode == GM_WG2) {
    if (!p.wg_sorted || p.m_tiles % 2 != 0) return cudaErrorInvalidValue;
  } else if (mode == GM_FWD_RING) {
    if (!p.pair_m0 || !p.fwd_sorted || p.ring_count_word != kHdrPairs || (p.ring_rows / kTileRows) % 2)
      return cudaErrorInvalidValue;
  } else if (!p.pair_m0 || (mode == GM_BWD_DA && !p.rows_sorted)) {
    return cudaErrorInvalidValue;
  }
  switch (mode) {
    case GM_FWD_RING: return launch_pair_mode<GM_FWD_RING>(maps, p, grid, st);
    case GM_WG13: return launch_pair_mode<GM_WG13>(maps, p, grid, st);
    case GM_WG2: return launch_pair_mode<GM_WG2>(maps, p, grid, st);
    case GM_BWD_DA: return launch_pair_mode<GM_BWD_DA>(maps, p, grid, st);
    case GM_BWD_DX: return launch_pair_mode<GM_BWD_DX>(maps, p, grid, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace mok

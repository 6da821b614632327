// C ABI of libmok.so: argument checks, workspace layout, tensor maps and the
// launch sequence of each call.  Everything here runs on the host and only
// enqueues work on the caller's stream.
#include <math.h>
#include <limits.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <mutex>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "gemm.cuh"

namespace mok {

namespace {

constexpr int kMaxDevices = 64;

size_t align256(size_t b) { return (b + 255) & ~size_t(255); }

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

}  // namespace

int device_sm_count() {
  static int cache[kMaxDevices] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev < kMaxDevices && cache[dev]) return cache[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev < kMaxDevices) cache[dev] = n;
  return n;
}

bool make_tmap(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* ptr, const uint64_t* dims,
               const uint64_t* strides_bytes, const uint32_t* box, bool swizzle128) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t d[5], s[4];
  cuuint32_t b[5], es[5] = {1, 1, 1, 1, 1};
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
  }
  for (int i = 0; i + 1 < rank; ++i) s[i] = strides_bytes[i];
  const CUresult r = fn(m, dt, (cuuint32_t)rank, const_cast<void*>(ptr), d, s, b, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int effective_minibatch_rows(const mok_shape& s, const mok_config& c, int num_sms) {
  // a minibatch is a whole number of 128-row tiles (a requested size is rounded up)
  if (c.minibatch_rows > 0) return (c.minibatch_rows + kTileRows - 1) / kTileRows * kTileRows;
  // two full waves of 128 x 256 output tiles over the narrower grouped GEMM
  const double rows = 2.0 * num_sms * 128.0 * 256.0 / (double)(2 * s.I < s.H ? 2 * s.I : s.H);
  int m = (int)ceil(rows / kTileRows) * kTileRows;
  return m < kTileRows ? kTileRows : m;
}

WsLayout ws_layout(const mok_shape& s, const mok_config& c, mok_precision prec, int num_sms) {
  WsLayout L;
  memset(&L, 0, sizeof(L));
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += align256(bytes);
    return o;
  };
  const int64_t R = (int64_t)s.T * s.k;
  L.pad_capacity = (R + (int64_t)s.E * (kTileRows - 1)) / kTileRows * kTileRows;
  L.tile_capacity = L.pad_capacity / kTileRows;
  L.nchunks = (R + kSchedChunk - 1) / kSchedChunk;
  int M = effective_minibatch_rows(s, c, num_sms);
  if (M > L.pad_capacity) M = (int)L.pad_capacity;
  L.minibatch_rows = M;
  L.ring_slots = c.ring_slots > 0 ? c.ring_slots : 4;
  const size_t I = s.I, H = s.H, P = L.pad_capacity;
  L.header = take(kHeaderWords * 4);
  L.counts = take(s.E * 4);
  L.offsets = take((s.E + 1) * 4);
  L.padded_offsets = take((s.E + 1) * 4);
  L.perm = take(R * 4);
  L.inv_perm = take(R * 4);
  L.pad_perm = take(P * 4);
  L.pad_inv = take(R * 4);
  L.tile_expert = take(L.tile_capacity * 4);
  L.chunk_hist = take(L.nchunks * s.E * 4);
  L.chunk_base = take(L.nchunks * s.E * 4);
  // ring flags: two halves (rows published, rows consumed) of 2 *
  // tile_capacity walk positions each -- a CTA-pair ring's walk has two
  // positions per unit, a solo unit's second one empty
  L.ring_flags = take(4 * L.tile_capacity * 4);
  L.ring = take((size_t)L.ring_slots * M * I * 2);
  if (prec == MOK_BF16) {
    L.ring_flags2 = take(4 * L.tile_capacity * 4);
    L.ring2 = take((size_t)L.ring_slots * M * I * 2);
  }
  L.yk = take((size_t)R * H * 2);
  L.dhu = take(P * 2 * I * 2);
  L.as = take(P * I * 2);
  L.dsp = take(P * (I / 128) * 4);
  L.sorted = prec == MOK_BF16 ? take(P * H * 2) : 0;
  L.sorted2 = prec == MOK_BF16 ? take(P * H * 2) : 0;
  L.pair_m0 = take(L.tile_capacity * 4);
  L.pair_mb = take((L.tile_capacity + 2) * 4);
  if (prec == MOK_MXFP8) {
    L.ring_sf = take((size_t)L.ring_slots * M * (I / 32));
    L.xq = take((size_t)s.T * H);
    L.xsf = take((size_t)s.T * (H / 32));
    L.xq_sorted = take(P * H);
    L.wsf1 = take(2 * (size_t)s.E * H * I / 32);
    L.wsf3 = L.wsf1 + (size_t)s.E * H * I / 32;
    L.wsf2 = take((size_t)s.E * I * H / 32);
    L.dhuq = take(P * 2 * I);
    L.dhusf = take(P * (2 * I / 32));
    L.sfa_rows_t = take(P * (std::max(H, 2 * I) / 32));
    L.wqa = take(P * H);
    L.wsfa = take(P * H / 32);
    L.wqb = take(P * 2 * I);
    L.wsfb = take(P * 2 * I / 32);
  }
  L.total = off;
  return L;
}

}  // namespace mok

using namespace mok;

namespace {

// ---------------------------------------------------------------- tracing
std::atomic<int64_t> g_launches{0};
std::mutex g_trace_mu;
bool g_trace_on = false;
struct TraceRec {
  int phase;
  cudaEvent_t a, b;
};
std::vector<TraceRec> g_trace;

// Records an event pair around one phase of a call (when tracing is on) and
// counts the phase's kernel launches.
// Names of the phases, for the NVTX ranges each call opens around them
// (host-side ranges: they mark when the launches were issued; a profiler
// that follows NVTX into the device shows the kernels under them).
const char* const kPhaseNames[MOK_NUM_PHASES] = {
    "mok schedule",  "mok fwd gemm",   "mok fwd combine", "mok bwd dA'",      "mok bwd ds",
    "mok bwd dX",    "mok bwd dX combine", "mok bwd dW1|dW3", "mok bwd dW2",   "mok mxfp8 quant",
    "mok bwd sort",  "mok router fwd", "mok router bwd",  "mok bwd replay",   "mok fwd fused",
    "mok fwd sort"};

class Phase {
 public:
  Phase(int phase, cudaStream_t st, int kernels) : st_(st) {
    g_launches += kernels;
    nvtxRangePushA(phase >= 0 && phase < MOK_NUM_PHASES ? kPhaseNames[phase] : "mok");
    std::lock_guard<std::mutex> lk(g_trace_mu);
    if (!g_trace_on) return;
    rec_.phase = phase;
    if (cudaEventCreate(&rec_.a) != cudaSuccess || cudaEventCreate(&rec_.b) != cudaSuccess) return;
    cudaEventRecord(rec_.a, st_);
    on_ = true;
  }
  ~Phase() {
    nvtxRangePop();
    if (!on_) return;
    cudaEventRecord(rec_.b, st_);
    std::lock_guard<std::mutex> lk(g_trace_mu);
    g_trace.push_back(rec_);
  }

 private:
  cudaStream_t st_;
  TraceRec rec_{};
  bool on_ = false;
};

}  // namespace

namespace {

const char* kStatusNames[] = {"MOK_OK",           "MOK_ERR_INVALID_ARG", "MOK_ERR_UNSUPPORTED",
                              "MOK_ERR_WORKSPACE_TOO_SMALL", "MOK_ERR_CUDA", "MOK_ERR_BAD_INDEX",
                              "MOK_ERR_TIMEOUT"};

mok_status check_shape(const mok_shape* s) {
  if (!s) return MOK_ERR_INVALID_ARG;
  if (s->T < 1 || s->H < 1 || s->I < 1 || s->E < 1 || s->k < 1) return MOK_ERR_INVALID_ARG;
  if (s->H % 128 || s->I % 128) return MOK_ERR_UNSUPPORTED;
  if (s->E > 1024 || s->k > 32) return MOK_ERR_UNSUPPORTED;
  if ((int64_t)s->T * s->k > (1 << 24)) return MOK_ERR_UNSUPPORTED;
  return MOK_OK;
}

mok_status check_config(const mok_config* c) {
  if (!c) return MOK_ERR_INVALID_ARG;
  if (c->comm_sms != 0) return MOK_ERR_INVALID_ARG;
  if (c->minibatch_rows < 0) return MOK_ERR_INVALID_ARG;
  if (c->ring_slots < 0 || c->ring_slots == 1) return MOK_ERR_INVALID_ARG;
  if (!(c->capacity_mult == 0.0f || c->capacity_mult >= 1.0f)) return MOK_ERR_INVALID_ARG;
  if (c->replay != 0 && c->replay != 1) return MOK_ERR_INVALID_ARG;
  if (c->overlap_sms < 0) return MOK_ERR_INVALID_ARG;
  return MOK_OK;
}

mok_status check_prec(mok_precision p) {
  if (p == MOK_BF16 || p == MOK_MXFP8) return MOK_OK;
  return MOK_ERR_INVALID_ARG;
}

const mok_mx* as_mx(const void* p) { return static_cast<const mok_mx*>(p); }

bool mx_ok(const void* p) { return p && as_mx(p)->q && as_mx(p)->scale; }

const CUtensorMapDataType kU8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;

// u8 [rows, cols] row-major, box {box_cols, box_rows}, 128-byte swizzle.
bool map2d_u8(CUtensorMap* m, const void* p, uint64_t cols, uint64_t rows, uint32_t box_cols, uint32_t box_rows) {
  const uint64_t dims[2] = {cols, rows};
  const uint64_t str[1] = {cols};
  const uint32_t box[2] = {box_cols, box_rows};
  return make_tmap(m, kU8, 2, p, dims, str, box, true);
}

// u8 [E, rows, cols], box {128, box_rows, 1}, 128-byte swizzle.
bool map3d_u8(CUtensorMap* m, const void* p, uint64_t cols, uint64_t rows, uint64_t E, uint32_t box_rows) {
  const uint64_t dims[3] = {cols, rows, E};
  const uint64_t str[2] = {cols, cols * rows};
  const uint32_t box[3] = {128, box_rows, 1};
  return make_tmap(m, kU8, 3, p, dims, str, box, true);
}

#define MOK_TRY(expr)                       \
  do {                                      \
    const mok_status st_ = (expr);          \
    if (st_ != MOK_OK) return st_;          \
  } while (0)

#define MOK_CUDA(expr)                          \
  do {                                          \
    if ((expr) != cudaSuccess) return MOK_ERR_CUDA; \
  } while (0)

const CUtensorMapDataType kBF16 = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;

// bf16 [rows, cols] row-major, box {64, box_rows}.
bool map2d(CUtensorMap* m, const void* p, uint64_t cols, uint64_t rows, uint32_t box_rows) {
  const uint64_t dims[2] = {cols, rows};
  const uint64_t str[1] = {cols * 2};
  const uint32_t box[2] = {64, box_rows};
  return make_tmap(m, kBF16, 2, p, dims, str, box, true);
}

// bf16 [E, rows, cols], box {64, box_rows, 1}.
bool map3d(CUtensorMap* m, const void* p, uint64_t cols, uint64_t rows, uint64_t E, uint32_t box_rows) {
  const uint64_t dims[3] = {cols, rows, E};
  const uint64_t str[2] = {cols * 2, cols * rows * 2};
  const uint32_t box[3] = {64, box_rows, 1};
  return make_tmap(m, kBF16, 3, p, dims, str, box, true);
}

// Tensor map of a token-row operand that the gather warps copy with
// cp.async (bf16 [rows, cols], box {64, 1}): no TMA load reads it; it keeps
// the map slot of the gathered operand valid for the descriptor prefetch.
bool map_gather(CUtensorMap* m, const void* p, uint64_t cols, uint64_t rows) {
  const uint64_t dims[2] = {cols, rows};
  const uint64_t str[1] = {cols * 2};
  const uint32_t box[2] = {64, 1};
  return make_tmap(m, kBF16, 2, p, dims, str, box, true);
}

int gemm_grid(long items) {
  const int sms = device_sm_count();
  if (items < 1) items = 1;
  return (int)(items < sms ? items : sms);
}

// The forward ring puts experts of at least this many 128-row tiles on CTA
// pairs, the others on single CTAs: a pair launch holding only a few short
// experts is bound by its critical path (measured on the mid-sized and
// Kimi-shaped workloads), and long experts leave few solo pairs.
constexpr int kRingPairTiles = 8;

// Experts with at least this many padded rows have their BF16 weight
// gradients computed on CTA pairs (cta_group::2, one 256 x 256 tile per
// pair): their long K loops are bound by operand delivery, which the pair
// halves per SM.  Shorter experts' tiles are bound by their dW stores and
// run on single CTAs, with all SMs resident.
constexpr int kPairMinRows = 512;

// BF16 weight-gradient GEMM of one mode: the long-K experts on CTA pairs,
// then the others (and the empty experts' zeros) on single CTAs, when the
// operands are token-sorted copies and the tile counts allow pairs; else
// every expert on single CTAs.  Returns the number of launches in *n.
cudaError_t launch_wgrad(int mode, const TmapSet& m, GemmParams q, int grid, int debug_flags, int light_counter,
                         int* n, cudaStream_t st) {
  *n = 0;
  if (!(debug_flags & MOK_DEBUG_SINGLE_CTA_WGRAD) && q.wg_sorted && q.m_tiles % 2 == 0 && q.bn == 256) {
    GemmParams qh = q;
    qh.wg_rows_min = kPairMinRows;
    qh.wg_rows_max = INT_MAX;
    const cudaError_t e = launch_gemm_pair(mode, m, qh, grid, st);
    if (e == cudaSuccess) {
      q.wg_rows_min = 0;
      q.wg_rows_max = kPairMinRows;
      q.counter = light_counter;
      *n = 2;
      return launch_gemm(mode, m, q, grid, st);
    }
    if (e != cudaErrorNotSupported) return e;
    (void)cudaGetLastError();
  }
  q.wg_rows_min = 0;
  q.wg_rows_max = INT_MAX;
  *n = 1;
  return launch_gemm(mode, m, q, grid, st);
}

void base_params(GemmParams& g, const mok_shape& s, const WsLayout& L, uint8_t* ws) {
  memset(&g, 0, sizeof(g));
  g.T = s.T;
  g.H = s.H;
  g.I = s.I;
  g.E = s.E;
  g.k = s.k;
  g.hdr = reinterpret_cast<int32_t*>(ws + L.header);
  g.tile_expert = reinterpret_cast<const int32_t*>(ws + L.tile_expert);
  g.pad_perm = reinterpret_cast<const int32_t*>(ws + L.pad_perm);
  g.padded_offsets = reinterpret_cast<const int32_t*>(ws + L.padded_offsets);
  g.counts = reinterpret_cast<const int32_t*>(ws + L.counts);
  g.wg_rows_min = 0;
  g.wg_rows_max = INT_MAX;
  g.ring_count_word = kHdrTiles;  // a ring launch walks every tile unless given a list
}

// Whether launches may overlap (programmatic dependent launch).
bool overlap(const mok_config& c) { return (c.debug_flags & MOK_DEBUG_NO_OVERLAP) == 0; }

// Whether the device holds a cluster of two GEMM CTAs (the pair launches).
bool pair_grid_available() {
  static int device = -1;
  static bool ok = false;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  if (dev != device) {
    ok = gemm_pair_capacity() >= 2;
    device = dev;
  }
  return ok;
}

// Whether the BF16 backward's dA' and dX run on CTA pairs.
bool row_pairs(const mok_config& c) { return (c.debug_flags & MOK_DEBUG_SINGLE_CTA_ROWS) == 0; }

void set_pair_table(GemmParams& g, const WsLayout& L, uint8_t* ws) {
  g.pair_m0 = reinterpret_cast<const int32_t*>(ws + L.pair_m0);
}

// A row-tiled launch on CTA pairs (pair_maps: weight boxes of 128 rows,
// each CTA's half of the tile), else -- without pairs, or without clusters
// of two on the device -- one CTA per tile (maps: boxes of bn rows).
// With pairs, the units of the split table (every expert's tiles two at a
// time, built with min_pair_tiles = 1, so no single tiles) run on CTA pairs.
cudaError_t launch_rows(int mode, bool pairs, const TmapSet& pair_maps, const TmapSet& maps, const GemmParams& q,
                        int grid, cudaStream_t st) {
  if (pairs) {
    const cudaError_t e = launch_gemm_pair(mode, pair_maps, q, grid, st);
    if (e != cudaErrorNotSupported) return e;
    (void)cudaGetLastError();
  }
  return launch_gemm(mode, maps, q, grid, st);
}

mok_status reset_counters(uint8_t* ws, const WsLayout& L, cudaStream_t st) {
  // the abort word and the tile counters (words [3, 48)); the error word,
  // the used-row count and the used-tile count are kept
  MOK_CUDA(cudaMemsetAsync(ws + L.header + kHdrAbort * 4, 0, (kHdrCounters + kNumCounters - kHdrAbort) * 4, st));
  return MOK_OK;
}


// MXFP8 backward: every GEMM block-scaled along its own K.  Weights come in
// the orientation the backward contracts over (W1, W3 along I; W2 along H);
// dout is quantised along H, dh|du along I (in the dA' epilogue), and the
// weight-gradient operands along the expert's routed rows.
mok_status backward_mx(const mok_shape& s, const WsLayout& L, uint8_t* w, const mok_config& cfg, const void* ctx,
                       const void* x, const float* scores, const mok_mx& q1, const mok_mx& q3, const mok_mx& q2,
                       const mok_mx* f1, const mok_mx* f3, const void* dout, void* dX, void* dW1, void* dW3,
                       void* dW2, float* dscores, cudaStream_t st) {
  // dA' reads dout's codes in padded-row order by plain TMA, unless asked to
  // gather them in its load path
  const int debug_flags = cfg.debug_flags;
  const bool sorted_codes = !(debug_flags & MOK_DEBUG_FUSED_WGRAD_GATHER);
  const uint64_t P = L.pad_capacity;
  const int bn_i = (s.I % 256 == 0) ? 256 : 128;
  const int bn_h = (s.H % 256 == 0) ? 256 : 128;
  const int32_t* rows_used = reinterpret_cast<const int32_t*>(w + L.header) + kHdrPaddedRows;
  GemmParams g;
  base_params(g, s, L, w);
  g.ctx_hu = const_cast<__nv_bfloat16*>(static_cast<const __nv_bfloat16*>(ctx));
  g.dhu = reinterpret_cast<__nv_bfloat16*>(w + L.dhu);
  g.as = reinterpret_cast<__nv_bfloat16*>(w + L.as);
  g.dsp = reinterpret_cast<float*>(w + L.dsp);
  g.scores = scores;
  g.yk = reinterpret_cast<__nv_bfloat16*>(w + L.yk);
  if (cfg.replay) {
    // Bounded-memory backward, as in BF16: the context's last ring_slots
    // minibatches of [h|u] go back to their rows of dh|du, and GEMM1 is
    // recomputed for the earlier ones straight into those rows -- with the
    // forward's operands (x quantised along H, W1 / W3 along H) and tiles,
    // so the values are the forward's bit for bit.
    const bool srt = !(debug_flags & MOK_DEBUG_GATHER_X_RING);
    {
      Phase ph(MOK_PHASE_BWD_REPLAY, st, srt ? 6 : 5);
      MOK_CUDA(launch_replay_copy(s, L, w, static_cast<const __nv_bfloat16*>(ctx), g.dhu, st));
      MOK_CUDA(launch_mxfp8_quantize(static_cast<const __nv_bfloat16*>(x), 1, s.T, s.H, 1, w + L.xq, w + L.xsf, st));
      MOK_CUDA(launch_tile_scales(f1->scale, s.E, s.H / 32, s.I, w + L.wsf1, st, 1, 2, 0));
      MOK_CUDA(launch_tile_scales(f3->scale, s.E, s.H / 32, s.I, w + L.wsf1, st, 1, 2, 1));
      MOK_CUDA(launch_tile_row_scales(w + L.xsf, s.H / 32, reinterpret_cast<const int32_t*>(w + L.pad_perm), s.k,
                                      rows_used, L.pad_capacity, w + L.sfa_rows_t, st));
      if (srt) MOK_CUDA(launch_gather_code_rows(s, L, w, w + L.xq, w + L.xq_sorted, st));
    }
    TmapSet m;
    memset(&m, 0, sizeof(m));
    if (!(srt ? map2d_u8(&m.m[0], w + L.xq_sorted, s.H, P, 128, 128) : map2d_u8(&m.m[0], w + L.xq, s.H, s.T, 128, 128)) ||
        !map3d_u8(&m.m[1], f1->q, s.I, s.H, s.E, 128) || !map3d_u8(&m.m[2], f3->q, s.I, s.H, s.E, 128))
      return MOK_ERR_CUDA;
    GemmParams q = g;
    q.ctx_hu = g.dhu;
    q.ring = reinterpret_cast<__nv_bfloat16*>(w + L.ring);  // a and its scales: scratch here
    q.ring_sf = w + L.ring_sf;
    q.ring_rows = L.minibatch_rows;
    q.ring_slots = L.ring_slots;
    q.gq_src = w + L.xq;
    q.fwd_sorted = srt ? 1 : 0;
    q.sfa_tiled = w + L.sfa_rows_t;
    q.sfb_tiled0 = w + L.wsf1;  // W1 | W3 interleaved
    q.nmaps = 3;
    q.bn = 256;
    q.n_tiles = s.I / 128;
    q.m_tile_begin = 0;
    q.m_tile_end = (int)L.tile_capacity;
    q.replay_keep = L.ring_slots;
    q.counter = 6;
    {
      Phase ph(MOK_PHASE_BWD_REPLAY, st, 1);
      MOK_CUDA(launch_gemm_mx(GM_FWD1, m, q, gemm_grid(L.tile_capacity * q.n_tiles), st));
    }
    g.ctx_hu = g.dhu;
  }
  {
    Phase ph(MOK_PHASE_QUANT, st, 1);
    MOK_CUDA(launch_mxfp8_quantize(static_cast<const __nv_bfloat16*>(dout), 1, s.T, s.H, 1, w + L.xq, w + L.xsf, st));
  }
  // dA' = gather(dout) W2^T (E4M3), SwiGLU backward, router partials, dh|du quantised along I
  {
    TmapSet m;
    memset(&m, 0, sizeof(m));
    if (!map3d_u8(&m.m[1], q2.q, s.H, s.I, s.E, bn_i)) return MOK_ERR_CUDA;
    if (!(sorted_codes ? map2d_u8(&m.m[0], w + L.xq_sorted, s.H, P, 128, 128)
                       : map2d_u8(&m.m[0], w + L.xq, s.H, s.T, 128, 128)))
      return MOK_ERR_CUDA;
    GemmParams q = g;
    q.nmaps = 2;
    q.bn = bn_i;
    q.n_tiles = s.I / bn_i;
    q.m_tiles = 0;
    q.rows_sorted = sorted_codes ? 1 : 0;
    q.m_tile_begin = 0;
    q.m_tile_end = (int)L.tile_capacity;
    q.counter = 0;
    q.gq_src = w + L.xq;
    // dout's scales in padded-row order and W2's scales (along H, in the
    // region the forward uses for its own W2 scales), tiled for the TMA
    // producer
    {
      Phase ph(MOK_PHASE_QUANT, st, sorted_codes ? 3 : 2);
      MOK_CUDA(launch_tile_row_scales(w + L.xsf, s.H / 32, reinterpret_cast<const int32_t*>(w + L.pad_perm), s.k,
                                      rows_used, L.pad_capacity, w + L.sfa_rows_t, st));
      MOK_CUDA(launch_tile_scales_rows(q2.scale, s.E, s.I, s.H / 32, w + L.wsf2, st, bn_i / 128, bn_i / 128, 0));
      if (sorted_codes) MOK_CUDA(launch_gather_code_rows(s, L, w, w + L.xq, w + L.xq_sorted, st));
    }
    q.sfa_tiled = w + L.sfa_rows_t;
    q.sfb_tiled0 = w + L.wsf2;
    q.dhu_q = w + L.dhuq;
    q.dhu_sf = w + L.dhusf;
    {
      Phase ph(MOK_PHASE_BWD_DA, st, 1);
      MOK_CUDA(launch_gemm_mx(GM_BWD_DA, m, q, gemm_grid(L.tile_capacity * q.n_tiles), st));
    }
    Phase ph(MOK_PHASE_BWD_DS, st, 1);
    MOK_CUDA(launch_ds_reduce(s, L, w, dscores, q.n_tiles, st));
  }
  // dX parts = [dh|du] [W1|W3]^T (E4M3 along I), scattered, then summed over k
  {
    TmapSet m;
    memset(&m, 0, sizeof(m));
    if (!map2d_u8(&m.m[0], w + L.dhuq, 2 * (uint64_t)s.I, P, 128, 128) ||
        !map3d_u8(&m.m[1], q1.q, s.I, s.H, s.E, bn_h) || !map3d_u8(&m.m[2], q3.q, s.I, s.H, s.E, bn_h))
      return MOK_ERR_CUDA;
    GemmParams q = g;
    q.nmaps = 3;
    q.bn = bn_h;
    q.n_tiles = s.H / bn_h;
    q.m_tile_begin = 0;
    q.m_tile_end = (int)L.tile_capacity;
    q.counter = 1;
    // dh|du's scales (padded rows already) and W1's and W3's scales (along
    // I), tiled for the TMA producer
    {
      Phase ph(MOK_PHASE_QUANT, st, 3);
      MOK_CUDA(launch_tile_row_scales(w + L.dhusf, 2 * s.I / 32, nullptr, 1, rows_used, L.pad_capacity,
                                      w + L.sfa_rows_t, st));
      MOK_CUDA(launch_tile_scales_rows(q1.scale, s.E, s.H, s.I / 32, w + L.wsf1, st, bn_h / 128, bn_h / 128, 0));
      MOK_CUDA(launch_tile_scales_rows(q3.scale, s.E, s.H, s.I / 32, w + L.wsf3, st, bn_h / 128, bn_h / 128, 0));
    }
    q.sfa_tiled = w + L.sfa_rows_t;
    q.sfb_tiled0 = w + L.wsf1;
    q.sfb_tiled1 = w + L.wsf3;
    {
      Phase ph(MOK_PHASE_BWD_DX, st, 1);
      MOK_CUDA(launch_gemm_mx(GM_BWD_DX, m, q, gemm_grid(L.tile_capacity * q.n_tiles), st));
    }
    Phase ph(MOK_PHASE_BWD_DX_COMBINE, st, 1);
    MOK_CUDA(launch_combine(s, L, w, g.yk, nullptr, static_cast<__nv_bfloat16*>(dX), st));
  }
  // the weight gradients' token-row operands (x, dout) are gathered in
  // padded-row order as they are quantised along the rows
  const int32_t* pad_perm = reinterpret_cast<const int32_t*>(w + L.pad_perm);
  // dW1 | dW3: token-sorted x and dh|du, both quantised along the routed rows
  {
    {
      Phase ph(MOK_PHASE_BWD_SORT, st, 2);
      MOK_CUDA(launch_quant_rows_gather(static_cast<const __nv_bfloat16*>(x), rows_used, P, s.H, pad_perm, s.k,
                                        w + L.wqa, w + L.wsfa, st));
      MOK_CUDA(launch_quant_rows_tiled(g.dhu, rows_used, P, 2 * s.I, w + L.wqb, w + L.wsfb, st));
    }
    TmapSet m;
    memset(&m, 0, sizeof(m));
    if (!map2d_u8(&m.m[0], w + L.wqa, s.H, P, 128, 128) || !map2d_u8(&m.m[1], w + L.wqb, 2 * (uint64_t)s.I, P, 128, 128))
      return MOK_ERR_CUDA;
    GemmParams q = g;
    q.nmaps = 2;
    q.bn = 256;
    q.n_tiles = 2 * s.I / 256;
    q.m_tiles = s.H / 128;
    q.counter = 2;
    q.wg_sorted = 1;
    q.sfa_tiled = w + L.wsfa;
    q.sfb_tiled0 = w + L.wsfb;
    q.dW1 = static_cast<__nv_bfloat16*>(dW1);
    q.dW3 = static_cast<__nv_bfloat16*>(dW3);
    Phase ph(MOK_PHASE_BWD_WG13, st, 1);
    MOK_CUDA(launch_gemm_mx(GM_WG13, m, q, gemm_grid((long)s.E * q.m_tiles * q.n_tiles), st));
  }
  // dW2: s*a and token-sorted dout, both quantised along the routed rows
  {
    {
      Phase ph(MOK_PHASE_BWD_SORT, st, 2);
      MOK_CUDA(launch_quant_rows_tiled(g.as, rows_used, P, s.I, w + L.wqb, w + L.wsfb, st));
      MOK_CUDA(launch_quant_rows_gather(static_cast<const __nv_bfloat16*>(dout), rows_used, P, s.H, pad_perm, s.k,
                                        w + L.wqa, w + L.wsfa, st));
    }
    TmapSet m;
    memset(&m, 0, sizeof(m));
    if (!map2d_u8(&m.m[0], w + L.wqb, s.I, P, 128, 128) || !map2d_u8(&m.m[1], w + L.wqa, s.H, P, 128, 128))
      return MOK_ERR_CUDA;
    GemmParams q = g;
    q.nmaps = 2;
    q.bn = bn_h;
    q.n_tiles = s.H / bn_h;
    q.m_tiles = s.I / 128;
    q.counter = 3;
    q.wg_sorted = 1;
    q.sfa_tiled = w + L.wsfb;
    q.sfb_tiled0 = w + L.wsfa;
    q.dW2 = static_cast<__nv_bfloat16*>(dW2);
    Phase ph(MOK_PHASE_BWD_WG2, st, 1);
    MOK_CUDA(launch_gemm_mx(GM_WG2, m, q, gemm_grid((long)s.E * q.m_tiles * q.n_tiles), st));
  }
  return MOK_OK;
}

}  // namespace

extern "C" {

const char* mok_version(void) { return "mok-gb300 0.1.0 (sm_103a)"; }

const char* mok_status_string(mok_status s) {
  if ((int)s < 0 || (int)s > 6) return "MOK_ERR_UNKNOWN";
  return kStatusNames[(int)s];
}

int32_t mok_device_sm_count(void) { return device_sm_count(); }

size_t mok_workspace_size(const mok_shape* shape, const mok_config* cfg, mok_precision prec) {
  if (check_shape(shape) != MOK_OK || check_config(cfg) != MOK_OK) return 0;
  if (prec != MOK_BF16 && prec != MOK_MXFP8) return 0;
  return ws_layout(*shape, *cfg, prec, device_sm_count()).total;
}

size_t mok_ctx_size(const mok_shape* shape, const mok_config* cfg, mok_precision prec) {
  if (check_shape(shape) != MOK_OK || check_config(cfg) != MOK_OK) return 0;
  if (prec != MOK_BF16 && prec != MOK_MXFP8) return 0;
  const WsLayout L = ws_layout(*shape, *cfg, prec, device_sm_count());
  if (cfg->replay) {
    // ring-slot order: slot rows are below min(ring_slots * minibatch_rows,
    // padded rows)
    const int64_t rows = std::min<int64_t>((int64_t)L.ring_slots * L.minibatch_rows, L.pad_capacity);
    return (size_t)rows * 2 * shape->I * 2;
  }
  return (size_t)L.pad_capacity * 2 * shape->I * 2;
}

mok_status mok_workspace_layout(const mok_shape* shape, const mok_config* cfg, mok_precision prec,
                                mok_layout* out) {
  MOK_TRY(check_shape(shape));
  MOK_TRY(check_config(cfg));
  if (!out || (prec != MOK_BF16 && prec != MOK_MXFP8)) return MOK_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(*shape, *cfg, prec, device_sm_count());
  out->header = L.header;
  out->counts = L.counts;
  out->offsets = L.offsets;
  out->padded_offsets = L.padded_offsets;
  out->perm = L.perm;
  out->inv_perm = L.inv_perm;
  out->pad_perm = L.pad_perm;
  out->pad_inv = L.pad_inv;
  out->tile_expert = L.tile_expert;
  out->pad_capacity = L.pad_capacity;
  out->tile_capacity = L.tile_capacity;
  return MOK_OK;
}

mok_status mok_build_schedule(const mok_shape* shape, const mok_config* cfg, void* ws, size_t ws_bytes,
                              const int32_t* topk_idx, void* stream) {
  MOK_TRY(check_shape(shape));
  MOK_TRY(check_config(cfg));
  if (!ws || !topk_idx) return MOK_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(*shape, *cfg, MOK_BF16, device_sm_count());
  // the schedule part of the layout is the same for both precisions
  if (ws_bytes < L.chunk_base + align256(L.nchunks * shape->E * 4)) return MOK_ERR_WORKSPACE_TOO_SMALL;
  Phase ph(MOK_PHASE_SCHEDULE, static_cast<cudaStream_t>(stream), 3);
  MOK_CUDA(launch_schedule(*shape, L, static_cast<uint8_t*>(ws), topk_idx, static_cast<cudaStream_t>(stream)));
  return MOK_OK;
}

mok_status mok_forward(const mok_shape* shape, const mok_config* cfg, mok_precision prec, void* ws,
                       size_t ws_bytes, const void* x, const float* scores, const void* W1, const void* W3,
                       const void* W2, void* out, void* ctx, void* stream) {
  MOK_TRY(check_shape(shape));
  MOK_TRY(check_config(cfg));
  MOK_TRY(check_prec(prec));
  if (!ws || !x || !scores || !W1 || !W3 || !W2 || !out || !ctx) return MOK_ERR_INVALID_ARG;
  const mok_shape& s = *shape;
  const WsLayout L = ws_layout(s, *cfg, prec, device_sm_count());
  if (ws_bytes < L.total) return MOK_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* w = static_cast<uint8_t*>(ws);
  MOK_TRY(reset_counters(w, L, st));
  MOK_CUDA(cudaMemsetAsync(w + L.ring_flags, 0, 4 * L.tile_capacity * 4, st));
  if (prec == MOK_BF16) MOK_CUDA(cudaMemsetAsync(w + L.ring_flags2, 0, 4 * L.tile_capacity * 4, st));

  const int M = L.minibatch_rows, S = L.ring_slots;
  const int bn2 = (s.H % 256 == 0) ? 256 : 128;
  if (prec == MOK_MXFP8) {
    MOK_CUDA(cudaMemsetAsync(reinterpret_cast<int32_t*>(w + L.header) + kHdrSortedX, 0, 4, st));
    if (!mx_ok(W1) || !mx_ok(W3) || !mx_ok(W2)) return MOK_ERR_INVALID_ARG;
    const mok_mx &q1 = *as_mx(W1), &q3 = *as_mx(W3), &q2 = *as_mx(W2);
    {
      // x along H; forward weight scales tiled for the N-major B operands
      Phase ph(MOK_PHASE_QUANT, st, 4);
      MOK_CUDA(launch_mxfp8_quantize(static_cast<const __nv_bfloat16*>(x), 1, s.T, s.H, 1, w + L.xq, w + L.xsf, st));
      MOK_CUDA(launch_tile_scales(q1.scale, s.E, s.H / 32, s.I, w + L.wsf1, st, 1, 2, 0));
      MOK_CUDA(launch_tile_scales(q3.scale, s.E, s.H / 32, s.I, w + L.wsf1, st, 1, 2, 1));
      MOK_CUDA(launch_tile_scales(q2.scale, s.E, s.I / 32, s.H, w + L.wsf2, st, bn2 / 128, bn2 / 128, 0));
    }
    const bool sorted_codes = !(cfg->debug_flags & MOK_DEBUG_GATHER_X_RING);
    {
      // x's scales in padded-row order, tiled for the TMA producer (GEMM1 A),
      // and x's codes in padded-row order (GEMM1's A by plain TMA)
      Phase ph(MOK_PHASE_QUANT, st, sorted_codes ? 2 : 1);
      MOK_CUDA(launch_tile_row_scales(w + L.xsf, s.H / 32, reinterpret_cast<const int32_t*>(w + L.pad_perm), s.k,
                                      reinterpret_cast<const int32_t*>(w + L.header) + kHdrPaddedRows,
                                      L.pad_capacity, w + L.sfa_rows_t, st));
      if (sorted_codes) MOK_CUDA(launch_gather_code_rows(s, L, w, w + L.xq, w + L.xq_sorted, st));
    }
    GemmParams g;
    base_params(g, s, L, w);
    g.ctx_hu = static_cast<__nv_bfloat16*>(ctx);
    g.ctx_ring = cfg->replay;  // bounded context: [h|u] rows in ring-slot order
    g.ring = reinterpret_cast<__nv_bfloat16*>(w + L.ring);  // E4M3 codes in MXFP8 mode
    g.ring_sf = w + L.ring_sf;
    g.ring_rows = M;
    g.ring_slots = S;
    g.ring_flags = reinterpret_cast<uint32_t*>(w + L.ring_flags);
    g.yk = reinterpret_cast<__nv_bfloat16*>(w + L.yk);
    g.debug_flags = cfg->debug_flags;
    g.gq_src = w + L.xq;
    g.sfa_tiled = w + L.sfa_rows_t;
    g.sfb_tiled0 = w + L.wsf1;  // W1 | W3 interleaved
    g.sfb_tiled2 = w + L.wsf2;
    TmapSet maps;
    memset(&maps, 0, sizeof(maps));
    if (!map3d_u8(&maps.m[1], q1.q, s.I, s.H, s.E, 128) || !map3d_u8(&maps.m[2], q3.q, s.I, s.H, s.E, 128) ||
        !map2d_u8(&maps.m[3], w + L.ring, s.I, (uint64_t)S * M, 128, 128) ||
        !map3d_u8(&maps.m[4], q2.q, s.H, s.I, s.E, 128))
      return MOK_ERR_CUDA;
    if (sorted_codes) {
      if (!map2d_u8(&maps.m[0], w + L.xq_sorted, s.H, (uint64_t)L.pad_capacity, 128, 128)) return MOK_ERR_CUDA;
      g.fwd_sorted = 1;
    } else if (!map2d_u8(&maps.m[0], w + L.xq, s.H, s.T, 128, 128)) {  // a valid map for the prefetch
      return MOK_ERR_CUDA;
    }
    g.nmaps = 5;
    g.bn = bn2;
    g.n_tiles = s.H / bn2;
    g.g1_tiles = s.I / 128;
    g.m_tiles = 2 * (int)L.tile_capacity;  // ring: where the consumed half of the flags starts
    g.counter = 0;
    {
      Phase ph(MOK_PHASE_FWD_GEMM, st, 1);
      MOK_CUDA(launch_gemm_mx(GM_FWD_RING, maps, g, gemm_grid(L.tile_capacity * (g.g1_tiles + g.n_tiles)), st));
    }
    Phase ph(MOK_PHASE_FWD_COMBINE, st, 1);
    MOK_CUDA(launch_combine(s, L, w, g.yk, scores, static_cast<__nv_bfloat16*>(out), st));
    return MOK_OK;
  }
  GemmParams g;
  base_params(g, s, L, w);
  // set again below once the token-sorted copy of x is made
  int32_t* sorted_x_flag = reinterpret_cast<int32_t*>(w + L.header) + kHdrSortedX;
  MOK_CUDA(cudaMemsetAsync(sorted_x_flag, 0, 4, st));
  g.ctx_hu = static_cast<__nv_bfloat16*>(ctx);
  g.ctx_ring = cfg->replay;  // bounded context: [h|u] rows in ring-slot order
  g.ring = reinterpret_cast<__nv_bfloat16*>(w + L.ring);
  g.ring_rows = M;
  g.ring_slots = S;
  g.ring_flags = reinterpret_cast<uint32_t*>(w + L.ring_flags);
  g.yk = reinterpret_cast<__nv_bfloat16*>(w + L.yk);
  g.debug_flags = cfg->debug_flags;
  g.gather_src = static_cast<const __nv_bfloat16*>(x);

  TmapSet maps;
  memset(&maps, 0, sizeof(maps));
  if (!map_gather(&maps.m[0], x, s.H, s.T)) return MOK_ERR_CUDA;
  if (!map3d(&maps.m[1], W1, s.I, s.H, s.E, 64) || !map3d(&maps.m[2], W3, s.I, s.H, s.E, 64)) return MOK_ERR_CUDA;

  const bool serial = (cfg->debug_flags & MOK_DEBUG_SERIAL_RING) != 0;
  if (!serial) {
    // one persistent launch: GEMM1 and GEMM2 interleaved through the ring
    if (!map2d(&maps.m[3], g.ring, s.I, (uint64_t)S * M, 128) || !map3d(&maps.m[4], W2, s.H, s.I, s.E, 64))
      return MOK_ERR_CUDA;
    g.nmaps = 5;
    g.bn = bn2;
    g.n_tiles = s.H / bn2;
    g.g1_tiles = s.I / 128;
    g.m_tiles = 2 * (int)L.tile_capacity;  // ring: where the consumed half of the flags starts
    g.counter = 0;
    const int grid = gemm_grid(L.tile_capacity * (g.g1_tiles + g.n_tiles));
    bool launched = false;
    // The ring in two launches (unless single CTAs are asked for, or the
    // context must keep the minibatches in one order for replay, or no
    // expert can reach kRingPairTiles tiles): the experts of at least
    // kRingPairTiles tiles on CTA pairs (two tiles of one expert per
    // 256 x 256 tile, an even number of tiles per minibatch), the others on
    // single CTAs; every expert in one launch, so its weights stream once.
    // Both read the token-sorted copy of x with plain TMA.
    const int Mt_pair = (M / kTileRows) & ~1;
    const bool big_expert_possible = (int64_t)s.T >= (int64_t)kRingPairTiles * kTileRows;
    if (!(cfg->debug_flags & MOK_DEBUG_SINGLE_CTA_RING) && !cfg->replay && bn2 == 256 && Mt_pair >= 2 &&
        big_expert_possible) {
      __nv_bfloat16* srt = reinterpret_cast<__nv_bfloat16*>(w + L.sorted);
      {
        Phase ph(MOK_PHASE_FWD_SORT, st, 2);
        MOK_CUDA(launch_gather_rows(s, L, w, static_cast<const __nv_bfloat16*>(x), srt, st));
        MOK_CUDA(cudaMemsetAsync(sorted_x_flag, 1, 1, st));
        MOK_CUDA(launch_split_table(L, w, kRingPairTiles, st));
      }
      TmapSet sm = maps;
      if (!map2d(&sm.m[0], srt, s.H, (uint64_t)L.pad_capacity, 128)) return MOK_ERR_CUDA;
      GemmParams gp = g;
      gp.fwd_sorted = 1;
      gp.pair_m0 = reinterpret_cast<const int32_t*>(w + L.pair_m0);
      gp.ring_count_word = kHdrPairs;
      gp.ring_rows = Mt_pair * kTileRows;
      // the short experts' tiles: a ring walk of their own (ring, flags and
      // tile counter), on single CTAs
      GemmParams gs = g;
      gs.fwd_sorted = 1;
      gs.ring_list = reinterpret_cast<const int32_t*>(w + L.pair_mb);
      gs.ring_count_word = kHdrSingles;
      gs.counter = 7;
      gs.ring = reinterpret_cast<__nv_bfloat16*>(w + L.ring2);
      gs.ring_flags = reinterpret_cast<uint32_t*>(w + L.ring_flags2);
      TmapSet ss = sm;
      if (!map2d(&ss.m[3], gs.ring, s.I, (uint64_t)S * M, 128)) return MOK_ERR_CUDA;
      Phase ph(MOK_PHASE_FWD_GEMM, st, 2);
      if (overlap(*cfg) && pair_grid_available()) {
        // the single-CTA launch first, on its share of the SMs; the pair
        // launch starts beside it at once and takes each SM it leaves
        gs.pdl_trigger = 1;
        gs.active_ctas = cfg->overlap_sms > 0 ? cfg->overlap_sms : -1;
        MOK_CUDA(launch_gemm(GM_FWD_RING, ss, gs, grid, st));
        gp.pdl_launch = 1;
        gp.pdl_wait_end = 1;
        MOK_CUDA(launch_gemm_pair(GM_FWD_RING, sm, gp, grid, st));
        launched = true;
      }
      const cudaError_t e = launched ? cudaSuccess : launch_gemm_pair(GM_FWD_RING, sm, gp, grid, st);
      if (e != cudaSuccess && e != cudaErrorNotSupported) return MOK_ERR_CUDA;
      if (launched) {
        // overlapped above
      } else if (e == cudaSuccess) {
        // one after the other: the pair launch, then the short experts
        MOK_CUDA(launch_gemm(GM_FWD_RING, ss, gs, grid, st));
        launched = true;
      } else {
        (void)cudaGetLastError();  // no cluster of two fits: all tiles on single CTAs below
        GemmParams ga = g;
        ga.fwd_sorted = 1;
        MOK_CUDA(launch_gemm(GM_FWD_RING, sm, ga, grid, st));
        launched = true;
      }
    }
    if (!launched && !(cfg->debug_flags & MOK_DEBUG_GATHER_X_RING)) {
      // single CTAs reading the token-sorted copy of x with plain TMA (the
      // backward's dW1|dW3 reads the same copy)
      __nv_bfloat16* srt = reinterpret_cast<__nv_bfloat16*>(w + L.sorted);
      {
        Phase ph(MOK_PHASE_FWD_SORT, st, 1);
        MOK_CUDA(launch_gather_rows(s, L, w, static_cast<const __nv_bfloat16*>(x), srt, st));
        MOK_CUDA(cudaMemsetAsync(sorted_x_flag, 1, 1, st));
      }
      TmapSet sm = maps;
      if (!map2d(&sm.m[0], srt, s.H, (uint64_t)L.pad_capacity, 128)) return MOK_ERR_CUDA;
      GemmParams gs = g;
      gs.fwd_sorted = 1;
      Phase ph(MOK_PHASE_FWD_GEMM, st, 1);
      MOK_CUDA(launch_gemm(GM_FWD_RING, sm, gs, grid, st));
      launched = true;
    }
    if (!launched) {
      Phase ph(MOK_PHASE_FWD_GEMM, st, 1);
      MOK_CUDA(launch_gemm(GM_FWD_RING, maps, g, grid, st));
    }
  } else {
    // minibatch by minibatch in stream order (same ring, no device flags)
    TmapSet m2;
    memset(&m2, 0, sizeof(m2));
    if (!map2d(&m2.m[0], g.ring, s.I, (uint64_t)S * M, 128) || !map3d(&m2.m[1], W2, s.H, s.I, s.E, 64))
      return MOK_ERR_CUDA;
    maps.m[3] = m2.m[0];
    const int Mt = M / kTileRows;
    const int nmb = (int)((L.tile_capacity + Mt - 1) / Mt);
    Phase ph(MOK_PHASE_FWD_GEMM, st, 2 * nmb);
    int counter = 0;
    for (int b = 0; b < nmb; ++b) {
      GemmParams g1 = g;
      g1.nmaps = 3;
      g1.bn = 256;
      g1.n_tiles = s.I / 128;
      g1.m_tile_begin = b * Mt;
      g1.m_tile_end = (b + 1) * Mt;
      g1.counter = counter++ % kNumCounters;
      if (g1.counter == 0 && b > 0) MOK_TRY(reset_counters(w, L, st));
      MOK_CUDA(launch_gemm(GM_FWD1, maps, g1, gemm_grid((long)Mt * g1.n_tiles), st));
      GemmParams g2 = g1;
      g2.nmaps = 2;
      g2.bn = bn2;
      g2.n_tiles = s.H / bn2;
      g2.counter = counter++ % kNumCounters;
      MOK_CUDA(launch_gemm(GM_FWD2, m2, g2, gemm_grid((long)Mt * g2.n_tiles), st));
    }
  }
  {
    Phase ph(MOK_PHASE_FWD_COMBINE, st, 1);
    MOK_CUDA(launch_combine(s, L, w, g.yk, scores, static_cast<__nv_bfloat16*>(out), st));
  }
  return MOK_OK;
}

mok_status mok_forward_fused(const mok_shape* shape, const mok_config* cfg, mok_precision prec, void* ws,
                             size_t ws_bytes, const int32_t* topk_idx, const void* x, const float* scores,
                             const void* W1, const void* W3, const void* W2, void* out, void* ctx, void* stream) {
  MOK_TRY(check_shape(shape));
  MOK_TRY(check_config(cfg));
  MOK_TRY(check_prec(prec));
  if (!ws || !topk_idx || !x || !scores || !W1 || !W3 || !W2 || !out || !ctx) return MOK_ERR_INVALID_ARG;
  if (prec == MOK_MXFP8 && (!mx_ok(W1) || !mx_ok(W3) || !mx_ok(W2))) return MOK_ERR_INVALID_ARG;
  const mok_shape& s = *shape;
  const WsLayout L = ws_layout(s, *cfg, prec, device_sm_count());
  if (ws_bytes < L.total) return MOK_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* w = static_cast<uint8_t*>(ws);
  // the whole header (error word, schedule totals, item counters) and the ring flags
  MOK_CUDA(cudaMemsetAsync(w + L.header, 0, kHeaderWords * 4, st));
  MOK_CUDA(cudaMemsetAsync(w + L.ring_flags, 0, 4 * L.tile_capacity * 4, st));
  const int M = L.minibatch_rows, S = L.ring_slots;
  const int bn2 = (s.H % 256 == 0) ? 256 : 128;
  if (prec == MOK_MXFP8) {
    const mok_mx &q1 = *as_mx(W1), &q3 = *as_mx(W3), &q2 = *as_mx(W2);
    {
      // what does not depend on the routing, ahead of the launch: x along H
      // and the forward weight scales tiled; the tiled A scales cleared (the
      // launch's placement items fill the routed rows')
      Phase ph(MOK_PHASE_QUANT, st, 4);
      MOK_CUDA(launch_mxfp8_quantize(static_cast<const __nv_bfloat16*>(x), 1, s.T, s.H, 1, w + L.xq, w + L.xsf, st));
      MOK_CUDA(launch_tile_scales(q1.scale, s.E, s.H / 32, s.I, w + L.wsf1, st, 1, 2, 0));
      MOK_CUDA(launch_tile_scales(q3.scale, s.E, s.H / 32, s.I, w + L.wsf1, st, 1, 2, 1));
      MOK_CUDA(launch_tile_scales(q2.scale, s.E, s.I / 32, s.H, w + L.wsf2, st, bn2 / 128, bn2 / 128, 0));
      MOK_CUDA(cudaMemsetAsync(w + L.sfa_rows_t, 0, (size_t)L.pad_capacity * (s.H / 32), st));
    }
  }
  auto I32 = [&](size_t off) { return reinterpret_cast<int32_t*>(w + off); };
  GemmParams g;
  base_params(g, s, L, w);
  g.ctx_hu = static_cast<__nv_bfloat16*>(ctx);
  g.ctx_ring = cfg->replay;
  g.ring = reinterpret_cast<__nv_bfloat16*>(w + L.ring);
  g.ring_rows = M;
  g.ring_slots = S;
  g.ring_flags = reinterpret_cast<uint32_t*>(w + L.ring_flags);
  g.yk = reinterpret_cast<__nv_bfloat16*>(w + L.yk);
  g.debug_flags = cfg->debug_flags;
  g.gather_src = static_cast<const __nv_bfloat16*>(x);
  g.scores = scores;
  g.out = static_cast<__nv_bfloat16*>(out);
  g.topk_idx = topk_idx;
  g.nchunks = (int)L.nchunks;
  g.chunk_hist = I32(L.chunk_hist);
  g.chunk_base = I32(L.chunk_base);
  g.s_counts = I32(L.counts);
  g.s_offsets = I32(L.offsets);
  g.s_poff = I32(L.padded_offsets);
  g.s_perm = I32(L.perm);
  g.s_inv_perm = I32(L.inv_perm);
  g.s_pad_perm = I32(L.pad_perm);
  g.s_pad_inv = I32(L.pad_inv);
  g.s_tile_expert = I32(L.tile_expert);
  TmapSet maps;
  memset(&maps, 0, sizeof(maps));
  if (prec == MOK_MXFP8) {
    // GEMM1 gathers x's E4M3 rows by token; its A scales come tiled by the
    // placement items, the weights' from the tilings above
    const mok_mx &q1 = *as_mx(W1), &q3 = *as_mx(W3), &q2 = *as_mx(W2);
    g.ring_sf = w + L.ring_sf;
    g.gq_src = w + L.xq;
    g.sfa_rows = w + L.xsf;
    g.sfa_ld = s.H / 32;
    g.sfa_tiled = w + L.sfa_rows_t;
    g.sfb_tiled0 = w + L.wsf1;  // W1 | W3 interleaved
    g.sfb_tiled2 = w + L.wsf2;
    if (!map2d_u8(&maps.m[0], w + L.xq, s.H, s.T, 128, 128) ||  // a valid map for the prefetch
        !map3d_u8(&maps.m[1], q1.q, s.I, s.H, s.E, 128) || !map3d_u8(&maps.m[2], q3.q, s.I, s.H, s.E, 128) ||
        !map2d_u8(&maps.m[3], w + L.ring, s.I, (uint64_t)S * M, 128, 128) ||
        !map3d_u8(&maps.m[4], q2.q, s.H, s.I, s.E, 128))
      return MOK_ERR_CUDA;
  } else {
    if (!map_gather(&maps.m[0], x, s.H, s.T)) return MOK_ERR_CUDA;
    if (!map3d(&maps.m[1], W1, s.I, s.H, s.E, 64) || !map3d(&maps.m[2], W3, s.I, s.H, s.E, 64)) return MOK_ERR_CUDA;
    if (!map2d(&maps.m[3], g.ring, s.I, (uint64_t)S * M, 128) || !map3d(&maps.m[4], W2, s.H, s.I, s.E, 64))
      return MOK_ERR_CUDA;
  }
  g.nmaps = 5;
  g.bn = bn2;
  g.n_tiles = s.H / bn2;
  g.g1_tiles = s.I / 128;
  g.m_tiles = 2 * (int)L.tile_capacity;  // ring: where the consumed half of the flags starts
  g.counter = 0;
  Phase ph(MOK_PHASE_FWD_FUSED, st, 1);
  const int grid = gemm_grid(L.tile_capacity * (g.g1_tiles + g.n_tiles));
  if (prec == MOK_MXFP8)
    MOK_CUDA(launch_gemm_mx(GM_FWD_FUSED, maps, g, grid, st));
  else
    MOK_CUDA(launch_gemm(GM_FWD_FUSED, maps, g, grid, st));
  return MOK_OK;
}

mok_status mok_backward(const mok_shape* shape, const mok_config* cfg, mok_precision prec, void* ws,
                        size_t ws_bytes, const void* ctx, const void* x, const float* scores, const void* W1,
                        const void* W3, const void* W2, const void* dout, void* dX, void* dW1, void* dW3,
                        void* dW2, float* dscores, void* stream) {
  MOK_TRY(check_shape(shape));
  MOK_TRY(check_config(cfg));
  MOK_TRY(check_prec(prec));
  if (!ws || !ctx || !x || !scores || !W1 || !W3 || !W2 || !dout || !dX || !dW1 || !dW3 || !dW2 || !dscores)
    return MOK_ERR_INVALID_ARG;
  const mok_shape& s = *shape;
  const WsLayout L = ws_layout(s, *cfg, prec, device_sm_count());
  if (ws_bytes < L.total) return MOK_ERR_WORKSPACE_TOO_SMALL;
  // MXFP8 descriptors are checked before anything touches the device; with
  // replay, W1 and W3 each point to two descriptors: the backward's
  // orientation (along I) and the forward's (along H, for the replayed GEMM1)
  const mok_mx* f1 = nullptr;
  const mok_mx* f3 = nullptr;
  if (prec == MOK_MXFP8) {
    if (!mx_ok(W1) || !mx_ok(W3) || !mx_ok(W2)) return MOK_ERR_INVALID_ARG;
    if (cfg->replay) {
      f1 = as_mx(W1) + 1;
      f3 = as_mx(W3) + 1;
      if (!mx_ok(f1) || !mx_ok(f3)) return MOK_ERR_INVALID_ARG;
    }
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* w = static_cast<uint8_t*>(ws);
  MOK_TRY(reset_counters(w, L, st));
  const uint64_t P = L.pad_capacity;
  const int bn_i = (s.I % 256 == 0) ? 256 : 128;
  const int bn_h = (s.H % 256 == 0) ? 256 : 128;

  if (prec == MOK_MXFP8) {
    return backward_mx(s, L, w, *cfg, ctx, x, scores, *as_mx(W1), *as_mx(W3), *as_mx(W2), f1, f3, dout, dX, dW1,
                       dW3, dW2, dscores, st);
  }
  GemmParams g;
  base_params(g, s, L, w);
  g.ctx_hu = const_cast<__nv_bfloat16*>(static_cast<const __nv_bfloat16*>(ctx));
  g.dhu = reinterpret_cast<__nv_bfloat16*>(w + L.dhu);
  g.as = reinterpret_cast<__nv_bfloat16*>(w + L.as);
  g.dsp = reinterpret_cast<float*>(w + L.dsp);
  g.scores = scores;
  g.yk = reinterpret_cast<__nv_bfloat16*>(w + L.yk);

  if (cfg->replay) {
    // Bounded-memory backward: [h|u] of the minibatches the forward context
    // no longer holds is recomputed by GEMM1 straight into the rows of
    // dh|du, and the last ring_slots minibatches are copied there from the
    // context; the dA' epilogue reads [h|u] there and overwrites it in place.
    Phase ph(MOK_PHASE_BWD_REPLAY, st, 2);
    MOK_CUDA(launch_replay_copy(s, L, w, static_cast<const __nv_bfloat16*>(ctx), g.dhu, st));
    TmapSet m;
    memset(&m, 0, sizeof(m));
    if (!map_gather(&m.m[0], x, s.H, s.T) || !map3d(&m.m[1], W1, s.I, s.H, s.E, 64) ||
        !map3d(&m.m[2], W3, s.I, s.H, s.E, 64))
      return MOK_ERR_CUDA;
    GemmParams q = g;
    q.ctx_hu = g.dhu;
    q.ring = reinterpret_cast<__nv_bfloat16*>(w + L.ring);  // a: scratch here
    q.ring_rows = L.minibatch_rows;
    q.ring_slots = L.ring_slots;
    q.gather_src = static_cast<const __nv_bfloat16*>(x);
    q.nmaps = 3;
    q.bn = 256;
    q.n_tiles = s.I / 128;
    q.m_tile_begin = 0;
    q.m_tile_end = (int)L.tile_capacity;
    q.replay_keep = L.ring_slots;
    q.counter = 6;
    MOK_CUDA(launch_gemm(GM_FWD1, m, q, gemm_grid(L.tile_capacity * q.n_tiles), st));
    g.ctx_hu = g.dhu;
  }

  // Token-sorted copies (rows in padded schedule order, zero padding rows)
  // feed dA' and dW2 (dout), then dW1|dW3 (x), through one buffer; with
  // MOK_DEBUG_FUSED_WGRAD_GATHER those GEMMs gather rows in their load path.
  const bool sorted = (cfg->debug_flags & MOK_DEBUG_FUSED_WGRAD_GATHER) == 0;
  __nv_bfloat16* srt = reinterpret_cast<__nv_bfloat16*>(w + L.sorted2);    // dout
  __nv_bfloat16* srt_x = reinterpret_cast<__nv_bfloat16*>(w + L.sorted);   // x
  // dA' and dX on CTA pairs: two tiles of one expert per cluster, each CTA
  // loading a 128-row half of the 256-row weight tile.  dA' only for long K
  // (H): with short main loops it is bound by its SwiGLU-backward epilogue,
  // where a pair only adds the coupling of two CTAs (measured: 13% slower
  // at H = 2048, 3% faster at H = 7168).
  const bool pairs_da = sorted && bn_i == 256 && s.H >= 4096 && row_pairs(*cfg);
  const bool pairs_dx = bn_h == 256 && row_pairs(*cfg);
  if (sorted) {
    Phase ph(MOK_PHASE_BWD_SORT, st, 1);
    MOK_CUDA(launch_gather_rows(s, L, w, static_cast<const __nv_bfloat16*>(dout), srt, st));
  }
  // dA' = sorted(dout) W2^T, SwiGLU backward + router-score partials
  {
    TmapSet m, mp;
    memset(&m, 0, sizeof(m));
    if (sorted ? !map2d(&m.m[0], srt, s.H, P, 128) : !map_gather(&m.m[0], dout, s.H, s.T)) return MOK_ERR_CUDA;
    if (!map3d(&m.m[1], W2, s.H, s.I, s.E, bn_i)) return MOK_ERR_CUDA;
    mp = m;
    if (pairs_da && !map3d(&mp.m[1], W2, s.H, s.I, s.E, 128)) return MOK_ERR_CUDA;
    GemmParams q = g;
    q.gather_src = static_cast<const __nv_bfloat16*>(dout);
    q.rows_sorted = sorted ? 1 : 0;
    q.nmaps = 2;
    q.bn = bn_i;
    q.n_tiles = s.I / bn_i;
    q.m_tile_begin = 0;
    q.m_tile_end = (int)L.tile_capacity;
    q.counter = 0;
    {
      Phase ph(MOK_PHASE_BWD_DA, st, (pairs_da || pairs_dx) ? 2 : 1);
      // every expert on pairs (an odd last tile a solo pair): measured faster
      // for dA' and dX than splitting the short experts off onto single CTAs
      if (pairs_da || pairs_dx) MOK_CUDA(launch_split_table(L, w, 1, st));
      if (pairs_da) set_pair_table(q, L, w);
      MOK_CUDA(launch_rows(GM_BWD_DA, pairs_da, mp, m, q, gemm_grid(L.tile_capacity * q.n_tiles), st));
    }
    Phase ph(MOK_PHASE_BWD_DS, st, 1);
    MOK_CUDA(launch_ds_reduce(s, L, w, dscores, q.n_tiles, st));
  }
  // dX parts = [dh|du] [W1|W3]^T scattered to token order, then summed over k
  {
    TmapSet m, mp;
    memset(&m, 0, sizeof(m));
    if (!map2d(&m.m[0], g.dhu, 2 * (uint64_t)s.I, P, 128) || !map3d(&m.m[1], W1, s.I, s.H, s.E, bn_h) ||
        !map3d(&m.m[2], W3, s.I, s.H, s.E, bn_h))
      return MOK_ERR_CUDA;
    mp = m;
    if (pairs_dx && (!map3d(&mp.m[1], W1, s.I, s.H, s.E, 128) || !map3d(&mp.m[2], W3, s.I, s.H, s.E, 128)))
      return MOK_ERR_CUDA;
    GemmParams q = g;
    q.nmaps = 3;
    q.bn = bn_h;
    q.n_tiles = s.H / bn_h;
    q.m_tile_begin = 0;
    q.m_tile_end = (int)L.tile_capacity;
    q.counter = 1;
    if (pairs_dx) set_pair_table(q, L, w);
    {
      Phase ph(MOK_PHASE_BWD_DX, st, 1);
      MOK_CUDA(launch_rows(GM_BWD_DX, pairs_dx, mp, m, q, gemm_grid(L.tile_capacity * q.n_tiles), st));
    }
    Phase ph(MOK_PHASE_BWD_DX_COMBINE, st, 1);
    MOK_CUDA(launch_combine(s, L, w, g.yk, nullptr, static_cast<__nv_bfloat16*>(dX), st));
  }
  // dW2 = (s a)^T sorted(dout), per expert
  {
    TmapSet m;
    memset(&m, 0, sizeof(m));
    if (!map2d(&m.m[0], g.as, s.I, P, 64)) return MOK_ERR_CUDA;
    if (sorted ? !map2d(&m.m[1], srt, s.H, P, 64) : !map_gather(&m.m[1], dout, s.H, s.T)) return MOK_ERR_CUDA;
    GemmParams q = g;
    q.nmaps = 2;
    q.bn = bn_h;
    q.n_tiles = s.H / bn_h;
    q.m_tiles = s.I / 128;
    q.counter = 3;
    q.wg_sorted = sorted ? 1 : 0;
    q.gather_src = static_cast<const __nv_bfloat16*>(dout);
    q.dW2 = static_cast<__nv_bfloat16*>(dW2);
    Phase ph(MOK_PHASE_BWD_WG2, st, 0);
    int n = 0;
    MOK_CUDA(launch_wgrad(GM_WG2, m, q, gemm_grid((long)s.E * q.m_tiles * q.n_tiles), cfg->debug_flags, 5, &n, st));
    g_launches += n;
  }
  // dW1 | dW3 = sorted(x)^T [dh|du], per expert; the sort of x does
  // nothing when the forward left its sorted copy in place
  {
    TmapSet m;
    memset(&m, 0, sizeof(m));
    if (sorted) {
      Phase ph(MOK_PHASE_BWD_SORT, st, 1);
      MOK_CUDA(launch_gather_rows(s, L, w, static_cast<const __nv_bfloat16*>(x), srt_x, st,
                                  reinterpret_cast<const int32_t*>(w + L.header) + kHdrSortedX));
    }
    if (sorted ? !map2d(&m.m[0], srt_x, s.H, P, 64) : !map_gather(&m.m[0], x, s.H, s.T)) return MOK_ERR_CUDA;
    if (!map2d(&m.m[1], g.dhu, 2 * (uint64_t)s.I, P, 64)) return MOK_ERR_CUDA;
    GemmParams q = g;
    q.nmaps = 2;
    q.bn = 256;
    q.n_tiles = 2 * s.I / 256;
    q.m_tiles = s.H / 128;
    q.counter = 2;
    q.wg_sorted = sorted ? 1 : 0;
    q.gather_src = static_cast<const __nv_bfloat16*>(x);
    q.dW1 = static_cast<__nv_bfloat16*>(dW1);
    q.dW3 = static_cast<__nv_bfloat16*>(dW3);
    Phase ph(MOK_PHASE_BWD_WG13, st, 0);
    int n = 0;
    MOK_CUDA(launch_wgrad(GM_WG13, m, q, gemm_grid((long)s.E * q.m_tiles * q.n_tiles), cfg->debug_flags, 4, &n, st));
    g_launches += n;
  }
  return MOK_OK;
}

mok_status mok_mxfp8_quantize(const void* src, int32_t batch, int32_t rows, int32_t cols, int32_t block_axis,
                              uint8_t* q, uint8_t* scale, void* stream) {
  if (!src || !q || !scale) return MOK_ERR_INVALID_ARG;
  if (batch < 1 || rows < 1 || cols < 1) return MOK_ERR_INVALID_ARG;
  if (block_axis != 0 && block_axis != 1) return MOK_ERR_INVALID_ARG;
  if (block_axis == 0 && rows % 32) return MOK_ERR_UNSUPPORTED;
  if (block_axis == 1 && cols % 32) return MOK_ERR_UNSUPPORTED;
  g_launches += 1;
  MOK_CUDA(launch_mxfp8_quantize(static_cast<const __nv_bfloat16*>(src), batch, rows, cols, block_axis, q, scale,
                                 static_cast<cudaStream_t>(stream)));
  return MOK_OK;
}

size_t mok_schedule_workspace_size(const mok_shape* shape, const mok_config* cfg) {
  if (check_shape(shape) != MOK_OK || check_config(cfg) != MOK_OK) return 0;
  const WsLayout L = ws_layout(*shape, *cfg, MOK_BF16, device_sm_count());
  return L.chunk_base + align256(L.nchunks * shape->E * 4);
}

mok_status mok_ep_pack_rows(const mok_shape* shape, const mok_config* cfg, const void* ws, size_t ws_bytes,
                            const void* x, const float* scores, void* rows, float* row_scores, void* stream) {
  MOK_TRY(check_shape(shape));
  MOK_TRY(check_config(cfg));
  if (!ws || !x || !rows || (row_scores && !scores)) return MOK_ERR_INVALID_ARG;
  if (ws_bytes < mok_schedule_workspace_size(shape, cfg)) return MOK_ERR_WORKSPACE_TOO_SMALL;
  const WsLayout L = ws_layout(*shape, *cfg, MOK_BF16, device_sm_count());
  g_launches += 1;
  MOK_CUDA(launch_ep_pack(*shape, L, static_cast<const uint8_t*>(ws), static_cast<const __nv_bfloat16*>(x),
                          scores, static_cast<__nv_bfloat16*>(rows), row_scores, static_cast<cudaStream_t>(stream)));
  return MOK_OK;
}

mok_status mok_ep_combine_rows(const mok_shape* shape, const mok_config* cfg, const void* ws, size_t ws_bytes,
                               const void* rows, const float* scores, void* out, void* stream) {
  MOK_TRY(check_shape(shape));
  MOK_TRY(check_config(cfg));
  if (!ws || !rows || !out) return MOK_ERR_INVALID_ARG;
  if (ws_bytes < mok_schedule_workspace_size(shape, cfg)) return MOK_ERR_WORKSPACE_TOO_SMALL;
  const WsLayout L = ws_layout(*shape, *cfg, MOK_BF16, device_sm_count());
  g_launches += 1;
  MOK_CUDA(launch_ep_combine(*shape, L, static_cast<const uint8_t*>(ws), static_cast<const __nv_bfloat16*>(rows),
                             scores, static_cast<__nv_bfloat16*>(out), static_cast<cudaStream_t>(stream)));
  return MOK_OK;
}

mok_status mok_ep_unsort_scores(const mok_shape* shape, const mok_config* cfg, const void* ws, size_t ws_bytes,
                                const float* row_vals, float* out, void* stream) {
  MOK_TRY(check_shape(shape));
  MOK_TRY(check_config(cfg));
  if (!ws || !row_vals || !out) return MOK_ERR_INVALID_ARG;
  if (ws_bytes < mok_schedule_workspace_size(shape, cfg)) return MOK_ERR_WORKSPACE_TOO_SMALL;
  const WsLayout L = ws_layout(*shape, *cfg, MOK_BF16, device_sm_count());
  g_launches += 1;
  MOK_CUDA(launch_ep_unsort(*shape, L, static_cast<const uint8_t*>(ws), row_vals, out,
                            static_cast<cudaStream_t>(stream)));
  return MOK_OK;
}

mok_status mok_gather_rows(const mok_shape* shape, const mok_config* cfg, const void* ws, size_t ws_bytes,
                           const void* x, void* xg, void* stream) {
  MOK_TRY(check_shape(shape));
  MOK_TRY(check_config(cfg));
  if (!ws || !x || !xg) return MOK_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(*shape, *cfg, MOK_BF16, device_sm_count());
  if (ws_bytes < L.chunk_base) return MOK_ERR_WORKSPACE_TOO_SMALL;
  g_launches += 1;
  MOK_CUDA(launch_gather_rows(*shape, L, static_cast<const uint8_t*>(ws), static_cast<const __nv_bfloat16*>(x),
                              static_cast<__nv_bfloat16*>(xg), static_cast<cudaStream_t>(stream)));
  return MOK_OK;
}

mok_status mok_gemm_bf16(int32_t M, int32_t N, int32_t K, const void* A, int32_t a_mn_major, const void* B,
                         int32_t b_mn_major, float* C, void* scratch, void* stream) {
  if (!A || !B || !C || !scratch) return MOK_ERR_INVALID_ARG;
  if (M < 128 || N < 128 || K < 64 || M % 128 || N % 128 || K % 64) return MOK_ERR_UNSUPPORTED;
  const int bn = (N % 256 == 0) ? 256 : 128;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int32_t* hdr = static_cast<int32_t*>(scratch);
  MOK_CUDA(cudaMemsetAsync(hdr, 0, kHeaderWords * 4, st));
  TmapSet m;
  memset(&m, 0, sizeof(m));
  bool ok = a_mn_major ? map2d(&m.m[0], A, M, K, 64) : map2d(&m.m[0], A, K, M, 128);
  ok = ok && (b_mn_major ? map2d(&m.m[1], B, N, K, 64) : map2d(&m.m[1], B, K, N, bn));
  if (!ok) return MOK_ERR_CUDA;
  GemmParams g;
  memset(&g, 0, sizeof(g));
  g.nmaps = 2;
  g.bn = bn;
  g.n_tiles = N / bn;
  g.m_tiles = M / 128;
  g.k_iters = K / 64;
  g.hdr = hdr;
  g.out_f32 = C;
  g.ld_out = N;
  g.a_mn = a_mn_major ? 1 : 0;
  g.b_mn = b_mn_major ? 1 : 0;
  g_launches += 1;
  MOK_CUDA(launch_gemm(GM_DENSE, m, g, gemm_grid((long)g.m_tiles * g.n_tiles), st));
  return MOK_OK;
}

mok_status mok_trace_enable(int32_t on) {
  std::lock_guard<std::mutex> lk(g_trace_mu);
  g_trace_on = on != 0;
  return MOK_OK;
}

mok_status mok_trace_read(float* ms, int32_t* count) {
  if (!ms || !count) return MOK_ERR_INVALID_ARG;
  std::vector<TraceRec> recs;
  {
    std::lock_guard<std::mutex> lk(g_trace_mu);
    recs.swap(g_trace);
  }
  for (int i = 0; i < MOK_NUM_PHASES; ++i) {
    ms[i] = 0.0f;
    count[i] = 0;
  }
  mok_status st = MOK_OK;
  for (const TraceRec& r : recs) {
    float t = 0.0f;
    if (cudaEventSynchronize(r.b) != cudaSuccess || cudaEventElapsedTime(&t, r.a, r.b) != cudaSuccess)
      st = MOK_ERR_CUDA;
    if (r.phase >= 0 && r.phase < MOK_NUM_PHASES) {
      ms[r.phase] += t;
      count[r.phase] += 1;
    }
    cudaEventDestroy(r.a);
    cudaEventDestroy(r.b);
  }
  return st;
}

int64_t mok_launch_count(void) { return g_launches.load(); }

mok_status mok_gemm_mxfp8(int32_t M, int32_t N, int32_t K, const uint8_t* Aq, const uint8_t* Asf,
                          int32_t a_mn_major, const uint8_t* Bq, const uint8_t* Bsf, int32_t b_mn_major, float* C,
                          void* scratch, size_t scratch_bytes, void* stream) {
  if (!Aq || !Asf || !Bq || !Bsf || !C || !scratch) return MOK_ERR_INVALID_ARG;
  if (M < 128 || N < 128 || K < 128 || M % 128 || N % 128 || K % 128) return MOK_ERR_UNSUPPORTED;
  const size_t need = 256 + (size_t)M * K / 32 + (size_t)N * K / 32;
  if (scratch_bytes < need) return MOK_ERR_WORKSPACE_TOO_SMALL;
  const int bn = (N % 256 == 0) ? 256 : 128;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* sc = static_cast<uint8_t*>(scratch);
  uint8_t* sfa_t = sc + 256;
  uint8_t* sfb_t = sfa_t + (size_t)M * K / 32;
  MOK_CUDA(cudaMemsetAsync(sc, 0, kHeaderWords * 4, st));
  // both operands' scales re-tiled for the TMA thread's bulk loads
  if (a_mn_major)
    MOK_CUDA(launch_tile_scales(Asf, 1, K / 32, M, sfa_t, st));
  else
    MOK_CUDA(launch_tile_scales_rows(Asf, 1, M, K / 32, sfa_t, st));
  if (b_mn_major)
    MOK_CUDA(launch_tile_scales(Bsf, 1, K / 32, N, sfb_t, st, bn / 128, bn / 128, 0));
  else
    MOK_CUDA(launch_tile_scales_rows(Bsf, 1, N, K / 32, sfb_t, st, bn / 128, bn / 128, 0));
  const int kernels = 3;
  TmapSet m;
  memset(&m, 0, sizeof(m));
  bool ok = a_mn_major ? map2d_u8(&m.m[0], Aq, M, K, 128, 128) : map2d_u8(&m.m[0], Aq, K, M, 128, 128);
  ok = ok && (b_mn_major ? map2d_u8(&m.m[1], Bq, N, K, 128, 128) : map2d_u8(&m.m[1], Bq, K, N, 128, bn));
  if (!ok) return MOK_ERR_CUDA;
  GemmParams g;
  memset(&g, 0, sizeof(g));
  g.nmaps = 2;
  g.bn = bn;
  g.n_tiles = N / bn;
  g.m_tiles = M / 128;
  g.k_iters = K / 128;
  g.hdr = reinterpret_cast<int32_t*>(sc);
  g.out_f32 = C;
  g.ld_out = N;
  g.a_mn = a_mn_major ? 1 : 0;
  g.b_mn = b_mn_major ? 1 : 0;
  g.sfa_rows = Asf;
  g.sfa_ld = K / 32;
  g.sfb_rows0 = Bsf;
  g.sfb_ld = K / 32;
  g.sfa_tiled = sfa_t;
  g.sfb_tiled0 = sfb_t;
  g_launches += kernels;
  MOK_CUDA(launch_gemm_mx(GM_DENSE, m, g, gemm_grid((long)g.m_tiles * g.n_tiles), st));
  return MOK_OK;
}

// ------------------------------------------------------------------ router
namespace {

struct RouterLayout {
  int Tpad, Epad;
  size_t header, wpad, logits, dl, dwr, total;
};

RouterLayout router_layout(const mok_shape& s) {
  RouterLayout r;
  r.Tpad = (s.T + 127) / 128 * 128;
  r.Epad = (s.E + 127) / 128 * 128;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += (bytes + 255) / 256 * 256;
    return o;
  };
  r.header = take(kHeaderWords * 4);
  r.wpad = take((size_t)s.H * r.Epad * 2);
  r.logits = take((size_t)r.Tpad * r.Epad * 4);
  r.dl = take((size_t)r.Tpad * r.Epad * 2);
  r.dwr = take((size_t)s.H * r.Epad * 4);
  r.total = off;
  return r;
}

mok_status check_router(const mok_shape* s) {
  MOK_TRY(check_shape(s));
  if (s->k > s->E) return MOK_ERR_INVALID_ARG;
  return MOK_OK;
}

// N tile of a router GEMM: 128 columns when 256-column tiles would leave SMs
// idle (the logits and dWr GEMMs have few output tiles: N is the expert
// count).  A K-major B operand's tensor map box must be this many rows.
int router_bn(int M, int N) {
  return (N % 256 == 0 && (long)(M / 128) * (N / 256) >= device_sm_count()) ? 256 : 128;
}

// One tcgen05 GEMM of the router (GM_DENSE) on the router workspace.
mok_status router_gemm(uint8_t* rw, const TmapSet& m, int M, int N, int K, int a_mn, int b_mn, float* out_f32,
                       __nv_bfloat16* out_bf16, long ld_out, long m_valid, int counter, cudaStream_t st) {
  GemmParams g;
  memset(&g, 0, sizeof(g));
  g.nmaps = 2;
  g.bn = router_bn(M, N);
  g.n_tiles = N / g.bn;
  g.m_tiles = M / 128;
  g.k_iters = K / 64;
  g.hdr = reinterpret_cast<int32_t*>(rw);
  g.counter = counter;
  g.out_f32 = out_f32;
  g.out_bf16 = out_bf16;
  g.ld_out = ld_out;
  g.m_valid = m_valid;
  g.a_mn = a_mn;
  g.b_mn = b_mn;
  MOK_CUDA(launch_gemm(GM_DENSE, m, g, gemm_grid((long)g.m_tiles * g.n_tiles), st));
  return MOK_OK;
}

}  // namespace

size_t mok_router_workspace_size(const mok_shape* shape) {
  if (check_router(shape) != MOK_OK) return 0;
  return router_layout(*shape).total;
}

mok_status mok_router_forward(const mok_shape* shape, void* rws, size_t rws_bytes, const void* x, const void* Wr,
                              const float* bias, int32_t* topk_idx, float* scores, float* logits, void* stream) {
  MOK_TRY(check_router(shape));
  if (!rws || !x || !Wr || !topk_idx || !scores) return MOK_ERR_INVALID_ARG;
  const mok_shape& s = *shape;
  const RouterLayout R = router_layout(s);
  if (rws_bytes < R.total) return MOK_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* rw = static_cast<uint8_t*>(rws);
  // a forward starts a router step: the whole header, error word included
  // (as the layer's schedule call does)
  MOK_CUDA(cudaMemsetAsync(rw, 0, kHeaderWords * 4, st));
  __nv_bfloat16* wpad = reinterpret_cast<__nv_bfloat16*>(rw + R.wpad);
  float* lg = reinterpret_cast<float*>(rw + R.logits);
  Phase ph(MOK_PHASE_ROUTER_FWD, st, logits ? 4 : 3);
  MOK_CUDA(launch_router_pad_weights(s.H, s.E, R.Epad, static_cast<const __nv_bfloat16*>(Wr), wpad, st));
  // logits [Tpad, Epad] = x [T, H] Wr: A K-major (rows past T read as zero), B N-major
  TmapSet m;
  memset(&m, 0, sizeof(m));
  if (!map2d(&m.m[0], x, s.H, s.T, 128) || !map2d(&m.m[1], wpad, R.Epad, s.H, 64)) return MOK_ERR_CUDA;
  MOK_TRY(router_gemm(rw, m, R.Tpad, R.Epad, s.H, 0, 1, lg, nullptr, R.Epad, 0, 0, st));
  MOK_CUDA(launch_router_topk(s.T, s.E, R.Epad, s.k, lg, bias, topk_idx, scores, st));
  if (logits) MOK_CUDA(launch_router_take_cols(s.T, s.E, R.Epad, lg, logits, st));
  return MOK_OK;
}

mok_status mok_router_backward(const mok_shape* shape, void* rws, size_t rws_bytes, const void* x, const void* Wr,
                               const int32_t* topk_idx, const float* scores, const float* dscores, float* dWr,
                               void* dx_router, void* stream) {
  MOK_TRY(check_router(shape));
  if (!rws || !x || !Wr || !topk_idx || !scores || !dscores || !dWr || !dx_router) return MOK_ERR_INVALID_ARG;
  const mok_shape& s = *shape;
  const RouterLayout R = router_layout(s);
  if (rws_bytes < R.total) return MOK_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* rw = static_cast<uint8_t*>(rws);
  MOK_CUDA(cudaMemsetAsync(rw + kHdrAbort * 4, 0, (kHdrCounters + kNumCounters - kHdrAbort) * 4, st));
  __nv_bfloat16* wpad = reinterpret_cast<__nv_bfloat16*>(rw + R.wpad);
  __nv_bfloat16* dl = reinterpret_cast<__nv_bfloat16*>(rw + R.dl);
  float* dwr = reinterpret_cast<float*>(rw + R.dwr);
  Phase ph(MOK_PHASE_ROUTER_BWD, st, 5);
  MOK_CUDA(launch_router_pad_weights(s.H, s.E, R.Epad, static_cast<const __nv_bfloat16*>(Wr), wpad, st));
  MOK_CUDA(launch_router_logit_grad(s.T, R.Tpad, s.E, R.Epad, s.k, topk_idx, scores, dscores, dl, st));
  // dWr [H, Epad] = x^T dL: A = x read M-major (rows past T read as zero), B = dL N-major
  {
    TmapSet m;
    memset(&m, 0, sizeof(m));
    if (!map2d(&m.m[0], x, s.H, s.T, 64) || !map2d(&m.m[1], dl, R.Epad, R.Tpad, 64)) return MOK_ERR_CUDA;
    MOK_TRY(router_gemm(rw, m, s.H, R.Epad, R.Tpad, 1, 1, dwr, nullptr, R.Epad, 0, 1, st));
    MOK_CUDA(launch_router_take_cols(s.H, s.E, R.Epad, dwr, dWr, st));
  }
  // dx [T, H] = dL Wr^T: A = dL K-major, B = padded Wr K-major; bf16 rows < T
  {
    TmapSet m;
    memset(&m, 0, sizeof(m));
    const int bn = router_bn(R.Tpad, s.H);
    if (!map2d(&m.m[0], dl, R.Epad, R.Tpad, 128) || !map2d(&m.m[1], wpad, R.Epad, s.H, bn)) return MOK_ERR_CUDA;
    MOK_TRY(router_gemm(rw, m, R.Tpad, s.H, R.Epad, 0, 0, nullptr, static_cast<__nv_bfloat16*>(dx_router), s.H,
                        s.T, 2, st));
  }
  return MOK_OK;
}

mok_status mok_check(void* ws, void* stream) {
  if (!ws) return MOK_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  MOK_CUDA(cudaStreamSynchronize(st));
  int32_t word = 0;
  MOK_CUDA(cudaMemcpy(&word, ws, sizeof(word), cudaMemcpyDeviceToHost));
  MOK_CUDA(cudaMemset(ws, 0, sizeof(word)));
  if (word & MOK_ERRBIT_TIMEOUT) return MOK_ERR_TIMEOUT;
  if (word & MOK_ERRBIT_BAD_INDEX) return MOK_ERR_BAD_INDEX;
  return MOK_OK;
}

}  // extern "C"

/*
 * mok.h -- C ABI of the GB300 (sm_103a) MoE layer library, libmok.so.
 *
 * The layer is the routed SwiGLU mixture-of-experts layer of the
 * Mixture-of-Kittens pages, on one GPU: a device-side schedule, dispatch
 * (gather by expert), expert-grouped GEMMs W1|W3 -> SwiGLU -> W2, a
 * deterministic weighted combine, and the full backward with the
 * router-score gradient fused into the SwiGLU backward.  BF16 and MXFP8.
 *
 * Citations name the page and its section:
 *   [MoK]  "Mixture-of-Kittens (MoK)" project summary (English): sections
 *          "What it is", "Use the functional API", "Core concepts",
 *          "Limitations / considerations".
 *   [MTP]  "Cursor Open-Sources Mixture-of-Kittens (MoK): A Deterministic MoE
 *          Training Megakernel for GB300 NVL72 Racks": section "Three design
 *          decisions that matter" (paragraphs: communication direction,
 *          overlap granularity, ring token buffer) and the paragraph after it.
 *   [NOTE] "Mixture-of-Kittens: our open-source MoE megakernel for NVL72s",
 *          section 2 (minibatch) and section 3 (ring token buffer).
 *
 * Conventions for every call
 *  - Pointers marked (device) are CUDA device pointers on the current device;
 *    the library reads or writes them only from kernels enqueued on `stream`
 *    (a cudaStream_t passed as void*; NULL is the legacy default stream).
 *  - Ownership: the caller allocates and frees every buffer, including the
 *    workspace and the forward context ("you manage all tensors yourself",
 *    [MoK] "Core concepts", ops-layer row).  The library allocates no device
 *    memory and keeps no per-call global state.
 *  - Asynchrony: calls only enqueue work; none synchronises or reads device
 *    data back to the host.
 *  - Errors found on the host (null pointers, unsupported shapes, too small a
 *    workspace, comm_sms != 0) return before anything is enqueued.  Errors
 *    found on the device (an expert id outside [0, E), a bounded wait that
 *    ran out) are recorded in the workspace's error word and reported by
 *    mok_check().  Outputs of a call that recorded a device error are
 *    unspecified.
 *  - Layouts are row-major and dense.  Shapes: T tokens, H hidden size,
 *    I expert intermediate size, E experts, k experts per token,
 *    R = T*k routed rows, flat routed index f = t*k + j.
 *  - Supported sizes: H % 128 == 0, I % 128 == 0, 1 <= k <= 32,
 *    1 <= E <= 1024, T >= 1, T*k < 2^31 / max(H, 2I).
 */
#ifndef MOK_H_
#define MOK_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOK_OK = 0,
  MOK_ERR_INVALID_ARG = 1,         /* null pointer, bad shape or config value */
  MOK_ERR_UNSUPPORTED = 2,         /* a size or mode this build does not support */
  MOK_ERR_WORKSPACE_TOO_SMALL = 3, /* ws_bytes < mok_workspace_size() */
  MOK_ERR_CUDA = 4,                /* a CUDA runtime/driver call failed */
  MOK_ERR_BAD_INDEX = 5,           /* device: an expert id outside [0, E) */
  MOK_ERR_TIMEOUT = 6              /* device: a bounded wait ran out */
} mok_status;

typedef enum { MOK_BF16 = 0, MOK_MXFP8 = 1 } mok_precision;

typedef struct {
  int32_t T, H, I, E, k;
} mok_shape;

/*
 * Tunable knobs ([MoK] "Core concepts", Config row: communication SM count,
 * minibatch granularity, macrobatch size, schedule capacity multiplier; the
 * pages name a fifth knob without saying what it is, so it is not invented).
 *
 * minibatch_rows  Routed (expert-sorted, padded) rows per minibatch of the
 *                 forward ring, rounded up to a whole number of 128-row
 *                 tiles (2368 runs as 2432), or 0 for the default:
 *                 the two-wave floor 2*C*128*256/min(2I, H) ([MTP]
 *                 overlap-granularity paragraph, [NOTE] section 2) with C
 *                 the device's SM count, rounded up to a multiple of 128.
 * ring_slots      Minibatch slots in the ring token buffer (the macrobatch,
 *                 [MTP] ring-token-buffer paragraph); >= 2, or 0 for 4.
 * capacity_mult   Schedule capacity multiplier.  On one GPU the schedule is
 *                 always sized for the worst case (R + E*127 padded rows),
 *                 so no token is ever dropped; accepted values are 0 (= 1)
 *                 and >= 1, and values above 1 change nothing.
 * comm_sms        SMs reserved for inter-GPU transfers.  There are none on
 *                 one GPU: must be 0.
 * debug_flags     0 in normal use.  Bit 0 (MOK_DEBUG_SKIP_RING_SIGNAL):
 *                 the forward ring producer skips one completion signal, so
 *                 its consumer's bounded wait runs out and the call records
 *                 MOK_ERR_TIMEOUT -- a host-chosen fault used to test the
 *                 failure path without faulting the GPU.
 *                 Bit 1 (MOK_DEBUG_SERIAL_RING): run the forward's two GEMMs
 *                 as one launch pair per minibatch (same ring, stream order)
 *                 instead of the single persistent ring launch.
 *                 Bit 2 (MOK_DEBUG_FUSED_WGRAD_GATHER): the BF16 backward's
 *                 dA' and weight-gradient GEMMs gather token rows in their
 *                 load path instead of reading token-sorted copies (dA' then
 *                 runs one CTA per tile); the MXFP8 dA' gathers dout's E4M3
 *                 rows instead of reading their token-sorted copy.
 *                 Bit 3 (MOK_DEBUG_SINGLE_CTA_WGRAD): the BF16 weight-gradient
 *                 GEMMs run one CTA per 128-row tile instead of clusters of
 *                 two CTAs sharing a 256-row tile (cta_group::2).
 *                 Bit 4 (MOK_DEBUG_SINGLE_CTA_ROWS): the BF16 backward's dA'
 *                 and dX GEMMs run one CTA per 128-row tile instead of
 *                 clusters of two CTAs sharing two tiles of one expert.
 *                 Bit 5 (MOK_DEBUG_SINGLE_CTA_RING): the BF16 forward ring
 *                 runs every tile on one CTA, in one launch.  By default
 *                 (T >= 1024, replay = 0) it runs in two launches, every
 *                 expert wholly in one: experts of at least 8 tiles of 128
 *                 rows on clusters of two CTAs (two tiles of one expert per
 *                 256 x 256 tile; an odd last tile leaves one CTA idle), then
 *                 the others on single CTAs.
 *                 Both forms read a token-sorted copy of x with plain TMA.
 *                 Bit 6 (MOK_DEBUG_GATHER_X_RING): the single-CTA ring
 *                 gathers token rows of x (MXFP8: of x's E4M3 codes) in its
 *                 load path instead of reading a token-sorted copy with
 *                 plain TMA (in BF16 the backward's dW1|dW3 then sorts x
 *                 itself).
 *                 Bit 7 (MOK_DEBUG_NO_OVERLAP): no two launches overlap (see
 *                 overlap_sms): the forward ring's pair launch runs first,
 *                 then the single-CTA one.
 *                 Results are bitwise the same in every mode.
 * replay          0: the forward context holds [h|u] of every routed row.
 *                 1: it holds [h|u] of the last ring_slots minibatches
 *                 only, in ring-slot order (mok_ctx_size shrinks to
 *                 ring_slots * minibatch_rows rows), and the backward
 *                 recomputes GEMM1 for the earlier minibatches -- the pages'
 *                 bounded-memory backward ([MTP] ring-token-buffer
 *                 paragraph; [NOTE] §3).  Recomputed values are bitwise
 *                 those of the forward.  In MXFP8 mode the recomputation
 *                 needs the forward's weight orientation too: mok_backward's
 *                 W1 and W3 then each point to TWO consecutive mok_mx, the
 *                 backward orientation (along I) followed by the forward
 *                 one (along H).
 * overlap_sms     SMs given to the first launch of the overlapped pair, or
 *                 0 for the default rule.  In the BF16 forward with the ring
 *                 in two launches, the single-CTA launch of the short
 *                 experts (bound by streaming their weights) and the
 *                 CTA-pair launch of the long ones overlap on the caller's
 *                 stream (programmatic dependent launch: the first lets the
 *                 second start at once on the SMs it leaves free; the second
 *                 takes each SM the first leaves and waits for it before it
 *                 ends).  By default the first keeps the share of the SMs
 *                 that its tiles make of both launches' tiles (a pair tile
 *                 counted at 4/5 of a single one), all of them when there is
 *                 no pair.  Must be >= 0.
 */
typedef struct {
  int32_t minibatch_rows;
  int32_t ring_slots;
  float capacity_mult;
  int32_t comm_sms;
  int32_t debug_flags;
  int32_t replay;
  int32_t overlap_sms;
} mok_config;

#define MOK_DEBUG_SKIP_RING_SIGNAL 1
#define MOK_DEBUG_SERIAL_RING 2
#define MOK_DEBUG_FUSED_WGRAD_GATHER 4
#define MOK_DEBUG_SINGLE_CTA_WGRAD 8
#define MOK_DEBUG_SINGLE_CTA_ROWS 16
#define MOK_DEBUG_SINGLE_CTA_RING 32
#define MOK_DEBUG_GATHER_X_RING 64
#define MOK_DEBUG_NO_OVERLAP 128

/* MXFP8 tensor: E4M3 codes plus E8M0 scales (see mok_mxfp8_quantize). */
typedef struct {
  const uint8_t* q;     /* (device) E4M3 codes, the shape of the source */
  const uint8_t* scale; /* (device) E8M0 scales, one per 32-element block */
} mok_mx;

/* Byte offsets of the schedule arrays inside the workspace, for inspection
 * (all int32, device).  Capacities are host-known upper bounds; the used
 * lengths are on the device (header words). */
typedef struct {
  size_t header;          /* int32[16]: [0] error bits, [1] padded rows used,
                             [2] M-tiles used */
  size_t counts;          /* [E]    rows routed to each expert */
  size_t offsets;         /* [E+1]  exclusive scan of counts */
  size_t padded_offsets;  /* [E+1]  exclusive scan of ceil(counts/128)*128 */
  size_t perm;            /* [R]    sorted row r -> flat index f */
  size_t inv_perm;        /* [R]    f -> r */
  size_t pad_perm;        /* [pad_capacity] padded row -> f, or -1 */
  size_t pad_inv;         /* [R]    f -> padded row */
  size_t tile_expert;     /* [tile_capacity] expert of each 128-row tile */
  int64_t pad_capacity;   /* rows: (R + E*127) rounded down to 128 */
  int64_t tile_capacity;  /* pad_capacity / 128 */
} mok_layout;

/* Bytes of device workspace a layer of this shape/config/precision needs. */
size_t mok_workspace_size(const mok_shape* shape, const mok_config* cfg, mok_precision prec);

/* Bytes of the forward context (saved activations) forward writes and
 * backward reads: [h|u] for every padded routed row, bf16. */
size_t mok_ctx_size(const mok_shape* shape, const mok_config* cfg, mok_precision prec);

/* Offsets of the schedule arrays in the workspace (host-only, no device work). */
mok_status mok_workspace_layout(const mok_shape* shape, const mok_config* cfg, mok_precision prec,
                                mok_layout* out);

/*
 * Build the schedule: the one table that serves forward dispatch and
 * combine and the backward's reverse combine and reverse dispatch ([MTP]
 * communication-direction paragraph), on the device with no host readback
 * ([MTP] ring-token-buffer paragraph: the CPU stays out of the loop).
 *
 *   topk_idx  (device) int32 [T, k]: expert of each routed row.
 * Computes the expert histogram, its exclusive scan, the stable
 * permutation (key = expert, ties by ascending f), the 128-row padded
 * offsets, the tile table and the inverse permutations, in the workspace.
 * An id outside [0, E) records MOK_ERR_BAD_INDEX; that row is routed
 * nowhere and contributes zero.  Clears the workspace error word first.
 */
mok_status mok_build_schedule(const mok_shape* shape, const mok_config* cfg, void* ws, size_t ws_bytes,
                              const int32_t* topk_idx, void* stream);

/*
 * Forward ([MoK] "Use the functional API": forward(config, workspace,
 * schedule, ...) -> (out, fwd_ctx)).  Needs the schedule of the same routing.
 *
 *   x       (device) bf16 [T, H]
 *   scores  (device) f32  [T, k]   router scores s[t, j] (combine weights)
 *   W1, W3  (device) gate / up projections [E, H, I]:
 *             MOK_BF16:  const bf16*
 *             MOK_MXFP8: const mok_mx* (host struct), quantised along H
 *                        (block_axis 0 of each [H, I] matrix)
 *   W2      (device) down projection [E, I, H]:
 *             MOK_BF16:  const bf16*
 *             MOK_MXFP8: const mok_mx*, quantised along I (block_axis 0)
 *   out     (device) bf16 [T, H]
 *           out[t] = sum_{j=0..k-1} s[t,j] * y[t*k+j], summed in f32 in
 *           increasing j and rounded once, where
 *           y = (silu(x W1_e) * (x W3_e)) W2_e for e = topk_idx[t, j].
 *   ctx     (device) mok_ctx_size() bytes, written; read by mok_backward.
 * Deterministic: bitwise-identical results for identical inputs.
 */
mok_status mok_forward(const mok_shape* shape, const mok_config* cfg, mok_precision prec, void* ws,
                       size_t ws_bytes, const void* x, const float* scores, const void* W1, const void* W3,
                       const void* W2, void* out, void* ctx, void* stream);

/*
 * The schedule and the forward in one persistent launch ([MTP]: the layer
 * as a single kernel; the ring-token-buffer paragraph).  Same inputs as
 * mok_build_schedule followed by mok_forward (weights as for mok_forward
 * in the given precision), same results bitwise -- the schedule arrays in
 * the workspace (so mok_backward can follow), out and ctx.  The launch's
 * work items, taken in order from a device counter, are: a histogram per
 * 1,024 routed rows, the scan, the placement per 1,024 routed rows (MXFP8:
 * also the placed rows' x scales, tiled for GEMM1) and the ring's GEMM1 /
 * GEMM2 tiles; each waits (bounded) only on items before it.  A CTA that
 * draws past the last item combines tokens, taken from a second counter,
 * once every GEMM2 row is stored.  MXFP8: what does not depend on the
 * routing -- x quantised along H, the weights' scales tiled -- runs as
 * four small launches ahead of the persistent one.
 * Clears the workspace error word first; an id outside [0, E) records
 * MOK_ERR_BAD_INDEX as in mok_build_schedule.
 */
mok_status mok_forward_fused(const mok_shape* shape, const mok_config* cfg, mok_precision prec, void* ws,
                             size_t ws_bytes, const int32_t* topk_idx, const void* x, const float* scores,
                             const void* W1, const void* W3, const void* W2, void* out, void* ctx, void* stream);

/*
 * Backward ([MoK] "Use the functional API": backward(config, workspace,
 * schedule, fwd_ctx, ...) -> grads).  The router-score gradient is taken in
 * the SwiGLU-backward epilogue ([MTP], the paragraph after "Three design
 * decisions that matter": router gradients fused into the SwiGLU backward).
 *
 *   ctx      (device) the forward's context, same routing and inputs
 *   x, scores, W1, W3, W2   as for mok_forward (the same x: a BF16 backward
 *            reuses the token-sorted copy of x its forward left in the
 *            workspace), except that in MXFP8 mode
 *            the weights are passed in the orientation the backward GEMMs
 *            contract over: W1, W3 quantised along I (block_axis 1), W2
 *            quantised along H (block_axis 1).
 *   dout     (device) bf16 [T, H]   dL/d out
 *   dX       (device) bf16 [T, H]   dL/dx
 *   dW1,dW3  (device) bf16 [E, H, I]; dW2 (device) bf16 [E, I, H].
 *            Experts with no routed rows get exact zeros.
 *   dscores  (device) f32 [T, k]    dL/ds[t, j] = <dout_t, y_(t,j)>
 * Deterministic: fixed reduction orders, no floating-point atomics.
 */
mok_status mok_backward(const mok_shape* shape, const mok_config* cfg, mok_precision prec, void* ws,
                        size_t ws_bytes, const void* ctx, const void* x, const float* scores, const void* W1,
                        const void* W3, const void* W2, const void* dout, void* dX, void* dW1, void* dW3,
                        void* dW2, float* dscores, void* stream);

/*
 * MXFP8 block quantisation ([MoK] "Core concepts", MXFP8 row: weights are
 * pre-quantised with ops.mxfp8_quantize before the kernel).
 *
 *   src    (device) bf16 [batch, rows, cols]
 *   block_axis 0: blocks of 32 consecutive rows in each column
 *                 (rows % 32 == 0); scale is [batch, rows/32, cols]
 *              1: blocks of 32 consecutive columns in each row
 *                 (cols % 32 == 0); scale is [batch, rows, cols/32]
 *   q      (device) u8 [batch, rows, cols] E4M3 codes
 *   scale  (device) u8 E8M0 codes (biased exponent, bias 127)
 * Rule (OCP MX v1.0): X = floor(log2(amax)) - 8 clamped to [-127, 127]
 * (X = -127 for an all-zero block); q = RNE(v / 2^X) on the E4M3 grid,
 * saturating at +-448; a negative value that rounds to zero is 0x80.
 */
mok_status mok_mxfp8_quantize(const void* src, int32_t batch, int32_t rows, int32_t cols, int32_t block_axis,
                              uint8_t* q, uint8_t* scale, void* stream);

/*
 * Dispatch as a standalone copy: xg[r] = x[token of padded row r] for every
 * padded row of the schedule (zeros for padding rows).  The layer itself
 * fuses this gather into its GEMMs' loads; this entry point exposes it on
 * its own ([MTP] communication-direction paragraph: pull-based dispatch).
 *   x   (device) bf16 [T, H];  xg (device) bf16 [pad_capacity, H]
 */
mok_status mok_gather_rows(const mok_shape* shape, const mok_config* cfg, const void* ws, size_t ws_bytes,
                           const void* x, void* xg, void* stream);

/*
 * The tensor-core GEMM the layer's grouped GEMMs are built on, on one dense
 * problem (a diagnostic of the core: tile pipeline, operand layouts).
 *   C (device) f32 [M, N] = A * B
 *   A (device) bf16: a_mn_major = 0 -> [M, K] row-major; 1 -> [K, M]
 *   B (device) bf16: b_mn_major = 0 -> [N, K] row-major; 1 -> [K, N]
 *   scratch (device) >= 256 bytes, caller-owned (tile counter, error word)
 * M % 128 == 0, N % 128 == 0, K % 64 == 0.
 */
mok_status mok_gemm_bf16(int32_t M, int32_t N, int32_t K, const void* A, int32_t a_mn_major, const void* B,
                         int32_t b_mn_major, float* C, void* scratch, void* stream);

/*
 * Phase tracing (a diagnostic for measurement).  While enabled, every call
 * records a pair of CUDA events on its stream around each of its kernel
 * phases; mok_trace_read synchronises on them and returns, per phase, the
 * summed duration in ms and the number of times the phase ran since the
 * last read, then forgets them.  This is the library's only host-side
 * global state; enable it from one thread at a time.  Independently of
 * this, every call opens an NVTX range per phase ("mok fwd gemm", ...) on
 * the calling host thread, around the launches it issues for that phase.
 */
enum {
  MOK_PHASE_SCHEDULE = 0,      /* histogram, scan, placement */
  MOK_PHASE_FWD_GEMM = 1,      /* ring kernel: GEMM1 + SwiGLU, GEMM2 + scatter */
  MOK_PHASE_FWD_COMBINE = 2,   /* weighted combine */
  MOK_PHASE_BWD_DA = 3,        /* dA' GEMM + SwiGLU backward + ds partials */
  MOK_PHASE_BWD_DS = 4,        /* ds reduction */
  MOK_PHASE_BWD_DX = 5,        /* dX GEMM + scatter */
  MOK_PHASE_BWD_DX_COMBINE = 6,/* dX combine */
  MOK_PHASE_BWD_WG13 = 7,      /* dW1 | dW3 grouped GEMM */
  MOK_PHASE_BWD_WG2 = 8,       /* dW2 grouped GEMM */
  MOK_PHASE_QUANT = 9,         /* MXFP8 quantisation of activations */
  MOK_PHASE_BWD_SORT = 10,     /* token-sorted copies of dout and x (dA', weight gradients) */
  MOK_PHASE_ROUTER_FWD = 11,   /* router: logits GEMM, top-k, softmax */
  MOK_PHASE_ROUTER_BWD = 12,   /* router: logit gradient, dWr and dx GEMMs */
  MOK_PHASE_BWD_REPLAY = 13,   /* bounded-memory backward: GEMM1 recomputed, context copied back */
  MOK_PHASE_FWD_FUSED = 14,    /* single-launch forward: schedule, GEMMs, combine */
  MOK_PHASE_FWD_SORT = 15,     /* token-sorted copy of x and the ring's pair table (CTA-pair ring) */
  MOK_NUM_PHASES = 16
};
mok_status mok_trace_enable(int32_t on);
mok_status mok_trace_read(float* ms /* [MOK_NUM_PHASES] */, int32_t* count /* [MOK_NUM_PHASES] */);

/* Number of kernels the library has launched in this process so far. */
int64_t mok_launch_count(void);

/*
 * Build the schedule without any device allocation, into caller-owned
 * buffers.  No counterpart on the pages: this is an addition for callers that
 * cannot allocate device memory themselves -- code whose device memory is all
 * owned by another allocator (a pool carved out once at start-up, as
 * training frameworks do), or code that must not call cudaMalloc because it
 * synchronises the device and stalls every other stream.  Such callers still
 * own their inputs and outputs, but the workspace that mok_build_schedule
 * asks for is one more buffer they cannot create; this entry point needs
 * none.
 *
 * Same computation and same results as mok_build_schedule: bit-identical
 * arrays.  Its only scratch (the per-chunk expert histograms and their
 * scans, 2 * ceil(T*k/1024) * E int32) lives in one static device array of
 * MOK_NOALLOC_SCRATCH_BYTES (1 MiB) built into the library; every GPU that
 * loads the library holds it until the process exits.
 *   - Sizes whose scratch exceeds the array (ceil(T*k/1024) * E > 131072)
 *     return MOK_ERR_UNSUPPORTED before anything is enqueued.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.  The address is cached per device and
 *     context: after a cudaDeviceReset the next call (again the first on a
 *     new context) looks it up anew.
 *   - The kernels use the current device's array, so `stream` must belong to
 *     the current device; a stream of another device returns
 *     MOK_ERR_INVALID_ARG before anything is enqueued.
 *   - All calls share the one array: calls that overlap on the GPU (other
 *     streams, other threads, same device) race and give wrong schedules.
 *     Serialise them.
 *   - The function allocates nothing: no cudaMalloc/cudaFree, no library
 *     routine that allocates.
 *   - MOK_ERR_CUDA means one of this call's own launches failed (each launch
 *     is checked on its own; an earlier error pending in the runtime is not
 *     reported as this call's).
 * Outputs (device, int32, caller-owned): the arrays of mok_layout, with the
 * same lengths; `header` gets [0] error bits (1 = an expert id outside
 * [0, E)), [1] padded rows used, [2] 128-row tiles used.
 */
#define MOK_NOALLOC_SCRATCH_BYTES (1u << 20)
typedef struct {
  int32_t* header;         /* [64] */
  int32_t* counts;         /* [E] */
  int32_t* offsets;        /* [E+1] */
  int32_t* padded_offsets; /* [E+1] */
  int32_t* perm;           /* [R] */
  int32_t* inv_perm;       /* [R] */
  int32_t* pad_perm;       /* [pad_capacity] */
  int32_t* pad_inv;        /* [R] */
  int32_t* tile_expert;    /* [tile_capacity] */
} mok_schedule_buffers;
mok_status mok_build_schedule_noalloc(const mok_shape* shape, const int32_t* topk_idx,
                                      const mok_schedule_buffers* out, void* stream);

/*
 * The block-scaled (MXFP8) tensor-core GEMM the layer's MXFP8 mode is built
 * on, on one dense problem (a diagnostic of the core: E4M3 operands, one
 * E8M0 scale per 32 K-elements, f32 accumulation).
 *   C (device) f32 [M, N] = dequant(A) * dequant(B)
 *   A: a_mn_major = 0: Aq u8 [M, K] + Asf u8 [M, K/32] (quantised with
 *      block_axis 1); a_mn_major = 1: Aq u8 [K, M] + Asf u8 [K/32, M]
 *      (block_axis 0).  B likewise with N: [N, K] + [N, K/32], or
 *      [K, N] + [K/32, N].
 *   scratch (device, caller-owned) >= 256 + M*K/32 + N*K/32 bytes (tile
 *      counter, error word, and both operands' scales re-tiled for the
 *      GEMM's bulk loads).
 * M, N, K multiples of 128.
 */
mok_status mok_gemm_mxfp8(int32_t M, int32_t N, int32_t K, const uint8_t* Aq, const uint8_t* Asf,
                          int32_t a_mn_major, const uint8_t* Bq, const uint8_t* Bsf, int32_t b_mn_major, float* C,
                          void* scratch, size_t scratch_bytes, void* stream);

/*
 * Router on either side of the layer.  The pages take the routing as the
 * schedule's input ("Mixture-of-Kittens (MoK)", "Use the functional API") and
 * compute the router weight gradients from the score gradient of the SwiGLU
 * backward ("Cursor Open-Sources Mixture-of-Kittens (MoK)", the paragraph
 * after "Three design decisions that matter"); these calls supply the plain
 * top-k softmax router around that path:
 *
 *   logits L = x Wr                        (bf16 in, f32 accumulate)
 *   topk_idx[t] = the k largest L[t] + bias (bias selects only; ties go to the
 *                 lower expert; columns in descending key order)
 *   scores[t, j] = softmax over j of L[t, topk_idx[t, j]]   (f32)
 *
 * and, from the layer's dscores (mok_backward):
 *
 *   dL[t, topk_idx[t, j]] = s_j (ds_j - sum_i s_i ds_i), zero elsewhere
 *   dWr = x^T dL  (f32 [H, E]),   dx_router = dL Wr^T  (bf16 [T, H], the
 *   router's share of the input gradient; the caller adds it to dX)
 *
 * Layout: x [T, H] bf16, Wr [H, E] bf16, bias [E] f32 or NULL, topk_idx
 * [T, k] int32, scores and dscores [T, k] f32, logits [T, E] f32 (optional
 * copy out, NULL to skip).  Requires k <= E <= 1024 and the shape rules of
 * mok_forward.  `rws` is a caller-owned device workspace of
 * mok_router_workspace_size bytes (its first word is an error word read by
 * mok_check; each mok_router_forward clears it, as it starts a router step);
 * the backward re-reads nothing of the forward but its outputs.
 * Host errors return before any launch; the calls only enqueue on `stream`.
 */
size_t mok_router_workspace_size(const mok_shape* shape); /* 0 for an invalid shape */
mok_status mok_router_forward(const mok_shape* shape, void* rws, size_t rws_bytes, const void* x, const void* Wr,
                              const float* bias, int32_t* topk_idx, float* scores, float* logits, void* stream);
mok_status mok_router_backward(const mok_shape* shape, void* rws, size_t rws_bytes, const void* x, const void* Wr,
                               const int32_t* topk_idx, const float* scores, const float* dscores, float* dWr,
                               void* dx_router, void* stream);

/* Bytes of workspace mok_build_schedule needs: the schedule's prefix of the
 * full layout (the source side of expert parallelism needs no more).  0 for
 * an invalid shape or config. */
size_t mok_schedule_workspace_size(const mok_shape* shape, const mok_config* cfg);

/*
 * Expert parallelism (EP): the E experts split over G ranks in contiguous
 * blocks, each rank holding its own tokens; one exchange of routed rows each
 * way per pass, all four directions driven by the one schedule ([MTP]
 * communication-direction paragraph; "Results": the layer at EP 64).  The
 * exchange itself is the caller's collective (an all-to-all with uneven
 * splits); these calls are the plan and the source side around it:
 *
 *   forward   source: mok_build_schedule (global expert ids), then
 *             mok_ep_pack_rows -> rows in expert-sorted order, which is
 *             destination-major; exchange the per-expert counts, plan with
 *             mok_ep_plan, send send_rows[g] rows to rank g.
 *             receiver: the ordinary layer calls on its n_recv received rows
 *             with shape (T = n_recv, k = 1, E = its own experts), routing
 *             recv_expert, scores 1.0 -> one output row per received row
 *             (exactly the expert output: a one-term combine with weight 1).
 *             return the rows; source: mok_ep_combine_rows with the scores.
 *   backward  source: mok_ep_pack_rows of dout with the scores; receiver:
 *             mok_backward with those scores -> dX rows, its experts' dW, the
 *             score gradient per row; return the dX rows and score gradients;
 *             source: mok_ep_combine_rows with no scores (dX) and
 *             mok_ep_unsort_scores (dscores).
 * Received rows are ordered by (source rank, source's sorted order), so each
 * expert sees its rows in ascending global flat index when token t of rank g
 * is global token g*T + t: every result is bitwise that of one GPU holding
 * all tokens and experts.
 */

/* First expert of rank g (g = G gives E): rank g owns experts
 * [first(g), first(g+1)), blocks whose sizes differ by at most one.
 * Requires 1 <= G <= E and 0 <= g <= G; -1 otherwise.  Host only. */
int32_t mok_ep_first_expert(int32_t E, int32_t G, int32_t g);

/*
 * The exchange plan of rank `rank` (host only, no device work):
 *   local_counts  (host) int32 [E]: rows this rank routes to each global
 *                 expert (the schedule's counts array)
 *   recv_counts   (host) int32 [G, E_rank]: rows source rank s routes to each
 *                 of this rank's experts (row s = source s's local_counts
 *                 over this rank's block)
 *   send_rows     (host) int64 [G]: rows to send to each rank, in order, from
 *                 the front of the packed rows
 *   recv_rows     (host) int64 [G]: rows arriving from each rank, in order
 *   recv_expert   (host) int32 [recv_capacity] or NULL: local expert id of
 *                 each received row in arrival order (the receiver's routing)
 *   n_recv        (host) total received rows
 * MOK_ERR_UNSUPPORTED if n_recv > recv_capacity (recv_expert given);
 * MOK_ERR_INVALID_ARG for bad sizes, null pointers or negative counts.
 */
mok_status mok_ep_plan(int32_t E, int32_t G, int32_t rank, const int32_t* local_counts, const int32_t* recv_counts,
                       int64_t* send_rows, int64_t* recv_rows, int32_t* recv_expert, int64_t recv_capacity,
                       int64_t* n_recv);

/*
 * Source side of the dispatch (forward) and of the reverse combine
 * (backward): rows[r] = x[perm[r] / k] (bf16 [T*k, H], device) for every
 * routed row r of the schedule in `ws`, in its expert-sorted order; rows
 * past the routed ones (ids outside [0, E)) are not written.  With
 * row_scores (device f32 [T*k]) also row_scores[r] = scores[perm[r]].
 * ws needs mok_schedule_workspace_size bytes.
 */
mok_status mok_ep_pack_rows(const mok_shape* shape, const mok_config* cfg, const void* ws, size_t ws_bytes,
                            const void* x, const float* scores, void* rows, float* row_scores, void* stream);

/*
 * Source side of the combine (forward) and reverse dispatch (backward):
 * out[t] = sum_j w[t,j] * rows[inv_perm[t*k + j]] in f32, increasing j,
 * rounded once to bf16, with w = scores (device f32 [T, k]) or 1 when scores
 * is NULL; a row routed nowhere adds nothing.  rows (device bf16 [T*k, H]) in
 * the schedule's sorted order (the returned expert outputs or dX rows).
 */
mok_status mok_ep_combine_rows(const mok_shape* shape, const mok_config* cfg, const void* ws, size_t ws_bytes,
                               const void* rows, const float* scores, void* out, void* stream);

/* out[f] = row_vals[inv_perm[f]] (device f32 [T*k] -> [T, k]), 0 for a row
 * routed nowhere: the returned per-row score gradients back in token order. */
mok_status mok_ep_unsort_scores(const mok_shape* shape, const mok_config* cfg, const void* ws, size_t ws_bytes,
                                const float* row_vals, float* out, void* stream);

/* Synchronise `stream`, then return (and clear) the status recorded in the
 * workspace's error word; MOK_OK if none. */
mok_status mok_check(void* ws, void* stream);

/* Number of SMs of the current device (the C in the minibatch floor). */
int32_t mok_device_sm_count(void);

const char* mok_status_string(mok_status s);
const char* mok_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MOK_H_ */

// Top-k softmax router on either side of the layer (the selection is the
// schedule's input; "Mixture-of-Kittens (MoK)", "Use the functional API").
// The logits GEMM and the two backward GEMMs run on the tcgen05 GEMM core
// (GM_DENSE); the kernels here are the small HBM-bound steps around them:
//   pad_weights   Wr [H, E] -> [H, Epad] (zero columns up to a 128 multiple)
//   topk_softmax  per token: the k largest logit + bias keys (ties to the
//                 lower expert, descending key order), softmax over the k
//                 chosen unbiased logits
//   logit_grad    per token: dL[idx_j] = s_j (ds_j - sum_i s_i ds_i), zero
//                 elsewhere, as bf16 rows of the backward GEMMs' operand
//   take_cols     f32 [rows, Epad] -> [rows, E]
// The router gradient reaches the weights through the layer's score
// gradient ("Cursor Open-Sources Mixture-of-Kittens (MoK)", the paragraph
// after "Three design decisions that matter": router weight gradients from
// the SonicMoE-style score gradient in the SwiGLU backward).
#include "mok_internal.cuh"

namespace mok {

namespace {

constexpr int kMaxRouterExperts = 1024;  // keys held in registers: 32 per lane

__global__ void __launch_bounds__(256) pad_weights_kernel(int H, int E, int Epad, const __nv_bfloat16* __restrict__ w,
                                                          __nv_bfloat16* __restrict__ wp) {
  const long n = (long)H * Epad;
  for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < n; i += (long)gridDim.x * blockDim.x) {
    const int h = (int)(i / Epad), e = (int)(i - (long)h * Epad);
    wp[i] = e < E ? w[(long)h * E + e] : __float2bfloat16(0.0f);
  }
}

// (key, expert) pairs ordered by descending key, then ascending expert.
__device__ __forceinline__ bool ranks_before(float ka, int ea, float kb, int eb) {
  return ka > kb || (ka == kb && ea < eb);
}

// One warp per token; lane l holds the keys of experts l, l + 32, ...
__global__ void __launch_bounds__(256) topk_softmax_kernel(int T, int E, int Epad, int k,
                                                           const float* __restrict__ logits,
                                                           const float* __restrict__ bias, int32_t* __restrict__ idx,
                                                           float* __restrict__ scores) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;
  const float* row = logits + (long)t * Epad;
  float key[kMaxRouterExperts / 32];
  const int per_lane = (E + 31) >> 5;
#pragma unroll
  for (int i = 0; i < kMaxRouterExperts / 32; ++i) {
    const int e = lane + 32 * i;
    const float v = (i < per_lane && e < E) ? row[e] + (bias ? bias[e] : 0.0f) : 0.0f;
    key[i] = isnan(v) ? -INFINITY : v;  // a NaN key ranks last
  }
  uint32_t taken = 0;  // bit i: expert lane + 32 i already chosen
  int my_e = -1;       // lane j < k ends with the j-th choice
  float my_l = 0.0f;
  for (int j = 0; j < k; ++j) {
    float bk = 0.0f;
    int be = INT_MAX;
#pragma unroll
    for (int i = 0; i < kMaxRouterExperts / 32; ++i) {
      const int e = lane + 32 * i;
      if (i < per_lane && e < E && !((taken >> i) & 1u) && (be == INT_MAX || ranks_before(key[i], e, bk, be))) {
        bk = key[i];
        be = e;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ok = __shfl_xor_sync(0xffffffffu, bk, o);
      const int oe = __shfl_xor_sync(0xffffffffu, be, o);
      if (oe != INT_MAX && (be == INT_MAX || ranks_before(ok, oe, bk, be))) {
        bk = ok;
        be = oe;
      }
    }
    if (be == INT_MAX) break;  // fewer than k experts (the host rules it out)
    if ((be & 31) == lane) taken |= 1u << (be >> 5);
    if (lane == j) {
      my_e = be;
      my_l = row[be];
    }
  }
  // softmax over the k chosen, unbiased logits (lanes j < k)
  float m = lane < k ? my_l : -INFINITY;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  const float ez = lane < k ? expf(my_l - m) : 0.0f;
  float sum = ez;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  if (lane < k) {
    idx[(long)t * k + lane] = my_e;
    scores[(long)t * k + lane] = ez / sum;
  }
}

// One warp per row of dL [Tpad, Epad] (rows past T are zero).
__global__ void __launch_bounds__(256) logit_grad_kernel(int T, int Tpad, int E, int Epad, int k,
                                                         const int32_t* __restrict__ idx, const float* __restrict__ s,
                                                         const float* __restrict__ ds, __nv_bfloat16* __restrict__ dl) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= Tpad) return;
  __nv_bfloat16* row = dl + (long)t * Epad;
  for (int e = lane; e < Epad; e += 32) row[e] = __float2bfloat16(0.0f);
  __syncwarp();
  if (t >= T) return;
  const float sj = lane < k ? s[(long)t * k + lane] : 0.0f;
  const float dsj = lane < k ? ds[(long)t * k + lane] : 0.0f;
  float dot = sj * dsj;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
  if (lane < k) {
    const int e = idx[(long)t * k + lane];
    if (e >= 0 && e < E) row[e] = __float2bfloat16(sj * (dsj - dot));
  }
}

__global__ void __launch_bounds__(256) take_cols_kernel(int rows, int E, int Epad, const float* __restrict__ src,
                                                        float* __restrict__ dst) {
  const long n = (long)rows * E;
  for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < n; i += (long)gridDim.x * blockDim.x) {
    const int r = (int)(i / E), e = (int)(i - (long)r * E);
    dst[i] = src[(long)r * Epad + e];
  }
}

int elementwise_grid(long items) {
  long blocks = (items + 255) / 256;
  const long cap = (long)device_sm_count() * 16;
  if (blocks > cap) blocks = cap;
  return (int)(blocks < 1 ? 1 : blocks);
}

}  // namespace

cudaError_t launch_router_pad_weights(int H, int E, int Epad, const __nv_bfloat16* w, __nv_bfloat16* wp,
                                      cudaStream_t st) {
  pad_weights_kernel<<<elementwise_grid((long)H * Epad), 256, 0, st>>>(H, E, Epad, w, wp);
  return cudaGetLastError();
}

cudaError_t launch_router_topk(int T, int E, int Epad, int k, const float* logits, const float* bias, int32_t* idx,
                               float* scores, cudaStream_t st) {
  if (E > kMaxRouterExperts || k > 32) return cudaErrorInvalidValue;
  topk_softmax_kernel<<<(T + 7) / 8, 256, 0, st>>>(T, E, Epad, k, logits, bias, idx, scores);
  return cudaGetLastError();
}

cudaError_t launch_router_logit_grad(int T, int Tpad, int E, int Epad, int k, const int32_t* idx, const float* s,
                                     const float* ds, __nv_bfloat16* dl, cudaStream_t st) {
  logit_grad_kernel<<<(Tpad + 7) / 8, 256, 0, st>>>(T, Tpad, E, Epad, k, idx, s, ds, dl);
  return cudaGetLastError();
}

cudaError_t launch_router_take_cols(int rows, int E, int Epad, const float* src, float* dst, cudaStream_t st) {
  take_cols_kernel<<<elementwise_grid((long)rows * E), 256, 0, st>>>(rows, E, Epad, src, dst);
  return cudaGetLastError();
}

}  // namespace mok

// route.cu -- router scores and top-k gating
// ("Making Every Verified Token Count: Adaptive Verification for MoE
// Speculative Decoding", Sec. 2.2, eq. (4): s = W_g h, E(h) = TopK(s, k), the
// selected scores normalised by softmax or sigmoid).
//
//   router_scores_kernel  one CTA per (expert, group of 8 tokens); its warps
//                         split d in 256-column chunks, each lane takes 8
//                         contiguous elements (16-byte loads of bf16, 2 x 16
//                         bytes of fp32); the warps' partial sums are added in
//                         a fixed order, so the fp32 logits are reproducible
//                         run to run.
//   topk_gate_kernel      one warp per token (topk_gate_warp, route_plan.cuh).
//   route_plan_kernel     both of the above and the union plan in one launch
//                         (the last CTA to finish its scores does the rest);
//                         for moe_verify_pass with E4M3 weights, one more CTA
//                         per 8 tokens writes their fp16 rows for the expert
//                         kernels (act_scale.cuh).
#include <math.h>

#include <type_traits>

#include "act_scale.cuh"
#include "kernels.h"
#include "moe_common.cuh"
#include "route_plan.cuh"

namespace moe {

namespace {

constexpr int TOKENS_PER_CTA = 8;

// One CTA per (expert, group of 8 tokens), one warp per 256-column chunk of
// d (8 to 16 warps; larger d loops), so a lane issues its loads together and
// the whole dot product costs one or two L2 round trips.
constexpr int ROUTER_MAX_WARPS = 16;

// 8 consecutive elements kept as loaded (bf16: one 16-byte word; fp32: two)
// and widened to fp32 only at use, so a thread can hold its 8 tokens' pieces
// in few registers and two CTAs fit on an SM.
struct Raw8Bf16 {
  uint4 v;
  __device__ __forceinline__ void load(const __nv_bfloat16 *p) {
    v = __ldg(reinterpret_cast<const uint4 *>(p));
  }
  __device__ __forceinline__ float at(int i) const {
    const uint32_t w = i < 2 ? v.x : i < 4 ? v.y : i < 6 ? v.z : v.w;
    return (i & 1) ? __uint_as_float(w & 0xFFFF0000u) : __uint_as_float(w << 16);
  }
};
struct Raw8F32 {
  float4 a, b;
  __device__ __forceinline__ void load(const float *p) {
    a = __ldg(reinterpret_cast<const float4 *>(p));
    b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
  }
  __device__ __forceinline__ float at(int i) const {
    const float4 &q = i < 4 ? a : b;
    const int j = i & 3;
    return j == 0 ? q.x : j == 1 ? q.y : j == 2 ? q.z : q.w;
  }
};
template <typename T> struct Raw8;
template <> struct Raw8<__nv_bfloat16> { using type = Raw8Bf16; };
template <> struct Raw8<float> { using type = Raw8F32; };

template <typename T>
__device__ __forceinline__ void router_scores_cta(const T *__restrict__ wg,
                                                  const T *__restrict__ h, int n, int d,
                                                  int n_experts, float *__restrict__ logits) {
  using R = typename Raw8<T>::type;
  __shared__ float part[ROUTER_MAX_WARPS][TOKENS_PER_CTA];
  const int e = blockIdx.x;
  const int t0 = blockIdx.y * TOKENS_PER_CTA;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_warps = blockDim.x >> 5;
  const int nt = min(TOKENS_PER_CTA, n - t0);
  float acc[TOKENS_PER_CTA];
#pragma unroll
  for (int t = 0; t < TOKENS_PER_CTA; ++t) acc[t] = 0.f;
#pragma unroll 2
  for (int c = threadIdx.x * 8; c < d; c += blockDim.x * 8) {
    R wv;
    wv.load(wg + int64_t(e) * d + c);
    R hv[TOKENS_PER_CTA];
#pragma unroll
    for (int t = 0; t < TOKENS_PER_CTA; ++t)
      if (t < nt) hv[t].load(h + int64_t(t0 + t) * d + c);
#pragma unroll
    for (int t = 0; t < TOKENS_PER_CTA; ++t)
      if (t < nt) {
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[t] = fmaf(wv.at(i), hv[t].at(i), acc[t]);
      }
  }
#pragma unroll
  for (int t = 0; t < TOKENS_PER_CTA; ++t) {
    float v = acc[t];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) part[warp][t] = v;
  }
  __syncthreads();
  if (threadIdx.x < nt) {
    float s = 0.f;
    for (int w = 0; w < n_warps; ++w) s += part[w][threadIdx.x];
    logits[int64_t(t0 + threadIdx.x) * n_experts + e] = s;
  }
}

template <typename T>
__global__ void __launch_bounds__(ROUTER_MAX_WARPS * 32, 2) router_scores_kernel(const T *__restrict__ wg,
                                                             const T *__restrict__ h, int n, int d,
                                                             int n_experts,
                                                             float *__restrict__ logits) {
  router_scores_cta(wg, h, n, d, n_experts, logits);
}

__global__ void __launch_bounds__(256) topk_gate_kernel(const float *__restrict__ logits, int n,
                                                        int n_experts, int k, int gate,
                                                        int32_t *__restrict__ ids,
                                                        float *__restrict__ w) {
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= n) return;
  topk_gate_warp(logits + int64_t(t) * n_experts, n_experts, k, gate, ids + int64_t(t) * k,
                 w + int64_t(t) * k);
}

// Router scores, top-k + gate and the union plan in one launch.  Every CTA
// computes its (expert, 8-token) scores as router_scores_kernel does, then
// takes a ticket of its 8-token group; the CTA that takes the group's last
// ticket (so the group's scores are all written) runs the top-k of the
// group's tokens, one warp a token, and takes a ticket of the kernel; the
// CTA that takes the kernel's last ticket (so every token is ranked) runs
// union_plan_block (BUDGET: the budgeted plan).  Each counter is reset by
// the CTA that took its last ticket, for the next call.  (One CTA ranking
// all n tokens, 8 warps, took ~20 us of a 64-token pass.)  With `A.acts` set, the grid has one more CTA
// column (blockIdx.x == n_experts): it writes the fp16 rows of its 8 tokens
// (act_scale_block) and counts them in *A.acts with release semantics, for
// the E4M3 expert kernel that starts before this kernel ends.  It takes no
// ticket: the plan does not wait for it.
template <typename T, bool BUDGET>
__global__ void __launch_bounds__(ROUTER_MAX_WARPS * 32, 2) route_plan_kernel(
    const T *__restrict__ wg, const T *__restrict__ h, int n, int d, int n_experts, int k,
    int gate, int n_shared, int64_t expert_bytes, float *logits, int32_t *ids, float *w,
    int32_t *hist, int32_t *uniq, int32_t *n_uniq, int32_t *offs, int32_t *perm,
    int64_t *union_bytes, int budget, float *w_kept, int32_t *routed_u, int32_t *err,
    unsigned int *counter, unsigned int *group_counter, unsigned int *ready, ActScaleOut A) {
  pdl_trigger();  // the expert kernel behind this one may launch (it waits for the plan)
  if (blockIdx.x < unsigned(n_experts)) {
    router_scores_cta(wg, h, n, d, n_experts, logits);
  } else if constexpr (std::is_same<T, __nv_bfloat16>::value) {
    const int t0 = blockIdx.y * TOKENS_PER_CTA;
    act_scale_block(h, d, t0, min(TOKENS_PER_CTA, n - t0), A.h16, A.hshift);
    __syncthreads();
    if (threadIdx.x == 0) {
      // the rows are read by bulk copies (async proxy) of another kernel
      fence_proxy_async_global();
      __threadfence();
      atomicAdd(A.acts, 1u);
    }
    return;
  }
  __shared__ int s_last;
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();  // this CTA's scores before its ticket
    const unsigned int ticket = atomicAdd(group_counter + blockIdx.y, 1u);
    s_last = ticket == unsigned(n_experts) - 1;  // the group's router CTAs
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  {
    // the group's tokens, one warp each (a router CTA has at least 8 warps)
    const int warp = threadIdx.x >> 5;
    const int t = blockIdx.y * TOKENS_PER_CTA + warp;
    if (warp < TOKENS_PER_CTA && t < n)
      topk_gate_warp(logits + int64_t(t) * n_experts, n_experts, k, gate, ids + int64_t(t) * k,
                     w + int64_t(t) * k);
  }
  __syncthreads();
  if (gridDim.y > 1) {
    // more than one group: the last group to be ranked builds the plan (one
    // group needs no second ticket: that CTA is the last)
    if (threadIdx.x == 0) {
      group_counter[blockIdx.y] = 0u;
      __threadfence();  // this group's ids and weights before its ticket
      const unsigned int ticket = atomicAdd(counter, 1u);
      s_last = ticket == gridDim.y - 1;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
  } else if (threadIdx.x == 0) {
    group_counter[0] = 0u;
  }
  __shared__ PlanSmem S;
  if constexpr (BUDGET) {
    __shared__ BudgetSmem B;
    union_plan_block<true>(S, &B, ids, w, n * k, n_experts, n_shared, expert_bytes, budget, hist,
                           uniq, n_uniq, offs, perm, union_bytes, w_kept, routed_u, err);
  } else {
    union_plan_block<false>(S, nullptr, ids, nullptr, n * k, n_experts, n_shared, expert_bytes,
                            0, hist, uniq, n_uniq, offs, perm, union_bytes, nullptr, nullptr,
                            err);
  }
  __syncthreads();  // the whole plan is written
  if (threadIdx.x == 0) {
    *counter = 0u;
    if (ready) {
      __threadfence();
      st_release_gpu(ready, 1u);
    }
  }
}

// Warps per router CTA: one per 256 columns of d, at least 8 (the fused
// kernel's last CTA gives one thread per expert to the union plan) and at
// most 16.  Both router kernels use the same count, so they add the same
// partial sums in the same order and produce identical scores.
int router_warps(int d) {
  const int w = (d + 255) / 256;
  return w < 8 ? 8 : w > ROUTER_MAX_WARPS ? ROUTER_MAX_WARPS : w;
}

}  // namespace

cudaError_t launch_router_scores(bool bf16, const void *router_w, const void *h, int n, int d,
                                 int n_experts, float *logits, cudaStream_t stream) {
  dim3 grid(n_experts, (n + TOKENS_PER_CTA - 1) / TOKENS_PER_CTA);
  const int warps = router_warps(d);
  if (bf16)
    router_scores_kernel<__nv_bfloat16><<<grid, warps * 32, 0, stream>>>(
        static_cast<const __nv_bfloat16 *>(router_w), static_cast<const __nv_bfloat16 *>(h), n, d,
        n_experts, logits);
  else
    router_scores_kernel<float><<<grid, warps * 32, 0, stream>>>(
        static_cast<const float *>(router_w), static_cast<const float *>(h), n, d, n_experts,
        logits);
  return cudaGetLastError();
}

cudaError_t launch_route_plan(bool bf16, const void *router_w, const void *h, int n, int d,
                              int n_experts, int k, int gate, int n_shared, int64_t expert_bytes,
                              float *logits, int32_t *ids, float *w, int32_t *hist, int32_t *uniq,
                              int32_t *n_uniq, int32_t *offs, int32_t *perm, int64_t *union_bytes,
                              int budget, float *w_kept, int32_t *routed_u, int32_t *err,
                              unsigned int *counter, unsigned int *group_counter,
                              unsigned int *ready, const ActScaleOut &S, cudaStream_t stream) {
  // E4M3 rows are written only beside bf16 activations (the only kind E4M3 weights take)
  const bool scale = S.acts != nullptr && bf16;
  dim3 grid(n_experts + (scale ? 1 : 0), (n + TOKENS_PER_CTA - 1) / TOKENS_PER_CTA);
  const int threads = router_warps(d) * 32;
  const __nv_bfloat16 *wb = static_cast<const __nv_bfloat16 *>(router_w);
  const __nv_bfloat16 *hb = static_cast<const __nv_bfloat16 *>(h);
  const float *wf = static_cast<const float *>(router_w);
  const float *hf = static_cast<const float *>(h);
  ActScaleOut Sx = S;
  if (!scale) Sx.acts = nullptr;
#define MOE_ROUTE_PLAN_ARGS                                                                  \
  n, d, n_experts, k, gate, n_shared, expert_bytes, logits, ids, w, hist, uniq, n_uniq, offs, \
      perm, union_bytes, budget, w_kept, routed_u, err, counter, group_counter, ready, Sx
  if (budget < 0) {
    if (bf16)
      route_plan_kernel<__nv_bfloat16, false><<<grid, threads, 0, stream>>>(wb, hb,
                                                                           MOE_ROUTE_PLAN_ARGS);
    else
      route_plan_kernel<float, false><<<grid, threads, 0, stream>>>(wf, hf, MOE_ROUTE_PLAN_ARGS);
  } else {
    if (bf16)
      route_plan_kernel<__nv_bfloat16, true><<<grid, threads, 0, stream>>>(wb, hb,
                                                                          MOE_ROUTE_PLAN_ARGS);
    else
      route_plan_kernel<float, true><<<grid, threads, 0, stream>>>(wf, hf, MOE_ROUTE_PLAN_ARGS);
  }
#undef MOE_ROUTE_PLAN_ARGS
  return cudaGetLastError();
}

cudaError_t launch_topk_gate(const float *logits, int n, int n_experts, int k, int gate,
                             int32_t *ids, float *w, cudaStream_t stream) {
  topk_gate_kernel<<<(n + 7) / 8, 256, 0, stream>>>(logits, n, n_experts, k, gate, ids, w);
  return cudaGetLastError();
}

}  // namespace moe

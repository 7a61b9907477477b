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
//   topk_gate_kernel      one warp per token; each lane holds up to 8 of the
//                         N <= 256 logits; k rounds of a warp arg-max over
//                         (logit desc, id asc) with xor shuffles pick the
//                         experts in output order; lane j keeps the j-th
//                         selected logit for the gate.
#include <math.h>

#include "kernels.h"
#include "moe_common.cuh"

namespace moe {

namespace {

constexpr int TOKENS_PER_CTA = 8;

__device__ __forceinline__ void load8(const float *p, float (&v)[8]) {
  const float4 a = __ldg(reinterpret_cast<const float4 *>(p));
  const float4 b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

__device__ __forceinline__ void load8(const __nv_bfloat16 *p, float (&v)[8]) {
  const uint4 a = __ldg(reinterpret_cast<const uint4 *>(p));
  const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// One CTA per (expert, group of 8 tokens), one warp per 256-column chunk of
// d (up to 16 warps; larger d loops), so a lane issues its loads together and
// the whole dot product costs one or two L2 round trips.
constexpr int ROUTER_MAX_WARPS = 16;

template <typename T>
__global__ void __launch_bounds__(ROUTER_MAX_WARPS * 32) router_scores_kernel(const T *__restrict__ wg,
                                                             const T *__restrict__ h, int n, int d,
                                                             int n_experts,
                                                             float *__restrict__ logits) {
  __shared__ float part[ROUTER_MAX_WARPS][TOKENS_PER_CTA];
  const int e = blockIdx.x;
  const int t0 = blockIdx.y * TOKENS_PER_CTA;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_warps = blockDim.x >> 5;
  const int nt = min(TOKENS_PER_CTA, n - t0);
  float acc[TOKENS_PER_CTA];
#pragma unroll
  for (int t = 0; t < TOKENS_PER_CTA; ++t) acc[t] = 0.f;
  for (int c = threadIdx.x * 8; c < d; c += blockDim.x * 8) {
    float wv[8];
    load8(wg + int64_t(e) * d + c, wv);
    float hv[TOKENS_PER_CTA][8];
#pragma unroll
    for (int t = 0; t < TOKENS_PER_CTA; ++t)
      if (t < nt) load8(h + int64_t(t0 + t) * d + c, hv[t]);
#pragma unroll
    for (int t = 0; t < TOKENS_PER_CTA; ++t)
      if (t < nt) {
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[t] = fmaf(wv[i], hv[t][i], acc[t]);
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

// (v, id) beats (bv, bid): larger logit, or equal logit and lower id.
__device__ __forceinline__ bool beats(float v, int id, float bv, int bid) {
  return v > bv || (v == bv && id < bid);
}

constexpr int MAX_PER_LANE = 8;  // N <= 256

__global__ void __launch_bounds__(256) topk_gate_kernel(const float *__restrict__ logits, int n,
                                                        int n_experts, int k, int gate,
                                                        int32_t *__restrict__ ids,
                                                        float *__restrict__ w) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + warp;
  if (t >= n) return;
  const float *z = logits + int64_t(t) * n_experts;
  float v[MAX_PER_LANE];
  bool taken[MAX_PER_LANE];
#pragma unroll
  for (int i = 0; i < MAX_PER_LANE; ++i) {
    const int e = lane + 32 * i;
    v[i] = e < n_experts ? z[e] : -INFINITY;
    taken[i] = e >= n_experts;
  }
  float my_sel = -INFINITY;  // lane j < k: logit of the j-th selected expert
  for (int j = 0; j < k; ++j) {
    float bv = -INFINITY;
    int bid = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < MAX_PER_LANE; ++i)
      if (!taken[i] && beats(v[i], lane + 32 * i, bv, bid)) {
        bv = v[i];
        bid = lane + 32 * i;
      }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oid = __shfl_xor_sync(0xffffffffu, bid, o);
      if (beats(ov, oid, bv, bid)) {
        bv = ov;
        bid = oid;
      }
    }
    if ((bid & 31) == lane) {
#pragma unroll
      for (int i = 0; i < MAX_PER_LANE; ++i)
        if (i == (bid >> 5)) taken[i] = true;
    }
    if (lane == j) my_sel = bv;
    if (lane == 0) ids[int64_t(t) * k + j] = bid;
  }
  // gate weights
  const bool mine = lane < k;
  float num = 0.f, den = 0.f;
  if (gate == MOE_GATE_SOFTMAX) {
    float zmax = -INFINITY;
#pragma unroll
    for (int i = 0; i < MAX_PER_LANE; ++i)
      if (lane + 32 * i < n_experts) zmax = fmaxf(zmax, v[i]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) zmax = fmaxf(zmax, __shfl_xor_sync(0xffffffffu, zmax, o));
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < MAX_PER_LANE; ++i)
      if (lane + 32 * i < n_experts) s += expf(v[i] - zmax);
    den = s;
    num = mine ? expf(my_sel - zmax) : 0.f;
  } else if (gate == MOE_GATE_SOFTMAX_RENORM) {
    const float zmax = __shfl_sync(0xffffffffu, my_sel, 0);  // the largest selected
    num = mine ? expf(my_sel - zmax) : 0.f;
    den = num;
  } else {
    num = mine ? 1.f / (1.f + expf(-my_sel)) : 0.f;
    den = num;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
  if (mine) w[int64_t(t) * k + lane] = num / den;
}

}  // namespace

cudaError_t launch_router_scores(bool bf16, const void *router_w, const void *h, int n, int d,
                                 int n_experts, float *logits, cudaStream_t stream) {
  dim3 grid(n_experts, (n + TOKENS_PER_CTA - 1) / TOKENS_PER_CTA);
  int warps = (d + 255) / 256;
  warps = warps < 1 ? 1 : warps > ROUTER_MAX_WARPS ? ROUTER_MAX_WARPS : warps;
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

cudaError_t launch_topk_gate(const float *logits, int n, int n_experts, int k, int gate,
                             int32_t *ids, float *w, cudaStream_t stream) {
  topk_gate_kernel<<<(n + 7) / 8, 256, 0, stream>>>(logits, n, n_experts, k, gate, ids, w);
  return cudaGetLastError();
}

}  // namespace moe

// route_plan.cuh -- device-side building blocks of routing and planning,
// shared by the stand-alone kernels (route.cu, plan.cu) and the fused
// route + top-k + plan kernel (route.cu).  Internal to the library.
#pragma once

#include <math.h>

#include "moe_common.cuh"

namespace moe {

constexpr int TOPK_MAX_PER_LANE = 8;  // N <= 256 scores per token, 8 per lane
constexpr int PLAN_MAX_SLOTS = 64 * 32;

// (v, id) beats (bv, bid): larger score, or equal score and lower id.
__device__ __forceinline__ bool topk_beats(float v, int id, float bv, int bid) {
  return v > bv || (v == bv && id < bid);
}

// One warp: top-k of token t's scores z[0..N) (largest first, equal scores
// by lower id: "Making Every Verified Token Count", Sec. 2.2, eq. (4)) and
// the gate weights of the selected experts.  k rounds of a warp arg-max
// with xor shuffles; lane j keeps the j-th selected score for the gate.
__device__ __forceinline__ void topk_gate_warp(const float *z, int n_experts, int k, int gate,
                                               int32_t *ids_t, float *w_t) {
  const int lane = threadIdx.x & 31;
  float v[TOPK_MAX_PER_LANE];
  bool taken[TOPK_MAX_PER_LANE];
#pragma unroll
  for (int i = 0; i < TOPK_MAX_PER_LANE; ++i) {
    const int e = lane + 32 * i;
    v[i] = e < n_experts ? __ldcg(z + e) : -INFINITY;  // L2: other CTAs may have written z
    taken[i] = e >= n_experts;
  }
  float my_sel = -INFINITY;  // lane j < k: score of the j-th selected expert
  for (int j = 0; j < k; ++j) {
    float bv = -INFINITY;
    int bid = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < TOPK_MAX_PER_LANE; ++i)
      if (!taken[i] && topk_beats(v[i], lane + 32 * i, bv, bid)) {
        bv = v[i];
        bid = lane + 32 * i;
      }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oid = __shfl_xor_sync(0xffffffffu, bid, o);
      if (topk_beats(ov, oid, bv, bid)) {
        bv = ov;
        bid = oid;
      }
    }
    if ((bid & 31) == lane) {
#pragma unroll
      for (int i = 0; i < TOPK_MAX_PER_LANE; ++i)
        if (i == (bid >> 5)) taken[i] = true;
    }
    if (lane == j) my_sel = bv;
    if (lane == 0) ids_t[j] = bid;
  }
  // gate weights
  const bool mine = lane < k;
  float num = 0.f, den = 0.f;
  if (gate == MOE_GATE_SOFTMAX) {
    float zmax = -INFINITY;
#pragma unroll
    for (int i = 0; i < TOPK_MAX_PER_LANE; ++i)
      if (lane + 32 * i < n_experts) zmax = fmaxf(zmax, v[i]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) zmax = fmaxf(zmax, __shfl_xor_sync(0xffffffffu, zmax, o));
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < TOPK_MAX_PER_LANE; ++i)
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
  if (mine) w_t[lane] = num / den;
}

// Shared memory of union_plan_block.
struct PlanSmem {
  int32_t hist[256];
  int32_t offs[256];
  int32_t ids[PLAN_MAX_SLOTS];
  int32_t warp_cnt[8];
  int32_t warp_sum[8];
};

// The whole block (blockDim.x >= 256, a multiple of 32): the expert union of
// the n_slots routed ids and the grouping of the slots by expert
// ("Less Experts, Faster Decoding", eq. (1); "Making Every Verified Token
// Count", eq. (5); "The Limits of Speculation", App. A.4.1, eq. (A2)):
//   1. histogram with shared-memory atomics;
//   2. the used experts compacted in ascending order: warp w ballots experts
//      32w..32w+31, __popc of the ballot below a lane gives the rank inside
//      the warp, a scan over the 8 warp counts gives the warp base;
//   3. exclusive prefix sum of the histogram (warp shuffle scan + warp
//      totals) gives each expert's group offset;
//   4. stable scatter: slot p goes to offs[ids[p]] + (earlier slots with the
//      same id), so slots stay ascending inside a group;
//   5. U and the union bytes (U + n_shared) * expert bytes.
// `ids` may be written by this block just before (after a __syncthreads).
__device__ __forceinline__ void union_plan_block(PlanSmem &S, const int32_t *ids, int n_slots,
                                                 int n_experts, int n_shared, int64_t expert_bytes,
                                                 int32_t *hist, int32_t *uniq, int32_t *n_uniq,
                                                 int32_t *offs, int32_t *perm,
                                                 int64_t *union_bytes, int32_t *err) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid < 256) S.hist[tid] = 0;
  __syncthreads();
  for (int p = tid; p < n_slots; p += blockDim.x) {
    const int e = ids[p];
    const bool ok = e >= 0 && e < n_experts;
    S.ids[p] = ok ? e : -1;
    if (ok) atomicAdd(&S.hist[e], 1);
    else record_error(err, MOE_ERR_DEVICE_INPUT);
  }
  __syncthreads();
  int incl = 0, cnt = 0;
  unsigned used = 0;
  if (tid < 256) {  // warps 0..7: thread e handles expert e
    const int e = tid;
    cnt = e < n_experts ? S.hist[e] : 0;
    used = __ballot_sync(0xffffffffu, cnt > 0);
    incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int x = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += x;
    }
    if (lane == 31) {
      S.warp_cnt[warp] = __popc(used);
      S.warp_sum[warp] = incl;
    }
  }
  __syncthreads();
  if (tid < 256) {
    const int e = tid;
    int rank_base = 0, off_base = 0, U = 0;
    for (int w = 0; w < 8; ++w) {
      if (w < warp) {
        rank_base += S.warp_cnt[w];
        off_base += S.warp_sum[w];
      }
      U += S.warp_cnt[w];
    }
    const int off = off_base + incl - cnt;
    S.offs[e] = off;
    if (e < n_experts) hist[e] = cnt;
    if (cnt > 0) {
      const int r = rank_base + __popc(used & ((1u << lane) - 1u));
      uniq[r] = e;
      offs[r] = off;
    }
    if (tid == 0) {
      int total = 0;
      for (int w = 0; w < 8; ++w) total += S.warp_sum[w];
      offs[U] = total;
      *n_uniq = U;
      *union_bytes = int64_t(U + n_shared) * expert_bytes;
    }
  }
  __syncthreads();
  for (int p = tid; p < n_slots; p += blockDim.x) {
    const int id = S.ids[p];
    if (id < 0) continue;
    int before = 0;
    for (int q = 0; q < p; ++q) before += S.ids[q] == id;
    perm[S.offs[id] + before] = p;
  }
}

}  // namespace moe

// route_plan.cuh -- device-side building blocks of routing and planning,
// shared by the stand-alone kernels (route.cu, plan.cu) and the fused
// route + top-k + plan kernel (route.cu).  Internal to the library.
#pragma once

#include <math.h>

#include "moe_common.cuh"

namespace moe {

constexpr int TOPK_MAX_PER_LANE = 8;  // N <= 256 scores per token, 8 per lane
constexpr int PLAN_MAX_SLOTS = 64 * 32;

// An unsigned integer with the order of the float v: the sign bit flipped
// for v >= 0, all bits flipped for v < 0, -0 taken as +0 (so that equal
// scores give equal keys) and NaN mapped to 0 (it never wins).
__device__ __forceinline__ uint32_t score_key(float v) {
  if (v != v) return 0u;
  if (v == 0.f) v = 0.f;
  const uint32_t b = __float_as_uint(v);
  return (b >> 31) ? ~b : (b | 0x80000000u);
}

// The float of a key from score_key (exact; -0 comes back as +0).
__device__ __forceinline__ float key_score(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// One warp: top-k of token t's scores z[0..N) (largest first, equal scores
// by lower id: "Making Every Verified Token Count", Sec. 2.2, eq. (4)) and
// the gate weights of the selected experts.  Each lane holds the scores of
// experts lane + 32 i as order keys; each of the k rounds takes the lane's
// best remaining (key, id), then the warp's largest key and, among lanes
// holding it, the smallest id, with one warp-reduction instruction each.
// Lane j keeps the j-th selected score for the gate.
__device__ __forceinline__ void topk_gate_warp(const float *z, int n_experts, int k, int gate,
                                               int32_t *ids_t, float *w_t) {
  const int lane = threadIdx.x & 31;
  float v[TOPK_MAX_PER_LANE];
  uint32_t key[TOPK_MAX_PER_LANE];
#pragma unroll
  for (int i = 0; i < TOPK_MAX_PER_LANE; ++i) {
    const int e = lane + 32 * i;
    v[i] = e < n_experts ? __ldcg(z + e) : -INFINITY;  // L2: other CTAs may have written z
    key[i] = e < n_experts ? score_key(v[i]) : 0u;     // 0: not a candidate
  }
  uint32_t taken = 0;        // bit i: expert lane + 32 i already selected
  float my_sel = -INFINITY;  // lane j < k: score of the j-th selected expert
  float zmax = -INFINITY;    // the largest score (the first selected)
  for (int j = 0; j < k; ++j) {
    uint32_t lk = 0u, li = 0xffffffffu;
#pragma unroll
    for (int i = 0; i < TOPK_MAX_PER_LANE; ++i)
      if (!((taken >> i) & 1u) && key[i] > lk) {  // ascending i: the first of equal keys
        lk = key[i];
        li = uint32_t(lane + 32 * i);
      }
    const uint32_t gk = __reduce_max_sync(0xffffffffu, lk);
    const uint32_t gi = __reduce_min_sync(0xffffffffu, lk == gk ? li : 0xffffffffu);
    if (gk != 0u && (gi & 31u) == uint32_t(lane)) taken |= 1u << (gi >> 5);
    if (j == 0) zmax = key_score(gk);
    if (lane == j) my_sel = key_score(gk);
    if (lane == 0) ids_t[j] = int32_t(gi);
  }
  // gate weights
  const bool mine = lane < k;
  float num = 0.f, den = 0.f;
  if (gate == MOE_GATE_SOFTMAX) {
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
  int32_t n_uniq;
  int32_t total;
};

// Extra shared memory of the budgeted plan.
struct BudgetSmem {
  int32_t perm[PLAN_MAX_SLOTS];   // the grouping of all valid slots
  float w[PLAN_MAX_SLOTS];        // the slots' gate weights
  unsigned long long key[256];    // order key of the contribution of the used expert of rank r
  int32_t expert[256];            // the used expert of rank r
  int32_t keep[256];              // by expert id
};

// What thread e (< 256) knows of expert e after plan_scan.
struct ExpertScan {
  int cnt;   // slots naming e
  int off;   // first position of e's group
  int rank;  // position of e among the used experts (valid when cnt > 0)
};

// Exclusive scan of S.hist and the compaction of the used experts: warp w
// ballots experts 32w..32w+31, __popc of the ballot below a lane gives the
// rank inside the warp, a shuffle scan gives the offsets inside the warp and
// the 8 warp totals give the bases.  Writes S.n_uniq (U) and S.total (the
// slots counted).  Every thread of the block calls it.
__device__ __forceinline__ ExpertScan plan_scan(PlanSmem &S, int n_experts) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  ExpertScan x{0, 0, 0};
  int incl = 0;
  unsigned used = 0;
  if (tid < 256) {
    x.cnt = tid < n_experts ? S.hist[tid] : 0;
    used = __ballot_sync(0xffffffffu, x.cnt > 0);
    incl = x.cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) {
      S.warp_cnt[warp] = __popc(used);
      S.warp_sum[warp] = incl;
    }
  }
  __syncthreads();
  if (tid < 256) {
    int rank_base = 0, off_base = 0, U = 0, total = 0;
    for (int w = 0; w < 8; ++w) {
      if (w < warp) {
        rank_base += S.warp_cnt[w];
        off_base += S.warp_sum[w];
      }
      U += S.warp_cnt[w];
      total += S.warp_sum[w];
    }
    x.off = off_base + incl - x.cnt;
    x.rank = rank_base + __popc(used & ((1u << lane) - 1u));
    if (tid == 0) {
      S.n_uniq = U;
      S.total = total;
    }
  }
  __syncthreads();
  return x;
}

// (key a, expert e) ranks before (key b, expert f): larger contribution, or
// equal and lower id.
__device__ __forceinline__ bool budget_beats(unsigned long long a, int e, unsigned long long b,
                                             int f) {
  return a > b || (a == b && e < f);
}

// The whole block (blockDim.x >= 256, a multiple of 32): the expert union of
// the n_slots routed ids and the grouping of the slots by expert
// ("Less Experts, Faster Decoding", eq. (1); "Making Every Verified Token
// Count", eq. (5); "The Limits of Speculation", App. A.4.1, eq. (A2)):
//   1. histogram with shared-memory atomics;
//   2. plan_scan: the used experts in ascending order and their offsets;
//   3. stable scatter: slot p goes to offs[ids[p]] + (earlier slots with the
//      same id), so slots stay ascending inside a group: one warp walks the
//      slots in order, 32 at a time; __match_any_sync gives each slot its
//      rank among the chunk's slots of the same expert, and a running count
//      per expert (in shared memory, over the offsets) carries it across
//      chunks.  (Counting the earlier slots of each slot was O(slots^2)
//      compares: ~1,000 a thread at 512 slots.);
//   4. U and the union bytes (U + n_shared) * expert bytes.
// BUDGET: at most `budget` routed experts are kept (MoE-Spec's per-layer
// expert cap).  The weights are staged in shared memory with the ids.  When
// U > budget, each used expert's contribution is the sum of its slots'
// weights w[p], added in double in ascending slot order (its group in the
// full grouping); the kept experts are the first `budget` by
// (contribution descending, id ascending); the plan is rebuilt over the kept
// slots only, and w_kept[p] = w[p] for a kept slot, 0 for a dropped one (or
// an invalid id).  routed_u (may be NULL) receives U before the cut.
// `ids` and `w` may have been written by other CTAs of the same kernel (the
// fused route + plan kernel, behind its ticket), so they are read through L2.
template <bool BUDGET>
__device__ __forceinline__ void union_plan_block(
    PlanSmem &S, BudgetSmem *B, const int32_t *ids, const float *w, int n_slots, int n_experts,
    int n_shared, int64_t expert_bytes, int budget, int32_t *hist, int32_t *uniq,
    int32_t *n_uniq, int32_t *offs, int32_t *perm, int64_t *union_bytes, float *w_kept,
    int32_t *routed_u, int32_t *err) {
  const int tid = threadIdx.x;
  if (tid < 256) S.hist[tid] = 0;
  __syncthreads();
  for (int p = tid; p < n_slots; p += blockDim.x) {
    const int e = __ldcg(ids + p);
    const bool ok = e >= 0 && e < n_experts;
    S.ids[p] = ok ? e : -1;
    if constexpr (BUDGET) B->w[p] = __ldcg(w + p);
    if (ok) atomicAdd(&S.hist[e], 1);
    else record_error(err, MOE_ERR_DEVICE_INPUT);
  }
  __syncthreads();
  ExpertScan x = plan_scan(S, n_experts);
  if (tid < 256) S.offs[tid] = x.off;
  const bool cut = BUDGET && S.n_uniq > budget;
  if (BUDGET && tid == 0 && routed_u) *routed_u = S.n_uniq;
  int32_t *group = cut ? B->perm : perm;  // where the full grouping goes
  __syncthreads();
  if (tid < 32) {
    // S.offs[e] runs on as expert e's next free position (restored below)
    const unsigned lt = (1u << tid) - 1u;
    for (int c = 0; c < n_slots; c += 32) {
      const int p = c + tid;
      const int id = p < n_slots ? S.ids[p] : -1;
      const unsigned peers = __match_any_sync(0xffffffffu, id);
      const int pos = id >= 0 ? S.offs[id] + __popc(peers & lt) : 0;
      __syncwarp();
      if (id >= 0) {
        group[pos] = p;
        if ((peers & lt) == 0u) S.offs[id] += __popc(peers);  // the group's first lane
      }
      __syncwarp();
    }
  }
  __syncthreads();
  if (tid < 256) S.offs[tid] = x.off;  // the scan's offsets again
  if constexpr (BUDGET) {
    if (cut) {
      __syncthreads();  // the grouping in B->perm is complete
      const int e = tid;
      const int U = S.n_uniq;
      unsigned long long mine = 0;
      if (e < 256 && x.cnt > 0) {
        double sum = 0.0;
        for (int i = 0; i < x.cnt; ++i) sum += double(B->w[B->perm[x.off + i]]);
        mine = order_key(sum);
        B->key[x.rank] = mine;
        B->expert[x.rank] = e;
      }
      __syncthreads();
      int keep = 0;
      if (e < 256 && x.cnt > 0) {
        int r = 0;  // used experts that rank before e
        for (int q = 0; q < U; ++q) r += budget_beats(B->key[q], B->expert[q], mine, e);
        keep = r < budget;
      }
      if (e < 256) {
        B->keep[e] = keep;
        if (!keep) S.hist[e] = 0;
      }
      __syncthreads();
      for (int p = tid; p < n_slots; p += blockDim.x) {
        const int id = S.ids[p];
        w_kept[p] = (id >= 0 && B->keep[id]) ? B->w[p] : 0.f;
      }
      const ExpertScan full = x;
      x = plan_scan(S, n_experts);  // the kept experts only
      if (tid < 256) {
        if (e < n_experts) hist[e] = x.cnt;
        if (x.cnt > 0) {
          uniq[x.rank] = e;
          offs[x.rank] = x.off;
          for (int i = 0; i < x.cnt; ++i) perm[x.off + i] = B->perm[full.off + i];
        }
        if (tid == 0) {
          offs[S.n_uniq] = S.total;
          *n_uniq = S.n_uniq;
          *union_bytes = int64_t(S.n_uniq + n_shared) * expert_bytes;
        }
      }
      return;
    }
    for (int p = tid; p < n_slots; p += blockDim.x)
      w_kept[p] = S.ids[p] >= 0 ? B->w[p] : 0.f;
  }
  if (tid < 256) {
    const int e = tid;
    if (e < n_experts) hist[e] = x.cnt;
    if (x.cnt > 0) {
      uniq[x.rank] = e;
      offs[x.rank] = x.off;
    }
    if (tid == 0) {
      offs[S.n_uniq] = S.total;
      *n_uniq = S.n_uniq;
      *union_bytes = int64_t(S.n_uniq + n_shared) * expert_bytes;
    }
  }
}

}  // namespace moe

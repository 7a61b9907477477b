// plan.cu -- the expert union of one verification pass and the grouping of
// its (token, slot) pairs by expert
// ("Less Experts, Faster Decoding: Cost-Aware Speculative Decoding for
// Mixture-of-Experts", eq. (1); "Making Every Verified Token Count", eq. (5);
// "The Limits of Speculation", App. A.4.1, eq. (A2)).
//
// One CTA of 256 threads (N <= 256, n*k <= 64*32):
//   1. histogram of the ids with shared-memory atomics;
//   2. the used experts compacted in ascending order: each warp ballots its 32
//      experts' "used" flags, __popc of the ballot below a lane gives the rank
//      inside the warp, and a scan over the 8 warp counts gives the warp base;
//   3. exclusive prefix sum of the histogram (warp shuffle scan + warp
//      totals) gives each expert's group offset;
//   4. a stable scatter: slot p goes to offs[ids[p]] + (number of earlier
//      slots with the same id), so slots stay ascending inside a group;
//   5. U and the union bytes (U + n_shared) * expert bytes.
#include "kernels.h"
#include "moe_common.cuh"

namespace moe {

namespace {

constexpr int PLAN_THREADS = 256;
constexpr int MAX_SLOTS = 64 * 32;

__global__ void __launch_bounds__(PLAN_THREADS) union_plan_kernel(
    const int32_t *__restrict__ ids, int n_slots, int n_experts, int n_shared,
    int64_t expert_bytes, int32_t *hist, int32_t *uniq, int32_t *n_uniq, int32_t *offs,
    int32_t *perm, int64_t *union_bytes, int32_t *err) {
  __shared__ int32_t s_hist[256];
  __shared__ int32_t s_offs[256];
  __shared__ int32_t s_ids[MAX_SLOTS];
  __shared__ int32_t s_warp[8];
  __shared__ int32_t s_warp_sum[8];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  s_hist[tid] = 0;
  __syncthreads();
  for (int p = tid; p < n_slots; p += PLAN_THREADS) {
    const int e = ids[p];
    const bool ok = e >= 0 && e < n_experts;
    s_ids[p] = ok ? e : -1;
    if (ok) atomicAdd(&s_hist[e], 1);
    else record_error(err, MOE_ERR_DEVICE_INPUT);
  }
  __syncthreads();

  // 2. ascending compaction of the used experts
  const int e = tid;  // expert handled by this thread (256 threads cover N <= 256)
  const int cnt = e < n_experts ? s_hist[e] : 0;
  const unsigned used = __ballot_sync(0xffffffffu, cnt > 0);
  // 3. exclusive scan of the counts inside the warp
  int incl = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int x = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += x;
  }
  if (lane == 31) {
    s_warp[warp] = __popc(used);
    s_warp_sum[warp] = incl;
  }
  __syncthreads();
  int rank_base = 0, off_base = 0;
  for (int w = 0; w < warp; ++w) {
    rank_base += s_warp[w];
    off_base += s_warp_sum[w];
  }
  int U = 0;
  for (int w = 0; w < 8; ++w) U += s_warp[w];
  const int off = off_base + incl - cnt;
  s_offs[e] = off;
  if (e < n_experts) hist[e] = cnt;
  if (cnt > 0) {
    const int r = rank_base + __popc(used & ((1u << lane) - 1u));
    uniq[r] = e;
    offs[r] = off;
  }
  if (tid == 0) {
    int total = 0;
    for (int w = 0; w < 8; ++w) total += s_warp_sum[w];
    offs[U] = total;
    *n_uniq = U;
    *union_bytes = int64_t(U + n_shared) * expert_bytes;
  }
  __syncthreads();

  // 4. stable scatter
  for (int p = tid; p < n_slots; p += PLAN_THREADS) {
    const int id = s_ids[p];
    if (id < 0) continue;
    int before = 0;
    for (int q = 0; q < p; ++q) before += s_ids[q] == id;
    perm[s_offs[id] + before] = p;
  }
}

}  // namespace

cudaError_t launch_union_plan(const int32_t *ids, int n_slots, int n_experts, int n_shared,
                              int64_t expert_bytes, int32_t *hist, int32_t *uniq, int32_t *n_uniq,
                              int32_t *offs, int32_t *perm, int64_t *union_bytes, int32_t *err,
                              cudaStream_t stream) {
  union_plan_kernel<<<1, PLAN_THREADS, 0, stream>>>(ids, n_slots, n_experts, n_shared,
                                                    expert_bytes, hist, uniq, n_uniq, offs, perm,
                                                    union_bytes, err);
  return cudaGetLastError();
}

}  // namespace moe

// plan.cu -- the stand-alone union-plan kernel: one CTA of 256 threads runs
// union_plan_block (route_plan.cuh) over the routed ids of one pass, with or
// without an expert budget.
#include "kernels.h"
#include "moe_common.cuh"
#include "route_plan.cuh"

namespace moe {

namespace {

constexpr int PLAN_THREADS = 256;

template <bool BUDGET>
__global__ void __launch_bounds__(PLAN_THREADS) union_plan_kernel(
    const int32_t *__restrict__ ids, const float *w, int n_slots, int n_experts, int n_shared,
    int64_t expert_bytes, int budget, int32_t *hist, int32_t *uniq, int32_t *n_uniq,
    int32_t *offs, int32_t *perm, int64_t *union_bytes, float *w_kept, int32_t *routed_u,
    int32_t *err) {
  pdl_trigger();  // the expert kernel behind this one may launch (it waits for the plan)
  __shared__ PlanSmem S;
  if constexpr (BUDGET) {
    __shared__ BudgetSmem B;
    union_plan_block<true>(S, &B, ids, w, n_slots, n_experts, n_shared, expert_bytes, budget,
                           hist, uniq, n_uniq, offs, perm, union_bytes, w_kept, routed_u, err);
  } else {
    union_plan_block<false>(S, nullptr, ids, nullptr, n_slots, n_experts, n_shared, expert_bytes,
                            0, hist, uniq, n_uniq, offs, perm, union_bytes, nullptr, nullptr,
                            err);
  }
}

}  // namespace

cudaError_t launch_union_plan(const int32_t *ids, int n_slots, int n_experts, int n_shared,
                              int64_t expert_bytes, int32_t *hist, int32_t *uniq, int32_t *n_uniq,
                              int32_t *offs, int32_t *perm, int64_t *union_bytes, int32_t *err,
                              cudaStream_t stream) {
  union_plan_kernel<false><<<1, PLAN_THREADS, 0, stream>>>(
      ids, nullptr, n_slots, n_experts, n_shared, expert_bytes, 0, hist, uniq, n_uniq, offs, perm,
      union_bytes, nullptr, nullptr, err);
  return cudaGetLastError();
}

cudaError_t launch_union_plan_budgeted(const int32_t *ids, const float *w, int n_slots,
                                       int n_experts, int n_shared, int64_t expert_bytes,
                                       int budget, int32_t *hist, int32_t *uniq, int32_t *n_uniq,
                                       int32_t *offs, int32_t *perm, int64_t *union_bytes,
                                       float *w_kept, int32_t *routed_u, int32_t *err,
                                       cudaStream_t stream) {
  union_plan_kernel<true><<<1, PLAN_THREADS, 0, stream>>>(
      ids, w, n_slots, n_experts, n_shared, expert_bytes, budget, hist, uniq, n_uniq, offs, perm,
      union_bytes, w_kept, routed_u, err);
  return cudaGetLastError();
}

}  // namespace moe

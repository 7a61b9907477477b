// plan.cu -- the stand-alone union-plan kernel: one CTA of 256 threads runs
// union_plan_block (route_plan.cuh) over the routed ids of one pass.
#include "kernels.h"
#include "moe_common.cuh"
#include "route_plan.cuh"

namespace moe {

namespace {

constexpr int PLAN_THREADS = 256;

__global__ void __launch_bounds__(PLAN_THREADS) union_plan_kernel(
    const int32_t *__restrict__ ids, int n_slots, int n_experts, int n_shared,
    int64_t expert_bytes, int32_t *hist, int32_t *uniq, int32_t *n_uniq, int32_t *offs,
    int32_t *perm, int64_t *union_bytes, int32_t *err) {
  __shared__ PlanSmem S;
  union_plan_block(S, ids, n_slots, n_experts, n_shared, expert_bytes, hist, uniq, n_uniq, offs,
                   perm, union_bytes, err);
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

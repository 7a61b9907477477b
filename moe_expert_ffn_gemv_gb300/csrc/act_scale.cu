// act_scale.cu -- the E4M3 engines' fp16 activation rows (act_scale.cuh), as
// kernels of their own:
//   act_scale_kernel  the hidden rows h16 = h * 2^hshift[t], a CTA per token,
//                     ahead of the gate/up kernel (moe_verify_pass writes
//                     them inside its plan kernel instead);
//   a16_scale_kernel  each slot's row of the intermediate a, in place, between
//                     the gate/up and down kernels.
// Both are launched as programmatic dependents of the kernel ahead of them
// and wait for it before reading what it wrote.
#include "act_scale.cuh"
#include "kernels.h"
#include "moe_common.cuh"

namespace moe {

namespace {

constexpr int A16_WARPS = 8;

// A CTA per token (rows held in registers): the gate/up kernel waits for
// this one, so its latency, not its bandwidth, is what counts.
__global__ void __launch_bounds__(ACT_ROW_THREADS) act_scale_kernel(const __nv_bfloat16 *__restrict__ h,
                                                                    int d, __half *h16,
                                                                    int32_t *hshift) {
  pdl_trigger();
  pdl_wait();
  act_scale_row(h, d, blockIdx.x, h16, hshift);
}

// A warp per slot row; few CTAs, so that they fit beside the gate/up
// kernel's CTAs and wait there for it to end.
__global__ void __launch_bounds__(A16_WARPS * 32) a16_scale_kernel(uint16_t *a, int slots, int inter,
                                                                   int32_t *ashift) {
  pdl_trigger();
  pdl_wait();
  const int warp = threadIdx.x >> 5;
  for (int s = blockIdx.x * A16_WARPS + warp; s < slots; s += gridDim.x * A16_WARPS)
    a16_scale_warp(a, inter, s, ashift);
}

}  // namespace

cudaError_t launch_act_scale(const void *h, int n, int d, const ActScaleOut &S,
                             cudaStream_t stream) {
  if (d > 8 * ACT_ROW_THREADS * ACT_ROW_WORDS) return cudaErrorInvalidValue;
  return launch_dependent(act_scale_kernel, dim3(n), dim3(ACT_ROW_THREADS), 0, stream,
                          static_cast<const __nv_bfloat16 *>(h), d, S.h16, S.hshift);
}

cudaError_t launch_a16_scale(void *a, int slots, int inter, int32_t *ashift, int max_ctas,
                             cudaStream_t stream) {
  int ctas = (slots + A16_WARPS - 1) / A16_WARPS;
  if (ctas > max_ctas) ctas = max_ctas;
  if (ctas < 1) ctas = 1;
  return launch_dependent(a16_scale_kernel, dim3(ctas), dim3(A16_WARPS * 32), 0, stream,
                          static_cast<uint16_t *>(a), slots, inter, ashift);
}

}  // namespace moe

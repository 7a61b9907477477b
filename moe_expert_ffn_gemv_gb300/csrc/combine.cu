// combine.cu -- the weighted sum of the layer output ("Making Every Verified
// Token Count", Sec. 2.2: the layer output is the router-weighted sum of the
// selected experts' outputs).
//
// combine_kernel: y[t][c] = sum_{j<k} w[t][j] * yslot[t*k+j][c]
//                           (+ yslot[n*k+t][c] for the shared expert),
// fp32 fused multiply-adds in that fixed order, then one rounding to the
// output dtype (round to nearest even for bf16).  A slot whose weight is 0
// is skipped, not multiplied: an expert budget leaves a dropped slot's
// yslot row unwritten and gives it weight 0.  (Skipping changes no sum:
// the accumulator starts at +0 and adding 0 * finite leaves it as it is.)
// Each thread owns 4 consecutive columns of one token (16-byte loads, all
// slots' loads issued before the multiply-adds); small CTAs so that a pass
// of a few tokens still spreads over the SMs.
#include "kernels.h"
#include "moe_common.cuh"

namespace moe {

namespace {

constexpr int COMBINE_THREADS = 64;

template <bool BF16>
__global__ void __launch_bounds__(COMBINE_THREADS) combine_kernel(const float *__restrict__ yslot,
                                                                  const float *__restrict__ w,
                                                                  int n, int k, int d,
                                                                  int n_shared,
                                                                  void *__restrict__ y,
                                                                  uint32_t *flags) {
  pdl_wait();  // the expert kernel's rows (launched as its programmatic dependent)
  // Both expert kernels have ended, so no reader of moe_verify_pass's
  // plan-ready flag and scaled-rows counter is left: clear them for the
  // next pass.
  if (flags && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) {
    flags[0] = 0u;
    flags[1] = 0u;
  }
  const int t = blockIdx.y;
  const int c = (blockIdx.x * COMBINE_THREADS + threadIdx.x) * 4;
  if (c >= d) return;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int j0 = 0; j0 < k; j0 += 8) {
    // all loads of the group first, then the multiply-adds in slot order
    float wt[8];
    float4 v[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      if (j0 + q < k) {
        wt[q] = __ldg(w + int64_t(t) * k + j0 + q);
        v[q] = __ldg(reinterpret_cast<const float4 *>(yslot + (int64_t(t) * k + j0 + q) * d + c));
      }
    }
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      if (j0 + q < k && wt[q] != 0.f) {
        acc.x = fmaf(wt[q], v[q].x, acc.x);
        acc.y = fmaf(wt[q], v[q].y, acc.y);
        acc.z = fmaf(wt[q], v[q].z, acc.z);
        acc.w = fmaf(wt[q], v[q].w, acc.w);
      }
    }
  }
  if (n_shared) {
    const float4 v =
        __ldg(reinterpret_cast<const float4 *>(yslot + (int64_t(n) * k + t) * d + c));
    acc.x += v.x;
    acc.y += v.y;
    acc.z += v.z;
    acc.w += v.w;
  }
  if (BF16) {
    __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
    __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
    uint2 out;
    out.x = *reinterpret_cast<uint32_t *>(&lo);
    out.y = *reinterpret_cast<uint32_t *>(&hi);
    *reinterpret_cast<uint2 *>(static_cast<__nv_bfloat16 *>(y) + int64_t(t) * d + c) = out;
  } else {
    *reinterpret_cast<float4 *>(static_cast<float *>(y) + int64_t(t) * d + c) = acc;
  }
}

}  // namespace

cudaError_t launch_combine(const float *yslot, const float *w, int n, int k, int d, int n_shared,
                           bool out_bf16, void *y, uint32_t *flags, cudaStream_t stream) {
  dim3 grid((d / 4 + COMBINE_THREADS - 1) / COMBINE_THREADS, n);
  if (out_bf16)
    return launch_dependent(combine_kernel<true>, grid, dim3(COMBINE_THREADS), 0, stream, yslot,
                            w, n, k, d, n_shared, y, flags);
  return launch_dependent(combine_kernel<false>, grid, dim3(COMBINE_THREADS), 0, stream, yslot, w,
                          n, k, d, n_shared, y, flags);
}

}  // namespace moe

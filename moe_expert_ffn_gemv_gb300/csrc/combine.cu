// combine.cu -- the weighted sum of the layer output ("Making Every Verified
// Token Count", Sec. 2.2: "the layer output is the corresponding weighted
// sum"), plus the bf16 -> fp16 copy of the hidden states used by the E4M3
// tensor-core path.
//
// combine_kernel: y[t][c] = sum_{j<k} w[t][j] * yslot[t*k+j][c]
//                           (+ yslot[n*k+t][c] for the shared expert),
// fp32 fused multiply-adds in that fixed order, then one rounding to the
// output dtype (round to nearest even for bf16).  Each thread owns 4
// consecutive columns of one token (16-byte loads).
#include "kernels.h"
#include "moe_common.cuh"

namespace moe {

namespace {

template <bool BF16>
__global__ void __launch_bounds__(256) combine_kernel(const float *__restrict__ yslot,
                                                      const float *__restrict__ w, int n, int k,
                                                      int d, int n_shared, void *__restrict__ y) {
  const int t = blockIdx.y;
  const int c = (blockIdx.x * 256 + threadIdx.x) * 4;
  if (c >= d) return;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int j = 0; j < k; ++j) {
    const float wt = __ldg(w + int64_t(t) * k + j);
    const float4 v = __ldg(reinterpret_cast<const float4 *>(yslot + (int64_t(t) * k + j) * d + c));
    acc.x = fmaf(wt, v.x, acc.x);
    acc.y = fmaf(wt, v.y, acc.y);
    acc.z = fmaf(wt, v.z, acc.z);
    acc.w = fmaf(wt, v.w, acc.w);
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

__global__ void bf16_to_f16_kernel(const uint4 *__restrict__ src, uint4 *__restrict__ dst,
                                   int64_t n8) {
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n8;
       i += int64_t(gridDim.x) * blockDim.x) {
    const uint4 v = __ldg(src + i);
    const uint32_t in[4] = {v.x, v.y, v.z, v.w};
    uint32_t out[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float lo = __uint_as_float(in[q] << 16);
      const float hi = __uint_as_float(in[q] & 0xFFFF0000u);
      __half2 h2 = __floats2half2_rn(lo, hi);
      out[q] = *reinterpret_cast<uint32_t *>(&h2);
    }
    dst[i] = make_uint4(out[0], out[1], out[2], out[3]);
  }
}

}  // namespace

cudaError_t launch_combine(const float *yslot, const float *w, int n, int k, int d, int n_shared,
                           bool out_bf16, void *y, cudaStream_t stream) {
  dim3 grid((d / 4 + 255) / 256, n);
  if (out_bf16) combine_kernel<true><<<grid, 256, 0, stream>>>(yslot, w, n, k, d, n_shared, y);
  else combine_kernel<false><<<grid, 256, 0, stream>>>(yslot, w, n, k, d, n_shared, y);
  return cudaGetLastError();
}

cudaError_t launch_bf16_to_f16(const void *src, void *dst, int64_t count, cudaStream_t stream) {
  const int64_t n8 = count / 8;
  int blocks = int((n8 + 255) / 256);
  if (blocks > 1024) blocks = 1024;
  if (blocks < 1) blocks = 1;
  bf16_to_f16_kernel<<<blocks, 256, 0, stream>>>(static_cast<const uint4 *>(src),
                                                  static_cast<uint4 *>(dst), n8);
  return cudaGetLastError();
}

}  // namespace moe

// expert_f32.cu -- the grouped expert FFN for fp32 weights, on CUDA cores.
//
// The same segments as the tensor-core kernel (deduplicating: one union
// expert with all its tokens; per-slot: one (token, slot) pair), the same two
// phases (a = silu(W1 x) * (W3 x), then y_slot = W2 a), fp32 throughout so
// that the result stays within fp32 rounding of the exact sum.  Work item =
// (segment, block of 8 rows); warp w of the CTA owns row 8 rb + w and walks
// its columns with 16-byte loads, each weight row read once per segment and
// applied to up to 8 tokens per sweep; lane partial sums are added with xor
// shuffles (fixed order).
#include "kernels.h"
#include "moe_common.cuh"

namespace moe {

namespace {

constexpr int WARPS = 8;
constexpr int TOK = 8;

__device__ __forceinline__ float dot4(float4 a, float4 b, float acc) {
  acc = fmaf(a.x, b.x, acc);
  acc = fmaf(a.y, b.y, acc);
  acc = fmaf(a.z, b.z, acc);
  return fmaf(a.w, b.w, acc);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

template <int PHASE>
__global__ void __launch_bounds__(WARPS * 32) expert_f32_kernel(const F32Params P) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rows = PHASE == 1 ? P.inter : P.d;      // output rows of this phase
  const int kdim = PHASE == 1 ? P.d : P.inter;
  const int row_blocks = (rows + WARPS - 1) / WARPS;
  const int n_items = n_segments(P.T) * row_blocks;
  if (P.T.dedup && blockIdx.x == 0 && threadIdx.x == 0) {
    const int32_t U = __ldg(P.T.n_uniq);
    if (U < 0 || U > P.T.n_experts) record_error(P.err, MOE_ERR_DEVICE_INPUT);
  }
  for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
    const int u = item / row_blocks, rb = item - u * row_blocks;
    const Seg sg = get_segment(P.T, u);
    if (sg.expert == -2) {
      if (threadIdx.x == 0 && rb == 0) record_error(P.err, MOE_ERR_DEVICE_INPUT);
      continue;
    }
    const int row = rb * WARPS + warp;
    if (row >= rows) continue;
    const float *wr, *wu = nullptr;
    if (PHASE == 1) {
      const float *base = sg.expert >= 0 ? P.w13 + int64_t(sg.expert) * 2 * P.inter * P.d : P.sh_w13;
      wr = base + int64_t(row) * P.d;
      wu = base + int64_t(P.inter + row) * P.d;
    } else {
      const float *base = sg.expert >= 0 ? P.w2 + int64_t(sg.expert) * P.d * P.inter : P.sh_w2;
      wr = base + int64_t(row) * P.inter;
    }
    for (int t0 = 0; t0 < sg.m; t0 += TOK) {
      const int nt = min(TOK, sg.m - t0);
      int src[TOK];
#pragma unroll
      for (int t = 0; t < TOK; ++t) {
        src[t] = 0;
        if (t < nt) {
          const int slot = segment_slot(P.T, sg, t0 + t);
          src[t] = PHASE == 1 ? slot_token(P.T, slot) : slot;
        }
      }
      float ag[TOK], au[TOK];
#pragma unroll
      for (int t = 0; t < TOK; ++t) ag[t] = au[t] = 0.f;
      const float *x = PHASE == 1 ? P.h : P.inter_out;
      for (int c = lane * 4; c < kdim; c += 128) {
        const float4 w4 = __ldg(reinterpret_cast<const float4 *>(wr + c));
        float4 u4 = make_float4(0.f, 0.f, 0.f, 0.f);
        if (PHASE == 1) u4 = __ldg(reinterpret_cast<const float4 *>(wu + c));
#pragma unroll
        for (int t = 0; t < TOK; ++t) {
          if (t < nt) {
            const float4 x4 = *reinterpret_cast<const float4 *>(x + int64_t(src[t]) * kdim + c);
            ag[t] = dot4(w4, x4, ag[t]);
            if (PHASE == 1) au[t] = dot4(u4, x4, au[t]);
          }
        }
      }
#pragma unroll
      for (int t = 0; t < TOK; ++t) {
        if (t < nt) {
          const float gs = warp_sum(ag[t]);
          const float us = PHASE == 1 ? warp_sum(au[t]) : 0.f;
          if (lane == 0) {
            const int slot = segment_slot(P.T, sg, t0 + t);
            if (PHASE == 1) {
              // silu(g) * u with the accurate expf: fp32 end to end
              P.inter_out[int64_t(slot) * P.inter + row] = gs / (1.0f + expf(-gs)) * us;
            } else {
              P.yslot[int64_t(slot) * P.d + row] = gs;
            }
          }
        }
      }
    }
  }
}

}  // namespace

cudaError_t launch_expert_f32(int phase, const F32Params &P, int grid, cudaStream_t stream) {
  if (phase == 1) expert_f32_kernel<1><<<grid, WARPS * 32, 0, stream>>>(P);
  else expert_f32_kernel<2><<<grid, WARPS * 32, 0, stream>>>(P);
  return cudaGetLastError();
}

}  // namespace moe

// act_scale.cuh -- the E4M3 engines' fp16 activation rows (internal).
//
// The E4M3 expert kernels multiply on fp16 tensor cores.  Before them, each
// token's bf16 hidden row is scaled by the exact power of two 2^hshift[t]
// that puts its largest magnitude in [2^14, 2^15) (fp16_range_shift) and
// stored as fp16 (h16), so that no hidden state overflows fp16 and every
// element above 2^-28 of the row's largest keeps all its bits; the gate/up
// kernel scales its sums back.  Between the gate/up and down kernels, each
// slot's row of the intermediate a is brought into fp16 range the same way
// (a16_scale_warp), and the down kernel scales its sums back.
#pragma once

#include "moe_common.cuh"

namespace moe {

constexpr int ACT_SCALE_TOKENS = 8;    // tokens per CTA
constexpr int ACT_SCALE_MAX_WARPS = 16;

// Tokens [t0, t0 + nt) (nt <= 8) of h [n][d] (bf16, d % 8 == 0), by every
// thread of the block (at most 16 warps).  All loads of a chunk are issued
// before they are used, as in the router.
__device__ __forceinline__ void act_scale_block(const __nv_bfloat16 *__restrict__ h, int d,
                                                int t0, int nt, __half *__restrict__ h16,
                                                int32_t *hshift) {
  __shared__ float s_part[ACT_SCALE_MAX_WARPS][ACT_SCALE_TOKENS];
  __shared__ int s_shift[ACT_SCALE_TOKENS];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_warps = blockDim.x >> 5;
  float m[ACT_SCALE_TOKENS];
#pragma unroll
  for (int t = 0; t < ACT_SCALE_TOKENS; ++t) m[t] = 0.f;
  for (int c = threadIdx.x * 8; c < d; c += blockDim.x * 8) {
    uint4 v[ACT_SCALE_TOKENS];
#pragma unroll
    for (int t = 0; t < ACT_SCALE_TOKENS; ++t)
      if (t < nt) v[t] = __ldg(reinterpret_cast<const uint4 *>(h + int64_t(t0 + t) * d + c));
#pragma unroll
    for (int t = 0; t < ACT_SCALE_TOKENS; ++t)
      if (t < nt) {
        const uint32_t w[4] = {v[t].x, v[t].y, v[t].z, v[t].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          // fmaxf drops a NaN operand, so a NaN leaves the maximum alone
          m[t] = fmaxf(m[t], fabsf(__uint_as_float(w[i] << 16)));
          m[t] = fmaxf(m[t], fabsf(__uint_as_float(w[i] & 0xFFFF0000u)));
        }
      }
  }
#pragma unroll
  for (int t = 0; t < ACT_SCALE_TOKENS; ++t) {
    float x = m[t];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    if (lane == 0) s_part[warp][t] = x;
  }
  __syncthreads();
  if (threadIdx.x < nt) {
    float x = 0.f;
    for (int w = 0; w < n_warps; ++w) x = fmaxf(x, s_part[w][threadIdx.x]);
    const int s = fp16_range_shift(__float_as_uint(x));
    s_shift[threadIdx.x] = s;
    hshift[t0 + threadIdx.x] = s;
  }
  __syncthreads();
  for (int c = threadIdx.x * 8; c < d; c += blockDim.x * 8) {
    uint4 v[ACT_SCALE_TOKENS];
#pragma unroll
    for (int t = 0; t < ACT_SCALE_TOKENS; ++t)
      if (t < nt) v[t] = __ldg(reinterpret_cast<const uint4 *>(h + int64_t(t0 + t) * d + c));
#pragma unroll
    for (int t = 0; t < ACT_SCALE_TOKENS; ++t)
      if (t < nt) {
        const float mul = pow2f(s_shift[t]);
        const uint32_t w[4] = {v[t].x, v[t].y, v[t].z, v[t].w};
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const __half2 p = __floats2half2_rn(__uint_as_float(w[i] << 16) * mul,
                                              __uint_as_float(w[i] & 0xFFFF0000u) * mul);
          o[i] = *reinterpret_cast<const uint32_t *>(&p);
        }
        *reinterpret_cast<uint4 *>(h16 + int64_t(t0 + t) * d + c) = make_uint4(o[0], o[1], o[2], o[3]);
      }
  }
}

// Token t's row of h [n][d] (bf16, d % 8 == 0, d <= 8 * ACT_ROW_THREADS *
// ACT_ROW_WORDS), by the ACT_ROW_THREADS threads of the block: the row's
// 16-byte words stay in registers between the maximum and the rewrite, so
// the row is read once.  Same shift and same fp16 values as act_scale_block.
constexpr int ACT_ROW_THREADS = 256;
constexpr int ACT_ROW_WORDS = 4;  // 16-byte words a thread keeps: rows of up to 8192

__device__ __forceinline__ void act_scale_row(const __nv_bfloat16 *__restrict__ h, int d, int t,
                                              __half *__restrict__ h16, int32_t *hshift) {
  __shared__ float s_part[ACT_ROW_THREADS / 32];
  __shared__ int s_shift;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const __nv_bfloat16 *row = h + int64_t(t) * d;
  uint4 v[ACT_ROW_WORDS];
  float m = 0.f;
#pragma unroll
  for (int i = 0; i < ACT_ROW_WORDS; ++i) {
    const int c = (i * ACT_ROW_THREADS + int(threadIdx.x)) * 8;
    if (c < d) v[i] = __ldg(reinterpret_cast<const uint4 *>(row + c));
  }
#pragma unroll
  for (int i = 0; i < ACT_ROW_WORDS; ++i) {
    const int c = (i * ACT_ROW_THREADS + int(threadIdx.x)) * 8;
    if (c < d) {
      const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        // fmaxf drops a NaN operand, so a NaN leaves the maximum alone
        m = fmaxf(m, fabsf(__uint_as_float(w[j] << 16)));
        m = fmaxf(m, fabsf(__uint_as_float(w[j] & 0xFFFF0000u)));
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (lane == 0) s_part[warp] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float x = 0.f;
    for (int w = 0; w < ACT_ROW_THREADS / 32; ++w) x = fmaxf(x, s_part[w]);
    const int sh = fp16_range_shift(__float_as_uint(x));
    s_shift = sh;
    hshift[t] = sh;
  }
  __syncthreads();
  const float mul = pow2f(s_shift);
#pragma unroll
  for (int i = 0; i < ACT_ROW_WORDS; ++i) {
    const int c = (i * ACT_ROW_THREADS + int(threadIdx.x)) * 8;
    if (c < d) {
      const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
      uint32_t o[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const __half2 p = __floats2half2_rn(__uint_as_float(w[j] << 16) * mul,
                                            __uint_as_float(w[j] & 0xFFFF0000u) * mul);
        o[j] = *reinterpret_cast<const uint32_t *>(&p);
      }
      *reinterpret_cast<uint4 *>(h16 + int64_t(t) * d + c) = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

// One warp: row `slot` of a [slots][I] (bf16 as the gate/up kernel wrote
// it; I % 8 == 0), rewritten in place as fp16 times 2^ashift[slot].  Each
// lane handles its own 16-byte words: rows of up to 2048 elements are held
// in registers between the maximum and the rewrite (one read of the row);
// longer rows are read twice.
constexpr int A16_REG_WORDS = 8;  // 16-byte words a lane keeps

__device__ __forceinline__ uint4 a16_convert(uint4 v, float mul) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t o[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const __half2 p = __floats2half2_rn(__uint_as_float(w[j] << 16) * mul,
                                        __uint_as_float(w[j] & 0xFFFF0000u) * mul);
    o[j] = *reinterpret_cast<const uint32_t *>(&p);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

__device__ __forceinline__ float a16_absmax(uint4 v, float m) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    m = fmaxf(m, fabsf(__uint_as_float(w[i] << 16)));
    m = fmaxf(m, fabsf(__uint_as_float(w[i] & 0xFFFF0000u)));
  }
  return m;
}

__device__ __forceinline__ void a16_scale_warp(uint16_t *a, int inter, int slot,
                                               int32_t *ashift) {
  const int lane = threadIdx.x & 31;
  uint4 *row = reinterpret_cast<uint4 *>(a + int64_t(slot) * inter);
  const int words = inter / 8;  // 16-byte words of the row
  float m = 0.f;
  if (words <= A16_REG_WORDS * 32) {
    uint4 v[A16_REG_WORDS];
#pragma unroll
    for (int q = 0; q < A16_REG_WORDS; ++q) {
      const int i = q * 32 + lane;
      v[q] = i < words ? row[i] : make_uint4(0u, 0u, 0u, 0u);
      m = a16_absmax(v[q], m);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const int s = fp16_range_shift(__float_as_uint(m));
    if (lane == 0) ashift[slot] = s;
    const float mul = pow2f(s);
#pragma unroll
    for (int q = 0; q < A16_REG_WORDS; ++q) {
      const int i = q * 32 + lane;
      if (i < words) row[i] = a16_convert(v[q], mul);
    }
    return;
  }
  for (int i = lane; i < words; i += 32) m = a16_absmax(row[i], m);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  const int s = fp16_range_shift(__float_as_uint(m));
  if (lane == 0) ashift[slot] = s;
  const float mul = pow2f(s);
  for (int i = lane; i < words; i += 32) row[i] = a16_convert(row[i], mul);
}

}  // namespace moe

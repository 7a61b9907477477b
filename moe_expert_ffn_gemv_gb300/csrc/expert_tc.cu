// expert_tc.cu -- the grouped expert FFN on tensor cores, for BF16 and
// FP8-E4M3 (128x128 block-scaled) expert weights.
//
// One kernel template serves both engines of "Speculative Decoding for
// Mixture-of-Experts Models: Expert Bytes, Kernel Bandwidth and the Best
// Draft Length" (abstract; Fig. 3):
//   deduplicating  a segment is one union expert with all m tokens routed to
//                  it, so each expert's weights cross HBM once per pass;
//   per-slot       a segment is one (token, slot) pair, so an expert's weights
//                  are requested once per pair that names it.
// and both halves of the SwiGLU FFN:
//   PHASE 1  a = silu(W1 x) * (W3 x)  over gate rows [32 rb, 32 rb + 32) and the
//            matching up rows, K = d; writes a[slot][I] (bf16 or fp16);
//   PHASE 2  y_slot = W2 a           over rows [64 rb, 64 rb + 64) of W2, K = I;
//            writes yslot[slot][d] (fp32).
//
// Structure (one CTA per SM, persistent over work items (segment, row block)):
//   - warp 8 is the producer: it streams 64 weight rows x 512 bytes per stage
//     with 1-D TMA bulk copies (cp.async.bulk, completing on an mbarrier) into
//     a 4- or 5-stage shared-memory ring;
//   - warps 0..7 consume: warp w owns bytes [64 w, 64 w + 64) of every row of a
//     stage, i.e. a K-split across warps, and runs mma.sync m16n8k16 with the
//     weights as the 16-row A operand (4 row tiles) and the segment's tokens as
//     the 8-wide N operand (NT tiles).  Because a dot product does not depend
//     on the order of its terms, each thread's 16 contiguous weight bytes feed
//     the A fragment directly (no ldmatrix); the activations (B fragment) are
//     read with the same permutation of K;
//   - E4M3 bytes become fp16 with cvt.rn.f16x2.e4m3x2 (exact); the block scale
//     multiplies the fp32 partial sum of each 64-column chunk, which lies in a
//     single 128x128 scale block;
//   - after the last stage of an item the 8 warps' partial sums are added in
//     shared memory in a fixed order (deterministic), and the epilogue applies
//     silu(g)*u (phase 1) or stores the fp32 rows (phase 2).
// Every wait is bounded; on time-out the kernel records MOE_ERR_TIMEOUT in the
// workspace error word, keeps its barrier structure, lets its own copies land
// and returns.
#include "moe_common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int ROWS = 64;          // weight rows per stage (4 MMA row tiles)
constexpr int KBYTES = 512;       // bytes of each row per stage
constexpr int ROW_STRIDE = 576;   // shared-memory stride of a row: the two rows a
                                  // quarter-warp reads sit 16 banks apart
constexpr int STAGE_BYTES = ROWS * ROW_STRIDE;
constexpr int CONSUMERS = 8;
constexpr int THREADS = (CONSUMERS + 1) * 32;
constexpr uint64_t DRAIN_LIMIT_NS = 200ull * 1000 * 1000;

template <int NT>
constexpr int n_stages() { return NT >= 4 ? 4 : 5; }

template <int NT>
constexpr size_t red_bytes() { return size_t(CONSUMERS) * 4 * NT * 32 * 16; }

template <int NT>
constexpr size_t smem_bytes() {
  return size_t(n_stages<NT>()) * STAGE_BYTES + red_bytes<NT>() + 2 * n_stages<NT>() * 8;
}

__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(CONSUMERS * 32) : "memory");
}

__device__ __forceinline__ float silu_times(float g, float u) {
  return g / (1.0f + __expf(-g)) * u;
}

template <bool FP8, int PHASE, int NT>
__global__ void __launch_bounds__(THREADS, 1) expert_tc_kernel(const TcParams P) {
  constexpr int S = n_stages<NT>();
  constexpr int ES = FP8 ? 1 : 2;       // bytes per weight element
  constexpr int TOK = 8 * NT;           // tokens per pass over an item
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t *ring = smem;
  float4 *red = reinterpret_cast<float4 *>(smem + S * STAGE_BYTES);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + S * STAGE_BYTES + red_bytes<NT>());
  uint64_t *empty = full + S;
  __shared__ volatile int s_abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], CONSUMERS);
    }
    s_abort = 0;
    fence_barrier_init();
  }
  __syncthreads();

  const int n_items = n_segments(P.T) * P.row_blocks;
  const int kbytes = P.kdim * ES;
  const int kstages = (kbytes + KBYTES - 1) / KBYTES;
  const int scale_cols = P.kdim / 128;              // E4M3 scale table width
  const int64_t scale_stride = int64_t(P.rows_total / 128) * scale_cols;

  if (warp == CONSUMERS) {
    // ------------------------------------------------------------ producer
    const uint64_t policy = policy_evict_first();
    uint32_t it = 0;
    bool ok = true;
    for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
      const int u = item / P.row_blocks, rb = item - u * P.row_blocks;
      const Seg sg = get_segment(P.T, u);
      if (sg.expert == -2) continue;
      const int groups = (sg.m + TOK - 1) / TOK;
      const uint8_t *base = sg.expert >= 0 ? P.w + int64_t(sg.expert) * P.expert_stride : P.w_sh;
      for (int grp = 0; grp < groups && ok; ++grp) {
        for (int ks = 0; ks < kstages; ++ks, ++it) {
          const int s = it % S;
          const uint32_t round = it / S;
          if (round > 0 && !mbar_wait_bounded(&empty[s], (round - 1) & 1, P.timeout_ns)) {
            ok = false;
            break;
          }
          if (s_abort) { ok = false; break; }
          const int k0 = ks * KBYTES;
          const int nb = min(KBYTES, kbytes - k0);
          if (lane == 0) mbar_arrive_expect_tx(&full[s], uint32_t(ROWS * nb));
          __syncwarp();
          for (int r = lane; r < ROWS; r += 32) {
            int grow;
            if (PHASE == 1) grow = r < 32 ? rb * 32 + r : P.inter + rb * 32 + (r - 32);
            else grow = rb * ROWS + r;
            bulk_g2s(ring + s * STAGE_BYTES + r * ROW_STRIDE, base + int64_t(grow) * kbytes + k0,
                     uint32_t(nb), &full[s], policy);
          }
        }
      }
    }
    if (!ok) {
      if (lane == 0) {
        record_error(P.err, MOE_ERR_TIMEOUT);
        s_abort = 1;
      }
    }
    // Let every copy this warp issued land before the CTA may exit.
    const uint32_t issued = it;
    const uint32_t first = issued > uint32_t(S) ? issued - S : 0;
    for (uint32_t j = first; j < issued; ++j)
      if (!mbar_wait_bounded(&full[j % S], (j / S) & 1, DRAIN_LIMIT_NS)) {
        if (lane == 0) record_error(P.err, MOE_ERR_TIMEOUT);
        break;
      }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int g = lane >> 2, c = lane & 3;
  const int tid = threadIdx.x;
  const uint16_t *act = static_cast<const uint16_t *>(P.act);
  uint32_t it = 0;
  bool aborted = false;

  for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
    const int u = item / P.row_blocks, rb = item - u * P.row_blocks;
    const Seg sg = get_segment(P.T, u);
    if (sg.expert == -2) {
      if (tid == 0 && rb == 0) record_error(P.err, MOE_ERR_DEVICE_INPUT);
      continue;
    }
    const int groups = (sg.m + TOK - 1) / TOK;
    const float *scales = nullptr;
    if (FP8) scales = sg.expert >= 0 ? P.sc + int64_t(sg.expert) * scale_stride : P.sc_sh;
    // E4M3 scale rows of the two halves of the stage (phase 1: gate, up)
    const int srow_a = PHASE == 1 ? (rb * 32) / 128 : (rb * ROWS) / 128;
    const int srow_b = PHASE == 1 ? (P.inter + rb * 32) / 128 : srow_a;

    for (int grp = 0; grp < groups; ++grp) {
      const int m_left = sg.m - grp * TOK;   // tokens of this pass (may exceed TOK)
      // activation row of this lane's token in each N tile
      int arow[NT];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int col = nt * 8 + g;
        arow[nt] = -1;
        if (col < m_left) {
          const int slot = segment_slot(P.T, sg, grp * TOK + col);
          arow[nt] = PHASE == 1 ? slot_token(P.T, slot) : slot;
        }
      }
      float acc[4][NT][4];
#pragma unroll
      for (int mt = 0; mt < 4; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int q = 0; q < 4; ++q) acc[mt][nt][q] = 0.f;

      for (int ks = 0; ks < kstages; ++ks, ++it) {
        const int s = it % S;
        const uint32_t round = it / S;
        const int kb0 = ks * KBYTES + warp * 64;          // first byte of this warp's chunk
        const bool active = kb0 < kbytes;
        const int kcol0 = kb0 / ES;                        // first weight column of the chunk
        // B fragments: this lane's token, the chunk's columns in the same order
        // as the thread's weight bytes.
        constexpr int BW = FP8 ? 8 : 4;
        uint32_t bfr[NT][BW];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
          for (int q = 0; q < BW; ++q) bfr[nt][q] = 0u;
          if (active && arow[nt] >= 0) {
            const uint4 *src = reinterpret_cast<const uint4 *>(
                act + int64_t(arow[nt]) * P.kdim + kcol0 + (FP8 ? 16 * c : 8 * c));
#pragma unroll
            for (int v = 0; v < BW / 4; ++v) {
              const uint4 x = __ldg(src + v);
              bfr[nt][4 * v + 0] = x.x;
              bfr[nt][4 * v + 1] = x.y;
              bfr[nt][4 * v + 2] = x.z;
              bfr[nt][4 * v + 3] = x.w;
            }
          }
        }
        if (!aborted && s_abort) aborted = true;
        if (!aborted && !mbar_wait_bounded(&full[s], round & 1, P.timeout_ns)) {
          aborted = true;
          s_abort = 1;
          if (lane == 0) record_error(P.err, MOE_ERR_TIMEOUT);
        }
        if (!aborted && active) {
          const uint8_t *st = ring + s * STAGE_BYTES + warp * 64 + c * 16;
          float sc_a = 1.f, sc_b = 1.f;
          if (FP8) {
            sc_a = __ldg(scales + int64_t(srow_a) * scale_cols + kcol0 / 128);
            sc_b = __ldg(scales + int64_t(srow_b) * scale_cols + kcol0 / 128);
          }
#pragma unroll
          for (int mt = 0; mt < 4; ++mt) {
            const uint4 lo = *reinterpret_cast<const uint4 *>(st + (mt * 16 + g) * ROW_STRIDE);
            const uint4 hi = *reinterpret_cast<const uint4 *>(st + (mt * 16 + g + 8) * ROW_STRIDE);
            const uint32_t wl[4] = {lo.x, lo.y, lo.z, lo.w};
            const uint32_t wh[4] = {hi.x, hi.y, hi.z, hi.w};
            if (FP8) {
              float tmp[NT][4];
#pragma unroll
              for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int q = 0; q < 4; ++q) tmp[nt][q] = 0.f;
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                uint32_t a[4];
                a[0] = e4m3x2_to_f16x2(wl[j]);
                a[1] = e4m3x2_to_f16x2(wh[j]);
                a[2] = e4m3x2_to_f16x2(wl[j] >> 16);
                a[3] = e4m3x2_to_f16x2(wh[j] >> 16);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
                  if (nt * 8 < m_left) mma_16816<false>(tmp[nt], a, bfr[nt][2 * j], bfr[nt][2 * j + 1]);
              }
              const float scl = mt < 2 ? sc_a : sc_b;
#pragma unroll
              for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int q = 0; q < 4; ++q) acc[mt][nt][q] = fmaf(scl, tmp[nt][q], acc[mt][nt][q]);
            } else {
#pragma unroll
              for (int j = 0; j < 2; ++j) {
                const uint32_t a[4] = {wl[2 * j], wh[2 * j], wl[2 * j + 1], wh[2 * j + 1]};
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
                  if (nt * 8 < m_left)
                    mma_16816<true>(acc[mt][nt], a, bfr[nt][2 * j], bfr[nt][2 * j + 1]);
              }
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
      }

      // ---- epilogue: add the 8 warps' K-partials in a fixed order
#pragma unroll
      for (int mt = 0; mt < 4; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
          red[((warp * 4 + mt) * NT + nt) * 32 + lane] =
              make_float4(acc[mt][nt][0], acc[mt][nt][1], acc[mt][nt][2], acc[mt][nt][3]);
      consumer_sync();
      if (!aborted) {
        constexpr int MT_OUT = PHASE == 1 ? 2 : 4;
        for (int q = tid; q < MT_OUT * NT * 32; q += CONSUMERS * 32) {
          const int ln = q & 31, nt = (q >> 5) % NT, mt = q / (32 * NT);
          float4 v = make_float4(0.f, 0.f, 0.f, 0.f), w4 = v;
#pragma unroll
          for (int w = 0; w < CONSUMERS; ++w) {
            const float4 x = red[((w * 4 + mt) * NT + nt) * 32 + ln];
            v.x += x.x; v.y += x.y; v.z += x.z; v.w += x.w;
            if (PHASE == 1) {
              const float4 y = red[((w * 4 + mt + 2) * NT + nt) * 32 + ln];
              w4.x += y.x; w4.y += y.y; w4.z += y.z; w4.w += y.w;
            }
          }
          const int gg = ln >> 2, cc = ln & 3;
          const float vals[4] = {v.x, v.y, v.z, v.w};
          const float ups[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int row = mt * 16 + gg + (e >> 1) * 8;
            const int col = nt * 8 + 2 * cc + (e & 1);
            if (col >= m_left || col >= TOK) continue;
            const int slot = segment_slot(P.T, sg, grp * TOK + col);
            if (PHASE == 1) {
              const float a = silu_times(vals[e], ups[e]);
              uint16_t *out = static_cast<uint16_t *>(P.out) + int64_t(slot) * P.inter + rb * 32 + row;
              if (FP8) *reinterpret_cast<__half *>(out) = __float2half_rn(a);
              else *reinterpret_cast<__nv_bfloat16 *>(out) = __float2bfloat16_rn(a);
            } else {
              float *out = static_cast<float *>(P.out) + int64_t(slot) * P.rows_total + rb * ROWS + row;
              *out = vals[e];
            }
          }
        }
      }
      consumer_sync();
    }
  }
}

template <bool FP8, int PHASE, int NT>
cudaError_t launch_one(const TcParams &P, int grid, cudaStream_t stream) {
  auto kern = expert_tc_kernel<FP8, PHASE, NT>;
  const size_t smem = smem_bytes<NT>();
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return e;
  kern<<<grid, THREADS, smem, stream>>>(P);
  return cudaGetLastError();
}

template <bool FP8, int PHASE>
cudaError_t launch_nt(const TcParams &P, int nt, int grid, cudaStream_t stream) {
  if (nt <= 1) return launch_one<FP8, PHASE, 1>(P, grid, stream);
  if (nt == 2) return launch_one<FP8, PHASE, 2>(P, grid, stream);
  return launch_one<FP8, PHASE, 4>(P, grid, stream);
}

}  // namespace

cudaError_t launch_expert_tc(bool fp8, int phase, int n_tiles, const TcParams &P, int grid,
                             cudaStream_t stream) {
  if (fp8) {
    return phase == 1 ? launch_nt<true, 1>(P, n_tiles, grid, stream)
                      : launch_nt<true, 2>(P, n_tiles, grid, stream);
  }
  return phase == 1 ? launch_nt<false, 1>(P, n_tiles, grid, stream)
                    : launch_nt<false, 2>(P, n_tiles, grid, stream);
}

}  // namespace moe

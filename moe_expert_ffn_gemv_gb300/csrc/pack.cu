// pack.cu -- the one-time repacking of expert weights into the tile layout
// the tensor-core expert kernel streams.
//
// An expert matrix (W13 [2I][d] or W2 [d][I], row-major, `es` bytes per
// element, K = row bytes) is cut into tiles of 64 rows x 512 bytes of K (the
// last K tile of a row block may be narrower: a multiple of 64 bytes for
// E4M3, of 128 bytes for BF16).  For W13 a tile's 64 rows are gate rows
// [32 rb, 32 rb + 32) followed by the up rows I + [32 rb, 32 rb + 32), so
// that one tile feeds both halves of silu(g) * u; for W2 they are rows
// [64 rb, 64 rb + 64).  Tiles of one row block are consecutive (K order); row
// blocks follow each other.  Inside a tile:
//   BF16  the canonical K-major layout with 128-byte swizzle of the tensor
//         cores' shared-memory operands: [128-byte column q][8-row group m]
//         [row r][16-byte chunk], chunk j of row 8 m + r stored at position
//         j ^ r, so that a 1024-byte aligned copy of a column is an operand
//         tcgen05.mma reads as it is; the mma.sync consumers read it without
//         bank conflicts too (expert_tc.cu);
//   E4M3  16-byte pieces ordered [warp w][row tile mt][half h][lane]
//         [16 bytes]: lane (g, c) = (lane / 4, lane % 4) of warp w takes row
//         16 mt + g + 8 h, bytes 512 kc + 64 w + 16 c .. +15 -- exactly the
//         A-fragment bytes that thread needs, read with one lane-contiguous
//         16-byte load.
// E4M3 tiles are each followed by their 8 block scales (32 bytes):
// the 128-column blocks 4 kc .. 4 kc + 3 of the 128-row block of the tile's
// first 32 rows, then of its last 32 rows (0 past the last column block), so
// that one bulk copy brings a stage its weights and its scales.  Without
// scales the packed matrix has exactly the size of the original.
#include "kernels.h"
#include "moe_common.cuh"

namespace moe {

namespace {

__global__ void pack_kernel(const uint4 *__restrict__ src, const float *__restrict__ scales,
                            uint4 *__restrict__ dst, int64_t n16, int64_t per_matrix16, int rows,
                            int kbytes, int inter, int gate_up) {
  const int trailer16 = scales ? PACK_SCALE_BYTES / 16 : 0;
  const int kstages = (kbytes + PACK_KBYTES - 1) / PACK_KBYTES;
  const int64_t rb16 = (int64_t(PACK_ROWS) * kbytes) / 16 + int64_t(kstages) * trailer16;
  const int64_t full_tile16 = int64_t(PACK_ROWS) * PACK_KBYTES / 16 + trailer16;
  const int64_t row16 = kbytes / 16;
  const int scale_cols = (kbytes + 127) / 128;  // E4M3: one byte per element
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n16;
       i += int64_t(gridDim.x) * blockDim.x) {
    const int64_t e = i / per_matrix16;
    const int64_t j = i - e * per_matrix16;
    const int64_t rb = j / rb16;
    const int64_t rem = j - rb * rb16;
    const int64_t kc = rem / full_tile16;
    const int q = int(rem - kc * full_tile16);
    const int nb = min(PACK_KBYTES, kbytes - int(kc) * PACK_KBYTES);
    const int tile_w16 = PACK_ROWS * nb / 16;
    if (q >= tile_w16) {
      // a scale piece: half 0 the first 32 rows' block row, half 1 the last
      const int half = q - tile_w16;
      const int64_t srow = gate_up ? (half * int64_t(inter) + 32 * rb) / 128 : (PACK_ROWS * rb) / 128;
      const float *sm = scales + e * int64_t(rows / 128) * scale_cols + srow * scale_cols;
      float v[4];
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const int64_t c = kc * 4 + t;
        v[t] = c < scale_cols ? sm[c] : 0.f;
      }
      dst[i] = make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]),
                          __float_as_uint(v[3]));
      continue;
    }
    int rit;      // row inside the tile
    int64_t kb;   // byte of K
    if (scales) {
      const int w = q >> 8, mt = (q >> 6) & 3, h = (q >> 5) & 1, lane = q & 31;
      rit = mt * 16 + (lane >> 2) + 8 * h;
      kb = kc * PACK_KBYTES + w * 64 + (lane & 3) * 16;
    } else {
      // [column q / 512][group (q / 64) % 8][row (q / 8) % 8][position q % 8]
      const int r8 = (q >> 3) & 7, pos = q & 7;
      rit = ((q >> 6) & 7) * 8 + r8;
      kb = kc * PACK_KBYTES + (q >> 9) * 128 + (pos ^ r8) * 16;
    }
    int64_t row;
    if (gate_up) row = rit < 32 ? 32 * rb + rit : inter + 32 * rb + (rit - 32);
    else row = int64_t(PACK_ROWS) * rb + rit;
    const int64_t col16 = kb / 16;
    dst[i] = src[e * (int64_t(rows) * row16) + row * row16 + col16];
  }
}

}  // namespace

cudaError_t launch_pack(const void *src, const float *scales, void *dst, int n_matrices, int rows,
                        int kbytes, int inter, bool gate_up, cudaStream_t stream) {
  const int64_t per16 = packed_matrix_bytes(rows, kbytes, scales != nullptr) / 16;
  const int64_t n16 = per16 * n_matrices;
  if (n16 == 0) return cudaSuccess;
  int64_t blocks = (n16 + 255) / 256;
  if (blocks > 65535) blocks = 65535;
  pack_kernel<<<int(blocks), 256, 0, stream>>>(static_cast<const uint4 *>(src), scales,
                                               static_cast<uint4 *>(dst), n16, per16, rows, kbytes, inter,
                                               gate_up ? 1 : 0);
  return cudaGetLastError();
}

}  // namespace moe

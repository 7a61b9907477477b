// pack.cu -- the one-time repacking of expert weights into the tile layout
// the tensor-core expert kernel streams.
//
// An expert matrix (W13 [2I][d] or W2 [d][I], row-major, `es` bytes per
// element, K = row bytes) is cut into tiles of 64 rows x 512 bytes of K (the
// last K tile of a row block may be narrower, a multiple of 64 bytes).  For
// W13 a tile's 64 rows are gate rows [32 rb, 32 rb + 32) followed by the up
// rows I + [32 rb, 32 rb + 32), so that one tile feeds both halves of
// silu(g) * u; for W2 they are rows [64 rb, 64 rb + 64).  Tiles of one row
// block are consecutive (K order); row blocks follow each other, so tile
// (rb, kc) starts at byte rb * 64 * K + kc * 64 * 512 and the packed matrix
// has exactly the size of the original.  Inside a tile the 16-byte pieces
// are ordered [warp w][row tile mt][half h][lane][16 bytes]: lane (g, c) =
// (lane / 4, lane % 4) of warp w takes row 16 mt + g + 8 h, bytes
// 512 kc + 64 w + 16 c .. +15 -- exactly the A-fragment bytes that thread
// needs, read with one lane-contiguous 16-byte load.
#include "kernels.h"
#include "moe_common.cuh"

namespace moe {

namespace {

__global__ void pack_kernel(const uint4 *__restrict__ src, uint4 *__restrict__ dst, int64_t n16,
                            int64_t per_matrix16, int kbytes, int inter, int gate_up) {
  const int64_t tile_row16 = int64_t(PACK_ROWS) * kbytes / 16;   // 16-byte pieces per row block
  const int64_t full_tile16 = int64_t(PACK_ROWS) * PACK_KBYTES / 16;  // 2048
  const int64_t row16 = kbytes / 16;
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n16;
       i += int64_t(gridDim.x) * blockDim.x) {
    const int64_t e = i / per_matrix16;
    const int64_t j = i - e * per_matrix16;
    const int64_t rb = j / tile_row16;
    const int64_t rem = j - rb * tile_row16;
    const int64_t kc = rem / full_tile16;
    const int q = int(rem - kc * full_tile16);
    const int w = q >> 8, mt = (q >> 6) & 3, h = (q >> 5) & 1, lane = q & 31;
    const int rit = mt * 16 + (lane >> 2) + 8 * h;  // row inside the tile
    int64_t row;
    if (gate_up) row = rit < 32 ? 32 * rb + rit : inter + 32 * rb + (rit - 32);
    else row = int64_t(PACK_ROWS) * rb + rit;
    const int64_t col16 = (kc * PACK_KBYTES + w * 64 + (lane & 3) * 16) / 16;
    dst[i] = src[e * per_matrix16 + row * row16 + col16];
  }
}

}  // namespace

cudaError_t launch_pack(const void *src, void *dst, int n_matrices, int rows, int kbytes, int inter,
                        bool gate_up, cudaStream_t stream) {
  const int64_t per16 = int64_t(rows) * kbytes / 16;
  const int64_t n16 = per16 * n_matrices;
  if (n16 == 0) return cudaSuccess;
  int64_t blocks = (n16 + 255) / 256;
  if (blocks > 65535) blocks = 65535;
  pack_kernel<<<int(blocks), 256, 0, stream>>>(static_cast<const uint4 *>(src),
                                               static_cast<uint4 *>(dst), n16, per16, kbytes, inter,
                                               gate_up ? 1 : 0);
  return cudaGetLastError();
}

}  // namespace moe

// The MMA-ready ("tiled") layout of e8m0 block scales used inside the layer.
//
// The tensor cores read a stage's scale factors from tensor memory, where
// tcgen05.cp.32x128b.warpx4 places them from a 512-byte shared-memory chunk
// covering 128 rows x 4 scales (one 128-element K slice): byte
// (r % 32) * 16 + (r / 32) * 4 + kb for row r of the block and 32-element
// block kb of the slice.  The tiled layout stores exactly those chunks,
// contiguous, so one 512-byte bulk copy stages a chunk:
//   chunk (row block rb, K slice kt) at byte (rb * KT + kt) * 512, KT = K / 128.
// Weights [E, N, K]: rb = row / 128 over the E*N rows (N % 128 == 0).
// Grouped activations: each expert's rows start a new row block, so row p of
// expert e is row (p - off_e) % 128 of block tile_base_e + (p - off_e) / 128,
// tile_base_e = sum over e' < e of ceil(count_e' / 128).  Bytes of a block
// past its expert's last row are never written or used.
#pragma once

#include <cstdint>

namespace mxmoe {

// Byte offset of (row, 32-element block j) for a matrix with KT 128-element
// K slices; `row` counts rows of the padded (128-aligned per block) space.
__host__ __device__ inline int64_t tiled_scale_offset(int64_t row, int j, int KT) {
  const int64_t rb = row >> 7;
  const int r = (int)(row & 127);
  return (rb * KT + (j >> 2)) * 512 + (r & 31) * 16 + (r >> 5) * 4 + (j & 3);
}

}  // namespace mxmoe

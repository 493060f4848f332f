// pack.cu -- regroup a row-major weight array into contiguous GEMM tiles.
//
// A matrix of `rows` rows x `row_bytes` bytes is cut into tiles of 128 rows x
// `tile_row_bytes` bytes (the box the grouped GEMMs load per k-block); tile
// (i, j) is written contiguously at byte (i * row_bytes / tile_row_bytes + j)
// * 128 * tile_row_bytes, its rows tile_row_bytes apart.  A pure permutation
// of 16-byte pieces: the values are not touched.
#include <cstdint>

#include "moe_internal.cuh"

namespace beam {
namespace {

__global__ void __launch_bounds__(256) pack_tiles_kernel(const uint4* src, uint4* dst, size_t n16, size_t row_bytes,
                                                         uint32_t tile_row_bytes) {
  const size_t tile_bytes = static_cast<size_t>(kBlockM) * tile_row_bytes;
  const size_t tiles_per_row = row_bytes / tile_row_bytes;
  for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n16;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const size_t d = i * 16;  // destination byte
    const size_t tile = d / tile_bytes, rem = d % tile_bytes;
    const size_t r_in = rem / tile_row_bytes, b_in = rem % tile_row_bytes;
    const size_t ti = tile / tiles_per_row, tj = tile % tiles_per_row;
    const size_t s = (ti * kBlockM + r_in) * row_bytes + tj * tile_row_bytes + b_in;
    dst[i] = src[s / 16];
  }
}

}  // namespace

cudaError_t launch_pack_tiles(const void* src, void* dst, size_t rows, size_t row_bytes, uint32_t tile_row_bytes,
                              int num_sms, cudaStream_t stream) {
  const size_t n16 = rows * row_bytes / 16;
  size_t blocks = (n16 + 255) / 256;
  const size_t cap = static_cast<size_t>(num_sms) * 16;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  pack_tiles_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(static_cast<const uint4*>(src),
                                                                        static_cast<uint4*>(dst), n16, row_bytes,
                                                                        tile_row_bytes);
  return cudaGetLastError();
}

}  // namespace beam

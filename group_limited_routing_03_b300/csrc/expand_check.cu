// expand_check.cu -- test hooks for the NVFP4 paths: the weight expansion
// (the converter warps' own device functions, nvfp4.cuh, over caller-given
// codes and block scales, so that a test can compare every E2M1 x E4M3
// product the grouped GEMMs can form with its exact value) and the W4A4
// activation quantiser (quant.cu's, over caller-given rows).
#include <cuda_runtime.h>

#include "beam_moe.h"
#include "moe_internal.cuh"
#include "nvfp4.cuh"

namespace beam {
namespace {

// Thread b expands block b (16 elements): its 8 code bytes, and its scale,
// found as the converters find it, in byte (b % 4) of the 4-byte scale word
// of four consecutive blocks.
__global__ void __launch_bounds__(256) expand_nvfp4_kernel(const uint8_t* codes, const uint8_t* scales, int n_blocks,
                                                           uint32_t* out) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= n_blocks) return;
  const uint2 w = *reinterpret_cast<const uint2*>(codes + 8 * static_cast<size_t>(b));
  const uint32_t sc4 = *reinterpret_cast<const uint32_t*>(scales + 4 * static_cast<size_t>(b >> 2));
  uint32_t sp[4];
  scales4_to_f16_pairs(sc4, sp);
  uint32_t o[8];
  nvfp4x16_to_f16(w.x, w.y, sp[b & 3], o);
  uint4* dst = reinterpret_cast<uint4*>(out + 8 * static_cast<size_t>(b));
  dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
  dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
}

}  // namespace
}  // namespace beam

extern "C" beam_status_t beam_debug_nvfp4_expand(const uint8_t* codes, const uint8_t* scales, int32_t n_blocks,
                                                 uint16_t* out, void* stream) {
  using namespace beam;
  if (!codes || !scales || !out || n_blocks < 4 || n_blocks % 4 != 0) return BEAM_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(codes) & 15u) || (reinterpret_cast<uintptr_t>(scales) & 15u) ||
      (reinterpret_cast<uintptr_t>(out) & 15u))
    return BEAM_ERR_INVALID_ARG;
  expand_nvfp4_kernel<<<(n_blocks + 255) / 256, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      codes, scales, n_blocks, reinterpret_cast<uint32_t*>(out));
  return cudaGetLastError() == cudaSuccess ? BEAM_OK : BEAM_ERR_CUDA;
}

extern "C" beam_status_t beam_debug_quantize_nvfp4(const void* a, beam_dtype_t a_dtype, int32_t rows, int32_t K,
                                                   uint8_t* codes, uint8_t* scales, float* global, uint16_t* values,
                                                   void* stream) {
  using namespace beam;
  if (!a || !codes || !scales || !global || !values || rows < 1 || K < 16 || K % 16 != 0) return BEAM_ERR_INVALID_ARG;
  if (a_dtype != BEAM_F32 && a_dtype != BEAM_BF16) return BEAM_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(a) & 15u) || (reinterpret_cast<uintptr_t>(values) & 15u) ||
      (reinterpret_cast<uintptr_t>(global) & 3u))
    return BEAM_ERR_INVALID_ARG;
  return launch_quantize_a4(a, a_dtype == BEAM_BF16, rows, K, codes, scales, global, reinterpret_cast<__half*>(values),
                            static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? BEAM_OK
             : BEAM_ERR_CUDA;
}

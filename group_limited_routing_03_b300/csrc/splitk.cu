// splitk.cu -- the finishing step of a grouped GEMM whose K range was split
// across CTAs (few units for many SMs, e.g. a dense MLP at decode size).
//
// The GEMM's parts left FP32 partial sums (row scales applied) in planes of
// [R, N]; this kernel adds the parts in part order (a fixed order, so the
// result does not depend on scheduling) and applies what the GEMM epilogue
// applies to a whole sum: for gate/up the SwiGLU product silu(gate) * up in
// FP32 (Beam launch post, section "Residual Stream": the SwiGLU product is
// computed in FP32), then the BF16 rounding of the stored result.
#include <cuda_bf16.h>

#include "moe_internal.cuh"

namespace beam {
namespace {

template <int kMode>
__global__ void __launch_bounds__(256) splitk_finish_kernel(const float* partial, int k_splits, size_t plane,
                                                            size_t n4, __nv_bfloat16* out) {
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n4;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < k_splits; ++s) {
      const float4* base = reinterpret_cast<const float4*>(partial + static_cast<size_t>(s) * (kMode == 0 ? 2 : 1) * plane);
      const float4 v = base[i];
      a.x += v.x, a.y += v.y, a.z += v.z, a.w += v.w;
      if (kMode == 0) {
        const float4 w = base[plane / 4 + i];
        b.x += w.x, b.y += w.y, b.z += w.z, b.w += w.w;
      }
    }
    float r[4] = {a.x, a.y, a.z, a.w};
    if (kMode == 0) {
      const float u[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) r[j] = __fdividef(r[j], 1.0f + __expf(-r[j])) * u[j];
    }
    __nv_bfloat162 q0 = __floats2bfloat162_rn(r[0], r[1]), q1 = __floats2bfloat162_rn(r[2], r[3]);
    uint2 o;
    o.x = *reinterpret_cast<uint32_t*>(&q0);
    o.y = *reinterpret_cast<uint32_t*>(&q1);
    reinterpret_cast<uint2*>(out)[i] = o;
  }
}

}  // namespace

cudaError_t launch_splitk_finish(int mode, const float* partial, int k_splits, int R, int N, __nv_bfloat16* out,
                                 cudaStream_t stream) {
  const size_t plane = static_cast<size_t>(R) * N;
  const size_t n4 = plane / 4;
  size_t blocks = (n4 + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  if (blocks < 1) blocks = 1;
  if (mode == 0)
    splitk_finish_kernel<0><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(partial, k_splits, plane, n4, out);
  else
    splitk_finish_kernel<1><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(partial, k_splits, plane, n4, out);
  return cudaGetLastError();
}

}  // namespace beam

// combine.cu -- weighted un-permute of the expert outputs.
//
// Beam launch post, section "Mixture of Experts": the expert outputs are
// combined with the normalised router weights (already scaled by 2.5 by the
// router); there is no shared expert.  y[t, :] = sum_k w[t,k] * yr[pos[t*8+k], :],
// FP32 accumulation in k order 0..7.  CTA (t, j) covers the 8-element groups
// c = 128 j + threadIdx.x + 128 gridDim.y i of token t (16-byte loads of the
// BF16 expert outputs); for few tokens (decode) gridDim.y splits each row so
// the work still spreads over many SMs, for many tokens one CTA per token.
#include <cuda_bf16.h>

#include "moe_internal.cuh"
#include "tc.cuh"

namespace beam {
namespace {

template <bool kBf16Out>
__global__ void __launch_bounds__(128) combine_kernel(const __nv_bfloat16* yr, const int32_t* pos, const float* w,
                                                      int H, void* y) {
  __shared__ int ps[kTopK];
  __shared__ float ws[kTopK];
  const int t = blockIdx.x;

  if (threadIdx.x < kTopK) {
    ps[threadIdx.x] = pos[static_cast<size_t>(t) * kTopK + threadIdx.x];
    ws[threadIdx.x] = w[static_cast<size_t>(t) * kTopK + threadIdx.x];
  }
  __syncthreads();
  for (int c = blockIdx.y * blockDim.x + threadIdx.x; c < H / 8; c += gridDim.y * blockDim.x) {
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
#pragma unroll
    for (int k = 0; k < kTopK; ++k) {
      if (ps[k] < 0) continue;
      const uint4 raw = *reinterpret_cast<const uint4*>(yr + static_cast<size_t>(ps[k]) * H + c * 8);
      const __nv_bfloat162* v = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(v[i]);
        acc[2 * i] = fmaf(ws[k], f.x, acc[2 * i]);
        acc[2 * i + 1] = fmaf(ws[k], f.y, acc[2 * i + 1]);
      }
    }
    const size_t o = static_cast<size_t>(t) * H + c * 8;
    if (kBf16Out) {
      uint4 out;
      __nv_bfloat162 q[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) q[i] = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
      out.x = *reinterpret_cast<uint32_t*>(&q[0]);
      out.y = *reinterpret_cast<uint32_t*>(&q[1]);
      out.z = *reinterpret_cast<uint32_t*>(&q[2]);
      out.w = *reinterpret_cast<uint32_t*>(&q[3]);
      *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(y) + o) = out;
    } else {
      float4* dst = reinterpret_cast<float4*>(static_cast<float*>(y) + o);
      dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
      dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    }
  }
}

// One CTA waits on an mbarrier nothing arrives on; the bounded wait gives up,
// records the timeout in the status word and the kernel returns normally.
__global__ void debug_timeout_kernel(uint32_t* status, uint64_t timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    mbar_wait(&bar, 0, timeout_ns, nullptr, status, kWhereDebug);
    // Complete the barrier's phase so it is not left pending.
    mbar_arrive(&bar);
  }
}

}  // namespace

cudaError_t launch_combine(const __nv_bfloat16* yr, const int32_t* pos, const float* w, int T, int H, void* y,
                           bool y_bf16, cudaStream_t stream) {
  const dim3 grid(T, T >= 1024 ? 1 : (H / 8 + 127) / 128);
  if (y_bf16)
    combine_kernel<true><<<grid, 128, 0, stream>>>(yr, pos, w, H, y);
  else
    combine_kernel<false><<<grid, 128, 0, stream>>>(yr, pos, w, H, y);
  return cudaGetLastError();
}

cudaError_t launch_debug_timeout(uint32_t* status, uint64_t timeout_ns, cudaStream_t stream) {
  debug_timeout_kernel<<<1, 32, 0, stream>>>(status, timeout_ns);
  return cudaGetLastError();
}

}  // namespace beam

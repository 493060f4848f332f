// quant.cu -- run-time E4M3 quantisation of the grouped GEMMs' inputs for FP8
// expert weights.
//
// The Beam launch post (section "Mixture of Experts") lists an FP8 checkpoint
// beside BF16 and NVFP4 without its layout.  The library reads it as E4M3
// weights with an FP32 scale per output row and runs the GEMMs on E4M3 x E4M3
// tensor cores, so the activations are quantised per row at run time:
//   scale = amax(row) / 448 (FP32 division; 1 when that is 0),
//   code  = E4M3(a / scale) (FP32 division, round to nearest even, saturating
//           at +-448, the largest finite E4M3 value).
// Both kernels give one warp a row: pass 1 finds the row's largest magnitude
// (a warp max), pass 2 re-reads the row (from L1) and converts 16 elements
// per lane and step into one 16-byte store.
//
// NVFP4 expert weights run on FP16 tensor cores (their E2M1 x E4M3 values
// are exact in FP16, and the MMA takes A and B of one type), so the GEMM
// inputs go to FP16 with a power-of-two scale per row, which keeps them
// exactly the BF16 values the BF16 weight path multiplies:
//   a = BF16 value of the input (x as given, or rounded to BF16 when FP32;
//       h as stored), E = exponent of the row's largest |a| (2^E <= amax <
//       2^(E+1)), k = 15 - E (clamped to [-100, 100]; 0 for a zero row),
//   code = FP16(a * 2^k) (nearest even), row scale = 2^-k (FP32).
// a * 2^k is exact in FP32; it is exact in FP16 when |a * 2^k| <= 65504
// (always: a BF16 amax scaled into [2^15, 2^16) is at most 65280) and a's
// lowest significand bit is at least 2^-24 after scaling, which holds for
// every |a| >= 2^(E-32) (a row spanning fewer than 32 binades).  Smaller
// values round to FP16 subnormals (absolute error <= 2^(E-40)).  The GEMM
// epilogue multiplies the FP32 sums by the row scale, undoing the exact
// power of two.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "moe_internal.cuh"
#include "tc.cuh"

namespace beam {
namespace {

constexpr int kWarpsPerCta = 8;

// 16 consecutive elements of a row, as FP32.
template <bool kBf16>
__device__ __forceinline__ void load16(const void* row, int g, float* v) {
  if (kBf16) {
    const uint4* src = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(row) + 16 * g);
    const uint4 r0 = src[0], r1 = src[1];
    const __nv_bfloat162* a = reinterpret_cast<const __nv_bfloat162*>(&r0);
    const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&r1);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 fa = __bfloat1622float2(a[i]), fb = __bfloat1622float2(b[i]);
      v[2 * i] = fa.x, v[2 * i + 1] = fa.y, v[8 + 2 * i] = fb.x, v[8 + 2 * i + 1] = fb.y;
    }
  } else {
    const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(row) + 16 * g);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float4 f = src[i];
      v[4 * i] = f.x, v[4 * i + 1] = f.y, v[4 * i + 2] = f.z, v[4 * i + 3] = f.w;
    }
  }
}

template <bool kBf16>
__device__ __forceinline__ float row_scale(const void* row, int groups, int lane) {
  float amax = 0.0f;
  for (int g = lane; g < groups; g += 32) {
    float v[16];
    load16<kBf16>(row, g, v);
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float s = __fdiv_rn(amax, 448.0f);
  return s == 0.0f ? 1.0f : s;
}

// 16 elements / scale -> 16 E4M3 codes (element i in byte i).
template <bool kBf16>
__device__ __forceinline__ uint4 codes16(const void* row, int g, float s) {
  float v[16];
  load16<kBf16>(row, g, v);
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_fp8x2_storage_t lo =
        __nv_cvt_float2_to_fp8x2(make_float2(__fdiv_rn(v[4 * i], s), __fdiv_rn(v[4 * i + 1], s)), __NV_SATFINITE,
                                 __NV_E4M3);
    const __nv_fp8x2_storage_t hi =
        __nv_cvt_float2_to_fp8x2(make_float2(__fdiv_rn(v[4 * i + 2], s), __fdiv_rn(v[4 * i + 3], s)),
                                 __NV_SATFINITE, __NV_E4M3);
    w[i] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// One warp per token: its codes go to the token's kRoutes route rows (8 for
// the MoE block, at pos[t*8 + k], skipping routes whose expert id was out of
// range (pos < 0); 1 for the dense MLP, row t).
template <bool kBf16, int kRoutes>
__global__ void __launch_bounds__(32 * kWarpsPerCta) gather_q8_kernel(const void* x, int H, const int32_t* pos,
                                                                      int T, uint8_t* xq, float* xs, uint32_t* status) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;
  const void* row = kBf16 ? static_cast<const void*>(static_cast<const __nv_bfloat16*>(x) + static_cast<size_t>(t) * H)
                          : static_cast<const void*>(static_cast<const float*>(x) + static_cast<size_t>(t) * H);
  const int groups = H / 16;
  const float s = row_scale<kBf16>(row, groups, lane);
  int p[kRoutes];
#pragma unroll
  for (int k = 0; k < kRoutes; ++k) {
    p[k] = kRoutes == 1 ? t : __ldg(&pos[static_cast<size_t>(t) * kTopK + k]);
    if (p[k] >= 0 && !dcheck(p[k] < T * kRoutes, lane == 0 ? status : nullptr, kCheckQ8Pos)) p[k] = -1;
  }
  if (lane < kRoutes && p[lane] >= 0) xs[p[lane]] = s;
  for (int g = lane; g < groups; g += 32) {
    const uint4 c = codes16<kBf16>(row, g, s);
#pragma unroll
    for (int k = 0; k < kRoutes; ++k)
      if (p[k] >= 0) *reinterpret_cast<uint4*>(xq + static_cast<size_t>(p[k]) * H + 16 * g) = c;
  }
}

__global__ void __launch_bounds__(32 * kWarpsPerCta) quantize_rows_kernel(const __nv_bfloat16* h, int R, int I,
                                                                          uint8_t* hq, float* hs) {
  const int lane = threadIdx.x & 31;
  const int r = blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
  if (r >= R) return;
  const void* row = h + static_cast<size_t>(r) * I;
  const int groups = I / 16;
  const float s = row_scale<true>(row, groups, lane);
  if (lane == 0) hs[r] = s;
  for (int g = lane; g < groups; g += 32)
    *reinterpret_cast<uint4*>(hq + static_cast<size_t>(r) * I + 16 * g) = codes16<true>(row, g, s);
}

// ---------------------------------------------------------------- FP16 rows
// 16 elements as the BF16 values the GEMM multiplies (FP32 x rounded).
template <bool kBf16>
__device__ __forceinline__ void load16_bf16_values(const void* row, int g, float* v) {
  load16<kBf16>(row, g, v);
  if (!kBf16) {
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __bfloat162float(__float2bfloat16_rn(v[i]));
  }
}

// k of the row (see the file comment) from its largest magnitude.
__device__ __forceinline__ int pow2_shift(float amax) {
  if (!(amax > 0.0f)) return 0;
  const int E = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFFu) - 127;
  const int k = 15 - E;
  return k < -100 ? -100 : (k > 100 ? 100 : k);
}
__device__ __forceinline__ float pow2f(int k) { return __uint_as_float(static_cast<uint32_t>(k + 127) << 23); }

template <bool kBf16>
__device__ __forceinline__ int row_shift16(const void* row, int groups, int lane) {
  float amax = 0.0f;
  for (int g = lane; g < groups; g += 32) {
    float v[16];
    load16_bf16_values<kBf16>(row, g, v);
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  return pow2_shift(amax);
}

// 16 elements times 2^k -> 16 FP16 (element i in half i of the 32 bytes).
template <bool kBf16>
__device__ __forceinline__ void f16x16(const void* row, int g, float up, uint4& lo, uint4& hi) {
  float v[16];
  load16_bf16_values<kBf16>(row, g, v);
  uint32_t w[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const __half2 q = __floats2half2_rn(v[2 * i] * up, v[2 * i + 1] * up);
    w[i] = *reinterpret_cast<const uint32_t*>(&q);
  }
  lo = make_uint4(w[0], w[1], w[2], w[3]);
  hi = make_uint4(w[4], w[5], w[6], w[7]);
}

// One warp per token: its FP16 row goes to the token's kRoutes route rows
// (pos[t*8 + k]; routes whose expert id was out of range have pos < 0 and
// are skipped; kRoutes = 1: row t), its row scale 2^-k beside them.
template <bool kBf16, int kRoutes>
__global__ void __launch_bounds__(32 * kWarpsPerCta) gather_f16_kernel(const void* x, int H, const int32_t* pos,
                                                                       int T, __half* xh, float* xs, uint32_t* status) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;
  const void* row = kBf16 ? static_cast<const void*>(static_cast<const __nv_bfloat16*>(x) + static_cast<size_t>(t) * H)
                          : static_cast<const void*>(static_cast<const float*>(x) + static_cast<size_t>(t) * H);
  const int groups = H / 16;
  const int k = row_shift16<kBf16>(row, groups, lane);
  const float up = pow2f(k);
  int p[kRoutes];
#pragma unroll
  for (int r = 0; r < kRoutes; ++r) {
    p[r] = kRoutes == 1 ? t : __ldg(&pos[static_cast<size_t>(t) * kTopK + r]);
    if (p[r] >= 0 && !dcheck(p[r] < T * kRoutes, lane == 0 ? status : nullptr, kCheckF16Pos)) p[r] = -1;
  }
  if (lane < kRoutes && p[lane] >= 0) xs[p[lane]] = pow2f(-k);
  for (int g = lane; g < groups; g += 32) {
    uint4 lo, hi;
    f16x16<kBf16>(row, g, up, lo, hi);
#pragma unroll
    for (int r = 0; r < kRoutes; ++r) {
      if (p[r] < 0) continue;
      uint4* dst = reinterpret_cast<uint4*>(xh + static_cast<size_t>(p[r]) * H + 16 * g);
      dst[0] = lo;
      dst[1] = hi;
    }
  }
}

// Rows of h (BF16 [R, I]) to FP16 in place, row scale 2^-k in hs[r]: every
// lane reads its elements of the row (for the warp's maximum) before any
// lane writes, and then rewrites only the elements it read.
__global__ void __launch_bounds__(32 * kWarpsPerCta) rows_to_f16_kernel(void* h, int R, int I, float* hs) {
  const int lane = threadIdx.x & 31;
  const int r = blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
  if (r >= R) return;
  void* row = static_cast<__nv_bfloat16*>(h) + static_cast<size_t>(r) * I;
  const int groups = I / 16;
  const int k = row_shift16<true>(row, groups, lane);
  const float up = pow2f(k);
  if (lane == 0) hs[r] = pow2f(-k);
  for (int g = lane; g < groups; g += 32) {
    uint4 lo, hi;
    f16x16<true>(row, g, up, lo, hi);
    uint4* dst = reinterpret_cast<uint4*>(static_cast<__half*>(row) + 16 * g);
    dst[0] = lo;
    dst[1] = hi;
  }
}

}  // namespace

cudaError_t launch_gather_f16(const void* x, bool x_bf16, int H, const int32_t* pos, int T, __half* xh, float* xs,
                              uint32_t* status, cudaStream_t stream) {
  const int warps = T <= 4096 ? 2 : kWarpsPerCta;
  const int grid = (T + warps - 1) / warps;
  const int threads = 32 * warps;
  if (pos == nullptr) {  // dense MLP: row t to row t
    if (x_bf16)
      gather_f16_kernel<true, 1><<<grid, threads, 0, stream>>>(x, H, pos, T, xh, xs, status);
    else
      gather_f16_kernel<false, 1><<<grid, threads, 0, stream>>>(x, H, pos, T, xh, xs, status);
  } else if (x_bf16) {
    gather_f16_kernel<true, kTopK><<<grid, threads, 0, stream>>>(x, H, pos, T, xh, xs, status);
  } else {
    gather_f16_kernel<false, kTopK><<<grid, threads, 0, stream>>>(x, H, pos, T, xh, xs, status);
  }
  return cudaGetLastError();
}

cudaError_t launch_rows_to_f16(void* h, int R, int I, float* hs, cudaStream_t stream) {
  const int grid = (R + kWarpsPerCta - 1) / kWarpsPerCta;
  rows_to_f16_kernel<<<grid, 32 * kWarpsPerCta, 0, stream>>>(h, R, I, hs);
  return cudaGetLastError();
}

cudaError_t launch_gather_q8(const void* x, bool x_bf16, int H, const int32_t* pos, int T, uint8_t* xq, float* xs,
                             uint32_t* status, cudaStream_t stream) {
  // few tokens (decode): two warps per CTA, so the rows spread over more SMs
  const int warps = T <= 4096 ? 2 : kWarpsPerCta;
  const int grid = (T + warps - 1) / warps;
  const int threads = 32 * warps;
  if (pos == nullptr) {  // dense MLP: row t to row t
    if (x_bf16)
      gather_q8_kernel<true, 1><<<grid, threads, 0, stream>>>(x, H, pos, T, xq, xs, status);
    else
      gather_q8_kernel<false, 1><<<grid, threads, 0, stream>>>(x, H, pos, T, xq, xs, status);
  } else if (x_bf16) {
    gather_q8_kernel<true, kTopK><<<grid, threads, 0, stream>>>(x, H, pos, T, xq, xs, status);
  } else {
    gather_q8_kernel<false, kTopK><<<grid, threads, 0, stream>>>(x, H, pos, T, xq, xs, status);
  }
  return cudaGetLastError();
}

cudaError_t launch_quantize_rows(const __nv_bfloat16* h, int R, int I, uint8_t* hq, float* hs, cudaStream_t stream) {
  const int grid = (R + kWarpsPerCta - 1) / kWarpsPerCta;
  quantize_rows_kernel<<<grid, 32 * kWarpsPerCta, 0, stream>>>(h, R, I, hq, hs);
  return cudaGetLastError();
}

}  // namespace beam

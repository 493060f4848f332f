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
//
// NVFP4 activations (W4A4, BEAM_NVFP4_A4): the launch post names NVFP4 as a
// weight format; for activations the library applies the weights' recipe per
// GEMM input row at run time (x as given, FP32 or BF16; h as stored, BF16):
//   g   = amax(row) / (6 * 448) in FP32 (1 when that is 0),
//   s_b = E4M3((bmax_b / 6) / g) for each block b of 16 elements (FP32
//         divisions, nearest even, saturating at 448),
//   q   = E2M1(a / (s_b * g)) for each element (FP32 product and division;
//         nearest of 0, 0.5, 1, 1.5, 2, 3, 4, 6, ties to the even code,
//         saturating at 6; code 0 when s_b * g is 0).
// The element stands for q * s_b * g.  The GEMM reads q * s_b, exact in FP16
// (at most 2 + 4 significant bits, magnitude 0 or in [2^-10, 2688]), and the
// epilogue multiplies the FP32 sums by g, the row scale, so the products the
// tensor cores form are exactly those of the two NVFP4 operands.
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

// ------------------------------------------------------------- NVFP4 rows
// Nearest E2M1 code of e, ties to the even code (the code's low bit is its
// mantissa bit), magnitudes above 6 to 6; sign in bit 3.  A NaN gives 0.
__device__ __forceinline__ uint32_t e2m1_code(float e) {
  const float m = fabsf(e);
  const uint32_t c = static_cast<uint32_t>(m > 0.25f) + static_cast<uint32_t>(m >= 0.75f) +
                     static_cast<uint32_t>(m > 1.25f) + static_cast<uint32_t>(m >= 1.75f) +
                     static_cast<uint32_t>(m > 2.5f) + static_cast<uint32_t>(m >= 3.5f) +
                     static_cast<uint32_t>(m > 5.0f);
  return (signbit(e) ? 8u : 0u) | c;
}

// The E2M1 value of a code (bit 3 the sign).
__device__ __forceinline__ float e2m1_value(uint32_t c) {
  const uint32_t m = c & 7u;  // 0, 0.5, 1, 1.5 (m / 2), then 2, 3, 4, 6
  const float v = m < 4u ? 0.5f * static_cast<float>(m)
                         : static_cast<float>(2u << ((m - 4u) >> 1)) * ((m & 1u) ? 1.5f : 1.0f);
  return (c & 8u) ? -v : v;
}

// The global scale g of a row from its largest magnitude.
__device__ __forceinline__ float a4_global(float amax) {
  const float g = __fdiv_rn(amax, 6.0f * 448.0f);
  return g == 0.0f ? 1.0f : g;
}

// One block of 16 elements (v) of a row with global scale g: its E4M3 scale
// code, its 16 E2M1 codes (element i in bits 4i..4i+3) and the 16 FP16 values
// q * s the GEMM reads.
__device__ __forceinline__ void a4_block(const float (&v)[16], float g, uint32_t& scale_code, uint64_t& codes,
                                         uint32_t (&f16)[8]) {
  float bmax = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) bmax = fmaxf(bmax, fabsf(v[i]));
  const float q = __fdiv_rn(__fdiv_rn(bmax, 6.0f), g);
  scale_code = static_cast<uint32_t>(__nv_cvt_float_to_fp8(q, __NV_SATFINITE, __NV_E4M3));
  const float sv = __half2float(__half(__nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(scale_code), __NV_E4M3)));
  const float d = __fmul_rn(sv, g);
  codes = 0;
#pragma unroll
  for (int i = 0; i < 16; i += 2) {
    uint32_t c0 = 0u, c1 = 0u;
    if (sv != 0.0f && d != 0.0f) {
      c0 = e2m1_code(__fdiv_rn(v[i], d));
      c1 = e2m1_code(__fdiv_rn(v[i + 1], d));
    }
    codes |= static_cast<uint64_t>(c0 | (c1 << 4)) << (4 * i);
    const __half2 h = __floats2half2_rn(__fmul_rn(e2m1_value(c0), sv), __fmul_rn(e2m1_value(c1), sv));
    f16[i / 2] = *reinterpret_cast<const uint32_t*>(&h);
  }
}

template <bool kBf16>
__device__ __forceinline__ float row_amax(const void* row, int groups, int lane) {
  float amax = 0.0f;
  for (int g = lane; g < groups; g += 32) {
    float v[16];
    load16<kBf16>(row, g, v);
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  return amax;
}

// One warp per token: the token's NVFP4 row (as FP16 q * s) goes to its
// kRoutes route rows (pos[t*8 + k]; pos < 0 skipped; kRoutes = 1: row t),
// its global scale g beside them.
template <bool kBf16, int kRoutes>
__global__ void __launch_bounds__(32 * kWarpsPerCta) gather_a4_kernel(const void* x, int H, const int32_t* pos,
                                                                      int T, __half* xh, float* xs, uint32_t* status) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;
  const void* row = kBf16 ? static_cast<const void*>(static_cast<const __nv_bfloat16*>(x) + static_cast<size_t>(t) * H)
                          : static_cast<const void*>(static_cast<const float*>(x) + static_cast<size_t>(t) * H);
  const int groups = H / 16;
  const float g = a4_global(row_amax<kBf16>(row, groups, lane));
  int p[kRoutes];
#pragma unroll
  for (int r = 0; r < kRoutes; ++r) {
    p[r] = kRoutes == 1 ? t : __ldg(&pos[static_cast<size_t>(t) * kTopK + r]);
    if (p[r] >= 0 && !dcheck(p[r] < T * kRoutes, lane == 0 ? status : nullptr, kCheckF16Pos)) p[r] = -1;
  }
  if (lane < kRoutes && p[lane] >= 0) xs[p[lane]] = g;
  for (int b = lane; b < groups; b += 32) {
    float v[16];
    load16<kBf16>(row, b, v);
    uint32_t sc, f16[8];
    uint64_t codes;
    a4_block(v, g, sc, codes, f16);
    const uint4 lo = make_uint4(f16[0], f16[1], f16[2], f16[3]), hi = make_uint4(f16[4], f16[5], f16[6], f16[7]);
#pragma unroll
    for (int r = 0; r < kRoutes; ++r) {
      if (p[r] < 0) continue;
      uint4* dst = reinterpret_cast<uint4*>(xh + static_cast<size_t>(p[r]) * H + 16 * b);
      dst[0] = lo;
      dst[1] = hi;
    }
  }
}

// Rows of h (BF16 [R, I]) to NVFP4 in place (as FP16 q * s), global scale in
// hs[r]: every lane reads the whole row's maximum before any lane writes, and
// then rewrites only the blocks it reads.
__global__ void __launch_bounds__(32 * kWarpsPerCta) rows_to_a4_kernel(void* h, int R, int I, float* hs) {
  const int lane = threadIdx.x & 31;
  const int r = blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
  if (r >= R) return;
  void* row = static_cast<__nv_bfloat16*>(h) + static_cast<size_t>(r) * I;
  const int groups = I / 16;
  const float g = a4_global(row_amax<true>(row, groups, lane));
  if (lane == 0) hs[r] = g;
  for (int b = lane; b < groups; b += 32) {
    float v[16];
    load16<true>(row, b, v);
    uint32_t sc, f16[8];
    uint64_t codes;
    a4_block(v, g, sc, codes, f16);
    uint4* dst = reinterpret_cast<uint4*>(static_cast<__half*>(row) + 16 * b);
    dst[0] = make_uint4(f16[0], f16[1], f16[2], f16[3]);
    dst[1] = make_uint4(f16[4], f16[5], f16[6], f16[7]);
  }
}

// Test hook: the same quantisation of rows [rows, K] into codes (one per
// byte, [rows, K]), block scales [rows, K/16], global scales [rows] and the
// FP16 values [rows, K].
template <bool kBf16>
__global__ void __launch_bounds__(32 * kWarpsPerCta) quantize_a4_kernel(const void* a, int rows, int K, uint8_t* codes,
                                                                        uint8_t* scales, float* global, __half* values) {
  const int lane = threadIdx.x & 31;
  const int r = blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
  if (r >= rows) return;
  const void* row = kBf16 ? static_cast<const void*>(static_cast<const __nv_bfloat16*>(a) + static_cast<size_t>(r) * K)
                          : static_cast<const void*>(static_cast<const float*>(a) + static_cast<size_t>(r) * K);
  const int groups = K / 16;
  const float g = a4_global(row_amax<kBf16>(row, groups, lane));
  if (lane == 0) global[r] = g;
  for (int b = lane; b < groups; b += 32) {
    float v[16];
    load16<kBf16>(row, b, v);
    uint32_t sc, f16[8];
    uint64_t c;
    a4_block(v, g, sc, c, f16);
    scales[static_cast<size_t>(r) * groups + b] = static_cast<uint8_t>(sc);
    uint8_t* cd = codes + static_cast<size_t>(r) * K + 16 * b;
#pragma unroll
    for (int i = 0; i < 16; ++i) cd[i] = static_cast<uint8_t>((c >> (4 * i)) & 0xFu);
    uint4* dst = reinterpret_cast<uint4*>(values + static_cast<size_t>(r) * K + 16 * b);
    dst[0] = make_uint4(f16[0], f16[1], f16[2], f16[3]);
    dst[1] = make_uint4(f16[4], f16[5], f16[6], f16[7]);
  }
}

}  // namespace

cudaError_t launch_gather_a4(const void* x, bool x_bf16, int H, const int32_t* pos, int T, __half* xh, float* xs,
                             uint32_t* status, cudaStream_t stream) {
  const int warps = T <= 4096 ? 2 : kWarpsPerCta;
  const int grid = (T + warps - 1) / warps;
  const int threads = 32 * warps;
  if (pos == nullptr) {  // dense MLP: row t to row t
    if (x_bf16)
      gather_a4_kernel<true, 1><<<grid, threads, 0, stream>>>(x, H, pos, T, xh, xs, status);
    else
      gather_a4_kernel<false, 1><<<grid, threads, 0, stream>>>(x, H, pos, T, xh, xs, status);
  } else if (x_bf16) {
    gather_a4_kernel<true, kTopK><<<grid, threads, 0, stream>>>(x, H, pos, T, xh, xs, status);
  } else {
    gather_a4_kernel<false, kTopK><<<grid, threads, 0, stream>>>(x, H, pos, T, xh, xs, status);
  }
  return cudaGetLastError();
}

cudaError_t launch_rows_to_a4(void* h, int R, int I, float* hs, cudaStream_t stream) {
  const int grid = (R + kWarpsPerCta - 1) / kWarpsPerCta;
  rows_to_a4_kernel<<<grid, 32 * kWarpsPerCta, 0, stream>>>(h, R, I, hs);
  return cudaGetLastError();
}

cudaError_t launch_quantize_a4(const void* a, bool a_bf16, int rows, int K, uint8_t* codes, uint8_t* scales,
                               float* global, __half* values, cudaStream_t stream) {
  const int grid = (rows + kWarpsPerCta - 1) / kWarpsPerCta;
  if (a_bf16)
    quantize_a4_kernel<true><<<grid, 32 * kWarpsPerCta, 0, stream>>>(a, rows, K, codes, scales, global, values);
  else
    quantize_a4_kernel<false><<<grid, 32 * kWarpsPerCta, 0, stream>>>(a, rows, K, codes, scales, global, values);
  return cudaGetLastError();
}

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

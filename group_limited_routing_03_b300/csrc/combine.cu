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
                                                      int H, void* y, uint32_t* status) {
  __shared__ int ps[kTopK];
  __shared__ float ws[kTopK];
  const int t = blockIdx.x;

  if (threadIdx.x < kTopK) {
    int q = pos[static_cast<size_t>(t) * kTopK + threadIdx.x];
    // route rows: T * 8, one CTA row per token
    if (q >= 0 && !dcheck(q < static_cast<int>(gridDim.x) * kTopK, blockIdx.y == 0 ? status : nullptr, kCheckCombinePos))
      q = -1;
    ps[threadIdx.x] = q;
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

// Combine fused with the post-norm residual update of the Beam post's section
// "Residual Stream": the block's output y (the weighted sum above, kept in
// FP32) is RMS-normalised with the learned scale g and added to the stream,
//   out[t,:] = keep * stream[t,:] + add * g * y[t,:] / sqrt(mean(y[t,:]^2) + eps),
// keep = sqrt((k-1)/k), add = 1/sqrt(k) at step k.  The row's sum of squares
// needs all of y[t,:] before anything is written: each CTA keeps its part of
// the row in shared memory, and when a row is split over the kClusterY CTAs of
// a cluster (few tokens) their partial sums are exchanged through distributed
// shared memory and added in rank order, so every CTA of the row uses the
// same normaliser.  `out` may be `stream` itself (each element is read and
// written by one thread); `y_out` (nullable) receives the plain combine.
template <bool kBf16, int kClusterY>
__global__ void __launch_bounds__(128) combine_residual_kernel(const __nv_bfloat16* yr, const int32_t* pos,
                                                               const float* w, int H, ResidualParams r,
                                                               void* y_out, uint32_t* status) {
  extern __shared__ float4 ys4[];  // this CTA's part of y[t,:], 8 floats per group
  float* ys = reinterpret_cast<float*>(ys4);
  __shared__ int ps[kTopK];
  __shared__ float ws[kTopK];
  __shared__ float red[4];
  __shared__ float row_ss;
  const int t = blockIdx.x;
  const int rank = kClusterY > 1 ? static_cast<int>(cluster_ctarank()) : 0;
  const int G = H / 8, step = kClusterY * 128;

  if (threadIdx.x < kTopK) {
    int q = pos[static_cast<size_t>(t) * kTopK + threadIdx.x];
    if (q >= 0 && !dcheck(q < static_cast<int>(gridDim.x) * kTopK, rank == 0 ? status : nullptr, kCheckResidualPos))
      q = -1;
    ps[threadIdx.x] = q;
    ws[threadIdx.x] = w[static_cast<size_t>(t) * kTopK + threadIdx.x];
  }
  __syncthreads();
  float ss = 0.0f;
  for (int c = rank * 128 + threadIdx.x, slot = threadIdx.x; c < G; c += step, slot += 128) {
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
#pragma unroll
    for (int i = 0; i < 8; ++i) ss = fmaf(acc[i], acc[i], ss);
    ys4[2 * slot] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    ys4[2 * slot + 1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x == 0) row_ss = (red[0] + red[1]) + (red[2] + red[3]);
  if (kClusterY > 1) {
    cluster_sync();  // every CTA's row_ss written and visible
    if (threadIdx.x == 0) {
      float total = 0.0f;
      for (int q = 0; q < kClusterY; ++q) total += ld_shared_cluster_f32(mapa_shared(&row_ss, q));
      red[0] = total;
    }
    cluster_sync();  // no CTA leaves (or reuses row_ss) while a peer still reads it
    if (threadIdx.x == 0) row_ss = red[0];
  }
  __syncthreads();
  const float scale = rsqrtf(row_ss / static_cast<float>(H) + r.eps) * r.add;

  for (int c = rank * 128 + threadIdx.x, slot = threadIdx.x; c < G; c += step, slot += 128) {
    float acc[8];
    const float4 a0 = ys4[2 * slot], a1 = ys4[2 * slot + 1];
    acc[0] = a0.x, acc[1] = a0.y, acc[2] = a0.z, acc[3] = a0.w;
    acc[4] = a1.x, acc[5] = a1.y, acc[6] = a1.z, acc[7] = a1.w;
    const float4 g0 = *reinterpret_cast<const float4*>(r.norm_w + c * 8);
    const float4 g1 = *reinterpret_cast<const float4*>(r.norm_w + c * 8 + 4);
    const float g[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
    float s[8];
    const size_t o = static_cast<size_t>(t) * H + c * 8;
    if (kBf16) {
      const uint4 raw = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(r.stream) + o);
      const __nv_bfloat162* v = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(v[i]);
        s[2 * i] = f.x, s[2 * i + 1] = f.y;
      }
    } else {
      const float4 s0 = *reinterpret_cast<const float4*>(static_cast<const float*>(r.stream) + o);
      const float4 s1 = *reinterpret_cast<const float4*>(static_cast<const float*>(r.stream) + o + 4);
      s[0] = s0.x, s[1] = s0.y, s[2] = s0.z, s[3] = s0.w, s[4] = s1.x, s[5] = s1.y, s[6] = s1.z, s[7] = s1.w;
    }
    float n[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) n[i] = fmaf(r.keep, s[i], acc[i] * scale * g[i]);
    if (kBf16) {
      __nv_bfloat162 q[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) q[i] = __floats2bfloat162_rn(n[2 * i], n[2 * i + 1]);
      *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(r.out) + o) = *reinterpret_cast<const uint4*>(q);
      if (y_out != nullptr) {
#pragma unroll
        for (int i = 0; i < 4; ++i) q[i] = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
        *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(y_out) + o) = *reinterpret_cast<const uint4*>(q);
      }
    } else {
      float4* dst = reinterpret_cast<float4*>(static_cast<float*>(r.out) + o);
      dst[0] = make_float4(n[0], n[1], n[2], n[3]);
      dst[1] = make_float4(n[4], n[5], n[6], n[7]);
      if (y_out != nullptr) {
        float4* yd = reinterpret_cast<float4*>(static_cast<float*>(y_out) + o);
        yd[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        yd[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
      }
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
                           bool y_bf16, uint32_t* status, cudaStream_t stream) {
  const dim3 grid(T, T >= 1024 ? 1 : (H / 8 + 127) / 128);
  if (y_bf16)
    combine_kernel<true><<<grid, 128, 0, stream>>>(yr, pos, w, H, y, status);
  else
    combine_kernel<false><<<grid, 128, 0, stream>>>(yr, pos, w, H, y, status);
  return cudaGetLastError();
}

int residual_cluster_y(int T, int H) {
  const int G = H / 8;
  int ny = 1;
  if (T < 1024)  // few tokens: split each row so the work spreads over the SMs
    while (ny < 8 && ny * 128 < G) ny *= 2;
  while (ny < 8 && (G + ny * 128 - 1) / (ny * 128) > 32) ny *= 2;  // row part <= 128 KB of shared memory
  return ny;
}

size_t residual_smem_bytes(int T, int H) {
  const int ny = residual_cluster_y(T, H);
  return static_cast<size_t>((H / 8 + ny * 128 - 1) / (ny * 128)) * 128 * 32;
}

namespace {
template <bool kBf16, int kCY>
cudaError_t launch_residual_t(const __nv_bfloat16* yr, const int32_t* pos, const float* w, int T, int H,
                              const ResidualParams& r, void* y_out, uint32_t* status, size_t smem, cudaStream_t stream) {
  auto kern = combine_residual_kernel<kBf16, kCY>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(T), kCY);
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = kCY;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = kCY > 1 ? 1 : 0;
  err = cudaLaunchKernelEx(&cfg, kern, yr, pos, w, H, r, y_out, status);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

template <bool kBf16>
cudaError_t launch_residual_d(const __nv_bfloat16* yr, const int32_t* pos, const float* w, int T, int H,
                              const ResidualParams& r, void* y_out, uint32_t* status, cudaStream_t stream) {
  const size_t smem = residual_smem_bytes(T, H);
  switch (residual_cluster_y(T, H)) {
    case 1: return launch_residual_t<kBf16, 1>(yr, pos, w, T, H, r, y_out, status, smem, stream);
    case 2: return launch_residual_t<kBf16, 2>(yr, pos, w, T, H, r, y_out, status, smem, stream);
    case 4: return launch_residual_t<kBf16, 4>(yr, pos, w, T, H, r, y_out, status, smem, stream);
    default: return launch_residual_t<kBf16, 8>(yr, pos, w, T, H, r, y_out, status, smem, stream);
  }
}
}  // namespace

cudaError_t launch_combine_residual(const __nv_bfloat16* yr, const int32_t* pos, const float* w, int T, int H,
                                    const ResidualParams& r, void* y_out, bool bf16, uint32_t* status,
                                    cudaStream_t stream) {
  return bf16 ? launch_residual_d<true>(yr, pos, w, T, H, r, y_out, status, stream)
              : launch_residual_d<false>(yr, pos, w, T, H, r, y_out, status, stream);
}

cudaError_t launch_debug_timeout(uint32_t* status, uint64_t timeout_ns, cudaStream_t stream) {
  debug_timeout_kernel<<<1, 32, 0, stream>>>(status, timeout_ns);
  return cudaGetLastError();
}

}  // namespace beam

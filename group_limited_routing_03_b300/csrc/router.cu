// router.cu -- group-limited router of the Beam MoE block.
//
// Beam launch post ("Willkommen Beam ..." (spke.com), section "Mixture of
// Experts"; FP32 per section "Residual Stream"): sigmoid scores over all 256
// experts, 8 groups of 32 ranked by the sum of their two best scores, the best
// 4 groups kept, the top-8 experts inside them, weights normalised and scaled.
//
// One CTA owns 32 tokens.  Phase 1 computes the FP32 logits of those tokens
// against all 256 experts: thread (warp w, lane l) owns experts
// 128*(w%2) + l + 32*i (i = 0..3) and tokens 8*(w/2) .. +7, i.e. 32
// accumulators; the router weight and the activations stream through shared
// memory in 32-wide k-chunks, the next chunk prefetched into registers while
// the current one is consumed.  When the hidden dimension is split across
// CTAs (small T) the partial logits go to the workspace and a second kernel,
// one CTA per token, sums them in split order.  Phase 2 is the selection: one
// warp per token, lane l holding experts 8l..8l+7 (so the four lanes
// 4j..4j+3 hold group j); group top-2 sums, group ranking and the masked
// top-8 all run on warp shuffles.  The tile's routes are counted per expert
// for the dispatch step.
#include <cuda_bf16.h>

#include <cmath>

#include "moe_internal.cuh"
#include "select.cuh"

namespace beam {
namespace {

constexpr int kLogitLd = kExperts + 4;       // row stride of the logits tile (16-byte aligned rows)
constexpr int kWLd = kRouterKChunk + 1;      // row stride of the weight chunk [e][k] (conflict-free)
constexpr int kXLd = kRouterTile + 4;        // row stride of the activation chunk [k][token]

struct RouterSmem {
  union {
    float w[kExperts * kWLd];              // weight chunk, [e][k]
    float logits[kRouterTile * kLogitLd];  // [token][e]
  };
  float x[kRouterKChunk * kXLd];           // activation chunk, [k][token]
  int hist[kExperts];
};

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// Register staging of one k-chunk: 8 float4 of the router weight (rows
// tid/8 + 32*j, columns 4*(tid%8)..+3) and 4 activations (token tid/8,
// columns 4*(tid%8)..+3).
struct ChunkRegs {
  float4 w[8];
  float x[4];
};

template <bool kBf16>
__device__ __forceinline__ void load_chunk(const RouterParams& p, int t0, int k0, ChunkRegs& r) {
  const int tid = threadIdx.x;
  const int c4 = 4 * (tid & 7);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int row = (tid >> 3) + 32 * j;
    r.w[j] = __ldg(reinterpret_cast<const float4*>(p.wr + static_cast<size_t>(row) * p.H + k0 + c4));
  }
  const int t = t0 + (tid >> 3);
  if (t < p.T) {
    const size_t base = static_cast<size_t>(t) * p.H + k0 + c4;
    if (kBf16) {
      const uint2 raw = __ldg(reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(p.x) + base));
      r.x[0] = bf16_bits_to_float(raw.x & 0xFFFFu);
      r.x[1] = bf16_bits_to_float(raw.x >> 16);
      r.x[2] = bf16_bits_to_float(raw.y & 0xFFFFu);
      r.x[3] = bf16_bits_to_float(raw.y >> 16);
    } else {
      const float4 f = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(p.x) + base));
      r.x[0] = f.x; r.x[1] = f.y; r.x[2] = f.z; r.x[3] = f.w;
    }
  } else {
    r.x[0] = r.x[1] = r.x[2] = r.x[3] = 0.0f;
  }
}

__device__ __forceinline__ void store_chunk(RouterSmem& s, const ChunkRegs& r) {
  const int tid = threadIdx.x;
  const int c4 = 4 * (tid & 7);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    float* dst = &s.w[((tid >> 3) + 32 * j) * kWLd + c4];
    dst[0] = r.w[j].x;
    dst[1] = r.w[j].y;
    dst[2] = r.w[j].z;
    dst[3] = r.w[j].w;
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) s.x[(c4 + j) * kXLd + (tid >> 3)] = r.x[j];
}

// Selection for the CTA's 32 tokens from s.logits; also the tile histogram.
__device__ __forceinline__ void select_tile(const RouterParams& p, RouterSmem& s, int tile) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = tile * kRouterTile;
  for (int j = warp; j < kRouterTile; j += blockDim.x / 32) {
    const int t = t0 + j;
    if (t >= p.T) break;
    int id;
    float wv;
    select_token(&s.logits[j * kLogitLd], p.bias, p.scale, lane, id, wv);
    if (lane < kTopK) {
      p.ids[static_cast<size_t>(t) * kTopK + lane] = id;
      p.w[static_cast<size_t>(t) * kTopK + lane] = wv;
      atomicAdd(&s.hist[id], 1);
    }
  }
  __syncthreads();
  p.tile_hist[static_cast<size_t>(threadIdx.x) * p.n_tiles + tile] = s.hist[threadIdx.x];
}

template <bool kBf16>
__global__ void __launch_bounds__(256) router_gemm_kernel(RouterParams p) {
  __shared__ __align__(16) RouterSmem s;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ebase = 128 * (warp & 1) + lane;  // experts ebase + 32*i
  const int tbase = 8 * (warp >> 1);          // tokens tbase .. tbase+7 of the tile
  const int tile = blockIdx.x, split = blockIdx.y;
  const int t0 = tile * kRouterTile;
  const int kc_begin = split * p.n_kchunks / p.splits;
  const int kc_end = (split + 1) * p.n_kchunks / p.splits;
  s.hist[threadIdx.x] = 0;
  if (p.splits > 1 && split == 0) p.tile_hist[static_cast<size_t>(threadIdx.x) * p.n_tiles + tile] = 0;

  float acc[4][8];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.0f;

  ChunkRegs r;
  if (kc_begin < kc_end) load_chunk<kBf16>(p, t0, kc_begin * kRouterKChunk, r);
  for (int kc = kc_begin; kc < kc_end; ++kc) {
    store_chunk(s, r);
    __syncthreads();
    if (kc + 1 < kc_end) load_chunk<kBf16>(p, t0, (kc + 1) * kRouterKChunk, r);
#pragma unroll 8
    for (int kk = 0; kk < kRouterKChunk; ++kk) {
      float wv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) wv[i] = s.w[(ebase + 32 * i) * kWLd + kk];
      const float4 xa = *reinterpret_cast<const float4*>(&s.x[kk * kXLd + tbase]);
      const float4 xb = *reinterpret_cast<const float4*>(&s.x[kk * kXLd + tbase + 4]);
      const float xv[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(xv[j], wv[i], acc[i][j]);
    }
    __syncthreads();
  }

  if (p.splits > 1) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int t = t0 + tbase + j;
      if (t < p.T) {
        float* dst = p.part + (static_cast<size_t>(split) * p.T + t) * kExperts;
#pragma unroll
        for (int i = 0; i < 4; ++i) dst[ebase + 32 * i] = acc[i][j];
      }
    }
    return;
  }
#pragma unroll
  for (int j = 0; j < 8; ++j)
#pragma unroll
    for (int i = 0; i < 4; ++i) s.logits[(tbase + j) * kLogitLd + ebase + 32 * i] = acc[i][j];
  __syncthreads();
  select_tile(p, s, tile);
}

// splits > 1: the partial logits of each token are summed (FP32, a fixed
// order), then one warp selects; the tile histogram (zeroed by the logits
// kernel) is counted with atomics.
__device__ __forceinline__ void select_and_count(const RouterParams& p, const float* lrow, int t, int lane) {
  int id;
  float wv;
  select_token(lrow, p.bias, p.scale, lane, id, wv);
  if (lane < kTopK) {
    p.ids[static_cast<size_t>(t) * kTopK + lane] = id;
    p.w[static_cast<size_t>(t) * kTopK + lane] = wv;
    atomicAdd(&p.tile_hist[static_cast<size_t>(id) * p.n_tiles + t / kRouterTile], 1);
  }
}

// Many tokens: one warp per token, 8 tokens per CTA; lane l sums experts
// 8l..8l+7 over the splits in order.
constexpr int kSelTokens = 8;
__global__ void __launch_bounds__(32 * kSelTokens) router_select_tokens_kernel(RouterParams p) {
  __shared__ __align__(16) float lrow[kSelTokens][kExperts];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kSelTokens + warp;
  if (t >= p.T) return;
  const size_t stride = static_cast<size_t>(p.T) * kExperts;
  const float4* src = reinterpret_cast<const float4*>(p.part + static_cast<size_t>(t) * kExperts + 8 * lane);
  float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
  for (int sp = 0; sp < p.splits; ++sp) {
    const float4 u = src[sp * stride / 4], v = src[sp * stride / 4 + 1];
    a.x += u.x; a.y += u.y; a.z += u.z; a.w += u.w;
    b.x += v.x; b.y += v.y; b.z += v.z; b.w += v.w;
  }
  float* row = lrow[warp];
  *reinterpret_cast<float4*>(row + 8 * lane) = a;
  *reinterpret_cast<float4*>(row + 8 * lane + 4) = b;
  __syncwarp();
  select_and_count(p, row, t, lane);
}

// Few tokens, many splits: one CTA per token, 4 x 256 threads; thread group g
// sums splits g, g+4, g+8, ... for one expert, then the 4 sums are added in
// group order.
constexpr int kSelGroups = 4;
__global__ void __launch_bounds__(kSelGroups * kExperts) router_select_wide_kernel(RouterParams p) {
  __shared__ __align__(16) float part[kSelGroups][kExperts];
  __shared__ __align__(16) float lrow[kExperts];
  const int e = threadIdx.x % kExperts, g = threadIdx.x / kExperts;
  const int t = blockIdx.x;
  const float* src = p.part + static_cast<size_t>(t) * kExperts + e;
  const size_t stride = static_cast<size_t>(p.T) * kExperts;
  float v = 0.0f;
  int sp = g;
  for (; sp + 4 * kSelGroups <= p.splits; sp += 4 * kSelGroups) {
    float q[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) q[u] = src[static_cast<size_t>(sp + u * kSelGroups) * stride];
#pragma unroll
    for (int u = 0; u < 4; ++u) v += q[u];
  }
  for (; sp < p.splits; sp += kSelGroups) v += src[static_cast<size_t>(sp) * stride];
  part[g][e] = v;
  __syncthreads();
  if (g == 0) {
    float s = part[0][e];
#pragma unroll
    for (int k = 1; k < kSelGroups; ++k) s += part[k][e];
    lrow[e] = s;
  }
  __syncthreads();
  if (threadIdx.x < 32) select_and_count(p, lrow, t, threadIdx.x);
}

cudaError_t launch_select(const RouterParams& p, cudaStream_t stream) {
  if (p.T >= 1024)
    router_select_tokens_kernel<<<(p.T + kSelTokens - 1) / kSelTokens, 32 * kSelTokens, 0, stream>>>(p);
  else
    router_select_wide_kernel<<<p.T, kSelGroups * kExperts, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

int router_split_cap(int T, int H) {
  const int n_tiles = (T + kRouterTile - 1) / kRouterTile;
  int cap = (2 * kMaxSmsForSizing + n_tiles - 1) / n_tiles;
  const int nkc = H / kRouterKChunk;
  if (cap > nkc) cap = nkc;
  return cap < 1 ? 1 : cap;
}

int router_splits(int T, int H, int num_sms) {
  const int n_tiles = (T + kRouterTile - 1) / kRouterTile;
  if (n_tiles >= num_sms) return 1;
  int s = (2 * num_sms + n_tiles - 1) / n_tiles;
  const int cap = router_split_cap(T, H);
  if (s > cap) s = cap;
  return s < 1 ? 1 : s;
}

cudaError_t launch_router(const RouterParams& p, bool x_bf16, cudaStream_t stream) {
  const dim3 grid(p.n_tiles, p.splits);
  if (x_bf16)
    router_gemm_kernel<true><<<grid, 256, 0, stream>>>(p);
  else
    router_gemm_kernel<false><<<grid, 256, 0, stream>>>(p);
  if (p.splits > 1) {
    const cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    return launch_select(p, stream);
  }
  return cudaGetLastError();
}

cudaError_t launch_router_select(const RouterParams& p, cudaStream_t stream) { return launch_select(p, stream); }

}  // namespace beam

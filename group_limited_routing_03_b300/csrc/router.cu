// router.cu -- group-limited router of the Beam MoE block.
//
// Beam launch post ("Willkommen Beam ..." (spke.com), section "Mixture of
// Experts"; FP32 per section "Residual Stream"): sigmoid scores over all 256
// experts, 8 groups of 32 ranked by the sum of their two best scores, the best
// 4 groups kept, the top-8 experts inside them, weights normalised and scaled.
//
// One CTA owns 32 tokens.  Phase 1 computes the FP32 logits of those tokens
// against all 256 experts (thread e owns expert e, 32 accumulators, the
// router weight streamed through shared memory in 32-wide k-chunks).  When the
// hidden dimension is split across CTAs (small T) the partial logits go to the
// workspace and a second kernel sums them in a fixed order.  Phase 2 is the
// selection: one warp per token, lane l holding experts 8l..8l+7 (so the four
// lanes 4j..4j+3 hold group j); group top-2 sums, group ranking and the
// masked top-8 all run on warp shuffles.  The CTA also counts its routes per
// expert for the dispatch step.
#include <cuda_bf16.h>

#include <cmath>

#include "moe_internal.cuh"

namespace beam {
namespace {

constexpr int kLogitLd = kExperts + 4;  // row stride of the logits tile (16-byte aligned rows)
constexpr int kWLd = kExperts + 1;      // row stride of the transposed weight chunk

struct RouterSmem {
  union {
    float w[kRouterKChunk * kWLd];       // weight chunk, [k][e]
    float logits[kRouterTile * kLogitLd];  // [token][e]
  };
  float x[kRouterKChunk * kRouterTile];  // activation chunk, [k][token]
  int hist[kExperts];
};

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// Loads activations [t0, t0+32) x [k0, k0+32) into s.x as [k][token] (f32).
template <bool kBf16>
__device__ __forceinline__ void load_x_chunk(const RouterParams& p, RouterSmem& s, int t0, int k0) {
  const int tid = threadIdx.x;
  const int tok = tid >> 3;        // 0..31
  const int kq = (tid & 7) * 4;    // 0..28
  const int t = t0 + tok;
  float v[4] = {0.f, 0.f, 0.f, 0.f};
  if (t < p.T) {
    const size_t base = static_cast<size_t>(t) * p.H + k0 + kq;
    if (kBf16) {
      const uint2 raw = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(p.x) + base);
      v[0] = bf16_bits_to_float(raw.x & 0xFFFFu);
      v[1] = bf16_bits_to_float(raw.x >> 16);
      v[2] = bf16_bits_to_float(raw.y & 0xFFFFu);
      v[3] = bf16_bits_to_float(raw.y >> 16);
    } else {
      const float4 f = *reinterpret_cast<const float4*>(static_cast<const float*>(p.x) + base);
      v[0] = f.x; v[1] = f.y; v[2] = f.z; v[3] = f.w;
    }
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) s.x[(kq + j) * kRouterTile + tok] = v[j];
}

// Selection for one token, by one warp.  `lrow` = the token's 256 logits in
// shared memory.  Lane k < 8 returns the k-th chosen expert and its weight.
__device__ __forceinline__ void select_token(const float* lrow, const float* bias, float scale, int lane,
                                             int& out_id, float& out_w) {
  float sc[8], sel[8];
  const float4 a = *reinterpret_cast<const float4*>(lrow + 8 * lane);
  const float4 b = *reinterpret_cast<const float4*>(lrow + 8 * lane + 4);
  const float lg[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    sc[i] = 1.0f / (1.0f + expf(-lg[i]));  // sigmoid, FP32
    sel[i] = sc[i] + (bias != nullptr ? bias[8 * lane + i] : 0.0f);
  }
  // Two best selection scores of this lane, then of the lane's group (4 lanes).
  float m1 = -INFINITY, m2 = -INFINITY;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float v = sel[i];
    if (v > m1) {
      m2 = m1;
      m1 = v;
    } else if (v > m2) {
      m2 = v;
    }
  }
#pragma unroll
  for (int off = 1; off <= 2; off <<= 1) {
    const float o1 = __shfl_xor_sync(0xFFFFFFFFu, m1, off);
    const float o2 = __shfl_xor_sync(0xFFFFFFFFu, m2, off);
    const float n1 = fmaxf(m1, o1);
    const float n2 = fmaxf(fminf(m1, o1), fmaxf(m2, o2));
    m1 = n1;
    m2 = n2;
  }
  const float gscore = m1 + m2;
  // Rank of this lane's group among the 8 (ties: lower group index first).
  const int mygroup = lane >> 2;
  int rank = 0;
#pragma unroll
  for (int j = 0; j < kGroups; ++j) {
    const float gj = __shfl_sync(0xFFFFFFFFu, gscore, 4 * j);
    rank += (gj > gscore || (gj == gscore && j < mygroup)) ? 1 : 0;
  }
  const bool kept = rank < kGroupsKept;
  float cand[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) cand[i] = kept ? sel[i] : -INFINITY;

  // Top-8 over the kept groups: 8 rounds of warp arg-max (ties: lower id).
  float ssum = 0.0f;
  int my_id = 0;
  float my_s = 0.0f;
#pragma unroll 1
  for (int k = 0; k < kTopK; ++k) {
    float bv = cand[0];
    int bi = 0;
#pragma unroll
    for (int i = 1; i < 8; ++i)
      if (cand[i] > bv) {
        bv = cand[i];
        bi = i;
      }
    int bidx = 8 * lane + bi;
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
      const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, off);
      const int oi = __shfl_xor_sync(0xFFFFFFFFu, bidx, off);
      if (ov > bv || (ov == bv && oi < bidx)) {
        bv = ov;
        bidx = oi;
      }
    }
    const int owner = bidx >> 3;
    float s_w = 0.0f;
    if (lane == owner) {
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (i == (bidx & 7)) {
          s_w = sc[i];
          cand[i] = -INFINITY;
        }
    }
    s_w = __shfl_sync(0xFFFFFFFFu, s_w, owner);
    ssum += s_w;
    if (lane == k) {
      my_id = bidx;
      my_s = s_w;
    }
  }
  out_id = my_id;
  out_w = my_s / ssum * scale;
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
  const int e = threadIdx.x;  // expert owned by this thread
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile = blockIdx.x, split = blockIdx.y;
  const int t0 = tile * kRouterTile;
  const int kc_begin = split * p.n_kchunks / p.splits;
  const int kc_end = (split + 1) * p.n_kchunks / p.splits;
  s.hist[threadIdx.x] = 0;

  float acc[kRouterTile];
#pragma unroll
  for (int j = 0; j < kRouterTile; ++j) acc[j] = 0.0f;

  for (int kc = kc_begin; kc < kc_end; ++kc) {
    const int k0 = kc * kRouterKChunk;
    // Weight chunk: warp w loads rows 32w..32w+31, lanes along k (coalesced),
    // stored transposed [k][e] (row stride 257 keeps the stores conflict-free).
#pragma unroll 8
    for (int i = 0; i < 32; ++i) {
      const int row = warp * 32 + i;
      s.w[lane * kWLd + row] = p.wr[static_cast<size_t>(row) * p.H + k0 + lane];
    }
    load_x_chunk<kBf16>(p, s, t0, k0);
    __syncthreads();
#pragma unroll 4
    for (int kk = 0; kk < kRouterKChunk; ++kk) {
      const float wv = s.w[kk * kWLd + e];
      const float4* xr = reinterpret_cast<const float4*>(&s.x[kk * kRouterTile]);
#pragma unroll
      for (int q = 0; q < kRouterTile / 4; ++q) {
        const float4 xv = xr[q];
        acc[4 * q + 0] = fmaf(xv.x, wv, acc[4 * q + 0]);
        acc[4 * q + 1] = fmaf(xv.y, wv, acc[4 * q + 1]);
        acc[4 * q + 2] = fmaf(xv.z, wv, acc[4 * q + 2]);
        acc[4 * q + 3] = fmaf(xv.w, wv, acc[4 * q + 3]);
      }
    }
    __syncthreads();
  }

  if (p.splits > 1) {
#pragma unroll
    for (int j = 0; j < kRouterTile; ++j) {
      const int t = t0 + j;
      if (t < p.T) p.part[(static_cast<size_t>(split) * p.T + t) * kExperts + e] = acc[j];
    }
    return;
  }
#pragma unroll
  for (int j = 0; j < kRouterTile; ++j) s.logits[j * kLogitLd + e] = acc[j];
  __syncthreads();
  select_tile(p, s, tile);
}

// splits > 1: sum the partial logits in split order, then select.
__global__ void __launch_bounds__(256) router_select_kernel(RouterParams p) {
  __shared__ __align__(16) RouterSmem s;
  const int e = threadIdx.x;
  const int tile = blockIdx.x;
  const int t0 = tile * kRouterTile;
  s.hist[threadIdx.x] = 0;
  for (int j = 0; j < kRouterTile; ++j) {
    const int t = t0 + j;
    float v = 0.0f;
    if (t < p.T)
      for (int sp = 0; sp < p.splits; ++sp) v += p.part[(static_cast<size_t>(sp) * p.T + t) * kExperts + e];
    s.logits[j * kLogitLd + e] = v;
  }
  __syncthreads();
  select_tile(p, s, tile);
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
  if (p.splits > 1) router_select_kernel<<<p.n_tiles, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace beam

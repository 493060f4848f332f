// dispatch.cu -- per-expert route lists.
//
// Beam launch post, section "Mixture of Experts": each token runs only its 8
// experts.  The grouped GEMMs therefore need, per expert, the list of routes
// r = t*8 + k that chose it.  Routes are cut into tiles of 256 (the router's
// 32-token tiles).  The router (or tile_hist_kernel, when the caller supplies
// the ids) counts each tile's routes per expert; scan_kernel turns those
// counts into per-expert totals and per-tile exclusive prefixes; and
// scatter_kernel places every route at
//     offsets[e] + (routes of e in earlier tiles) + (rank inside the tile),
// which keeps the routes of an expert in ascending r: a deterministic
// permutation with no global atomics.  gather_kernel then copies the token
// rows into that order (BF16) as the B operand of the gate/up GEMM, reading
// each token row once and writing it to its 8 route positions (reading per
// route would fetch x from DRAM several times, as the 8x larger output
// streams through L2 and evicts it).
#include <cuda_bf16.h>

#include "moe_internal.cuh"
#include "tc.cuh"

namespace beam {
namespace {

__device__ __forceinline__ int warp_inclusive_scan(int v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xFFFFFFFFu, v, off);
    if (lane >= off) v += o;
  }
  return v;
}

// Exclusive scan of one value per thread over a 256-thread block; returns the
// thread's exclusive prefix, writes the block total to *total.
__device__ __forceinline__ int block_exclusive_scan_256(int v, int* warp_sums, int* total) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int incl = warp_inclusive_scan(v);
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int ws = lane < 8 ? warp_sums[lane] : 0;
    const int wi = warp_inclusive_scan(ws);
    if (lane < 8) warp_sums[lane] = wi - ws;
    if (lane == 7) *total = wi;
  }
  __syncthreads();
  const int r = warp_sums[warp] + incl - v;
  __syncthreads();
  return r;
}

// Per-tile expert histogram for caller-supplied ids (the router fuses this).
__global__ void __launch_bounds__(256) tile_hist_kernel(const int32_t* ids, int R, int n_tiles,
                                                        int32_t* tile_hist, uint32_t* status) {
  __shared__ int hist[kExperts];
  hist[threadIdx.x] = 0;
  __syncthreads();
  const int r = blockIdx.x * kTileRoutes + threadIdx.x;
  if (r < R) {
    const int e = ids[r];
    if (e >= 0 && e < kExperts)
      atomicAdd(&hist[e], 1);
    else
      report_status(status, kStatusDeviceCheck, kCheckTileHistId);
  }
  __syncthreads();
  tile_hist[static_cast<size_t>(threadIdx.x) * n_tiles + blockIdx.x] = hist[threadIdx.x];
}

// One CTA per expert: exclusive scan of its per-tile counts (in place) and
// its total.
__global__ void __launch_bounds__(256) scan_kernel(int32_t* tile_hist, int n_tiles, int32_t* counts) {
  __shared__ int warp_sums[8];
  __shared__ int total;
  int32_t* row = tile_hist + static_cast<size_t>(blockIdx.x) * n_tiles;
  int carry = 0;
  for (int base = 0; base < n_tiles; base += 256) {
    const int i = base + threadIdx.x;
    const int v = i < n_tiles ? row[i] : 0;
    const int ex = block_exclusive_scan_256(v, warp_sums, &total);
    if (i < n_tiles) row[i] = carry + ex;
    carry += total;
  }
  if (threadIdx.x == 0) counts[blockIdx.x] = carry;
}

// One CTA per tile of 256 routes (thread = route).
__global__ void __launch_bounds__(256) scatter_kernel(const int32_t* ids, int R, int n_tiles,
                                                      const int32_t* tile_prefix, const int32_t* counts,
                                                      int nmax, int32_t* offsets, int32_t* chunk_prefix,
                                                      int32_t* perm, int32_t* pos, uint32_t* status) {
  __shared__ int warp_sums[8];
  __shared__ int total;
  __shared__ int off_s[kExperts];
  __shared__ int wcnt[8][kExperts];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tile = blockIdx.x;

  const int c = counts[tid];
  const int ex = block_exclusive_scan_256(c, warp_sums, &total);
  off_s[tid] = ex;
  if (tile == 0) {
    offsets[tid] = ex;
    if (tid == kExperts - 1) offsets[kExperts] = ex + c;
    const int nch = (c + nmax - 1) / nmax;
    const int cex = block_exclusive_scan_256(nch, warp_sums, &total);
    chunk_prefix[tid] = cex;
    if (tid == kExperts - 1) chunk_prefix[kExperts] = cex + nch;
  }
#pragma unroll
  for (int w = 0; w < 8; ++w) wcnt[w][tid] = 0;
  __syncthreads();

  const int r = tile * kTileRoutes + tid;
  const bool valid = r < R;
  int e = valid ? ids[r] : -1;
  if (e < 0 || e >= kExperts) {
    if (valid) dcheck(false, status, kCheckScatterId);
    e = -1;
  }
  const unsigned peers = __match_any_sync(0xFFFFFFFFu, e);
  const unsigned lt = (1u << lane) - 1u;
  const int rank_in_warp = __popc(peers & lt);
  if (e >= 0 && (peers & lt) == 0u) wcnt[warp][e] = __popc(peers);
  __syncthreads();
  if (valid) {
    if (e >= 0) {
      int rank = rank_in_warp;
      for (int w = 0; w < warp; ++w) rank += wcnt[w][e];
      const int p = off_s[e] + tile_prefix[static_cast<size_t>(e) * n_tiles + tile] + rank;
      perm[p] = r;
      pos[r] = p;
    } else {
      pos[r] = -1;
    }
  }
}

// xp[pos[t*8+k], :] = bf16(x[t, :]) for k = 0..7 (routes with pos < 0, whose
// expert id was out of range, are skipped); 8 elements (16 bytes) per step.
template <bool kBf16>
__global__ void __launch_bounds__(256) gather_kernel(const void* x, int H, const int32_t* pos, int T,
                                                     __nv_bfloat16* xp, uint32_t* status) {
  const int R = T * kTopK;
  const int vecs_per_row = H / 8;
  const size_t n = static_cast<size_t>(T) * vecs_per_row;
#pragma unroll 2
  for (size_t v = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; v < n;
       v += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const int t = static_cast<int>(v / vecs_per_row);
    const int c = static_cast<int>(v % vecs_per_row);
    uint4 out;
    if (kBf16) {
      out = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(x) + static_cast<size_t>(t) * H + c * 8);
    } else {
      const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(x) + static_cast<size_t>(t) * H + c * 8);
      const float4 a = src[0], b = src[1];
      __nv_bfloat162 q0 = __floats2bfloat162_rn(a.x, a.y), q1 = __floats2bfloat162_rn(a.z, a.w);
      __nv_bfloat162 q2 = __floats2bfloat162_rn(b.x, b.y), q3 = __floats2bfloat162_rn(b.z, b.w);
      out.x = *reinterpret_cast<uint32_t*>(&q0);
      out.y = *reinterpret_cast<uint32_t*>(&q1);
      out.z = *reinterpret_cast<uint32_t*>(&q2);
      out.w = *reinterpret_cast<uint32_t*>(&q3);
    }
    const int4 p0 = *reinterpret_cast<const int4*>(pos + static_cast<size_t>(t) * kTopK);
    const int4 p1 = *reinterpret_cast<const int4*>(pos + static_cast<size_t>(t) * kTopK + 4);
    const int dst[kTopK] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
#pragma unroll
    for (int k = 0; k < kTopK; ++k)
      if (dst[k] >= 0 && dcheck(dst[k] < R, status, kCheckGatherPos))
        *reinterpret_cast<uint4*>(xp + static_cast<size_t>(dst[k]) * H + c * 8) = out;
  }
}

}  // namespace

cudaError_t launch_tile_hist(const int32_t* ids, int R, int n_tiles, int32_t* tile_hist, uint32_t* status,
                             cudaStream_t stream) {
  tile_hist_kernel<<<n_tiles, 256, 0, stream>>>(ids, R, n_tiles, tile_hist, status);
  return cudaGetLastError();
}

cudaError_t launch_dispatch(const int32_t* ids, int R, int n_tiles, int32_t* tile_hist, int32_t* counts,
                            int32_t* offsets, int32_t* chunk_prefix, int nmax, int32_t* perm, int32_t* pos,
                            uint32_t* status, cudaStream_t stream) {
  scan_kernel<<<kExperts, 256, 0, stream>>>(tile_hist, n_tiles, counts);
  scatter_kernel<<<n_tiles, 256, 0, stream>>>(ids, R, n_tiles, tile_hist, counts, nmax, offsets,
                                              chunk_prefix, perm, pos, status);
  return cudaGetLastError();
}

namespace {
// The dense MLP as one "expert" that takes every row: counts = (R, 0, ...),
// offsets = (0, R, ..., R), chunk_prefix = (0, n, ..., n) with n = ceil(R / nmax).
__global__ void __launch_bounds__(288) dense_dispatch_kernel(int R, int nmax, int32_t* counts, int32_t* offsets,
                                                             int32_t* chunk_prefix) {
  const int e = threadIdx.x;
  if (e > kExperts) return;
  if (e < kExperts) counts[e] = e == 0 ? R : 0;
  offsets[e] = e == 0 ? 0 : R;
  chunk_prefix[e] = e == 0 ? 0 : (R + nmax - 1) / nmax;
}
}  // namespace

namespace {
// Debug builds, before each grouped GEMM: the schedule the GEMM will read
// must describe R routes in order -- counts >= 0, offsets the exclusive
// prefix sum of counts ending at most at R, chunk_prefix the prefix sum of
// ceil(count / nmax).  If it does not, the check is recorded and
// chunk_prefix[E] is set to 0, so that the GEMM runs no unit (it would
// otherwise store outside the route rows).
__global__ void __launch_bounds__(kExperts) validate_schedule_kernel(const int32_t* counts, const int32_t* offsets,
                                                                     int32_t* chunk_prefix, int R, int nmax,
                                                                     uint32_t* status) {
  __shared__ int bad;
  const int e = threadIdx.x;
  if (e == 0) bad = 0;
  __syncthreads();
  const int c = counts[e];
  const int o0 = offsets[e], o1 = offsets[e + 1];
  const int q0 = chunk_prefix[e], q1 = chunk_prefix[e + 1];
  const bool ok = c >= 0 && o0 >= 0 && o1 == o0 + c && o1 <= R && (e != 0 || (o0 == 0 && q0 == 0)) &&
                  q1 - q0 == (c + nmax - 1) / nmax;
  if (!ok) atomicExch(&bad, 1);
  __syncthreads();
  if (e == 0 && bad != 0) {
    report_status(status, kStatusDeviceCheck, kCheckSchedule);
    chunk_prefix[kExperts] = 0;
  }
}
}  // namespace

cudaError_t launch_validate_schedule(const int32_t* counts, const int32_t* offsets, int32_t* chunk_prefix, int R,
                                     int nmax, uint32_t* status, cudaStream_t stream) {
  validate_schedule_kernel<<<1, kExperts, 0, stream>>>(counts, offsets, chunk_prefix, R, nmax, status);
  return cudaGetLastError();
}

cudaError_t launch_dense_dispatch(int R, int nmax, int32_t* counts, int32_t* offsets, int32_t* chunk_prefix,
                                  cudaStream_t stream) {
  dense_dispatch_kernel<<<1, 288, 0, stream>>>(R, nmax, counts, offsets, chunk_prefix);
  return cudaGetLastError();
}

cudaError_t launch_gather(const void* x, bool x_bf16, int H, const int32_t* pos, int T, __nv_bfloat16* xp,
                          int num_sms, uint32_t* status, cudaStream_t stream) {
  const size_t n = static_cast<size_t>(T) * (H / 8);
  size_t blocks = (n + 255) / 256;
  const size_t cap = static_cast<size_t>(num_sms) * 16;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  if (x_bf16)
    gather_kernel<true><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(x, H, pos, T, xp, status);
  else
    gather_kernel<false><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(x, H, pos, T, xp, status);
  return cudaGetLastError();
}

}  // namespace beam

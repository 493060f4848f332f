// gemm.cu -- grouped expert GEMMs on the Blackwell tensor cores (tcgen05,
// accumulators in TMEM, operands staged by TMA).
//
// Beam launch post, section "Mixture of Experts": every expert is a SwiGLU MLP
// (hidden 5120, intermediate 2560); section "Residual Stream": the SwiGLU
// product is computed in FP32.
//
//   mode 0 (gate/up):  h[r, i]  = silu(x_r . Wg[e,i,:]) * (x_r . Wu[e,i,:])
//   mode 1 (down):     yr[r, j] = h_r . Wd[e,j,:]
//
// for every route r of expert e (routes in the dispatch order).  The weight
// rows are the MMA's M side (128 rows per tile = the 128 TMEM lanes) and the
// routed tokens are its N side ("swap AB"): an expert sees 1..3 tokens at
// decode and ~256 at prefill, and N can be any multiple of 16 up to 256,
// while M is fixed at 128.  A work unit is (expert, token chunk of <= nmax
// routes, 128-row weight tile); units are enumerated in the order
// (expert, chunk, row tile) so that CTAs running side by side share the
// activation chunk (and, for several chunks of one expert, the weight tile)
// through L2.  The grid is persistent (one CTA per SM), units are dealt
// round-robin.
//
// Warp roles (192 threads):
//   warp 0      TMA producer: weight tile(s) 128x64 and ceil(n/32) boxes of
//               32 activation rows x 64 per stage, 128-byte swizzle;
//   warp 1      TMEM allocator and MMA issuer (one thread):
//               tcgen05.mma kind::f16, M=128, N=round_up(n,16), K=16 steps;
//   warps 2-5   epilogue: tcgen05.ld of the accumulators (warp w reads TMEM
//               lanes 32*(w%4)..+31), SwiGLU in FP32 (mode 0), BF16 stores.
// Shared-memory stages are recycled through full/empty mbarriers, TMEM
// accumulator buffers through acc_full/acc_empty.  Every wait is bounded.
#include <cuda.h>
#include <cuda_bf16.h>

#include "moe_internal.cuh"
#include "tc.cuh"

namespace beam {
namespace {

constexpr int kThreads = 192;
constexpr uint32_t kATileBytes = kBlockM * kBlockK * 2;  // 16 KiB
constexpr uint32_t kBoxBytes = kBoxRows * kBlockK * 2;   // 4 KiB

struct Unit {
  int e, m, start, n;
};

__device__ __forceinline__ Unit unit_at(const GemmParams& p, int u) {
  const int q = u / p.m_tiles;
  Unit U;
  U.m = u - q * p.m_tiles;
  // expert e with chunk_prefix[e] <= q < chunk_prefix[e+1]
  int lo = 0, hi = kExperts;  // invariant: chunk_prefix[lo] <= q < chunk_prefix[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(&p.chunk_prefix[mid]) <= q)
      lo = mid;
    else
      hi = mid;
  }
  U.e = lo;
  const int c = q - __ldg(&p.chunk_prefix[lo]);
  U.start = __ldg(&p.offsets[lo]) + c * p.nmax;
  const int left = __ldg(&p.counts[lo]) - c * p.nmax;
  U.n = left < p.nmax ? left : p.nmax;
  return U;
}

template <int kMode>
__global__ void __launch_bounds__(kThreads, 1)
    moe_gemm_kernel(const __grid_constant__ CUtensorMap tm_a0, const __grid_constant__ CUtensorMap tm_a1,
                    const __grid_constant__ CUtensorMap tm_b, const GemmParams p) {
  constexpr int kNumA = kMode == 0 ? 2 : 1;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t b_tile_bytes = static_cast<uint32_t>(p.nmax) * kBlockK * 2;
  const uint32_t stage_bytes = kNumA * kATileBytes + b_tile_bytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(p.stages) * stage_bytes);
  uint64_t* full = bars;
  uint64_t* empty = full + p.stages;
  uint64_t* acc_full = empty + p.stages;
  uint64_t* acc_empty = acc_full + p.acc_stages;
  uint64_t* drain = acc_empty + p.acc_stages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile uint32_t* abort_flag = tmem_slot + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto a_tile = [&](int s, int which) { return smem + static_cast<size_t>(s) * stage_bytes + which * kATileBytes; };
  auto b_tile = [&](int s) { return smem + static_cast<size_t>(s) * stage_bytes + kNumA * kATileBytes; };

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < p.acc_stages; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], 4);
    }
    mbar_init(drain, 1);
    *abort_flag = 0u;
    fence_mbar_init();
    tma_prefetch_desc(&tm_a0);
    if (kMode == 0) tma_prefetch_desc(&tm_a1);
    tma_prefetch_desc(&tm_b);
  }
  if (warp == 1) tmem_alloc(tmem_slot, p.tmem_cols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int total_units = __ldg(&p.chunk_prefix[kExperts]) * p.m_tiles;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol_w = l2_policy_evict_first();
      const uint64_t pol_x = l2_policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      long long issued = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < total_units && ok; u += gridDim.x) {
        const Unit U = unit_at(p, u);
        const int a_row = U.e * p.a_rows_per_expert + U.m * kBlockM;
        const int nbox = (U.n + kBoxRows - 1) / kBoxRows;
        const uint32_t bytes = kNumA * kATileBytes + static_cast<uint32_t>(nbox) * kBoxBytes;
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, p.timeout_ns, abort_flag, p.status, kWhereProducerEmpty)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[stage], bytes);
          const int kx = kb * kBlockK;
          tma_load_2d(a_tile(stage, 0), &tm_a0, &full[stage], kx, a_row, pol_w);
          if (kMode == 0) tma_load_2d(a_tile(stage, 1), &tm_a1, &full[stage], kx, a_row, pol_w);
          for (int b = 0; b < nbox; ++b)
            tma_load_2d(b_tile(stage) + b * kBoxBytes, &tm_b, &full[stage], kx, U.start + b * kBoxRows, pol_x);
          ++issued;
          if (++stage == p.stages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Drain: the latest load issued on every slot has landed (immediate in
      // the normal case, where the MMA warp consumed them all).
      for (int s = 0; s < p.stages; ++s) {
        if (issued <= s && issued < p.stages) continue;  // slot never used
        const uint32_t par = s < stage ? phase : (phase ^ 1u);
        mbar_wait(&full[s], par, p.timeout_ns, nullptr, p.status, kWhereDrain);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < total_units && ok; u += gridDim.x) {
        const Unit U = unit_at(p, u);
        const uint32_t n_mma = static_cast<uint32_t>((U.n + 15) & ~15);
        const uint32_t idesc = idesc_bf16_f32(kBlockM, n_mma);
        if (!mbar_wait(&acc_empty[acc], acc_phase ^ 1u, p.timeout_ns, abort_flag, p.status, kWhereMmaAccEmpty))
          break;
        tc_fence_after();
        const uint32_t d0 = tmem_base + static_cast<uint32_t>(acc) * p.acc_cols;
        const uint32_t d1 = d0 + static_cast<uint32_t>(p.nmax);
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          if (!mbar_wait(&full[stage], phase, p.timeout_ns, abort_flag, p.status, kWhereMmaFull)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t da0 = sdesc_k_sw128(smem_u32(a_tile(stage, 0)));
          const uint64_t da1 = sdesc_k_sw128(smem_u32(a_tile(stage, kNumA - 1)));
          const uint64_t db = sdesc_k_sw128(smem_u32(b_tile(stage)));
#pragma unroll
          for (int k = 0; k < kBlockK / 16; ++k) {
            const uint32_t accumulate = (kb | k) != 0 ? 1u : 0u;
            mma_bf16(d0, da0 + 2u * k, db + 2u * k, idesc, accumulate);
            if (kMode == 0) mma_bf16(d1, da1 + 2u * k, db + 2u * k, idesc, accumulate);
          }
          mma_commit(&empty[stage]);
          if (++stage == p.stages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(&acc_full[acc]);
        if (++acc == p.acc_stages) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      // Every MMA issued by this thread has completed before TMEM is freed.
      mma_commit(drain);
      mbar_wait(drain, 0, p.timeout_ns, nullptr, p.status, kWhereDrain);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int u = blockIdx.x; u < total_units; u += gridDim.x) {
      const Unit U = unit_at(p, u);
      int ok = 1;
      if (lane == 0)
        ok = mbar_wait(&acc_full[acc], acc_phase, p.timeout_ns, abort_flag, p.status, kWhereEpiAccFull) ? 1 : 0;
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + static_cast<uint32_t>(acc) * p.acc_cols;
      const int feat = U.m * kBlockM + row;
      const float s0 = p.gs0 != nullptr ? __ldg(&p.gs0[U.e]) : 1.0f;
      const float s1 = (kMode == 0 && p.gs1 != nullptr) ? __ldg(&p.gs1[U.e]) : 1.0f;
      const int ncols = (U.n + 15) & ~15;
      __nv_bfloat16* out = p.out + static_cast<size_t>(U.start) * p.out_ld + feat;
      for (int c0 = 0; c0 < ncols; c0 += 16) {
        float g[16];
        tmem_ld16(tbase + static_cast<uint32_t>(c0), g);
        if (kMode == 0) {
          float up[16];
          tmem_ld16(tbase + static_cast<uint32_t>(p.nmax + c0), up);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            if (c0 + j < U.n) {
              const float a = g[j] * s0;
              const float b = up[j] * s1;
              const float hval = a / (1.0f + expf(-a)) * b;  // SiLU(gate) * up, FP32
              out[static_cast<size_t>(c0 + j) * p.out_ld] = __float2bfloat16_rn(hval);
            }
          }
        } else {
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (c0 + j < U.n) out[static_cast<size_t>(c0 + j) * p.out_ld] = __float2bfloat16_rn(g[j] * s0);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[acc]);
      if (++acc == p.acc_stages) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, p.tmem_cols);
  }
}

}  // namespace

size_t gemm_stage_bytes(int mode, int nmax) {
  return static_cast<size_t>(mode == 0 ? 2 : 1) * kATileBytes + static_cast<size_t>(nmax) * kBlockK * 2;
}

cudaError_t launch_gemm(int mode, const CUtensorMap& a0, const CUtensorMap& a1, const CUtensorMap& b,
                        const GemmParams& p, int grid, size_t smem_bytes, cudaStream_t stream) {
  cudaError_t err;
  if (mode == 0) {
    err = cudaFuncSetAttribute(moe_gemm_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(smem_bytes));
    if (err != cudaSuccess) return err;
    moe_gemm_kernel<0><<<grid, kThreads, smem_bytes, stream>>>(a0, a1, b, p);
  } else {
    err = cudaFuncSetAttribute(moe_gemm_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(smem_bytes));
    if (err != cudaSuccess) return err;
    moe_gemm_kernel<1><<<grid, kThreads, smem_bytes, stream>>>(a0, a1, b, p);
  }
  return cudaGetLastError();
}

}  // namespace beam

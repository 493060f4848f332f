// router_tc.cu -- router logits on the tensor cores for large token counts.
//
// Beam launch post ("Willkommen Beam ..." (spke.com), section "Mixture of
// Experts", FP32 per section "Residual Stream"): router logits
// l[t,e] = sum_h x[t,h] * Wr[e,h], sigmoid scores, group-limited top-8.
//
// FP32 accuracy from BF16 tensor-core products: the FP32 router weight is
// split exactly into three BF16 terms, W = w1 + w2 + w3 with
//   w1 = bf16(W), w2 = bf16(W - w1), w3 = bf16(W - w1 - w2)
// (24 significant bits; the split-precision scheme of Henry, Tang and
// Heinecke, "Leveraging the bfloat16 Artificial Intelligence Datatype For
// Higher-Precision Computations", 2019).  x is BF16 already, so every
// product x*w_i is exact; the reduction over K' = 3H runs as short partial
// sums of kPartial k-blocks (16 MMAs), each accumulated in a TMEM buffer from
// zero and then added, round-to-nearest, into FP32 registers while the MMA
// fills the other buffer.  (Accumulating all of K' in one TMEM accumulator
// measured ~1e-4 logit error on B300, far above FP32 FMA's; short partials
// keep every tensor-core rounding relative to a small partial sum.)
// One CTA owns 128 tokens x 256 experts (tcgen05.mma M=128, N=256, BF16,
// FP32 accumulation) over a range of the K' reduction: with one range it holds
// whole logits, which 8 epilogue warps (lane = token, half the experts each)
// write to shared memory for the same warp-per-token group-limited selection
// as the CUDA-core router; with p.splits ranges (blockIdx.y) it writes FP32
// partial logits, which the select kernel (router.cu) sums.  Every k-block
// moves 48 KiB through shared memory (TMA in, MMA out), so the router is bound
// by shared-memory bandwidth per SM; splitting K spreads it over more SMs.
#include <cuda.h>
#include <cuda_bf16.h>

#include "moe_internal.cuh"
#include "select.cuh"
#include "tc.cuh"

namespace beam {
namespace {

constexpr int kTok = 128;                          // tokens per CTA (TMEM lanes)
constexpr int kThreads = 320;                      // producer, MMA, 8 epilogue warps
constexpr int kPartial = 4;                        // k-blocks per TMEM partial sum
constexpr uint32_t kATile = kTok * kBlockK * 2;    // 16 KiB
constexpr uint32_t kBTile = kExperts * kBlockK * 2;  // 32 KiB
constexpr uint32_t kStage = kATile + kBTile;
constexpr int kStages = 4;
constexpr int kLd = kExperts + 4;                  // logits row stride (floats)
constexpr int kDispatchTiles = kTok / kRouterTile;  // 4 dispatch tiles per CTA

// W (fp32 [E, H]) -> three BF16 terms [3][E][H].
__global__ void __launch_bounds__(256) router_split_kernel(const float* w, int n, __nv_bfloat16* out) {
  for (int i = 4 * (blockIdx.x * blockDim.x + threadIdx.x); i < n; i += 4 * gridDim.x * blockDim.x) {
    const float4 v = *reinterpret_cast<const float4*>(w + i);
    const float x[4] = {v.x, v.y, v.z, v.w};
    __nv_bfloat16 t[3][4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const __nv_bfloat16 a = __float2bfloat16_rn(x[j]);
      const float r1 = x[j] - __bfloat162float(a);  // exact
      const __nv_bfloat16 b = __float2bfloat16_rn(r1);
      const float r2 = r1 - __bfloat162float(b);    // exact
      t[0][j] = a;
      t[1][j] = b;
      t[2][j] = __float2bfloat16_rn(r2);
    }
#pragma unroll
    for (int s = 0; s < 3; ++s) *reinterpret_cast<uint2*>(out + static_cast<size_t>(s) * n + i) = *reinterpret_cast<uint2*>(t[s]);
  }
}

struct TcSmemTail {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t pfull[2];   // TMEM partial buffer b holds a finished partial sum
  uint64_t pempty[2];  // ... and has been added into the registers
  uint64_t drain;
  uint32_t tmem_slot;
  uint32_t abort_flag;
  int hist[kDispatchTiles][kExperts];
};

__global__ void __launch_bounds__(kThreads, 1)
    router_tc_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                     RouterParams p, uint32_t* status, uint64_t timeout_ns) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  TcSmemTail& tail = *reinterpret_cast<TcSmemTail*>(smem + kStages * kStage);
  float* logits = reinterpret_cast<float*>(smem);  // reuses the stage memory after the mainloop
  volatile uint32_t* abort_flag = &tail.abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blockIdx.x * kTok;
  const int kb_per = p.H / kBlockK;
  const int split = blockIdx.y;
  // this CTA's k-blocks [kb_lo, kb_hi) of the 3 x kb_per (term-major) sequence
  const int kb_lo = static_cast<int>(static_cast<long long>(3 * kb_per) * split / p.splits);
  const int kb_hi = static_cast<int>(static_cast<long long>(3 * kb_per) * (split + 1) / p.splits);
  const int total_kb = kb_hi - kb_lo;

  for (int i = threadIdx.x; i < kDispatchTiles * kExperts; i += kThreads) (&tail.hist[0][0])[i] = 0;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&tail.full[s], 1);
      mbar_init(&tail.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tail.pfull[b], 1);
      mbar_init(&tail.pempty[b], 8);
    }
    mbar_init(&tail.drain, 1);
    tail.abort_flag = 0u;
    fence_mbar_init();
    tma_prefetch_desc(&tm_x);
    tma_prefetch_desc(&tm_w);
  }
  if (warp == 1) tmem_alloc(&tail.tmem_slot, 2 * kExperts);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = tail.tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      for (int kb = 0; kb < total_kb; ++kb) {
        if (!mbar_wait(&tail.empty[stage], phase ^ 1u, timeout_ns, abort_flag, status, kWhereProducerEmpty)) break;
        mbar_arrive_expect_tx(&tail.full[stage], kStage);
        const int g = kb_lo + kb;  // position in the 3 x kb_per sequence
        const int kx = (g % kb_per) * kBlockK;
        uint8_t* st = smem + stage * kStage;
        tma_load_2d_nohint(st, &tm_x, &tail.full[stage], kx, t0);
        tma_load_2d_nohint(st + kATile, &tm_w, &tail.full[stage], kx, (g / kb_per) * kExperts);
        ++issued;
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      for (int s = 0; s < kStages; ++s) {  // drain
        if (issued <= s && issued < kStages) continue;
        const uint32_t par = s < stage ? phase : (phase ^ 1u);
        mbar_wait(&tail.full[s], par, timeout_ns, nullptr, status, kWhereDrain);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(kTok, kExperts);
      int stage = 0, buf = 0;
      uint32_t phase = 0, buf_phase = 0;
      bool ok = true;
      for (int kb = 0; kb < total_kb && ok; ++kb) {
        const int in_part = kb % kPartial;
        if (in_part == 0) {
          if (!mbar_wait(&tail.pempty[buf], buf_phase ^ 1u, timeout_ns, abort_flag, status, kWhereMmaAccEmpty)) {
            ok = false;
            break;
          }
          tc_fence_after();
        }
        if (!mbar_wait(&tail.full[stage], phase, timeout_ns, abort_flag, status, kWhereMmaFull)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint8_t* st = smem + stage * kStage;
        const uint64_t da = sdesc_k_sw128(smem_u32(st));
        const uint64_t db = sdesc_k_sw128(smem_u32(st + kATile));
        const uint32_t d = tmem_base + static_cast<uint32_t>(buf) * kExperts;
#pragma unroll
        for (int k = 0; k < kBlockK / 16; ++k) mma_bf16(d, da + 2u * k, db + 2u * k, idesc, (in_part | k) != 0 ? 1u : 0u);
        mma_commit(&tail.empty[stage]);
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
        if (in_part == kPartial - 1 || kb == total_kb - 1) {
          mma_commit(&tail.pfull[buf]);
          if (++buf == 2) {
            buf = 0;
            buf_phase ^= 1u;
          }
        }
      }
      mma_commit(&tail.drain);
      mbar_wait(&tail.drain, 0, timeout_ns, nullptr, status, kWhereDrain);
    }
  } else {
    // warp w: TMEM lanes (tokens) 32*(w%4).., experts 128*h .. +127
    const int quad = warp & 3;
    const int half = (warp - 2) >> 2;
    float acc[kExperts / 2];
#pragma unroll
    for (int i = 0; i < kExperts / 2; ++i) acc[i] = 0.0f;
    const int nparts = (total_kb + kPartial - 1) / kPartial;
    int buf = 0;
    uint32_t buf_phase = 0;
    bool ok = true;
    for (int part = 0; part < nparts; ++part) {
      int good = 1;
      if (lane == 0) good = mbar_wait(&tail.pfull[buf], buf_phase, timeout_ns, abort_flag, status, kWhereEpiAccFull) ? 1 : 0;
      good = __shfl_sync(0xFFFFFFFFu, good, 0);
      if (!good) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + static_cast<uint32_t>(buf) * kExperts +
                             static_cast<uint32_t>(half * (kExperts / 2));
#pragma unroll
      for (int c0 = 0; c0 < kExperts / 2; c0 += 16) {
        float v[16];
        tmem_ld16(tbase + static_cast<uint32_t>(c0), v);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j) acc[c0 + j] += v[j];  // FP32, round to nearest
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tail.pempty[buf]);
      if (++buf == 2) {
        buf = 0;
        buf_phase ^= 1u;
      }
    }
    if (ok && p.splits > 1) {
      // partial logits of this K range -> part[split][t][:]
      const int t = t0 + quad * 32 + lane;
      if (t < p.T) {
        float* row = p.part + (static_cast<size_t>(split) * p.T + t) * kExperts + half * (kExperts / 2);
#pragma unroll
        for (int j = 0; j < kExperts / 2; j += 4)
          *reinterpret_cast<float4*>(row + j) = make_float4(acc[j], acc[j + 1], acc[j + 2], acc[j + 3]);
      }
    } else if (ok) {
      // every stage's TMA bytes were consumed by the MMAs before the last
      // partial sum completed, so the stage memory can hold the logits
      float* row = logits + (quad * 32 + lane) * kLd + half * (kExperts / 2);
#pragma unroll
      for (int j = 0; j < kExperts / 2; j += 4) *reinterpret_cast<float4*>(row + j) = make_float4(acc[j], acc[j + 1], acc[j + 2], acc[j + 3]);
    }
  }
  __syncthreads();
  if (p.splits > 1) {
    // the select kernel counts the tile histogram with atomics: the first
    // K range zeroes this CTA's dispatch tiles
    if (split == 0) {
      for (int i = threadIdx.x; i < kDispatchTiles * kExperts; i += kThreads) {
        const int sub = i / kExperts, e = i % kExperts;
        const int dt = blockIdx.x * kDispatchTiles + sub;
        if (dt < p.n_tiles) p.tile_hist[static_cast<size_t>(e) * p.n_tiles + dt] = 0;
      }
    }
  } else if (tail.abort_flag == 0u) {
    // warp-per-token selection, all 6 warps
    for (int j = warp; j < kTok; j += kThreads / 32) {
      const int t = t0 + j;
      if (t >= p.T) break;
      int id;
      float wv;
      select_token(logits + j * kLd, p.bias, p.scale, lane, id, wv);
      if (lane < kTopK) {
        p.ids[static_cast<size_t>(t) * kTopK + lane] = id;
        p.w[static_cast<size_t>(t) * kTopK + lane] = wv;
        atomicAdd(&tail.hist[j / kRouterTile][id], 1);
      }
    }
  }
  __syncthreads();
  if (p.splits == 1) {
    for (int i = threadIdx.x; i < kDispatchTiles * kExperts; i += kThreads) {
      const int sub = i / kExperts, e = i % kExperts;
      const int dt = blockIdx.x * kDispatchTiles + sub;
      if (dt < p.n_tiles) p.tile_hist[static_cast<size_t>(e) * p.n_tiles + dt] = tail.hist[sub][e];
    }
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 2 * kExperts);
  }
}

}  // namespace

size_t router_tc_smem_bytes() { return 1024 + kStages * kStage + sizeof(TcSmemTail); }

int router_tc_splits(int T, int H, int num_sms, int split_cap) {
  const int tiles = (T + kTok - 1) / kTok;
  int s = num_sms / tiles;  // about one CTA per SM
  if (s > split_cap) s = split_cap;
  const int kbs = 3 * (H / kBlockK);
  if (s > kbs / kPartial) s = kbs / kPartial;  // at least one whole partial sum per range
  return s < 1 ? 1 : s;
}

cudaError_t launch_router_tc(const CUtensorMap& tm_x, const CUtensorMap& tm_w, const RouterParams& p,
                             __nv_bfloat16* wsplit, uint32_t* status, uint64_t timeout_ns, int num_sms,
                             cudaStream_t stream) {
  const int n = kExperts * p.H;
  int blocks = (n / 4 + 255) / 256;
  if (blocks > 4 * num_sms) blocks = 4 * num_sms;
  router_split_kernel<<<blocks, 256, 0, stream>>>(p.wr, n, wsplit);
  const size_t smem = router_tc_smem_bytes();
  cudaError_t err = cudaFuncSetAttribute(router_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  const dim3 grid((p.T + kTok - 1) / kTok, p.splits);
  router_tc_kernel<<<grid, kThreads, smem, stream>>>(tm_x, tm_w, p, status, timeout_ns);
  if (p.splits > 1) {
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    return launch_router_select(p, stream);
  }
  return cudaGetLastError();
}

}  // namespace beam

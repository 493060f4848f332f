// noalloc.cu -- routing for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc or hand this library a workspace: a
// host framework that owns all device memory and passes a plugin only its
// inputs and outputs, or a latency-critical serving loop that must never
// allocate (an allocation can stall the whole device).  For them
// beam_moe_route_noalloc runs the same router kernels as beam_moe_route, but
// its scratch (the per-split partial logits and the per-tile expert
// histograms) lives in the file-scope device array below, which the library
// holds on every GPU that loads it, until the process exits.
//
// Limits: at most kNoAllocMaxTokens tokens; the split of the hidden
// dimension across CTAs is reduced so that the partial logits fit in
// kNoAllocPartRows rows of E floats.  Nothing in the scratch has to start at
// zero (every call writes every element it later reads), but every call
// shares it, so two calls that overlap on the GPU race.
#include <cuda_runtime.h>

#include <mutex>

#include "beam_moe.h"
#include "moe_internal.cuh"

namespace beam {
namespace {

constexpr int kNoAllocMaxTokens = 65536;
constexpr int kNoAllocMaxTiles = kNoAllocMaxTokens / kRouterTile;  // 2048
constexpr size_t kNoAllocPartRows = 4096;                          // rows of E partial logits
constexpr size_t kHistBytes = static_cast<size_t>(kExperts) * kNoAllocMaxTiles * 4;   // 2 MiB
constexpr size_t kPartBytes = kNoAllocPartRows * kExperts * 4;                        // 4 MiB
constexpr size_t kScratchBytes = kHistBytes + kPartBytes;                             // 6 MiB

static __device__ __align__(256) unsigned char g_route_scratch[kScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_ptr[64] = {};

// Device address of g_route_scratch on the current device (looked up once
// per device, with that device current).
beam_status_t scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return BEAM_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || p == nullptr) return BEAM_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return BEAM_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace beam

using namespace beam;

extern "C" beam_status_t beam_moe_route_noalloc(const beam_moe_shape_t* shape, const void* x, beam_dtype_t xdtype,
                                                const float* router_w, const float* router_bias, int32_t* topk_ids,
                                                float* topk_w, void* stream) {
  if (shape == nullptr) return BEAM_ERR_INVALID_ARG;
  if (shape->T < 1 || shape->H < 1 || shape->I < 1) return BEAM_ERR_INVALID_ARG;
  if (shape->E != kExperts || shape->n_group != kGroups || shape->topk_group != kGroupsKept ||
      shape->top_k != kTopK || shape->H % 128 != 0 || shape->H > 65536)
    return BEAM_ERR_UNSUPPORTED;
  if (shape->T > kNoAllocMaxTokens) return BEAM_ERR_UNSUPPORTED;  // beyond the static scratch
  if (!(shape->routed_scale == shape->routed_scale) || shape->routed_scale > 3.4e38f ||
      shape->routed_scale < -3.4e38f)
    return BEAM_ERR_INVALID_ARG;
  if (!x || !router_w || !topk_ids || !topk_w) return BEAM_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(router_w) || !aligned16(topk_ids) || !aligned16(topk_w) ||
      (router_bias && !aligned16(router_bias)))
    return BEAM_ERR_INVALID_ARG;
  if (xdtype != BEAM_F32 && xdtype != BEAM_BF16) return BEAM_ERR_UNSUPPORTED;

  void* scratch = nullptr;
  const beam_status_t st = scratch_address(&scratch);
  if (st != BEAM_OK) return st;
  int sms = 0, dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return BEAM_ERR_CUDA;

  RouterParams p;
  p.x = x;
  p.wr = router_w;
  p.bias = router_bias;
  p.T = shape->T;
  p.H = shape->H;
  p.scale = shape->routed_scale;
  p.n_kchunks = shape->H / kRouterKChunk;
  p.n_tiles = (shape->T + kRouterTile - 1) / kRouterTile;
  int splits = router_splits(shape->T, shape->H, sms);
  const int fit = static_cast<int>(kNoAllocPartRows / static_cast<size_t>(shape->T));
  if (splits > fit) splits = fit;
  if (splits < 1) splits = 1;
  p.splits = splits;
  p.tile_hist = static_cast<int32_t*>(scratch);
  p.part = reinterpret_cast<float*>(static_cast<unsigned char*>(scratch) + kHistBytes);
  p.ids = topk_ids;
  p.w = topk_w;
  return launch_router(p, xdtype == BEAM_BF16, static_cast<cudaStream_t>(stream)) == cudaSuccess ? BEAM_OK
                                                                                                : BEAM_ERR_CUDA;
}

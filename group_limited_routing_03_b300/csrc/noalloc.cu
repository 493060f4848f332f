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
// kNoAllocPartRows rows of E floats: at most 4096 / T splits, so every
// T > 2048 runs one split per 32-token tile (beam_moe_route splits the
// hidden dimension up to T = 4704 on a 148-SM B300), and the selection is
// fused into the logits kernel.  Nothing in the scratch has to start at zero
// (every call writes every element it later reads), but every call shares
// it, so two calls that overlap on the GPU race.
#include <cuda.h>
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

// Device address of g_route_scratch, per CUDA context.  Host code only sees
// a host-side stand-in under that name, so the address is looked up with
// cudaGetSymbolAddress in the context that will run the kernels.  The cache
// is keyed by the context's unique id (cuCtxGetId), which no later context
// reuses: after cudaDeviceReset, or under another context of the same device,
// the address is looked up afresh instead of reusing one that belongs to a
// dead or different context.
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

struct DriverFns {
  CtxGetCurrentFn get_current = nullptr;
  CtxGetIdFn get_id = nullptr;
};

const DriverFns& driver_fns() {
  static DriverFns fns;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fns.get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fns.get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  return fns;
}

constexpr int kCacheSlots = 64;
struct CacheEntry {
  unsigned long long ctx_id;
  void* ptr;
};
std::mutex g_scratch_mu;
CacheEntry g_scratch_cache[kCacheSlots] = {};
int g_scratch_next = 0;

// Unique id of the context current to this thread (false: none yet, or the
// driver does not report it).
bool current_context_id(unsigned long long* id) {
  const DriverFns& fns = driver_fns();
  CUcontext ctx = nullptr;
  return fns.get_current != nullptr && fns.get_id != nullptr && fns.get_current(&ctx) == CUDA_SUCCESS &&
         ctx != nullptr && fns.get_id(ctx, id) == CUDA_SUCCESS;
}

beam_status_t scratch_address(void** out) {
  unsigned long long id = 0;
  bool keyed = current_context_id(&id);
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (keyed) {
    for (int i = 0; i < kCacheSlots; ++i)
      if (g_scratch_cache[i].ptr != nullptr && g_scratch_cache[i].ctx_id == id) {
        *out = g_scratch_cache[i].ptr;
        return BEAM_OK;
      }
  }
  // set-up for this context (the runtime binds its primary context to the
  // thread here if none was current)
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || p == nullptr) return BEAM_ERR_CUDA;
  if (!keyed) keyed = current_context_id(&id);
  if (keyed) {  // replaces the oldest entry once every slot is taken
    g_scratch_cache[g_scratch_next] = CacheEntry{id, p};
    g_scratch_next = (g_scratch_next + 1) % kCacheSlots;
  }
  *out = p;
  return BEAM_OK;
}

}  // namespace
}  // namespace beam

using namespace beam;

extern "C" beam_status_t beam_moe_route_noalloc(const beam_moe_shape_t* shape, const void* x, beam_dtype_t xdtype,
                                                const float* router_w, const float* router_bias, int32_t* topk_ids,
                                                float* topk_w, void* stream) {
  beam_status_t st = check_shape(shape);  // the rules of beam_moe_route ...
  if (st != BEAM_OK) return st;
  if (shape->T > kNoAllocMaxTokens) return BEAM_ERR_UNSUPPORTED;  // ... and the static scratch's limit
  st = check_route_args(x, xdtype, router_w, router_bias, topk_ids, topk_w);
  if (st != BEAM_OK) return st;

  void* scratch = nullptr;
  st = scratch_address(&scratch);
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

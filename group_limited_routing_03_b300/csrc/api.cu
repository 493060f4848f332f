// api.cu -- the C ABI declared in include/beam_moe.h: argument validation,
// workspace carve-up, TMA descriptors and the launch sequence
//   router -> [tile histogram] -> scan -> scatter -> gather (FP8 weights: E4M3
//   codes of x) -> gate/up GEMM -> [FP8: E4M3 codes of h] -> down GEMM ->
//   combine (or the combine fused with the post-norm residual update)
// and, for the dense MLP, schedule -> [FP8: codes of x] -> gate/up GEMM
// [-> K-split finish] -> [FP8: codes of h] -> down GEMM [-> K-split finish],
// all on the caller's stream, with no host synchronisation and no allocation.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>

#include "beam_moe.h"
#include "moe_internal.cuh"

namespace beam {
namespace {

constexpr uint64_t kDefaultTimeoutNs = 1000000000ull;  // 1 s per bounded wait

// NVFP4 weights, with BF16 activations carried exactly in FP16 (W4A16) or
// with activations quantised to NVFP4 at run time (W4A4): the same weight
// arrays, GEMM kernels and workspace; only the activation rows differ.
inline bool is_nvfp4(beam_dtype_t t) { return t == BEAM_NVFP4 || t == BEAM_NVFP4_A4; }
inline bool known_wdtype(beam_dtype_t t) { return t == BEAM_BF16 || t == BEAM_FP8 || is_nvfp4(t); }
#if defined(BEAM_DEBUG) && BEAM_DEBUG
constexpr bool kDebugBuild = true;  // device checks of every workspace index (see tc.cuh)
#else
constexpr bool kDebugBuild = false;
#endif

// ------------------------------------------------------------------ device
struct DeviceInfo {
  int sms = 0;
  int smem_optin = 0;
  int cc_major = 0;
};

std::mutex g_mu;
DeviceInfo g_dev[64];
bool g_dev_ok[64] = {};

bool device_info(DeviceInfo& out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_dev_ok[dev]) {
    DeviceInfo d;
    if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return false;
    if (cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
      return false;
    if (cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return false;
    g_dev[dev] = d;
    g_dev_ok[dev] = true;
  }
  out = g_dev[dev];
  return true;
}

// ------------------------------------------------------------------ TMA
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 2-D row-major matrix of 16-bit elements [rows, inner] (BF16, or FP16 for
// the NVFP4 path's activations); boxes of box_rows x 64 elements, 128-byte
// swizzle.
bool make_bf16_map(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint32_t box_rows,
                   CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {inner * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kBlockK), box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D row-major byte matrix [rows, inner_bytes], boxes box_rows x box_inner
// bytes, no swizzle (NVFP4 packed codes and block scales).
bool make_u8_map(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint32_t box_inner,
                 uint32_t box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {inner};
  const cuuint32_t box[2] = {box_inner, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D view of a tensor: dims d (innermost first), byte strides of dims 1 and
// 2 (any order: the innermost dimension is contiguous), box b.
bool make_3d_map(CUtensorMap* map, CUtensorMapDataType dt, const void* base, const uint64_t (&d)[3],
                 const uint64_t (&stride)[2], const uint32_t (&b)[3], CUtensorMapSwizzle swz) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  const cuuint64_t dims[3] = {d[0], d[1], d[2]};
  const cuuint64_t strides[2] = {stride[0], stride[1]};
  const cuuint32_t box[3] = {b[0], b[1], b[2]};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, dt, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D row-major byte matrix [rows, inner], boxes box_rows x 128 bytes with the
// 128-byte swizzle the MMA descriptors expect (FP8 operand tiles).
bool make_u8_sw128_map(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint32_t box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {inner};
  const cuuint32_t box[2] = {128, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ------------------------------------------------------------------ layout
// FP8 weights: the E4M3 codes of x (xq, R_pad x H bytes) and of h (hq, R_pad x
// I bytes, I <= H) share the xp region, which the BF16 rows do not use then;
// xs / hs hold their row scales (R_pad + 32 floats: the GEMM epilogue reads
// the scales of whole 16-column groups).
struct Layout {
  size_t status, sched, counts, offsets, chunk_prefix, tile_hist, part, wsplit, perm, pos, xp, h, yr, xs, hs, total;
  size_t xq, hq;
  int n_tiles, split_cap;
};

size_t align256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

void make_layout(const beam_moe_shape_t& s, Layout& L) {
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align256(off + bytes);
    return o;
  };
  const size_t T = static_cast<size_t>(s.T), H = static_cast<size_t>(s.H), I = static_cast<size_t>(s.I);
  const size_t R = T * kTopK;
  // Activation buffers hold whole 32-row TMA boxes; rows past R are never
  // read into a used accumulator column.
  const size_t R_pad = (R + kBoxRows - 1) / kBoxRows * kBoxRows;
  L.n_tiles = static_cast<int>((T + kRouterTile - 1) / kRouterTile);
  L.split_cap = router_split_cap(s.T, s.H);
  L.status = take(16);
  L.sched = take(16);
  L.counts = take(kExperts * 4);
  L.offsets = take((kExperts + 1) * 4);
  L.chunk_prefix = take((kExperts + 1) * 4);
  L.tile_hist = take(static_cast<size_t>(kExperts) * L.n_tiles * 4);
  L.part = take(L.split_cap > 1 ? static_cast<size_t>(L.split_cap) * T * kExperts * 4 : 0);
  L.wsplit = take(s.T >= kRouterTcMinTokens ? 3 * static_cast<size_t>(kExperts) * H * 2 : 0);
  L.perm = take(R * 4);
  L.pos = take(R * 4);
  L.xp = take(R_pad * H * 2);
  L.h = take(R_pad * I * 2);
  L.yr = take(R_pad * H * 2);
  L.xs = take((R_pad + 32) * 4);
  L.hs = take((R_pad + 32) * 4);
  L.xq = L.xp;
  L.hq = L.xp + align256(R_pad * H);
  L.total = off;
}

// ------------------------------------------------------------------ checks
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int chunk_rows(int T, bool fp4);
int split_parts(int units, int k_blocks);

// Dense MLP workspace: status, unit counters, the one-expert schedule, h, and
// for FP8 weights the codes of x and h with their row scales.
struct DenseLayout {
  size_t status, sched, counts, offsets, chunk_prefix, h, xq, hq, xs, hs, x16, partial, total;
};

// NVFP4 weights also need x as FP16 rows (x16, T_pad x H).
void make_dense_layout(const beam_dense_shape_t& s, beam_dtype_t wdtype, DenseLayout& L) {
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align256(off + bytes);
    return o;
  };
  const size_t T = static_cast<size_t>(s.T), H = static_cast<size_t>(s.H), I = static_cast<size_t>(s.I);
  const size_t T_pad = (T + kBoxRows - 1) / kBoxRows * kBoxRows;
  L.status = take(16);
  L.sched = take(16);
  L.counts = take(kExperts * 4);
  L.offsets = take((kExperts + 1) * 4);
  L.chunk_prefix = take((kExperts + 1) * 4);
  L.h = take(T_pad * I * 2);
  L.xq = take(T_pad * H);
  L.hq = take(T_pad * I);
  L.xs = take((T_pad + 32) * 4);
  L.hs = take((T_pad + 32) * 4);
  L.x16 = take(is_nvfp4(wdtype) ? T_pad * H * 2 : 0);
  // K-split partial planes: the larger of gate/up (two planes of T x I per
  // part) and down (one of T x H), parts as run_gemm picks them for BF16
  // weights (FP8 has half the k-blocks, so never more parts)
  const int nmax = chunk_rows(s.T, false);
  const int chunks = (s.T + nmax - 1) / nmax;
  const size_t gu = static_cast<size_t>(split_parts(chunks * (s.I / kBlockM), s.H / kBlockK));
  const size_t dn = static_cast<size_t>(split_parts(chunks * (s.H / kBlockM), s.I / kBlockK));
  const size_t need = std::max(gu > 1 ? gu * 2 * T * I : 0, dn > 1 ? dn * T * H : 0);
  L.partial = take(need * 4);
  L.total = off;
}

// The dense shape as a block shape (the block's constants; only T, H, I are read).
beam_moe_shape_t dense_as_moe(const beam_dense_shape_t& s) {
  beam_moe_shape_t m;
  m.T = s.T;
  m.H = s.H;
  m.I = s.I;
  m.E = kExperts;
  m.n_group = kGroups;
  m.topk_group = kGroupsKept;
  m.top_k = kTopK;
  m.routed_scale = 1.0f;
  return m;
}

beam_status_t check_workspace(const beam_moe_shape_t* s, const void* ws, size_t bytes, Layout& L) {
  make_layout(*s, L);
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0 || bytes < L.total) return BEAM_ERR_WORKSPACE;
  return BEAM_OK;
}

// shared_codes: FP8 h codes live in the x-code buffer (the block's workspace),
// which needs I <= H; the dense MLP's workspace has its own.
beam_status_t check_weights(const beam_moe_shape_t* s, const beam_expert_weights_t* w, bool shared_codes = true) {
  if (w == nullptr) return BEAM_ERR_INVALID_ARG;
  if (w->layout != BEAM_LAYOUT_ROWS && w->layout != BEAM_LAYOUT_TILED) return BEAM_ERR_INVALID_ARG;
  if (w->dtype == BEAM_FP8) {
    if (!w->gate || !w->up || !w->down || !w->gate_rs || !w->up_rs || !w->down_rs) return BEAM_ERR_INVALID_ARG;
    if (!aligned16(w->gate) || !aligned16(w->up) || !aligned16(w->down) || !aligned16(w->gate_rs) ||
        !aligned16(w->up_rs) || !aligned16(w->down_rs))
      return BEAM_ERR_INVALID_ARG;
    if (w->gate_sf || w->up_sf || w->down_sf || w->gate_gs || w->up_gs || w->down_gs) return BEAM_ERR_INVALID_ARG;
    // h's codes share the x-code buffer (I <= H); the k-block is 128 elements
    if (shared_codes && s->I > s->H) return BEAM_ERR_UNSUPPORTED;
    return BEAM_OK;
  }
  if (w->gate_rs || w->up_rs || w->down_rs) return BEAM_ERR_INVALID_ARG;
  if (w->dtype == BEAM_BF16) {
    if (!w->gate || !w->up || !w->down) return BEAM_ERR_INVALID_ARG;
    if (!aligned16(w->gate) || !aligned16(w->up) || !aligned16(w->down)) return BEAM_ERR_INVALID_ARG;
    if (w->gate_sf || w->up_sf || w->down_sf || w->gate_gs || w->up_gs || w->down_gs) return BEAM_ERR_INVALID_ARG;
    return BEAM_OK;
  }
  if (is_nvfp4(w->dtype)) {
    if (!w->gate || !w->up || !w->down || !w->gate_sf || !w->up_sf || !w->down_sf || !w->gate_gs || !w->up_gs ||
        !w->down_gs)
      return BEAM_ERR_INVALID_ARG;
    if (!aligned16(w->gate) || !aligned16(w->up) || !aligned16(w->down) || !aligned16(w->gate_sf) ||
        !aligned16(w->up_sf) || !aligned16(w->down_sf) || !aligned16(w->gate_gs) || !aligned16(w->up_gs) ||
        !aligned16(w->down_gs))
      return BEAM_ERR_INVALID_ARG;
    // scale rows of K/16 bytes must be whole 16-byte TMA strides
    if (s->H % 256 != 0 || s->I % 256 != 0) return BEAM_ERR_UNSUPPORTED;
    return BEAM_OK;
  }
  return BEAM_ERR_UNSUPPORTED;
}

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

beam_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? BEAM_OK : BEAM_ERR_CUDA; }

// ------------------------------------------------------------------ stages
// Large batches of BF16 tokens route on the tensor cores (three-term BF16
// split of the FP32 router weight); small batches and FP32 x on CUDA cores.
bool use_router_tc(const beam_moe_shape_t& s, bool x_bf16, const DeviceInfo& d) {
  return x_bf16 && s.T >= kRouterTcMinTokens && d.cc_major >= 10 &&
         router_tc_smem_bytes() <= static_cast<size_t>(d.smem_optin);
}

beam_status_t run_route(const beam_moe_shape_t& s, const void* x, bool x_bf16, const float* wr, const float* bias,
                        int32_t* ids, float* w, void* ws, const Layout& L, const DeviceInfo& d,
                        cudaStream_t stream) {
  RouterParams p;
  p.x = x;
  p.wr = wr;
  p.bias = bias;
  p.T = s.T;
  p.H = s.H;
  p.scale = s.routed_scale;
  p.splits = router_splits(s.T, s.H, d.sms);
  if (p.splits > L.split_cap) p.splits = L.split_cap;
  p.n_kchunks = s.H / kRouterKChunk;
  p.n_tiles = L.n_tiles;
  p.part = at<float>(ws, L.part);
  p.ids = ids;
  p.w = w;
  p.tile_hist = at<int32_t>(ws, L.tile_hist);
  if (use_router_tc(s, x_bf16, d)) {
    CUtensorMap tm_x, tm_w;
    __nv_bfloat16* wsplit = at<__nv_bfloat16>(ws, L.wsplit);
    if (!make_bf16_map(&tm_x, x, static_cast<uint64_t>(s.H), static_cast<uint64_t>(s.T), 128) ||
        !make_bf16_map(&tm_w, wsplit, static_cast<uint64_t>(s.H), 3ull * kExperts, kExperts))
      return BEAM_ERR_CUDA;
    p.splits = router_tc_splits(s.T, s.H, d.sms, L.split_cap);
    return cuda_status(
        launch_router_tc(tm_x, tm_w, p, wsplit, at<uint32_t>(ws, L.status), kDefaultTimeoutNs, d.sms, stream));
  }
  return cuda_status(launch_router(p, x_bf16, stream));
}

beam_status_t run_dispatch(const beam_moe_shape_t& s, const int32_t* ids, void* ws, const Layout& L, int nmax,
                           bool hist_ready, cudaStream_t stream) {
  const int R = s.T * kTopK;
  cudaError_t e;
  if (!hist_ready) {
    e = launch_tile_hist(ids, R, L.n_tiles, at<int32_t>(ws, L.tile_hist), at<uint32_t>(ws, L.status), stream);
    if (e != cudaSuccess) return BEAM_ERR_CUDA;
  }
  e = launch_dispatch(ids, R, L.n_tiles, at<int32_t>(ws, L.tile_hist), at<int32_t>(ws, L.counts),
                      at<int32_t>(ws, L.offsets), at<int32_t>(ws, L.chunk_prefix), nmax, at<int32_t>(ws, L.perm),
                      at<int32_t>(ws, L.pos), at<uint32_t>(ws, L.status), stream);
  return cuda_status(e);
}

// Routes per GEMM unit: all of an expert's routes up to a cap (BF16 256, the
// widest MMA; NVFP4 160, so that TMEM also holds a ring of FP16 weight tiles).
int chunk_rows(int T, bool fp4) {
  // NVFP4 with few routes per expert (T <= 256: 8 on average): chunks of 16
  // leave TMEM room for the decode variant's accumulators and tile rings
  if (fp4 && T <= kFp4SmallT) return kDecChunkRows;
  const int cap = fp4 ? kChunkRowsFp4 : kChunkRowsBf16;
  int n = ((T + kBoxRows - 1) / kBoxRows) * kBoxRows;
  return n > cap ? cap : n;
}

uint32_t pow2_at_least(uint32_t v) {
  uint32_t p = 32;
  while (p < v) p <<= 1;
  return p;
}

// Token rows into route order: BF16 (BF16 weights), E4M3 codes with row
// scales (FP8 weights) or FP16 rows times a power of two (NVFP4 weights).
beam_status_t run_gather(const beam_moe_shape_t& s, const void* x, bool x_bf16, beam_dtype_t wdtype, void* ws,
                         const Layout& L, const DeviceInfo& d, cudaStream_t stream) {
  if (wdtype == BEAM_FP8)
    return cuda_status(launch_gather_q8(x, x_bf16, s.H, at<int32_t>(ws, L.pos), s.T, at<uint8_t>(ws, L.xq),
                                        at<float>(ws, L.xs), at<uint32_t>(ws, L.status), stream));
  if (wdtype == BEAM_NVFP4_A4)
    return cuda_status(launch_gather_a4(x, x_bf16, s.H, at<int32_t>(ws, L.pos), s.T, at<__half>(ws, L.xp),
                                        at<float>(ws, L.xs), at<uint32_t>(ws, L.status), stream));
  if (wdtype == BEAM_NVFP4)
    return cuda_status(launch_gather_f16(x, x_bf16, s.H, at<int32_t>(ws, L.pos), s.T, at<__half>(ws, L.xp),
                                         at<float>(ws, L.xs), at<uint32_t>(ws, L.status), stream));
  return cuda_status(launch_gather(x, x_bf16, s.H, at<int32_t>(ws, L.pos), s.T, at<__nv_bfloat16>(ws, L.xp), d.sms,
                                   at<uint32_t>(ws, L.status), stream));
}

// mode 0: gate/up (+SwiGLU) -> h; mode 1: down -> yr.
// The buffers and sizes one pair of grouped GEMMs works on: the MoE block
// (T*8 route rows over 256 experts, in the workspace) or the dense MLP (T
// rows, one "expert", x itself as the gate/up input).
struct GemmIO {
  int R;                // route rows
  int nmax;             // routes per unit at most
  uint64_t n_exp;       // experts stacked in the weight arrays
  const void* xp;       // BF16 gate/up input rows [xp_rows, H]
  uint64_t xp_rows;     // rows of that tensor (whole TMA boxes past R read zeros or unused rows)
  __nv_bfloat16* h;     // [R_pad, I]
  __nv_bfloat16* out;   // down output [R, H]
  uint8_t* xq;          // FP8: codes of the gate/up input rows [R_pad, H]
  uint8_t* hq;          // FP8: codes of h [R_pad, I]
  float* xs;            // FP8: their row scales [R_pad + 32]
  float* hs;
  int32_t* counts;
  int32_t* offsets;
  int32_t* chunk_prefix;
  int* sched;           // two unit counters (gate/up, down)
  uint32_t* status;
  int split_chunks;     // K split allowed: the number of token chunks (known on the host), else 0
  float* partial;       // K split: FP32 partial planes (see split_parts)
};

// K split of a grouped GEMM with few units: enough parts for about four
// units per SM of a 148-SM B300, each part at least four k-blocks, at most
// 16 parts.  1: no split.
constexpr int kSplitTargetUnits = 592;
int split_parts(int units, int k_blocks) {
  if (units <= 0 || units >= kSplitTargetUnits) return 1;
  int ks = (kSplitTargetUnits + units - 1) / units;
  if (ks > 16) ks = 16;
  if (ks > k_blocks / 4) ks = k_blocks / 4;
  return ks < 2 ? 1 : ks;
}

GemmIO moe_io(const beam_moe_shape_t& s, void* ws, const Layout& L, bool fp4) {
  GemmIO io;
  io.R = s.T * kTopK;
  io.nmax = chunk_rows(s.T, fp4);
  io.n_exp = kExperts;
  io.xp = at<__nv_bfloat16>(ws, L.xp);
  io.xp_rows = static_cast<uint64_t>((io.R + kBoxRows - 1) / kBoxRows * kBoxRows);
  io.h = at<__nv_bfloat16>(ws, L.h);
  io.out = at<__nv_bfloat16>(ws, L.yr);
  io.xq = at<uint8_t>(ws, L.xq);
  io.hq = at<uint8_t>(ws, L.hq);
  io.xs = at<float>(ws, L.xs);
  io.hs = at<float>(ws, L.hs);
  io.counts = at<int32_t>(ws, L.counts);
  io.offsets = at<int32_t>(ws, L.offsets);
  io.chunk_prefix = at<int32_t>(ws, L.chunk_prefix);
  io.sched = at<int>(ws, L.sched);
  io.status = at<uint32_t>(ws, L.status);
  io.split_chunks = 0;  // the block's chunk count is known only on the device
  io.partial = nullptr;
  return io;
}

// The GEMM variant run_gemm launches.  CTA pairs (one M=256 MMA per unit over
// two SMs) halve each SM's shared-memory operand traffic; used for BF16 / FP8
// weights when chunks reach 256 routes and a pair fits on the device (a pair
// tile's stage is fixed: two weight tiles, 128 token rows per CTA, one 2 x
// 256-column accumulator).  K split: only with a host-known chunk count
// (split_chunks > 0), one CTA per unit, BF16 / FP8.
struct GemmChoice {
  bool pair;
  int clusters;
  int k_splits;
};

GemmChoice choose_gemm(int mode, const beam_moe_shape_t& s, bool fp4, bool fp8, int nmax, int split_chunks,
                       const DeviceInfo& d) {
  GemmChoice c{false, 0, 1};
  // shared memory for the stages: all but the barriers, unit ring and
  // alignment slack of the deepest pipeline (gemm_smem_bytes with no stage bytes)
  const size_t budget = static_cast<size_t>(d.smem_optin) - gemm_smem_bytes(kMaxStages, 4, 0);
  c.pair = !fp4 && nmax == 256 && s.H % 512 == 0 && s.I % 256 == 0 && d.sms >= 2;
  if (c.pair) {
    const size_t sbp = gemm_stage_bytes(2, false, nmax / 2);
    int stp = static_cast<int>(budget / sbp);
    if (stp > kMaxStages) stp = kMaxStages;
    c.clusters = stp >= 2 ? gemm_pair_max_clusters(mode, gemm_smem_bytes(stp, 1, sbp)) : 0;
    if (c.clusters <= 0) c.pair = false;
  }
  const int k_blocks = (mode == 0 ? s.H : s.I) / (fp8 ? 2 * kBlockK : kBlockK);
  if (split_chunks > 0 && !c.pair && !fp4)
    c.k_splits = split_parts(split_chunks * ((mode == 0 ? s.I : s.H) / kBlockM), k_blocks);
  return c;
}

beam_status_t run_gemm(int mode, const beam_moe_shape_t& s, const beam_expert_weights_t* wts, const GemmIO& io,
                       const DeviceInfo& d, cudaStream_t stream) {
  const int R = io.R;
  const uint64_t R_pad = static_cast<uint64_t>((R + kBoxRows - 1) / kBoxRows * kBoxRows);
  const bool fp4 = is_nvfp4(wts->dtype);
  const bool fp8 = wts->dtype == BEAM_FP8;
  const int nmax = io.nmax;
  // FP8 / NVFP4: h's row conversion comes first (its scales need whole rows
  // of h): E4M3 codes into hq, or FP16 in place
  if (fp8 && mode == 1) {
    const cudaError_t e = launch_quantize_rows(io.h, R, s.I, io.hq, io.hs, stream);
    if (e != cudaSuccess) return BEAM_ERR_CUDA;
  }
  if (fp4 && mode == 1) {
    const cudaError_t e = wts->dtype == BEAM_NVFP4_A4 ? launch_rows_to_a4(io.h, R, s.I, io.hs, stream)
                                                       : launch_rows_to_f16(io.h, R, s.I, io.hs, stream);
    if (e != cudaSuccess) return BEAM_ERR_CUDA;
  }
  // NVFP4: the activation operand holds FP16 rows (kind::f16 takes A and B
  // of one type)
  const CUtensorMapDataType act_dt = fp4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const void* xp = io.xp;
  __nv_bfloat16* h = io.h;
  __nv_bfloat16* yr = io.out;
  const uint64_t E = io.n_exp, H = s.H, I = s.I;
  GemmMaps maps;
  std::memset(&maps, 0, sizeof(maps));
  bool ok;
  // Weight maps of an [E * N, K] matrix (N rows per expert): row-major, or
  // the tiled layout seen as a column of 128-row tiles whose rows are one
  // box wide (64 BF16 / 32 code bytes / 16 scale bytes), each box one tile.
  const bool tiled = wts->layout == BEAM_LAYOUT_TILED;
  auto wmap_bf16 = [&](CUtensorMap* m, const void* base, uint64_t N, uint64_t K) {
    return tiled ? make_bf16_map(m, base, kBlockK, E * N * (K / kBlockK), kBlockM)
                 : make_bf16_map(m, base, K, E * N, kBlockM);
  };
  auto wmap_codes = [&](CUtensorMap* m, const void* base, uint64_t N, uint64_t K) {
    return tiled ? make_u8_map(m, base, kBlockK / 2, E * N * (K / kBlockK), kBlockK / 2, kBlockM)
                 : make_u8_map(m, base, K / 2, E * N, kBlockK / 2, kBlockM);
  };
  auto wmap_scales = [&](CUtensorMap* m, const void* base, uint64_t N, uint64_t K) {
    return tiled ? make_u8_map(m, base, kScaleBoxCols, E * N * (K / (16 * kScaleBoxCols)), kScaleBoxCols, kBlockM)
                 : make_u8_map(m, base, K / 16, E * N, kScaleBoxCols, kBlockM);
  };
  // FP8: E4M3 weight tiles of 128 rows x 128 bytes (128 K elements)
  auto wmap_f8 = [&](CUtensorMap* m, const void* base, uint64_t N, uint64_t K) {
    return tiled ? make_u8_sw128_map(m, base, 128, E * N * (K / 128), kBlockM) : make_u8_sw128_map(m, base, K, E * N, kBlockM);
  };
  uint8_t* xq = io.xq;
  uint8_t* hq = io.hq;
  if (fp8) {
    if (mode == 0)
      ok = make_u8_sw128_map(&maps.b, xq, H, R_pad, kBoxRows) && wmap_f8(&maps.a0, wts->gate, I, H) &&
           wmap_f8(&maps.a1, wts->up, I, H);
    else
      ok = make_u8_sw128_map(&maps.b, hq, I, R_pad, kBoxRows) && wmap_f8(&maps.a0, wts->down, H, I);
    if (mode == 1) maps.a1 = maps.a0;
  } else if (mode == 0) {
    ok = make_bf16_map(&maps.b, xp, H, io.xp_rows, kBoxRows, act_dt);
    if (fp4)
      ok = ok && wmap_codes(&maps.a0, wts->gate, I, H) && wmap_codes(&maps.a1, wts->up, I, H) &&
           wmap_scales(&maps.s0, wts->gate_sf, I, H) && wmap_scales(&maps.s1, wts->up_sf, I, H);
    else
      ok = ok && wmap_bf16(&maps.a0, wts->gate, I, H) && wmap_bf16(&maps.a1, wts->up, I, H);
  } else {
    ok = make_bf16_map(&maps.b, h, I, R_pad, kBoxRows, act_dt);
    if (fp4)
      ok = ok && wmap_codes(&maps.a0, wts->down, H, I) && wmap_scales(&maps.s0, wts->down_sf, H, I);  // a1 / s1 = a0 / s0
    else
      ok = ok && wmap_bf16(&maps.a0, wts->down, H, I);
    maps.a1 = maps.a0;
    maps.s1 = maps.s0;
  }
  if (!ok) return BEAM_ERR_CUDA;
  // CTA pairs (one M=256 MMA per unit over two SMs) halve each SM's shared-
  // memory operand traffic; used for BF16 weights when chunks reach 256 routes.
  // Decided first, so the tiling below is derived once for the kernel that
  // runs: a pair tile's stage is fixed (two weight tiles, 128 token rows per
  // CTA, one 2 x 256-column accumulator), and if no pair fits on the device
  // the GEMM runs one CTA per unit.
  // shared memory for the stages: all but the barriers, unit ring and
  // alignment slack of the deepest pipeline (gemm_smem_bytes with no stage bytes)
  const size_t budget = static_cast<size_t>(d.smem_optin) - gemm_smem_bytes(kMaxStages, 4, 0);
  const GemmChoice gc = choose_gemm(mode, s, fp4, fp8, nmax, io.partial != nullptr ? io.split_chunks : 0, d);
  const bool pair = gc.pair;
  const int clusters = gc.clusters;
  // pair units: gate/up 256 features (gate and up tiles), down 512 features.
  // Down on one CTA per unit: 256 features (two weight tiles, two
  // accumulators: two MMA chains per k-block) for NVFP4, and for BF16 when H
  // allows ("wide"); else 128.  K split: 128-row units.
  const int k_blocks = (mode == 0 ? s.H : s.I) / (fp8 ? 2 * kBlockK : kBlockK);
  const int k_splits = gc.k_splits;
  // NVFP4 with chunks of at most 64 routes (decode): more converter warps
  const bool dec = fp4 && nmax <= kDecChunkRows;
  const bool wide = mode == 1 && !pair && !fp4 && s.H % 256 == 0 && k_splits == 1;
  const int rows_per_unit =
      pair ? (mode == 0 ? 2 * kBlockM : 4 * kBlockM) : ((fp4 || wide) && mode == 1 ? 2 * kBlockM : kBlockM);
  GemmParams p;
  p.counts = io.counts;
  p.offsets = io.offsets;
  p.chunk_prefix = io.chunk_prefix;
  p.m_tiles = (mode == 0 ? s.I : s.H) / rows_per_unit;
  p.a_rows_per_expert = mode == 0 ? s.I : s.H;
  p.k_blocks = k_blocks;
  p.k_splits = k_splits;
  p.rows = R;
  p.partial = k_splits > 1 ? io.partial : nullptr;
  p.a_tiled = tiled ? 1 : 0;
  p.nmax = nmax;
  const int num_a = (mode == 0 || pair || fp4 || wide) ? 2 : 1;  // weight tiles per stage
  // NVFP4 in the tiled layout: several k-blocks per stage (four with small
  // chunks, two otherwise), so one stage is five TMA loads (codes and scales
  // of both matrices, the activations as a 3-D box) for several k-blocks
  const int sub = (fp4 && tiled) ? (nmax <= kDecChunkRows ? 4 : 2) : 1;
  const size_t sb = gemm_stage_bytes(num_a, fp4, pair ? nmax / 2 : nmax, sub);
  int stages = static_cast<int>(budget / sb);
  if (stages > kMaxStages) stages = kMaxStages;
  if (stages < 2) return BEAM_ERR_UNSUPPORTED;
  p.stages = stages;
  // NVFP4 decode variant: two accumulators per matrix (alternate K steps)
  p.acc_cols = static_cast<uint32_t>(num_a * nmax * (dec ? 2 : 1));
  int acc_stages = static_cast<int>(512 / p.acc_cols);
  if (acc_stages > 4) acc_stages = 4;
  if (acc_stages < 1) acc_stages = 1;
  p.acc_stages = acc_stages;
  p.tmem_cols = pow2_at_least(static_cast<uint32_t>(acc_stages) * p.acc_cols);
  p.a_stages = 0;
  p.a_col0 = 0;
  if (fp4) {
    // TMEM (512 columns): the accumulator buffer(s), then a ring of BF16
    // weight tiles (32 columns per 128x64 tile) with room for at least three
    const uint32_t a_cols = static_cast<uint32_t>(num_a * (kBlockK / 2));
    acc_stages = static_cast<int>((512 - 3 * a_cols) / p.acc_cols);
    if (acc_stages > 2) acc_stages = 2;
    if (acc_stages < 1) return BEAM_ERR_UNSUPPORTED;
    p.acc_stages = acc_stages;
    p.a_col0 = static_cast<uint32_t>(acc_stages) * p.acc_cols;
    p.a_stages = static_cast<int>((512 - p.a_col0) / a_cols);
    if (p.a_stages > kMaxAStages) p.a_stages = kMaxAStages;
    // converter groups G = 3 (decode) or 2; a group's consecutive k-blocks
    // lie at most 2G - 1 apart, and a tile must come back to it no sooner
    if (p.a_stages < (dec ? 5 : 3)) return BEAM_ERR_UNSUPPORTED;
    p.tmem_cols = 512;
  }
  p.sub_blocks = sub;
  p.sched = io.sched + mode;
  p.out = mode == 0 ? h : yr;
  p.out_ld = mode == 0 ? s.I : s.H;
  p.gs0 = fp4 ? (mode == 0 ? wts->gate_gs : wts->down_gs) : nullptr;
  p.gs1 = fp4 && mode == 0 ? wts->up_gs : nullptr;
  p.rs0 = fp8 ? (mode == 0 ? wts->gate_rs : wts->down_rs) : nullptr;
  p.rs1 = fp8 && mode == 0 ? wts->up_rs : nullptr;
  p.bscale = (fp8 || fp4) ? (mode == 0 ? io.xs : io.hs) : nullptr;
  p.status = io.status;
  p.timeout_ns = kDefaultTimeoutNs;
  const size_t smem = gemm_smem_bytes(stages, acc_stages, sb);
  // persistent: one CTA per SM, or as many pairs as can be resident at once
  // (a TPC with a disabled SM cannot host one)
  const int grid = pair ? 2 * (clusters < d.sms / 2 ? clusters : d.sms / 2) : d.sms;
  // activations in one box per k-block: the B tile's full height
  p.b_big_rows = pair ? nmax / 2 : nmax;
  if (fp8) {
    if (!make_u8_sw128_map(&maps.bb, mode == 0 ? xq : hq, mode == 0 ? H : I, R_pad, static_cast<uint32_t>(p.b_big_rows)))
      return BEAM_ERR_CUDA;
  } else if (!make_bf16_map(&maps.bb, mode == 0 ? xp : static_cast<const void*>(h), mode == 0 ? H : I,
                            mode == 0 ? io.xp_rows : R_pad, static_cast<uint32_t>(p.b_big_rows), act_dt)) {
    return BEAM_ERR_CUDA;
  }
  if (sub > 1) {
    // packed codes: the tiled layout as (byte, row, tile), boxes of `sub`
    // consecutive tiles; activations as (element, row, k-block), boxes of the
    // chunk's rows for `sub` k-blocks (their B tiles one after another)
    const uint64_t N = mode == 0 ? I : H, K = mode == 0 ? H : I;
    const uint64_t tiles = E * N / kBlockM * (K / kBlockK);
    const uint64_t cd[3] = {kBlockK / 2, kBlockM, tiles};
    const uint64_t cs[2] = {kBlockK / 2, kPackedTileBytes};
    const uint32_t cb[3] = {kBlockK / 2, kBlockM, static_cast<uint32_t>(sub)};
    const void* c0 = mode == 0 ? wts->gate : wts->down;
    const void* c1 = mode == 0 ? wts->up : wts->down;
    const void* act = mode == 0 ? xp : static_cast<const void*>(h);
    const uint64_t ad[3] = {kBlockK, mode == 0 ? io.xp_rows : R_pad, K / kBlockK};
    const uint64_t as[2] = {K * 2, kBlockK * 2};
    const uint32_t ab[3] = {kBlockK, static_cast<uint32_t>(p.b_big_rows), static_cast<uint32_t>(sub)};
    if (!make_3d_map(&maps.a0, CU_TENSOR_MAP_DATA_TYPE_UINT8, c0, cd, cs, cb, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_3d_map(&maps.a1, CU_TENSOR_MAP_DATA_TYPE_UINT8, c1, cd, cs, cb, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_3d_map(&maps.bb, act_dt, act, ad, as, ab, CU_TENSOR_MAP_SWIZZLE_128B))
      return BEAM_ERR_CUDA;
  }
  if (cudaMemsetAsync(p.sched, 0, sizeof(int), stream) != cudaSuccess) return BEAM_ERR_CUDA;
  if (kDebugBuild &&
      launch_validate_schedule(io.counts, io.offsets, io.chunk_prefix, R, nmax, io.status, stream) != cudaSuccess)
    return BEAM_ERR_CUDA;
  if (launch_gemm(mode, fp4, pair, wide, fp8, dec, maps, p, grid, smem, stream) != cudaSuccess) return BEAM_ERR_CUDA;
  if (k_splits > 1)
    return cuda_status(launch_splitk_finish(mode, io.partial, k_splits, R, p.out_ld, mode == 0 ? h : yr, stream));
  return BEAM_OK;
}

beam_status_t run_combine(const beam_moe_shape_t& s, const float* w, void* y, bool y_bf16, void* ws, const Layout& L,
                          cudaStream_t stream) {
  return cuda_status(
      launch_combine(at<__nv_bfloat16>(ws, L.yr), at<int32_t>(ws, L.pos), w, s.T, s.H, y, y_bf16,
                     at<uint32_t>(ws, L.status), stream));
}

beam_status_t run_experts(const beam_moe_shape_t& s, const void* x, bool x_bf16, const beam_expert_weights_t* wts,
                          const int32_t* ids, const float* w, void* y, void* ws, const Layout& L,
                          const DeviceInfo& d, bool hist_ready, cudaStream_t stream) {
  beam_status_t st = run_dispatch(s, ids, ws, L, chunk_rows(s.T, is_nvfp4(wts->dtype)), hist_ready, stream);
  if (st == BEAM_OK) st = run_gather(s, x, x_bf16, wts->dtype, ws, L, d, stream);
  if (st == BEAM_OK) st = run_gemm(0, s, wts, moe_io(s, ws, L, is_nvfp4(wts->dtype)), d, stream);
  if (st == BEAM_OK) st = run_gemm(1, s, wts, moe_io(s, ws, L, is_nvfp4(wts->dtype)), d, stream);
  if (st == BEAM_OK) st = run_combine(s, w, y, x_bf16, ws, L, stream);
  return st;
}

// The residual-update arguments: pointers set and aligned, out either the
// stream itself or disjoint from it, y (when written) disjoint from both,
// step >= 2, eps finite and >= 0.
beam_status_t check_residual(const beam_moe_shape_t* s, const beam_residual_t& r, beam_dtype_t xdtype,
                             const void* y) {
  if (!r.stream || !r.out || !r.norm_weight) return BEAM_ERR_INVALID_ARG;
  if (!aligned16(r.stream) || !aligned16(r.out) || !aligned16(r.norm_weight)) return BEAM_ERR_INVALID_ARG;
  if (r.step < 2 || !std::isfinite(r.eps) || r.eps < 0.0f) return BEAM_ERR_INVALID_ARG;
  const size_t len = static_cast<size_t>(s->T) * s->H * (xdtype == BEAM_BF16 ? 2 : 4);
  auto overlap = [len](const void* p, const void* q) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p), b = reinterpret_cast<uintptr_t>(q);
    return a < b + len && b < a + len;
  };
  if (r.out != r.stream && overlap(r.out, r.stream)) return BEAM_ERR_INVALID_ARG;
  if (y && (overlap(y, r.out) || overlap(y, r.stream))) return BEAM_ERR_INVALID_ARG;
  return BEAM_OK;
}

beam_status_t run_combine_residual(const beam_moe_shape_t& s, const float* w, const beam_residual_t& res, void* y,
                                   bool bf16, void* ws, const Layout& L, cudaStream_t stream) {
  ResidualParams r;
  r.stream = res.stream;
  r.out = res.out;
  r.norm_w = res.norm_weight;
  r.eps = res.eps;
  r.keep = static_cast<float>(std::sqrt(static_cast<double>(res.step - 1) / res.step));
  r.add = static_cast<float>(1.0 / std::sqrt(static_cast<double>(res.step)));
  return cuda_status(launch_combine_residual(at<__nv_bfloat16>(ws, L.yr), at<int32_t>(ws, L.pos), w, s.T, s.H, r, y,
                                             bf16, at<uint32_t>(ws, L.status), stream));
}

// Validation shared by beam_moe_forward, beam_moe_forward_stage and
// beam_moe_forward_residual.
beam_status_t check_forward(const beam_moe_shape_t* shape, const beam_moe_args_t& a, void* workspace,
                            size_t workspace_bytes, Layout& L, DeviceInfo& d) {
  beam_status_t st = check_shape(shape);
  if (st != BEAM_OK) return st;
  if (!a.x || !a.router_w || !a.topk_ids || !a.topk_w || (!a.y && !a.residual)) return BEAM_ERR_INVALID_ARG;
  if (!aligned16(a.x) || !aligned16(a.router_w) || !aligned16(a.topk_ids) || !aligned16(a.topk_w) ||
      (a.y && !aligned16(a.y)) || (a.router_bias && !aligned16(a.router_bias)))
    return BEAM_ERR_INVALID_ARG;
  if (a.xdtype != BEAM_F32 && a.xdtype != BEAM_BF16) return BEAM_ERR_UNSUPPORTED;
  if (a.residual) {
    st = check_residual(shape, *a.residual, a.xdtype, a.y);
    if (st != BEAM_OK) return st;
  }
  st = check_weights(shape, a.weights);
  if (st != BEAM_OK) return st;
  st = check_workspace(shape, workspace, workspace_bytes, L);
  if (st != BEAM_OK) return st;
  if (!device_info(d)) return BEAM_ERR_CUDA;
  if (d.cc_major < 10) return BEAM_ERR_UNSUPPORTED;
  return BEAM_OK;
}

beam_status_t run_stage(const beam_moe_shape_t& s, const beam_moe_args_t& a, int stage, void* ws, const Layout& L,
                        const DeviceInfo& d, cudaStream_t cs) {
  const bool xb = a.xdtype == BEAM_BF16;
  switch (stage) {
    case BEAM_STAGE_ROUTE:
      return run_route(s, a.x, xb, a.router_w, a.router_bias, a.topk_ids, a.topk_w, ws, L, d, cs);
    case BEAM_STAGE_DISPATCH:
      return run_dispatch(s, a.topk_ids, ws, L, chunk_rows(s.T, is_nvfp4(a.weights->dtype)), true, cs);
    case BEAM_STAGE_GATHER:
      return run_gather(s, a.x, xb, a.weights->dtype, ws, L, d, cs);
    case BEAM_STAGE_GATE_UP:
      return run_gemm(0, s, a.weights, moe_io(s, ws, L, is_nvfp4(a.weights->dtype)), d, cs);
    case BEAM_STAGE_DOWN:
      return run_gemm(1, s, a.weights, moe_io(s, ws, L, is_nvfp4(a.weights->dtype)), d, cs);
    case BEAM_STAGE_COMBINE:
      if (a.residual) return run_combine_residual(s, a.topk_w, *a.residual, a.y, xb, ws, L, cs);
      return run_combine(s, a.topk_w, a.y, xb, ws, L, cs);
  }
  return BEAM_ERR_INVALID_ARG;
}

}  // namespace

beam_status_t check_shape(const beam_moe_shape_t* s) {
  if (s == nullptr) return BEAM_ERR_INVALID_ARG;
  if (s->T < 1 || s->H < 1 || s->I < 1) return BEAM_ERR_INVALID_ARG;
  if (s->E != kExperts || s->n_group != kGroups || s->topk_group != kGroupsKept || s->top_k != kTopK)
    return BEAM_ERR_UNSUPPORTED;
  if (s->H % 128 != 0 || s->I % 128 != 0 || s->H > 65536 || s->I > 65536 || s->T > (1 << 20))
    return BEAM_ERR_UNSUPPORTED;
  if (!std::isfinite(s->routed_scale)) return BEAM_ERR_INVALID_ARG;
  return BEAM_OK;
}

beam_status_t check_route_args(const void* x, beam_dtype_t xdtype, const float* router_w, const float* router_bias,
                               const int32_t* topk_ids, const float* topk_w) {
  if (!x || !router_w || !topk_ids || !topk_w) return BEAM_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(router_w) || !aligned16(topk_ids) || !aligned16(topk_w) ||
      (router_bias && !aligned16(router_bias)))
    return BEAM_ERR_INVALID_ARG;
  if (xdtype != BEAM_F32 && xdtype != BEAM_BF16) return BEAM_ERR_UNSUPPORTED;
  return BEAM_OK;
}

}  // namespace beam

using namespace beam;

extern "C" {

size_t beam_moe_workspace_size(const beam_moe_shape_t* shape, beam_dtype_t wdtype) {
  if (check_shape(shape) != BEAM_OK) return 0;
  if (!known_wdtype(wdtype)) return 0;
  Layout L;
  make_layout(*shape, L);
  return L.total;
}

beam_status_t beam_moe_workspace_layout(const beam_moe_shape_t* shape, beam_dtype_t wdtype, beam_ws_layout_t* out) {
  const beam_status_t st = check_shape(shape);
  if (st != BEAM_OK) return st;
  if (out == nullptr) return BEAM_ERR_INVALID_ARG;
  if (!known_wdtype(wdtype)) return BEAM_ERR_UNSUPPORTED;
  Layout L;
  make_layout(*shape, L);
  out->xq = L.xq;
  out->hq = L.hq;
  out->xs = L.xs;
  out->hs = L.hs;
  out->status = L.status;
  out->counts = L.counts;
  out->offsets = L.offsets;
  out->perm = L.perm;
  out->pos = L.pos;
  out->xp = L.xp;
  out->h = L.h;
  out->yr = L.yr;
  out->total = L.total;
  return BEAM_OK;
}

beam_status_t beam_moe_route(const beam_moe_shape_t* shape, const void* x, beam_dtype_t xdtype,
                             const float* router_w, const float* router_bias, int32_t* topk_ids, float* topk_w,
                             void* workspace, size_t workspace_bytes, void* stream) {
  beam_status_t st = check_shape(shape);
  if (st != BEAM_OK) return st;
  st = check_route_args(x, xdtype, router_w, router_bias, topk_ids, topk_w);
  if (st != BEAM_OK) return st;
  Layout L;
  st = check_workspace(shape, workspace, workspace_bytes, L);
  if (st != BEAM_OK) return st;
  DeviceInfo d;
  if (!device_info(d)) return BEAM_ERR_CUDA;
  return run_route(*shape, x, xdtype == BEAM_BF16, router_w, router_bias, topk_ids, topk_w, workspace, L, d,
                   static_cast<cudaStream_t>(stream));
}

beam_status_t beam_moe_dispatch(const beam_moe_shape_t* shape, const int32_t* topk_ids, void* workspace,
                                size_t workspace_bytes, void* stream) {
  beam_status_t st = check_shape(shape);
  if (st != BEAM_OK) return st;
  if (!topk_ids || !aligned16(topk_ids)) return BEAM_ERR_INVALID_ARG;
  Layout L;
  st = check_workspace(shape, workspace, workspace_bytes, L);
  if (st != BEAM_OK) return st;
  DeviceInfo d;
  if (!device_info(d)) return BEAM_ERR_CUDA;
  return run_dispatch(*shape, topk_ids, workspace, L, chunk_rows(shape->T, false), false, static_cast<cudaStream_t>(stream));
}

beam_status_t beam_moe_experts(const beam_moe_shape_t* shape, const void* x, beam_dtype_t xdtype,
                               const beam_expert_weights_t* weights, const int32_t* topk_ids, const float* topk_w,
                               void* y, void* workspace, size_t workspace_bytes, void* stream) {
  beam_status_t st = check_shape(shape);
  if (st != BEAM_OK) return st;
  if (!x || !topk_ids || !topk_w || !y) return BEAM_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(topk_ids) || !aligned16(topk_w) || !aligned16(y)) return BEAM_ERR_INVALID_ARG;
  if (xdtype != BEAM_F32 && xdtype != BEAM_BF16) return BEAM_ERR_UNSUPPORTED;
  st = check_weights(shape, weights);
  if (st != BEAM_OK) return st;
  Layout L;
  st = check_workspace(shape, workspace, workspace_bytes, L);
  if (st != BEAM_OK) return st;
  DeviceInfo d;
  if (!device_info(d)) return BEAM_ERR_CUDA;
  if (d.cc_major < 10) return BEAM_ERR_UNSUPPORTED;
  return run_experts(*shape, x, xdtype == BEAM_BF16, weights, topk_ids, topk_w, y, workspace, L, d, false,
                     static_cast<cudaStream_t>(stream));
}

beam_status_t beam_moe_forward(const beam_moe_shape_t* shape, const void* x, beam_dtype_t xdtype,
                               const float* router_w, const float* router_bias, const beam_expert_weights_t* weights,
                               void* y, int32_t* topk_ids, float* topk_w, void* workspace, size_t workspace_bytes,
                               void* stream) {
  const beam_moe_args_t a = {x, xdtype, router_w, router_bias, weights, y, topk_ids, topk_w};
  Layout L;
  DeviceInfo d;
  beam_status_t st = check_forward(shape, a, workspace, workspace_bytes, L, d);
  if (st != BEAM_OK) return st;
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  for (int stage = 0; stage < BEAM_STAGE_COUNT && st == BEAM_OK; ++stage)
    st = run_stage(*shape, a, stage, workspace, L, d, cs);
  return st;
}

beam_status_t beam_moe_forward_residual(const beam_moe_shape_t* shape, const beam_moe_args_t* args, void* workspace,
                                        size_t workspace_bytes, void* stream) {
  if (args == nullptr || args->residual == nullptr) return BEAM_ERR_INVALID_ARG;
  Layout L;
  DeviceInfo d;
  beam_status_t st = check_forward(shape, *args, workspace, workspace_bytes, L, d);
  if (st != BEAM_OK) return st;
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  for (int stage = 0; stage < BEAM_STAGE_COUNT && st == BEAM_OK; ++stage)
    st = run_stage(*shape, *args, stage, workspace, L, d, cs);
  return st;
}

beam_status_t beam_moe_forward_stage(const beam_moe_shape_t* shape, const beam_moe_args_t* args, beam_stage_t stage,
                                     void* workspace, size_t workspace_bytes, void* stream) {
  if (args == nullptr) return BEAM_ERR_INVALID_ARG;
  if (static_cast<int>(stage) < 0 || static_cast<int>(stage) >= BEAM_STAGE_COUNT) return BEAM_ERR_INVALID_ARG;
  Layout L;
  DeviceInfo d;
  const beam_status_t st = check_forward(shape, *args, workspace, workspace_bytes, L, d);
  if (st != BEAM_OK) return st;
  return run_stage(*shape, *args, stage, workspace, L, d, static_cast<cudaStream_t>(stream));
}

int32_t beam_moe_stage_kernel_count(const beam_moe_shape_t* shape, beam_dtype_t xdtype, beam_dtype_t wdtype,
                                    beam_stage_t stage) {
  if (check_shape(shape) != BEAM_OK) return -1;
  if (xdtype != BEAM_F32 && xdtype != BEAM_BF16) return -1;
  if (!known_wdtype(wdtype)) return -1;
  DeviceInfo d;
  if (!device_info(d)) return -1;
  switch (stage) {
    case BEAM_STAGE_ROUTE: {
      Layout L;
      make_layout(*shape, L);
      if (use_router_tc(*shape, xdtype == BEAM_BF16, d))  // weight split + logits (+ selection of split K)
        return router_tc_splits(shape->T, shape->H, d.sms, L.split_cap) > 1 ? 3 : 2;
      int sp = router_splits(shape->T, shape->H, d.sms);
      if (sp > L.split_cap) sp = L.split_cap;
      return sp > 1 ? 2 : 1;
    }
    case BEAM_STAGE_DISPATCH: return 2;
    // FP8 / NVFP4: h's rows converted first; debug builds check the schedule before each GEMM
    case BEAM_STAGE_DOWN: return (wdtype == BEAM_BF16 ? 1 : 2) + (kDebugBuild ? 1 : 0);
    case BEAM_STAGE_GATE_UP: return 1 + (kDebugBuild ? 1 : 0);
    case BEAM_STAGE_GATHER:
    case BEAM_STAGE_COMBINE: return 1;
    default: return -1;
  }
}

beam_status_t beam_moe_read_device_status(void* workspace, uint32_t* where, void* stream) {
  if (workspace == nullptr) return BEAM_ERR_WORKSPACE;
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  uint32_t word[4] = {0, 0, 0, 0};
  if (cudaStreamSynchronize(cs) != cudaSuccess) return BEAM_ERR_CUDA;
  if (cudaMemcpy(word, workspace, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return BEAM_ERR_CUDA;
  if (cudaMemset(workspace, 0, sizeof(word)) != cudaSuccess) return BEAM_ERR_CUDA;
  if (where != nullptr) *where = word[1];
  return static_cast<beam_status_t>(word[0]);
}

// Weight packing for n_exp stacked experts (256 for the block, 1 for the
// dense MLP).
static beam_status_t pack_impl(const beam_moe_shape_t* shape, size_t n_exp, const beam_expert_weights_t* src,
                               beam_expert_weights_t* dst, void* stream) {
  beam_status_t st = check_shape(shape);
  if (st != BEAM_OK) return st;
  if (src == nullptr || dst == nullptr || src->layout != BEAM_LAYOUT_ROWS || dst->dtype != src->dtype)
    return BEAM_ERR_INVALID_ARG;
  beam_expert_weights_t probe = *dst;
  probe.layout = BEAM_LAYOUT_TILED;
  st = check_weights(shape, src, n_exp == kExperts);
  if (st == BEAM_OK) st = check_weights(shape, &probe, n_exp == kExperts);
  if (st != BEAM_OK) return st;
  const size_t E = n_exp, H = shape->H, I = shape->I;
  const bool fp4 = is_nvfp4(src->dtype), fp8 = src->dtype == BEAM_FP8;
  // FP8 row scales keep their order: the same arrays serve both layouts
  if (fp8 && (dst->gate_rs != src->gate_rs || dst->up_rs != src->up_rs || dst->down_rs != src->down_rs))
    return BEAM_ERR_INVALID_ARG;
  // (array, rows, row bytes, tile row bytes) for gate, up, down [, their scales]
  struct Job {
    const void* s;
    const void* d;
    size_t rows, row_bytes;
    uint32_t tile_row_bytes;
  };
  Job jobs[6];
  int n = 0;
  const uint32_t wb = fp4 ? kBlockK / 2 : kBlockK * 2;  // tile row: 64 K elements (BF16, E2M1), 128 (E4M3)
  auto row_bytes = [&](size_t K) { return fp4 ? K / 2 : (fp8 ? K : K * 2); };
  jobs[n++] = {src->gate, dst->gate, E * I, row_bytes(H), wb};
  jobs[n++] = {src->up, dst->up, E * I, row_bytes(H), wb};
  jobs[n++] = {src->down, dst->down, E * H, row_bytes(I), wb};
  if (fp4) {
    jobs[n++] = {src->gate_sf, dst->gate_sf, E * I, H / 16, kScaleBoxCols};
    jobs[n++] = {src->up_sf, dst->up_sf, E * I, H / 16, kScaleBoxCols};
    jobs[n++] = {src->down_sf, dst->down_sf, E * H, I / 16, kScaleBoxCols};
  }
  for (int j = 0; j < n; ++j) {
    if (jobs[j].row_bytes % jobs[j].tile_row_bytes != 0 || jobs[j].rows % kBlockM != 0) return BEAM_ERR_UNSUPPORTED;
    // the arrays must not overlap
    const uintptr_t a = reinterpret_cast<uintptr_t>(jobs[j].s), b = reinterpret_cast<uintptr_t>(jobs[j].d);
    const size_t len = jobs[j].rows * jobs[j].row_bytes;
    if (a < b + len && b < a + len) return BEAM_ERR_INVALID_ARG;
  }
  DeviceInfo d;
  if (!device_info(d)) return BEAM_ERR_CUDA;
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  for (int j = 0; j < n; ++j) {
    const cudaError_t e = launch_pack_tiles(jobs[j].s, const_cast<void*>(jobs[j].d), jobs[j].rows, jobs[j].row_bytes,
                                            jobs[j].tile_row_bytes, d.sms, cs);
    if (e != cudaSuccess) return BEAM_ERR_CUDA;
  }
  dst->layout = BEAM_LAYOUT_TILED;
  return BEAM_OK;
}

beam_status_t beam_moe_pack_weights(const beam_moe_shape_t* shape, const beam_expert_weights_t* src,
                                    beam_expert_weights_t* dst, void* stream) {
  return pack_impl(shape, kExperts, src, dst, stream);
}

beam_status_t beam_dense_pack_weights(const beam_dense_shape_t* shape, const beam_expert_weights_t* src,
                                      beam_expert_weights_t* dst, void* stream) {
  if (shape == nullptr) return BEAM_ERR_INVALID_ARG;
  const beam_moe_shape_t ms = dense_as_moe(*shape);
  return pack_impl(&ms, 1, src, dst, stream);
}

int32_t beam_dense_kernel_count(const beam_dense_shape_t* shape, beam_dtype_t wdtype) {
  if (shape == nullptr) return -1;
  const beam_moe_shape_t ms = dense_as_moe(*shape);
  if (check_shape(&ms) != BEAM_OK) return -1;
  if (!known_wdtype(wdtype)) return -1;
  DeviceInfo d;
  if (!device_info(d)) return -1;
  const bool fp4 = is_nvfp4(wdtype), fp8 = wdtype == BEAM_FP8;
  const int nmax = chunk_rows(shape->T, fp4);
  const int chunks = (shape->T + nmax - 1) / nmax;
  int n = 1 + 1 + 1;        // schedule, gate/up, down
  if (kDebugBuild) n += 2;  // the schedule checked before each GEMM
  if (fp8 || fp4) n += 2;   // x and h rows converted (E4M3 codes / FP16)
  for (int mode = 0; mode < 2; ++mode)
    if (choose_gemm(mode, ms, fp4, fp8, nmax, chunks, d).k_splits > 1) n += 1;  // the finishing kernel
  return n;
}

size_t beam_dense_workspace_size(const beam_dense_shape_t* shape, beam_dtype_t wdtype) {
  if (shape == nullptr) return 0;
  const beam_moe_shape_t ms = dense_as_moe(*shape);
  if (check_shape(&ms) != BEAM_OK) return 0;
  if (!known_wdtype(wdtype)) return 0;
  DenseLayout L;
  make_dense_layout(*shape, wdtype, L);
  return L.total;
}

beam_status_t beam_dense_mlp_forward(const beam_dense_shape_t* shape, const void* x, beam_dtype_t xdtype,
                                     const beam_expert_weights_t* weights, void* y, void* workspace,
                                     size_t workspace_bytes, void* stream) {
  if (shape == nullptr) return BEAM_ERR_INVALID_ARG;
  const beam_moe_shape_t ms = dense_as_moe(*shape);
  beam_status_t st = check_shape(&ms);
  if (st != BEAM_OK) return st;
  if (!x || !y || !aligned16(x) || !aligned16(y)) return BEAM_ERR_INVALID_ARG;
  st = check_weights(&ms, weights, false);
  if (st != BEAM_OK) return st;
  const bool fp8 = weights->dtype == BEAM_FP8;
  if (xdtype != BEAM_BF16 && !(fp8 && xdtype == BEAM_F32)) return BEAM_ERR_UNSUPPORTED;
  DenseLayout L;
  make_dense_layout(*shape, weights->dtype, L);
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || workspace_bytes < L.total)
    return BEAM_ERR_WORKSPACE;
  DeviceInfo d;
  if (!device_info(d)) return BEAM_ERR_CUDA;
  if (d.cc_major < 10) return BEAM_ERR_UNSUPPORTED;
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  void* ws = workspace;
  GemmIO io;
  io.R = shape->T;
  io.nmax = chunk_rows(shape->T, is_nvfp4(weights->dtype));
  io.n_exp = 1;
  io.xp = x;  // BF16 x is the gate/up input itself, rows in token order
  io.xp_rows = static_cast<uint64_t>(shape->T);
  io.h = at<__nv_bfloat16>(ws, L.h);
  io.out = static_cast<__nv_bfloat16*>(y);
  io.xq = at<uint8_t>(ws, L.xq);
  io.hq = at<uint8_t>(ws, L.hq);
  io.xs = at<float>(ws, L.xs);
  io.hs = at<float>(ws, L.hs);
  io.counts = at<int32_t>(ws, L.counts);
  io.offsets = at<int32_t>(ws, L.offsets);
  io.chunk_prefix = at<int32_t>(ws, L.chunk_prefix);
  io.sched = at<int>(ws, L.sched);
  io.status = at<uint32_t>(ws, L.status);
  io.split_chunks = (io.R + io.nmax - 1) / io.nmax;
  io.partial = at<float>(ws, L.partial);
  if (launch_dense_dispatch(io.R, io.nmax, io.counts, io.offsets, io.chunk_prefix, cs) != cudaSuccess)
    return BEAM_ERR_CUDA;
  if (fp8 && launch_gather_q8(x, xdtype == BEAM_BF16, shape->H, nullptr, shape->T, io.xq, io.xs, io.status, cs) !=
                 cudaSuccess)
    return BEAM_ERR_CUDA;
  if (is_nvfp4(weights->dtype)) {  // x as FP16 rows: times a power of two (W4A16) or NVFP4 values (W4A4)
    io.xp = at<__half>(ws, L.x16);
    const cudaError_t e =
        weights->dtype == BEAM_NVFP4_A4
            ? launch_gather_a4(x, true, shape->H, nullptr, shape->T, at<__half>(ws, L.x16), io.xs, io.status, cs)
            : launch_gather_f16(x, true, shape->H, nullptr, shape->T, at<__half>(ws, L.x16), io.xs, io.status, cs);
    if (e != cudaSuccess) return BEAM_ERR_CUDA;
  }
  st = run_gemm(0, ms, weights, io, d, cs);
  if (st == BEAM_OK) st = run_gemm(1, ms, weights, io, d, cs);
  return st;
}

beam_status_t beam_moe_debug_timeout(void* workspace, size_t workspace_bytes, uint32_t timeout_us, void* stream) {
  if (workspace == nullptr || workspace_bytes < 16 || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return BEAM_ERR_WORKSPACE;
  if (timeout_us == 0 || timeout_us > 10000000u) return BEAM_ERR_INVALID_ARG;
  return cuda_status(launch_debug_timeout(static_cast<uint32_t*>(workspace), static_cast<uint64_t>(timeout_us) * 1000ull,
                                          static_cast<cudaStream_t>(stream)));
}

int32_t beam_moe_debug_build(void) { return kDebugBuild ? 1 : 0; }

const char* beam_status_string(beam_status_t status) {
  switch (status) {
    case BEAM_OK: return "ok";
    case BEAM_ERR_INVALID_ARG: return "invalid argument (null, misaligned or out-of-range value)";
    case BEAM_ERR_UNSUPPORTED: return "unsupported shape or data type";
    case BEAM_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case BEAM_ERR_CUDA: return "CUDA runtime or launch error";
    case BEAM_ERR_TIMEOUT: return "device: a bounded wait ran out";
    case BEAM_ERR_DEVICE_CHECK: return "device: a consistency check failed (e.g. an expert id out of range)";
  }
  return "unknown status";
}

}  // extern "C"

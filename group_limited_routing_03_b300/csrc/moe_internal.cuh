// moe_internal.cuh -- constants, parameter blocks and host-side launchers
// shared by the CUDA sources of the MoE library (not part of the C ABI).
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "beam_moe.h"

namespace beam {

constexpr int kExperts = 256;      // E
constexpr int kGroups = 8;         // groups of 32 contiguous experts
constexpr int kGroupsKept = 4;     // best groups kept
constexpr int kTopK = 8;           // experts per token
constexpr int kRouterTile = 32;    // tokens per router CTA (= one dispatch tile)
constexpr int kRouterKChunk = 32;  // hidden elements per router k-step
constexpr int kTileRoutes = kRouterTile * kTopK;  // routes per dispatch tile (256)
constexpr int kBlockM = 128;       // weight rows per MMA tile (TMEM lanes)
constexpr int kBlockK = 64;        // K elements per pipeline stage (128 bytes of bf16; FP8 stages hold 128)
constexpr int kBoxRows = 32;       // token rows per TMA box of the activation operand
constexpr int kMaxSmsForSizing = 256;  // bound on the SM count used to size the workspace
constexpr uint32_t kPackedTileBytes = kBlockM * kBlockK / 2;  // NVFP4: 128 rows x 32 bytes
constexpr uint32_t kScaleBoxCols = 16;                       // NVFP4: scale bytes per TMA box row (4 k-blocks)
constexpr uint32_t kScaleTileBytes = kBlockM * kScaleBoxCols;  // NVFP4: 2 KiB
constexpr int kMaxAStages = 8;     // NVFP4: BF16 weight tiles in TMEM in flight (at most)
constexpr int kMaxStages = 8;      // shared-memory ring depth
constexpr int kChunkRowsBf16 = 256;  // routes per GEMM unit (BF16 weights)
constexpr int kChunkRowsFp4 = 160;   // NVFP4: TMEM holds the accumulators and the weight tiles
constexpr int kFp4SmallT = 256;      // NVFP4: up to this many tokens, the decode variant (chunks of kDecChunkRows)

// ---------------------------------------------------------------------------
// Argument checks shared by the entry points (api.cu)
// ---------------------------------------------------------------------------
// The layer shape: BEAM_OK, BEAM_ERR_INVALID_ARG (null, non-positive size,
// non-finite scale) or BEAM_ERR_UNSUPPORTED (outside the supported set).
beam_status_t check_shape(const beam_moe_shape_t* s);
// The routing call's tensors: set, 16-byte aligned (bias may be null), x FP32
// or BF16.
beam_status_t check_route_args(const void* x, beam_dtype_t xdtype, const float* router_w, const float* router_bias,
                               const int32_t* topk_ids, const float* topk_w);

// ---------------------------------------------------------------------------
// Router
// ---------------------------------------------------------------------------
struct RouterParams {
  const void* x;        // [T, H] f32 or bf16
  const float* wr;      // [E, H]
  const float* bias;    // [E] or null
  int T, H;
  float scale;
  int splits;           // K splits (1: fused selection in the GEMM CTA)
  int n_kchunks;        // H / kRouterKChunk
  int n_tiles;          // ceil(T / kRouterTile)
  float* part;          // [splits, T, E] partial logits when splits > 1
  int32_t* ids;         // [T, 8]
  float* w;             // [T, 8]
  int32_t* tile_hist;   // [E, n_tiles] routes of tile per expert
};

// ---------------------------------------------------------------------------
// Grouped GEMM (gate/up with SwiGLU epilogue, or down)
// ---------------------------------------------------------------------------
struct GemmParams {
  const int32_t* counts;        // [E]
  const int32_t* offsets;       // [E+1]
  const int32_t* chunk_prefix;  // [E+1] exclusive scan of ceil(counts / nmax)
  int m_tiles;                  // weight rows per expert / rows per unit (128, or 256 for CTA pairs)
  int a_rows_per_expert;        // I (gate/up) or H (down)
  int k_blocks;                 // K / kBlockK
  int nmax;                     // tokens per chunk (multiple of kBoxRows, <= 256)
  int stages;                   // shared-memory pipeline depth
  int acc_stages;               // TMEM accumulator buffers
  uint32_t acc_cols;            // TMEM columns per accumulator buffer
  uint32_t tmem_cols;           // TMEM columns allocated (power of two)
  int b_big_rows;               // rows of the bb box (the B tile's capacity: nmax, or nmax / 2 for CTA pairs)
  int a_tiled;                  // weights (codes, scales) in BEAM_LAYOUT_TILED: every box is one contiguous tile
  int sub_blocks;               // NVFP4: k-blocks per pipeline stage (1, 2 or 4; divides k_blocks)
  int a_stages;                 // NVFP4: FP16 weight tiles in TMEM (ring depth)
  uint32_t a_col0;              // NVFP4: first TMEM column of that ring
  int* sched;                   // unit counter (zeroed before the launch)
  __nv_bfloat16* out;           // h [R, I] or yr [R, H], perm order
  int out_ld;                   // I or H
  const float* gs0;             // NVFP4 global scales (gate or down) [E], else null
  const float* gs1;             // NVFP4 global scale (up) [E], else null
  const float* rs0;             // FP8 row scales (gate or down) [E * rows], else null
  const float* rs1;             // FP8 row scales (up) [E * I], else null
  const float* bscale;          // FP8 token-row scales [R_pad + 32] (x or h rows, perm order), else null
  int k_splits;                 // parts of the K range per tile (1: none); > 1 only without CTA pairs / NVFP4
  int rows;                     // route rows R (K split: rows of one partial plane)
  float* partial;               // K split: FP32 sums [k_splits][planes][R][out_ld] (planes: 2 gate/up, 1 down), else null
  uint32_t* status;
  uint64_t timeout_ns;
};

// TMA descriptors of one grouped GEMM: weights a0 (gate or down) and a1 (up),
// activations b (boxes of kBoxRows rows) and bb (one box of a whole chunk,
// b_big_rows rows), and for NVFP4 the block scales s0 / s1 of a0 / a1.
struct GemmMaps {
  CUtensorMap a0, a1, b, bb, s0, s1;
};

// Bytes of one pipeline stage: the activation boxes plus, for BF16 weights,
// the weight tile(s), or for NVFP4 the packed tile(s) and scale tile(s) that
// the converters expand into TMEM; NVFP4 stages may hold `sub` consecutive
// k-blocks (activations and packed tiles of each, one scale tile per matrix).
__host__ __device__ inline size_t gemm_stage_bytes(int num_a, bool fp4, int nmax, int sub = 1) {
  const size_t b = static_cast<size_t>(sub) * nmax * kBlockK * 2;
  if (fp4) return b + static_cast<size_t>(num_a) * (sub * kPackedTileBytes + kScaleTileBytes);
  return b + static_cast<size_t>(num_a) * kBlockM * kBlockK * 2;
}

// ---------------------------------------------------------------------------
// Host launchers (each returns cudaGetLastError() of its launches)
// ---------------------------------------------------------------------------
int router_splits(int T, int H, int num_sms);
int router_split_cap(int T, int H);

cudaError_t launch_router(const RouterParams& p, bool x_bf16, cudaStream_t stream);
// Sum p.splits partial logits per token (in split order), select, count the
// tile histogram with atomics (zeroed by the logits kernel).
cudaError_t launch_router_select(const RouterParams& p, cudaStream_t stream);
// Tensor-core router (router_tc.cu) for BF16 x and large T: splits the FP32
// router weight into three BF16 terms (wsplit [3, E, H]) and runs the logits
// on tcgen05; tm_x = x [T, H] boxes 64x128, tm_w = wsplit [3E, H] boxes 64x256.
constexpr int kRouterTcMinTokens = 512;
size_t router_tc_smem_bytes();
// K ranges of the tensor-core router: about one CTA per SM, at most split_cap
// (the partial-logit rows the workspace holds).
int router_tc_splits(int T, int H, int num_sms, int split_cap);
cudaError_t launch_router_tc(const CUtensorMap& tm_x, const CUtensorMap& tm_w, const RouterParams& p,
                             __nv_bfloat16* wsplit, uint32_t* status, uint64_t timeout_ns, int num_sms,
                             cudaStream_t stream);
cudaError_t launch_tile_hist(const int32_t* ids, int R, int n_tiles, int32_t* tile_hist,
                             uint32_t* status, cudaStream_t stream);
cudaError_t launch_dispatch(const int32_t* ids, int R, int n_tiles, int32_t* tile_hist,
                            int32_t* counts, int32_t* offsets, int32_t* chunk_prefix, int nmax,
                            int32_t* perm, int32_t* pos, uint32_t* status, cudaStream_t stream);
// Debug builds, before each grouped GEMM: check the schedule (counts,
// offsets, chunk prefix) describes R routes with chunks of nmax; if not,
// record it in the status word and leave the GEMM no unit.
cudaError_t launch_validate_schedule(const int32_t* counts, const int32_t* offsets, int32_t* chunk_prefix, int R,
                                     int nmax, uint32_t* status, cudaStream_t stream);
// Dense MLP: the unit schedule of one expert holding all R rows.
cudaError_t launch_dense_dispatch(int R, int nmax, int32_t* counts, int32_t* offsets, int32_t* chunk_prefix,
                                  cudaStream_t stream);
cudaError_t launch_gather(const void* x, bool x_bf16, int H, const int32_t* pos, int T,
                          __nv_bfloat16* xp, int num_sms, uint32_t* status, cudaStream_t stream);
// FP8 weights: token rows (x in BF16 or FP32) to E4M3 codes in route order,
// one FP32 scale per row (amax / 448, 1 for a zero row); every token's codes
// are written to its 8 route rows (xq [R_pad, H], xs [R_pad]); pos == NULL
// (dense MLP): row t to row t.
cudaError_t launch_gather_q8(const void* x, bool x_bf16, int H, const int32_t* pos, int T, uint8_t* xq, float* xs,
                             uint32_t* status, cudaStream_t stream);
// FP8 weights: rows of h (BF16 [R, I]) to E4M3 codes hq [R_pad, I] and row
// scales hs [R_pad], the same rule.
cudaError_t launch_quantize_rows(const __nv_bfloat16* h, int R, int I, uint8_t* hq, float* hs, cudaStream_t stream);
// NVFP4 weights (FP16 tensor cores): token rows (x in BF16 or FP32, the
// latter rounded to BF16 first) to FP16 times a power of two per row, in
// route order (xh [R_pad, H]), the inverse power of two per row in xs
// [R_pad]; pos == NULL (dense MLP): row t to row t.  Exact (see quant.cu).
cudaError_t launch_gather_f16(const void* x, bool x_bf16, int H, const int32_t* pos, int T, __half* xh, float* xs,
                              uint32_t* status, cudaStream_t stream);
// NVFP4 weights: rows of h (BF16 [R, I]) to FP16 in place, the same rule,
// inverse scales in hs [R_pad].
cudaError_t launch_rows_to_f16(void* h, int R, int I, float* hs, cudaStream_t stream);
// NVFP4 activations (W4A4): token rows quantised per row to NVFP4 (x as
// given), each element written as the FP16 value e2m1 * e4m3 in route order
// (xh [R_pad, H]), the row's FP32 global scale in xs; pos == NULL: row t to
// row t (see quant.cu for the rule).
cudaError_t launch_gather_a4(const void* x, bool x_bf16, int H, const int32_t* pos, int T, __half* xh, float* xs,
                             uint32_t* status, cudaStream_t stream);
// W4A4: rows of h (BF16 [R, I]) quantised to NVFP4 in place (as FP16), global
// scales in hs.
cudaError_t launch_rows_to_a4(void* h, int R, int I, float* hs, cudaStream_t stream);
// The W4A4 quantiser on rows [rows, K] (FP32 or BF16): codes (one per byte),
// block scales, global scales and FP16 values (test hook).
cudaError_t launch_quantize_a4(const void* a, bool a_bf16, int rows, int K, uint8_t* codes, uint8_t* scales,
                               float* global, __half* values, cudaStream_t stream);
// wide: BF16 / FP8 down on one CTA per unit with 256-row units (two tiles per
// k-block); fp8: E4M3 weights and activations (kind::f8f6f4); dec: NVFP4 with
// chunks of at most 64 routes (4 epilogue warps, 12 converter warps)
cudaError_t launch_gemm(int mode, bool fp4, bool pair, bool wide, bool fp8, bool dec, const GemmMaps& maps,
                        const GemmParams& p, int grid, size_t smem_bytes, cudaStream_t stream);
constexpr int kDecChunkRows = 16;  // NVFP4 decode variant: routes per unit at most
size_t gemm_smem_bytes(int stages, int acc_stages, size_t stage_bytes);
// Clusters of two CTAs of the pair kernel that can be resident at once (0: none).
int gemm_pair_max_clusters(int mode, size_t smem_bytes);
cudaError_t launch_combine(const __nv_bfloat16* yr, const int32_t* pos, const float* w, int T, int H,
                           void* y, bool y_bf16, uint32_t* status, cudaStream_t stream);
// K split: add the k_splits FP32 partial planes in part order; mode 0: h =
// BF16(silu(sum gate) * sum up) [R, N]; mode 1: out = BF16(sum) [R, N].
cudaError_t launch_splitk_finish(int mode, const float* partial, int k_splits, int R, int N, __nv_bfloat16* out,
                                 cudaStream_t stream);
// Post-norm residual update fused into the combine (see combine.cu).
struct ResidualParams {
  const void* stream;   // [T, H] residual stream, the activations' dtype
  void* out;            // [T, H] new stream; may equal `stream`
  const float* norm_w;  // [H] RMSNorm scale
  float eps, keep, add;
};
cudaError_t launch_combine_residual(const __nv_bfloat16* yr, const int32_t* pos, const float* w, int T, int H,
                                    const ResidualParams& r, void* y_out, bool bf16, uint32_t* status,
                                    cudaStream_t stream);
// Row split (CTAs per token, one cluster) and dynamic shared memory of the
// fused kernel.
int residual_cluster_y(int T, int H);
size_t residual_smem_bytes(int T, int H);
cudaError_t launch_debug_timeout(uint32_t* status, uint64_t timeout_ns, cudaStream_t stream);
// Regroup `rows` x `row_bytes` (row-major) into contiguous tiles of 128 rows
// x `tile_row_bytes` (pack.cu); rows % 128 == 0, row_bytes % tile_row_bytes
// == 0, tile_row_bytes % 16 == 0.
cudaError_t launch_pack_tiles(const void* src, void* dst, size_t rows, size_t row_bytes, uint32_t tile_row_bytes,
                              int num_sms, cudaStream_t stream);

}  // namespace beam

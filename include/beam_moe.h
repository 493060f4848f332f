/*
 * beam_moe.h -- C ABI of a single-GPU (B300, sm_103a) implementation of the
 * group-limited Mixture-of-Experts block of the Beam model.
 *
 * Source of the operation (two translations of one launch post):
 *   "Willkommen Beam: ein offenes 501B-Modell, das Sie besitzen, anpassen und
 *   skalieren können" (spke.com), section "Mixture of Experts", and the
 *   Chinese "Reflection 发布 501B 开放模型 Beam，支持自托管定制与扩展"
 *   (sihot.dev), section 混合专家.  The post fixes: 256 experts, each a
 *   SwiGLU MLP (intermediate 2560, hidden 5120); sigmoid router scores;
 *   8 groups of 32 ranked by the sum of each group's two best scores; the
 *   best 4 groups kept; the top-8 experts inside them; no shared expert;
 *   expert outputs combined with the normalised router weights times 2.5.
 *   Section "Residual Stream" of the same post: the router and the SwiGLU
 *   product are computed in FP32.
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers, owned by the caller, row-major,
 *     16-byte aligned.  The library allocates no memory and keeps no state
 *     between calls other than a per-device cache of kernel attributes (and,
 *     for beam_moe_route_noalloc only, a 6 MiB static device buffer whose
 *     address is cached per CUDA context).
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls
 *     only enqueue work; none synchronises the host except
 *     beam_moe_read_device_status.
 *   - Argument, shape and alignment errors are detected on the host before
 *     anything is enqueued (BEAM_ERR_INVALID_ARG / BEAM_ERR_UNSUPPORTED /
 *     BEAM_ERR_WORKSPACE).  A failed launch returns BEAM_ERR_CUDA.  Errors the
 *     kernels detect (a bounded wait that ran out) are written to a status
 *     word inside the workspace; read it with beam_moe_read_device_status.
 *   - Two calls that run concurrently must use distinct workspaces.
 *
 * Supported shape: E = 256, n_group = 8, topk_group = 4, top_k = 8,
 * H % 128 == 0, I % 128 == 0, 1 <= T <= 1048576.  routed_scale is any finite
 * value (2.5 for Beam).
 */
#ifndef BEAM_MOE_H
#define BEAM_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  BEAM_OK = 0,
  BEAM_ERR_INVALID_ARG = 1,  /* null / misaligned pointer, negative size */
  BEAM_ERR_UNSUPPORTED = 2,  /* shape or dtype outside the supported set */
  BEAM_ERR_WORKSPACE = 3,    /* workspace null, misaligned or too small */
  BEAM_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed */
  BEAM_ERR_TIMEOUT = 5,      /* device: a bounded wait ran out (status word) */
  BEAM_ERR_DEVICE_CHECK = 6  /* device: a kernel's own consistency check failed */
} beam_status_t;

/* BEAM_NVFP4_A4 (expert weights only): the NVFP4 weights of BEAM_NVFP4 with
 * the GEMM inputs quantised to NVFP4 at run time (W4A4): each row of x (as
 * given) and of h (as stored in BF16) gets the weights' recipe per row:
 * global scale g = amax / (6 * 448) in FP32 (1 for a zero row), an E4M3 scale
 * s = E4M3((block max / 6) / g) per 16 consecutive elements and E2M1 codes of
 * a / (s * g) (FP32 divisions and product, nearest even, saturating; code 0
 * where s * g is 0), the element standing for e2m1 * s * g.  The launch post
 * (section "Mixture of Experts") names NVFP4 as a weight format; this
 * activation recipe is the library's reading.  The GEMMs multiply the
 * quantised operands exactly (FP16 tensor cores, FP32 accumulation; not the
 * block-scaled FP4 MMA).  Results move by tens of percent from W4A16's. */
typedef enum { BEAM_F32 = 0, BEAM_BF16 = 1, BEAM_NVFP4 = 2, BEAM_FP8 = 3, BEAM_NVFP4_A4 = 4 } beam_dtype_t;

/* Layer shape.  T tokens, hidden H, expert intermediate I, E experts in
 * n_group contiguous groups (group j = experts [j*E/n_group, (j+1)*E/n_group)),
 * topk_group groups kept, top_k experts per token, combine scale. */
typedef struct {
  int32_t T, H, I, E, n_group, topk_group, top_k;
  float routed_scale;
} beam_moe_shape_t;

/* Storage order of the expert weight arrays (codes and block scales for
 * NVFP4; the global scales are always [E]).
 *   BEAM_LAYOUT_ROWS : row-major as described at beam_expert_weights_t.
 *   BEAM_LAYOUT_TILED: the same bytes regrouped so that every tile the GEMMs
 *     load is contiguous: the matrix of R = E*N rows (N = I for gate / up, H
 *     for down) and B bytes per row is cut into tiles of 128 rows x b bytes,
 *     b = 128 for BF16 (64 elements) and FP8 (128 elements), 32 for E2M1
 *     codes (64 elements), 16 for E4M3 scales (256 elements); the FP8 row
 *     scales keep their order; tile (i, j) (rows 128i.., bytes bj..) is
 *     stored at byte (i * B/b + j) * 128 * b, its rows b bytes apart.  Made by
 *     beam_moe_pack_weights; streams ~3% faster from HBM (each tile is one
 *     contiguous block instead of 128 pieces). */
typedef enum { BEAM_LAYOUT_ROWS = 0, BEAM_LAYOUT_TILED = 1 } beam_weight_layout_t;

/* Expert weights, all experts stacked, linear-layer orientation [out, in]:
 *   BF16 : gate [E, I, H], up [E, I, H], down [E, H, I]  (bf16 elements)
 *   NVFP4: gate/up [E, I, H/2], down [E, H, I/2] bytes, two E2M1 codes per
 *          byte, the even K index in the low nibble; *_sf = E4M3 block scales
 *          [E, I, H/16] / [E, H, I/16], one per 16 consecutive K elements;
 *          *_gs = FP32 global scale per expert and matrix [E].
 *          Element value = e2m1 * e4m3 * global.
 *   FP8  : gate/up [E, I, H], down [E, H, I] E4M3 bytes (OCP FP8 E4M3: bias 7,
 *          no infinities, largest finite 448); *_rs = FP32 scale per output
 *          row [E, I] / [E, H].  Element value = e4m3 * row scale.  The
 *          launch post (section "Mixture of Experts") lists an FP8 checkpoint
 *          without its layout; this per-row layout is the library's reading.
 *          The GEMM inputs are quantised per row to E4M3 at run time (x
 *          rows before gate/up, h rows before down): scale = row amax / 448
 *          (1 for a zero row), code = E4M3(a / scale), round to nearest even,
 *          saturating, both divisions in FP32; the MMAs run E4M3 x E4M3 with
 *          FP32 accumulation and both scales are applied in FP32 after the
 *          sum.  Supported when I <= H (h's codes share the x-code buffer).
 * (in `layout` order; BEAM_LAYOUT_ROWS when the field is zero-initialised).
 * Pointers the dtype does not use must be NULL. */
typedef struct {
  beam_dtype_t dtype; /* BEAM_BF16, BEAM_NVFP4, BEAM_NVFP4_A4 (NVFP4 arrays) or BEAM_FP8 */
  const void* gate;
  const void* up;
  const void* down;
  const uint8_t* gate_sf;
  const uint8_t* up_sf;
  const uint8_t* down_sf;
  const float* gate_gs;
  const float* up_gs;
  const float* down_gs;
  beam_weight_layout_t layout;
  const float* gate_rs; /* FP8 only */
  const float* up_rs;
  const float* down_rs;
} beam_expert_weights_t;

/* Where the intermediates of the last call live inside the workspace (byte
 * offsets from its start); for inspection by tests and tools.
 *   counts int32[E]        routes per expert
 *   offsets int32[E+1]     exclusive prefix sum of counts
 *   perm int32[T*top_k]    route ids r = t*top_k + k grouped by expert,
 *                          ascending r inside an expert
 *   pos int32[T*top_k]     inverse of perm: perm[pos[r]] == r
 *   xp bf16[T*top_k, H]    token rows in perm order
 *   h bf16[T*top_k, I]     SwiGLU activations in perm order
 *   yr bf16[T*top_k, H]    expert outputs in perm order (before weighting)
 *   status uint32[4]       device status word (code, where, 0, 0)
 * FP8 weights only (the GEMM inputs quantised per row):
 *   xq u8[T*top_k, H]      E4M3 codes of the token rows, perm order (inside xp)
 *   hq u8[T*top_k, I]      E4M3 codes of h, perm order (inside xp, after xq)
 *   xs, hs f32[T*top_k]    their row scales */
typedef struct {
  size_t status, counts, offsets, perm, pos, xp, h, yr, total;
  size_t xq, hq, xs, hs;
} beam_ws_layout_t;

/* Bytes of workspace beam_moe_forward / beam_moe_experts need for `shape`
 * with expert weights of type `wdtype` (0 on an unsupported shape).  The
 * same workspace serves beam_moe_route and beam_moe_dispatch. */
size_t beam_moe_workspace_size(const beam_moe_shape_t* shape, beam_dtype_t wdtype);

/* Fill `layout` for `shape`; returns BEAM_OK or BEAM_ERR_UNSUPPORTED. */
beam_status_t beam_moe_workspace_layout(const beam_moe_shape_t* shape, beam_dtype_t wdtype,
                                        beam_ws_layout_t* layout);

/* Routing only (Beam post, "Mixture of Experts"): for every token t
 *   s[e]   = sigmoid(sum_h x[t,h] * router_w[e,h])        (FP32)
 *   sel[e] = s[e] + router_bias[e]   (bias 0 when router_bias == NULL; it
 *            steers the selection only, as in DeepSeek-V3's scheme)
 *   group score = sum of the two largest sel in the group; keep the
 *   topk_group best groups (ties: lower group index); take the top_k largest
 *   sel among their experts (ties: lower expert index), best first.
 *   topk_ids[t,k] = chosen expert; topk_w[t,k] = s[id] / sum_k s * scale.
 * x: [T, H] FP32 or BF16 (xdtype); router_w: FP32 [E, H]; router_bias:
 * FP32 [E] or NULL; topk_ids: int32 [T, top_k]; topk_w: FP32 [T, top_k].
 * Also leaves per-tile expert histograms in the workspace for dispatch. */
beam_status_t beam_moe_route(const beam_moe_shape_t* shape, const void* x, beam_dtype_t xdtype,
                             const float* router_w, const float* router_bias, int32_t* topk_ids,
                             float* topk_w, void* workspace, size_t workspace_bytes, void* stream);

/* Dispatch only: from topk_ids [T, top_k] build counts, offsets, perm and
 * pos in the workspace (see beam_ws_layout_t), deterministic order. */
beam_status_t beam_moe_dispatch(const beam_moe_shape_t* shape, const int32_t* topk_ids,
                                void* workspace, size_t workspace_bytes, void* stream);

/* Experts and combine for a given routing:
 *   y[t,:] = sum_k topk_w[t,k] * FFN_{topk_ids[t,k]}(x[t,:]),  k = 0..top_k-1
 *   FFN_e(v) = Wd[e] (silu(Wg[e] v) * (Wu[e] v)),  SwiGLU product in FP32,
 *   FP32 accumulation, activations rounded to BF16 between the matmuls.
 * No shared-expert term.  y has x's dtype ([T, H]). */
beam_status_t beam_moe_experts(const beam_moe_shape_t* shape, const void* x, beam_dtype_t xdtype,
                               const beam_expert_weights_t* weights, const int32_t* topk_ids,
                               const float* topk_w, void* y, void* workspace,
                               size_t workspace_bytes, void* stream);

/* The whole block: beam_moe_route followed by beam_moe_experts. */
beam_status_t beam_moe_forward(const beam_moe_shape_t* shape, const void* x, beam_dtype_t xdtype,
                               const float* router_w, const float* router_bias,
                               const beam_expert_weights_t* weights, void* y, int32_t* topk_ids,
                               float* topk_w, void* workspace, size_t workspace_bytes,
                               void* stream);

/* The steps of beam_moe_forward, in order.  beam_moe_forward enqueues all of
 * them; beam_moe_forward_stage enqueues one, so that a caller can put events
 * between them (per-step timing) or run the steps on its own schedule. */
typedef enum {
  BEAM_STAGE_ROUTE = 0,    /* router GEMV + selection (+ per-tile histogram) */
  BEAM_STAGE_DISPATCH = 1, /* counts, offsets, perm, pos from the histograms */
  BEAM_STAGE_GATHER = 2,   /* token rows into route order (BF16; FP8 weights:
                              E4M3 codes and row scales) */
  BEAM_STAGE_GATE_UP = 3,  /* grouped gate/up GEMM with the SwiGLU epilogue */
  BEAM_STAGE_DOWN = 4,     /* grouped down GEMM (FP8 weights: after h is
                              quantised per row) */
  BEAM_STAGE_COMBINE = 5,  /* weighted sum of each token's expert outputs
                              (+ the residual update when args->residual) */
  BEAM_STAGE_COUNT = 6
} beam_stage_t;

/* Post-norm residual update after the block, fused into its combine step.
 * Source: the Beam post, section "Residual Stream": the stream starts from the
 * embedding (step 1); at step k >= 2 the stream is kept with weight
 * sqrt((k-1)/k) and the sublayer's output, normalised after the sublayer,
 * added with weight 1/sqrt(k) (the two weights' squares sum to one, so the
 * embedding and every sublayer output end with equal weight); norms in FP32.
 * The post does not say which norm follows a sublayer; it is read as RMSNorm
 * (the norm the post names, in section "Attention", for queries and keys)
 * with a learned scale g and an eps inside the root:
 *   out[t,:] = sqrt((k-1)/k) * stream[t,:]
 *            + (1/sqrt(k)) * g * y[t,:] / sqrt(mean_j y[t,j]^2 + eps)
 * where y is the block's output (kept in FP32 inside the kernel, not rounded
 * to the activations' dtype first).  All arithmetic FP32; out rounded to the
 * stream's dtype (round to nearest even).  A row with y = 0 and eps = 0
 * gives NaN, as the formula does. */
typedef struct {
  const void* stream;       /* [T, H] stream before the update, x's dtype */
  void* out;                /* [T, H] stream after it, x's dtype; may be `stream`
                               itself (in place), else must not overlap it */
  const float* norm_weight; /* [H] the post-norm's scale g, FP32 */
  float eps;                /* finite, >= 0 */
  int32_t step;             /* k >= 2 (the embedding is step 1) */
} beam_residual_t;

/* All tensors of one forward call (the arguments of beam_moe_forward).
 * `residual` (nullable, last so that older initialisers stay valid): when set,
 * the combine step applies the residual update above and `y` becomes
 * optional (NULL: the block's output is not written; else it is written too,
 * in x's dtype, and must not overlap the stream or out). */
typedef struct {
  const void* x;
  beam_dtype_t xdtype;
  const float* router_w;
  const float* router_bias;
  const beam_expert_weights_t* weights;
  void* y;
  int32_t* topk_ids;
  float* topk_w;
  const beam_residual_t* residual;
} beam_moe_args_t;

/* The whole block followed by the residual update: beam_moe_forward with
 * args->residual (required) applied in the combine kernel.  The routing
 * outputs are written as by beam_moe_forward.  BEAM_ERR_INVALID_ARG for a
 * null or misaligned residual pointer, step < 2, eps negative or not finite,
 * or overlapping stream / out / y. */
beam_status_t beam_moe_forward_residual(const beam_moe_shape_t* shape, const beam_moe_args_t* args,
                                        void* workspace, size_t workspace_bytes, void* stream);

/* Enqueue stage `stage` of the forward pass.  Each stage reads what the
 * previous stages left in `workspace` (and in topk_ids / topk_w), so the
 * stages of one forward must be issued in order, on one stream (or with the
 * caller's own ordering).  Arguments are validated as beam_moe_forward does. */
beam_status_t beam_moe_forward_stage(const beam_moe_shape_t* shape, const beam_moe_args_t* args,
                                     beam_stage_t stage, void* workspace, size_t workspace_bytes,
                                     void* stream);

/* Number of kernels stage `stage` launches for `shape`, activations of type
 * `xdtype` and expert weights of type `wdtype` on the current device: the
 * router adds a selection kernel when it splits its reduction across CTAs,
 * and its tensor-core path (BF16 x, T >= 512) a kernel that splits the
 * router weight into BF16 terms; the dispatch is two kernels; with FP8
 * weights the down stage first quantises h (two kernels); -1 on an
 * unsupported shape, dtype or stage. */
int32_t beam_moe_stage_kernel_count(const beam_moe_shape_t* shape, beam_dtype_t xdtype, beam_dtype_t wdtype,
                                    beam_stage_t stage);

/* Regroup row-major expert weights into BEAM_LAYOUT_TILED (a one-time step
 * when loading a model; not part of the Beam post's method, which fixes the
 * arithmetic, not the storage).  `src`: layout BEAM_LAYOUT_ROWS; `dst`: the
 * same dtype, caller-allocated arrays of the same sizes (gate, up, down and,
 * for NVFP4, the three scale arrays; dst's global-scale pointers are used as
 * given and may alias src's; for FP8, dst's row-scale pointers must be src's,
 * as the row scales keep their order); dst->layout is set to
 * BEAM_LAYOUT_TILED.  The arrays must not overlap.  Async on `stream`.
 * Errors as for the forward call's weights; BEAM_ERR_UNSUPPORTED unless N and
 * K are multiples of 128 / 64 elements (BF16), 128 / 256 (NVFP4) or
 * 128 / 128 (FP8). */
beam_status_t beam_moe_pack_weights(const beam_moe_shape_t* shape, const beam_expert_weights_t* src,
                                    beam_expert_weights_t* dst, void* stream);

/* Synchronises `stream`, returns the device status word of `workspace`
 * (BEAM_OK when no kernel reported a problem) and clears it.  `where`
 * (nullable) receives the code of the wait that gave up. */
beam_status_t beam_moe_read_device_status(void* workspace, uint32_t* where, void* stream);

/* Test hook for the bounded-wait machinery: launches one CTA that waits on
 * an mbarrier nothing ever arrives on, with a limit of `timeout_us`
 * microseconds; the kernel then records BEAM_ERR_TIMEOUT in the workspace
 * status word and returns normally. */
beam_status_t beam_moe_debug_timeout(void* workspace, size_t workspace_bytes, uint32_t timeout_us,
                                     void* stream);

/* Test hook for the NVFP4 weight expansion (not part of the Beam post's
 * method): expands n_blocks blocks of 16 E2M1 elements with the same device
 * code the grouped GEMMs' converter warps run.  codes: device, n_blocks * 8
 * bytes (block b in bytes 8b..8b+7, element 2j in the low nibble of byte j);
 * scales: device, n_blocks E4M3 codes (block b's at byte b); out: device,
 * n_blocks * 16 FP16 values (bit patterns), element i of block b at 16b + i,
 * = e2m1 * e4m3 exactly (NaN for the E4M3 NaN codes).  n_blocks a positive
 * multiple of 4, all pointers 16-byte aligned, else BEAM_ERR_INVALID_ARG.
 * Async on `stream`. */
beam_status_t beam_debug_nvfp4_expand(const uint8_t* codes, const uint8_t* scales, int32_t n_blocks, uint16_t* out,
                                      void* stream);

/* Test hook for the W4A4 activation quantiser (see BEAM_NVFP4_A4): quantises
 * `rows` rows of K elements (a: device, FP32 or BF16 by a_dtype, row-major)
 * with the device code the W4A4 forward runs on x and h.  codes: device,
 * [rows, K] bytes, one E2M1 code per byte (bit 3 the sign); scales: device,
 * [rows, K/16] E4M3 codes; global: device, [rows] FP32; values: device,
 * [rows, K] FP16 bit patterns of e2m1 * e4m3 (what the GEMMs multiply; the
 * global scale is applied after the sums).  K a positive multiple of 16; a and
 * values 16-byte aligned, else BEAM_ERR_INVALID_ARG; a_dtype other than
 * BEAM_F32 / BEAM_BF16: BEAM_ERR_UNSUPPORTED.  Async on `stream`. */
beam_status_t beam_debug_quantize_nvfp4(const void* a, beam_dtype_t a_dtype, int32_t rows, int32_t K, uint8_t* codes,
                                        uint8_t* scales, float* global, uint16_t* values, void* stream);

/* Routing without a workspace, for callers that cannot allocate device memory
 * (a host framework that owns all device memory and hands a plugin only its
 * inputs and outputs, or a serving loop that must never allocate, since an
 * allocation can stall the device).  The Beam post has no counterpart: this
 * is an integration convenience.  Same result as beam_moe_route (the hidden
 * dimension may be split across fewer CTAs, so FP32 logits can differ in the
 * last bits).  Arguments and shape rules as beam_moe_route, without the
 * workspace.
 *   - Scratch: a library-owned static device buffer of 6 MiB (2 MiB of tile
 *     histograms + 4 MiB of partial logits) on every GPU that loads the
 *     library, held until the process exits.  No allocation in any call.
 *   - Limit: T <= 65536, else BEAM_ERR_UNSUPPORTED.  The hidden dimension is
 *     split across at most 4096 / T CTAs per 32-token tile, so every T > 2048
 *     runs one split per tile (beam_moe_route splits it up to T = 4704 on a
 *     148-SM B300, and runs BF16 x with T >= 512 on the tensor cores).
 *   - The first call in each CUDA context (per device, or per driver context
 *     a caller makes current) looks up the buffer's device address in that
 *     context; make that first call before any stream capture.
 *   - All calls share the buffer and it keeps the last call's contents
 *     (nothing in it needs to start at zero); calls that overlap on the GPU,
 *     on any stream or thread, race and must be serialised by the caller. */
beam_status_t beam_moe_route_noalloc(const beam_moe_shape_t* shape, const void* x, beam_dtype_t xdtype,
                                     const float* router_w, const float* router_bias, int32_t* topk_ids,
                                     float* topk_w, void* stream);

/* Dense SwiGLU MLP.  Source: the Beam post, section "Mixture of Experts":
 * the first 3 of the 52 layers use a dense SwiGLU MLP in place of the MoE
 * block (its width is not given; I is the caller's).  Same arithmetic as one
 * expert of the block:
 *   y[t,:] = Wd (silu(Wg x[t,:]) * (Wu x[t,:])),  SwiGLU product in FP32,
 *   FP32 accumulation, h rounded to BF16 between the matmuls,
 * run by the block's grouped GEMMs as a single expert that takes every row.
 * x and y: BF16 [T, H] (FP32 x only with FP8 weights, whose first step
 * re-encodes x).  Weights: a beam_expert_weights_t of one expert (gate/up
 * [1, I, H], down [1, H, I], the per-expert arrays of NVFP4 / FP8 with one
 * entry), any dtype and layout the block takes.  Shape limits as for the
 * block (H % 128, I % 128, 1 <= T <= 1048576; NVFP4 H, I % 256). */
typedef struct {
  int32_t T, H, I;
} beam_dense_shape_t;

/* Workspace bytes of beam_dense_mlp_forward (0 on an unsupported shape). */
size_t beam_dense_workspace_size(const beam_dense_shape_t* shape, beam_dtype_t wdtype);

beam_status_t beam_dense_mlp_forward(const beam_dense_shape_t* shape, const void* x, beam_dtype_t xdtype,
                                     const beam_expert_weights_t* weights, void* y, void* workspace,
                                     size_t workspace_bytes, void* stream);

/* Kernels one beam_dense_mlp_forward launches on the current device: the
 * one-expert schedule, the gate/up and down GEMMs, with FP8 weights the two
 * row quantisations, and a finishing kernel after each GEMM whose K range is
 * split across CTAs (few rows: the partial sums are added in part order);
 * -1 on an unsupported shape or dtype. */
int32_t beam_dense_kernel_count(const beam_dense_shape_t* shape, beam_dtype_t wdtype);

/* beam_moe_pack_weights for the dense MLP's one-expert weight arrays. */
beam_status_t beam_dense_pack_weights(const beam_dense_shape_t* shape, const beam_expert_weights_t* src,
                                      beam_expert_weights_t* dst, void* stream);

/* 1 when this library is the debug build (libbeam_moe_debug.so, compiled
 * with BEAM_DEBUG=1), else 0.  The debug build checks on the device every
 * index a kernel takes from the workspace before using it as an address --
 * route positions in the gathers and combines, and, before each grouped GEMM
 * (one more kernel per GEMM), that counts / offsets / chunk prefixes describe
 * the routes -- and on a failed check records BEAM_ERR_DEVICE_CHECK in the
 * status word (second word: where: 21 expert id met by the dispatch, 22 / 26
 * / 27 route position met by the gather of BF16 rows / E4M3 codes / FP16
 * rows, 23 / 28 by the combine / the combine with the residual update, 24 the
 * GEMM schedule), skips the access (a GEMM with a bad schedule runs no work)
 * and returns normally.  Both builds check expert ids given to the dispatch
 * (where 20).  Otherwise the two builds compute the same results. */
int32_t beam_moe_debug_build(void);

/* Static description of a status code. */
const char* beam_status_string(beam_status_t status);

#ifdef __cplusplus
}
#endif
#endif /* BEAM_MOE_H */

// gemm.cu -- grouped expert GEMMs on the Blackwell tensor cores (tcgen05,
// accumulators in TMEM, operands staged by TMA).
//
// Beam launch post, section "Mixture of Experts": every expert is a SwiGLU MLP
// (hidden 5120, intermediate 2560); section "Residual Stream": the SwiGLU
// product is computed in FP32.  The same post names three checkpoint formats:
// BF16; NVFP4 for Blackwell (4-bit weights), here expanded exactly to FP16
// in TMEM and multiplied with the BF16 activations carried exactly in FP16
// (each row times a power of two, undone in the epilogue; W4A16); and FP8,
// here E4M3 weights
// with per-row scales multiplied with per-row-quantised E4M3 activations on
// kind::f8f6f4 MMAs.
//
//   mode 0 (gate/up):  h[r, i]  = silu(x_r . Wg[e,i,:]) * (x_r . Wu[e,i,:])
//   mode 1 (down):     yr[r, j] = h_r . Wd[e,j,:]
//
// for every route r of expert e (routes in the dispatch order).  The weight
// rows are the MMA's M side (128 rows per tile = the 128 TMEM lanes) and the
// routed tokens are its N side ("swap AB"): an expert sees 1..3 tokens at
// decode and ~256 at prefill, and N can be any multiple of 16 up to 256,
// while M is 128 per CTA.  A work unit is (expert, token chunk of <= nmax
// routes, weight row tile[, part of the K range]): 128 rows, or on CTA pairs
// 256 (gate/up) / 512 (down) rows, and 256 rows for two-tile down units; each
// k-block issues its MMAs into two accumulators (gate and up, or two row
// halves) where the unit has two tiles.  Units are numbered in the order
// (expert, row tile, chunk, K part) -- (expert, chunk, row tile, K part) for
// experts with many chunks (see unit_at) -- and taken from a global counter in
// that order by a persistent grid (one CTA, or CTA pair, per SM), so CTAs
// running side by side share weight tiles and token chunks through L2.  A K
// range split into parts (few units for many SMs) leaves FP32 partial sums
// that splitk.cu adds up.
//
// Warp roles (BF16 / FP8: 10 warps; NVFP4: 19 warps, 21 in the decode variant):
//   warp 0       TMA producer: weight tile(s) of 128 rows x 128 bytes and the
//                chunk's token rows x 128 bytes (one box of the tile's
//                height, or 32-row boxes for a small chunk) per stage,
//                128-byte swizzle (NVFP4: the packed 128x32-byte tiles and
//                their E4M3 scales);
//   warp 1       TMEM allocator and MMA issuer (one thread): tcgen05.mma
//                kind::f16 (BF16, K=16 steps) or kind::f8f6f4 (E4M3, K=32
//                steps), M=128 (256 on pairs), N=round_up(n,16);
//   warps 2..    epilogue (8 warps; 4 in the NVFP4 decode variant):
//                tcgen05.ld of the accumulators (warp w reads TMEM lanes
//                32*(w%4)..+31 and every (warps/4)-th 16-column chunk),
//                NVFP4 global scale or FP8 row x token-row scales, SwiGLU in
//                FP32 (mode 0), BF16 stores (K parts: FP32 partial stores);
//   then         (NVFP4 only) converters, 8 warps in two groups (12 in three
//                groups in the decode variant) taking alternate k-blocks:
//                packed E2M1 x E4M3 -> FP16 weight tile (hardware cvt of
//                code pairs and scale pairs, one exact FP16 multiply),
//                written straight into TMEM (tcgen05.st; the thread of TMEM
//                lane m expands weight row m), where the MMA (kind::f16, FP16
//                A and B) reads its A operand.  Shared
//                memory then carries only the packed bytes and the
//                activations, and its bandwidth stays with the MMA's B operand;
//   last         (NVFP4 only) a second MMA issuer for the second tile (decode
//                variant: three more, so that two threads share each tile).
// Shared-memory stages are recycled through full/empty mbarriers, TMEM
// accumulator buffers through acc_full/acc_empty.  NVFP4: the converters wait
// for the TMA bytes of a stage before expanding its weights, and the MMA
// threads wait only for the converters (afull), whose arrival follows their
// observation of the TMA completion; a TMEM weight tile is reused once the
// empty barrier of the k-block that last read it has completed, so each
// MMA-issuing thread waits once and commits once per k-block.  Every wait is
// bounded; waits after the first poll let the thread sleep (see mbar_wait).
#include <cuda.h>
#include <cuda_bf16.h>

#include "moe_internal.cuh"
#include "nvfp4.cuh"
#include "tc.cuh"

namespace beam {
namespace {

constexpr int kEpilogueWarps = 8;
constexpr int kConvertWarps = 8;
constexpr int kThreadsBf16 = 32 * (2 + kEpilogueWarps);
// NVFP4: a second MMA-issuing warp (after the converters): one thread issues
// the first tile's MMAs (gate, or the first row half), the other the
// second's, each its own accumulator chain, so MMA issue is not bound by one
// thread's instruction rate at N ~ 144.
constexpr int kMma2Warp = 2 + kEpilogueWarps + kConvertWarps;
constexpr int kThreadsFp4 = 32 * (kMma2Warp + 1);
// NVFP4 decode variant: four MMA-issuing threads (warps 1 and kMma2Warp..+2),
// two per weight matrix, one per accumulator of that matrix.  With chunks of
// at most 16 routes a tcgen05.mma keeps its issuing thread ~80 cycles while
// the tensor pipe needs ~33, so one thread per matrix left the pipe idle.
constexpr int kThreadsFp4Dec = 32 * (kMma2Warp + 3);
constexpr uint32_t kATileBytes = kBlockM * kBlockK * 2;     // 16 KiB of BF16
constexpr uint32_t kBoxBytes = kBoxRows * kBlockK * 2;      // 4 KiB
constexpr int kSchedRing = 8;                               // scheduled unit indices in flight
constexpr int kSlotInts = 8;                                // ints per unit ring slot: index + Unit
constexpr int kSiblingChunks = 2;                           // experts with more chunks run chunk by chunk

struct Unit {
  int e, m, start, n;
  int ks, kb0, kb1;  // K split: part ks covers k-blocks [kb0, kb1)
};

__device__ __forceinline__ Unit unit_at(const GemmParams& p, int u) {
  Unit U;
  // K split (p.k_splits > 1: few units for many SMs): the parts of one tile
  // are adjacent unit indices
  U.ks = u % p.k_splits;
  u /= p.k_splits;
  U.kb0 = U.ks * p.k_blocks / p.k_splits;
  U.kb1 = (U.ks + 1) * p.k_blocks / p.k_splits;
  // Expert e owns units [chunk_prefix[e], chunk_prefix[e+1]) * m_tiles.  With
  // at most kSiblingChunks chunks they are numbered (row tile, chunk): the
  // chunks of one weight tile are adjacent units, which the schedule starts
  // side by side, so they read the tile's k-blocks from DRAM once and share
  // them through L2 (prefill-sized layers, ~2 chunks per expert: 2.5% faster).
  // Experts with more chunks (the hot experts of skewed routing) keep the
  // order (chunk, row tile), in which the row tiles of one chunk share its
  // token rows instead (numbered the other way, the skewed layer ran 2% slower).
  const int q = u / p.m_tiles;
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
  // The expert's routes are cut into nch = ceil(count / nmax) chunks of
  // near-equal size (sizes differ by at most one), so the CTAs that run the
  // chunks of one weight tile side by side progress in step.
  const int cp0 = __ldg(&p.chunk_prefix[lo]);
  const int nch = __ldg(&p.chunk_prefix[lo + 1]) - cp0;
  const int local = u - cp0 * p.m_tiles;
  int c;
  if (nch <= kSiblingChunks) {
    U.m = local / nch;
    c = local - U.m * nch;
  } else {
    c = local / p.m_tiles;
    U.m = local - c * p.m_tiles;
  }
  const int count = __ldg(&p.counts[lo]);
  const int base = count / nch, rem = count - base * nch;
  U.start = __ldg(&p.offsets[lo]) + c * base + (c < rem ? c : rem);
  U.n = base + (c < rem ? 1 : 0);
  return U;
}

// kPair: a cluster of two CTAs runs each unit as one M=256 pair MMA
// (tcgen05 cta_group::2): CTA r holds weight rows 128r..128r+127 of the
// 256-row tile and half of the token chunk (N/2 rows); each CTA's TMEM gets
// its 128 rows x N accumulator.  The even CTA issues the MMAs; both CTAs'
// TMA loads signal the even CTA's full barrier; commits are multicast to
// both CTAs; both epilogues release the even CTA's acc_empty barrier.
// kWide (down, one CTA per unit, BF16): 256-row units of two 128-row tiles,
// two accumulators, so each k-block carries eight MMAs in two chains.
// kFp8: E4M3 weights and E4M3 activations (kind::f8f6f4): the same tiles of
// 128-byte rows, now 128 K elements per k-block; the epilogue multiplies each
// accumulator element by its weight row's scale and its token row's scale.
// kDec (NVFP4 at decode sizes, chunks of at most 16 routes): the MMAs are
// tiny and the conversion of the weights sets the pace, so the same 19 warps
// are split 4 epilogue warps (enough for 64 columns) and 12 converter warps in
// three groups that take every third k-block.
template <int kMode, bool kFp4, bool kPair, bool kWide = false, bool kFp8 = false, bool kDec = false>
__global__ void __launch_bounds__(kFp4 ? (kDec ? kThreadsFp4Dec : kThreadsFp4) : kThreadsBf16, 1)
    moe_gemm_kernel(const __grid_constant__ GemmMaps maps, const GemmParams p) {
  static_assert(!kDec || kFp4, "the decode split of warps is for NVFP4");
  constexpr int kEpi = kDec ? 4 : kEpilogueWarps;            // epilogue warps
  constexpr int kConv = kDec ? 12 : kConvertWarps;           // converter warps (NVFP4)
  constexpr int kGroups = kConv / 4;                         // converter groups, one k-block each
  constexpr int kEpiHalves = kEpi / 4;                       // epilogue warps per TMEM lane quarter
  static_assert(2 + kEpi + kConv == kMma2Warp, "NVFP4 warp layout");
  // Weight tiles per stage: gate/up always two (gate, up); down two on CTA
  // pairs (two 256-row halves of a 512-row unit sharing the token tile) and
  // for NVFP4 (two 128-row halves of a 256-row unit), so that every k-block
  // carries two accumulators' worth of MMAs.
  constexpr int kNumA = (kMode == 0 || kPair || kFp4 || kWide) ? 2 : 1;
  constexpr int kRowsPerUnit = kPair ? (kMode == 0 ? 2 * kBlockM : 4 * kBlockM) : (kNumA == 2 && kMode == 1 ? 2 * kBlockM : kBlockM);
  // down with two tiles: feature offset of the second tile's rows
  constexpr int kHalfRows = kPair ? 2 * kBlockM : kBlockM;
  static_assert(!(kPair && kFp4), "pair MMA path is BF16 / FP8 only");
  static_assert(!(kFp4 && kFp8), "one weight format");
  constexpr int kKElems = kFp8 ? 2 * kBlockK : kBlockK;  // K elements per k-block (128-byte rows)
  // MMA-issuing threads: commits per k-block / unit
  constexpr uint32_t kIssuers = kFp4 ? (kDec ? 4 : 2) : 1;
  // Roles that read every scheduled unit index (they release ring slots).
  constexpr uint32_t kRingConsumers =
      kPair ? (1 + kEpilogueWarps) + (1 + kEpilogueWarps)  // even CTA: MMA + epilogue; odd: producer + epilogue
            : kIssuers + kEpi + (kFp4 ? kConv : 0);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t b_tile_bytes = static_cast<uint32_t>(kPair ? p.nmax / 2 : p.nmax) * kBlockK * 2;
  // NVFP4: k-blocks per pipeline stage (1, 2 or 4; K loaded as a whole
  // number of stages per unit)
  const int S = kFp4 ? p.sub_blocks : 1;
  const uint32_t stage_bytes = static_cast<uint32_t>(gemm_stage_bytes(kNumA, kFp4, kPair ? p.nmax / 2 : p.nmax, S));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(p.stages) * stage_bytes);
  uint64_t* full = bars;
  uint64_t* empty = full + p.stages;
  uint64_t* afull = empty + p.stages;        // NVFP4: FP16 weight tile written to TMEM
  uint64_t* aempty = afull + kMaxAStages;    // NVFP4: the MMAs reading that tile have completed
  uint64_t* acc_full = aempty + kMaxAStages;
  uint64_t* acc_empty = acc_full + p.acc_stages;
  uint64_t* drain = acc_empty + p.acc_stages;
  uint64_t* ufull = drain + 1;        // unit ring: unit published
  uint64_t* uempty = ufull + kSchedRing;  // unit ring: unit read by every consumer
  // slot r: kSlotInts ints, the unit index and its decoded Unit
  volatile int* ring = reinterpret_cast<volatile int*>(uempty + kSchedRing);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(const_cast<int*>(ring) + kSchedRing * kSlotInts);
  volatile uint32_t* abort_flag = tmem_slot + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = kPair ? cluster_ctarank() : 0u;  // 0: the CTA that issues the MMAs
  // Stage layout: BF16 weights [A x kNumA][B]; NVFP4 [B x S][packed x kNumA x S][scales x kNumA]
  // (k-block `sub` of the stage: B at b_tile + sub * b_tile_bytes, packed
  // codes of matrix `which` at p_tile(s, which, sub); one scale tile per
  // matrix covers four k-blocks)
  auto a_tile = [&](int s, int which) { return smem + static_cast<size_t>(s) * stage_bytes + which * kATileBytes; };
  auto b_tile = [&](int s) {
    return smem + static_cast<size_t>(s) * stage_bytes + (kFp4 ? 0u : kNumA * kATileBytes);
  };
  auto p_tile = [&](int s, int which, int sub) {
    return b_tile(s) + S * b_tile_bytes + (which * S + sub) * kPackedTileBytes;
  };
  auto s_tile = [&](int s, int which) {
    return b_tile(s) + S * b_tile_bytes + kNumA * S * kPackedTileBytes + which * kScaleTileBytes;
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kIssuers);
    }
    for (int a = 0; a < kMaxAStages; ++a) {
      mbar_init(&afull[a], kConv / kGroups);  // one converter group per k-block
      mbar_init(&aempty[a], kIssuers);
    }
    for (int a = 0; a < p.acc_stages; ++a) {
      mbar_init(&acc_full[a], kIssuers);
      mbar_init(&acc_empty[a], kPair ? 2 * kEpilogueWarps : kEpi);
    }
    mbar_init(drain, kIssuers);
    for (int r = 0; r < kSchedRing; ++r) {
      mbar_init(&ufull[r], 1);
      mbar_init(&uempty[r], kRingConsumers);
    }
    *abort_flag = 0u;
    fence_mbar_init();
    tma_prefetch_desc(&maps.a0);
    if (kMode == 0) tma_prefetch_desc(&maps.a1);
    tma_prefetch_desc(&maps.b);
    tma_prefetch_desc(&maps.bb);
    if (kFp4) {
      tma_prefetch_desc(&maps.s0);
      if (kMode == 0) tma_prefetch_desc(&maps.s1);
    }
  }
  if (warp == 1) {
    if (kPair)
      tmem_alloc_pair(tmem_slot, p.tmem_cols);
    else
      tmem_alloc(tmem_slot, p.tmem_cols);
  }
  tc_fence_before();
  if (kPair)
    cluster_sync();  // both CTAs' barriers initialised before any cross-CTA arrive
  else
    __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  // --- dynamic unit schedule ------------------------------------------------
  // The fetching thread (producer of the even CTA) takes unit indices from a
  // global counter in order and publishes each one, or -1 at the end, into a
  // ring read by every role of both CTAs, so units (and the sibling chunks of
  // one expert, which share weight tiles through L2) start in index order.
  // NVFP4 decode variant: the unit is decoded (unit_at: a binary search over
  // the chunk prefix in global memory, ~10 dependent loads) once, by the
  // fetching thread, ahead of its consumers, and every role reads it from the
  // ring instead of decoding it again at its unit boundary (on the MMA
  // threads that search cost ~2 us per unit, ~6% of a decode-size launch of
  // short units).  The other kernels (measured no faster, or slower through
  // register spills) decode the index in each role.
  constexpr bool kRingUnits = kDec;
  constexpr int kStride = kRingUnits ? kSlotInts : 1;  // ints per ring slot in use
  int ring_slot = 0;
  uint32_t ring_phase = 0;
  auto ring_advance = [&]() {
    if (++ring_slot == kSchedRing) {
      ring_slot = 0;
      ring_phase ^= 1u;
    }
  };
  // One thread: the next unit index (-1: no more) and its Unit; false when a
  // wait gave up.
  auto ring_take_raw = [&](int& u, Unit& U) -> bool {
    if (!mbar_wait_cluster(&ufull[ring_slot], ring_phase, p.timeout_ns, abort_flag, p.status, kWhereSchedule))
      return false;
    const volatile int* r = ring + ring_slot * kStride;
    u = r[0];
    if (kRingUnits) {
      U.e = r[1];
      U.m = r[2];
      U.start = r[3];
      U.n = r[4];
      U.ks = r[5];
      U.kb0 = r[6];
      U.kb1 = r[7];
    }
    if (kPair)
      mbar_arrive_cluster(mapa_shared(&uempty[ring_slot], 0));
    else
      mbar_arrive(&uempty[ring_slot]);
    ring_advance();
    return true;
  };
  auto ring_take = [&](int& u, Unit& U) -> bool {
    if (!ring_take_raw(u, U)) return false;
    if (!kRingUnits && u >= 0) U = unit_at(p, u);
    return true;
  };
  // Fetching thread only.
  auto ring_publish = [&](int u, const Unit& U) -> bool {
    if (!mbar_wait(&uempty[ring_slot], ring_phase ^ 1u, p.timeout_ns, abort_flag, p.status, kWhereSchedule))
      return false;
    volatile int* r = ring + ring_slot * kStride;
    constexpr int kInts = kStride;
    const int v[kSlotInts] = {u, U.e, U.m, U.start, U.n, U.ks, U.kb0, U.kb1};
#pragma unroll
    for (int j = 0; j < kInts; ++j) r[j] = v[j];
    if (kPair) {
#pragma unroll
      for (int j = 0; j < kInts; ++j)
        st_shared_cluster_u32(mapa_shared(const_cast<int*>(&r[j]), 1), static_cast<uint32_t>(v[j]));
      mbar_arrive_cluster(mapa_shared(&ufull[ring_slot], 1));
    }
    mbar_arrive(&ufull[ring_slot]);
    ring_advance();
    return true;
  };
  // Warp-wide version of ring_take for the epilogue / converter warps.
  auto warp_take = [&](int& u, Unit& U) -> bool {
    int good = 1, v = -1;
    Unit W{};
    if (lane == 0) good = ring_take_raw(v, W) ? 1 : 0;
    good = __shfl_sync(0xFFFFFFFFu, good, 0);
    u = __shfl_sync(0xFFFFFFFFu, v, 0);
    if (kRingUnits) {
      U.e = __shfl_sync(0xFFFFFFFFu, W.e, 0);
      U.m = __shfl_sync(0xFFFFFFFFu, W.m, 0);
      U.start = __shfl_sync(0xFFFFFFFFu, W.start, 0);
      U.n = __shfl_sync(0xFFFFFFFFu, W.n, 0);
      U.ks = __shfl_sync(0xFFFFFFFFu, W.ks, 0);
      U.kb0 = __shfl_sync(0xFFFFFFFFu, W.kb0, 0);
      U.kb1 = __shfl_sync(0xFFFFFFFFu, W.kb1, 0);
    } else if (u >= 0) {
      U = unit_at(p, u);
    }
    return good != 0;
  };

  // TMA coordinates of the weight box of rows [row, row + 128) and k-block kb
  // (x_rows: its column in the row-major layout); tiled layout: box (i, kb)
  // of the 128-row block i is tile i * k_blocks + kb, 128 rows of the tiled
  // view.  Scale boxes cover four k-blocks.
  auto a_y = [&](int row, int kb) { return p.a_tiled ? ((row >> 7) * p.k_blocks + kb) << 7 : row; };
  auto a_x = [&](int x_rows) { return p.a_tiled ? 0 : x_rows; };
  auto s_y = [&](int row, int kb) { return p.a_tiled ? ((row >> 7) * (p.k_blocks >> 2) + (kb >> 2)) << 7 : row; };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol_x = l2_policy_evict_last();
      const int total_units = __ldg(&p.chunk_prefix[kExperts]) * p.m_tiles * p.k_splits;
      int stage = 0;
      uint32_t phase = 0;
      long long issued = 0;
      bool ok = true;
      while (ok) {
        int u;
        Unit U{};
        if (rank == 0) {
          u = atomicAdd(p.sched, 1);
          if (u >= total_units) u = -1;
          if (kRingUnits && u >= 0) U = unit_at(p, u);
          if (!ring_publish(u, U)) break;
          if (!kRingUnits && u >= 0) U = unit_at(p, u);
        } else if (!ring_take(u, U)) {
          break;
        }
        if (u < 0) break;
        const int a_row = U.e * p.a_rows_per_expert + U.m * kRowsPerUnit + static_cast<int>(rank) * kBlockM;
        // pair: this CTA loads token rows [start + rank*N/2, +N/2), N = round16(n)
        const int n_local = kPair ? ((U.n + 15) & ~15) / 2 : U.n;
        const int b_row0 = U.start + static_cast<int>(rank) * n_local;
        // activations: one box of the tile's full height when the chunk fills
        // more than half of it (rows past the chunk are loaded and not read),
        // else ceil(n / 32) boxes of 32 rows; NVFP4 stages of several
        // k-blocks always load the full height
        const bool big = 2 * n_local > p.b_big_rows || S > 1 || p.b_big_rows < kBoxRows;
        const int nbox = big ? 1 : (n_local + kBoxRows - 1) / kBoxRows;
        const uint32_t a_bytes = kFp4 ? kNumA * (S * kPackedTileBytes + kScaleTileBytes) : kNumA * kATileBytes;
        const uint32_t bytes =
            a_bytes + (big ? static_cast<uint32_t>(S * p.b_big_rows) * (kBlockK * 2) : static_cast<uint32_t>(nbox) * kBoxBytes);
        const CUtensorMap* bmap = big ? &maps.bb : &maps.b;
        const int box_rows = big ? 0 : kBoxRows;  // row step between boxes
        for (int kb = U.kb0; kb < U.kb1; kb += S) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, p.timeout_ns, abort_flag, p.status, kWhereProducerEmpty)) {
            ok = false;
            break;
          }
          const int kx = kb * kKElems;
          if (kPair) {
            // both CTAs' bytes land on the even CTA's full barrier
            const uint32_t bar0 = mapa_shared(&full[stage], 0);
            if (rank == 0) mbar_arrive_expect_tx(&full[stage], 2 * bytes);
            tma_load_2d_pair(a_tile(stage, 0), &maps.a0, bar0, a_x(kx), a_y(a_row, kb));
            if (kMode == 0)
              tma_load_2d_pair(a_tile(stage, 1), &maps.a1, bar0, a_x(kx), a_y(a_row, kb));
            else  // second 256-row half of the down unit
              tma_load_2d_pair(a_tile(stage, 1), &maps.a0, bar0, a_x(kx), a_y(a_row + 2 * kBlockM, kb));
            for (int b = 0; b < nbox; ++b)
              tma_load_2d_pair_hint(b_tile(stage) + b * kBoxBytes, bmap, bar0, kx, b_row0 + b * box_rows, pol_x);
          } else {
            mbar_arrive_expect_tx(&full[stage], bytes);
            if (kFp4) {
              const int sx = a_x((kb >> 2) * static_cast<int>(kScaleBoxCols));
              // gate/up: gate and up tiles of the same rows; down: rows a_row and a_row + 128
              const int a_row1 = kMode == 0 ? a_row : a_row + kHalfRows;
              // packed codes of S k-blocks: S consecutive tiles of the tiled
              // layout's 3-D view (bytes, row, tile), or one 2-D box when S = 1
              if (S > 1) {
                tma_load_3d(p_tile(stage, 0, 0), &maps.a0, &full[stage], 0, 0, (a_row >> 7) * p.k_blocks + kb);
                tma_load_3d(p_tile(stage, 1, 0), &maps.a1, &full[stage], 0, 0, (a_row1 >> 7) * p.k_blocks + kb);
              } else {
                tma_load_2d_nohint(p_tile(stage, 0, 0), &maps.a0, &full[stage], a_x(kx / 2), a_y(a_row, kb));
                tma_load_2d_nohint(p_tile(stage, 1, 0), &maps.a1, &full[stage], a_x(kx / 2), a_y(a_row1, kb));
              }
              tma_load_2d_nohint(s_tile(stage, 0), &maps.s0, &full[stage], sx, s_y(a_row, kb));
              tma_load_2d_nohint(s_tile(stage, 1), &maps.s1, &full[stage], sx, s_y(a_row1, kb));
            } else {
              tma_load_2d_nohint(a_tile(stage, 0), &maps.a0, &full[stage], a_x(kx), a_y(a_row, kb));
              // gate/up: the up tile of the same rows; wide down: rows a_row + 128 (a1 = a0)
              if (kNumA == 2)
                tma_load_2d_nohint(a_tile(stage, 1), &maps.a1, &full[stage], a_x(kx),
                                   a_y(kMode == 0 ? a_row : a_row + kHalfRows, kb));
            }
            if (kFp4 && S > 1)  // the chunk's rows for S k-blocks: 3-D view (element, row, k-block)
              tma_load_3d_hint(b_tile(stage), bmap, &full[stage], 0, U.start, kb, pol_x);
            else
              for (int b = 0; b < nbox; ++b)
                tma_load_2d(b_tile(stage) + b * kBoxBytes, bmap, &full[stage], kx, U.start + b * box_rows, pol_x);
          }
          ++issued;
          if (++stage == p.stages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Drain: the latest load issued on every slot has landed (immediate in
      // the normal case, where the MMA warp consumed them all).  Pair: the
      // even CTA's barriers also count the other CTA's bytes.
      for (int s = 0; s < p.stages && rank == 0; ++s) {
        if (issued <= s && issued < p.stages) continue;  // slot never used
        const uint32_t par = s < stage ? phase : (phase ^ 1u);
        mbar_wait(&full[s], par, p.timeout_ns, nullptr, p.status, kWhereDrain);
      }
    }
  } else if (kFp4 && (warp == 1 || (warp >= kMma2Warp && warp < kMma2Warp + static_cast<int>(kIssuers) - 1))) {
    // ------------------------------------------------------------ MMA issuers (NVFP4)
    // One thread per weight matrix of the unit (gate / up, or the two row
    // halves of a down unit), each its own accumulator chain, A (the FP16
    // tile the converters wrote) from TMEM, B from the stage's activation
    // tile of that k-block; descriptors formed once per stage.  In the decode
    // variant each matrix has two accumulators, one for the K steps 0 and 2
    // of every k-block and one for the steps 1 and 3 (the epilogue adds the
    // two), and each accumulator its own issuing thread.  Per k-block: wait
    // for the converters, the thread's MMAs (four, or two in the decode
    // variant), a commit that frees the TMEM tile; per stage a commit that
    // frees the shared-memory stage.
    const int issuer = warp == 1 ? 0 : warp - kMma2Warp + 1;
    const int mat = kDec ? (issuer & 1) : issuer;  // the weight matrix (tile) of this thread
    const uint32_t ks0 = kDec ? static_cast<uint32_t>(issuer >> 1) : 0u;  // decode: K steps ks0, ks0 + 2
    if (lane == 0) {
      int stage = 0, acc = 0, astage = 0;
      uint32_t phase = 0, acc_phase = 0, aphase = 0;
      constexpr uint32_t kAStep = kNumA * (kBlockK / 2);  // TMEM columns of one expanded k-block
      const uint32_t b_step = b_tile_bytes >> 4;          // descriptor address units per k-block of a stage
      bool ok = true;
      while (ok) {
        int u;
        Unit U;
        if (!ring_take(u, U) || u < 0) break;
        const uint32_t idesc = idesc_f16_f32(kBlockM, static_cast<uint32_t>((U.n + 15) & ~15));
        if (!mbar_wait(&acc_empty[acc], acc_phase ^ 1u, p.timeout_ns, abort_flag, p.status, kWhereMmaAccEmpty))
          break;
        tc_fence_after();
        // decode: the accumulator of K steps 1 and 3 lies 2 * nmax columns after that of steps 0 and 2
        const uint32_t d = tmem_base + static_cast<uint32_t>(acc) * p.acc_cols + static_cast<uint32_t>(mat * p.nmax) +
                           ks0 * static_cast<uint32_t>(2 * p.nmax);
        for (int kb = U.kb0; kb < U.kb1 && ok; kb += S) {
          const uint64_t db0 = sdesc_k_sw128(smem_u32(b_tile(stage)));
          for (int sub = 0; sub < S; ++sub) {
            if (!mbar_wait(&afull[astage], aphase, p.timeout_ns, abort_flag, p.status, kWhereMmaFull)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t db = db0 + static_cast<uint64_t>(sub) * b_step;
            const uint32_t ta = tmem_base + p.a_col0 + static_cast<uint32_t>(astage) * kAStep +
                                static_cast<uint32_t>(mat * (kBlockK / 2));
            const uint32_t first = (kb + sub == U.kb0) ? 1u : 0u;  // the unit's first k-block starts the sum
            if (kDec) {  // K steps ks0 and ks0 + 2 (8 TMEM columns, 2 descriptor units each)
              mma_f16_ts(d, ta + 8u * ks0, db + 2u * ks0, idesc, first ^ 1u);
              mma_f16_ts(d, ta + 8u * (ks0 + 2u), db + 2u * (ks0 + 2u), idesc, 1u);
            } else {
              mma_f16_ts(d, ta, db, idesc, first ^ 1u);
              mma_f16_ts(d, ta + 8u, db + 2u, idesc, 1u);
              mma_f16_ts(d, ta + 16u, db + 4u, idesc, 1u);
              mma_f16_ts(d, ta + 24u, db + 6u, idesc, 1u);
            }
            mma_commit(&aempty[astage]);  // the TMEM tile is free once these MMAs complete
            if (++astage == p.a_stages) {
              astage = 0;
              aphase ^= 1u;
            }
          }
          if (!ok) break;
          mma_commit(&empty[stage]);  // the stage is free once its last k-block's MMAs complete
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
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && rank == 0) {
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      while (ok) {
        int u;
        Unit U;
        if (!ring_take(u, U) || u < 0) break;
        const uint32_t n_mma = static_cast<uint32_t>((U.n + 15) & ~15);
        const uint32_t idesc = kFp8 ? idesc_e4m3_f32(kPair ? 2 * kBlockM : kBlockM, n_mma)
                                    : idesc_bf16_f32(kPair ? 2 * kBlockM : kBlockM, n_mma);
        if (!mbar_wait(&acc_empty[acc], acc_phase ^ 1u, p.timeout_ns, abort_flag, p.status, kWhereMmaAccEmpty))
          break;
        tc_fence_after();
        const uint32_t d0 = tmem_base + static_cast<uint32_t>(acc) * p.acc_cols;
        const uint32_t d1 = d0 + static_cast<uint32_t>(p.nmax);
        for (int kb = U.kb0; kb < U.kb1; ++kb) {
          if (!mbar_wait(&full[stage], phase, p.timeout_ns, abort_flag, p.status, kWhereMmaFull)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t db = sdesc_k_sw128(smem_u32(b_tile(stage)));
          {
            const uint64_t da0 = sdesc_k_sw128(smem_u32(a_tile(stage, 0)));
            const uint64_t da1 = sdesc_k_sw128(smem_u32(a_tile(stage, kNumA - 1)));
#pragma unroll
            for (int k = 0; k < kBlockK / 16; ++k) {
              const uint32_t accumulate = (kb != U.kb0 || k != 0) ? 1u : 0u;
              if (kPair && kFp8) {
                mma_f8_pair(d0, da0 + 2u * k, db + 2u * k, idesc, accumulate);
                mma_f8_pair(d1, da1 + 2u * k, db + 2u * k, idesc, accumulate);
              } else if (kPair) {
                mma_bf16_pair(d0, da0 + 2u * k, db + 2u * k, idesc, accumulate);
                mma_bf16_pair(d1, da1 + 2u * k, db + 2u * k, idesc, accumulate);
              } else if (kFp8) {
                mma_f8(d0, da0 + 2u * k, db + 2u * k, idesc, accumulate);
                if (kNumA == 2) mma_f8(d1, da1 + 2u * k, db + 2u * k, idesc, accumulate);
              } else {
                mma_bf16(d0, da0 + 2u * k, db + 2u * k, idesc, accumulate);
                if (kNumA == 2) mma_bf16(d1, da1 + 2u * k, db + 2u * k, idesc, accumulate);
              }
            }
          }
          if (kPair)
            mma_commit_pair_multicast(&empty[stage], 0x3);
          else
            mma_commit(&empty[stage]);
          stage = stage + 1 == p.stages ? 0 : stage + 1;
          phase ^= stage == 0 ? 1u : 0u;
        }
        if (!ok) break;
        if (kPair)
          mma_commit_pair_multicast(&acc_full[acc], 0x3);
        else
          mma_commit(&acc_full[acc]);
        if (++acc == p.acc_stages) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      // Every MMA issued by this thread has completed before TMEM is freed.
      if (kPair)
        mma_commit_pair_multicast(drain, 0x1);
      else
        mma_commit(drain);
      mbar_wait(drain, 0, p.timeout_ns, nullptr, p.status, kWhereDrain);
    }
  } else if (warp < 2 + kEpi) {
    // ------------------------------------------------------------ epilogue
    const int quad = warp & 3;               // TMEM lanes this warp may read
    const int half = (warp - 2) >> 2;        // which 16-column chunks (even / odd)
    const int row = quad * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    while (true) {
      int u;
      Unit U;
      if (!warp_take(u, U) || u < 0) break;
      int ok = 1;
      if (lane == 0)
        ok = mbar_wait(&acc_full[acc], acc_phase, p.timeout_ns, abort_flag, p.status, kWhereEpiAccFull) ? 1 : 0;
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + static_cast<uint32_t>(acc) * p.acc_cols;
      const int feat = U.m * kRowsPerUnit + static_cast<int>(rank) * kBlockM + row;
      constexpr int kOut = (kMode == 1 && kNumA == 2) ? 2 : 1;      // down with two weight tiles
      // Row scales: NVFP4 the global scale of each matrix; FP8 this thread's
      // weight row (s0: gate or down, s1: up, or the down unit's second tile)
      float s0, s1;
      if (kFp8) {
        const size_t rrow = static_cast<size_t>(U.e) * p.a_rows_per_expert + feat;
        s0 = __ldg(&p.rs0[rrow]);
        s1 = kMode == 0 ? __ldg(&p.rs1[rrow]) : (kOut == 2 ? __ldg(&p.rs0[rrow + kHalfRows]) : 1.0f);
      } else {
        s0 = p.gs0 != nullptr ? __ldg(&p.gs0[U.e]) : 1.0f;
        s1 = (kMode == 0 && p.gs1 != nullptr) ? __ldg(&p.gs1[U.e]) : 1.0f;
      }
      const int ncols = (U.n + 15) & ~15;
      if (!kFp4 && !kPair && !kWide && p.partial != nullptr) {  // K split: 128-row units, BF16 / FP8
        // K split: FP32 partial sums (row scales applied, they are linear)
        // of this part, stored as they are read; the finishing kernel adds
        // the parts and applies SwiGLU / the BF16 rounding.
        const size_t plane = static_cast<size_t>(p.rows) * p.out_ld;
        float* part0 = p.partial + static_cast<size_t>(U.ks) * (kMode == 0 ? 2 : 1) * plane + feat;
        for (int c0 = 16 * half; c0 < ncols; c0 += 16 * kEpiHalves) {
          float g[16], g2[16];
          tmem_ld16(tbase + static_cast<uint32_t>(c0), g);
          if (kNumA == 2) tmem_ld16(tbase + static_cast<uint32_t>(p.nmax + c0), g2);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float cs = kFp8 ? __ldg(&p.bscale[U.start + c0 + j]) : 1.0f;
            if (c0 + j < U.n) {
              float* dst = part0 + static_cast<size_t>(U.start + c0 + j) * p.out_ld;
              dst[0] = g[j] * cs * s0;
              if (kMode == 0) dst[plane] = g2[j] * cs * s1;            // up: the second plane
              if (kMode == 1 && kOut == 2) dst[kHalfRows] = g2[j] * cs * s1;
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (kPair)
            mbar_arrive_cluster(mapa_shared(&acc_empty[acc], 0));
          else
            mbar_arrive(&acc_empty[acc]);
        }
        if (++acc == p.acc_stages) {
          acc = 0;
          acc_phase ^= 1u;
        }
        continue;
      }
      __nv_bfloat16* out = p.out + static_cast<size_t>(U.start) * p.out_ld + feat;
      // 1) TMEM -> packed BF16 results in registers (this warp's 16-column
      //    chunks), 2) release the accumulator so the next unit's MMAs start,
      //    3) global stores.
      // this warp's 16-column chunks: columns / (kEpiHalves x 16)
      constexpr int kMaxChunks = (kDec ? kDecChunkRows : (kFp4 ? kChunkRowsFp4 : kChunkRowsBf16)) / (16 * kEpiHalves);
      uint32_t hp[kOut][kMaxChunks][8];
#pragma unroll
      for (int ci = 0; ci < kMaxChunks; ++ci) {
        const int c0 = 16 * half + 16 * kEpiHalves * ci;
        if (c0 < ncols) {
          float g[16], g2[16];
          tmem_ld16(tbase + static_cast<uint32_t>(c0), g);
          if (kNumA == 2) tmem_ld16(tbase + static_cast<uint32_t>(p.nmax + c0), g2);
          if (kDec) {  // the odd-K-step accumulators of both matrices
            float o[16], o2[16];
            tmem_ld16(tbase + static_cast<uint32_t>(2 * p.nmax + c0), o);
            tmem_ld16(tbase + static_cast<uint32_t>(3 * p.nmax + c0), o2);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              g[j] += o[j];
              g2[j] += o2[j];
            }
          }
          tmem_ld_wait();
          if (kFp8 || kFp4) {
            // token row scales of these 16 columns (FP8: the E4M3 rows';
            // NVFP4: the inverse powers of two of the FP16 rows; the scale
            // array is padded past the last route, so columns beyond the
            // chunk read in bounds)
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float cs = __ldg(&p.bscale[U.start + c0 + j]);
              g[j] *= cs;
              if (kNumA == 2) g2[j] *= cs;
            }
          }
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            float v0, v1;
            if (kMode == 0) {
              // SiLU(gate) * up in FP32 (fast exp / divide: the result is
              // rounded to BF16 right after, far coarser than their error)
              const float a0 = g[2 * j] * s0, a1 = g[2 * j + 1] * s0;
              v0 = __fdividef(a0, 1.0f + __expf(-a0)) * (g2[2 * j] * s1);
              v1 = __fdividef(a1, 1.0f + __expf(-a1)) * (g2[2 * j + 1] * s1);
            } else {
              v0 = g[2 * j] * s0;
              v1 = g[2 * j + 1] * s0;
            }
            __nv_bfloat162 q = __floats2bfloat162_rn(v0, v1);
            hp[0][ci][j] = *reinterpret_cast<uint32_t*>(&q);
            if (kOut == 2) {
              const float sb = kFp8 ? s1 : s0;  // the second tile's row scale
              __nv_bfloat162 q2 = __floats2bfloat162_rn(g2[2 * j] * sb, g2[2 * j + 1] * sb);
              hp[kOut - 1][ci][j] = *reinterpret_cast<uint32_t*>(&q2);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (kPair)
          mbar_arrive_cluster(mapa_shared(&acc_empty[acc], 0));
        else
          mbar_arrive(&acc_empty[acc]);
      }
#pragma unroll
      for (int ci = 0; ci < kMaxChunks; ++ci) {
        const int c0 = 16 * half + 16 * kEpiHalves * ci;
        if (c0 < ncols) {
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            if (c0 + j < U.n) {
              const uint32_t w0 = hp[0][ci][j >> 1];
              const uint16_t b0 = static_cast<uint16_t>((j & 1) ? (w0 >> 16) : (w0 & 0xFFFFu));
              *reinterpret_cast<uint16_t*>(out + static_cast<size_t>(c0 + j) * p.out_ld) = b0;
              if (kOut == 2) {
                const uint32_t w1 = hp[kOut - 1][ci][j >> 1];
                const uint16_t b1 = static_cast<uint16_t>((j & 1) ? (w1 >> 16) : (w1 & 0xFFFFu));
                *reinterpret_cast<uint16_t*>(out + static_cast<size_t>(c0 + j) * p.out_ld + kHalfRows) = b1;
              }
            }
          }
        }
      }
      if (++acc == p.acc_stages) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  } else if (kFp4 && warp < kMma2Warp) {
    // ------------------------------------------------------------ converters
    // Warp w may write TMEM lanes 32*(w%4)..+31, so its lane i expands weight
    // row 32*(w%4)+i.  The converter groups (4 warps each) take the k-blocks
    // in turn (counted over all units), so G k-blocks are expanded at once;
    // a thread expands its row of every weight matrix of the unit (gate and
    // up, or down): 64 K elements = 32 TMEM columns each.
    const int cw = warp - (2 + kEpi);
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const int group = cw >> 2;
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    // This group's k-blocks: kb = group, group + G, ... of every unit (G =
    // kGroups; the same split in every unit, so a unit's sums do not depend
    // on which units the CTA ran before).  For the CTA's running k-block
    // index i: the stage holding it (S k-blocks per stage), its phase and its
    // place `sub` in the stage; its TMEM tile (i mod a_stages) and the parity
    // of that tile's previous release (aempty: the MMAs of k-block
    // i - a_stages completed; the MMA threads issue the k-blocks in order, so
    // the release of k-block i - 2*a_stages has completed by then and the
    // wait cannot be mistaken for it).  The host keeps G <= a_stages.
    int sub = 0, stage = 0, astage = 0, i = 0;
    uint32_t phase = 0, aphase = 1;
    auto advance_to = [&](int target) {  // target >= i
      const int by = target - i;
      sub += by;
      while (sub >= S) {
        sub -= S;
        if (++stage == p.stages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      astage += by;
      while (astage >= p.a_stages) {
        astage -= p.a_stages;
        aphase ^= 1u;
      }
      i = target;
    };
    int unit_base = 0;  // running index of the current unit's first k-block
    bool ok = true;
    while (ok) {
      int u;
      Unit U;
      if (!warp_take(u, U) || u < 0) break;
      for (int kb = group; kb < p.k_blocks; kb += kGroups) {
        advance_to(unit_base + kb);
        int good = 1;
        if (lane == 0)
          good = (mbar_wait(&full[stage], phase, p.timeout_ns, abort_flag, p.status, kWhereConvert) &&
                  (i < p.a_stages ||
                   mbar_wait(&aempty[astage], aphase, p.timeout_ns, abort_flag, p.status, kWhereConvert)))
                     ? 1
                     : 0;
        good = __shfl_sync(0xFFFFFFFFu, good, 0);
        if (!good) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t ta0 = tmem_base + lane_addr + p.a_col0 + static_cast<uint32_t>(astage * kNumA * (kBlockK / 2));
#pragma unroll
        for (int mat = 0; mat < kNumA; ++mat) {
          // packed row: 32 bytes (64 elements); scale row: this k-block's 4
          // E4M3 codes at byte 4*(kb%4), one per 16 elements
          const uint4* src = reinterpret_cast<const uint4*>(p_tile(stage, mat, sub) + row * (kBlockK / 2));
          const uint4 v0 = src[0], v1 = src[1];
          const uint32_t wv[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
          const uint32_t sc4 =
              *reinterpret_cast<const uint32_t*>(s_tile(stage, mat) + row * kScaleBoxCols + 4 * (kb & 3));
          uint32_t sp[4];
          scales4_to_f16_pairs(sc4, sp);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t out[16];
#pragma unroll
            for (int g = 0; g < 2; ++g)  // 16 elements per scale
              nvfp4x16_to_f16(wv[4 * h + 2 * g], wv[4 * h + 2 * g + 1], sp[2 * h + g], out + 8 * g);
            tmem_st16(ta0 + static_cast<uint32_t>(mat * (kBlockK / 2) + 16 * h), out);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&afull[astage]);
      }
      unit_base += p.k_blocks;
    }
  }

  tc_fence_before();
  if (kPair)
    cluster_sync();  // no CTA leaves while the other may still signal its barriers
  else
    __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    if (kPair)
      tmem_dealloc_pair(tmem_base, p.tmem_cols);
    else
      tmem_dealloc(tmem_base, p.tmem_cols);
  }
}

template <int kMode, bool kFp4, bool kPair, bool kWide = false, bool kFp8 = false, bool kDec = false>
cudaError_t launch_one(const GemmMaps& maps, const GemmParams& p, int grid, size_t smem_bytes, cudaStream_t stream) {
  auto kern = moe_gemm_kernel<kMode, kFp4, kPair, kWide, kFp8, kDec>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem_bytes));
  if (err != cudaSuccess) return err;
  if (!kPair) {
    kern<<<grid, kFp4 ? (kDec ? kThreadsFp4Dec : kThreadsFp4) : kThreadsBf16, smem_bytes, stream>>>(maps, p);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kThreadsBf16);
  cfg.dynamicSmemBytes = smem_bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  err = cudaLaunchKernelEx(&cfg, kern, maps, p);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

}  // namespace

size_t gemm_smem_bytes(int stages, int acc_stages, size_t stage_bytes) {
  return 1024 + static_cast<size_t>(stages) * stage_bytes +
         (2 * stages + 3 * kMaxAStages + 2 * acc_stages + 1 + 2 * kSchedRing) * 8 + kSchedRing * kSlotInts * 4 + 16;
}

int gemm_pair_max_clusters(int mode, size_t smem_bytes) {
  auto kern = mode == 0 ? moe_gemm_kernel<0, false, true> : moe_gemm_kernel<1, false, true>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem_bytes)) !=
      cudaSuccess)
    return 0;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 0) != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(kThreadsBf16);
  cfg.dynamicSmemBytes = smem_bytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

cudaError_t launch_gemm(int mode, bool fp4, bool pair, bool wide, bool fp8, bool dec, const GemmMaps& maps,
                        const GemmParams& p, int grid, size_t smem_bytes, cudaStream_t stream) {
  if (dec) {
    if (!fp4 || pair || fp8) return cudaErrorInvalidValue;
    return mode == 0 ? launch_one<0, true, false, false, false, true>(maps, p, grid, smem_bytes, stream)
                     : launch_one<1, true, false, false, false, true>(maps, p, grid, smem_bytes, stream);
  }
  if (fp8) {
    if (fp4) return cudaErrorInvalidValue;
    if (pair)
      return mode == 0 ? launch_one<0, false, true, false, true>(maps, p, grid, smem_bytes, stream)
                       : launch_one<1, false, true, false, true>(maps, p, grid, smem_bytes, stream);
    if (mode == 0) return launch_one<0, false, false, false, true>(maps, p, grid, smem_bytes, stream);
    return wide ? launch_one<1, false, false, true, true>(maps, p, grid, smem_bytes, stream)
                : launch_one<1, false, false, false, true>(maps, p, grid, smem_bytes, stream);
  }
  if (pair) {
    if (fp4) return cudaErrorInvalidValue;
    return mode == 0 ? launch_one<0, false, true>(maps, p, grid, smem_bytes, stream)
                     : launch_one<1, false, true>(maps, p, grid, smem_bytes, stream);
  }
  if (mode == 0)
    return fp4 ? launch_one<0, true, false>(maps, p, grid, smem_bytes, stream)
               : launch_one<0, false, false>(maps, p, grid, smem_bytes, stream);
  if (fp4) return launch_one<1, true, false>(maps, p, grid, smem_bytes, stream);
  return wide ? launch_one<1, false, false, true>(maps, p, grid, smem_bytes, stream)
              : launch_one<1, false, false>(maps, p, grid, smem_bytes, stream);
}

}  // namespace beam

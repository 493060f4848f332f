// select.cuh -- the group-limited top-k selection of one token by one warp,
// shared by the router kernels.
//
// Beam launch post ("Willkommen Beam ..." (spke.com), section "Mixture of
// Experts"): sigmoid scores over 256 experts, 8 groups of 32 ranked by the
// sum of their two best scores, the best 4 groups kept, the top-8 experts
// inside them, weights normalised and scaled.  An optional bias steers the
// selection only.  Lane l holds experts 8l..8l+7, so lanes 4j..4j+3 hold
// group j; ties go to the lower group / expert index.
#pragma once
#include <cmath>

#include "moe_internal.cuh"

namespace beam {

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


}  // namespace beam

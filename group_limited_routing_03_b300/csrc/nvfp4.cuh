// nvfp4.cuh -- exact expansion of NVFP4 weights to FP16 on the conversion
// units (cvt ... e2m1x2 / e4m3x2), used by the grouped GEMMs' converter
// warps and by the library's expansion test hook.
//
// Beam launch post, section "Mixture of Experts": NVFP4 is the Blackwell
// checkpoint format.  An element is e2m1 * e4m3 (block scale, one per 16 K
// elements) * global; the e2m1 * e4m3 product has at most 2 + 4 significant
// bits and lies in [2^-10, 2688] (or is zero), so it is exact in FP16 (11
// significant bits, normal from 2^-14 to 65504): one FP16 multiply of the
// converted code by the converted scale gives it exactly.
#pragma once
#include <cuda_fp16.h>

#include <cstdint>

namespace beam {

__device__ __forceinline__ uint32_t prmt_u32(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

// Four bytes of E2M1 pairs (byte j: element 2j in the low nibble, 2j+1 in
// the high nibble) -> four FP16x2 words (word j: element 2j in the low half).
__device__ __forceinline__ void e2m1x8_to_f16x8(uint32_t w, uint32_t (&o)[4]) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3])
      : "r"(w));
}

// Two E4M3 codes (the first in the low byte) -> FP16x2 (the first in the
// low half), exact (E4M3 values, subnormals included, are FP16 normals).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_codes) {
  uint32_t r;
  const uint16_t v = static_cast<uint16_t>(two_codes & 0xFFFFu);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(v));
  return r;
}

// Four E4M3 block scales (one 32-bit word, block i in byte i) -> each as an
// FP16 pair (s_i, s_i).
__device__ __forceinline__ void scales4_to_f16_pairs(uint32_t sc4, uint32_t (&s)[4]) {
  const uint32_t a = e4m3x2_to_f16x2(sc4), b = e4m3x2_to_f16x2(sc4 >> 16);
  s[0] = prmt_u32(a, 0u, 0x1010u);  // low half twice
  s[1] = prmt_u32(a, 0u, 0x3232u);  // high half twice
  s[2] = prmt_u32(b, 0u, 0x1010u);
  s[3] = prmt_u32(b, 0u, 0x3232u);
}

// One block of 16 E2M1 elements (two words, element i of word q in bits
// 4i..4i+3 = K index 8q + i) times its scale pair -> eight FP16x2 words in K
// order (the even K index in the low half).
__device__ __forceinline__ void nvfp4x16_to_f16(uint32_t w0, uint32_t w1, uint32_t scale_pair, uint32_t* o) {
  uint32_t a[4], b[4];
  e2m1x8_to_f16x8(w0, a);
  e2m1x8_to_f16x8(w1, b);
  const __half2 s2 = *reinterpret_cast<const __half2*>(&scale_pair);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    __half2 va = __hmul2(*reinterpret_cast<const __half2*>(&a[j]), s2);  // exact: at most 6 significant bits
    __half2 vb = __hmul2(*reinterpret_cast<const __half2*>(&b[j]), s2);
    o[j] = *reinterpret_cast<const uint32_t*>(&va);
    o[4 + j] = *reinterpret_cast<const uint32_t*>(&vb);
  }
}

}  // namespace beam

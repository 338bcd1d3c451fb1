// MXFP8 block-scale helpers (E4M3 elements, one E8M0 scale per 32 elements).
//
// Scale rule: shared exponent s = floor(log2(amax)) - 8 (8 = the largest E4M3
// exponent), clamped below at -127; scale code s + 127; element codes are
// RNE(v / 2^s) with saturation to +-448.  This is the OCP microscaling rule;
// the MXFP4 page ("GPT-OSS-120B with MXFP4 on DGX Spark (SM121/GB10)",
// "Numerical Accuracy") asks for full-scale block activation scaling without
// fixing the rule.
#pragma once

#include <stdint.h>

namespace moe {

// floor(log2(amax)) - 8, at least -127.  amax >= 0 (fp32 bit pattern ordering).
__device__ __forceinline__ int mx_scale_exp(float amax) {
  const int biased = (int)((__float_as_uint(amax) >> 23) & 0xFFu);
  if (biased == 0) return -127;  // zero or subnormal: floor(log2) <= -127
  return max(biased - 127 - 8, -127);
}

// 2^-s as an fp32 (exact for s in [-127, 126]).
__device__ __forceinline__ float mx_pow2_neg(int s) { return __uint_as_float((uint32_t)(127 - s) << 23); }

}  // namespace moe

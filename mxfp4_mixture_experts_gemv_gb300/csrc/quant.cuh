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

#include "ptx.cuh"

namespace moe {

// floor(log2(amax)) - emax, at least -127.  amax >= 0 (fp32 bit pattern ordering);
// emax is the element format's largest exponent: 8 for E4M3 (448 = 1.75 * 2^8),
// 2 for E2M1 (6 = 1.5 * 2^2).
template <int EMAX = 8>
__device__ __forceinline__ int mx_scale_exp(float amax) {
  const int biased = (int)((__float_as_uint(amax) >> 23) & 0xFFu);
  if (biased == 0) return -127;  // zero or subnormal: floor(log2) <= -127
  return max(biased - 127 - EMAX, -127);
}

// 2^-s as an fp32 (exact for s in [-127, 126]).
__device__ __forceinline__ float mx_pow2_neg(int s) { return __uint_as_float((uint32_t)(127 - s) << 23); }

// Eight bf16 (one 16-byte load) to fp32.
__device__ __forceinline__ void bf16x8(const uint4 v, float (&f)[8]) {
  const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(u[i] << 16);
    f[2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
  }
}

// Quantise one 32-element block of bf16 (four 16-byte words, already loaded) to
// MXFP8: the 32 codes in c, returns the scale code.
__device__ __forceinline__ uint8_t quant_block_vals(const uint4 (&v)[4], uint4 (&c)[2]) {
  float f[32];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    float g[8];
    bf16x8(v[q], g);
#pragma unroll
    for (int i = 0; i < 8; ++i) f[8 * q + i] = g[i];
  }
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(f[i]));
  const int s = mx_scale_exp(amax);
  const float inv = mx_pow2_neg(s);
  uint32_t pk[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t lo = cvt_e4m3x2(f[4 * i] * inv, f[4 * i + 1] * inv);
    const uint32_t hi = cvt_e4m3x2(f[4 * i + 2] * inv, f[4 * i + 3] * inv);
    pk[i] = lo | (hi << 16);
  }
  c[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
  c[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
  return (uint8_t)(s + 127);
}

// Quantise one 32-element block of bf16 to MXFP4 (the FP4-activation variant):
// shared exponent floor(log2(amax)) - 2, elements E2M1 with round-to-nearest-even
// and saturation to +-6, the same reading of the OCP microscaling rule as MXFP8.
// The 32 codes, two per byte (lower-index element in the low nibble), in c[0];
// returns the scale code.
__device__ __forceinline__ uint8_t quant_block_vals_fp4(const uint4 (&v)[4], uint4 (&c)[2]) {
  float f[32];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    float g[8];
    bf16x8(v[q], g);
#pragma unroll
    for (int i = 0; i < 8; ++i) f[8 * q + i] = g[i];
  }
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(f[i]));
  const int s = mx_scale_exp<2>(amax);
  const float inv = mx_pow2_neg(s);
#pragma unroll
  for (int i = 0; i < 32; ++i) f[i] *= inv;
  c[0] = make_uint4(cvt_e2m1x8(f), cvt_e2m1x8(f + 8), cvt_e2m1x8(f + 16), cvt_e2m1x8(f + 24));
  c[1] = make_uint4(0u, 0u, 0u, 0u);
  return (uint8_t)(s + 127);
}

// E4M3 code -> fp32 (exact; codes from a saturating conversion, never NaN).
__device__ __forceinline__ float e4m3_value(uint32_t c) {
  const uint32_t e = (c >> 3) & 15u, m = c & 7u;
  const float v = e ? __uint_as_float(((e + 120u) << 23) | (m << 20)) : (float)m * 0.001953125f;  // m * 2^-9
  return (c & 0x80u) ? -v : v;
}

// NVFP4 quantisation of one 16-element block with global scale gs: scale code =
// E4M3(amax / (6 gs)) with round-to-nearest-even and saturation at 448, element
// codes = E2M1(v / (scale * gs)) likewise (zero codes if the scale is zero), the
// divisions in IEEE fp32.  The 16 codes, two per byte (lower-index element in
// the low nibble), in pk[0..1]; returns the scale code.
__device__ __forceinline__ uint32_t nvfp4_block16(const float* v, float gs, uint32_t (&pk)[2]) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
  const uint32_t sc = cvt_e4m3x2(__fdiv_rn(amax, __fmul_rn(6.0f, gs)), 0.f) & 0xFFu;
  const float sv = __fmul_rn(e4m3_value(sc), gs);
  float x[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) x[i] = sv == 0.f ? 0.f : __fdiv_rn(v[i], sv);
  pk[0] = cvt_e2m1x8(x);
  pk[1] = cvt_e2m1x8(x + 8);
  return sc;
}

// Either activation format: MXFP8 (fp4 false; 32 code bytes in c[0..1]) or
// MXFP4 (fp4 true; 16 code bytes in c[0]).
__device__ __forceinline__ uint8_t quant_block_act(const uint4 (&v)[4], uint4 (&c)[2], bool fp4) {
  return fp4 ? quant_block_vals_fp4(v, c) : quant_block_vals(v, c);
}

// Store one block's codes at dst (16-byte aligned): 32 bytes (MXFP8) or 16 (MXFP4).
__device__ __forceinline__ void store_block_codes(uint8_t* dst, const uint4 (&c)[2], bool fp4) {
  reinterpret_cast<uint4*>(dst)[0] = c[0];
  if (!fp4) reinterpret_cast<uint4*>(dst)[1] = c[1];
}

// The same from a block in global or shared memory (16-byte aligned).
__device__ __forceinline__ uint8_t quant_block_regs_act(const uint16_t* src, uint4 (&c)[2], bool fp4) {
  uint4 v[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) v[q] = reinterpret_cast<const uint4*>(src)[q];
  return quant_block_act(v, c, fp4);
}

// The same from a block in global or shared memory (16-byte aligned).
__device__ __forceinline__ uint8_t quant_block_regs(const uint16_t* src, uint4 (&c)[2]) {
  uint4 v[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) v[q] = reinterpret_cast<const uint4*>(src)[q];
  return quant_block_vals(v, c);
}

// The same, with the 32 codes stored to dst (16-byte aligned).
__device__ __forceinline__ uint8_t quant_block(const uint16_t* src, uint8_t* dst) {
  uint4 c[2];
  const uint8_t sc = quant_block_regs(src, c);
  reinterpret_cast<uint4*>(dst)[0] = c[0];
  reinterpret_cast<uint4*>(dst)[1] = c[1];
  return sc;
}

// Exclusive prefix sums over E <= 256 counts by one warp (lane l owns entries
// 8l..8l+7): off[e] = sum of cnt[<e], toff[e] = sum of ceil(cnt[<e] / 2^tshift);
// off[E], toff[E] hold the totals and tile_e[t] the expert of every tile t.
__device__ __forceinline__ void warp_expert_scan(const int* cnt, int E, int tshift, int* off, int* toff,
                                                 int* tile_e, int lane) {
  int c[8], tc[8], sum = 0, tsum = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = 8 * lane + i;
    c[i] = e < E ? cnt[e] : 0;
    tc[i] = (c[i] + (1 << tshift) - 1) >> tshift;
    sum += c[i];
    tsum += tc[i];
  }
  int incl = sum, tincl = tsum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o), tv = __shfl_up_sync(0xffffffffu, tincl, o);
    if (lane >= o) {
      incl += v;
      tincl += tv;
    }
  }
  int run = incl - sum, trun = tincl - tsum;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = 8 * lane + i;
    if (e < E) {
      off[e] = run;
      toff[e] = trun;
      for (int t = 0; t < tc[i]; ++t) tile_e[trun + t] = e;
    }
    run += c[i];
    trun += tc[i];
  }
  if (lane == 31) {
    off[E] = incl;
    toff[E] = tincl;
  }
}

}  // namespace moe

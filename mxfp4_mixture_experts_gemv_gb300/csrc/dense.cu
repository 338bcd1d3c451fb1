// Dense MXFP4 linears: out = MXFP8(x) . W^T + b with W [N, K] in MXFP4.
//
// "GPT-OSS-120B with MXFP4 on DGX Spark (SM121/GB10)", "What's Included", "Full
// MXFP4 Quantization Stack": the QKV and O projections and the LM head in MXFP4
// as well as the MoE layers; "Performance Optimizations": a CUDA-core path for
// M <= 4 beside the tensor cores.  The checkpoint keeps those projections in BF16
// ("GPT-OSS-120B on DGX Spark: From MXFP4 to NVFP4", "MXFP4 Tensor Structure"),
// so this file also quantises BF16 weights to MXFP4 (the OCP-style block rule of
// the activations: shared exponent floor(log2 amax) - 2, E2M1 round-to-nearest-
// even, saturating at 6).
//
// The tensor-core path is the expert kernel's down projection with one expert
// (weights in the MMA's M slot, tokens in N; dense mode writes bf16 out + bias);
// this file supplies the weight packing, the identity grouping and the CUDA-core
// GEMV for a few tokens.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>

#include "common.cuh"
#include "quant.cuh"

namespace moe {
namespace {

// BF16 weights -> MXFP4 blocks [N][K/32][16] and E8M0 scales [N][K/32]: one thread
// per 32-element block.
__global__ void dense_quantize_weights_kernel(int N, int K, const uint16_t* __restrict__ w, uint8_t* __restrict__ blocks,
                                              uint8_t* __restrict__ scales) {
  const int64_t nb = (int64_t)N * (K / 32);
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < nb; i += (int64_t)gridDim.x * blockDim.x) {
    uint4 c[2];
    const uint8_t sc = quant_block_regs_act(w + i * 32, c, true);
    reinterpret_cast<uint4*>(blocks)[i] = c[0];
    scales[i] = sc;
  }
}

struct DensePackArgs {
  PackedHeader h;
  const uint8_t* blocks;
  const uint8_t* scales;
  const uint16_t* bias;
  uint8_t* packed;
};

// Data tiles: one thread per 16-byte chunk (32 elements) of the tile-contiguous layout.
__global__ void dense_pack_data_kernel(DensePackArgs a) {
  const PackedHeader& h = a.h;
  const int N = h.H, K = h.I, kt_n = h.d_ktiles, nb = K / 32;
  const uint4* src = reinterpret_cast<const uint4*>(a.blocks);
  uint4* dst = reinterpret_cast<uint4*>(a.packed + h.off_d_data);
  const int64_t per_mtile = (int64_t)kTileM * kt_n * 4;
  const int64_t total = (int64_t)N * kt_n * 4;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int m = (int)(i / per_mtile);
    const int rows_m = min(kTileM, N - m * kTileM);
    const int64_t rem = i - (int64_t)m * per_mtile;
    const int kt = (int)(rem / (rows_m * 4));
    const int rem2 = (int)(rem - (int64_t)kt * rows_m * 4);
    const int r = rem2 >> 2, j = rem2 & 3;
    const int kb = kt * 4 + j;
    dst[i] = kb < nb ? src[(int64_t)(m * kTileM + r) * nb + kb] : make_uint4(0, 0, 0, 0);
  }
}

// Scale atoms (one thread per atom byte), biases, and the header.
__global__ void dense_pack_sf_kernel(DensePackArgs a) {
  const PackedHeader& h = a.h;
  const int N = h.H, K = h.I, mt = h.d_mtiles, kt = h.d_ktiles, nb = K / 32;
  uint8_t* dst = a.packed + h.off_d_sf;
  float* bias = reinterpret_cast<float*>(a.packed + h.off_d_bias);
  const int64_t total = (int64_t)mt * kt * kAtomBytes;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total + N; i += (int64_t)gridDim.x * blockDim.x) {
    if (i >= total) {
      const int n = (int)(i - total);
      bias[n] = a.bias ? __uint_as_float((uint32_t)a.bias[n] << 16) : 0.f;
      continue;
    }
    const int j = (int)(i % kAtomBytes);
    const int64_t q = i / kAtomBytes;
    const int ktile = (int)(q % kt), mtile = (int)(q / kt);
    const int r = (j >> 4) + 32 * ((j & 15) >> 2);
    const int kb = ktile * 4 + (j & 3);
    const int pr = mtile * kTileM + r;
    dst[i] = (pr < N && kb < nb) ? a.scales[(int64_t)pr * nb + kb] : (uint8_t)127;
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) *reinterpret_cast<PackedHeader*>(a.packed) = h;
}

// Eight E2M1 codes (one 32-bit word, lower-index element in the low nibble) ->
// eight fp32 values, by the hardware E2M1 -> f16x2 conversion.
__device__ __forceinline__ void e2m1x8_to_f32(uint32_t w, float (&f)[8]) {
  uint32_t h[4];
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(w));
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 v = __half22float2(*reinterpret_cast<const __half2*>(&h[i]));
    f[2 * i] = v.x;
    f[2 * i + 1] = v.y;
  }
}

constexpr int kGemvMaxT = 4;
constexpr int kGemvThreads = 128;  // one 128-row weight tile per CTA, one row per thread

// CUDA-core path for a few tokens: CTA (m, c) takes weight tile m against the
// k-tiles of chunk c; every thread one weight row.  x is quantised to MXFP8 into
// shared memory (values, fp32), then each row's E2M1 codes are decoded in
// registers and contracted per 32-element block, times the block's E8M0 scale.
__global__ void __launch_bounds__(kGemvThreads) dense_gemv_kernel(PackedHeader h, const uint8_t* __restrict__ packed,
                                                                  const uint16_t* __restrict__ x, int T, int kt_per,
                                                                  float* __restrict__ partial,
                                                                  uint16_t* __restrict__ out) {
  extern __shared__ float s_x[];  // [T][kt_per * 128]
  const int N = h.H, K = h.I, kt_n = h.d_ktiles;
  const int m = blockIdx.x, c = blockIdx.y;
  const int kt0 = c * kt_per, kt1 = min(kt_n, kt0 + kt_per), len = (kt1 - kt0) * kTileK;
  // quantise this chunk of x: one 32-element block per thread and step
  const int nbc = len / 32;
  for (int u = threadIdx.x; u < T * nbc; u += kGemvThreads) {
    const int t = u / nbc, b = u - t * nbc;
    const int kb = kt0 * 4 + b;
    float* dst = s_x + (int64_t)t * len + 32 * b;
    if (kb < K / 32) {
      uint4 v[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) v[q] = reinterpret_cast<const uint4*>(x + (int64_t)t * K + 32 * kb)[q];
      uint4 cd[2];
      const int s = (int)quant_block_vals(v, cd) - 127;
      const float sc = s >= -126 ? __uint_as_float((uint32_t)(s + 127) << 23) : __uint_as_float(1u << (s + 149));
      const uint8_t* cb = reinterpret_cast<const uint8_t*>(cd);
#pragma unroll
      for (int i = 0; i < 32; ++i) dst[i] = e4m3_value(cb[i]) * sc;
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) dst[i] = 0.f;  // padding past K
    }
  }
  __syncthreads();
  const int r = threadIdx.x, rows_m = min(kTileM, N - m * kTileM);
  if (r >= rows_m) return;
  const int pr = m * kTileM + r;
  const uint8_t* data = packed + h.off_d_data;
  const uint8_t* sf = packed + h.off_d_sf;
  float acc[kGemvMaxT] = {0.f, 0.f, 0.f, 0.f};
  for (int kt = kt0; kt < kt1; ++kt) {
    const uint4* row = reinterpret_cast<const uint4*>(data + (tile_row0(0, m, kt, N, kt_n) + r) * kTileRowBytes);
    const uint32_t sw = *reinterpret_cast<const uint32_t*>(sf + ((int64_t)m * kt_n + kt) * kAtomBytes + (r & 31) * 16 + (r >> 5) * 4);
    uint4 q[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) q[j] = __ldcs(row + j);  // weights are read once: stream them
#pragma unroll
    for (int j = 0; j < 4; ++j) {  // 32-element block j of the k-tile
      const uint32_t wds[4] = {q[j].x, q[j].y, q[j].z, q[j].w};
      float part[kGemvMaxT] = {0.f, 0.f, 0.f, 0.f};
      const float* xb = s_x + (kt - kt0) * kTileK + 32 * j;
#pragma unroll
      for (int wq = 0; wq < 4; ++wq) {
        float f[8];
        e2m1x8_to_f32(wds[wq], f);
#pragma unroll
        for (int t = 0; t < kGemvMaxT; ++t)
          if (t < T)
#pragma unroll
            for (int i = 0; i < 8; ++i) part[t] = fmaf(f[i], xb[(int64_t)t * len + 8 * wq + i], part[t]);
      }
      const int s = (int)((sw >> (8 * j)) & 0xFFu);
      const float scale = s ? __uint_as_float((uint32_t)s << 23) : __uint_as_float(0x00400000u);  // 2^(s - 127)
#pragma unroll
      for (int t = 0; t < kGemvMaxT; ++t)
        if (t < T) acc[t] = fmaf(part[t], scale, acc[t]);
    }
  }
  if (partial) {
#pragma unroll
    for (int t = 0; t < kGemvMaxT; ++t)
      if (t < T) partial[((int64_t)c * T + t) * N + pr] = acc[t];
  } else {
    const float b = reinterpret_cast<const float*>(packed + h.off_d_bias)[pr];
#pragma unroll
    for (int t = 0; t < kGemvMaxT; ++t)
      if (t < T) out[(int64_t)t * N + pr] = __bfloat16_as_ushort(__float2bfloat16_rn(acc[t] + b));
  }
}

// Sum of the K chunks' partial sums in chunk order, plus the bias, to bf16.
__global__ void dense_gemv_reduce_kernel(PackedHeader h, const uint8_t* __restrict__ packed, int T, int chunks,
                                         const float* __restrict__ partial, uint16_t* __restrict__ out) {
  const int N = h.H;
  const float* bias = reinterpret_cast<const float*>(packed + h.off_d_bias);
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < T * N; i += gridDim.x * blockDim.x) {
    const int n = i % N;
    float a = 0.f;
    for (int c = 0; c < chunks; ++c) a += partial[(int64_t)c * T * N + i];
    out[i] = __bfloat16_as_ushort(__float2bfloat16_rn(a + bias[n]));
  }
}

}  // namespace

cudaError_t launch_dense_quantize_weights(int N, int K, const uint16_t* w, uint8_t* blocks, uint8_t* scales,
                                          cudaStream_t s) {
  dense_quantize_weights_kernel<<<2048, 256, 0, s>>>(N, K, w, blocks, scales);
  return cudaGetLastError();
}

cudaError_t launch_dense_pack(const PackedHeader& h, const uint8_t* blocks, const uint8_t* scales, const uint16_t* bias,
                              uint8_t* packed, cudaStream_t s) {
  DensePackArgs a{h, blocks, scales, bias, packed};
  dense_pack_data_kernel<<<2048, 256, 0, s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  dense_pack_sf_kernel<<<512, 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_dense_gemv(const PackedHeader& h, const uint8_t* packed, const uint16_t* x, int T, int k_chunks,
                              float* partial, uint16_t* out, cudaStream_t s) {
  if (T < 1 || T > kGemvMaxT) return cudaErrorInvalidValue;
  const int kt_per = (h.d_ktiles + k_chunks - 1) / k_chunks;
  const int chunks = (h.d_ktiles + kt_per - 1) / kt_per;
  const size_t smem = (size_t)T * kt_per * kTileK * sizeof(float);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(dense_gemv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  dense_gemv_kernel<<<dim3(h.d_mtiles, chunks), kGemvThreads, smem, s>>>(h, packed, x, T, kt_per,
                                                                         chunks > 1 ? partial : nullptr, out);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || chunks == 1) return e;
  dense_gemv_reduce_kernel<<<std::min(2048, (T * h.H + 255) / 256), 256, 0, s>>>(h, packed, T, chunks, partial, out);
  return cudaGetLastError();
}

}  // namespace moe

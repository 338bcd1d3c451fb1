// Router GEMV + bias (fp32 logits), top-k + softmax, and MXFP8 quantisation of
// the hidden states.
//
// The router weight is kept in BF16 ("GPT-OSS-120B on DGX Spark: From MXFP4 to
// NVFP4", section "GPT-OSS-120B Architecture": router weights are among the
// non-quantised BF16 tensors; 128 experts with 4 active per token).
#include "common.cuh"
#include "ptx.cuh"
#include "quant.cuh"

namespace moe {
namespace {

constexpr int kRouterTokens = 8;    // tokens per CTA
constexpr int kRouterExperts = 16;  // experts per CTA (2 per warp)

__device__ __forceinline__ void bf16x8_to_f32(const uint4 v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// logits[t][e] = sum_h x[t][h] * wr[e][h] + br[e]   (fp32 accumulation)
__global__ void __launch_bounds__(256) router_logits_kernel(const uint16_t* __restrict__ x,
                                                            const uint16_t* __restrict__ wr,
                                                            const uint16_t* __restrict__ br, int T,
                                                            int H, int E, float* __restrict__ logits) {
  extern __shared__ float4 xs4[];  // [kRouterTokens][H] fp32
  float* xs = reinterpret_cast<float*>(xs4);
  const int t0 = blockIdx.x * kRouterTokens;
  const int e0 = blockIdx.y * kRouterExperts;
  const int nt = min(kRouterTokens, T - t0);
  const int hc = H / 8;  // 8-element chunks per row
  for (int i = threadIdx.x; i < kRouterTokens * hc; i += blockDim.x) {
    const int t = i / hc, c = i % hc;
    float f[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    if (t < nt) bf16x8_to_f32(reinterpret_cast<const uint4*>(x + (int64_t)(t0 + t) * H)[c], f);
    float4* d = reinterpret_cast<float4*>(xs + t * H + c * 8);
    d[0] = make_float4(f[0], f[1], f[2], f[3]);
    d[1] = make_float4(f[4], f[5], f[6], f[7]);
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ea = e0 + 2 * warp, eb = ea + 1;
  if (ea >= E) return;
  const bool has_b = eb < E;
  float acc_a[kRouterTokens], acc_b[kRouterTokens];
#pragma unroll
  for (int t = 0; t < kRouterTokens; ++t) acc_a[t] = acc_b[t] = 0.f;
  const uint4* wa = reinterpret_cast<const uint4*>(wr + (int64_t)ea * H);
  const uint4* wb = reinterpret_cast<const uint4*>(wr + (int64_t)(has_b ? eb : ea) * H);
  for (int c = lane; c < hc; c += 32) {
    float fa[8], fb[8];
    bf16x8_to_f32(__ldg(wa + c), fa);
    bf16x8_to_f32(__ldg(wb + c), fb);
#pragma unroll
    for (int t = 0; t < kRouterTokens; ++t) {
      const float4* xr = reinterpret_cast<const float4*>(xs + t * H + c * 8);
      const float4 x0 = xr[0], x1 = xr[1];
      const float xv[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        acc_a[t] = fmaf(xv[i], fa[i], acc_a[t]);
        acc_b[t] = fmaf(xv[i], fb[i], acc_b[t]);
      }
    }
  }
#pragma unroll
  for (int t = 0; t < kRouterTokens; ++t) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      acc_a[t] += __shfl_xor_sync(0xffffffffu, acc_a[t], o);
      acc_b[t] += __shfl_xor_sync(0xffffffffu, acc_b[t], o);
    }
  }
  if (lane < nt) {
    // lane t writes token t (registers indexed by a compile-time loop)
#pragma unroll
    for (int t = 0; t < kRouterTokens; ++t) {
      if (t == lane) {
        logits[(int64_t)(t0 + t) * E + ea] = acc_a[t] + __uint_as_float((uint32_t)br[ea] << 16);
        if (has_b) logits[(int64_t)(t0 + t) * E + eb] = acc_b[t] + __uint_as_float((uint32_t)br[eb] << 16);
      }
    }
  }
}

// One warp per token: top-k of the logits (value desc, index asc), softmax over
// the k selected, then MXFP8 quantisation of the token's hidden row.
__global__ void __launch_bounds__(256) topk_quant_kernel(const float* __restrict__ logits,
                                                         const uint16_t* __restrict__ x, int T, int H,
                                                         int E, int k, int32_t* __restrict__ ids,
                                                         float* __restrict__ w, uint8_t* __restrict__ xq,
                                                         uint8_t* __restrict__ xsc) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + warp;
  if (t >= T) return;
  float v[8];
  uint32_t taken = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = lane + 32 * i;
    const float l = e < E ? logits[(int64_t)t * E + e] : -INFINITY;
    v[i] = isnan(l) ? -INFINITY : l;  // a NaN logit ranks last; every slot still gets a valid expert
  }
  float sel_v[8];
  int sel_i[8];
  for (int j = 0; j < k; ++j) {
    float bv = -INFINITY;
    int bi = 0x7FFFFFFF;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane + 32 * i;
      if (e < E && !(taken >> i & 1u) && (v[i] > bv || (v[i] == bv && e < bi))) {
        bv = v[i];
        bi = e;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (ov > bv || (ov == bv && oi < bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    sel_v[j] = bv;
    sel_i[j] = bi;
  }
  if (lane == 0) {
    float den = 0.f;
    for (int j = 0; j < k; ++j) den += expf(sel_v[j] - sel_v[0]);
    for (int j = 0; j < k; ++j) {
      ids[(int64_t)t * k + j] = sel_i[j];
      w[(int64_t)t * k + j] = expf(sel_v[j] - sel_v[0]) / den;
    }
  }
  // MXFP8: lane handles whole 32-element blocks.
  const int nb = H / 32;
  for (int b = lane; b < nb; b += 32) {
    const uint4* src = reinterpret_cast<const uint4*>(x + (int64_t)t * H + b * 32);
    float f[32];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      float g[8];
      const uint4 u = src[c];
      const uint32_t ww[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        g[2 * i] = __uint_as_float(ww[i] << 16);
        g[2 * i + 1] = __uint_as_float(ww[i] & 0xFFFF0000u);
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) f[8 * c + i] = g[i];
    }
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(f[i]));
    const int s = mx_scale_exp(amax);
    const float inv = mx_pow2_neg(s);
    uint32_t packed[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t lo = cvt_e4m3x2(f[4 * i] * inv, f[4 * i + 1] * inv);
      const uint32_t hi = cvt_e4m3x2(f[4 * i + 2] * inv, f[4 * i + 3] * inv);
      packed[i] = lo | (hi << 16);
    }
    uint4* dst = reinterpret_cast<uint4*>(xq + (int64_t)t * H + b * 32);
    dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
    dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
    xsc[(int64_t)t * nb + b] = (uint8_t)(s + 127);
  }
}

}  // namespace

cudaError_t launch_router(const uint16_t* x, const uint16_t* wr, const uint16_t* br, int T, int H,
                          int E, float* logits, cudaStream_t s) {
  const size_t smem = (size_t)kRouterTokens * H * sizeof(float);
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(router_logits_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         227 * 1024);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  dim3 grid((T + kRouterTokens - 1) / kRouterTokens, (E + kRouterExperts - 1) / kRouterExperts);
  router_logits_kernel<<<grid, 256, smem, s>>>(x, wr, br, T, H, E, logits);
  return cudaGetLastError();
}

cudaError_t launch_topk_quant(const float* logits, const uint16_t* x, int T, int H, int E, int k,
                              int32_t* ids, float* w, uint8_t* xq, uint8_t* xs, cudaStream_t s) {
  topk_quant_kernel<<<(T + 7) / 8, 256, 0, s>>>(logits, x, T, H, E, k, ids, w, xq, xs);
  return cudaGetLastError();
}

}  // namespace moe

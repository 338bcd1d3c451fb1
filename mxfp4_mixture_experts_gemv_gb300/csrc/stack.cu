// Residual stream of a stack of MoE layers, x <- x + moe(rmsnorm(x)): one kernel
// adds the previous layer's bf16 output to the fp32 residual and writes the
// RMSNorm (unit gain) of the result as the next layer's bf16 input.
#include <cuda_bf16.h>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads) residual_rmsnorm_kernel(float* __restrict__ x_res,
                                                                    const uint16_t* __restrict__ layer_out, int H,
                                                                    float eps, uint16_t* __restrict__ hidden) {
  const int t = blockIdx.x;
  float4* xr = reinterpret_cast<float4*>(x_res + (int64_t)t * H);
  const uint2* lo = layer_out ? reinterpret_cast<const uint2*>(layer_out + (int64_t)t * H) : nullptr;
  const int h4 = H / 4;
  float ss = 0.f;
  for (int c = threadIdx.x; c < h4; c += kThreads) {
    float4 v = xr[c];
    if (lo) {
      const uint2 o = lo[c];
      v.x += __uint_as_float(o.x << 16);
      v.y += __uint_as_float(o.x & 0xFFFF0000u);
      v.z += __uint_as_float(o.y << 16);
      v.w += __uint_as_float(o.y & 0xFFFF0000u);
      xr[c] = v;
    }
    ss = fmaf(v.x, v.x, fmaf(v.y, v.y, fmaf(v.z, v.z, fmaf(v.w, v.w, ss))));
  }
  __shared__ float red[kThreads / 32];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int i = 0; i < kThreads / 32; ++i) tot += red[i];
  const float inv = 1.0f / sqrtf(tot / (float)H + eps);
  uint2* hd = reinterpret_cast<uint2*>(hidden + (int64_t)t * H);
  for (int c = threadIdx.x; c < h4; c += kThreads) {
    const float4 v = xr[c];
    const __nv_bfloat162 a = __floats2bfloat162_rn(v.x * inv, v.y * inv);
    const __nv_bfloat162 b = __floats2bfloat162_rn(v.z * inv, v.w * inv);
    hd[c] = make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b));
  }
}

}  // namespace

cudaError_t launch_residual_rmsnorm(float* x_res, const uint16_t* layer_out, int T, int H, float eps,
                                    uint16_t* hidden, cudaStream_t s) {
  residual_rmsnorm_kernel<<<T, kThreads, 0, s>>>(x_res, layer_out, H, eps, hidden);
  return cudaGetLastError();
}

}  // namespace moe

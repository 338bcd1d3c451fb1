// Routing-weighted combine: out[t] = bf16( sum_j w[t][j] * y[pos(t, j)] ), the k
// slots summed in slot order in fp32, one rounding to bf16 at the end.
#include <cuda_bf16.h>

#include "common.cuh"

namespace moe {
namespace {

__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ y, const float* __restrict__ w,
                                                      const int32_t* __restrict__ inv_pos, int k, int H,
                                                      uint16_t* __restrict__ out) {
  const int t = blockIdx.x;
  float wt[8];
  int64_t pos[8];
  for (int j = 0; j < k; ++j) {
    wt[j] = w[(int64_t)t * k + j];
    pos[j] = inv_pos[(int64_t)t * k + j];
  }
  const int h4 = H / 4;
  for (int c = blockIdx.y * blockDim.x + threadIdx.x; c < h4; c += gridDim.y * blockDim.x) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < k; ++j) {
      const float4 v = reinterpret_cast<const float4*>(y + pos[j] * H)[c];
      acc.x = fmaf(wt[j], v.x, acc.x);
      acc.y = fmaf(wt[j], v.y, acc.y);
      acc.z = fmaf(wt[j], v.z, acc.z);
      acc.w = fmaf(wt[j], v.w, acc.w);
    }
    const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
    const __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
    uint2 o;
    o.x = *reinterpret_cast<const uint32_t*>(&lo);
    o.y = *reinterpret_cast<const uint32_t*>(&hi);
    reinterpret_cast<uint2*>(out + (int64_t)t * H)[c] = o;
  }
}

}  // namespace

cudaError_t launch_combine(const float* y, const float* w, const int32_t* inv_pos, int T, int k, int H,
                           uint16_t* out, cudaStream_t s) {
  const int h4 = H / 4;
  dim3 grid(T, (h4 + 255) / 256);
  combine_kernel<<<grid, 256, 0, s>>>(y, w, inv_pos, k, H, out);
  return cudaGetLastError();
}

}  // namespace moe

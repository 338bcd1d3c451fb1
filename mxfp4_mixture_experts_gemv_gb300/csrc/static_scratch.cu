// moe_forward_static_scratch: the layer forward without any device allocation,
// for callers that cannot allocate device memory themselves.  Its scratch lives
// in a fixed-size array in this library's own device image instead of a
// caller-provided workspace; everything else is moe_forward.
#include <mutex>

#include "common.cuh"

namespace {

// The scratch array (MOE_STATIC_SCRATCH_BYTES).  Every GPU that loads this
// library holds it until the process exits.  In host code the name is only a
// host-side stand-in for the symbol: its device address comes from
// cudaGetSymbolAddress, taken once per device with that device current.
static __device__ __align__(256) uint8_t g_static_scratch[MOE_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

moe_status scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return moe::report_error(MOE_ERR_CUDA, "cudaGetDevice failed: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return moe::report_error(MOE_ERR_INVALID_ARG, "device %d beyond %d", dev, kMaxDevices);
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess || !p)
      return moe::report_error(MOE_ERR_CUDA, "cudaGetSymbolAddress of the static scratch failed: %s",
                               cudaGetErrorString(e));
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return MOE_OK;
}

}  // namespace

extern "C" moe_status moe_forward_static_scratch(moe_dims d, const void* hidden, int32_t T, const void* router_w,
                                                 const void* router_b, const void* packed, int32_t top_k, void* out,
                                                 void* stream) {
  if (T <= 0 || top_k < 1) {
    // nothing to run (T = 0) or an argument error: moe_forward reports either
    return moe_forward(d, hidden, T, router_w, router_b, packed, top_k, out, nullptr, 0, stream);
  }
  const size_t need = moe_workspace_size(d, T, top_k);
  if (need > (size_t)MOE_STATIC_SCRATCH_BYTES)
    return moe::report_error(MOE_ERR_WORKSPACE_TOO_SMALL,
                             "this forward needs %zu bytes of scratch but the static scratch holds %zu "
                             "(MOE_STATIC_SCRATCH_BYTES); use fewer tokens per call or moe_forward",
                             need, (size_t)MOE_STATIC_SCRATCH_BYTES);
  void* ptr = nullptr;
  moe_status st = scratch_address(&ptr);
  if (st != MOE_OK) return st;
  return moe_forward(d, hidden, T, router_w, router_b, packed, top_k, out, ptr, (size_t)MOE_STATIC_SCRATCH_BYTES,
                     stream);
}

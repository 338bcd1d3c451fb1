// moe_forward_static_scratch: the layer forward without any device allocation,
// for callers that cannot allocate device memory themselves.  Its scratch lives
// in a fixed-size array in this library's own device image instead of a
// caller-provided workspace; everything else is moe_forward.
#include "common.cuh"

namespace {

// The scratch array (MOE_STATIC_SCRATCH_BYTES).  Every GPU that loads this
// library holds it until the process exits.  In host code the name is only a
// host-side stand-in for the symbol: its device address comes from
// cudaGetSymbolAddress, with the device that runs the call current.
static __device__ __align__(256) uint8_t g_static_scratch[MOE_STATIC_SCRATCH_BYTES];

// Device address of the array on the current device.  Looked up on every call:
// after the first (which loads the library's device code on that device) it is a
// host-side table lookup, and it stays right if the context is torn down and
// created again.
moe_status scratch_address(void** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
  if (e != cudaSuccess || !p)
    return moe::report_error(MOE_ERR_CUDA, "cudaGetSymbolAddress of the static scratch failed: %s",
                             cudaGetErrorString(e));
  *out = p;
  return MOE_OK;
}

}  // namespace

extern "C" {

size_t moe_static_scratch_bytes(void) { return (size_t)MOE_STATIC_SCRATCH_BYTES; }

moe_status moe_forward_static_scratch(moe_dims d, const void* hidden, int32_t T, const void* router_w,
                                      const void* router_b, const void* packed, int32_t top_k, void* out,
                                      void* stream) {
  // moe_forward's own argument checks first, so that errors read the same
  moe_status st = moe::check_forward_args(d, hidden, T, router_w, router_b, packed, top_k, out);
  if (st != MOE_OK || T == 0) return st;
  const size_t need = moe_workspace_size(d, T, top_k);
  if (need > (size_t)MOE_STATIC_SCRATCH_BYTES)
    return moe::report_error(MOE_ERR_WORKSPACE_TOO_SMALL,
                             "this forward needs %zu bytes of scratch but the static scratch holds %zu "
                             "(MOE_STATIC_SCRATCH_BYTES); use fewer tokens per call or moe_forward",
                             need, (size_t)MOE_STATIC_SCRATCH_BYTES);
  void* ptr = nullptr;
  st = scratch_address(&ptr);
  if (st != MOE_OK) return st;
  return moe_forward(d, hidden, T, router_w, router_b, packed, top_k, out, ptr, (size_t)MOE_STATIC_SCRATCH_BYTES,
                     stream);
}

moe_status moe_static_scratch_status(void* stream) {
  void* ptr = nullptr;
  const moe_status st = scratch_address(&ptr);
  if (st != MOE_OK) return st;
  // the status words sit at the start of a forward's scratch
  return moe::read_status_words(ptr, stream);
}

}  // extern "C"

// C ABI of the MXFP4 MoE layer: argument validation, workspace carving and the
// launch sequence  router -> top-k/quant -> grouping -> gather -> gate_up GEMM
// -> down GEMM -> combine, all on the caller's stream.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "common.cuh"

namespace {

thread_local std::string g_last_error;

moe_status fail(moe_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

moe_status cuda_fail(cudaError_t e, const char* what) {
  return fail(MOE_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

moe_status check_dims(const moe_dims& d) {
  if (d.E <= 0 || d.H <= 0 || d.I <= 0) return fail(MOE_ERR_INVALID_ARG, "dims must be positive (E=%d H=%d I=%d)", d.E, d.H, d.I);
  if (d.E > 256) return fail(MOE_ERR_UNSUPPORTED_SHAPE, "E=%d > 256 experts", d.E);
  if (d.H % 32) return fail(MOE_ERR_UNSUPPORTED_SHAPE, "H=%d is not a multiple of 32", d.H);
  if (d.I % 64) return fail(MOE_ERR_UNSUPPORTED_SHAPE, "I=%d is not a multiple of 64", d.I);
  if (d.H > moe::kRouteSmallMaxH) return fail(MOE_ERR_UNSUPPORTED_SHAPE, "H=%d > %d", d.H, moe::kRouteSmallMaxH);
  return MOE_OK;
}

constexpr int kStages = 2;  // routing (all routing kernels), expert MLP

std::atomic<uint64_t> g_wait_limit_ns{moe::kWaitLimitNsDefault};
std::atomic<int> g_hold_waits{0};
std::atomic<int> g_plan_tile_rows{0};
std::atomic<int> g_plan_route{0};
std::atomic<int> g_plan_expert{0};

// Per-stage CUDA events of profiled forward calls.
struct Profiler {
  bool armed = false;
  std::vector<cudaEvent_t> ev;  // (kStages + 1) events per call
  int capacity = 0, used = 0;
};
Profiler g_prof;

cudaEvent_t* profile_slot() {
  if (!g_prof.armed || g_prof.used >= g_prof.capacity) return nullptr;
  return &g_prof.ev[(size_t)(g_prof.used++) * (kStages + 1)];
}

int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 1;
  return n;
}

}  // namespace

namespace moe {
moe_status report_error(moe_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

uint64_t wait_limit_ns() { return g_wait_limit_ns.load(std::memory_order_relaxed); }
int debug_hold_waits() { return g_hold_waits.load(std::memory_order_relaxed); }
int plan_tile_rows() { return g_plan_tile_rows.load(std::memory_order_relaxed); }
int plan_route() { return g_plan_route.load(std::memory_order_relaxed); }
int plan_expert() { return g_plan_expert.load(std::memory_order_relaxed); }

moe_status check_forward_args(const moe_dims& d, const void* hidden, int32_t T, const void* router_w,
                              const void* router_b, const void* packed, int32_t top_k, const void* out) {
  moe_status st = check_dims(d);
  if (st != MOE_OK) return st;
  if (T < 0) return fail(MOE_ERR_INVALID_ARG, "T=%d < 0", T);
  if (top_k < 1 || top_k > 8 || top_k > d.E) return fail(MOE_ERR_INVALID_ARG, "top_k=%d outside [1, min(E, 8)]", top_k);
  if (T == 0) return MOE_OK;
  if ((int64_t)T * top_k * (int64_t)(d.H > d.I ? d.H : d.I) >= (int64_t)1 << 31)
    return fail(MOE_ERR_UNSUPPORTED_SHAPE, "T*top_k*max(H,I) must stay below 2^31");
  if (!hidden || !router_w || !router_b || !packed || !out) return fail(MOE_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned(hidden, 16) || !aligned(router_w, 16) || !aligned(out, 16))
    return fail(MOE_ERR_ALIGNMENT, "hidden, router_w and out must be 16-byte aligned");
  if (!aligned(packed, 256)) return fail(MOE_ERR_ALIGNMENT, "packed must be 256-byte aligned");
  return MOE_OK;
}

moe_status read_status_words(const void* status_words, void* stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
  uint32_t st[4] = {0, 0, 0, 0};
  e = cudaMemcpy(st, status_words, sizeof(st), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "status read");
  if (st[0] != 0)
    return fail(MOE_ERR_TIMEOUT, "device wait expired (status bits 0x%x, first expired wait 0x%08x)", st[0], st[1]);
  return MOE_OK;
}
}  // namespace moe

extern "C" {

uint32_t moe_version(void) { return (1u << 16) | moe::kPackedVersion; }

const char* moe_last_error(void) { return g_last_error.c_str(); }

size_t moe_packed_size(moe_dims d) {
  moe::PackedHeader h;
  if (check_dims(d) != MOE_OK || !moe::packed_layout(d, &h)) return 0;
  return (size_t)h.total;
}

moe_status moe_pack_weights(moe_dims d, const moe_mxfp4_weights* src, void* packed, size_t packed_bytes,
                            void* stream) {
  moe_status st = check_dims(d);
  if (st != MOE_OK) return st;
  if (!src || !packed) return fail(MOE_ERR_INVALID_ARG, "null src or packed pointer");
  if (!src->gate_up_blocks || !src->gate_up_scales || !src->gate_up_bias || !src->down_blocks ||
      !src->down_scales || !src->down_bias)
    return fail(MOE_ERR_INVALID_ARG, "null weight tensor pointer");
  if (!aligned(packed, 256)) return fail(MOE_ERR_ALIGNMENT, "packed buffer must be 256-byte aligned");
  if (!aligned(src->gate_up_blocks, 16) || !aligned(src->down_blocks, 16))
    return fail(MOE_ERR_ALIGNMENT, "*_blocks tensors must be 16-byte aligned");
  moe::PackedHeader h;
  moe::packed_layout(d, &h);
  if (packed_bytes < h.total)
    return fail(MOE_ERR_BAD_PACKED_HEADER, "packed buffer has %zu bytes, %llu needed", packed_bytes,
                (unsigned long long)h.total);
  cudaError_t e = moe::launch_pack(d, h, *src, static_cast<uint8_t*>(packed), static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "pack kernels");
  return MOE_OK;
}

size_t moe_packed_size_nvfp4(moe_dims d) {
  moe::PackedHeader h;
  if (check_dims(d) != MOE_OK || !moe::packed_layout(d, &h, moe::kWeightsNvfp4)) return 0;
  return (size_t)h.total;
}

moe_status moe_pack_weights_nvfp4(moe_dims d, const moe_mxfp4_weights* src, void* packed, size_t packed_bytes,
                                  void* stream) {
  moe_status st = check_dims(d);
  if (st != MOE_OK) return st;
  if (d.H % 64 || d.I % 64)
    return fail(MOE_ERR_UNSUPPORTED_SHAPE, "NVFP4 packing needs H and I multiples of 64 (H=%d I=%d)", d.H, d.I);
  if (!src || !packed) return fail(MOE_ERR_INVALID_ARG, "null src or packed pointer");
  if (!src->gate_up_blocks || !src->gate_up_scales || !src->gate_up_bias || !src->down_blocks ||
      !src->down_scales || !src->down_bias)
    return fail(MOE_ERR_INVALID_ARG, "null weight tensor pointer");
  if (!aligned(packed, 256)) return fail(MOE_ERR_ALIGNMENT, "packed buffer must be 256-byte aligned");
  if (!aligned(src->gate_up_blocks, 16) || !aligned(src->down_blocks, 16))
    return fail(MOE_ERR_ALIGNMENT, "*_blocks tensors must be 16-byte aligned");
  moe::PackedHeader h;
  moe::packed_layout(d, &h, moe::kWeightsNvfp4);
  if (packed_bytes < h.total)
    return fail(MOE_ERR_BAD_PACKED_HEADER, "packed buffer has %zu bytes, %llu needed", packed_bytes,
                (unsigned long long)h.total);
  cudaError_t e = moe::launch_pack_nvfp4(h, *src, static_cast<uint8_t*>(packed), static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "NVFP4 pack kernels");
  return MOE_OK;
}

size_t moe_workspace_size(moe_dims d, int32_t T, int32_t top_k) {
  moe_workspace_layout l;
  if (check_dims(d) != MOE_OK || T < 0 || top_k <= 0 || !moe::workspace_layout(d, T, top_k, &l)) return 0;
  return l.total;
}

moe_status moe_workspace_layout_get(moe_dims d, int32_t T, int32_t top_k, moe_workspace_layout* out) {
  return moe_workspace_layout_act(d, T, top_k, MOE_ACT_MXFP8, out);
}

moe_status moe_workspace_layout_act(moe_dims d, int32_t T, int32_t top_k, int32_t act_format,
                                    moe_workspace_layout* out) {
  moe_status st = check_dims(d);
  if (st != MOE_OK) return st;
  if (!out || T < 0 || top_k <= 0 || top_k > 8 || top_k > d.E)
    return fail(MOE_ERR_INVALID_ARG, "bad layout query (T=%d top_k=%d)", T, top_k);
  if (act_format != MOE_ACT_MXFP8 && act_format != MOE_ACT_MXFP4 && act_format != MOE_ACT_NVFP4)
    return fail(MOE_ERR_INVALID_ARG, "unknown activation format %d", act_format);
  moe::workspace_layout(d, T, top_k, out, act_format);
  return MOE_OK;
}

}  // extern "C"

namespace {

// The forward for every activation format (moe::ActFormat).
moe_status forward_impl(moe_dims d, int fmt, const void* hidden, int32_t T, const void* router_w,
                        const void* router_b, const void* packed, int32_t top_k, void* out, void* workspace,
                        size_t workspace_bytes, void* stream) {
  moe_status st = moe::check_forward_args(d, hidden, T, router_w, router_b, packed, top_k, out);
  if (st != MOE_OK || T == 0) return st;
  if (!workspace) return fail(MOE_ERR_INVALID_ARG, "null workspace");
  if (!aligned(workspace, 256)) return fail(MOE_ERR_ALIGNMENT, "workspace must be 256-byte aligned");
  moe_workspace_layout L;
  moe::workspace_layout(d, T, top_k, &L, fmt);
  if (workspace_bytes < L.total)
    return fail(MOE_ERR_WORKSPACE_TOO_SMALL, "workspace has %zu bytes, %zu needed", workspace_bytes, L.total);
  const bool fp4 = fmt == moe::kActMxfp4;  // the routing kernels' MXFP4 quantisation
  moe::PackedHeader h;
  moe::packed_layout(d, &h, fmt == moe::kActNvfp4 ? moe::kWeightsNvfp4 : moe::kWeightsMxfp4);

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const uint8_t* pk = static_cast<const uint8_t*>(packed);
  auto at = [&](size_t off) { return ws + off; };
  const int TK = T * top_k;
  uint32_t* status = reinterpret_cast<uint32_t*>(at(L.status));
  int32_t* ids = reinterpret_cast<int32_t*>(at(L.topk_ids));
  float* w = reinterpret_cast<float*>(at(L.topk_w));
  int32_t* tiles = reinterpret_cast<int32_t*>(at(L.tiles));
  int32_t* inv_pos = reinterpret_cast<int32_t*>(at(L.inv_pos));
  int32_t* sorted_rows = reinterpret_cast<int32_t*>(at(L.sorted_rows));
  const int sms = num_sms();

  // routing path: a few tokens in one cluster, batched decode in one cooperative
  // grid, else the tensor-core router with separate grouping and gather passes
  const int forced = moe::plan_route();
  const bool cluster_fits = moe::route_cluster_fits(T, d.E, d.H), grid_fits = moe::route_small_fits(T, d.H);
  // NVFP4 activations are quantised by the cluster kernel and by the gather pass of the
  // tensor-core path (not by the grid routing kernel)
  const bool nv = fmt == moe::kActNvfp4;
  const int route = forced != moe::kRouteAuto
                        ? forced
                        : (cluster_fits ? moe::kRouteCluster
                                        : (grid_fits && !nv ? moe::kRouteGrid : moe::kRouteTensorCore));
  if (nv && route == moe::kRouteGrid)
    return fail(MOE_ERR_UNSUPPORTED_SHAPE, "NVFP4 activations take the cluster or tensor-core routing path");
  if ((route == moe::kRouteCluster && !cluster_fits) || (route == moe::kRouteGrid && !grid_fits))
    return fail(MOE_ERR_UNSUPPORTED_SHAPE, "the forced routing path %d does not fit T=%d", route, T);
  // The cluster routing kernel clears the status words and counters itself; the
  // other paths start from a memset.
  const bool cluster_route = route == moe::kRouteCluster;
  cudaError_t e = cudaSuccess;
  if (!cluster_route) {
    e = cudaMemsetAsync(ws, 0, L.zero_bytes, s);
    if (e != cudaSuccess) return cuda_fail(e, "status reset");
  }
  cudaEvent_t* pev = profile_slot();
  auto mark = [&](int i) {
    // external record: inside a stream capture this becomes a timestamping graph node
    if (pev) cudaEventRecordWithFlags(pev[i], s, cudaEventRecordExternal);
  };
  mark(0);
  int route_ctas = 0;  // routing CTAs that publish through the flags (cluster path)
  if (cluster_route) {
    // a few tokens: routing, grouping and quantise-on-gather in one cluster
    moe::RouteClusterOut o;
    o.logits = reinterpret_cast<float*>(at(L.logits));
    o.ids = ids;
    o.w = w;
    o.xq = at(L.xq);
    o.xs = at(L.xs);
    o.counts = reinterpret_cast<int32_t*>(at(L.counts));
    o.offsets = reinterpret_cast<int32_t*>(at(L.offsets));
    o.sorted_rows = sorted_rows;
    o.inv_pos = inv_pos;
    o.tiles = tiles;
    o.xp = at(L.xp);
    o.xp_sf = at(L.xp_sf);
    o.zero = reinterpret_cast<uint32_t*>(ws);
    o.zero_words = (int)(L.zero_bytes / 4);
    o.status = status;
    o.flags = reinterpret_cast<int32_t*>(at(L.grid_bar)) + 2;
    e = moe::launch_route_cluster(static_cast<const uint16_t*>(hidden), static_cast<const uint16_t*>(router_w),
                                  static_cast<const uint16_t*>(router_b), T, d.H, d.E, top_k, L.tile_rows, fmt, o,
                                  &route_ctas, s);
    if (e != cudaSuccess) return cuda_fail(e, "cluster routing kernel");
  } else if (route == moe::kRouteGrid) {
    // decode: routing, quantisation, grouping and gather in one launch
    moe::RouteSmallOut o;
    o.logits = reinterpret_cast<float*>(at(L.logits));
    o.ids = ids;
    o.w = w;
    o.xq = at(L.xq);
    o.xs = at(L.xs);
    o.counts = reinterpret_cast<int32_t*>(at(L.counts));
    o.offsets = reinterpret_cast<int32_t*>(at(L.offsets));
    o.sorted_rows = sorted_rows;
    o.inv_pos = inv_pos;
    o.tiles = tiles;
    o.xp = at(L.xp);
    o.xp_sf = at(L.xp_sf);
    o.hq_sf = at(L.hq_sf);
    o.grid_bar = reinterpret_cast<int32_t*>(at(L.grid_bar));
    o.status = status;
    e = moe::launch_route_small(static_cast<const uint16_t*>(hidden), static_cast<const uint16_t*>(router_w),
                                static_cast<const uint16_t*>(router_b), T, d.H, d.E, d.I, top_k, L.tile_rows,
                                L.max_tiles, fp4, o, s);
    if (e != cudaSuccess) return cuda_fail(e, "small-batch routing kernel");
  } else {
    // larger T: tensor-core router with top-k in its epilogue, grouping, quantise-on-gather
    e = moe::launch_router_tc(static_cast<const uint16_t*>(hidden), static_cast<const uint16_t*>(router_w),
                              static_cast<const uint16_t*>(router_b), T, d.H, d.E, top_k,
                              reinterpret_cast<float*>(at(L.logits)), ids, w, status, s);
    if (e != cudaSuccess) return cuda_fail(e, "router kernel");
    // the grouping's per-chunk counts live at the start of y, which is written only later
    e = moe::launch_permute(ids, TK, top_k, d.E, L.tile_rows, L.max_tiles, reinterpret_cast<int32_t*>(at(L.counts)),
                            reinterpret_cast<int32_t*>(at(L.offsets)), sorted_rows, inv_pos, tiles,
                            reinterpret_cast<int32_t*>(at(L.y)), s);
    if (e != cudaSuccess) return cuda_fail(e, "grouping kernel");
    e = moe::launch_gather_quant(static_cast<const uint16_t*>(hidden), inv_pos, tiles, L.max_tiles, T, top_k, d.H,
                                 fmt, at(L.xq), at(L.xs), at(L.xp), at(L.xp_sf), s);
    if (e != cudaSuccess) return cuda_fail(e, "gather kernel");
  }
  mark(1);
  moe::ExpertMlpBuffers b = {};
  b.xp = at(L.xp);
  b.xp_sf = at(L.xp_sf);
  b.hq = at(L.hq);
  b.hq_sf = at(L.hq_sf);
  b.y = reinterpret_cast<float*>(at(L.y));
  b.out = static_cast<uint16_t*>(out);
  b.tiles = tiles;
  b.sorted_rows = sorted_rows;
  b.inv_pos = inv_pos;
  b.topk_w = w;
  b.done_gu = reinterpret_cast<int32_t*>(at(L.done_gu));
  b.done_tok = reinterpret_cast<int32_t*>(at(L.done_tok));
  b.sched = reinterpret_cast<int32_t*>(at(L.grid_bar)) + 1;  // word 0 is the grid routing barrier
  b.status = status;
  // The expert kernel follows the cluster routing kernel through the flags (words 2
  // and 3 of the section): weight copies once the tile list is published, activation
  // copies once every routing CTA has written its grouped rows.  A debug hold asks it
  // to wait for one routing CTA more than there are.
  b.route_flags = reinterpret_cast<int32_t*>(at(L.grid_bar)) + 2;
  b.route_ctas = route_ctas == 0 ? 0 : route_ctas + ((moe::debug_hold_waits() & MOE_DEBUG_HOLD_ROUTING_BARRIER) ? 1 : 0);
  // A few tokens: the down epilogue combines (no extra launch on the decode path).
  // Many tokens: a streaming pass after the expert kernel, which would otherwise
  // stall on the slot loads of every completed token.
  b.fused_combine = L.tile_rows <= 32;
  // expert kernel: tokens-on-M for 128-row token tiles with MXFP8 activations
  // (measured on GB300, gpt-oss-shaped layer: 2048 tokens 395 against 449 us,
  // 4096 564 against 657, 8192 916 against 1078), weights-on-M otherwise or when
  // the plan asks for it
  const int forced_expert = moe::plan_expert();
  const bool swap_ok = L.tile_rows == 128 && !b.fused_combine && moe::expert_swap_supported(h);
  // (NVFP4 only when the plan asks: its tokens-on-M form measured slower, T = 2048
  // 466 against 410 us)
  const bool tokens_m =
      swap_ok && (forced_expert == moe::kExpertTokensM || (forced_expert == moe::kExpertAuto && fmt != moe::kActNvfp4));
  if (forced_expert == moe::kExpertTokensM && !tokens_m)
    return fail(MOE_ERR_UNSUPPORTED_SHAPE, "the tokens-on-M expert kernel needs 128-row tiles");
  if (tokens_m)
    e = moe::launch_expert_swap(h, pk, b, T, top_k, L.max_tiles, sms, fmt, s);
  else
    e = moe::launch_expert_mlp(h, pk, b, T, top_k, L.max_tiles, L.tile_rows, sms, fmt, s);
  if (e != cudaSuccess) return cuda_fail(e, "expert MLP kernel");
  if (!b.fused_combine) {
    e = moe::launch_combine(b.y, inv_pos, w, T, top_k, d.H, static_cast<uint16_t*>(out), s);
    if (e != cudaSuccess) return cuda_fail(e, "combine kernel");
  }
  mark(2);
  return MOE_OK;
}

}  // namespace

extern "C" {

moe_status moe_forward(moe_dims d, const void* hidden, int32_t T, const void* router_w, const void* router_b,
                       const void* packed, int32_t top_k, void* out, void* workspace, size_t workspace_bytes,
                       void* stream) {
  return forward_impl(d, moe::kActMxfp8, hidden, T, router_w, router_b, packed, top_k, out, workspace,
                      workspace_bytes, stream);
}

moe_status moe_forward_act(moe_dims d, int32_t act_format, const void* hidden, int32_t T, const void* router_w,
                           const void* router_b, const void* packed, int32_t top_k, void* out, void* workspace,
                           size_t workspace_bytes, void* stream) {
  if (act_format != MOE_ACT_MXFP8 && act_format != MOE_ACT_MXFP4 && act_format != MOE_ACT_NVFP4)
    return fail(MOE_ERR_INVALID_ARG, "unknown activation format %d", act_format);
  const int fmt = act_format == MOE_ACT_MXFP4 ? moe::kActMxfp4 : act_format == MOE_ACT_NVFP4 ? moe::kActNvfp4 : moe::kActMxfp8;
  return forward_impl(d, fmt, hidden, T, router_w, router_b, packed, top_k, out, workspace, workspace_bytes, stream);
}

// ---------------------------------------------------------------- dense MXFP4 linears
size_t moe_dense_packed_size(int32_t N, int32_t K) {
  moe::PackedHeader h;
  return moe::dense_layout(N, K, &h) ? (size_t)h.total : 0;
}

moe_status moe_dense_quantize_weights(int32_t N, int32_t K, const void* w, void* blocks, void* scales, void* stream) {
  if (N <= 0 || K <= 0 || K % 32) return fail(MOE_ERR_UNSUPPORTED_SHAPE, "N=%d K=%d (K a multiple of 32)", N, K);
  if (!w || !blocks || !scales) return fail(MOE_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned(w, 16) || !aligned(blocks, 16)) return fail(MOE_ERR_ALIGNMENT, "w and blocks must be 16-byte aligned");
  cudaError_t e = moe::launch_dense_quantize_weights(N, K, static_cast<const uint16_t*>(w), static_cast<uint8_t*>(blocks),
                                                     static_cast<uint8_t*>(scales), static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "dense weight quantiser");
  return MOE_OK;
}

moe_status moe_dense_pack(int32_t N, int32_t K, const void* blocks, const void* scales, const void* bias, void* packed,
                          size_t packed_bytes, void* stream) {
  moe::PackedHeader h;
  if (!moe::dense_layout(N, K, &h))
    return fail(MOE_ERR_UNSUPPORTED_SHAPE, "N=%d K=%d (N a multiple of 64, K of 32)", N, K);
  if (!blocks || !scales || !packed) return fail(MOE_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned(packed, 256)) return fail(MOE_ERR_ALIGNMENT, "packed buffer must be 256-byte aligned");
  if (!aligned(blocks, 16)) return fail(MOE_ERR_ALIGNMENT, "blocks must be 16-byte aligned");
  if (packed_bytes < h.total)
    return fail(MOE_ERR_BAD_PACKED_HEADER, "packed buffer has %zu bytes, %llu needed", packed_bytes,
                (unsigned long long)h.total);
  cudaError_t e = moe::launch_dense_pack(h, static_cast<const uint8_t*>(blocks), static_cast<const uint8_t*>(scales),
                                         static_cast<const uint16_t*>(bias), static_cast<uint8_t*>(packed),
                                         static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "dense pack kernels");
  return MOE_OK;
}

size_t moe_dense_workspace_size(int32_t N, int32_t K, int32_t T) {
  moe::DenseWorkspace w;
  moe::PackedHeader h;
  if (!moe::dense_layout(N, K, &h) || T < 0 || !moe::dense_workspace(N, K, T, num_sms(), &w)) return 0;
  return w.total;
}

moe_status moe_dense_forward(int32_t N, int32_t K, const void* x, int32_t T, const void* packed, void* out,
                             void* workspace, size_t workspace_bytes, void* stream) {
  moe::PackedHeader h;
  if (!moe::dense_layout(N, K, &h))
    return fail(MOE_ERR_UNSUPPORTED_SHAPE, "N=%d K=%d (N a multiple of 64, K of 32)", N, K);
  if (T < 0) return fail(MOE_ERR_INVALID_ARG, "T=%d < 0", T);
  if (T == 0) return MOE_OK;
  if ((int64_t)T * (N > K ? N : K) >= (int64_t)1 << 31) return fail(MOE_ERR_UNSUPPORTED_SHAPE, "T*max(N,K) >= 2^31");
  if (!x || !packed || !out || !workspace) return fail(MOE_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned(x, 16) || !aligned(out, 16)) return fail(MOE_ERR_ALIGNMENT, "x and out must be 16-byte aligned");
  if (!aligned(packed, 256) || !aligned(workspace, 256))
    return fail(MOE_ERR_ALIGNMENT, "packed and workspace must be 256-byte aligned");
  const int sms = num_sms();
  moe::DenseWorkspace L;
  moe::dense_workspace(N, K, T, sms, &L);
  if (workspace_bytes < L.total)
    return fail(MOE_ERR_WORKSPACE_TOO_SMALL, "workspace has %zu bytes, %zu needed", workspace_bytes, L.total);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const uint8_t* pk = static_cast<const uint8_t*>(packed);
  // a few tokens on the CUDA cores (the plan may force either path; the measured
  // default is in dense_cuda_cores_for)
  const int forced = moe::plan_expert();
  const bool cores = forced == moe::kExpertCudaCores || (forced == moe::kExpertAuto && moe::dense_cuda_cores_for(T, N, K));
  if (cores && T > 4) return fail(MOE_ERR_UNSUPPORTED_SHAPE, "the CUDA-core dense path takes at most 4 tokens");
  cudaError_t e;
  if (cores) {
    e = moe::launch_dense_gemv(h, pk, static_cast<const uint16_t*>(x), T, L.k_chunks,
                               reinterpret_cast<float*>(ws + L.partial), static_cast<uint16_t*>(out), s);
    if (e != cudaSuccess) return cuda_fail(e, "dense GEMV kernels");
    return MOE_OK;
  }
  int32_t* tiles = reinterpret_cast<int32_t*>(ws + L.tiles);
  int32_t* inv_pos = reinterpret_cast<int32_t*>(ws + L.inv_pos);
  // the quantiser also lays out the identity grouping and clears the counters
  e = moe::launch_gather_quant(static_cast<const uint16_t*>(x), inv_pos, tiles, L.max_tiles, T, 1, K, moe::kActMxfp8,
                               ws + L.xq, ws + L.xs, ws + L.xp, ws + L.xp_sf, s, L.tile_rows,
                               reinterpret_cast<uint32_t*>(ws), (int)(L.zero_bytes / 4));
  if (e != cudaSuccess) return cuda_fail(e, "dense quantiser");
  moe::ExpertMlpBuffers b = {};
  b.xp = ws + L.xp;
  b.xp_sf = ws + L.xp_sf;
  b.hq = ws + L.xp;      // the down units' activation operand: the quantised input
  b.hq_sf = ws + L.xp_sf;
  b.out = static_cast<uint16_t*>(out);
  b.tiles = tiles;
  b.inv_pos = inv_pos;
  b.done_gu = reinterpret_cast<int32_t*>(ws + L.done);
  b.done_tok = reinterpret_cast<int32_t*>(ws + L.done);
  b.sched = reinterpret_cast<int32_t*>(ws + L.sched);
  b.status = reinterpret_cast<uint32_t*>(ws + L.status);
  b.fused_combine = false;
  e = moe::launch_expert_mlp(h, pk, b, T, 1, L.max_tiles, L.tile_rows, sms, moe::kActMxfp8, s);
  if (e != cudaSuccess) return cuda_fail(e, "dense GEMM kernel");
  return MOE_OK;
}

moe_status moe_residual_rmsnorm(float* x_res, const void* layer_out, int32_t T, int32_t H, float eps, void* hidden,
                                void* stream) {
  if (T < 0 || H <= 0 || H % 4 || !(eps > 0.f)) return fail(MOE_ERR_INVALID_ARG, "bad residual/rmsnorm arguments");
  if (T == 0) return MOE_OK;
  if (!x_res || !hidden) return fail(MOE_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned(x_res, 16) || !aligned(hidden, 8) || (layer_out && !aligned(layer_out, 8)))
    return fail(MOE_ERR_ALIGNMENT, "x_res must be 16-byte and hidden/layer_out 8-byte aligned");
  cudaError_t e = moe::launch_residual_rmsnorm(x_res, static_cast<const uint16_t*>(layer_out), T, H, eps,
                                               static_cast<uint16_t*>(hidden), static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "residual/rmsnorm kernel");
  return MOE_OK;
}

moe_status moe_profile_begin(int32_t max_calls) {
  if (max_calls <= 0) return fail(MOE_ERR_INVALID_ARG, "max_calls=%d", max_calls);
  const size_t need = (size_t)max_calls * (kStages + 1);
  while (g_prof.ev.size() < need) {
    cudaEvent_t ev;
    cudaError_t e = cudaEventCreate(&ev);
    if (e != cudaSuccess) return cuda_fail(e, "event create");
    g_prof.ev.push_back(ev);
  }
  g_prof.capacity = max_calls;
  g_prof.used = 0;
  g_prof.armed = true;
  return MOE_OK;
}

moe_status moe_profile_end(double* stage_ms, int32_t* calls) {
  if (!stage_ms || !calls) return fail(MOE_ERR_INVALID_ARG, "null output");
  g_prof.armed = false;
  for (int i = 0; i < kStages; ++i) stage_ms[i] = 0.0;
  *calls = g_prof.used;
  for (int c = 0; c < g_prof.used; ++c) {
    cudaEvent_t* ev = &g_prof.ev[(size_t)c * (kStages + 1)];
    cudaError_t e = cudaEventSynchronize(ev[kStages]);
    if (e != cudaSuccess) return cuda_fail(e, "event synchronize");
    for (int i = 0; i < kStages; ++i) {
      float ms = 0.f;
      e = cudaEventElapsedTime(&ms, ev[i], ev[i + 1]);
      if (e != cudaSuccess) return cuda_fail(e, "event elapsed");
      stage_ms[i] += ms;
    }
  }
  g_prof.used = 0;
  return MOE_OK;
}

moe_status moe_get_device_status(const void* workspace, void* stream) {
  if (!workspace) return fail(MOE_ERR_INVALID_ARG, "null workspace");
  return moe::read_status_words(workspace, stream);
}

moe_status moe_set_wait_limit_ns(uint64_t ns) {
  if (ns == 0) ns = moe::kWaitLimitNsDefault;
  if (ns < 1000ull || ns > 60000000000ull)
    return fail(MOE_ERR_INVALID_ARG, "wait limit %llu ns outside [1 us, 60 s]", (unsigned long long)ns);
  g_wait_limit_ns.store(ns, std::memory_order_relaxed);
  return MOE_OK;
}

uint64_t moe_get_wait_limit_ns(void) { return g_wait_limit_ns.load(std::memory_order_relaxed); }

moe_status moe_set_plan(int32_t tile_rows, int32_t route, int32_t expert_kernel) {
  if (tile_rows != 0 && tile_rows != 8 && tile_rows != 16 && tile_rows != 32 && tile_rows != 64 && tile_rows != 128)
    return fail(MOE_ERR_INVALID_ARG, "tile_rows=%d is not 0, 8, 16, 32, 64 or 128", tile_rows);
  if (route < MOE_ROUTE_AUTO || route > MOE_ROUTE_TENSOR_CORE) return fail(MOE_ERR_INVALID_ARG, "route=%d", route);
  if (expert_kernel < MOE_EXPERT_AUTO || expert_kernel > MOE_EXPERT_CUDA_CORES)
    return fail(MOE_ERR_INVALID_ARG, "expert_kernel=%d", expert_kernel);
  g_plan_tile_rows.store(tile_rows, std::memory_order_relaxed);
  g_plan_route.store(route, std::memory_order_relaxed);
  g_plan_expert.store(expert_kernel, std::memory_order_relaxed);
  return MOE_OK;
}

moe_status moe_debug_hold_waits(int32_t which) {
  if (which & ~(MOE_DEBUG_HOLD_DOWN_UNITS | MOE_DEBUG_HOLD_ROUTING_BARRIER))
    return fail(MOE_ERR_INVALID_ARG, "unknown wait mask 0x%x", which);
  g_hold_waits.store(which, std::memory_order_relaxed);
  return MOE_OK;
}

}  // extern "C"

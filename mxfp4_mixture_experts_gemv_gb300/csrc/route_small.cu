// Routing for small token counts (batched decode) in one cooperative launch: router GEMV
// + bias, top-k + softmax, MXFP8 quantisation of x, the stable grouping by
// expert with its tile list, and the gather of the quantised rows into grouped
// order with their scale atoms.
//
// Phase A: CTA e computes the logits of expert e for every token (all loads in
// flight at once: the router weight row and the token rows are a few KB).
// A grid barrier (all CTAs are resident: cooperative launch) publishes them.
// Phase B: every CTA recomputes the top-k and the grouping of all T*k pairs
// (tiny at these sizes, and identical everywhere since it is deterministic),
// which spares a second barrier; then each CTA quantises and places its share
// of the grouped rows and writes its share of the tiles' scale atoms.
//
// Same arithmetic as the other routing kernels: fp32 logits, top-k by (logit
// desc, index asc), softmax over the selected, OCP-style MXFP8 (quant.cuh).
#include <algorithm>

#include "common.cuh"
#include "ptx.cuh"
#include "quant.cuh"
#include "routing.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;

struct RouteSmallArgs {
  const uint16_t* x;
  const uint16_t* wr;
  const uint16_t* br;
  int T, H, E, I, k, tile_rows, max_tiles;
  float* logits;
  int32_t* ids;
  float* w;
  uint8_t* xq;
  uint8_t* xs;
  int32_t* counts;
  int32_t* offsets;
  int32_t* sorted_rows;
  int32_t* inv_pos;
  int32_t* tiles;
  uint8_t* xp;
  uint8_t* xp_sf;
  uint8_t* hq_sf;
  int32_t* grid_bar;
  uint32_t* status;
  uint64_t wait_ns;
  int bar_extra;  // failure-detection hook: wait for this many CTAs more than the grid has
  int fp4;        // activation format: 0 MXFP8 (32 code bytes per block), 1 MXFP4 (16)
};

__global__ void __launch_bounds__(kThreads) route_small_kernel(const RouteSmallArgs a) {
  __shared__ int s_ids[kRouteSmallMaxT * 8];
  __shared__ float s_w[kRouteSmallMaxT * 8];
  __shared__ int s_cnt[257], s_off[258], s_run[257], s_toff[258];
  __shared__ int s_tile_e[kRouteSmallMaxT * 8 + 256];
  __shared__ int s_sorted[kRouteSmallMaxT * 8], s_inv[kRouteSmallMaxT * 8];
  __shared__ uint8_t s_scale[kRouteSmallMaxH / 32];
  extern __shared__ uint4 s_dyn[];  // phase A: staged rows; phase B: logits [T][257]
  float* s_logit = reinterpret_cast<float*>(s_dyn);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int T = a.T, H = a.H, E = a.E, k = a.k;
  // the expert kernel may start its prologue now; it waits for this grid's results
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int TK = T * k;

  // the 256 bytes after the last grouped row are read (as zero padding) by the
  // expert kernel's k-tile-plane boxes: keep them zero
  if (blockIdx.x == 0 && tid < 16)
    reinterpret_cast<uint4*>(a.xp + (int64_t)TK * (H >> a.fp4))[tid] = make_uint4(0, 0, 0, 0);

  // ------------------------------------------------------------ phase A: logits of expert e
  {
    // stage the router row and the T token rows in shared memory with async copies
    // (every copy in flight at once), then contract from shared memory
    uint4* s_rows4 = s_dyn;  // [(T + 1) * H / 8]: row 0 = router row of e, rows 1.. = tokens
    const int e = blockIdx.x;
    const int hc = H / 8;
    const float bias = __uint_as_float((uint32_t)a.br[e] << 16);
    {
      const uint4* wsrc = reinterpret_cast<const uint4*>(a.wr + (int64_t)e * H);
      const uint4* xsrc = reinterpret_cast<const uint4*>(a.x);
      for (int i = tid; i < (T + 1) * hc; i += kThreads) {
        const uint4* src = i < hc ? wsrc + i : xsrc + (i - hc);
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(s_rows4 + i)), "l"(src) : "memory");
      }
      asm volatile("cp.async.commit_group;\n\tcp.async.wait_all;" ::: "memory");
    }
    __syncthreads();
    // warp w contracts the tokens t = w, w + 8, ...: no cross-warp reduction
    constexpr int kTpw = kRouteSmallMaxT / (kThreads / 32);
    float part[kTpw];
#pragma unroll
    for (int m = 0; m < kTpw; ++m) part[m] = 0.f;
    for (int c = lane; c < hc; c += 32) {
      float wv[8];
      bf16x8(s_rows4[c], wv);
#pragma unroll
      for (int m = 0; m < kTpw; ++m) {
        const int t = warp + 8 * m;
        if (t < T) {
          float xv[8];
          bf16x8(s_rows4[(t + 1) * hc + c], xv);
#pragma unroll
          for (int i = 0; i < 8; ++i) part[m] = fmaf(xv[i], wv[i], part[m]);
        }
      }
    }
#pragma unroll
    for (int m = 0; m < kTpw; ++m) {
      const int t = warp + 8 * m;
      if (t < T) {
        float v = part[m];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) a.logits[(int64_t)t * E + e] = v + bias;
      }
    }
  }

  // ------------------------------------------------------------ grid barrier (bounded)
  __shared__ int s_barrier_ok;
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    atomicAdd(a.grid_bar, 1);
    const uint64_t t0 = global_timer_ns();
    int ok = 1;
    while (true) {
      int v;
      asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(a.grid_bar) : "memory");
      if (v >= (int)gridDim.x + a.bar_extra) break;
      if (global_timer_ns() - t0 > a.wait_ns) {
        // some logits may be missing: report it (role 9: routing grid barrier) and
        // publish nothing computed from them
        atomicOr(a.status, kStatusTimeoutRouting);
        atomicCAS(a.status + 1, 0u, (9u << 28) | ((uint32_t)blockIdx.x << 12));
        ok = 0;
        break;
      }
      __nanosleep(32);
    }
    __threadfence();
    s_barrier_ok = ok;
  }
  __syncthreads();
  if (!s_barrier_ok) {
    // an empty tile list: the expert kernel then has no work and writes no output
    if (blockIdx.x == 0 && tid == 0) a.tiles[0] = 0;
    return;
  }

  // ------------------------------------------------------------ phase B
  // every logit (8 independent loads in flight per thread and round)
  for (int i0 = 0; i0 < T * E; i0 += 8 * kThreads) {
    float v[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const int i = i0 + r * kThreads + tid;
      v[r] = i < T * E ? __ldcg(a.logits + i) : 0.f;
    }
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const int i = i0 + r * kThreads + tid;
      if (i < T * E) s_logit[(i / E) * 257 + i % E] = v[r];
    }
  }
  for (int e = tid; e < E; e += kThreads) s_cnt[e] = 0;
  __syncthreads();
  for (int t = warp; t < T; t += kThreads / 32) topk_softmax_warp(s_logit + t * 257, E, k, s_ids + t * k, s_w + t * k, lane);
  __syncthreads();
  const int tshift = __ffs(a.tile_rows) - 1;
  if (warp == 0) group_pairs_warp(s_ids, TK, E, tshift, s_cnt, s_off, s_toff, s_tile_e, s_run, s_sorted, s_inv, lane);
  __syncthreads();
  if (blockIdx.x == 0)
    publish_routing(s_ids, s_w, s_sorted, s_inv, s_cnt, s_off, s_toff, s_tile_e, TK, E, a.tile_rows, a.ids, a.w,
                    a.sorted_rows, a.inv_pos, a.counts, a.offsets, a.tiles);
  // gather: grouped row p -> quantised x row of its token, plus its scale words
  const int nbh = H / 32, kth = (H + kTileK - 1) / kTileK;
  for (int p = blockIdx.x; p < TK; p += gridDim.x) {
    const int f = s_sorted[p], t = f / k;
    // tile of p and its row inside the tile
    int e = s_ids[f];
    const int r_in_e = p - s_off[e];
    const int b = s_toff[e] + r_in_e / a.tile_rows;
    const int n = r_in_e % a.tile_rows;
    for (int blk = tid; blk < nbh; blk += kThreads) {
      uint4 c[2];
      const uint8_t sc = quant_block_regs_act(a.x + (int64_t)t * H + blk * 32, c, a.fp4);
      store_block_codes(a.xp + (int64_t)p * (H >> a.fp4) + blk * (32 >> a.fp4), c, a.fp4);
      s_scale[blk] = sc;
      if (f % k == 0) {  // the token's first slot also publishes x's codes (stage output)
        store_block_codes(a.xq + (int64_t)t * (H >> a.fp4) + blk * (32 >> a.fp4), c, a.fp4);
        a.xs[(int64_t)t * nbh + blk] = sc;
      }
    }
    __syncthreads();
    // one 32-bit word per atom holds this row's 4 block scales
    for (int ka = tid; ka < kth; ka += kThreads) {
      uint32_t wv = 0;
      for (int j = 0; j < 4; ++j) {
        const int kb = 4 * ka + j;
        wv |= (uint32_t)(kb < nbh ? s_scale[kb] : 127) << (8 * j);
      }
      *reinterpret_cast<uint32_t*>(a.xp_sf + ((int64_t)b * kth + ka) * kAtomBytes + (n & 31) * 16 + (n >> 5) * 4) = wv;
    }
    __syncthreads();
  }
}

}  // namespace

cudaError_t launch_route_small(const uint16_t* x, const uint16_t* wr, const uint16_t* br, int T, int H, int E, int I,
                               int k, int tile_rows, int max_tiles, bool fp4, const RouteSmallOut& o, cudaStream_t s) {
  RouteSmallArgs a{x, wr, br, T, H, E, I, k, tile_rows, max_tiles, o.logits, o.ids, o.w, o.xq, o.xs, o.counts,
                   o.offsets, o.sorted_rows, o.inv_pos, o.tiles, o.xp, o.xp_sf, o.hq_sf, o.grid_bar, o.status,
                   wait_limit_ns(), (debug_hold_waits() & MOE_DEBUG_HOLD_ROUTING_BARRIER) ? 1 : 0, fp4 ? 1 : 0};
  const size_t smem = std::max((size_t)(T + 1) * H * 2, (size_t)T * 257 * 4);  // staged rows, later the logits
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(route_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kRouteSmallMaxSmem);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(E);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attrs[1];
  attrs[0].id = cudaLaunchAttributeCooperative;  // the grid barrier needs every CTA resident
  attrs[0].val.cooperative = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, route_small_kernel, a);
}

}  // namespace moe

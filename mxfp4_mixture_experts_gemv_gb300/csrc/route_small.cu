// Routing for small token counts (decode) in one cooperative launch: router GEMV
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
// Same arithmetic as router.cu / permute.cu: fp32 logits, top-k by (logit desc,
// index asc), softmax over the selected, OCP-style MXFP8 (see quant.cuh).
#include <algorithm>

#include "common.cuh"
#include "ptx.cuh"
#include "quant.cuh"

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
};

__global__ void __launch_bounds__(kThreads) route_small_kernel(const RouteSmallArgs a) {
  __shared__ float s_part[kThreads / 32][kRouteSmallMaxT];
  __shared__ int s_ids[kRouteSmallMaxT * 8];
  __shared__ float s_w[kRouteSmallMaxT * 8];
  __shared__ int s_cnt[257], s_off[258], s_run[257], s_toff[258];
  __shared__ int s_tile_e[kRouteSmallMaxT * 8 + 256];
  __shared__ int s_sorted[kRouteSmallMaxT * 8], s_inv[kRouteSmallMaxT * 8];
  __shared__ uint8_t s_scale[kRouteSmallMaxH / 32];
  extern __shared__ uint4 s_dyn[];  // phase A: staged rows; phase B: logits [T][257]
  float* s_logit = reinterpret_cast<float*>(s_dyn);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int T = a.T, H = a.H, E = a.E, I = a.I, k = a.k;
  // the expert kernel may start its prologue now; it waits for this grid's results
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int TK = T * k;

  // ------------------------------------------------------------ phase A: logits of expert e
  {
    // stage the router row and the T token rows in shared memory with async copies
    // (every copy in flight at once), then contract from shared memory
    uint4* s_rows4 = s_dyn;  // [(T + 1) * H / 8]: row 0 = router row of e, rows 1.. = tokens
    const int e = blockIdx.x;
    const int hc = H / 8;
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
    float part[kRouteSmallMaxT];
#pragma unroll
    for (int t = 0; t < kRouteSmallMaxT; ++t) part[t] = 0.f;
    for (int c = tid; c < hc; c += kThreads) {
      float wv[8];
      bf16x8(s_rows4[c], wv);
#pragma unroll
      for (int t = 0; t < kRouteSmallMaxT; ++t) {
        if (t < T) {
          float xv[8];
          bf16x8(s_rows4[(t + 1) * hc + c], xv);
#pragma unroll
          for (int i = 0; i < 8; ++i) part[t] = fmaf(xv[i], wv[i], part[t]);
        }
      }
    }
#pragma unroll
    for (int t = 0; t < kRouteSmallMaxT; ++t) {
      if (t < T) {
        float v = part[t];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) s_part[warp][t] = v;
      }
    }
    __syncthreads();
    if (tid < T) {
      float v = 0.f;
      for (int wi = 0; wi < kThreads / 32; ++wi) v += s_part[wi][tid];
      a.logits[(int64_t)tid * E + e] = v + __uint_as_float((uint32_t)a.br[e] << 16);
    }
  }

  // ------------------------------------------------------------ grid barrier (bounded)
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    atomicAdd(a.grid_bar, 1);
    const uint64_t t0 = global_timer_ns();
    while (true) {
      int v;
      asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(a.grid_bar) : "memory");
      if (v >= (int)gridDim.x) break;
      if (global_timer_ns() - t0 > kWaitLimitNs) {
        atomicOr(a.status, kStatusTimeoutDrain);
        break;
      }
      __nanosleep(32);
    }
    __threadfence();
  }
  __syncthreads();

  // ------------------------------------------------------------ phase B
  for (int i = tid; i < T * E; i += kThreads) s_logit[(i / E) * 257 + i % E] = __ldcg(a.logits + i);
  for (int e = tid; e < E; e += kThreads) s_cnt[e] = 0;
  __syncthreads();
  // top-k + softmax: warp per token
  for (int t = warp; t < T; t += kThreads / 32) {
    float v[8];
    uint32_t taken = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane + 32 * i;
      const float l = e < E ? s_logit[t * 257 + e] : -INFINITY;
      v[i] = isnan(l) ? -INFINITY : l;
    }
    float l0 = 0.f, den = 0.f;
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
      if (j == 0) l0 = bv;
      if (lane == 0) {
        s_ids[t * k + j] = bi;
        s_w[t * k + j] = bv;  // logit for now
      }
      den += expf(bv - l0);
    }
    __syncwarp();
    if (lane < k) s_w[t * k + lane] = expf(s_w[t * k + lane] - l0) / den;
  }
  __syncthreads();
  // grouping (stable counting sort of the T*k pairs by expert), warp 0
  if (warp == 0) {
    for (int f = lane; f < TK; f += 32) atomicAdd(&s_cnt[s_ids[f]], 1);
    __syncwarp();
    warp_expert_scan(s_cnt, E, __ffs(a.tile_rows) - 1, s_off, s_toff, s_tile_e, lane);
    __syncwarp();
    for (int e = lane; e < E; e += 32) s_run[e] = s_off[e];
    __syncwarp();
    const unsigned lt = (1u << lane) - 1u;
    for (int base = 0; base < TK; base += 32) {
      const int f = base + lane;
      const int e = f < TK ? s_ids[f] : -1;
      const unsigned peers = __match_any_sync(0xffffffffu, e);
      const int rank = __popc(peers & lt);
      if (f < TK) {
        const int pos = s_run[e] + rank;
        s_sorted[pos] = f;
        s_inv[f] = pos;
      }
      __syncwarp();
      if (f < TK && rank == 0) s_run[e] += __popc(peers);
      __syncwarp();
    }
  }
  __syncthreads();
  const int n_tiles = s_toff[E];
  // CTA 0 publishes the routing results
  if (blockIdx.x == 0) {
    for (int i = tid; i < TK; i += kThreads) {
      a.ids[i] = s_ids[i];
      a.w[i] = s_w[i];
      a.sorted_rows[i] = s_sorted[i];
      a.inv_pos[i] = s_inv[i];
    }
    for (int e = tid; e < E; e += kThreads) {
      a.counts[e] = s_cnt[e];
      a.offsets[e] = s_off[e];
    }
    for (int t = tid; t < n_tiles; t += kThreads) {
      const int e = s_tile_e[t];
      const int r0 = (t - s_toff[e]) * a.tile_rows;
      reinterpret_cast<int4*>(a.tiles + 4)[t] = make_int4(e, s_off[e] + r0, min(a.tile_rows, s_cnt[e] - r0), 0);
    }
    if (tid == 0) {
      a.offsets[E] = s_off[E];
      a.tiles[0] = n_tiles;
    }
  }
  // gather: grouped row p -> quantised x row of its token, plus its scale words
  const int nbh = H / 32, kth = (H + kTileK - 1) / kTileK, kti = (I + kTileK - 1) / kTileK;
  for (int p = blockIdx.x; p < TK; p += gridDim.x) {
    const int f = s_sorted[p], t = f / k;
    // tile of p and its row inside the tile
    int e = s_ids[f];
    const int r_in_e = p - s_off[e];
    const int b = s_toff[e] + r_in_e / a.tile_rows;
    const int n = r_in_e % a.tile_rows;
    for (int blk = tid; blk < nbh; blk += kThreads) {
      const uint8_t sc = quant_block(a.x + (int64_t)t * H + blk * 32, a.xp + (int64_t)p * H + blk * 32);
      s_scale[blk] = sc;
      if (f % k == 0) {  // the token's first slot also publishes x's codes (stage output)
        for (int i = 0; i < 32; i += 16)
          *reinterpret_cast<uint4*>(a.xq + (int64_t)t * H + blk * 32 + i) =
              *reinterpret_cast<const uint4*>(a.xp + (int64_t)p * H + blk * 32 + i);
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
                               int k, int tile_rows, int max_tiles, const RouteSmallOut& o, cudaStream_t s) {
  RouteSmallArgs a{x, wr, br, T, H, E, I, k, tile_rows, max_tiles, o.logits, o.ids, o.w, o.xq, o.xs, o.counts,
                   o.offsets, o.sorted_rows, o.inv_pos, o.tiles, o.xp, o.xp_sf, o.hq_sf, o.grid_bar, o.status};
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

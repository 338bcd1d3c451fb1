// Routing for a handful of tokens (decode, T <= 8) in one thread-block cluster:
// router GEMV + bias, top-k + softmax, the stable grouping by expert with its
// tile list, and the MXFP8 quantisation of the token rows straight into grouped
// order with their scale atoms.
//
// The cluster's CTAs split the experts: each CTA copies its slice of router rows
// and all T token rows into shared memory with two bulk copies, computes its
// experts' logits, and after one cluster barrier reads every CTA's logits
// through distributed shared memory.  The selection and the grouping are then
// recomputed by every CTA (a few dozen pairs; deterministic, so identical
// everywhere) and each CTA quantises its share of (token, 128-column) units
// from the token rows it already holds, writing every slot the token goes to.
// Nothing here goes through global memory twice and nothing waits on another
// grid, so the chain from launch to the tile list is a single DRAM round trip
// plus a cluster barrier.  The kernel also clears the counters the expert
// kernel uses, which the expert kernel reads only after this grid completes.
//
// Same arithmetic as the other routing kernels: fp32 logits, top-k by (logit
// desc, index asc), softmax over the selected, OCP-style MXFP8 (quant.cuh).
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "ptx.cuh"
#include "quant.cuh"
#include "routing.cuh"

namespace moe {
namespace {

constexpr int kRcThreads = 256;
constexpr int kRcMaxT = kRouteClusterMaxT;
constexpr int kRcMaxEpc = 32;  // experts per CTA: E <= 256 over at least 8 CTAs

struct RouteClusterArgs {
  const uint16_t* x;
  const uint16_t* wr;
  const uint16_t* br;
  int T, H, E, k, tshift;
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
  uint32_t* zero;  // words cleared for this forward (status and the expert kernel's counters)
  int zero_words;
  uint32_t* status;
};

__global__ void __launch_bounds__(kRcThreads, 1) route_cluster_kernel(const RouteClusterArgs a) {
  extern __shared__ __align__(128) uint8_t rc_dyn[];  // [epc][H] router rows, then [T][H] token rows (bf16)
  __shared__ float s_mine[kRcMaxEpc][kRcMaxT];       // logits of this CTA's experts
  __shared__ float s_log[kRcMaxT][257];              // every expert's logits
  __shared__ int s_ids[kRcMaxT * 8], s_sorted[kRcMaxT * 8], s_inv[kRcMaxT * 8];
  __shared__ float s_w[kRcMaxT * 8];
  __shared__ int s_cnt[257], s_off[258], s_run[257], s_toff[258];
  __shared__ int s_tile_e[kRcMaxT * 8 + 256];
  __shared__ __align__(8) uint64_t s_bar;
  // the expert kernel may start its prologue now; it waits for this grid's results
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int T = a.T, H = a.H, E = a.E, k = a.k, TK = T * k;
  const int rank = (int)cluster_ctarank(), ncta = (int)cluster_nctarank();
  const int epc = (E + ncta - 1) / ncta, e0 = rank * epc, ne = max(0, min(epc, E - e0));
  uint16_t* s_wr = reinterpret_cast<uint16_t*>(rc_dyn);
  uint16_t* s_x = s_wr + (size_t)epc * H;

  if (tid == 0) {
    mbar_init(&s_bar, 1);
    fence_mbar_init();
    const uint32_t bw = (uint32_t)ne * H * 2, bx = (uint32_t)T * H * 2;
    mbar_arrive_expect_tx(&s_bar, bw + bx);
    if (bw) bulk_g2s(s_wr, a.wr + (int64_t)e0 * H, bw, &s_bar);
    bulk_g2s(s_x, a.x, bx, &s_bar);
  }
  // biases of this warp's experts (in flight with the copies)
  float bias[kRcMaxEpc / 8];
#pragma unroll
  for (int m = 0; m < kRcMaxEpc / 8; ++m) {
    const int j = warp + 8 * m;
    bias[m] = j < ne ? __uint_as_float((uint32_t)a.br[e0 + j] << 16) : 0.f;
  }
  for (int i = rank + ncta * tid; i < a.zero_words; i += ncta * kRcThreads) a.zero[i] = 0u;
  for (int e = tid; e < E; e += kRcThreads) s_cnt[e] = 0;
  __syncthreads();  // the barrier's initialisation is visible to every thread
  const bool staged = mbar_wait(&s_bar, 0, kWaitLimitNs);

  // logits of this CTA's experts: warp per expert, lanes over 16-byte column chunks
  const int hc = H / 8;
#pragma unroll
  for (int m = 0; m < kRcMaxEpc / 8; ++m) {
    const int j = warp + 8 * m;
    if (j < ne) {
      float acc[kRcMaxT];
#pragma unroll
      for (int t = 0; t < kRcMaxT; ++t) acc[t] = 0.f;
      const uint4* w4 = reinterpret_cast<const uint4*>(s_wr + (size_t)j * H);
      for (int c = lane; c < hc; c += 32) {
        float wv[8];
        bf16x8(w4[c], wv);
#pragma unroll
        for (int t = 0; t < kRcMaxT; ++t) {
          if (t < T) {
            float xv[8];
            bf16x8(reinterpret_cast<const uint4*>(s_x + (size_t)t * H)[c], xv);
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[t] = fmaf(xv[i], wv[i], acc[t]);
          }
        }
      }
#pragma unroll
      for (int t = 0; t < kRcMaxT; ++t) {
        if (t < T) {
          float v = acc[t];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
          v += bias[m];
          if (lane == 0) {
            s_mine[j][t] = v;
            a.logits[(int64_t)t * E + e0 + j] = v;
          }
        }
      }
    }
  }
  cluster_arrive();
  cluster_wait();  // every CTA's logits (and every CTA's clearing) are done
  if (!staged && tid == 0) {
    atomicOr(a.status, kStatusTimeoutProducer);
    atomicCAS(a.status + 1, 0u, (6u << 28) | ((uint32_t)rank << 12));  // role 6: routing copies
  }
  for (int i = tid; i < T * E; i += kRcThreads) {
    const int t = i / E, e = i - t * E;
    s_log[t][e] = ld_dsmem_f32(&s_mine[e % epc][t], (uint32_t)(e / epc));
  }
  cluster_arrive();  // done reading the other CTAs' shared memory (matched by the wait at the end)
  __syncthreads();
  for (int t = warp; t < T; t += kRcThreads / 32) topk_softmax_warp(s_log[t], E, k, s_ids + t * k, s_w + t * k, lane);
  __syncthreads();
  if (warp == 0)
    group_pairs_warp(s_ids, TK, E, a.tshift, s_cnt, s_off, s_toff, s_tile_e, s_run, s_sorted, s_inv, lane);
  __syncthreads();
  if (rank == 0)
    publish_routing(s_ids, s_w, s_sorted, s_inv, s_cnt, s_off, s_toff, s_tile_e, TK, E, 1 << a.tshift, a.ids, a.w,
                    a.sorted_rows, a.inv_pos, a.counts, a.offsets, a.tiles);

  // quantise (token t, atom column ka) units: four 32-element blocks, written to
  // every grouped row of the token with one scale word each
  const int nbh = H / 32, kth = (H + kTileK - 1) / kTileK;
  for (int u = rank + ncta * tid; u < T * kth; u += ncta * kRcThreads) {
    const int t = u / kth, ka = u - t * kth;
    uint4 c[4][2];
    uint32_t word = 0;
#pragma unroll
    for (int jb = 0; jb < 4; ++jb) {
      const int kb = 4 * ka + jb;
      const uint8_t sc = kb < nbh ? quant_block_regs(s_x + (size_t)t * H + kb * 32, c[jb]) : (uint8_t)127;
      word |= (uint32_t)sc << (8 * jb);
    }
    for (int j = 0; j < k; ++j) {
      const int f = t * k + j, p = s_inv[f];
      uint4* dst = reinterpret_cast<uint4*>(a.xp + (int64_t)p * H + ka * kTileK);
#pragma unroll
      for (int jb = 0; jb < 4; ++jb) {
        if (4 * ka + jb < nbh) {
          dst[2 * jb] = c[jb][0];
          dst[2 * jb + 1] = c[jb][1];
        }
      }
      *reinterpret_cast<uint32_t*>(a.xp_sf + row_sf_word(p, ka, kth, s_ids, s_sorted, s_off, s_toff, a.tshift)) =
          word;
    }
    // the token's codes and scales (stage output)
    uint4* q = reinterpret_cast<uint4*>(a.xq + (int64_t)t * H + ka * kTileK);
#pragma unroll
    for (int jb = 0; jb < 4; ++jb) {
      const int kb = 4 * ka + jb;
      if (kb < nbh) {
        q[2 * jb] = c[jb][0];
        q[2 * jb + 1] = c[jb][1];
        a.xs[(int64_t)t * nbh + kb] = (uint8_t)(word >> (8 * jb));
      }
    }
  }
  cluster_wait();
}

int g_cluster_size[64];  // per device: 0 = not chosen yet
std::mutex g_cluster_mu;

}  // namespace

bool route_cluster_fits(int T, int E, int H) {
  const int epc = (E + 7) / 8;  // the smallest cluster this kernel runs on
  return T >= 1 && T <= kRouteClusterMaxT && E <= 256 &&
         (size_t)(epc + T) * H * 2 <= kRouteClusterMaxSmem;
}

cudaError_t launch_route_cluster(const uint16_t* x, const uint16_t* wr, const uint16_t* br, int T, int H, int E,
                                 int k, int tile_rows, const RouteClusterOut& o, cudaStream_t s) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  int csize;
  {
    std::lock_guard<std::mutex> lk(g_cluster_mu);
    csize = g_cluster_size[dev];
    if (csize == 0) {
      e = cudaFuncSetAttribute(route_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)kRouteClusterMaxSmem);
      if (e != cudaSuccess) return e;
      e = cudaFuncSetAttribute(route_cluster_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      // 16 CTAs when the device can place such a cluster with the largest shared
      // memory this kernel asks for, else the portable 8
      csize = 8;
      if (e == cudaSuccess) {
        cudaLaunchConfig_t q = {};
        q.gridDim = dim3(16);
        q.blockDim = dim3(kRcThreads);
        q.dynamicSmemBytes = kRouteClusterMaxSmem;
        cudaLaunchAttribute qa[1];
        qa[0].id = cudaLaunchAttributeClusterDimension;
        qa[0].val.clusterDim.x = 16;
        qa[0].val.clusterDim.y = 1;
        qa[0].val.clusterDim.z = 1;
        q.attrs = qa;
        q.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, route_cluster_kernel, &q) == cudaSuccess && n >= 1) csize = 16;
      }
      (void)cudaGetLastError();
      g_cluster_size[dev] = csize;
    }
  }
  const int epc = (E + csize - 1) / csize;
  RouteClusterArgs a{x, wr, br, T, H, E, k, __builtin_ctz((unsigned)tile_rows), o.logits, o.ids, o.w, o.xq, o.xs,
                     o.counts, o.offsets, o.sorted_rows, o.inv_pos, o.tiles, o.xp, o.xp_sf, o.zero,
                     o.zero_words, o.status};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(csize);
  cfg.blockDim = dim3(kRcThreads);
  cfg.dynamicSmemBytes = (size_t)(epc + T) * H * 2;
  cfg.stream = s;
  cudaLaunchAttribute attrs[1];
  attrs[0].id = cudaLaunchAttributeClusterDimension;
  attrs[0].val.clusterDim.x = csize;
  attrs[0].val.clusterDim.y = 1;
  attrs[0].val.clusterDim.z = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, route_cluster_kernel, a);
}

}  // namespace moe

// Routing for a handful of tokens (decode, T <= 8) in one thread-block cluster:
// router GEMV + bias, top-k + softmax, the stable grouping by expert with its
// tile list, and the MXFP8 quantisation of the token rows straight into grouped
// order with their scale atoms.
//
// The cluster's CTAs split the experts: each CTA copies its slice of router rows
// and all T token rows into shared memory with two bulk copies, computes its
// experts' logits and stores them into every CTA's shared memory (distributed
// shared memory) before one cluster barrier.  While the barrier completes, each
// thread quantises its (token, 32-element block) unit of the token rows it
// already holds.  The selection and the grouping (a few dozen pairs, ranked
// inside one warp) are then recomputed by every CTA -- deterministic, so
// identical everywhere -- and each thread writes its unit to every grouped row
// of its token.  Nothing goes through global memory twice and nothing waits on
// another grid: the chain from launch to the tile list is one DRAM round trip
// plus one cluster barrier.  The kernel also clears the counters the expert
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

constexpr int kRcThreads = 384;
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
  int32_t* flags;  // [0] tile list published, [1] routing CTAs whose grouped rows are written
  uint64_t wait_ns;
  int fp4;  // activation codes: 0 MXFP8 (32 code bytes per block), 1 E2M1 (16)
  int nv;   // 1: NVFP4 (two E4M3 scales per 32-element block, unit global scale)
};

// Sum-reduce N values held by every lane of a warp so that each lane ends up
// with N / 32 complete sums: after the call lane l holds the sums of the values
// with index l * (N / 32) + m in v[m].
template <int N>
__device__ __forceinline__ void warp_reduce_scatter(float (&v)[N], int lane) {
  int n = N;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < N / 2; ++i) {
      if (i < n / 2) {
        const float lo = v[i], hi = v[i + n / 2];
        const float got = __shfl_xor_sync(0xffffffffu, up ? lo : hi, o);
        v[i] = (up ? hi : lo) + got;
      }
    }
    n >>= 1;
  }
}

__device__ __forceinline__ void st_dsmem_f32(const void* p, uint32_t cta, float v) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(cta));
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(r), "f"(v) : "memory");
}

template <int TM>  // token capacity of this instance (4 or 8)
__global__ void __launch_bounds__(kRcThreads, 1) route_cluster_kernel(const RouteClusterArgs a) {
  constexpr int kG = 8;           // experts contracted together
  constexpr int kN = kG * TM;     // partial sums per thread
  extern __shared__ __align__(128) uint8_t rc_dyn[];  // [epc][H] router rows, then [T][H] token rows (bf16)
  __shared__ float s_log[TM][257];                    // every expert's logits (pushed by their CTAs)
  __shared__ float s_red[kRcThreads / 32][kN];
  __shared__ float s_bias[kRcMaxEpc];
  __shared__ int s_ids[TM * 8], s_sorted[TM * 8], s_inv[TM * 8];
  __shared__ float s_w[TM * 8];
  __shared__ int s_off[256], s_toff[256];  // of the experts the pairs use
  __shared__ __align__(8) uint64_t s_bar;
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
  // The expert kernel may start once every CTA has let it (programmatic dependent
  // launch).  It then follows this grid through the two flags, so CTA 0 first
  // clears them, this forward's status words and the expert kernel's counters
  // (while the copies are in flight), and makes that visible.
  if (rank == 0) {
    for (int i = tid; i < a.zero_words; i += kRcThreads) a.zero[i] = 0u;
    // the 256 bytes after the last grouped row are read (as zero padding) by the
    // expert kernel's k-tile-plane boxes: keep them zero
    if (tid >= 32 && tid < 48)
      reinterpret_cast<uint4*>(a.xp + (int64_t)TK * (H >> a.fp4))[tid - 32] = make_uint4(0, 0, 0, 0);
    __threadfence();
  }
  // biases of this CTA's experts (in flight with the copies)
  if (tid < ne) s_bias[tid] = __uint_as_float((uint32_t)a.br[e0 + tid] << 16);
  __syncthreads();  // the barrier's initialisation (and CTA 0's clearing) is visible to every thread
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const bool staged = mbar_wait(&s_bar, 0, a.wait_ns);

  // logits of this CTA's experts, kG at a time: thread = 16-byte column chunk(s),
  // the token chunks stay in registers across the kG router rows
  const int hc = H / 8;
  for (int g0 = 0; g0 < ne; g0 += kG) {
    float acc[kN];
#pragma unroll
    for (int i = 0; i < kN; ++i) acc[i] = 0.f;
    for (int c = tid; c < hc; c += kRcThreads) {
      float xv[TM][8];
#pragma unroll
      for (int t = 0; t < TM; ++t) {
        if (t < T) bf16x8(reinterpret_cast<const uint4*>(s_x + (size_t)t * H)[c], xv[t]);
        else
#pragma unroll
          for (int i = 0; i < 8; ++i) xv[t][i] = 0.f;
      }
#pragma unroll
      for (int j = 0; j < kG; ++j) {
        if (g0 + j < ne) {
          float wv[8];
          bf16x8(reinterpret_cast<const uint4*>(s_wr + (size_t)(g0 + j) * H)[c], wv);
#pragma unroll
          for (int t = 0; t < TM; ++t)
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[j * TM + t] = fmaf(xv[t][i], wv[i], acc[j * TM + t]);
        }
      }
    }
    warp_reduce_scatter<kN>(acc, lane);
#pragma unroll
    for (int m = 0; m < kN / 32; ++m) s_red[warp][lane * (kN / 32) + m] = acc[m];
    __syncthreads();
    if (tid < kN) {
      const int j = tid / TM, t = tid % TM;
      float v = 0.f;
#pragma unroll
      for (int wi = 0; wi < kRcThreads / 32; ++wi) v += s_red[wi][tid];
      if (g0 + j < ne && t < T) {
        v += s_bias[g0 + j];
        const int e = e0 + g0 + j;
        for (int r = 0; r < ncta; ++r) st_dsmem_f32(&s_log[t][e], (uint32_t)r, v);
      }
    }
    __syncthreads();
  }
  cluster_arrive();

  // While the logits travel: this thread's quantisation unit (token t, 32-element
  // block kb) into registers, the token's codes and scale (stage output), and the
  // expert kernel's counters (read by it only after this grid completes).
  const int nbh = H / 32, kth = (H + kTileK - 1) / kTileK;
  const int u = rank + ncta * tid;
  const bool has_u = u < T * nbh;
  const int ut = has_u ? u / nbh : 0, ukb = has_u ? u - ut * nbh : 0;
  uint4 qc[2];
  uint32_t qs = 0;  // the block's scale code (NVFP4: the two 16-element blocks' codes, low byte first)
  if (has_u) {
    if (a.nv) {
      float f[32];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float g[8];
        bf16x8(reinterpret_cast<const uint4*>(s_x + (size_t)ut * H + ukb * 32)[q], g);
#pragma unroll
        for (int i = 0; i < 8; ++i) f[8 * q + i] = g[i];
      }
      uint32_t p0[2], p1[2];
      qs = nvfp4_block16(f, 1.0f, p0) | (nvfp4_block16(f + 16, 1.0f, p1) << 8);
      qc[0] = make_uint4(p0[0], p0[1], p1[0], p1[1]);
      *reinterpret_cast<uint16_t*>(a.xs + (int64_t)ut * (H / 16) + 2 * ukb) = (uint16_t)qs;
    } else {
      qs = quant_block_regs_act(s_x + (size_t)ut * H + ukb * 32, qc, a.fp4);
      a.xs[(int64_t)ut * nbh + ukb] = (uint8_t)qs;
    }
    store_block_codes(a.xq + (int64_t)ut * (H >> a.fp4) + ukb * (32 >> a.fp4), qc, a.fp4);
  }

  cluster_wait();  // every CTA has every logit; no CTA touches another's shared memory after this
  if (!staged && tid == 0) {
    atomicOr(a.status, kStatusTimeoutProducer);
    atomicCAS(a.status + 1, 0u, (8u << 28) | ((uint32_t)rank << 12));  // role 8: routing copies
  }
  for (int t = warp; t < T; t += kRcThreads / 32) topk_softmax_warp(s_log[t], E, k, s_ids + t * k, s_w + t * k, lane);
  __syncthreads();
  if (warp == 0) {
    group_pairs_small_warp(s_ids, TK, E, a.tshift, s_off, s_toff, s_sorted, s_inv, rank == 0 ? a.tiles : nullptr, lane);
    if (rank == 0) {
      // publish the tile list (the counters were cleared and fenced at the start):
      // the expert kernel may now read it and start its weight copies.  The release
      // store orders the warp's tile writes, ordered before it by the warp barrier.
      __syncwarp();
      if (lane == 0) st_release_gpu(a.flags, 1);
    }
  } else {
    // meanwhile: this CTA's experts' logits, and (CTA 0) the selection and the
    // per-expert counts and offsets (stage outputs)
    const int v = tid - 32, nv = kRcThreads - 32;
    for (int i = v; i < T * ne; i += nv) {
      const int t = i / ne, e = e0 + i % ne;
      a.logits[(int64_t)t * E + e] = s_log[t][e];
    }
    if (rank == 0) {
      for (int i = v; i < TK; i += nv) {
        a.ids[i] = s_ids[i];
        a.w[i] = s_w[i];
      }
      expert_counts_offsets(s_ids, TK, E, a.counts, a.offsets, v, nv);
    }
  }
  __syncthreads();
  if (rank == 0)
    for (int i = tid; i < TK; i += kRcThreads) {
      a.sorted_rows[i] = s_sorted[i];
      a.inv_pos[i] = s_inv[i];
    }
  // the unit's codes go to every grouped row of its token, the scale byte to each
  // row's atom word; the last real block also sets the padding bytes of its word
  if (has_u) {
    const int ka = ukb >> 2;
    for (int j = 0; j < k; ++j) {
      const int f = ut * k + j, p = s_inv[f], e = s_ids[f];
      store_block_codes(a.xp + (int64_t)p * (H >> a.fp4) + ukb * (32 >> a.fp4), qc, a.fp4);
      const int r_in_e = p - s_off[e];
      const int b = s_toff[e] + (r_in_e >> a.tshift), n = r_in_e & ((1 << a.tshift) - 1);
      const int row_off = (n & 31) * 16 + (n >> 5) * 4;
      if (a.nv) {
        // a k-tile's eight 16-element blocks fill two atoms; 32-element block s of the
        // k-tile is half-word s & 1 of atom (s >> 1) & 1.  The last real block also
        // gives the padding blocks after it the zero scale.
        uint8_t* atoms = a.xp_sf + ((int64_t)b * kth + ka) * 2 * kAtomBytes + row_off;
        const int sl = ukb & 3;
        reinterpret_cast<uint16_t*>(atoms + ((sl >> 1) & 1) * kAtomBytes)[sl & 1] = (uint16_t)qs;
        if (ukb == nbh - 1)
          for (int jj = sl + 1; jj < 4; ++jj) reinterpret_cast<uint16_t*>(atoms + ((jj >> 1) & 1) * kAtomBytes)[jj & 1] = 0;
      } else {
        uint8_t* wd = a.xp_sf + ((int64_t)b * kth + ka) * kAtomBytes + row_off;
        wd[ukb & 3] = (uint8_t)qs;
        if (ukb == nbh - 1)
          for (int jj = (ukb & 3) + 1; jj < 4; ++jj) wd[jj] = 127;
      }
    }
  }
  // this CTA's grouped rows and scale bytes (and CTA 0's weights and permutation,
  // which the combine reads) are written: count it in, so that the expert kernel's
  // activation copies may read them
  __threadfence();
  __syncthreads();
  if (tid == 0) red_add_release_gpu(a.flags + 1, 1);
}

int g_cluster_size[64];  // per device: 0 = not chosen yet
std::mutex g_cluster_mu;

}  // namespace

bool route_cluster_fits(int T, int E, int H) {
  const int epc = (E + 7) / 8;  // the smallest cluster this kernel runs on
  // (T * k <= 64 pairs follows from T <= 8, k <= 8; one quantisation unit per thread)
  return T >= 1 && T <= kRouteClusterMaxT && E <= 256 && (size_t)(epc + T) * H * 2 <= kRouteClusterMaxSmem &&
         T * (H / 32) <= 8 * kRcThreads;
}

cudaError_t launch_route_cluster(const uint16_t* x, const uint16_t* wr, const uint16_t* br, int T, int H, int E,
                                 int k, int tile_rows, int fmt, const RouteClusterOut& o, int* ctas, cudaStream_t s) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  int csize;
  {
    std::lock_guard<std::mutex> lk(g_cluster_mu);
    csize = g_cluster_size[dev];
    if (csize == 0) {
      for (auto fn : {route_cluster_kernel<4>, route_cluster_kernel<8>}) {
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kRouteClusterMaxSmem);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) break;
      }
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
        if (cudaOccupancyMaxActiveClusters(&n, route_cluster_kernel<8>, &q) == cudaSuccess && n >= 1) csize = 16;
      }
      (void)cudaGetLastError();
      g_cluster_size[dev] = csize;
    }
  }
  const int epc = (E + csize - 1) / csize;
  RouteClusterArgs a{x, wr, br, T, H, E, k, __builtin_ctz((unsigned)tile_rows), o.logits, o.ids, o.w, o.xq, o.xs,
                     o.counts, o.offsets, o.sorted_rows, o.inv_pos, o.tiles, o.xp, o.xp_sf, o.zero,
                     o.zero_words, o.status, o.flags, wait_limit_ns(), fmt != kActMxfp8 ? 1 : 0,
                     fmt == kActNvfp4 ? 1 : 0};
  *ctas = csize;
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
  return T <= 4 ? cudaLaunchKernelEx(&cfg, route_cluster_kernel<4>, a) : cudaLaunchKernelEx(&cfg, route_cluster_kernel<8>, a);
}

}  // namespace moe

// Router for larger token counts on tcgen05 (kind::f16, bf16 inputs, fp32
// accumulation in tensor memory): logits[T, E] = x[T, H] . Wr[E, H]^T + br, then
// the top-k selection and the softmax over the selected.
//
// Routing rule: top-k experts by logit (descending, lower index first on ties),
// then softmax over the k selected ("GPT-OSS-120B on DGX Spark: From MXFP4 to
// NVFP4", section "GPT-OSS-120B Architecture": 128 experts, 4 active per token;
// router weights in BF16).
//
// A 128-token tile is contracted by a cluster of `splits` CTAs (384 threads
// each), CTA r taking the r-th run of k-slices: warp 0 streams x and Wr k-slices
// by TMA (128-byte swizzle, 64 bf16 per row), one lane of warp 1 issues the MMAs,
// and warps 2..5 read the accumulator (thread = token).  A lone CTA selects from
// its accumulator, a thread per token.  In a cluster every CTA parks its partial
// logits in its own shared memory; after a cluster barrier each CTA receives, by
// bulk shared-to-shared copies, the peers' partials of the tokens it finishes,
// adds them in rank order (the same sum on every run) and selects with one warp
// per token, on all 12 warps.  Splitting lets the grid cover the GPU: a single
// CTA per tile is bound by one SM's copy bandwidth.  Waits are bounded.
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kRTileM = 128;   // tokens per tile (MMA M)
constexpr int kRK = 64;        // bf16 elements per k-slice (one 128-byte swizzled row)
constexpr int kRMaxSplits = 8;  // portable cluster size
constexpr int kRThreads = 384;  // warps 0..5 as below; all 12 warps finish split tiles
constexpr int kRWarps = kRThreads / 32;

struct RouterArgs {
  const uint16_t* br;
  float* logits;
  int32_t* ids;
  float* w;
  uint32_t* status;
  int T, H, E, k, n_pad;  // n_pad: E rounded up to 16 (MMA N)
  int splits, slices;     // CTAs per tile (the cluster), k-slices per CTA
  uint64_t wait_ns;       // limit of every bounded wait
};

// Instruction descriptor of kind::f16 with bf16 A and B, fp32 accumulator, both K-major.
__host__ __device__ constexpr uint32_t idesc_bf16(uint32_t M, uint32_t N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

template <int NPAD>
struct RouterCfg {
  static constexpr uint32_t kA = kRTileM * kRK * 2;  // 16 KB
  static constexpr uint32_t kB = NPAD * kRK * 2;     // up to 32 KB
  static constexpr uint32_t kStage = kA + kB;
  static constexpr int kStages = NPAD <= 128 ? 6 : 4;
  static constexpr uint32_t kSmem = 1024 + kStages * kStage + 256;
  static constexpr uint32_t kTmemCols = NPAD <= 128 ? 128 : 256;
  // Split tiles reuse the idle stage buffers: this CTA's partial logits (128
  // rows), then an inbox of the peers' partials for the rows this CTA finishes
  // (splits * ceil(128 / splits) <= 128 + kRMaxSplits rows).  Rows of NPAD + 4
  // floats: 16-byte stores of 8 consecutive rows cover all banks, and row runs
  // are whole 16-byte units for the bulk copies.
  static constexpr uint32_t kRedStride = NPAD + 4;
  static constexpr uint32_t kParkBytes = kRTileM * kRedStride * 4;
  static constexpr bool kCanSplit = kParkBytes + (kRTileM + kRMaxSplits) * kRedStride * 4 <= kStages * kStage;
  static_assert(kSmem <= 227 * 1024, "shared memory");
};

// Running top-8 of one token's logits, sorted by (logit desc, index asc).  The
// experts arrive in ascending order, so only a strictly larger logit moves
// ahead of an earlier one; a NaN logit ranks last.
struct Top8 {
  float v[8];
  int i[8];
};

__device__ __forceinline__ void top8_init(Top8& b) {
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    b.v[j] = -INFINITY;
    b.i[j] = 0x7FFFFFFF;
  }
}

__device__ __forceinline__ void top8_push(Top8& b, float v, int e) {
  if (isnan(v)) v = -INFINITY;
  if (!(v > b.v[7] || b.i[7] == 0x7FFFFFFF)) return;
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    const bool take = v > b.v[s] || b.i[s] == 0x7FFFFFFF;
    const float tv = b.v[s];
    const int ti = b.i[s];
    b.v[s] = take ? v : tv;
    b.i[s] = take ? e : ti;
    v = take ? tv : v;
    e = take ? ti : e;
  }
}

// ids and softmax weights of the first k
__device__ __forceinline__ void top8_emit(const Top8& b, int k, int32_t* ids, float* w) {
  float den = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j)
    if (j < k) den += expf(b.v[j] - b.v[0]);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    if (j < k) {
      ids[j] = b.i[j];
      w[j] = expf(b.v[j] - b.v[0]) / den;
    }
  }
}

template <int NPAD>
__global__ void __launch_bounds__(kRThreads, 1)
    router_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                     const RouterArgs a) {
  using C = RouterCfg<NPAD>;
  constexpr int kRStages = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + kRStages * C::kA;
  uint64_t* full = reinterpret_cast<uint64_t*>(sB + kRStages * C::kB);
  uint64_t* empty = full + kRStages;
  uint64_t* done = empty + kRStages;
  uint64_t* inbox_full = done + 1;  // split tiles: the peers' partials have landed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(inbox_full + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile = blockIdx.x / a.splits, rank = blockIdx.x - tile * a.splits;  // rank in the cluster
  const int t0 = tile * kRTileM;
  const int ksl = (a.H + kRK - 1) / kRK;
  const int k0 = rank * a.slices, k1 = min(ksl, k0 + a.slices);
  float* park = reinterpret_cast<float*>(sA);
  float* inbox = reinterpret_cast<float*>(sA + C::kParkBytes);
  const int rows_per = (kRTileM + a.splits - 1) / a.splits;  // rows each CTA of a split tile finishes
  if (threadIdx.x == 0) {
    for (int s = 0; s < kRStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(done, 1);
    mbar_init(inbox_full, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  __shared__ float s_bias[NPAD];  // router bias in fp32 (zero past E)
  for (int e = threadIdx.x; e < NPAD; e += blockDim.x)
    s_bias[e] = e < a.E ? __uint_as_float((uint32_t)a.br[e] << 16) : 0.f;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    int s = 0;
    uint32_t ph = 0;
    int issued = 0;
    for (int kk = k0; kk < k1; ++kk) {
      if (!mbar_wait_warp(&empty[s], ph ^ 1u, a.wait_ns)) {
        if (lane == 0) atomicOr(a.status, kStatusTimeoutProducer);
        break;
      }
      if (elect_one()) {
        mbar_arrive_expect_tx(&full[s], C::kStage);
        tma_load_2d(sA + s * C::kA, &tmX, &full[s], kk * kRK, t0);
        tma_load_2d(sB + s * C::kB, &tmW, &full[s], kk * kRK, 0);
      }
      __syncwarp();
      ++issued;
      if (++s == kRStages) {
        s = 0;
        ph ^= 1u;
      }
    }
    for (int st = 0; st < kRStages && st < issued; ++st) {
      const int last = ((issued - 1 - st) / kRStages) * kRStages + st;
      if (!mbar_wait_warp(&full[st], (uint32_t)((last / kRStages) & 1), kDrainLimitNs) && lane == 0)
        atomicOr(a.status, kStatusTimeoutDrain);
    }
  } else if (warp == 1) {
    int s = 0;
    uint32_t ph = 0;
    const uint32_t idesc = idesc_bf16(kRTileM, NPAD);
    for (int kk = k0; kk < k1; ++kk) {
      if (!mbar_wait_warp(&full[s], ph, a.wait_ns)) {
        if (lane == 0) atomicOr(a.status, kStatusTimeoutMma);
        break;
      }
      tc_fence_after();
      const uint64_t ad = sdesc_sw128(smem_u32(sA + s * C::kA));
      const uint64_t bd = sdesc_sw128(smem_u32(sB + s * C::kB));
      if (elect_one()) {
#pragma unroll
        for (uint32_t j = 0; j < kRK / 16; ++j)  // K = 16 per MMA: 32 bytes along the swizzled row
          umma_bf16(tmem, ad + 2u * j, bd + 2u * j, idesc, ((kk - k0) | (int)j) != 0);
        umma_commit(&empty[s]);
      }
      __syncwarp();
      if (++s == kRStages) {
        s = 0;
        ph ^= 1u;
      }
    }
    if (elect_one()) umma_commit(done);
    __syncwarp();
  } else if (warp < 6) {
    // epilogue: thread = token row of the tile (tmem lane quarter warp % 4)
    const int q = warp & 3, row = 32 * q + lane, t = t0 + row;
    const bool ok = mbar_wait_warp(done, 0, a.wait_ns);
    if (!ok && lane == 0) atomicOr(a.status, kStatusTimeoutEpilogue);
    tc_fence_after();
    const uint32_t tb = tmem + ((uint32_t)(32 * q) << 16);
    if (a.splits == 1) {
      Top8 best;
      top8_init(best);
      for (int c0 = 0; c0 < NPAD; c0 += 16) {
        uint32_t r[16];
        if (ok) {
          tmem_ld_32x32b_x16(tb + (uint32_t)c0, r);
          tmem_ld_wait();
        }
        if (ok && t < a.T) {
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int e = c0 + j;
            if (e < a.E) {
              const float v = __uint_as_float(r[j]) + s_bias[e];
              a.logits[(int64_t)t * a.E + e] = v;
              top8_push(best, v, e);
            }
          }
        }
      }
      if (ok && t < a.T) top8_emit(best, a.k, a.ids + (int64_t)t * a.k, a.w + (int64_t)t * a.k);
    } else {
      // park this CTA's partial logits in its own (idle) stage buffers
      for (int c0 = 0; c0 < NPAD; c0 += 16) {
        uint32_t r[16];
        if (ok) {
          tmem_ld_32x32b_x16(tb + (uint32_t)c0, r);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int j = 0; j < 16; ++j) r[j] = 0u;
        }
        uint4* dst = reinterpret_cast<uint4*>(park + row * C::kRedStride + c0);
#pragma unroll
        for (int j = 0; j < 4; ++j) dst[j] = make_uint4(r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
      }
      fence_proxy_async_smem();  // the bulk copies below read these rows
    }
  }
  if (a.splits > 1) {
    // Every CTA of the cluster has parked its partials (and so finished with its
    // stage buffers).  CTA `rank` finishes rows [r0, r0 + rows_per) of the tile:
    // each peer sends those rows of its partials into slot `peer` of this CTA's
    // inbox with one bulk copy; then one warp per token adds the partials in rank
    // order (lane l holding experts l, l + 32, ...) and selects.
    constexpr int kPer = NPAD / 32;
    const int r0 = rank * rows_per;
    const int rows_mine = min(rows_per, kRTileM - r0);
    if (threadIdx.x == 0)
      mbar_arrive_expect_tx(inbox_full, (uint32_t)((a.splits - 1) * rows_mine) * C::kRedStride * 4u);
    __syncwarp();
    cluster_arrive();
    cluster_wait();
    if (threadIdx.x == 0) {
      for (int q = 0; q < a.splits; ++q) {
        if (q == rank) continue;
        const int rows_q = min(rows_per, kRTileM - q * rows_per);
        bulk_s2cluster(cluster_addr(inbox + rank * rows_per * C::kRedStride, (uint32_t)q),
                       park + q * rows_per * C::kRedStride, (uint32_t)rows_q * C::kRedStride * 4u,
                       cluster_addr(inbox_full, (uint32_t)q));
      }
    }
    const bool got = __all_sync(0xffffffffu, mbar_wait(inbox_full, 0, a.wait_ns));  // warp-uniform
    if (!got && lane == 0) atomicOr(a.status, kStatusTimeoutEpilogue);
    const int n = min(rows_mine, a.T - t0 - r0);  // tokens this CTA finishes
    for (int lr = warp; got && lr < n; lr += kRWarps) {
      const int t = t0 + r0 + lr;
      // logits, and order-preserving unsigned keys (a NaN logit ranks last; a
      // padding expert or a taken one has key 0, below every real expert)
      float lg[kPer];
      uint32_t key[kPer];
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        const int e = lane + 32 * i;
        float acc = 0.f;
        for (int c = 0; c < a.splits; ++c)
          acc += c == rank ? park[(r0 + lr) * C::kRedStride + e] : inbox[(c * rows_per + lr) * C::kRedStride + e];
        lg[i] = acc + s_bias[e];
        const uint32_t bits = __float_as_uint(isnan(lg[i]) ? -INFINITY : lg[i]);
        key[i] = e < a.E ? ((bits & 0x80000000u) ? ~bits : (bits | 0x80000000u)) : 0u;
        if (e < a.E) a.logits[(int64_t)t * a.E + e] = lg[i];
      }
      // k rounds: the largest key over the warp, then the lowest expert holding it
      Top8 best;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (j < a.k) {
          uint32_t bk = 0u;
          int bi = 0;
#pragma unroll
          for (int i = 0; i < kPer; ++i)
            if (key[i] > bk) {
              bk = key[i];
              bi = i;
            }
          const uint32_t m = __reduce_max_sync(0xffffffffu, bk);
          const uint32_t e = __reduce_min_sync(0xffffffffu, bk == m ? (uint32_t)(lane + 32 * bi) : 0xffffffffu);
#pragma unroll
          for (int i = 0; i < kPer; ++i)
            if (e == (uint32_t)(lane + 32 * i)) key[i] = 0u;
          best.v[j] = __uint_as_float((m & 0x80000000u) ? (m & 0x7fffffffu) : ~m);
          best.i[j] = (int)e;
        }
      }
      // softmax over the selected, lane j holding selection j; the denominator
      // adds the terms in selection order, as the single-CTA path does
      float my_v = -INFINITY;
      int my_i = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (j == lane) {
          my_v = best.v[j];
          my_i = best.i[j];
        }
      const float ex = lane < a.k ? expf(my_v - best.v[0]) : 0.f;
      float den = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float exj = __shfl_sync(0xffffffffu, ex, j);
        if (j < a.k) den += exj;
      }
      if (lane < a.k) {
        a.ids[(int64_t)t * a.k + lane] = my_i;
        a.w[(int64_t)t * a.k + lane] = ex / den;
      }
    }
    // every inbox is complete, so every bulk copy has finished reading its
    // source: only then may a CTA leave
    __syncwarp();
    cluster_arrive();
    cluster_wait();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn_router() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }
  return fn;
}

bool make_bf16_map(CUtensorMap* map, const uint16_t* base, int K, int rows, int box_rows) {
  auto enc = encode_fn_router();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  cuuint32_t box[2] = {kRK, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Clusters of `splits` CTAs of this kernel that the device holds at once (0 if
// none), cached per device.
template <int NPAD>
int max_active_clusters(int splits) {
  static std::mutex mu;
  static int cache[16][kRMaxSplits + 1];
  static bool filled[16][kRMaxSplits + 1];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 16) return 0;
  std::lock_guard<std::mutex> lk(mu);
  if (!filled[dev][splits]) {
    using C = RouterCfg<NPAD>;
    cudaLaunchConfig_t q = {};
    q.gridDim = dim3(splits);
    q.blockDim = dim3(kRThreads);
    q.dynamicSmemBytes = C::kSmem;
    cudaLaunchAttribute qa[1];
    qa[0].id = cudaLaunchAttributeClusterDimension;
    qa[0].val.clusterDim.x = splits;
    qa[0].val.clusterDim.y = 1;
    qa[0].val.clusterDim.z = 1;
    q.attrs = qa;
    q.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, router_tc_kernel<NPAD>, &q) != cudaSuccess) n = 0;
    (void)cudaGetLastError();
    cache[dev][splits] = n;
    filled[dev][splits] = true;
  }
  return cache[dev][splits];
}

// CTAs per token tile and k-slices per CTA.  About one CTA per SM over the grid,
// at least four k-slices per CTA, and every tile's cluster resident at once (a
// tile left for a second wave costs a whole CTA time); no empty split.
template <int NPAD>
void choose_split(RouterArgs& a) {
  const int tiles = (a.T + kRTileM - 1) / kRTileM;
  const int ksl = (a.H + kRK - 1) / kRK;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    sms = 1;
  int ks = RouterCfg<NPAD>::kCanSplit ? std::min(std::min(sms / std::max(tiles, 1), ksl / 4), kRMaxSplits) : 1;
  while (ks > 1 && max_active_clusters<NPAD>(ks) < tiles) --ks;
  ks = std::max(ks, 1);
  a.slices = (ksl + ks - 1) / ks;
  a.splits = (ksl + a.slices - 1) / a.slices;
}

template <int NPAD>
cudaError_t launch_np(const CUtensorMap& mx, const CUtensorMap& mw, RouterArgs a, cudaStream_t s) {
  using C = RouterCfg<NPAD>;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(router_tc_kernel<NPAD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)C::kSmem);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  choose_split<NPAD>(a);
  const int tiles = (a.T + kRTileM - 1) / kRTileM;
  if (a.splits == 1) {
    router_tc_kernel<NPAD><<<tiles, kRThreads, C::kSmem, s>>>(mx, mw, a);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(tiles * a.splits);
  cfg.blockDim = dim3(kRThreads);
  cfg.dynamicSmemBytes = C::kSmem;
  cfg.stream = s;
  cudaLaunchAttribute attrs[1];
  attrs[0].id = cudaLaunchAttributeClusterDimension;
  attrs[0].val.clusterDim.x = a.splits;
  attrs[0].val.clusterDim.y = 1;
  attrs[0].val.clusterDim.z = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, router_tc_kernel<NPAD>, mx, mw, a);
}

}  // namespace

cudaError_t launch_router_tc(const uint16_t* x, const uint16_t* wr, const uint16_t* br, int T, int H, int E, int k,
                             float* logits, int32_t* ids, float* w, uint32_t* status, cudaStream_t s) {
  const int n_pad = (E + 15) / 16 * 16;
  const int np = n_pad <= 64 ? 64 : (n_pad <= 128 ? 128 : 256);
  CUtensorMap mx, mw;
  if (!make_bf16_map(&mx, x, H, T, kRTileM) || !make_bf16_map(&mw, wr, H, E, np)) return cudaErrorInvalidValue;
  RouterArgs a{br, logits, ids, w, status, T, H, E, k, np, 1, 0, wait_limit_ns()};
  switch (np) {
    case 64: return launch_np<64>(mx, mw, a, s);
    case 128: return launch_np<128>(mx, mw, a, s);
    default: return launch_np<256>(mx, mw, a, s);
  }
}

}  // namespace moe

// Router for larger token counts on tcgen05 (kind::f16, bf16 inputs, fp32
// accumulation in tensor memory): logits[T, E] = x[T, H] . Wr[E, H]^T + br, with
// the top-k selection and the softmax over the selected done in the epilogue,
// where each thread holds one token's row of logits.
//
// Routing rule: top-k experts by logit (descending, lower index first on ties),
// then softmax over the k selected ("GPT-OSS-120B on DGX Spark: From MXFP4 to
// NVFP4", section "GPT-OSS-120B Architecture": 128 experts, 4 active per token;
// router weights in BF16).
//
// One CTA per 128-token tile (192 threads): warp 0 streams x and Wr k-slices by
// TMA (128-byte swizzle, 64 bf16 per row), one lane of warp 1 issues the MMAs,
// warps 2..5 read the accumulator (thread = token).  Waits are bounded.
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kRTileM = 128;   // tokens per tile (MMA M)
constexpr int kRK = 64;        // bf16 elements per k-slice (one 128-byte swizzled row)
constexpr int kRStages = 6;

struct RouterArgs {
  const uint16_t* br;
  float* logits;
  int32_t* ids;
  float* w;
  uint32_t* status;
  int T, H, E, k, n_pad;  // n_pad: E rounded up to 16 (MMA N)
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
  static constexpr uint32_t kSmem = 1024 + kRStages * kStage + 256;
  static constexpr uint32_t kTmemCols = NPAD <= 128 ? 128 : 256;
};

template <int NPAD>
__global__ void __launch_bounds__(192, 1)
    router_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                     const RouterArgs a) {
  using C = RouterCfg<NPAD>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + kRStages * C::kA;
  uint64_t* full = reinterpret_cast<uint64_t*>(sB + kRStages * C::kB);
  uint64_t* empty = full + kRStages;
  uint64_t* done = empty + kRStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blockIdx.x * kRTileM;
  const int ksl = (a.H + kRK - 1) / kRK;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kRStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(done, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    int s = 0;
    uint32_t ph = 0;
    int issued = 0;
    for (int kk = 0; kk < ksl; ++kk) {
      if (!mbar_wait_warp(&empty[s], ph ^ 1u, kWaitLimitNs)) {
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
      if (!mbar_wait_warp(&full[st], (uint32_t)((last / kRStages) & 1), 200000000ull) && lane == 0)
        atomicOr(a.status, kStatusTimeoutDrain);
    }
  } else if (warp == 1) {
    int s = 0;
    uint32_t ph = 0;
    const uint32_t idesc = idesc_bf16(kRTileM, NPAD);
    for (int kk = 0; kk < ksl; ++kk) {
      if (!mbar_wait_warp(&full[s], ph, kWaitLimitNs)) {
        if (lane == 0) atomicOr(a.status, kStatusTimeoutMma);
        break;
      }
      tc_fence_after();
      const uint64_t ad = sdesc_sw128(smem_u32(sA + s * C::kA));
      const uint64_t bd = sdesc_sw128(smem_u32(sB + s * C::kB));
      if (elect_one()) {
#pragma unroll
        for (uint32_t j = 0; j < kRK / 16; ++j)  // K = 16 per MMA: 32 bytes along the swizzled row
          umma_bf16(tmem, ad + 2u * j, bd + 2u * j, idesc, (kk | (int)j) != 0);
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
  } else {
    // epilogue: thread = token row of the tile (tmem lane)
    const int q = warp & 3, row = 32 * q + lane, t = t0 + row;
    const bool ok = mbar_wait_warp(done, 0, kWaitLimitNs);
    if (!ok && lane == 0) atomicOr(a.status, kStatusTimeoutEpilogue);
    tc_fence_after();
    // running top-8 in registers, sorted by (logit desc, index asc): experts arrive
    // in ascending order and only a strictly larger logit moves ahead
    float best_v[8];
    int best_i[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      best_v[j] = -INFINITY;
      best_i[j] = 0x7FFFFFFF;
    }
    const uint32_t tb = tmem + ((uint32_t)(32 * q) << 16);
    for (int c0 = 0; c0 < NPAD; c0 += 16) {
      uint32_t r[16];
      if (ok) {
        tmem_ld_32x32b_x16(tb + (uint32_t)c0, r);
        tmem_ld_wait();
      }
      if (ok && t < a.T) {
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int e0 = c0 + j;
          if (e0 < a.E) {
            float v = __uint_as_float(r[j]) + __uint_as_float((uint32_t)a.br[e0] << 16);
            a.logits[(int64_t)t * a.E + e0] = v;
            if (isnan(v)) v = -INFINITY;  // a NaN logit ranks last
            int e = e0;
            const bool any = v > best_v[7] || best_i[7] == 0x7FFFFFFF;
            if (any) {
#pragma unroll
              for (int s2 = 0; s2 < 8; ++s2) {
                const bool take = v > best_v[s2] || best_i[s2] == 0x7FFFFFFF;
                const float tv = best_v[s2];
                const int ti = best_i[s2];
                best_v[s2] = take ? v : tv;
                best_i[s2] = take ? e : ti;
                v = take ? tv : v;
                e = take ? ti : e;
              }
            }
          }
        }
      }
    }
    if (ok && t < a.T) {
      float den = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (j < a.k) den += expf(best_v[j] - best_v[0]);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (j < a.k) {
          a.ids[(int64_t)t * a.k + j] = best_i[j];
          a.w[(int64_t)t * a.k + j] = expf(best_v[j] - best_v[0]) / den;
        }
      }
    }
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

template <int NPAD>
cudaError_t launch_np(const CUtensorMap& mx, const CUtensorMap& mw, const RouterArgs& a, cudaStream_t s) {
  using C = RouterCfg<NPAD>;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(router_tc_kernel<NPAD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)C::kSmem);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  router_tc_kernel<NPAD><<<(a.T + kRTileM - 1) / kRTileM, 192, C::kSmem, s>>>(mx, mw, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_router_tc(const uint16_t* x, const uint16_t* wr, const uint16_t* br, int T, int H, int E, int k,
                             float* logits, int32_t* ids, float* w, uint32_t* status, cudaStream_t s) {
  const int n_pad = (E + 15) / 16 * 16;
  const int np = n_pad <= 64 ? 64 : (n_pad <= 128 ? 128 : 256);
  CUtensorMap mx, mw;
  if (!make_bf16_map(&mx, x, H, T, kRTileM) || !make_bf16_map(&mw, wr, H, E, np)) return cudaErrorInvalidValue;
  RouterArgs a{br, logits, ids, w, status, T, H, E, k, np};
  switch (np) {
    case 64: return launch_np<64>(mx, mw, a, s);
    case 128: return launch_np<128>(mx, mw, a, s);
    default: return launch_np<256>(mx, mw, a, s);
  }
}

}  // namespace moe

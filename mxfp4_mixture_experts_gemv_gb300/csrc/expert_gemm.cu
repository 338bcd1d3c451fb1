// Block-scaled grouped GEMM of the expert MLP on tcgen05 (kind::mxf8f6f4):
// E2M1 weights (A, 128 rows per tile) x E4M3 activations (B, up to BN token rows
// per tile), one E8M0 scale per 32 contraction elements on both sides, fp32
// accumulation in tensor memory.
//
//   gate_up: g = Xp . Wgu[e]^T + bgu[e]; epilogue h = silu(gate) * up, MXFP8(h)
//   down:    y = hq . Wd[e]^T + bd[e];   epilogue adds the bias, writes fp32
//
// The MoE layer as an FP8-activation x FP4-weight grouped GEMM follows "GPT-OSS-
// 120B with MXFP4 on DGX Spark (SM121/GB10)", "What's Included"; that page's
// CUTLASS tile schemes for GB10 are not used.  Here the weights take the MMA M
// slot (swap-AB) because an expert sees few tokens, and the token count of a
// tile sets the MMA N at run time (16..BN, step 16).
//
// Warp roles (192 threads, one CTA per SM, persistent over the tile list):
//   warp 0      TMA producer: weight tile (4-bit, unpacked to the 16-byte
//               aligned smem form), activation tile, both scale atoms
//   warp 1      TMEM allocation; one thread issues tcgen05.cp (scales ->
//               tmem) and tcgen05.mma, commits to mbarriers
//   warps 2..5  epilogue: tcgen05.ld of the accumulator, bias, SwiGLU +
//               MXFP8 (gate_up) or fp32 store (down)
// Every mbarrier wait is bounded; an expired wait records a status bit and the
// roles wind down without hanging.
#include <cudaTypedefs.h>

#include <algorithm>

#include "common.cuh"
#include "ptx.cuh"
#include "quant.cuh"

namespace moe {
namespace {

// One pipeline stage covers kKS consecutive 128-element k-tiles: one TMA box for
// the weights (their tiles are adjacent in the packed layout), one box per k-tile
// for the activations, one bulk copy per operand for the scale atoms, and a single
// commit.  Fewer, larger copies per byte keep the single issuing lanes ahead of HBM.
constexpr int kKS = 2;

template <int BN>
struct GemmCfg {
  static constexpr uint32_t kA1 = kTileM * kTileK;      // 16 KB smem per weight k-tile (4-bit unpacked form)
  static constexpr uint32_t kB1 = BN * kTileK;          // BN rows x 128 B of E4M3 per k-tile
  static constexpr uint32_t kA = kKS * kA1;
  static constexpr uint32_t kB = kKS * kB1;
  static constexpr uint32_t kSF = 2 * kKS * kAtomBytes;  // scale atoms of A (first half) and B
  static constexpr uint32_t kStage = kA + kB + kSF;
  static constexpr uint32_t kXbuf = 64 * 33 * 4;    // gate_up: up-half exchange
  static constexpr uint32_t kBars = 256;
  static constexpr uint32_t kBudget = 227 * 1024 - 1024 - kXbuf - kBars;
  static constexpr int kStages = (kBudget / kStage) > 8 ? 8 : (int)(kBudget / kStage);
  static constexpr uint32_t kSmem = 1024 + kStages * kStage + kBars + kXbuf;
  static_assert(kStages >= 2, "pipeline too shallow");
  static_assert(256 + 8 * kKS * kStages <= 512, "tmem columns");
};

struct GemmParams {
  const uint8_t* sfa;      // weight scale atoms [E][m_tiles][k_tiles][512]
  const float* bias;       // [E][out_rows] fp32 (gate_up rows interleaved)
  const uint8_t* sfb;      // activation scale atoms [tiles][k_tiles][512]
  const int32_t* tiles;    // [0] = count; tile i at 4 + 4i: {expert, row0, rows, 0}
  uint8_t* hq;             // gate_up out: E4M3 codes [TK][I]
  uint8_t* hq_sf;          // gate_up out: scale atoms [tiles][hq_ktiles][512]
  float* y;                // down out: [TK][H]
  uint32_t* status;
  int m_tiles, k_tiles, out_rows, rows_stored, I, H, hq_ktiles;
};

// Where a bounded wait expired: role (1 producer/empty, 2 mma/accumulator, 3 mma/full,
// 4 epilogue), tile and k-step, packed for the second status word.
__device__ __forceinline__ uint32_t wait_site(uint32_t role, int tile, int kt) {
  return (role << 28) | ((uint32_t)min(tile, 0xFFFF) << 12) | (uint32_t)min(kt, 0xFFF);
}

__device__ __forceinline__ uint32_t warp_max_u32(uint32_t v) {
  uint32_t r;
  asm("redux.sync.max.u32 %0, %1, 0xffffffff;" : "=r"(r) : "r"(v));
  return r;
}

template <int BN, bool GATE_UP>
__global__ void __launch_bounds__(192, 1)
    expert_gemm_kernel(const __grid_constant__ CUtensorMap tmA2, const __grid_constant__ CUtensorMap tmA,
                       const __grid_constant__ CUtensorMap tmAt, const __grid_constant__ CUtensorMap tmB,
                       const GemmParams p) {
  using C = GemmCfg<BN>;
  constexpr int S = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + S * C::kA;
  uint8_t* sSF = sB + S * C::kB;
  uint64_t* full = reinterpret_cast<uint64_t*>(sSF + S * C::kSF);
  uint64_t* empty = full + S;
  uint64_t* tfull = empty + S;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  float* xbuf = reinterpret_cast<float*>(sSF + S * C::kSF + C::kBars);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 4);
    }
    mbar_init(drain, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int n_btiles = p.tiles[0];
  const int total = n_btiles * p.m_tiles;
  const int4* tl = reinterpret_cast<const int4*>(p.tiles + 4);

  if (warp == 0) {
    // -------------------------------------------------------------- producer
    // The whole warp walks the schedule (so every operand stays warp-uniform);
    // one elected lane issues the copies.
    if (elect_one()) {
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmA2);
      tma_prefetch_desc(&tmAt);
      tma_prefetch_desc(&tmB);
    }
    __syncwarp();
    int s = 0;
    uint32_t ph = 0;
    int64_t issued = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
      const int b = tile / p.m_tiles, m = tile - b * p.m_tiles;
      const int4 td = tl[b];
      const uint8_t* sfa = p.sfa + ((int64_t)td.x * p.m_tiles + m) * p.k_tiles * kAtomBytes;
      const uint8_t* sfb = p.sfb + (int64_t)b * p.k_tiles * kAtomBytes;
      const int rows_m = min(kTileM, p.rows_stored - m * kTileM);  // 64 for a tail m-tile
      for (int kt = 0; kt < p.k_tiles; kt += kKS) {
        const int nk = min(kKS, p.k_tiles - kt);
        if (!mbar_wait_warp(&empty[s], ph ^ 1u, kWaitLimitNs)) {
          if (lane == 0) {
            atomicOr(p.status, kStatusTimeoutProducer);
            atomicCAS(p.status + 1, 0u, wait_site(1, tile, kt));
          }
          ok = false;
          break;
        }
        if (elect_one()) {
          // the nk weight tiles are rows_m * nk consecutive 64-byte rows: one box
          const int box_rows = rows_m * nk;
          const CUtensorMap* amap = box_rows == 256 ? &tmA2 : (box_rows == 128 ? &tmA : &tmAt);
          mbar_arrive_expect_tx(&full[s], (uint32_t)(box_rows * kTileRowBytes + nk * (C::kB1 + 2 * kAtomBytes)));
          tma_load_2d(sA + s * C::kA, amap, &full[s], 0, (int)tile_row0(td.x, m, kt, p.rows_stored, p.k_tiles));
          for (int j = 0; j < nk; ++j)
            tma_load_2d(sB + s * C::kB + j * C::kB1, &tmB, &full[s], (kt + j) * kTileK, td.y);
          uint8_t* sf = sSF + s * C::kSF;
          bulk_g2s(sf, sfa + kt * kAtomBytes, nk * kAtomBytes, &full[s]);
          bulk_g2s(sf + kKS * kAtomBytes, sfb + kt * kAtomBytes, nk * kAtomBytes, &full[s]);
        }
        __syncwarp();
        ++issued;
        if (++s == S) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
    // Let every copy this warp issued land before the CTA can exit.
    for (int st = 0; st < S && st < issued; ++st) {
      const int64_t last = ((issued - 1 - st) / S) * S + st;
      if (!mbar_wait_warp(&full[st], (uint32_t)((last / S) & 1), 200000000ull) && lane == 0)
        atomicOr(p.status, kStatusTimeoutDrain);
    }
  } else if (warp == 1) {
    // -------------------------------------------------------------- MMA issuer
    // Warp-uniform loop; the elected lane (always the same one, the lowest) issues
    // tcgen05.cp / tcgen05.mma and the commits that track them.
    int s = 0, acc = 0;
    uint32_t ph = 0, aph = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
      const int4 td = tl[tile / p.m_tiles];
      if (!mbar_wait_warp(&tempty[acc], aph ^ 1u, kWaitLimitNs)) {
        if (lane == 0) {
          atomicOr(p.status, kStatusTimeoutMma);
          atomicCAS(p.status + 1, 0u, wait_site(2, tile, 0xFFF));
        }
        break;
      }
      tc_fence_after();
      const uint32_t n_mma = (uint32_t)min(BN, max(16, (td.z + 15) & ~15));
      const uint32_t d_tmem = tmem + (uint32_t)acc * 128u;
      const uint32_t idesc0 = idesc_mxf8f6f4(128, n_mma, 5 /*E2M1*/, 0 /*E4M3*/, 0, 0);
      const int rows_m = min(kTileM, p.rows_stored - (tile % p.m_tiles) * kTileM);
      for (int kt = 0; kt < p.k_tiles; kt += kKS) {
        const int nk = min(kKS, p.k_tiles - kt);
        if (!mbar_wait_warp(&full[s], ph, kWaitLimitNs)) {
          if (lane == 0) {
            atomicOr(p.status, kStatusTimeoutMma);
            atomicCAS(p.status + 1, 0u, wait_site(3, tile, kt));
          }
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sf_t = tmem + 256u + (uint32_t)s * (8u * kKS);
        const uint32_t sf_s = smem_u32(sSF + s * C::kSF);
        const uint32_t a_s = smem_u32(sA + s * C::kA);
        const uint32_t b_s = smem_u32(sB + s * C::kB);
        if (elect_one()) {
          for (int j = 0; j < nk; ++j) {
            const uint32_t sfa_t = sf_t + 8u * j, sfb_t = sfa_t + 4u;
            tmem_cp_32x128b_x4(sfa_t, sdesc_sf_atom(sf_s + j * kAtomBytes));
            tmem_cp_32x128b_x4(sfb_t, sdesc_sf_atom(sf_s + (kKS + j) * kAtomBytes));
            // weight k-tile j starts rows_m rows into the stage (8 or 16 KB, a swizzle-atom multiple)
            const uint64_t ad = sdesc_sw128(a_s + (uint32_t)(j * rows_m * kTileK));
            const uint64_t bd = sdesc_sw128(b_s + j * C::kB1);
#pragma unroll
            for (uint32_t kk = 0; kk < 4; ++kk) {
              // block-scale ids pick byte kk of the scale columns (bits 4-5 for B, 29-30 for A)
              const uint32_t idesc = idesc0 | (kk << 4) | (kk << 29);
              umma_mxf8f6f4(d_tmem, ad + 2u * kk, bd + 2u * kk, idesc, sfa_t, sfb_t, (kt + j + (int)kk) != 0);
            }
          }
          umma_commit(&empty[s]);
        }
        __syncwarp();
        if (++s == S) {
          s = 0;
          ph ^= 1u;
        }
      }
      if (!ok) break;
      if (elect_one()) umma_commit(&tfull[acc]);
      __syncwarp();
      acc ^= 1;
      if (acc == 0) aph ^= 1u;
    }
    // No MMA may still be running when the tensor memory is released.
    if (elect_one()) umma_commit(drain);
    __syncwarp();
    if (!mbar_wait_warp(drain, 0, 200000000ull) && lane == 0) atomicOr(p.status, kStatusTimeoutDrain);
  } else {
    // -------------------------------------------------------------- epilogue
    const int q = warp & 3;              // tmem lane quadrant this warp may read
    const int row = 32 * q + lane;       // tile row == tmem lane
    int acc = 0;
    uint32_t aph = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      const int b = tile / p.m_tiles, m = tile - b * p.m_tiles;
      const int4 td = tl[b];
      const int rows = td.z;
      if (ok) {
        // all lanes take the same decision, so the warp-collective tcgen05.ld stays uniform
        ok = __all_sync(0xffffffffu, mbar_wait(&tfull[acc], aph, kWaitLimitNs));
        if (!ok && lane == 0) {
          atomicOr(p.status, kStatusTimeoutEpilogue);
          atomicCAS(p.status + 1, 0u, wait_site(4, tile, 0));
        }
      }
      tc_fence_after();
      const uint32_t tb = tmem + (uint32_t)acc * 128u + ((uint32_t)(32 * q) << 16);
      if constexpr (GATE_UP) {
        const float bias_v = p.bias[(int64_t)td.x * p.out_rows + m * kTileM + row];
        const int kb = 2 * m + q;  // MX block of the intermediate this gate warp covers
        for (int c0 = 0; c0 < rows; c0 += 32) {
          uint32_t r0[16], r1[16];
          if (ok) {
            tmem_ld_32x32b_x16(tb + (uint32_t)c0, r0);
            tmem_ld_32x32b_x16(tb + (uint32_t)c0 + 16u, r1);
            tmem_ld_wait();
          } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) r0[j] = r1[j] = 0;
          }
          if (q >= 2) {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              xbuf[(row - 64) * 33 + j] = __uint_as_float(j < 16 ? r0[j] : r1[j - 16]) + bias_v;
          }
          named_barrier_sync(1, 128);
          if (q < 2) {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const int n = c0 + j;
              if (n < rows) {
                const float g = __uint_as_float(j < 16 ? r0[j] : r1[j - 16]) + bias_v;
                const float u = xbuf[row * 33 + j];
                const float h = g / (1.0f + expf(-g)) * u;
                const uint32_t amax = warp_max_u32(__float_as_uint(fabsf(h)));
                const int sx = mx_scale_exp(__uint_as_float(amax));
                const uint8_t code = (uint8_t)(cvt_e4m3x2(h * mx_pow2_neg(sx), 0.0f) & 0xFFu);
                if (ok) {
                  p.hq[(int64_t)(td.y + n) * p.I + m * 64 + row] = code;
                  if (lane == 0)
                    p.hq_sf[((int64_t)b * p.hq_ktiles + (kb >> 2)) * kAtomBytes + (n & 31) * 16 + (n >> 5) * 4 +
                            (kb & 3)] = (uint8_t)(sx + 127);
                }
              }
            }
          }
          named_barrier_sync(1, 128);
        }
      } else {
        const int orow = m * kTileM + row;
        const bool rv = orow < p.H;
        const float bias_v = rv ? p.bias[(int64_t)td.x * p.H + orow] : 0.0f;
        for (int c0 = 0; c0 < rows; c0 += 32) {
          uint32_t r0[16], r1[16];
          if (ok) {
            tmem_ld_32x32b_x16(tb + (uint32_t)c0, r0);
            tmem_ld_32x32b_x16(tb + (uint32_t)c0 + 16u, r1);
            tmem_ld_wait();
            if (rv) {
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                const int n = c0 + j;
                if (n < rows) p.y[(int64_t)(td.y + n) * p.H + orow] = __uint_as_float(j < 16 ? r0[j] : r1[j - 16]) + bias_v;
              }
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
      acc ^= 1;
      if (acc == 0) aph ^= 1u;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

// Weights: the tile-contiguous layout seen as a 2-D array of 128-element (64-byte)
// rows of 4-bit codes; one box is one tile (128 rows, or 64 for a tail m-tile),
// unpacked by TMA into the 16-byte-aligned smem form the MMA reads (16 codes in
// each 16-byte chunk, 8 bytes used).
bool make_weight_map(CUtensorMap* map, const uint8_t* base, int64_t total_rows, int box_rows) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)kTileK, (cuuint64_t)total_rows};
  cuuint64_t strides[1] = {(cuuint64_t)kTileRowBytes};
  cuuint32_t box[2] = {kTileK, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 2, const_cast<uint8_t*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Activations: 2-D [rows][K] bytes (E4M3 codes), rows of the grouped order.
bool make_act_map(CUtensorMap* map, const uint8_t* base, int K, int rows, int box_rows) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)K};
  cuuint32_t box[2] = {kTileK, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BN, bool GU>
cudaError_t launch_bn(const CUtensorMap& a2, const CUtensorMap& a, const CUtensorMap& at, const CUtensorMap& b,
                      const GemmParams& p, int grid, cudaStream_t s) {
  using C = GemmCfg<BN>;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(expert_gemm_kernel<BN, GU>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)C::kSmem);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  expert_gemm_kernel<BN, GU><<<grid, 192, C::kSmem, s>>>(a2, a, at, b, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_expert_gemm(bool gate_up, const PackedHeader& h, const uint8_t* packed, const uint8_t* b_rows,
                               int b_rows_total, const uint8_t* b_sf, const int32_t* tiles, int max_tiles,
                               int tile_rows, uint8_t* hq, uint8_t* hq_sf, float* y, uint32_t* status, int num_sms,
                               cudaStream_t s) {
  CUtensorMap ma2, ma, mat, mb;
  GemmParams p{};
  p.tiles = tiles;
  p.status = status;
  p.I = h.I;
  p.H = h.H;
  p.hq_ktiles = h.d_ktiles;
  p.hq = hq;
  p.hq_sf = hq_sf;
  p.y = y;
  p.sfb = b_sf;
  if (gate_up) {
    const int64_t rows = (int64_t)h.E * h.gu_rows_stored * h.gu_ktiles;
    if (!make_weight_map(&ma2, packed + h.off_gu_data, rows, 2 * kTileM)) return cudaErrorInvalidValue;
    if (!make_weight_map(&ma, packed + h.off_gu_data, rows, kTileM)) return cudaErrorInvalidValue;
    if (!make_weight_map(&mat, packed + h.off_gu_data, rows, 64)) return cudaErrorInvalidValue;
    if (!make_act_map(&mb, b_rows, h.H, b_rows_total, tile_rows)) return cudaErrorInvalidValue;
    p.sfa = packed + h.off_gu_sf;
    p.bias = reinterpret_cast<const float*>(packed + h.off_gu_bias);
    p.m_tiles = h.gu_mtiles;
    p.k_tiles = h.gu_ktiles;
    p.out_rows = 2 * h.I;
    p.rows_stored = h.gu_rows_stored;
  } else {
    const int64_t rows = (int64_t)h.E * h.d_rows_stored * h.d_ktiles;
    if (!make_weight_map(&ma2, packed + h.off_d_data, rows, 2 * kTileM)) return cudaErrorInvalidValue;
    if (!make_weight_map(&ma, packed + h.off_d_data, rows, kTileM)) return cudaErrorInvalidValue;
    if (!make_weight_map(&mat, packed + h.off_d_data, rows, 64)) return cudaErrorInvalidValue;
    if (!make_act_map(&mb, b_rows, h.I, b_rows_total, tile_rows)) return cudaErrorInvalidValue;
    p.sfa = packed + h.off_d_sf;
    p.bias = reinterpret_cast<const float*>(packed + h.off_d_bias);
    p.m_tiles = h.d_mtiles;
    p.k_tiles = h.d_ktiles;
    p.out_rows = h.H;
    p.rows_stored = h.d_rows_stored;
  }
  const int grid = (int)std::min<int64_t>(num_sms, (int64_t)max_tiles * p.m_tiles);
  switch (tile_rows) {
    case 16: return gate_up ? launch_bn<16, true>(ma2, ma, mat, mb, p, grid, s) : launch_bn<16, false>(ma2, ma, mat, mb, p, grid, s);
    case 32: return gate_up ? launch_bn<32, true>(ma2, ma, mat, mb, p, grid, s) : launch_bn<32, false>(ma2, ma, mat, mb, p, grid, s);
    case 64: return gate_up ? launch_bn<64, true>(ma2, ma, mat, mb, p, grid, s) : launch_bn<64, false>(ma2, ma, mat, mb, p, grid, s);
    case 128: return gate_up ? launch_bn<128, true>(ma2, ma, mat, mb, p, grid, s) : launch_bn<128, false>(ma2, ma, mat, mb, p, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace moe

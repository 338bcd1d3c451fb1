// The expert MLP for large token counts, with the tokens in the MMA's M slot.
//
// Same layer as the weights-on-M kernel (expert_gemm.cu): E2M1 weights x E4M3
// activations, one E8M0 scale per 32 contraction elements on both sides
// (tcgen05 kind::mxf8f6f4 block-scaled MMA, fp32 accumulation in tensor memory),
// or with MXFP4 activations E2M1 x E2M1 (kind::mxf4, FP4 = true), or NVFP4
// weights and activations (kind::mxf4nvf4, NV = true: UE4M3 scales per 16
// elements and a global scale per weight projection):
//
//   gate_up units: g = Xp . Wgu[e]^T + bgu[e]; epilogue h = silu(gate) * up, MXFP8(h)
//                  (MXFP4(h) or NVFP4(h) with FP4 activations)
//   down units:    y = hq . Wd[e]^T + bd[e]
//
// A unit is one token tile of up to 128 rows (MMA M = 128; rows past the tile are
// computed and never stored) against TWO consecutive 128-row weight tiles of its
// expert (MMA N = 256).  Per contraction step one MMA then reads 16 KB of
// activations and 32 KB of unpacked weights from shared memory for 128 x 256
// outputs, where the weights-on-M layout reads 32 KB for 128 x 128: shared-memory
// traffic per flop, which bounds the block-scaled MMA with unpacked E2M1 operands,
// drops by a quarter.  It also puts gate and up of an intermediate, and the 32
// intermediates of an MX block, in one thread's accumulator columns, so the SwiGLU
// and the MXFP8 quantisation of h run in registers without a transpose.
// The 256-column accumulator leaves no room in tensor memory for a second one and
// the scale columns, so the accumulator is single-buffered: each epilogue warp
// copies its 128 columns to registers and releases the accumulator before the
// SwiGLU, quantisation and stores, so the next unit's MMAs overlap them.
//
// Scheduling is the weights-on-M kernel's: units claimed by running CTAs from one
// counter in increasing order, gate_up units first; a down unit's producer waits
// (bounded) until every gate_up unit of its token tile is counted.
//
// Warp roles (320 threads, one CTA per SM):
//   warp 0      TMA producer
//   warp 1      TMEM allocation, tcgen05.cp / tcgen05.mma issue
//   warps 2..9  epilogue: warp w reads accumulator lanes 32 (w % 4).. (its token
//               rows) and column half (w - 2) / 4 (one of the two weight tiles)
#include <cuda_bf16.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "expert_common.cuh"
#include "ptx.cuh"
#include "quant.cuh"

namespace moe {
namespace {

constexpr int kSwThreads = 320;
constexpr int kSwEpiThreads = 256;
constexpr int kSwQ = 4;                            // tile queue entries
constexpr uint32_t kSwBars = 1024;

// Stage shapes.  MXFP8 activations (kind::mxf8f6f4): 128 token rows of 128 E4M3
// codes (16 KB) and 256 weight rows with the E2M1 codes unpacked to bytes (32 KB),
// four stages.  MXFP4 activations (kind::mxf4) and NVFP4 (kind::mxf4nvf4): both
// operands packed, two codes per byte (8 KB + 16 KB), so twice the stages fit.
// Scale atoms per stage: tokens, then weight tile 0 and 1 (one atom each per
// k-tile; NVFP4 two each, one per 64 elements: tokens a0 a1, tile 0 a0 a1, tile 1
// a0 a1), four tensor-memory columns per atom.
template <bool FP4, bool NV>
struct SwCfg {
  static constexpr int kStages = FP4 ? 8 : 4;
  static constexpr int kSA = NV ? 2 : 1;  // scale atoms per k-tile and 128 rows
  static constexpr uint32_t kRowA = FP4 ? 64 : kTileK;  // bytes of a token row's k-tile
  static constexpr uint32_t kA = kTileM * kRowA;
  static constexpr uint32_t kB = 2 * kTileM * (FP4 ? 64 : kTileK);
  static constexpr uint32_t kSF = 3 * kSA * kAtomBytes;
  static constexpr uint32_t kSfCols = 12 * kSA;
  static constexpr uint32_t kStage = kA + kB + kSF;
  static constexpr uint32_t kSmem = 1024 + kStages * kStage + kSwBars;
  static_assert(!NV || FP4, "NVFP4 operands are packed");
  static_assert(kSmem <= 227 * 1024, "shared memory");
  static_assert(256 + kSfCols * kStages <= 512, "tensor memory columns");
  static_assert((2 * kStages + 3 + 2 * kSwQ) * 8 + 16 + 16 * (kSwQ + 1) <= kSwBars, "barrier area");
};

struct SwapParams {
  const uint8_t* gu_sfa;  // gate_up weight scale atoms [E][gu_mtiles][gu_ktiles][512]
  const float* gu_bias;   // [E][2I] fp32, rows interleaved like the weights
  const uint8_t* d_sfa;   // down weight scale atoms [E][d_mtiles][d_ktiles][512]
  const float* d_bias;    // [E][H] fp32
  const uint8_t* xp_sf;   // gate_up A scale atoms [tiles][gu_ktiles][512]
  uint8_t* hq;            // gate_up out / down A: E4M3 codes [TK][I]
  uint8_t* hq_sf;         // gate_up out / down A: scale atoms [tiles][d_ktiles][512]
  float* y;               // down out: [TK][H]
  const int32_t* tiles;   // [0] = count; tile i at 4 + 4i: {expert, row0, rows, 0}
  int32_t* done_gu;       // [tiles] gate_up units finished per token tile
  int32_t* sched;         // units claimed so far (zero at launch)
  uint32_t* status;
  uint64_t wait_ns;
  int dep_extra;          // failure-detection hook: down units wait for this many extra gate_up units
  int gu_mtiles, gu_ktiles, gu_rows_stored;
  int d_mtiles, d_ktiles, d_rows_stored;
  int I, H;
  int weights_evict_first;
  const float* nv_amax;   // NVFP4 weights: each projection's amax (gate_up, down), for its global scale
};

struct Unit {
  bool gu;
  int b, j;  // token tile, weight tile pair (weight tiles 2j, 2j+1)
};

__device__ __forceinline__ Unit unit_ref(int u, int n_gu, int gp, int dp) {
  Unit r;
  r.gu = u < n_gu;
  const int v = r.gu ? u : u - n_gu;
  const int per = r.gu ? gp : dp;
  r.b = v / per;
  r.j = v - r.b * per;
  return r;
}

template <bool FP4, bool NV>
__global__ void __launch_bounds__(kSwThreads, 1)
    expert_swap_kernel(const __grid_constant__ Maps maps, const SwapParams p) {
  using C = SwCfg<FP4, NV>;
  constexpr int kSwStages = C::kStages, SA = C::kSA;
  constexpr uint32_t kSwA = C::kA, kSwB = C::kB, kSwSF = C::kSF, kSwSfCols = C::kSfCols;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + kSwStages * kSwA;
  uint8_t* sSF = sB + kSwStages * kSwB;
  uint64_t* full = reinterpret_cast<uint64_t*>(sSF + kSwStages * kSwSF);
  uint64_t* empty = full + kSwStages;
  uint64_t* tfull = empty + kSwStages;
  uint64_t* tempty = tfull + 1;
  uint64_t* drain = tempty + 1;
  uint64_t* q_full = drain + 1;
  uint64_t* q_empty = q_full + kSwQ;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(q_empty + kSwQ);
  int4* s_tq = reinterpret_cast<int4*>((reinterpret_cast<uintptr_t>(tmem_slot + 4) + 15) & ~uintptr_t(15));
  int4* s_eq = s_tq + kSwQ;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kSwStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(tfull, 1);
    mbar_init(tempty, kSwEpiThreads / 32);
    mbar_init(drain, 1);
    for (int i = 0; i < kSwQ; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], 2);
    }
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
  if (warp == 0 && elect_one()) {
    tma_prefetch_desc(&maps.gu);
    tma_prefetch_desc(&maps.gut);
    tma_prefetch_desc(&maps.d);
    tma_prefetch_desc(&maps.dt);
    for (int i = 0; i < kActBoxes; ++i) {
      tma_prefetch_desc(&maps.xp[i]);
      tma_prefetch_desc(&maps.hq[i]);
    }
  }
  __syncwarp();
  // Everything above overlaps the previous kernel (programmatic dependent launch).
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int n_btiles = p.tiles[0];
  const int gp = (p.gu_mtiles + 1) / 2, dp = (p.d_mtiles + 1) / 2;  // weight tile pairs per projection
  const int n_gu = n_btiles * gp;
  const int total = n_gu + n_btiles * dp;
  const int4* tl = reinterpret_cast<const int4*>(p.tiles + 4);

  if (warp == 0) {
    // -------------------------------------------------------------- producer
    int s = 0;
    uint32_t ph = 0;
    int64_t issued = 0;
    bool ok = true;
    const uint64_t wpol = l2_policy(p.weights_evict_first != 0);
    int claim = 0;
    if (lane == 0) claim = atomicAdd(p.sched, 1);
    int u = __shfl_sync(0xffffffffu, claim, 0);
    int4 td_next = u < total ? tl[unit_ref(u, n_gu, gp, dp).b] : make_int4(0, 0, 0, 0);
    for (int i = 0; ok; ++i) {
      const int4 td = td_next;
      const int slot = i & (kSwQ - 1);
      if (!mbar_wait_warp(&q_empty[slot], (uint32_t)((i / kSwQ) & 1) ^ 1u, p.wait_ns)) {
        if (lane == 0) {
          atomicOr(p.status, kStatusTimeoutProducer);
          atomicCAS(p.status + 1, 0u, wait_site(6, i, 0));
        }
        break;
      }
      if (lane == 0) {
        s_tq[slot] = make_int4(u < total ? u : -1, td.x, td.y, td.z);
        mbar_arrive(&q_full[slot]);
      }
      __syncwarp();
      if (u >= total) break;
      const Unit r = unit_ref(u, n_gu, gp, dp);
      const int k_tiles = r.gu ? p.gu_ktiles : p.d_ktiles;
      const int m_tiles = r.gu ? p.gu_mtiles : p.d_mtiles;
      const int rows_stored = r.gu ? p.gu_rows_stored : p.d_rows_stored;
      const int m0 = 2 * r.j, nm = min(2, m_tiles - m0);
      const int rw0 = min(kTileM, rows_stored - m0 * kTileM);             // 64 for a tail weight tile
      const int rw1 = nm == 2 ? min(kTileM, rows_stored - (m0 + 1) * kTileM) : 0;
      const uint8_t* sfw = (r.gu ? p.gu_sfa : p.d_sfa) + ((int64_t)td.x * m_tiles + m0) * k_tiles * SA * kAtomBytes;
      const uint8_t* sfx = (r.gu ? p.xp_sf : p.hq_sf) + (int64_t)r.b * k_tiles * SA * kAtomBytes;
      const int bi = min(act_box_index(td.z), kActBoxes - 1);
      const CUtensorMap* amap = r.gu ? &maps.xp[bi] : &maps.hq[bi];
      const CUtensorMap* w0map = r.gu ? (rw0 == kTileM ? &maps.gu : &maps.gut) : (rw0 == kTileM ? &maps.d : &maps.dt);
      const CUtensorMap* w1map = r.gu ? (rw1 == kTileM ? &maps.gu : &maps.gut) : (rw1 == kTileM ? &maps.d : &maps.dt);
      const int w0row = (int)tile_row0(td.x, m0, 0, rows_stored, k_tiles);
      const int w1row = nm == 2 ? (int)tile_row0(td.x, m0 + 1, 0, rows_stored, k_tiles) : 0;
      const uint32_t bytes =
          (uint32_t)(act_box_rows(bi) * C::kRowA + (rw0 + rw1) * kTileRowBytes + (1 + nm) * SA * kAtomBytes);
      // two full weight tiles take the pair boxes
      const bool pair = nm == 2 && rw0 == kTileM && rw1 == kTileM;
      const int claim_st = max(0, k_tiles - 8), fetch_st = max(0, k_tiles - 3);
      int next = total;
      if (!r.gu) {
        // the intermediate of this token tile must be complete (all its gate_up units)
        if (!wait_counter_warp(p.done_gu + r.b, gp + p.dep_extra, p.wait_ns)) {
          if (lane == 0) {
            atomicOr(p.status, kStatusTimeoutProducer);
            atomicCAS(p.status + 1, 0u, wait_site(5, u, 0));
          }
          ok = false;
          break;
        }
        fence_proxy_async_global();  // hq was written by generic stores; TMA reads it
      }
      for (int kt = 0; kt < k_tiles; ++kt) {
        if (kt == claim_st && lane == 0) claim = atomicAdd(p.sched, 1);
        if (kt == fetch_st) {
          next = __shfl_sync(0xffffffffu, claim, 0);
          if (next < total) td_next = tl[unit_ref(next, n_gu, gp, dp).b];
        }
        if (!mbar_wait_warp(&empty[s], ph ^ 1u, p.wait_ns)) {
          if (lane == 0) {
            atomicOr(p.status, kStatusTimeoutProducer);
            atomicCAS(p.status + 1, 0u, wait_site(1, u, kt));
          }
          ok = false;
          break;
        }
        if (elect_one()) {
          mbar_arrive_expect_tx(&full[s], bytes);
          uint8_t* b_s = sB + s * kSwB;
          uint8_t* sf = sSF + s * kSwSF;
          if (pair) {
            // k-tile kt of both weight tiles (rows kt*128.. of tiles m0 and m0+1 of
            // expert e) and their two scale atoms, one box each
            tma_load_4d_hint(b_s, r.gu ? &maps.gup : &maps.dp, &full[s], 0, kt * kTileM, m0, td.x, wpol);
            tma_load_3d_hint(sf + SA * kAtomBytes, r.gu ? &maps.gusf : &maps.dsf, &full[s], 0, kt * SA,
                             td.x * m_tiles + m0, wpol);
          } else {
            tma_load_2d_hint(b_s, w0map, &full[s], 0, w0row + kt * rw0, wpol);
            if (nm == 2)
              tma_load_2d_hint(b_s + rw0 * (FP4 ? kTileRowBytes : kTileK), w1map, &full[s], 0, w1row + kt * rw1, wpol);
            bulk_g2s_hint(sf + SA * kAtomBytes, sfw + kt * SA * kAtomBytes, SA * kAtomBytes, &full[s], wpol);
            if (nm == 2)
              bulk_g2s_hint(sf + 2 * SA * kAtomBytes, sfw + (k_tiles + kt) * SA * kAtomBytes, SA * kAtomBytes,
                            &full[s], wpol);
          }
          tma_load_2d(sA + s * kSwA, amap, &full[s], kt * (int)C::kRowA, td.y);
          bulk_g2s(sf, sfx + kt * SA * kAtomBytes, SA * kAtomBytes, &full[s]);
        }
        __syncwarp();
        ++issued;
        if (++s == kSwStages) {
          s = 0;
          ph ^= 1u;
        }
      }
      u = next;
    }
    // Let every copy this warp issued land before the CTA can exit.
    for (int st = 0; st < kSwStages && st < issued; ++st) {
      const int64_t last = ((issued - 1 - st) / kSwStages) * kSwStages + st;
      if (!mbar_wait_warp(&full[st], (uint32_t)((last / kSwStages) & 1), kDrainLimitNs) && lane == 0)
        atomicOr(p.status, kStatusTimeoutDrain);
    }
  } else if (warp == 1) {
    // -------------------------------------------------------------- MMA issuer
    int s = 0;
    uint32_t ph = 0, aph = 0;
    bool ok = true;
    for (int i = 0; ok; ++i) {
      const int slot = i & (kSwQ - 1);
      if (!mbar_wait_warp(&q_full[slot], (uint32_t)((i / kSwQ) & 1), p.wait_ns)) {
        if (lane == 0) {
          atomicOr(p.status, kStatusTimeoutMma);
          atomicCAS(p.status + 1, 0u, wait_site(7, i, 0));
        }
        break;
      }
      const int4 q = s_tq[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(&q_empty[slot]);
      if (q.x < 0) break;
      const Unit r = unit_ref(q.x, n_gu, gp, dp);
      const int k_tiles = r.gu ? p.gu_ktiles : p.d_ktiles;
      const int m_tiles = r.gu ? p.gu_mtiles : p.d_mtiles;
      const int rows_stored = r.gu ? p.gu_rows_stored : p.d_rows_stored;
      const int m0 = 2 * r.j, nm = min(2, m_tiles - m0);
      const int n_mma = min(kTileM, rows_stored - m0 * kTileM) + (nm == 2 ? min(kTileM, rows_stored - (m0 + 1) * kTileM) : 0);
      // the single accumulator must have been drained by the previous unit's epilogue
      if (!mbar_wait_warp(tempty, aph ^ 1u, p.wait_ns)) {
        if (lane == 0) {
          atomicOr(p.status, kStatusTimeoutMma);
          atomicCAS(p.status + 1, 0u, wait_site(2, q.x, 0xFFF));
        }
        break;
      }
      tc_fence_after();
      uint32_t idesc0 = FP4 ? idesc_mxf8f6f4(128, (uint32_t)n_mma, 1 /*E2M1*/, 1 /*E2M1*/, 0, 0)
                            : idesc_mxf8f6f4(128, (uint32_t)n_mma, 0 /*E4M3*/, 5 /*E2M1*/, 0, 0);
      if (NV) idesc0 &= ~(1u << 23);  // block scales in UE4M3, not UE8M0
      for (int kt = 0; kt < k_tiles; ++kt) {
        if (!mbar_wait_warp(&full[s], ph, p.wait_ns)) {
          if (lane == 0) {
            atomicOr(p.status, kStatusTimeoutMma);
            atomicCAS(p.status + 1, 0u, wait_site(3, q.x, kt));
          }
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sf_t = tmem + 256u + (uint32_t)s * kSwSfCols;
        const uint32_t sf_s = smem_u32(sSF + s * kSwSF);
        if (elect_one()) {
          if constexpr (NV) {
            // columns: token atoms a0 a1 at 0 and 4; for each 64-element half j the
            // B scales of weight rows 0..127 then 128..255 side by side at 8 + 8j
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              tmem_cp_32x128b_x4(sf_t + 4u * j, sdesc_sf_atom(sf_s + j * kAtomBytes));
              tmem_cp_32x128b_x4(sf_t + 8u + 8u * j, sdesc_sf_atom(sf_s + (2 + j) * kAtomBytes));
              if (nm == 2) tmem_cp_32x128b_x4(sf_t + 12u + 8u * j, sdesc_sf_atom(sf_s + (4 + j) * kAtomBytes));
            }
          } else {
            tmem_cp_32x128b_x4(sf_t, sdesc_sf_atom(sf_s));                      // A: token scales
            tmem_cp_32x128b_x4(sf_t + 4u, sdesc_sf_atom(sf_s + kAtomBytes));    // B: weight rows 0..127
            if (nm == 2) tmem_cp_32x128b_x4(sf_t + 8u, sdesc_sf_atom(sf_s + 2 * kAtomBytes));  // rows 128..255
          }
          if constexpr (NV) {
            // two MMAs of K = 64, each with the four 16-element block scales of one atom
            const uint64_t ad = sdesc_sw64(smem_u32(sA + s * kSwA));
            const uint64_t bd = sdesc_sw64(smem_u32(sB + s * kSwB));
#pragma unroll
            for (uint32_t kk = 0; kk < 2; ++kk)
              umma_mxf4nvf4(tmem, ad + 2u * kk, bd + 2u * kk, idesc0, sf_t + 4u * kk, sf_t + 8u + 8u * kk,
                            (kt + (int)kk) != 0);
          } else if constexpr (FP4) {
            // two MMAs of K = 64 (32 bytes of each 64-byte row); MMA kk takes block
            // scales 2kk and 2kk + 1 of each row
            const uint64_t ad = sdesc_sw64(smem_u32(sA + s * kSwA));
            const uint64_t bd = sdesc_sw64(smem_u32(sB + s * kSwB));
#pragma unroll
            for (uint32_t kk = 0; kk < 2; ++kk) {
              const uint32_t idesc = idesc0 | ((2u * kk) << 4) | ((2u * kk) << 29);
              umma_mxf4(tmem, ad + 2u * kk, bd + 2u * kk, idesc, sf_t, sf_t + 4u, (kt + (int)kk) != 0);
            }
          } else {
            const uint64_t ad = sdesc_sw128(smem_u32(sA + s * kSwA));
            const uint64_t bd = sdesc_sw128(smem_u32(sB + s * kSwB));
#pragma unroll
            for (uint32_t kk = 0; kk < 4; ++kk) {
              const uint32_t idesc = idesc0 | (kk << 4) | (kk << 29);
              umma_mxf8f6f4(tmem, ad + 2u * kk, bd + 2u * kk, idesc, sf_t, sf_t + 4u, (kt + (int)kk) != 0);
            }
          }
          umma_commit(&empty[s]);
        }
        __syncwarp();
        if (++s == kSwStages) {
          s = 0;
          ph ^= 1u;
        }
      }
      if (!ok) break;
      if (elect_one()) umma_commit(tfull);
      __syncwarp();
      aph ^= 1u;
    }
    if (elect_one()) umma_commit(drain);
    __syncwarp();
    if (!mbar_wait_warp(drain, 0, kDrainLimitNs) && lane == 0) atomicOr(p.status, kStatusTimeoutDrain);
  } else {
    // -------------------------------------------------------------- epilogue
    // NVFP4 weights carry a global scale per projection (the activations' is 1)
    const float gs_gu = NV ? nvfp4_global_scale(p.nv_amax[0]) : 1.0f;
    const float gs_d = NV ? nvfp4_global_scale(p.nv_amax[1]) : 1.0f;
    const int q = warp & 3;            // tmem lane quadrant this warp may read
    const int half = (warp - 2) >> 2;  // accumulator columns [128 half, 128 half + 128)
    const int n = 32 * q + lane;       // token row of the tile == tmem lane
    const int et = threadIdx.x - 64;   // 0..255
    uint32_t aph = 0;
    bool ok = true;
    for (int i = 0;; ++i) {
      const int slot = i & (kSwQ - 1);
      if (warp == 2) {
        const bool got = mbar_wait_warp(&q_full[slot], (uint32_t)((i / kSwQ) & 1), p.wait_ns);
        if (lane == 0) {
          *s_eq = got ? s_tq[slot] : make_int4(-2, 0, 0, 0);
          if (got) {
            mbar_arrive(&q_empty[slot]);
          } else {
            atomicOr(p.status, kStatusTimeoutEpilogue);
            atomicCAS(p.status + 1, 0u, wait_site(4, i, 0xFFE));
          }
        }
      }
      named_barrier_sync(1, kSwEpiThreads);
      const int4 qe = *s_eq;
      named_barrier_sync(1, kSwEpiThreads);  // every warp has its copy before the next entry overwrites it
      if (qe.x < 0) break;
      const Unit r = unit_ref(qe.x, n_gu, gp, dp);
      const int e = qe.y, row0 = qe.z, rows = qe.w;
      const int m_tiles = r.gu ? p.gu_mtiles : p.d_mtiles;
      const int rows_stored = r.gu ? p.gu_rows_stored : p.d_rows_stored;
      const int mt = 2 * r.j + half;  // this warp's weight tile
      const bool present = mt < m_tiles;
      const int wrows = present ? min(kTileM, rows_stored - mt * kTileM) : 0;
      if (ok) {
        ok = mbar_wait_warp(tfull, aph, p.wait_ns);
        if (!ok && lane == 0) {
          atomicOr(p.status, kStatusTimeoutEpilogue);
          atomicCAS(p.status + 1, 0u, wait_site(4, qe.x, 0));
        }
      }
      tc_fence_after();
      const uint32_t tb = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(kTileM * half);
      const bool store = ok && n < rows;
      // the warp's 128 accumulator columns go to registers first and the accumulator
      // is released at once, so the next unit's MMAs overlap the math and the stores
      uint32_t acc[128];
      if (present && ok) {
#pragma unroll
        for (int c = 0; c < 128; c += 16) tmem_ld_32x32b_x16(tb + (uint32_t)c, *reinterpret_cast<uint32_t(*)[16]>(acc + c));
        tmem_ld_wait();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty);
      if (present && r.gu) {
        // columns 0..63 of this tile are gate rows 64 mt.., 64..127 the matching up rows
        const float* bias = p.gu_bias + (int64_t)e * 2 * p.I + (int64_t)mt * kTileM;
#pragma unroll
        for (int blk = 0; blk < 2; ++blk) {
          float h[32];
          float amax = 0.f;
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const float g = __uint_as_float(acc[32 * blk + c]) * gs_gu + __ldg(bias + 32 * blk + c);
            const float up = __uint_as_float(acc[64 + 32 * blk + c]) * gs_gu + __ldg(bias + 64 + 32 * blk + c);
            h[c] = __fdividef(g, 1.0f + __expf(-g)) * up;  // rel. error ~1e-6, far below an E4M3 step
            amax = fmaxf(amax, fabsf(h[c]));
          }
          const int sx = FP4 ? mx_scale_exp<2>(amax) : mx_scale_exp<8>(amax);
          const float inv = mx_pow2_neg(sx);
          uint32_t pk[8];
          uint32_t nsc[2] = {0u, 0u};  // NVFP4: the E4M3 scales of the two 16-element halves
          if constexpr (NV) {
            uint32_t q0[2], q1[2];
            nsc[0] = nvfp4_block16(h, 1.0f, q0);
            nsc[1] = nvfp4_block16(h + 16, 1.0f, q1);
            pk[0] = q0[0];
            pk[1] = q0[1];
            pk[2] = q1[0];
            pk[3] = q1[1];
          } else if constexpr (FP4) {
#pragma unroll
            for (int c = 0; c < 32; ++c) h[c] *= inv;
#pragma unroll
            for (int c = 0; c < 4; ++c) pk[c] = cvt_e2m1x8(h + 8 * c);
          } else {
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              const uint32_t lo = cvt_e4m3x2(h[4 * c] * inv, h[4 * c + 1] * inv);
              const uint32_t hi = cvt_e4m3x2(h[4 * c + 2] * inv, h[4 * c + 3] * inv);
              pk[c] = lo | (hi << 16);
            }
          }
          if (store) {
            if constexpr (FP4) {
              // 32 codes, two per byte: 16 bytes at intermediate column mt * 64 + 32 blk
              *reinterpret_cast<uint4*>(p.hq + (int64_t)(row0 + n) * (p.I / 2) + mt * 32 + 16 * blk) =
                  make_uint4(pk[0], pk[1], pk[2], pk[3]);
            } else {
              uint4* dst = reinterpret_cast<uint4*>(p.hq + (int64_t)(row0 + n) * p.I + mt * 64 + 32 * blk);
              dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
              dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
            }
            const int kb = 2 * mt + blk;  // MX block of the intermediate
            if constexpr (NV) {
              // 16-element block q = 2 kb + hh: k-tile q / 8, atom (q / 4) % 2, byte q % 4
#pragma unroll
              for (int hh = 0; hh < 2; ++hh) {
                const int qb = 2 * kb + hh;
                uint8_t* wd = p.hq_sf + (((int64_t)r.b * p.d_ktiles + (qb >> 3)) * 2 + ((qb >> 2) & 1)) * kAtomBytes +
                              (n & 31) * 16 + (n >> 5) * 4;
                wd[qb & 3] = (uint8_t)nsc[hh];
                // the last real block also zeroes the scales of the padding blocks after
                // it in its k-tile (zero data past I; their scale must not be a NaN code)
                if (qb == (p.I >> 4) - 1) {
                  for (int jj = (qb & 3) + 1; jj < 4; ++jj) wd[jj] = 0;
                  if (((qb >> 2) & 1) == 0) *reinterpret_cast<uint32_t*>(wd + kAtomBytes) = 0u;
                }
              }
            } else {
              uint8_t* wd = p.hq_sf + ((int64_t)r.b * p.d_ktiles + (kb >> 2)) * kAtomBytes + (n & 31) * 16 + (n >> 5) * 4;
              wd[kb & 3] = (uint8_t)(sx + 127);
              // the last real block also sets the padding blocks of its word (zero data
              // past I; their scale must not be the NaN code)
              if (kb == (p.I >> 5) - 1)
                for (int jj = (kb & 3) + 1; jj < 4; ++jj) wd[jj] = 127;
            }
          }
        }
      } else if (present && store) {
        const float* bias = p.d_bias + (int64_t)e * p.H + (int64_t)mt * kTileM;
        float* yrow = p.y + (int64_t)(row0 + n) * p.H + (int64_t)mt * kTileM;
#pragma unroll
        for (int c0 = 0; c0 < 128; c0 += 32) {
          if (c0 < wrows) {
#pragma unroll
            for (int c = 0; c < 32; c += 4) {
              const int f = mt * kTileM + c0 + c;
              if (f < p.H) {  // H is a multiple of 32: whole groups of four are in or out
                float4 o;
                o.x = __uint_as_float(acc[c0 + c]) * gs_d + __ldg(bias + c0 + c);
                o.y = __uint_as_float(acc[c0 + c + 1]) * gs_d + __ldg(bias + c0 + c + 1);
                o.z = __uint_as_float(acc[c0 + c + 2]) * gs_d + __ldg(bias + c0 + c + 2);
                o.w = __uint_as_float(acc[c0 + c + 3]) * gs_d + __ldg(bias + c0 + c + 3);
                *reinterpret_cast<float4*>(yrow + c0 + c) = o;
              }
            }
          }
        }
      }
      if (r.gu) {
        // every hq byte of this unit is stored: count it
        named_barrier_sync(1, kSwEpiThreads);
        if (et == 0 && ok) red_add_release_gpu(p.done_gu + r.b, 1);
      }
      aph ^= 1u;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

// One k-tile of two consecutive 128-row weight tiles of an expert as one box: the
// tile-contiguous layout seen as 4-D {128 codes, row within the m-tile (k-tile kt
// at rows 128 kt..), m-tile, expert}; full m-tiles only (a 64-row tail tile is read
// by the 2-D maps).
bool make_weight_pair_map(CUtensorMap* map, const uint8_t* base, int E, int rows_stored, int k_tiles, bool packed) {
  auto enc = encode_fn();
  if (!enc) return false;
  // unpacked by TMA for kind::mxf8f6f4 (128 codes per row, 128-byte swizzle), or the
  // packed bytes for kind::mxf4 (64 bytes per row, 64-byte swizzle)
  const cuuint64_t inner = packed ? (cuuint64_t)kTileRowBytes : (cuuint64_t)kTileK;
  cuuint64_t dims[4] = {inner, (cuuint64_t)kTileM * k_tiles, (cuuint64_t)(rows_stored / kTileM), (cuuint64_t)E};
  cuuint64_t strides[3] = {(cuuint64_t)kTileRowBytes, (cuuint64_t)kTileM * k_tiles * kTileRowBytes,
                           (cuuint64_t)rows_stored * k_tiles * kTileRowBytes};
  cuuint32_t box[4] = {(cuuint32_t)inner, kTileM, 2, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(map, packed ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 4,
             const_cast<uint8_t*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             packed ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The scale atoms [E][m_tiles][k_tiles][atoms][512 bytes] (atoms = 1, or 2 for
// NVFP4) as 3-D {128 words, (k-tile, atom), (expert, m-tile)}: a box holds the atoms
// of one k-tile of two consecutive m-tiles.
bool make_scale_pair_map(CUtensorMap* map, const uint8_t* base, int E, int m_tiles, int k_tiles, int atoms) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)(kAtomBytes / 4), (cuuint64_t)k_tiles * atoms, (cuuint64_t)E * m_tiles};
  cuuint64_t strides[2] = {(cuuint64_t)kAtomBytes, (cuuint64_t)k_tiles * atoms * kAtomBytes};
  cuuint32_t box[3] = {kAtomBytes / 4, (cuuint32_t)atoms, 2};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<uint8_t*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool expert_swap_supported(const PackedHeader& h) {
  // the weight tiles of a projection pair up, a 64-row tail tile only as the last
  return h.gu_rows_stored % kTileM == 0;
}

cudaError_t launch_expert_swap(const PackedHeader& h, const uint8_t* packed, const ExpertMlpBuffers& b, int T, int k,
                               int max_tiles, int num_sms, int fmt, cudaStream_t s) {
  if (fmt != kActMxfp8 && fmt != kActMxfp4 && fmt != kActNvfp4) return cudaErrorInvalidValue;
  const bool fp4 = fmt != kActMxfp8, nv = fmt == kActNvfp4;
  const int atoms = nv ? 2 : 1;
  const int TK = T * k;
  struct Key {
    const uint8_t *packed, *xp, *hq;
    int E, H, I, TK, fmt;
    bool operator==(const Key& o) const {
      return packed == o.packed && xp == o.xp && hq == o.hq && E == o.E && H == o.H && I == o.I && TK == o.TK &&
             fmt == o.fmt;
    }
  };
  static std::mutex mu;
  static Key keys[32];
  static Maps cache[32];
  static int n_cached = 0, next_slot = 0;
  const Key key{packed, b.xp, b.hq, h.E, h.H, h.I, TK, fmt};
  Maps m;
  bool hit = false;
  {
    std::lock_guard<std::mutex> lk(mu);
    for (int i = 0; i < n_cached; ++i)
      if (keys[i] == key) {
        m = cache[i];
        hit = true;
        break;
      }
  }
  if (!hit) {
    m = Maps{};
    const int64_t gu_rows = (int64_t)h.E * h.gu_rows_stored * h.gu_ktiles;
    const int64_t d_rows = (int64_t)h.E * h.d_rows_stored * h.d_ktiles;
    auto wmap = fp4 ? make_weight_map_packed : make_weight_map;
    if (!wmap(&m.gu, packed + h.off_gu_data, gu_rows, kTileM) || !wmap(&m.gut, packed + h.off_gu_data, gu_rows, 64) ||
        !wmap(&m.d, packed + h.off_d_data, d_rows, kTileM) || !wmap(&m.dt, packed + h.off_d_data, d_rows, 64))
      return cudaErrorInvalidValue;
    // pair boxes exist for projections with at least two full 128-row weight tiles
    // (the only ones whose units take them)
    if (h.gu_rows_stored >= 2 * kTileM &&
        (!make_weight_pair_map(&m.gup, packed + h.off_gu_data, h.E, h.gu_rows_stored, h.gu_ktiles, fp4) ||
         !make_scale_pair_map(&m.gusf, packed + h.off_gu_sf, h.E, h.gu_mtiles, h.gu_ktiles, atoms)))
      return cudaErrorInvalidValue;
    if (h.d_rows_stored >= 2 * kTileM &&
        (!make_weight_pair_map(&m.dp, packed + h.off_d_data, h.E, h.d_rows_stored, h.d_ktiles, fp4) ||
         !make_scale_pair_map(&m.dsf, packed + h.off_d_sf, h.E, h.d_mtiles, h.d_ktiles, atoms)))
      return cudaErrorInvalidValue;
    for (int i = 0; i < kActBoxes; ++i) {
      const int rows = act_box_rows(i);
      // MXFP4 rows hold two codes per byte; a box is one k-tile (64 bytes) of a row
      if (!make_act_map(&m.xp[i], b.xp, fp4 ? h.H / 2 : h.H, TK, rows, fp4) ||
          !make_act_map(&m.hq[i], b.hq, fp4 ? h.I / 2 : h.I, TK, rows, fp4))
        return cudaErrorInvalidValue;
    }
    std::lock_guard<std::mutex> lk(mu);
    keys[next_slot] = key;
    cache[next_slot] = m;
    next_slot = (next_slot + 1) % 32;
    if (n_cached < 32) ++n_cached;
  }
  SwapParams p{};
  p.gu_sfa = packed + h.off_gu_sf;
  p.gu_bias = reinterpret_cast<const float*>(packed + h.off_gu_bias);
  p.d_sfa = packed + h.off_d_sf;
  p.d_bias = reinterpret_cast<const float*>(packed + h.off_d_bias);
  p.xp_sf = b.xp_sf;
  p.hq = b.hq;
  p.hq_sf = b.hq_sf;
  p.y = b.y;
  p.tiles = b.tiles;
  p.done_gu = b.done_gu;
  p.sched = b.sched;
  p.status = b.status;
  p.wait_ns = wait_limit_ns();
  p.dep_extra = (debug_hold_waits() & MOE_DEBUG_HOLD_DOWN_UNITS) ? 1 : 0;
  p.gu_mtiles = h.gu_mtiles;
  p.gu_ktiles = h.gu_ktiles;
  p.gu_rows_stored = h.gu_rows_stored;
  p.d_mtiles = h.d_mtiles;
  p.d_ktiles = h.d_ktiles;
  p.d_rows_stored = h.d_rows_stored;
  p.I = h.I;
  p.H = h.H;
  p.weights_evict_first = (int64_t)T * k <= (int64_t)h.E * kTileM;
  p.nv_amax = reinterpret_cast<const float*>(packed + kAmaxOffset);
  static bool attr[3] = {false, false, false};
  const uint32_t smem = nv ? SwCfg<true, true>::kSmem : fp4 ? SwCfg<true, false>::kSmem : SwCfg<false, false>::kSmem;
  auto kernel = nv ? expert_swap_kernel<true, true> : fp4 ? expert_swap_kernel<true, false>
                                                          : expert_swap_kernel<false, false>;
  if (!attr[fmt]) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr[fmt] = true;
  }
  const int units = max_tiles * ((h.gu_mtiles + 1) / 2 + (h.d_mtiles + 1) / 2);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)std::max(1, std::min(num_sms, units)));
  cfg.blockDim = dim3(kSwThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  // programmatic dependent launch, as for the weights-on-M kernel: units are
  // claimed at run time by running CTAs, so any subset of resident CTAs finishes
  cudaLaunchAttribute attrs[1];
  attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, m, p);
}

}  // namespace moe

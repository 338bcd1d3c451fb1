// The expert MLP of the MoE layer in one persistent kernel on tcgen05
// (kind::mxf8f6f4 block-scaled MMA): E2M1 weights (A, 128 rows per tile) x E4M3
// activations (B, up to BN token rows per tile), one E8M0 scale per 32
// contraction elements on both sides, fp32 accumulation in tensor memory.
// The FP4 x FP4 variant (FP4 = true) quantises the activations to MXFP4 as well
// and runs kind::mxf4 on packed E2M1 operands ("GPT-OSS-120B with MXFP4 on DGX
// Spark (SM121/GB10)", "Performance Optimizations": native FP4 x FP4
// block-scale MMA); both operands then stay packed in shared memory.
//
//   gate_up tiles: g = Xp . Wgu[e]^T + bgu[e]; epilogue h = silu(gate) * up, MXFP8(h)
//   down tiles:    y = hq . Wd[e]^T + bd[e];   epilogue writes y, then the
//                  routing-weighted combine of every (token, 128-feature block)
//                  whose k contributions are complete
//
// The MoE layer as an FP8-activation x FP4-weight grouped GEMM follows "GPT-OSS-
// 120B with MXFP4 on DGX Spark (SM121/GB10)", "What's Included"; that page's
// CUTLASS tile schemes for GB10 are not used.  Here the weights take the MMA M
// slot (swap-AB) because an expert sees few tokens, and the token count of a
// tile sets the MMA N at run time (16..BN, step 16).
//
// One launch walks the tile list: every gate_up tile first, then every down
// tile.  A down tile needs the whole intermediate of its token rows, i.e. all
// gate_up m-tiles of the same token tile; their epilogues count themselves in a
// per-token-tile counter that the down tile's producer waits on (acquire) before
// it streams hq.  Its weights do not depend on hq, so the producer issues the
// weight copies of its first stages before that wait.  Every unit is taken by a
// running CTA from one claim counter, in increasing order: the first down unit
// is claimed only after every gate_up unit has been claimed, so every unit a
// down unit waits for is owned by a CTA that is already running and never waits
// itself (whether or not all CTAs of the grid are resident at once).
//
// Warp roles (192 threads, one CTA per SM):
//   warp 0      TMA producer (whole warp walks the schedule, one elected lane issues)
//   warp 1      TMEM allocation; elected lane issues tcgen05.cp / tcgen05.mma / commits
//   warps 2..5  epilogue: tcgen05.ld of the accumulator, bias, SwiGLU + MXFP8 (gate_up)
//               or fp32 y + combine (down)
// Every wait (mbarrier or global counter) is bounded; an expired wait records a
// status bit and the roles wind down without hanging.
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "expert_common.cuh"
#include "ptx.cuh"
#include "quant.cuh"

namespace moe {
namespace {

// One pipeline stage covers kKS consecutive 128-element k-tiles: weight boxes of
// up to 256 rows (the k-tiles of a weight tile are adjacent in the packed
// layout), one box per k-tile for the activations, one bulk copy per operand for
// the scale atoms, and a single commit.  Fewer, larger copies per byte stream
// faster (measured with the same copies alone: three stages of four k-tiles
// reach 6.8 TB/s where six stages of two reach 5.9 TB/s), so the smallest token
// tile, whose activation slots are small, takes four k-tiles per stage.
// k-tiles per pipeline stage for token tiles of bn rows (the kernel's stage layout
// and the host's k-tile-plane activation boxes both follow it).  Measured at
// decode (8-row tiles): unpacked E2M1 weights (32 KB of smem per 4 k-tiles) run
// best with three stages of four k-tiles (T = 4: 50.0 us against 51.2 with two of
// six, 54 with two of five, 52.6 with four of three, 58.2 with six of two); packed
// FP4 operands (half the smem) with stages of six (FP4 x FP4 49.3 against 50.9 us,
// NVFP4 69.1 against 71.9).  FP4 stages hold an even number of k-tiles: the MXFP4
// activation boxes span two k-tiles (256 elements, 128-byte rows).
constexpr int stage_ktiles_for(int bn, bool fp4) { return bn == 8 ? (fp4 ? 6 : 4) : (bn <= 32 ? (fp4 ? 4 : 3) : 2); }

// Shared-memory bytes of one 128-element k-tile row of an operand: 128 for E4M3
// and for E2M1 weights unpacked by TMA for kind::mxf8f6f4 (16 codes per 16-byte
// chunk), 64 for packed E2M1 (kind::mxf4).
template <bool FP4>
constexpr uint32_t smem_row_bytes() { return FP4 ? 64u : 128u; }

// Tiles are claimed from a global counter by the producer warp and handed to the
// MMA and epilogue warps through a small queue in shared memory.
constexpr int kTileQ = 4;

template <int BN, bool FP4, bool NV>
struct GemmCfg {
  static_assert(FP4 || !NV, "NVFP4 operands are FP4");
  static constexpr int kKS = stage_ktiles_for(BN, FP4);
  static constexpr int kSfAtoms = NV ? 2 : 1;  // scale atoms per k-tile and operand (16- or 32-element blocks)
  static constexpr uint32_t kRow = smem_row_bytes<FP4>();
  // MXFP4 activations (kind::mxf4): 128-byte shared-memory rows of 256 elements, one
  // TMA box row per two k-tiles (TMA lands box rows at a fixed rate per SM, whatever
  // their width); NVFP4 keeps 64-byte rows, one per k-tile
  static constexpr bool kWideB = FP4 && !NV;
  static constexpr uint32_t kBRow = kWideB ? 128u : kRow;
  static constexpr int kBPlanes = kWideB ? kKS / 2 : kKS;  // activation planes of a grouped-x stage
  static_assert(!kWideB || kKS % 2 == 0, "MXFP4 activation stages span whole pairs of k-tiles");
  static constexpr uint32_t kA1 = kTileM * kRow;        // smem per weight k-tile (16 KB unpacked, 8 KB packed)
  static constexpr uint32_t kB1 = BN * kRow;            // BN activation rows per k-tile
  static constexpr uint32_t kA = kKS * kA1;
  static constexpr uint32_t kB = kKS * kB1;
  static constexpr uint32_t kSF = 2 * kKS * kSfAtoms * kAtomBytes;  // scale atoms of A (first half) and B
  static constexpr uint32_t kSfCols = 8 * kKS * kSfAtoms;            // tmem columns of one stage's scales
  static constexpr uint32_t kStage = kA + kB + kSF;
  // gate_up epilogue: accumulator chunks of kCW token columns are transposed
  // through shared memory (a token tile of at most 16 rows needs one 16-wide chunk)
  static constexpr int kCW = BN >= 32 ? 32 : 16;
  static constexpr uint32_t kXbuf = 128 * (kCW + 1) * 4;
  static_assert(kXbuf >= BN * 16 * 4, "combine staging lives in the transpose buffer");
  static constexpr uint32_t kBars = 1024;
  static constexpr uint32_t kBudget = 227 * 1024 - 1024 - kXbuf - kBars;
  static constexpr int kStagesSmem = (kBudget / kStage) > 8 ? 8 : (int)(kBudget / kStage);
  static constexpr int kStagesTmem = (int)(256 / kSfCols);
  static constexpr int kStages = kStagesSmem < kStagesTmem ? kStagesSmem : kStagesTmem;
  static constexpr uint32_t kSmem = 1024 + kStages * kStage + kBars + kXbuf;
  static_assert(kStages >= 2, "pipeline too shallow");
  static_assert(256 + kSfCols * kStages <= 512, "tmem columns");
  // barriers (stages, accumulators, drain, tile queue), tmem slot, tile queue, combine list
  static_assert((2 * kStages + 5 + 2 * kTileQ) * 8 + 16 + 16 * (kTileQ + 1) + 4 * (BN + 1) + 16 <= kBars, "barrier area");
};

struct MlpParams {
  const uint8_t* gu_sfa;     // gate_up weight scale atoms [E][gu_mtiles][gu_ktiles][512]
  const float* gu_bias;      // [E][2I] fp32, rows interleaved like the weights
  const uint8_t* d_sfa;      // down weight scale atoms [E][d_mtiles][d_ktiles][512]
  const float* d_bias;       // [E][H] fp32
  const uint8_t* xp_sf;      // gate_up B scale atoms [tiles][gu_ktiles][512]
  uint8_t* hq;               // gate_up out / down B: E4M3 codes [TK][I]
  uint8_t* hq_sf;            // gate_up out / down B: scale atoms [tiles][d_ktiles][512]
  float* y;                  // down out: [TK][H]
  uint16_t* out;             // combine out: bf16 [T][H]
  const int32_t* tiles;      // [0] = count; tile i at 4 + 4i: {expert, row0, rows, 0}
  const int32_t* sorted_rows;  // grouped position -> flat (t*k + j)
  const int32_t* inv_pos;      // flat (t*k + j) -> grouped position
  const float* topk_w;         // [T][k]
  int32_t* done_gu;          // [tiles] gate_up m-tiles finished per token tile
  int32_t* done_tok;         // [T][d_mtiles] down contributions finished per (token, feature block)
  int32_t* sched;            // tiles claimed so far (zero at launch)
  uint32_t* status;
  uint64_t wait_ns;          // limit of every bounded wait
  int dep_extra;             // failure-detection hook: down units wait for this many extra gate_up tiles
  int gu_mtiles, gu_ktiles, gu_rows_stored;
  int d_mtiles, d_ktiles, d_rows_stored;
  int I, H, k;
  int weights_evict_first;  // weights are read once per forward: let them leave L2 first
  int fused_combine;  // the down epilogue also combines the k slots of completed tokens
  const PackedHeader* hdr;   // the packed buffer's header, checked against what this launch expects
  PackedHeader want;         // (magic, version, dims and weight format)
  int dense;                 // a dense linear: down units only, B = the quantised input, bf16 out + bias
  int max_tiles;             // capacity of the tile list (entries past its count are not meaningful)
  int TK;                    // grouped rows (token, slot pairs)
  const int32_t* route_flags;  // routing still running: [0] tile list published, [1] CTAs done
  int route_ctas;              // the count [1] reaches; 0 = the routing grid completed first
};

struct TileRef {
  bool gu;      // gate_up tile (else down)
  int b, m;     // token tile, weight m-tile
};

__device__ __forceinline__ TileRef tile_ref(int tile, int n_gu, const MlpParams& p) {
  TileRef r;
  r.gu = tile < n_gu;
  if (r.gu) {
    r.b = tile / p.gu_mtiles;
    r.m = tile - r.b * p.gu_mtiles;
  } else {
    const int t = tile - n_gu;
    r.b = t / p.d_mtiles;
    r.m = t - r.b * p.d_mtiles;
  }
  return r;
}

template <int BN, bool FP4, bool NV>
__global__ void __launch_bounds__(192, 1)
    expert_mlp_kernel(const __grid_constant__ Maps maps, const MlpParams p) {
  using C = GemmCfg<BN, FP4, NV>;
  constexpr int SA = C::kSfAtoms;
  constexpr int kKS = C::kKS;
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
  uint64_t* q_full = drain + 1;  // [kTileQ] tile queue: entry written
  uint64_t* q_empty = q_full + kTileQ;  // [kTileQ] entry read by the MMA warp and by the epilogue
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(q_empty + kTileQ);
  int4* s_tq = reinterpret_cast<int4*>((reinterpret_cast<uintptr_t>(tmem_slot + 4) + 15) & ~uintptr_t(15));
  int4* s_eq = s_tq + kTileQ;  // the epilogue's copy of its current entry
  int* comb_list = reinterpret_cast<int*>(s_eq + 1);  // [BN + 1]: count, tokens to combine
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
    for (int i = 0; i < kTileQ; ++i) {
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
    tma_prefetch_desc(&maps.gu2);
    tma_prefetch_desc(&maps.gu);
    tma_prefetch_desc(&maps.gut);
    tma_prefetch_desc(&maps.d2);
    tma_prefetch_desc(&maps.d);
    tma_prefetch_desc(&maps.dt);
    for (int i = 0; i < kActBoxes && act_box_rows(i) <= BN; ++i) {
      tma_prefetch_desc(&maps.xp[i]);
      tma_prefetch_desc(&maps.hq[i]);
    }
  }
  __syncwarp();
  // The packed buffer was written before the previous kernel began, so its header
  // can be read while that kernel runs.  A buffer of other dims or another weight
  // format runs no unit.
  const PackedHeader& hd = *p.hdr;
  const bool hdr_ok = hd.magic == p.want.magic && hd.version == p.want.version && hd.E == p.want.E &&
                      hd.H == p.want.H && hd.I == p.want.I && hd.wfmt == p.want.wfmt;
  // Everything above overlaps the previous kernel (programmatic dependent
  // launch).  Its tile list is read only after that grid completes, or, for a
  // routing kernel that publishes its results while it runs, after its first flag
  // (the grouped activations then wait for the second, in the producer).
  // Every counter of the forward, the claim counter included, was cleared before
  // this kernel could start (by a memset or a kernel earlier in the stream, or by
  // the cluster routing kernel before it let this one launch), so the first claim
  // is taken now, while the routing results are still on their way.
  int first_claim = 0;
  if (warp == 0 && lane == 0) first_claim = atomicAdd(p.sched, 1);
  __shared__ int s_routed;
  bool routed = true;
  if (p.route_ctas == 0) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
  } else {
    if (threadIdx.x == 0) {
      bool got = ld_acquire_gpu(p.route_flags) != 0;
      const uint64_t t0 = global_timer_ns();
      while (!got && global_timer_ns() - t0 <= p.wait_ns) got = ld_acquire_gpu(p.route_flags) != 0;
      if (!got) {
        atomicOr(p.status, kStatusTimeoutProducer);
        atomicCAS(p.status + 1, 0u, wait_site(9, 0, 0));
      }
      s_routed = got ? 1 : 0;
    }
    __syncthreads();
    routed = s_routed != 0;
  }
  if (!hdr_ok && threadIdx.x == 0) atomicOr(p.status, kStatusBadWeights);
  const int n_btiles = hdr_ok && routed ? p.tiles[0] : 0;
  const int n_gu = n_btiles * p.gu_mtiles;
  const int total = n_gu + n_btiles * p.d_mtiles;
  const int4* tl = reinterpret_cast<const int4*>(p.tiles + 4);

  if (warp == 0) {
    // -------------------------------------------------------------- producer
    int s = 0;
    uint32_t ph = 0;
    int64_t issued = 0;
    bool ok = true;
    const uint64_t wpol = l2_policy(p.weights_evict_first != 0);
    // Units are claimed from the counter in increasing order, the first one before
    // the routing results are read; later claims are issued several stages before the current
    // unit's last loads and their descriptor fetched two stages before them, so
    // neither round trip stalls the copies.
    // The first claim and the first tile-list entries travel together: lane i
    // loads entry i, so a first unit among them needs no further round trip.
    bool xp_ready = p.route_ctas == 0;  // the grouped activations may be read
    int claim = first_claim;
    const int4 pre = lane < min(p.max_tiles, 32) ? tl[lane] : make_int4(0, 0, 0, 0);
    int tile = __shfl_sync(0xffffffffu, claim, 0);
    int4 td_next = make_int4(0, 0, 0, 0);
    if (tile < total) {
      const int b0 = tile_ref(tile, n_gu, p).b;
      if (b0 < 32) {
        td_next.x = __shfl_sync(0xffffffffu, pre.x, b0);
        td_next.y = __shfl_sync(0xffffffffu, pre.y, b0);
        td_next.z = __shfl_sync(0xffffffffu, pre.z, b0);
        td_next.w = __shfl_sync(0xffffffffu, pre.w, b0);
      } else {
        td_next = tl[b0];
      }
    }
    for (int i = 0; ok; ++i) {
      const int4 td = td_next;
      // hand the tile (or the end, -1) to the MMA and epilogue warps
      const int slot = i & (kTileQ - 1);
      if (!mbar_wait_warp(&q_empty[slot], (uint32_t)((i / kTileQ) & 1) ^ 1u, p.wait_ns)) {
        if (lane == 0) {
          atomicOr(p.status, kStatusTimeoutProducer);
          atomicCAS(p.status + 1, 0u, wait_site(6, i, 0));
        }
        break;
      }
      if (lane == 0) {
        s_tq[slot] = make_int4(tile < total ? tile : -1, td.x, td.y, td.z);
        mbar_arrive(&q_full[slot]);
      }
      __syncwarp();
      if (tile >= total) break;
      const TileRef r = tile_ref(tile, n_gu, p);
      const int k_tiles = r.gu ? p.gu_ktiles : p.d_ktiles;
      const int n_st = (k_tiles + kKS - 1) / kKS;
      const int claim_st = max(0, n_st - 6), fetch_st = max(0, n_st - 2);
      int next = total;
      const int m_tiles = r.gu ? p.gu_mtiles : p.d_mtiles;
      const int rows_stored = r.gu ? p.gu_rows_stored : p.d_rows_stored;
      const uint8_t* sfa = (r.gu ? p.gu_sfa : p.d_sfa) + ((int64_t)td.x * m_tiles + r.m) * k_tiles * SA * kAtomBytes;
      const uint8_t* sfb = (r.gu ? p.xp_sf : p.hq_sf) + (int64_t)r.b * k_tiles * SA * kAtomBytes;
      const int rows_m = min(kTileM, rows_stored - r.m * kTileM);  // 64 for a tail m-tile
      const int bi = min(act_box_index(td.z), kActBoxes - 1);
      const uint32_t b_bytes = (uint32_t)act_box_rows(bi) * C::kBRow;  // one box plane
      const int row0_unit = (int)tile_row0(td.x, r.m, 0, rows_stored, k_tiles);
      // weight (A) copies of stage slot `ss`: the nk weight tiles are rows_m * nk
      // consecutive 64-byte rows (128 bytes each in shared memory when unpacked),
      // boxes of 256, 128 or 64 rows, then their scale atoms
      auto issue_a = [&](int ss, int kt, int nk) {
        const int a_rows = rows_m * nk;
        const int row0 = row0_unit + kt * rows_m;
        if (a_rows == 512) {  // two 256-row planes in one box
          tma_load_3d_hint(sA + ss * C::kA, r.gu ? &maps.gu4 : &maps.d4, &full[ss], 0, row0, 0, wpol);
          return;
        }
        for (int off = 0; off < a_rows;) {
          const int c = a_rows - off >= 256 ? 256 : a_rows - off >= 128 ? 128 : 64;
          const CUtensorMap* amap = r.gu ? (c == 256 ? &maps.gu2 : (c == 128 ? &maps.gu : &maps.gut))
                                         : (c == 256 ? &maps.d2 : (c == 128 ? &maps.d : &maps.dt));
          tma_load_2d_hint(sA + ss * C::kA + off * C::kRow, amap, &full[ss], 0, row0 + off, wpol);
          off += c;
        }
      };
      // activation (B) copies of stage slot `ss` covering k-tiles kt..kt+nk-1: one box
      // of the stage's planes (plane j, one k-tile or two for MXFP4, at j * box rows) of
      // grouped x or of the intermediate; a short last stage reads planes past K, which
      // TMA fills with zeros, and a last row's last plane reads the zeroed 256 bytes
      // after the rows
      const uint32_t b_plane = (uint32_t)act_box_rows(bi) * C::kBRow;
      auto issue_b = [&](int ss, int kt, int nk) {
        (void)nk;
        tma_load_3d(sB + ss * C::kB, r.gu ? &maps.xp3[bi] : &maps.hq3[bi], &full[ss], 0, td.y,
                    C::kWideB ? kt / 2 : kt);
      };
      auto stage_bytes = [&](int nk) {
        return (uint32_t)(rows_m * nk * kTileRowBytes + C::kBPlanes * b_bytes + nk * 2 * SA * kAtomBytes);
      };
      // A down unit's hq is ready once all gate_up m-tiles of its token tile are
      // counted.  If it is not ready yet, the unit's first stages get their weight
      // copies only, and the activation copies of those stages follow the
      // (bounded) wait.
      // (a gate_up unit's grouped activations are ready once every routing CTA that
      // publishes through the flags has counted in)
      const int32_t* dep_ctr = r.gu ? p.route_flags + 1 : p.done_gu + r.b;
      const int dep_target = r.gu ? p.route_ctas : p.gu_mtiles + p.dep_extra;
      // (until a gate_up unit has seen the routing flag, its first stages stream
      // weights only and the flag is read after their copies are out)
      bool dep_ok = r.gu ? xp_ready : __all_sync(0xffffffffu, ld_acquire_gpu(dep_ctr) >= dep_target);
      // hq and the flagged xp were written by generic stores; TMA reads them
      if (dep_ok && (!r.gu || p.route_ctas != 0)) fence_proxy_async_global();
      bool dep_timeout = false;
      int pend_s = 0, pend_kt = 0, pend_n = 0;  // stages waiting for their activation copies
      // activation copies of the stages that wait for them.  After an expired wait
      // the copies still go out (they read in-bounds workspace bytes), so that every
      // stage's phase completes before the roles wind down.
      auto flush_pending = [&]() {
        fence_proxy_async_global();
        if (elect_one())
          for (int j = 0; j < pend_n; ++j) {
            const int kk = pend_kt + j * kKS, nn = min(kKS, k_tiles - kk), ss = (pend_s + j) % S;
            issue_b(ss, kk, nn);
            bulk_g2s(sSF + ss * C::kSF + kKS * SA * kAtomBytes, sfb + kk * SA * kAtomBytes, nn * SA * kAtomBytes,
                     &full[ss]);
          }
        __syncwarp();
        pend_n = 0;
      };
      for (int kt = 0; kt < k_tiles; kt += kKS) {
        const int nk = min(kKS, k_tiles - kt);
        const int st = kt / kKS;
        if (st == claim_st && lane == 0) claim = atomicAdd(p.sched, 1);
        if (st == fetch_st) {
          next = __shfl_sync(0xffffffffu, claim, 0);
          if (next < total) td_next = tl[tile_ref(next, n_gu, p).b];
        }
        if (!mbar_wait_warp(&empty[s], ph ^ 1u, p.wait_ns)) {
          if (lane == 0) {
            atomicOr(p.status, kStatusTimeoutProducer);
            atomicCAS(p.status + 1, 0u, wait_site(1, tile, kt));
          }
          flush_pending();
          ok = false;
          break;
        }
        if (dep_ok) {
          if (elect_one()) {
            mbar_arrive_expect_tx(&full[s], stage_bytes(nk));
            issue_a(s, kt, nk);
            issue_b(s, kt, nk);
            uint8_t* sf = sSF + s * C::kSF;
            bulk_g2s_hint(sf, sfa + kt * SA * kAtomBytes, nk * SA * kAtomBytes, &full[s], wpol);
            bulk_g2s(sf + kKS * SA * kAtomBytes, sfb + kt * SA * kAtomBytes, nk * SA * kAtomBytes, &full[s]);
          }
          __syncwarp();
        } else {
          if (elect_one()) {
            mbar_arrive_expect_tx(&full[s], stage_bytes(nk));
            issue_a(s, kt, nk);
            bulk_g2s_hint(sSF + s * C::kSF, sfa + kt * SA * kAtomBytes, nk * SA * kAtomBytes, &full[s], wpol);
          }
          __syncwarp();
          if (pend_n == 0) {
            pend_s = s;
            pend_kt = kt;
          }
          ++pend_n;
          dep_ok = __all_sync(0xffffffffu, ld_acquire_gpu(dep_ctr) >= dep_target);
          // keep streaming weights while the activations are not ready, until every
          // stage slot is taken or this is the unit's last stage
          if (!dep_ok && (pend_n >= S || kt + kKS >= k_tiles)) {
            if (!wait_counter_warp(dep_ctr, dep_target, p.wait_ns)) {
              if (lane == 0) {
                atomicOr(p.status, kStatusTimeoutProducer);
                atomicCAS(p.status + 1, 0u, wait_site(r.gu ? 9 : 5, tile, kt));
              }
              dep_timeout = true;
            }
            dep_ok = true;
          }
          if (dep_ok && r.gu) xp_ready = true;
          if (dep_ok) flush_pending();
        }
        ++issued;
        if (++s == S) {
          s = 0;
          ph ^= 1u;
        }
        if (dep_timeout) {
          ok = false;
          break;
        }
      }
      tile = next;
    }
    // Let every copy this warp issued land before the CTA can exit.
    for (int st = 0; st < S && st < issued; ++st) {
      const int64_t last = ((issued - 1 - st) / S) * S + st;
      if (!mbar_wait_warp(&full[st], (uint32_t)((last / S) & 1), kDrainLimitNs) && lane == 0)
        atomicOr(p.status, kStatusTimeoutDrain);
    }
  } else if (warp == 1) {
    // -------------------------------------------------------------- MMA issuer
    int s = 0, acc = 0;
    uint32_t ph = 0, aph = 0;
    bool ok = true;
    for (int i = 0; ok; ++i) {
      const int slot = i & (kTileQ - 1);
      if (!mbar_wait_warp(&q_full[slot], (uint32_t)((i / kTileQ) & 1), p.wait_ns)) {
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
      const int tile = q.x;
      const TileRef r = tile_ref(tile, n_gu, p);
      const int4 td = make_int4(q.y, q.z, q.w, 0);
      const int k_tiles = r.gu ? p.gu_ktiles : p.d_ktiles;
      const int rows_m = min(kTileM, (r.gu ? p.gu_rows_stored : p.d_rows_stored) - r.m * kTileM);
      // activation plane j sits j box heights into the stage (the producer's layout)
      const uint32_t b_plane = (uint32_t)act_box_rows(min(act_box_index(td.z), kActBoxes - 1)) * C::kBRow;
      if (!mbar_wait_warp(&tempty[acc], aph ^ 1u, p.wait_ns)) {
        if (lane == 0) {
          atomicOr(p.status, kStatusTimeoutMma);
          atomicCAS(p.status + 1, 0u, wait_site(2, tile, 0xFFF));
        }
        break;
      }
      tc_fence_after();
      // N of the MMA: the unit's rows rounded up to 16 (the smallest N for M = 128);
      // B rows past the unit's rows are never read back
      const uint32_t n_mma = (uint32_t)max(16, min(BN, (td.z + 15) & ~15));
      const uint32_t d_tmem = tmem + (uint32_t)acc * 128u;
      uint32_t idesc0 = FP4 ? idesc_mxf8f6f4(128, n_mma, 1 /*E2M1*/, 1 /*E2M1*/, 0, 0)
                            : idesc_mxf8f6f4(128, n_mma, 5 /*E2M1*/, 0 /*E4M3*/, 0, 0);
      if (NV) idesc0 &= ~(1u << 23);  // block scales in UE4M3, not UE8M0
      for (int kt = 0; kt < k_tiles; kt += kKS) {
        const int nk = min(kKS, k_tiles - kt);
        if (!mbar_wait_warp(&full[s], ph, p.wait_ns)) {
          if (lane == 0) {
            atomicOr(p.status, kStatusTimeoutMma);
            atomicCAS(p.status + 1, 0u, wait_site(3, tile, kt));
          }
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sf_t = tmem + 256u + (uint32_t)s * C::kSfCols;
        const uint32_t sf_s = smem_u32(sSF + s * C::kSF);
        const uint32_t a_s = smem_u32(sA + s * C::kA);
        const uint32_t b_s = smem_u32(sB + s * C::kB);
        if (elect_one()) {
          for (int j = 0; j < nk; ++j) {
            // this k-tile's scale atoms: A then B, SA each, four columns per atom
            const uint32_t sfa_t = sf_t + 8u * SA * j, sfb_t = sfa_t + 4u * SA;
#pragma unroll
            for (int aa = 0; aa < SA; ++aa) {
              tmem_cp_32x128b_x4(sfa_t + 4u * aa, sdesc_sf_atom(sf_s + (j * SA + aa) * kAtomBytes));
              tmem_cp_32x128b_x4(sfb_t + 4u * aa, sdesc_sf_atom(sf_s + ((kKS + j) * SA + aa) * kAtomBytes));
            }
            // weight k-tile j starts rows_m rows into the stage (a swizzle-atom multiple)
            const uint32_t a_j = a_s + (uint32_t)(j * rows_m) * C::kRow,
                           b_j = b_s + (uint32_t)(C::kWideB ? j >> 1 : j) * b_plane;
            if constexpr (NV) {
              // two MMAs of K = 64, each with the four 16-element block scales of one atom
              const uint64_t ad = sdesc_sw64(a_j), bd = sdesc_sw64(b_j);
#pragma unroll
              for (uint32_t kk = 0; kk < 2; ++kk)
                umma_mxf4nvf4(d_tmem, ad + 2u * kk, bd + 2u * kk, idesc0, sfa_t + 4u * kk, sfb_t + 4u * kk,
                              (kt + j + (int)kk) != 0);
            } else if constexpr (FP4) {
              // two MMAs of K = 64 (32 bytes of each 64-byte weight row; the activation row
              // holds two k-tiles, this one in its first or second 64 bytes); each takes
              // two of the row's four block scales, starting at byte 2kk
              const uint64_t ad = sdesc_sw64(a_j), bd = sdesc_sw128(b_j) + 4u * (uint32_t)(j & 1);
#pragma unroll
              for (uint32_t kk = 0; kk < 2; ++kk) {
                const uint32_t idesc = idesc0 | ((2u * kk) << 4) | ((2u * kk) << 29);
                umma_mxf4(d_tmem, ad + 2u * kk, bd + 2u * kk, idesc, sfa_t, sfb_t, (kt + j + (int)kk) != 0);
              }
            } else {
              const uint64_t ad = sdesc_sw128(a_j), bd = sdesc_sw128(b_j);
#pragma unroll
              for (uint32_t kk = 0; kk < 4; ++kk) {
                // block-scale ids pick byte kk of the scale columns (bits 4-5 for B, 29-30 for A)
                const uint32_t idesc = idesc0 | (kk << 4) | (kk << 29);
                umma_mxf8f6f4(d_tmem, ad + 2u * kk, bd + 2u * kk, idesc, sfa_t, sfb_t, (kt + j + (int)kk) != 0);
              }
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
    if (!mbar_wait_warp(drain, 0, kDrainLimitNs) && lane == 0) atomicOr(p.status, kStatusTimeoutDrain);
  } else {
    // -------------------------------------------------------------- epilogue
    const int q = warp & 3;              // tmem lane quadrant this warp may read
    const int row = 32 * q + lane;       // tile row == tmem lane
    const int et = threadIdx.x - 64;     // 0..127 within the epilogue warps
    int acc = 0;
    uint32_t aph = 0;
    bool ok = true;
    // NVFP4 weights carry a global scale per projection (the activations' is 1)
    const float gs_gu = NV ? nvfp4_global_scale(__uint_as_float(reinterpret_cast<const uint32_t*>(
                                 reinterpret_cast<const uint8_t*>(p.hdr) + kAmaxOffset)[0]))
                           : 1.0f;
    const float gs_d = NV ? nvfp4_global_scale(__uint_as_float(reinterpret_cast<const uint32_t*>(
                                reinterpret_cast<const uint8_t*>(p.hdr) + kAmaxOffset)[1]))
                          : 1.0f;
    auto bias_of = [&](const TileRef& rr, const int4& t4) -> float {
      if (rr.gu) return p.gu_bias[(int64_t)t4.x * 2 * p.I + rr.m * kTileM + row];
      const int o = rr.m * kTileM + row;
      return o < p.H ? p.d_bias[(int64_t)t4.x * p.H + o] : 0.0f;
    };
    for (int i = 0;; ++i) {
      // one warp takes the next queue entry for all four, so that they agree on
      // every tile (and on stopping) and meet at the same named barriers
      const int slot = i & (kTileQ - 1);
      if (warp == 2) {
        const bool got = mbar_wait_warp(&q_full[slot], (uint32_t)((i / kTileQ) & 1), p.wait_ns);
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
      named_barrier_sync(1, 128);
      const int4 qe = *s_eq;
      if (qe.x < 0) break;
      const int tile = qe.x;
      const TileRef r = tile_ref(tile, n_gu, p);
      const int4 td = make_int4(qe.y, qe.z, qe.w, 0);
      const float bias_v = bias_of(r, td);
      const int rows = td.z;
      if (ok) {
        // all lanes take the same decision, so the warp-collective tcgen05.ld stays uniform
        ok = mbar_wait_warp(&tfull[acc], aph, p.wait_ns);
        if (!ok && lane == 0) {
          atomicOr(p.status, kStatusTimeoutEpilogue);
          atomicCAS(p.status + 1, 0u, wait_site(4, tile, 0));
        }
      }
      tc_fence_after();
      const uint32_t tb = tmem + (uint32_t)acc * 128u + ((uint32_t)(32 * q) << 16);
      if (r.gu) {
        // the 256 bytes after the last intermediate row are read (as zero padding) by the
        // down units' plane boxes: the tile holding the last row clears them before it
        // counts its m-tile 0 (which every down unit of that tile waits for)
        if (r.m == 0 && td.y + td.z == p.TK && et < 16)
          reinterpret_cast<uint4*>(p.hq + (int64_t)p.TK * (FP4 ? p.I / 2 : p.I))[et] = make_uint4(0, 0, 0, 0);
        // accumulator rows 0..63 = gate, 64..127 = up of intermediate columns 64m..64m+63
        // SwiGLU + MXFP8 of a 32-column chunk, transposed through shared memory:
        // thread et takes token column jt of the chunk and 16 rows (half hh = et & 1)
        // of MX block rb (gate rows 32rb..32rb+31); the two halves of a block are
        // neighbouring lanes and share their amax with one shuffle.  A 16-wide chunk
        // needs the first 64 threads only.
        constexpr int CW = C::kCW, XS = CW + 1;
        const int hh = et & 1, jt = (et >> 1) & (CW - 1), rb = (et >> (CW == 32 ? 6 : 5)) & 1;
        const bool active = et < 4 * CW;
        const int kb = 2 * r.m + rb;  // MX block of the intermediate
        for (int c0 = 0; c0 < rows; c0 += CW) {
          uint32_t r0[16], r1[16];
          if (ok) {
            tmem_ld_32x32b_x16(tb + (uint32_t)c0, r0);
            if (CW == 32) tmem_ld_32x32b_x16(tb + (uint32_t)c0 + 16u, r1);
            tmem_ld_wait();
          } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) r0[j] = r1[j] = 0;
          }
#pragma unroll
          for (int j = 0; j < CW; ++j)
            xbuf[row * XS + j] = (NV ? __uint_as_float(j < 16 ? r0[j] : r1[j - 16]) * gs_gu
                                     : __uint_as_float(j < 16 ? r0[j] : r1[j - 16])) + bias_v;
          named_barrier_sync(1, 128);
          const int n = c0 + jt;
          float h[16];
          float amax = 0.f;
          if (active && n < rows) {  // same for both lanes of a pair
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int rr = 32 * rb + 16 * hh + i;
              const float g = xbuf[rr * XS + jt];
              const float u = xbuf[(64 + rr) * XS + jt];
              h[i] = __fdividef(g, 1.0f + __expf(-g)) * u;  // rel. error ~1e-6, far below an E4M3 step
              amax = fmaxf(amax, fabsf(h[i]));
            }
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) h[i] = 0.f;
          }
          if (!NV) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));  // MX blocks span the lane pair
          const int sx = FP4 ? mx_scale_exp<2>(amax) : mx_scale_exp<8>(amax);
          const float inv = mx_pow2_neg(sx);
          uint32_t pk[4];
          uint32_t nsc = 0;  // NVFP4: this half block is one 16-element block with its own E4M3 scale
          if constexpr (NV) {
            uint32_t p2[2];
            nsc = nvfp4_block16(h, 1.0f, p2);
            pk[0] = p2[0];
            pk[1] = p2[1];
          } else if constexpr (FP4) {
#pragma unroll
            for (int i = 0; i < 16; ++i) h[i] *= inv;
            pk[0] = cvt_e2m1x8(h);
            pk[1] = cvt_e2m1x8(h + 8);
          } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const uint32_t lo = cvt_e4m3x2(h[4 * i] * inv, h[4 * i + 1] * inv);
              const uint32_t hi = cvt_e4m3x2(h[4 * i + 2] * inv, h[4 * i + 3] * inv);
              pk[i] = lo | (hi << 16);
            }
          }
          if (ok && active && n < rows) {
            const int64_t col = r.m * 64 + 32 * rb + 16 * hh;  // first intermediate of this half block
            if constexpr (FP4)
              *reinterpret_cast<uint2*>(p.hq + (int64_t)(td.y + n) * (p.I / 2) + col / 2) = make_uint2(pk[0], pk[1]);
            else
              *reinterpret_cast<uint4*>(p.hq + (int64_t)(td.y + n) * p.I + col) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            if (NV) {
              // 16-element block q = 2 kb + hh: k-tile q / 8, atom (q / 4) % 2, byte q % 4
              const int qb = 2 * kb + hh;
              uint8_t* wd = p.hq_sf + (((int64_t)r.b * p.d_ktiles + (qb >> 3)) * 2 + ((qb >> 2) & 1)) * kAtomBytes +
                            (n & 31) * 16 + (n >> 5) * 4;
              wd[qb & 3] = (uint8_t)nsc;
              // the last real block also zeroes the scales of the padding blocks after it
              // in its k-tile (zero data past I; their scale must not be a NaN code)
              const int last = (p.I >> 4) - 1;
              if (qb == last) {
                for (int j = (qb & 3) + 1; j < 4; ++j) wd[j] = 0;
                if (((qb >> 2) & 1) == 0) *reinterpret_cast<uint32_t*>(wd + kAtomBytes) = 0u;
              }
            } else if (hh == 0) {
              uint8_t* wd = p.hq_sf + ((int64_t)r.b * p.d_ktiles + (kb >> 2)) * kAtomBytes + (n & 31) * 16 + (n >> 5) * 4;
              wd[kb & 3] = (uint8_t)(sx + 127);
              // the last real block also sets the padding blocks of its word (zero
              // data past I; their scale must not be the NaN code)
              if (kb == (p.I >> 5) - 1)
                for (int j = (kb & 3) + 1; j < 4; ++j) wd[j] = 127;
            }
          }
          named_barrier_sync(1, 128);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[acc]);
        // every hq byte of this m-tile is stored (the last barrier above): count it
        if (et == 0 && ok) red_add_release_gpu(p.done_gu + r.b, 1);
      } else {
        const int orow = r.m * kTileM + row;
        const bool rv = orow < p.H;
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
                if (n < rows) {
                  const float v =
                      (NV ? __uint_as_float(j < 16 ? r0[j] : r1[j - 16]) * gs_d : __uint_as_float(j < 16 ? r0[j] : r1[j - 16])) +
                      bias_v;
                  if (p.dense)  // a dense linear: row td.y + n of the grouped order is that token
                    p.out[(int64_t)(td.y + n) * p.H + orow] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
                  else
                    p.y[(int64_t)(td.y + n) * p.H + orow] = v;
                }
              }
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[acc]);
        if (p.fused_combine) {
        // combine: each token of the tile has one more of its k contributions to
        // feature block m; the epilogue that completes the k-th sums them (slot order).
        // The completing thread stages the token's slot positions and weights in
        // shared memory (the transpose buffer is free here); then every epilogue
        // thread takes one feature column of all completed tokens, four tokens'
        // loads in flight at a time.
        int* cpos = reinterpret_cast<int*>(xbuf);    // [BN][8] grouped positions of the slots
        float* cwt = xbuf + BN * 8;                  // [BN][8] routing weights
        if (et == 0) comb_list[0] = 0;
        named_barrier_sync(1, 128);
        if (et < rows && ok) {
          const int flat = p.sorted_rows[td.y + et];
          const int t = flat / p.k;
          // y of this tile is stored (barrier above); release it, and acquire the
          // other slots' rows if this is the last of the k contributions
          const int prev = atom_add_acq_rel_gpu(p.done_tok + (int64_t)t * p.d_mtiles + r.m, 1);
          if (prev == p.k - 1) {
            const int c = atomicAdd(comb_list, 1);
            comb_list[1 + c] = t;
            for (int j = 0; j < p.k; ++j) {
              cpos[c * 8 + j] = p.inv_pos[(int64_t)t * p.k + j];
              cwt[c * 8 + j] = p.topk_w[(int64_t)t * p.k + j];
            }
          }
        }
        named_barrier_sync(1, 128);
        const int ncomb = comb_list[0];
        const int f = r.m * kTileM + et;
        if (f < p.H) {
          for (int i0 = 0; i0 < ncomb; i0 += 4) {
            float v[4][8];
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
              for (int j = 0; j < 8; ++j)
                v[u][j] = (i0 + u < ncomb && j < p.k) ? __ldcg(p.y + (int64_t)cpos[(i0 + u) * 8 + j] * p.H + f) : 0.f;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              if (i0 + u < ncomb) {
                float a = 0.f;
#pragma unroll
                for (int j = 0; j < 8; ++j)
                  if (j < p.k) a = fmaf(cwt[(i0 + u) * 8 + j], v[u][j], a);
                p.out[(int64_t)comb_list[1 + i0 + u] * p.H + f] = __bfloat16_as_ushort(__float2bfloat16_rn(a));
              }
            }
          }
        }
        named_barrier_sync(1, 128);
        }  // fused_combine (otherwise a separate streaming pass combines y)
      }
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
  // a routing grid followed through its flags completes before this one does
  if (p.route_ctas != 0) asm volatile("griddepcontrol.wait;" ::: "memory");
}

template <int BN, bool FP4, bool NV>
cudaError_t launch_bn(const Maps& m, const MlpParams& p, int grid, cudaStream_t s) {
  using C = GemmCfg<BN, FP4, NV>;
  static bool attr = false;
  if (!attr) {
    cudaError_t e =
        cudaFuncSetAttribute(expert_mlp_kernel<BN, FP4, NV>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::kSmem);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(192);
  cfg.dynamicSmemBytes = C::kSmem;
  cfg.stream = s;
  // Programmatic dependent launch: the CTAs start (barrier init, TMEM allocation,
  // descriptor prefetch) while the routing kernel finishes.  The grid is at most
  // one CTA per SM.  Units are claimed at run time by the CTAs that are running,
  // so the dependencies between units hold even when only part of the grid is
  // resident (another kernel holding SMs); every wait is bounded regardless.
  cudaLaunchAttribute attrs[1];
  attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, expert_mlp_kernel<BN, FP4, NV>, m, p);
}

}  // namespace

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
// rows of 4-bit codes; a box is 256, 128 or 64 rows (whole adjacent k-tiles),
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

// The same layout seen as packed bytes (kind::mxf4 reads E2M1 two per byte): 64-byte
// rows, 64-byte swizzle.
bool make_weight_map_packed(CUtensorMap* map, const uint8_t* base, int64_t total_rows, int box_rows) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)kTileRowBytes, (cuuint64_t)total_rows};
  cuuint64_t strides[1] = {(cuuint64_t)kTileRowBytes};
  cuuint32_t box[2] = {(cuuint32_t)kTileRowBytes, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Activations: 2-D [rows][row_bytes] (E4M3 codes, or E2M1 codes two per byte),
// rows of the grouped order; a box covers one 128-element k-tile.
bool make_act_map(CUtensorMap* map, const uint8_t* base, int row_bytes, int rows, int box_rows, bool fp4) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)row_bytes, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
  cuuint32_t box[2] = {fp4 ? (cuuint32_t)kTileRowBytes : (cuuint32_t)kTileK, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, fp4 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_weight_map_x2(CUtensorMap* map, const uint8_t* base, int64_t total_rows, bool packed) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {packed ? (cuuint64_t)kTileRowBytes : (cuuint64_t)kTileK, (cuuint64_t)total_rows, 2};
  cuuint64_t strides[2] = {(cuuint64_t)kTileRowBytes, (cuuint64_t)256 * kTileRowBytes};
  cuuint32_t box[3] = {packed ? (cuuint32_t)kTileRowBytes : (cuuint32_t)kTileK, 256, 2};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(map, packed ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 3,
             const_cast<uint8_t*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             packed ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_act_map_planes(CUtensorMap* map, const uint8_t* base, int row_bytes, int rows, int K, int box_rows,
                         int planes, bool fp4) {
  auto enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t kbytes = fp4 ? (cuuint64_t)kTileRowBytes : (cuuint64_t)kTileK;  // one k-tile of a row
  cuuint64_t dims[3] = {kbytes, (cuuint64_t)rows, (cuuint64_t)((K + kTileK - 1) / kTileK)};
  cuuint64_t strides[2] = {(cuuint64_t)row_bytes, kbytes};
  cuuint32_t box[3] = {(cuuint32_t)kbytes, (cuuint32_t)box_rows, (cuuint32_t)planes};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, fp4 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Encoded descriptors depend only on these values, so they are reused across calls.
struct MapKey {
  const uint8_t* packed;
  const uint8_t* xp;
  const uint8_t* hq;
  int E, H, I, TK, tile_rows;
  int fmt;                       // activation format, which also fixes the weight layout
  uint64_t off_gu_data, off_d_data;  // the packed sections the weight maps point into
  bool operator==(const MapKey& o) const {
    return packed == o.packed && xp == o.xp && hq == o.hq && E == o.E && H == o.H && I == o.I && TK == o.TK &&
           tile_rows == o.tile_rows && fmt == o.fmt && off_gu_data == o.off_gu_data && off_d_data == o.off_d_data;
  }
};

cudaError_t launch_expert_mlp(const PackedHeader& h, const uint8_t* packed, const ExpertMlpBuffers& b, int T, int k,
                              int max_tiles, int tile_rows, int num_sms, int fmt, cudaStream_t s) {
  const int TK = T * k;
  const bool fp4 = fmt != kActMxfp8;
  static std::mutex mu;
  static MapKey keys[32];
  static Maps cache[32];
  static int n_cached = 0, next_slot = 0;
  const MapKey key{packed, b.xp, b.hq, h.E, h.H, h.I, TK, tile_rows, fmt, h.off_gu_data, h.off_d_data};
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
  const int64_t d_rows = (int64_t)h.E * h.d_rows_stored * h.d_ktiles;
  auto wmap = fp4 ? make_weight_map_packed : make_weight_map;
  // a dense linear has no gate_up section: its (unused) gate_up maps alias the weights
  const uint64_t off_gu = h.gu_rows_stored ? h.off_gu_data : h.off_d_data;
  const int64_t gu_rows = h.gu_rows_stored ? (int64_t)h.E * h.gu_rows_stored * h.gu_ktiles
                                           : (int64_t)h.E * h.d_rows_stored * h.d_ktiles;
  if (!make_weight_map_x2(&m.gu4, packed + off_gu, gu_rows, fp4) ||
      !make_weight_map_x2(&m.d4, packed + h.off_d_data, (int64_t)h.E * h.d_rows_stored * h.d_ktiles, fp4))
    return cudaErrorInvalidValue;
  if (!wmap(&m.gu2, packed + off_gu, gu_rows, 2 * kTileM) || !wmap(&m.gu, packed + off_gu, gu_rows, kTileM) ||
      !wmap(&m.gut, packed + off_gu, gu_rows, 64) ||
      !wmap(&m.d2, packed + h.off_d_data, d_rows, 2 * kTileM) || !wmap(&m.d, packed + h.off_d_data, d_rows, kTileM) ||
      !wmap(&m.dt, packed + h.off_d_data, d_rows, 64))
    return cudaErrorInvalidValue;
  for (int i = 0; i < kActBoxes; ++i) {
    // boxes taller than the token tile are never used; encode them at its height
    const int rows = std::min(act_box_rows(i), tile_rows);
    // MXFP4 activations travel as 128-byte rows of 256 elements (byte-typed boxes with
    // the 128-byte swizzle, one plane per two k-tiles); NVFP4 as 64-byte rows
    const bool wide = fp4 && fmt != kActNvfp4, narrow = fp4 && !wide;
    const int kst = stage_ktiles_for(tile_rows, fp4);
    if (!make_act_map_planes(&m.xp3[i], b.xp, fp4 ? h.H / 2 : h.H, TK, wide ? h.H / 2 : h.H, rows,
                             wide ? kst / 2 : kst, narrow) ||
        !make_act_map_planes(&m.hq3[i], b.hq, fp4 ? h.I / 2 : h.I, TK, wide ? h.I / 2 : h.I, rows,
                             wide ? kst / 2 : kst, narrow) ||
        !make_act_map(&m.xp[i], b.xp, fp4 ? h.H / 2 : h.H, TK, rows, narrow) ||
        !make_act_map(&m.hq[i], b.hq, fp4 ? h.I / 2 : h.I, TK, rows, narrow))
      return cudaErrorInvalidValue;
  }
    std::lock_guard<std::mutex> lk(mu);
    keys[next_slot] = key;
    cache[next_slot] = m;
    next_slot = (next_slot + 1) % 32;
    if (n_cached < 32) ++n_cached;
  }
  MlpParams p{};
  p.gu_sfa = packed + h.off_gu_sf;
  p.gu_bias = reinterpret_cast<const float*>(packed + h.off_gu_bias);
  p.d_sfa = packed + h.off_d_sf;
  p.d_bias = reinterpret_cast<const float*>(packed + h.off_d_bias);
  p.xp_sf = b.xp_sf;
  p.hq = b.hq;
  p.hq_sf = b.hq_sf;
  p.y = b.y;
  p.out = b.out;
  p.tiles = b.tiles;
  p.sorted_rows = b.sorted_rows;
  p.inv_pos = b.inv_pos;
  p.topk_w = b.topk_w;
  p.done_gu = b.done_gu;
  p.done_tok = b.done_tok;
  p.sched = b.sched;
  p.max_tiles = max_tiles;
  p.TK = TK;
  p.route_flags = b.route_flags;
  p.route_ctas = b.route_ctas;
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
  p.k = k;
  // when the token rows of an expert fit one tile on average, each weight byte is
  // read once per forward
  p.weights_evict_first = (int64_t)T * k <= (int64_t)h.E * tile_rows;
  p.fused_combine = b.fused_combine ? 1 : 0;
  p.hdr = reinterpret_cast<const PackedHeader*>(packed);
  p.want = h;
  p.dense = h.wfmt == kWeightsDense ? 1 : 0;
  const int grid = (int)std::min<int64_t>(num_sms, (int64_t)max_tiles * (h.gu_mtiles + h.d_mtiles));
  switch (tile_rows) {
    case 8: return fmt == kActNvfp4 ? launch_bn<8, true, true>(m, p, grid, s)
                 : fp4 ? launch_bn<8, true, false>(m, p, grid, s) : launch_bn<8, false, false>(m, p, grid, s);
    case 16: return fmt == kActNvfp4 ? launch_bn<16, true, true>(m, p, grid, s)
                  : fp4 ? launch_bn<16, true, false>(m, p, grid, s) : launch_bn<16, false, false>(m, p, grid, s);
    case 32: return fmt == kActNvfp4 ? launch_bn<32, true, true>(m, p, grid, s)
                  : fp4 ? launch_bn<32, true, false>(m, p, grid, s) : launch_bn<32, false, false>(m, p, grid, s);
    case 64: return fmt == kActNvfp4 ? launch_bn<64, true, true>(m, p, grid, s)
                  : fp4 ? launch_bn<64, true, false>(m, p, grid, s) : launch_bn<64, false, false>(m, p, grid, s);
    case 128: return fmt == kActNvfp4 ? launch_bn<128, true, true>(m, p, grid, s)
                   : fp4 ? launch_bn<128, true, false>(m, p, grid, s) : launch_bn<128, false, false>(m, p, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace moe

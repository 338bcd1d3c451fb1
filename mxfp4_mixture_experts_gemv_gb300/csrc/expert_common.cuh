// Device helpers and tensor-map builders shared by the expert-MLP kernels.
#pragma once

#include <cudaTypedefs.h>

#include "common.cuh"
#include "ptx.cuh"

namespace moe {

// Where a bounded wait expired: role (1 producer/empty, 2 mma/accumulator, 3 mma/full,
// 4 epilogue, 5 producer/dependency, 6 producer/tile queue, 7 mma/tile queue; 8 is the
// cluster routing kernel's copies, 9 the expert kernel's wait for the routing flags), tile (or queue position) and k-step, packed for the
// second status word.
__device__ __forceinline__ uint32_t wait_site(uint32_t role, int tile, int kt) {
  return (role << 28) | ((uint32_t)min(tile, 0xFFFF) << 12) | (uint32_t)min(kt, 0xFFF);
}

// Increment with acquire and release: returns the previous value; the caller sees
// every write published by earlier increments.
__device__ __forceinline__ int atom_add_acq_rel_gpu(int32_t* p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Bounded wait (all lanes of the warp) until *ctr >= target.
__device__ __forceinline__ bool wait_counter_warp(const int32_t* ctr, int target, uint64_t limit_ns) {
  bool ok = ld_acquire_gpu(ctr) >= target;
  if (!__all_sync(0xffffffffu, ok)) {
    const uint64_t t0 = global_timer_ns();
    while (true) {
      ok = ld_acquire_gpu(ctr) >= target;
      if (__all_sync(0xffffffffu, ok)) break;
      if (global_timer_ns() - t0 > limit_ns) return false;
      __nanosleep(64);
    }
  }
  return true;
}

// Activation tiles are fetched with the smallest of these box heights that covers
// the unit's token rows (the MMA's N rounds rows up to 16; columns past the rows
// are never read back), so a sparse token tile does not pull a full BN x 128 box.
constexpr int kActBoxes = 5;  // 8, 16, 32, 64, 128 rows
__host__ __device__ constexpr int act_box_rows(int i) { return 8 << i; }
__device__ __forceinline__ int act_box_index(int rows) {
  return rows <= 8 ? 0 : rows <= 16 ? 1 : rows <= 32 ? 2 : rows <= 64 ? 3 : 4;
}

// Tensor maps of one launch: weight boxes of 256, 128 and 64 rows (two k-tiles,
// one k-tile, a 64-row tail tile), and the activation maps (grouped x for
// gate_up, hq for down) for each box height.
struct Maps {
  CUtensorMap gu2, gu, gut, d2, d, dt;
  CUtensorMap xp[kActBoxes], hq[kActBoxes];
  // Fewer, larger copies stream faster: four k-tiles of a 128-row weight tile (512
  // consecutive rows) as one box of two 256-row planes, and the activation rows of
  // every k-tile of a pipeline stage as one box of k-tile planes (grouped x, and the
  // intermediate read by the down units).
  CUtensorMap gu4, d4;
  CUtensorMap xp3[kActBoxes], hq3[kActBoxes];
  // The tokens-on-M kernel's pairs of consecutive 128-row weight tiles: one k-tile of
  // both tiles as one box, and both tiles' scale atoms of that k-tile as one box.
  CUtensorMap gup, dp, gusf, dsf;
};

// Tensor maps (host).  Weights: the tile-contiguous packed layout as 2-D rows of
// 128 E2M1 codes, either unpacked by TMA into the 16-byte-per-16-codes form that
// kind::mxf8f6f4 reads (make_weight_map) or as packed bytes for kind::mxf4
// (make_weight_map_packed); activations: [rows][row_bytes] of E4M3 codes or E2M1
// codes two per byte, one 128-element k-tile per box.
PFN_cuTensorMapEncodeTiled_v12000 encode_fn();
bool make_weight_map(CUtensorMap* map, const uint8_t* base, int64_t total_rows, int box_rows);
bool make_weight_map_packed(CUtensorMap* map, const uint8_t* base, int64_t total_rows, int box_rows);
bool make_act_map(CUtensorMap* map, const uint8_t* base, int row_bytes, int rows, int box_rows, bool fp4);
// Weights as planes of 256 rows (two planes per box): dims {128 codes, rows, 2}.
bool make_weight_map_x2(CUtensorMap* map, const uint8_t* base, int64_t total_rows, bool packed);
// Activations as k-tile planes: dims {128 elements, rows, ceil(K/128)} with the
// k-tile plane stride one k-tile of a row; a box covers `planes` consecutive k-tiles
// of box_rows rows.  The last k-tile of a row runs past the row end into the next
// row (or into the buffer's zeroed slack after the last row), where the weights it
// multiplies are zero padding.
bool make_act_map_planes(CUtensorMap* map, const uint8_t* base, int row_bytes, int rows, int K, int box_rows,
                         int planes, bool fp4);

}  // namespace moe

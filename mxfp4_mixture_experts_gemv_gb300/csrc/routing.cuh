// Warp-level steps shared by the small-batch routing kernels: the top-k +
// softmax of one token's logits and the stable grouping of the T*k (token,
// slot) pairs by expert, with the tile list the expert kernel walks.
//
// Routing rule: top-k experts by logit (descending, lower index first on ties),
// then softmax over the k selected ("GPT-OSS-120B on DGX Spark: From MXFP4 to
// NVFP4", section "GPT-OSS-120B Architecture": 128 experts, 4 active per token).
#pragma once

#include <stdint.h>

#include "common.cuh"
#include "quant.cuh"

namespace moe {

// Order-preserving map of a non-NaN fp32 onto uint32 (a larger float gives a larger
// key; -0 and +0 must be merged by the caller).  Key 0 is never produced.
__device__ __forceinline__ uint32_t f32_order_key(float f) {
  const uint32_t b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ float f32_from_order_key(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// One warp selects the k <= 8 largest of E <= 256 logits (a NaN ranks as -inf,
// ties go to the lower expert index) and writes their ids and their softmax
// weights, exp(l_j - l_0) / sum_i exp(l_i - l_0) with l_0 the largest.
__device__ __forceinline__ void topk_softmax_warp(const float* logit, int E, int k, int32_t* ids, float* w,
                                                  int lane) {
  uint32_t key[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = lane + 32 * i;
    float v = e < E ? logit[e] : 0.f;
    if (isnan(v)) v = -INFINITY;
    if (v == 0.f) v = 0.f;  // -0 ranks equal to +0
    key[i] = e < E ? f32_order_key(v) : 0u;
  }
  float l0 = 0.f, den = 0.f, mine = 0.f;
  int mine_id = 0;
  for (int j = 0; j < k; ++j) {
    uint32_t bk = 0u;
    int bi = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (key[i] > bk) {  // strict: the lower index of this lane wins a tie
        bk = key[i];
        bi = i;
      }
    const uint32_t mk = __reduce_max_sync(0xffffffffu, bk);
    const int e = __reduce_min_sync(0xffffffffu, bk == mk ? lane + 32 * bi : 0x7FFFFFFF);
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if ((e & 31) == lane && (e >> 5) == i) key[i] = 0u;
    const float lv = f32_from_order_key(mk);
    if (j == 0) l0 = lv;
    den += expf(lv - l0);
    if (lane == j) {
      mine = lv;
      mine_id = e;
    }
  }
  if (lane < k) {
    ids[lane] = mine_id;
    w[lane] = expf(mine - l0) / den;
  }
}

// Warp 0: stable counting sort of the TK pairs f = t*k + j by expert ids[f].
// cnt must be zero on entry.  Produces the counts, the offsets off[0..E], the
// tile offsets toff[0..E] (tiles of 2^tshift rows), the expert of every tile,
// sorted[p] = pair at grouped row p and its inverse inv[f].
__device__ __forceinline__ void group_pairs_warp(const int32_t* ids, int TK, int E, int tshift, int* cnt, int* off,
                                                 int* toff, int* tile_e, int* run, int* sorted, int* inv, int lane) {
  for (int f = lane; f < TK; f += 32) atomicAdd(&cnt[ids[f]], 1);
  __syncwarp();
  warp_expert_scan(cnt, E, tshift, off, toff, tile_e, lane);
  __syncwarp();
  for (int e = lane; e < E; e += 32) run[e] = off[e];
  __syncwarp();
  const unsigned lt = (1u << lane) - 1u;
  for (int base = 0; base < TK; base += 32) {
    const int f = base + lane;
    const int e = f < TK ? ids[f] : -1;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & lt);
    if (f < TK) {
      const int pos = run[e] + rank;
      sorted[pos] = f;
      inv[f] = pos;
    }
    __syncwarp();
    if (f < TK && rank == 0) run[e] += __popc(peers);
    __syncwarp();
  }
}

// Warp: the same grouping for at most 64 pairs (lane l holds pairs l and l + 32)
// and E <= 256 experts, without a pass over the pairs per pair.  A pair's grouped
// row is its expert's offset plus the number of earlier pairs (smaller f) of the
// same expert: within each half of the pairs that ordinal comes from the lanes
// holding the same expert (match.any), and the second half adds the first half's
// count of that expert.  The per-expert counts are a histogram in off[], turned
// into exclusive offsets, together with the tile offsets, by one warp scan over
// the experts (lane l holds experts l*per .. l*per + per - 1).  Writes sorted[p],
// inv[f], off[e] and toff[e] for every e < E; when `tiles` is given also the tile
// list ({expert, row0, rows, 0} at tiles + 4 + 4i, the count in tiles[0]).
__device__ __forceinline__ void group_pairs_small_warp(const int32_t* ids, int TK, int E, int tshift, int* off,
                                                       int* toff, int* sorted, int* inv, int32_t* tiles, int lane) {
  const int f0 = lane, f1 = lane + 32;
  const bool v0 = f0 < TK, v1 = f1 < TK;
  const int id0 = v0 ? ids[f0] : 0, id1 = v1 ? ids[f1] : 0;
  for (int e = lane; e < E; e += 32) off[e] = 0;
  __syncwarp();
  // lanes without a pair get keys no expert has
  const unsigned lt = (1u << lane) - 1u;
  const unsigned m0 = __match_any_sync(0xffffffffu, v0 ? id0 : -1 - lane);
  const unsigned m1 = __match_any_sync(0xffffffffu, v1 ? id1 : -1 - lane);
  if (v0 && (m0 & lt) == 0) off[id0] = __popc(m0);  // first-half count, by the group's first lane
  __syncwarp();
  const int ord0 = __popc(m0 & lt);
  const int ord1 = v1 ? off[id1] + __popc(m1 & lt) : 0;
  __syncwarp();
  if (v1 && (m1 & lt) == 0) off[id1] += __popc(m1);  // plus the second half's
  __syncwarp();
  // exclusive scan of (tiles << 16 | count) over the experts
  const int per = (E + 31) >> 5, e_lo = lane * per;
  const int tr = 1 << tshift;
  int cnt[8];
  int mine = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = e_lo + i;
    cnt[i] = i < per && e < E ? off[e] : 0;
    mine += (((cnt[i] + tr - 1) >> tshift) << 16) + cnt[i];
  }
  int incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  int run = incl - mine;
  __syncwarp();
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = e_lo + i;
    if (i < per && e < E) {
      const int o = run & 0xFFFF, to = run >> 16;
      off[e] = o;
      toff[e] = to;
      if (tiles)
        for (int t = 0; t * tr < cnt[i]; ++t)
          reinterpret_cast<int4*>(tiles + 4)[to + t] = make_int4(e, o + t * tr, min(tr, cnt[i] - t * tr), 0);
      run += (((cnt[i] + tr - 1) >> tshift) << 16) + cnt[i];
    }
  }
  if (tiles && lane == 31) tiles[0] = incl >> 16;
  __syncwarp();
  if (v0) {
    const int r = off[id0] + ord0;
    sorted[r] = f0;
    inv[f0] = r;
  }
  if (v1) {
    const int r = off[id1] + ord1;
    sorted[r] = f1;
    inv[f1] = r;
  }
}

// Thread t of nt: counts[e] and offsets[e] of every expert e < E and offsets[E] =
// TK, straight from the ids of the TK pairs.
__device__ __forceinline__ void expert_counts_offsets(const int32_t* ids, int TK, int E, int32_t* counts,
                                                      int32_t* offsets, int t, int nt) {
  for (int e = t; e <= E; e += nt) {
    int c = 0, o = 0;
    for (int f = 0; f < TK; ++f) {
      const int id = ids[f];
      c += id == e;
      o += id < e;
    }
    if (e < E) counts[e] = c;
    offsets[e] = o;
  }
}

// Block: write the routing results held in shared memory to global memory.
__device__ __forceinline__ void publish_routing(const int* s_ids, const float* s_w, const int* s_sorted,
                                                const int* s_inv, const int* s_cnt, const int* s_off,
                                                const int* s_toff, const int* s_tile_e, int TK, int E,
                                                int tile_rows, int32_t* ids, float* w, int32_t* sorted_rows,
                                                int32_t* inv_pos, int32_t* counts, int32_t* offsets,
                                                int32_t* tiles) {
  const int n_tiles = s_toff[E];
  for (int i = threadIdx.x; i < TK; i += blockDim.x) {
    ids[i] = s_ids[i];
    w[i] = s_w[i];
    sorted_rows[i] = s_sorted[i];
    inv_pos[i] = s_inv[i];
  }
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    counts[e] = s_cnt[e];
    offsets[e] = s_off[e];
  }
  for (int t = threadIdx.x; t < n_tiles; t += blockDim.x) {
    const int e = s_tile_e[t];
    const int r0 = (t - s_toff[e]) * tile_rows;
    reinterpret_cast<int4*>(tiles + 4)[t] = make_int4(e, s_off[e] + r0, min(tile_rows, s_cnt[e] - r0), 0);
  }
  if (threadIdx.x == 0) {
    offsets[E] = s_off[E];
    tiles[0] = n_tiles;
  }
}

// Byte offset of grouped row p's 32-bit scale word for atom column ka, in the
// scale atoms of the tile list (tiles of 2^tshift rows, kt atoms per tile).
__device__ __forceinline__ int64_t row_sf_word(int p, int ka, int kt, const int* s_ids, const int* s_sorted,
                                               const int* s_off, const int* s_toff, int tshift) {
  const int e = s_ids[s_sorted[p]];
  const int r_in_e = p - s_off[e];
  const int b = s_toff[e] + (r_in_e >> tshift);
  const int n = r_in_e & ((1 << tshift) - 1);
  return ((int64_t)b * kt + ka) * kAtomBytes + (n & 31) * 16 + (n >> 5) * 4;
}

}  // namespace moe

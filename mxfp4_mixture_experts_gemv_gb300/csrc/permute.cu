// Expert grouping: histogram, exclusive prefix, stable permutation of the
// (token, slot) pairs by expert, the GEMM tile list, and the gather of the
// quantised activations into grouped order with their scale atoms.
//
// The grouping is deterministic: counts are order-free and every pair's
// position is its rank among equal experts in ascending flat index t*k+j,
// decided with warp match/popcount, never by atomics racing for slots.
#include <cuda_bf16.h>

#include "common.cuh"
#include "quant.cuh"

namespace moe {
namespace {

constexpr int kPermThreads = 256;
constexpr int kPermWarps = kPermThreads / 32;
constexpr int kPermChunk = 2048;          // pairs per CTA
constexpr int kPermPerLane = kPermChunk / kPermThreads;  // 8 pairs per thread

// Pass 1: expert counts of each CTA's chunk of pairs, to part[blk][E].
__global__ void __launch_bounds__(kPermThreads) perm_count_kernel(const int32_t* __restrict__ ids, int TK, int E,
                                                                  int32_t* __restrict__ part) {
  __shared__ int h[256];
  for (int e = threadIdx.x; e < E; e += kPermThreads) h[e] = 0;
  __syncthreads();
  const int base = blockIdx.x * kPermChunk;
  int e[kPermPerLane];
#pragma unroll
  for (int u = 0; u < kPermPerLane; ++u) {
    const int i = base + u * kPermThreads + threadIdx.x;
    // ids come from the top-k kernel and are always in [0, E); the clamp only keeps
    // shared-memory indexing safe whatever the input
    e[u] = i < TK ? min(max(ids[i], 0), E - 1) : -1;
  }
#pragma unroll
  for (int u = 0; u < kPermPerLane; ++u)
    if (e[u] >= 0) atomicAdd(&h[e[u]], 1);
  __syncthreads();
  for (int x = threadIdx.x; x < E; x += kPermThreads) part[(int64_t)blockIdx.x * E + x] = h[x];
}

// Pass 2: every CTA takes the totals and the counts of the CTAs before it, so the
// first grouped row of (its chunk, expert e) is off[e] + the earlier chunks' count;
// inside the chunk each warp owns a contiguous run of pairs and ranks them with
// match/popcount, so every pair's row is its rank among equal experts in
// ascending flat index.  CTA 0 also writes the counts, offsets and tile list.
__global__ void __launch_bounds__(kPermThreads) perm_scatter_kernel(
    const int32_t* __restrict__ ids, int TK, int E, int tile_rows, int max_tiles, const int32_t* __restrict__ part,
    int nb, int32_t* __restrict__ counts, int32_t* __restrict__ offsets, int32_t* __restrict__ sorted_rows,
    int32_t* __restrict__ inv_pos, int32_t* __restrict__ tiles) {
  __shared__ int hist[kPermWarps][257];
  __shared__ int s_tot[257], s_off[258], s_tile_off[258], s_pre[257];
  extern __shared__ int s_tile_e[];  // [max_tiles]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int blk = blockIdx.x;
  for (int e = threadIdx.x; e < E; e += kPermThreads) {
    int tot = 0, pre = 0;
    for (int b = 0; b < nb; ++b) {
      const int c = part[(int64_t)b * E + e];
      tot += c;
      pre += b < blk ? c : 0;
    }
    s_tot[e] = tot;
    s_pre[e] = pre;
  }
  for (int i = threadIdx.x; i < kPermWarps * 257; i += kPermThreads) (&hist[0][0])[i] = 0;
  __syncthreads();
  if (warp == 0) warp_expert_scan(s_tot, E, __ffs(tile_rows) - 1, s_off, s_tile_off, s_tile_e, lane);
  // this warp's run of pairs: ids in registers
  const int per_warp = kPermChunk / kPermWarps;  // 256
  const int start = min(TK, blk * kPermChunk + warp * per_warp), end = min(TK, start + per_warp);
  int ev[per_warp / 32];
#pragma unroll
  for (int u = 0; u < per_warp / 32; ++u) {
    const int i = start + 32 * u + lane;
    ev[u] = i < end ? min(max(ids[i], 0), E - 1) : -1;
  }
#pragma unroll
  for (int u = 0; u < per_warp / 32; ++u)
    if (ev[u] >= 0) atomicAdd(&hist[warp][ev[u]], 1);
  __syncthreads();
  // hist[w][e] becomes the first grouped row of warp w's pairs of expert e
  for (int e = threadIdx.x; e < E; e += kPermThreads) {
    int run = s_off[e] + s_pre[e];
    for (int w = 0; w < kPermWarps; ++w) {
      const int c = hist[w][e];
      hist[w][e] = run;
      run += c;
    }
  }
  if (blk == 0) {
    for (int e = threadIdx.x; e < E; e += kPermThreads) {
      counts[e] = s_tot[e];
      offsets[e] = s_off[e];
      const int cnt = s_tot[e];
      int t = s_tile_off[e];
      for (int r0 = 0; r0 < cnt && t < max_tiles; r0 += tile_rows, ++t)
        reinterpret_cast<int4*>(tiles + 4)[t] = make_int4(e, s_off[e] + r0, min(tile_rows, cnt - r0), 0);
    }
    if (threadIdx.x == 0) {
      offsets[E] = s_off[E];
      tiles[0] = min(s_tile_off[E], max_tiles);
    }
  }
  __syncthreads();
  const unsigned lt_mask = (1u << lane) - 1u;
#pragma unroll
  for (int u = 0; u < per_warp / 32; ++u) {
    if (start + 32 * u >= end) break;  // warp-uniform
    const int i = start + 32 * u + lane;
    const int e = ev[u];
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & lt_mask);
    if (e >= 0) {
      const int pos = hist[warp][e] + rank;
      sorted_rows[pos] = i;
      inv_pos[i] = pos;
    }
    __syncwarp();
    if (e >= 0 && rank == 0) hist[warp][e] += __popc(peers);
    __syncwarp();
  }
}

// Quantise-on-gather, one warp per token: the token's row is quantised to MXFP8
// once and its codes go to each of its k grouped rows, with one scale byte per
// block in each row's atom word (a row's tile and place in it are found by binary
// search over the tile list, staged in shared memory).  The token's codes and
// scales are also published (xq, xs).  Atom words of rows past a tile's rows are
// left as they are: they only feed accumulator columns that are discarded.
constexpr int kGatherWarps = 8;

// dense_tr > 0 (a dense linear, k = 1): the grouping is the identity in tiles of
// dense_tr rows; block 0 writes that tile list and inv_pos and clears the expert
// kernel's zero_words counters (which it reads only after this grid completes).
__global__ void __launch_bounds__(32 * kGatherWarps) gather_tok_kernel(
    const uint16_t* __restrict__ x, int32_t* __restrict__ inv_pos, int32_t* __restrict__ tiles,
    int max_tiles, int T, int k, int H, int fmt, uint8_t* __restrict__ xq, uint8_t* __restrict__ xs,
    uint8_t* __restrict__ xp, uint8_t* __restrict__ xp_sf, int dense_tr, uint32_t* __restrict__ zero,
    int zero_words) {
  const int fp4 = fmt != kActMxfp8 ? 1 : 0;  // codes two per byte
  const bool nv = fmt == kActNvfp4;          // two E4M3 scales per 32-element block
  // the 256 bytes after the last grouped row are read (as zero padding) by the
  // expert kernel's k-tile-plane boxes: keep them zero
  if (blockIdx.x == 0 && threadIdx.x < 16)
    reinterpret_cast<uint4*>(xp + (int64_t)T * k * (H >> fp4))[threadIdx.x] = make_uint4(0, 0, 0, 0);
  if (dense_tr > 0 && blockIdx.x == 0) {
    // the expert kernel takes its first work ticket before it waits for this grid:
    // the counters are cleared and made visible before the dependents may launch
    const int n_tiles = min((T + dense_tr - 1) / dense_tr, max_tiles);
    for (int i = threadIdx.x; i < max(n_tiles, zero_words); i += blockDim.x) {
      if (i < zero_words) zero[i] = 0u;
      if (i < n_tiles) reinterpret_cast<int4*>(tiles + 4)[i] = make_int4(0, i * dense_tr, min(dense_tr, T - i * dense_tr), 0);
    }
    if (threadIdx.x == 0) tiles[0] = n_tiles;
    __threadfence();
    __syncthreads();
  }
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  extern __shared__ int2 s_tl[];  // [max_tiles]: {row0, rows}
  const int n_tiles = dense_tr > 0 ? 0 : min(tiles[0], max_tiles);
  for (int i = threadIdx.x; i < n_tiles; i += blockDim.x) {
    const int4 td = reinterpret_cast<const int4*>(tiles + 4)[i];
    s_tl[i] = make_int2(td.y, td.z);
  }
  __syncthreads();
  const int t = blockIdx.x * kGatherWarps + warp;
  if (t >= T) return;  // whole warp
  const int nbh = H / 32, kth = (H + kTileK - 1) / kTileK;
  // lanes j < k: grouped row p of slot j, its tile b and row n in the tile
  int p = 0, b = 0, n = 0;
  if (dense_tr > 0) {
    if (lane == 0) inv_pos[t] = t;
    p = t;
    b = t / dense_tr;
    n = t - b * dense_tr;
  } else if (lane < k) {
    p = inv_pos[(int64_t)t * k + lane];
    int lo = 0, hi = n_tiles - 1;
    while (lo < hi) {  // last tile whose first row is <= p (tiles are in row order)
      const int mid = (lo + hi + 1) >> 1;
      if (s_tl[mid].x <= p) lo = mid;
      else hi = mid - 1;
    }
    b = lo;
    n = p - s_tl[lo].x;
  }
  const uint4* xr = reinterpret_cast<const uint4*>(x + (int64_t)t * H);
  for (int b0 = 0; b0 < nbh; b0 += 128) {
    uint4 v[4][4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int blk = b0 + 32 * u + lane;
      if (blk < nbh)
#pragma unroll
        for (int q = 0; q < 4; ++q) v[u][q] = __ldg(xr + blk * 4 + q);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int blk = b0 + 32 * u + lane;
      if (b0 + 32 * u >= nbh) break;  // whole warp
      uint4 c[2];
      // padding blocks past H carry the neutral E8M0 scale, or the zero E4M3 scale
      uint32_t sc = nv ? 0u : 127u;
      if (blk < nbh) {
        if (nv) {
          float f[32];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            float g[8];
            bf16x8(v[u][q], g);
#pragma unroll
            for (int i = 0; i < 8; ++i) f[8 * q + i] = g[i];
          }
          uint32_t p0[2], p1[2];
          const uint32_t s0 = nvfp4_block16(f, 1.0f, p0), s1 = nvfp4_block16(f + 16, 1.0f, p1);
          c[0] = make_uint4(p0[0], p0[1], p1[0], p1[1]);
          sc = s0 | (s1 << 8);
          *reinterpret_cast<uint16_t*>(xs + (int64_t)t * (H / 16) + 2 * blk) = (uint16_t)sc;
        } else {
          sc = quant_block_act(v[u], c, fp4);
          xs[(int64_t)t * nbh + blk] = (uint8_t)sc;
        }
        store_block_codes(xq + (int64_t)t * (H >> fp4) + blk * (32 >> fp4), c, fp4);
      }
      // the scales of a 128-element k-tile form one word of the row's atom entry
      // (lanes 4i..4i+3 hold them, lane 4i stores it), or for NVFP4 two words in the
      // tile's two atoms (lanes 4i and 4i+2 store them, padding blocks included)
      const uint32_t word = nv ? (sc | (__shfl_down_sync(0xffffffffu, sc, 1) << 16))
                               : (sc | (__shfl_down_sync(0xffffffffu, sc, 1) << 8) |
                                  (__shfl_down_sync(0xffffffffu, sc, 2) << 16) |
                                  (__shfl_down_sync(0xffffffffu, sc, 3) << 24));
      const bool writes_word = nv ? ((lane & 1) == 0 && (blk >> 2) < kth) : ((lane & 3) == 0 && blk < nbh);
      for (int j = 0; j < k; ++j) {
        const int pj = __shfl_sync(0xffffffffu, p, j), bj = __shfl_sync(0xffffffffu, b, j),
                  nj = __shfl_sync(0xffffffffu, n, j);
        if (blk < nbh) store_block_codes(xp + (int64_t)pj * (H >> fp4) + blk * (32 >> fp4), c, fp4);
        if (writes_word) {
          const int64_t atom = nv ? ((int64_t)bj * kth + (blk >> 2)) * 2 + ((lane >> 1) & 1) : (int64_t)bj * kth + (blk >> 2);
          *reinterpret_cast<uint32_t*>(xp_sf + atom * kAtomBytes + (nj & 31) * 16 + (nj >> 5) * 4) = word;
        }
      }
    }
  }
}

// Routing-weighted combine of the down projection's slot rows, one CTA per token:
// each thread sums four consecutive features over the k slots (fixed slot order,
// fp32) and rounds once to bf16.  A streaming pass over y, used when many tokens
// finish in each down tile and summing inside the expert kernel would stall it.
__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ y, const int32_t* __restrict__ inv_pos,
                                                      const float* __restrict__ topk_w, int k, int H,
                                                      uint16_t* __restrict__ out) {
  const int t = blockIdx.x;
  __shared__ int s_pos[8];
  __shared__ float s_w[8];
  if (threadIdx.x < k) {
    s_pos[threadIdx.x] = inv_pos[(int64_t)t * k + threadIdx.x];
    s_w[threadIdx.x] = topk_w[(int64_t)t * k + threadIdx.x];
  }
  __syncthreads();
  for (int f = 4 * threadIdx.x; f < H; f += 4 * blockDim.x) {
    float4 v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (j < k) v[j] = __ldcs(reinterpret_cast<const float4*>(y + (int64_t)s_pos[j] * H + f));
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (j < k) {
        a.x = fmaf(s_w[j], v[j].x, a.x);
        a.y = fmaf(s_w[j], v[j].y, a.y);
        a.z = fmaf(s_w[j], v[j].z, a.z);
        a.w = fmaf(s_w[j], v[j].w, a.w);
      }
    }
    const uint32_t lo = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(a.x)) |
                        ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(a.y)) << 16);
    const uint32_t hi = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(a.z)) |
                        ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(a.w)) << 16);
    *reinterpret_cast<uint2*>(out + (int64_t)t * H + f) = make_uint2(lo, hi);
  }
}

}  // namespace

cudaError_t launch_combine(const float* y, const int32_t* inv_pos, const float* topk_w, int T, int k, int H,
                           uint16_t* out, cudaStream_t s) {
  combine_kernel<<<T, 256, 0, s>>>(y, inv_pos, topk_w, k, H, out);
  return cudaGetLastError();
}

cudaError_t launch_permute(const int32_t* ids, int TK, int k, int E, int tile_rows, int max_tiles,
                           int32_t* counts, int32_t* offsets, int32_t* sorted_rows, int32_t* inv_pos,
                           int32_t* tiles, int32_t* scratch, cudaStream_t s) {
  (void)k;
  const int nb = (TK + kPermChunk - 1) / kPermChunk;
  perm_count_kernel<<<nb, kPermThreads, 0, s>>>(ids, TK, E, scratch);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  perm_scatter_kernel<<<nb, kPermThreads, (size_t)max_tiles * sizeof(int), s>>>(
      ids, TK, E, tile_rows, max_tiles, scratch, nb, counts, offsets, sorted_rows, inv_pos, tiles);
  return cudaGetLastError();
}

cudaError_t launch_gather_quant(const uint16_t* x, int32_t* inv_pos, int32_t* tiles, int max_tiles, int T,
                                int k, int H, int fmt, uint8_t* xq, uint8_t* xs, uint8_t* xp, uint8_t* xp_sf,
                                cudaStream_t s, int dense_tile_rows, uint32_t* zero, int zero_words) {
  const size_t smem = dense_tile_rows > 0 ? 16 : (size_t)max_tiles * sizeof(int2);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(gather_tok_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  gather_tok_kernel<<<(T + kGatherWarps - 1) / kGatherWarps, 32 * kGatherWarps, smem, s>>>(
      x, inv_pos, tiles, max_tiles, T, k, H, fmt, xq, xs, xp, xp_sf, dense_tile_rows, zero, zero_words);
  return cudaGetLastError();
}

}  // namespace moe

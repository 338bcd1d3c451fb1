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

constexpr int kPermThreads = 1024;
constexpr int kPermWarps = kPermThreads / 32;

__global__ void __launch_bounds__(kPermThreads) permute_kernel(
    const int32_t* __restrict__ ids, int TK, int E, int tile_rows, int max_tiles, int32_t* __restrict__ counts,
    int32_t* __restrict__ offsets, int32_t* __restrict__ sorted_rows, int32_t* __restrict__ inv_pos,
    int32_t* __restrict__ tiles) {
  __shared__ int hist[kPermWarps][257];
  __shared__ int s_off[258];
  __shared__ int s_tile_off[258];
  extern __shared__ int s_tile_e[];  // [max_tiles]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < kPermWarps * 257; i += kPermThreads) (&hist[0][0])[i] = 0;
  __syncthreads();
  const int chunk = (TK + kPermWarps - 1) / kPermWarps;
  const int start = min(TK, warp * chunk), end = min(TK, start + chunk);
  // ids come from the top-k kernel and are always in [0, E); the clamp only keeps
  // shared-memory indexing safe whatever the input.  Each lane loads its ids in
  // batches of kBatch independent loads.
  constexpr int kBatch = 16;
  for (int b0 = start; b0 < end; b0 += 32 * kBatch) {
    int e[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int i = b0 + 32 * u + lane;
      e[u] = i < end ? min(max(ids[i], 0), E - 1) : -1;
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u)
      if (e[u] >= 0) atomicAdd(&hist[warp][e[u]], 1);
  }
  __syncthreads();
  __shared__ int s_cnt[257];
  if (threadIdx.x < E) {
    int c = 0;
    for (int w = 0; w < kPermWarps; ++w) c += hist[w][threadIdx.x];
    counts[threadIdx.x] = c;
    s_cnt[threadIdx.x] = c;
  }
  __syncthreads();
  if (warp == 0) warp_expert_scan(s_cnt, E, __ffs(tile_rows) - 1, s_off, s_tile_off, s_tile_e, lane);
  __syncthreads();
  if (threadIdx.x < E) {
    const int e = threadIdx.x;
    int run = s_off[e];
    for (int w = 0; w < kPermWarps; ++w) {
      const int c = hist[w][e];
      hist[w][e] = run;
      run += c;
    }
    offsets[e] = s_off[e];
    // tile list entries of expert e
    const int cnt = s_off[e + 1] - s_off[e];
    int t = s_tile_off[e];
    for (int r0 = 0; r0 < cnt && t < max_tiles; r0 += tile_rows, ++t) {
      int4 td = make_int4(e, s_off[e] + r0, min(tile_rows, cnt - r0), 0);
      reinterpret_cast<int4*>(tiles + 4)[t] = td;
    }
  }
  if (threadIdx.x == 0) {
    offsets[E] = s_off[E];
    tiles[0] = min(s_tile_off[E], max_tiles);
  }
  __syncthreads();
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int b0 = start; b0 < end; b0 += 32 * kBatch) {
    int eb[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int i = b0 + 32 * u + lane;
      eb[u] = i < end ? min(max(ids[i], 0), E - 1) : -1;
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      if (b0 + 32 * u >= end) break;  // warp-uniform
      const int i = b0 + 32 * u + lane;
      const int e = eb[u];
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
}

// One CTA per tile: quantise the tile's token rows to MXFP8 straight into grouped
// order (x -> Xp rows and their scale atoms); the row of a token's first slot also
// publishes the token's codes (xq, xs).  Atom words of rows past the tile's rows
// are left as they are: they only feed accumulator columns that are discarded.
__global__ void __launch_bounds__(512) gather_quant_kernel(const uint16_t* __restrict__ x,
                                                           const int32_t* __restrict__ sorted_rows,
                                                           const int32_t* __restrict__ tiles, int k, int H, int I,
                                                           uint8_t* __restrict__ xq, uint8_t* __restrict__ xs,
                                                           uint8_t* __restrict__ xp, uint8_t* __restrict__ xp_sf,
                                                           uint8_t* __restrict__ hq_sf) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int b = blockIdx.x;
  if (b >= tiles[0]) return;
  const int4 td = reinterpret_cast<const int4*>(tiles + 4)[b];
  const int row0 = td.y, rows = td.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nbh = H / 32;
  const int kth = (H + kTileK - 1) / kTileK;
  (void)I;
  (void)hq_sf;
  __shared__ uint8_t s_scale[16][kRouteSmallMaxH / 32];
  for (int r = warp; r < rows; r += 16) {
    const int f = sorted_rows[row0 + r], t = f / k;
    const bool first = (f % k) == 0;
    const uint4* xr = reinterpret_cast<const uint4*>(x + (int64_t)t * H);
    // up to four blocks per lane per round, every load of the round in flight
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
        if (blk < nbh) {
          uint4 c[2];
          const uint8_t sc = quant_block_vals(v[u], c);
          uint4* dst = reinterpret_cast<uint4*>(xp + (int64_t)(row0 + r) * H + blk * 32);
          dst[0] = c[0];
          dst[1] = c[1];
          s_scale[warp][blk] = sc;
          if (first) {
            uint4* q = reinterpret_cast<uint4*>(xq + (int64_t)t * H + blk * 32);
            q[0] = c[0];
            q[1] = c[1];
            xs[(int64_t)t * nbh + blk] = sc;
          }
        }
      }
    }
    __syncwarp();
    for (int ka = lane; ka < kth; ka += 32) {
      uint32_t wv = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int kb = 4 * ka + j;
        wv |= (uint32_t)(kb < nbh ? s_scale[warp][kb] : 127) << (8 * j);
      }
      *reinterpret_cast<uint32_t*>(xp_sf + ((int64_t)b * kth + ka) * kAtomBytes + (r & 31) * 16 + (r >> 5) * 4) = wv;
    }
    __syncwarp();
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
                           int32_t* tiles, cudaStream_t s) {
  (void)k;
  permute_kernel<<<1, kPermThreads, (size_t)max_tiles * sizeof(int), s>>>(ids, TK, E, tile_rows, max_tiles, counts,
                                                                           offsets, sorted_rows, inv_pos, tiles);
  return cudaGetLastError();
}

cudaError_t launch_gather_quant(const uint16_t* x, const int32_t* sorted_rows, const int32_t* tiles, int max_tiles,
                                int k, int H, int I, uint8_t* xq, uint8_t* xs, uint8_t* xp, uint8_t* xp_sf,
                                uint8_t* hq_sf, cudaStream_t s) {
  gather_quant_kernel<<<max_tiles, 512, 0, s>>>(x, sorted_rows, tiles, k, H, I, xq, xs, xp, xp_sf, hq_sf);
  return cudaGetLastError();
}

}  // namespace moe

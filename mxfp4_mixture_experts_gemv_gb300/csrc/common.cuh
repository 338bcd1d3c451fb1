// Internal definitions shared by the kernels of the MXFP4 MoE layer (sm_103a).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "../../include/moe.h"

namespace moe {

// ---------------------------------------------------------------------------------------
// Packed weight buffer (written by moe_pack_weights), layout version 2.
//
// Expert weights are stored tile-contiguous so that every pipeline stage of the
// grouped GEMM fetches one contiguous block with one TMA box:
//   data  [E][m_tile][k_tile][rows_m][64 B]: 128 weight rows (64 for a tail
//         m-tile) x 128 contraction elements of packed E2M1 per tile, 8 KB.
//         The contraction axis is padded with zero nibbles to Kp = round_up(K, 128)
//         (TMA's 4-bit unpacking mode works on 128-element rows); the row count per
//         expert is padded to a multiple of 64 with zero rows.
//   sf    [E][m_tile][k_tile][512 B]: E8M0 scales in scale-factor atoms; byte
//         (r%32)*16 + (r/32)*4 + (kb%4) holds the scale of tile row r, 32-element
//         block kb of the tile.  Padding holds code 127 (1.0).
//   bias  [E][rows] fp32.
// gate_up rows are interleaved: m-tile t holds gate rows 64t..64t+63 in tile rows
// 0..63 and the matching up rows in tile rows 64..127, so one accumulator tile
// carries both halves of the SwiGLU.
// ---------------------------------------------------------------------------------------
constexpr uint32_t kPackedMagic = 0x4D584645u;  // "EFXM"
constexpr uint32_t kPackedVersion = 2;
constexpr int kTileM = 128;   // weight rows per tile (MMA M)
constexpr int kTileK = 128;   // contraction elements per pipeline stage
constexpr int kAtomBytes = 512;
constexpr int kTileRowBytes = kTileK / 2;  // packed bytes of one tile row

// Weight formats of a packed buffer: MXFP4 (E2M1, one E8M0 scale per 32
// elements) or NVFP4 (E2M1, one E4M3 scale per 16 elements and a global fp32
// scale per projection).  An NVFP4 buffer holds two scale atoms per k-tile: atom
// j covers the 16-element blocks 4j..4j+3 of the tile's 128 elements, byte
// (r%32)*16 + (r/32)*4 + (block%4) for tile row r.
enum : int32_t { kWeightsMxfp4 = 0, kWeightsNvfp4 = 1, kWeightsDense = 2 };

struct PackedHeader {
  uint32_t magic, version;
  int32_t E, H, I, Hp, Ip, gu_mtiles, d_mtiles, gu_ktiles, d_ktiles;
  int32_t gu_rows_stored, d_rows_stored, wfmt;
  uint64_t off_gu_data, off_gu_sf, off_gu_bias, off_d_data, off_d_sf, off_d_bias, total;
};

// NVFP4 buffers: the largest magnitude of each projection's weights (fp32 bits,
// gate_up then down) sits at this offset of the 1 KB header area; the global
// scale of a projection is amax / (6 * 448) (nvfp4_global_scale).
constexpr uint32_t kAmaxOffset = 512;
__host__ __device__ inline float nvfp4_global_scale(float amax) { return amax > 0.f ? amax / 2688.0f : 1.0f; }

inline int64_t round_up(int64_t a, int64_t b) { return (a + b - 1) / b * b; }

inline bool packed_layout(const moe_dims& d, PackedHeader* hd, int32_t wfmt = kWeightsMxfp4) {
  if (d.E <= 0 || d.H <= 0 || d.I <= 0) return false;
  if (d.E > 256 || d.H % 32 || d.I % 64) return false;
  PackedHeader h = {};
  h.magic = kPackedMagic;
  h.version = kPackedVersion;
  h.E = d.E; h.H = d.H; h.I = d.I;
  h.Hp = (int32_t)round_up(d.H, kTileK);
  h.Ip = (int32_t)round_up(d.I, kTileK);
  h.gu_mtiles = 2 * d.I / kTileM;
  h.d_mtiles = (int32_t)((d.H + kTileM - 1) / kTileM);
  h.gu_ktiles = h.Hp / kTileK;
  h.d_ktiles = h.Ip / kTileK;
  h.gu_rows_stored = 2 * d.I;
  h.d_rows_stored = (int32_t)round_up(d.H, 64);
  h.wfmt = wfmt;
  const int atoms = wfmt == kWeightsNvfp4 ? 2 : 1;  // scale atoms per k-tile
  uint64_t off = 1024;
  auto take = [&](uint64_t bytes) { uint64_t o = off; off = (uint64_t)round_up(off + bytes, 1024); return o; };
  h.off_gu_data = take((uint64_t)d.E * h.gu_rows_stored * h.gu_ktiles * kTileRowBytes);
  h.off_gu_sf = take((uint64_t)d.E * h.gu_mtiles * h.gu_ktiles * atoms * kAtomBytes);
  h.off_gu_bias = take((uint64_t)d.E * 2 * d.I * 4);
  h.off_d_data = take((uint64_t)d.E * h.d_rows_stored * h.d_ktiles * kTileRowBytes);
  h.off_d_sf = take((uint64_t)d.E * h.d_mtiles * h.d_ktiles * atoms * kAtomBytes);
  h.off_d_bias = take((uint64_t)d.E * d.H * 4);
  h.total = off;
  *hd = h;
  return true;
}

// A dense MXFP4 linear (N outputs, K inputs) packed like one expert's down
// projection: E = 1, H = N output rows (padded to a multiple of 64; a 64-row tail
// tile), I = K contraction elements (padded to a multiple of 128), one scale atom
// per 128 x 128 tile, fp32 bias; no gate_up section.
inline bool dense_layout(int N, int K, PackedHeader* hd) {
  if (N <= 0 || K <= 0 || N % 64 || K % 32) return false;
  PackedHeader h = {};
  h.magic = kPackedMagic;
  h.version = kPackedVersion;
  h.E = 1; h.H = N; h.I = K;
  h.Hp = (int32_t)round_up(N, kTileK);
  h.Ip = (int32_t)round_up(K, kTileK);
  h.gu_mtiles = 0;
  h.d_mtiles = (int32_t)((N + kTileM - 1) / kTileM);
  h.gu_ktiles = 0;
  h.d_ktiles = h.Ip / kTileK;
  h.gu_rows_stored = 0;
  h.d_rows_stored = N;
  h.wfmt = kWeightsDense;
  uint64_t off = 1024;
  auto take = [&](uint64_t bytes) { uint64_t o = off; off = (uint64_t)round_up(off + bytes, 1024); return o; };
  h.off_gu_data = h.off_gu_sf = h.off_gu_bias = off;
  h.off_d_data = take((uint64_t)h.d_rows_stored * h.d_ktiles * kTileRowBytes);
  h.off_d_sf = take((uint64_t)h.d_mtiles * h.d_ktiles * kAtomBytes);
  h.off_d_bias = take((uint64_t)N * 4);
  h.total = off;
  *hd = h;
  return true;
}

// Row (in 64-byte units) of the first row of data tile (e, m, kt) in the
// tile-contiguous layout; `rows_stored` rows per expert, the last m-tile may be short.
__host__ __device__ inline int64_t tile_row0(int e, int m, int kt, int rows_stored, int k_tiles) {
  const int rows_m = (rows_stored - m * kTileM) < kTileM ? (rows_stored - m * kTileM) : kTileM;
  return ((int64_t)e * rows_stored + (int64_t)m * kTileM) * k_tiles + (int64_t)kt * rows_m;
}

// Token counts up to this take the fused small-batch routing kernel.
constexpr int kRouteSmallMaxT = 32;
constexpr int kRouteSmallMaxH = 8192;
// dynamic shared memory of the small-batch routing kernel: (T + 1) rows of H bf16
constexpr size_t kRouteSmallMaxSmem = 200 * 1024;
inline bool route_small_fits(int T, int H) {
  return T <= kRouteSmallMaxT && H <= kRouteSmallMaxH && (size_t)(T + 1) * H * 2 <= kRouteSmallMaxSmem;
}

// Cluster routing (a few tokens): the router rows of a CTA's experts (E / 8 of
// them on the smallest cluster) and the T token rows sit in shared memory.
constexpr int kRouteClusterMaxT = 8;
constexpr size_t kRouteClusterMaxSmem = 200 * 1024;
bool route_cluster_fits(int T, int E, int H);

// Measurement overrides of the plan (moe_set_plan), process-wide: token rows per
// tile (0 = automatic) and the routing path (kRouteAuto = automatic).
enum : int { kRouteAuto = 0, kRouteCluster = 1, kRouteGrid = 2, kRouteTensorCore = 3 };
enum : int { kExpertAuto = 0, kExpertWeightsM = 1, kExpertTokensM = 2, kExpertCudaCores = 3 };
int plan_tile_rows();
int plan_route();
int plan_expert();

// Activation formats: MXFP8 (one E4M3 code byte per element, one E8M0 scale per
// 32), MXFP4 (two E2M1 codes per byte, one E8M0 scale per 32) and NVFP4 (two
// E2M1 codes per byte, one E4M3 scale per 16, unit global scale; scale atoms in
// pairs per k-tile as in an NVFP4 weight buffer).
enum ActFormat : int { kActMxfp8 = 0, kActMxfp4 = 1, kActNvfp4 = 2 };

// Token rows per tile of the grouped GEMM for the weights-on-M kernel, from the
// measured plan sweep on the gpt-oss-shaped layer (E = 128, top-4): twice the
// average rows per expert, rounded up to a power of two, within [8, 128].  Small
// tiles take the pipeline shape that streams weights fastest (four k-tiles per
// stage) and most experts still fit one tile, so each weight byte is read once;
// the fastest height in the sweep was 8 rows up to T = 128 (2 to 4 rows per
// expert on average), then 16, 32, 64 at T = 256, 512, 1024 and 128 from 2048.
inline int tile_rows_weights_m(int T, int k, int E) {
  const int64_t avg = ((int64_t)T * k + E - 1) / E;  // average token rows per expert
  int tr = 8;
  while (tr < 128 && tr < 2 * avg) tr *= 2;
  return tr;
}

// Average token rows per expert from which MXFP8 and MXFP4 layers take 128-row tiles
// and the tokens-on-M kernel: measured fastest from 8 rows per expert up to T = 8192
// on the gpt-oss layer (MXFP8: T = 256 327.7 against 330.2 us for 16-row tiles,
// T = 512 340 against 348, T = 1024 364 against 371; MXFP4: T = 256 287 against 297,
// T = 512 295 against 319, T = 1024 322 against 346).  NVFP4 layers keep the
// weights-on-M kernel.
constexpr int kTokensMMinAvgRows = 8;

// The tile height of a layer forward in activation format fmt (the plan's, if it
// forces one).
inline int tile_rows_for(int T, int k, int E, int fmt) {
  if (const int forced = plan_tile_rows()) return forced;
  const int64_t avg = ((int64_t)T * k + E - 1) / E;
  if ((fmt == kActMxfp8 || fmt == kActMxfp4) && avg >= kTokensMMinAvgRows) return 128;
  return tile_rows_weights_m(T, k, E);
}

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

inline bool workspace_layout(const moe_dims& d, int T, int k, moe_workspace_layout* L, int fmt = kActMxfp8) {
  if (T < 0 || k <= 0) return false;
  const int64_t TK = (int64_t)T * k;
  const int tr = tile_rows_for(T, k, d.E, fmt);
  const int64_t max_tiles = TK / tr + (TK < d.E ? TK : d.E) + 1;
  // the sections that scale with the tile count are sized for the smallest tile
  // height any activation format takes, so every format has the same offsets
  const int tr_min = plan_tile_rows() ? tr : std::min(tr, tile_rows_weights_m(T, k, d.E));
  const int64_t cap_tiles = TK / tr_min + (TK < d.E ? TK : d.E) + 1;
  const int64_t kth = (d.H + kTileK - 1) / kTileK, kti = (d.I + kTileK - 1) / kTileK;
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t r = o; o = align256(o + bytes); return r; };
  moe_workspace_layout l = {};
  l.status = take(16);
  l.done_gu = take((size_t)cap_tiles * 4);
  l.done_tok = take((size_t)T * ((d.H + kTileM - 1) / kTileM) * 4);
  l.grid_bar = take(16);
  l.zero_bytes = o;  // status words and the counters above start at zero every forward
  l.logits = take((size_t)T * d.E * 4);
  l.topk_ids = take((size_t)TK * 4);
  l.topk_w = take((size_t)TK * 4);
  // sized for every activation format: one code byte per element, one scale per
  // 16 elements (NVFP4; the 32-element formats use half), two scale atoms per
  // k-tile (NVFP4; the others use the first of each pair's space)
  l.xq = take((size_t)T * d.H);
  l.xs = take((size_t)T * (d.H / 16));
  l.counts = take((size_t)d.E * 4);
  l.offsets = take((size_t)(d.E + 1) * 4);
  l.sorted_rows = take((size_t)TK * 4);
  l.inv_pos = take((size_t)TK * 4);
  l.tiles = take((size_t)(4 + 4 * cap_tiles) * 4);
  l.xp = take((size_t)TK * d.H + 256);
  l.xp_sf = take((size_t)cap_tiles * kth * 2 * kAtomBytes);
  l.hq = take((size_t)TK * d.I + 256);
  l.hq_sf = take((size_t)cap_tiles * kti * 2 * kAtomBytes);
  l.y = take((size_t)TK * d.H * 4);
  l.total = o;
  l.max_tiles = (int32_t)max_tiles;
  l.tile_rows = tr;
  *L = l;
  return true;
}

// Status words (first 16 bytes of the workspace).
enum : uint32_t {
  kStatusTimeoutProducer = 1u << 0,
  kStatusTimeoutMma = 1u << 1,
  kStatusTimeoutEpilogue = 1u << 2,
  kStatusTimeoutDrain = 1u << 3,
  kStatusTimeoutRouting = 1u << 4,  // the small-batch routing grid's barrier
  kStatusBadWeights = 1u << 5,      // the packed buffer's header does not match the forward
};

// Bounded waits give up after this many nanoseconds unless the host sets
// another limit (a healthy wait lasts microseconds).
constexpr uint64_t kWaitLimitNsDefault = 2000000000ull;
// Drains (waiting for copies and MMAs already issued, which always complete)
// are bounded separately.
constexpr uint64_t kDrainLimitNs = 200000000ull;

// The limit every kernel launched from now on passes to its bounded waits
// (moe_set_wait_limit_ns), and the failure-detection hook's mask of waits made
// unreachable (moe_debug_hold_waits).  Both are process-wide host settings.
uint64_t wait_limit_ns();
int debug_hold_waits();

// moe_forward's argument checks (everything but the workspace), in its order.
moe_status check_forward_args(const moe_dims& d, const void* hidden, int32_t T, const void* router_w,
                              const void* router_b, const void* packed, int32_t top_k, const void* out);
// Synchronise `stream`, then read four status words at a device address.
moe_status read_status_words(const void* status_words, void* stream);

// Record a status and its message for moe_last_error (defined with the C ABI).
moe_status report_error(moe_status st, const char* fmt, ...);

// Kernel launchers (defined in the .cu files).
cudaError_t launch_pack(const moe_dims& d, const PackedHeader& h, const moe_mxfp4_weights& w,
                        uint8_t* packed, cudaStream_t s);
// The MXFP4 checkpoint converted to NVFP4 while packing (h.wfmt == kWeightsNvfp4).
cudaError_t launch_pack_nvfp4(const PackedHeader& h, const moe_mxfp4_weights& w, uint8_t* packed, cudaStream_t s);
cudaError_t launch_router_tc(const uint16_t* x, const uint16_t* wr, const uint16_t* br, int T, int H, int E, int k,
                             float* logits, int32_t* ids, float* w, uint32_t* status, cudaStream_t s);
// Grouping in two passes over chunks of pairs; `scratch` holds one count per
// (chunk, expert): ceil(TK / 2048) * E ints.
cudaError_t launch_permute(const int32_t* ids, int TK, int k, int E, int tile_rows, int max_tiles,
                           int32_t* counts, int32_t* offsets, int32_t* sorted_rows, int32_t* inv_pos,
                           int32_t* tiles, int32_t* scratch, cudaStream_t s);
// dense_tile_rows > 0: a dense linear (k = 1, identity grouping); the kernel also
// writes the tile list and inv_pos and clears the first zero_words words at zero.
cudaError_t launch_gather_quant(const uint16_t* x, int32_t* inv_pos, int32_t* tiles, int max_tiles, int T,
                                int k, int H, int fmt, uint8_t* xq, uint8_t* xs, uint8_t* xp, uint8_t* xp_sf,
                                cudaStream_t s, int dense_tile_rows = 0, uint32_t* zero = nullptr,
                                int zero_words = 0);

cudaError_t launch_residual_rmsnorm(float* x_res, const uint16_t* layer_out, int T, int H, float eps,
                                    uint16_t* hidden, cudaStream_t s);

// Token counts up to this take the dense linears' CUDA-core path by default.
constexpr int kDenseCudaCoresMaxT = 4;

// Workspace of a dense linear for T tokens: offsets from its base.
struct DenseWorkspace {
  size_t status, done, sched, zero_bytes, tiles, inv_pos, xq, xs, xp, xp_sf, partial, total;
  int max_tiles, tile_rows, k_chunks;
};
inline bool dense_workspace(int N, int K, int T, int num_sms, DenseWorkspace* w) {
  if (N <= 0 || K <= 0 || T < 0) return false;
  DenseWorkspace d = {};
  d.tile_rows = plan_tile_rows() ? plan_tile_rows() : tile_rows_weights_m(T, 1, 1);
  d.max_tiles = T / d.tile_rows + 2;
  const int kt = (K + kTileK - 1) / kTileK, mt = (N + kTileM - 1) / kTileM;
  // K chunks of the CUDA-core path: about two CTAs per SM, and at most 96 k-tiles
  // (4 tokens x 96 x 128 fp32 = 192 KiB of shared memory) per chunk
  d.k_chunks = std::max((kt + 95) / 96, std::max(1, std::min(kt, (2 * num_sms + mt - 1) / mt)));
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t r = o; o = align256(o + bytes); return r; };
  d.status = take(16);
  d.done = take((size_t)d.max_tiles * 4);
  d.sched = take(16);
  d.zero_bytes = o;
  d.tiles = take((size_t)(4 + 4 * d.max_tiles) * 4);
  d.inv_pos = take((size_t)T * 4);
  d.xq = take((size_t)T * K);
  d.xs = take((size_t)T * (K / 16));
  d.xp = take((size_t)T * K + 256);
  d.xp_sf = take((size_t)d.max_tiles * kt * 2 * kAtomBytes);
  d.partial = take((size_t)d.k_chunks * std::min(T, 4) * N * 4);
  d.total = o;
  *w = d;
  return true;
}

// Dense linear for T tokens on the CUDA cores (else the tensor cores), from the
// measured crossover on GB300 (graph-replayed calls, weights streamed from HBM): the
// GEMV has no quantise-and-place pass but decodes every element on the CUDA cores
// (E2M1 -> f16 -> f32), so it wins up to about 2^25 multiply-adds (T * N * K): 2880 x
// 2880 at T = 4 14.9 against 15.3 us, 5120 x 2880 at T = 2 15.2 against 15.2; from
// about 4.7e7 the tensor cores win (2880 x 4096 at T = 4 16.7 against 18.7 us, 16384 x
// 2880 at T = 1 16.8 against 24.7, the LM head 201,088 x 2880 at T = 1 65 against 134).
constexpr int64_t kDenseCudaCoresMaxMacs = (int64_t)1 << 25;
inline bool dense_cuda_cores_for(int T, int N, int K) {
  return T <= kDenseCudaCoresMaxT && (int64_t)T * N * K <= kDenseCudaCoresMaxMacs;
}

// Dense linears (dense.cu).
cudaError_t launch_dense_quantize_weights(int N, int K, const uint16_t* w, uint8_t* blocks, uint8_t* scales,
                                          cudaStream_t s);
cudaError_t launch_dense_pack(const PackedHeader& h, const uint8_t* blocks, const uint8_t* scales, const uint16_t* bias,
                              uint8_t* packed, cudaStream_t s);
// CUDA-core path for a few tokens: out (or fp32 partial sums over K chunks) of
// MXFP8(x) . W^T + b; k_chunks > 1 writes partial[c][t][n] and a second pass sums.
cudaError_t launch_dense_gemv(const PackedHeader& h, const uint8_t* packed, const uint16_t* x, int T, int k_chunks,
                              float* partial, uint16_t* out, cudaStream_t s);

struct RouteSmallOut {
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
  uint8_t* hq_sf;
  int32_t* grid_bar;
  uint32_t* status;
};
cudaError_t launch_route_small(const uint16_t* x, const uint16_t* wr, const uint16_t* br, int T, int H, int E, int I,
                               int k, int tile_rows, int max_tiles, bool fp4, const RouteSmallOut& o, cudaStream_t s);

struct RouteClusterOut {
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
  uint32_t* zero;  // the workspace's zero-initialised words, cleared by the kernel
  int zero_words;
  uint32_t* status;
  int32_t* flags;  // two words inside the zero-initialised ones: tile list published, CTAs done
};
// *ctas: the routing CTAs the launch runs (the count the second flag reaches)
cudaError_t launch_route_cluster(const uint16_t* x, const uint16_t* wr, const uint16_t* br, int T, int H, int E,
                                 int k, int tile_rows, int fmt, const RouteClusterOut& o, int* ctas,
                                 cudaStream_t s);

struct ExpertMlpBuffers {
  const uint8_t* xp;        // gate_up B rows [TK][H]
  const uint8_t* xp_sf;     // gate_up B scale atoms
  uint8_t* hq;              // [TK][I]
  uint8_t* hq_sf;           // down B scale atoms
  float* y;                 // [TK][H]
  uint16_t* out;            // bf16 [T][H]
  const int32_t* tiles;
  const int32_t* sorted_rows;
  const int32_t* inv_pos;
  const float* topk_w;
  int32_t* done_gu;
  int32_t* done_tok;
  int32_t* sched;  // tile claim counter, zero at launch
  uint32_t* status;
  bool fused_combine;  // false: launch_combine sums the slots after the expert kernel
  // Routing that publishes its results through two flags (tile list, then CTAs
  // whose grouped rows are written) while it still runs: the expert kernel starts
  // its weight copies on the first and its activation copies when the second
  // reaches route_ctas.  route_ctas = 0: the routing grid completes first.
  const int32_t* route_flags;
  int route_ctas;
};
// out[t] = bf16(sum_j w[t][j] * y[inv_pos[t][j]]), slots in order, fp32 sums.
cudaError_t launch_combine(const float* y, const int32_t* inv_pos, const float* topk_w, int T, int k, int H,
                           uint16_t* out, cudaStream_t s);
// fmt: activations (xp, hq) in MXFP8 (tcgen05 kind::mxf8f6f4), MXFP4
// (kind::mxf4) or NVFP4 with NVFP4 weights (kind::mxf4nvf4).
cudaError_t launch_expert_mlp(const PackedHeader& h, const uint8_t* packed, const ExpertMlpBuffers& b, int T, int k,
                              int max_tiles, int tile_rows, int num_sms, int fmt, cudaStream_t s);
// The same layer for 128-row token tiles with the tokens in the MMA M slot and two
// weight tiles in N (any activation format); y is combined by launch_combine.
cudaError_t launch_expert_swap(const PackedHeader& h, const uint8_t* packed, const ExpertMlpBuffers& b, int T, int k,
                               int max_tiles, int num_sms, int fmt, cudaStream_t s);
// whether the packed layer's weight tiles pair up as the tokens-on-M kernel reads them
bool expert_swap_supported(const PackedHeader& h);

}  // namespace moe

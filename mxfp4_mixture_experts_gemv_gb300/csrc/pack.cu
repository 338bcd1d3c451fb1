// Weight repacker: checkpoint-layout MXFP4 expert weights -> the tiled layout the
// grouped GEMM streams (see common.cuh for the layout).
#include "common.cuh"

namespace moe {
namespace {

// Packed gate_up row -> checkpoint row: tile t = gate rows 64t.. then up rows I+64t..
__device__ __forceinline__ int gu_source_row(int pr, int I) {
  const int t = pr >> 7, w = pr & 127;
  return w < 64 ? 64 * t + w : I + 64 * t + (w - 64);
}

struct PackArgs {
  PackedHeader h;
  moe_mxfp4_weights w;
  uint8_t* packed;
};

// Data tiles: one thread per 16-byte chunk (32 elements) of the tile-contiguous layout.
__global__ void pack_data_kernel(PackArgs a, int gate_up) {
  const PackedHeader& h = a.h;
  const int rows = gate_up ? 2 * h.I : h.H;
  const int rows_stored = gate_up ? h.gu_rows_stored : h.d_rows_stored;
  const int K = gate_up ? h.H : h.I;
  const int kt_n = gate_up ? h.gu_ktiles : h.d_ktiles;
  const int nb = K / 32;
  const uint4* src = reinterpret_cast<const uint4*>(gate_up ? a.w.gate_up_blocks : a.w.down_blocks);
  uint4* dst = reinterpret_cast<uint4*>(a.packed + (gate_up ? h.off_gu_data : h.off_d_data));
  const int64_t per_expert = (int64_t)rows_stored * kt_n * 4;  // chunks
  const int64_t per_mtile = (int64_t)kTileM * kt_n * 4;
  const int64_t total = (int64_t)h.E * per_expert;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int e = (int)(i / per_expert);
    const int64_t q = i - (int64_t)e * per_expert;
    const int m = (int)(q / per_mtile);
    const int rows_m = min(kTileM, rows_stored - m * kTileM);
    const int64_t rem = q - (int64_t)m * per_mtile;
    const int kt = (int)(rem / (rows_m * 4));
    const int rem2 = (int)(rem - (int64_t)kt * rows_m * 4);
    const int r = rem2 >> 2, j = rem2 & 3;
    const int pr = m * kTileM + r;          // packed row
    const int kb = kt * 4 + j;              // source 32-element block
    uint4 v = make_uint4(0, 0, 0, 0);
    if (pr < rows && kb < nb) {
      const int sr = gate_up ? gu_source_row(pr, h.I) : pr;
      v = src[((int64_t)e * rows + sr) * nb + kb];
    }
    dst[i] = v;
  }
}

// Scale atoms: one thread per atom byte.
__global__ void pack_sf_kernel(PackArgs a, int gate_up) {
  const PackedHeader& h = a.h;
  const int rows = gate_up ? 2 * h.I : h.H;
  const int K = gate_up ? h.H : h.I;
  const int nb = K / 32;
  const int mt = gate_up ? h.gu_mtiles : h.d_mtiles;
  const int kt = gate_up ? h.gu_ktiles : h.d_ktiles;
  const uint8_t* src = gate_up ? a.w.gate_up_scales : a.w.down_scales;
  uint8_t* dst = a.packed + (gate_up ? h.off_gu_sf : h.off_d_sf);
  const int64_t total = (int64_t)h.E * mt * kt * kAtomBytes;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int j = (int)(i % kAtomBytes);
    int64_t q = i / kAtomBytes;
    const int ktile = (int)(q % kt);
    q /= kt;
    const int mtile = (int)(q % mt);
    const int e = (int)(q / mt);
    const int r = (j >> 4) + 32 * ((j & 15) >> 2);
    const int kb = ktile * 4 + (j & 3);
    const int pr = mtile * kTileM + r;
    uint8_t v = 127;
    if (pr < rows && kb < nb) {
      const int sr = gate_up ? gu_source_row(pr, h.I) : pr;
      v = src[((int64_t)e * rows + sr) * nb + kb];
    }
    dst[i] = v;
  }
}

__global__ void pack_bias_kernel(PackArgs a) {
  const PackedHeader& h = a.h;
  float* gub = reinterpret_cast<float*>(a.packed + h.off_gu_bias);
  float* db = reinterpret_cast<float*>(a.packed + h.off_d_bias);
  const int64_t ngu = (int64_t)h.E * 2 * h.I, nd = (int64_t)h.E * h.H;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < ngu + nd;
       i += (int64_t)gridDim.x * blockDim.x) {
    if (i < ngu) {
      const int pr = (int)(i % (2 * h.I));
      const int64_t e = i / (2 * h.I);
      const uint16_t b = a.w.gate_up_bias[e * 2 * h.I + gu_source_row(pr, h.I)];
      gub[i] = __uint_as_float((uint32_t)b << 16);
    } else {
      const int64_t j = i - ngu;
      db[j] = __uint_as_float((uint32_t)a.w.down_bias[j] << 16);
    }
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) *reinterpret_cast<PackedHeader*>(a.packed) = h;
}

}  // namespace

cudaError_t launch_pack(const moe_dims& d, const PackedHeader& h, const moe_mxfp4_weights& w,
                        uint8_t* packed, cudaStream_t s) {
  (void)d;
  PackArgs a{h, w, packed};
  const int threads = 256, blocks = 4096;
  pack_data_kernel<<<blocks, threads, 0, s>>>(a, 1);
  pack_data_kernel<<<blocks, threads, 0, s>>>(a, 0);
  pack_sf_kernel<<<blocks, threads, 0, s>>>(a, 1);
  pack_sf_kernel<<<blocks, threads, 0, s>>>(a, 0);
  pack_bias_kernel<<<512, threads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace moe

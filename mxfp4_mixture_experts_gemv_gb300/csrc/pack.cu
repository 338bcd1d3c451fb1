// Weight repacker: checkpoint-layout MXFP4 expert weights -> the tiled layout the
// grouped GEMM streams (see common.cuh for the layout); optionally converted to
// NVFP4 on the way.
#include "common.cuh"
#include "quant.cuh"

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

// ---------------------------------------------------------------- NVFP4 conversion
// "GPT-OSS-120B on DGX Spark: From MXFP4 to NVFP4", "Conversion Methodology":
// dequantise each MXFP4 block (E2M1 value times 2^(scale - 127)), then per
// 16-element block take the amax, choose the E4M3 block scale and quantise the
// elements to E2M1; a global scale per projection (its amax / (6 * 448), a
// reading: the page names the global factor without its rule) lets the E4M3
// block scales span the tensor.

__device__ __forceinline__ float e2m1_mag(uint32_t nib) {
  // magnitudes of the E2M1 codes 0..7: 0, 0.5, 1, 1.5, 2, 3, 4, 6 (code 1 is the
  // subnormal 0.5; codes 2..7 are 2^((m >> 1) - 1) times 1 or 1.5)
  const uint32_t m = nib & 7u;
  return m < 2u ? 0.5f * (float)m : (float)(1u << ((m >> 1) - 1u)) * (m & 1u ? 1.5f : 1.0f);
}

__device__ __forceinline__ float e8m0_f32(uint32_t s) {
  // 2^(s - 127); s = 0 is the subnormal 2^-127
  return s ? __uint_as_float(s << 23) : __uint_as_float(0x00400000u);
}

// Largest magnitude of each projection: one thread per 32-element block.
__global__ void nvfp4_amax_kernel(PackArgs a, int gate_up) {
  const PackedHeader& h = a.h;
  const int rows = gate_up ? 2 * h.I : h.H;
  const int nb = (gate_up ? h.H : h.I) / 32;
  const uint4* blk = reinterpret_cast<const uint4*>(gate_up ? a.w.gate_up_blocks : a.w.down_blocks);
  const uint8_t* sc = gate_up ? a.w.gate_up_scales : a.w.down_scales;
  uint32_t* amax = reinterpret_cast<uint32_t*>(a.packed + kAmaxOffset) + (gate_up ? 0 : 1);
  const int64_t total = (int64_t)h.E * rows * nb;
  float m = 0.f;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const uint4 v = blk[i];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t mm = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q)
#pragma unroll
      for (int n = 0; n < 8; ++n) mm = max(mm, (w[q] >> (4 * n)) & 7u);
    m = fmaxf(m, e2m1_mag(mm) * e8m0_f32(sc[i]));
  }
  // non-negative floats order like their bit patterns
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0 && m > 0.f) atomicMax(amax, __float_as_uint(m));
}

// Data tiles and scale atoms: one thread per 16-byte chunk of the tile-contiguous
// layout (one source 32-element block = two NVFP4 blocks).  The scale section is
// zeroed first (padding rows and blocks keep the zero scale).
__global__ void pack_nvfp4_kernel(PackArgs a, int gate_up) {
  const PackedHeader& h = a.h;
  const int rows = gate_up ? 2 * h.I : h.H;
  const int rows_stored = gate_up ? h.gu_rows_stored : h.d_rows_stored;
  const int K = gate_up ? h.H : h.I;
  const int kt_n = gate_up ? h.gu_ktiles : h.d_ktiles;
  const int mt_n = gate_up ? h.gu_mtiles : h.d_mtiles;
  const int nb = K / 32;
  const uint4* src = reinterpret_cast<const uint4*>(gate_up ? a.w.gate_up_blocks : a.w.down_blocks);
  const uint8_t* ssrc = gate_up ? a.w.gate_up_scales : a.w.down_scales;
  uint4* dst = reinterpret_cast<uint4*>(a.packed + (gate_up ? h.off_gu_data : h.off_d_data));
  uint8_t* sf = a.packed + (gate_up ? h.off_gu_sf : h.off_d_sf);
  const float amax = __uint_as_float(reinterpret_cast<const uint32_t*>(a.packed + kAmaxOffset)[gate_up ? 0 : 1]);
  const float gs = nvfp4_global_scale(amax);
  const int64_t per_expert = (int64_t)rows_stored * kt_n * 4;
  const int64_t per_mtile = (int64_t)kTileM * kt_n * 4;
  const int64_t total = (int64_t)h.E * per_expert;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int e = (int)(i / per_expert);
    const int64_t q = i - (int64_t)e * per_expert;
    const int m = (int)(q / per_mtile);
    const int rows_m = min(kTileM, rows_stored - m * kTileM);
    const int64_t rem = q - (int64_t)m * per_mtile;
    const int kt = (int)(rem / (rows_m * 4));
    const int rem2 = (int)(rem - (int64_t)kt * rows_m * 4);
    const int r = rem2 >> 2, j = rem2 & 3;
    const int pr = m * kTileM + r;
    const int kb = kt * 4 + j;
    if (pr >= rows || kb >= nb) {
      dst[i] = make_uint4(0, 0, 0, 0);
      continue;
    }
    const int sr = gate_up ? gu_source_row(pr, h.I) : pr;
    const int64_t si = ((int64_t)e * rows + sr) * nb + kb;
    const uint4 v = src[si];
    const float scale = e8m0_f32(ssrc[si]);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float x[32];
#pragma unroll
    for (int c = 0; c < 32; ++c) {
      const uint32_t nib = (w[c >> 3] >> (4 * (c & 7))) & 15u;
      const float mag = e2m1_mag(nib) * scale;
      x[c] = (nib & 8u) ? -mag : mag;
    }
    uint32_t p0[2], p1[2];
    const uint32_t s0 = nvfp4_block16(x, gs, p0), s1 = nvfp4_block16(x + 16, gs, p1);
    dst[i] = make_uint4(p0[0], p0[1], p1[0], p1[1]);
    // 16-element blocks 2j, 2j+1 of this k-tile: atom j / 2, bytes (2j) % 4 and (2j) % 4 + 1
    uint8_t* at = sf + ((((int64_t)e * mt_n + m) * kt_n + kt) * 2 + (j >> 1)) * kAtomBytes + (r & 31) * 16 + (r >> 5) * 4;
    at[(2 * j) & 3] = (uint8_t)s0;
    at[((2 * j) & 3) + 1] = (uint8_t)s1;
  }
}

}  // namespace

cudaError_t launch_pack_nvfp4(const PackedHeader& h, const moe_mxfp4_weights& w, uint8_t* packed, cudaStream_t s) {
  PackArgs a{h, w, packed};
  const int threads = 256, blocks = 4096;
  cudaError_t e = cudaMemsetAsync(packed + kAmaxOffset, 0, 8, s);
  if (e != cudaSuccess) return e;
  e = cudaMemsetAsync(packed + h.off_gu_sf, 0, h.off_gu_bias - h.off_gu_sf, s);
  if (e != cudaSuccess) return e;
  e = cudaMemsetAsync(packed + h.off_d_sf, 0, h.off_d_bias - h.off_d_sf, s);
  if (e != cudaSuccess) return e;
  nvfp4_amax_kernel<<<blocks, threads, 0, s>>>(a, 1);
  nvfp4_amax_kernel<<<blocks, threads, 0, s>>>(a, 0);
  pack_nvfp4_kernel<<<blocks, threads, 0, s>>>(a, 1);
  pack_nvfp4_kernel<<<blocks, threads, 0, s>>>(a, 0);
  pack_bias_kernel<<<512, threads, 0, s>>>(a);
  return cudaGetLastError();
}

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

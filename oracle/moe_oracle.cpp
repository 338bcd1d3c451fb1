// CPU oracle for the MXFP4 mixture-of-experts layer.
//
// TEST INFRASTRUCTURE ONLY.  This is a plain, slow, single-threaded fp64
// restatement of what the layer computes, used by tests/, the smoke check and
// the benchmark's CPU baseline.  It shares no code with the CUDA library and
// must never be called from the library's product path.
//
// Sources (titles of the pages the method is described on):
//  * "GPT-OSS-120B on DGX Spark: From MXFP4 to NVFP4 — A Deep-Dive Benchmark",
//    section "MXFP4 Tensor Structure": the *_blocks / *_scales / *_bias
//    layout, the E2M1 value set {0, +-0.5, +-1, +-1.5, +-2, +-3, +-4, +-6} and
//    the E8M0 power-of-two scale with bias 127; section "Conversion
//    Methodology", step 1: dequantisation = unpack nibbles, look the code up
//    in the 16-value table, multiply by 2^(stored-127).
//  * same page, "GPT-OSS-120B Architecture": 128 experts, 4 active per token,
//    router weights kept in BF16.
//  * "GPT-OSS-120B with MXFP4 on DGX Spark (SM121/GB10)", "What's Included":
//    the MoE layer is an FP8-activation x FP4-weight grouped GEMM;
//    "Numerical Accuracy": full-scale (block-scaled) activation quantisation.
//  * "GPT-OSS-120B with MXFP4 on DGX Spark (SM121/GB10)", "Performance
//    Optimizations": native FP4 x FP4 block-scaled MMA as the next step, for
//    which the layer can also quantise its activations to MXFP4 (the
//    `act_fp4` variant below).
//  * "GPT-OSS-120B with MXFP4 on DGX Spark (SM121/GB10)", "What's Included",
//    "Full MXFP4 Quantization Stack": the dense projections (QKV, O, LM head)
//    in MXFP4 as well (oracle_dense_linear, oracle_quantize_mxfp4_weights).
//  * "GPT-OSS-120B on DGX Spark: From MXFP4 to NVFP4", "The MXFP4 -> NVFP4
//    Conversion": NVFP4 = E2M1 data in 16-element blocks with an E4M3 scale per
//    block and a global scale; "Conversion Methodology": dequantise MXFP4, then
//    per 16-element block take the amax, choose the E4M3 scale, quantise the
//    elements to E2M1 (oracle_nvfp4_*).
//  The layer definition the pages leave open (routing rule, SwiGLU, MXFP8
//  scale rule, nibble order, gate/up row order) follows the readings listed
//  in the design notes; each function below states the one it uses.
//
// Every entry point is extern "C" and takes plain host pointers.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

namespace {

// E2M1 magnitudes in the order the MXFP4 page lists the value set.  Code bit 3
// is the sign; bits 2..0 index this table.
const double kE2M1Magnitude[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

double e2m1(int code) {
  const double m = kE2M1Magnitude[code & 7];
  return (code & 8) ? -m : m;
}

double e8m0(int code) {
  if (code == 255) return std::nan("");
  return std::ldexp(1.0, code - 127);
}

double bf16_to_double(uint16_t b) {
  uint32_t u = static_cast<uint32_t>(b) << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return static_cast<double>(f);
}

// Round a double to the nearest bfloat16, ties to even (one rounding step).
uint16_t double_to_bf16(double v) {
  if (std::isnan(v)) return 0x7FC0;
  // bf16 has an 8-bit significand; scale so the kept bits are an integer.
  const uint16_t sign = std::signbit(v) ? 0x8000 : 0;
  double a = std::fabs(v);
  if (a == 0.0) return sign;
  int ex;
  std::frexp(a, &ex);           // a in [2^(ex-1), 2^ex)
  int e = ex - 1;
  if (e < -126) e = -126;       // subnormal range: fixed quantum 2^-133
  const double quantum = std::ldexp(1.0, e - 7);
  double q = std::nearbyint(a / quantum) * quantum;   // RNE on the significand
  if (q >= std::ldexp(1.0, 128)) return sign | 0x7F80;  // overflow to inf
  float f = static_cast<float>(q);  // exact: q has <= 8 significant bits
  uint32_t u;
  std::memcpy(&u, &f, 4);
  return sign | static_cast<uint16_t>((u >> 16) & 0x7FFF);
}

// E4M3 (OCP "fn" variant): bias 7, no infinities, S.1111.111 is NaN, largest
// finite 448, subnormals m/8 * 2^-6.  Encoding: round to nearest, ties to even
// mantissa, magnitudes above 448 saturate to 448.
double e4m3(int code) {
  const int s = (code >> 7) & 1, e = (code >> 3) & 15, m = code & 7;
  if (e == 15 && m == 7) return std::nan("");
  const double v = (e == 0) ? std::ldexp(m / 8.0, -6) : std::ldexp(1.0 + m / 8.0, e - 7);
  return s ? -v : v;
}

int e4m3_encode(double v) {
  if (std::isnan(v)) return 0x7F;
  const int sign = std::signbit(v) ? 0x80 : 0;
  const double a = std::fabs(v);
  if (a >= 448.0) return sign | 0x7E;
  if (a < std::ldexp(1.0, -6)) {
    // subnormal grid: multiples of 2^-9; a count of 8 is the smallest normal
    const int q = static_cast<int>(std::nearbyint(a * 512.0));
    return sign | q;
  }
  int ex;
  std::frexp(a, &ex);
  int e = ex - 1;                                     // a in [2^e, 2^(e+1))
  int m = static_cast<int>(std::nearbyint((a / std::ldexp(1.0, e) - 1.0) * 8.0));
  if (m == 8) { e += 1; m = 0; }
  return sign | ((e + 7) << 3) | m;
}

// MXFP8 quantisation of one 32-element block (reading: OCP-MX style shared
// exponent floor(log2(amax)) - 8, 8 being E4M3's largest exponent; scale code
// = that exponent + 127, clamped to [0, 254]).  Returns the scale exponent.
int mxfp8_block(const double* v, uint8_t* q) {
  double amax = 0.0;
  for (int i = 0; i < 32; ++i) amax = std::max(amax, std::fabs(v[i]));
  int sexp = -127;
  if (amax > 0.0) {
    int ex;
    std::frexp(amax, &ex);
    sexp = std::max(ex - 1 - 8, -127);
    sexp = std::min(sexp, 127);
  }
  for (int i = 0; i < 32; ++i) q[i] = static_cast<uint8_t>(e4m3_encode(std::ldexp(v[i], -sexp)));
  return sexp;
}

// E2M1 encoding: the nearest magnitude of the value set, ties to the even
// mantissa (code bit 0 clear), magnitudes above 6 saturating to 6.  The sign
// is kept, so a negative value that rounds to zero gives code 8 (-0).
int e2m1_encode(double v) {
  if (std::isnan(v)) return 7;  // never produced by these inputs
  const int sign = std::signbit(v) ? 8 : 0;
  const double a = std::fabs(v);
  if (a >= 6.0) return sign | 7;  // (far out, the distances to 4 and 6 round equal)
  int best = 0;
  for (int c = 1; c < 8; ++c) {
    const double d = std::fabs(a - kE2M1Magnitude[c]), db = std::fabs(a - kE2M1Magnitude[best]);
    if (d < db || (d == db && (c & 1) == 0)) best = c;
  }
  return sign | best;
}

// MXFP4 quantisation of one 32-element block of activations (reading: the
// same OCP-MX shared-exponent rule as MXFP8, floor(log2(amax)) - 2, 2 being
// E2M1's largest exponent; scale code = that exponent + 127).  Codes are one
// E2M1 code per byte.  Returns the scale exponent.
int mxfp4_block(const double* v, uint8_t* q) {
  double amax = 0.0;
  for (int i = 0; i < 32; ++i) amax = std::max(amax, std::fabs(v[i]));
  int sexp = -127;
  if (amax > 0.0) {
    int ex;
    std::frexp(amax, &ex);
    sexp = std::max(ex - 1 - 2, -127);
    sexp = std::min(sexp, 127);
  }
  for (int i = 0; i < 32; ++i) q[i] = static_cast<uint8_t>(e2m1_encode(std::ldexp(v[i], -sexp)));
  return sexp;
}

// One MXFP4 weight W[r][c] of a [rows, K] matrix stored as blocks [rows, K/32, 16]
// and scales [rows, K/32].  Reading: the low nibble of a byte holds the even
// element of the pair.
inline double mxfp4_weight(const uint8_t* blocks, const uint8_t* scales, int64_t K, int64_t r,
                           int64_t c) {
  const int64_t nb = K / 32;
  const uint8_t byte = blocks[(r * nb + c / 32) * 16 + (c % 32) / 2];
  const int code = (c % 2 == 0) ? (byte & 0xF) : (byte >> 4);
  return e2m1(code) * e8m0(scales[r * nb + c / 32]);
}

double silu(double z) { return z / (1.0 + std::exp(-z)); }

}  // namespace

extern "C" {

double oracle_e2m1_value(int code) { return e2m1(code & 15); }
double oracle_e8m0_value(int code) { return e8m0(code & 255); }
double oracle_e4m3_value(int code) { return e4m3(code & 255); }
int oracle_e4m3_encode(double v) { return e4m3_encode(v); }
int oracle_e2m1_encode(double v) { return e2m1_encode(v); }
double oracle_bf16_value(uint16_t b) { return bf16_to_double(b); }
uint16_t oracle_bf16_round(double v) { return double_to_bf16(v); }
double oracle_silu(double z) { return silu(z); }

// Dequantise a [rows, K] MXFP4 matrix (checkpoint layout) to fp64, row-major.
void oracle_dequant_mxfp4(const uint8_t* blocks, const uint8_t* scales, int64_t rows, int64_t K,
                          double* W) {
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t c = 0; c < K; ++c) W[r * K + c] = mxfp4_weight(blocks, scales, K, r, c);
}

// MXFP8-quantise n values (n a multiple of 32): codes q[n], scale codes s[n/32].
void oracle_mxfp8_quantize(const double* v, int64_t n, uint8_t* q, uint8_t* s) {
  for (int64_t b = 0; b < n / 32; ++b) s[b] = static_cast<uint8_t>(mxfp8_block(v + 32 * b, q + 32 * b) + 127);
}

// MXFP4-quantise n values (n a multiple of 32): E2M1 codes q[n] (one per byte),
// scale codes s[n/32].
void oracle_mxfp4_quantize(const double* v, int64_t n, uint8_t* q, uint8_t* s) {
  for (int64_t b = 0; b < n / 32; ++b) s[b] = static_cast<uint8_t>(mxfp4_block(v + 32 * b, q + 32 * b) + 127);
}

// Router: logits l[t][e] = sum_h x[t][h] * Wr[e][h] + br[e] (bf16 inputs widened
// exactly, fp64 sum).  Selection: experts ordered by logit descending, lower
// index first on ties, first k kept, in that order.  The comparison is made on
// the logits rounded to fp32, the precision the kernel decides in.  Weights:
// softmax over the k selected fp64 logits.
void oracle_route(const uint16_t* x, const uint16_t* wr, const uint16_t* br, int64_t T, int64_t H,
                  int64_t E, int32_t k, double* logits, int32_t* ids, double* w) {
  std::vector<int32_t> order(E);
  for (int64_t t = 0; t < T; ++t) {
    double* l = logits + t * E;
    for (int64_t e = 0; e < E; ++e) {
      double acc = 0.0;
      for (int64_t h = 0; h < H; ++h) acc += bf16_to_double(x[t * H + h]) * bf16_to_double(wr[e * H + h]);
      l[e] = acc + bf16_to_double(br[e]);
    }
    for (int64_t e = 0; e < E; ++e) order[e] = static_cast<int32_t>(e);
    std::stable_sort(order.begin(), order.end(), [&](int32_t a, int32_t b) {
      return static_cast<float>(l[a]) > static_cast<float>(l[b]);
    });
    double denom = 0.0;
    for (int32_t j = 0; j < k; ++j) denom += std::exp(l[order[j]] - l[order[0]]);
    for (int32_t j = 0; j < k; ++j) {
      ids[t * k + j] = order[j];
      w[t * k + j] = std::exp(l[order[j]] - l[order[0]]) / denom;
    }
  }
}

// Stable grouping of the T*k (token, slot) pairs by expert: cnt[e], exclusive
// offsets off[0..E], sorted_rows[off[e] + r] = flat index t*k+j of the r-th pair
// routed to e (ascending flat index), inv_pos[t*k+j] = its position.
void oracle_permute(const int32_t* ids, int64_t T, int32_t k, int32_t E, int32_t* cnt, int32_t* off,
                    int32_t* sorted_rows, int32_t* inv_pos) {
  for (int32_t e = 0; e < E; ++e) cnt[e] = 0;
  for (int64_t f = 0; f < T * k; ++f) cnt[ids[f]] += 1;
  off[0] = 0;
  for (int32_t e = 0; e < E; ++e) off[e + 1] = off[e] + cnt[e];
  std::vector<int32_t> fill(off, off + E);
  for (int64_t f = 0; f < T * k; ++f) {
    const int32_t pos = fill[ids[f]]++;
    sorted_rows[pos] = static_cast<int32_t>(f);
    inv_pos[f] = pos;
  }
}

// One expert's MLP on one quantised row; act_fp4 = 0 for MXFP8 activations
// (E4M3 codes), 1 for MXFP4 activations (E2M1 codes, one per byte) -- both x
// and the intermediate h use that format.
//   xq, xs : the row's codes [H] and E8M0 scale codes [H/32]
//   g      : gate_up pre-activation [2I] = xq . Wgu^T + bgu   (rows [0,I) gate, [I,2I) up)
//   h      : silu(g[i]) * g[I+i] [I], rounded to fp32 (the precision the kernel
//            quantises from), then MXFP8-quantised to hq [I] / hs [I/32]
//   y      : down output [H] = hq . Wd^T + bd
// Any of g / h / hq / hs may be NULL.
void oracle_expert_mlp_fmt(const uint8_t* xq, const uint8_t* xs, int64_t H, int64_t I,
                           const uint8_t* gu_blocks, const uint8_t* gu_scales, const uint16_t* gu_bias,
                           const uint8_t* d_blocks, const uint8_t* d_scales, const uint16_t* d_bias,
                           double* g_out, double* h_out, uint8_t* hq_out, uint8_t* hs_out, double* y,
                           int32_t act_fp4) {
  std::vector<double> xv(H), g(2 * I), h(I), hv(I);
  std::vector<uint8_t> hq(I), hs(I / 32);
  auto act = [&](uint8_t code) { return act_fp4 ? e2m1(code) : e4m3(code); };
  for (int64_t c = 0; c < H; ++c) xv[c] = act(xq[c]) * e8m0(xs[c / 32]);
  for (int64_t r = 0; r < 2 * I; ++r) {
    double acc = 0.0;
    for (int64_t c = 0; c < H; ++c) acc += xv[c] * mxfp4_weight(gu_blocks, gu_scales, H, r, c);
    g[r] = acc + bf16_to_double(gu_bias[r]);
  }
  for (int64_t i = 0; i < I; ++i) h[i] = static_cast<double>(static_cast<float>(silu(g[i]) * g[I + i]));
  if (act_fp4)
    oracle_mxfp4_quantize(h.data(), I, hq.data(), hs.data());
  else
    oracle_mxfp8_quantize(h.data(), I, hq.data(), hs.data());
  for (int64_t i = 0; i < I; ++i) hv[i] = act(hq[i]) * e8m0(hs[i / 32]);
  for (int64_t c = 0; c < H; ++c) {
    double acc = 0.0;
    for (int64_t i = 0; i < I; ++i) acc += hv[i] * mxfp4_weight(d_blocks, d_scales, I, c, i);
    y[c] = acc + bf16_to_double(d_bias[c]);
  }
  if (g_out) std::copy(g.begin(), g.end(), g_out);
  if (h_out) std::copy(h.begin(), h.end(), h_out);
  if (hq_out) std::copy(hq.begin(), hq.end(), hq_out);
  if (hs_out) std::copy(hs.begin(), hs.end(), hs_out);
}

void oracle_expert_mlp(const uint8_t* xq, const uint8_t* xs, int64_t H, int64_t I,
                       const uint8_t* gu_blocks, const uint8_t* gu_scales, const uint16_t* gu_bias,
                       const uint8_t* d_blocks, const uint8_t* d_scales, const uint16_t* d_bias,
                       double* g_out, double* h_out, uint8_t* hq_out, uint8_t* hs_out, double* y) {
  oracle_expert_mlp_fmt(xq, xs, H, I, gu_blocks, gu_scales, gu_bias, d_blocks, d_scales, d_bias, g_out, h_out,
                        hq_out, hs_out, y, 0);
}

// The whole layer for T tokens.
//   x [T,H] bf16; router_w [E,H] bf16; router_b [E] bf16
//   expert weights in the checkpoint layout, all E experts:
//     gu_blocks [E,2I,H/32,16], gu_scales [E,2I,H/32], gu_bias bf16 [E,2I]
//     d_blocks  [E,H,I/32,16],  d_scales  [E,H,I/32],  d_bias  bf16 [E,H]
//   out [T,H] fp64: sum_j w[t][j] * y(t, ids[t][j]), accumulated in slot order.
//   Optional (may be NULL): logits [T,E], ids [T,k], w [T,k], xq [T,H], xs [T,H/32],
//   and the intermediate of every (token, slot): h [T,k,I], hq [T,k,I], hs [T,k,I/32].
//   act_fp4 selects MXFP4 instead of MXFP8 for the activations (x and h).
void oracle_moe_forward_fmt(const uint16_t* x, int64_t T, int64_t H, int64_t I, int64_t E, int32_t k,
                            const uint16_t* router_w, const uint16_t* router_b,
                            const uint8_t* gu_blocks, const uint8_t* gu_scales, const uint16_t* gu_bias,
                            const uint8_t* d_blocks, const uint8_t* d_scales, const uint16_t* d_bias,
                            double* out, double* logits_out, int32_t* ids_out, double* w_out,
                            uint8_t* xq_out, uint8_t* xs_out, double* h_out, uint8_t* hq_out,
                            uint8_t* hs_out, int32_t act_fp4) {
  std::vector<double> logits(T * E), w(T * k), xrow(H), y(H);
  std::vector<int32_t> ids(T * k);
  std::vector<uint8_t> xq(H), xs(H / 32);
  oracle_route(x, router_w, router_b, T, H, E, k, logits.data(), ids.data(), w.data());
  const int64_t gu_rows = 2 * I, nbh = H / 32, nbi = I / 32;
  for (int64_t t = 0; t < T; ++t) {
    for (int64_t c = 0; c < H; ++c) xrow[c] = bf16_to_double(x[t * H + c]);
    if (act_fp4)
      oracle_mxfp4_quantize(xrow.data(), H, xq.data(), xs.data());
    else
      oracle_mxfp8_quantize(xrow.data(), H, xq.data(), xs.data());
    if (xq_out) std::copy(xq.begin(), xq.end(), xq_out + t * H);
    if (xs_out) std::copy(xs.begin(), xs.end(), xs_out + t * nbh);
    for (int64_t c = 0; c < H; ++c) out[t * H + c] = 0.0;
    for (int32_t j = 0; j < k; ++j) {
      const int64_t e = ids[t * k + j];
      const int64_t tj = t * k + j;
      oracle_expert_mlp_fmt(xq.data(), xs.data(), H, I,
                            gu_blocks + e * gu_rows * nbh * 16, gu_scales + e * gu_rows * nbh,
                            gu_bias + e * gu_rows,
                            d_blocks + e * H * nbi * 16, d_scales + e * H * nbi, d_bias + e * H,
                            nullptr, h_out ? h_out + tj * I : nullptr, hq_out ? hq_out + tj * I : nullptr,
                            hs_out ? hs_out + tj * nbi : nullptr, y.data(), act_fp4);
      for (int64_t c = 0; c < H; ++c) out[t * H + c] += w[t * k + j] * y[c];
    }
  }
  if (logits_out) std::copy(logits.begin(), logits.end(), logits_out);
  if (ids_out) std::copy(ids.begin(), ids.end(), ids_out);
  if (w_out) std::copy(w.begin(), w.end(), w_out);
}

void oracle_moe_forward(const uint16_t* x, int64_t T, int64_t H, int64_t I, int64_t E, int32_t k,
                        const uint16_t* router_w, const uint16_t* router_b,
                        const uint8_t* gu_blocks, const uint8_t* gu_scales, const uint16_t* gu_bias,
                        const uint8_t* d_blocks, const uint8_t* d_scales, const uint16_t* d_bias,
                        double* out, double* logits_out, int32_t* ids_out, double* w_out,
                        uint8_t* xq_out, uint8_t* xs_out, double* h_out, uint8_t* hq_out,
                        uint8_t* hs_out) {
  oracle_moe_forward_fmt(x, T, H, I, E, k, router_w, router_b, gu_blocks, gu_scales, gu_bias, d_blocks, d_scales,
                         d_bias, out, logits_out, ids_out, w_out, xq_out, xs_out, h_out, hq_out, hs_out, 0);
}

// ---------------------------------------------------------------- dense MXFP4 linears
// Pack E2M1 codes (one per byte, [rows, K]) into the checkpoint block layout
// [rows, K/32, 16]: two codes per byte, the even element in the low nibble.
void oracle_pack_e2m1(const uint8_t* codes, int64_t rows, int64_t K, uint8_t* blocks) {
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t c = 0; c < K; c += 2)
      blocks[(r * K + c) / 2] = static_cast<uint8_t>((codes[r * K + c] & 0xF) | ((codes[r * K + c + 1] & 0xF) << 4));
}

// Quantise a [rows, K] weight matrix (fp64 values, e.g. widened bf16) to MXFP4 in the
// checkpoint layout: per 32-element block the same shared-exponent rule as the
// MXFP4 activations (floor(log2 amax) - 2; E2M1 round-to-nearest-even, saturating
// at 6).  blocks [rows, K/32, 16], scales [rows, K/32].
void oracle_quantize_mxfp4_weights(const double* w, int64_t rows, int64_t K, uint8_t* blocks, uint8_t* scales) {
  std::vector<uint8_t> q(K);
  for (int64_t r = 0; r < rows; ++r) {
    oracle_mxfp4_quantize(w + r * K, K, q.data(), scales + r * (K / 32));
    oracle_pack_e2m1(q.data(), 1, K, blocks + r * (K / 2));
  }
}

// A dense MXFP4 linear: out[t][n] = sum_k xq[t][k] * W[n][k] + b[n], with x (bf16
// [T, K]) quantised per row to MXFP8 (act_fp4 = 0) or MXFP4 (1) as in the expert
// MLP, W [N, K] MXFP4 in the checkpoint layout, b bf16 [N] (may be NULL).  fp64
// sums; out [T, N] fp64.
void oracle_dense_linear(const uint16_t* x, int64_t T, int64_t K, int64_t N, const uint8_t* blocks,
                         const uint8_t* scales, const uint16_t* bias, double* out, int32_t act_fp4) {
  std::vector<double> xr(K), xv(K);
  std::vector<uint8_t> xq(K), xs(K / 32);
  for (int64_t t = 0; t < T; ++t) {
    for (int64_t c = 0; c < K; ++c) xr[c] = bf16_to_double(x[t * K + c]);
    if (act_fp4)
      oracle_mxfp4_quantize(xr.data(), K, xq.data(), xs.data());
    else
      oracle_mxfp8_quantize(xr.data(), K, xq.data(), xs.data());
    for (int64_t c = 0; c < K; ++c) xv[c] = (act_fp4 ? e2m1(xq[c]) : e4m3(xq[c])) * e8m0(xs[c / 32]);
    for (int64_t n = 0; n < N; ++n) {
      double acc = 0.0;
      for (int64_t c = 0; c < K; ++c) acc += xv[c] * mxfp4_weight(blocks, scales, K, n, c);
      out[t * N + n] = acc + (bias ? bf16_to_double(bias[n]) : 0.0);
    }
  }
}

// ---------------------------------------------------------------- NVFP4
// Global scale of a tensor whose largest magnitude is amax: amax / (6 * 448), so
// that the largest block scale is E4M3's largest value (reading: the page's
// conversion returns "a global scale factor" without its rule; this is the
// plainest one that lets the E4M3 block scales span the tensor).  fp32, the
// precision the scale is stored in; 1 for an all-zero tensor.
double oracle_nvfp4_global_scale(double amax) {
  if (!(amax > 0.0)) return 1.0;
  return static_cast<double>(static_cast<float>(amax) / 2688.0f);
}

// NVFP4 quantisation of n values (n a multiple of 16) with global scale gs:
// per 16-element block, scale code = E4M3(amax / (6 gs)) (round-to-nearest-even,
// saturating at 448); element codes = E2M1(v / (scale * gs)) (ties to even,
// saturating at 6), all-zero codes where the block scale is zero.  The divisions
// that decide codes are taken in fp32, the precision a GPU quantiser computes
// in.  codes q[n] one per byte, scale codes s[n/16].
void oracle_nvfp4_quantize(const double* v, int64_t n, double gs, uint8_t* q, uint8_t* s) {
  const float g = static_cast<float>(gs);
  for (int64_t b = 0; b < n / 16; ++b) {
    double amax = 0.0;
    for (int i = 0; i < 16; ++i) amax = std::max(amax, std::fabs(v[16 * b + i]));
    const float t = static_cast<float>(amax) / (6.0f * g);
    const int sc = e4m3_encode(static_cast<double>(t));
    s[b] = static_cast<uint8_t>(sc);
    const float sv = static_cast<float>(e4m3(sc)) * g;
    for (int i = 0; i < 16; ++i) {
      const int64_t k = 16 * b + i;
      q[k] = sv == 0.0f ? 0 : static_cast<uint8_t>(e2m1_encode(static_cast<double>(static_cast<float>(v[k]) / sv)));
    }
  }
}

// Value of NVFP4 element k of a row: e2m1(code) * e4m3(scale of its block) * gs.
double oracle_nvfp4_value(int code, int scale_code, double gs) { return e2m1(code & 15) * e4m3(scale_code & 255) * gs; }

// One expert's MLP with NVFP4 weights and NVFP4 activations (unit global scale
// for the activations): x codes xq [H] (one per byte) with scales xs [H/16];
// weights as codes [rows, K] (one per byte) with scale codes [rows, K/16] and a
// global scale per projection.  h (rounded to fp32) is NVFP4-quantised the same
// way.  Outputs as in oracle_expert_mlp_fmt.
void oracle_expert_mlp_nvfp4(const uint8_t* xq, const uint8_t* xs, int64_t H, int64_t I, const uint8_t* gu_codes,
                             const uint8_t* gu_sc, double gu_gs, const uint16_t* gu_bias, const uint8_t* d_codes,
                             const uint8_t* d_sc, double d_gs, const uint16_t* d_bias, double* h_out, uint8_t* hq_out,
                             uint8_t* hs_out, double* y) {
  std::vector<double> xv(H), g(2 * I), h(I), hv(I);
  std::vector<uint8_t> hq(I), hs(I / 16);
  for (int64_t c = 0; c < H; ++c) xv[c] = oracle_nvfp4_value(xq[c], xs[c / 16], 1.0);
  for (int64_t r = 0; r < 2 * I; ++r) {
    double acc = 0.0;
    for (int64_t c = 0; c < H; ++c) acc += xv[c] * oracle_nvfp4_value(gu_codes[r * H + c], gu_sc[r * (H / 16) + c / 16], gu_gs);
    g[r] = acc + bf16_to_double(gu_bias[r]);
  }
  for (int64_t i = 0; i < I; ++i) h[i] = static_cast<double>(static_cast<float>(silu(g[i]) * g[I + i]));
  oracle_nvfp4_quantize(h.data(), I, 1.0, hq.data(), hs.data());
  for (int64_t i = 0; i < I; ++i) hv[i] = oracle_nvfp4_value(hq[i], hs[i / 16], 1.0);
  for (int64_t c = 0; c < H; ++c) {
    double acc = 0.0;
    for (int64_t i = 0; i < I; ++i) acc += hv[i] * oracle_nvfp4_value(d_codes[c * I + i], d_sc[c * (I / 16) + i / 16], d_gs);
    y[c] = acc + bf16_to_double(d_bias[c]);
  }
  if (h_out) std::copy(h.begin(), h.end(), h_out);
  if (hq_out) std::copy(hq.begin(), hq.end(), hq_out);
  if (hs_out) std::copy(hs.begin(), hs.end(), hs_out);
}

// Convert one MXFP4 projection's rows [rows, K] (checkpoint layout) to NVFP4 with
// global scale gs: codes [rows, K] one per byte, E4M3 scale codes [rows, K/16].
void oracle_convert_mxfp4_to_nvfp4(const uint8_t* blocks, const uint8_t* scales, int64_t rows, int64_t K, double gs,
                                   uint8_t* codes, uint8_t* sc) {
  std::vector<double> w(K);
  for (int64_t r = 0; r < rows; ++r) {
    for (int64_t c = 0; c < K; ++c) w[c] = mxfp4_weight(blocks, scales, K, r, c);
    oracle_nvfp4_quantize(w.data(), K, gs, codes + r * K, sc + r * (K / 16));
  }
}

// Largest magnitude of an MXFP4 tensor of n_rows rows of K elements.
double oracle_mxfp4_amax(const uint8_t* blocks, const uint8_t* scales, int64_t rows, int64_t K) {
  double m = 0.0;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t c = 0; c < K; ++c) m = std::max(m, std::fabs(mxfp4_weight(blocks, scales, K, r, c)));
  return m;
}

// The whole layer in the NVFP4 variant: the MXFP4 expert weights converted to
// NVFP4 per projection (global scale from the projection's amax over all experts),
// the activations x and h quantised to NVFP4 with unit global scale, routing and
// combine as in oracle_moe_forward_fmt.  Arguments as there; xs has H/16 scale
// codes per token and hs I/16 per (token, slot); codes one per byte.
void oracle_moe_forward_nvfp4(const uint16_t* x, int64_t T, int64_t H, int64_t I, int64_t E, int32_t k,
                              const uint16_t* router_w, const uint16_t* router_b, const uint8_t* gu_blocks,
                              const uint8_t* gu_scales, const uint16_t* gu_bias, const uint8_t* d_blocks,
                              const uint8_t* d_scales, const uint16_t* d_bias, double* out, double* logits_out,
                              int32_t* ids_out, double* w_out, uint8_t* xq_out, uint8_t* xs_out, double* h_out,
                              uint8_t* hq_out, uint8_t* hs_out) {
  std::vector<double> logits(T * E), w(T * k), xrow(H), y(H);
  std::vector<int32_t> ids(T * k);
  std::vector<uint8_t> xq(H), xs(H / 16);
  oracle_route(x, router_w, router_b, T, H, E, k, logits.data(), ids.data(), w.data());
  const double gs_gu = oracle_nvfp4_global_scale(oracle_mxfp4_amax(gu_blocks, gu_scales, E * 2 * I, H));
  const double gs_d = oracle_nvfp4_global_scale(oracle_mxfp4_amax(d_blocks, d_scales, E * H, I));
  std::vector<std::vector<uint8_t>> guc(E), gus(E), dc(E), ds(E);
  for (int64_t t = 0; t < T; ++t)
    for (int32_t j = 0; j < k; ++j) {
      const int64_t e = ids[t * k + j];
      if (!guc[e].empty()) continue;
      guc[e].resize(2 * I * H);
      gus[e].resize(2 * I * (H / 16));
      dc[e].resize(H * I);
      ds[e].resize(H * (I / 16));
      oracle_convert_mxfp4_to_nvfp4(gu_blocks + e * 2 * I * (H / 2), gu_scales + e * 2 * I * (H / 32), 2 * I, H,
                                    gs_gu, guc[e].data(), gus[e].data());
      oracle_convert_mxfp4_to_nvfp4(d_blocks + e * H * (I / 2), d_scales + e * H * (I / 32), H, I, gs_d,
                                    dc[e].data(), ds[e].data());
    }
  for (int64_t t = 0; t < T; ++t) {
    for (int64_t c = 0; c < H; ++c) xrow[c] = bf16_to_double(x[t * H + c]);
    oracle_nvfp4_quantize(xrow.data(), H, 1.0, xq.data(), xs.data());
    if (xq_out) std::copy(xq.begin(), xq.end(), xq_out + t * H);
    if (xs_out) std::copy(xs.begin(), xs.end(), xs_out + t * (H / 16));
    for (int64_t c = 0; c < H; ++c) out[t * H + c] = 0.0;
    for (int32_t j = 0; j < k; ++j) {
      const int64_t e = ids[t * k + j], tj = t * k + j;
      oracle_expert_mlp_nvfp4(xq.data(), xs.data(), H, I, guc[e].data(), gus[e].data(), gs_gu, gu_bias + e * 2 * I,
                              dc[e].data(), ds[e].data(), gs_d, d_bias + e * H, h_out ? h_out + tj * I : nullptr,
                              hq_out ? hq_out + tj * I : nullptr, hs_out ? hs_out + tj * (I / 16) : nullptr,
                              y.data());
      for (int64_t c = 0; c < H; ++c) out[t * H + c] += w[t * k + j] * y[c];
    }
  }
  if (logits_out) std::copy(logits.begin(), logits.end(), logits_out);
  if (ids_out) std::copy(ids.begin(), ids.end(), ids_out);
  if (w_out) std::copy(w.begin(), w.end(), w_out);
}

// RMSNorm with unit gain: x / sqrt(mean(x^2) + eps), rounded to bf16 (RNE).
void oracle_rmsnorm_bf16(const double* x, int64_t T, int64_t H, double eps, uint16_t* out) {
  for (int64_t t = 0; t < T; ++t) {
    double ss = 0.0;
    for (int64_t c = 0; c < H; ++c) ss += x[t * H + c] * x[t * H + c];
    const double inv = 1.0 / std::sqrt(ss / static_cast<double>(H) + eps);
    for (int64_t c = 0; c < H; ++c) out[t * H + c] = double_to_bf16(x[t * H + c] * inv);
  }
}

}  // extern "C"

/*
 * moe.h — C ABI of the GB300 (sm_103a) MXFP4 mixture-of-experts layer.
 *
 * The layer (gpt-oss-style MoE block):
 *   logits = x . Wr^T + br                        router GEMV, bf16 in, fp32 accumulate
 *   ids    = top-k experts by logit (desc; lower index first on ties)
 *   w      = softmax over the k selected logits
 *   xq     = MXFP8(x)                              E4M3 elements, one E8M0 scale per 32
 *   for each (token, slot j), e = ids[t][j]:
 *     g    = xq . Wgu[e]^T + bgu[e]                MXFP4 weights, 2I outputs
 *     h    = silu(g[0:I]) * g[I:2I]                SwiGLU
 *     hq   = MXFP8(h)
 *     y    = hq . Wd[e]^T + bd[e]                  MXFP4 weights, H outputs
 *   out[t] = bf16( sum_j w[t][j] * y(t, j) )
 *
 * Sources: "GPT-OSS-120B on DGX Spark: From MXFP4 to NVFP4 — A Deep-Dive
 * Benchmark", sections "GPT-OSS-120B Architecture" (128 experts, 4 active,
 * hidden 2880, router in BF16) and "MXFP4 Tensor Structure" (the weight
 * layout below, E2M1 values, E8M0 scales with bias 127); "GPT-OSS-120B with
 * MXFP4 on DGX Spark (SM121/GB10)", section "What's Included" (the MoE layer
 * as an FP8-activation x FP4-weight grouped GEMM) and "Numerical Accuracy"
 * (full-scale block activation quantisation).  The routing rule, SwiGLU form,
 * MXFP8 scale rule, nibble order and gate/up row order are readings of those
 * pages, documented with the oracle.
 *
 * Conventions for every entry point:
 *  - All tensor pointers are DEVICE pointers owned by the caller; the library
 *    never allocates or frees device memory and keeps no pointer after return.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  Work is
 *    enqueued asynchronously; no entry point synchronises the host except
 *    moe_get_device_status, moe_static_scratch_status and moe_profile_end.
 *  - Argument errors are detected on the host before anything is enqueued and
 *    return a non-zero moe_status; moe_last_error() gives the message.
 *  - bf16 values are passed as uint16_t bit patterns.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,         /* null pointer, T < 0, top_k out of range, ... */
  MOE_ERR_UNSUPPORTED_SHAPE = 2,   /* H or I not a multiple of 32, I not a multiple of 64, E > 256 */
  MOE_ERR_ALIGNMENT = 3,           /* a pointer is not 256-byte (packed/workspace) or 16-byte aligned */
  MOE_ERR_WORKSPACE_TOO_SMALL = 4, /* workspace_bytes < moe_workspace_size(...) */
  MOE_ERR_BAD_PACKED_HEADER = 5,   /* packed buffer too small for these dims */
  MOE_ERR_CUDA = 6,                /* a CUDA runtime/driver call failed */
  MOE_ERR_TIMEOUT = 7              /* a device-side bounded wait expired (see moe_get_device_status) */
} moe_status;

/* Layer dimensions: E experts, hidden size H, expert intermediate size I. */
typedef struct {
  int32_t E;
  int32_t H;
  int32_t I;
} moe_dims;

/*
 * Expert weights in the checkpoint layout of the MXFP4 gpt-oss release
 * ("MXFP4 Tensor Structure"): per projection a *_blocks tensor
 * uint8 [E, out, in/32, 16] of packed E2M1 codes (two per byte, low nibble =
 * even element), a *_scales tensor uint8 [E, out, in/32] of E8M0 codes
 * (value 2^(code-127)), and a *_bias tensor bf16 [E, out].
 * gate_up: out = 2I (rows [0, I) gate, [I, 2I) up), in = H.
 * down:    out = H, in = I.
 */
typedef struct {
  const uint8_t *gate_up_blocks;  /* [E, 2I, H/32, 16] */
  const uint8_t *gate_up_scales;  /* [E, 2I, H/32]     */
  const uint16_t *gate_up_bias;   /* bf16 [E, 2I]      */
  const uint8_t *down_blocks;     /* [E, H, I/32, 16]  */
  const uint8_t *down_scales;     /* [E, H, I/32]      */
  const uint16_t *down_bias;      /* bf16 [E, H]       */
} moe_mxfp4_weights;

/* Byte offsets of the intermediates inside a forward workspace (for tests
 * and debugging; all relative to the workspace base). */
typedef struct {
  size_t status;       /* uint32 [4]: device status words (0 = ok)                  */
  size_t done_gu;      /* int32 [max_tiles]: finished gate_up tiles per token tile  */
  size_t done_tok;     /* int32 [T, ceil(H/128)]: finished down slots per block     */
  size_t grid_bar;     /* int32[4]: grid routing arrivals, expert tiles claimed,
                          cluster routing's tile-list flag and finished-CTA count */
  size_t zero_bytes;   /* bytes from offset 0 the forward zeroes before it starts   */
  size_t logits;       /* fp32 [T, E] router logits                                 */
  size_t topk_ids;     /* int32 [T, k]                                              */
  size_t topk_w;       /* fp32 [T, k]                                               */
  size_t xq;           /* uint8 [T, H] E4M3 codes of x                              */
  size_t xs;           /* uint8 [T, H/32] E8M0 scale codes of x                     */
  size_t counts;       /* int32 [E] tokens per expert                               */
  size_t offsets;      /* int32 [E+1] exclusive prefix of counts                    */
  size_t sorted_rows;  /* int32 [T*k] flat (t*k+j) index at each grouped position   */
  size_t inv_pos;      /* int32 [T*k] grouped position of each flat index           */
  size_t tiles;        /* int32 [4 + 4*max_tiles]: count, 3 pad, then {expert,row0,rows,0} */
  size_t xp;           /* uint8 [T*k, H] x codes in grouped order                   */
  size_t xp_sf;        /* uint8 [max_tiles, ceil(H/128), 512] scale atoms of xp     */
  size_t hq;           /* uint8 [T*k, I] E4M3 codes of h                            */
  size_t hq_sf;        /* uint8 [max_tiles, ceil(I/128), 512] scale atoms of hq     */
  size_t y;            /* fp32 [T*k, H] per-(token, slot) expert outputs            */
  size_t total;        /* bytes needed                                              */
  int32_t max_tiles;   /* capacity of the tile list                                 */
  int32_t tile_rows;   /* token rows per tile used for this T                       */
} moe_workspace_layout;

/* Bytes of the packed (repacked) weight buffer for these dims; 0 if the
 * dims are unsupported.  (The packed form has no counterpart on the pages; it
 * holds the tensors of "MXFP4 Tensor Structure" rearranged, see below.) */
size_t moe_packed_size(moe_dims d);

/*
 * Repack checkpoint-layout MXFP4 expert weights ("GPT-OSS-120B on DGX Spark:
 * From MXFP4 to NVFP4", section "MXFP4 Tensor Structure": *_blocks
 * [E, out, in/32, 16] packed E2M1, *_scales [E, out, in/32] E8M0, *_bias bf16)
 * into the layout the forward kernels stream: rows padded along the
 * contraction axis to a multiple of 128 elements, gate and up rows interleaved
 * per 128-row tile, E8M0 scales
 * rearranged into the tensor-core scale-factor atoms, biases widened to fp32.
 * The source tensors are only read.  `packed` (device, 256-byte aligned,
 * >= moe_packed_size(d) bytes) is fully written, header included.
 * Asynchronous on `stream`; the source must stay valid until the work ends.
 */
moe_status moe_pack_weights(moe_dims d, const moe_mxfp4_weights *src, void *packed,
                            size_t packed_bytes, void *stream);

/*
 * NVFP4 variant of the weights: the checkpoint-layout MXFP4 tensors converted to
 * NVFP4 while packing, by the method of "GPT-OSS-120B on DGX Spark: From MXFP4 to
 * NVFP4", "Conversion Methodology": dequantise each MXFP4 block (E2M1 value times
 * 2^(scale - 127)), then per 16-element block take the amax, choose the E4M3
 * block scale E4M3(amax / (6 gs)) and quantise the elements to E2M1 (round to
 * nearest even, saturating at 6), with a global scale gs = amax / (6 * 448) per
 * projection over all experts (this library's reading: the page returns "a global
 * scale factor" without its rule).  Same layout otherwise (gate/up interleave,
 * tile-contiguous data, fp32 biases); two scale atoms per k-tile; the global
 * scales' source amax is kept in the header.  H and I must be multiples of 64
 * (else MOE_ERR_UNSUPPORTED_SHAPE).  Sizes, ownership, ordering and errors as
 * moe_pack_weights.
 */
size_t moe_packed_size_nvfp4(moe_dims d);
moe_status moe_pack_weights_nvfp4(moe_dims d, const moe_mxfp4_weights *src, void *packed,
                                  size_t packed_bytes, void *stream);

/* Workspace bytes moe_forward needs for up to T tokens with top_k (0 for
 * unsupported dims or arguments).  The workspace has no counterpart on the
 * pages: it holds this library's intermediates (logits, grouping, quantised
 * activations, the expert outputs before the combine). */
size_t moe_workspace_size(moe_dims d, int32_t T, int32_t top_k);

/* Offsets of the intermediates for T tokens (same layout moe_forward uses). */
moe_status moe_workspace_layout_get(moe_dims d, int32_t T, int32_t top_k,
                                    moe_workspace_layout *out);

/* The same for moe_forward_act in activation format act_format (MOE_ACT_*): the
 * section offsets and total are those of moe_workspace_layout_get; tile_rows and
 * max_tiles are the ones that format's forward uses.  An unknown format is
 * MOE_ERR_INVALID_ARG. */
moe_status moe_workspace_layout_act(moe_dims d, int32_t T, int32_t top_k, int32_t act_format,
                                    moe_workspace_layout *out);

/*
 * One MoE layer forward for T tokens: the layer defined at the top of this
 * file.  Passages: "GPT-OSS-120B on DGX Spark: From MXFP4 to NVFP4", section
 * "GPT-OSS-120B Architecture" (128 experts, top-4 routing, hidden 2880, router
 * weights in BF16) and section "MXFP4 Tensor Structure" (E2M1 values, E8M0
 * scales with bias 127); "GPT-OSS-120B with MXFP4 on DGX Spark (SM121/GB10)",
 * section "What's Included" (the MoE layer as an FP8 x FP4 grouped GEMM) and
 * section "Numerical Accuracy" (full-scale block activation quantisation).
 *   hidden    bf16 [T, H]            (16-byte aligned)
 *   router_w  bf16 [E, H]            (16-byte aligned)
 *   router_b  bf16 [E]
 *   packed    output of moe_pack_weights for the same dims
 *   top_k     1 <= top_k <= min(E, 8)
 *   out       bf16 [T, H]            (written; may not alias the inputs)
 *   workspace device scratch, 256-byte aligned, >= moe_workspace_size(d, T, top_k)
 * T = 0 is a no-op returning MOE_OK.  Nothing is allocated; no host
 * synchronisation happens, so the call can be captured into a CUDA graph.
 * Device-side bounded waits that expire set a status word in the workspace
 * (read it with moe_get_device_status) and the kernels return early; they
 * never trap or hang.
 */
moe_status moe_forward(moe_dims d, const void *hidden, int32_t T, const void *router_w,
                       const void *router_b, const void *packed, int32_t top_k, void *out,
                       void *workspace, size_t workspace_bytes, void *stream);

/*
 * The layer with a choice of activation format (act_format):
 *   MOE_ACT_MXFP8  x and h quantised to MXFP8 (E4M3, one E8M0 scale per 32): the
 *                  FP8-activation x FP4-weight layer, identical to moe_forward;
 *   MOE_ACT_MXFP4  x and h quantised to MXFP4 (E2M1 with the same OCP-style
 *                  shared exponent, floor(log2 amax) - 2, round-to-nearest-even,
 *                  saturating at +-6), run on the tensor cores as FP4 x FP4
 *                  (tcgen05 kind::mxf4) with both operands packed.
 * Passage: "GPT-OSS-120B with MXFP4 on DGX Spark (SM121/GB10)", section
 * "Performance Optimizations" (native FP4 x FP4 block-scale MMA as the next
 * step after FP8 x FP4); the activation rule is this library's reading of
 * "Numerical Accuracy" (full-scale block activation quantisation), the same as
 * for MXFP8.
 *   MOE_ACT_NVFP4  the NVFP4 variant: `packed` must come from moe_pack_weights_nvfp4
 *                  (the weights converted to NVFP4); x and h are quantised to
 *                  NVFP4 (E2M1 in 16-element blocks with an E4M3 scale each,
 *                  amax / 6 rounded to nearest even, unit global scale), and the
 *                  MMA is tcgen05 kind::mxf4nvf4.  Passages: "GPT-OSS-120B on DGX
 *                  Spark: From MXFP4 to NVFP4", "The MXFP4 -> NVFP4 Conversion";
 *                  "GPT-OSS-120B with MXFP4 on DGX Spark (SM121/GB10)", "New
 *                  Features" (NVFP4 format support, group size 16).  Routing takes
 *                  the tensor-core path at every T.
 * Same arguments, workspace and errors as moe_forward (an unknown act_format is
 * MOE_ERR_INVALID_ARG); in the FP4 formats the workspace's xq, xp and hq sections
 * hold two codes per byte (rows of H/2 and I/2 bytes).  A packed buffer whose
 * header does not match the forward (other dims, or MXFP4 weights for the NVFP4
 * format and the reverse) runs no expert unit and reports MOE_ERR_TIMEOUT-class
 * status bit 0x20 through moe_get_device_status; the output is then not written.
 */
#define MOE_ACT_MXFP8 0
#define MOE_ACT_MXFP4 1
#define MOE_ACT_NVFP4 2
moe_status moe_forward_act(moe_dims d, int32_t act_format, const void *hidden, int32_t T,
                           const void *router_w, const void *router_b, const void *packed, int32_t top_k,
                           void *out, void *workspace, size_t workspace_bytes, void *stream);

/*
 * Allocation-free forward.  This entry point has no counterpart in the pages
 * the layer follows; it exists for callers that cannot allocate device memory
 * themselves: code whose device memory is owned by a host runtime that forbids
 * or budgets cudaMalloc (plugins, fixed-pool serving runtimes), or code that
 * must not call an allocator in its launch path because cudaMalloc can
 * synchronise the device.  It computes exactly what moe_forward computes, with
 * the same arguments minus the workspace: its scratch is a file-scope device
 * array of MOE_STATIC_SCRATCH_BYTES inside this library (held by every GPU that
 * loads the library until the process exits; enough for a gpt-oss-sized layer
 * up to T = 128 with top_k = 4).
 *  - A call whose scratch need (moe_workspace_size) exceeds that size returns
 *    MOE_ERR_WORKSPACE_TOO_SMALL with a message; nothing is enqueued.
 *  - Nothing is allocated: no cudaMalloc, cudaFree or allocating library call.
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress, with that device current); make that first call
 *    before any stream capture on the device.
 *  - Every call on a device shares the one array, which keeps the last call's
 *    contents (the forward resets the words it needs zeroed itself).  Calls that
 *    overlap on the GPU (concurrent streams or host threads) race on it:
 *    serialise them.
 */
#define MOE_STATIC_SCRATCH_BYTES ((size_t)24 << 20)
moe_status moe_forward_static_scratch(moe_dims d, const void *hidden, int32_t T, const void *router_w,
                                      const void *router_b, const void *packed, int32_t top_k, void *out,
                                      void *stream);

/* Failure detection (no counterpart on the pages).  Synchronise `stream`, then
 * read the workspace status words: MOE_OK, or MOE_ERR_TIMEOUT if a kernel of
 * the last forward that used `workspace` gave up on a bounded wait (its output
 * is then not valid).  `workspace` is the device workspace passed to that
 * forward; NULL is MOE_ERR_INVALID_ARG.  Takes a workspace, unlike a global
 * status query, because concurrent forwards on different workspaces report
 * separately. */
moe_status moe_get_device_status(const void *workspace, void *stream);

/* The same for the allocation-free entry point: synchronise `stream`, then read
 * the status words at the start of the library's static scratch array on the
 * current device (the last moe_forward_static_scratch call on it). */
moe_status moe_static_scratch_status(void *stream);

/* Size of the static scratch array (MOE_STATIC_SCRATCH_BYTES of the library as
 * built), for callers that load the library without this header. */
size_t moe_static_scratch_bytes(void);

/*
 * Failure detection (no counterpart on the pages): the limit, in nanoseconds,
 * of every bounded device-side wait (pipeline barriers, the expert kernel's
 * dependency counters, the small-batch routing grid's barrier) in kernels
 * launched after the call.  0 restores the default of 2 s; other values must lie
 * in [1 us, 60 s], else MOE_ERR_INVALID_ARG.  A healthy wait lasts microseconds,
 * so a limit of a millisecond or more never fires in a correct run.  Process-wide;
 * forwards already enqueued (or captured in a graph) keep the limit they were
 * launched with.
 */
moe_status moe_set_wait_limit_ns(uint64_t ns);
uint64_t moe_get_wait_limit_ns(void);

/*
 * Test hook for failure detection (no counterpart on the pages).  `which` is a
 * mask of the waits that later forwards make unreachable, so that they always
 * expire:
 *   MOE_DEBUG_HOLD_DOWN_UNITS       the expert kernel's down units wait for one
 *                                   more gate_up completion than exists;
 *   MOE_DEBUG_HOLD_ROUTING_BARRIER  the small-batch routing grid (8 < T <= 32)
 *                                   waits at its grid barrier for one more CTA
 *                                   than it has; after the cluster routing kernel
 *                                   (T <= 8) the expert kernel waits for one more
 *                                   routing CTA than published its grouped rows.
 * Such a forward reports MOE_ERR_TIMEOUT through moe_get_device_status after a
 * few wait limits (pair the hook with a short moe_set_wait_limit_ns), its output
 * is not valid, and the device stays usable.  0 restores normal forwards.
 * Process-wide.
 */
#define MOE_DEBUG_HOLD_DOWN_UNITS 1
#define MOE_DEBUG_HOLD_ROUTING_BARRIER 2
moe_status moe_debug_hold_waits(int32_t which);

/*
 * Dense MXFP4 linears: out = MXFP8(x) . W^T + b, for the attention projections and
 * the LM head ("GPT-OSS-120B with MXFP4 on DGX Spark (SM121/GB10)", section "What's
 * Included", "Full MXFP4 Quantization Stack": QKV projections, O projections and
 * the LM head in MXFP4; section "Performance Optimizations": a CUDA-core path for
 * M <= 4 beside the tensor cores).  W is [N, K] (N outputs, K inputs), x bf16
 * [T, K], b bf16 [N] (optional), out bf16 [T, N]; x is quantised per 32-element
 * block to MXFP8 exactly as in the MoE layer.  N must be a multiple of 64 and K
 * of 32 (else MOE_ERR_UNSUPPORTED_SHAPE).  All pointers are device pointers owned
 * by the caller; everything is asynchronous on `stream`.
 *
 * moe_dense_quantize_weights: BF16 weights w [N, K] -> MXFP4 in the checkpoint
 *   layout, blocks [N, K/32, 16] (two E2M1 codes per byte, even element in the low
 *   nibble) and E8M0 scales [N, K/32], by the activations' block rule (shared
 *   exponent floor(log2 amax) - 2, E2M1 round-to-nearest-even, saturating at 6);
 *   the checkpoint keeps these projections in BF16 ("GPT-OSS-120B on DGX Spark:
 *   From MXFP4 to NVFP4", "MXFP4 Tensor Structure").
 * moe_dense_pack: MXFP4 checkpoint-layout W (+ bias, may be NULL) -> the packed
 *   form moe_dense_forward streams (moe_dense_packed_size bytes, 256-byte aligned).
 * moe_dense_forward: T = 0 is a no-op; the workspace (256-byte aligned,
 *   moe_dense_workspace_size bytes) holds the quantised input and, for a few
 *   tokens, K-chunk partial sums.  A few tokens (T <= 4) take the CUDA-core path
 *   (a GEMV streaming the packed weights), more the tensor-core path (the MoE
 *   layer's block-scaled GEMM with one expert); moe_set_plan can force either
 *   (MOE_EXPERT_CUDA_CORES / MOE_EXPERT_WEIGHTS_M).
 */
size_t moe_dense_packed_size(int32_t N, int32_t K);
moe_status moe_dense_quantize_weights(int32_t N, int32_t K, const void *w, void *blocks, void *scales,
                                      void *stream);
moe_status moe_dense_pack(int32_t N, int32_t K, const void *blocks, const void *scales, const void *bias,
                          void *packed, size_t packed_bytes, void *stream);
size_t moe_dense_workspace_size(int32_t N, int32_t K, int32_t T);
moe_status moe_dense_forward(int32_t N, int32_t K, const void *x, int32_t T, const void *packed, void *out,
                             void *workspace, size_t workspace_bytes, void *stream);

/*
 * Residual stream of a stack of MoE layers, x <- x + moe(rmsnorm(x)) (the
 * stacked-layer workload; RMSNorm with unit gain; 36 MoE layers per model,
 * "GPT-OSS-120B on DGX Spark: From MXFP4 to NVFP4", section "GPT-OSS-120B
 * Architecture", which names the layernorms without their form): if layer_out (bf16 [T, H],
 * the previous layer's moe_forward output) is not NULL, x_res (fp32 [T, H]) +=
 * layer_out; then hidden (bf16 [T, H]) = bf16(x_res / sqrt(mean(x_res^2) + eps))
 * per token, ready to be the next layer's input.  H a multiple of 4.
 */
moe_status moe_residual_rmsnorm(float *x_res, const void *layer_out, int32_t T, int32_t H, float eps,
                                void *hidden, void *stream);

/*
 * Measurement hook for the tile and schedule selection (the pages' planned
 * autotuner and small-tile variants: "GPT-OSS-120B with MXFP4 on DGX Spark
 * (SM121/GB10)", "Performance Optimizations").  Forces the token rows per expert
 * tile of the grouped GEMM (8, 16, 32, 64 or 128; 0 = the measured default for
 * T), the routing path (MOE_ROUTE_AUTO = the measured default; _CLUSTER needs
 * T <= 8, _GRID T <= 32, _TENSOR_CORE any T) and the expert kernel
 * (MOE_EXPERT_AUTO = the measured default; _WEIGHTS_M = weight rows in the MMA's
 * M slot and token rows in N, any tile height; _TOKENS_M = 128 token rows in M and
 * two 128-row weight tiles in N, 128-row tiles only).
 * Process-wide.  moe_workspace_size
 * and moe_workspace_layout_get follow the tile override, so size workspaces
 * after setting it.  A forced routing path or expert kernel that does not fit
 * the call makes that forward return MOE_ERR_UNSUPPORTED_SHAPE.  Results do not depend on the
 * plan; only the launch shapes do.  Invalid values are MOE_ERR_INVALID_ARG.
 */
#define MOE_ROUTE_AUTO 0
#define MOE_ROUTE_CLUSTER 1
#define MOE_ROUTE_GRID 2
#define MOE_ROUTE_TENSOR_CORE 3
#define MOE_EXPERT_AUTO 0
#define MOE_EXPERT_WEIGHTS_M 1
#define MOE_EXPERT_TOKENS_M 2
#define MOE_EXPERT_CUDA_CORES 3 /* dense linears only: the CUDA-core path (T <= 4) */
moe_status moe_set_plan(int32_t tile_rows, int32_t route, int32_t expert_kernel);

/*
 * Optional per-stage timing of moe_forward with CUDA events (measurement; no
 * counterpart on the pages) (host-side event
 * objects only; no device memory).  moe_profile_begin(n) arms event recording
 * for the next n forward calls (three events each: start, expert-kernel start,
 * end; inside a stream capture they become timestamping graph nodes);
 * moe_profile_end synchronises on the recorded events and writes, per stage,
 * the summed milliseconds over the recorded calls into stage_ms[0..1] and the
 * number of calls into *calls.  Stages: 0 routing (router GEMV, top-k +
 * softmax, MXFP8 of x, grouping, gather), 1 expert MLP (gate_up GEMM + SwiGLU +
 * MXFP8, down GEMM, combine in one persistent kernel).  Not thread-safe.
 */
moe_status moe_profile_begin(int32_t max_calls);
moe_status moe_profile_end(double *stage_ms, int32_t *calls);

/* Thread-local message of the last non-OK status returned on this thread. */
const char *moe_last_error(void);

/* Library version (packed layout version in the low 16 bits). */
uint32_t moe_version(void);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */

/*
 * moe_decode.h -- C ABI of the GB300 (sm_103a) routing-and-combine path of a
 * decode-step latent-MoE layer.
 *
 * The path, per decode step of T token rows:
 *   router logits (BF16 x, BF16 gate -> FP32)  ->  sigmoid + bias top-k with
 *   renormalised weights  ->  per-expert routing lists  ||  MXFP8 quantisation of the
 *   latent rows  ->  Finalize (the weighted top-k sum of the experts' rows).
 *
 * Source pages (vLLM API documentation):
 *   [wide] "vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.moe.wide"
 *   [ep]   "vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.moe.ep.layer"
 *   [fin]  "vllm.models.glm5next.nvidia.specialized_decode.cutedsl.finalize_publish"
 *
 * Conventions shared by every call
 *   - Pointers named as device buffers must be device (or managed) memory of the
 *     current CUDA device; the caller owns every buffer. The library never allocates,
 *     frees or synchronises in these calls, and keeps no per-call state.
 *   - Every call is asynchronous and stream ordered on `stream` (a cudaStream_t;
 *     NULL is the legacy default stream). Kernels are launched with programmatic
 *     dependent launch, so consecutive calls on one stream overlap their launch
 *     latency; each kernel waits for its predecessor before touching dependent data.
 *   - Arguments are validated synchronously before anything is launched; on an
 *     error nothing is launched and the status says why. No exception crosses the ABI.
 *   - BF16 tensors are passed as uint16_t bit patterns, E4M3 / E8M0 bytes as uint8_t.
 *     Tensors are dense row-major.
 *   - Data-dependent errors that only the GPU can see (an out-of-range index) do not
 *     fault: the kernel skips the offending element and sets a bit in the library's
 *     device error word, read with moe_device_error().
 */
#ifndef MOE_DECODE_H
#define MOE_DECODE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream (identical to cudaStream_t / CUstream). */
typedef struct CUstream_st* moe_stream_t;

/* Status codes returned by every call. */
#define MOE_OK 0
#define MOE_ERR_INVALID_ARGUMENT 1 /* bad size, null required pointer, bad flag (the pages' ValueError on a bad width) */
#define MOE_ERR_ALIGNMENT 2        /* a vectorised pointer is not 16-byte aligned */
#define MOE_ERR_CAPACITY 3         /* a size beyond what the call supports (the pages' ValueError on tokens outside capacity) */
#define MOE_ERR_WORKSPACE 4        /* workspace missing or smaller than the *_workspace() query (the pages' RuntimeError on scratch misuse) */
#define MOE_ERR_UNSUPPORTED 5      /* no GPU, or a device that is not sm_103 */
#define MOE_ERR_CUDA 6             /* a CUDA runtime/driver call or a launch failed */

/* Bits of the device error word (see moe_device_error). */
#define MOE_DEVERR_ROW_INDEX 0x1u /* moe_finalize: a row index outside [-1, n_rows); that term was skipped */
#define MOE_DEVERR_EXPERT_ID 0x2u /* moe_build_routing_lists: an expert id outside [0, E); that pair was dropped */
#define MOE_DEVERR_TIMEOUT 0x4u   /* a bounded wait inside a kernel gave up; that kernel's output is invalid */
#define MOE_DEVERR_CAPACITY 0x8u  /* moe_build_unit_windows: more units than max_units; those past it were not written */

/* Weight dtypes for moe_finalize. */
#define MOE_DTYPE_F32 0
#define MOE_DTYPE_BF16 1

/* Limits. */
#define MOE_MAX_EXPERTS 4096 /* E of moe_topk_route, moe_build_routing_lists and moe_build_unit_windows */
#define MOE_MAX_TOPK 32      /* K of every call */

/* Human-readable name of a status code (static string, never NULL). */
const char* moe_status_string(int status);

/* Library ABI version: major * 10000 + minor * 100 + patch. */
int moe_version(void);

/*
 * Read the device error word of the current device into *bits (may be NULL) and, if
 * clear != 0, reset it to zero. Synchronous: waits for all work on the device.
 * Returns MOE_OK or MOE_ERR_CUDA / MOE_ERR_UNSUPPORTED.
 */
int moe_device_error(uint32_t* bits, int clear);

/* -------------------------------------------------------------------------------
 * Router logits.
 *   logits[t, e] = sum_j x[t, j] * w[e, j]      (FP32 accumulate and output, no bias)
 * Source: [ep] EpMoeLayer.stock_order (mm(x, gate^T) with an FP32 output) and
 * EpMoeLayer.__init__ (the FP32-output split-K router projection, its partials reduced
 * in FP32, module docstring); [wide] module docstring (the router logits are FP32).
 *
 *   x         device, BF16 [T, H]        hidden rows
 *   w         device, BF16 [E, H]        router weight (gate), expert rows
 *   logits    device, FP32 [T, E]        output
 *   workspace device scratch of at least moe_router_logits_workspace(T, H, E) bytes
 *             (may be NULL when that query returns 0); its contents on entry do not
 *             matter and are clobbered. Calls that share a workspace must not overlap.
 * Requirements: T >= 1, E >= 1, H >= 8, H % 8 == 0; x, w 16-byte aligned
 * (MOE_ERR_ALIGNMENT), logits 4-byte aligned.
 * Numerics: BF16 products are exact in FP32; sums are accumulated in FP32 -- for up
 * to 4 tokens on the CUDA cores (one pass over the gate, no split-K: per-lane chains
 * of at most H / 224 fragments x 8 products, then fixed shuffle and warp trees), else
 * on the tensor cores in K-chunks with the split-K partials reduced in a fixed order
 * -- so the result is deterministic run to run. The error is well inside
 * 1e-5 * sum_j |x[t,j] w[e,j]|.
 * ------------------------------------------------------------------------------- */
size_t moe_router_logits_workspace(int T, int H, int E);
int moe_router_logits(const uint16_t* x, const uint16_t* w, float* logits, int T, int H, int E,
                      void* workspace, size_t workspace_bytes, moe_stream_t stream);

/* The same computation with an explicit kernel family: MOE_ROUTER_AUTO (what
 * moe_router_logits uses: the CUDA cores for T <= 4, the tensor cores above),
 * MOE_ROUTER_SIMT (CUDA cores: the GEMV form for T <= 8, else split-K with per-lane
 * FP32 chains of at most 128 products and a fixed butterfly) or MOE_ROUTER_TCGEN05
 * (tensor-core split-K with a TMEM accumulator). The workspace query covers every
 * family. */
#define MOE_ROUTER_AUTO 0
#define MOE_ROUTER_SIMT 1
#define MOE_ROUTER_TCGEN05 2
int moe_router_logits_ex(const uint16_t* x, const uint16_t* w, float* logits, int T, int H, int E,
                         void* workspace, size_t workspace_bytes, int algo, moe_stream_t stream);

/* The router logits for callers that cannot allocate device memory when they call it
 * -- an engine whose pool owns all device memory after start-up, or a plug-in that is
 * handed only its inputs and outputs -- and so cannot pass a workspace. The pages have
 * no counterpart of this call. It computes exactly what moe_router_logits computes
 * (same kernels, same split-K plan, bit-identical results), but keeps the split-K
 * partials in a fixed array of MOE_ROUTER_NOALLOC_SCRATCH_BYTES that the library
 * reserves in the device memory of every GPU that loads it, until the process exits.
 *   - It allocates nothing: no cudaMalloc, no cudaFree, no allocating library call.
 *   - The first call on a device looks up the array's device address with that device
 *     current (cudaGetSymbolAddress) and caches it; make that first call before any
 *     stream capture.
 *   - Sizes whose tensor-core split-K partials would not fit in the array, and
 *     T * E > 2^40 as for moe_router_logits, return MOE_ERR_CAPACITY and launch
 *     nothing. The tensor-core plan keeps (splits x token tiles x 128-expert tiles) at
 *     or below the SM count and a tile's partial at or below 256 x 128 FP32, so its
 *     partials never exceed SM count x 128 KiB: 19 MiB on a 152-SM GB300, inside the
 *     20 MiB array for every T and E. (moe_router_logits_workspace may report more: it
 *     also covers the CUDA-core family, which this call never runs.)
 *   - Every call on a device shares the array and leaves its contents behind; nothing
 *     in it needs to start at zero. Calls whose kernels overlap on the GPU (other
 *     streams, other threads) race on it: order them on one stream.
 * Arguments, requirements and numerics as moe_router_logits. */
#define MOE_ROUTER_NOALLOC_SCRATCH_BYTES (20u * 1024u * 1024u)
int moe_router_logits_noalloc(const uint16_t* x, const uint16_t* w, float* logits, int T, int H, int E,
                              moe_stream_t stream);

/* -------------------------------------------------------------------------------
 * Front projection: the router logits and the latent down projection of the same
 * hidden rows in one tensor-core launch (one pass over x for both weights).
 *   logits[t, e] = sum_j x[t, j] * w_router[e, j]                 FP32 [T, E]
 *   latent[t, l] = bf16_rn( sum_j x[t, j] * w_down[l, j] )        BF16 [T, L]
 * Source: [wide] module docstring (the front is a single GEMM with FP32 output over
 * the rank's router rows and its share of the latent down projection; precision
 * paragraph: logits stay FP32, the latent is rounded to BF16 once, like the stock
 * GEMM's epilogue); [wide] WideMoE.__init__ (`packed`: the router rows stacked on the
 * latent down rows); [ep] EpMoeLayer.stock_order (front = mm(x, front^T), the latent
 * its last 3584 columns, BF16).
 *
 *   x         device, BF16 [T, H]        hidden rows
 *   w_router  device, BF16 [E, H]        router weight (gate)
 *   w_down    device, BF16 [L, H]        latent down projection
 *   logits    device, FP32 [T, E]        output
 *   latent    device, BF16 [T, L]        output
 *   workspace device scratch of at least moe_front_projection_workspace(T, H, E, L)
 *             bytes (NULL allowed when that is 0); clobbered. Calls that share a
 *             workspace must not overlap.
 * Requirements: T, E, L >= 1, H >= 8, H % 8 == 0 (MOE_ERR_INVALID_ARGUMENT);
 * E + L < 2^24 (MOE_ERR_CAPACITY); x, w_router, w_down 16-byte aligned, logits 4-byte,
 * latent 2-byte (MOE_ERR_ALIGNMENT).
 * Numerics: each output is an FP32 tensor-core sum of exact BF16 products, split-K
 * partials (if any) reduced in a fixed order: deterministic, within 1e-5 *
 * sum_j |x w| of the exact sum before the latent's one round-to-nearest-even to BF16.
 * The logits need not be bit-identical to moe_router_logits (another split plan).
 * ------------------------------------------------------------------------------- */
size_t moe_front_projection_workspace(int T, int H, int E, int L);
int moe_front_projection(const uint16_t* x, const uint16_t* w_router, const uint16_t* w_down, float* logits,
                         uint16_t* latent, int T, int H, int E, int L, void* workspace, size_t workspace_bytes,
                         moe_stream_t stream);

/* -------------------------------------------------------------------------------
 * Sigmoid + e_score_correction_bias top-K with renormalised weights.
 * Source: [ep] EpMoeLayer.topk (one group, sigmoid scoring, correction bias,
 * renormalize, routed scaling); [wide] WideRoute docstring (an exact top-16 with
 * renormalised weights); [wide] WideMoE.__init__ (bias, renorm, scale taken from the
 * module); [wide] WideScratch (ids int32 [cap, 16], weights BF16 [cap, 16]).
 *
 * Per token t:
 *   s_e = sigmoid(logits[t, e])  (the library's specified sigmoid: exp by Cody-Waite
 *         reduction + degree-7 Taylor, FP32 add, correctly rounded division;
 *         s = 1 for x >= 17.5, s = 0 for x <= -88.5)
 *   c_e = s_e + bias[e]          (c_e = s_e when bias is NULL)
 *   ids[t, k]  = the k-th expert in the order (c descending, expert index ascending)
 *   S          = s_{ids[t,0]} + ... + s_{ids[t,K-1]}   (FP32, slot order)
 *   weights[t, k] = renormalize ? (S == 0 ? 0 : s_{ids[t,k]} / S) : s_{ids[t,k]},
 *                   then times `scale` when scale != 1
 *   weights_bf16[t, k] = weights[t, k] rounded to nearest even BF16.
 * Weights use the unbiased scores. NaN keys rank below every number.
 *
 *   logits       device, FP32 [T, E]
 *   bias         device, FP32 [E] or NULL
 *   ids          device, int32 [T, K]   output
 *   weights      device, FP32 [T, K]    output (may be NULL)
 *   weights_bf16 device, BF16 [T, K]    output (may be NULL)
 * Requirements: T >= 0 (T == 0 launches nothing), 1 <= K <= min(E, MOE_MAX_TOPK),
 * 1 <= E <= MOE_MAX_EXPERTS (MOE_ERR_CAPACITY beyond); logits, bias, ids and weights
 * 4-byte aligned, weights_bf16 2-byte aligned (MOE_ERR_ALIGNMENT otherwise).
 * Bit-exact and deterministic.
 * ------------------------------------------------------------------------------- */
int moe_topk_route(const float* logits, const float* bias, int T, int E, int K, int renormalize,
                   float scale, int32_t* ids, float* weights, uint16_t* weights_bf16,
                   moe_stream_t stream);

/* moe_topk_route and mxfp8_quantize_rows(latent, rows, cols, q, scales) in ONE launch
 * ([wide] WideRoute: the top-K CTAs and the latent-quantisation CTAs of a batch share
 * one grid): the quantisation CTAs stream the latent on the SMs the selection leaves
 * free. Results are identical to the two separate calls; arguments
 * and requirements are theirs (T >= 1; rows may be 0). */
int moe_topk_route_quantize(const float* logits, const float* bias, int T, int E, int K, int renormalize,
                            float scale, int32_t* ids, float* weights, uint16_t* weights_bf16,
                            const uint16_t* latent, int rows, int cols, uint8_t* q, uint8_t* scales,
                            moe_stream_t stream);

/* -------------------------------------------------------------------------------
 * Per-expert routing lists (counting sort, CSR).
 * Source: [wide] WideRoute docstring and kernel: each of token t's K (token, slot)
 * pairs is appended to its expert's list as the pair code t*K + k, which is also the
 * expanded-row index that Finalize reads.
 *
 *   pairs[offsets[e] .. offsets[e+1]) = the codes t*K + k with ids[t, k] == e, in
 *   ascending t (so ascending code). offsets = exclusive prefix sum of the per-expert
 *   counts; offsets[0] = 0, offsets[E] = T*K.
 *
 *   ids       device, int32 [T, K]   (an id may repeat within a row: each pair is listed)
 *   offsets   device, int32 [E + 1]  output
 *   pairs     device, int32 [T * K]  output
 *   workspace device scratch of moe_build_routing_lists_workspace(T, K, E) bytes; that
 *             size is 0 (NULL is fine): the lists need no scratch.
 * Requirements: T >= 0 (T == 0 writes offsets = 0), 1 <= K <= MOE_MAX_TOPK,
 * 1 <= E <= MOE_MAX_EXPERTS, T*K < 2^31; ids, offsets and pairs 4-byte aligned.
 * An id outside [0, E) is dropped and sets MOE_DEVERR_EXPERT_ID (the lists are then
 * incomplete). Deterministic and free of global atomics.
 * ------------------------------------------------------------------------------- */
size_t moe_build_routing_lists_workspace(int T, int K, int E);
int moe_build_routing_lists(const int32_t* ids, int T, int K, int E, int32_t* offsets,
                            int32_t* pairs, void* workspace, size_t workspace_bytes,
                            moe_stream_t stream);

/* -------------------------------------------------------------------------------
 * Unit windows: the work units a grouped expert engine takes from the routing lists,
 * each touched expert once per `window` of its listed pairs.
 * Source: [wide] module docstring (the grouped engine's unit windows come from the
 * routing lists; each expert with tokens is read once per 8 of them).
 *
 *   n_e = offsets[e+1] - offsets[e];  expert e has ceil(n_e / window) units;
 *   unit_offsets = exclusive prefix sum of those counts (unit_offsets[E] = units);
 *   unit u = unit_offsets[e] + j of expert e:
 *     unit_expert[u] = e, unit_start[u] = offsets[e] + j*window,
 *     unit_len[u] = min(window, offsets[e+1] - unit_start[u])
 *   i.e. the list positions pairs[unit_start[u] .. unit_start[u] + unit_len[u]).
 *
 *   offsets      device, int32 [E + 1]   routing-list offsets (moe_build_routing_lists)
 *   unit_offsets device, int32 [E + 1]   output
 *   unit_expert, unit_start, unit_len    device, int32 [max_units]  outputs
 *   max_units    their capacity; moe_unit_windows_capacity(T, K, E, window) units
 *                always suffice for lists of T*K pairs (ceil(T*K/window) + E, at most
 *                T*K). Units past max_units are not written and set
 *                MOE_DEVERR_CAPACITY; unit_offsets is complete either way.
 * Requirements: 1 <= E <= MOE_MAX_EXPERTS, window >= 1, max_units >= 0; pointers
 * 4-byte aligned. offsets must be non-decreasing (as the lists call writes them).
 * One launch of one CTA; deterministic, bit-exact.
 * moe_unit_windows_capacity returns -1 for invalid sizes.
 * ------------------------------------------------------------------------------- */
int moe_unit_windows_capacity(int T, int K, int E, int window);
int moe_build_unit_windows(const int32_t* offsets, int E, int window, int32_t* unit_offsets, int32_t* unit_expert,
                           int32_t* unit_start, int32_t* unit_len, int max_units, moe_stream_t stream);

/* -------------------------------------------------------------------------------
 * MXFP8 (OCP Microscaling) quantisation of BF16 rows.
 * Source: [wide] module docstring (the activations are MXFP8) and WideRoute (the token's
 * MXFP8 plan row written from its BF16 latent); [ep] module docstring ("the MXFP8
 * latent"). Read as OCP MX v1.0: per block of 32 consecutive elements of a row,
 *   se = clamp(floor(log2(max |v|)) - 8, -127, 127),   scale byte = se + 127 (E8M0),
 *   q  = E4M3(v * 2^-se), round to nearest even, saturating to +-448, sign kept.
 * An all-zero block has scale byte 0 and signed-zero elements; a block holding an
 * infinity or NaN has scale byte 0xFF and elements 0x7F.
 *
 *   x       device, BF16 [rows, cols]
 *   q       device, E4M3 bytes [rows, cols]      output
 *   scales  device, E8M0 bytes [rows, cols/32]   output, row-major
 * Requirements: rows >= 0, cols >= 32, cols % 32 == 0; x 16-byte aligned, q and scales
 * 8-byte aligned. Bit-exact.
 * ------------------------------------------------------------------------------- */
int mxfp8_quantize_rows(const uint16_t* x, int rows, int cols, uint8_t* q, uint8_t* scales,
                        moe_stream_t stream);

/* The same with a choice of the scale rule:
 *   MXFP8_SCALE_FLOOR (what mxfp8_quantize_rows does): se = floor(log2 amax) - 8, the
 *     OCP rule; elements above 448 * 2^se saturate to +-448.
 *   MXFP8_SCALE_CEIL: se = ceil(log2(amax / 448)), the smallest power of two with
 *     amax / 2^se <= 448, so no element saturates (one step above the OCP scale when
 *     the block maximum's significand exceeds 1.75, the same scale otherwise).
 * Source: [ep] module docstring (the latent's MXFP8 bit-identical to the stock
 * mxfp8_quantize, whose scale rule the pages do not show: both readings are offered).
 * Clamping, special blocks, layouts and requirements as mxfp8_quantize_rows; another
 * rule returns MOE_ERR_INVALID_ARGUMENT. */
#define MXFP8_SCALE_FLOOR 0
#define MXFP8_SCALE_CEIL 1
int mxfp8_quantize_rows_ex(const uint16_t* x, int rows, int cols, uint8_t* q, uint8_t* scales, int scale_rule,
                           moe_stream_t stream);

/* The same quantisation with the scales laid out for a block-scaled tensor-core
 * consumer: the tile layout that tcgen05.mma kind::mxf8f6f4 (one E8M0 scale per 32
 * elements) reads through tcgen05.cp, as the PTX ISA describes it. The [rows, cols/32]
 * scale matrix is cut into tiles of 128 rows x 4 scale columns, rows padded to a
 * multiple of 128 and scale columns to a multiple of 4; tile (i, j) is the 512 bytes
 * at (i * ceil(cols/128) + j) * 512, and inside it the scale of row r (0..127) and
 * column c (0..3) is byte 16 * (r mod 32) + 4 * (r div 32) + c. Padding bytes are 0.
 * Source: [wide] WideRoute (the token's plan row written with the swizzled plan_xsf
 * scale layout the grouped expert GEMM reads; that layout itself is not shown, so this
 * call offers the tensor cores' own layout); [ep] module docstring (the MXFP8 latent).
 *   scales  device, mxfp8_tcgen05_scales_bytes(rows, cols) bytes, 16-byte aligned
 * q, scale_rule, requirements and numerics as mxfp8_quantize_rows_ex; every scale byte
 * equals the row-major call's. mxfp8_tcgen05_scales_bytes returns 0 for invalid sizes. */
size_t mxfp8_tcgen05_scales_bytes(int rows, int cols);
int mxfp8_quantize_rows_tcgen05(const uint16_t* x, int rows, int cols, uint8_t* q, uint8_t* scales, int scale_rule,
                                moe_stream_t stream);

/* -------------------------------------------------------------------------------
 * Finalize: the routing-weighted top-K sum, optionally with the shared expert.
 * Source: [wide] Finalize (out[t] = sum_k w[t,k] * rows[16t + k], FP32, k in order,
 * fma, one BF16 rounding; all of a thread's row loads in flight before the math);
 * [fin] _QuadFinalizePublishDeviceKernel (weights read as BF16 or FP32, times
 * routed_scaling_factor when it is not 1, zero for a -1 permuted index whose row is
 * skipped, the shared-expert row added once in FP32 after all k, then one rounding).
 *
 * Per token t and column c, with r(t,k) = row_index ? row_index[t*K+k] : t*K + k:
 *   w_k  = float(weights[t,k]); if scale != 1: w_k = w_k * scale
 *   acc  = +0; for k = 0..K-1 in order: if r(t,k) != -1: acc = fma(w_k, rows[r(t,k), c], acc)
 *   if shared: acc = acc + shared[t, c]
 *   out[t, c] = bf16_rne(acc)
 *
 *   rows       device, BF16 [n_rows, H]
 *   row_index  device, int32 [T, K] or NULL (then row t*K + k; n_rows >= T*K required)
 *   weights    device, [T, K] FP32 (weights_dtype MOE_DTYPE_F32) or BF16 (MOE_DTYPE_BF16)
 *   shared     device, BF16 [T, H] or NULL
 *   out        device, BF16 [T, H]   output (must not alias the inputs)
 * Requirements: T >= 0, 1 <= K <= MOE_MAX_TOPK, H >= 8, H % 8 == 0; rows, shared, out
 * 16-byte aligned. An index outside [-1, n_rows) skips its term and sets
 * MOE_DEVERR_ROW_INDEX. Bit-exact and deterministic.
 * ------------------------------------------------------------------------------- */
int moe_finalize(const uint16_t* rows, int64_t n_rows, const int32_t* row_index,
                 const void* weights, int weights_dtype, const uint16_t* shared,
                 float routed_scaling_factor, int T, int K, int H, uint16_t* out,
                 moe_stream_t stream);

/* -------------------------------------------------------------------------------
 * Finalize with the RMSNorm epilogue: the routed latent (as moe_finalize without a
 * shared row) and its RMS-normalised copy, in one pass over the rows.
 * Source: [ep] EpMoeLayer.forward / stock_order (routed = the experts' weighted sum,
 * then rms_norm(normed, routed, w["norm"], eps = 1e-5)); [wide] WideMoE.tail (the
 * latent's RMSNorm, fused with its all-reduce; one GPU has no all-reduce).
 *
 *   routed[t, c] = the moe_finalize output (bit-identical; FP32 fma over k, one BF16 rounding)
 *   x = routed[t, :] as FP32,  ss = sum_c x[c]^2 (FP32, fixed blocked order)
 *   out[t, c] = bf16_rn( (x[c] * rsqrt_rn(ss / H + eps)) * norm_weight[c] )
 *
 *   rows, row_index, weights, weights_dtype, routed_scaling_factor: as moe_finalize
 *   norm_weight device, BF16 [H]; eps >= 0 (the pages' default 1e-5)
 *   routed      device, BF16 [T, H] output, or NULL (not written)
 *   out         device, BF16 [T, H] output
 * Requirements: T >= 0 (T == 0 launches nothing), 1 <= K <= MOE_MAX_TOPK, H % 256 ==
 * 0 and 256 <= H <= 8192 (MOE_ERR_CAPACITY above); rows, out, routed and norm_weight
 * 16-byte aligned. Row indices as moe_finalize (-1 skipped; out of range sets
 * MOE_DEVERR_ROW_INDEX). `routed` is bit-exact; `out` is within 2^-16 relative of the
 * exact normalisation of `routed` before its one rounding. Deterministic.
 * ------------------------------------------------------------------------------- */
int moe_finalize_rmsnorm(const uint16_t* rows, int64_t n_rows, const int32_t* row_index, const void* weights,
                         int weights_dtype, float routed_scaling_factor, const uint16_t* norm_weight, float eps, int T,
                         int K, int H, uint16_t* routed, uint16_t* out, moe_stream_t stream);

/* -------------------------------------------------------------------------------
 * The whole routing-and-combine step in one call.
 * Source: [wide] WideMoE.run (router logits -> route -> ... -> Finalize of the
 * token's top-K expert rows, on one stream) and [ep] EpMoeLayer.__call__.
 *
 * Computes, on `stream`, what these four calls compute, in this order:
 *   moe_router_logits(x, w, logits, T, H, E, workspace, ...)
 *   moe_topk_route_quantize(logits, bias, T, E, K, renormalize, scale, ids, weights,
 *                           weights_bf16, latent, T, L, q, scales)
 *   moe_build_routing_lists(ids, T, K, E, offsets, pairs)
 *   moe_finalize(rows, T*K, NULL, weights_bf16, MOE_DTYPE_BF16, NULL, 1, T, K, L, out)
 * i.e. Finalize combines the expanded expert rows (row t*K + k = token t's k-th
 * expert) with the BF16 routing weights, as the wide page's Finalize does. Every
 * output equals the four calls' bit for bit. It takes three launches (programmatic
 * dependent launch between them): the router, whose warps that wait for its tensor-core
 * mainloop meanwhile quantise the latent to MXFP8 (for up to 4 tokens, whose router runs
 * on the CUDA cores, the next launch does); top-K, whose routing CTAs (four tokens each)
 * also write each token's slots by expert to the workspace; and Finalize, whose launch
 * also builds the routing lists from those slots
 * in CTAs of its own (Finalize does not read the lists, so they are built beside its row
 * stream). Where top-K runs one CTA per token (E > 1024 or E % 4 != 0), or a range's
 * slot map with its per-chunk counts does not fit the Finalize CTAs' shared memory in
 * chunks (T above 65280 at K = 16, above 16256 at K = 8), the lists kernel runs between
 * the last two launches instead. For token tiles wider
 * than 64 the router stores its split-K partials in the workspace instead of reducing
 * them, and the top-K launch sums each token's partials in the same split order before
 * selecting: the same logits, one on-chip exchange fewer. Arguments, layouts and
 * requirements are those of the four calls (weights may be NULL; weights_bf16 may
 * not); they are all checked before the first launch. `workspace` holds
 * moe_route_finalize_workspace(T, H, E, K) bytes, 16-byte aligned (the router's
 * split-K partials and the top-K launch's slot map for the lists); it is clobbered. Returns the first non-OK status (nothing is launched after it). Allocates
 * nothing, so the call can be captured in a CUDA graph.
 * ------------------------------------------------------------------------------- */
size_t moe_route_finalize_workspace(int T, int H, int E, int K);
int moe_route_finalize(const uint16_t* x, const uint16_t* w, const float* bias, const uint16_t* latent,
                       const uint16_t* rows, int T, int H, int L, int E, int K, int renormalize, float scale,
                       float* logits, int32_t* ids, float* weights, uint16_t* weights_bf16, int32_t* offsets,
                       int32_t* pairs, uint8_t* q, uint8_t* scales, uint16_t* out, void* workspace,
                       size_t workspace_bytes, moe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_DECODE_H */

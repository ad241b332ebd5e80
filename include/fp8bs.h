/*
 * fp8bs.h -- C ABI of the GB300 (sm_103a) FP8 block-scaled linear library.
 *
 * The operations follow DeepSeek-V3's FP8 inference path as these pages
 * state it:
 *   - "Data flow -- deepseek-ai/DeepSeek-V3" (codevetter.com), bullet
 *     "FP8 quantization data flow": act_quant produces a float8_e4m3fn tensor
 *     and fp32 scales per 128-element block; fp8_gemm multiplies the scaled
 *     blocks accumulating in fp32; each FP8 weight carries a .scale grid.
 *   - "DeepSeek-V3" source tour (pyshine.com), section "The Three Ideas That
 *     Make V3 Fast", paragraph "FP8 with per-block scales": a tile's max is
 *     clamped and divided by 448 (the e4m3 ceiling); weights are e4m3 with a
 *     scale grid over 128-element blocks; linear() either dequantises the
 *     weight (weight_dequant) or stays in FP8 (act_quant + fp8_gemm).
 *   - "Behavior traces -- deepseek-ai/DeepSeek-V3" (codevetter.com), bullets
 *     "MoE trace" (tokens routed to experts, y[idx] += expert(x[idx]) * w)
 *     and "fp8->bf16 trace" (weight_dequant over a checkpoint); source tour,
 *     "Honest Limits": serious deployments replace the per-expert loop with
 *     a fused grouped GEMM.
 *
 * Conventions shared by every entry point:
 *   - All pointers marked "device" are CUDA device pointers owned by the
 *     caller; the library allocates no device memory and keeps no pointer
 *     after a call returns.  Tensors are dense and row-major.
 *   - bf16 data is bfloat16; e4m3 data is float8_e4m3fn (one byte); scales
 *     are fp32.  A scale multiplies to dequantise: value = code * scale.
 *   - Blocks are 128 elements: activation scales are [rows, K/128]; weight
 *     scales are [ceil(N/128), K/128] for a weight [N, K] (y = x W^T).
 *   - `stream` is a cudaStream_t (NULL: the legacy default stream).  Calls
 *     only enqueue work; they never synchronise, except fp8_device_status.
 *   - Errors are returned, never raised: FP8_ERR_INVALID_ARG for a bad
 *     pointer, size or alignment (nothing is launched), FP8_ERR_CUDA when a
 *     launch fails.  A kernel whose internal wait ran out of time records
 *     FP8_ERR_TIMEOUT, and fp8_gemm_ue8m0 given a scale that is not a power
 *     of two records FP8_ERR_INVALID_ARG; fp8_device_status reports either.
 *   - Pointers to e4m3 or bf16 matrices read by the GEMMs must be 16-byte
 *     aligned; K must be a multiple of 128.
 */
#ifndef FP8BS_H
#define FP8BS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FP8_OK = 0,
    FP8_ERR_INVALID_ARG = 1,
    FP8_ERR_UNSUPPORTED = 2,
    FP8_ERR_CUDA = 3,
    FP8_ERR_TIMEOUT = 4,
    FP8_ERR_WORKSPACE = 5
} fp8_status;

/* Scale format (the model's scale_fmt knob): FP32 stores max/448 as is;
 * UE8M0 rounds that scale up to the next power of two (stored as fp32). */
typedef enum { FP8_SCALE_FP32 = 0, FP8_SCALE_UE8M0 = 1 } fp8_scale_fmt;

/* act_quant (data-flow page, "FP8 quantization data flow"; source tour,
 * "FP8 with per-block scales").
 * x [M, K] bf16 (device) -> y [M, K] e4m3 (device), s [M, K/128] fp32
 * (device).  Per 128-block: s = max(max|x|, 1e-4) / 448 (IEEE fp32 divide),
 * ue8m0: s -> smallest power of two >= s; y = e4m3_rne_satfinite(x / s).
 * Requires K % 128 == 0; x, y 16-byte aligned.  M == 0 is a no-op. */
fp8_status fp8_act_quant(const void* x, void* y, float* s, int64_t M, int64_t K,
                         int scale_fmt, void* stream);

/* Weight quantisation with 128x128 blocks (preparing e4m3 weights from
 * bf16 ones, the inverse of weight_dequant).  w [N, K] bf16 -> q [N, K]
 * e4m3, s [ceil(N/128), ceil(K/128)] fp32; a partial block at the N or K
 * edge covers its valid elements only.  Same scale rule as act_quant.
 * Requires K % 16 == 0 and 16-byte aligned w, q. */
fp8_status fp8_weight_quant(const void* w, void* q, float* s, int64_t N, int64_t K,
                            int scale_fmt, void* stream);

/* weight_dequant (behavior-traces page, "fp8->bf16 trace"; source tour,
 * "FP8 with per-block scales").  w [M, N] e4m3, s [ceil(M/128), ceil(N/128)]
 * fp32 -> y [M, N] bf16 = bf16_rne(fp32(w) * s) (one fp32 multiply).
 * Requires N % 16 == 0 and 16-byte aligned w, y. */
fp8_status fp8_weight_dequant(const void* w, const float* s, void* y, int64_t M, int64_t N,
                              void* stream);

/* Bytes of workspace fp8_gemm needs for this shape on the current device
 * (0 when the schedule needs none).  Layout: 16 KiB of split-tile counters,
 * then fp32 partial tiles.  The workspace must be zero-filled by the caller
 * before its first use; every call that completes without a device error
 * leaves the counters zero again, so one workspace can serve calls of any
 * shape in stream order (calls that overlap on the GPU need separate
 * workspaces). */
size_t fp8_gemm_workspace_size(int64_t M, int64_t N, int64_t K);

/* fp8_gemm (data-flow page, "FP8 quantization data flow"; source tour,
 * "FP8 with per-block scales").
 * a [M, K] e4m3 with a_s [M, K/128]; b [N, K] e4m3 (the weight) with
 * b_s [ceil(N/128), K/128].  Computes, accumulating in fp32,
 *   C[m, n] = sum_kb a_s[m, kb] * b_s[n/128, kb] * sum_{k in kb} a[m,k] b[n,k]
 * and writes it to c_bf16 [M, N] (bf16, round to nearest even) and/or
 * c_fp32 [M, N] (either may be NULL, not both).  workspace: device buffer of
 * at least fp8_gemm_workspace_size(M, N, K) bytes (see there), else
 * FP8_ERR_WORKSPACE.  M == 0 or N == 0 is a no-op. */
fp8_status fp8_gemm(const void* a, const float* a_s, const void* b, const float* b_s,
                    void* c_bf16, float* c_fp32, int64_t M, int64_t N, int64_t K,
                    void* workspace, size_t workspace_bytes, void* stream);

/* fp8_gemm for power-of-two scales (the pages' optional scale_fmt "ue8m0":
 * every scale rounded up to a power of two), computed by the tensor core's
 * block-scaled MMA: each 128-K block's scales a_s[m, kb] and b_s[n/128, kb]
 * are applied by the MMA as E8M0 exponents, so a tile accumulates over all
 * of K without per-block promotion.  Same arguments, layouts and result as
 * fp8_gemm (the fp32 accumulation order differs; the tolerance is the same),
 * minus the workspace (none is needed).  Requires K % 512 == 0 and 16-byte
 * aligned a, b, a_s and b_s (else FP8_ERR_INVALID_ARG).  Every a_s and b_s
 * value must be a positive normal power of two; any other value makes
 * fp8_device_status report FP8_ERR_INVALID_ARG, and the output is then
 * unspecified.  Meant for prefill shapes: 256 x 256 output tiles on pairs of
 * SMs (thread-block clusters of 2) when there is at least one such tile per
 * SM pair, else 128 x 256 tiles on one SM each. */
fp8_status fp8_gemm_ue8m0(const void* a, const float* a_s, const void* b, const float* b_s,
                          void* c_bf16, float* c_fp32, int64_t M, int64_t N, int64_t K, void* stream);

/* The FP8 branch of the model's linear() (source tour, "FP8 with per-block
 * scales": act_quant of the activations, then fp8_gemm against the e4m3
 * weight and its block scales).  x [M, K] bf16 (device), w [N, K] e4m3,
 * w_s [ceil(N/128), K/128] fp32 -> c_bf16 and/or c_fp32 [M, N].  scale_fmt
 * is the activation scale format.  The result equals fp8_act_quant followed
 * by fp8_gemm bit for bit.  For M <= 16 the quantisation runs inside the
 * decode GEMM kernel (one kernel, no workspace); otherwise the activation
 * codes and scales are staged in the workspace first (act_quant, then the
 * GEMM), whose size fp8_linear_workspace_size() gives (0 when none is
 * needed).  Layout:
 * fp8_gemm's workspace first (same zero-fill rule, and never shorter than
 * its 16 KiB of split-tile counters), then codes and scales, so one
 * workspace can serve both entry points and any shapes in stream order. */
size_t fp8_linear_workspace_size(int64_t M, int64_t N, int64_t K);
fp8_status fp8_linear(const void* x, const void* w, const float* w_s, void* c_bf16, float* c_fp32,
                      int64_t M, int64_t N, int64_t K, int scale_fmt, void* workspace,
                      size_t workspace_bytes, void* stream);


/* fp8_gemm without any allocation (the paper has no counterpart: this is a
 * convenience of this library).  For callers that cannot hand the library a
 * workspace -- code that must not call cudaMalloc on its hot path (it can
 * synchronise the device), code under a fixed memory budget, or hosts whose
 * allocator gives out no scratch.  Same arguments and result as fp8_gemm,
 * minus the workspace: the split-tile scratch comes from a fixed 8 MiB
 * (8388608-byte) device array inside the library, held on every GPU that
 * loads the library until the process exits.
 *   - The first call on each device looks up that array's device address
 *     (cudaGetSymbolAddress, with the device current); make that first call
 *     before any stream capture.
 *   - Shapes whose split-K schedule needs more scratch than the array holds
 *     (fp8_gemm_workspace_size(M, N, K) > 8 MiB) return FP8_ERR_WORKSPACE and
 *     launch nothing; use fp8_gemm with a caller workspace for those.
 *   - Arguments are checked first, exactly as fp8_gemm checks them; a call
 *     that returns an error has enqueued nothing and left the array alone.
 *   - Every accepted call clears the counters it needs on `stream` and then
 *     uses the shared array: calls that may overlap on the GPU (different
 *     streams, different host threads) race on it and must be serialised by
 *     the caller.  No cudaMalloc, cudaFree or allocating routine is called. */
fp8_status fp8_gemm_noalloc(const void* a, const float* a_s, const void* b, const float* b_s,
                            void* c_bf16, float* c_fp32, int64_t M, int64_t N, int64_t K,
                            void* stream);

/* Grouped fp8_gemm over routed experts (behavior-traces page, "MoE trace";
 * source tour, "Honest Limits").  Expert g owns the packed activation rows
 * [offsets[g], offsets[g+1]) of a [R_max, K] (e4m3, scales a_s [R_max,
 * K/128]) and multiplies them by its weight b[g] ([G, N, K] e4m3, scales
 * b_s [G, ceil(N/128), K/128]); the rows of C [R_max, N] are written in the
 * same packed order.  offsets: int32 [G+1] in DEVICE memory, non-decreasing,
 * offsets[0] == 0, offsets[G] <= R_max (rows past offsets[G] are not
 * written).  No host synchronisation.  Requires N % 128 == 0. */
fp8_status fp8_grouped_gemm(const void* a, const float* a_s, const void* b, const float* b_s,
                            const int32_t* offsets, int32_t G, int64_t R_max,
                            void* c_bf16, float* c_fp32, int64_t N, int64_t K, void* stream);

/* The first half of the MLP / expert body with its gate fused in
 * (behavior-traces page, "MoE trace": each expert computes
 * w2(silu(w1 x) * w3 x); source tour, "FP8 with per-block scales": every
 * linear's input is quantised per 128 block): the block-scaled products
 * h1 = a w1^T and h3 = a w3^T, then g = bf16(bf16(silu(h1)) * h3) with h1, h3
 * rounded to bf16, then act_quant(g) -> g_q [M, I] e4m3 and g_s [M, I/128]
 * fp32 -- the same bytes as fp8_gemm (bf16 out) followed by
 * fp8_silu_mul_quant, without h ever leaving the chip.
 * w13 [2I, K] e4m3 holds w1 and w3 INTERLEAVED by 128-row blocks: rows
 * [256 j, 256 j + 128) are w1's rows [128 j, 128 j + 128) and rows
 * [256 j + 128, 256 j + 256) are w3's same rows; w13_s [2I/128, K/128]
 * follows the same block order.  a [M, K] e4m3 with a_s [M, K/128].
 * Requires I % 128 == 0, K % 128 == 0, 16-byte aligned a, w13, g_q.
 * scale_fmt is g's scale format.  No workspace.  M == 0 is a no-op. */
fp8_status fp8_gemm_swiglu(const void* a, const float* a_s, const void* w13, const float* w13_s, void* g_q,
                           float* g_s, int64_t M, int64_t I, int64_t K, int scale_fmt, void* stream);

/* The routed experts' first half in one launch (behavior-traces page, "MoE
 * trace": each expert runs w2(silu(w1 x) * w3 x) on its tokens; source tour,
 * "Honest Limits": a fused grouped GEMM instead of the per-expert loop).
 * Expert g owns the packed rows [offsets[g], offsets[g+1]) of a [R_max, K]
 * e4m3 (scales a_s [R_max, K/128]); its w13 ([G, 2I, K], interleaved as for
 * fp8_gemm_swiglu; scales [G, 2I/128, K/128]) makes h1, h3, and the gate and
 * act_quant run on chip on each finished tile -> g_q [R_max, I] e4m3,
 * g_s [R_max, I/128]
 * in packed row order (rows past offsets[G] are not written).  offsets:
 * int32 [G+1] in device memory.  The same bytes as fp8_grouped_gemm (bf16
 * out) followed by fp8_silu_mul_quant.  Requires I % 128 == 0,
 * K % 128 == 0, 16-byte aligned a, w13, g_q. */
fp8_status fp8_moe_expert_up(const void* a, const float* a_s, const void* w13, const float* w13_s,
                             const int32_t* offsets, int32_t G, int64_t R_max, void* g_q, float* g_s,
                             int64_t I, int64_t K, int scale_fmt, void* stream);

/* Expert body between the two grouped GEMMs, fused with act_quant: for
 * rows r < R and columns i < I,
 *   g = bf16(bf16(silu(h1)) * h3),  silu(v) = v / (1 + exp(-v)) in fp32,
 * then act_quant(g) -> y [R, I] e4m3 and s [R, I/128].  h1 and h3 are bf16
 * with row stride ld_h elements (w1 and w3 outputs side by side: h3 = h1 + I,
 * ld_h = 2I).  g_bf16 [R, I] (nullable) receives g itself.  Requires
 * I % 128 == 0, ld_h % 8 == 0, 16-byte aligned pointers. */
fp8_status fp8_silu_mul_quant(const void* h1, const void* h3, int64_t ld_h, int64_t R,
                              int64_t I, void* y, float* s, void* g_bf16, int scale_fmt,
                              void* stream);

/* MoE routing as a stable counting sort (behavior-traces page, "MoE
 * trace": bincount per expert, then each expert's tokens in order).
 * ids [T, topk] int32 expert ids (distinct within a token, in [0, E)) ->
 * offsets [E+1] (expert e owns packed rows [offsets[e], offsets[e+1])),
 * pair_row [T, topk] (packed row of pair (t, j)), row_token [T*topk]
 * (token of each packed row).  Inside an expert rows follow t*topk + j.
 * All device int32.  E <= 1024. */
fp8_status fp8_moe_route(const int32_t* ids, int64_t T, int32_t topk, int32_t E,
                         int32_t* offsets, int32_t* pair_row, int32_t* row_token,
                         void* stream);

/* Gather of quantised activation rows for the experts: row r of (aq, as)
 * is row row_token[r] of (xq [T, K] e4m3, xs [T, K/128]).  Quantising first
 * and gathering after is exact: act_quant works row by row.
 * Requires K % 128 == 0 and 16-byte aligned xq, aq. */
fp8_status fp8_moe_gather(const void* xq, const float* xs, const int32_t* row_token,
                          int64_t R, int64_t K, void* aq, float* as, void* stream);

/* act_quant of the tokens written straight to their experts' packed rows
 * (behavior-traces page, "MoE trace": each expert takes x[idx] of its
 * tokens): row t of x [T, K] bf16 is quantised once (fp8_act_quant's rule and
 * routine) and its codes and scales are written to packed rows
 * pair_row[t, j], j < topk, of aq [T*topk, K] e4m3 and as [T*topk, K/128]
 * fp32 (pair_row from fp8_moe_route).  The same bytes as fp8_act_quant
 * followed by fp8_moe_gather, with one pass over x.  Requires K % 128 == 0,
 * 16-byte aligned x and aq. */
fp8_status fp8_moe_quant_scatter(const void* x, const int32_t* pair_row, int64_t T, int32_t topk, int64_t K,
                                 void* aq, float* as, int scale_fmt, void* stream);

/* Weighted combine of expert outputs (behavior-traces page, "MoE trace":
 * y[idx] += expert(x[idx]) * weight): y[t, :] = sum_j w[t, j] *
 * out[pair_row[t, j], :] in fp32, written to y_bf16 [T, D] and/or y_fp32
 * [T, D].  out [R, D] bf16; w [T, topk] fp32.  Requires D % 8 == 0. */
fp8_status fp8_moe_combine(const void* out, const float* w, const int32_t* pair_row, int64_t T,
                           int32_t topk, int64_t D, void* y_bf16, float* y_fp32, void* stream);

/* Synchronises `stream`, then returns and clears the library's device
 * status words: FP8_ERR_TIMEOUT if a kernel's bounded wait gave up since
 * the last call, FP8_ERR_INVALID_ARG if fp8_gemm_ue8m0 met a scale that is
 * not a power of two, FP8_ERR_CUDA if the stream reported an error, else
 * FP8_OK.  After FP8_ERR_TIMEOUT the outputs of the calls since the last
 * check are unspecified, and so are the split-tile counters of the
 * workspaces they used: zero those workspaces again before reusing them. */
fp8_status fp8_device_status(void* stream);

/* Test hooks of the failure path (no counterpart in the pages: they exist so
 * that a test can make a kernel's bounded wait run out without faulting or
 * hanging the GPU).  fp8_debug_set_wait_limit sets, on the current device,
 * how many SM clock cycles a kernel waits on one barrier before it gives up
 * (cycles <= 0 restores the default of 2e9, about a second); it copies to
 * device memory synchronously, so call it with no library kernel running.
 * fp8_debug_skip_one_arrive makes the next fp8_gemm call (and only that one)
 * withhold the tensor core's hand-off of its first 128-K slab to the
 * epilogue: the epilogue's wait runs out, the kernel winds down (waits for
 * its own copies and MMAs, frees its tensor memory, returns) and
 * fp8_device_status then reports FP8_ERR_TIMEOUT; that call's output is
 * unspecified.  Neither is meant for production use. */
fp8_status fp8_debug_set_wait_limit(long long cycles);
void fp8_debug_skip_one_arrive(void);

/* Static description of a status code. */
const char* fp8_status_string(fp8_status status);

/* Number of SMs of the current device (the persistent grid size). */
int fp8_num_sms(void);

#ifdef __cplusplus
}
#endif

#endif /* FP8BS_H */

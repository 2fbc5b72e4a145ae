/*
 * wna16_moe.h -- C ABI of the GB300 (sm_103a) WNA16 routed-expert MoE forward.
 *
 * The operation is the indexed routed-expert MoE of the page "Incubate
 * DeepSeek V4 WNA16 runtime on SM86" (section "What this branch adds": items 1
 * "symmetric W2A16 compressed-tensors MoE loading", 2 "separate WNA16 schemas
 * for fused gate/up (w13) and down (w2)", 3 "W2, group-128, BF16 indexed MoE",
 * 9 "SwiGLU alpha, beta, and clamp semantics ... corrected N/K group-shape
 * metadata"), on the weight format of the page
 * "hampsonw/DeepSeek-V4-Flash-0731-WNA16" (section "What changed": symmetric
 * W2A16 with group size 128, "FP16 group scales and INT32 packed values";
 * section "How it was created", step 4: signed codes packed with
 * compressed-tensors).  4-bit experts follow the page "DeepSeek-V4-Flash-
 * W4A16-FP8-MTP -- Ada (SM89) Serving Edition" (section "What this checkpoint
 * is": "W4A16 INT4 experts").
 *
 * Notation: T tokens, K hidden size, N intermediate size, E experts, topk
 * slots per token, b = bits (2 or 4), p = 32/b codes per INT32 word,
 * R = T*topk routed slots (slot f = t*topk + j).
 *
 * Formats (all tensors row-major and contiguous):
 *   x            bf16  [T, K]
 *   topk_ids     int32 [T, topk]       expert of each slot, in [0, E)
 *   topk_weights fp32  [T, topk]
 *   w13_packed   int32 [E, 2N, K/p]    rows [0, N) gate (w1), rows [N, 2N) up (w3)
 *   w13_scales   fp16  [E, 2N, K/g13]  one scale per group of g13 consecutive k
 *   w2_packed    int32 [E, K, N/p]
 *   w2_scales    fp16  [E, K, N/g2]
 *   out          bf16  [T, K]
 * Word layout: element k of a row is field (k mod p) of word (k / p), field j
 * at bits [b*j, b*j + b) (least significant first); the field stores
 * code + 2^(b-1), code in [-2^(b-1), 2^(b-1)).  Dequantised weight:
 * bf16_rne(code * scale), exact product rounded once.
 *
 * Semantics (per slot f = t*topk + j, e = topk_ids[t][j]):
 *   g = W1_e x_t,  u = W3_e x_t                      (fp32 accumulation)
 *   h = bf16( silu(min(g, L)) * clamp(u, -L, L) )    L = swiglu_limit (+inf: no clamp)
 *   y = bf16( W2_e h )
 *   out_t = bf16( sum_j topk_weights[t][j] * y_f )  (fp32, j ascending)
 *
 * Conventions for every call:
 *   - Tensor pointers are DEVICE pointers owned by the caller; the library
 *     never allocates, frees or retains them.  Scratch comes from `workspace`
 *     (size from wna16_moe_workspace_size), also owned by the caller.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream).  The return value reports host-side validation and
 *     launch errors only; device-side conditions (an expert id outside
 *     [0, E), a pipeline wait that timed out) are written to a status word in
 *     the workspace and read with wna16_moe_read_status.
 *   - On any non-zero return nothing has been launched, except
 *     WNA16_ERR_CUDA, which reports a failed launch.
 *   - Thread safety: calls are re-entrant; concurrent calls must not share a
 *     workspace.  All kernels are compiled ahead of time for sm_103a; nothing
 *     is compiled or loaded at run time.
 *   - Bounds-checked build: the same sources compiled with -DWNA16_DEBUG
 *     (libwna16_moe_debug.so) check every index the kernels compute from
 *     routing and tile data (expert rows, permuted rows, split-K slots,
 *     correction rows) and, instead of an out-of-bounds access, skip it and
 *     store WNA16_ERR_INDEX in the status word.
 */
#ifndef WNA16_MOE_H
#define WNA16_MOE_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define WNA16_API __attribute__((visibility("default")))
#else
#define WNA16_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    WNA16_OK = 0,
    WNA16_ERR_INVALID_ARG = -1,       /* null/misaligned pointer, bad size, overlap     */
    WNA16_ERR_UNSUPPORTED = -2,       /* valid but not implemented (bits, group, dims)  */
    WNA16_ERR_WORKSPACE_TOO_SMALL = -3,
    WNA16_ERR_CUDA = -4,              /* a CUDA runtime call or launch failed            */
    /* device status word values (wna16_moe_read_status): */
    WNA16_ERR_BAD_ROUTING = -5,       /* an expert id was outside [0, E); its slot adds 0 */
    WNA16_ERR_DEVICE_TIMEOUT = -6,    /* a pipeline wait gave up; the output is invalid  */
    WNA16_ERR_INDEX = -7              /* bounds-checked build only: a computed index fell
                                         outside its buffer; that access was skipped      */
} wna16_status;

/* Pack signed codes into INT32 words (page "hampsonw/DeepSeek-V4-Flash-0731-
 * WNA16", section "How it was created", step 4).
 *   codes   int8 device [rows, K], each in [-2^(bits-1), 2^(bits-1))
 *   packed  int32 device [rows, K*bits/32] (written)
 * bits in {2, 4}; K a multiple of 32/bits.  Codes outside the range are
 * masked to their low `bits` bits after the offset is added (garbage in,
 * garbage out; never out of bounds). */
WNA16_API int wna16_moe_pack(const int8_t* codes, int64_t rows, int64_t K, int bits, int32_t* packed,
                   void* stream);

/* Bytes of workspace a forward with these sizes needs (0 if unsupported). */
WNA16_API size_t wna16_moe_workspace_size(int64_t T, int64_t K, int64_t N, int64_t E, int topk, int bits);

/* The routed-expert forward (the whole hot path: route/permute, gather,
 * grouped w13 GEMM + clamped SwiGLU, grouped w2 GEMM, weighted combine).
 *   group_size     g13, the group of w13 along K
 *   group_size_w2  g2, the group of w2 along N (0 = same as group_size); the
 *                  per-projection groups are the "projection-specific group
 *                  sizes" of page "Incubate DeepSeek V4 WNA16 runtime on SM86",
 *                  section "Validation completed"
 *   swiglu_limit   L > 0 (may be +inf)
 * Supported: bits in {2,4}; group sizes 32 or multiples of 64 that divide
 * the reduction dim (K for w13, N for w2) -- a group equal to the reduction
 * dim is one scale per output channel -- as long as the scales of one work
 * item (256 weight rows x its groups, double-buffered) leave room for two
 * pipeline stages in shared memory (WNA16_ERR_UNSUPPORTED otherwise; group 32
 * fits up to a reduction dim of 4096);
 * K % 256 == 0; N % 128 == 0; 1 <= topk <= E <= 1024; T*topk < 2^31.
 * x, out, weights and scales 16-byte aligned; out must not overlap x.
 * Returns WNA16_OK or an error (nothing launched). */
WNA16_API int wna16_moe_forward(const void* x, const int32_t* topk_ids, const float* topk_weights,
                      const int32_t* w13_packed, const uint16_t* w13_scales,
                      const int32_t* w2_packed, const uint16_t* w2_scales,
                      int64_t T, int64_t K, int64_t N, int64_t E, int topk,
                      int group_size, int group_size_w2, int bits, float swiglu_limit,
                      void* out, void* workspace, size_t workspace_bytes, void* stream);

/* Expert-parallel partial forward: the experts are split across devices and
 * this call runs the path for the local ones, [expert_begin, expert_begin +
 * E_local) of E_total, only (the expert-parallel deployment of the page
 * "Incubate DeepSeek V4 WNA16 runtime on SM86", section "Measured server60
 * result", shards the same layer across four GPUs; here the experts, not the
 * intermediate dimension, are split).  The weight pointers hold the local
 * experts only ([E_local, ...], local expert i = global expert
 * expert_begin + i); topk_ids hold global ids in [0, E_total).  A slot whose
 * expert is not local contributes nothing.  Output:
 *   out_partial fp32 device [T, K] = sum over the slots t*topk + j with a
 *                local expert (j ascending, fp32) of topk_weights[t][j] * y
 *                where y = bf16(W2 h) as in wna16_moe_forward; not rounded to
 *                BF16, so that the ranks' partials can be summed (in rank
 *                order, fp32) before the final BF16 rounding.
 * Workspace: wna16_moe_workspace_size(T, K, N, E_local, topk, bits).  Other
 * arguments, limits and errors as for wna16_moe_forward (topk <= E_total;
 * E_local <= 1024). */
WNA16_API int wna16_moe_forward_partial(const void* x, const int32_t* topk_ids, const float* topk_weights,
                                        const int32_t* w13_packed, const uint16_t* w13_scales,
                                        const int32_t* w2_packed, const uint16_t* w2_scales,
                                        int64_t T, int64_t K, int64_t N, int64_t E_total, int64_t expert_begin,
                                        int64_t E_local, int topk, int group_size, int group_size_w2, int bits,
                                        float swiglu_limit, float* out_partial, void* workspace,
                                        size_t workspace_bytes, void* stream);

/* Synchronise `stream` and read the device status word of the last call that
 * used `workspace` (WNA16_OK, WNA16_ERR_BAD_ROUTING or
 * WNA16_ERR_DEVICE_TIMEOUT) into *device_status.  Returns WNA16_OK or
 * WNA16_ERR_CUDA. */
WNA16_API int wna16_moe_read_status(const void* workspace, int* device_status, void* stream);

/* Router: the step that produces topk_ids / topk_weights from router logits
 * (the workloads' "top-k softmax routing from N(0,1) logits", renormalised,
 * with the expert-popularity skew entering as a logit bias).  Per token t:
 *   z_e  = logits[t][e] + bias[e]                (one fp32 addition; bias may be NULL)
 *   ids  = the topk experts of largest z, descending; equal z -> lower index
 *          (the order of softmax(z), since exp is increasing)
 *   w_j  = softmax(z) renormalised over the chosen experts
 *        = exp(z_j - z_max) / sum_i exp(z_i - z_max)       (fp32, i in choice order)
 *   logits        fp32 device [T, E], finite
 *   bias          fp32 device [E] or NULL
 *   topk_ids      int32 device [T, topk] (written)
 *   topk_weights  fp32 device [T, topk] (written)
 * 1 <= topk <= min(E, 32); E <= 1024.  Asynchronous on `stream`; returns
 * WNA16_OK, WNA16_ERR_INVALID_ARG, WNA16_ERR_UNSUPPORTED or WNA16_ERR_CUDA
 * (nothing launched on a non-zero return other than WNA16_ERR_CUDA). */
WNA16_API int wna16_moe_route_topk(const float* logits, const float* bias, int64_t T, int64_t E, int topk,
                                   int32_t* topk_ids, float* topk_weights, void* stream);

/* Quantiser: the conversion step that produces the packed words and FP16
 * scales this library consumes -- symmetric RTN with an importance-weighted
 * scale search (page "hampsonw/DeepSeek-V4-Flash-0731-WNA16", section "How it
 * was created", steps 2-5, and its note that importance-weighted RTN was
 * selected).  Per row and group of group_size consecutive k, with
 * lo = -2^(bits-1), hi = 2^(bits-1) - 1:
 *   m = max|w|, s0 = m / 2^(bits-1)
 *   candidates s_i = fp16(fp32(s0 * fp32((10 + i) / 20))), i = 0..30 (factors
 *     0.5 .. 2.0); search = 0: s_10 only (plain RTN)
 *   code = clamp(round-half-even(fp32(w / s)), lo, hi); what = bf16(code * s)
 *     (the forward's dequantisation)
 *   E(s) = sum_k importance[k] * (w - what)^2, fp64, k ascending (importance
 *     1 when NULL); the smallest E wins, ties to the lower i; a group of zeros
 *     gets scale 0.
 *   w           fp32 device [rows, K], 16-byte aligned
 *   importance  fp32 device [K] (per input channel, >= 0) or NULL
 *   packed      int32 device [rows, K*bits/32] (written; the format of
 *               wna16_moe_pack)
 *   scales      fp16 device [rows, K/group_size] (written)
 *   metrics     fp64 device [rows, 4] or NULL (written): per row, weighted
 *               error sum a (w - what)^2, unweighted error sum (w - what)^2,
 *               sum a w^2 and sum w^2, each as per-group fp64 sums added in
 *               group order
 * group_size a multiple of 32 dividing K, K/group_size <= 128.  The result is
 * bit-for-bit reproducible (IEEE operations in a fixed order).  Asynchronous
 * on `stream`; returns WNA16_OK, WNA16_ERR_INVALID_ARG, WNA16_ERR_UNSUPPORTED
 * or WNA16_ERR_CUDA. */
WNA16_API int wna16_moe_quantize(const float* w, int64_t rows, int64_t K, const float* importance, int bits,
                                 int group_size, int search, int32_t* packed, uint16_t* scales, double* metrics,
                                 void* stream);

/* Message for the last host-side error on the calling thread ("" if none). */
WNA16_API const char* wna16_moe_last_error(void);

/* ---- stage entry points, for per-stage parity tests (same conventions). ---- */

/* Stage 1: routing lists.  counts int32[E], offsets int32[E+1] (offsets[E] =
 * number of valid slots), perm int32[R] (slots sorted by (expert, slot),
 * stable), inv int32[R] (inv[perm[i]] = i; -1 for a slot with a bad id),
 * all written into the workspace; copied to the optional outputs. */
WNA16_API int wna16_moe_route(const int32_t* topk_ids, int64_t T, int topk, int64_t E, int64_t K, int64_t N,
                    int bits, int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv,
                    void* workspace, size_t workspace_bytes, void* stream);

/* Stages 1-3 only: h bf16 [R, N] in permuted order (row i = slot perm[i]). */
WNA16_API int wna16_moe_w13(const void* x, const int32_t* topk_ids, const int32_t* w13_packed,
                  const uint16_t* w13_scales, int64_t T, int64_t K, int64_t N, int64_t E, int topk,
                  int group_size, int bits, float swiglu_limit, void* h_out,
                  void* workspace, size_t workspace_bytes, void* stream);

/* Stage 4 alone: y bf16 [R, K] = W2 h for permuted rows; needs the routing
 * lists from wna16_moe_route in the same workspace and h [R, N] in permuted
 * order. */
WNA16_API int wna16_moe_w2(const void* h, const int32_t* w2_packed, const uint16_t* w2_scales,
                 int64_t T, int64_t K, int64_t N, int64_t E, int topk, int group_size_w2, int bits,
                 void* y_out, void* workspace, size_t workspace_bytes, void* stream);

/* Stage 5 alone: out bf16 [T, K] from y bf16 [R, K] (permuted order) using
 * the inverse map of the routing lists in the workspace. */
WNA16_API int wna16_moe_combine(const void* y, const float* topk_weights, int64_t T, int64_t K, int topk,
                      int64_t E, int64_t N, int bits, void* out, void* workspace,
                      size_t workspace_bytes, void* stream);

/* ---- allocation-free forward (no counterpart on the pages). ----
 * For callers that cannot allocate device memory while they run: a serving
 * loop whose device memory is all owned by another allocator, or a
 * latency-critical path that must not risk cudaMalloc failing or
 * synchronising the device.  Same arguments and results as
 * wna16_moe_forward, minus the workspace: the scratch is one fixed 32 MiB
 * device array inside the library, which every GPU that loads the library
 * holds until the process exits.  Sizes whose workspace
 * (wna16_moe_workspace_size) exceeds 32 MiB are rejected with
 * WNA16_ERR_WORKSPACE_TOO_SMALL and a message, and nothing is launched
 * (decode batches up to about 160 tokens of hidden 4096 / intermediate 2048 /
 * 256 experts / top-8 fit).  The call itself allocates nothing: no cudaMalloc
 * or cudaFree and no allocating library routine.  The first call on a device
 * (and the first after that device's context changes) looks up the array's
 * device address (cudaGetSymbolAddress) with that device current; under
 * lazy module loading that lookup is also when the driver loads the array's
 * module and reserves its 32 MiB, so the first call can fail with
 * WNA16_ERR_CUDA when the device is out of memory.  Make one call (or any
 * call that succeeds) at start-up, while memory is free and before any
 * stream capture; later calls reuse the address.  Every call uses the same
 * array and it keeps the previous call's contents (the forward clears what
 * must start at zero); calls that overlap on the GPU -- on different streams
 * or from different host threads -- race on it, so the caller must serialise
 * them.  The device status word lives in that shared array and cannot be read
 * back by the caller. */
WNA16_API int wna16_moe_forward_noalloc(const void* x, const int32_t* topk_ids, const float* topk_weights,
                                        const int32_t* w13_packed, const uint16_t* w13_scales,
                                        const int32_t* w2_packed, const uint16_t* w2_scales,
                                        int64_t T, int64_t K, int64_t N, int64_t E, int topk,
                                        int group_size, int group_size_w2, int bits, float swiglu_limit,
                                        void* out, void* stream);

/* ---- failure detection check (not part of the method). ----
 * Every pipeline wait in the GEMM kernels gives up after a bounded time
 * (2 s), stores WNA16_ERR_DEVICE_TIMEOUT in the workspace status word, makes
 * the CTA's other waits return, drains its copies and MMAs and frees its
 * TMEM, so that a stalled pipeline is reported instead of hanging the GPU.
 * wna16_moe_check_wait_timeout runs one such wait, with a limit of limit_us
 * microseconds (0 < limit_us <= 5e6), on a barrier that nothing completes,
 * and so sets the status word of `workspace` (at least 4 bytes, device) to
 * WNA16_ERR_DEVICE_TIMEOUT; read it with wna16_moe_read_status.  The next
 * forward on that workspace resets the word.  Asynchronous on `stream`.
 * Returns WNA16_OK, WNA16_ERR_INVALID_ARG or WNA16_ERR_CUDA. */
WNA16_API int wna16_moe_check_wait_timeout(void* workspace, size_t workspace_bytes, int64_t limit_us,
                                           void* stream);

/* ---- instrumentation (not part of the method): per-stage device times. ----
 * wna16_moe_profile(slots) with slots > 0 makes every later
 * wna16_moe_forward on the calling thread record CUDA events on its stream
 * before each of its five stages (route, gather, w13, w2, combine) and after
 * the last, into a ring of `slots` forwards; 0 turns it off.  Forwards can be
 * queued without waiting.  wna16_moe_profile_read(ms, n) waits for the last
 * n recorded forwards (n <= slots) and writes their stage durations in
 * milliseconds to ms[5*i + stage], oldest first.
 * Both return WNA16_OK, WNA16_ERR_INVALID_ARG or WNA16_ERR_CUDA. */
WNA16_API int wna16_moe_profile(int slots);
WNA16_API int wna16_moe_profile_read(float* ms, int n);

/* Number of kernels the last successful wna16_moe_forward on the calling
 * thread launched (4 to 10 depending on the plan: routing in one kernel with
 * the gather for small batches, or in one or three kernels plus the gather;
 * w13, with a split-K finalize when decode-sized tiles split it (the two
 * splits of prefill-sized tiles are added inside the w13 kernel); w2;
 * combine; for 2-bit prefill batches with experts of at most 8 rows, one
 * more w13 and one more w2 launch for those experts); 0 before any. */
WNA16_API int wna16_moe_launches_last_forward(void);

#ifdef __cplusplus
}
#endif

#endif /* WNA16_MOE_H */

// Internal interface of the grouped WNA16 GEMM kernel (not part of the C ABI).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace wna16 {

struct GemmParams {
    const int4* tiles;          // token tiles: {expert, first permuted row, rows, 0}
    const int* n_tiles;         // number of valid tiles (device)
    const uint16_t* scales;     // fp16 [E * rows_per_expert, ngroups]
    __nv_bfloat16* out;         // h [R, N] (w13) or y [R, K] (w2), permuted rows
    int out_ld;                 // row length of `out`
    int rows_per_expert;        // 2N (w13) or K (w2)
    int half_rows;              // N (w13: first up row)
    int kred;                   // reduction length: K (w13) or N (w2)
    int ngroups;                // kred / group
    int group;                  // scale group along the reduction dim (32, or a multiple of 64)
    int mt_count;               // 256-row units per expert: N/128 (w13) or K/256 (w2)
    int kp;                     // K elements per pipeline stage
    int nt;                     // token tile (MMA N): 16, 32, 64 or 128
    int nstage;                 // smem pipeline depth
    int nabuf;                  // TMEM A buffers (128 k each)
    int nacc;                   // TMEM accumulator sets (2: the epilogue overlaps the next item)
    int n_issuers;              // MMA-issuing threads (2, 4 or 6 in GA mode)
    int ga;                     // group-accumulate mode (2-bit codes, nt 16, group % 128 == 0): plain codes
                                // into the MMA, one TMEM slot per scale group, scales applied by the epilogue
    int off_b, off_w, off_s, off_bar;   // smem layout (bytes from the 1024-aligned base)
    float limit;                // SwiGLU limit (w13 only)
    int* status;                // device status word
    int ksplit;                 // K splits per unit (1: no split)
    int fuse_splits;            // w13, 2 splits: CTA 2i + 1 (split 1) adds CTA 2i's parked split-0 sums and writes h
    int* unit_flags;            // per unit: epilogue warps of split 0 that have parked their sums (zeroed per forward)
    int early_w;                // the tile list is older than the previous kernel: weights of the first
                                // stages are loaded and converted before the dependency wait
    int w_reuse;                // weight tiles are read again by the expert's other token tiles: load
                                // them with the normal L2 policy instead of evict-first
    float* partial;             // split-K partial sums [ksplit][mt_count][partial_rows][256] fp32
    int partial_rows;           // rows of the permuted token order (R)
    int64_t n_weight_rows;      // E * rows_per_expert (bound of the scale rows, bounds-checked build)
    int h_interleaved;          // w13: h column order of w2's input: 0 natural, 1 / 2 the interleaved
                                // 16-k / 8-k order of the 2-bit / 4-bit A operand (interleave_pos)
    int scale_copy_bytes;       // 16, 8 or 4: cp.async size for the scale rows; 0: plain loads
    const float* csum;          // GA mode with offset codes: per scale group and permuted token row,
                                // sum_k w(k) b[row, k] with w(k) = 130, 34, 10, 130, 34, 10, 130, 34
                                // by k mod 8 ([ngroups][partial_rows]); null: plain codes
};

struct GemmSmem {
    int nstage = 0;
    int off_b = 0, off_w = 0, off_s = 0, off_bar = 0;
    int total = 0;
};

// Shared-memory plan for one launch (ng_item = scale groups per work item);
// nstage < 2 means it does not fit.
GemmSmem gemm_smem_layout(int bits, int nt, int kp, int ng_item, int max_smem);

cudaError_t launch_grouped_gemm(int bits, bool w13, const CUtensorMap& tm_w, const CUtensorMap& tm_b,
                                const GemmParams& p, int grid, int smem_bytes, cudaStream_t stream);

// Record a host-side error message for wna16_moe_last_error (api.cu); returns `code`.
int set_error(int code, const char* fmt, ...);

// Allow kernel `fn` at least `bytes` of dynamic shared memory on the current
// device (api.cu): the opt-in is a per-device function attribute, set once per
// device and kernel (thread-safe).
cudaError_t ensure_dynamic_smem(const void* fn, int bytes);

// Routing / gather / combine / pack kernels (kernels.cu).
// Routing lists of the local experts [e_begin, e_begin + E) among E_total
// (e_begin = 0, E_total = E on a single device).  Batches of more than
// kRouteChunkedMin slots are sorted by chunks in three kernels, with
// route_chunks(R) * (E + 1) ints of chunk_scratch; smaller ones by one CTA.
constexpr int kRouteChunkedMin = 8192;
int route_chunks(int R);
// With light_max > 0 (at most 8), experts of at most light_max rows get one
// tile each in light_tiles (n_light of them) instead of the main list.
cudaError_t launch_route(const int32_t* ids, int R, int E, int e_begin, int E_total, int nt, int* counts,
                         int* offsets, int* perm, int* inv, int4* tiles, int* n_tiles, int* status,
                         int* chunk_scratch, cudaStream_t stream, int light_max = 0, int4* light_tiles = nullptr,
                         int* n_light = nullptr);
// Routing lists and the gather of x rows in one kernel for small batches
// (R <= kSmallRouteMax slots, E <= 1024): one CTA per slot.
constexpr int kSmallRouteMax = 512;
cudaError_t launch_route_gather_small(const int32_t* ids, int R, int E, int e_begin, int E_total, int nt, int topk,
                                      int* counts, int* offsets, int* perm, int* inv, int4* tiles, int* n_tiles,
                                      int* status, const __nv_bfloat16* x, int K, int interleave, __nv_bfloat16* xp,
                                      float* csum, int* flags, int n_flags, cudaStream_t stream);
// Router: ids/weights [T, k] from fp32 logits [T, E] (+ bias [E] or null);
// 1 <= k <= min(E, 32), E <= 1024.
cudaError_t launch_route_topk(const float* logits, const float* bias, int T, int E, int k, int32_t* ids,
                              float* weights, cudaStream_t stream);
// Xp[inv[t * topk + j], :] = x[t, :] (in K order `interleave`) for every slot
// of every token routed to a local expert (inv >= 0), one warp per token.
// With csum (2-bit interleaved order only, group 128): also the offset-code
// corrections of those rows, csum[g * R + i] = sum over group g of w(k) x.
// Both gathers also zero flags[0, n_flags) (the w13 GEMM's per-unit flags).
cudaError_t launch_gather(const __nv_bfloat16* x, const int* inv, int T, int topk, int K, int interleave,
                          __nv_bfloat16* xp, float* csum, int R, int* status, int* flags, int n_flags,
                          cudaStream_t stream);
// dst[i, :] = src[i, :] in the A operand's interleaved K order: mode 1 (2-bit)
// (0, 8, 1, 9, ..., 7, 15) in every 16-element block, mode 2 (4-bit)
// (0, 4, 1, 5, 2, 6, 3, 7) in every 8-element block.
cudaError_t launch_interleave_rows(const __nv_bfloat16* src, int64_t rows, int64_t cols, int mode,
                                   __nv_bfloat16* dst, cudaStream_t stream);
// out bf16 [T, K], or with f32_out the unrounded fp32 sums (partial output)
cudaError_t launch_combine(const __nv_bfloat16* y, const float* weights, const int* inv, int T, int topk, int K,
                           void* out, bool f32_out, int R, int* status, cudaStream_t stream);
// Split-K epilogues (partial sums [ksplit][mt][R][256] fp32, rows < offsets_end):
//   h[r, n] = bf16(swiglu(sum_s gate, sum_s up)) (column n at its position in K order `interleave`, 0-2),
//   and with csum the offset-code corrections of h for w2 (group 128), csum[g * R + r]
cudaError_t launch_finalize_w13(const float* partial, int ksplit, int R, const int* offsets_end, int N, float limit,
                                int interleave, __nv_bfloat16* h, float* csum, cudaStream_t stream);
//   y[r, m] = bf16(sum_s partial)
cudaError_t launch_finalize_w2(const float* partial, int ksplit, int R, const int* offsets_end, int K,
                               __nv_bfloat16* y, cudaStream_t stream);
//   out[t, m] = bf16( sum_j w[t, j] * bf16(sum_s partial[s][m/256][inv[t, j]][m%256]) )
cudaError_t launch_combine_partials(const float* partial, int ksplit, int R, const float* weights, const int* inv,
                                    int T, int topk, int K, void* out, bool f32_out, int* status, cudaStream_t stream);
// Quantiser (quant.cu): packed [rows, K/p], scales fp16 [rows, K/g], metrics
// fp64 [rows, 4] (or null) from fp32 w [rows, K] and importance [K] (or null).
cudaError_t launch_quantize(const float* w, int64_t rows, int K, const float* importance, int bits, int g, int search,
                            int32_t* packed, uint16_t* scales, double* metrics, cudaStream_t stream);
cudaError_t launch_pack(const int8_t* codes, int64_t rows, int64_t K, int bits, int32_t* packed,
                        cudaStream_t stream);
// One bounded mbarrier wait that nothing completes (device failure-detection check).
cudaError_t launch_wait_timeout_check(int* status, uint64_t limit_ns, cudaStream_t stream);

}  // namespace wna16

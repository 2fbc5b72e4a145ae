// Routing/permute, gather, weighted combine and pack kernels of the WNA16
// routed-expert MoE forward ("Incubate DeepSeek V4 WNA16 runtime on SM86",
// section "What this branch adds", item 3: the indexed MoE; page
// "hampsonw/DeepSeek-V4-Flash-0731-WNA16", section "How it was created",
// step 4: packing signed codes into INT32 words).
#include <cuda_bf16.h>

#include "gemm.h"
#include "ptx.cuh"

namespace wna16 {

namespace {

constexpr int kRouteThreads = 1024;
constexpr int kRouteWarps = kRouteThreads / 32;

// Block-wide exclusive scan of two values with warp-level inclusive scans
// (shuffles) and one pass over the warp totals (blocks of up to 32 warps).
__device__ __forceinline__ void block_exclusive_scan2(int a, int b, int& ea, int& eb, int& total_a, int& total_b,
                                                      int* scratch /* 64 ints */) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int ia = a, ib = b;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int ta = __shfl_up_sync(0xffffffffu, ia, d);
        const int tb = __shfl_up_sync(0xffffffffu, ib, d);
        if (lane >= d) {
            ia += ta;
            ib += tb;
        }
    }
    if (lane == 31) {
        scratch[warp] = ia;
        scratch[32 + warp] = ib;
    }
    __syncthreads();
    if (warp == 0) {
        const int nw = static_cast<int>(blockDim.x >> 5);
        int va = lane < nw ? scratch[lane] : 0, vb = lane < nw ? scratch[32 + lane] : 0;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int ta = __shfl_up_sync(0xffffffffu, va, d);
            const int tb = __shfl_up_sync(0xffffffffu, vb, d);
            if (lane >= d) {
                va += ta;
                vb += tb;
            }
        }
        scratch[lane] = va;           // inclusive warp prefix
        scratch[32 + lane] = vb;
    }
    __syncthreads();
    const int pa = warp ? scratch[warp - 1] : 0;
    const int pb = warp ? scratch[32 + warp - 1] : 0;
    ea = pa + ia - a;
    eb = pb + ib - b;
    total_a = scratch[31];
    total_b = scratch[63];
}

// Expert of slot id `g` among the local experts [e_begin, e_begin + E): its
// local index, or -1 when it belongs to another range (skipped) or is not a
// valid expert id at all (`bad`).
__device__ __forceinline__ int local_expert(int g, int e_begin, int E, int E_total, bool& bad) {
    if (g < 0 || g >= E_total) {
        bad = true;
        return -1;
    }
    const int e = g - e_begin;
    return (e >= 0 && e < E) ? e : -1;
}

// One CTA.  Slot f = t*topk + j.  Each warp owns a contiguous run of slots;
// pass 1 counts its slots per expert (warp-match groups), a scan over warps and
// over experts turns the counts into start positions, pass 2 places each slot
// (stable: ascending slot within an expert) and records the inverse map.
// Also emits the token-tile list {expert, first row, rows} in expert order.
// Only the experts [e_begin, e_begin + E) of the E_total are routed here
// (all of them on a single device); slots of the other experts get inv = -1.
// Light experts (at most light_max > 0 rows, and at most kLightTileRows: the
// skewed tail of a prefill batch) leave the main tile list for a second one
// with one tile per expert, run by launches of their own; both lists are in
// expert order.
constexpr int kLightTileRows = 8;
__device__ __forceinline__ bool is_light(int c, int light_max) {
    return light_max > 0 && c > 0 && c <= light_max && c <= kLightTileRows;
}
// Exclusive scan of the experts' light tile counts (the whole block calls it;
// `scratch` is free again on return).
__device__ __forceinline__ void light_scan(bool light, int c, int& loff, int& ltotal, int* scratch) {
    __syncthreads();
    int z0, z1;
    block_exclusive_scan2(light ? (c + kLightTileRows - 1) / kLightTileRows : 0, 0, loff, z0, ltotal, z1, scratch);
    __syncthreads();
}
__device__ __forceinline__ void write_light_tiles(int e, int c, int off, int4* dst) {
    for (int j = 0; j * kLightTileRows < c; ++j)
        dst[j] = make_int4(e, off + j * kLightTileRows, min(kLightTileRows, c - j * kLightTileRows), 0);
}

__global__ void __launch_bounds__(kRouteThreads, 1)
    route_kernel(const int32_t* __restrict__ ids, int R, int E, int e_begin, int E_total, int nt,
                 int* __restrict__ counts, int* __restrict__ offsets, int* __restrict__ perm, int* __restrict__ inv,
                 int4* __restrict__ tiles, int* __restrict__ n_tiles, int* __restrict__ status, int light_max,
                 int4* __restrict__ light_tiles, int* __restrict__ n_light) {
    extern __shared__ int sm[];
    int* cnt = sm;                          // [kRouteWarps][E]
    int* scratch = sm + kRouteWarps * E;    // 64 ints
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    pdl_trigger();
    if (tid == 0) *status = kStatusOk;

    // W warps hold slots (32 each, more once R > 32 * kRouteWarps); the
    // per-expert passes below walk only their W count rows
    const int W = max(1, min(kRouteWarps, (R + 31) / 32));
    const int per_warp = (((R + W - 1) / W) + 31) & ~31;
    const int f0 = warp * per_warp;
    const int f1 = min(R, f0 + per_warp);
    int* my = cnt + warp * E;
    if (warp < W)
        for (int e = lane; e < E; e += 32) my[e] = 0;
    __syncwarp();

    bool bad = false;
    for (int base = f0; base < f1; base += 32) {
        const int f = base + lane;
        int e = -1;
        if (f < f1) e = local_expert(ids[f], e_begin, E, E_total, bad);
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        if (e >= 0 && lane == __ffs(peers) - 1) my[e] += __popc(peers);
        __syncwarp();
    }
    __syncthreads();
    if (bad) atomicExch(status, kStatusBadRouting);

    int c = 0;
    if (tid < E) {
        for (int w = 0; w < W; ++w) {
            const int v = cnt[w * E + tid];
            cnt[w * E + tid] = c;
            c += v;
        }
    }
    const bool light = tid < E && is_light(c, light_max);
    const int ntl = tid < E && !light ? (c + nt - 1) / nt : 0;
    int off, toff, total, ttotal;
    block_exclusive_scan2(c, ntl, off, toff, total, ttotal, scratch);
    int loff = 0, ltotal = 0;
    if (light_max > 0) light_scan(light, c, loff, ltotal, scratch);
    if (tid < E) {
        counts[tid] = c;
        offsets[tid] = off;
        for (int j = 0; j < ntl; ++j) tiles[toff + j] = make_int4(tid, off + j * nt, min(nt, c - j * nt), 0);
        if (light) write_light_tiles(tid, c, off, light_tiles + loff);
        for (int w = 0; w < W; ++w) cnt[w * E + tid] += off;
    }
    if (tid == 0) {
        offsets[E] = total;
        *n_tiles = ttotal;
        if (light_max > 0) *n_light = ltotal;
    }
    __syncthreads();

    const unsigned lt = (1u << lane) - 1u;
    for (int base = f0; base < f1; base += 32) {
        const int f = base + lane;
        int e = -1;
        bool ignored = false;
        if (f < f1) e = local_expert(ids[f], e_begin, E, E_total, ignored);
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        const int pos = e >= 0 ? my[e] + __popc(peers & lt) : -1;
        __syncwarp();
        if (e >= 0 && lane == __ffs(peers) - 1) my[e] += __popc(peers);
        __syncwarp();
        if (f < f1) {
            if (e >= 0 && in_bounds(pos >= 0 && pos < R, status)) perm[pos] = f;
            inv[f] = pos;
        }
    }
}

// ---- routing lists for large batches: a stable counting sort in three
// kernels over chunks of kChunk slots (the single-CTA route_kernel walks every
// slot on one SM, which dominates at tens of thousands of slots).
//   count: per chunk, the slots of each local expert  -> ccount[chunk][E]
//   scan:  per expert, the chunks' starting positions (chunk order), the
//          counts, offsets and the token-tile list        (one CTA)
//   place: per chunk, each slot's position, stable in slot order
constexpr int kChunk = 1024;
constexpr int kChunkThreads = 256;
constexpr int kChunkWarps = kChunkThreads / 32;

__global__ void __launch_bounds__(kChunkThreads)
    route_count_kernel(const int32_t* __restrict__ ids, int R, int E, int e_begin, int E_total,
                       int* __restrict__ ccount, int* __restrict__ cbad) {
    extern __shared__ int hist[];   // [E]
    for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
    __syncthreads();
    const int f0 = blockIdx.x * kChunk;
    const int f1 = min(R, f0 + kChunk);
    bool bad = false;
    for (int f = f0 + threadIdx.x; f < f1; f += blockDim.x) {
        const int e = local_expert(ids[f], e_begin, E, E_total, bad);
        if (e >= 0) atomicAdd(&hist[e], 1);
    }
    const int any_bad = __syncthreads_or(bad ? 1 : 0);
    for (int e = threadIdx.x; e < E; e += blockDim.x) ccount[static_cast<int64_t>(blockIdx.x) * E + e] = hist[e];
    if (threadIdx.x == 0) cbad[blockIdx.x] = any_bad;
}

__global__ void __launch_bounds__(kRouteThreads, 1)
    route_scan_kernel(int nchunks, int E, int nt, int* __restrict__ ccount, const int* __restrict__ cbad,
                      int* __restrict__ counts, int* __restrict__ offsets, int4* __restrict__ tiles,
                      int* __restrict__ n_tiles, int* __restrict__ status, int light_max,
                      int4* __restrict__ light_tiles, int* __restrict__ n_light) {
    __shared__ int scratch[64];
    const int tid = threadIdx.x;
    if (tid == 0) {
        int bad = 0;
        for (int c = 0; c < nchunks; ++c) bad |= cbad[c];
        *status = bad ? kStatusBadRouting : kStatusOk;
    }
    // per expert: the total over the chunks, then each chunk's start (the
    // expert's offset plus the chunks before it, in chunk order); the counts
    // are read in batches of kScanBatch independent loads
    constexpr int kScanBatch = 16;
    int c_tot = 0;
    if (tid < E) {
        for (int c0 = 0; c0 < nchunks; c0 += kScanBatch) {
            int v[kScanBatch];
#pragma unroll
            for (int i = 0; i < kScanBatch; ++i)
                v[i] = c0 + i < nchunks ? ccount[static_cast<int64_t>(c0 + i) * E + tid] : 0;
#pragma unroll
            for (int i = 0; i < kScanBatch; ++i) c_tot += v[i];
        }
    }
    const bool light = tid < E && is_light(c_tot, light_max);
    const int ntl = tid < E && !light ? (c_tot + nt - 1) / nt : 0;
    int off, toff, total, ttotal;
    block_exclusive_scan2(c_tot, ntl, off, toff, total, ttotal, scratch);
    int loff = 0, ltotal = 0;
    if (light_max > 0) light_scan(light, c_tot, loff, ltotal, scratch);
    if (tid < E) {
        counts[tid] = c_tot;
        offsets[tid] = off;
        for (int j = 0; j < ntl; ++j) tiles[toff + j] = make_int4(tid, off + j * nt, min(nt, c_tot - j * nt), 0);
        if (light) write_light_tiles(tid, c_tot, off, light_tiles + loff);
        int run = off;
        for (int c0 = 0; c0 < nchunks; c0 += kScanBatch) {
            int v[kScanBatch];
#pragma unroll
            for (int i = 0; i < kScanBatch; ++i)
                v[i] = c0 + i < nchunks ? ccount[static_cast<int64_t>(c0 + i) * E + tid] : 0;
#pragma unroll
            for (int i = 0; i < kScanBatch; ++i) {
                if (c0 + i < nchunks) ccount[static_cast<int64_t>(c0 + i) * E + tid] = run;
                run += v[i];
            }
        }
    }
    if (tid == 0) {
        offsets[E] = total;
        *n_tiles = ttotal;
        if (light_max > 0) *n_light = ltotal;
    }
}

__global__ void __launch_bounds__(kChunkThreads)
    route_place_kernel(const int32_t* __restrict__ ids, int R, int E, int e_begin, int E_total,
                       const int* __restrict__ cstart, int* __restrict__ perm, int* __restrict__ inv,
                       int* __restrict__ status) {
    extern __shared__ int wcnt[];   // [kChunkWarps][E]
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int per_warp = kChunk / kChunkWarps;
    const int f0 = blockIdx.x * kChunk + warp * per_warp;
    const int f1 = min(R, f0 + per_warp);
    int* my = wcnt + warp * E;
    for (int e = lane; e < E; e += 32) my[e] = 0;
    __syncwarp();
    for (int base = f0; base < f1; base += 32) {
        const int f = base + lane;
        bool ignored = false;
        const int e = f < f1 ? local_expert(ids[f], e_begin, E, E_total, ignored) : -1;
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        if (e >= 0 && lane == __ffs(peers) - 1) my[e] += __popc(peers);
        __syncwarp();
    }
    __syncthreads();
    // per expert: the warps' starts (warp order) after the chunk's start
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int c = cstart[static_cast<int64_t>(blockIdx.x) * E + e];
        for (int w = 0; w < kChunkWarps; ++w) {
            const int v = wcnt[w * E + e];
            wcnt[w * E + e] = c;
            c += v;
        }
    }
    __syncthreads();
    const unsigned lt = (1u << lane) - 1u;
    for (int base = f0; base < f1; base += 32) {
        const int f = base + lane;
        bool ignored = false;
        const int e = f < f1 ? local_expert(ids[f], e_begin, E, E_total, ignored) : -1;
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        const int pos = e >= 0 ? my[e] + __popc(peers & lt) : -1;
        __syncwarp();
        if (e >= 0 && lane == __ffs(peers) - 1) my[e] += __popc(peers);
        __syncwarp();
        if (f < f1) {
            if (e >= 0 && in_bounds(pos >= 0 && pos < R, status)) perm[pos] = f;
            inv[f] = pos;
        }
    }
}

// Router: one warp per token.  Lane l holds the scores z = logit + bias of
// experts l, l + 32, ... (PL per lane).  k rounds of a warp-wide argmax (the
// larger score wins, equal scores go to the lower expert index) pick the
// experts in descending order; the weights are the softmax renormalised over
// the chosen k, exp(z_j - z_max) / sum_i exp(z_i - z_max), which equals the
// full softmax divided by its sum over the chosen experts.  Lane j keeps the
// j-th choice; the sum runs in choice order.
template <int PL>
__global__ void __launch_bounds__(256)
    route_topk_kernel(const float* __restrict__ logits, const float* __restrict__ bias, int T, int E, int k,
                      int32_t* __restrict__ ids, float* __restrict__ weights) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= T) return;   // whole warps leave together
    const float* row = logits + static_cast<int64_t>(t) * E;
    float z[PL];
#pragma unroll
    for (int i = 0; i < PL; ++i) {
        const int e = i * 32 + lane;
        z[i] = e < E ? __fadd_rn(__ldg(row + e), bias ? __ldg(bias + e) : 0.0f) : 0.0f;
    }
    uint32_t taken = 0;
    float my_z = 0.0f;
    int my_id = 0;
    for (int j = 0; j < k; ++j) {
        float bv = 0.0f;
        int bi = -1;
#pragma unroll
        for (int i = 0; i < PL; ++i) {
            const int e = i * 32 + lane;
            if (e < E && !((taken >> i) & 1u) && (bi < 0 || z[i] > bv)) {
                bv = z[i];
                bi = e;
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
            if (oi >= 0 && (bi < 0 || ov > bv || (ov == bv && oi < bi))) {
                bv = ov;
                bi = oi;
            }
        }
        // k <= E, so a candidate always exists; the owner marks it taken
        if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
        if (lane == j) {
            my_z = bv;
            my_id = bi;
        }
    }
    const float zmax = __shfl_sync(0xffffffffu, my_z, 0);
    const float ex = lane < k ? expf(my_z - zmax) : 0.0f;
    float sum = 0.0f;
    for (int j = 0; j < k; ++j) sum += __shfl_sync(0xffffffffu, ex, j);
    if (lane < k) {
        ids[static_cast<int64_t>(t) * k + lane] = my_id;
        weights[static_cast<int64_t>(t) * k + lane] = ex / sum;
    }
}

// 16 BF16 (elements 0..15 of a block, as two 8-element vectors) -> the
// interleaved order (0, 8, 1, 9, ..., 7, 15) of the 2-bit A operand.
__device__ __forceinline__ void interleave_block(const uint4& lo, const uint4& hi, uint4& a, uint4& b) {
    a.x = __byte_perm(lo.x, hi.x, 0x5410);  // lo0 hi0
    a.y = __byte_perm(lo.x, hi.x, 0x7632);  // lo1 hi1
    a.z = __byte_perm(lo.y, hi.y, 0x5410);
    a.w = __byte_perm(lo.y, hi.y, 0x7632);
    b.x = __byte_perm(lo.z, hi.z, 0x5410);
    b.y = __byte_perm(lo.z, hi.z, 0x7632);
    b.z = __byte_perm(lo.w, hi.w, 0x5410);
    b.w = __byte_perm(lo.w, hi.w, 0x7632);
}
// 8 BF16 (one 8-element vector) -> the interleaved order (0, 4, 1, 5, 2, 6, 3, 7)
// of the 4-bit A operand.
__device__ __forceinline__ uint4 interleave8(const uint4& v) {
    uint4 a;
    a.x = __byte_perm(v.x, v.z, 0x5410);  // 0 4
    a.y = __byte_perm(v.x, v.z, 0x7632);  // 1 5
    a.z = __byte_perm(v.y, v.w, 0x5410);  // 2 6
    a.w = __byte_perm(v.y, v.w, 0x7632);  // 3 7
    return a;
}

// Weight of element k in the offset-code correction of the grouped GEMM's
// group-accumulate mode: off(k) + 2 for the magic offset off = 128, 32, 8 of
// the code field's mantissa position, i.e. 130, 34, 10 for (k mod 8) mod 3 =
// 0, 1, 2.
__device__ __forceinline__ float offset_weight(int k) {
    const int c = (k & 7) % 3;
    return c == 0 ? 130.0f : (c == 1 ? 34.0f : 10.0f);
}

// sum_e offset_weight(e) (lo_e + hi_e) over a 16-element block held as its
// elements 0..7 (lo) and 8..15 (hi), in the natural order.
__device__ __forceinline__ float offset_sum16(const uint4& lo, const uint4& hi) {
    const uint32_t a[4] = {lo.x, lo.y, lo.z, lo.w};
    const uint32_t b[4] = {hi.x, hi.y, hi.z, hi.w};
    float s = 0.0f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float2 fa = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&a[j]));
        const float2 fb = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&b[j]));
        s = __fmaf_rn(offset_weight(2 * j), fa.x + fb.x, s);
        s = __fmaf_rn(offset_weight(2 * j + 1), fa.y + fb.y, s);
    }
    return s;
}

// Xp[i, :] = x[perm[i] / topk, :] for the valid rows i < offsets[E], in the
// K order of the A operand (interleave: 0 natural, 1 the 16-k order of 2-bit
// weights, 2 the 8-k order of 4-bit ones); with csum (order 1 only) also
// csum[g * R + i] = sum over the 128-element group g of offset_weight(k) x[k].
// Copies token row t of x into permuted row i of xp (one CTA; see gather_kernel).
// `tid` of `nthr` threads (whole warps) copy the row.
__device__ __forceinline__ void gather_row(const uint4* __restrict__ x, int64_t t, int i, int R, int vec_per_row,
                                           int interleave, uint4* __restrict__ xp, float* __restrict__ csum, int tid,
                                           int nthr) {
    const uint4* src = x + t * vec_per_row;
    uint4* dst = xp + static_cast<int64_t>(i) * vec_per_row;
    if (interleave != 1) {
        // four loads in flight per thread before the stores
        for (int v0 = tid; v0 < vec_per_row; v0 += 4 * nthr) {
            uint4 a[4];
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (v0 + j * nthr < vec_per_row) a[j] = __ldg(src + v0 + j * nthr);
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (v0 + j * nthr < vec_per_row) dst[v0 + j * nthr] = interleave == 2 ? interleave8(a[j]) : a[j];
        }
    } else {
        // every warp runs the same number of rounds (the shuffles need all
        // lanes); 8 consecutive threads hold one group's 16 vectors; two
        // rounds' loads are in flight before their stores
        for (int base = 0; base < vec_per_row; base += 4 * nthr) {
            uint4 lo[2], hi[2];
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int v = base + r * 2 * nthr + 2 * tid;
                if (v < vec_per_row) {
                    lo[r] = __ldg(src + v);
                    hi[r] = __ldg(src + v + 1);
                }
            }
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int v = base + r * 2 * nthr + 2 * tid;
                float part = 0.0f;
                if (v < vec_per_row) {
                    uint4 a, b;
                    interleave_block(lo[r], hi[r], a, b);
                    dst[v] = a;
                    dst[v + 1] = b;
                    if (csum) part = offset_sum16(lo[r], hi[r]);
                }
                if (csum) {
                    part += __shfl_xor_sync(0xffffffffu, part, 1);
                    part += __shfl_xor_sync(0xffffffffu, part, 2);
                    part += __shfl_xor_sync(0xffffffffu, part, 4);
                    if ((tid & 7) == 0 && v < vec_per_row) csum[static_cast<int64_t>(v >> 4) * R + i] = part;
                }
            }
        }
    }
}

// Zeroes the w13 GEMM's per-unit flags (paired K splits) before it runs.
__device__ __forceinline__ void zero_flags(int* __restrict__ flags, int n_flags) {
    for (int j = blockIdx.x * blockDim.x + threadIdx.x; j < n_flags; j += gridDim.x * blockDim.x) flags[j] = 0;
}

// One warp per token, kGatherRows tokens per CTA: the warp reads the token's
// x row once and writes it (in the A operand's K order) to the permuted row
// of each of its slots routed to a local expert (inv >= 0), with csum (order 1
// only) also those rows' offset-code corrections.  Reading each x row once,
// rather than once per slot, keeps the R = T * topk row writes from evicting
// x from L2 between its reads.
constexpr int kGatherRows = 8;

__global__ void __launch_bounds__(32 * kGatherRows)
    scatter_kernel(const uint4* __restrict__ x, const int* __restrict__ inv, int T, int topk, int vec_per_row,
                   int interleave, uint4* __restrict__ xp, float* __restrict__ csum, int R, int* __restrict__ status,
                   int* __restrict__ flags, int n_flags) {
    pdl_wait();
    pdl_trigger();
    zero_flags(flags, n_flags);
    const int t = blockIdx.x * kGatherRows + (threadIdx.x >> 5);
    if (t >= T) return;   // whole warps
    const int lane = threadIdx.x & 31;
    int mine = -1;        // lane j < topk: the permuted row of slot j (-1: not local)
    if (lane < topk) {
        const int r = inv[static_cast<int64_t>(t) * topk + lane];
        mine = r >= 0 && in_bounds(r < R, status) ? r : -1;
    }
    const uint4* src = x + static_cast<int64_t>(t) * vec_per_row;
    if (interleave != 1) {
        // vec_per_row is a multiple of 32, so every lane runs the same rounds
        for (int v0 = lane; v0 < vec_per_row; v0 += 4 * 32) {
            uint4 a[4];
#pragma unroll
            for (int c = 0; c < 4; ++c)
                if (v0 + c * 32 < vec_per_row) {
                    a[c] = __ldg(src + v0 + c * 32);
                    if (interleave == 2) a[c] = interleave8(a[c]);
                }
            for (int j = 0; j < topk; ++j) {
                const int i = __shfl_sync(0xffffffffu, mine, j);
                if (i < 0) continue;
                uint4* dst = xp + static_cast<int64_t>(i) * vec_per_row;
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    if (v0 + c * 32 < vec_per_row) dst[v0 + c * 32] = a[c];
            }
        }
    } else {
        // two vectors (one 16-element block) per lane and round; 8 consecutive
        // lanes hold one 128-element group
        for (int base = 0; base < vec_per_row; base += 2 * 32) {
            const int v = base + 2 * lane;
            uint4 a = make_uint4(0, 0, 0, 0), b = a;
            float part = 0.0f;
            if (v < vec_per_row) {
                const uint4 lo = __ldg(src + v), hi = __ldg(src + v + 1);
                interleave_block(lo, hi, a, b);
                if (csum) part = offset_sum16(lo, hi);
            }
            if (csum) {
                part += __shfl_xor_sync(0xffffffffu, part, 1);
                part += __shfl_xor_sync(0xffffffffu, part, 2);
                part += __shfl_xor_sync(0xffffffffu, part, 4);
            }
            for (int j = 0; j < topk; ++j) {
                const int i = __shfl_sync(0xffffffffu, mine, j);
                if (i < 0 || v >= vec_per_row) continue;
                uint4* dst = xp + static_cast<int64_t>(i) * vec_per_row;
                dst[v] = a;
                dst[v + 1] = b;
                if (csum && (lane & 7) == 0) csum[static_cast<int64_t>(v >> 4) * R + i] = part;
            }
        }
    }
}

// Routing lists and the gather in one kernel, for small batches (decode):
// one CTA per slot f.  Every CTA reads all R ids; slot f's position in the
// stable (expert, slot) order is the number of valid slots that sort before
// it, so no scan across CTAs is needed.  CTA f records perm / inv for its slot
// and copies its token's row of x to that position; CTA 0 also writes the
// per-expert counts and offsets, the token-tile list and the status word.
constexpr int kSmallRouteThreads = 256;

__global__ void __launch_bounds__(kSmallRouteThreads)
    route_gather_small_kernel(const int32_t* __restrict__ ids, int R, int E, int e_begin, int E_total, int nt,
                              int topk, int* __restrict__ counts, int* __restrict__ offsets, int* __restrict__ perm,
                              int* __restrict__ inv, int4* __restrict__ tiles, int* __restrict__ n_tiles,
                              int* __restrict__ status, const uint4* __restrict__ x, int vec_per_row, int interleave,
                              uint4* __restrict__ xp, float* __restrict__ csum, int* __restrict__ flags, int n_flags) {
    extern __shared__ int sm[];
    zero_flags(flags, n_flags);
    int* le = sm;                      // [R] local expert of each slot (-1: skipped or bad)
    int* cnt = sm + R;                 // [E] (CTA 0)
    __shared__ int red[kSmallRouteThreads / 32];
    __shared__ int scratch[64];
    pdl_trigger();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int f = blockIdx.x;
    bool bad = false;
    for (int q = tid; q < R; q += blockDim.x) le[q] = local_expert(ids[q], e_begin, E, E_total, bad);
    const int any_bad = __syncthreads_or(bad ? 1 : 0);
    const int e = le[f];
    // rank of slot f among the valid slots in (expert, slot) order
    int c = 0;
    if (e >= 0)
        for (int q = tid; q < R; q += blockDim.x) {
            const int eq = le[q];
            c += (eq >= 0 && (eq < e || (eq == e && q < f))) ? 1 : 0;
        }
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) c += __shfl_xor_sync(0xffffffffu, c, d);
    if (lane == 0) red[warp] = c;
    __syncthreads();
    int rank = 0;
    for (int w = 0; w < kSmallRouteThreads / 32; ++w) rank += red[w];
    const bool rank_ok = e < 0 || in_bounds(rank < R, status);
    if (tid == 0) {
        inv[f] = e >= 0 && rank_ok ? rank : -1;
        if (e >= 0 && rank_ok) perm[rank] = f;
    }
    if (f == 0) {
        // counts, offsets, tiles, status
        for (int q = tid; q < E; q += blockDim.x) cnt[q] = 0;
        __syncthreads();
        for (int q = tid; q < R; q += blockDim.x)
            if (le[q] >= 0) atomicAdd(&cnt[le[q]], 1);
        __syncthreads();
        // E <= 1024 experts over 256 threads: each thread sums a run of 4 experts
        int run[4], rtot = 0, rtiles = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int q = tid * 4 + j;
            run[j] = q < E ? cnt[q] : 0;
            rtot += run[j];
            rtiles += (run[j] + nt - 1) / nt;
        }
        int off, toff, total, ttotal;
        block_exclusive_scan2(rtot, rtiles, off, toff, total, ttotal, scratch);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int q = tid * 4 + j;
            if (q < E) {
                counts[q] = run[j];
                offsets[q] = off;
                const int ntl = (run[j] + nt - 1) / nt;
                for (int k = 0; k < ntl; ++k) tiles[toff + k] = make_int4(q, off + k * nt, min(nt, run[j] - k * nt), 0);
                off += run[j];
                toff += ntl;
            }
        }
        if (tid == 0) {
            offsets[E] = total;
            *n_tiles = ttotal;
            *status = any_bad ? kStatusBadRouting : kStatusOk;
        }
    }
    if (e >= 0 && rank_ok && xp) gather_row(x, f / topk, rank, R, vec_per_row, interleave, xp, csum, threadIdx.x, blockDim.x);
}

// Rows of BF16 into the A operand's K order (mode 1: 16-element blocks, 2:
// 8-element vectors); one thread per 16 elements.
__global__ void interleave_rows_kernel(const uint4* __restrict__ src, int64_t blocks, int mode,
                                       uint4* __restrict__ dst) {
    const int64_t b = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (b >= blocks) return;
    uint4 a, c;
    if (mode == 2) {
        a = interleave8(src[2 * b]);
        c = interleave8(src[2 * b + 1]);
    } else {
        interleave_block(src[2 * b], src[2 * b + 1], a, c);
    }
    dst[2 * b] = a;
    dst[2 * b + 1] = c;
}

// out[t, m] = bf16( sum_j w[t, j] * y[inv[t*topk + j], m] ), fp32, j ascending;
// a slot whose inverse index is -1 (bad expert id, or an expert of another
// range) adds nothing.  With F32OUT the fp32 sum is stored unrounded (the
// partial output of an expert range).
template <bool F32OUT>
__global__ void combine_kernel(const uint4* __restrict__ y, const float* __restrict__ w, const int* __restrict__ inv,
                               int topk, int vec_per_row, void* __restrict__ out, int R, int* __restrict__ status) {
    pdl_wait();
    const int t = blockIdx.x;
    const int v = blockIdx.y * blockDim.x + threadIdx.x;
    if (v >= vec_per_row) return;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    // up to 8 slots' rows in flight before the adds, which stay in slot order
    for (int j0 = 0; j0 < topk; j0 += 8) {
        uint4 q[8];
        float wj[8];
        bool ok[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const int j = j0 + c;
            ok[c] = false;
            if (j < topk) {
                const int r = inv[t * topk + j];
                ok[c] = r >= 0 && in_bounds(r < R, status);
                if (ok[c]) {
                    wj[c] = w[t * topk + j];
                    q[c] = __ldg(y + static_cast<int64_t>(r) * vec_per_row + v);
                }
            }
        }
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            if (!ok[c]) continue;
            const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&q[c]);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 f = __bfloat1622float2(h[i]);
                acc[2 * i] = __fmaf_rn(wj[c], f.x, acc[2 * i]);
                acc[2 * i + 1] = __fmaf_rn(wj[c], f.y, acc[2 * i + 1]);
            }
        }
    }
    if constexpr (F32OUT) {
        float4* o = reinterpret_cast<float4*>(out) + (static_cast<int64_t>(t) * vec_per_row + v) * 2;
        o[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        o[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    } else {
        uint4 o;
        __nv_bfloat162* ob = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
        for (int i = 0; i < 4; ++i) ob[i] = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
        reinterpret_cast<uint4*>(out)[static_cast<int64_t>(t) * vec_per_row + v] = o;
    }
}

__device__ __forceinline__ float swiglu_clamped(float g, float u, float L) {
    g = fminf(g, L);
    u = fminf(fmaxf(u, -L), L);
    // fast exp / divide: their fp32 errors (a few ulp) are far below the BF16
    // rounding of h; for very negative g the divisor overflows and the
    // quotient is 0, as silu's is
    return __fdividef(g, 1.0f + __expf(-g)) * u;
}

// Split-K epilogue of w13: blockIdx.x = permuted row (valid rows only), each
// thread 4 consecutive n; all KS partial loads of a thread are issued before
// the first is used, and the splits are added in ascending order.
// With csum, each warp (128 consecutive n = one group of w2's reduction) also
// writes csum[g * R + r] = sum_n offset_weight(n) bf16(h[r, n]) for w2's
// offset codes.
template <int KS>
__global__ void finalize_w13_kernel(const float* __restrict__ partial, int R, const int* __restrict__ offsets_end,
                                    int N, float L, int interleave, __nv_bfloat16* __restrict__ h,
                                    float* __restrict__ csum) {
    pdl_wait();
    pdl_trigger();
    const int r = blockIdx.x;
    if (r >= *offsets_end) return;
    const int n0 = (blockIdx.y * blockDim.x + threadIdx.x) * 4;
    if (n0 >= N) return;
    const int mtc = N / 128;
    const float* q = partial + (static_cast<int64_t>(n0 >> 7) * R + r) * 256 + (n0 & 127);
    const int64_t split_stride = static_cast<int64_t>(mtc) * R * 256;
    float4 g[KS], u[KS];
#pragma unroll
    for (int s = 0; s < KS; ++s) {
        g[s] = __ldg(reinterpret_cast<const float4*>(q + s * split_stride));
        u[s] = __ldg(reinterpret_cast<const float4*>(q + s * split_stride + 128));
    }
    float gs[4] = {0.f, 0.f, 0.f, 0.f}, us[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int s = 0; s < KS; ++s) {
        gs[0] += g[s].x; gs[1] += g[s].y; gs[2] += g[s].z; gs[3] += g[s].w;
        us[0] += u[s].x; us[1] += u[s].y; us[2] += u[s].z; us[3] += u[s].w;
    }
    __nv_bfloat16* hr = h + static_cast<int64_t>(r) * N;
    float part = 0.0f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const int n = n0 + e;
        int col = n;
        if (interleave == 1) {
            const int b = n & 15;
            col = (n & ~15) | (b < 8 ? 2 * b : 2 * (b - 8) + 1);
        } else if (interleave == 2) {
            const int b = n & 7;
            col = (n & ~7) | (b < 4 ? 2 * b : 2 * (b - 4) + 1);
        }
        const __nv_bfloat16 hv = __float2bfloat16_rn(swiglu_clamped(gs[e], us[e], L));
        hr[col] = hv;
        part = __fmaf_rn(offset_weight(n), __bfloat162float(hv), part);
    }
    if (csum) {   // N % 128 == 0: whole warps return above, so all 32 lanes are here
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) part += __shfl_xor_sync(0xffffffffu, part, d);
        if ((threadIdx.x & 31) == 0) csum[static_cast<int64_t>(n0 >> 7) * R + r] = part;
    }
}

// Split-K epilogue of w2 (for the stage entry point): y = bf16(sum of splits).
__global__ void finalize_w2_kernel(const float* __restrict__ partial, int ksplit, int R, const int* __restrict__ offsets_end,
                                   int K, __nv_bfloat16* __restrict__ y) {
    pdl_wait();
    const int r = blockIdx.x;
    if (r >= *offsets_end) return;
    const int mtc = K / 256;
    for (int m = threadIdx.x; m < K; m += blockDim.x) {
        float a = 0.f;
        for (int s = 0; s < ksplit; ++s) a += partial[((static_cast<int64_t>(s) * mtc + (m >> 8)) * R + r) * 256 + (m & 255)];
        y[static_cast<int64_t>(r) * K + m] = __float2bfloat16_rn(a);
    }
}

// Combine straight from the w2 split partial sums: y is rounded to BF16 exactly
// where the unsplit path stores it, then weighted and summed (j ascending).
// The lanes of a warp fetch up to 32 (slot row, weight) pairs at once and
// pass them round by shuffles; the KS partial loads of a slot are issued
// together.
template <int KS, bool F32OUT>
__global__ void combine_partials_kernel(const float* __restrict__ partial, int R, const float* __restrict__ w,
                                        const int* __restrict__ inv, int topk, int K, void* __restrict__ out,
                                        int* __restrict__ status) {
    pdl_wait();
    const int t = blockIdx.x;
    const int lane = threadIdx.x & 31;
    const int m0 = (blockIdx.y * blockDim.x + threadIdx.x) * 4;
    const bool active = m0 < K;   // warp-uniform: K / 4 is a multiple of 32
    const int mtc = K / 256;
    const int64_t split_stride = static_cast<int64_t>(mtc) * R * 256;
    const float* col = partial + static_cast<int64_t>(m0 >> 8) * R * 256 + (m0 & 255);
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int j0 = 0; j0 < topk; j0 += 32) {
        const int jn = min(32, topk - j0);
        int rl = -1;
        float wl = 0.f;
        if (lane < jn) {
            rl = inv[t * topk + j0 + lane];
            wl = w[t * topk + j0 + lane];
        }
        // JB slots per round: their loads are all in flight before the first sum
        constexpr int JB = KS <= 4 ? 4 : 2;
        for (int j = 0; j < jn; j += JB) {
            int r[JB];
            float wj[JB];
#pragma unroll
            for (int b = 0; b < JB; ++b) {
                r[b] = __shfl_sync(0xffffffffu, rl, (j + b) & 31);
                wj[b] = __shfl_sync(0xffffffffu, wl, (j + b) & 31);
                if (j + b >= jn || !active) r[b] = -1;
                if (r[b] >= 0 && !in_bounds(r[b] < R, status)) r[b] = -1;
            }
            float4 q[JB][KS];
#pragma unroll
            for (int b = 0; b < JB; ++b)
#pragma unroll
                for (int s = 0; s < KS; ++s)
                    q[b][s] = r[b] >= 0 ? __ldg(reinterpret_cast<const float4*>(
                                              col + s * split_stride + static_cast<int64_t>(r[b]) * 256))
                                        : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int b = 0; b < JB; ++b) {
                if (r[b] < 0) continue;
                float ysum[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int s = 0; s < KS; ++s) {
                    ysum[0] += q[b][s].x; ysum[1] += q[b][s].y; ysum[2] += q[b][s].z; ysum[3] += q[b][s].w;
                }
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    acc[i] = __fmaf_rn(wj[b], __bfloat162float(__float2bfloat16_rn(ysum[i])), acc[i]);
            }
        }
    }
    if (!active) return;
    if constexpr (F32OUT) {
        *reinterpret_cast<float4*>(reinterpret_cast<float*>(out) + static_cast<int64_t>(t) * K + m0) =
            make_float4(acc[0], acc[1], acc[2], acc[3]);
    } else {
        __nv_bfloat162* o =
            reinterpret_cast<__nv_bfloat162*>(reinterpret_cast<__nv_bfloat16*>(out) + static_cast<int64_t>(t) * K + m0);
        o[0] = __floats2bfloat162_rn(acc[0], acc[1]);
        o[1] = __floats2bfloat162_rn(acc[2], acc[3]);
    }
}

// word i <- codes [i*p, (i+1)*p): field j = (code_j + 2^(b-1)) & (2^b - 1) at bits [b*j, b*j+b).
__global__ void pack_kernel(const int8_t* __restrict__ codes, int64_t n_words, int bits, int32_t* __restrict__ packed) {
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= n_words) return;
    const int p = 32 / bits;
    const int off = 1 << (bits - 1);
    const uint32_t mask = (1u << bits) - 1u;
    const int8_t* c = codes + i * p;
    uint32_t w = 0;
    for (int j = 0; j < p; ++j) w |= (static_cast<uint32_t>(c[j] + off) & mask) << (bits * j);
    packed[i] = static_cast<int32_t>(w);
}

}  // namespace

int route_chunks(int R) { return R > kRouteChunkedMin ? (R + kChunk - 1) / kChunk : 0; }

cudaError_t launch_route(const int32_t* ids, int R, int E, int e_begin, int E_total, int nt, int* counts, int* offsets,
                         int* perm, int* inv, int4* tiles, int* n_tiles, int* status, int* chunk_scratch,
                         cudaStream_t stream, int light_max, int4* light_tiles, int* n_light) {
    const int nchunks = route_chunks(R);
    if (nchunks > 0) {
        int* ccount = chunk_scratch;                                  // [nchunks][E]
        int* cbad = chunk_scratch + static_cast<int64_t>(nchunks) * E; // [nchunks]
        const int hsmem = E * static_cast<int>(sizeof(int));
        const int psmem = kChunkWarps * E * static_cast<int>(sizeof(int));
        cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(route_place_kernel), psmem);
        if (e != cudaSuccess) return e;
        route_count_kernel<<<nchunks, kChunkThreads, hsmem, stream>>>(ids, R, E, e_begin, E_total, ccount, cbad);
        route_scan_kernel<<<1, kRouteThreads, 0, stream>>>(nchunks, E, nt, ccount, cbad, counts, offsets, tiles,
                                                          n_tiles, status, light_max, light_tiles, n_light);
        route_place_kernel<<<nchunks, kChunkThreads, psmem, stream>>>(ids, R, E, e_begin, E_total, ccount, perm, inv,
                                                                      status);
        return cudaGetLastError();
    }
    const int smem = (kRouteWarps * E + 64) * static_cast<int>(sizeof(int));
    cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(route_kernel), smem);
    if (e != cudaSuccess) return e;
    route_kernel<<<1, kRouteThreads, smem, stream>>>(ids, R, E, e_begin, E_total, nt, counts, offsets, perm, inv,
                                                    tiles, n_tiles, status, light_max, light_tiles, n_light);
    return cudaGetLastError();
}

cudaError_t launch_route_topk(const float* logits, const float* bias, int T, int E, int k, int32_t* ids,
                              float* weights, cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    const dim3 grid((T + 7) / 8), block(256);
    const int pl = (E + 31) / 32;
    if (pl <= 1) return launch_pdl(route_topk_kernel<1>, grid, block, 0, stream, logits, bias, T, E, k, ids, weights);
    if (pl <= 2) return launch_pdl(route_topk_kernel<2>, grid, block, 0, stream, logits, bias, T, E, k, ids, weights);
    if (pl <= 4) return launch_pdl(route_topk_kernel<4>, grid, block, 0, stream, logits, bias, T, E, k, ids, weights);
    if (pl <= 8) return launch_pdl(route_topk_kernel<8>, grid, block, 0, stream, logits, bias, T, E, k, ids, weights);
    if (pl <= 16)
        return launch_pdl(route_topk_kernel<16>, grid, block, 0, stream, logits, bias, T, E, k, ids, weights);
    if (pl <= 32)
        return launch_pdl(route_topk_kernel<32>, grid, block, 0, stream, logits, bias, T, E, k, ids, weights);
    return cudaErrorInvalidValue;
}

cudaError_t launch_route_gather_small(const int32_t* ids, int R, int E, int e_begin, int E_total, int nt, int topk,
                                      int* counts, int* offsets, int* perm, int* inv, int4* tiles, int* n_tiles,
                                      int* status, const __nv_bfloat16* x, int K, int interleave, __nv_bfloat16* xp,
                                      float* csum, int* flags, int n_flags, cudaStream_t stream) {
    if (R == 0) return cudaSuccess;
    const int smem = (R + E) * static_cast<int>(sizeof(int));
    cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(route_gather_small_kernel), smem);
    if (e != cudaSuccess) return e;
    route_gather_small_kernel<<<R, kSmallRouteThreads, smem, stream>>>(
        ids, R, E, e_begin, E_total, nt, topk, counts, offsets, perm, inv, tiles, n_tiles, status,
        reinterpret_cast<const uint4*>(x), K / 8, interleave, reinterpret_cast<uint4*>(xp),
        interleave == 1 ? csum : nullptr, flags, n_flags);
    return cudaGetLastError();
}

cudaError_t launch_gather(const __nv_bfloat16* x, const int* inv, int T, int topk, int K, int interleave,
                          __nv_bfloat16* xp, float* csum, int R, int* status, int* flags, int n_flags,
                          cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    const int vpr = K / 8;
    return launch_pdl(scatter_kernel, dim3((T + kGatherRows - 1) / kGatherRows), dim3(32 * kGatherRows), 0, stream,
                      reinterpret_cast<const uint4*>(x), inv, T, topk, vpr, interleave, reinterpret_cast<uint4*>(xp),
                      interleave == 1 ? csum : nullptr, R, status, flags, n_flags);
}

cudaError_t launch_interleave_rows(const __nv_bfloat16* src, int64_t rows, int64_t cols, int mode,
                                   __nv_bfloat16* dst, cudaStream_t stream) {
    const int64_t blocks = rows * cols / 16;
    if (blocks == 0) return cudaSuccess;
    const int threads = 256;
    interleave_rows_kernel<<<static_cast<unsigned>((blocks + threads - 1) / threads), threads, 0, stream>>>(
        reinterpret_cast<const uint4*>(src), blocks, mode, reinterpret_cast<uint4*>(dst));
    return cudaGetLastError();
}

cudaError_t launch_combine(const __nv_bfloat16* y, const float* weights, const int* inv, int T, int topk, int K,
                           void* out, bool f32_out, int R, int* status, cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    const int vpr = K / 8;
    const int threads = 128;
    const dim3 grid(T, (vpr + threads - 1) / threads);
    if (f32_out)
        return launch_pdl(combine_kernel<true>, grid, dim3(threads), 0, stream, reinterpret_cast<const uint4*>(y),
                          weights, inv, topk, vpr, out, R, status);
    return launch_pdl(combine_kernel<false>, grid, dim3(threads), 0, stream, reinterpret_cast<const uint4*>(y), weights,
                      inv, topk, vpr, out, R, status);
}

cudaError_t launch_finalize_w13(const float* partial, int ksplit, int R, const int* offsets_end, int N, float limit,
                                int interleave, __nv_bfloat16* h, float* csum, cudaStream_t stream) {
    if (R == 0) return cudaSuccess;
    const int threads = 128;
    const dim3 grid(R, (N / 4 + threads - 1) / threads);
    switch (ksplit) {
        case 2: return launch_pdl(finalize_w13_kernel<2>, grid, dim3(threads), 0, stream, partial, R, offsets_end, N,
                                  limit, interleave, h, csum);
        case 4: return launch_pdl(finalize_w13_kernel<4>, grid, dim3(threads), 0, stream, partial, R, offsets_end, N,
                                  limit, interleave, h, csum);
        case 8: return launch_pdl(finalize_w13_kernel<8>, grid, dim3(threads), 0, stream, partial, R, offsets_end, N,
                                  limit, interleave, h, csum);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_finalize_w2(const float* partial, int ksplit, int R, const int* offsets_end, int K,
                               __nv_bfloat16* y, cudaStream_t stream) {
    if (R == 0) return cudaSuccess;
    return launch_pdl(finalize_w2_kernel, dim3(R), dim3(256), 0, stream, partial, ksplit, R, offsets_end, K, y);
}

template <bool F32OUT>
static cudaError_t launch_combine_partials_t(const float* partial, int ksplit, int R, const float* weights,
                                             const int* inv, int T, int topk, int K, void* out, int* status,
                                             cudaStream_t stream) {
    const int threads = 128;
    const dim3 grid(T, (K / 4 + threads - 1) / threads);
    switch (ksplit) {
        case 2: return launch_pdl(combine_partials_kernel<2, F32OUT>, grid, dim3(threads), 0, stream, partial, R,
                                  weights, inv, topk, K, out, status);
        case 4: return launch_pdl(combine_partials_kernel<4, F32OUT>, grid, dim3(threads), 0, stream, partial, R,
                                  weights, inv, topk, K, out, status);
        case 8: return launch_pdl(combine_partials_kernel<8, F32OUT>, grid, dim3(threads), 0, stream, partial, R,
                                  weights, inv, topk, K, out, status);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_combine_partials(const float* partial, int ksplit, int R, const float* weights, const int* inv,
                                    int T, int topk, int K, void* out, bool f32_out, int* status, cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    return f32_out ? launch_combine_partials_t<true>(partial, ksplit, R, weights, inv, T, topk, K, out, status, stream)
                   : launch_combine_partials_t<false>(partial, ksplit, R, weights, inv, T, topk, K, out, status, stream);
}

// One bounded pipeline wait on a barrier that nothing completes: the wait
// gives up after limit_ns and reports WNA16_ERR_DEVICE_TIMEOUT in *status,
// exactly as a stalled GEMM pipeline would.
__global__ void wait_timeout_check_kernel(int* status, uint64_t limit_ns) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x != 0) return;
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_barrier_init();
    mbar_wait_bounded(&bar, 0, &abort_flag, status, false, limit_ns);
}

cudaError_t launch_wait_timeout_check(int* status, uint64_t limit_ns, cudaStream_t stream) {
    wait_timeout_check_kernel<<<1, 32, 0, stream>>>(status, limit_ns);
    return cudaGetLastError();
}

cudaError_t launch_pack(const int8_t* codes, int64_t rows, int64_t K, int bits, int32_t* packed,
                        cudaStream_t stream) {
    const int64_t n_words = rows * (K * bits / 32);
    if (n_words == 0) return cudaSuccess;
    const int threads = 256;
    const int64_t blocks = (n_words + threads - 1) / threads;
    pack_kernel<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(codes, n_words, bits, packed);
    return cudaGetLastError();
}

}  // namespace wna16

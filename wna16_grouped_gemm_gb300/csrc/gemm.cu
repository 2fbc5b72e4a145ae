// Grouped WNA16 expert GEMM for sm_103a (tcgen05 + TMEM + TMA), used for both
// projections of the routed-expert MoE ("Incubate DeepSeek V4 WNA16 runtime on
// SM86", section "What this branch adds", items 1-3 and 9):
//
//   w13 unit:  D_gate[n, t] = sum_k W1_e[n, k] X[t, k],  D_up likewise with W3_e
//              h[t, n]      = bf16( silu(min(D_gate, L)) * clamp(D_up, -L, L) )
//   w2  unit:  y[t, m]      = bf16( sum_n W2_e[m, n] H[t, n] )
//
// The weights are the M side of the MMA ("swap AB"): a unit is 2 x 128 weight
// rows (gate+up rows n0.., or 256 consecutive w2 rows) against one token tile
// of up to NT rows of a single expert; a work item is a unit and a range of K
// (split K for decode).  Per 128-k A buffer:
//
//   TMA producer (warp 0)      packed INT32 tiles of both weight row blocks and
//                              the token tile (128B-swizzled BF16) -> smem ring
//   scale loader (warp 1)      the item's FP16 scales -> smem (cp.async)
//   dequant warps (4..11)      each thread owns one weight row: reads its packed
//                              words, builds bf16(code*scale) exactly (or the
//                              plain code in group-accumulate mode) and writes
//                              them into a TMEM A buffer with tcgen05.st
//   MMA issuers (2, 3, 16-19)  tcgen05.mma kind::f16, A from TMEM, B from smem,
//                              fp32 accumulators (or group slots) in TMEM
//   epilogue (warps 12..15)    tcgen05.ld -> per-group scaling (group-accumulate
//                              mode) -> SwiGLU / plain -> BF16, or split-K sums
//
// Keeping the dequantised A operand in TMEM means shared memory only carries
// the packed words and the token tile: the BF16 weights never cross the
// shared-memory port, which would otherwise cap decode far below HBM speed.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "dequant.cuh"
#include "gemm.h"
#include "ptx.cuh"

namespace wna16 {

namespace {

// Warp roles: producer, scale loader, issuers 0-1, DW = 8 dequant warps (one
// per 128-row block and TMEM lane quarter), 4 epilogue warps (one per lane
// quarter), issuers 2-5.  A warp can only reach the TMEM lanes of its quarter
// (warp index % 4), which the dequant and epilogue ranges, starting at
// multiples of 4, respect.
constexpr int kProducerWarp = 0;       // TMA
constexpr int kScaleWarp = 1;          // cp.async of the scales
constexpr int kIssuerWarp0 = 2;        // MMA issuers; warp 2 also owns the TMEM allocation
constexpr int kIssuerWarp1 = 3;
constexpr int kAllocWarp = kIssuerWarp0;
constexpr int kFirstDequantWarp = 4;
constexpr int kEpilogueWarps = 4;
constexpr int kMaxIssuers = 6;
template <int DW>
struct Roles {
    static constexpr int kFirstEpilogueWarp = kFirstDequantWarp + DW;
    static constexpr int kIssuerWarp2 = kFirstEpilogueWarp + kEpilogueWarps;
    static constexpr int kThreads = 32 * (kIssuerWarp2 + 4);
};
constexpr int kRowsPerTile = 128;
constexpr int kKA = 128;         // K elements per TMEM A buffer (per row block): 64 columns
constexpr int kMaxABuf = 3;      // TMEM A ring depth (fewer when the accumulators need the columns)
constexpr int kTmemCols = 512;
// Group-partial slots of the group-accumulate mode (2 x 16 columns each): one
// per issuer parity, so that a slot is always refilled by the issuer that
// filled it before.  An mbarrier parity wait is only sound when the barrier
// can be neither two phases behind the waiter (the wait would pass early) nor
// two phases ahead (it would wait for a later phase).  Every wait here is on
// a barrier whose phases the waiter's own earlier waits and arrivals order:
// the dequant warps and the epilogue wait on every phase of theirs; an issuer
// waits on the A buffers and group slots of its own parity only, which with
// 3 A buffers and 3 parities (GA) or in-order afull completions (4 issuers)
// keeps it within one phase.
constexpr int kGaSlots = 3;

struct Ring {
    uint32_t idx = 0, phase = 0;
    __device__ __forceinline__ void next(uint32_t n) {
        if (++idx == n) {
            idx = 0;
            phase ^= 1u;
        }
    }
};


// Weight rows of the two 128-row blocks of unit (expert e, row tile mt).
template <bool W13>
__device__ __forceinline__ void unit_rows(const GemmParams& p, int e, int mt, int& r0, int& r1) {
    const int base = e * p.rows_per_expert;
    if constexpr (W13) {
        r0 = base + mt * kRowsPerTile;                  // gate rows
        r1 = base + p.half_rows + mt * kRowsPerTile;    // up rows
    } else {
        r0 = base + mt * 2 * kRowsPerTile;
        r1 = r0 + kRowsPerTile;
    }
}

}  // namespace

template <int BITS, bool W13, int DW, int GA>
__global__ void __launch_bounds__(Roles<DW>::kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_b,
                        const GemmParams p) {
    constexpr int kCodes = 32 / BITS;
    constexpr int kDequantWarps = DW;
    constexpr int kFirstEpilogueWarp = Roles<DW>::kFirstEpilogueWarp;
    constexpr int kIssuerWarp2 = Roles<DW>::kIssuerWarp2;
    constexpr int kEW = DW == 16 ? 8 : 16;   // epilogue column chunk (fits the register budget)
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int nt = p.nt;
    const int kp = p.kp;
    const int nstage = p.nstage;
    const int pitch = kp * BITS / 8;                     // packed bytes per row per stage
    const int b_stage_bytes = (kp / 64) * nt * 128;
    const int w_tile_bytes = kRowsPerTile * pitch;
    const int ksteps = p.kred / kp;
    const int chunks = kp / kKA;
    const int nabuf = p.nabuf;
    const int nacc = p.nacc;
    const int n_iss = p.n_issuers;
    static_assert(GA == 0 || BITS == 2, "group-accumulate mode: 2-bit codes");
    static_assert(DW == 8, "8 dequant warps: one per row block and TMEM lane quarter");
    // group-accumulate mode (GA 1 or 2; see the issuer and epilogue sections),
    // GA 2 with offset codes and per-token corrections (p.csum)
    constexpr bool ga = GA != 0;
    constexpr bool goff = GA == 2;

    uint8_t* sB = smem + p.off_b;
    uint8_t* sW = smem + p.off_w;
    uint16_t* sS = reinterpret_cast<uint16_t*>(smem + p.off_s);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.off_bar);
    uint64_t* full = bars;
    uint64_t* empty = full + nstage;
    uint64_t* afull = empty + nstage;
    uint64_t* aempty = afull + 2 * kMaxABuf;   // afull/aempty: [A buffer][row block]
    uint64_t* accfull = aempty + 2 * kMaxABuf; // [2]
    uint64_t* accempty = accfull + 2;          // [2]
    uint64_t* sfull = accempty + 2;
    uint64_t* sempty = sfull + 2;
    uint64_t* drain = sempty + 2;              // [kMaxIssuers]
    uint64_t* gfull = drain + kMaxIssuers;     // [kGaSlots]
    uint64_t* gempty = gfull + kGaSlots;       // [kGaSlots]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gempty + kGaSlots);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    if (threadIdx.x == 0) {
        for (int i = 0; i < nstage; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kDequantWarps + n_iss);
        }
        for (int i = 0; i < 2 * kMaxABuf; ++i) {
            mbar_init(&afull[i], 4);               // the 4 dequant warps of the row block
            mbar_init(&aempty[i], 1);              // the one issuer of the row block that reads it
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&accfull[i], n_iss);
            mbar_init(&accempty[i], n_iss == 2 ? 2 * kEpilogueWarps : kEpilogueWarps);   // + helpers
            mbar_init(&sfull[i], 32);
            mbar_init(&sempty[i], ga ? kEpilogueWarps : kDequantWarps);   // whoever applies the scales
        }
        for (int i = 0; i < kMaxIssuers; ++i) mbar_init(&drain[i], 1);
        for (int i = 0; i < kGaSlots; ++i) {
            mbar_init(&gfull[i], 2);                   // the group's two issuers (row blocks)
            mbar_init(&gempty[i], kEpilogueWarps);
        }
        *abort_flag = 0;
        fence_barrier_init();
        tma_prefetch_desc(&tm_w);
        tma_prefetch_desc(&tm_b);
    }
    if (warp == kAllocWarp) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = __shfl_sync(0xffffffffu, *tmem_slot, 0);   // warp-uniform
    // Everything above overlapped the previous kernel; its outputs are read
    // only below.  With early_w (the w2 GEMM, whose tile list was written
    // kernels earlier) only the token tiles depend on the previous kernel: the
    // producer issues the weights of its first stages before it waits, and
    // the scale and dequant warps, which read only weights, scales and the
    // tile list, start converting them without waiting; the issuers (token
    // tiles) and the epilogue (which writes buffers the previous kernel may
    // read) wait here.
    const bool early_w = p.early_w != 0;
    const bool is_dequant = warp >= kFirstDequantWarp && warp < kFirstDequantWarp + kDequantWarps;
    if (!early_w || !(warp == kProducerWarp || warp == kScaleWarp || is_dequant)) pdl_wait();
    pdl_trigger();

    const int n_units = (*p.n_tiles) * p.mt_count;
    const int ksplit = p.ksplit;
    const int n_items = n_units * ksplit;         // item = (unit, K split)
    const int kps = ksteps / ksplit;              // stages per item
    const int nbuf_item = kps * chunks;           // TMEM A buffers per item
    int* status = p.status;
    // TMEM columns: [nacc sets x n_iss accumulators of nt columns] [A buffers of 128 columns],
    // in GA mode [kGaSlots group slots of 2 x 16 columns, padded to 128] [A buffers]
    const uint32_t acc_set_cols = static_cast<uint32_t>(n_iss * nt);
    const uint32_t abase_col = ga ? 128u : static_cast<uint32_t>(nacc) * acc_set_cols;
    const int issuer = warp == kIssuerWarp0                                ? 0
                       : warp == kIssuerWarp1                             ? 1
                       : (warp >= kIssuerWarp2 && warp < kIssuerWarp2 + 4) ? 2 + (warp - kIssuerWarp2)
                                                                           : -1;
    // group-accumulate mode: groups of this CTA counted over all its items
    const int ng_item = p.ngroups / ksplit;       // scale groups per item
    const uint32_t nt8 = static_cast<uint32_t>(nt) * 8u;   // one 64-k token atom (nt x 128 B) >> 4

    if (warp == kProducerWarp) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint64_t pol_w = p.w_reuse ? policy_evict_normal() : policy_evict_first();
            const uint64_t pol_b = policy_evict_last();
            const uint32_t tx = static_cast<uint32_t>(2 * w_tile_bytes + b_stage_bytes);
            Ring st;
            uint32_t issued = 0, last_parity = 0;   // per slot: issued at least once / parity of last issue
            bool ok = true;
            // early_w: the weights of the first item's first stages (every slot
            // is free at the start), then the dependency wait
            int pre = 0;
            if (early_w) {
                if (static_cast<int>(blockIdx.x) < n_items) {
                    const int u = static_cast<int>(blockIdx.x) / ksplit;
                    const int split = static_cast<int>(blockIdx.x) - u * ksplit;
                    const int4 tile = p.tiles[u / p.mt_count];
                    int r0, r1;
                    unit_rows<W13>(p, tile.x, u % p.mt_count, r0, r1);
                    pre = min(nstage, kps);
                    for (int i = 0; i < pre; ++i) {
                        mbar_arrive_expect_tx(&full[i], tx);
                        tma_load_3d(sW + i * 2 * w_tile_bytes, &tm_w, &full[i], (split * kps + i) * (kp / kCodes), r0,
                                    0, pol_w);
                    }
                }
                pdl_wait();
            }
            for (int v = blockIdx.x; v < n_items && ok; v += gridDim.x) {
                const int u = v / ksplit;
                const int split = v - u * ksplit;
                const int4 tile = p.tiles[u / p.mt_count];
                int r0, r1;
                unit_rows<W13>(p, tile.x, u % p.mt_count, r0, r1);
                for (int ks = split * kps; ks < (split + 1) * kps; ++ks) {
                    if (pre > 0 && v == static_cast<int>(blockIdx.x) && ks - split * kps < pre) {
                        // weights already in flight: the token tile only
                        tma_load_3d(sB + st.idx * b_stage_bytes, &tm_b, &full[st.idx], 0, tile.y, ks * (kp / 64),
                                    pol_b);
                        issued |= 1u << st.idx;
                        last_parity = (last_parity & ~(1u << st.idx)) | (st.phase << st.idx);
                        st.next(nstage);
                        continue;
                    }
                    if (!mbar_try_wait(smem_u32(&empty[st.idx]), st.phase ^ 1u) &&
                        !mbar_wait_bounded(&empty[st.idx], st.phase ^ 1u, abort_flag, status, true)) {
                        ok = false;
                        break;
                    }
                    // two TMA instructions per stage: both weight row blocks in one
                    // 3-D box, all 64-k atoms of the token tile in another
                    mbar_arrive_expect_tx(&full[st.idx], tx);
                    tma_load_3d(sW + st.idx * 2 * w_tile_bytes, &tm_w, &full[st.idx], ks * (kp / kCodes), r0, 0,
                                pol_w);
                    tma_load_3d(sB + st.idx * b_stage_bytes, &tm_b, &full[st.idx], 0, tile.y, ks * (kp / 64), pol_b);
                    issued |= 1u << st.idx;
                    last_parity = (last_parity & ~(1u << st.idx)) | (st.phase << st.idx);
                    st.next(nstage);
                }
            }
            // No copy may still be in flight when the CTA exits: wait for the
            // last issue of every slot (already complete on the normal path).
            for (int i = 0; i < nstage; ++i) {
                if (!(issued & (1u << i))) continue;
                const uint32_t a = smem_u32(&full[i]);
                const uint32_t ph = (last_parity >> i) & 1u;
                const uint64_t t0 = globaltimer_ns();
                while (!mbar_try_wait(a, ph)) {
                    if (globaltimer_ns() - t0 > kWaitLimitNs) {
                        atomicExch(status, kStatusTimeout);
                        break;
                    }
                }
            }
        }
    } else if (issuer >= 0 && !(n_iss == 2 && warp >= kIssuerWarp2)) {
        // ------------------------------------------------------------ MMA issuers
        // Issuer i serves row block t = i & 1.  One thread can issue a
        // tcgen05.mma only every ~110 cycles, so several issuers keep the tensor
        // pipe fed: with 4 issuers, parity h = i >> 1 takes the item's A buffers
        // b with b % 2 == h, each issuer into its own accumulator (the epilogue
        // adds them).  In group-accumulate mode (6 issuers) issuer parity
        // h = i >> 1 takes the groups g with g % 3 == h, and every group is
        // accumulated from zero into a slot of kGaSlots that the epilogue warps
        // scale and add up.
        // The whole warp runs the loop: lane 0 waits and the warp follows its
        // verdict; one elected thread issues each A buffer's MMAs and their
        // commits (elect.sync keeps the operands in uniform registers, which
        // makes each MMA ~3x cheaper to issue than under `if (lane == 0)`).
        auto warp_wait = [&](uint64_t* bar, uint32_t parity) -> bool {
            bool r = true;
            if (lane == 0) r = mbar_wait(bar, parity, abort_flag, status);
            return __shfl_sync(0xffffffffu, r ? 1 : 0, 0) != 0;
        };
        // after a failure: no MMA of this issuer may still run when TMEM is released
        auto drain_issuer = [&]() {
            if (elect_one(status)) {
                tc_commit(&drain[issuer]);
                const uint32_t a = smem_u32(&drain[issuer]);
                const uint64_t t0 = globaltimer_ns();
                while (!mbar_try_wait(a, 0)) {
                    if (globaltimer_ns() - t0 > kWaitLimitNs) break;
                }
            }
            __syncwarp();
        };
        if constexpr (ga) {
          if (issuer < n_iss) {
            const int t = issuer & 1;
            const int h = issuer >> 1;
            const uint32_t idesc = idesc_bf16_f32(128, static_cast<uint32_t>(nt));
            // One group per A buffer (group == 128 k); groups (and buffers) are
            // counted over all items, group g going to parity g % 3, so this
            // issuer's groups all use group slot h and A buffer h, and the
            // k-th of them waits for phase k of those barriers.  Counters
            // instead of divisions: the issuing thread pays every
            // instruction's full latency.
            uint32_t par = 0;    // parity of the current group
            uint32_t own = 0;    // groups of this parity issued so far
            const uint32_t d = tmem + static_cast<uint32_t>(h) * (2 * 16) + static_cast<uint32_t>(t * 16);
            const uint32_t a0 = tmem + abase_col + static_cast<uint32_t>(h) * 128 + t * 64;
            Ring st;
            bool ok = true;
            bool issued = false;
            for (int v = blockIdx.x; v < n_items && ok; v += gridDim.x) {
                for (int ks = 0; ks < kps && ok; ++ks) {
                    if (!warp_wait(&full[st.idx], st.phase)) {
                        ok = false;
                        break;
                    }
                    const uint32_t blo = smem_desc_sw128_lo(smem_u32(sB + st.idx * b_stage_bytes));
                    for (int c = 0; c < chunks; ++c) {
                        if (par == static_cast<uint32_t>(h)) {
                            if (!warp_wait(&gempty[h], (own & 1u) ^ 1u) || !warp_wait(&afull[h * 2 + t], own & 1u)) {
                                ok = false;
                                break;
                            }
                            // B: 64-k swizzle atoms 2c and 2c+1, 32 B per 16 k inside each
                            const uint32_t lo0 = blo + static_cast<uint32_t>(2 * c) * nt8;
                            const uint32_t lo1 = lo0 + nt8;
                            if (elect_one(status)) {
                                tc_fence_after();
#pragma unroll
                                for (int k16 = 0; k16 < 8; ++k16)
                                    tc_mma_ts_lohi(d, a0 + k16 * 8, (k16 < 4 ? lo0 : lo1) + (k16 & 3) * 2,
                                                   kSmemDescSw128Hi, idesc, k16 == 0 ? 0u : 1u);
                                tc_commit(&aempty[h * 2 + t]);
                                tc_commit(&gfull[h]);
                            }
                            __syncwarp();
                            issued = true;
                            ++own;
                        }
                        par = par == 2u ? 0u : par + 1u;
                    }
                    if (!ok) break;
                    if (elect_one(status)) tc_commit(&empty[st.idx]);
                    __syncwarp();
                    st.next(nstage);
                }
            }
            if (!ok && issued) drain_issuer();
          }
        } else if (issuer < n_iss) {
            const int t = issuer & 1;
            const int h = issuer >> 1;
            Ring st, ab, acc;
            bool ok = true;
            bool issued = false;
            for (int v = blockIdx.x; v < n_items && ok; v += gridDim.x) {
                // MMA N: the item's token rows rounded up to 16, not the whole
                // tile (an expert's last tile is often far from full); the
                // columns beyond are neither written nor read for this item
                const int rows = __shfl_sync(0xffffffffu, p.tiles[(v / ksplit) / p.mt_count].z, 0);
                const uint32_t n_mma = static_cast<uint32_t>(min(nt, (rows + 15) & ~15));
                const uint32_t idesc = idesc_bf16_f32(128, n_mma < 16u ? 16u : n_mma);
                if (!warp_wait(&accempty[acc.idx], acc.phase ^ 1u)) break;
                const uint32_t d = tmem + acc.idx * acc_set_cols + static_cast<uint32_t>(issuer * nt);
                uint32_t accumulate = 0;
                int bl = 0;   // A buffer index within the item
                for (int ks = 0; ks < kps && ok; ++ks) {
                    if (!warp_wait(&full[st.idx], st.phase)) {
                        ok = false;
                        break;
                    }
                    const uint32_t blo = smem_desc_sw128_lo(smem_u32(sB + st.idx * b_stage_bytes));
                    for (int c = 0; c < chunks; ++c, ++bl) {
                        if (n_iss == 2 || (bl & 1) == h) {
                            if (!warp_wait(&afull[ab.idx * 2 + t], ab.phase)) {
                                ok = false;
                                break;
                            }
                            const uint32_t a0 = tmem + abase_col + ab.idx * 128 + t * 64;
                            // B: 64-k swizzle atoms 2c and 2c+1, 32 B per 16 k inside each
                            const uint32_t lo0 = blo + static_cast<uint32_t>(2 * c) * nt8;
                            const uint32_t lo1 = lo0 + nt8;
                            if (elect_one(status)) {
                                tc_fence_after();
#pragma unroll
                                for (int k16 = 0; k16 < 8; ++k16)
                                    tc_mma_ts_lohi(d, a0 + k16 * 8, (k16 < 4 ? lo0 : lo1) + (k16 & 3) * 2,
                                                   kSmemDescSw128Hi, idesc, (accumulate | k16) != 0 ? 1u : 0u);
                                tc_commit(&aempty[ab.idx * 2 + t]);
                            }
                            __syncwarp();
                            accumulate = 1;
                            issued = true;
                        }
                        ab.next(nabuf);
                    }
                    if (!ok) break;
                    if (elect_one(status)) tc_commit(&empty[st.idx]);
                    __syncwarp();
                    st.next(nstage);
                }
                if (!ok) break;
                if (elect_one(status)) tc_commit(&accfull[acc.idx]);
                __syncwarp();
                acc.next(nacc);
            }
            if (!ok && issued) drain_issuer();
        }
    } else if (warp == kScaleWarp) {
        // ------------------------------------------------------------ scale loader
        Ring sb;
        const int ng = p.ngroups;
        const int rb = ng_item * 2;                // scale bytes of one row for one item
        const int cb = p.scale_copy_bytes;         // cp.async size (0: plain loads)
        for (int v = blockIdx.x; v < n_items; v += gridDim.x) {
            if (!mbar_wait_bounded(&sempty[sb.idx], sb.phase ^ 1u, abort_flag, status, true)) break;
            const int u = v / ksplit;
            const int g0 = (v - u * ksplit) * ng_item;
            const int4 tile = p.tiles[u / p.mt_count];
            int r0, r1;
            unit_rows<W13>(p, tile.x, u % p.mt_count, r0, r1);
            // buffer layout [256 rows][ng_item] fp16
            uint8_t* dst = reinterpret_cast<uint8_t*>(sS + sb.idx * (ng_item * 2 * kRowsPerTile));
            if (cb) {
                const int cpr = rb / cb;           // copies per row
                for (int i = lane; i < 2 * kRowsPerTile * cpr; i += 32) {
                    const int r = i / cpr;
                    const int c = i - r * cpr;
                    const int grow = r < kRowsPerTile ? r0 + r : r1 + (r - kRowsPerTile);
                    if (!in_bounds(grow >= 0 && grow < p.n_weight_rows, status)) continue;
                    const uint8_t* src =
                        reinterpret_cast<const uint8_t*>(p.scales + static_cast<int64_t>(grow) * ng + g0) + c * cb;
                    uint8_t* dd = dst + r * rb + c * cb;
                    if (cb == 16)
                        cp_async<16>(dd, src);
                    else if (cb == 8)
                        cp_async<8>(dd, src);
                    else
                        cp_async<4>(dd, src);
                }
                cp_async_arrive(&sfull[sb.idx]);
            } else {
                uint16_t* d16 = reinterpret_cast<uint16_t*>(dst);
                for (int r = lane; r < 2 * kRowsPerTile; r += 32) {
                    const int grow = r < kRowsPerTile ? r0 + r : r1 + (r - kRowsPerTile);
                    if (!in_bounds(grow >= 0 && grow < p.n_weight_rows, status)) continue;
                    const uint16_t* src = p.scales + static_cast<int64_t>(grow) * ng + g0;
                    for (int g = 0; g < ng_item; ++g) d16[r * ng_item + g] = __ldg(src + g);
                }
                mbar_arrive(&sfull[sb.idx]);
            }
            sb.next(2);
        }
    } else if (warp >= kFirstDequantWarp && warp < kFirstDequantWarp + kDequantWarps) {
        // ------------------------------------------------------------ dequant
        const int blk = (warp - kFirstDequantWarp) >> 2;   // row block 0 or 1
        const int quarter = warp & 3;                     // TMEM lanes 32*quarter ..
        const int row = quarter * 32 + lane;              // row within the block
        const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t xr = static_cast<uint32_t>((row * pitch) >> 7) & static_cast<uint32_t>(pitch / 16 - 1);
        const uint32_t abase = tmem + abase_col + lane_base + static_cast<uint32_t>(blk * 64);
        Ring st, ab, sb;
        bool ok = true;
        const bool g32 = p.group == 32;
        const int halves_per_group = g32 ? 1 : p.group / 64;
        for (int v = blockIdx.x; v < n_items && ok; v += gridDim.x) {
            const int u = v / ksplit;
            const int split = v - u * ksplit;
            // GA mode: the epilogue warps apply the scales, not these warps
            if (!ga && !mbar_wait_bounded(&sfull[sb.idx], sb.phase, abort_flag, status)) break;
            const uint16_t* srow = sS + sb.idx * (ng_item * 2 * kRowsPerTile) + (blk * kRowsPerTile + row) * ng_item;
            // scale group of the current 64-k half (group 32: the first of its two groups)
            int gi = 0, gleft = halves_per_group;
            auto next_half = [&]() {
                if (g32) {
                    gi += 2;
                } else if (--gleft == 0) {
                    gleft = halves_per_group;
                    ++gi;
                }
            };
            // one 64-k half of weights: one scale, or (group 32) one per 32 k
            auto half_chunk = [&](const uint8_t* wr, int chunk, uint32_t (&v)[32]) {
                if (g32)
                    dequant_chunk_g32<BITS>(wr, xr, chunk, __half2float(__ushort_as_half(srow[gi])),
                                            __half2float(__ushort_as_half(srow[gi + 1])), v);
                else
                    dequant_chunk<BITS>(wr, xr, chunk, __half2float(__ushort_as_half(srow[gi])), v);
            };
            for (int ks = split * kps; ks < (split + 1) * kps && ok; ++ks) {
                if (!mbar_wait(&full[st.idx], st.phase, abort_flag, status)) {
                    ok = false;
                    break;
                }
                const uint8_t* wrow = sW + st.idx * 2 * w_tile_bytes + blk * w_tile_bytes + row * pitch;
                for (int c = 0; c < chunks; ++c) {
                    // one TMEM A buffer = 128 k = two 64-k halves (scales may differ
                    // for group 64), this warp's 32 rows of its row block.  The
                    // buffer's aempty phase is probed before the arithmetic (the
                    // answer takes ~50-100 cycles); the stores are waited for and
                    // afull is arrived on at once, which measured faster than
                    // deferring them past the next buffer.  Every warp arrives on
                    // the buffers in order, so afull phases complete in order.
                    const uint32_t abar = ab.idx * 2 + blk;   // per row block
                    const bool a_ready = mbar_test_wait(smem_u32(&aempty[abar]), ab.phase ^ 1u);
                    uint32_t v32[32];
                    if constexpr (BITS == 2) {
                        if constexpr (goff) {
                            codes_chunk2<true>(wrow, xr, 2 * c, v32);
                        } else if (ga) {
                            codes_chunk2<false>(wrow, xr, 2 * c, v32);
                        } else {
                            half_chunk(wrow, 2 * c, v32);
                        }
                    } else {
                        half_chunk(wrow, 2 * c, v32);
                    }
                    next_half();
                    if (!a_ready && !mbar_wait_bounded(&aempty[abar], ab.phase ^ 1u, abort_flag, status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    tc_st_32x32b_x32(abase + ab.idx * 128, v32);
                    if constexpr (BITS == 2) {
                        if constexpr (goff) {
                            codes_chunk2<true>(wrow, xr, 2 * c + 1, v32);
                        } else if (ga) {
                            codes_chunk2<false>(wrow, xr, 2 * c + 1, v32);
                        } else {
                            half_chunk(wrow, 2 * c + 1, v32);
                        }
                    } else {
                        half_chunk(wrow, 2 * c + 1, v32);
                    }
                    next_half();
                    tc_st_32x32b_x32(abase + ab.idx * 128 + 32, v32);
                    tc_wait_st();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&afull[abar]);
                    ab.next(nabuf);
                }
                if (!ok) break;
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[st.idx]);
                st.next(nstage);
            }
            if (!ok) break;
            if (!ga) {
                __syncwarp();
                if (lane == 0) mbar_arrive(&sempty[sb.idx]);
                sb.next(2);
            }
        }
    } else if ((warp >= kFirstEpilogueWarp && warp < kFirstEpilogueWarp + kEpilogueWarps) ||
               (n_iss == 2 && warp >= kIssuerWarp2)) {
        // Epilogue warps 12-15; with only 2 issuers (large token tiles) warps
        // 16-19 are idle as issuers and take the upper half of the token
        // columns (their lane quarters are warp % 4 as well).
        // ------------------------------------------------------------ epilogue
        // thread = TMEM lane = weight row `row` of both row blocks
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
        const float L = p.limit;
        const bool helper = warp >= kIssuerWarp2;
        const bool halves = n_iss == 2;   // token columns split between the two warp sets
        // Writes one item's result for its token columns (all of 0..rows-1, or
        // this warp set's half of them); load(j0, s0, s1) yields both row
        // blocks' sums for columns j0..j0+kEW-1.
        auto emit = [&](int split, int mt, int rows_all, int row0, auto&& load) {
            const int jbeg = halves && helper ? nt / 2 : 0;
            const int rows = halves && !helper ? min(rows_all, nt / 2) : rows_all;
            if (ksplit > 1) {
                // Split K: park this split's fp32 sums for the tile's real token
                // rows in partial[split][mt][permuted row][256 weight rows]; a
                // separate kernel adds the splits in split order (deterministic)
                // and applies the epilogue.
                const int64_t R_rows = p.partial_rows;
                float* mine = p.partial + ((static_cast<int64_t>(split) * p.mt_count + mt) * R_rows + row0) *
                                              (2 * kRowsPerTile) + row;
                for (int j0 = jbeg; j0 < rows; j0 += kEW) {
                    float s0[kEW], s1[kEW];
                    load(j0, s0, s1);
#pragma unroll
                    for (int i = 0; i < kEW; ++i) {
                        if (j0 + i < rows && in_bounds(row0 + j0 + i < R_rows, p.status)) {
                            mine[(j0 + i) * (2 * kRowsPerTile)] = s0[i];
                            mine[(j0 + i) * (2 * kRowsPerTile) + kRowsPerTile] = s1[i];
                        }
                    }
                }
                return;
            }
            if constexpr (W13) {
                // gate = block 0, up = block 1 of the same lane
                const int n0 = mt * kRowsPerTile + row;
                const int n = interleave_pos(n0, p.h_interleaved);
                for (int j0 = jbeg; j0 < rows; j0 += kEW) {
                    float g[kEW], uu[kEW];
                    load(j0, g, uu);
#pragma unroll
                    for (int i = 0; i < kEW; ++i)
                        if (j0 + i < rows && in_bounds(row0 + j0 + i < p.partial_rows && n < p.out_ld, p.status))
                            p.out[static_cast<int64_t>(row0 + j0 + i) * p.out_ld + n] =
                                __float2bfloat16_rn(swiglu(g[i], uu[i], L));
                }
            } else {
                const int m = mt * 2 * kRowsPerTile + row;
                for (int j0 = jbeg; j0 < rows; j0 += kEW) {
                    float y0[kEW], y1[kEW];
                    load(j0, y0, y1);
#pragma unroll
                    for (int i = 0; i < kEW; ++i) {
                        if (j0 + i < rows &&
                            in_bounds(row0 + j0 + i < p.partial_rows && m + kRowsPerTile < p.out_ld, p.status)) {
                            __nv_bfloat16* o = p.out + static_cast<int64_t>(row0 + j0 + i) * p.out_ld + m;
                            o[0] = __float2bfloat16_rn(y0[i]);
                            o[kRowsPerTile] = __float2bfloat16_rn(y1[i]);
                        }
                    }
                }
            }
        };
        // Paired splits (fuse_splits), after this CTA parked split 1 of w13 unit
        // (mt, tile) and released its accumulator: add the split-0 sums that
        // the partner CTA's thread of the same warp and lane parked and this
        // thread's own split-1 sums (the finalize kernel's order: split 0,
        // then 1) and write h, off the issuers' path.
        auto finish = [&](int mt, int rows_all, int row0) {
            if constexpr (W13) {
                const int jbeg = halves && helper ? nt / 2 : 0;
                const int rows = halves && !helper ? min(rows_all, nt / 2) : rows_all;
                const int64_t R_rows = p.partial_rows;
                const float* q0 = p.partial + (static_cast<int64_t>(mt) * R_rows + row0) * (2 * kRowsPerTile) + row;
                const float* q1 = q0 + static_cast<int64_t>(p.mt_count) * R_rows * (2 * kRowsPerTile);
                const int n = interleave_pos(mt * kRowsPerTile + row, p.h_interleaved);
                for (int j0 = jbeg; j0 < rows; j0 += kEW) {
                    float g[kEW], uu[kEW];
#pragma unroll
                    for (int i = 0; i < kEW; ++i) {
                        const bool ok = j0 + i < rows && in_bounds(row0 + j0 + i < R_rows, p.status);
                        const int64_t o = static_cast<int64_t>(j0 + i) * (2 * kRowsPerTile);
                        g[i] = ok ? __ldcg(q0 + o) + q1[o] : 0.0f;
                        uu[i] = ok ? __ldcg(q0 + o + kRowsPerTile) + q1[o + kRowsPerTile] : 0.0f;
                    }
#pragma unroll
                    for (int i = 0; i < kEW; ++i)
                        if (j0 + i < rows && in_bounds(row0 + j0 + i < R_rows && n < p.out_ld, p.status))
                            p.out[static_cast<int64_t>(row0 + j0 + i) * p.out_ld + n] =
                                __float2bfloat16_rn(swiglu(g[i], uu[i], L));
                }
            }
        };
        // Same, from sums held in registers (columns 0..N-1).
        auto emit_regs = [&](int split, int mt, int rows, int row0, const auto& y0, const auto& y1) {
            constexpr int N = sizeof(y0) / sizeof(y0[0]);
            if (ksplit > 1) {
                const int64_t R_rows = p.partial_rows;
                float* mine = p.partial + ((static_cast<int64_t>(split) * p.mt_count + mt) * R_rows + row0) *
                                              (2 * kRowsPerTile) + row;
#pragma unroll
                for (int i = 0; i < N; ++i) {
                    if (i < rows && in_bounds(row0 + i < R_rows, p.status)) {
                        mine[i * (2 * kRowsPerTile)] = y0[i];
                        mine[i * (2 * kRowsPerTile) + kRowsPerTile] = y1[i];
                    }
                }
                return;
            }
            if constexpr (W13) {
                const int n0 = mt * kRowsPerTile + row;
                const int n = interleave_pos(n0, p.h_interleaved);
#pragma unroll
                for (int i = 0; i < N; ++i)
                    if (i < rows && in_bounds(row0 + i < p.partial_rows && n < p.out_ld, p.status))
                        p.out[static_cast<int64_t>(row0 + i) * p.out_ld + n] = __float2bfloat16_rn(swiglu(y0[i], y1[i], L));
            } else {
                const int m = mt * 2 * kRowsPerTile + row;
#pragma unroll
                for (int i = 0; i < N; ++i) {
                    if (i < rows && in_bounds(row0 + i < p.partial_rows && m + kRowsPerTile < p.out_ld, p.status)) {
                        __nv_bfloat16* o = p.out + static_cast<int64_t>(row0 + i) * p.out_ld + m;
                        o[0] = __float2bfloat16_rn(y0[i]);
                        o[kRowsPerTile] = __float2bfloat16_rn(y1[i]);
                    }
                }
            }
        };
        if constexpr (ga) {
            {
                // Group-accumulate mode (2-bit codes, 16-token tiles): every group's
                // code sums arrive in a TMEM slot; this row's sums add
                // bf16(scale) * slot in group order.  For 2-bit codes (0 or +-2^j)
                // code * bf16(scale) is exactly the BF16-rounded dequantised
                // weight, so this is the same sum as with dequantised weights.
                // With offset codes the slot holds sum (code + off + 2) x; the
                // token's correction
                // sum (off + 2) x over the group (csum[group][permuted row]) is
                // subtracted first, the same for both row blocks.
                Ring sb, gs;   // gs: group slot ring (kGaSlots), advanced per group
                const int R_rows = p.partial_rows;
                bool ok = true;
                auto scale_of = [](uint16_t h) {
                    return __bfloat162float(__float2bfloat16_rn(__half2float(__ushort_as_half(h))));
                };
                for (int v = blockIdx.x; v < n_items && ok; v += gridDim.x) {
                    const int u = v / ksplit;
                    const int split = v - u * ksplit;
                    const int4 tile = p.tiles[u / p.mt_count];
                    if (!mbar_wait_bounded(&sfull[sb.idx], sb.phase, abort_flag, status)) break;
                    const uint16_t* s0row = sS + sb.idx * (ng_item * 2 * kRowsPerTile) + row * ng_item;
                    const uint16_t* s1row = s0row + kRowsPerTile * ng_item;
                    // corrections of this item's groups for the tile's token rows
                    const float* crow = goff ? p.csum + static_cast<int64_t>(split * ng_item) * R_rows + tile.y : nullptr;
                    // tiles of 2-bit 16-token plans hold at most 8 token rows (the
                    // routing cuts them so), which read 8 columns per block
                    in_bounds(tile.z <= 8, status);
                    float y0[8], y1[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) y0[i] = y1[i] = 0.0f;
                    for (int g = 0; g < ng_item; ++g) {
                        float cs[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            cs[i] = goff && i < tile.z &&
                                            in_bounds(tile.y + i < R_rows && split * ng_item + g < p.ngroups, status)
                                        ? __ldg(crow + static_cast<int64_t>(g) * R_rows + i)
                                        : 0.0f;
                        if (!mbar_wait(&gfull[gs.idx], gs.phase, abort_flag, status)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        uint32_t d0[8], d1[8];
                        const uint32_t col = gs.idx * (2 * 16);
                        tc_ld_32x32b_x8(tmem + lane_base + col, d0);
                        tc_ld_32x32b_x8(tmem + lane_base + col + 16, d1);
                        tc_wait_ld();
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&gempty[gs.idx]);
                        gs.next(kGaSlots);
                        const float c0 = scale_of(s0row[g]);
                        const float c1 = scale_of(s1row[g]);
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            y0[i] = __fmaf_rn(c0, __uint_as_float(d0[i]) - cs[i], y0[i]);
                            y1[i] = __fmaf_rn(c1, __uint_as_float(d1[i]) - cs[i], y1[i]);
                        }
                    }
                    if (!ok) break;
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&sempty[sb.idx]);
                    sb.next(2);
                    emit_regs(split, u % p.mt_count, tile.z, tile.y, y0, y1);
                }
            }
        } else {
            // a row block's sum is its issuers' accumulators added (one or two parities)
            const int nh = (n_iss == 4 && nbuf_item >= 2) ? 2 : 1;
            Ring acc;
            for (int v = blockIdx.x; v < n_items; v += gridDim.x) {
                const int u = v / ksplit;
                const int split = v - u * ksplit;
                const int4 tile = p.tiles[u / p.mt_count];
                if (!mbar_wait_bounded(&accfull[acc.idx], acc.phase, abort_flag, status, true)) break;
                tc_fence_after();
                const uint32_t a0 = tmem + lane_base + acc.idx * acc_set_cols;   // issuer i at + i * nt
                // every load of a column chunk is issued before the one wait
                // (TMEM loads take hundreds of cycles to complete)
                auto loader = [&](int j0, float (&s0)[kEW], float (&s1)[kEW]) {
                    if (nh == 1) {
                        uint32_t d0[kEW], d1[kEW];
                        if constexpr (kEW == 16) {
                            tc_ld_32x32b_x16(a0 + static_cast<uint32_t>(j0), d0);
                            tc_ld_32x32b_x16(a0 + static_cast<uint32_t>(nt + j0), d1);
                        } else {
                            tc_ld_32x32b_x8(a0 + static_cast<uint32_t>(j0), d0);
                            tc_ld_32x32b_x8(a0 + static_cast<uint32_t>(nt + j0), d1);
                        }
                        tc_wait_ld();
#pragma unroll
                        for (int i = 0; i < kEW; ++i) {
                            s0[i] = __uint_as_float(d0[i]);
                            s1[i] = __uint_as_float(d1[i]);
                        }
                    } else {
#pragma unroll
                        for (int q = 0; q < kEW; q += 8) {
                            uint32_t d0[8], d1[8], d2[8], d3[8];
                            tc_ld_32x32b_x8(a0 + static_cast<uint32_t>(j0 + q), d0);
                            tc_ld_32x32b_x8(a0 + static_cast<uint32_t>(nt + j0 + q), d1);
                            tc_ld_32x32b_x8(a0 + static_cast<uint32_t>(2 * nt + j0 + q), d2);
                            tc_ld_32x32b_x8(a0 + static_cast<uint32_t>(3 * nt + j0 + q), d3);
                            tc_wait_ld();
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                s0[q + i] = __uint_as_float(d0[i]) + __uint_as_float(d2[i]);
                                s1[q + i] = __uint_as_float(d1[i]) + __uint_as_float(d3[i]);
                            }
                        }
                    }
                };
                const bool fused = W13 && p.fuse_splits;
                emit(split, u % p.mt_count, tile.z, tile.y, loader);
                // the accumulator is free once its loads have landed in
                // registers: release it before the stores are made visible
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&accempty[acc.idx]);
                acc.next(nacc);
                if (fused && split == 0) {
                    // publish: every lane's stores, then one count per warp
                    __threadfence();
                    __syncwarp();
                    if (lane == 0) atomicAdd(p.unit_flags + u, 1);
                }
                if (fused && split == 1) {
                    // wait (bounded) until all epilogue warps of the split-0 CTA
                    // have parked this unit's sums, then write h
                    int okw = 1;
                    if (lane == 0) {
                        const uint64_t t0 = globaltimer_ns();
                        while (ld_acquire_gpu(p.unit_flags + u) < 2 * kEpilogueWarps) {
                            if (*abort_flag) {
                                okw = 0;
                                break;
                            }
                            if (globaltimer_ns() - t0 > kWaitLimitNs) {
                                *abort_flag = 1;
                                atomicExch(status, kStatusTimeout);
                                okw = 0;
                                break;
                            }
                            __nanosleep(64);
                        }
                    }
                    if (!__shfl_sync(0xffffffffu, okw, 0)) break;
                    finish(u % p.mt_count, tile.z, tile.y);
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kAllocWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ------------------------------------------------------------------ host side

GemmSmem gemm_smem_layout(int bits, int nt, int kp, int ng_item, int max_smem) {
    GemmSmem L{};
    const int pitch = kp * bits / 8;
    const int b_stage = (kp / 64) * nt * 128;
    const int w_stage = 2 * kRowsPerTile * pitch;
    const int s_bytes = 2 * ng_item * 2 * kRowsPerTile * 2;   // two item buffers [256 rows][ng_item] fp16
    const int bar_bytes = 8 * (2 * 16 + 4 * kMaxABuf + 4 + 4 + kMaxIssuers + 2 * kGaSlots) + 16;
    const int fixed = s_bytes + bar_bytes + 1024 /*alignment slack*/;
    int ns = (max_smem - fixed) / (b_stage + w_stage);
    if (ns > 8) ns = 8;
    L.nstage = ns;
    if (ns < 2) return L;
    L.off_b = 0;
    L.off_w = ns * b_stage;
    L.off_s = L.off_w + ns * w_stage;
    L.off_bar = (L.off_s + s_bytes + 7) & ~7;
    L.total = L.off_bar + 8 * (2 * ns + 4 * kMaxABuf + 4 + 4 + kMaxIssuers + 2 * kGaSlots) + 16 + 1024;
    return L;
}

template <int BITS, bool W13, int DW, int GA>
static cudaError_t launch_impl(const CUtensorMap& tm_w, const CUtensorMap& tm_b, const GemmParams& p, int grid,
                               int smem_bytes, cudaStream_t stream) {
    auto kern = grouped_gemm_kernel<BITS, W13, DW, GA>;
    cudaError_t err = ensure_dynamic_smem(reinterpret_cast<const void*>(kern), smem_bytes);
    if (err != cudaSuccess) return err;
    return launch_pdl(kern, dim3(grid), dim3(Roles<DW>::kThreads), static_cast<size_t>(smem_bytes), stream, tm_w,
                      tm_b, p);
}

template <int BITS, bool W13>
static cudaError_t launch_dw(const CUtensorMap& tm_w, const CUtensorMap& tm_b, const GemmParams& p, int grid,
                             int smem_bytes, cudaStream_t stream) {
    if constexpr (BITS == 2) {
        if (p.ga && p.csum) return launch_impl<BITS, W13, 8, 2>(tm_w, tm_b, p, grid, smem_bytes, stream);
        if (p.ga) return launch_impl<BITS, W13, 8, 1>(tm_w, tm_b, p, grid, smem_bytes, stream);
    }
    return launch_impl<BITS, W13, 8, 0>(tm_w, tm_b, p, grid, smem_bytes, stream);
}

cudaError_t launch_grouped_gemm(int bits, bool w13, const CUtensorMap& tm_w, const CUtensorMap& tm_b,
                                const GemmParams& p, int grid, int smem_bytes, cudaStream_t stream) {
    if (bits == 2)
        return w13 ? launch_dw<2, true>(tm_w, tm_b, p, grid, smem_bytes, stream)
                   : launch_dw<2, false>(tm_w, tm_b, p, grid, smem_bytes, stream);
    return w13 ? launch_dw<4, true>(tm_w, tm_b, p, grid, smem_bytes, stream)
               : launch_dw<4, false>(tm_w, tm_b, p, grid, smem_bytes, stream);
}

}  // namespace wna16

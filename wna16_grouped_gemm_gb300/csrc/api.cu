// C ABI of the WNA16 routed-expert MoE forward: argument validation,
// workspace layout, TMA descriptors and the launch sequence
//   route -> gather -> grouped w13 (+SwiGLU) -> grouped w2 -> combine
// on the caller's stream.  See include/wna16_moe.h for the contract.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>

#include "../../include/wna16_moe.h"
#include "gemm.h"

using namespace wna16;

namespace {

thread_local char g_err[512] = "";

// Per-thread stage events for wna16_moe_profile (instrumentation only): a
// ring of `slots` forwards x 6 events, so that a caller can queue many
// forwards without waiting and read all their stage times afterwards.
struct StageEvents {
    int slots = 0;          // 0: off
    int next = 0;           // ring position of the next forward
    long long recorded = 0; // forwards recorded since enabled
    cudaEvent_t* ev = nullptr;
};
thread_local StageEvents g_prof;
thread_local int g_launches = 0;   // kernels the last wna16_moe_forward on this thread launched

inline void mark(int i, cudaStream_t s) {
    if (g_prof.slots) cudaEventRecord(g_prof.ev[g_prof.next * 6 + i], s);
}
inline void mark_done() {
    if (g_prof.slots) {
        g_prof.next = (g_prof.next + 1) % g_prof.slots;
        ++g_prof.recorded;
    }
}

int fail(int code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return code;
}

int cuda_fail(cudaError_t e, const char* what) {
    return fail(WNA16_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

constexpr size_t kAlign = 256;
size_t align_up(size_t v) { return (v + kAlign - 1) & ~(kAlign - 1); }

// Light experts of 2-bit prefill batches: at most this many rows (one 8-row
// tile; measured 1 % faster on the 2-bit Zipf prefill than 16, whose 9-16-row
// experts took two light tiles).
constexpr int kLightRows = 8;

// Token tile (MMA N) from the mean rows per expert.
int choose_nt(int64_t R, int64_t E) {
    const double avg = static_cast<double>(R) / static_cast<double>(E);
    if (avg <= 4.0) return 16;
    if (avg <= 16.0) return 32;
    if (avg <= 48.0) return 64;
    return 128;
}

// Split-K plan of one grouped GEMM: the smallest power of two (<= 8) that gives
// at least kTargetItems work items over the largest possible unit count, with
// every split a whole number of pipeline stages and scale groups.  Decided from
// the sizes alone, so the workspace size needs no device query.
constexpr int64_t kTargetItems = 1280;

int stage_k(int nt, int bits, int64_t kred) {
    if (nt > 32) return 128;
    int kp = 1024 / bits;                       // 128 packed bytes per row per stage
    while (kred % kp) kp /= 2;
    return kp;
}

// The tensor cores' fp32 accumulation in TMEM loses low-order bits on every
// MMA K-step (the error grows with the number of steps added into one
// accumulator and leans toward smaller magnitudes); measured against the
// oracle on the 8192-token W4 prefill, 256 K-steps into one accumulator put
// the output at relative L2 1.03e-3, 128 steps at 7.3e-4, 64 at 5.5e-4.  So
// no accumulator takes more than kMaxChain K-steps of 16 before its sum is
// added in fp32 on the CUDA cores: with one accumulator per row block (token
// tiles above 32 rows) the K range is split until each split has at most
// kMaxChain * 16 elements; smaller tiles alternate two accumulators per row
// block (2 * kMaxChain steps per split), and the 2-bit group-accumulate mode
// restarts its accumulator every scale group.
constexpr int64_t kMaxChain = 128;

int min_split_for_chain(int nt, int64_t kred) {
    const int64_t per_acc = nt > 32 ? kMaxChain * 16 : 2 * kMaxChain * 16;
    int S = 1;
    while (S < 8 && kred / S > per_acc) S *= 2;
    return S;
}

// The w2 GEMM's splits are added by the combine, which reads ksplit x topk
// partial rows per output, so its target stops at 4 splits (measured: 8 made
// the one-token decode forward 4 % slower, the combine taking the extra).
int choose_split(int64_t max_units, int64_t kred, int kp, int group, int nt, int max_split = 8) {
    int S = 1;
    const int need = min_split_for_chain(nt, kred);
    while (S < 8 && ((max_units * S < kTargetItems && S < max_split) || S < need)) {
        const int64_t next = 2 * S;
        if ((kred / kp) % next || (kred / next) % group) break;
        S = static_cast<int>(next);
    }
    return S;
}

struct Layout {
    int64_t R = 0;
    int nt = 16;
    int tile_rows = 16;
    int64_t max_tiles = 0;
    int64_t units13 = 0, units2 = 0;      // largest possible unit counts of the two GEMMs
    size_t status = 0, n_tiles = 0, counts = 0, offsets = 0, perm = 0, inv = 0, tiles = 0, xp = 0, h = 0, y = 0;
    size_t chunks = 0;                    // chunked routing scratch: [chunks][E] + [chunks] ints
    size_t partial = 0;
    size_t flags = 0;
    int64_t n_flags = 0;
    size_t csum13 = 0, csum2 = 0;         // offset-code corrections (2-bit, 16-token tiles): [groups][R]
    int light_max = 0;                    // 2-bit prefill plans: experts of at most this many rows get
    int64_t max_light = 0;                //   a light tile list (8-row tiles) and launches of their own
    size_t light_tiles = 0, n_light = 0;
    size_t total = 0;
};

Layout make_layout(int64_t T, int64_t K, int64_t N, int64_t E, int topk, int bits) {
    Layout L;
    L.R = T * topk;
    L.nt = choose_nt(L.R, E);
    // token rows per tile: nt, except 8 for 2-bit 16-token tiles (the
    // group-accumulate epilogue keeps one fp32 sum per row and token, and
    // 8 tokens fit its registers; an expert with more rows gets more tiles)
    L.tile_rows = (bits == 2 && L.nt == 16) ? 8 : L.nt;
    L.max_tiles = (L.R < E ? L.R : E) + L.R / L.tile_rows + 1;
    L.units13 = L.max_tiles * (N / 128);
    L.units2 = L.max_tiles * (K / 256);
    // split-K partial sums for the largest split any group size could give (32
    // is the smallest supported group): splits x row tiles x R token rows x 256
    const int64_t s13 = choose_split(L.units13, K, stage_k(L.nt, bits, K), 32, L.nt);
    const int64_t s2 = choose_split(L.units2, N, stage_k(L.nt, bits, N), 32, L.nt, 4);
    const int64_t p13 = s13 > 1 ? s13 * (N / 128) * L.R * 256 : 0;
    const int64_t p2 = s2 > 1 ? s2 * (K / 256) * L.R * 256 : 0;
    const int64_t partial_floats = p13 > p2 ? p13 : p2;
    size_t o = 0;
    L.status = o;   o = align_up(o + sizeof(int));
    L.n_tiles = o;  o = align_up(o + sizeof(int));
    L.counts = o;   o = align_up(o + sizeof(int) * E);
    L.offsets = o;  o = align_up(o + sizeof(int) * (E + 1));
    L.perm = o;     o = align_up(o + sizeof(int) * L.R);
    L.inv = o;      o = align_up(o + sizeof(int) * L.R);
    L.tiles = o;    o = align_up(o + sizeof(int4) * L.max_tiles);
    L.chunks = o;   o = align_up(o + sizeof(int) * static_cast<size_t>(route_chunks(static_cast<int>(L.R))) * (E + 1));
    L.xp = o;       o = align_up(o + sizeof(__nv_bfloat16) * L.R * K);
    L.h = o;        o = align_up(o + sizeof(__nv_bfloat16) * L.R * N);
    L.y = o;        o = align_up(o + sizeof(__nv_bfloat16) * L.R * K);
    L.partial = o;  o = align_up(o + sizeof(float) * partial_floats);
    // per w13 unit: how many epilogue warps of its first K split have parked
    // their sums (paired splits, see plan_gemm); zeroed by the gather kernels
    L.n_flags = L.max_tiles * (N / 128);
    L.flags = o;    o = align_up(o + sizeof(int) * L.n_flags);
    // group-accumulate mode (2-bit, 16-token tiles, group 128) with offset codes
    const bool ga = bits == 2 && L.nt == 16;
    L.csum13 = o;   o = align_up(o + (ga ? sizeof(float) * L.R * (K / 128) : 0));
    L.csum2 = o;    o = align_up(o + (ga ? sizeof(float) * L.R * (N / 128) : 0));
    // 2-bit batches routed by the large-batch kernels with 64- or 128-token
    // tiles: experts with at most kLightRows rows (the skewed tail) are run by
    // separate group-accumulate launches over 8-row tiles, whose work item
    // costs about half of a full tile's for the same weights
    L.light_max = (bits == 2 && L.nt >= 64 && L.R > kSmallRouteMax) ? kLightRows : 0;
    L.max_light = L.light_max ? E : 0;   // one tile per light expert
    L.light_tiles = o; o = align_up(o + sizeof(int4) * L.max_light);
    L.n_light = o;     o = align_up(o + sizeof(int));
    L.total = o;
    return L;
}

template <typename P>
P* at(void* ws, size_t off) {
    return reinterpret_cast<P*>(static_cast<char*>(ws) + off);
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// ---------------------------------------------------------------- device info

struct DevInfo {
    int sms = 0;
    int max_smem = 0;
};

int device_info(DevInfo& d) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    static std::mutex mu;
    static DevInfo cache[64];
    std::lock_guard<std::mutex> lock(mu);
    if (dev < 64 && cache[dev].sms) {
        d = cache[dev];
        return WNA16_OK;
    }
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (major != 10 || minor != 3)
        return fail(WNA16_ERR_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a", dev, major,
                    minor);
    e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    e = cudaDeviceGetAttribute(&d.max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    if (dev < 64) cache[dev] = d;
    return WNA16_OK;
}

}  // namespace

cudaError_t wna16::ensure_dynamic_smem(const void* fn, int bytes) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    static std::mutex mu;
    static std::map<std::pair<const void*, int>, int> allowed;   // (kernel, device) -> bytes already allowed
    std::lock_guard<std::mutex> lock(mu);
    int& cur = allowed[{fn, dev}];
    if (bytes <= cur) return cudaSuccess;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) cur = bytes;
    return e;
}

namespace {

// ---------------------------------------------------------------- TMA descriptors

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// 3-D tensor: dims[0] contiguous elements; dims[1], dims[2] with byte strides s1, s2.
int encode_3d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, const uint64_t (&dims)[3],
              const uint64_t (&strides)[2], const uint32_t (&box)[3], CUtensorMapSwizzle swz) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return fail(WNA16_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    cuuint64_t d[3] = {dims[0], dims[1], dims[2]};
    cuuint64_t st[2] = {strides[0], strides[1]};
    cuuint32_t b[3] = {box[0], box[1], box[2]};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = fn(map, dtype, 3, const_cast<void*>(base), d, st, b, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(WNA16_ERR_CUDA, "cuTensorMapEncodeTiled (3-D) failed (%d)", static_cast<int>(r));
    return WNA16_OK;
}

CUtensorMapSwizzle swizzle_for_pitch(int pitch) {
    switch (pitch) {
        case 32: return CU_TENSOR_MAP_SWIZZLE_32B;
        case 64: return CU_TENSOR_MAP_SWIZZLE_64B;
        case 128: return CU_TENSOR_MAP_SWIZZLE_128B;
        default: return CU_TENSOR_MAP_SWIZZLE_NONE;
    }
}

// ---------------------------------------------------------------- validation

int check_dims(int64_t T, int64_t K, int64_t N, int64_t E, int topk, int bits) {
    if (T < 0 || K <= 0 || N <= 0 || E <= 0 || topk <= 0)
        return fail(WNA16_ERR_INVALID_ARG, "sizes must be positive (T may be 0): T=%lld K=%lld N=%lld E=%lld topk=%d",
                    (long long)T, (long long)K, (long long)N, (long long)E, topk);
    if (bits != 2 && bits != 4) return fail(WNA16_ERR_UNSUPPORTED, "bits=%d: only 2 and 4 are supported", bits);
    if (topk > E) return fail(WNA16_ERR_INVALID_ARG, "topk=%d exceeds E=%lld", topk, (long long)E);
    if (E > 1024) return fail(WNA16_ERR_UNSUPPORTED, "E=%lld: at most 1024 experts", (long long)E);
    if (K % 256) return fail(WNA16_ERR_UNSUPPORTED, "K=%lld must be a multiple of 256", (long long)K);
    if (N % 128) return fail(WNA16_ERR_UNSUPPORTED, "N=%lld must be a multiple of 128", (long long)N);
    if (T * topk >= (int64_t(1) << 31)) return fail(WNA16_ERR_UNSUPPORTED, "T*topk must be < 2^31");
    if (E * 2 * N >= (int64_t(1) << 31) || E * K >= (int64_t(1) << 31))
        return fail(WNA16_ERR_UNSUPPORTED, "E*2N and E*K must be < 2^31 weight rows");
    return WNA16_OK;
}

// Group sizes: 32, or multiples of 64 (up to the whole reduction dim: one
// scale per output channel), dividing the reduction dim.  Whether the scales
// of one work item fit in shared memory is checked when the launch is planned.
int check_group(int g, int64_t kred, const char* name) {
    if (g <= 0 || (g != 32 && g % 64) || kred % g)
        return fail(WNA16_ERR_UNSUPPORTED, "%s=%d: groups must be 32 or multiples of 64 that divide %lld", name, g,
                    (long long)kred);
    return WNA16_OK;
}

int check_ptr(const void* p, size_t align, const char* name) {
    if (!p) return fail(WNA16_ERR_INVALID_ARG, "%s is NULL", name);
    if (!aligned(p, align)) return fail(WNA16_ERR_INVALID_ARG, "%s must be %zu-byte aligned", name, align);
    return WNA16_OK;
}

int check_workspace(const void* ws, size_t bytes, const Layout& L) {
    if (int rc = check_ptr(ws, kAlign, "workspace")) return rc;
    if (bytes < L.total)
        return fail(WNA16_ERR_WORKSPACE_TOO_SMALL, "workspace has %zu bytes, needs %zu", bytes, L.total);
    return WNA16_OK;
}

// ---------------------------------------------------------------- launch helpers

// Routing lists of the local experts [e_begin, e_begin + E) among E_total.
int run_route(const int32_t* ids, int64_t E, const Layout& L, void* ws, cudaStream_t s, int64_t e_begin = 0,
              int64_t E_total = -1, int light_max = 0) {
    cudaError_t e = launch_route(ids, static_cast<int>(L.R), static_cast<int>(E), static_cast<int>(e_begin),
                                 static_cast<int>(E_total < 0 ? E : E_total), L.tile_rows, at<int>(ws, L.counts),
                                 at<int>(ws, L.offsets), at<int>(ws, L.perm), at<int>(ws, L.inv),
                                 at<int4>(ws, L.tiles), at<int>(ws, L.n_tiles), at<int>(ws, L.status),
                                 at<int>(ws, L.chunks), s, light_max, at<int4>(ws, L.light_tiles),
                                 at<int>(ws, L.n_light));
    return e == cudaSuccess ? WNA16_OK : cuda_fail(e, "route kernel launch");
}

// One grouped GEMM, prepared on the host (tensor maps, parameters, launch
// shape) before anything is launched: w13 (B = Xp [R, K], out = h [R, N]) or
// w2 (B = h [R, N], out = y [R, K]).
struct GemmPlan {
    bool w13 = true;
    int bits = 2;
    CUtensorMap tm_w, tm_b;
    GemmParams gp{};
    int grid = 0;
    int smem = 0;
};

int plan_gemm(GemmPlan& P, bool w13, int bits, const int32_t* wpacked, const uint16_t* wscales, const void* b_src,
              void* out, int64_t K, int64_t N, int64_t E, int group, float limit, const Layout& L, void* ws,
              int h_interleaved = 0, const float* csum = nullptr, bool light = false) {
    DevInfo dev;
    if (int rc = device_info(dev)) return rc;
    const int64_t kred = w13 ? K : N;
    const int64_t rows_per_expert = w13 ? 2 * N : K;
    // light: the light experts' launch, 16-token tiles (of at most 8 rows)
    // over the light tile list, no K split (every output written directly)
    const int nt = light ? 16 : L.nt;
    const int kp = stage_k(nt, bits, kred);
    const int pitch = kp * bits / 8;
    const int64_t mt_units = w13 ? N / 128 : K / 256;
    const int64_t max_units = light ? L.max_light * mt_units : (w13 ? L.units13 : L.units2);
    const int ksplit = light ? 1 : choose_split(max_units, kred, kp, group, nt, w13 ? 8 : 4);
    const int ngroups = static_cast<int>(kred / group);
    GemmSmem sm = gemm_smem_layout(bits, nt, kp, ngroups / ksplit, dev.max_smem);
    if (sm.nstage < 2)
        return fail(WNA16_ERR_UNSUPPORTED,
                    "shared-memory plan does not fit (%d scale groups per work item of 256 rows; group %d along %lld)",
                    ngroups / ksplit, group, (long long)kred);

    const int p = 32 / bits;
    {
        // weights: [words of a row][rows][the unit's two 128-row blocks], the
        // second block N rows (w13: up) or 128 rows (w2) after the first
        const uint64_t row_bytes = static_cast<uint64_t>(kred / p) * 4;
        const uint64_t brows = 128;
        const uint64_t block_rows = w13 ? static_cast<uint64_t>(N) : brows;
        const uint64_t dims[3] = {static_cast<uint64_t>(kred / p),
                                  static_cast<uint64_t>(E * rows_per_expert) - block_rows, 2};
        const uint64_t strides[2] = {row_bytes, block_rows * row_bytes};
        const uint32_t box[3] = {static_cast<uint32_t>(pitch / 4), static_cast<uint32_t>(brows), 2};
        if (int rc = encode_3d(&P.tm_w, CU_TENSOR_MAP_DATA_TYPE_INT32, wpacked, dims, strides, box,
                               swizzle_for_pitch(pitch)))
            return rc;
    }
    {
        // token rows: [64 elements][rows][64-k atoms] so that one box is the
        // stage's atoms one after another, each nt rows x 128 B (128B-swizzled)
        const uint64_t dims[3] = {64, static_cast<uint64_t>(L.R), static_cast<uint64_t>(kred / 64)};
        const uint64_t strides[2] = {static_cast<uint64_t>(kred) * 2, 128};
        const uint32_t box[3] = {64, static_cast<uint32_t>(nt), static_cast<uint32_t>(kp / 64)};
        if (int rc = encode_3d(&P.tm_b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, b_src, dims, strides, box,
                               CU_TENSOR_MAP_SWIZZLE_128B))
            return rc;
    }

    GemmParams& gp = P.gp;
    gp.tiles = at<const int4>(ws, light ? L.light_tiles : L.tiles);
    gp.n_tiles = at<const int>(ws, light ? L.n_light : L.n_tiles);
    gp.scales = wscales;
    gp.out = static_cast<__nv_bfloat16*>(out);
    gp.out_ld = static_cast<int>(w13 ? N : K);
    gp.rows_per_expert = static_cast<int>(rows_per_expert);
    gp.half_rows = static_cast<int>(N);
    gp.kred = static_cast<int>(kred);
    gp.ngroups = ngroups;
    gp.group = group;
    gp.mt_count = static_cast<int>(w13 ? N / 128 : K / 256);
    gp.kp = kp;
    gp.nt = nt;
    gp.nstage = sm.nstage;
    // TMEM (512 columns): nacc sets of n_issuers accumulators of nt columns,
    // then A buffers of 128 columns (2 or 3).  A thread can issue a tcgen05.mma
    // only every ~110 cycles, so small token tiles use 4 issuers (row block x
    // buffer parity) and large ones 2 (one per row block).  2-bit codes with
    // 16-token tiles take the group-accumulate mode: 6 issuers (row block x
    // group parity), 3 group slots of 32 columns, 3 A buffers.
    // group-accumulate mode: one A buffer per scale group (group == 128 k)
    gp.ga = (bits == 2 && nt == 16 && group == 128) ? 1 : 0;
    // offset codes when the caller provides the token corrections
    gp.csum = gp.ga ? csum : nullptr;
    if (gp.ga) {
        gp.n_issuers = 6;
        gp.nacc = 1;
        gp.nabuf = 3;   // A buffers (128 columns each) after the 128 columns of group slots
    } else {
        gp.n_issuers = nt <= 32 ? 4 : 2;
        gp.nacc = 2 * gp.n_issuers * nt + 2 * 128 <= 512 ? 2 : 1;
        const int acc_cols = gp.nacc * gp.n_issuers * nt;
        gp.nabuf = (512 - acc_cols) / 128 < 3 ? (512 - acc_cols) / 128 : 3;
    }
    gp.off_b = sm.off_b;
    gp.off_w = sm.off_w;
    gp.off_s = sm.off_s;
    gp.off_bar = sm.off_bar;
    gp.limit = limit;
    gp.status = at<int>(ws, L.status);
    gp.ksplit = ksplit;
    gp.partial = ksplit > 1 ? at<float>(ws, L.partial) : nullptr;
    // Prefill tiles: an expert's weights are read once per token tile of that
    // expert, by CTAs running at about the same time, so they are kept in L2
    // (evict-first made every tile re-read them from HBM); decode streams
    // each weight once.
    gp.w_reuse = nt >= 64 ? 1 : 0;
    // w2 reads the tile list written by the routing kernels, which ran before
    // the w13 GEMM; only its token operand (h) comes from the kernel before it
    gp.early_w = w13 ? 0 : 1;
    gp.partial_rows = static_cast<int>(L.R);
    gp.n_weight_rows = E * rows_per_expert;
    gp.h_interleaved = h_interleaved;
    // Prefill w13 split in two (the accumulation cap): the CTAs 2i and 2i + 1
    // of a launch with an even grid run the two splits of the same unit at the
    // same time; the second one's epilogue adds the first one's parked sums
    // (fresh in L2) to its own accumulator and writes h, so no finalize
    // kernel runs.  Only odd CTAs wait, and only on even ones.
    gp.fuse_splits = (w13 && ksplit == 2 && nt > 32) ? 1 : 0;
    gp.unit_flags = at<int>(ws, L.flags);
    // widest async copy that divides the scale row stride, one split's row
    // segment and the base alignment
    gp.scale_copy_bytes = 0;
    for (int c : {16, 8, 4}) {
        if ((ngroups * 2) % c == 0 && ((ngroups / ksplit) * 2) % c == 0 && aligned(wscales, c)) {
            gp.scale_copy_bytes = c;
            break;
        }
    }

    const int64_t max_items = max_units * ksplit;
    P.grid = static_cast<int>(max_items < dev.sms ? max_items : dev.sms);
    if (gp.fuse_splits) P.grid &= ~1;   // split parity = CTA parity (max_items is even)
    if (P.grid < 1) P.grid = 1;
    P.smem = sm.total;
    P.w13 = w13;
    P.bits = bits;
    return WNA16_OK;
}

int launch_plan(const GemmPlan& P, cudaStream_t s) {
    cudaError_t e = launch_grouped_gemm(P.bits, P.w13, P.tm_w, P.tm_b, P.gp, P.grid, P.smem, s);
    return e == cudaSuccess ? WNA16_OK : cuda_fail(e, "grouped GEMM launch");
}

}  // namespace

int wna16::set_error(int code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return code;
}

// ====================================================================== C ABI

extern "C" {

const char* wna16_moe_last_error(void) { return g_err; }

size_t wna16_moe_workspace_size(int64_t T, int64_t K, int64_t N, int64_t E, int topk, int bits) {
    if (check_dims(T, K, N, E, topk, bits) != WNA16_OK) return 0;
    return make_layout(T, K, N, E, topk, bits).total;
}

int wna16_moe_pack(const int8_t* codes, int64_t rows, int64_t K, int bits, int32_t* packed, void* stream) {
    g_err[0] = 0;
    if (bits != 2 && bits != 4) return fail(WNA16_ERR_UNSUPPORTED, "bits=%d: only 2 and 4 are supported", bits);
    if (rows < 0 || K <= 0 || K % (32 / bits))
        return fail(WNA16_ERR_INVALID_ARG, "K=%lld must be a positive multiple of %d", (long long)K, 32 / bits);
    if (rows == 0) return WNA16_OK;
    if (int rc = check_ptr(codes, 1, "codes")) return rc;
    if (int rc = check_ptr(packed, 4, "packed")) return rc;
    cudaError_t e = launch_pack(codes, rows, K, bits, packed, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? WNA16_OK : cuda_fail(e, "pack kernel launch");
}

int wna16_moe_read_status(const void* workspace, int* device_status, void* stream) {
    g_err[0] = 0;
    if (!workspace || !device_status) return fail(WNA16_ERR_INVALID_ARG, "NULL argument");
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    e = cudaMemcpy(device_status, workspace, sizeof(int), cudaMemcpyDeviceToHost);  // status is at offset 0
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy(status)");
    return WNA16_OK;
}

int wna16_moe_check_wait_timeout(void* workspace, size_t workspace_bytes, int64_t limit_us, void* stream) {
    g_err[0] = 0;
    if (!workspace || workspace_bytes < sizeof(int)) return fail(WNA16_ERR_INVALID_ARG, "workspace too small or NULL");
    if (limit_us <= 0 || limit_us > 5000000) return fail(WNA16_ERR_INVALID_ARG, "limit_us must be in (0, 5e6]");
    cudaError_t e = launch_wait_timeout_check(static_cast<int*>(workspace), static_cast<uint64_t>(limit_us) * 1000u,
                                              static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? WNA16_OK : cuda_fail(e, "wait check kernel launch");
}

}  // extern "C"

namespace {

// The forward over the local experts [e_begin, e_begin + E) of E_total (all
// of them on a single device): bf16 out, or with f32_out the fp32 partial
// output of that expert range.
int forward_impl(const void* x, const int32_t* topk_ids, const float* topk_weights, const int32_t* w13_packed,
                 const uint16_t* w13_scales, const int32_t* w2_packed, const uint16_t* w2_scales, int64_t T, int64_t K,
                 int64_t N, int64_t E, int64_t e_begin, int64_t E_total, int topk, int group_size, int group_size_w2,
                 int bits, float swiglu_limit, void* out, bool f32_out, void* workspace, size_t workspace_bytes,
                 void* stream) {
    g_err[0] = 0;
    if (int rc = check_dims(T, K, N, E, f32_out ? 1 : topk, bits)) return rc;
    if (topk <= 0) return fail(WNA16_ERR_INVALID_ARG, "topk=%d must be positive", topk);
    if (e_begin < 0 || E_total < E || e_begin > E_total - E || E_total >= (int64_t(1) << 31))
        return fail(WNA16_ERR_INVALID_ARG, "expert range [%lld, %lld) is not inside [0, %lld)", (long long)e_begin,
                    (long long)(e_begin + E), (long long)E_total);
    if (topk > E_total) return fail(WNA16_ERR_INVALID_ARG, "topk=%d exceeds E=%lld", topk, (long long)E_total);
    const int g2 = group_size_w2 ? group_size_w2 : group_size;
    if (int rc = check_group(group_size, K, "group_size")) return rc;
    if (int rc = check_group(g2, N, "group_size_w2")) return rc;
    if (!(swiglu_limit > 0.0f)) return fail(WNA16_ERR_INVALID_ARG, "swiglu_limit must be > 0 (or +inf)");
    if (T == 0) return WNA16_OK;
    if (int rc = check_ptr(x, 16, "x")) return rc;
    if (int rc = check_ptr(out, 16, "out")) return rc;
    if (T * topk >= (int64_t(1) << 31)) return fail(WNA16_ERR_UNSUPPORTED, "T*topk must be < 2^31");
    if (int rc = check_ptr(topk_ids, 4, "topk_ids")) return rc;
    if (int rc = check_ptr(topk_weights, 4, "topk_weights")) return rc;
    if (int rc = check_ptr(w13_packed, 16, "w13_packed")) return rc;
    if (int rc = check_ptr(w2_packed, 16, "w2_packed")) return rc;
    if (int rc = check_ptr(w13_scales, 2, "w13_scales")) return rc;
    if (int rc = check_ptr(w2_scales, 2, "w2_scales")) return rc;
    {
        const uintptr_t xb = reinterpret_cast<uintptr_t>(x), ob = reinterpret_cast<uintptr_t>(out);
        const uintptr_t xbytes = static_cast<uintptr_t>(T * K * 2);
        const uintptr_t obytes = static_cast<uintptr_t>(T * K * (f32_out ? 4 : 2));
        if (xb < ob + obytes && ob < xb + xbytes) return fail(WNA16_ERR_INVALID_ARG, "out overlaps x");
    }
    const Layout L = make_layout(T, K, N, E, topk, bits);
    if (int rc = check_workspace(workspace, workspace_bytes, L)) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    GemmPlan p13, p2;
    // The A operand's K order is interleaved (2-bit: 16-k blocks, 4-bit: 8-k
    // words): x is gathered and h is written in that order (w2's input); y and
    // out are not affected.
    const int il = bits == 2 ? 1 : 2;
    // Group-accumulate mode takes offset codes when the token operand's
    // corrections are written with it: by the gather for w13, by the split-K
    // finalize (which writes h) for w2.
    if (int rc = plan_gemm(p13, true, bits, w13_packed, w13_scales, at<void>(workspace, L.xp),
                           at<void>(workspace, L.h), K, N, E, group_size, swiglu_limit, L, workspace, il,
                           at<float>(workspace, L.csum13)))
        return rc;
    if (int rc = plan_gemm(p2, false, bits, w2_packed, w2_scales, at<void>(workspace, L.h), at<void>(workspace, L.y),
                           K, N, E, g2, swiglu_limit, L, workspace, false,
                           p13.gp.ksplit > 1 ? at<float>(workspace, L.csum2) : nullptr))
        return rc;
    // Light experts of 2-bit prefill batches: two more launches, group-
    // accumulate with plain codes over 8-row tiles and no K split, which write
    // their rows of h and y themselves. The light w13 runs after the main w13's
    // split-K finalize (which writes every row of h, the light ones from sums
    // nobody parked) and overwrites those rows; the main w2 must write y
    // itself (no split), since the combine reads every row of y. Kept only
    // when both light plans fit and take the group-accumulate mode.
    GemmPlan p13l, p2l;
    int light_max = 0;
    if (L.light_max > 0 && p2.gp.ksplit == 1) {
        if (plan_gemm(p13l, true, bits, w13_packed, w13_scales, at<void>(workspace, L.xp), at<void>(workspace, L.h), K,
                      N, E, group_size, swiglu_limit, L, workspace, il, nullptr, true) == WNA16_OK &&
            plan_gemm(p2l, false, bits, w2_packed, w2_scales, at<void>(workspace, L.h), at<void>(workspace, L.y), K,
                      N, E, g2, swiglu_limit, L, workspace, false, nullptr, true) == WNA16_OK &&
            p13l.gp.ga && p2l.gp.ga)
            light_max = L.light_max;
        g_err[0] = 0;   // a light plan that does not fit only leaves the light path out
    }

    mark(0, s);
    int launches = 0;
    cudaError_t e = cudaSuccess;
    if (L.R <= kSmallRouteMax) {
        // small batch: routing lists and gather in one kernel (the gather stage is folded into route)
        e = launch_route_gather_small(topk_ids, static_cast<int>(L.R), static_cast<int>(E), static_cast<int>(e_begin),
                                      static_cast<int>(E_total), L.tile_rows, topk, at<int>(workspace, L.counts),
                                      at<int>(workspace, L.offsets), at<int>(workspace, L.perm),
                                      at<int>(workspace, L.inv), at<int4>(workspace, L.tiles),
                                      at<int>(workspace, L.n_tiles), at<int>(workspace, L.status),
                                      static_cast<const __nv_bfloat16*>(x), static_cast<int>(K), il,
                                      at<__nv_bfloat16>(workspace, L.xp),
                                      p13.gp.csum ? at<float>(workspace, L.csum13) : nullptr,
                                      at<int>(workspace, L.flags), static_cast<int>(L.n_flags), s);
        if (e != cudaSuccess) return cuda_fail(e, "route/gather kernel launch");
        launches += 1;
        mark(1, s);
    } else {
        if (int rc = run_route(topk_ids, E, L, workspace, s, e_begin, E_total, light_max)) return rc;
        launches += route_chunks(static_cast<int>(L.R)) > 0 ? 3 : 1;
        mark(1, s);
        e = launch_gather(static_cast<const __nv_bfloat16*>(x), at<int>(workspace, L.inv), static_cast<int>(T), topk,
                          static_cast<int>(K), il, at<__nv_bfloat16>(workspace, L.xp),
                          p13.gp.csum ? at<float>(workspace, L.csum13) : nullptr, static_cast<int>(L.R),
                          at<int>(workspace, L.status), at<int>(workspace, L.flags), static_cast<int>(L.n_flags), s);
        if (e != cudaSuccess) return cuda_fail(e, "gather kernel launch");
        launches += 1;
    }
    mark(2, s);
    if (int rc = launch_plan(p13, s)) return rc;
    if (p13.gp.ksplit > 1 && !p13.gp.fuse_splits) {   // split K: fixed-order sum of the splits + SwiGLU -> h
        e = launch_finalize_w13(at<float>(workspace, L.partial), p13.gp.ksplit, static_cast<int>(L.R),
                                at<int>(workspace, L.offsets) + E, static_cast<int>(N), swiglu_limit, il,
                                at<__nv_bfloat16>(workspace, L.h), p2.gp.csum ? at<float>(workspace, L.csum2) : nullptr,
                                s);
        if (e != cudaSuccess) return cuda_fail(e, "finalize kernel launch");
    }
    if (light_max)
        if (int rc = launch_plan(p13l, s)) return rc;
    mark(3, s);
    if (int rc = launch_plan(p2, s)) return rc;
    if (light_max)
        if (int rc = launch_plan(p2l, s)) return rc;
    mark(4, s);
    if (p2.gp.ksplit > 1)      // split K: the combine adds the splits itself
        e = launch_combine_partials(at<float>(workspace, L.partial), p2.gp.ksplit, static_cast<int>(L.R), topk_weights,
                                    at<int>(workspace, L.inv), static_cast<int>(T), topk, static_cast<int>(K), out,
                                    f32_out, at<int>(workspace, L.status), s);
    else
        e = launch_combine(at<__nv_bfloat16>(workspace, L.y), topk_weights, at<int>(workspace, L.inv),
                           static_cast<int>(T), topk, static_cast<int>(K), out, f32_out, static_cast<int>(L.R),
                           at<int>(workspace, L.status), s);
    if (e != cudaSuccess) return cuda_fail(e, "combine kernel launch");
    mark(5, s);
    mark_done();
    // + w13 (+ finalize), w2, combine (+ the two light launches)
    g_launches = launches + 3 + (p13.gp.ksplit > 1 && !p13.gp.fuse_splits ? 1 : 0) + (light_max ? 2 : 0);
    return WNA16_OK;
}

}  // namespace

extern "C" {

int wna16_moe_forward(const void* x, const int32_t* topk_ids, const float* topk_weights, const int32_t* w13_packed,
                      const uint16_t* w13_scales, const int32_t* w2_packed, const uint16_t* w2_scales, int64_t T,
                      int64_t K, int64_t N, int64_t E, int topk, int group_size, int group_size_w2, int bits,
                      float swiglu_limit, void* out, void* workspace, size_t workspace_bytes, void* stream) {
    if (topk > E) {
        g_err[0] = 0;
        return fail(WNA16_ERR_INVALID_ARG, "topk=%d exceeds E=%lld", topk, (long long)E);
    }
    return forward_impl(x, topk_ids, topk_weights, w13_packed, w13_scales, w2_packed, w2_scales, T, K, N, E, 0, E,
                        topk, group_size, group_size_w2, bits, swiglu_limit, out, false, workspace, workspace_bytes,
                        stream);
}

int wna16_moe_forward_partial(const void* x, const int32_t* topk_ids, const float* topk_weights,
                              const int32_t* w13_packed, const uint16_t* w13_scales, const int32_t* w2_packed,
                              const uint16_t* w2_scales, int64_t T, int64_t K, int64_t N, int64_t E_total,
                              int64_t expert_begin, int64_t E_local, int topk, int group_size, int group_size_w2,
                              int bits, float swiglu_limit, float* out_partial, void* workspace,
                              size_t workspace_bytes, void* stream) {
    return forward_impl(x, topk_ids, topk_weights, w13_packed, w13_scales, w2_packed, w2_scales, T, K, N, E_local,
                        expert_begin, E_total, topk, group_size, group_size_w2, bits, swiglu_limit, out_partial, true,
                        workspace, workspace_bytes, stream);
}

int wna16_moe_route_topk(const float* logits, const float* bias, int64_t T, int64_t E, int topk, int32_t* topk_ids,
                         float* topk_weights, void* stream) {
    g_err[0] = 0;
    if (T < 0 || E <= 0) return fail(WNA16_ERR_INVALID_ARG, "T=%lld must be >= 0 and E=%lld > 0", (long long)T,
                                     (long long)E);
    if (E > 1024) return fail(WNA16_ERR_UNSUPPORTED, "E=%lld: at most 1024 experts", (long long)E);
    if (topk < 1 || topk > E || topk > 32)
        return fail(WNA16_ERR_INVALID_ARG, "topk=%d must be in [1, min(E, 32)]", topk);
    if (T * E >= (int64_t(1) << 40) || T >= (int64_t(1) << 31))
        return fail(WNA16_ERR_UNSUPPORTED, "T=%lld too large", (long long)T);
    if (T == 0) return WNA16_OK;
    if (int rc = check_ptr(logits, 4, "logits")) return rc;
    if (bias)
        if (int rc = check_ptr(bias, 4, "bias")) return rc;
    if (int rc = check_ptr(topk_ids, 4, "topk_ids")) return rc;
    if (int rc = check_ptr(topk_weights, 4, "topk_weights")) return rc;
    cudaError_t e = launch_route_topk(logits, bias, static_cast<int>(T), static_cast<int>(E), topk, topk_ids,
                                      topk_weights, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? WNA16_OK : cuda_fail(e, "router kernel launch");
}

int wna16_moe_quantize(const float* w, int64_t rows, int64_t K, const float* importance, int bits, int group_size,
                       int search, int32_t* packed, uint16_t* scales, double* metrics, void* stream) {
    g_err[0] = 0;
    if (bits != 2 && bits != 4) return fail(WNA16_ERR_UNSUPPORTED, "bits=%d: only 2 and 4 are supported", bits);
    if (rows < 0 || K <= 0) return fail(WNA16_ERR_INVALID_ARG, "rows=%lld must be >= 0 and K=%lld > 0",
                                        (long long)rows, (long long)K);
    if (group_size <= 0 || group_size % 32 || K % group_size)
        return fail(WNA16_ERR_UNSUPPORTED, "group_size=%d must be a multiple of 32 dividing K=%lld", group_size,
                    (long long)K);
    if (K / group_size > 128)
        return fail(WNA16_ERR_UNSUPPORTED, "K/group_size=%lld: at most 128 groups per row",
                    (long long)(K / group_size));
    if (K >= (int64_t(1) << 31) || rows * K >= (int64_t(1) << 62))
        return fail(WNA16_ERR_UNSUPPORTED, "sizes too large");
    if (search != 0 && search != 1) return fail(WNA16_ERR_INVALID_ARG, "search=%d must be 0 or 1", search);
    if (rows == 0) return WNA16_OK;
    if (int rc = check_ptr(w, 16, "w")) return rc;
    if (importance)
        if (int rc = check_ptr(importance, 16, "importance")) return rc;
    if (int rc = check_ptr(packed, 4, "packed")) return rc;
    if (int rc = check_ptr(scales, 2, "scales")) return rc;
    if (metrics)
        if (int rc = check_ptr(metrics, 8, "metrics")) return rc;
    cudaError_t e = launch_quantize(w, rows, static_cast<int>(K), importance, bits, group_size, search, packed, scales,
                                    metrics, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? WNA16_OK : cuda_fail(e, "quantize kernel launch");
}

int wna16_moe_launches_last_forward(void) { return g_launches; }

int wna16_moe_profile(int slots) {
    g_err[0] = 0;
    if (slots < 0 || slots > 65536) return fail(WNA16_ERR_INVALID_ARG, "slots=%d must be in [0, 65536]", slots);
    if (g_prof.ev) {
        for (int i = 0; i < g_prof.slots * 6; ++i) cudaEventDestroy(g_prof.ev[i]);
        delete[] g_prof.ev;
        g_prof.ev = nullptr;
    }
    g_prof.slots = 0;
    g_prof.next = 0;
    g_prof.recorded = 0;
    if (slots == 0) return WNA16_OK;
    g_prof.ev = new cudaEvent_t[static_cast<size_t>(slots) * 6];
    for (int i = 0; i < slots * 6; ++i) {
        cudaError_t e = cudaEventCreate(&g_prof.ev[i]);
        if (e != cudaSuccess) {
            for (int j = 0; j < i; ++j) cudaEventDestroy(g_prof.ev[j]);
            delete[] g_prof.ev;
            g_prof.ev = nullptr;
            return cuda_fail(e, "cudaEventCreate");
        }
    }
    g_prof.slots = slots;
    return WNA16_OK;
}

int wna16_moe_profile_read(float* ms, int n) {
    g_err[0] = 0;
    if (!ms || n <= 0) return fail(WNA16_ERR_INVALID_ARG, "ms is NULL or n <= 0");
    if (!g_prof.slots || n > g_prof.slots || n > g_prof.recorded)
        return fail(WNA16_ERR_INVALID_ARG, "only %lld profiled forwards available (ring of %d)", g_prof.recorded,
                    g_prof.slots);
    for (int f = 0; f < n; ++f) {
        const int slot = ((g_prof.next - n + f) % g_prof.slots + g_prof.slots) % g_prof.slots;
        cudaEvent_t* ev = g_prof.ev + slot * 6;
        cudaError_t e = cudaEventSynchronize(ev[5]);
        if (e != cudaSuccess) return cuda_fail(e, "cudaEventSynchronize");
        for (int i = 0; i < 5; ++i) {
            e = cudaEventElapsedTime(&ms[f * 5 + i], ev[i], ev[i + 1]);
            if (e != cudaSuccess) return cuda_fail(e, "cudaEventElapsedTime");
        }
    }
    return WNA16_OK;
}

int wna16_moe_route(const int32_t* topk_ids, int64_t T, int topk, int64_t E, int64_t K, int64_t N, int bits,
                    int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv, void* workspace,
                    size_t workspace_bytes, void* stream) {
    g_err[0] = 0;
    if (int rc = check_dims(T, K, N, E, topk, bits)) return rc;
    const Layout L = make_layout(T, K, N, E, topk, bits);
    if (int rc = check_workspace(workspace, workspace_bytes, L)) return rc;
    if (T > 0)
        if (int rc = check_ptr(topk_ids, 4, "topk_ids")) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (int rc = run_route(topk_ids, E, L, workspace, s)) return rc;
    struct {
        void* dst;
        size_t off, bytes;
    } copies[4] = {{counts, L.counts, sizeof(int) * E},
                   {offsets, L.offsets, sizeof(int) * (E + 1)},
                   {perm, L.perm, sizeof(int) * L.R},
                   {inv, L.inv, sizeof(int) * L.R}};
    for (auto& c : copies) {
        if (!c.dst || c.bytes == 0) continue;
        cudaError_t e = cudaMemcpyAsync(c.dst, at<char>(workspace, c.off), c.bytes, cudaMemcpyDeviceToDevice, s);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyAsync");
    }
    return WNA16_OK;
}

int wna16_moe_w13(const void* x, const int32_t* topk_ids, const int32_t* w13_packed, const uint16_t* w13_scales,
                  int64_t T, int64_t K, int64_t N, int64_t E, int topk, int group_size, int bits, float swiglu_limit,
                  void* h_out, void* workspace, size_t workspace_bytes, void* stream) {
    g_err[0] = 0;
    if (int rc = check_dims(T, K, N, E, topk, bits)) return rc;
    if (int rc = check_group(group_size, K, "group_size")) return rc;
    if (!(swiglu_limit > 0.0f)) return fail(WNA16_ERR_INVALID_ARG, "swiglu_limit must be > 0 (or +inf)");
    if (T == 0) return WNA16_OK;
    if (int rc = check_ptr(x, 16, "x")) return rc;
    if (int rc = check_ptr(h_out, 16, "h_out")) return rc;
    if (int rc = check_ptr(topk_ids, 4, "topk_ids")) return rc;
    if (int rc = check_ptr(w13_packed, 16, "w13_packed")) return rc;
    if (int rc = check_ptr(w13_scales, 2, "w13_scales")) return rc;
    const Layout L = make_layout(T, K, N, E, topk, bits);
    if (int rc = check_workspace(workspace, workspace_bytes, L)) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    GemmPlan p13;
    if (int rc = plan_gemm(p13, true, bits, w13_packed, w13_scales, at<void>(workspace, L.xp), h_out, K, N, E,
                           group_size, swiglu_limit, L, workspace, false, at<float>(workspace, L.csum13)))
        return rc;
    if (int rc = run_route(topk_ids, E, L, workspace, s)) return rc;
    cudaError_t e = launch_gather(static_cast<const __nv_bfloat16*>(x), at<int>(workspace, L.inv),
                                  static_cast<int>(T), topk, static_cast<int>(K), bits == 2 ? 1 : 2,
                                  at<__nv_bfloat16>(workspace, L.xp),
                                  p13.gp.csum ? at<float>(workspace, L.csum13) : nullptr, static_cast<int>(L.R),
                                  at<int>(workspace, L.status), at<int>(workspace, L.flags),
                                  static_cast<int>(L.n_flags), s);
    if (e != cudaSuccess) return cuda_fail(e, "gather kernel launch");
    if (int rc = launch_plan(p13, s)) return rc;
    if (p13.gp.ksplit > 1 && !p13.gp.fuse_splits) {
        e = launch_finalize_w13(at<float>(workspace, L.partial), p13.gp.ksplit, static_cast<int>(L.R),
                                at<int>(workspace, L.offsets) + E, static_cast<int>(N), swiglu_limit, 0,
                                static_cast<__nv_bfloat16*>(h_out), nullptr, s);
        if (e != cudaSuccess) return cuda_fail(e, "finalize kernel launch");
    }
    return WNA16_OK;
}

int wna16_moe_w2(const void* h, const int32_t* w2_packed, const uint16_t* w2_scales, int64_t T, int64_t K, int64_t N,
                 int64_t E, int topk, int group_size_w2, int bits, void* y_out, void* workspace,
                 size_t workspace_bytes, void* stream) {
    g_err[0] = 0;
    if (int rc = check_dims(T, K, N, E, topk, bits)) return rc;
    if (int rc = check_group(group_size_w2, N, "group_size_w2")) return rc;
    if (T == 0) return WNA16_OK;
    if (int rc = check_ptr(h, 16, "h")) return rc;
    if (int rc = check_ptr(y_out, 16, "y_out")) return rc;
    if (int rc = check_ptr(w2_packed, 16, "w2_packed")) return rc;
    if (int rc = check_ptr(w2_scales, 2, "w2_scales")) return rc;
    const Layout L = make_layout(T, K, N, E, topk, bits);
    if (int rc = check_workspace(workspace, workspace_bytes, L)) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const void* b_src = h;
    {   // the weights read h in the A operand's interleaved K order
        cudaError_t e = launch_interleave_rows(static_cast<const __nv_bfloat16*>(h), L.R, N, bits == 2 ? 1 : 2,
                                               at<__nv_bfloat16>(workspace, L.h), s);
        if (e != cudaSuccess) return cuda_fail(e, "interleave kernel launch");
        b_src = at<void>(workspace, L.h);
    }
    GemmPlan p2;
    if (int rc = plan_gemm(p2, false, bits, w2_packed, w2_scales, b_src, y_out, K, N, E, group_size_w2, INFINITY, L,
                           workspace))
        return rc;
    if (int rc = launch_plan(p2, s)) return rc;
    if (p2.gp.ksplit > 1) {
        cudaError_t e = launch_finalize_w2(at<float>(workspace, L.partial), p2.gp.ksplit, static_cast<int>(L.R),
                                           at<int>(workspace, L.offsets) + E, static_cast<int>(K),
                                           static_cast<__nv_bfloat16*>(y_out), s);
        if (e != cudaSuccess) return cuda_fail(e, "finalize kernel launch");
    }
    return WNA16_OK;
}

int wna16_moe_combine(const void* y, const float* topk_weights, int64_t T, int64_t K, int topk, int64_t E, int64_t N,
                      int bits, void* out, void* workspace, size_t workspace_bytes, void* stream) {
    g_err[0] = 0;
    if (int rc = check_dims(T, K, N, E, topk, bits)) return rc;
    if (T == 0) return WNA16_OK;
    if (int rc = check_ptr(y, 16, "y")) return rc;
    if (int rc = check_ptr(out, 16, "out")) return rc;
    if (int rc = check_ptr(topk_weights, 4, "topk_weights")) return rc;
    const Layout L = make_layout(T, K, N, E, topk, bits);
    if (int rc = check_workspace(workspace, workspace_bytes, L)) return rc;
    cudaError_t e = launch_combine(static_cast<const __nv_bfloat16*>(y), topk_weights, at<int>(workspace, L.inv),
                                   static_cast<int>(T), topk, static_cast<int>(K), out, false, static_cast<int>(L.R),
                                   at<int>(workspace, L.status), static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? WNA16_OK : cuda_fail(e, "combine kernel launch");
}

}  // extern "C"

// Quantiser: symmetric RTN with an importance-weighted scale search, the
// conversion step that produces the packed INT32 words and FP16 group scales
// the forward consumes (page "hampsonw/DeepSeek-V4-Flash-0731-WNA16", section
// "How it was created": symmetric 2-bit weights with group size 128 (step 2),
// the scale search weighted by a routed-expert activation importance vector
// (step 3), the signed codes packed (step 4), weighted and unweighted
// reconstruction error recorded (step 5); the same section's note that
// importance-weighted RTN was selected).
//
// Per row and group of g consecutive k (lo = -2^(b-1), hi = 2^(b-1) - 1):
//   m = max |w|, s0 = m / 2^(b-1);  candidate i = fp16(fp32(s0 * f_i)),
//   f_i = fp32((10 + i) / 20), i = 0..30 (plain RTN: i = 10 only);
//   code = clamp(rne(fp32(w / s)), lo, hi), what = bf16(code * s);
//   E(s) = sum_k a_k (w_k - what_k)^2 in fp64, k ascending;
//   the candidate of smallest E wins, ties to the lower i.
// The codes and the winning candidate are integer decisions taken on
// floating point: every step here is the IEEE operation the definition names
// (correctly rounded fp32 division, round-to-nearest-even, fp64 products and
// sums in the stated order, no contraction into fused multiply-adds), so the
// decisions are reproducible on any IEEE machine.
//
// One warp per row; lane l takes the groups l, l + 32, ... (at most 4 per
// lane).  Each lane streams its group once per pass with 16-byte loads; the 31
// candidate sums live in registers.  The row's metrics add the per-group sums
// in group order through warp shuffles.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "gemm.h"

namespace wna16 {

namespace {

constexpr int kCands = 31;
constexpr int kPlainCand = 10;
constexpr int kQuantWarpsPerBlock = 4;

__device__ __forceinline__ float cand_factor(int i) { return __fdiv_rn(static_cast<float>(10 + i), 20.0f); }

// fp32 code of w for scale s (clamped round-to-nearest-even of the IEEE quotient)
__device__ __forceinline__ float code_of(float w, float s, float lo, float hi) {
    return fminf(fmaxf(rintf(__fdiv_rn(w, s)), lo), hi);
}

// the forward's dequantised weight: bf16 of the exact product code * s
__device__ __forceinline__ double recon(float q, float s) {
    return static_cast<double>(__bfloat162float(__float2bfloat16_rn(__fmul_rn(q, s))));
}

// e + (a * d) * d, each operation rounded on its own
__device__ __forceinline__ double add_weighted_sq(double e, double a, double d) {
    return __dadd_rn(e, __dmul_rn(__dmul_rn(a, d), d));
}

template <int BITS>
__global__ void __launch_bounds__(32 * kQuantWarpsPerBlock)
    quantize_kernel(const float* __restrict__ w, int64_t rows, int K, const float* __restrict__ imp, int g, int search,
                    int32_t* __restrict__ packed, uint16_t* __restrict__ scales, double* __restrict__ metrics) {
    constexpr int kP = 32 / BITS;
    const float lo = -static_cast<float>(1 << (BITS - 1));
    const float hi = static_cast<float>((1 << (BITS - 1)) - 1);
    const int lane = threadIdx.x & 31;
    const int64_t row = static_cast<int64_t>(blockIdx.x) * kQuantWarpsPerBlock + (threadIdx.x >> 5);
    if (row >= rows) return;   // whole warps leave together
    const int groups = K / g;
    const float* wr = w + row * K;
    double gm[4][4];           // per own group: weighted err, unweighted err, sum a w^2, sum w^2
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int c = 0; c < 4; ++c) gm[j][c] = 0.0;

#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int gi = lane + 32 * j;
        if (gi >= groups) continue;
        const float4* wg = reinterpret_cast<const float4*>(wr + static_cast<int64_t>(gi) * g);
        const float4* ag = imp ? reinterpret_cast<const float4*>(imp + static_cast<int64_t>(gi) * g) : nullptr;
        // largest magnitude
        float m = 0.0f;
        for (int k4 = 0; k4 < g / 4; ++k4) {
            const float4 v = __ldg(wg + k4);
            m = fmaxf(m, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
        }
        float best_s = 0.0f;
        uint16_t best_h = 0;
        if (m > 0.0f) {
            const float s0 = __fdiv_rn(m, static_cast<float>(1 << (BITS - 1)));
            float cs[kCands];
            double ce[kCands];
#pragma unroll
            for (int i = 0; i < kCands; ++i) {
                cs[i] = __half2float(__float2half_rn(__fmul_rn(s0, cand_factor(i))));
                ce[i] = 0.0;
            }
            for (int k4 = 0; k4 < g / 4; ++k4) {
                const float4 v = __ldg(wg + k4);
                const float4 av = ag ? __ldg(ag + k4) : make_float4(1.f, 1.f, 1.f, 1.f);
                const float wv[4] = {v.x, v.y, v.z, v.w};
                const float aa[4] = {av.x, av.y, av.z, av.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const double wd = static_cast<double>(wv[e]);
                    const double ad = static_cast<double>(aa[e]);
                    if (search) {
#pragma unroll
                        for (int i = 0; i < kCands; ++i) {
                            if (!(cs[i] > 0.0f) || isinf(cs[i])) continue;
                            const double d = __dsub_rn(wd, recon(code_of(wv[e], cs[i], lo, hi), cs[i]));
                            ce[i] = add_weighted_sq(ce[i], ad, d);
                        }
                    } else if (cs[kPlainCand] > 0.0f && !isinf(cs[kPlainCand])) {
                        const double d = __dsub_rn(wd, recon(code_of(wv[e], cs[kPlainCand], lo, hi), cs[kPlainCand]));
                        ce[kPlainCand] = add_weighted_sq(ce[kPlainCand], ad, d);
                    }
                }
            }
            bool first = true;
            double best_e = 0.0;
#pragma unroll
            for (int i = 0; i < kCands; ++i) {
                if (!search && i != kPlainCand) continue;
                if (!(cs[i] > 0.0f) || isinf(cs[i])) continue;
                if (first || ce[i] < best_e) {
                    best_e = ce[i];
                    best_s = cs[i];
                    first = false;
                }
            }
            best_h = __half_as_ushort(__float2half_rn(best_s));
        }
        scales[row * groups + gi] = best_h;
        // codes, packed words and this group's metrics for the chosen scale
        int32_t* pw = packed + (row * K + static_cast<int64_t>(gi) * g) / kP;
        uint32_t word = 0;
        int field = 0;
        double e_w = 0.0, e_u = 0.0, s_aw = 0.0, s_w = 0.0;
        for (int k4 = 0; k4 < g / 4; ++k4) {
            const float4 v = __ldg(wg + k4);
            const float4 av = ag ? __ldg(ag + k4) : make_float4(1.f, 1.f, 1.f, 1.f);
            const float wv[4] = {v.x, v.y, v.z, v.w};
            const float aa[4] = {av.x, av.y, av.z, av.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float q = 0.0f;
                double what = 0.0;
                if (best_s > 0.0f) {
                    q = code_of(wv[e], best_s, lo, hi);
                    what = recon(q, best_s);
                }
                const uint32_t f = static_cast<uint32_t>(static_cast<int>(q) + (1 << (BITS - 1))) & ((1u << BITS) - 1u);
                word |= f << (BITS * field);
                if (++field == kP) {
                    *pw++ = static_cast<int32_t>(word);
                    word = 0;
                    field = 0;
                }
                const double wd = static_cast<double>(wv[e]);
                const double ad = static_cast<double>(aa[e]);
                const double d = __dsub_rn(wd, what);
                e_w = add_weighted_sq(e_w, ad, d);
                e_u = __dadd_rn(e_u, __dmul_rn(d, d));
                s_aw = add_weighted_sq(s_aw, ad, wd);
                s_w = __dadd_rn(s_w, __dmul_rn(wd, wd));
            }
        }
        gm[j][0] = e_w;
        gm[j][1] = e_u;
        gm[j][2] = s_aw;
        gm[j][3] = s_w;
    }
    if (!metrics) return;
    // the row's sums: group sums added in group order (group 32*j + l is lane l's slot j)
    double acc[4] = {0.0, 0.0, 0.0, 0.0};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        for (int l = 0; l < 32; ++l) {
            const bool valid = 32 * j + l < groups;   // warp-uniform
            if (!valid) break;
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[c] = __dadd_rn(acc[c], __shfl_sync(0xffffffffu, gm[j][c], l));
        }
    }
    if (lane < 4) metrics[row * 4 + lane] = lane == 0 ? acc[0] : lane == 1 ? acc[1] : lane == 2 ? acc[2] : acc[3];
}

}  // namespace

cudaError_t launch_quantize(const float* w, int64_t rows, int K, const float* importance, int bits, int g, int search,
                            int32_t* packed, uint16_t* scales, double* metrics, cudaStream_t stream) {
    if (rows == 0) return cudaSuccess;
    const int64_t blocks = (rows + kQuantWarpsPerBlock - 1) / kQuantWarpsPerBlock;
    if (blocks > 0x7FFFFFFF) return cudaErrorInvalidValue;
    const dim3 grid(static_cast<unsigned>(blocks)), block(32 * kQuantWarpsPerBlock);
    if (bits == 2)
        quantize_kernel<2><<<grid, block, 0, stream>>>(w, rows, K, importance, g, search, packed, scales, metrics);
    else
        quantize_kernel<4><<<grid, block, 0, stream>>>(w, rows, K, importance, g, search, packed, scales, metrics);
    return cudaGetLastError();
}

}  // namespace wna16

/*
 * CPU oracle for the WNA16 routed-expert MoE forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference leg of bench.py may load this library.  The CUDA
 * product path never calls, links or includes anything from this directory,
 * and this file shares no code, header, table or helper with that path.
 *
 * What it computes, step by step, in the plainest order (no tiling, no fusion):
 *
 *   1. unpack   INT32 words -> signed codes           (format: "compressed-tensors
 *               WNA16 format with FP16 group scales and INT32 packed values",
 *               hampsonw/DeepSeek-V4-Flash-0731-WNA16, section "What changed";
 *               "packed the signed codes with compressed-tensors",
 *               section "How it was created", step 4)
 *   2. dequant  W[n][k] = bf16_rne(code * scale[n][k / group])  (symmetric, no
 *               zero point, one FP16 scale per group of input-dim weights;
 *               same page, "What changed": "symmetric W2A16 quantization with
 *               group size 128")
 *   3. gather   each routed slot f = t*topk + j uses expert ids[t][j]
 *               ("indexed MoE", Incubate DeepSeek V4 WNA16 runtime on SM86,
 *               section "What this branch adds", item 3)
 *   4. w13      g = W1 x, u = W3 x with W1 = rows [0, N) and W3 = rows [N, 2N)
 *               of the fused gate/up tensor (same section, item 2)
 *   5. SwiGLU   h = bf16_rne( silu(min(g, L)) * clamp(u, -L, L) )  (same
 *               section, item 9: "SwiGLU alpha, beta, and clamp semantics";
 *               alpha = 1, beta = 0, L = swiglu_limit)
 *   6. w2       y = bf16_rne( W2 h )
 *   7. combine  out[t] = bf16_rne( sum_j  w[t][j] * y[t*topk + j] ), j ascending
 *
 * Readings of points the pages leave open:
 *   - in-word order: field j of a word holds element p*word + j at bits
 *     [b*j, b*j + b), least significant first;
 *   - stored field = code + 2^(b-1) (2-bit: code + 2, 4-bit: code + 8);
 *   - the group axis is the reduction (input) dim of each projection;
 *   - dequantised weights, h and y are rounded to BF16 (the operands the
 *     BF16 tensor cores consume); accumulation is exact-ish (fp64 by default,
 *     fp32 in the optional mode), each dot product in ascending k;
 *   - routing weights are applied in the combine, in fp32/fp64, j ascending.
 *
 * The only source of randomness is the inputs; nothing here draws numbers.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------ */
/* Planted mistakes, used only by the pin tests to show that each pin   */
/* catches a plausible bug.  0 = the correct oracle.                     */
/* ------------------------------------------------------------------ */
enum {
    MUT_NONE = 0,
    MUT_MSB_FIRST = 1,      /* unpack fields most-significant first            */
    MUT_CODE_OFFSET = 2,    /* subtract 2^(b-1) - 1 instead of 2^(b-1)          */
    MUT_GATE_UP_SWAP = 3,   /* use rows [N,2N) as gate and [0,N) as up          */
    MUT_NO_CLAMP = 4,       /* drop the SwiGLU clamp                            */
    MUT_GROUP_AXIS = 5,     /* index scales with (k % groups) instead of k/g    */
    MUT_W2_TRANSPOSE = 6,   /* read w2 as [N, K] instead of [K, N]              */
    MUT_NO_ROUTE_WEIGHT = 7,/* drop the routing weight in the combine           */
    MUT_UNSTABLE_PERM = 8,  /* emit each expert's slots in descending order     */
    MUT_SILU_SIGN = 9,      /* silu(z) = z / (1 + exp(z))                        */
    MUT_TOPK_TIE_HIGH = 10, /* router: equal scores go to the higher index       */
    MUT_TOPK_NO_RENORM = 11,/* router: weights left as full-softmax probabilities */
    MUT_TOPK_NO_BIAS = 12,  /* router: the bias is ignored                       */
    MUT_Q_NO_IMPORTANCE = 13,/* quantiser: the importance weights are ignored     */
    MUT_Q_CLAMP_HIGH = 14,  /* quantiser: codes clamped to 2^(b-1) (one too far) */
    MUT_LAST = 15
};
static int g_mutation = MUT_NONE;

int oracle_set_mutation(int m)
{
    if (m < 0 || m >= MUT_LAST) return -1;
    g_mutation = m;
    return 0;
}

/* ------------------------------------------------------------------ */
/* Number formats (written from the IEEE-754 definitions).               */
/* ------------------------------------------------------------------ */

/* IEEE binary16 -> double, exact. */
double oracle_fp16_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int exp = (h >> 10) & 0x1f;
    int man = h & 0x3ff;
    double v;
    if (exp == 0)
        v = ldexp((double)man, -24);                 /* subnormal or zero */
    else if (exp == 31)
        v = man ? NAN : INFINITY;
    else
        v = ldexp((double)(man | 0x400), exp - 25);  /* 1.man * 2^(exp-15) */
    return sign ? -v : v;
}

/* bfloat16 -> double, exact (bf16 is the top half of a binary32). */
double oracle_bf16_to_double(uint16_t b)
{
    uint32_t bits = (uint32_t)b << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* Round a real value (given as a double) to the nearest bfloat16, ties to
 * even, in ONE rounding step.  bfloat16 has 8 significant bits and the
 * binary32 exponent range (normal exponents -126..127, subnormals down to
 * 2^-133).  Overflow goes to infinity. */
uint16_t oracle_bf16_rne(double v)
{
    uint32_t bits;
    float f;
    if (isnan(v)) return 0x7fc0;
    if (v == 0.0) return signbit(v) ? 0x8000 : 0x0000;
    int neg = v < 0;
    double a = neg ? -v : v;
    if (isinf(a)) return neg ? 0xff80 : 0x7f80;
    int e;
    frexp(a, &e);                      /* a = m * 2^e, m in [0.5, 1) */
    int q = e - 8;                     /* quantum of an 8-bit significand */
    if (q < -133) q = -133;            /* subnormal bf16 quantum */
    double n = nearbyint(ldexp(a, -q)); /* default mode: to nearest, ties even */
    double r = ldexp(n, q);
    if (r > 0x1.fep127)                /* rounded beyond the largest finite bf16 */
        return neg ? 0xff80 : 0x7f80;
    f = (float)r;                      /* exact: r has <= 8 significant bits */
    memcpy(&bits, &f, sizeof bits);
    return (uint16_t)((bits >> 16) | (neg ? 0x8000u : 0u));
}

/* ------------------------------------------------------------------ */
/* Pack / unpack.                                                        */
/* ------------------------------------------------------------------ */

static int codes_per_word(int bits) { return 32 / bits; }

/* Signed code of element k of one packed row. */
static int unpack_one(const int32_t* row_words, int64_t k, int bits)
{
    int p = codes_per_word(bits);
    uint32_t w = (uint32_t)row_words[k / p];
    int j = (int)(k % p);
    if (g_mutation == MUT_MSB_FIRST) j = p - 1 - j;
    uint32_t field = (w >> (bits * j)) & ((1u << bits) - 1u);
    int offset = 1 << (bits - 1);
    if (g_mutation == MUT_CODE_OFFSET) offset -= 1;
    return (int)field - offset;
}

/* codes int8 [rows, K] (values in [-2^(b-1), 2^(b-1)) ) -> words [rows, K/p].
 * Returns 0, or -1 on a bad argument or an out-of-range code. */
int oracle_pack(const int8_t* codes, int64_t rows, int64_t K, int bits, int32_t* packed)
{
    if (bits != 2 && bits != 4) return -1;
    int p = codes_per_word(bits);
    if (K % p) return -1;
    int lo = -(1 << (bits - 1)), hi = (1 << (bits - 1)) - 1;
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t wi = 0; wi < K / p; ++wi) {
            uint32_t w = 0;
            for (int j = 0; j < p; ++j) {
                int c = codes[r * K + wi * p + j];
                if (c < lo || c > hi) return -1;
                uint32_t field = (uint32_t)(c - lo);
                w |= field << (bits * j);
            }
            packed[r * (K / p) + wi] = (int32_t)w;
        }
    }
    return 0;
}

int oracle_unpack(const int32_t* packed, int64_t rows, int64_t K, int bits, int8_t* codes)
{
    if (bits != 2 && bits != 4) return -1;
    int p = codes_per_word(bits);
    if (K % p) return -1;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t k = 0; k < K; ++k)
            codes[r * K + k] = (int8_t)unpack_one(packed + r * (K / p), k, bits);
    return 0;
}

/* ------------------------------------------------------------------ */
/* Dequantisation of whole rows (step 2).                                */
/* ------------------------------------------------------------------ */

static int64_t scale_index(int64_t k, int64_t group, int64_t n_groups)
{
    if (g_mutation == MUT_GROUP_AXIS) return k % n_groups;
    return k / group;
}

/* One row: packed words [K/p], scales fp16 [K/group] -> BF16 values as double. */
static void dequant_row(const int32_t* words, const uint16_t* scales, int64_t K,
                        int64_t group, int bits, double* out)
{
    int64_t n_groups = K / group;
    for (int64_t k = 0; k < K; ++k) {
        int code = unpack_one(words, k, bits);
        double s = oracle_fp16_to_double(scales[scale_index(k, group, n_groups)]);
        /* code * s is exact in double; a single RNE step gives the BF16 weight */
        out[k] = oracle_bf16_to_double(oracle_bf16_rne((double)code * s));
    }
}

/* Public: dequantise [rows, K] to BF16 bit patterns (for the dequant pins). */
int oracle_dequant(const int32_t* packed, const uint16_t* scales, int64_t rows, int64_t K,
                   int64_t group, int bits, uint16_t* out_bf16)
{
    if (bits != 2 && bits != 4) return -1;
    if (group <= 0 || K % group || K % codes_per_word(bits)) return -1;
    double* tmp = (double*)malloc(sizeof(double) * (size_t)K);
    if (!tmp) return -1;
    int p = codes_per_word(bits);
    for (int64_t r = 0; r < rows; ++r) {
        dequant_row(packed + r * (K / p), scales + r * (K / group), K, group, bits, tmp);
        for (int64_t k = 0; k < K; ++k) out_bf16[r * K + k] = oracle_bf16_rne(tmp[k]);
    }
    free(tmp);
    return 0;
}

/* ------------------------------------------------------------------ */
/* Routing lists (the "indexed" gather): counts, offsets, stable perm.    */
/* ------------------------------------------------------------------ */

/* ids int32 [R] (R = T*topk, flat slot f = t*topk + j).
 * counts [E]; offsets [E+1] exclusive prefix; perm [R]: slots sorted by
 * (expert, slot) ascending; inv [R]: inv[perm[i]] = i.
 * Returns 0, or -1 if an id is outside [0, E). */
int oracle_route(const int32_t* ids, int64_t R, int64_t E, int32_t* counts,
                 int32_t* offsets, int32_t* perm, int32_t* inv)
{
    for (int64_t e = 0; e < E; ++e) counts[e] = 0;
    for (int64_t f = 0; f < R; ++f) {
        if (ids[f] < 0 || ids[f] >= E) return -1;
        counts[ids[f]]++;
    }
    offsets[0] = 0;
    for (int64_t e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
    /* counting sort, one expert at a time, slots visited in ascending order */
    for (int64_t e = 0; e < E; ++e) {
        int32_t pos = offsets[e];
        if (g_mutation == MUT_UNSTABLE_PERM) {
            for (int64_t f = R - 1; f >= 0; --f)
                if (ids[f] == e) perm[pos++] = (int32_t)f;
        } else {
            for (int64_t f = 0; f < R; ++f)
                if (ids[f] == e) perm[pos++] = (int32_t)f;
        }
    }
    for (int64_t i = 0; i < R; ++i) inv[perm[i]] = (int32_t)i;
    return 0;
}

/* ------------------------------------------------------------------ */
/* The forward.                                                          */
/* ------------------------------------------------------------------ */

static double silu(double z)
{
    if (g_mutation == MUT_SILU_SIGN) return z / (1.0 + exp(z));
    return z / (1.0 + exp(-z));
}

static float silu_f(float z)
{
    if (g_mutation == MUT_SILU_SIGN) return z / (1.0f + expf(z));
    return z / (1.0f + expf(-z));
}

/* Clamped SwiGLU with limit L (L = +inf: no clamp). */
static double swiglu(double g, double u, double L)
{
    if (g_mutation != MUT_NO_CLAMP) {
        g = g < L ? g : L;             /* gate: clamped from above only */
        u = u < -L ? -L : (u > L ? L : u);
    }
    return silu(g) * u;
}

static float swiglu_f(float g, float u, float L)
{
    if (g_mutation != MUT_NO_CLAMP) {
        g = g < L ? g : L;
        u = u < -L ? -L : (u > L ? L : u);
    }
    return silu_f(g) * u;
}

/*
 * x        bf16 [T, K]          activations
 * ids      int32 [T, topk]      expert of each slot
 * wts      fp32 [T, topk]       routing weight of each slot
 * w13p     int32 [E, 2N, K/p]   fused gate/up codes; rows [0,N) gate, [N,2N) up
 * w13s     fp16  [E, 2N, K/g13]
 * w2p      int32 [E, K, N/p]    down codes
 * w2s      fp16  [E, K, N/g2]
 * accum    0: fp64 dot products and combine; 1: fp32 (ascending order)
 * tokens   optional list of n_tok token indices to evaluate (NULL: all T)
 * h_in     optional bf16 [n_tok*topk, N] (slot order): when given, steps 4 and 5
 *          are skipped and these values are h (to run steps 6 and 7 on an h
 *          computed elsewhere)
 * out      bf16 [n_tok, K]
 * h_out    optional bf16 [n_tok*topk, N]  (slot order t*topk + j)
 * y_out    optional bf16 [n_tok*topk, K]
 * Returns 0, or -1 on a bad argument / out-of-range expert id.
 */
int oracle_forward(const uint16_t* x, const int32_t* ids, const float* wts,
                   const int32_t* w13p, const uint16_t* w13s,
                   const int32_t* w2p, const uint16_t* w2s,
                   int64_t T, int64_t K, int64_t N, int64_t E, int topk,
                   int64_t g13, int64_t g2, int bits, float swiglu_limit, int accum,
                   const int64_t* tokens, int64_t n_tok, const uint16_t* h_in,
                   uint16_t* out, uint16_t* h_out, uint16_t* y_out)
{
    if (bits != 2 && bits != 4) return -1;
    int p = codes_per_word(bits);
    if (K % p || N % p || g13 <= 0 || g2 <= 0 || K % g13 || N % g2 || topk <= 0) return -1;
    if (!tokens) n_tok = T;
    for (int64_t i = 0; i < n_tok; ++i) {
        int64_t t = tokens ? tokens[i] : i;
        if (t < 0 || t >= T) return -1;
        for (int j = 0; j < topk; ++j)
            if (ids[t * topk + j] < 0 || ids[t * topk + j] >= E) return -1;
    }
    const double L = (double)swiglu_limit;
    const int64_t R = n_tok * topk;

    /* Slots of the selected tokens, grouped by expert only so that each
     * expert's weights are dequantised once; every output element is still
     * one dot product in ascending order, so the result does not depend on
     * this grouping or on the thread count. */
    double* W13 = (double*)malloc(sizeof(double) * (size_t)(2 * N * K));
    double* W2 = (double*)malloc(sizeof(double) * (size_t)(K * N));
    double* hbuf = (double*)malloc(sizeof(double) * (size_t)(R * N)); /* bf16 values */
    double* ybuf = (double*)malloc(sizeof(double) * (size_t)(R * K)); /* bf16 values */
    double* xrow = (double*)malloc(sizeof(double) * (size_t)(n_tok * K));
    if (!W13 || !W2 || !hbuf || !ybuf || !xrow) {
        free(W13); free(W2); free(hbuf); free(ybuf); free(xrow);
        return -1;
    }
    for (int64_t i = 0; i < n_tok; ++i) {
        int64_t t = tokens ? tokens[i] : i;
        for (int64_t k = 0; k < K; ++k) xrow[i * K + k] = oracle_bf16_to_double(x[t * K + k]);
    }

    for (int64_t e = 0; e < E; ++e) {
        int used = 0;
        for (int64_t s = 0; s < R && !used; ++s) {
            int64_t t = tokens ? tokens[s / topk] : s / topk;
            used = ids[t * topk + s % topk] == e;
        }
        if (!used) continue;

        /* step 2 for this expert */
        #pragma omp parallel for schedule(static)
        for (int64_t r = 0; r < (h_in ? 0 : 2 * N); ++r)
            dequant_row(w13p + (e * 2 * N + r) * (K / p), w13s + (e * 2 * N + r) * (K / g13),
                        K, g13, bits, W13 + r * K);
        #pragma omp parallel for schedule(static)
        for (int64_t m = 0; m < K; ++m)
            dequant_row(w2p + (e * K + m) * (N / p), w2s + (e * K + m) * (N / g2),
                        N, g2, bits, W2 + m * N);

        for (int64_t s = 0; s < R; ++s) {
            int64_t i = s / topk;
            int64_t t = tokens ? tokens[i] : i;
            if (ids[t * topk + s % topk] != e) continue;
            const double* xs = xrow + i * K;
            int64_t gate0 = 0, up0 = N;
            if (g_mutation == MUT_GATE_UP_SWAP) { gate0 = N; up0 = 0; }

            /* steps 4 and 5: h = swiglu(W1 x, W3 x), rounded to bf16 */
            #pragma omp parallel for schedule(static)
            for (int64_t n = 0; n < N; ++n) {
                if (h_in) {
                    hbuf[s * N + n] = oracle_bf16_to_double(h_in[s * N + n]);
                    continue;
                }
                const double* w1 = W13 + (gate0 + n) * K;
                const double* w3 = W13 + (up0 + n) * K;
                if (accum == 0) {
                    double g = 0.0, u = 0.0;
                    for (int64_t k = 0; k < K; ++k) { g += w1[k] * xs[k]; u += w3[k] * xs[k]; }
                    hbuf[s * N + n] = oracle_bf16_to_double(oracle_bf16_rne(swiglu(g, u, L)));
                } else {
                    float g = 0.0f, u = 0.0f;
                    for (int64_t k = 0; k < K; ++k) {
                        g += (float)w1[k] * (float)xs[k];
                        u += (float)w3[k] * (float)xs[k];
                    }
                    hbuf[s * N + n] = oracle_bf16_to_double(
                        oracle_bf16_rne((double)swiglu_f(g, u, (float)L)));
                }
            }
            /* step 6: y = W2 h, rounded to bf16 */
            #pragma omp parallel for schedule(static)
            for (int64_t m = 0; m < K; ++m) {
                const double* hs = hbuf + s * N;
                if (accum == 0) {
                    double acc = 0.0;
                    if (g_mutation == MUT_W2_TRANSPOSE) {
                        /* reads the [K, N] tensor as if it were [N, K] */
                        for (int64_t n = 0; n < N; ++n) acc += W2[n * K + m] * hs[n];
                    } else {
                        for (int64_t n = 0; n < N; ++n) acc += W2[m * N + n] * hs[n];
                    }
                    ybuf[s * K + m] = oracle_bf16_to_double(oracle_bf16_rne(acc));
                } else {
                    float acc = 0.0f;
                    for (int64_t n = 0; n < N; ++n) acc += (float)W2[m * N + n] * (float)hs[n];
                    ybuf[s * K + m] = oracle_bf16_to_double(oracle_bf16_rne((double)acc));
                }
            }
        }
    }

    /* step 7: combine, j ascending */
    for (int64_t i = 0; i < n_tok; ++i) {
        int64_t t = tokens ? tokens[i] : i;
        for (int64_t m = 0; m < K; ++m) {
            if (accum == 0) {
                double acc = 0.0;
                for (int j = 0; j < topk; ++j) {
                    double wj = g_mutation == MUT_NO_ROUTE_WEIGHT ? 1.0 : (double)wts[t * topk + j];
                    acc += wj * ybuf[(i * topk + j) * K + m];
                }
                out[i * K + m] = oracle_bf16_rne(acc);
            } else {
                float acc = 0.0f;
                for (int j = 0; j < topk; ++j) {
                    float wj = g_mutation == MUT_NO_ROUTE_WEIGHT ? 1.0f : wts[t * topk + j];
                    acc += wj * (float)ybuf[(i * topk + j) * K + m];
                }
                out[i * K + m] = oracle_bf16_rne((double)acc);
            }
        }
    }
    if (h_out)
        for (int64_t q = 0; q < R * N; ++q) h_out[q] = oracle_bf16_rne(hbuf[q]);
    if (y_out)
        for (int64_t q = 0; q < R * K; ++q) y_out[q] = oracle_bf16_rne(ybuf[q]);

    free(W13); free(W2); free(hbuf); free(ybuf); free(xrow);
    return 0;
}

/* ------------------------------------------------------------------ */
/* Quantiser: symmetric RTN with an importance-weighted scale search.    */
/* ------------------------------------------------------------------ */

/* binary16 bit pattern of the nearest fp16 to a double, ties to even (one
 * rounding; overflow to infinity). */
uint16_t oracle_fp16_rne(double v)
{
    if (isnan(v)) return 0x7e00;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (a == 0.0) return sign;
    int e;
    frexp(a, &e);                       /* a = m * 2^e, m in [0.5, 1) */
    int q = e - 11;                     /* quantum of an 11-bit significand */
    if (q < -24) q = -24;               /* subnormal quantum */
    double n = nearbyint(ldexp(a, -q));
    double r = ldexp(n, q);
    if (r >= 65520.0) return sign | 0x7c00;   /* beyond the largest finite half (65504) after rounding */
    if (r < ldexp(1.0, -14))                   /* subnormal: mantissa = r / 2^-24 */
        return sign | (uint16_t)(r * 16777216.0);
    int ee;
    double m = frexp(r, &ee);           /* r = m * 2^ee, m in [0.5, 1) */
    uint16_t man = (uint16_t)(ldexp(m, 11) - 1024.0);
    return sign | (uint16_t)((ee + 14) << 10) | man;
}

/*
 * The quantiser that produces the packed words and FP16 scales the forward
 * consumes, following the conversion the weight-format page describes
 * ("hampsonw/DeepSeek-V4-Flash-0731-WNA16", section "How it was created":
 * symmetric b-bit weights fitted with group size 128 (step 2), the scale
 * search weighted by a routed-expert activation importance vector (step 3),
 * signed codes packed (step 4), weighted and unweighted reconstruction error
 * recorded (step 5); "imatrix-weighted RTN").  Per row and group of g
 * consecutive k, with lo = -2^(b-1), hi = 2^(b-1) - 1:
 *
 *   m      = max |w_k|
 *   s0     = m / 2^(b-1)                 the largest magnitude lands on lo
 *   cand i = fp16( fp32(s0 * f_i) ),  f_i = fp32((10 + i) / 20), i = 0..30
 *            (f from 0.5 to 2.0 in steps of 0.05; f_10 = 1 is plain RTN);
 *            search = 0 tries f_10 only
 *   code_k = clamp( rne( fp32(w_k / s) ), lo, hi )     for a candidate s
 *   what_k = bf16( code_k * s )                        the forward's dequantisation
 *   E(s)   = sum_k a_k (w_k - what_k)^2    fp64, k ascending (a = 1 without importance)
 *   chosen = the candidate of smallest E; ties to the lower i
 *
 * A group whose largest magnitude is 0 gets scale 0 and codes 0.  The codes
 * and the candidate are integer decisions taken on fp32 divisions and fp64
 * sums that the kernel performs in the same precision and order.
 *
 * w fp32 [rows, K]; importance fp32 [K] or NULL; packed int32 [rows, K/p];
 * scales fp16 bits [rows, K/g]; metrics fp64 [rows, 4] or NULL: per row,
 * sum a (w - what)^2, sum (w - what)^2, sum a w^2, sum w^2, each summed per
 * group (k ascending, fp64) and the group sums added in group order.
 * Returns 0, or -1 on a bad argument.
 */
int oracle_quantize(const float* w, int64_t rows, int64_t K, const float* importance, int bits, int64_t g,
                    int search, int32_t* packed, uint16_t* scales, double* metrics)
{
    if ((bits != 2 && bits != 4) || g <= 0 || K % g || g % codes_per_word(bits) || rows < 0) return -1;
    const int p = codes_per_word(bits);
    const int lo = -(1 << (bits - 1));
    const int hi = (1 << (bits - 1)) - 1 + (g_mutation == MUT_Q_CLAMP_HIGH ? 1 : 0);
    const int64_t groups = K / g;
    int8_t* codes = (int8_t*)malloc((size_t)K);
    if (!codes) return -1;
    for (int64_t r = 0; r < rows; ++r) {
        const float* wr = w + r * K;
        double row_ew = 0.0, row_eu = 0.0, row_aw = 0.0, row_w = 0.0;
        for (int64_t gi = 0; gi < groups; ++gi) {
            const float* wg = wr + gi * g;
            float m = 0.0f;
            for (int64_t k = 0; k < g; ++k) {
                float a = fabsf(wg[k]);
                if (a > m) m = a;
            }
            float best_s = 0.0f;
            if (m > 0.0f) {
                const float s0 = m / (float)(1 << (bits - 1));
                double best_e = 0.0;
                int first = 1;
                for (int i = 0; i <= 30; ++i) {
                    if (!search && i != 10) continue;
                    const float f = (float)(10 + i) / 20.0f;
                    const float prod = s0 * f;
                    const uint16_t sh = oracle_fp16_rne((double)prod);
                    const float s = (float)oracle_fp16_to_double(sh);
                    if (!(s > 0.0f) || isinf(s)) continue;
                    double e = 0.0;
                    for (int64_t k = 0; k < g; ++k) {
                        float qf = nearbyintf(wg[k] / s);
                        if (qf < (float)lo) qf = (float)lo;
                        if (qf > (float)hi) qf = (float)hi;
                        const double what = oracle_bf16_to_double(oracle_bf16_rne((double)qf * (double)s));
                        const double d = (double)wg[k] - what;
                        const double a = (importance && g_mutation != MUT_Q_NO_IMPORTANCE)
                                             ? (double)importance[gi * g + k] : 1.0;
                        e = e + (a * d) * d;
                    }
                    if (first || e < best_e) {
                        best_e = e;
                        best_s = s;
                        first = 0;
                    }
                }
            }
            scales[r * groups + gi] = oracle_fp16_rne((double)best_s);
            /* codes, reconstruction and the group's metrics for the chosen scale */
            double gew = 0.0, geu = 0.0, gaw = 0.0, gw = 0.0;
            for (int64_t k = 0; k < g; ++k) {
                int c = 0;
                double what = 0.0;
                if (best_s > 0.0f) {
                    float qf = nearbyintf(wg[k] / best_s);
                    if (qf < (float)lo) qf = (float)lo;
                    if (qf > (float)hi) qf = (float)hi;
                    c = (int)qf;
                    what = oracle_bf16_to_double(oracle_bf16_rne((double)qf * (double)best_s));
                }
                codes[gi * g + k] = (int8_t)c;
                const double d = (double)wg[k] - what;
                const double a = importance ? (double)importance[gi * g + k] : 1.0;
                gew = gew + (a * d) * d;
                geu = geu + d * d;
                gaw = gaw + (a * (double)wg[k]) * (double)wg[k];
                gw = gw + (double)wg[k] * (double)wg[k];
            }
            row_ew = row_ew + gew;
            row_eu = row_eu + geu;
            row_aw = row_aw + gaw;
            row_w = row_w + gw;
        }
        /* pack: field j of word i holds code p*i + j + 2^(b-1) at bits [b*j, b*j + b) */
        for (int64_t wi = 0; wi < K / p; ++wi) {
            uint32_t word = 0;
            for (int j = 0; j < p; ++j)
                word |= ((uint32_t)(codes[wi * p + j] - lo) & ((1u << bits) - 1u)) << (bits * j);
            packed[r * (K / p) + wi] = (int32_t)word;
        }
        if (metrics) {
            metrics[r * 4 + 0] = row_ew;
            metrics[r * 4 + 1] = row_eu;
            metrics[r * 4 + 2] = row_aw;
            metrics[r * 4 + 3] = row_w;
        }
    }
    free(codes);
    return 0;
}

/* ------------------------------------------------------------------ */
/* Expert-parallel profile: partial outputs per expert range, summed in   */
/* rank order.                                                           */
/* ------------------------------------------------------------------ */

/*
 * When the experts are split across ranks (each rank holds the experts
 * [e_begin, e_end) and runs the path on them alone), rank r's combine covers
 * only the slots routed to its experts and is kept in fp32 for the reduction
 * across ranks:
 *
 *   partial_r[t][m] = fp32( sum_{j ascending, e_begin <= ids[t][j] < e_end} w[t][j] * y[t*topk+j][m] )
 *   out[t][m]       = bf16( (((partial_0 + partial_1) + partial_2) + ...) )   each + in fp32
 *
 * y is the BF16 down-projection output of step 6 (computed per slot, here
 * given as BF16 bits [n*topk, K]); the partial sum is fp64, rounded once to
 * fp32.  This changes one rounding point of the single-device combine (the
 * fp32 partials before the final BF16 rounding), so it is its own profile.
 * ids/wts [n, topk]; partial fp32 [n, K].
 */
int oracle_combine_partial(const int32_t* ids, const float* wts, const uint16_t* y, int64_t n, int64_t K,
                           int topk, int64_t e_begin, int64_t e_end, float* partial)
{
    if (n < 0 || K <= 0 || topk <= 0 || e_begin > e_end) return -1;
    for (int64_t t = 0; t < n; ++t)
        for (int64_t m = 0; m < K; ++m) {
            double acc = 0.0;
            for (int j = 0; j < topk; ++j) {
                int32_t e = ids[t * topk + j];
                if (e < e_begin || e >= e_end) continue;
                acc += (double)wts[t * topk + j] * oracle_bf16_to_double(y[(t * topk + j) * K + m]);
            }
            partial[t * K + m] = (float)acc;
        }
    return 0;
}

/* out = bf16( partial_0 + partial_1 + ... ) with the ranks added in order in
 * fp32; partials fp32 [P][count]. */
int oracle_sum_partials(const float* partials, int P, int64_t count, uint16_t* out)
{
    if (P <= 0 || count < 0) return -1;
    for (int64_t q = 0; q < count; ++q) {
        float s = partials[q];
        for (int r = 1; r < P; ++r) s = s + partials[(int64_t)r * count + q];
        out[q] = oracle_bf16_rne((double)s);
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* Router: softmax over the experts, top-k, renormalisation.             */
/* ------------------------------------------------------------------ */

/*
 * The routing that produces topk_ids / topk_weights from router logits, in
 * the order the workload description gives it ("top-k softmax routing from
 * N(0,1) logits", renormalised; the popularity skew enters as a logit bias):
 *
 *   z_e   = fp32( logits[t][e] + bias[e] )             (bias optional)
 *   p_e   = exp(z_e - max z) / sum_e' exp(z_e' - max z)  softmax, fp64
 *   ids   = the k experts of largest p, in descending order; equal values
 *           go to the lower expert index
 *   w_j   = fp32( p_ids[j] / sum_i p_ids[i] )          renormalised, fp64
 *
 * Which experts are chosen is an integer decision taken on floating point,
 * so it is taken on z itself, in the fp32 that both this definition and the
 * kernel compute it in: exp is increasing and the softmax denominator is
 * shared, so the order of p is the order of z (exactly so while the fp64
 * exponentials do not underflow, i.e. while the logits span less than about
 * 700).
 *
 * logits fp32 [T, E]; bias fp32 [E] or NULL; ids int32 [T, k]; weights fp32
 * [T, k].  Returns 0, or -1 on a bad argument (k outside [1, E]).
 */
int oracle_route_topk(const float* logits, const float* bias, int64_t T, int64_t E, int k,
                      int32_t* ids, float* weights)
{
    if (T < 0 || E <= 0 || k < 1 || k > E) return -1;
    float* z = (float*)malloc(sizeof(float) * (size_t)E);
    double* p = (double*)malloc(sizeof(double) * (size_t)E);
    unsigned char* taken = (unsigned char*)malloc((size_t)E);
    if (!z || !p || !taken) {
        free(z); free(p); free(taken);
        return -1;
    }
    for (int64_t t = 0; t < T; ++t) {
        /* scores */
        for (int64_t e = 0; e < E; ++e) {
            float b = (bias && g_mutation != MUT_TOPK_NO_BIAS) ? bias[e] : 0.0f;
            z[e] = logits[t * E + e] + b;      /* one fp32 addition */
        }
        /* softmax */
        double zmax = z[0];
        for (int64_t e = 1; e < E; ++e)
            if (z[e] > zmax) zmax = z[e];
        double denom = 0.0;
        for (int64_t e = 0; e < E; ++e) {
            p[e] = exp((double)z[e] - zmax);
            denom += p[e];
        }
        for (int64_t e = 0; e < E; ++e) p[e] /= denom;
        /* top-k */
        memset(taken, 0, (size_t)E);
        for (int j = 0; j < k; ++j) {
            int64_t best = -1;
            for (int64_t e = 0; e < E; ++e) {
                if (taken[e]) continue;
                if (best < 0 || z[e] > z[best] ||
                    (g_mutation == MUT_TOPK_TIE_HIGH && z[e] == z[best]))
                    best = e;
            }
            taken[best] = 1;
            ids[t * k + j] = (int32_t)best;
        }
        /* renormalisation over the chosen k */
        double sel = 0.0;
        for (int j = 0; j < k; ++j) sel += p[ids[t * k + j]];
        for (int j = 0; j < k; ++j) {
            double w = g_mutation == MUT_TOPK_NO_RENORM ? p[ids[t * k + j]] : p[ids[t * k + j]] / sel;
            weights[t * k + j] = (float)w;
        }
    }
    free(z); free(p); free(taken);
    return 0;
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

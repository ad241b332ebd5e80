/*
 * oracle.c -- plain, slow CPU oracle for the FP8 block-scaled linear layer of
 * DeepSeek-V3 inference.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call this file:
 * only the tests, the smoke check and the CPU-baseline leg of the benchmark
 * load it.  It shares no code, header, table or constant with the CUDA
 * library; it is written from the statement of the method on these pages:
 *
 *   [DF]  "Data flow -- deepseek-ai/DeepSeek-V3" (codevetter.com), bullet
 *         "FP8 quantization data flow": act_quant yields an e4m3 tensor plus
 *         one fp32 scale per 128-element block; fp8_gemm multiplies the scaled
 *         blocks and accumulates in fp32; weights carry a .scale grid.
 *   [BT]  "Behavior traces -- deepseek-ai/DeepSeek-V3" (codevetter.com),
 *         bullets "MoE trace" (y[idx] += expert(x[idx]) * weight) and
 *         "fp8->bf16 trace" (weight_dequant of each 1-byte tensor).
 *   [TOUR] "DeepSeek-V3" source tour (pyshine.com), section "The Three Ideas
 *         That Make V3 Fast", paragraph "FP8 with per-block scales": each
 *         128-element tile's max is clamped and divided by 448 (the e4m3
 *         ceiling); weights are e4m3 with a scale grid of 128-element blocks;
 *         the GEMM rescales FP8 products by their block scales.
 *
 * Readings of points the pages leave open (each is restated where used):
 *   R1  the clamp is a floor on amax of 1e-4 (an all-zero block gets a
 *       positive scale and all-zero codes);
 *   R2  amax/448 and x/s are IEEE fp32 divisions rounded to nearest;
 *   R3  fp32 -> e4m3 rounds to nearest, ties to even, and saturates finite
 *       values beyond +-448 to +-448;
 *   R4  scale_fmt "ue8m0": the fp32 scale is replaced by the smallest power
 *       of two that is >= it (the scale is still stored as fp32);
 *   R5  weights are [N, K] (y = x W^T), their scales [ceil(N/128), K/128];
 *       activation scales are [M, K/128]; a scale multiplies to dequantise;
 *   R6  the GEMM result is the exact block-scaled sum (fp32 accumulation is
 *       the kernel's business; here it is carried in double).
 *
 * Floating point is carried in double except where a reading fixes fp32.
 * Build flags must keep IEEE semantics: -O2 -ffp-contract=off, no fast-math.
 */
#include <stdint.h>
#include <string.h>
#include <math.h>

#define ORACLE_BLOCK 128          /* [TOUR] 128-element blocks */
#define ORACLE_E4M3_MAX 448.0f    /* [TOUR] the e4m3 ceiling */
#define ORACLE_AMAX_FLOOR 1e-4f   /* R1 */

/* ------------------------------------------------------------------ */
/* Number formats                                                       */
/* ------------------------------------------------------------------ */

/* float8_e4m3fn: sign | 4 exponent bits (bias 7) | 3 mantissa bits.
 * Exponent field 0 holds the subnormals m/8 * 2^-6; the bit pattern
 * S.1111.111 is NaN; there is no infinity.  Largest finite: 1.75 * 2^8. */
double oracle_e4m3_decode(uint8_t code)
{
    int sign = (code >> 7) & 1;
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    double mag;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        mag = ldexp((double)m, -9);              /* (m/8) * 2^(1-7) */
    else
        mag = ldexp((double)(8 + m), e - 10);    /* (1 + m/8) * 2^(e-7) */
    return sign ? -mag : mag;
}

/* The 256 decoded values, tabulated once from the definition above so the
 * loops below do not recompute it per element. */
static double e4m3_table[256];
static int e4m3_table_ready = 0;

static void e4m3_table_init(void)
{
    if (e4m3_table_ready)
        return;
    for (int c = 0; c < 256; ++c)
        e4m3_table[c] = oracle_e4m3_decode((uint8_t)c);
    e4m3_table_ready = 1;
}

/* Nearest e4m3 code to v (R3).  The non-negative finite codes 0x00..0x7E
 * are increasing in value, so the answer is one of the two codes that
 * bracket |v|; a tie goes to the code with an even last mantissa bit. */
uint8_t oracle_e4m3_encode(float v)
{
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs((double)v);
    if (isnan(v))
        return (uint8_t)(sign | 0x7F);
    e4m3_table_init();
    if (a >= e4m3_table[0x7E])                  /* saturate (incl. inf) */
        return (uint8_t)(sign | 0x7E);
    /* binary search keeping decode(lo) <= a < decode(hi) */
    int lo = 0, hi = 0x7E;
    while (hi - lo > 1) {
        int mid = (lo + hi) / 2;
        if (e4m3_table[mid] <= a) lo = mid; else hi = mid;
    }
    double below = e4m3_table[lo];
    double above = e4m3_table[lo + 1];
    double d_lo = a - below, d_hi = above - a;  /* exact: all dyadic, few bits */
    int code;
    if (d_lo < d_hi) code = lo;
    else if (d_hi < d_lo) code = lo + 1;
    else code = (lo % 2 == 0) ? lo : lo + 1;    /* tie: even mantissa */
    return (uint8_t)(sign | code);
}

/* Array forms of the scalar codec (plain loops, for the tests). */
void oracle_e4m3_encode_array(const float *v, int64_t n, uint8_t *out)
{
    e4m3_table_init();
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_e4m3_encode(v[i]);
}

/* bfloat16: the top 16 bits of an fp32.  Widening is exact. */
float oracle_bf16_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

static float f32_from_bits(uint32_t u) { float f; memcpy(&f, &u, sizeof f); return f; }
static uint32_t bits_from_f32(float f) { uint32_t u; memcpy(&u, &f, sizeof u); return u; }

/* fp32 -> bf16, round to nearest, ties to even.  The two bf16 candidates are
 * the fp32 truncated to 16 bits (toward zero) and the next bf16 away from
 * zero; pick the nearer in exact (double) arithmetic. */
uint16_t oracle_f32_to_bf16(float f)
{
    if (isnan(f))
        return 0x7FC0;
    uint32_t u = bits_from_f32(f);
    uint32_t toward = u & 0xFFFF0000u;
    uint32_t away = toward + 0x10000u;          /* next magnitude up, same sign */
    if (toward == u)
        return (uint16_t)(toward >> 16);
    double a = fabs((double)f);
    double lo = fabs((double)f32_from_bits(toward));
    double hi = fabs((double)f32_from_bits(away));
    if (isinf(hi))              /* IEEE: past max finite the next step is 2^128 */
        hi = ldexp(1.0, 128);
    double d_lo = a - lo, d_hi = hi - a;
    if (d_lo < d_hi) return (uint16_t)(toward >> 16);
    if (d_hi < d_lo) return (uint16_t)(away >> 16);
    return (uint16_t)((((toward >> 16) & 1u) == 0u ? toward : away) >> 16);
}

void oracle_f32_to_bf16_array(const float *v, int64_t n, uint16_t *out)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_f32_to_bf16(v[i]);
}

/* double -> bf16, round to nearest, ties to even, for finite values inside
 * the normal bf16 range (the oracle's uses never leave it); zero keeps its
 * sign.  Written as: scale |d| to [128, 256), round to an integer with ties
 * to even, scale back, then take the bf16 bits of that (exact) fp32. */
uint16_t oracle_f64_to_bf16(double d)
{
    if (d == 0.0)
        return signbit(d) ? 0x8000 : 0x0000;
    int e;
    double frac = frexp(fabs(d), &e);           /* |d| = frac * 2^e, frac in [0.5,1) */
    double scaled = ldexp(frac, 8);             /* [128, 256) */
    double q = floor(scaled);
    double rem = scaled - q;
    if (rem > 0.5 || (rem == 0.5 && fmod(q, 2.0) != 0.0))
        q += 1.0;
    double r = ldexp(q, e - 8);
    float rf = (float)r;                        /* exact: 8 significant bits */
    uint32_t u = bits_from_f32(rf);
    if (d < 0) u |= 0x80000000u;
    return (uint16_t)(u >> 16);
}

/* ------------------------------------------------------------------ */
/* Scale of one block                                                   */
/* ------------------------------------------------------------------ */

/* R4: smallest power of two that is >= s (s > 0, finite, normal). */
float oracle_pow2_ceil(float s)
{
    int e;
    float frac = frexpf(s, &e);                 /* s = frac * 2^e, frac in [0.5, 1) */
    if (frac == 0.5f)
        return s;                               /* already a power of two */
    return ldexpf(1.0f, e);
}

/* [TOUR]: scale = clamped amax / 448 (R1, R2), optionally ue8m0 (R4). */
static float block_scale(float amax, int ue8m0)
{
    if (amax < ORACLE_AMAX_FLOOR)
        amax = ORACLE_AMAX_FLOOR;
    float s = amax / ORACLE_E4M3_MAX;           /* fp32 divide, RN */
    if (ue8m0)
        s = oracle_pow2_ceil(s);
    return s;
}

/* ------------------------------------------------------------------ */
/* act_quant  [DF "FP8 quantization data flow"], [TOUR]                 */
/* ------------------------------------------------------------------ */

/* x: bf16 bits [M, K] row-major, K % 128 == 0.
 * y: e4m3 codes [M, K]; s: fp32 [M, K/128].  ue8m0: 0 or 1. */
void oracle_act_quant(const uint16_t *x, int64_t M, int64_t K, int ue8m0,
                      uint8_t *y, float *s)
{
    e4m3_table_init();
    int64_t KB = K / ORACLE_BLOCK;
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t kb = 0; kb < KB; ++kb) {
            const uint16_t *xb = x + m * K + kb * ORACLE_BLOCK;
            float amax = 0.0f;
            for (int i = 0; i < ORACLE_BLOCK; ++i) {
                float a = fabsf(oracle_bf16_to_f32(xb[i]));
                if (a > amax) amax = a;
            }
            float sc = block_scale(amax, ue8m0);
            s[m * KB + kb] = sc;
            for (int i = 0; i < ORACLE_BLOCK; ++i)
                y[m * K + kb * ORACLE_BLOCK + i] =
                    oracle_e4m3_encode(oracle_bf16_to_f32(xb[i]) / sc);
        }
    }
}

/* ------------------------------------------------------------------ */
/* weight quantisation (input preparation: bf16 weight -> e4m3 + grid)  */
/* ------------------------------------------------------------------ */

/* w: bf16 bits [N, K]; q: e4m3 [N, K]; s: fp32 [ceil(N/128), ceil(K/128)].
 * One scale per 128x128 block (R5); a partial block at the N or K edge
 * covers only its valid elements.  Same scale rule as act_quant. */
void oracle_weight_quant(const uint16_t *w, int64_t N, int64_t K, int ue8m0,
                         uint8_t *q, float *s)
{
    e4m3_table_init();
    int64_t NB = (N + ORACLE_BLOCK - 1) / ORACLE_BLOCK;
    int64_t KB = (K + ORACLE_BLOCK - 1) / ORACLE_BLOCK;
#pragma omp parallel for schedule(static)
    for (int64_t nb = 0; nb < NB; ++nb) {
        int64_t n0 = nb * ORACLE_BLOCK;
        int64_t n1 = n0 + ORACLE_BLOCK < N ? n0 + ORACLE_BLOCK : N;
        for (int64_t kb = 0; kb < KB; ++kb) {
            int64_t k0 = kb * ORACLE_BLOCK;
            int64_t k1 = k0 + ORACLE_BLOCK < K ? k0 + ORACLE_BLOCK : K;
            float amax = 0.0f;
            for (int64_t n = n0; n < n1; ++n)
                for (int64_t k = k0; k < k1; ++k) {
                    float a = fabsf(oracle_bf16_to_f32(w[n * K + k]));
                    if (a > amax) amax = a;
                }
            float sc = block_scale(amax, ue8m0);
            s[nb * KB + kb] = sc;
            for (int64_t n = n0; n < n1; ++n)
                for (int64_t k = k0; k < k1; ++k)
                    q[n * K + k] = oracle_e4m3_encode(oracle_bf16_to_f32(w[n * K + k]) / sc);
        }
    }
}

/* ------------------------------------------------------------------ */
/* weight_dequant  [BT "fp8->bf16 trace"], [TOUR]                       */
/* ------------------------------------------------------------------ */

/* w: e4m3 [M, N]; s: fp32 [ceil(M/128), ceil(N/128)]; y: bf16 bits [M, N].
 * y = bf16_rne(fp32(w) * s) with one fp32 multiply rounded to nearest. */
void oracle_weight_dequant(const uint8_t *w, const float *s, int64_t M, int64_t N,
                           uint16_t *y)
{
    e4m3_table_init();
    int64_t NB = (N + ORACLE_BLOCK - 1) / ORACLE_BLOCK;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < M; ++i)
        for (int64_t j = 0; j < N; ++j) {
            float v = (float)oracle_e4m3_decode(w[i * N + j]);
            float sc = s[(i / ORACLE_BLOCK) * NB + (j / ORACLE_BLOCK)];
            y[i * N + j] = oracle_f32_to_bf16(v * sc);
        }
}

/* ------------------------------------------------------------------ */
/* fp8_gemm  [DF "FP8 quantization data flow"], [TOUR]                  */
/* ------------------------------------------------------------------ */

/* One output element of the block-scaled product (R5, R6):
 *   ref = sum_kb a_s[m,kb] * b_s[n/128,kb] * sum_{k in kb} a[m,k] * b[n,k]
 * The inner sums of e4m3 products are exact in double.  mag is the same
 * expression over absolute values, the yardstick for rounding error. */
static void gemm_element(const uint8_t *a_row, const float *as_row,
                         const uint8_t *b_row, const float *bs_row, int64_t K,
                         double *ref, double *mag)
{
    e4m3_table_init();
    int64_t KB = K / ORACLE_BLOCK;
    double r = 0.0, g = 0.0;
    for (int64_t kb = 0; kb < KB; ++kb) {
        double dot = 0.0, adot = 0.0;
        for (int i = 0; i < ORACLE_BLOCK; ++i) {
            double p = e4m3_table[a_row[kb * ORACLE_BLOCK + i]] *
                       e4m3_table[b_row[kb * ORACLE_BLOCK + i]];
            dot += p;
            adot += fabs(p);
        }
        double scale = (double)as_row[kb] * (double)bs_row[kb];
        r += scale * dot;
        g += fabs(scale) * adot;
    }
    *ref = r;
    *mag = g;
}

/* a: e4m3 [M, K]; a_s: fp32 [M, K/128]; b: e4m3 [N, K]; b_s: fp32
 * [ceil(N/128), K/128].  rows: the nrows row indices of A to evaluate (all
 * rows when rows == NULL, nrows == M).  ref, mag: double [nrows, N]. */
void oracle_gemm(const uint8_t *a, const float *a_s, const uint8_t *b, const float *b_s,
                 int64_t M, int64_t N, int64_t K, const int64_t *rows, int64_t nrows,
                 double *ref, double *mag)
{
    e4m3_table_init();
    int64_t KB = K / ORACLE_BLOCK;
    (void)M;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t m = rows ? rows[i] : i;
        for (int64_t n = 0; n < N; ++n)
            gemm_element(a + m * K, a_s + m * KB, b + n * K, b_s + (n / ORACLE_BLOCK) * KB,
                         K, ref + i * N + n, mag + i * N + n);
    }
}

/* Grouped form for the routed experts ([BT "MoE trace"]): rows
 * [offsets[g], offsets[g+1]) of the packed A use expert g's weight
 * b + g*N*K and scales b_s + g*ceil(N/128)*(K/128).  rows: which packed rows
 * to evaluate (NULL: all offsets[G] rows). */
void oracle_grouped_gemm(const uint8_t *a, const float *a_s, const uint8_t *b,
                         const float *b_s, const int32_t *offsets, int32_t G,
                         int64_t N, int64_t K, const int64_t *rows, int64_t nrows,
                         double *ref, double *mag)
{
    e4m3_table_init();
    int64_t KB = K / ORACLE_BLOCK;
    int64_t NB = (N + ORACLE_BLOCK - 1) / ORACLE_BLOCK;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t r = rows ? rows[i] : i;
        int32_t g = 0;
        while (g < G && !(offsets[g] <= r && r < offsets[g + 1]))
            ++g;
        if (g == G) {                           /* row outside every group */
            for (int64_t n = 0; n < N; ++n) { ref[i * N + n] = NAN; mag[i * N + n] = NAN; }
            continue;
        }
        const uint8_t *bg = b + (int64_t)g * N * K;
        const float *bsg = b_s + (int64_t)g * NB * KB;
        for (int64_t n = 0; n < N; ++n)
            gemm_element(a + r * K, a_s + r * KB, bg + n * K, bsg + (n / ORACLE_BLOCK) * KB,
                         K, ref + i * N + n, mag + i * N + n);
    }
}

/* ------------------------------------------------------------------ */
/* Expert body and MoE combine  [BT "MoE trace"], [DF MoE bullet]       */
/* ------------------------------------------------------------------ */

/* silu(h1) * h3 between the two expert projections, with bf16 tensors as
 * in the model: silu is rounded to bf16, then the product of two bf16
 * values is rounded to bf16.  silu(v) = v / (1 + exp(-v)) in double. */
void oracle_silu_mul(const uint16_t *h1, const uint16_t *h3, int64_t n, uint16_t *g)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        double v = (double)oracle_bf16_to_f32(h1[i]);
        double sl = v / (1.0 + exp(-v));
        double sl_b = (double)oracle_bf16_to_f32(oracle_f64_to_bf16(sl));
        double prod = sl_b * (double)oracle_bf16_to_f32(h3[i]);   /* exact */
        g[i] = oracle_f64_to_bf16(prod);
    }
}

/* Routing of T tokens with topk experts each (ids [T, topk], no duplicates
 * within a token) to packed expert-major rows: expert e owns packed rows
 * [offsets[e], offsets[e+1]); inside an expert, pairs (t, j) keep the
 * order of t*topk + j.  pair_row[t*topk+j] = packed row of that pair,
 * row_token[r] = the token whose activation row r holds. */
void oracle_moe_route(const int32_t *ids, int64_t T, int32_t topk, int32_t E,
                      int32_t *offsets, int32_t *pair_row, int32_t *row_token)
{
    int64_t P = T * topk;
    offsets[0] = 0;
    for (int32_t e = 0; e < E; ++e) {
        int32_t count = 0;
        for (int64_t p = 0; p < P; ++p)
            if (ids[p] == e) ++count;
        offsets[e + 1] = offsets[e] + count;
    }
    for (int32_t e = 0; e < E; ++e) {
        int32_t r = offsets[e];
        for (int64_t p = 0; p < P; ++p)
            if (ids[p] == e) {
                pair_row[p] = r;
                row_token[r] = (int32_t)(p / topk);
                ++r;
            }
    }
}

/* y[t, :] = sum_j w[t, j] * out[pair_row[t*topk+j], :] in double, the
 * weighted scatter-add of the routed expert outputs (bf16 bits [R, D]). */
void oracle_moe_combine(const uint16_t *out, const float *w, const int32_t *pair_row,
                        int64_t T, int32_t topk, int64_t D, const int64_t *tokens,
                        int64_t ntok, double *y, double *ymag)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < ntok; ++i) {
        int64_t t = tokens ? tokens[i] : i;
        for (int64_t d = 0; d < D; ++d) {
            double acc = 0.0, amag = 0.0;
            for (int32_t j = 0; j < topk; ++j) {
                double v = (double)w[t * topk + j] *
                           (double)oracle_bf16_to_f32(out[(int64_t)pair_row[t * topk + j] * D + d]);
                acc += v;
                amag += fabs(v);
            }
            y[i * D + d] = acc;
            ymag[i * D + d] = amag;
        }
    }
    (void)T;
}

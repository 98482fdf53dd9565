/*
 * qlin_oracle.c -- the CPU oracle for the group-wise quantized linear layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library calls, links or
 * includes this file; only the tests, the smoke check and the CPU-baseline leg
 * of the benchmark load it.  It shares no code, header, table or helper with
 * the CUDA path: every conversion below is written out here from the IEEE-754
 * definitions.
 *
 * It is deliberately plain and slow: one output element at a time, integer
 * dot products in int64, the cross-group rescale as a single fp32 chain, and
 * an fp64 evaluation of the same sums with a rounding-error bound beside it.
 *
 * What it computes, and where that is stated:
 *
 *  - Weight format: GPTQ qweight/qzeros/scales, no g_idx, desc_act=false,
 *    symmetric, group size 128 ("Flint-DFlash2-GPTQ-INT8-PTQR" model card,
 *    parameter table; "every matrix uses contiguous groups of exactly 128
 *    weights", same card, text under the table).
 *  - Activations: dynamic per-token INT8 quantization with round-to-nearest
 *    (same card: PTQR paragraph and the VLLM_GFX908_ACT_QUANT=round recipe
 *    line; "Qwen3.8-27B-GPTQ-INT8-W8A8-GS128-PTQR" card, "Serving": GEMM
 *    inputs are dynamically quantized to INT8).
 *  - W8A8: int8 x int8 products with one weight scale per 128-wide K block
 *    ("Qwen3.8-27B-GPTQ-INT8-W8A8-GS128-PTQR" card, "Quantization details").
 *  - W4A16: 4-bit symmetric weights, group 128, bf16 activations, dequantized
 *    as "unpack_from_int32 + group scales" ("Qwen3.8-27B-DFlash2-W4A16-g128-
 *    sym-GPTQ" card, property table and the apply_dense_kv_fix format table).
 *
 * Readings taken where the pages are silent (all listed in the design notes):
 *  - activation scale s = amax / 127 in fp32 (an IEEE divide), q = rint(x / s)
 *    with ties to even, clamped to [-127, 127]; an all-zero row gives s = 0 and
 *    q = 0 without dividing;
 *  - GPTQ packing is LSB-first along K: field i of word kk holds row
 *    (32/bits)*kk + i, stored with the zero point 2^(bits-1) added;
 *  - the W8A8 group partials are rescaled by an fp32 fma chain over ascending
 *    groups, then multiplied once by the activation scale, then rounded to
 *    bf16 (round to nearest even);
 *  - W4A16 dequantizes each weight to bf16(q * s) and accumulates x * w in
 *    fp32 over all K in ascending k, then rounds to bf16.
 *
 * Build: plain C11, -ffp-contract=off so that no a*b+c is fused behind the
 * code's back (fmaf is called where a fused multiply-add is meant).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define GROUP 128

/* ---------------------------------------------------------------- formats */

/* bf16 is the upper half of an IEEE binary32. */
float orc_bf16_to_f32(uint16_t h)
{
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* binary32 -> bf16, round to nearest, ties to even (NaN kept quiet). */
uint16_t orc_f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7f800000u) == 0x7f800000u) {            /* inf or NaN */
        if (u & 0x007fffffu) return (uint16_t)((u >> 16) | 0x0040u);
        return (uint16_t)(u >> 16);
    }
    uint32_t upper = u >> 16;
    uint32_t lower = u & 0xffffu;                        /* the dropped bits */
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u)))
        upper += 1u;                                     /* carries into the exponent correctly */
    return (uint16_t)upper;
}

/* IEEE binary16 -> binary32 (exact). */
float orc_f16_to_f32(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int mant = h & 0x3ff;
    float v;
    if (expo == 0)
        v = ldexpf((float)mant, -24);                    /* subnormal: mant * 2^-24 */
    else if (expo == 31)
        v = mant ? NAN : INFINITY;
    else
        v = ldexpf((float)(1024 + mant), expo - 25);     /* (1 + mant/1024) * 2^(expo-15) */
    return sign ? -v : v;
}

/* ---------------------------------------------------------- activations */

/* Dynamic per-token symmetric INT8 quantization of a bf16 [M, K] matrix.
 * For each row m: amax = max_k |x|, s[m] = amax / 127, q = rint(x / s) in
 * [-127, 127].  An all-zero row gives s = 0 and q = 0. */
void orc_act_quant_i8(const uint16_t *x, int64_t M, int64_t K, int8_t *q, float *s)
{
    for (int64_t m = 0; m < M; ++m) {
        const uint16_t *row = x + m * K;
        float amax = 0.0f;
        for (int64_t k = 0; k < K; ++k) {
            float a = fabsf(orc_bf16_to_f32(row[k]));
            if (a > amax) amax = a;
        }
        if (amax == 0.0f) {
            s[m] = 0.0f;
            for (int64_t k = 0; k < K; ++k) q[m * K + k] = 0;
            continue;
        }
        float scale = amax / 127.0f;
        s[m] = scale;
        for (int64_t k = 0; k < K; ++k) {
            float r = rintf(orc_bf16_to_f32(row[k]) / scale);
            if (r > 127.0f) r = 127.0f;
            if (r < -127.0f) r = -127.0f;
            q[m * K + k] = (int8_t)r;
        }
    }
}

/* ------------------------------------------------------------ GPTQ pack */

/* Pack q[K, N] (row-major, K = input features) into GPTQ words along K.
 * bits = 8: 4 fields per int32, stored q + 128; bits = 4: 8 fields, q + 8.
 * qweight is [K*bits/32, N]; qzeros (may be NULL) is [K/128, N*bits/32] with
 * every field equal to the zero point.  Returns the number of q values that
 * fell outside [-2^(bits-1), 2^(bits-1) - 1] (those are packed masked). */
int64_t orc_pack_gptq(const int8_t *q, int64_t K, int64_t N, int bits,
                      int32_t *qweight, int32_t *qzeros)
{
    const int per = 32 / bits;
    const int zero = 1 << (bits - 1);
    const uint32_t mask = (1u << bits) - 1u;
    int64_t bad = 0;
    for (int64_t kk = 0; kk < K / per; ++kk) {
        for (int64_t n = 0; n < N; ++n) {
            uint32_t word = 0;
            for (int i = 0; i < per; ++i) {
                int v = (int)q[(kk * per + i) * N + n] + zero;
                if (v < 0 || v > (int)mask) ++bad;
                word |= ((uint32_t)v & mask) << (bits * i);
            }
            qweight[kk * N + n] = (int32_t)word;
        }
    }
    if (qzeros) {
        uint32_t zword = 0;
        for (int i = 0; i < per; ++i) zword |= (uint32_t)zero << (bits * i);
        for (int64_t g = 0; g < K / GROUP; ++g)
            for (int64_t j = 0; j < N / per; ++j)
                qzeros[g * (N / per) + j] = (int32_t)zword;
    }
    return bad;
}

/* One weight value q[k, n] read back out of the packed words. */
static int weight_at(const int32_t *qweight, int64_t N, int bits, int64_t k, int64_t n)
{
    const int per = 32 / bits;
    uint32_t word = (uint32_t)qweight[(k / per) * N + n];
    uint32_t field = (word >> (bits * (int)(k % per))) & ((1u << bits) - 1u);
    return (int)field - (1 << (bits - 1));
}

/* Unpack qweight back to q[K, N]. */
void orc_unpack_gptq(const int32_t *qweight, int64_t K, int64_t N, int bits, int8_t *q)
{
    for (int64_t k = 0; k < K; ++k)
        for (int64_t n = 0; n < N; ++n)
            q[k * N + n] = (int8_t)weight_at(qweight, N, bits, k, n);
}

/* ------------------------------------------------------------ W8A8 GS128 */

/* Exact per-group integer dot products:
 * P[g, m, n] = sum_{k in group g} qa[m, k] * qw[k, n]   (int32, g = 0..K/128-1). */
void orc_group_partials_i8(const int8_t *qa, const int32_t *qweight,
                           int64_t M, int64_t N, int64_t K, int32_t *P)
{
    const int64_t G = K / GROUP;
    for (int64_t g = 0; g < G; ++g)
        for (int64_t m = 0; m < M; ++m)
            for (int64_t n = 0; n < N; ++n) {
                int64_t acc = 0;
                for (int64_t k = g * GROUP; k < (g + 1) * GROUP; ++k)
                    acc += (int64_t)qa[m * K + k] * (int64_t)weight_at(qweight, N, 8, k, n);
                P[(g * M + m) * N + n] = (int32_t)acc;   /* |acc| <= 128*127*127 */
            }
}

/* W8A8 GS128 linear on the listed rows and columns.
 * Outputs, each [nrows, ncols]:
 *   y_bf16 : bf16 of y_f32,
 *   y_f32  : acc * sa[m] with acc = fma(P_g, sw[g, n], acc) over g ascending,
 *   y64    : sa[m] * sum_g P_g * sw[g, n] in fp64,
 *   bound  : (G + 2) * 2^-24 * |sa[m]| * sum_g |P_g * sw[g, n]|,
 *            a bound on |y_f32 - y64| for any summation order of the G terms,
 *   abs_sum: |sa[m]| * sum_g |P_g * sw[g, n]| in fp64 (the size of the terms,
 *            against which cancellation in y is measured). */
void orc_gemm_w8a8_gs128(const int8_t *qa, const float *sa, const int32_t *qweight,
                         const uint16_t *scales_f16, int64_t M, int64_t N, int64_t K,
                         const int64_t *rows, int64_t nrows,
                         const int64_t *cols, int64_t ncols,
                         uint16_t *y_bf16, float *y_f32, double *y64, double *bound,
                         double *abs_sum)
{
    const int64_t G = K / GROUP;
    (void)M;
    for (int64_t r = 0; r < nrows; ++r) {
        const int64_t m = rows[r];
        for (int64_t c = 0; c < ncols; ++c) {
            const int64_t n = cols[c];
            float acc = 0.0f;
            double exact = 0.0, magnitude = 0.0;
            for (int64_t g = 0; g < G; ++g) {
                int64_t p = 0;
                for (int64_t k = g * GROUP; k < (g + 1) * GROUP; ++k)
                    p += (int64_t)qa[m * K + k] * (int64_t)weight_at(qweight, N, 8, k, n);
                const float sw = orc_f16_to_f32(scales_f16[g * N + n]);
                acc = fmaf((float)p, sw, acc);
                exact += (double)p * (double)sw;
                magnitude += fabs((double)p * (double)sw);
            }
            const float y = acc * sa[m];
            const int64_t o = r * ncols + c;
            y_f32[o] = y;
            y_bf16[o] = orc_f32_to_bf16(y);
            y64[o] = exact * (double)sa[m];
            bound[o] = (double)(G + 2) * ldexp(1.0, -24) * magnitude * fabs((double)sa[m]);
            abs_sum[o] = magnitude * fabs((double)sa[m]);
        }
    }
}

/* ----------------------------------------------------------- W4A16 g128 */

/* W4A16 g128 linear on the listed rows and columns.
 * w[k, n] = bf16(q[k, n] * s[k/128, n]) (the product is exact in fp32, so
 * this is one rounding); y_f32 = sum_k x[m, k] * w[k, n] in fp32 over k
 * ascending (each product is exact in fp32); y_bf16 = bf16(y_f32);
 * y64 = the same sum in fp64; bound = (K + 2) * 2^-23 * sum_k |x * w|, a
 * bound on |y_f32 - y64| that also covers accumulators that truncate instead
 * of rounding; abs_sum = sum_k |x * w| in fp64. */
void orc_gemm_w4a16_g128(const uint16_t *x, const int32_t *qweight,
                         const uint16_t *scales_bf16, int64_t M, int64_t N, int64_t K,
                         const int64_t *rows, int64_t nrows,
                         const int64_t *cols, int64_t ncols,
                         uint16_t *y_bf16, float *y_f32, double *y64, double *bound,
                         double *abs_sum)
{
    (void)M;
    for (int64_t r = 0; r < nrows; ++r) {
        const int64_t m = rows[r];
        for (int64_t c = 0; c < ncols; ++c) {
            const int64_t n = cols[c];
            float acc = 0.0f;
            double exact = 0.0, magnitude = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                const float s = orc_bf16_to_f32(scales_bf16[(k / GROUP) * N + n]);
                const float w = orc_bf16_to_f32(orc_f32_to_bf16((float)weight_at(qweight, N, 4, k, n) * s));
                const float xv = orc_bf16_to_f32(x[m * K + k]);
                const float prod = xv * w;
                acc = acc + prod;
                exact += (double)xv * (double)w;
                magnitude += fabs((double)xv * (double)w);
            }
            const int64_t o = r * ncols + c;
            y_f32[o] = acc;
            y_bf16[o] = orc_f32_to_bf16(acc);
            y64[o] = exact;
            bound[o] = (double)(K + 2) * ldexp(1.0, -23) * magnitude;
            abs_sum[o] = magnitude;
        }
    }
}

/* Dequantized W4A16 weight w[k, n] = bf16(q * s) for the whole matrix (used
 * by the identity-probe checks). */
void orc_dequant_w4a16(const int32_t *qweight, const uint16_t *scales_bf16,
                       int64_t K, int64_t N, uint16_t *w_bf16)
{
    for (int64_t k = 0; k < K; ++k)
        for (int64_t n = 0; n < N; ++n) {
            const float s = orc_bf16_to_f32(scales_bf16[(k / GROUP) * N + n]);
            w_bf16[k * N + n] = orc_f32_to_bf16((float)weight_at(qweight, N, 4, k, n) * s);
        }
}

/* Greedy decoding reads only the argmax of the vocabulary head's output
 * ("DFlash2 decoding" recipe page: single-GPU, batch-one greedy inference,
 * with an INT8 or INT4 group-128 shared vocabulary head): for each row m of
 * y (bf16 [M, N]) the index n of the largest value, the lowest such index
 * when several are equal.  Values compare as the numbers they encode. */
void orc_argmax_bf16_rows(const uint16_t *y, int64_t M, int64_t N, int32_t *idx)
{
    for (int64_t m = 0; m < M; ++m) {
        int64_t best = 0;
        float best_v = orc_bf16_to_f32(y[m * N]);
        for (int64_t n = 1; n < N; ++n) {
            const float v = orc_bf16_to_f32(y[m * N + n]);
            if (v > best_v) {
                best_v = v;
                best = n;
            }
        }
        idx[m] = (int32_t)best;
    }
}

/* Ingest of the compressed-tensors "pack-quantized" orientation
 * ("Qwen3.8-27B-DFlash2-W4A16-g128-sym-GPTQ" card, property table, Format row: compressed-tensors
 * pack-quantized, Marlin-compatible): the packed weight is stored per output
 * row, word (n, kk) holding the same fields as the GPTQ word (kk, n) (field i
 * = q[(32/bits) kk + i, n] + 2^(bits-1)), and the scales are [N, K/128].  The
 * GEMMs read [K*bits/32, N] words and [K/128, N] scales: ingest is the
 * transpose of both, bit for bit. */
void orc_ingest_nk(const int32_t *packed_nk, const uint16_t *scales_ng, int64_t K, int64_t N,
                   int bits, int32_t *qweight, uint16_t *scales)
{
    const int64_t R = K * bits / 32, G = K / GROUP;
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t kk = 0; kk < R; ++kk) qweight[kk * N + n] = packed_nk[n * R + kk];
        for (int64_t g = 0; g < G; ++g) scales[g * N + n] = scales_ng[n * G + g];
    }
}

/* The tile layout of the weights (a reordering of the GPTQ words, with no
 * counterpart in the pages beyond the card's note that serving kernels take
 * the words in their own, Marlin-compatible, order): tile (f, g) holds the
 * words of output features 128f..128f+127 and K group g as W x 128 int32, W =
 * 128 * bits / 32 words; word (kk, j) of the tile is GPTQ word (g*W + kk,
 * 128f + j), or 0 past N; tiles follow each other by f, then g. */
void orc_pack_tiles(const int32_t *qweight, int64_t K, int64_t N, int bits, int32_t *tiles)
{
    const int64_t W = GROUP * bits / 32, G = K / GROUP, F = (N + 127) / 128;
    int64_t o = 0;
    for (int64_t f = 0; f < F; ++f)
        for (int64_t g = 0; g < G; ++g)
            for (int64_t kk = 0; kk < W; ++kk)
                for (int64_t j = 0; j < 128; ++j, ++o) {
                    const int64_t n = 128 * f + j;
                    tiles[o] = n < N ? qweight[(g * W + kk) * N + n] : 0;
                }
}

/* W8A16 weight-only int8 linear ("Qwen3.5-4B-DFlash-W8A16" card: a
 * weight-only int8 drafter made by round-to-nearest on the weights; "DFlash2
 * decoding" recipe page: int8 drafter projections with group-32 scales).
 * Read like W4A16: w[k, n] = bf16(q[k, n] * s[k / gs, n]) (one rounding of an
 * exact product), y = bf16(sum_k x[m, k] * w[k, n]) accumulated in fp32 over
 * k ascending.  q comes from the 8-bit GPTQ words ([K/4, N], byte = q + 128);
 * scales are bf16 [K/gs, N], with gs = 0 meaning one scale per output column
 * (scales [1, N]).  y64 / bound / abs_sum as for W4A16. */
void orc_gemm_w8a16(const uint16_t *x, const int32_t *qweight, const uint16_t *scales_bf16,
                    int64_t M, int64_t N, int64_t K, int64_t gs,
                    const int64_t *rows, int64_t nrows, const int64_t *cols, int64_t ncols,
                    uint16_t *y_bf16, float *y_f32, double *y64, double *bound,
                    double *abs_sum)
{
    (void)M;
    for (int64_t r = 0; r < nrows; ++r) {
        const int64_t m = rows[r];
        for (int64_t c = 0; c < ncols; ++c) {
            const int64_t n = cols[c];
            float acc = 0.0f;
            double exact = 0.0, magnitude = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                const int64_t g = gs > 0 ? k / gs : 0;
                const float s = orc_bf16_to_f32(scales_bf16[g * N + n]);
                const float w = orc_bf16_to_f32(orc_f32_to_bf16((float)weight_at(qweight, N, 8, k, n) * s));
                const float xv = orc_bf16_to_f32(x[m * K + k]);
                const float prod = xv * w;
                acc = acc + prod;
                exact += (double)xv * (double)w;
                magnitude += fabs((double)xv * (double)w);
            }
            const int64_t o = r * ncols + c;
            y_f32[o] = acc;
            y_bf16[o] = orc_f32_to_bf16(acc);
            y64[o] = exact;
            bound[o] = (double)(K + 2) * ldexp(1.0, -23) * magnitude;
            abs_sum[o] = magnitude;
        }
    }
}

/* ------------------------------------------------------ fused producers */

/* binary64 -> bf16, rounded once to nearest, ties to even.  The value is
 * scaled so that its bf16 unit in the last place becomes 1 (2^-133 at the
 * bottom of the subnormal range), rounded to an integer by nearbyint under the
 * default rounding mode, and scaled back: every step is exact except the one
 * rounding.  Values that round past the largest finite bf16 give infinity. */
uint16_t orc_f64_to_bf16(double d)
{
    if (isnan(d)) return (uint16_t)0x7fc0u;
    const int neg = signbit(d) != 0;
    const double a = fabs(d);
    if (a == 0.0) return neg ? (uint16_t)0x8000u : (uint16_t)0;
    int e;
    (void)frexp(a, &e);                   /* a = f * 2^e, f in [0.5, 1) */
    int ulp_exp = e - 8;                  /* 8 significant bits */
    if (ulp_exp < -133) ulp_exp = -133;   /* subnormal bf16 spacing */
    const double r = ldexp(nearbyint(ldexp(a, -ulp_exp)), ulp_exp);
    const float f = (float)r;             /* exact, or infinity on overflow */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    uint16_t h = (uint16_t)(u >> 16);
    if (neg) h |= (uint16_t)0x8000u;
    return h;
}

/* RMSNorm of each bf16 row, as the decoder norms of the model family define
 * it ("Qwen3.8-27B-DFlash2-W4A16-g128-sym-GPTQ" card: input_layernorm and
 * post_attention_layernorm are kept in BF16, in front of the q/k/v and
 * gate/up projections):
 *   variance = mean_k x[m,k]^2,   t = bf16(x / sqrt(variance + eps)),
 *   z[m,k] = bf16(gamma[k] * t).
 * Evaluated in fp64 and rounded where the definition stores bf16 (the
 * product of two bf16 values is exact in fp64). */
void orc_rmsnorm_bf16(const uint16_t *x, const uint16_t *gamma, double eps, int64_t M, int64_t K,
                      uint16_t *z)
{
    for (int64_t m = 0; m < M; ++m) {
        const uint16_t *row = x + m * K;
        double ss = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            const double v = (double)orc_bf16_to_f32(row[k]);
            ss += v * v;
        }
        const double rstd = 1.0 / sqrt(ss / (double)K + eps);
        for (int64_t k = 0; k < K; ++k) {
            const double t = (double)orc_bf16_to_f32(orc_f64_to_bf16((double)orc_bf16_to_f32(row[k]) * rstd));
            z[m * K + k] = orc_f64_to_bf16((double)orc_bf16_to_f32(gamma[k]) * t);
        }
    }
}

/* The gated MLP activation in front of down_proj (same card: the
 * mlp.{gate,up,down}_proj linears): z[m,i] = bf16(SiLU(g) * u) with
 * SiLU(g) = g / (1 + exp(-g)), g = gate_up[m, i], u = gate_up[m, I + i]:
 * the gate and up halves of one row of the fused gate/up projection's output
 * ([M, 2I], gate first).  Evaluated in fp64, rounded once. */
void orc_silu_mul_bf16(const uint16_t *gate_up, int64_t M, int64_t I, uint16_t *z)
{
    for (int64_t m = 0; m < M; ++m) {
        const uint16_t *row = gate_up + m * 2 * I;
        for (int64_t i = 0; i < I; ++i) {
            const double g = (double)orc_bf16_to_f32(row[i]);
            const double u = (double)orc_bf16_to_f32(row[I + i]);
            z[m * I + i] = orc_f64_to_bf16(g / (1.0 + exp(-g)) * u);
        }
    }
}

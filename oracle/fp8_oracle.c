/*
 * CPU oracle for fine-grained FP8 quantization and the block-scaled FP8 GEMM.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the plain, slow, obviously correct
 * statement of what the hot path computes. Only the test suite, the smoke
 * check and the benchmark's CPU-baseline leg may load it. The product library
 * never links, includes or calls anything here, and nothing here includes or
 * calls the product library.
 *
 * Sources (extracted web pages about DeepSeek-V3 mixed-precision training):
 *  - news.qq.com/rain/a/20241229A05OQF00, section "FP8 低精度训练",
 *    item "细粒度量化" (Fig. 7a): activations are quantized per 1x128 tile
 *    (one scale per token per 128 channels), weights per 128x128 block.
 *  - same page, item "提高累加精度" (Fig. 7b): the tensor-core MMA results are
 *    accumulated into FP32 registers (promotion of partial sums).
 *  - developer.aliyun.com/article/1776647, section 4.1 "FP8 混合精度训练":
 *    128x128 block quantization plus high-precision multiply-accumulate.
 *  - m.jxzklqfsx.com/aigc/3586, section 三(二) "FP8 混合精度訓練突破":
 *    tile- and block-grouped fine-grained quantization with high-precision
 *    accumulation.
 * The pages do not name the FP8 encoding, the scale formula or the promotion
 * interval. This oracle takes the plainest reading that fits them:
 *  - encoding E4M3 (OCP FP8 E4M3FN: bias 7, max 448, no infinities);
 *  - scale s = fl32(amax / 448), amax over the tile's present elements;
 *  - code q = E4M3_RNE_saturating(fl32(x / s)); an all-zero tile has s = 0
 *    and all codes 0x00;
 *  - GEMM: per 128-wide K block the dot product of decoded codes is taken
 *    exactly (in FP64, where it is exact), then scaled by sa*sb and summed
 *    in FP32 in ascending K-block order.
 *
 * Build: gcc -O2 -std=c11 -fno-fast-math -ffp-contract=off -shared -fPIC.
 * Contraction must stay off: the FP32 steps below are written as separate
 * roundings on purpose.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define TILE 128 /* the 1x128 / 128x128 granularity of the pages' Fig. 7a */
#define E4M3_MAX 448.0

/* bf16 -> fp32 is exact: the bf16 bits are the top half of the fp32 bits. */
static float bf16_to_f32(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

float fp8o_bf16_to_f32(uint16_t h) { return bf16_to_f32(h); }

/*
 * Decode one E4M3 code (OCP FP8 E4M3FN).
 *   exponent field e in 0..15, mantissa m in 0..7, bias 7
 *   e == 0            : (-1)^s * m * 2^-9           (subnormal)
 *   e in 1..15        : (-1)^s * (8 + m) * 2^(e-10) (= (1 + m/8) * 2^(e-7))
 *   e == 15 && m == 7 : NaN (0x7F, 0xFF); the format has no infinities.
 */
double fp8o_e4m3_decode(uint8_t c) {
    int sign = c >> 7;
    int e = (c >> 3) & 15;
    int m = c & 7;
    if (e == 15 && m == 7) return NAN;
    double mag = (e == 0) ? ldexp((double)m, -9) : ldexp((double)(8 + m), e - 10);
    return sign ? -mag : mag;
}

/*
 * Encode a finite fp32 value to E4M3: round to nearest, ties to even, onto
 * the E4M3 grid (subnormals included), and saturate to +-448 (a magnitude
 * at or above 448 gives 448: values in [448, 464) round to 448 anyway, and
 * everything above would round past the largest finite value). The sign is
 * kept, so -0 and negative values that round to zero give 0x80.
 *
 * Method: with a = |f| < 448, let E = max(floor(log2 a), -6). The grid step
 * in that binade is 2^(E-3) (2^-9 in the subnormal range), so n = a / 2^(E-3)
 * is exact in double, and rounding n to the nearest even integer is the RNE
 * step. The code magnitude is then ((E + 7) << 3) + (n - 8) for a normal
 * binade, where n == 16 carries into the exponent field by itself, and n for
 * the subnormal range, where n == 8 is the smallest normal code 0x08.
 */
uint8_t fp8o_e4m3_encode(float f) {
    uint8_t sign = signbit(f) ? 0x80 : 0x00;
    double a = fabs((double)f);
    if (a >= E4M3_MAX) return sign | 0x7E;
    int code;
    if (a < ldexp(1.0, -6)) {
        double n = nearbyint(ldexp(a, 9)); /* a / 2^-9 */
        code = (int)n;                     /* 0..8 */
    } else {
        int ex;
        frexp(a, &ex); /* a = frac * 2^ex, frac in [0.5, 1) */
        int E = ex - 1; /* floor(log2 a), in -6..8 */
        double n = nearbyint(ldexp(a, 3 - E)); /* a / 2^(E-3), in [8, 16] */
        code = ((E + 7) << 3) + ((int)n - 8);
    }
    return (uint8_t)(sign | (uint8_t)code);
}

/* Encode n fp32 values (vectorised test helper, no extra arithmetic). */
void fp8o_e4m3_encode_n(const float* f, int64_t n, uint8_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = fp8o_e4m3_encode(f[i]);
}

/* The tile scale: s = fl32(amax / 448), an IEEE round-to-nearest divide. */
static float tile_scale(float amax) { return amax / 448.0f; }

/* One element: q = E4M3(fl32(x / s)); an all-zero tile (s == 0) gives 0x00. */
static uint8_t encode_scaled(float x, float s) {
    if (s == 0.0f) return 0x00;
    float y = x / s;
    return fp8o_e4m3_encode(y);
}

/*
 * Activation quantization, one scale per 1x128 tile (news.qq.com page,
 * "细粒度量化", Fig. 7a: "1x128 tile-wise" for activations).
 *   x  : bf16 [M, K] row-major (raw uint16 bits)
 *   q  : uint8 E4M3 codes [M, K] row-major
 *   s  : fp32 [M, ceil(K/128)] row-major
 * Rows [m_begin, m_end) are processed, so a caller may split the work.
 * A tail tile (K % 128 != 0) takes its amax over its present elements only.
 */
void fp8o_quant_act(const uint16_t* x, int64_t M, int64_t K, int64_t m_begin,
                    int64_t m_end, uint8_t* q, float* s) {
    (void)M;
    int64_t KB = (K + TILE - 1) / TILE;
    for (int64_t m = m_begin; m < m_end; ++m) {
        for (int64_t kb = 0; kb < KB; ++kb) {
            int64_t k0 = kb * TILE;
            int64_t k1 = k0 + TILE < K ? k0 + TILE : K;
            float amax = 0.0f;
            for (int64_t k = k0; k < k1; ++k) {
                float v = fabsf(bf16_to_f32(x[m * K + k]));
                if (v > amax) amax = v;
            }
            float sc = tile_scale(amax);
            s[m * KB + kb] = sc;
            for (int64_t k = k0; k < k1; ++k)
                q[m * K + k] = encode_scaled(bf16_to_f32(x[m * K + k]), sc);
        }
    }
}

/*
 * Weight quantization, one scale per 128x128 block (news.qq.com page,
 * "细粒度量化", Fig. 7a: "128x128 block-wise" for weights; aliyun page §4.1).
 *   w  : bf16 [N, K] row-major
 *   q  : uint8 [N, K] row-major
 *   s  : fp32 [ceil(N/128), ceil(K/128)] row-major
 * Block rows [nb_begin, nb_end) are processed. Tail blocks (N or K not a
 * multiple of 128) take their amax over the present elements only.
 */
void fp8o_quant_weight(const uint16_t* w, int64_t N, int64_t K, int64_t nb_begin,
                       int64_t nb_end, uint8_t* q, float* s) {
    int64_t KB = (K + TILE - 1) / TILE;
    for (int64_t nb = nb_begin; nb < nb_end; ++nb) {
        int64_t n0 = nb * TILE;
        int64_t n1 = n0 + TILE < N ? n0 + TILE : N;
        for (int64_t kb = 0; kb < KB; ++kb) {
            int64_t k0 = kb * TILE;
            int64_t k1 = k0 + TILE < K ? k0 + TILE : K;
            float amax = 0.0f;
            for (int64_t n = n0; n < n1; ++n)
                for (int64_t k = k0; k < k1; ++k) {
                    float v = fabsf(bf16_to_f32(w[n * K + k]));
                    if (v > amax) amax = v;
                }
            float sc = tile_scale(amax);
            s[nb * KB + kb] = sc;
            for (int64_t n = n0; n < n1; ++n)
                for (int64_t k = k0; k < k1; ++k)
                    q[n * K + k] = encode_scaled(bf16_to_f32(w[n * K + k]), sc);
        }
    }
}

/*
 * Power-of-two (UE8M0) scales: a variant that the pages do not describe. It
 * keeps the 1x128 / 128x128 granularity but rounds each scale up to a power
 * of two, so that a tensor core with block scaling in hardware (8-bit
 * exponent scale factors) can apply it:
 *   e = ceil(log2(amax / 448)), the smallest integer with amax / 2^e <= 448,
 *   stored as the byte e + 127 (clamped below at 0, i.e. 2^-127);
 *   q = E4M3_RNE_sat(fl32(x / 2^e)); an all-zero tile gets byte 0, codes 0.
 * With amax = f * 2^E (frexp, f in [0.5, 1)) and 448 = 0.875 * 2^9, the
 * ratio amax / 448 = (f / 0.875) * 2^(E - 9) lies in (2^(E - 10), 2^(E - 8)),
 * so e = E - 9 when f <= 0.875 and E - 8 otherwise (exact comparisons).
 */
static uint8_t ue8m0_scale_byte(float amax) {
    if (amax == 0.0f) return 0;
    int E;
    double f = frexp((double)amax, &E);
    int e = f > 0.875 ? E - 8 : E - 9;
    if (e < -127) e = -127;
    return (uint8_t)(e + 127);
}

static uint8_t encode_pow2(float x, uint8_t sbyte, int zero_tile) {
    if (zero_tile) return 0x00;
    float s = ldexpf(1.0f, (int)sbyte - 127); /* exact, 2^-127 is an fp32 subnormal */
    return fp8o_e4m3_encode(x / s);
}

/* 1x128 tiles with UE8M0 scales; s: uint8 [M, ceil(K/128)]. */
void fp8o_quant_act_ue8m0(const uint16_t* x, int64_t M, int64_t K, int64_t m_begin,
                          int64_t m_end, uint8_t* q, uint8_t* s) {
    (void)M;
    int64_t KB = (K + TILE - 1) / TILE;
    for (int64_t m = m_begin; m < m_end; ++m) {
        for (int64_t kb = 0; kb < KB; ++kb) {
            int64_t k0 = kb * TILE;
            int64_t k1 = k0 + TILE < K ? k0 + TILE : K;
            float amax = 0.0f;
            for (int64_t k = k0; k < k1; ++k) {
                float v = fabsf(bf16_to_f32(x[m * K + k]));
                if (v > amax) amax = v;
            }
            uint8_t sb = ue8m0_scale_byte(amax);
            s[m * KB + kb] = sb;
            for (int64_t k = k0; k < k1; ++k)
                q[m * K + k] = encode_pow2(bf16_to_f32(x[m * K + k]), sb, amax == 0.0f);
        }
    }
}

/* 128x128 blocks with UE8M0 scales; s: uint8 [ceil(N/128), ceil(K/128)]. */
void fp8o_quant_weight_ue8m0(const uint16_t* w, int64_t N, int64_t K, int64_t nb_begin,
                             int64_t nb_end, uint8_t* q, uint8_t* s) {
    int64_t KB = (K + TILE - 1) / TILE;
    for (int64_t nb = nb_begin; nb < nb_end; ++nb) {
        int64_t n0 = nb * TILE;
        int64_t n1 = n0 + TILE < N ? n0 + TILE : N;
        for (int64_t kb = 0; kb < KB; ++kb) {
            int64_t k0 = kb * TILE;
            int64_t k1 = k0 + TILE < K ? k0 + TILE : K;
            float amax = 0.0f;
            for (int64_t n = n0; n < n1; ++n)
                for (int64_t k = k0; k < k1; ++k) {
                    float v = fabsf(bf16_to_f32(w[n * K + k]));
                    if (v > amax) amax = v;
                }
            uint8_t sb = ue8m0_scale_byte(amax);
            s[nb * KB + kb] = sb;
            for (int64_t n = n0; n < n1; ++n)
                for (int64_t k = k0; k < k1; ++k)
                    q[n * K + k] = encode_pow2(bf16_to_f32(w[n * K + k]), sb, amax == 0.0f);
        }
    }
}

/*
 * The exact per-K-block partial P_kb[m, n] = sum_{k in block kb} dec(qa[m,k]) *
 * dec(qb[n,k]) for kb = 0..ceil(K/128)-1, written to P[kb].
 * Exactness: every E4M3 value is an integer below 2^18 times 2^-9, so each
 * product is an integer below 2^36 times 2^-18 and 128 of them sum to below
 * 2^43 times 2^-18: no FP64 rounding happens, in any order.
 */
void fp8o_block_partials(const uint8_t* qa, const uint8_t* qb, int64_t K, int64_t m,
                         int64_t n, double* P) {
    int64_t KB = (K + TILE - 1) / TILE;
    for (int64_t kb = 0; kb < KB; ++kb) {
        int64_t k0 = kb * TILE;
        int64_t k1 = k0 + TILE < K ? k0 + TILE : K;
        double acc = 0.0;
        for (int64_t k = k0; k < k1; ++k)
            acc += fp8o_e4m3_decode(qa[m * K + k]) * fp8o_e4m3_decode(qb[n * K + k]);
        P[kb] = acc;
    }
}

/*
 * One output element of the block-scaled GEMM C = A * B^T with promotion of
 * each K block into an FP32 accumulator (news.qq.com page, "提高累加精度",
 * Fig. 7b):
 *   acc = 0
 *   for kb ascending:
 *     P   = exact block dot product of the decoded codes (FP64, exact)
 *     sab = fl32(sa[m, kb] * sb[n / 128, kb])
 *     acc = fl32(acc + fl32(fl32(P) * sab))
 * Also returns S = sum_k |dec(qa) * sa * dec(qb) * sb| in FP64, the scale of
 * the acceptance bound.
 *   qa [M, K], sa [M, KB]; qb [N, K], sb [ceil(N/g), KB]; row-major, where
 *   g is the number of B rows sharing one scale row: 128 for a weight
 *   quantized in 128x128 blocks, 1 for an operand quantized in 1x128 tiles.
 */
static void gemm_element(const double* dec, const uint8_t* qa, const float* sa,
                         const uint8_t* qb, const float* sb, int64_t g, int64_t K, int64_t m,
                         int64_t n, float* c32, double* S) {
    int64_t KB = (K + TILE - 1) / TILE;
    float acc = 0.0f;
    double bound = 0.0;
    for (int64_t kb = 0; kb < KB; ++kb) {
        int64_t k0 = kb * TILE;
        int64_t k1 = k0 + TILE < K ? k0 + TILE : K;
        double P = 0.0, Pabs = 0.0;
        for (int64_t k = k0; k < k1; ++k) {
            double prod = dec[qa[m * K + k]] * dec[qb[n * K + k]];
            P += prod;
            Pabs += fabs(prod);
        }
        float a_s = sa[m * KB + kb];
        float b_s = sb[(n / g) * KB + kb];
        float sab = a_s * b_s;
        float t = (float)P * sab;
        acc = acc + t;
        bound += Pabs * fabs((double)a_s) * fabs((double)b_s);
    }
    *c32 = acc;
    *S = bound;
}

/* The 256 decoded code values, dec[c] = fp8o_e4m3_decode(c). */
static void decode_table(double dec[256]) {
    for (int c = 0; c < 256; ++c) dec[c] = fp8o_e4m3_decode((uint8_t)c);
}

/*
 * The GEMM at selected outputs: for i < nrows, j < ncols, the element
 * (rows[i], cols[j]) goes to c32[i * ncols + j] and its bound to S[...].
 */
void fp8o_gemm(const uint8_t* qa, const float* sa, const uint8_t* qb, const float* sb,
               int64_t K, const int64_t* rows, int64_t nrows, const int64_t* cols,
               int64_t ncols, float* c32, double* S) {
    double dec[256];
    decode_table(dec);
    for (int64_t i = 0; i < nrows; ++i)
        for (int64_t j = 0; j < ncols; ++j)
            gemm_element(dec, qa, sa, qb, sb, TILE, K, rows[i], cols[j], &c32[i * ncols + j],
                         &S[i * ncols + j]);
}

/*
 * The weight-gradient GEMM of the backward pass, at selected outputs. The
 * news.qq.com page's pipeline figure ("DualPipe" overlap, "backward for
 * weights") and its FP8 section (Fig. 7: the linear layers' GEMMs run in
 * FP8) put this contraction in FP8 too; the pages do not spell out its
 * quantization. Reading taken: dW = dY^T X contracts over tokens, so both
 * operands are activations quantized in 1x128 tiles along the token axis
 * (128x1 tiles of dY [T, N] and X [T, K]), stored transposed:
 *   qa = codes of dY^T [N, T], sa [N, ceil(T/128)]
 *   qb = codes of X^T  [K, T], sb [K, ceil(T/128)]
 * and the result is dW [N, K] = A * B^T, promoted per 128-token block
 * exactly as the forward GEMM, with one B scale per row instead of per
 * 128-row block. Here M, N and K are the rows of A, the rows of B and the
 * contraction length.
 */
void fp8o_wgrad_gemm(const uint8_t* qa, const float* sa, const uint8_t* qb, const float* sb,
                     int64_t K, const int64_t* rows, int64_t nrows, const int64_t* cols,
                     int64_t ncols, float* c32, double* S) {
    double dec[256];
    decode_table(dec);
    for (int64_t i = 0; i < nrows; ++i)
        for (int64_t j = 0; j < ncols; ++j)
            gemm_element(dec, qa, sa, qb, sb, 1, K, rows[i], cols[j], &c32[i * ncols + j],
                         &S[i * ncols + j]);
}

/*
 * The grouped (per-expert) GEMM at selected outputs. Row m of A belongs to
 * the expert e with off[e] <= m < off[e+1] (offsets nondecreasing, off[0] = 0,
 * off[E] = total rows); its output row is A[m] * B_e^T with
 *   B_e  = qb + e * N * K        (expert weights [E][N][K])
 *   sb_e = sb + e * NB * KB      (expert scales [E][ceil(N/128)][KB]).
 * The MoE FFN runs the routed experts' GEMMs this way (news.qq.com page,
 * "DeepSeekMoE 架构": 256 routed experts, 8 per token).
 */
void fp8o_grouped_gemm(const uint8_t* qa, const float* sa, const uint8_t* qb,
                       const float* sb, const int32_t* off, int32_t E, int64_t N,
                       int64_t K, const int64_t* rows, int64_t nrows, const int64_t* cols,
                       int64_t ncols, float* c32, double* S) {
    int64_t KB = (K + TILE - 1) / TILE;
    int64_t NB = (N + TILE - 1) / TILE;
    double dec[256];
    decode_table(dec);
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t m = rows[i];
        int32_t e = 0;
        while (e < E && !(off[e] <= m && m < off[e + 1])) ++e;
        for (int64_t j = 0; j < ncols; ++j) {
            if (e == E) { /* row outside every expert: no output defined */
                c32[i * ncols + j] = NAN;
                S[i * ncols + j] = NAN;
                continue;
            }
            gemm_element(dec, qa, sa, qb + (int64_t)e * N * K, sb + (int64_t)e * NB * KB, TILE,
                         K, m, cols[j], &c32[i * ncols + j], &S[i * ncols + j]);
        }
    }
}

/*
 * nvfp4_oracle.c -- plain, slow, single-threaded CPU reference for the NVFP4
 * weight x bf16 activation path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may include, link,
 * load or call this file: only the test suite, the smoke check and the CPU
 * baseline leg of the benchmark use it.  It shares no code, header, table or
 * helper with the CUDA library.
 *
 * What it follows:
 *   - The NVFP4 weight format: 4-bit E2M1 codes packed two per byte, one
 *     FP8-E4M3 scale per 16 consecutive elements along K, and one FP32 scale
 *     per tensor.  The pages name the format and its block scaling (bw24
 *     README, section on the NVFP4 / Q4_0 decode path; bw24 wiki Home, feature
 *     list, NVFP4 decode path entry; qwentin README, section "Why it's
 *     interesting", where 4-bit E2M1 weights are the NVFP4 quality tier).
 *   - The quantisation recipe of the library's problem statement: tensor
 *     scale = amax / (6*448); block scale = E4M3 round-to-nearest-even of
 *     (block amax / 6) / tensor scale; code = nearest E2M1 value of
 *     w / (block scale * tensor scale), clamped to +-6.  Every step is done
 *     in fp32, in the order written, with IEEE round-to-nearest-even.
 *   - The FP6 E2M3 block-scaled variant of the weights (section at the end
 *     of this file): codes, 128-wide UE8M0 block scales, its quantiser and
 *     product, with the readings it takes stated there.
 *   - The product y[N,M] = x[N,K] . dequant(W[M,K])^T, computed here in fp64
 *     in k order.  Checking every quantised kernel against a CPU reference is
 *     the first gate of the bw24 wiki Home page (list of checks every kernel
 *     change must pass).
 *
 * Readings where the statement is silent (each one is listed in the design
 * notes of the repository):
 *   - ties go to the even code, for E4M3 and for E2M1;
 *   - a small negative value that rounds to magnitude 0 keeps its sign
 *     (code 0x8), as any round-to-nearest conversion does;
 *   - a block whose decoded scale times the tensor scale is 0 (scale byte 0,
 *     or an all-zero tensor) gets all-zero codes (0x0) and is not divided;
 *   - non-finite weights are outside the format: quantise returns an error;
 *   - layout: codes[m][k/2] with even k in the low nibble; scales[m][k/16].
 *
 * Parity pins (what makes this file trustworthy) live in tests/: brute-force
 * nearest-value searches over all 16 E2M1 codes and all 127 finite positive
 * E4M3 bytes, PyTorch's float8_e4m3fn decode and cast, a hand-worked 16-value
 * block, exact rational arithmetic on tiny products, and closed forms.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

/* ------------------------------------------------------------------------- */
/* Element formats                                                           */
/* ------------------------------------------------------------------------- */

/* E2M1: bit 3 sign, bits 2..1 exponent (bias 1), bit 0 mantissa.
 * Exponent field 0 is subnormal: value = m * 0.5.
 * Otherwise value = 2^(e-1) * (1 + m/2).  Magnitudes: 0 .5 1 1.5 2 3 4 6. */
double nvfp4_oracle_e2m1_value(int code)
{
    int s = (code >> 3) & 1;
    int e = (code >> 1) & 3;
    int m = code & 1;
    double mag = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return s ? -mag : mag;
}

/* E4M3 (OCP FP8 "E4M3FN"): bit 7 sign, bits 6..3 exponent (bias 7), bits 2..0
 * mantissa.  Exponent field 0 is subnormal: value = m/8 * 2^-6.  No infinity;
 * exponent 15 with mantissa 7 is NaN.  Largest finite magnitude 448. */
double nvfp4_oracle_e4m3_value(int byte)
{
    int s = (byte >> 7) & 1;
    int e = (byte >> 3) & 15;
    int m = byte & 7;
    if (e == 15 && m == 7)
        return NAN;
    double mag = (e == 0) ? ldexp(m / 8.0, -6) : ldexp(1.0 + m / 8.0, e - 7);
    return s ? -mag : mag;
}

/* fp32 -> E4M3, round to nearest with ties to the even mantissa, saturating to
 * the largest finite value 448 (byte 0x7E) instead of overflowing.
 * Subnormals (multiples of 2^-9 below 2^-6) are produced. */
uint8_t nvfp4_oracle_e4m3_encode(float qf)
{
    uint8_t sign = signbit(qf) ? 0x80 : 0x00;
    if (isnan(qf))
        return (uint8_t)(sign | 0x7F);
    double q = fabs((double)qf);
    if (q >= 448.0)
        return (uint8_t)(sign | 0x7E);
    if (q == 0.0)
        return sign;
    int E;
    frexp(q, &E);              /* q in [2^(E-1), 2^E) */
    int e = E - 1;             /* unbiased exponent of q */
    if (e < -6)
        e = -6;                /* subnormals share the smallest binade's spacing */
    double quantum = ldexp(1.0, e - 3);          /* 3 mantissa bits */
    double v = rint(q / quantum) * quantum;      /* q/quantum is exact; rint = ties-to-even */
    if (v == 0.0)
        return sign;
    if (v >= 448.0)
        return (uint8_t)(sign | 0x7E);
    if (v < ldexp(1.0, -6))                      /* subnormal: m * 2^-9 */
        return (uint8_t)(sign | (int)(v / ldexp(1.0, -9)));
    frexp(v, &E);
    int ev = E - 1;
    int mant = (int)((v / ldexp(1.0, ev) - 1.0) * 8.0);
    return (uint8_t)(sign | ((ev + 7) << 3) | mant);
}

/* fp32 -> E2M1: nearest magnitude on {0, .5, 1, 1.5, 2, 3, 4, 6}, ties to the
 * even code (the even mantissa bit), magnitudes of 6 and above clamp to 6,
 * sign bit = sign bit of the input (so -0.2 -> 0x8). */
uint8_t nvfp4_oracle_e2m1_encode(float vf)
{
    uint8_t sign = signbit(vf) ? 0x8 : 0x0;
    double a = fabs((double)vf);
    int code;
    if (a >= 6.0) {
        code = 7;
    } else {
        double quantum = (a < 2.0) ? 0.5 : (a < 4.0) ? 1.0 : 2.0;
        double v = rint(a / quantum) * quantum;  /* ties to the even multiple */
        if (v < 2.0)
            code = (int)(v * 2.0);               /* 0, .5, 1, 1.5 -> 0..3 */
        else if (v < 4.0)
            code = (int)(v + 2.0);               /* 2, 3 -> 4, 5 */
        else
            code = (int)(v / 2.0 + 4.0);         /* 4, 6 -> 6, 7 */
    }
    return (uint8_t)(sign | code);
}

/* bf16 bit pattern -> exact double. */
static double bf16_value(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* ------------------------------------------------------------------------- */
/* Quantiser                                                                  */
/* ------------------------------------------------------------------------- */

/* Quantise an fp32 row-major w[M][K] (K a multiple of 16) to
 *   codes[M][K/2]  (element 2j in the low nibble of byte j, 2j+1 in the high)
 *   scales[M][K/16] (E4M3 bytes)
 *   *tensor_scale  (fp32).
 * Returns 0, or -1 for a bad shape, -2 for a non-finite weight. */
int nvfp4_oracle_quantize(const float *w, int64_t M, int64_t K,
                          uint8_t *codes, uint8_t *scales, float *tensor_scale)
{
    if (M < 0 || K < 0 || K % 16 != 0)
        return -1;

    /* Step 1: amax over the whole tensor (exact). */
    float amax = 0.0f;
    for (int64_t i = 0; i < M * K; ++i) {
        float a = fabsf(w[i]);
        if (!isfinite(a))
            return -2;
        if (a > amax)
            amax = a;
    }

    /* Step 2: tensor scale, one fp32 division (6*448 = 2688 is exact). */
    float ts = amax / 2688.0f;
    *tensor_scale = ts;

    const int64_t nb = K / 16;
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t b = 0; b < nb; ++b) {
            const float *blk = w + m * K + 16 * b;

            /* Step 3a: block amax. */
            float bamax = 0.0f;
            for (int j = 0; j < 16; ++j) {
                float a = fabsf(blk[j]);
                if (a > bamax)
                    bamax = a;
            }

            /* Step 3b: block scale byte = E4M3_RNE_sat((bamax / 6) / ts). */
            uint8_t sb = 0;
            if (ts > 0.0f) {
                float q = (bamax / 6.0f) / ts;
                sb = nvfp4_oracle_e4m3_encode(q);
            }
            scales[m * nb + b] = sb;

            /* Step 3c: decoded divisor d = dec(sb) * ts, one fp32 rounding. */
            float s = (float)nvfp4_oracle_e4m3_value(sb);
            float d = s * ts;

            /* Step 3d: codes = nearestE2M1(w / d); a zero divisor gives 0x0. */
            uint8_t c[16];
            for (int j = 0; j < 16; ++j)
                c[j] = (d == 0.0f) ? 0 : nvfp4_oracle_e2m1_encode(blk[j] / d);

            /* Step 4: pack two codes per byte, even k in the low nibble. */
            uint8_t *out = codes + m * (K / 2) + 8 * b;
            for (int j = 0; j < 8; ++j)
                out[j] = (uint8_t)(c[2 * j] | (c[2 * j + 1] << 4));
        }
    }
    return 0;
}

/* Decode one weight exactly: ts is applied by the caller. */
static double weight_unscaled(const uint8_t *codes, const uint8_t *scales,
                              int64_t K, int64_t m, int64_t k)
{
    uint8_t byte = codes[m * (K / 2) + k / 2];
    int code = (k & 1) ? (byte >> 4) : (byte & 0xF);
    return nvfp4_oracle_e2m1_value(code) *
           nvfp4_oracle_e4m3_value(scales[m * (K / 16) + k / 16]);
}

/* ------------------------------------------------------------------------- */
/* Products                                                                   */
/* ------------------------------------------------------------------------- */

/* y[i][j] = ts * sum_k w_unscaled(rows[j], k) * x[tokens[i]][k]   (fp64, k order)
 * A[i][j] = |ts| * sum_k |w_unscaled(rows[j], k) * x[tokens[i]][k]|
 *
 * x is bf16 bits, row-major [N_total][K].  rows / tokens may be NULL, meaning
 * all M rows / all N_total tokens in order; otherwise n_rows / n_tokens
 * indices.  A is the scale of the accuracy bound |y - y_ref| <= 1e-5*A + 1e-7
 * and may be NULL. */
void nvfp4_oracle_gemv(const uint16_t *x, int64_t N_total, int64_t K,
                       const int64_t *tokens, int64_t n_tokens,
                       const uint8_t *codes, const uint8_t *scales, float ts,
                       int64_t M, const int64_t *rows, int64_t n_rows,
                       double *y, double *A)
{
    if (tokens == NULL)
        n_tokens = N_total;
    if (rows == NULL)
        n_rows = M;
    for (int64_t i = 0; i < n_tokens; ++i) {
        int64_t n = tokens ? tokens[i] : i;
        const uint16_t *xn = x + n * K;
        for (int64_t j = 0; j < n_rows; ++j) {
            int64_t m = rows ? rows[j] : j;
            double sum = 0.0, asum = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double t = weight_unscaled(codes, scales, K, m, k) * bf16_value(xn[k]);
                sum += t;
                asum += fabs(t);
            }
            y[i * n_rows + j] = (double)ts * sum;
            if (A)
                A[i * n_rows + j] = fabs((double)ts) * asum;
        }
    }
}

/* SwiGLU of two products that share x, rows and tokens:
 *   h = silu(g) * u,  silu(g) = g / (1 + exp(-g)),
 * where g and u are nvfp4_oracle_gemv of the gate and up weights.  Also
 * returns g, u and their bound scales Ag, Au (any of them may be NULL). */
void nvfp4_oracle_swiglu(const uint16_t *x, int64_t N_total, int64_t K,
                         const int64_t *tokens, int64_t n_tokens,
                         const uint8_t *g_codes, const uint8_t *g_scales, float g_ts,
                         const uint8_t *u_codes, const uint8_t *u_scales, float u_ts,
                         int64_t M, const int64_t *rows, int64_t n_rows,
                         double *h, double *g, double *u, double *Ag, double *Au)
{
    if (tokens == NULL)
        n_tokens = N_total;
    if (rows == NULL)
        n_rows = M;
    for (int64_t i = 0; i < n_tokens; ++i) {
        int64_t tok = tokens ? tokens[i] : i;
        for (int64_t j = 0; j < n_rows; ++j) {
            int64_t row = rows ? rows[j] : j;
            double gv, uv, ag, au;
            nvfp4_oracle_gemv(x, N_total, K, &tok, 1, g_codes, g_scales, g_ts,
                              M, &row, 1, &gv, &ag);
            nvfp4_oracle_gemv(x, N_total, K, &tok, 1, u_codes, u_scales, u_ts,
                              M, &row, 1, &uv, &au);
            int64_t o = i * n_rows + j;
            h[o] = gv / (1.0 + exp(-gv)) * uv;
            if (g) g[o] = gv;
            if (u) u[o] = uv;
            if (Ag) Ag[o] = ag;
            if (Au) Au[o] = au;
        }
    }
}

/* ------------------------------------------------------------------------- */
/* FP6 E2M3 block-scaled weights                                              */
/* ------------------------------------------------------------------------- */
/*
 * The FP6 variant of the weight format (qwentin README, "Highlights" and
 * "How it works": E2M3 weights, block-scaled, 128-wide block scales, fed to the
 * block-scaled tensor-core MMA of kind mxf8f6f4).  The pages give no more than
 * that; the readings below take the OCP microscaling (MX) conversion rule the
 * named MMA kind is built for, with blocks of 128 instead of 32:
 *   - element: E2M3, bit 5 sign, bits 4..3 exponent (bias 1), bits 2..0
 *     mantissa; exponent 0 is subnormal (m/8); largest magnitude 7.5;
 *   - block scale: one UE8M0 byte s per 128 consecutive k of a row, value
 *     2^(s-127); no tensor scale;
 *   - quantise a block: shared exponent = floor(log2(block amax)) - 2 (2 is
 *     the exponent of E2M3's largest normal, 7.5 = 1.875 * 2^2), raised to -127
 *     when lower (and -127 for an all-zero block); each element is the nearest
 *     E2M3 value to w / 2^shared (an fp32 division), ties to the even code,
 *     magnitudes above 7.5 saturating to 7.5, the sign kept;
 *   - layout: codes[m][3K/4], each row a little-endian bit stream of 6-bit
 *     codes (element k at bits 6k..6k+5, so four codes fill three bytes);
 *     scales[m][K/128].  K must be a multiple of 128.
 */

double nvfp4_oracle_e2m3_value(int code)
{
    int e = (code >> 3) & 3, m = code & 7;
    double mag = (e == 0) ? m / 8.0 : ldexp(1.0 + m / 8.0, e - 1);
    return (code & 0x20) ? -mag : mag;
}

/* fp32 -> E2M3: nearest of the 32 magnitudes (a search over all of them),
 * ties to the even code, saturating at 7.5, sign bit of the input kept. */
uint8_t nvfp4_oracle_e2m3_encode(float vf)
{
    double a = fabs((double)vf);
    int best = 0;
    double best_d = INFINITY;
    for (int c = 0; c < 32; ++c) {
        double d = fabs(nvfp4_oracle_e2m3_value(c) - a);
        if (d < best_d || (d == best_d && (c & 1) == 0)) {
            best = c;
            best_d = d;
        }
    }
    return (uint8_t)(best | (signbit(vf) ? 0x20 : 0));
}

static void put_code6(uint8_t *row, int64_t k, unsigned code)
{
    int64_t bit = 6 * k;
    unsigned v = (code & 63u) << (bit % 8);  /* at most 14 bits */
    row[bit / 8] |= (uint8_t)(v & 0xFF);
    if (v >> 8)
        row[bit / 8 + 1] |= (uint8_t)(v >> 8);
}

static int get_code6(const uint8_t *row, int64_t k)
{
    int64_t bit = 6 * k;
    unsigned v = row[bit / 8];
    if (bit % 8 > 2)
        v |= (unsigned)row[bit / 8 + 1] << 8;
    return (int)((v >> (bit % 8)) & 63u);
}

/* Quantise fp32 w[M][K] (K % 128 == 0) to FP6 E2M3 codes and UE8M0 scales.
 * Returns 0, -1 for a bad shape, -2 for a non-finite weight. */
int nvfp4_oracle_fp6_quantize(const float *w, int64_t M, int64_t K,
                              uint8_t *codes, uint8_t *scales)
{
    if (M < 0 || K < 0 || K % 128 != 0)
        return -1;
    for (int64_t i = 0; i < M * K; ++i)
        if (!isfinite(w[i]))
            return -2;
    const int64_t row_bytes = K / 8 * 6;
    memset(codes, 0, (size_t)(M * row_bytes));
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t b = 0; b < K / 128; ++b) {
            const float *blk = w + m * K + 128 * b;
            /* Step 1: block amax. */
            float amax = 0.0f;
            for (int i = 0; i < 128; ++i)
                if (fabsf(blk[i]) > amax)
                    amax = fabsf(blk[i]);
            /* Step 2: shared exponent and the UE8M0 scale byte. */
            int shared = -127;
            if (amax > 0.0f) {
                int e;
                frexpf(amax, &e);           /* amax = f * 2^e, f in [0.5, 1) */
                shared = (e - 1) - 2;       /* floor(log2(amax)) - 2 */
                if (shared < -127)
                    shared = -127;
            }
            scales[m * (K / 128) + b] = (uint8_t)(shared + 127);
            const float X = ldexpf(1.0f, shared);  /* exact; 2^-127 is subnormal */
            /* Step 3: elements. */
            for (int i = 0; i < 128; ++i)
                put_code6(codes + m * row_bytes, 128 * b + i,
                          nvfp4_oracle_e2m3_encode(blk[i] / X));
        }
    }
    return 0;
}

/* One FP6 weight, exactly. */
static double fp6_weight(const uint8_t *codes, const uint8_t *scales,
                         int64_t K, int64_t m, int64_t k)
{
    int code = get_code6(codes + m * (K / 8 * 6), k);
    return nvfp4_oracle_e2m3_value(code) *
           ldexp(1.0, (int)scales[m * (K / 128) + k / 128] - 127);
}

/* y[i][j] = sum_k w(rows[j], k) * x[tokens[i]][k]  (fp64, k order), and
 * A[i][j] = sum_k |w * x| (may be NULL); rows / tokens as for nvfp4_oracle_gemv. */
void nvfp4_oracle_fp6_gemv(const uint16_t *x, int64_t N_total, int64_t K,
                           const int64_t *tokens, int64_t n_tokens,
                           const uint8_t *codes, const uint8_t *scales,
                           int64_t M, const int64_t *rows, int64_t n_rows,
                           double *y, double *A)
{
    if (tokens == NULL)
        n_tokens = N_total;
    if (rows == NULL)
        n_rows = M;
    for (int64_t i = 0; i < n_tokens; ++i) {
        int64_t n = tokens ? tokens[i] : i;
        const uint16_t *xrow = x + n * K;
        for (int64_t j = 0; j < n_rows; ++j) {
            int64_t m = rows ? rows[j] : j;
            double sum = 0.0, asum = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double t = fp6_weight(codes, scales, K, m, k) * bf16_value(xrow[k]);
                sum += t;
                asum += fabs(t);
            }
            y[i * n_rows + j] = sum;
            if (A)
                A[i * n_rows + j] = asum;
        }
    }
}

/* ------------------------------------------------------------------------- */
/* W4A4: activations quantised to NVFP4 as well                               */
/* ------------------------------------------------------------------------- */
/*
 * The opt-in prefill arm that quantises the activations to FP4 too (bw24
 * README, Gemma section, the paragraph on prefill against llama.cpp: W4A4 with
 * FP4 activations is faster but a different numeric class, which forks outputs
 * on long prompts).  Readings, since the page names the class and nothing
 * more:
 *   - the activation matrix x[N][K] is one NVFP4 tensor, quantised by the same
 *     recipe as the weights (its bf16 elements taken as their exact fp32
 *     values): one tensor scale for the whole matrix, one E4M3 scale per 16
 *     consecutive k of a token row, E2M1 codes, the same layout;
 *   - the product is the plain definition with both operands decoded exactly:
 *     y[n][m] = ts_x * ts_w * sum_k e2m1(cx) e4m3(sx) e2m1(cw) e4m3(sw).
 * Every term is exact in fp64 (at most 12 significant bits); the sum runs in
 * k order and the two fp32 tensor scales multiply it at the end. */
void nvfp4_oracle_w4a4_gemm(const uint8_t *x_codes, const uint8_t *x_scales, float x_ts,
                            int64_t N_total, int64_t K, const int64_t *tokens, int64_t n_tokens,
                            const uint8_t *codes, const uint8_t *scales, float ts,
                            int64_t M, const int64_t *rows, int64_t n_rows,
                            double *y, double *A)
{
    if (tokens == NULL)
        n_tokens = N_total;
    if (rows == NULL)
        n_rows = M;
    const double scale = (double)x_ts * (double)ts;  /* exact: 24 + 24 bits */
    for (int64_t i = 0; i < n_tokens; ++i) {
        int64_t n = tokens ? tokens[i] : i;
        for (int64_t j = 0; j < n_rows; ++j) {
            int64_t m = rows ? rows[j] : j;
            double sum = 0.0, asum = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double t = weight_unscaled(x_codes, x_scales, K, n, k) *
                           weight_unscaled(codes, scales, K, m, k);
                sum += t;
                asum += fabs(t);
            }
            y[i * n_rows + j] = scale * sum;
            if (A)
                A[i * n_rows + j] = fabs(scale) * asum;
        }
    }
}

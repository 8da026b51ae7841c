/*
 * Plain CPU oracle for the W8A8 INT8 Linear path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header, table or helper with the
 * CUDA library.
 *
 * What it computes follows "TurboDiffusion Integration Notes" (TurboT2AV
 * docs/acceleration.md):
 *   - section "Reused Components", bullet "W8A8 Linear": weights are quantized
 *     to INT8 once, activations are quantized dynamically before every Linear;
 *   - section "Differences From TurboDiffusion", row "W8A8 kernel" and the
 *     paragraph under the table: the post-scale kernel keeps the integer
 *     accumulation continuous over K and applies the activation and weight
 *     scales in the epilogue; the original kernel is blockwise-scaled.
 * The pages give no formula.  The readings taken here (every one is listed in
 * the design notes) are:
 *   - symmetric quantizer: s = absmax / 127 (IEEE fp32 division),
 *     q = clamp(round_half_even(x / s), -127, 127), x / s an IEEE fp32 division;
 *     absmax == 0 gives s = 0 and q = 0 for the whole group;
 *   - groups: activations per token (a whole row) or per 1x128 block of a row;
 *     weights per output channel (a whole row of W[N,K]) or per 128x128 block;
 *   - post-scale epilogue: y = ((float(acc) * sx[m]) * sw[n]) + bias[n], each
 *     operation rounded to fp32 on its own, the bias add skipped when there is
 *     no bias, then y rounded to bf16 (nearest, ties to even);
 *   - blockwise: for each 128-wide K block kb in ascending order,
 *     P = sum of the block's int8 products (exact int32),
 *     t = (float(P) * sx[m,kb]) * sw[n/128,kb], acc = acc + t from acc = 0.0f;
 *     then (+ bias) and bf16 rounding as above.
 *
 * Build with -O2 -ffp-contract=off -fno-fast-math so that no multiply-add is
 * fused and every fp32 operation is rounded on its own.  Rows are spread over
 * OpenMP threads; nothing else is reordered.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_QMAX 127
#define ORC_BLOCK 128

/* bf16 is the top half of an IEEE binary32, so widening is a shift. */
static float orc_bf16_to_f32(uint16_t h) {
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round a binary32 to the nearest bf16, ties to even (IEEE 754 roundTiesToEven
 * applied to the 16 dropped bits).  NaN stays a quiet NaN. */
static uint16_t orc_f32_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7f800000u) == 0x7f800000u) {
        uint16_t hi = (uint16_t)(u >> 16);
        if (u & 0x007fffffu) hi |= 0x0040u; /* NaN: keep it a NaN */
        return hi;
    }
    uint32_t dropped = u & 0xffffu;
    uint32_t keep = u >> 16;
    if (dropped > 0x8000u || (dropped == 0x8000u && (keep & 1u))) keep += 1u;
    return (uint16_t)keep;
}

/* Scale of a group from its absolute maximum: s = absmax / 127. */
static float orc_scale_of(float absmax) { return absmax / (float)ORC_QMAX; }

/* One quantized value: round_half_even(x / s) clamped to [-127, 127].
 * nearbyintf rounds in the current mode, which is round-to-nearest-even by
 * default; the division is an IEEE binary32 division. */
static int8_t orc_q(float x, float s) {
    if (s == 0.0f) return 0;
    float r = nearbyintf(x / s);
    if (r > (float)ORC_QMAX) r = (float)ORC_QMAX;
    if (r < -(float)ORC_QMAX) r = -(float)ORC_QMAX;
    return (int8_t)r;
}

int orc_version(void) { return 1; }

int orc_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void orc_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

void orc_bf16_from_f32(const float* x, int64_t n, uint16_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_f32_to_bf16(x[i]);
}

void orc_f32_from_bf16(const uint16_t* x, int64_t n, float* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_bf16_to_f32(x[i]);
}

/* Quantize the rows of A[R,K] (bf16 bits) in groups of `group` consecutive
 * elements (group == K: one scale per row; group == 128: one per 1x128 block).
 * Writes Aq[R,K] and s[R, K/group]. */
static void orc_quant_rows(const uint16_t* A, int64_t R, int64_t K, int64_t group,
                           int8_t* Aq, float* s) {
    int64_t ng = K / group;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < R; ++r) {
        const uint16_t* a = A + r * K;
        for (int64_t g = 0; g < ng; ++g) {
            float amax = 0.0f;
            for (int64_t k = g * group; k < (g + 1) * group; ++k) {
                float v = fabsf(orc_bf16_to_f32(a[k]));
                if (v > amax) amax = v;
            }
            float sc = orc_scale_of(amax);
            s[r * ng + g] = sc;
            for (int64_t k = g * group; k < (g + 1) * group; ++k)
                Aq[r * K + k] = orc_q(orc_bf16_to_f32(a[k]), sc);
        }
    }
}

/* Activation quantization.  mode 0: per token, sx[M].  mode 1: per 1x128 block,
 * sx[M][K/128] (K must be a multiple of 128).  Returns 0, or -1 on bad shape. */
int orc_quantize_act(const uint16_t* X, int64_t M, int64_t K, int mode, int8_t* Xq, float* sx) {
    if (M < 0 || K <= 0) return -1;
    if (mode == 0) {
        orc_quant_rows(X, M, K, K, Xq, sx);
        return 0;
    }
    if (mode == 1) {
        if (K % ORC_BLOCK) return -1;
        orc_quant_rows(X, M, K, ORC_BLOCK, Xq, sx);
        return 0;
    }
    return -1;
}

/* Weight quantization.  mode 0: per output channel, sw[N].  mode 1: per
 * 128x128 block, sw[ceil(N/128)][K/128]; a last, partial row block takes the
 * absmax over the rows it has.  Returns 0, or -1 on bad shape. */
int orc_quantize_weight(const uint16_t* W, int64_t N, int64_t K, int mode, int8_t* Wq, float* sw) {
    if (N < 0 || K <= 0) return -1;
    if (mode == 0) {
        orc_quant_rows(W, N, K, K, Wq, sw);
        return 0;
    }
    if (mode != 1 || K % ORC_BLOCK) return -1;
    int64_t nb_count = (N + ORC_BLOCK - 1) / ORC_BLOCK;
    int64_t kb_count = K / ORC_BLOCK;
#pragma omp parallel for schedule(static)
    for (int64_t nb = 0; nb < nb_count; ++nb) {
        int64_t n0 = nb * ORC_BLOCK;
        int64_t n1 = n0 + ORC_BLOCK < N ? n0 + ORC_BLOCK : N;
        for (int64_t kb = 0; kb < kb_count; ++kb) {
            float amax = 0.0f;
            for (int64_t n = n0; n < n1; ++n)
                for (int64_t k = kb * ORC_BLOCK; k < (kb + 1) * ORC_BLOCK; ++k) {
                    float v = fabsf(orc_bf16_to_f32(W[n * K + k]));
                    if (v > amax) amax = v;
                }
            float sc = orc_scale_of(amax);
            sw[nb * kb_count + kb] = sc;
            for (int64_t n = n0; n < n1; ++n)
                for (int64_t k = kb * ORC_BLOCK; k < (kb + 1) * ORC_BLOCK; ++k)
                    Wq[n * K + k] = orc_q(orc_bf16_to_f32(W[n * K + k]), sc);
        }
    }
    return 0;
}

/* acc[m,n] = sum_k Xq[m,k] * Wq[n,k] in int32, k ascending (the sum is exact:
 * |acc| <= 127*127*K < 2^31 for K <= 131072). */
void orc_gemm_s32(const int8_t* Xq, const int8_t* Wq, int64_t M, int64_t N, int64_t K, int32_t* acc) {
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m) {
        const int8_t* x = Xq + m * K;
        for (int64_t n = 0; n < N; ++n) {
            const int8_t* w = Wq + n * K;
            int32_t a = 0;
            for (int64_t k = 0; k < K; ++k) a += (int32_t)x[k] * (int32_t)w[k];
            acc[m * N + n] = a;
        }
    }
}

/* Post-scale epilogue: Y[m,n] = bf16(((float(acc) * sx[m]) * sw[n]) + bias[n]).
 * bias is bf16 bits or NULL (then the add is skipped). */
void orc_epilogue_postscale(const int32_t* acc, const float* sx, const float* sw,
                            const uint16_t* bias, int64_t M, int64_t N, uint16_t* Y) {
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            float y = (float)acc[m * N + n];
            y = y * sx[m];
            y = y * sw[n];
            if (bias) y = y + orc_bf16_to_f32(bias[n]);
            Y[m * N + n] = orc_f32_to_bf16(y);
        }
    }
}

/* Blockwise-scaled accumulation (pre-bf16): for kb ascending,
 * P = sum over the block of Xq*Wq (int32), t = (float(P) * sx[m,kb]) * sw[n/128,kb],
 * acc += t, from acc = 0.0f.  sx is [M][K/128], sw is [ceil(N/128)][K/128]. */
void orc_gemm_blockwise_f32(const int8_t* Xq, const float* sx, const int8_t* Wq, const float* sw,
                            int64_t M, int64_t N, int64_t K, float* acc) {
    int64_t kb_count = K / ORC_BLOCK;
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m) {
        const int8_t* x = Xq + m * K;
        for (int64_t n = 0; n < N; ++n) {
            const int8_t* w = Wq + n * K;
            const float* swb = sw + (n / ORC_BLOCK) * kb_count;
            float a = 0.0f;
            for (int64_t kb = 0; kb < kb_count; ++kb) {
                int32_t p = 0;
                for (int64_t k = kb * ORC_BLOCK; k < (kb + 1) * ORC_BLOCK; ++k)
                    p += (int32_t)x[k] * (int32_t)w[k];
                float t = (float)p * sx[m * kb_count + kb];
                t = t * swb[kb];
                a = a + t;
            }
            acc[m * N + n] = a;
        }
    }
}

/* Blockwise epilogue: Y = bf16(acc + bias[n]) (add skipped without bias). */
void orc_epilogue_blockwise(const float* acc, const uint16_t* bias, int64_t M, int64_t N, uint16_t* Y) {
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            float y = acc[m * N + n];
            if (bias) y = y + orc_bf16_to_f32(bias[n]);
            Y[m * N + n] = orc_f32_to_bf16(y);
        }
}

/* ------------------------------------------------------------------------
 * FFN up-projection activation: GELU, then 1x128 quantization of its output.
 *
 * The pages tune the post-scale kernel for "LTX FFN shapes" ("TurboDiffusion
 * Integration Notes", section "Differences From TurboDiffusion") and name no
 * activation.  Reading taken: the FFN's activation is GELU in its erf form,
 *   gelu(x) = x * Phi(x),  Phi(x) = (1 + erf(x / sqrt 2)) / 2,
 * applied to the bf16 output of the up-projection; the value is rounded to
 * binary32 and then to bf16 (round to nearest even both times), and that
 * tensor is what the down-projection quantizes in 1x128 blocks.
 *
 * This is the plain definition, evaluated in binary64 with the C library:
 * Phi(x) is written as erfc(-x / sqrt 2) / 2, the same function as
 * (1 + erf(x / sqrt 2)) / 2 without the cancellation of 1 + erf for
 * negative x (below x = -8 the erf form is 0 in binary64 while Phi is still
 * above 1e-16).
 * ------------------------------------------------------------------------ */
static double orc_gelu_f64_one(double x) { return 0.5 * x * erfc(-x * 0.70710678118654752440); }

/* g[i] = gelu(x[i]) in binary64 (for the pins of the definition). */
void orc_gelu_f64(const double* x, int64_t n, double* g) {
    for (int64_t i = 0; i < n; ++i) g[i] = orc_gelu_f64_one(x[i]);
}

/* G = bf16(fp32(gelu(Y))) for bf16 Y (bit patterns in, bit patterns out). */
void orc_gelu_bf16(const uint16_t* y, int64_t n, uint16_t* g) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i)
        g[i] = orc_f32_to_bf16((float)orc_gelu_f64_one((double)orc_bf16_to_f32(y[i])));
}

/* ------------------------------------------------------------------------
 * Normalization fused with per-token activation quantization.
 *
 * "TurboDiffusion Integration Notes", section "Reused Components": FastNorm
 * replaces RMSNorm/LayerNorm with fused implementations, and W8A8 + FastNorm
 * is the one combined stage of the section "End-to-End Result".  The
 * acceleration overview's LayerNorm sketch (section "Custom Kernel
 * Optimizations") computes the statistics, normalizes, then applies the
 * affine transform.  Readings taken (the pages give no formula):
 *   RMSNorm:   y = (x / sqrt(mean(x^2) + eps)) * gamma
 *   LayerNorm: y = ((x - mu) / sqrt(var + eps)) * gamma + beta,
 *              mu = mean(x), var = mean((x - mu)^2)  (biased, about the mean)
 * (gamma and beta optional: a missing one is 1, resp. 0), then y is quantized
 * per token like any activation.
 *
 * orc_norm_quant is the plain definition: the statistics are sums over the
 * row in binary64 taken left to right, and every operation up to y is a
 * binary64 operation; y is then rounded to binary32 and to bf16.
 *
 * orc_norm_quant_fixed_order is a second, binary32 statement of the same
 * formulas with one fixed summation order, kept as a bit-exact description
 * of a particular evaluation (independent of any thread layout):
 *   RMSNorm:   r = 1 / sqrt(S(x*x) / K + eps),      y = bf16((x * r) * gamma)
 *   LayerNorm: mu = S(x) / K, d = x - mu,
 *              r = 1 / sqrt(S(d*d) / K + eps),      y = bf16(((d * r) * gamma) + beta)
 * with every operation rounded to binary32 on its own, sqrt and the
 * divisions IEEE, and S() the row cut into chunks of 8 consecutive elements,
 * each chunk summed left to right, the chunk sums zero-padded to P = the next
 * power of two of K/8 entries and added pairwise level by level (entry i of
 * the next level = entry 2i + entry 2i+1) down to one value.
 * ------------------------------------------------------------------------ */

/* kind 0: RMSNorm, 1: LayerNorm.  X, gamma, beta, Y are bf16 bit patterns;
 * gamma / beta may be NULL.  Writes Y[M,K] (the normalized bf16 output), then
 * its per-token quantization Xq[M,K] and sx[M].  Returns 0, or -1 for a bad
 * shape (K <= 0). */
int orc_norm_quant(const uint16_t* X, const uint16_t* gamma, const uint16_t* beta, float eps, int kind,
                   int64_t M, int64_t K, uint16_t* Y, int8_t* Xq, float* sx) {
    if (K <= 0) return -1;
    const double Kd = (double)K;
    const double epsd = (double)eps;
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m) {
        const uint16_t* x = X + m * K;
        uint16_t* y = Y + m * K;
        double mu = 0.0;
        if (kind == 1) {
            double s = 0.0;
            for (int64_t k = 0; k < K; ++k) s += (double)orc_bf16_to_f32(x[k]);
            mu = s / Kd;
        }
        double ss = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double d = (double)orc_bf16_to_f32(x[k]) - mu;
            ss += d * d;
        }
        const double rs = sqrt(ss / Kd + epsd);
        for (int64_t k = 0; k < K; ++k) {
            double v = ((double)orc_bf16_to_f32(x[k]) - mu) / rs;
            if (gamma) v = v * (double)orc_bf16_to_f32(gamma[k]);
            if (kind == 1 && beta) v = v + (double)orc_bf16_to_f32(beta[k]);
            y[k] = orc_f32_to_bf16((float)v);
        }
    }
    return orc_quantize_act(Y, M, K, 0, Xq, sx);
}

static float orc_tree_sum(float* part, int64_t P) {
    for (int64_t w = P; w > 1; w >>= 1)
        for (int64_t i = 0; i < w / 2; ++i) part[i] = part[2 * i] + part[2 * i + 1];
    return part[0];
}

static int64_t orc_pow2_at_least(int64_t n) {
    int64_t p = 1;
    while (p < n) p <<= 1;
    return p;
}

/* The fixed-order binary32 statement above.  Same arguments; returns -1 for
 * a bad shape (K % 8 != 0 or K > 65536). */
int orc_norm_quant_fixed_order(const uint16_t* X, const uint16_t* gamma, const uint16_t* beta, float eps, int kind,
                               int64_t M, int64_t K, uint16_t* Y, int8_t* Xq, float* sx) {
    if (K <= 0 || K % 8 != 0 || K > 65536) return -1;
    const int64_t C = K / 8;
    const int64_t P = orc_pow2_at_least(C);
    const float Kf = (float)K;
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m) {
        float part[65536 / 8];
        const uint16_t* x = X + m * K;
        uint16_t* y = Y + m * K;
        float mu = 0.0f;
        if (kind == 1) {
            for (int64_t c = 0; c < P; ++c) {
                float s = 0.0f;
                if (c < C) {
                    s = orc_bf16_to_f32(x[8 * c]);
                    for (int j = 1; j < 8; ++j) s = s + orc_bf16_to_f32(x[8 * c + j]);
                }
                part[c] = s;
            }
            mu = orc_tree_sum(part, P) / Kf;
        }
        for (int64_t c = 0; c < P; ++c) {
            float s = 0.0f;
            if (c < C) {
                for (int j = 0; j < 8; ++j) {
                    float d = orc_bf16_to_f32(x[8 * c + j]);
                    if (kind == 1) d = d - mu;
                    float t = d * d;
                    s = (j == 0) ? t : s + t;
                }
            }
            part[c] = s;
        }
        const float var = orc_tree_sum(part, P) / Kf;
        const float r = 1.0f / sqrtf(var + eps);
        for (int64_t k = 0; k < K; ++k) {
            float d = orc_bf16_to_f32(x[k]);
            if (kind == 1) d = d - mu;
            float v = d * r;
            if (gamma) v = v * orc_bf16_to_f32(gamma[k]);
            if (kind == 1 && beta) v = v + orc_bf16_to_f32(beta[k]);
            y[k] = orc_f32_to_bf16(v);
        }
    }
    return orc_quantize_act(Y, M, K, 0, Xq, sx);
}

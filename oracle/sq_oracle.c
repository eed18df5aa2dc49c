/*
 * CPU oracle for the SmoothQuant W8A8 INT8 linear block.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file; only the tests, the package's smoke check and the
 * benchmark's timed CPU-baseline leg do.  It shares no code, header, table or
 * constant with the CUDA path.
 *
 * What it follows ("Efficient INT8 Inference of Small NLP Models on Server
 * CPUs with PyTorch Native Stack", Xia, Cui, Cao):
 *   - Table 10 (Smooth-Dynamic): SmoothQuant smoothing followed by dynamic
 *     activation quantisation; the per-token granularity and the
 *     per-output-channel weight scale are the ones the INT8 W8A8 recipe on the
 *     same listing states (per-channel weights, per-token dynamic activations,
 *     per-token x per-channel dequantisation).
 *   - Table 3 caption: the linear block is the GEMM plus its fused post-ops
 *     (bias, activation, residual addition).
 *   - Reference list, "SmoothQuant" and "Gaussian Error Linear Units": the
 *     smoothing factor s_j = max|X_j|^alpha / max|W_j|^(1-alpha) with
 *     migration strength alpha (Table 15 lists alpha per model), and the erf
 *     form of GELU.
 * The pages print no formula for the quantiser.  Readings taken here:
 *   - X is divided by s, W is multiplied by s (the product X W^T is unchanged);
 *   - symmetric int8, clamp [-127, 127], round-half-to-even;
 *   - scale = amax / 127 as one IEEE fp32 division; codes = round(v / scale)
 *     with v and v / scale each one IEEE fp32 division (the precision in which
 *     the kernel decides the integer code);
 *   - an all-zero row gets scale 1.0f and all-zero codes;
 *   - a channel whose activation or weight max is zero gets s_j = 1.
 * GEMM: exact integer sum in int64, checked against the int32 range.
 * Epilogue: evaluated in double from the exact integer sum and the fp32
 * scales, rounded once to fp32.
 *
 * Scalar loops, no blocking.  Rows are independent, so the outer row loops
 * carry an OpenMP pragma (it changes no arithmetic: every output is still
 * computed by the same scalar loop in the same order).
 *
 * Build: gcc -O2 -fopenmp -ffp-contract=off -fno-fast-math -shared -fPIC.
 * fp-contract is off so that no multiply-add is fused and every fp32
 * operation rounds exactly once, as written.
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_OK 0
#define ORC_ERR_ARG 1
#define ORC_ERR_OVERFLOW 2

enum { ORC_EPI_NONE = 0, ORC_EPI_BIAS = 1, ORC_EPI_BIAS_GELU = 2, ORC_EPI_BIAS_RESIDUAL = 3 };

/* Column-wise absolute maximum of a row-major rows x cols fp32 matrix:
 * out[j] = max_i |A[i][j]|.  Used for max|X_j| (over tokens) and max|W_j|
 * (over output channels) in the smoothing factor. */
int oracle_channel_absmax(const float *A, int64_t rows, int64_t cols, float *out)
{
    if (rows < 0 || cols < 0) return ORC_ERR_ARG;
    for (int64_t j = 0; j < cols; ++j) out[j] = 0.0f;
    for (int64_t i = 0; i < rows; ++i)
        for (int64_t j = 0; j < cols; ++j) {
            float a = fabsf(A[i * cols + j]);
            if (a > out[j]) out[j] = a;
        }
    return ORC_OK;
}

/* SmoothQuant smoothing factor, one per input channel j:
 *   s_j = max|X_j|^alpha / max|W_j|^(1 - alpha),
 * in double, rounded once to fp32.  A zero maximum on either side gives
 * s_j = 1 (no migration for a dead channel). */
int oracle_smooth_factor(const float *x_amax, const float *w_amax, int64_t K,
                         double alpha, float *s)
{
    if (K < 0 || !(alpha >= 0.0 && alpha <= 1.0)) return ORC_ERR_ARG;
    for (int64_t j = 0; j < K; ++j) {
        double ax = (double)x_amax[j], aw = (double)w_amax[j];
        if (ax == 0.0 || aw == 0.0) { s[j] = 1.0f; continue; }
        double v = pow(ax, alpha) / pow(aw, 1.0 - alpha);
        s[j] = (float)v;
    }
    return ORC_OK;
}

/* Smoothing alone, without quantisation (fp32, one rounding per element).
 * direction 0: activations, out = X / s (X diag(s)^-1)
 * direction 1: weights,     out = W * s (W diag(s))   */
int oracle_smooth(const float *A, const float *s, int64_t rows, int64_t K,
                  int direction, float *out)
{
    if (rows < 0 || K < 0 || (direction != 0 && direction != 1)) return ORC_ERR_ARG;
    for (int64_t i = 0; i < rows; ++i)
        for (int64_t j = 0; j < K; ++j) {
            float a = A[i * K + j];
            out[i * K + j] = direction == 0 ? a / s[j] : a * s[j];
        }
    return ORC_OK;
}

/* Symmetric per-row int8 quantisation of a smoothed row-major matrix.
 * For each row i, with v_ij the smoothed value (X/s or W*s, fp32):
 *   amax_i  = max_j |v_ij|
 *   scale_i = fp32(amax_i / 127), or 1 when amax_i == 0
 *   q_ij    = clamp(round_half_even(fp32(v_ij / scale_i)), -127, 127)
 * direction 0 quantises activations per token (Smooth-Dynamic, Table 10);
 * direction 1 quantises weights per output channel. */
int oracle_quantize_rows(const float *A, const float *s, int64_t rows, int64_t K,
                         int direction, int8_t *q, float *scale)
{
    if (rows < 0 || K < 0 || (direction != 0 && direction != 1)) return ORC_ERR_ARG;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < rows; ++i) {
        const float *a = A + i * K;
        float amax = 0.0f;
        for (int64_t j = 0; j < K; ++j) {
            float v = direction == 0 ? a[j] / s[j] : a[j] * s[j];
            float av = fabsf(v);
            if (av > amax) amax = av;
        }
        float sc = amax == 0.0f ? 1.0f : amax / 127.0f;
        scale[i] = sc;
        for (int64_t j = 0; j < K; ++j) {
            float v = direction == 0 ? a[j] / s[j] : a[j] * s[j];
            float r = v / sc;
            /* nearbyintf honours the default FE_TONEAREST mode:
             * ties go to the even integer. */
            float n = nearbyintf(r);
            if (n > 127.0f) n = 127.0f;
            if (n < -127.0f) n = -127.0f;
            q[i * K + j] = (int8_t)n;
        }
    }
    return ORC_OK;
}

/* Smooth-Static calibration (Table 10, "SmoothQuant, static quantization"):
 * the per-tensor running maximum of the smoothed activations,
 *   amax = max(amax, max_{i,j} |fl(X[i][j] / s[j])|),
 * over one calibration batch.  The static scale is fl(amax / 127), or 1 when
 * amax is 0. */
int oracle_act_absmax(const float *X, const float *s, int64_t rows, int64_t K, float *amax)
{
    if (rows < 0 || K < 0) return ORC_ERR_ARG;
    float m = *amax;
    for (int64_t i = 0; i < rows; ++i)
        for (int64_t j = 0; j < K; ++j) {
            float v = fabsf(X[i * K + j] / s[j]);
            if (v > m) m = v;
        }
    *amax = m;
    return ORC_OK;
}

/* Smooth-Static quantisation with one per-tensor scale fixed offline:
 *   q[i][j] = clamp(round_half_even(fl(fl(X[i][j] / s[j]) / scale)), -127, 127)
 * Values beyond the calibrated range saturate at +-127. */
int oracle_quantize_static(const float *X, const float *s, int64_t rows, int64_t K,
                           float scale, int8_t *q)
{
    if (rows < 0 || K < 0 || !(scale > 0.0f)) return ORC_ERR_ARG;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < rows; ++i)
        for (int64_t j = 0; j < K; ++j) {
            float v = X[i * K + j] / s[j];
            float n = nearbyintf(v / scale);
            if (n > 127.0f) n = 127.0f;
            if (n < -127.0f) n = -127.0f;
            q[i * K + j] = (int8_t)n;
        }
    return ORC_OK;
}

/* Exact integer contraction acc[m][n] = sum_k xq[m][k] * wq[n][k]
 * (both operands K-contiguous: X is tokens x K, W is the nn.Linear
 * out x in layout).  Summed in int64; any result outside int32 is an error. */
int oracle_gemm_i32(const int8_t *xq, const int8_t *wq, int64_t M, int64_t N,
                    int64_t K, int32_t *acc)
{
    if (M < 0 || N < 0 || K < 0) return ORC_ERR_ARG;
    int overflow = 0;
#pragma omp parallel for schedule(static) reduction(| : overflow)
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            int64_t sum = 0;
            for (int64_t k = 0; k < K; ++k)
                sum += (int64_t)xq[m * K + k] * (int64_t)wq[n * K + k];
            if (sum > INT32_MAX || sum < INT32_MIN) overflow = 1;
            acc[m * N + n] = (int32_t)sum;
        }
    }
    return overflow ? ORC_ERR_OVERFLOW : ORC_OK;
}

/* GELU in its exact erf form: 0.5 t (1 + erf(t / sqrt 2)). */
static double gelu_erf(double t)
{
    return 0.5 * t * (1.0 + erf(t / sqrt(2.0)));
}

/* Dequantising epilogue (the linear block's fused post-ops, Table 3 caption):
 *   d = acc * sx_m * sw_n                   (per-token x per-channel)
 *   NONE:          y = d
 *   BIAS:          y = d + b_n
 *   BIAS_GELU:     y = gelu(d + b_n)
 *   BIAS_RESIDUAL: y = d + b_n + r_mn
 * in double, rounded once to fp32. */
int oracle_epilogue(const int32_t *acc, const float *sx, const float *sw,
                    const float *bias, const float *residual, int64_t M,
                    int64_t N, int mode, float *y)
{
    if (M < 0 || N < 0 || mode < ORC_EPI_NONE || mode > ORC_EPI_BIAS_RESIDUAL)
        return ORC_ERR_ARG;
    if (mode != ORC_EPI_NONE && !bias) return ORC_ERR_ARG;
    if (mode == ORC_EPI_BIAS_RESIDUAL && !residual) return ORC_ERR_ARG;
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            double d = (double)acc[m * N + n] * (double)sx[m] * (double)sw[n];
            double t;
            switch (mode) {
            case ORC_EPI_NONE: t = d; break;
            case ORC_EPI_BIAS: t = d + (double)bias[n]; break;
            case ORC_EPI_BIAS_GELU: t = gelu_erf(d + (double)bias[n]); break;
            default: t = d + (double)bias[n] + (double)residual[m * N + n]; break;
            }
            y[m * N + n] = (float)t;
        }
    }
    return ORC_OK;
}

/* One pass of the linear block for already-packed weights:
 * activation quantisation, integer GEMM, epilogue.  The caller provides all
 * buffers (xq: M*K, sx: M, acc: M*N, y: M*N). */
int oracle_linear_block(const float *X, const float *s, const int8_t *wq,
                        const float *sw, const float *bias, const float *residual,
                        int64_t M, int64_t N, int64_t K, int mode,
                        int8_t *xq, float *sx, int32_t *acc, float *y)
{
    int rc = oracle_quantize_rows(X, s, M, K, 0, xq, sx);
    if (rc != ORC_OK) return rc;
    rc = oracle_gemm_i32(xq, wq, M, N, K, acc);
    if (rc != ORC_OK) return rc;
    return oracle_epilogue(acc, sx, sw, bias, residual, M, N, mode, y);
}

/* LayerNorm of each row, the encoder's normalisation that precedes the FFN
 * and QKV linears (Table 3 lists it among BERT-large's operators; SmoothQuant
 * folds the smoothing factor into it, so its output is what the next linear
 * quantises):
 *   y = (h - mean) / sqrt(var + eps) * gamma[j] + beta[j],
 * mean and the biased variance over the row's K elements, all in double,
 * rounded once to fp32. */
int oracle_layernorm(const float *H, const float *gamma, const float *beta, double eps,
                     int64_t rows, int64_t K, float *Y)
{
    if (!H || !gamma || !beta || !Y || rows < 0 || K <= 0 || !(eps >= 0.0))
        return ORC_ERR_ARG;
    #pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < rows; ++m) {
        const float *h = H + m * K;
        double sum = 0.0;
        for (int64_t j = 0; j < K; ++j) sum += (double)h[j];
        const double mean = sum / (double)K;
        double sq = 0.0;
        for (int64_t j = 0; j < K; ++j) {
            const double d = (double)h[j] - mean;
            sq += d * d;
        }
        const double rstd = 1.0 / sqrt(sq / (double)K + eps);
        for (int64_t j = 0; j < K; ++j)
            Y[m * K + j] = (float)(((double)h[j] - mean) * rstd * (double)gamma[j] +
                                   (double)beta[j]);
    }
    return ORC_OK;
}

/* Encoder self-attention of one layer, the part of the encoder beside the
 * linear block in "Efficient INT8 Inference of Small NLP Models on Server
 * CPUs with PyTorch Native Stack", Table 3: it reads the fused QKV
 * projection's output and writes the out-projection's input.
 *   QKV [B*S][3*H*D] row-major, token-major (sequence b, token i in row
 *   b*S + i); head h's query in columns h*D.., its key in H*D + h*D.., its
 *   value in 2*H*D + h*D..;  O [B*S][H*D], head h in columns h*D..
 *   O[b,i,h,:] = sum_j p_ij V[b,j,h,:],  p_ij = exp(z_ij - max_j z_ij) / sum,
 *   z_ij = scale * <Q[b,i,h,:], K[b,j,h,:]>
 * Every token attends to every token of its sequence (no mask).  All in
 * double, rounded once to fp32. */
int oracle_attention(const float *QKV, int64_t B, int64_t S, int64_t H, int64_t D,
                     double scale, float *O)
{
    if (!QKV || !O || B < 0 || S <= 0 || H <= 0 || D <= 0) return ORC_ERR_ARG;
    const int64_t ld = 3 * H * D;
    int err = ORC_OK;
    #pragma omp parallel
    {
        double *z = (double *)malloc((size_t)S * sizeof(double));
        if (!z) {
            #pragma omp atomic write
            err = ORC_ERR_ARG;
        }
        #pragma omp for schedule(static)
        for (int64_t r = 0; r < B * H * S; ++r) {
            if (!z) continue;
            const int64_t b = r / (H * S), h = (r / S) % H, i = r % S;
            const float *q = QKV + (b * S + i) * ld + h * D;
            double zmax = -INFINITY;
            for (int64_t j = 0; j < S; ++j) {
                const float *k = QKV + (b * S + j) * ld + H * D + h * D;
                double dot = 0.0;
                for (int64_t d = 0; d < D; ++d) dot += (double)q[d] * (double)k[d];
                z[j] = scale * dot;
                if (z[j] > zmax) zmax = z[j];
            }
            double sum = 0.0;
            for (int64_t j = 0; j < S; ++j) {
                z[j] = exp(z[j] - zmax);
                sum += z[j];
            }
            float *o = O + (b * S + i) * (H * D) + h * D;
            for (int64_t d = 0; d < D; ++d) {
                double acc = 0.0;
                for (int64_t j = 0; j < S; ++j)
                    acc += z[j] * (double)QKV[(b * S + j) * ld + 2 * H * D + h * D + d];
                o[d] = (float)(acc / sum);
            }
        }
        free(z);
    }
    return err;
}

/* Number of OpenMP threads a parallel region of this library uses. */
int oracle_num_threads(void)
{
    int n = 1;
#ifdef _OPENMP
#pragma omp parallel
    {
#pragma omp single
        n = omp_get_num_threads();
    }
#endif
    return n;
}

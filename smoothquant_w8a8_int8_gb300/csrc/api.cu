// C-ABI boundary: argument checks, then one launch per call on the caller's
// stream.  Declarations and the contract of every entry point are in sq.h.
#include "common.cuh"

#include <cmath>
#include <mutex>

namespace sq {

sq_status device_info(DeviceInfo *out) {
    static std::mutex mu;
    static DeviceInfo cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SQ_ERR_CUDA;
    if (dev < 0 || dev >= 64) return SQ_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(mu);
    DeviceInfo &c = cache[dev];
    if (c.device != dev) {
        cudaDeviceProp p;
        if (cudaGetDeviceProperties(&p, dev) != cudaSuccess) return SQ_ERR_CUDA;
        c.sms = p.multiProcessorCount;
        c.major = p.major;
        c.minor = p.minor;
        c.smem_optin = p.sharedMemPerBlockOptin;
        c.device = dev;
    }
    *out = c;
    return SQ_OK;
}

}  // namespace sq

using namespace sq;

namespace {

inline cudaStream_t as_stream(void *s) { return static_cast<cudaStream_t>(s); }

// The kernels are built for sm_103a only.
sq_status require_sm103() {
    DeviceInfo di;
    sq_status rc = device_info(&di);
    if (rc != SQ_OK) return rc;
    if (di.major != 10 || di.minor != 3) return SQ_ERR_UNSUPPORTED;
    return SQ_OK;
}

constexpr int64_t kMaxK = 133144;  // K * 127^2 < 2^31

sq_status check_linear_args(const void *X, const float *sx, const void *W, const float *sw,
                            const float *bias, const float *residual, int64_t M, int64_t N,
                            int64_t K, int mode, const void *Y) {
    if (M < 0 || N < 0 || K <= 0) return SQ_ERR_INVALID_ARG;
    if (mode < SQ_EPI_NONE || mode > SQ_EPI_RAW_I32) return SQ_ERR_INVALID_ARG;
    if (K % 16 != 0) return SQ_ERR_ALIGNMENT;
    if (K > kMaxK) return SQ_ERR_UNSUPPORTED;
    if (M == 0 || N == 0) return SQ_OK;  // empty: pointers may be NULL, nothing is launched
    if (!X || !W || !Y) return SQ_ERR_INVALID_ARG;
    if (mode != SQ_EPI_RAW_I32 && (!sx || !sw)) return SQ_ERR_INVALID_ARG;
    if ((mode == SQ_EPI_BIAS || mode == SQ_EPI_BIAS_GELU || mode == SQ_EPI_BIAS_RESIDUAL) &&
        !bias)
        return SQ_ERR_INVALID_ARG;
    if (mode == SQ_EPI_BIAS_RESIDUAL && !residual) return SQ_ERR_INVALID_ARG;
    if (!aligned16(X) || !aligned16(W) || !aligned16(Y)) return SQ_ERR_ALIGNMENT;
    if (mode != SQ_EPI_RAW_I32 && (!aligned4(sx) || !aligned4(sw))) return SQ_ERR_ALIGNMENT;
    if (bias && !aligned4(bias)) return SQ_ERR_ALIGNMENT;
    if (mode == SQ_EPI_BIAS_RESIDUAL && !aligned16(residual)) return SQ_ERR_ALIGNMENT;
    return SQ_OK;
}

sq_status check_quant_args(const float *A, const float *s, int64_t rows, int64_t K,
                           const int8_t *q, const float *scale, const void *op) {
    if (rows < 0 || K <= 0) return SQ_ERR_INVALID_ARG;
    if (K % 16 != 0) return SQ_ERR_ALIGNMENT;
    if (K > (int64_t)1 << 30) return SQ_ERR_UNSUPPORTED;
    if (rows == 0) return SQ_OK;  // empty: pointers may be NULL, nothing is launched
    if (!A || !s || !scale) return SQ_ERR_INVALID_ARG;
    if (!q && !op) return SQ_ERR_INVALID_ARG;
    if (!aligned16(A) || !aligned16(s) || (q && !aligned16(q)) || (op && !aligned16(op)))
        return SQ_ERR_ALIGNMENT;
    if (!aligned4(scale)) return SQ_ERR_ALIGNMENT;
    return SQ_OK;
}

}  // namespace

namespace sq {

sq_status validate_linear(const void *Xop, const float *x_scale, const int32_t *x_row_l1,
                          const void *Wop, const float *w_scale, const int32_t *w_row_l1,
                          const float *bias, const float *residual, int64_t M, int64_t N,
                          int64_t K, int mode, const void *Y) {
    sq_status rc = check_linear_args(Xop, x_scale, Wop, w_scale, bias, residual, M, N, K, mode, Y);
    if (rc != SQ_OK) return rc;
    if (M == 0 || N == 0) return SQ_OK;
    if ((x_row_l1 && !aligned4(x_row_l1)) || (w_row_l1 && !aligned4(w_row_l1)))
        return SQ_ERR_ALIGNMENT;
    return SQ_OK;
}

sq_status require_gb300() { return require_sm103(); }

}  // namespace sq

namespace {

sq_status linear_impl(const void *Xop, const float *x_scale, const int32_t *x_row_l1,
                      const void *Wop, const float *w_scale, const int32_t *w_row_l1,
                      const float *bias, const float *residual, int64_t M, int64_t N, int64_t K,
                      int mode, void *Y, void *workspace, size_t workspace_bytes, void *stream) {
    sq_status rc = validate_linear(Xop, x_scale, x_row_l1, Wop, w_scale, w_row_l1, bias, residual,
                                   M, N, K, mode, Y);
    if (rc != SQ_OK) return rc;
    if (M == 0 || N == 0) return SQ_OK;
    if (workspace && !aligned16(workspace)) return SQ_ERR_ALIGNMENT;
    if ((rc = require_sm103()) != SQ_OK) return rc;
    return launch_gemm_tc(static_cast<const __nv_bfloat16 *>(Xop), x_scale, x_row_l1,
                          static_cast<const __nv_bfloat16 *>(Wop), w_scale, w_row_l1, bias,
                          residual, M, N, K, mode, Y, nullptr, workspace, workspace_bytes,
                          as_stream(stream));
}

sq_status requant_impl(const void *Xop, const float *x_scale, const int32_t *x_row_l1,
                       const void *Wop, const float *w_scale, const int32_t *w_row_l1,
                       const float *bias, const float *residual, int64_t M, int64_t N, int64_t K,
                       int mode, const float *s_next, float scale, int8_t *Yq, void *Yop,
                       float *x_scale_next, void *workspace, size_t workspace_bytes,
                       void *stream) {
    if (mode == SQ_EPI_RAW_I32) return SQ_ERR_INVALID_ARG;
    if (!(scale > 0.0f) || !(scale <= 3.4028234663852886e38f)) return SQ_ERR_INVALID_ARG;
    const void *out = Yop ? Yop : static_cast<const void *>(Yq);
    sq_status rc = check_linear_args(Xop, x_scale, Wop, w_scale, bias, residual, M, N, K, mode,
                                     out);
    if (rc != SQ_OK) return rc;
    if (M == 0 || N == 0) return SQ_OK;
    if (!s_next || (!Yq && !Yop)) return SQ_ERR_INVALID_ARG;
    if (!aligned4(s_next) || (x_scale_next && !aligned4(x_scale_next)) ||
        (Yop && (reinterpret_cast<uintptr_t>(Yop) & 1u)))
        return SQ_ERR_ALIGNMENT;
    if ((x_row_l1 && !aligned4(x_row_l1)) || (w_row_l1 && !aligned4(w_row_l1)))
        return SQ_ERR_ALIGNMENT;
    if (workspace && !aligned16(workspace)) return SQ_ERR_ALIGNMENT;
    if ((rc = require_sm103()) != SQ_OK) return rc;
    RequantOut rq;
    rq.s_next = s_next;
    rq.scale = scale;
    rq.rscale = 1.0f / scale;  // IEEE division: the correctly rounded reciprocal
    rq.Yq = Yq;
    rq.Yop = static_cast<__nv_bfloat16 *>(Yop);
    rq.x_scale = x_scale_next;
    return launch_gemm_tc(static_cast<const __nv_bfloat16 *>(Xop), x_scale, x_row_l1,
                          static_cast<const __nv_bfloat16 *>(Wop), w_scale, w_row_l1, bias,
                          residual, M, N, K, mode, nullptr, &rq, workspace, workspace_bytes,
                          as_stream(stream));
}

}  // namespace

extern "C" {

const char *sq_status_string(int status) {
    switch (status) {
    case SQ_OK: return "SQ_OK";
    case SQ_ERR_INVALID_ARG: return "SQ_ERR_INVALID_ARG: invalid argument";
    case SQ_ERR_ALIGNMENT: return "SQ_ERR_ALIGNMENT: K not a multiple of 16 or misaligned pointer";
    case SQ_ERR_UNSUPPORTED: return "SQ_ERR_UNSUPPORTED: size limit exceeded or device not sm_103";
    case SQ_ERR_CUDA: return "SQ_ERR_CUDA: CUDA call or kernel launch failed";
    case SQ_ERR_TIMEOUT: return "SQ_ERR_TIMEOUT: a kernel's bounded pipeline wait ran out";
    default: return "unknown sq_status";
    }
}

int sq_version(void) { return (1 << 16) | 0; }

size_t sq_operand_bytes(int64_t rows, int64_t K) {
    if (rows < 0 || K < 0) return 0;
    return (size_t)rows * (size_t)K * sizeof(__nv_bfloat16);
}

size_t sq_packed_weight_bytes(int64_t N, int64_t K) { return sq_operand_bytes(N, K); }

sq_status sq_channel_absmax(const float *A, int64_t rows, int64_t cols, float *amax,
                            void *stream) {
    if (rows < 0 || cols <= 0) return SQ_ERR_INVALID_ARG;
    if (rows == 0) return SQ_OK;
    if (!A || !amax) return SQ_ERR_INVALID_ARG;
    if (!aligned4(A) || !aligned4(amax)) return SQ_ERR_ALIGNMENT;
    sq_status rc = require_sm103();
    if (rc != SQ_OK) return rc;
    return launch_channel_absmax(A, rows, cols, amax, as_stream(stream));
}

sq_status sq_smooth_factor(const float *x_amax, const float *w_amax, int64_t K, float alpha,
                           float *s, void *stream) {
    if (!x_amax || !w_amax || !s || K <= 0) return SQ_ERR_INVALID_ARG;
    if (!(alpha >= 0.0f && alpha <= 1.0f)) return SQ_ERR_INVALID_ARG;
    if (!aligned4(x_amax) || !aligned4(w_amax) || !aligned4(s)) return SQ_ERR_ALIGNMENT;
    sq_status rc = require_sm103();
    if (rc != SQ_OK) return rc;
    return launch_smooth_factor(x_amax, w_amax, K, alpha, s, as_stream(stream));
}

sq_status sq_pack_weight(const float *W, const float *s, int64_t N, int64_t K, int8_t *Wq,
                         float *w_scale, void *Wop, int32_t *w_row_l1, void *stream) {
    sq_status rc = check_quant_args(W, s, N, K, Wq, w_scale, Wop);
    if (rc != SQ_OK) return rc;
    if (N == 0) return SQ_OK;
    if ((rc = require_sm103()) != SQ_OK) return rc;
    if (w_row_l1 && !aligned4(w_row_l1)) return SQ_ERR_ALIGNMENT;
    return launch_quantize_rows(1, W, s, N, K, Wq, w_scale, static_cast<__nv_bfloat16 *>(Wop),
                                w_row_l1, 0.0f, as_stream(stream));
}

sq_status sq_quantize_act(const float *X, const float *s, int64_t M, int64_t K, int8_t *Xq,
                          float *x_scale, void *Xop, int32_t *x_row_l1, void *stream) {
    sq_status rc = check_quant_args(X, s, M, K, Xq, x_scale, Xop);
    if (rc != SQ_OK) return rc;
    if (M == 0) return SQ_OK;
    if ((rc = require_sm103()) != SQ_OK) return rc;
    if (x_row_l1 && !aligned4(x_row_l1)) return SQ_ERR_ALIGNMENT;
    return launch_quantize_rows(0, X, s, M, K, Xq, x_scale, static_cast<__nv_bfloat16 *>(Xop),
                                x_row_l1, 0.0f, as_stream(stream));
}

sq_status sq_act_absmax(const float *X, const float *s, int64_t M, int64_t K, float *amax,
                        void *stream) {
    if (M < 0 || K <= 0) return SQ_ERR_INVALID_ARG;
    if (K % 16 != 0) return SQ_ERR_ALIGNMENT;
    if (M == 0) return SQ_OK;
    if (!X || !s || !amax) return SQ_ERR_INVALID_ARG;
    if (!aligned16(X) || !aligned16(s) || !aligned4(amax)) return SQ_ERR_ALIGNMENT;
    sq_status rc = require_sm103();
    if (rc != SQ_OK) return rc;
    return launch_act_absmax(X, s, M, K, amax, as_stream(stream));
}

sq_status sq_division_table(const float *s, int64_t K, float *table, void *stream) {
    if (K < 0) return SQ_ERR_INVALID_ARG;
    if (K == 0) return SQ_OK;
    if (!s || !table) return SQ_ERR_INVALID_ARG;
    if (!aligned4(s) || !aligned16(table)) return SQ_ERR_ALIGNMENT;
    sq_status rc = require_sm103();
    if (rc != SQ_OK) return rc;
    return launch_division_table(s, K, table, as_stream(stream));
}

sq_status sq_linear_i8_rowmax(const void *Xop, const float *x_scale, const int32_t *x_row_l1,
                              const void *Wop, const float *w_scale, const int32_t *w_row_l1,
                              const float *bias, const float *residual, int64_t M, int64_t N,
                              int64_t K, int mode, void *Y, const float *next_table,
                              float *row_amax, void *stream) {
    if (mode == SQ_EPI_RAW_I32) return SQ_ERR_INVALID_ARG;
    sq_status rc = validate_linear(Xop, x_scale, x_row_l1, Wop, w_scale, w_row_l1, bias, residual,
                                   M, N, K, mode, Y);
    if (rc != SQ_OK) return rc;
    if (M == 0 || N == 0) return SQ_OK;
    if (!next_table || !row_amax) return SQ_ERR_INVALID_ARG;
    if (!aligned16(next_table) || !aligned4(row_amax)) return SQ_ERR_ALIGNMENT;
    if ((rc = require_sm103()) != SQ_OK) return rc;
    return launch_gemm_tc(static_cast<const __nv_bfloat16 *>(Xop), x_scale, x_row_l1,
                          static_cast<const __nv_bfloat16 *>(Wop), w_scale, w_row_l1, bias,
                          residual, M, N, K, mode, Y, nullptr, nullptr, 0, as_stream(stream),
                          next_table, row_amax);
}

sq_status sq_quantize_act_rowmax(const float *X, const float *s, const float *row_amax,
                                 int64_t M, int64_t K, int8_t *Xq, float *x_scale, void *Xop,
                                 int32_t *x_row_l1, void *stream) {
    sq_status rc = check_quant_args(X, s, M, K, Xq, x_scale, Xop);
    if (rc != SQ_OK) return rc;
    if (M == 0) return SQ_OK;
    if (!row_amax) return SQ_ERR_INVALID_ARG;
    if (!aligned4(row_amax) || (x_row_l1 && !aligned4(x_row_l1))) return SQ_ERR_ALIGNMENT;
    if ((rc = require_sm103()) != SQ_OK) return rc;
    return launch_quantize_act_given_max(X, s, row_amax, M, K, Xq, x_scale,
                                         static_cast<__nv_bfloat16 *>(Xop), x_row_l1,
                                         as_stream(stream));
}

sq_status sq_quantize_act_table(const float *X, const float *s, const float *s_table,
                                const float *row_amax, int64_t M, int64_t K, int8_t *Xq,
                                float *x_scale, void *Xop, int32_t *x_row_l1, void *stream) {
    sq_status rc = check_quant_args(X, s, M, K, Xq, x_scale, Xop);
    if (rc != SQ_OK) return rc;
    if (M == 0) return SQ_OK;
    if (!s_table) return SQ_ERR_INVALID_ARG;
    if (!aligned16(s_table) || (row_amax && !aligned4(row_amax)) ||
        (x_row_l1 && !aligned4(x_row_l1)))
        return SQ_ERR_ALIGNMENT;
    if ((rc = require_sm103()) != SQ_OK) return rc;
    return launch_quantize_act_table(X, s, s_table, row_amax, M, K, Xq, x_scale,
                                     static_cast<__nv_bfloat16 *>(Xop), x_row_l1,
                                     as_stream(stream));
}

sq_status sq_attention(const float *QKV, int64_t B, int64_t S, int64_t H, int64_t D,
                       float scale, float *O, void *stream) {
    if (B < 0 || S < 0 || H < 0 || D <= 0) return SQ_ERR_INVALID_ARG;
    if (!(scale == scale) || !(fabsf(scale) <= 3.4028234663852886e38f)) return SQ_ERR_INVALID_ARG;
    if (D != 64 || S % 64 != 0 || S > 448) return SQ_ERR_UNSUPPORTED;
    if (B == 0 || S == 0 || H == 0) return SQ_OK;
    if (B * S >= ((int64_t)1 << 31) || H > 65536) return SQ_ERR_UNSUPPORTED;
    if (!QKV || !O) return SQ_ERR_INVALID_ARG;
    if (!aligned16(QKV) || !aligned16(O)) return SQ_ERR_ALIGNMENT;
    sq_status rc = require_sm103();
    if (rc != SQ_OK) return rc;
    return launch_attention(QKV, B, S, H, scale, O, as_stream(stream));
}

sq_status sq_static_scale(const float *amax, float *scale, void *stream) {
    if (!amax || !scale) return SQ_ERR_INVALID_ARG;
    if (!aligned4(amax) || !aligned4(scale)) return SQ_ERR_ALIGNMENT;
    sq_status rc = require_sm103();
    if (rc != SQ_OK) return rc;
    return launch_static_scale(amax, scale, as_stream(stream));
}

sq_status sq_quantize_act_static(const float *X, const float *s, int64_t M, int64_t K,
                                 float scale, int8_t *Xq, float *x_scale, void *Xop,
                                 int32_t *x_row_l1, void *stream) {
    if (!(scale > 0.0f) || !(scale <= 3.4028234663852886e38f)) return SQ_ERR_INVALID_ARG;
    sq_status rc = check_quant_args(X, s, M, K, Xq, x_scale, Xop);
    if (rc != SQ_OK) return rc;
    if (M == 0) return SQ_OK;
    if (x_row_l1 && !aligned4(x_row_l1)) return SQ_ERR_ALIGNMENT;
    if ((rc = require_sm103()) != SQ_OK) return rc;
    return launch_quantize_rows(2, X, s, M, K, Xq, x_scale, static_cast<__nv_bfloat16 *>(Xop),
                                x_row_l1, scale, as_stream(stream));
}

sq_status sq_layernorm_quant(const float *H, const float *gamma, const float *beta, float eps,
                             const float *s, int64_t M, int64_t K, float static_scale, float *Y,
                             int8_t *Xq, float *x_scale, void *Xop, int32_t *x_row_l1,
                             void *stream) {
    if (!(eps >= 0.0f) || !(eps <= 3.4028234663852886e38f)) return SQ_ERR_INVALID_ARG;
    if (!(static_scale >= 0.0f) || !(static_scale <= 3.4028234663852886e38f))
        return SQ_ERR_INVALID_ARG;
    sq_status rc = check_quant_args(H, s, M, K, Xq, x_scale, Xop);
    if (rc != SQ_OK) return rc;
    if (M == 0) return SQ_OK;
    if (!gamma || !beta) return SQ_ERR_INVALID_ARG;
    if (!aligned16(gamma) || !aligned16(beta) || (Y && !aligned16(Y)) ||
        (x_row_l1 && !aligned4(x_row_l1)))
        return SQ_ERR_ALIGNMENT;
    if (K > 8192) return SQ_ERR_UNSUPPORTED;
    if ((rc = require_sm103()) != SQ_OK) return rc;
    return launch_layernorm_quant(H, gamma, beta, eps, s, M, K, static_scale, Y, Xq, x_scale,
                                  static_cast<__nv_bfloat16 *>(Xop), x_row_l1, as_stream(stream));
}

sq_status sq_linear_i8(const void *Xop, const float *x_scale, const int32_t *x_row_l1,
                       const void *Wop, const float *w_scale, const int32_t *w_row_l1,
                       const float *bias, const float *residual, int64_t M, int64_t N, int64_t K,
                       int mode, void *Y, void *stream) {
    return linear_impl(Xop, x_scale, x_row_l1, Wop, w_scale, w_row_l1, bias, residual, M, N, K,
                       mode, Y, nullptr, 0, stream);
}

sq_status sq_linear_workspace_bytes(int64_t M, int64_t N, int64_t K, size_t *bytes) {
    if (!bytes) return SQ_ERR_INVALID_ARG;
    *bytes = 0;
    if (M < 0 || N < 0 || K <= 0) return SQ_ERR_INVALID_ARG;
    if (K > kMaxK) return SQ_ERR_UNSUPPORTED;
    if (M == 0 || N == 0) return SQ_OK;
    return gemm_tc_workspace_bytes(M, N, K, bytes);
}

sq_status sq_linear_i8_ws(const void *Xop, const float *x_scale, const int32_t *x_row_l1,
                          const void *Wop, const float *w_scale, const int32_t *w_row_l1,
                          const float *bias, const float *residual, int64_t M, int64_t N,
                          int64_t K, int mode, void *Y, void *workspace, size_t workspace_bytes,
                          void *stream) {
    return linear_impl(Xop, x_scale, x_row_l1, Wop, w_scale, w_row_l1, bias, residual, M, N, K,
                       mode, Y, workspace, workspace_bytes, stream);
}

sq_status sq_linear_codes_workspace_bytes(int64_t M, int64_t K, size_t *bytes) {
    if (!bytes) return SQ_ERR_INVALID_ARG;
    *bytes = 0;
    if (M < 0 || K <= 0) return SQ_ERR_INVALID_ARG;
    if (K % 16 != 0) return SQ_ERR_ALIGNMENT;
    if (K > kMaxK || M > ((int64_t)1 << 40) / K) return SQ_ERR_UNSUPPORTED;
    *bytes = (size_t)((M * K * 2 + 255) / 256 * 256);
    return SQ_OK;
}

sq_status sq_linear_i8_codes(const int8_t *Xq, const float *x_scale, const int32_t *x_row_l1,
                             const void *Wop, const float *w_scale, const int32_t *w_row_l1,
                             const float *bias, const float *residual, int64_t M, int64_t N,
                             int64_t K, int mode, void *Y, void *workspace, size_t workspace_bytes,
                             void *stream) {
    size_t need = 0;
    sq_status rc = sq_linear_codes_workspace_bytes(M, K, &need);
    if (rc != SQ_OK) return rc;
    if (M > 0 && N > 0) {
        if (!Xq || !workspace) return SQ_ERR_INVALID_ARG;
        if (!aligned16(Xq) || !aligned16(workspace)) return SQ_ERR_ALIGNMENT;
        if (workspace_bytes < need) return SQ_ERR_INVALID_ARG;
    }
    // the operand the codes widen into is the workspace: the checks of sq_linear_i8 on it
    if ((rc = validate_linear(workspace, x_scale, x_row_l1, Wop, w_scale, w_row_l1, bias,
                              residual, M, N, K, mode, Y)) != SQ_OK ||
        M == 0 || N == 0)
        return rc;
    if ((rc = require_gb300()) != SQ_OK) return rc;
    __nv_bfloat16 *op = static_cast<__nv_bfloat16 *>(workspace);
    if ((rc = launch_widen_codes(Xq, op, M * K, as_stream(stream))) != SQ_OK) return rc;
    return linear_impl(op, x_scale, x_row_l1, Wop, w_scale, w_row_l1, bias, residual, M, N, K,
                       mode, Y, nullptr, 0, stream);
}

sq_status sq_linear_i8_requant(const void *Xop, const float *x_scale, const int32_t *x_row_l1,
                               const void *Wop, const float *w_scale, const int32_t *w_row_l1,
                               const float *bias, const float *residual, int64_t M, int64_t N,
                               int64_t K, int mode, const float *s_next, float scale, int8_t *Yq,
                               void *Yop, float *x_scale_next, void *stream) {
    return requant_impl(Xop, x_scale, x_row_l1, Wop, w_scale, w_row_l1, bias, residual, M, N, K,
                        mode, s_next, scale, Yq, Yop, x_scale_next, nullptr, 0, stream);
}

sq_status sq_linear_i8_requant_ws(const void *Xop, const float *x_scale,
                                  const int32_t *x_row_l1, const void *Wop, const float *w_scale,
                                  const int32_t *w_row_l1, const float *bias,
                                  const float *residual, int64_t M, int64_t N, int64_t K,
                                  int mode, const float *s_next, float scale, int8_t *Yq,
                                  void *Yop, float *x_scale_next, void *workspace,
                                  size_t workspace_bytes, void *stream) {
    return requant_impl(Xop, x_scale, x_row_l1, Wop, w_scale, w_row_l1, bias, residual, M, N, K,
                        mode, s_next, scale, Yq, Yop, x_scale_next, workspace, workspace_bytes,
                        stream);
}

sq_status sq_linear_i8_mma_sync(const int8_t *Xq, const float *x_scale, const int8_t *Wq,
                                const float *w_scale, const float *bias, const float *residual,
                                int64_t M, int64_t N, int64_t K, int mode, void *Y,
                                void *stream) {
    sq_status rc = check_linear_args(Xq, x_scale, Wq, w_scale, bias, residual, M, N, K, mode, Y);
    if (rc != SQ_OK) return rc;
    if (M == 0 || N == 0) return SQ_OK;
    if ((rc = require_sm103()) != SQ_OK) return rc;
    return launch_gemm_mma_sync(Xq, x_scale, Wq, w_scale, bias, residual, M, N, K, mode, Y,
                                as_stream(stream));
}

sq_status sq_check_division(uint32_t b_first, uint32_t b_count, uint32_t a_first,
                            uint32_t a_count, int corrected, unsigned long long *out,
                            void *stream) {
    const uint64_t lim = 1ull << 23;
    if ((uint64_t)b_first + b_count > lim || (uint64_t)a_first + a_count > lim)
        return SQ_ERR_INVALID_ARG;
    if (b_count == 0 || a_count == 0) return SQ_OK;
    if (!out) return SQ_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(out) & 7u) != 0) return SQ_ERR_ALIGNMENT;
    sq_status rc = require_sm103();
    if (rc != SQ_OK) return rc;
    return launch_check_division(b_first, b_count, a_first, a_count, corrected ? 1 : 0, out,
                                 as_stream(stream));
}

sq_status sq_device_status(void *stream) {
    if (cudaStreamSynchronize(as_stream(stream)) != cudaSuccess) return SQ_ERR_CUDA;
    const sq_status rq = quant_take_error(as_stream(stream));
    if (rq == SQ_ERR_CUDA) return rq;
    const sq_status ra = attention_take_error(as_stream(stream));
    if (ra == SQ_ERR_CUDA) return ra;
    sq_status rc = gemm_tc_take_error(as_stream(stream));
    if (rc == SQ_OK) rc = rq;
    if (rc == SQ_OK) rc = ra;
    if (rc == SQ_ERR_TIMEOUT) {
        // a split-K launch that gave up may have left counters in the static
        // scratch: clear them before the next sq_linear_i8_static_ws call
        const sq_status r2 = static_ws_reset_counters(as_stream(stream));
        if (r2 != SQ_OK) return r2;
    }
    return rc;
}

sq_status sq_get_device_status(void *stream) { return sq_device_status(stream); }

}  // extern "C"

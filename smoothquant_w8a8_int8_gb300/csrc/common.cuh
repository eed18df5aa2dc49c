// Shared host/device helpers of the CUDA path (not used by the oracle).
#pragma once
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "sq.h"

namespace sq {

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

inline sq_status cuda_status(cudaError_t e) { return e == cudaSuccess ? SQ_OK : SQ_ERR_CUDA; }

// SM count and compute capability of the current device, cached per device.
struct DeviceInfo {
    int device = -1;
    int sms = 0;
    int major = 0, minor = 0;
    size_t smem_optin = 0;
};
sq_status device_info(DeviceInfo *out);

// Launchers (internal): arguments were validated by the C-ABI layer.
sq_status launch_channel_absmax(const float *A, int64_t rows, int64_t cols, float *amax,
                                cudaStream_t st);
sq_status launch_smooth_factor(const float *ax, const float *aw, int64_t K, float alpha,
                               float *s, cudaStream_t st);
// direction: 0 dynamic activations, 1 weights, 2 static activations (fixed_scale)
sq_status launch_quantize_rows(int direction, const float *A, const float *s, int64_t rows,
                               int64_t K, int8_t *q, float *scale, __nv_bfloat16 *op,
                               int32_t *l1, float fixed_scale, cudaStream_t st);
sq_status launch_act_absmax(const float *A, const float *s, int64_t rows, int64_t K,
                            float *amax, cudaStream_t st);
sq_status launch_gemm_mma_sync(const int8_t *Xq, const float *sx, const int8_t *Wq,
                               const float *sw, const float *bias, const float *residual,
                               int64_t M, int64_t N, int64_t K, int mode, void *Y,
                               cudaStream_t st);
sq_status launch_gemm_tc(const __nv_bfloat16 *Xop, const float *sx, const int32_t *x_l1,
                         const __nv_bfloat16 *Wop, const float *sw, const int32_t *w_l1,
                         const float *bias, const float *residual, int64_t M, int64_t N,
                         int64_t K, int mode, void *Y, cudaStream_t st);
// Reads and clears the tcgen05 GEMM's device error word (synchronous).
sq_status gemm_tc_take_error(cudaStream_t st);

// fp32 epilogue shared by both GEMM paths: d = acc * sx * sw, then the mode.
__device__ __forceinline__ float epilogue_value(int32_t acc, float sx, float sw, float b,
                                                float r, int mode) {
    float d = __fmul_rn(__fmul_rn(__int2float_rn(acc), sx), sw);
    if (mode == SQ_EPI_NONE) return d;
    float t = __fadd_rn(d, b);
    if (mode == SQ_EPI_BIAS) return t;
    if (mode == SQ_EPI_BIAS_GELU) return 0.5f * t * (1.0f + erff(t * 0.70710678118654752f));
    return __fadd_rn(t, r);
}

}  // namespace sq

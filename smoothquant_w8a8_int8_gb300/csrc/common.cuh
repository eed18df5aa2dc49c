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

// Programmatic dependent launch.  Every kernel of the library is launched with
// programmatic stream serialisation allowed: once all CTAs of the kernel
// before it on the stream have started (and called pdl_launch_dependents) or
// finished, its CTAs may be scheduled, run their set-up (barrier
// initialisation, tensor-memory allocation) and then block in pdl_wait until
// the previous kernel has completed and its memory operations are visible.
// Every global-memory access comes after pdl_wait, so the ordering of the
// stream is kept for all data; only launch latency and set-up overlap.
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Launch with programmatic stream serialisation (and a cluster of
// `cluster_x` CTAs along x when cluster_x > 1).
template <typename... KArgs, typename... Args>
inline sq_status launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                            cudaStream_t st, unsigned cluster_x, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    unsigned n = 0;
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
    if (cluster_x > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = cluster_x;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cuda_status(cudaLaunchKernelEx(&cfg, kern, args...));
}

// ---- packed fp32 pairs (f32x2: two lanes of arithmetic per instruction) ----

__device__ __forceinline__ unsigned long long pk(float a, float b) {
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ void upk(unsigned long long r, float &a, float &b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ unsigned long long fma2(unsigned long long a, unsigned long long b,
                                                   unsigned long long c) {
    unsigned long long d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ unsigned long long mul2(unsigned long long a, unsigned long long b) {
    unsigned long long d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ unsigned long long add2(unsigned long long a, unsigned long long b) {
    unsigned long long d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ unsigned long long sub2(unsigned long long a, unsigned long long b) {
    unsigned long long d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// SM count and compute capability of the current device, cached per device.
struct DeviceInfo {
    int device = -1;
    int sms = 0;
    int major = 0, minor = 0;
    size_t smem_optin = 0;
};
sq_status device_info(DeviceInfo *out);

// x / s with y = RN(1/s) computed once per column:
//   q0 = RN(x y),  r = RN(x - s q0) (one fma),  q = RN(q0 + r y) (one fma).
// q is the IEEE quotient RN(x / s) when no step leaves the normal range.  With
// y = (1/s)(1 + d), |d| < 2^-24, and r exact, the value rounded last is
// x/s + d (x/s - q0), a few 2^-48 ulp from x/s, while x/s -- never itself a
// rounding midpoint -- lies at least ulp / 2^25 from every midpoint; q0 can be
// more than an ulp off only for the largest few dividend significands.  Scaling
// x or s by a power of two scales every step exactly, so correctness is a
// property of the 2^46 significand pairs, and sq_check_division runs this very
// function against IEEE division over all of them (or any subset).  Range used
// by the callers: |s| in [2^-20, 2^20], |x| >= 2^-100 (then r is exact) and
// |q0| <= 2^100; tinier x only matter as code 0.
__device__ __forceinline__ float div_smooth(float x, float s, float y) {
    const float q0 = __fmul_rn(x, y);
    const float r = __fmaf_rn(-q0, s, x);
    return __fmaf_rn(r, y, q0);
}

// Smooth-Static code of a smoothed value v (Table 10): round_half_even(fl(v /
// scale)) saturated to [-127, 127], for any finite v, given rscale =
// fl(1/scale).  p = fl(v * rscale) is within a relative 3u of the quotient;
// |p| >= 128 means the quotient exceeds 127.5 in magnitude (the code
// saturates); below that p is within 2.3e-5 of fl(v/scale), so its rounding
// decides unless p lies within 2^-14 of a half-integer, where the IEEE
// division does.  Shared by the activation quantiser and the GEMM epilogue
// that emits the next linear's codes.
__device__ __forceinline__ float static_code(float v, float scale, float rscale) {
    const float p = __fmul_rn(v, rscale);
    if (fabsf(p) >= 128.0f) return copysignf(127.0f, p);
    const float k = rintf(p);
    if (fabsf(__fsub_rn(p, k)) <= 0.49993896484375f)  // 0.5 - 2^-14
        return fminf(127.0f, fmaxf(-127.0f, k));
    const float e = rintf(__fdiv_rn(v, scale));
    return fminf(127.0f, fmaxf(-127.0f, e));
}

// Outputs of the requantising epilogue (sq_linear_i8_requant): the codes of
// the next linear's input, Smooth-Static with its smoothing factor s_next [N]
// and per-tensor scale; either code array may be NULL (not both).
struct RequantOut {
    const float *s_next;
    float scale, rscale;
    int8_t *Yq;
    __nv_bfloat16 *Yop;
    float *x_scale;  // [M], set to `scale` (nullable)
};


// Launchers (internal): arguments were validated by the C-ABI layer.
sq_status launch_channel_absmax(const float *A, int64_t rows, int64_t cols, float *amax,
                                cudaStream_t st);
sq_status launch_smooth_factor(const float *ax, const float *aw, int64_t K, float alpha,
                               float *s, cudaStream_t st);
// direction: 0 dynamic activations, 1 weights, 2 static activations (fixed_scale)
sq_status launch_quantize_rows(int direction, const float *A, const float *s, int64_t rows,
                               int64_t K, int8_t *q, float *scale, __nv_bfloat16 *op,
                               int32_t *l1, float fixed_scale, cudaStream_t st);
sq_status launch_check_division(uint32_t b_first, uint32_t b_count, uint32_t a_first,
                                uint32_t a_count, int corrected, unsigned long long *out,
                                cudaStream_t st);
sq_status launch_layernorm_quant(const float *H, const float *gamma, const float *beta,
                                 float eps, const float *s, int64_t rows, int64_t K,
                                 float static_scale, float *Y, int8_t *q, float *scale,
                                 __nv_bfloat16 *op, int32_t *l1, cudaStream_t st);
sq_status launch_act_absmax(const float *A, const float *s, int64_t rows, int64_t K,
                            float *amax, cudaStream_t st);
sq_status launch_static_scale(const float *amax, float *scale, cudaStream_t st);
sq_status launch_division_table(const float *s, int64_t K, float *table, cudaStream_t st);
sq_status launch_quantize_act_given_max(const float *A, const float *s, const float *row_amax,
                                        int64_t rows, int64_t K, int8_t *q, float *scale,
                                        __nv_bfloat16 *op, int32_t *l1, cudaStream_t st);
// the Smooth-Dynamic quantiser (row_amax NULL) or its given-maximum form with
// s's division table (launch_division_table) beside s
sq_status launch_quantize_act_table(const float *A, const float *s, const float *table,
                                    const float *row_amax, int64_t rows, int64_t K, int8_t *q,
                                    float *scale, __nv_bfloat16 *op, int32_t *l1,
                                    cudaStream_t st);
sq_status launch_gemm_mma_sync(const int8_t *Xq, const float *sx, const int8_t *Wq,
                               const float *sw, const float *bias, const float *residual,
                               int64_t M, int64_t N, int64_t K, int mode, void *Y,
                               cudaStream_t st);
// rq == NULL: Y gets the epilogue's fp32 (or int32) values; otherwise the
// epilogue's values are requantised into rq's code arrays and Y is unused.
// rm_pairs / row_amax (both non-NULL, rq NULL): Y as usual, and each row's
// maximum of |fl(Y / s_next)| merged into row_amax (pairs: the division table
// of s_next, see sq_division_table).
sq_status launch_gemm_tc(const __nv_bfloat16 *Xop, const float *sx, const int32_t *x_l1,
                         const __nv_bfloat16 *Wop, const float *sw, const int32_t *w_l1,
                         const float *bias, const float *residual, int64_t M, int64_t N,
                         int64_t K, int mode, void *Y, const RequantOut *rq, void *workspace,
                         size_t workspace_bytes, cudaStream_t st,
                         const float *rm_pairs = nullptr, float *row_amax = nullptr);
// Bytes of the split-K workspace of an M x N x K launch on the current device (0: none used).
sq_status gemm_tc_workspace_bytes(int64_t M, int64_t N, int64_t K, size_t *bytes);
// Read and clear the device error words of the tcgen05 GEMM and of the
// activation quantiser (synchronous).
sq_status gemm_tc_take_error(cudaStream_t st);
sq_status quant_take_error(cudaStream_t st);
// int8 codes [count] -> the bf16 GEMM operand (exact); count % 16 == 0, both
// pointers 16-byte aligned.
sq_status launch_widen_codes(const int8_t *q, __nv_bfloat16 *op, int64_t count, cudaStream_t st);
sq_status attention_take_error(cudaStream_t st);
// A 2-D TMA tensor map (a CUtensorMap, 128 bytes) over a row-major fp32 matrix
// of rows x cols, boxes of box_rows x box_cols, 128-byte swizzle.
sq_status make_map_f32(void *map, const float *base, int64_t rows, int64_t cols, int box_rows,
                       int box_cols);
// Encoder self-attention (head dimension 64): QKV [B*S][3*H*64] -> O [B*S][H*64].
sq_status launch_attention(const float *QKV, int64_t B, int64_t S, int64_t H, float scale,
                           float *O, cudaStream_t st);
// The host-side argument checks of sq_linear_i8 / sq_linear_i8_ws (everything
// but the workspace and the device): SQ_OK for a valid call, empty calls
// included.  require_gb300: SQ_ERR_UNSUPPORTED unless the current device is
// an sm_103 GPU.
sq_status validate_linear(const void *Xop, const float *x_scale, const int32_t *x_row_l1,
                          const void *Wop, const float *w_scale, const int32_t *w_row_l1,
                          const float *bias, const float *residual, int64_t M, int64_t N,
                          int64_t K, int mode, const void *Y);
sq_status require_gb300();
// Zero-fills the split-K counter block of the static scratch on the current
// device, if its address has been looked up there (no allocation; synchronous).
sq_status static_ws_reset_counters(cudaStream_t st);

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

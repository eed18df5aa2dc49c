// Smoothing statistics, smoothing factor, and the per-row symmetric int8
// quantiser used for both activations (dynamic, per token) and weights
// (offline, per output channel).
//
// "Efficient INT8 Inference of Small NLP Models on Server CPUs with PyTorch
// Native Stack": Table 10 (Smooth-Dynamic: SmoothQuant + dynamic activation
// quantisation), with per-token activation / per-channel weight scales; the
// smoothing factor and its migration strength alpha follow SmoothQuant (the
// pages' reference list; alpha per model in Table 15).
//
// The quantiser is HBM-bound (4 B read + 1-3 B written per element, a few
// flops), so it is written as a coalesced row reduction: a group of TPR
// threads owns a row, each thread holds up to VPT float4 of it in registers,
// the row maximum is a warp-shuffle (and, for TPR > 32, a shared-memory)
// reduction, and the codes are produced from the registers, so every input
// byte is read from HBM exactly once.  Blocks loop over rows so that the
// per-channel smoothing factors stay in registers across rows.
#include "common.cuh"

#include <algorithm>

namespace sq {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxVPT = 8;  // float4 per thread held in registers: K <= 256 * 8 * 4

// Row kinds: dynamic activations (per-token scale from the row maximum),
// weights (per-output-channel scale), static activations (one given scale).
constexpr int kActDynamic = 0, kWeight = 1, kActStatic = 2;

__device__ __forceinline__ float smooth_one(float x, float s, int kind) {
    // activations: x / s (IEEE division); weights: x * s
    return kind == kWeight ? __fmul_rn(x, s) : __fdiv_rn(x, s);
}

// round_half_even(fl(v / scale)), clamped to [-127, 127], returned as an
// integer-valued float, with the division replaced by a multiplication where
// that provably gives the same integer.  With r = fl(1/scale) (correctly
// rounded) and p = fl(v * r), p differs from the exact quotient v/scale by a
// relative 2^-23 + 2^-48 at most, and fl(v/scale) by 2^-24: for
// |v/scale| <= 128 the two lie within 2.3e-5 of each other.  Their integer
// roundings can differ only if a half-integer lies between them, so when p is
// farther than 2^-14 from every half-integer the rounded p is the answer;
// otherwise (rare) the IEEE division decides.  (|v| <= amax and
// scale = fl(amax/127) keep every quotient within 127 * (1 + 2^-23), so the
// clamp never acts on the fast path.)
__device__ __forceinline__ float code_of(float v, float scale, float rscale) {
    const float p = __fmul_rn(v, rscale);
    const float k = rintf(p);
    if (fabsf(__fsub_rn(p, k)) <= 0.49993896484375f) return k;  // 0.5 - 2^-14
    const float e = rintf(__fdiv_rn(v, scale));                 // round half to even
    return fminf(127.0f, fmaxf(-127.0f, e));
}

// four integer-valued codes to the int8 and/or bf16 outputs (float4 index off4)
__device__ __forceinline__ void store_code_values(float c0, float c1, float c2, float c3,
                                                  int64_t off4, int8_t *q, __nv_bfloat16 *op) {
    if (q) {
        const uint32_t packed = (uint32_t)(__float2int_rn(c0) & 0xff) |
                                ((uint32_t)(__float2int_rn(c1) & 0xff) << 8) |
                                ((uint32_t)(__float2int_rn(c2) & 0xff) << 16) |
                                ((uint32_t)(__float2int_rn(c3) & 0xff) << 24);
        reinterpret_cast<uint32_t *>(q)[off4] = packed;
    }
    if (op) {
        // integers |c| <= 127 are exact in bf16
        __nv_bfloat162 lo = __floats2bfloat162_rn(c0, c1);
        __nv_bfloat162 hi = __floats2bfloat162_rn(c2, c3);
        uint2 u;
        u.x = *reinterpret_cast<uint32_t *>(&lo);
        u.y = *reinterpret_cast<uint32_t *>(&hi);
        reinterpret_cast<uint2 *>(op)[off4] = u;
    }
}

// Writes four codes; returns the sum of their magnitudes (for the row L1 norm).
template <int KIND>
__device__ __forceinline__ float store_codes(float4 v, float scale, float rscale, int64_t off4,
                                             int8_t *q, __nv_bfloat16 *op) {
    auto code = [&](float x) {
        return KIND == kActStatic ? static_code(x, scale, rscale) : code_of(x, scale, rscale);
    };
    const float c0 = code(v.x), c1 = code(v.y), c2 = code(v.z), c3 = code(v.w);
    store_code_values(c0, c1, c2, c3, off4, q, op);
    return (fabsf(c0) + fabsf(c1)) + (fabsf(c2) + fabsf(c3));
}

// Row maximum across the TPR threads of a row group.  red: [rows_per_block][8].
__device__ __forceinline__ float group_max(float m, int tpr, float *red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (tpr > 32) {
        const int warp = threadIdx.x >> 5;
        const int wpg = tpr >> 5;           // warps per group
        const int g = warp / wpg;
        if ((threadIdx.x & 31) == 0) red[warp] = m;
        __syncthreads();
        m = 0.0f;
        for (int w = 0; w < wpg; ++w) m = fmaxf(m, red[g * wpg + w]);
        __syncthreads();
    }
    return m;
}

// Row sum across the TPR threads of a row group (as group_max).
__device__ __forceinline__ float group_sum(float v, int tpr, float *red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (tpr > 32) {
        const int warp = threadIdx.x >> 5;
        const int wpg = tpr >> 5;
        const int g = warp / wpg;
        if ((threadIdx.x & 31) == 0) red[warp] = v;
        __syncthreads();
        v = 0.0f;
        for (int w = 0; w < wpg; ++w) v += red[g * wpg + w];
        __syncthreads();
    }
    return v;
}

// Registers path: K4 = K/4 <= tpr * kVPT.
template <int DIR, int kVPT>
__global__ void __launch_bounds__(kThreads) quantize_rows_reg(
    const float *__restrict__ A, const float *__restrict__ s, int64_t rows, int K4, int tpr,
    int8_t *__restrict__ q, float *__restrict__ scale, __nv_bfloat16 *__restrict__ op,
    int32_t *__restrict__ l1, float fixed_scale) {
    pdl_launch_dependents();
    pdl_wait();
    __shared__ float red[kThreads / 32];
    const int rpb = kThreads / tpr;
    const int g = threadIdx.x / tpr;
    const int t = threadIdx.x % tpr;
    const float4 *s4 = reinterpret_cast<const float4 *>(s);
    float4 sv[kVPT];
#pragma unroll
    for (int i = 0; i < kVPT; ++i) {
        int j = t + i * tpr;
        sv[i] = j < K4 ? __ldg(s4 + j) : make_float4(1.f, 1.f, 1.f, 1.f);
    }
    const int64_t tiles = (rows + rpb - 1) / rpb;
    for (int64_t tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
        const int64_t row = tile * rpb + g;
        const bool valid = row < rows;
        const float4 *a4 = reinterpret_cast<const float4 *>(A) + (valid ? row : 0) * K4;
        float4 v[kVPT];
        // issue every load of the row before any arithmetic (all in flight at once)
#pragma unroll
        for (int i = 0; i < kVPT; ++i) {
            int j = t + i * tpr;
            v[i] = (valid && j < K4) ? __ldcs(a4 + j) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        float m = 0.0f;
#pragma unroll
        for (int i = 0; i < kVPT; ++i) {
            v[i].x = smooth_one(v[i].x, sv[i].x, DIR);
            v[i].y = smooth_one(v[i].y, sv[i].y, DIR);
            v[i].z = smooth_one(v[i].z, sv[i].z, DIR);
            v[i].w = smooth_one(v[i].w, sv[i].w, DIR);
            if (DIR != kActStatic)
                m = fmaxf(m, fmaxf(fmaxf(fabsf(v[i].x), fabsf(v[i].y)),
                                   fmaxf(fabsf(v[i].z), fabsf(v[i].w))));
        }
        float sc = fixed_scale;
        if (DIR != kActStatic) {
            m = group_max(m, tpr, red);
            sc = m == 0.0f ? 1.0f : __fdiv_rn(m, 127.0f);
        }
        const float rsc = __frcp_rn(sc);
        float a1 = 0.0f;  // sum of |code| (exact: at most 127 * 8192 < 2^24)
        if (valid) {
            if (t == 0) scale[row] = sc;
#pragma unroll
            for (int i = 0; i < kVPT; ++i) {
                int j = t + i * tpr;
                if (j < K4) a1 += store_codes<DIR>(v[i], sc, rsc, row * K4 + j, q, op);
            }
        }
        if (l1) {
            a1 = group_sum(a1, tpr, red);
            if (valid && t == 0) l1[row] = (int32_t)a1;
        }
    }
}

// Long rows (K4 > kThreads * kMaxVPT): one block per row, the row is read twice.
template <int DIR>
__global__ void __launch_bounds__(kThreads) quantize_rows_loop(
    const float *__restrict__ A, const float *__restrict__ s, int64_t rows, int K4,
    int8_t *__restrict__ q, float *__restrict__ scale, __nv_bfloat16 *__restrict__ op,
    int32_t *__restrict__ l1, float fixed_scale) {
    pdl_launch_dependents();
    pdl_wait();
    __shared__ float red[kThreads / 32];
    const float4 *s4 = reinterpret_cast<const float4 *>(s);
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
        const float4 *a4 = reinterpret_cast<const float4 *>(A) + row * K4;
        float sc = fixed_scale;
        if (DIR != kActStatic) {
            float m = 0.0f;
            for (int j = threadIdx.x; j < K4; j += kThreads) {
                float4 x = __ldg(a4 + j), sv = __ldg(s4 + j);
                m = fmaxf(m, fmaxf(fmaxf(fabsf(smooth_one(x.x, sv.x, DIR)),
                                         fabsf(smooth_one(x.y, sv.y, DIR))),
                                   fmaxf(fabsf(smooth_one(x.z, sv.z, DIR)),
                                         fabsf(smooth_one(x.w, sv.w, DIR)))));
            }
            m = group_max(m, kThreads, red);
            sc = m == 0.0f ? 1.0f : __fdiv_rn(m, 127.0f);
        }
        const float rsc = __frcp_rn(sc);
        if (threadIdx.x == 0) scale[row] = sc;
        int a1 = 0;  // integer: long rows may exceed 2^24
        for (int j = threadIdx.x; j < K4; j += kThreads) {
            float4 x = __ldcs(a4 + j), sv = __ldg(s4 + j);
            float4 v = make_float4(smooth_one(x.x, sv.x, DIR), smooth_one(x.y, sv.y, DIR),
                                   smooth_one(x.z, sv.z, DIR), smooth_one(x.w, sv.w, DIR));
            a1 += (int)store_codes<DIR>(v, sc, rsc, row * K4 + j, q, op);
        }
        if (l1) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) a1 += __shfl_xor_sync(0xffffffffu, a1, o);
            if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = __int_as_float(a1);
            __syncthreads();
            if (threadIdx.x == 0) {
                long long tot = 0;
                for (int w = 0; w < kThreads / 32; ++w) tot += __float_as_int(red[w]);
                l1[row] = tot > 0x7fffffffLL ? 0x7fffffff : (int32_t)tot;
            }
            __syncthreads();
        }
    }
}

// Smooth-Static calibration: per-tensor maximum of |fl(x / s)| (IEEE
// division; offline), merged into *amax with an integer atomicMax.
__global__ void __launch_bounds__(kThreads) act_absmax_kernel(const float *__restrict__ A,
                                                              const float *__restrict__ s,
                                                              int64_t rows, int K4,
                                                              float *__restrict__ amax) {
    pdl_launch_dependents();
    pdl_wait();
    const float4 *a4 = reinterpret_cast<const float4 *>(A);
    const float4 *s4 = reinterpret_cast<const float4 *>(s);
    const int64_t total = rows * (int64_t)K4;
    float m = 0.0f;
    for (int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * kThreads) {
        const float4 x = __ldcs(a4 + i), sv = __ldg(s4 + (int)(i % K4));
        m = fmaxf(m, fmaxf(fmaxf(fabsf(__fdiv_rn(x.x, sv.x)), fabsf(__fdiv_rn(x.y, sv.y))),
                           fmaxf(fabsf(__fdiv_rn(x.z, sv.z)), fabsf(__fdiv_rn(x.w, sv.w)))));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((threadIdx.x & 31) == 0) atomicMax(reinterpret_cast<int *>(amax), __float_as_int(m));
}

// Smooth-Static per-tensor scale from the calibrated maximum: fl32(amax / 127)
// (IEEE division), 1 for a zero maximum.
__global__ void static_scale_kernel(const float *__restrict__ amax, float *__restrict__ scale) {
    pdl_launch_dependents();
    pdl_wait();
    const float a = *amax;
    *scale = a == 0.0f ? 1.0f : __fdiv_rn(a, 127.0f);
}

// Column maxima, merged into amax with an integer atomicMax (the bit patterns
// of non-negative floats order like the floats).
__global__ void __launch_bounds__(kThreads) channel_absmax_kernel(
    const float *__restrict__ A, int64_t rows, int64_t cols, int64_t rows_per_block,
    float *__restrict__ amax) {
    pdl_launch_dependents();
    pdl_wait();
    const int64_t j = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    if (j >= cols) return;
    const int64_t r0 = (int64_t)blockIdx.y * rows_per_block;
    const int64_t r1 = min(rows, r0 + rows_per_block);
    float m = 0.0f;
    for (int64_t i = r0; i < r1; ++i) m = fmaxf(m, fabsf(__ldg(A + i * cols + j)));
    atomicMax(reinterpret_cast<int *>(amax) + j, __float_as_int(m));
}

__global__ void smooth_factor_kernel(const float *__restrict__ ax, const float *__restrict__ aw,
                                     int64_t K, double alpha, float *__restrict__ s) {
    pdl_launch_dependents();
    pdl_wait();
    const int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (j >= K) return;
    double x = (double)ax[j], w = (double)aw[j];
    s[j] = (x == 0.0 || w == 0.0) ? 1.0f : (float)(pow(x, alpha) / pow(w, 1.0 - alpha));
}

template <typename Kern>
int resident_blocks(Kern k) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kThreads, 0) != cudaSuccess ||
        per_sm < 1)
        per_sm = 1;
    return per_sm;
}

// LayerNorm with the next linear's quantiser fused in (the encoder's
// normalisation, Table 3, emitting the smoothed int8 codes SmoothQuant's
// folding implies).  A group of tpr threads owns a row, held in registers:
//   mean = fl(sum / K), var = fl(sum (h - mean)^2 / K) (fp32 tree sums),
//   y = fma((h - mean) * rstd, gamma, beta), rstd = RN(1 / sqrt(var + eps)),
// then the quantiser of KIND on y: v = fl(y / s), per-token scale from the row
// maximum (dynamic) or the given scale (static), codes as quantize_rows_reg.
// y is also stored when Y is given.
template <int KIND, int kVPT>
__global__ void __launch_bounds__(kThreads) layernorm_quant_kernel(
    const float *__restrict__ H, const float *__restrict__ gamma, const float *__restrict__ beta,
    float eps, const float *__restrict__ s, int64_t rows, int K4, int tpr,
    float *__restrict__ Y, int8_t *__restrict__ q, float *__restrict__ scale,
    __nv_bfloat16 *__restrict__ op, int32_t *__restrict__ l1, float fixed_scale) {
    pdl_launch_dependents();
    pdl_wait();
    __shared__ float red[kThreads / 32];
    const int rpb = kThreads / tpr;
    const int g = threadIdx.x / tpr;
    const int t = threadIdx.x % tpr;
    const float4 *s4 = reinterpret_cast<const float4 *>(s);
    const float4 *g4 = reinterpret_cast<const float4 *>(gamma);
    const float4 *b4 = reinterpret_cast<const float4 *>(beta);
    const float Kf = (float)(4 * K4);
    const int64_t tiles = (rows + rpb - 1) / rpb;
    for (int64_t tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
        const int64_t row = tile * rpb + g;
        const bool valid = row < rows;
        const float4 *h4 = reinterpret_cast<const float4 *>(H) + (valid ? row : 0) * K4;
        float4 v[kVPT];
#pragma unroll
        for (int i = 0; i < kVPT; ++i) {
            const int j = t + i * tpr;
            v[i] = (valid && j < K4) ? __ldcs(h4 + j) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        float sum = 0.0f;
#pragma unroll
        for (int i = 0; i < kVPT; ++i) sum += (v[i].x + v[i].y) + (v[i].z + v[i].w);
        const float mean = __fdiv_rn(group_sum(sum, tpr, red), Kf);
        float sq = 0.0f;
#pragma unroll
        for (int i = 0; i < kVPT; ++i) {
            const int j = t + i * tpr;
            if (j < K4) {
                v[i] = make_float4(v[i].x - mean, v[i].y - mean, v[i].z - mean, v[i].w - mean);
                sq += (v[i].x * v[i].x + v[i].y * v[i].y) + (v[i].z * v[i].z + v[i].w * v[i].w);
            }
        }
        const float var = __fdiv_rn(group_sum(sq, tpr, red), Kf);
        const float rstd = __frsqrt_rn(__fadd_rn(var, eps));
        float m = 0.0f;
#pragma unroll
        for (int i = 0; i < kVPT; ++i) {
            const int j = t + i * tpr;
            if (j < K4) {
                const float4 gv = __ldg(g4 + j), bv = __ldg(b4 + j), sv = __ldg(s4 + j);
                float4 y;
                y.x = __fmaf_rn(__fmul_rn(v[i].x, rstd), gv.x, bv.x);
                y.y = __fmaf_rn(__fmul_rn(v[i].y, rstd), gv.y, bv.y);
                y.z = __fmaf_rn(__fmul_rn(v[i].z, rstd), gv.z, bv.z);
                y.w = __fmaf_rn(__fmul_rn(v[i].w, rstd), gv.w, bv.w);
                if (Y && valid) reinterpret_cast<float4 *>(Y)[row * K4 + j] = y;
                v[i] = make_float4(__fdiv_rn(y.x, sv.x), __fdiv_rn(y.y, sv.y),
                                   __fdiv_rn(y.z, sv.z), __fdiv_rn(y.w, sv.w));
                if (KIND == kActDynamic)
                    m = fmaxf(m, fmaxf(fmaxf(fabsf(v[i].x), fabsf(v[i].y)),
                                       fmaxf(fabsf(v[i].z), fabsf(v[i].w))));
            }
        }
        float sc = fixed_scale;
        if (KIND == kActDynamic) {
            m = group_max(m, tpr, red);
            sc = m == 0.0f ? 1.0f : __fdiv_rn(m, 127.0f);
        }
        const float rsc = __frcp_rn(sc);
        float a1 = 0.0f;
        if (valid) {
            if (t == 0) scale[row] = sc;
#pragma unroll
            for (int i = 0; i < kVPT; ++i) {
                const int j = t + i * tpr;
                if (j < K4) a1 += store_codes<KIND>(v[i], sc, rsc, row * K4 + j, q, op);
            }
        }
        if (l1) {
            a1 = group_sum(a1, tpr, red);
            if (valid && t == 0) l1[row] = (int32_t)a1;
        }
    }
}

}  // namespace

sq_status launch_quantize_rows(int direction, const float *A, const float *s, int64_t rows,
                               int64_t K, int8_t *q, float *scale, __nv_bfloat16 *op,
                               int32_t *l1, float fixed_scale, cudaStream_t st) {
    DeviceInfo di;
    sq_status rc = device_info(&di);
    if (rc != SQ_OK) return rc;
    const int K4 = (int)(K / 4);
    if (K4 <= kThreads * kMaxVPT) {
        // 4 float4 per thread when that covers the row with one block (more
        // resident warps), else 8
        const bool small = K4 <= kThreads * 4;
        const int vpt = small ? 4 : 8;
        int tpr = 32;
        while (tpr * vpt < K4) tpr <<= 1;
        const int rpb = kThreads / tpr;
        const int64_t tiles = (rows + rpb - 1) / rpb;
        void (*kern)(const float *, const float *, int64_t, int, int, int8_t *, float *,
                     __nv_bfloat16 *, int32_t *, float);
        if (direction == kActDynamic)
            kern = small ? quantize_rows_reg<kActDynamic, 4> : quantize_rows_reg<kActDynamic, 8>;
        else if (direction == kWeight)
            kern = small ? quantize_rows_reg<kWeight, 4> : quantize_rows_reg<kWeight, 8>;
        else
            kern = small ? quantize_rows_reg<kActStatic, 4> : quantize_rows_reg<kActStatic, 8>;
        static int per_sm[3][2] = {{0, 0}, {0, 0}, {0, 0}};
        int &occ = per_sm[direction][small ? 0 : 1];
        if (!occ) occ = resident_blocks(kern);
        const int64_t grid = std::min<int64_t>(tiles, (int64_t)di.sms * occ);
        return launch_pdl(kern, dim3((unsigned)grid), dim3(kThreads), 0, st, 1, A, s, rows, K4,
                          tpr, q, scale, op, l1, fixed_scale);
    } else {
        auto kern = direction == kActDynamic ? quantize_rows_loop<kActDynamic>
                    : direction == kWeight       ? quantize_rows_loop<kWeight>
                                                 : quantize_rows_loop<kActStatic>;
        const int64_t grid = std::min<int64_t>(rows, (int64_t)di.sms * 8);
        return launch_pdl(kern, dim3((unsigned)grid), dim3(kThreads), 0, st, 1, A, s, rows, K4, q,
                          scale, op, l1, fixed_scale);
    }
}

sq_status launch_layernorm_quant(const float *H, const float *gamma, const float *beta,
                                 float eps, const float *s, int64_t rows, int64_t K,
                                 float static_scale, float *Y, int8_t *q, float *scale,
                                 __nv_bfloat16 *op, int32_t *l1, cudaStream_t st) {
    DeviceInfo di;
    sq_status rc = device_info(&di);
    if (rc != SQ_OK) return rc;
    const int K4 = (int)(K / 4);
    if (K4 > kThreads * kMaxVPT) return SQ_ERR_UNSUPPORTED;
    const bool small = K4 <= kThreads * 4;
    const int vpt = small ? 4 : 8;
    int tpr = 32;
    while (tpr * vpt < K4) tpr <<= 1;
    const int rpb = kThreads / tpr;
    const int64_t tiles = (rows + rpb - 1) / rpb;
    using Kern = void (*)(const float *, const float *, const float *, float, const float *,
                          int64_t, int, int, float *, int8_t *, float *, __nv_bfloat16 *,
                          int32_t *, float);
    static const Kern kerns[2][2] = {
        {layernorm_quant_kernel<kActDynamic, 4>, layernorm_quant_kernel<kActDynamic, 8>},
        {layernorm_quant_kernel<kActStatic, 4>, layernorm_quant_kernel<kActStatic, 8>}};
    const Kern kern = kerns[static_scale > 0.0f ? 1 : 0][small ? 0 : 1];
    static int per_sm[2][2] = {};
    int &occ = per_sm[static_scale > 0.0f ? 1 : 0][small ? 0 : 1];
    if (!occ) occ = resident_blocks(kern);
    const int64_t grid = std::min<int64_t>(tiles, (int64_t)di.sms * occ);
    return launch_pdl(kern, dim3((unsigned)grid), dim3(kThreads), 0, st, 1, H, gamma, beta, eps, s,
                      rows, K4, tpr, Y, q, scale, op, l1, static_scale);
}

sq_status launch_act_absmax(const float *A, const float *s, int64_t rows, int64_t K,
                            float *amax, cudaStream_t st) {
    DeviceInfo di;
    sq_status rc = device_info(&di);
    if (rc != SQ_OK) return rc;
    const int64_t total4 = rows * (K / 4);
    const int64_t grid = std::max<int64_t>(
        1, std::min<int64_t>((total4 + kThreads - 1) / kThreads, (int64_t)di.sms * 8));
    return launch_pdl(act_absmax_kernel, dim3((unsigned)grid), dim3(kThreads), 0, st, 1, A, s, rows,
                      (int)(K / 4), amax);
}

sq_status launch_static_scale(const float *amax, float *scale, cudaStream_t st) {
    return launch_pdl(static_scale_kernel, dim3(1), dim3(1), 0, st, 1, amax, scale);
}

sq_status launch_channel_absmax(const float *A, int64_t rows, int64_t cols, float *amax,
                                cudaStream_t st) {
    DeviceInfo di;
    sq_status rc = device_info(&di);
    if (rc != SQ_OK) return rc;
    const int64_t gx = (cols + kThreads - 1) / kThreads;
    int64_t gy = std::max<int64_t>(1, ((int64_t)di.sms * 8 + gx - 1) / gx);
    gy = std::min<int64_t>(gy, std::min<int64_t>(rows, 65535));
    const int64_t rpb = (rows + gy - 1) / gy;
    gy = (rows + rpb - 1) / rpb;
    if (gx > 0x7fffffff) return SQ_ERR_UNSUPPORTED;
    return launch_pdl(channel_absmax_kernel, dim3((unsigned)gx, (unsigned)gy), dim3(kThreads), 0, st,
                      1, A, rows, cols, rpb, amax);
}

sq_status launch_smooth_factor(const float *ax, const float *aw, int64_t K, float alpha,
                               float *s, cudaStream_t st) {
    const int64_t grid = (K + kThreads - 1) / kThreads;
    return launch_pdl(smooth_factor_kernel, dim3((unsigned)grid), dim3(kThreads), 0, st, 1, ax, aw,
                      K, (double)alpha, s);
}

}  // namespace sq

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
#include <mutex>

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

__device__ __forceinline__ float max3_nan(float a, float b, float c) {
    float d;
    asm("max.NaN.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}
__device__ __forceinline__ float max2_nan(float a, float b) {
    float d;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
    return d;
}
// RN(1/s) where the corrected reciprocal division is proven (|s| in
// [2^-20, 2^20]), NaN elsewhere: the division tables' entry for s
__device__ __forceinline__ float smooth_recip(float x) {
    const float a = fabsf(x);
    return (a >= 0x1p-20f && a <= 0x1p20f) ? __frcp_rn(x) : __int_as_float(0x7fffffff);
}

// Reductions across the tpr threads of row group g for the register and
// LayerNorm kernels, synchronised on the group's own named barrier (1 + g, tpr threads)
// instead of the block's, so that the groups of a block run their tiles
// independently.  The caller alternates two slot arrays between consecutive
// reductions: a slot is rewritten only after the group has passed the next
// reduction's barrier, hence after every thread read it, so one barrier per
// reduction is enough.
__device__ __forceinline__ void row_group_sync(int g, int tpr) {
    asm volatile("bar.sync %0, %1;" ::"r"(1 + g), "r"(tpr) : "memory");
}
template <int OP>  // 0: max (NaN kept), 1: max, 2: sum
__device__ __forceinline__ float row_group_reduce(float v, int tpr, int g, float *red) {
    auto op = [](float a, float b) {
        return OP == 0 ? max2_nan(a, b) : OP == 1 ? fmaxf(a, b) : a + b;
    };
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = op(v, __shfl_xor_sync(0xffffffffu, v, o));
    if (tpr > 32) {
        const int wpg = tpr >> 5;
        if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
        row_group_sync(g, tpr);
        v = red[g * wpg];
        for (int w = 1; w < wpg; ++w) v = op(v, red[g * wpg + w]);
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


// ---------------------------------------------------------------------------
// Smooth-Dynamic activation quantiser (Table 10's run-time step).
//
// One persistent block per SM streams its rows through a ring of shared-memory
// stages: a producer thread copies `groups` consecutive rows per stage with one
// bulk copy (cp.async.bulk, completion counted on the stage's mbarrier), and
// each group of `wpr` consumer warps codes one row of the stage from shared
// memory, then frees the stage.  The copies of the next stages stay in flight
// while rows are coded, so the row maximum's dependency (every code waits for
// it) no longer empties the memory pipeline.  Lane l of warp w of a group
// holds the float4 f = (32 w + l) + 32 wpr i, i < VPT4, of its row.
//  * row maximum: max |fl(x / s)| by the corrected reciprocal division
//    q0 = RN(x y), q = RN(q0 + RN(x - s q0) y), y = RN(1/s) (div_smooth: the
//    IEEE quotient where |s| is in [2^-20, 2^20], |x| >= 2^-100 and |q0| <=
//    2^100), with s and y per column from tables in shared memory (y NaN where
//    |s| is outside that range).  Rows whose maximum is NaN or outside
//    [2^-60, 2^100] take the exact path, so the maximum, and the scale
//    fl(max / 127), are bit-exact.
//  * codes: p = RN(RN(x y) RN(1/scale)) is within 5u of fl(x / s) / scale,
//    |fl(x / s) / scale| <= 127.0001, and so within 4.2e-5 of
//    fl(fl(x / s) / scale); where p is farther than 2^-14 from every
//    half-integer, rint(p) is the round-half-even code (rint by the addition
//    and subtraction of 1.5 * 2^23, on f32x2 pairs).  A float4 holding a value
//    within 2^-14 of a half-integer recomputes those elements with IEEE
//    divisions.  Elements with subnormal products are below 2^-126 while the
//    scale is above 2^-67: their code is 0 either way.
// Every wait (stages, group reductions) is bounded; on expiry the block
// records an error for sq_device_status, lets its copies land and exits.
constexpr int kRingWarps = 16;  // consumer warps of a block at most
// modes of the register kernel: the row maximum found, given, or none (static)
constexpr int kRegDynamic = 0, kRegGiven = 1, kRegStatic = 2;
constexpr float kRoundMagic = 12582912.0f;      // 1.5 * 2^23
constexpr float kTieLimit = 0.49993896484375f;  // 0.5 - 2^-14
constexpr unsigned long long kRingTimeoutNs = 2000000000ull;

__device__ unsigned int g_quant_error;

__device__ __forceinline__ uint32_t saddr(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ bool mb_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ uint64_t gtimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Bounded wait for the phase of parity `parity`; false (and the block's abort
// flag and the error word set) when it runs out or the block has aborted.
__device__ __noinline__ bool mb_wait_slow(uint32_t bar, uint32_t parity, volatile int *abort) {
    const uint64_t t0 = gtimer();
    for (uint32_t it = 1;; ++it) {
        if (mb_try_wait(bar, parity)) return true;
        if ((it & 63u) == 0) {
            if (*abort) return false;
            if (gtimer() - t0 > kRingTimeoutNs) {
                *abort = 1;
                atomicOr(&g_quant_error, 1u);
                return false;
            }
        }
    }
}
__device__ __forceinline__ bool mb_wait(uint32_t bar, uint32_t parity, volatile int *abort) {
    if (mb_try_wait(bar, parity)) return true;
    return mb_wait_slow(bar, parity, abort);
}
// wait used while letting issued copies land (ignores the abort flag)
__device__ __noinline__ void mb_drain(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = gtimer();
    while (!mb_try_wait(bar, parity))
        if (gtimer() - t0 > kRingTimeoutNs) {
            atomicOr(&g_quant_error, 2u);
            return;
        }
}

// The warps of one row group and their reduction state: partials in red
// (two phases used in turn), an mbarrier of count wpr per group.
struct RingGroup {
    int wpr, g, wg, lane;
    uint32_t bar, bph;
    float *red;  // [2][8]
    int rp;
    volatile int *abort;
};

// Group-wide NaN-keeping maximum (sum when SUM); false if the block aborted.
// A phase of red is written again only after the next reduction's barrier,
// which every warp reaches after reading it.
template <bool SUM>
__device__ __forceinline__ bool group_reduce(float &v, RingGroup &G) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float w = __shfl_xor_sync(0xffffffffu, v, o);
        v = SUM ? v + w : max2_nan(v, w);
    }
    if (G.wpr == 1) return true;
    if (G.lane == 0) {
        G.red[8 * G.rp + G.wg] = v;
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(G.bar) : "memory");
    }
    int ok = 1;
    if (G.lane == 0) ok = mb_wait(G.bar, G.bph, G.abort);
    ok = __shfl_sync(0xffffffffu, ok, 0);
    __syncwarp();  // lane 0's acquire orders the other warps' partials for every lane
    G.bph ^= 1u;
    if (!ok) return false;
    v = G.red[8 * G.rp];
    for (int w = 1; w < G.wpr; ++w) v = SUM ? v + G.red[8 * G.rp + w] : max2_nan(v, G.red[8 * G.rp + w]);
    G.rp ^= 1;
    return true;
}

// Four codes (integer-valued floats) to the outputs at element offset off
// (a multiple of 4): bf16 operand (8 bytes) and/or int8 (4 bytes).
__device__ __forceinline__ void store4_codes(float t0, float t1, float t2, float t3, int64_t off,
                                             int8_t *q, __nv_bfloat16 *op) {
    if (op) {
        // integers |t| <= 127: the high half of the fp32 pattern is the exact bf16
        const uint2 w = make_uint2(__byte_perm(__float_as_uint(t0), __float_as_uint(t1), 0x7632),
                                   __byte_perm(__float_as_uint(t2), __float_as_uint(t3), 0x7632));
        *reinterpret_cast<uint2 *>(op + off) = w;
    }
    if (q) {
        // t + 1.5 * 2^23 holds the code in its low byte (two's complement)
        float f0, f1, f2, f3;
        upk(add2(pk(t0, t1), pk(kRoundMagic, kRoundMagic)), f0, f1);
        upk(add2(pk(t2, t3), pk(kRoundMagic, kRoundMagic)), f2, f3);
        *reinterpret_cast<uint32_t *>(q + off) =
            __byte_perm(__byte_perm(__float_as_uint(f0), __float_as_uint(f1), 0x0040),
                        __byte_perm(__float_as_uint(f2), __float_as_uint(f3), 0x0040), 0x5410);
    }
}

// The code of x as the definition states it: round_half_even(fl(fl(x / s) /
// scale)), clamped (IEEE divisions; the rare near-tie elements).  By value and
// not inlined, so that the caller's register arrays stay in registers.
__device__ __noinline__ float exact_code(float x, float s, float scale) {
    return fminf(127.0f, fmaxf(-127.0f, rintf(__fdiv_rn(__fdiv_rn(x, s), scale))));
}

// |fl(x / s)| (IEEE division), out of line for the rare exact path
__device__ __noinline__ float abs_quotient(float x, float s) { return fabsf(__fdiv_rn(x, s)); }

// Smooth-Dynamic activations, the row in registers (K4 <= tpr * kVPT): the
// arithmetic of the ring kernel below on the register kernel's layout (tpr
// threads per row, float4 f = t + i tpr of it in thread t), with the
// smoothing factors, negated, and their reciprocals in shared-memory tables
// (2 x K floats) built once per block.
//  * row maximum of |fl(x / s)| by the corrected reciprocal division with
//    y = RN(1/s) (NaN for |s| outside [2^-20, 2^20]), on f32x2 pairs;
//  * codes: rint of p = RN(RN(x y) RN(1/scale)), the IEEE divisions for a
//    value within 2^-14 of a half-integer.
// A row whose maximum is NaN or outside [2^-60, 2^100] takes IEEE divisions
// throughout (the maximum is uniform across the row group, and so is the
// choice; the group's reductions sync on its own barrier).  GIVEN: the row
// maxima come from row_amax (as the row-maximum GEMM epilogue leaves them) instead of the reduction, and the codes saturate
// at +-127 (a maximum below the true one cannot wrap them); an out-of-range
// maximum still sends the block to the IEEE path, which finds its own.
// STATIC (Smooth-Static): no maximum; the given per-tensor scale, codes
// saturating at +-127 (the launcher takes this kernel only for scales in
// [2^-60, 2^60]: a subnormal or overflowing product then decides no code, and
// a product at or beyond 2^22 fails the near-tie check and takes the IEEE
// division).  While a tile is coded, one thread per row group asks for the
// group's next row to be brought into L2 (a bulk prefetch, no registers held),
// so that DRAM stays busy through the reductions and stores (measured 7% on
// 8192 x 4096; a second row ahead measured slower).  TAB: the tables are
// copied from the caller's division table of s instead of formed in every
// block (the block's reciprocals cost 3% of the quantiser's time in the
// BERT-large step, 2.51 -> 2.43 ms; reading the table through L1 inside the
// tile loop, with no shared-memory copy, measured 8% slower than forming it).
template <int kVPT, int MODE, bool TAB>
__global__ void __launch_bounds__(kThreads, kVPT == 4 ? 4 : 2) quantize_act_reg(
    const float *__restrict__ A, const float *__restrict__ s, const float4 *__restrict__ tab,
    int64_t rows, int K4, int tpr, int8_t *__restrict__ q, float *__restrict__ scale,
    __nv_bfloat16 *__restrict__ op, int32_t *__restrict__ l1,
    const float *__restrict__ row_amax, float fixed_scale) {
    constexpr bool GIVEN = MODE == kRegGiven, STATIC = MODE == kRegStatic;
    extern __shared__ float4 qtab[];
    float4 *nstab = qtab;       // -s
    float4 *ytab = qtab + K4;   // RN(1/s) or NaN
    pdl_launch_dependents();
    pdl_wait();
    __shared__ float red2[2][kThreads / 32];
    int rb = 0;  // the slot array of the group's next reduction
    const int rpb = kThreads / tpr;
    const int g = threadIdx.x / tpr;
    const int t = threadIdx.x % tpr;
    {
        // the group's first row on its way into L2 while the tables are built
        const int64_t row0 = (int64_t)blockIdx.x * rpb + g;
        if (t == 0 && row0 < rows)
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(
                             reinterpret_cast<const float4 *>(A) + row0 * K4),
                         "r"((uint32_t)K4 * 16u)
                         : "memory");
    }
    if (TAB) {
        // the caller's division table: float4 2j and 2j + 1 hold the pairs
        // (-s, RN(1/s)) of columns 4j .. 4j + 3
        for (int j = threadIdx.x; j < K4; j += kThreads) {
            const float4 a = __ldg(tab + 2 * j), b = __ldg(tab + 2 * j + 1);
            nstab[j] = make_float4(a.x, a.z, b.x, b.z);
            ytab[j] = make_float4(a.y, a.w, b.y, b.w);
        }
    } else {
        const float4 *s4 = reinterpret_cast<const float4 *>(s);
        for (int j = threadIdx.x; j < K4; j += kThreads) {
            const float4 v = __ldg(s4 + j);
            nstab[j] = make_float4(-v.x, -v.y, -v.z, -v.w);
            ytab[j] = make_float4(smooth_recip(v.x), smooth_recip(v.y), smooth_recip(v.z),
                                  smooth_recip(v.w));
        }
    }
    __syncthreads();
    const unsigned long long magic2 = pk(kRoundMagic, kRoundMagic);
    const int64_t tiles = (rows + rpb - 1) / rpb;
    for (int64_t tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
        const int64_t row = tile * rpb + g;
        const bool valid = row < rows;
        const float4 *a4 = reinterpret_cast<const float4 *>(A) + (valid ? row : 0) * K4;
        {
            // the row this thread group codes next, into L2 while this one is coded
            const int64_t nrow = row + (int64_t)gridDim.x * rpb;
            if (t == 0 && nrow < rows)
                asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(
                                 reinterpret_cast<const float4 *>(A) + nrow * K4),
                             "r"((uint32_t)K4 * 16u)
                             : "memory");
        }
        float4 v[kVPT];
#pragma unroll
        for (int i = 0; i < kVPT; ++i) {
            int j = t + i * tpr;
            v[i] = (valid && j < K4) ? __ldcs(a4 + j) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        // row maximum, div_smooth on f32x2 pairs (GIVEN: read; STATIC: none)
        float m = 0.0f;
        if (GIVEN) m = valid ? __ldg(row_amax + row) : 0.0f;
#pragma unroll
        for (int i = 0; i < kVPT; ++i) {
            const int j = t + i * tpr;
            if (MODE != kRegDynamic || j >= K4) continue;
            const float4 y = ytab[j], ns = nstab[j];
            const unsigned long long x01 = pk(v[i].x, v[i].y), x23 = pk(v[i].z, v[i].w);
            const unsigned long long y01 = pk(y.x, y.y), y23 = pk(y.z, y.w);
            const unsigned long long q01 = mul2(x01, y01), q23 = mul2(x23, y23);
            float d0, d1, d2, d3;
            upk(fma2(fma2(q01, pk(ns.x, ns.y), x01), y01, q01), d0, d1);
            upk(fma2(fma2(q23, pk(ns.z, ns.w), x23), y23, q23), d2, d3);
            m = max3_nan(m, fabsf(d0), fabsf(d1));
            m = max3_nan(m, fabsf(d2), fabsf(d3));
        }
        if (MODE == kRegDynamic) {
            m = row_group_reduce<0>(m, tpr, g, red2[rb]);
            rb ^= 1;
        }
        const bool exact = !STATIC && valid && !(m >= 0x1p-60f && m <= 0x1p100f);
        float a1 = 0.0f;
        if (exact) {
            // IEEE divisions throughout (the definition as stated)
            float me = 0.0f;
            for (int i = 0; i < kVPT; ++i) {
                const int j = t + i * tpr;
                if (j >= K4) continue;
                const float4 ns = nstab[j];
                me = fmaxf(me, fmaxf(abs_quotient(v[i].x, -ns.x), abs_quotient(v[i].y, -ns.y)));
                me = fmaxf(me, fmaxf(abs_quotient(v[i].z, -ns.z), abs_quotient(v[i].w, -ns.w)));
            }
            me = row_group_reduce<1>(me, tpr, g, red2[rb]);
            rb ^= 1;
            const float sc = me == 0.0f ? 1.0f : abs_quotient(me, 127.0f);
            if (valid) {
                if (t == 0) scale[row] = sc;
                for (int i = 0; i < kVPT; ++i) {
                    const int j = t + i * tpr;
                    if (j >= K4) continue;
                    const float4 ns = nstab[j];
                    const float c0 = exact_code(v[i].x, -ns.x, sc);
                    const float c1 = exact_code(v[i].y, -ns.y, sc);
                    const float c2 = exact_code(v[i].z, -ns.z, sc);
                    const float c3 = exact_code(v[i].w, -ns.w, sc);
                    store4_codes(c0, c1, c2, c3, ((int64_t)row * K4 + j) * 4, q, op);
                    a1 += (fabsf(c0) + fabsf(c1)) + (fabsf(c2) + fabsf(c3));
                }
            }
        } else {
            const float sc = STATIC ? fixed_scale : __fdiv_rn(m, 127.0f);
            const float rsc = __frcp_rn(sc);
            const unsigned long long r2 = pk(rsc, rsc);
            if (valid) {
                if (t == 0) scale[row] = sc;
#pragma unroll
                for (int i = 0; i < kVPT; ++i) {
                    const int j = t + i * tpr;
                    if (j >= K4) continue;
                    const float4 y = ytab[j];
                    const unsigned long long p01 = mul2(mul2(pk(v[i].x, v[i].y), pk(y.x, y.y)), r2);
                    const unsigned long long p23 = mul2(mul2(pk(v[i].z, v[i].w), pk(y.z, y.w)), r2);
                    const unsigned long long t01 = sub2(add2(p01, magic2), magic2);
                    const unsigned long long t23 = sub2(add2(p23, magic2), magic2);
                    float c[4], d[4];
                    upk(t01, c[0], c[1]);
                    upk(t23, c[2], c[3]);
                    upk(sub2(p01, t01), d[0], d[1]);
                    upk(sub2(p23, t23), d[2], d[3]);
                    // NaN kept: with the maxima given, a column whose s has no
                    // reciprocal (NaN in the table) reaches this point
                    const float dm = max3_nan(fabsf(d[0]), fabsf(d[1]),
                                              max2_nan(fabsf(d[2]), fabsf(d[3])));
                    if (!(dm <= kTieLimit)) {
                        // rare: a value within 2^-14 of a half-integer (or NaN)
                        const float4 ns = nstab[j];
                        if (!(fabsf(d[0]) <= kTieLimit)) c[0] = exact_code(v[i].x, -ns.x, sc);
                        if (!(fabsf(d[1]) <= kTieLimit)) c[1] = exact_code(v[i].y, -ns.y, sc);
                        if (!(fabsf(d[2]) <= kTieLimit)) c[2] = exact_code(v[i].z, -ns.z, sc);
                        if (!(fabsf(d[3]) <= kTieLimit)) c[3] = exact_code(v[i].w, -ns.w, sc);
                    }
                    if (MODE != kRegDynamic) {
#pragma unroll
                        for (int e = 0; e < 4; ++e) c[e] = fminf(127.0f, fmaxf(-127.0f, c[e]));
                    }
                    store4_codes(c[0], c[1], c[2], c[3], ((int64_t)row * K4 + j) * 4, q, op);
                    a1 += (fabsf(c[0]) + fabsf(c[1])) + (fabsf(c[2]) + fabsf(c[3]));
                }
            }
        }
        if (l1) {
            a1 = row_group_reduce<2>(a1, tpr, g, red2[rb]);  // exact: <= 127 * 8192 < 2^24
            rb ^= 1;
            if (valid && t == 0) l1[row] = (int32_t)a1;
        }
    }
}

// LayerNorm with the next linear's quantiser fused in (the encoder's
// normalisation, Table 3, emitting the smoothed int8 codes SmoothQuant's
// folding implies).  A group of tpr threads owns a row, held in registers:
//   mean = fl(sum / K), var = fl(sum (h - mean)^2 / K) (fp32 tree sums),
//   y = fma((h - mean) * rstd, gamma, beta), rstd = RN(1 / sqrt(var + eps)),
// then the quantiser of KIND on y with the register kernel's arithmetic and
// shared-memory division tables: the row maximum of |fl(y / s)| by the
// corrected reciprocal division (dynamic) or the given scale (static), codes
// from p = RN(RN(y RN(1/s)) RN(1/scale)) with the near-tie elements on IEEE
// divisions.  A row whose maximum is NaN or outside [2^-60, 2^100], and every
// row when a static scale lies outside [2^-60, 2^60] (fast == 0), takes IEEE
// divisions throughout.  y is also stored when Y is given.  Row reductions
// sync on each row group's named barrier.
template <int KIND, int kVPT>
__global__ void __launch_bounds__(kThreads, kVPT == 4 ? 4 : 2) layernorm_quant_kernel(
    const float *__restrict__ H, const float *__restrict__ gamma, const float *__restrict__ beta,
    float eps, const float *__restrict__ s, int64_t rows, int K4, int tpr,
    float *__restrict__ Y, int8_t *__restrict__ q, float *__restrict__ scale,
    __nv_bfloat16 *__restrict__ op, int32_t *__restrict__ l1, float fixed_scale, int fast) {
    extern __shared__ float4 qtab[];
    float4 *nstab = qtab;       // -s
    float4 *ytab = qtab + K4;   // RN(1/s) or NaN
    pdl_launch_dependents();
    pdl_wait();
    __shared__ float red2[2][kThreads / 32];
    int rb = 0;  // the slot array of the group's next reduction (see row_group_reduce)
    const int rpb = kThreads / tpr;
    const int g = threadIdx.x / tpr;
    const int t = threadIdx.x % tpr;
    const float4 *s4 = reinterpret_cast<const float4 *>(s);
    const float4 *g4 = reinterpret_cast<const float4 *>(gamma);
    const float4 *b4 = reinterpret_cast<const float4 *>(beta);
    for (int j = threadIdx.x; j < K4; j += kThreads) {
        const float4 v = __ldg(s4 + j);
        nstab[j] = make_float4(-v.x, -v.y, -v.z, -v.w);
        ytab[j] = make_float4(smooth_recip(v.x), smooth_recip(v.y), smooth_recip(v.z),
                              smooth_recip(v.w));
    }
    __syncthreads();
    const unsigned long long magic2 = pk(kRoundMagic, kRoundMagic);
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
        const float mean = __fdiv_rn(row_group_reduce<2>(sum, tpr, g, red2[rb]), Kf);
        rb ^= 1;
        float sq = 0.0f;
#pragma unroll
        for (int i = 0; i < kVPT; ++i) {
            const int j = t + i * tpr;
            if (j < K4) {
                v[i] = make_float4(v[i].x - mean, v[i].y - mean, v[i].z - mean, v[i].w - mean);
                sq += (v[i].x * v[i].x + v[i].y * v[i].y) + (v[i].z * v[i].z + v[i].w * v[i].w);
            }
        }
        const float var = __fdiv_rn(row_group_reduce<2>(sq, tpr, g, red2[rb]), Kf);
        rb ^= 1;
        const float rstd = __frsqrt_rn(__fadd_rn(var, eps));
        // y = LayerNorm(h) (kept in v), and for Smooth-Dynamic the row maximum of
        // |fl(y / s)| by the corrected reciprocal division on f32x2 pairs
        float m = 0.0f;
#pragma unroll
        for (int i = 0; i < kVPT; ++i) {
            const int j = t + i * tpr;
            if (j >= K4) continue;
            const float4 gv = __ldg(g4 + j), bv = __ldg(b4 + j);
            float4 y;
            y.x = __fmaf_rn(__fmul_rn(v[i].x, rstd), gv.x, bv.x);
            y.y = __fmaf_rn(__fmul_rn(v[i].y, rstd), gv.y, bv.y);
            y.z = __fmaf_rn(__fmul_rn(v[i].z, rstd), gv.z, bv.z);
            y.w = __fmaf_rn(__fmul_rn(v[i].w, rstd), gv.w, bv.w);
            if (Y && valid) reinterpret_cast<float4 *>(Y)[row * K4 + j] = y;
            v[i] = y;
            if (KIND == kActDynamic) {
                const float4 ys = ytab[j], ns = nstab[j];
                const unsigned long long x01 = pk(y.x, y.y), x23 = pk(y.z, y.w);
                const unsigned long long y01 = pk(ys.x, ys.y), y23 = pk(ys.z, ys.w);
                const unsigned long long q01 = mul2(x01, y01), q23 = mul2(x23, y23);
                float d0, d1, d2, d3;
                upk(fma2(fma2(q01, pk(ns.x, ns.y), x01), y01, q01), d0, d1);
                upk(fma2(fma2(q23, pk(ns.z, ns.w), x23), y23, q23), d2, d3);
                m = max3_nan(m, max2_nan(fabsf(d0), fabsf(d1)), max2_nan(fabsf(d2), fabsf(d3)));
            }
        }
        bool exact;
        if (KIND == kActDynamic) {
            m = row_group_reduce<0>(m, tpr, g, red2[rb]);
            rb ^= 1;
            exact = !(m >= 0x1p-60f && m <= 0x1p100f);
        } else {
            exact = !fast;
        }
        float a1 = 0.0f;
        if (exact) {
            // IEEE divisions: v = fl(y / s), then the codes as the definition states
            float me = 0.0f;
#pragma unroll
            for (int i = 0; i < kVPT; ++i) {
                const int j = t + i * tpr;
                if (j >= K4) continue;
                const float4 sv = __ldg(s4 + j);
                v[i] = make_float4(__fdiv_rn(v[i].x, sv.x), __fdiv_rn(v[i].y, sv.y),
                                   __fdiv_rn(v[i].z, sv.z), __fdiv_rn(v[i].w, sv.w));
                if (KIND == kActDynamic)
                    me = fmaxf(me, fmaxf(fmaxf(fabsf(v[i].x), fabsf(v[i].y)),
                                         fmaxf(fabsf(v[i].z), fabsf(v[i].w))));
            }
            float sc = fixed_scale;
            if (KIND == kActDynamic) {
                me = row_group_reduce<1>(me, tpr, g, red2[rb]);
                rb ^= 1;
                sc = me == 0.0f ? 1.0f : __fdiv_rn(me, 127.0f);
            }
            const float rsc = __frcp_rn(sc);
            if (valid) {
                if (t == 0) scale[row] = sc;
#pragma unroll
                for (int i = 0; i < kVPT; ++i) {
                    const int j = t + i * tpr;
                    if (j < K4) a1 += store_codes<KIND>(v[i], sc, rsc, row * K4 + j, q, op);
                }
            }
        } else {
            // p = RN(RN(y RN(1/s)) RN(1/scale)), rint where p is 2^-14 clear of a
            // half-integer (NaN kept: a column without a reciprocal), else the
            // IEEE divisions; Smooth-Static codes saturate at +-127
            const float sc = KIND == kActDynamic ? __fdiv_rn(m, 127.0f) : fixed_scale;
            const float rsc = __frcp_rn(sc);
            const unsigned long long r2 = pk(rsc, rsc);
            if (valid) {
                if (t == 0) scale[row] = sc;
#pragma unroll
                for (int i = 0; i < kVPT; ++i) {
                    const int j = t + i * tpr;
                    if (j >= K4) continue;
                    const float4 ys = ytab[j];
                    const unsigned long long p01 = mul2(mul2(pk(v[i].x, v[i].y), pk(ys.x, ys.y)), r2);
                    const unsigned long long p23 = mul2(mul2(pk(v[i].z, v[i].w), pk(ys.z, ys.w)), r2);
                    const unsigned long long t01 = sub2(add2(p01, magic2), magic2);
                    const unsigned long long t23 = sub2(add2(p23, magic2), magic2);
                    float c[4], d[4];
                    upk(t01, c[0], c[1]);
                    upk(t23, c[2], c[3]);
                    upk(sub2(p01, t01), d[0], d[1]);
                    upk(sub2(p23, t23), d[2], d[3]);
                    const float dm = max3_nan(fabsf(d[0]), fabsf(d[1]),
                                              max2_nan(fabsf(d[2]), fabsf(d[3])));
                    if (!(dm <= kTieLimit)) {
                        const float4 ns = nstab[j];
                        if (!(fabsf(d[0]) <= kTieLimit)) c[0] = exact_code(v[i].x, -ns.x, sc);
                        if (!(fabsf(d[1]) <= kTieLimit)) c[1] = exact_code(v[i].y, -ns.y, sc);
                        if (!(fabsf(d[2]) <= kTieLimit)) c[2] = exact_code(v[i].z, -ns.z, sc);
                        if (!(fabsf(d[3]) <= kTieLimit)) c[3] = exact_code(v[i].w, -ns.w, sc);
                    }
                    if (KIND == kActStatic) {
#pragma unroll
                        for (int e = 0; e < 4; ++e) c[e] = fminf(127.0f, fmaxf(-127.0f, c[e]));
                    }
                    store4_codes(c[0], c[1], c[2], c[3], ((int64_t)row * K4 + j) * 4, q, op);
                    a1 += (fabsf(c[0]) + fabsf(c[1])) + (fabsf(c[2]) + fabsf(c[3]));
                }
            }
        }
        if (l1) {
            a1 = row_group_reduce<2>(a1, tpr, g, red2[rb]);  // exact: <= 127 * 8192 < 2^24
            rb ^= 1;
            if (valid && t == 0) l1[row] = (int32_t)a1;
        }
    }
}

// The exact path for one row (rare): IEEE divisions throughout, the codes as
// the definition states them.  Every warp of the group runs it together.
__device__ __noinline__ bool dynamic_row_exact(const float *__restrict__ xr,
                                               const float *__restrict__ s, int F4, int f0,
                                               int stride4, int vpt4, RingGroup &G, int64_t row,
                                               int64_t K, int8_t *q, float *scale,
                                               __nv_bfloat16 *op, int32_t *l1) {
    float m = 0.0f;
    for (int i = 0; i < vpt4; ++i) {
        const int f = f0 + i * stride4;
        if (f >= F4) break;
        for (int e = 0; e < 4; ++e)
            m = fmaxf(m, fabsf(__fdiv_rn(xr[4 * f + e], __ldg(s + 4 * f + e))));
    }
    if (!group_reduce<false>(m, G)) return false;
    const float sc = m == 0.0f ? 1.0f : __fdiv_rn(m, 127.0f);
    if (G.wg == 0 && G.lane == 0) scale[row] = sc;
    float a1 = 0.0f;
    for (int i = 0; i < vpt4; ++i) {
        const int f = f0 + i * stride4;
        if (f >= F4) break;
        float t[4];
        for (int e = 0; e < 4; ++e) {
            const float v = __fdiv_rn(xr[4 * f + e], __ldg(s + 4 * f + e));
            t[e] = fminf(127.0f, fmaxf(-127.0f, rintf(__fdiv_rn(v, sc))));
            a1 += fabsf(t[e]);
        }
        store4_codes(t[0], t[1], t[2], t[3], row * K + 4 * f, q, op);
    }
    if (l1) {
        if (!group_reduce<true>(a1, G)) return false;
        if (G.wg == 0 && G.lane == 0) l1[row] = (int32_t)a1;
    }
    return true;
}

// GIVEN: the row maxima come from row_amax (max_j |fl(x / s)|, as the GEMM's
// row-maximum epilogue merges them), so no reduction runs before the codes; a
// wrong maximum only makes the codes saturate at +-127.
template <int VPT4, bool GIVEN>
__global__ void __launch_bounds__(32 * (kRingWarps + 1), 1) quantize_act_ring(
    const float *__restrict__ X, const float *__restrict__ s, int64_t rows, int K, int wpr,
    int groups, int stages, int8_t *__restrict__ q, float *__restrict__ scale,
    __nv_bfloat16 *__restrict__ op, int32_t *__restrict__ l1,
    const float *__restrict__ row_amax) {
    extern __shared__ __align__(128) unsigned char ring_smem[];
    const int64_t stage_floats = (int64_t)groups * K;
    float *ring = reinterpret_cast<float *>(ring_smem);
    float *ytab = ring + stages * stage_floats;  // K reciprocals of s
    float *nstab = ytab + K;                     // K negated smoothing factors
    uint64_t *full = reinterpret_cast<uint64_t *>(nstab + K);
    uint64_t *empty = full + stages;
    uint64_t *gbar = empty + stages;                        // [kRingWarps]
    float *red = reinterpret_cast<float *>(gbar + kRingWarps);  // [kRingWarps][2][8]
    int *abort_flag = reinterpret_cast<int *>(red + kRingWarps * 16);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nconsumer = groups * wpr;  // warps 0 .. nconsumer-1; the producer is the last
    if (threadIdx.x == 0) {
        for (int i = 0; i < stages; ++i) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(saddr(&full[i])));
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(saddr(&empty[i])),
                         "r"(nconsumer));
        }
        for (int g = 0; g < groups; ++g)
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(saddr(&gbar[g])), "r"(wpr));
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    pdl_launch_dependents();
    pdl_wait();  // every global-memory access below follows the previous kernel
    for (int j = threadIdx.x; j < K; j += blockDim.x) {
        const float sj = __ldg(s + j);
        const float a = fabsf(sj);
        ytab[j] = (a >= 0x1p-20f && a <= 0x1p20f) ? __frcp_rn(sj) : __int_as_float(0x7fffffff);
        nstab[j] = -sj;
    }
    __syncthreads();
    volatile int *abort = abort_flag;
    const int64_t nst = (rows + groups - 1) / groups;  // stages of `groups` rows
    if (warp == nconsumer) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int slot = 0;
            uint32_t ph = 0, issued = 0, fill_par = 0;  // per slot: a copy issued, its phase
            for (int64_t t = blockIdx.x; t < nst; t += gridDim.x) {
                if (!mb_wait(saddr(&empty[slot]), ph ^ 1u, abort)) break;
                const int64_t r0 = t * groups;
                const int64_t nr = rows - r0 < groups ? rows - r0 : groups;
                const uint32_t bytes = (uint32_t)(nr * K * 4);
                const uint32_t fb = saddr(&full[slot]);
                asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(fb),
                             "r"(bytes)
                             : "memory");
                asm volatile(
                    "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], "
                    "%2, [%3];" ::"r"(saddr(ring + slot * stage_floats)),
                    "l"(X + r0 * K), "r"(bytes), "r"(fb)
                    : "memory");
                issued |= 1u << slot;
                fill_par = (fill_par & ~(1u << slot)) | (ph << slot);
                if (++slot == stages) {
                    slot = 0;
                    ph ^= 1u;
                }
            }
            // every issued copy lands before the block's shared memory goes away
            for (int i = 0; i < stages; ++i)
                if (issued & (1u << i)) mb_drain(saddr(&full[i]), (fill_par >> i) & 1u);
        }
        return;
    }
    // ---------------------------------------------------------------- consumers
    RingGroup G;
    G.wpr = wpr;
    G.g = warp / wpr;
    G.wg = warp - G.g * wpr;
    G.lane = lane;
    G.bar = saddr(&gbar[G.g]);
    G.bph = 0;
    G.red = red + 16 * G.g;
    G.rp = 0;
    G.abort = abort;
    const int F4 = K >> 2;
    const int stride4 = 32 * wpr;
    const int f0 = 32 * G.wg + lane;
    const float4 *y4 = reinterpret_cast<const float4 *>(ytab);
    const unsigned long long magic2 = pk(kRoundMagic, kRoundMagic);
    int slot = 0;
    uint32_t ph = 0;
    for (int64_t t = blockIdx.x; t < nst; t += gridDim.x) {
        int ok = 1;
        if (lane == 0) ok = mb_wait(saddr(&full[slot]), ph, abort);
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
        const int64_t row = t * groups + G.g;
        bool alive = true;
        if (row < rows) {
            const float4 *xs = reinterpret_cast<const float4 *>(ring + slot * stage_floats +
                                                                (int64_t)G.g * K);
            float x[VPT4][4];
#pragma unroll
            for (int i = 0; i < VPT4; ++i) {
                const int f = f0 + i * stride4;
                const float4 v = f < F4 ? xs[f] : make_float4(0.f, 0.f, 0.f, 0.f);
                x[i][0] = v.x;
                x[i][1] = v.y;
                x[i][2] = v.z;
                x[i][3] = v.w;
            }
            float m;
            if (GIVEN) {
                m = __ldg(row_amax + row);
            } else {
                // the row maximum of |fl(x / s)|: the corrected reciprocal division
                // (div_smooth) on f32x2 pairs, the IEEE quotient for |s| in
                // [2^-20, 2^20], |x| >= 2^-100 and a first product of at most
                // 2^100.  Tinier x give tinier quotients, which decide nothing
                // unless the whole row is below 2^-60 (the exact path then).
                float lm = 0.0f;
                const float4 *ns4 = reinterpret_cast<const float4 *>(nstab);
#pragma unroll
                for (int i = 0; i < VPT4; ++i) {
                    const int f = f0 + i * stride4;
                    if (f < F4) {
                        const float4 y = y4[f], ns = ns4[f];
                        const unsigned long long x01 = pk(x[i][0], x[i][1]);
                        const unsigned long long x23 = pk(x[i][2], x[i][3]);
                        const unsigned long long y01 = pk(y.x, y.y), y23 = pk(y.z, y.w);
                        const unsigned long long q01 = mul2(x01, y01), q23 = mul2(x23, y23);
                        float v0, v1, v2, v3;
                        upk(fma2(fma2(q01, pk(ns.x, ns.y), x01), y01, q01), v0, v1);
                        upk(fma2(fma2(q23, pk(ns.z, ns.w), x23), y23, q23), v2, v3);
                        lm = max3_nan(lm, fabsf(v0), fabsf(v1));
                        lm = max3_nan(lm, fabsf(v2), fabsf(v3));
                    }
                }
                alive = group_reduce<false>(lm, G);
                m = lm;
            }
            if (alive && !(m >= 0x1p-60f && m <= 0x1p100f)) {
                alive = dynamic_row_exact(X + row * K, s, F4, f0, stride4, VPT4, G, row, K, q,
                                          scale, op, l1);
            } else if (alive) {
                const float sc = __fdiv_rn(m, 127.0f);
                const float rsc = __frcp_rn(sc);
                if (G.wg == 0 && lane == 0) scale[row] = sc;
                const unsigned long long r2 = pk(rsc, rsc);
                float a1 = 0.0f;
#pragma unroll
                for (int i = 0; i < VPT4; ++i) {
                    const int f = f0 + i * stride4;
                    if (f >= F4) continue;
                    const float4 y = y4[f];
                    const unsigned long long p01 = mul2(mul2(pk(x[i][0], x[i][1]), pk(y.x, y.y)), r2);
                    const unsigned long long p23 = mul2(mul2(pk(x[i][2], x[i][3]), pk(y.z, y.w)), r2);
                    const unsigned long long t01 = sub2(add2(p01, magic2), magic2);
                    const unsigned long long t23 = sub2(add2(p23, magic2), magic2);
                    float t[4], d[4];
                    upk(t01, t[0], t[1]);
                    upk(t23, t[2], t[3]);
                    upk(sub2(p01, t01), d[0], d[1]);
                    upk(sub2(p23, t23), d[2], d[3]);
                    // NaN kept: with the maxima given, a column whose s has no
                    // reciprocal (NaN in the table) reaches this point
                    const float dm = max3_nan(fabsf(d[0]), fabsf(d[1]),
                                              max2_nan(fabsf(d[2]), fabsf(d[3])));
                    if (!(dm <= kTieLimit)) {
                        // rare: a value within 2^-14 of a half-integer (or NaN)
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            if (!(fabsf(d[e]) <= kTieLimit))
                                t[e] = exact_code(x[i][e], -nstab[4 * f + e], sc);
                    }
                    if (GIVEN) {
                        // a maximum below the row's true one: saturate
#pragma unroll
                        for (int e = 0; e < 4; ++e) t[e] = fminf(127.0f, fmaxf(-127.0f, t[e]));
                    }
                    store4_codes(t[0], t[1], t[2], t[3], row * K + 4 * f, q, op);
                    if (l1) a1 += (fabsf(t[0]) + fabsf(t[1])) + (fabsf(t[2]) + fabsf(t[3]));
                }
                if (l1) {
                    alive = group_reduce<true>(a1, G);  // exact: at most 127 * 8192 < 2^24
                    if (alive && G.wg == 0 && lane == 0) l1[row] = (int32_t)a1;
                }
            }
        }
        // this warp is done with the stage (its group's reads are its own)
        __syncwarp();
        if (lane == 0)
            asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(saddr(&empty[slot]))
                         : "memory");
        if (!alive) break;
        if (++slot == stages) {
            slot = 0;
            ph ^= 1u;
        }
    }
}

}  // namespace

// Smooth-Dynamic activations of up to 8192 elements per row: the ring kernel
// above.  wpr warps per row (a warp covers 1024 elements), VPT4 float4 per lane,
// `groups` rows per stage (16 / wpr, fewer when the rows would not give every
// SM a stage), as many stages of up to 64 KB as the shared memory holds.
sq_status launch_quantize_act_dynamic(const float *A, const float *s, int64_t rows, int64_t K,
                                      int8_t *q, float *scale, __nv_bfloat16 *op, int32_t *l1,
                                      const DeviceInfo &di, cudaStream_t st,
                                      const float *row_amax) {
    const int wpr = (int)((K + 1023) / 1024);
    const int F4 = (int)(K / 4);
    const int need4 = (F4 + 32 * wpr - 1) / (32 * wpr);  // float4 per lane, 1..8
    const int vpt4 = need4 <= 1 ? 1 : need4 <= 2 ? 2 : need4 <= 4 ? 4 : need4 <= 6 ? 6 : 8;
    int groups = kRingWarps / wpr;
    const int64_t per_sm = (rows + di.sms - 1) / di.sms;
    if (per_sm < groups) groups = (int)std::max<int64_t>(1, per_sm);
    const size_t stage_bytes = (size_t)groups * K * 4;
    const size_t fixed = (size_t)K * 8 + (size_t)kRingWarps * 8 + kRingWarps * 16 * 4 + 16 + 256;
    const size_t budget = di.smem_optin > 0 ? di.smem_optin : 227 * 1024;
    int stages = (int)std::min<size_t>(6, (budget - fixed - 2 * 6 * 8) / stage_bytes);
    if (stages < 2) return SQ_ERR_UNSUPPORTED;
    const size_t smem = stages * stage_bytes + (size_t)K * 8 + 2 * stages * 8 +
                        (size_t)kRingWarps * 8 + kRingWarps * 16 * 4 + 16;
    using Kern = void (*)(const float *, const float *, int64_t, int, int, int, int, int8_t *,
                          float *, __nv_bfloat16 *, int32_t *, const float *);
    static const Kern kerns[2][5] = {
        {quantize_act_ring<1, false>, quantize_act_ring<2, false>, quantize_act_ring<4, false>,
         quantize_act_ring<6, false>, quantize_act_ring<8, false>},
        {quantize_act_ring<1, true>, quantize_act_ring<2, true>, quantize_act_ring<4, true>,
         quantize_act_ring<6, true>, quantize_act_ring<8, true>}};
    const int vi = vpt4 == 1 ? 0 : vpt4 == 2 ? 1 : vpt4 == 4 ? 2 : vpt4 == 6 ? 3 : 4;
    const int given = row_amax ? 1 : 0;
    const Kern kern = kerns[given][vi];
    // the shared-memory opt-in, once per (device, kernel)
    static std::mutex mu;
    static bool attr_set[64][2][5] = {};
    {
        std::lock_guard<std::mutex> lock(mu);
        bool &done = attr_set[di.device & 63][given][vi];
        if (!done) {
            if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)budget) != cudaSuccess)
                return SQ_ERR_CUDA;
            done = true;
        }
    }
    const int64_t nst = (rows + groups - 1) / groups;
    const int64_t grid = std::min<int64_t>(nst, (int64_t)di.sms);
    const int threads = 32 * (groups * wpr + 1);
    return launch_pdl(kern, dim3((unsigned)grid), dim3(threads), smem, st, 1, A, s, rows, (int)K,
                      wpr, groups, stages, q, scale, op, l1, row_amax);
}

// int8 codes -> the bf16 GEMM operand, 16 codes per thread per pass (one
// 16-byte load, two 16-byte stores); every |q| <= 127 is exact in bf16, whose
// bit pattern is the high half of the fp32 value.
__global__ void __launch_bounds__(kThreads) widen_codes_kernel(const uint4 *__restrict__ q,
                                                             uint4 *__restrict__ op, int64_t n16) {
    pdl_launch_dependents();
    pdl_wait();
    for (int64_t i = blockIdx.x * (int64_t)kThreads + threadIdx.x; i < n16;
         i += (int64_t)gridDim.x * kThreads) {
        const uint4 c = __ldcs(q + i);
        const uint32_t w[4] = {c.x, c.y, c.z, c.w};
        uint32_t o[8];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t b0 = __float_as_uint((float)(int8_t)(w[k] & 0xff));
            const uint32_t b1 = __float_as_uint((float)(int8_t)((w[k] >> 8) & 0xff));
            const uint32_t b2 = __float_as_uint((float)(int8_t)((w[k] >> 16) & 0xff));
            const uint32_t b3 = __float_as_uint((float)(int8_t)(w[k] >> 24));
            o[2 * k] = __byte_perm(b0, b1, 0x7632);
            o[2 * k + 1] = __byte_perm(b2, b3, 0x7632);
        }
        op[2 * i] = make_uint4(o[0], o[1], o[2], o[3]);
        op[2 * i + 1] = make_uint4(o[4], o[5], o[6], o[7]);
    }
}

sq_status launch_widen_codes(const int8_t *q, __nv_bfloat16 *op, int64_t count, cudaStream_t st) {
    DeviceInfo di;
    sq_status rc = device_info(&di);
    if (rc != SQ_OK) return rc;
    const int64_t n16 = count / 16;
    if (n16 == 0) return SQ_OK;
    // one 16-byte group of codes per thread, the block scheduler filling the SMs
    // (measured on GB300 in the BERT-large step with int8 inputs: 700 -> 710
    // TOPS against a grid-stride loop over one wave of resident blocks)
    const int64_t grid = (n16 + kThreads - 1) / kThreads;
    if (grid > 0x7fffffff) return SQ_ERR_UNSUPPORTED;
    return launch_pdl(widen_codes_kernel, dim3((unsigned)grid), dim3(kThreads), 0, st, 1,
                      reinterpret_cast<const uint4 *>(q), reinterpret_cast<uint4 *>(op), n16);
}

sq_status quant_take_error(cudaStream_t st) {
    unsigned int word = 0;
    if (cudaMemcpyFromSymbolAsync(&word, g_quant_error, sizeof(word), 0, cudaMemcpyDeviceToHost,
                                  st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return SQ_ERR_CUDA;
    if (word != 0) {
        const unsigned int zero = 0;
        if (cudaMemcpyToSymbolAsync(g_quant_error, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice,
                                    st) != cudaSuccess ||
            cudaStreamSynchronize(st) != cudaSuccess)
            return SQ_ERR_CUDA;
        return SQ_ERR_TIMEOUT;
    }
    return SQ_OK;
}

// Division table of a smoothing factor: (-s[j], RN(1/s[j])) per column, NaN for
// the reciprocal where |s[j]| is outside [2^-20, 2^20].
__global__ void division_table_kernel(const float *__restrict__ s, int64_t K,
                                      float2 *__restrict__ table) {
    pdl_launch_dependents();
    pdl_wait();
    const int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (j >= K) return;
    const float sj = s[j];
    const float a = fabsf(sj);
    table[j] = make_float2(-sj, (a >= 0x1p-20f && a <= 0x1p20f) ? __frcp_rn(sj)
                                                                 : __int_as_float(0x7fffffff));
}

sq_status launch_division_table(const float *s, int64_t K, float *table, cudaStream_t st) {
    const int64_t grid = (K + kThreads - 1) / kThreads;
    return launch_pdl(division_table_kernel, dim3((unsigned)grid), dim3(kThreads), 0, st, 1, s, K,
                      reinterpret_cast<float2 *>(table));
}

// The register Smooth-Dynamic kernel (K <= 8192): its tables of -s and 1/s in
// shared memory (8 bytes per column; formed from s, or copied from s's
// division table when one is given), its residency at that size, and the grid.
// mode: kRegDynamic, kRegGiven (row_amax) or kRegStatic (fixed_scale).
sq_status launch_act_reg(int mode, const float *A, const float *s, const float *tab,
                         int64_t rows, int64_t K, int8_t *q, float *scale, __nv_bfloat16 *op,
                         int32_t *l1, const float *row_amax, float fixed_scale,
                         const DeviceInfo &di, cudaStream_t st) {
    const int K4 = (int)(K / 4);
    const bool small = K4 <= kThreads * 4;
    const int vpt = small ? 4 : 8;
    int tpr = 32;
    while (tpr * vpt < K4) tpr <<= 1;
    const int rpb = kThreads / tpr;
    const int64_t tiles = (rows + rpb - 1) / rpb;
    using Kern = void (*)(const float *, const float *, const float4 *, int64_t, int, int,
                          int8_t *, float *, __nv_bfloat16 *, int32_t *, const float *, float);
    static const Kern kerns[2][3][2] = {
        {{quantize_act_reg<4, kRegDynamic, false>, quantize_act_reg<8, kRegDynamic, false>},
         {quantize_act_reg<4, kRegGiven, false>, quantize_act_reg<8, kRegGiven, false>},
         {quantize_act_reg<4, kRegStatic, false>, quantize_act_reg<8, kRegStatic, false>}},
        {{quantize_act_reg<4, kRegDynamic, true>, quantize_act_reg<8, kRegDynamic, true>},
         {quantize_act_reg<4, kRegGiven, true>, quantize_act_reg<8, kRegGiven, true>},
         {quantize_act_reg<4, kRegStatic, true>, quantize_act_reg<8, kRegStatic, true>}}};
    const int ti = tab ? 1 : 0, gi = mode, vi = small ? 0 : 1;
    const Kern kern = kerns[ti][gi][vi];
    const int smem = K4 * 32;
    constexpr int kMaxTab = kThreads * kMaxVPT * 32;  // 64 KB at K = 8192
    static std::mutex mu;
    static bool opted[64][2][3][2] = {};
    static int occ_dyn[64][2][3][2][8] = {};  // per device, table, mode, vpt, 256-float4 bucket
    int occ = 0;
    {
        std::lock_guard<std::mutex> lock(mu);
        const int dv = di.device & 63;
        if (!opted[dv][ti][gi][vi]) {
            if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kMaxTab) != cudaSuccess)
                return SQ_ERR_CUDA;
            opted[dv][ti][gi][vi] = true;
        }
        // residency at the bucket's largest table (never above the true one)
        const int bucket = (K4 - 1) / 256;
        int &o = occ_dyn[dv][ti][gi][vi][bucket];
        if (!o && (cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                       &o, kern, kThreads, (bucket + 1) * 256 * 32) != cudaSuccess ||
                   o < 1))
            return SQ_ERR_CUDA;
        occ = o;
    }
    // twice the blocks that fit at once: measured on GB300 in the BERT-large
    // step (each quantiser between two GEMMs, launched with programmatic
    // dependent launch) 756 -> 782-788 TOPS against one resident wave, while
    // 1.5, 2.5, 3, 4 times or one tile per block ran slower (761, 765, 763,
    // 754, 698 TOPS); a launch timed on its own runs a little slower
    const int64_t grid = std::min<int64_t>(tiles, 2 * (int64_t)di.sms * occ);
    return launch_pdl(kern, dim3((unsigned)grid), dim3(kThreads), smem, st, 1, A, s,
                      reinterpret_cast<const float4 *>(tab), rows, K4, tpr, q, scale, op, l1,
                      row_amax, fixed_scale);
}

sq_status launch_quantize_act_given_max(const float *A, const float *s, const float *row_amax,
                                        int64_t rows, int64_t K, int8_t *q, float *scale,
                                        __nv_bfloat16 *op, int32_t *l1, cudaStream_t st) {
    DeviceInfo di;
    sq_status rc = device_info(&di);
    if (rc != SQ_OK) return rc;
    // the register kernel on the given maxima (measured on GB300 at 8192 x 4096:
    // faster than the ring kernel's given-maximum mode, which the shorter rows
    // that are not 1024 * 2^k keep, as in the dynamic dispatch)
    const bool pow2_rows = K >= 1024 && K <= 8192 && (K & (K - 1)) == 0;
    if (K <= 8192 && (pow2_rows || K > 2048))
        return launch_act_reg(kRegGiven, A, s, nullptr, rows, K, q, scale, op, l1, row_amax,
                              0.0f, di, st);
    if (K <= 8192 && rows >= 16 * (int64_t)di.sms)
        return launch_quantize_act_dynamic(A, s, rows, K, q, scale, op, l1, di, st, row_amax);
    // other launches: the full quantiser (it finds the same maxima itself)
    return launch_quantize_rows(kActDynamic, A, s, rows, K, q, scale, op, l1, 0.0f, st);
}

sq_status launch_quantize_act_table(const float *A, const float *s, const float *table,
                                    const float *row_amax, int64_t rows, int64_t K, int8_t *q,
                                    float *scale, __nv_bfloat16 *op, int32_t *l1,
                                    cudaStream_t st) {
    DeviceInfo di;
    sq_status rc = device_info(&di);
    if (rc != SQ_OK) return rc;
    // the register kernel reads the table wherever the dispatch below (and in
    // the given-maximum quantiser) would take it; the other kernels take s
    const bool pow2_rows = K >= 1024 && K <= 8192 && (K & (K - 1)) == 0;
    const bool reg = K <= 8192 && (row_amax ? (pow2_rows || K > 2048)
                                            : !(K <= 2048 && !pow2_rows &&
                                                rows >= 16 * (int64_t)di.sms));
    if (reg)
        return launch_act_reg(row_amax ? kRegGiven : kRegDynamic, A, s, table, rows, K, q, scale,
                              op, l1, row_amax, 0.0f, di, st);
    if (row_amax)
        return launch_quantize_act_given_max(A, s, row_amax, rows, K, q, scale, op, l1, st);
    return launch_quantize_rows(kActDynamic, A, s, rows, K, q, scale, op, l1, 0.0f, st);
}

sq_status launch_quantize_rows(int direction, const float *A, const float *s, int64_t rows,
                               int64_t K, int8_t *q, float *scale, __nv_bfloat16 *op,
                               int32_t *l1, float fixed_scale, cudaStream_t st) {
    DeviceInfo di;
    sq_status rc = device_info(&di);
    if (rc != SQ_OK) return rc;
    // Smooth-Dynamic activations: the register kernel (quantize_act_reg) for
    // rows of 1024 * 2^k elements, which fill its thread groups exactly, and
    // for rows above 2048 elements (measured on GB300, L2 flushed: 21 us at
    // 8192 x 1024, 52 us at 8192 x 4096, 152 us against the ring's 183 us at
    // 32768 x 3072); the ring kernel for the other rows up to 2048 elements
    // (44 against 46 us at 32768 x 768), and only with at least 16 rows per SM:
    // below that the ring's stages stay short and its set-up dominates
    const bool pow2_rows = K >= 1024 && K <= 8192 && (K & (K - 1)) == 0;
    if (direction == kActDynamic && K <= 2048 && !pow2_rows && rows >= 16 * (int64_t)di.sms)
        return launch_quantize_act_dynamic(A, s, rows, K, q, scale, op, l1, di, st, nullptr);
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
            return launch_act_reg(kRegDynamic, A, s, nullptr, rows, K, q, scale, op, l1, nullptr,
                                  0.0f, di, st);
        // Smooth-Static: the register kernel's static mode (f32x2 codes from the
        // division tables) for scales where its shortcut is proven
        if (direction == kActStatic && fixed_scale >= 0x1p-60f && fixed_scale <= 0x1p60f)
            return launch_act_reg(kRegStatic, A, s, nullptr, rows, K, q, scale, op, l1, nullptr,
                                  fixed_scale, di, st);
        if (direction == kWeight)
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
                          int32_t *, float, int);
    static const Kern kerns[2][2] = {
        {layernorm_quant_kernel<kActDynamic, 4>, layernorm_quant_kernel<kActDynamic, 8>},
        {layernorm_quant_kernel<kActStatic, 4>, layernorm_quant_kernel<kActStatic, 8>}};
    const int ki = static_scale > 0.0f ? 1 : 0, vi = small ? 0 : 1;
    const Kern kern = kerns[ki][vi];
    // the static shortcut's proven range of scales (as in launch_act_reg's static mode)
    const int fast = static_scale >= 0x1p-60f && static_scale <= 0x1p60f;
    const int smem = K4 * 32;
    constexpr int kMaxTab = kThreads * kMaxVPT * 32;  // 64 KB at K = 8192
    static std::mutex mu;
    static bool opted[64][2][2] = {};
    static int occ_dyn[64][2][2][8] = {};  // per device, kind, vpt, 256-float4 bucket of K4
    int occ = 0;
    {
        std::lock_guard<std::mutex> lock(mu);
        const int dv = di.device & 63;
        if (!opted[dv][ki][vi]) {
            if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kMaxTab) != cudaSuccess)
                return SQ_ERR_CUDA;
            opted[dv][ki][vi] = true;
        }
        const int bucket = (K4 - 1) / 256;
        int &o = occ_dyn[dv][ki][vi][bucket];
        if (!o && (cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                       &o, kern, kThreads, (bucket + 1) * 256 * 32) != cudaSuccess ||
                   o < 1))
            return SQ_ERR_CUDA;
        occ = o;
    }
    // twice the blocks that fit at once, as for the register quantiser (measured
    // on GB300, BERT-large step with LayerNorm inputs: 757 -> 765 TOPS)
    const int64_t grid = std::min<int64_t>(tiles, 2 * (int64_t)di.sms * occ);
    return launch_pdl(kern, dim3((unsigned)grid), dim3(kThreads), smem, st, 1, H, gamma, beta,
                      eps, s, rows, K4, tpr, Y, q, scale, op, l1, static_scale, fast);
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

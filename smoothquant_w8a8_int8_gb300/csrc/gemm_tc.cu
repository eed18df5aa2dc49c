// INT8 GEMM + fused dequantising epilogue on the 5th-generation tensor cores
// (tcgen05, sm_103a): TMA-fed shared-memory ring, accumulators in tensor
// memory, warp-specialised persistent CTAs.
//
// "Efficient INT8 Inference of Small NLP Models on Server CPUs with PyTorch
// Native Stack": the linear block is the int8 x int8 -> int32 GEMM plus its
// fused post-operations -- bias, activation, residual addition (Table 3
// caption) -- with per-token x per-output-channel dequantisation.
//
// Exact integer arithmetic on this chip.  The sm_103a tensor cores take no
// int8 operand kind, so the int8 codes arrive as bf16 numbers of the same
// integer value (exact: |q| <= 127 needs 7 of bf16's 8 significand bits).
// Every product |q_x q_w| <= 16129 < 2^14 is exact, and an fp32 accumulator
// adds integers exactly while every partial sum stays below 2^24 in
// magnitude.  K is therefore cut into chunks of at most 1024
// (1024 * 16129 = 16,516,096 < 2^24); each chunk is summed in fp32 in tensor
// memory, converted to int32 (exact) by the epilogue warps and added in
// int32.  The result equals the int32 dot product for every input.
//
// Roles (320 threads, one CTA per SM, persistent over 128 x 256 output tiles):
//   warp 0, lane 0  TMA producer: A [128 x 64] and B [256 x 64] bf16 tiles,
//                   128-byte swizzle, into a 4-stage ring (48 KB per stage)
//   warp 1, lane 0  MMA issuer: tcgen05.mma kind::f16, M=128 N=256 K=16,
//                   one chunk into one of two 256-column TMEM accumulators
//   warps 2..9      epilogue: warp w reads TMEM lanes 32*(w%4).. (its rows)
//                   and columns 128*((w-2)/4).. (its half), int32 partials in
//                   registers, then scales, bias, GELU / residual, stores.
// Every wait is bounded (about 4 s of %globaltimer); on expiry the kernel
// records SQ_ERR_TIMEOUT in a device word, lets its issued copies and MMAs
// drain, frees its tensor memory and returns.
#include "common.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

namespace sq {
namespace {

constexpr int BM = 128, BN = 256, BK = 64;  // BK in bf16 elements (128 bytes)
constexpr int STAGES = 4;
constexpr int KB_PER_CHUNK = 16;            // 16 * 64 = 1024 K per exact fp32 chunk
constexpr int UMMA_K = 16;
constexpr int NUM_EPI_WARPS = 8;
constexpr int THREADS = 64 + NUM_EPI_WARPS * 32;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int TMEM_COLS = 2 * BN;           // two accumulators
constexpr int BAR_BYTES = 256;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + BAR_BYTES;
constexpr unsigned long long kTimeoutNs = 4000000000ull;

// instruction descriptor, kind::f16: D fp32, A/B bf16, both K-major, N, M
constexpr uint32_t IDESC = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) |
                           ((uint32_t)(BM >> 4) << 24);

__device__ unsigned int g_tc_error;

// ---------------------------------------------------------------- PTX glue

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Slow path of mbar_wait: poll with a time limit.
__device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity,
                                            volatile int *abort_flag) {
    const uint64_t t0 = globaltimer();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 0) {
            if (*abort_flag) return false;
            if (globaltimer() - t0 > kTimeoutNs) {
                *abort_flag = 1;
                atomicOr(&g_tc_error, 1u);
                return false;
            }
        }
    }
}

// Bounded wait for the phase of parity `parity` to complete.  Returns false
// when the CTA has aborted or the wait ran out (then it aborts the CTA).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          volatile int *abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    return mbar_wait_slow(bar, parity, abort_flag);
}

// Bounded wait used while draining after an abort (ignores the abort flag).
__device__ __noinline__ void mbar_drain(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer() - t0 > kTimeoutNs) {
            atomicOr(&g_tc_error, 2u);
            return;
        }
    }
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                            int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows of
// 128 bytes, 8-row swizzle atoms 1024 bytes apart (SBO); LBO unused here.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)1 << 16;             // LBO (ignored for swizzled K-major)
    d |= (uint64_t)(1024 >> 4) << 32;   // SBO
    d |= (uint64_t)1 << 46;             // descriptor version
    d |= (uint64_t)2 << 61;             // 128-byte swizzle
    return d;
}

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(IDESC), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread i gets lane (base + i).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
        "%28, %29, %30, %31}, [%32];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
          "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]),
          "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]),
          "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),
          "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]),
          "=r"(v[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ------------------------------------------------------------------ kernel

struct Smem {
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t mma_done;
    uint32_t tmem_base;
    int abort_flag;
};
static_assert(sizeof(Smem) <= BAR_BYTES, "barrier block");

__device__ __forceinline__ void store4(float *y, int64_t off, int64_t n, int64_t N, bool vec_ok,
                                       float a, float b, float c, float d) {
    if (vec_ok && n + 3 < N) {
        *reinterpret_cast<float4 *>(y + off) = make_float4(a, b, c, d);
    } else {
        if (n < N) y[off] = a;
        if (n + 1 < N) y[off + 1] = b;
        if (n + 2 < N) y[off + 2] = c;
        if (n + 3 < N) y[off + 3] = d;
    }
}

__global__ void __launch_bounds__(THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const float *__restrict__ sx, const float *__restrict__ sw,
                   const float *__restrict__ bias, const float *residual, int M, int N, int K,
                   int mode, int vec_ok, void *Y) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    Smem &S = *reinterpret_cast<Smem *>(smem + STAGES * STAGE_BYTES);
    const uint32_t ring = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_u32(&S.full[s]), 1);
            mbar_init(smem_u32(&S.empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&S.tfull[b]), 1);
            mbar_init(smem_u32(&S.tempty[b]), NUM_EPI_WARPS);
        }
        mbar_init(smem_u32(&S.mma_done), 1);
        S.abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&S.tmem_base)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = S.tmem_base;
    volatile int *abort_flag = &S.abort_flag;

    const int m_tiles = (M + BM - 1) / BM;
    const int n_tiles = (N + BN - 1) / BN;
    const int num_tiles = m_tiles * n_tiles;
    const int nkb = (K + BK - 1) / BK;
    const int nchunks = (nkb + KB_PER_CHUNK - 1) / KB_PER_CHUNK;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued = 0, fill_parity = 0;  // per-stage bits: loads in flight
            for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
                const int m0 = (tile % m_tiles) * BM, n0 = (tile / m_tiles) * BN;
                for (int kb = 0; kb < nkb; ++kb) {
                    if (!mbar_wait(smem_u32(&S.empty[stage]), phase ^ 1, abort_flag)) goto done_p;
                    const uint32_t full = smem_u32(&S.full[stage]);
                    mbar_expect_tx(full, STAGE_BYTES);
                    const uint32_t sa = ring + stage * STAGE_BYTES;
                    tma_load_2d(sa, &tmA, full, kb * BK, m0);
                    tma_load_2d(sa + A_BYTES, &tmB, full, kb * BK, n0);
                    issued |= 1u << stage;
                    fill_parity = (fill_parity & ~(1u << stage)) | (phase << stage);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
        done_p:
            // let every issued copy land before the CTA's shared memory goes away
            for (int s = 0; s < STAGES; ++s)
                if (issued & (1u << s)) mbar_drain(smem_u32(&S.full[s]), (fill_parity >> s) & 1u);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------ MMA issuer
            int stage = 0;
            uint32_t phase = 0, item = 0;
            bool issued_any = false;
            for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
                for (int c = 0; c < nchunks; ++c, ++item) {
                    const uint32_t b = item & 1, use = (item >> 1) & 1;
                    if (!mbar_wait(smem_u32(&S.tempty[b]), use ^ 1, abort_flag)) goto done_m;
                    tc_fence_after();
                    const uint32_t d = tmem_base + b * BN;
                    const int kb0 = c * KB_PER_CHUNK;
                    const int kb1 = min(nkb, kb0 + KB_PER_CHUNK);
                    for (int kb = kb0; kb < kb1; ++kb) {
                        if (!mbar_wait(smem_u32(&S.full[stage]), phase, abort_flag)) goto done_m;
                        tc_fence_after();
                        const uint32_t sa = ring + stage * STAGE_BYTES;
                        const uint64_t adesc = sw128_desc(sa);
                        const uint64_t bdesc = sw128_desc(sa + A_BYTES);
#pragma unroll
                        for (int k = 0; k < BK / UMMA_K; ++k) {
                            // advance 16 bf16 = 32 bytes along K inside the swizzled row
                            umma_bf16(d, adesc + 2 * k, bdesc + 2 * k,
                                      (kb > kb0 || k > 0) ? 1u : 0u);
                        }
                        issued_any = true;
                        umma_commit(smem_u32(&S.empty[stage]));
                        if (++stage == STAGES) {
                            stage = 0;
                            phase ^= 1;
                        }
                    }
                    umma_commit(smem_u32(&S.tfull[b]));
                }
            }
        done_m:
            if (issued_any) {
                // all MMAs issued by this thread complete before TMEM is freed
                umma_commit(smem_u32(&S.mma_done));
                mbar_drain(smem_u32(&S.mma_done), 0);
            }
        }
    } else {
        // ---------------------------------------------------- epilogue
        const int q = warp & 3;              // TMEM lane quarter this warp may access
        const int half = (warp - 2) >> 2;    // which 128 of the 256 columns
        const int row_in_tile = q * 32 + lane;
        uint32_t item = 0;
        for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
            const int m0 = (tile % m_tiles) * BM, n0 = (tile / m_tiles) * BN;
            int32_t part[128];
            for (int c = 0; c < nchunks; ++c, ++item) {
                const uint32_t b = item & 1, use = (item >> 1) & 1;
                if (!mbar_wait(smem_u32(&S.tfull[b]), use, abort_flag)) goto done_e;
                tc_fence_after();
                const uint32_t taddr =
                    tmem_base + ((uint32_t)(q * 32) << 16) + b * BN + (uint32_t)(half * 128);
#pragma unroll
                for (int s = 0; s < 4; ++s) {
                    uint32_t v[32];
                    tmem_ld32(taddr + s * 32, v);
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        // an exact integer below 2^24 in magnitude
                        const int32_t a = __float2int_rn(__uint_as_float(v[i]));
                        part[s * 32 + i] = c == 0 ? a : part[s * 32 + i] + a;
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&S.tempty[b]));
            }
            const int64_t m = (int64_t)m0 + row_in_tile;
            if (m < M) {
                const int64_t nb = (int64_t)n0 + half * 128;
                const int64_t rowoff = m * (int64_t)N;
                if (mode == SQ_EPI_RAW_I32) {
                    int32_t *y = static_cast<int32_t *>(Y);
#pragma unroll
                    for (int j = 0; j < 128; j += 4) {
                        const int64_t n = nb + j;
                        if (vec_ok && n + 3 < N) {
                            *reinterpret_cast<int4 *>(y + rowoff + n) =
                                make_int4(part[j], part[j + 1], part[j + 2], part[j + 3]);
                        } else {
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                if (n + e < N) y[rowoff + n + e] = part[j + e];
                        }
                    }
                } else {
                    float *y = static_cast<float *>(Y);
                    const float xs = __ldg(sx + m);
#pragma unroll
                    for (int j = 0; j < 128; j += 4) {
                        const int64_t n = nb + j;
                        if (n >= N) break;
                        float r[4] = {0.f, 0.f, 0.f, 0.f}, bb[4] = {0.f, 0.f, 0.f, 0.f};
                        float ws[4];
                        if (vec_ok && n + 3 < N) {
                            const float4 w4 = __ldg(reinterpret_cast<const float4 *>(sw + n));
                            ws[0] = w4.x; ws[1] = w4.y; ws[2] = w4.z; ws[3] = w4.w;
                            if (mode != SQ_EPI_NONE) {
                                const float4 b4 = __ldg(reinterpret_cast<const float4 *>(bias + n));
                                bb[0] = b4.x; bb[1] = b4.y; bb[2] = b4.z; bb[3] = b4.w;
                            }
                            if (mode == SQ_EPI_BIAS_RESIDUAL) {
                                const float4 r4 =
                                    *reinterpret_cast<const float4 *>(residual + rowoff + n);
                                r[0] = r4.x; r[1] = r4.y; r[2] = r4.z; r[3] = r4.w;
                            }
                        } else {
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const bool ok = n + e < N;
                                ws[e] = ok ? __ldg(sw + n + e) : 0.f;
                                if (mode != SQ_EPI_NONE) bb[e] = ok ? __ldg(bias + n + e) : 0.f;
                                if (mode == SQ_EPI_BIAS_RESIDUAL)
                                    r[e] = ok ? residual[rowoff + n + e] : 0.f;
                            }
                        }
                        float o[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            o[e] = epilogue_value(part[j + e], xs, ws[e], bb[e], r[e], mode);
                        store4(y, rowoff + n, n, N, vec_ok, o[0], o[1], o[2], o[3]);
                    }
                }
            }
        }
    done_e:;
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                     "r"(TMEM_COLS)
                     : "memory");
    }
}

// ------------------------------------------------------------------ host

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

sq_status get_encoder() {
    static std::once_flag once;
    static sq_status rc = SQ_OK;
    std::call_once(once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !fn) {
            rc = SQ_ERR_CUDA;
            return;
        }
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return rc;
}

// rows x K bf16, K contiguous; box = box_rows x 64 with 128-byte swizzle
sq_status make_map(CUtensorMap *map, const void *base, int64_t rows, int64_t K, int box_rows) {
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? SQ_OK : SQ_ERR_CUDA;
}

}  // namespace

sq_status launch_gemm_tc(const __nv_bfloat16 *Xop, const float *sx, const __nv_bfloat16 *Wop,
                         const float *sw, const float *bias, const float *residual, int64_t M,
                         int64_t N, int64_t K, int mode, void *Y, cudaStream_t st) {
    if (M > 0x7fffffff || N > 0x7fffffff) return SQ_ERR_UNSUPPORTED;
    sq_status rc = get_encoder();
    if (rc != SQ_OK) return rc;
    DeviceInfo di;
    if ((rc = device_info(&di)) != SQ_OK) return rc;
    static int attr_dev = -1;
    if (attr_dev != di.device) {
        if (cudaFuncSetAttribute(gemm_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 SMEM_BYTES) != cudaSuccess)
            return SQ_ERR_CUDA;
        attr_dev = di.device;
    }
    CUtensorMap ta, tb;
    if ((rc = make_map(&ta, Xop, M, K, BM)) != SQ_OK) return rc;
    if ((rc = make_map(&tb, Wop, N, K, BN)) != SQ_OK) return rc;
    const int64_t tiles = ((M + BM - 1) / BM) * ((N + BN - 1) / BN);
    if (tiles > 0x7fffffff) return SQ_ERR_UNSUPPORTED;
    const int grid = (int)std::min<int64_t>(tiles, di.sms);
    // 16-byte vector loads/stores of the epilogue need N % 4 == 0 and aligned vectors
    const int vec_ok = (N % 4 == 0) && aligned16(Y) &&
                       (mode == SQ_EPI_RAW_I32 || aligned16(sw)) &&
                       (bias == nullptr || aligned16(bias)) &&
                       (residual == nullptr || aligned16(residual));
    gemm_tc_kernel<<<grid, THREADS, SMEM_BYTES, st>>>(ta, tb, sx, sw, bias, residual, (int)M,
                                                      (int)N, (int)K, mode, vec_ok, Y);
    return cuda_status(cudaGetLastError());
}

sq_status gemm_tc_take_error(cudaStream_t st) {
    unsigned int word = 0;
    if (cudaMemcpyFromSymbolAsync(&word, g_tc_error, sizeof(word), 0, cudaMemcpyDeviceToHost,
                                  st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return SQ_ERR_CUDA;
    if (word != 0) {
        const unsigned int zero = 0;
        if (cudaMemcpyToSymbolAsync(g_tc_error, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice,
                                    st) != cudaSuccess ||
            cudaStreamSynchronize(st) != cudaSuccess)
            return SQ_ERR_CUDA;
        return SQ_ERR_TIMEOUT;
    }
    return SQ_OK;
}

}  // namespace sq

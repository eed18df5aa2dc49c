// INT8 GEMM + fused dequantising epilogue on the legacy warp-level integer
// MMA (mma.sync.m16n8k32 s8 x s8 -> s32): exact by construction.  This is the
// comparison point for the tcgen05 path, not the primary kernel.
//
// "Efficient INT8 Inference of Small NLP Models on Server CPUs with PyTorch
// Native Stack": the linear block is the int8 GEMM plus its fused post-ops
// (Table 3 caption); scales are per token x per output channel.
//
// Tiling: 128 x 128 output tile per 256-thread CTA (8 warps as 2 x 4, 64 x 32
// per warp), K staged 128 bytes at a time through a 4-deep cp.async ring.
// Shared-memory rows are 128 bytes with the 16-byte chunks XOR-swizzled by
// (row & 7), so both the cp.async writes and the ldmatrix reads are free of
// bank conflicts.  Out-of-range rows and the K tail are zero-filled.
#include "common.cuh"

namespace sq {
namespace {

constexpr int BM = 128, BN = 128, BK = 128;  // BK in bytes (= int8 elements)
constexpr int STAGES = 4;
constexpr int THREADS = 256;
constexpr int TILE_BYTES = BM * BK;           // 16 KB per operand per stage
constexpr int SMEM_BYTES = STAGES * 2 * TILE_BYTES;

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
                 "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t &r0, uint32_t &r1,
                                            uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldmatrix_x2(uint32_t addr, uint32_t &r0, uint32_t &r1) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];\n"
                 : "=r"(r0), "=r"(r1)
                 : "r"(addr));
}

__device__ __forceinline__ void mma_s8(int32_t (&c)[4], const uint32_t (&a)[4],
                                       const uint32_t (&b)[2]) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+r"(c[0]), "+r"(c[1]), "+r"(c[2]), "+r"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// byte offset of (row, 16-byte chunk) inside a 128-byte-row swizzled tile
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
    return (uint32_t)(row * BK + ((chunk ^ (row & 7)) << 4));
}

__device__ __forceinline__ void load_stage(uint32_t sA, uint32_t sB, const int8_t *Xq,
                                           const int8_t *Wq, int64_t M, int64_t N, int64_t K,
                                           int64_t m0, int64_t n0, int64_t k0) {
    // 128 rows x 8 chunks per operand = 1024 chunks, 4 per thread
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int idx = threadIdx.x + i * THREADS;
        const int row = idx >> 3, chunk = idx & 7;
        const int64_t k = k0 + chunk * 16;
        {
            const int64_t m = m0 + row;
            const bool ok = m < M && k < K;
            const int8_t *src = ok ? Xq + m * K + k : Xq;
            cp_async16(sA + swz(row, chunk), src, ok ? 16 : 0);
        }
        {
            const int64_t n = n0 + row;
            const bool ok = n < N && k < K;
            const int8_t *src = ok ? Wq + n * K + k : Wq;
            cp_async16(sB + swz(row, chunk), src, ok ? 16 : 0);
        }
    }
}

__global__ void __launch_bounds__(THREADS) gemm_mma_sync_kernel(
    const int8_t *__restrict__ Xq, const float *__restrict__ sx, const int8_t *__restrict__ Wq,
    const float *__restrict__ sw, const float *__restrict__ bias,
    const float *__restrict__ residual, int64_t M, int64_t N, int64_t K, int mode, void *Y) {
    extern __shared__ __align__(128) uint8_t smem[];
    const uint32_t s0 = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int wm = warp >> 2, wn = warp & 3;  // 2 x 4 warps, 64 x 32 each
    const int64_t m0 = (int64_t)blockIdx.x * BM, n0 = (int64_t)blockIdx.y * BN;
    const int64_t ktiles = (K + BK - 1) / BK;

    int32_t acc[4][4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int v = 0; v < 4; ++v) acc[i][j][v] = 0;

#pragma unroll
    for (int st = 0; st < STAGES - 1; ++st) {
        if (st < ktiles)
            load_stage(s0 + st * 2 * TILE_BYTES, s0 + st * 2 * TILE_BYTES + TILE_BYTES, Xq, Wq,
                       M, N, K, m0, n0, (int64_t)st * BK);
        cp_async_commit();
    }

    for (int64_t kt = 0; kt < ktiles; ++kt) {
        cp_async_wait<STAGES - 2>();
        __syncthreads();
        {   // prefetch tile kt + STAGES - 1 into the slot freed by tile kt - 1
            const int64_t nk = kt + STAGES - 1;
            if (nk < ktiles) {
                const int slot = (int)(nk % STAGES);
                load_stage(s0 + slot * 2 * TILE_BYTES, s0 + slot * 2 * TILE_BYTES + TILE_BYTES,
                           Xq, Wq, M, N, K, m0, n0, nk * BK);
            }
            cp_async_commit();
        }
        const int slot = (int)(kt % STAGES);
        const uint32_t sA = s0 + slot * 2 * TILE_BYTES, sB = sA + TILE_BYTES;
#pragma unroll
        for (int ks = 0; ks < BK / 32; ++ks) {  // 4 k32 steps = chunks 2ks, 2ks+1
            uint32_t a[4][4], b[4][2];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                // x4: matrices (rows 0-7, chunk 2ks), (rows 8-15, 2ks),
                //     (rows 0-7, 2ks+1), (rows 8-15, 2ks+1)
                const int r = wm * 64 + i * 16 + (lane & 15);
                const int c = 2 * ks + (lane >> 4);
                ldmatrix_x4(sA + swz(r, c), a[i][0], a[i][1], a[i][2], a[i][3]);
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int r = wn * 32 + j * 8 + (lane & 7);
                const int c = 2 * ks + ((lane >> 3) & 1);
                ldmatrix_x2(sB + swz(r, c), b[j][0], b[j][1]);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) mma_s8(acc[i][j], a[i], b[j]);
        }
    }
    cp_async_wait<0>();

    // epilogue straight from the accumulator fragments:
    // c0,c1 -> (row g, cols 2t, 2t+1); c2,c3 -> (row g+8, same cols)
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int64_t m = m0 + wm * 64 + i * 16 + g + h * 8;
            if (m >= M) continue;
            const float xs = mode == SQ_EPI_RAW_I32 ? 0.f : __ldg(sx + m);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int64_t n = n0 + wn * 32 + j * 8 + 2 * t;
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int64_t nn = n + e;
                    if (nn >= N) continue;
                    const int32_t a = acc[i][j][2 * h + e];
                    if (mode == SQ_EPI_RAW_I32) {
                        static_cast<int32_t *>(Y)[m * N + nn] = a;
                    } else {
                        const float b = mode == SQ_EPI_NONE ? 0.f : __ldg(bias + nn);
                        const float r =
                            mode == SQ_EPI_BIAS_RESIDUAL ? __ldg(residual + m * N + nn) : 0.f;
                        static_cast<float *>(Y)[m * N + nn] =
                            epilogue_value(a, xs, __ldg(sw + nn), b, r, mode);
                    }
                }
            }
        }
    }
}

}  // namespace

sq_status launch_gemm_mma_sync(const int8_t *Xq, const float *sx, const int8_t *Wq,
                               const float *sw, const float *bias, const float *residual,
                               int64_t M, int64_t N, int64_t K, int mode, void *Y,
                               cudaStream_t st) {
    static bool attr_set = false;
    if (!attr_set) {
        if (cudaFuncSetAttribute(gemm_mma_sync_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 SMEM_BYTES) != cudaSuccess)
            return SQ_ERR_CUDA;
        attr_set = true;
    }
    // x walks M tiles (consecutive CTAs share a weight tile), y walks N tiles
    const int64_t gx = (M + BM - 1) / BM, gy = (N + BN - 1) / BN;
    if (gx > 0x7fffffff || gy > 65535) return SQ_ERR_UNSUPPORTED;
    gemm_mma_sync_kernel<<<dim3((unsigned)gx, (unsigned)gy), THREADS, SMEM_BYTES, st>>>(
        Xq, sx, Wq, sw, bias, residual, M, N, K, mode, Y);
    return cuda_status(cudaGetLastError());
}

}  // namespace sq

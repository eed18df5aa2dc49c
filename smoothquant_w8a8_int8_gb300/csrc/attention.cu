// Encoder self-attention, softmax(Q K^T * scale) V per sequence and head, on the
// 5th-generation tensor cores (tcgen05, sm_103a).
//
// "Efficient INT8 Inference of Small NLP Models on Server CPUs with PyTorch
// Native Stack", Table 3: attention is the largest share of BERT-large's time
// beside the linear block.  The input is the fused QKV projection's fp32
// output, row-major [B*S][3*H*D] (Q, K, V blocks; head h at columns h*D of
// each); the output O is fp32 [B*S][H*D].  Every token attends to every token
// of its sequence (no mask).
//
// Precision.  The two contractions run on kind::tf32 with each fp32 operand
// split exactly into x = hi + lo, hi = x with its 13 low significand bits
// cleared, lo = x - hi (exact in fp32), and the products summed as
// hi*hi' + hi*lo' + lo*hi' in fp32 tensor memory: the operand the tensor core
// sees for hi is exact and lo loses at most 2 of its 13 bits, so each product
// is within about 2^-21 (relative) of the fp32 product.  The row maximum is
// subtracted before exp2; the row sum and the division by it run in fp32.
//
// One CTA per (sequence, head, tile of 128 queries); S a multiple of 64, at
// most 448 (the logits of a query tile live in tensor memory: S columns, plus
// 64 for O).  Roles (288 threads):
//   warps 0-3  softmax and epilogue: thread r owns query row r of the tile and
//              tensor-memory lane r; reads all S logits for the exact row
//              maximum, then writes exp2((s - max) * scale * log2 e) chunk by
//              chunk as the split A operand of P V, and finally O / sum;
//   warps 4-7  loaders: the Q tile, then the K chunks and the V chunks (64
//              keys each; V transposed so that keys run along K), split into
//              hi / lo tf32 parts in shared memory (128-byte swizzle, K-major);
//   warp 8     tensor memory, and lane 0 issues the MMAs:
//              S[:, 64c..] = Q K_c^T, then O += P_c V_c.
// Every wait is bounded (about 4 s); on expiry the CTA records an error for
// sq_device_status, lets its MMAs drain, frees tensor memory and exits.
#include "common.cuh"

#include <mutex>

namespace sq {
namespace {

constexpr int AD = 64;    // head dimension
constexpr int ABQ = 128;  // queries per CTA (the MMA's M)
constexpr int ACH = 64;   // keys per chunk (the first MMA's N, the second's K)
constexpr int AMAXS = 448;
constexpr int A_THREADS = 288;
constexpr int Q_PART = ABQ * AD * 4;   // 32 KB: one tf32 part of the Q tile
constexpr int KV_PART = ACH * AD * 4;  // 16 KB: one part of a K or V^T chunk
constexpr int P_PART = ABQ * ACH * 4;  // 32 KB: one part of a P chunk
constexpr int OFF_QH = 0, OFF_QL = Q_PART;
constexpr int OFF_RING = 2 * Q_PART;  // 2 stages x (hi, lo)
constexpr int OFF_PH = OFF_RING + 4 * KV_PART, OFF_PL = OFF_PH + P_PART;
constexpr int OFF_BAR = OFF_PL + P_PART;
constexpr int A_SMEM = OFF_BAR + 256 + 1024;  // barriers; 1024-byte alignment slack
constexpr int TMEM_COLS = 512;                // S (<= 448) + O (64)
constexpr unsigned long long kAttnTimeoutNs = 4000000000ull;
constexpr float kLog2e = 1.4426950408889634f;

// instruction descriptor, kind::tf32: D fp32, A and B tf32, both K-major, N = 64, M = 128
constexpr uint32_t IDESC_TF32 =
    (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(64 >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);

__device__ unsigned int g_attn_error;

struct AttnBars {
    uint64_t q_full, ring_full[2], ring_empty[2], s_full, p_full, p_empty, o_full, mma_done;
    uint32_t tmem_base;
    int abort_flag;
};
static_assert(sizeof(AttnBars) <= 256, "barrier block");

__device__ __forceinline__ uint32_t su32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ uint64_t gtime() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ bool try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, volatile int *abort) {
    const uint64_t t0 = gtime();
    for (uint32_t it = 1;; ++it) {
        if (try_wait(bar, parity)) return true;
        if ((it & 63u) == 0) {
            if (*abort) return false;
            if (gtime() - t0 > kAttnTimeoutNs) {
                *abort = 1;
                atomicOr(&g_attn_error, 1u);
                return false;
            }
        }
    }
}
// Bounded wait for the phase of parity `parity`; false when the CTA aborted.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int *abort) {
    if (try_wait(bar, parity)) return true;
    return wait_slow(bar, parity, abort);
}
// One lane waits, the warp learns the outcome.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int *abort) {
    int ok = 1;
    if ((threadIdx.x & 31) == 0) ok = wait_bar(bar, parity, abort);
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}
__device__ __noinline__ void drain_bar(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = gtime();
    while (!try_wait(bar, parity))
        if (gtime() - t0 > kAttnTimeoutNs) {
            atomicOr(&g_attn_error, 2u);
            return;
        }
}
__device__ __forceinline__ void bar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void fence_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tc_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// K-major operand, 128-byte swizzle: rows of 128 bytes, 8-row atoms 1024 bytes apart
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
    uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)1 << 16;
    d |= (uint64_t)(1024 >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}
__device__ __forceinline__ void mma_tf32(uint32_t d, uint64_t a, uint64_t b, uint32_t acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
        "l"(a), "l"(b), "r"(IDESC_TF32), "r"(acc)
        : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
        "%28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
}

// Byte offset of element (row, k), k < 64, of an operand part of `rows` rows:
// two 32-float K blocks of rows x 128 bytes, 16-byte chunk j of a row at
// j ^ (row & 7) (the 128-byte swizzle; every part starts 1024-byte aligned).
__device__ __forceinline__ uint32_t sw_off(int row, int k, int rows) {
    return (uint32_t)((k >> 5) * rows * 128 + row * 128 + ((((k & 31) >> 2) ^ (row & 7)) << 4) +
                      ((k & 3) << 2));
}

// exact split of x into a tf32 part and the fp32 remainder
__device__ __forceinline__ float hi_part(float x) {
    return __uint_as_float(__float_as_uint(x) & 0xffffe000u);
}

__global__ void __launch_bounds__(A_THREADS, 1)
    attention_kernel(const float *__restrict__ QKV, int S, int H, float scale,
                     float *__restrict__ O) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    AttnBars &B = *reinterpret_cast<AttnBars *>(smem + OFF_BAR);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int qtiles = (S + ABQ - 1) / ABQ;
    const int qt = blockIdx.x % qtiles;
    const int h = (blockIdx.x / qtiles) % H;
    const int b = blockIdx.x / (qtiles * H);
    const int q0 = qt * ABQ;
    const int nch = S / ACH;
    const int64_t ld = 3LL * H * AD;  // QKV row stride (floats)
    const float *qkv_b = QKV + (int64_t)b * S * ld;

    if (threadIdx.x == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 4;" ::"r"(su32(&B.q_full)));
        for (int i = 0; i < 2; ++i) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 4;" ::"r"(su32(&B.ring_full[i])));
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(su32(&B.ring_empty[i])));
        }
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(su32(&B.s_full)));
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 4;" ::"r"(su32(&B.p_full)));
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(su32(&B.p_empty)));
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(su32(&B.o_full)));
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(su32(&B.mma_done)));
        B.abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 8) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         su32(&B.tmem_base)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_before();
    __syncthreads();
    tc_after();
    pdl_launch_dependents();
    pdl_wait();  // every global-memory access below follows the previous kernel
    const uint32_t tmem = B.tmem_base;
    volatile int *abort = &B.abort_flag;
    const uint32_t sbase = su32(smem);

    if (warp >= 4 && warp < 8) {
        // -------------------------------------------------------------- loaders
        const int t = threadIdx.x - 128;
        {
            // the Q tile: thread t owns query row t (rows past S load zeros)
            const bool ok = q0 + t < S;
            const float4 *src =
                reinterpret_cast<const float4 *>(qkv_b + (int64_t)(ok ? q0 + t : 0) * ld + h * AD);
#pragma unroll 4
            for (int i = 0; i < AD / 4; ++i) {
                const float4 v = ok ? __ldg(src + i) : make_float4(0.f, 0.f, 0.f, 0.f);
                const float4 vh = make_float4(hi_part(v.x), hi_part(v.y), hi_part(v.z),
                                              hi_part(v.w));
                const float4 vl = make_float4(v.x - vh.x, v.y - vh.y, v.z - vh.z, v.w - vh.w);
                const uint32_t off = sw_off(t, 4 * i, ABQ);
                *reinterpret_cast<float4 *>(smem + OFF_QH + off) = vh;
                *reinterpret_cast<float4 *>(smem + OFF_QL + off) = vl;
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) bar_arrive(su32(&B.q_full));
        }
        for (int n = 0; n < 2 * nch; ++n) {
            const int slot = n & 1;
            const uint32_t ph = (uint32_t)(n >> 1) & 1u;
            if (!warp_wait(su32(&B.ring_empty[slot]), ph ^ 1u, abort)) break;
            uint8_t *hi = smem + OFF_RING + slot * 2 * KV_PART;
            uint8_t *lo = hi + KV_PART;
            if (n < nch) {
                // K chunk n: thread t takes key t / 2, dimensions 32 (t % 2) ..
                const int key = t >> 1, half = t & 1;
                const float4 *src = reinterpret_cast<const float4 *>(
                    qkv_b + (int64_t)(n * ACH + key) * ld + (int64_t)H * AD + h * AD + 32 * half);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float4 v = __ldg(src + i);
                    const float4 vh = make_float4(hi_part(v.x), hi_part(v.y), hi_part(v.z),
                                                  hi_part(v.w));
                    const float4 vl = make_float4(v.x - vh.x, v.y - vh.y, v.z - vh.z, v.w - vh.w);
                    const uint32_t off = sw_off(key, 32 * half + 4 * i, ACH);
                    *reinterpret_cast<float4 *>(hi + off) = vh;
                    *reinterpret_cast<float4 *>(lo + off) = vl;
                }
            } else {
                // V chunk n - nch, transposed (rows: dimensions, K: keys): thread t
                // takes key t % 64, dimensions 32 (t / 64) ..; a warp writes 32
                // consecutive keys of one row per store
                const int key = t & 63, dh = t >> 6;
                const float4 *src = reinterpret_cast<const float4 *>(
                    qkv_b + (int64_t)((n - nch) * ACH + key) * ld + 2LL * H * AD + h * AD +
                    32 * dh);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float4 v = __ldg(src + i);
                    const float e[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const float eh = hi_part(e[j]);
                        const uint32_t off = sw_off(32 * dh + 4 * i + j, key, AD);
                        *reinterpret_cast<float *>(hi + off) = eh;
                        *reinterpret_cast<float *>(lo + off) = e[j] - eh;
                    }
                }
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) bar_arrive(su32(&B.ring_full[slot]));
        }
    } else if (warp == 8) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0) {
            if (!wait_bar(su32(&B.q_full), 0, abort)) goto done_m;
            tc_after();
            for (int c = 0; c < nch; ++c) {
                const int slot = c & 1;
                if (!wait_bar(su32(&B.ring_full[slot]), (uint32_t)(c >> 1) & 1u, abort))
                    goto done_m;
                tc_after();
                const uint32_t kh = sbase + OFF_RING + slot * 2 * KV_PART, kl = kh + KV_PART;
                const uint32_t d = tmem + (uint32_t)(c * ACH);
#pragma unroll
                for (int p = 0; p < 3; ++p) {
                    const uint32_t a = p == 2 ? sbase + OFF_QL : sbase + OFF_QH;
                    const uint32_t bb = p == 1 ? kl : kh;
#pragma unroll
                    for (int kb = 0; kb < 2; ++kb) {
                        const uint64_t ad = desc_sw128(a + kb * ABQ * 128);
                        const uint64_t bd = desc_sw128(bb + kb * ACH * 128);
#pragma unroll
                        for (int k = 0; k < 4; ++k)  // K = 8 tf32 = 32 bytes per MMA
                            mma_tf32(d, ad + 2 * k, bd + 2 * k, (p | kb | k) ? 1u : 0u);
                    }
                }
                mma_commit(su32(&B.ring_empty[slot]));
            }
            mma_commit(su32(&B.s_full));
            for (int c = 0; c < nch; ++c) {
                const int n = nch + c, slot = n & 1;
                if (!wait_bar(su32(&B.ring_full[slot]), (uint32_t)(n >> 1) & 1u, abort))
                    goto done_m;
                if (!wait_bar(su32(&B.p_full), (uint32_t)c & 1u, abort)) goto done_m;
                tc_after();
                const uint32_t vh = sbase + OFF_RING + slot * 2 * KV_PART, vl = vh + KV_PART;
                const uint32_t d = tmem + (uint32_t)AMAXS;  // O after the logits' columns
#pragma unroll
                for (int p = 0; p < 3; ++p) {
                    const uint32_t a = p == 2 ? sbase + OFF_PL : sbase + OFF_PH;
                    const uint32_t bb = p == 1 ? vl : vh;
#pragma unroll
                    for (int kb = 0; kb < 2; ++kb) {
                        const uint64_t ad = desc_sw128(a + kb * ABQ * 128);
                        const uint64_t bd = desc_sw128(bb + kb * AD * 128);
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            mma_tf32(d, ad + 2 * k, bd + 2 * k, (c | p | kb | k) ? 1u : 0u);
                    }
                }
                mma_commit(su32(&B.ring_empty[slot]));
                mma_commit(su32(&B.p_empty));
            }
            mma_commit(su32(&B.o_full));
        done_m:
            // every MMA issued above completes before tensor memory is freed
            mma_commit(su32(&B.mma_done));
            drain_bar(su32(&B.mma_done), 0);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ softmax and epilogue
        const int r = threadIdx.x;  // query row of the tile, tensor-memory lane
        const uint32_t lane_addr = tmem + ((uint32_t)(32 * warp) << 16);
        const float cl2e = scale * kLog2e;
        if (!warp_wait(su32(&B.s_full), 0, abort)) goto done_s;
        tc_after();
        {
            // the row maximum over all S logits
            float m = -INFINITY;
            for (int sl = 0; sl < S / 32; ++sl) {
                float v[32];
                tmem_ld32(lane_addr + 32 * sl, v);
#pragma unroll
                for (int j = 0; j < 32; ++j) m = fmaxf(m, v[j]);
            }
            const float mc = m * cl2e;
            float sum = 0.0f;
            for (int c = 0; c < nch; ++c) {
                // the P buffer is free once the previous chunk's MMAs are done
                if (!warp_wait(su32(&B.p_empty), ((uint32_t)c & 1u) ^ 1u, abort)) goto done_s;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    float v[32];
                    tmem_ld32(lane_addr + c * ACH + 32 * half, v);
#pragma unroll
                    for (int j = 0; j < 32; j += 4) {
                        float pp[4], ph[4], pl[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            pp[e] = exp2f(__fmaf_rn(v[j + e], cl2e, -mc));
                            sum += pp[e];
                            ph[e] = hi_part(pp[e]);
                            pl[e] = pp[e] - ph[e];
                        }
                        const uint32_t off = sw_off(r, 32 * half + j, ABQ);
                        *reinterpret_cast<float4 *>(smem + OFF_PH + off) =
                            make_float4(ph[0], ph[1], ph[2], ph[3]);
                        *reinterpret_cast<float4 *>(smem + OFF_PL + off) =
                            make_float4(pl[0], pl[1], pl[2], pl[3]);
                    }
                }
                fence_async_smem();
                tc_before();
                __syncwarp();
                if (lane == 0) bar_arrive(su32(&B.p_full));
            }
            if (!warp_wait(su32(&B.o_full), 0, abort)) goto done_s;
            tc_after();
            const float inv = __frcp_rn(sum);
            float o[64];
            tmem_ld32(lane_addr + AMAXS, *reinterpret_cast<float(*)[32]>(o));
            tmem_ld32(lane_addr + AMAXS + 32, *reinterpret_cast<float(*)[32]>(o + 32));
            if (q0 + r < S) {
                float4 *dst = reinterpret_cast<float4 *>(O + ((int64_t)b * S + q0 + r) * H * AD +
                                                         h * AD);
#pragma unroll
                for (int i = 0; i < AD / 4; ++i)
                    dst[i] = make_float4(o[4 * i] * inv, o[4 * i + 1] * inv, o[4 * i + 2] * inv,
                                         o[4 * i + 3] * inv);
            }
        }
    done_s:;
    }
    tc_before();
    __syncthreads();
    if (warp == 8) {
        tc_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(TMEM_COLS)
                     : "memory");
    }
}

}  // namespace

sq_status launch_attention(const float *QKV, int64_t B, int64_t S, int64_t H, float scale,
                           float *O, cudaStream_t st) {
    DeviceInfo di;
    sq_status rc = device_info(&di);
    if (rc != SQ_OK) return rc;
    static std::mutex mu;
    static bool attr[64] = {};
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!attr[di.device & 63]) {
            if (cudaFuncSetAttribute(attention_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     A_SMEM) != cudaSuccess)
                return SQ_ERR_CUDA;
            attr[di.device & 63] = true;
        }
    }
    const int64_t grid = B * H * ((S + ABQ - 1) / ABQ);
    if (grid > 0x7fffffff) return SQ_ERR_UNSUPPORTED;
    return launch_pdl(attention_kernel, dim3((unsigned)grid), dim3(A_THREADS), A_SMEM, st, 1, QKV,
                      (int)S, (int)H, scale, O);
}

sq_status attention_take_error(cudaStream_t st) {
    unsigned int word = 0;
    if (cudaMemcpyFromSymbolAsync(&word, g_attn_error, sizeof(word), 0, cudaMemcpyDeviceToHost,
                                  st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return SQ_ERR_CUDA;
    if (word != 0) {
        const unsigned int zero = 0;
        if (cudaMemcpyToSymbolAsync(g_attn_error, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice,
                                    st) != cudaSuccess ||
            cudaStreamSynchronize(st) != cudaSuccess)
            return SQ_ERR_CUDA;
        return SQ_ERR_TIMEOUT;
    }
    return SQ_OK;
}

}  // namespace sq

// INT8 GEMM + fused dequantising epilogue on the 5th-generation tensor cores
// (tcgen05, sm_103a): TMA-fed shared-memory ring, accumulators in tensor
// memory, warp-specialised persistent CTAs, TMA-staged epilogue stores.
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
// Two kernels share the epilogue code below.  The pair kernel (end of the
// kernel section: clusters of two CTAs, tcgen05.mma.cta_group::2, 256 x 256
// tiles) runs every launch with at least 256 rows that is not split over K;
// the one-CTA kernel runs the rest, including the split-K schedule (fewer
// tiles than SMs, K >= 2048, a caller workspace).  Both are launched with
// programmatic dependent launch: set-up overlaps the previous kernel on the
// stream, every global-memory access follows griddepcontrol.wait.
//
// One-CTA roles (320 threads, one CTA per SM, persistent over 128 x 256 output tiles):
//   warp 0, lane 0  TMA producer: A [128 x 64] and B [256 x 64] bf16 tiles,
//                   128-byte swizzle, into a 4-stage ring (48 KB per stage)
//   warp 1, lane 0  MMA issuer: tcgen05.mma kind::f16, M=128 N=256 K=16
//   warps 2..9      epilogue: warp w owns TMEM lanes 32*(w%4).. (32 rows of
//                   the tile) and columns 128*((w-2)/4).. (half of its width)
// Tensor memory (512 columns):
//   K <= 1024: two 256-column accumulators; the MMA fills one while the
//              epilogue drains the other.
//   K >  1024: one 256-column chunk accumulator A and a 256-column int32
//              partial P; after each chunk the epilogue adds A into P (in
//              tensor memory) and frees A, so the MMA of the next chunk only
//              waits for that short pass, and the final pass (scales, bias,
//              GELU / residual, stores) overlaps the next tile's first chunk.
//              When the caller passes the row L1 norms of the codes and
//              127 * max L1 < 2^24 for either operand, no partial sum can
//              reach 2^24 and all of K is one exact pass (the K <= 1024 case).
// Epilogue I/O per 32 x 32 slice: results are written to a per-warp 4 KB
// staging tile in shared memory (128-byte swizzle, conflict-free) and stored
// with one TMA bulk tensor store.  Shapes whose rows are not 16-byte
// multiples (N % 4 != 0) take plain per-element stores instead.
// Every wait is bounded (about 4 s of %globaltimer); on expiry the kernel
// records SQ_ERR_TIMEOUT in a device word, lets its issued copies and MMAs
// drain, frees its tensor memory and returns.
#include "common.cuh"
#include "schedule.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

namespace sq {
namespace {

using namespace sched;  // tile shape, chunking and the work schedules (schedule.cuh)
constexpr int STAGES = 4;
constexpr int UMMA_K = 16;
constexpr int THREADS = 64 + NUM_EPI_WARPS * 32;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int SLICE = 32;                   // epilogue slice: 32 rows x 32 columns
constexpr int COLS_PER_WARP = BN / 2;       // 128
constexpr int SLICES = COLS_PER_WARP / SLICE;
constexpr int STG_BYTES = SLICE * SLICE * 4;  // 4 KB staging tile per epilogue warp
constexpr int TMEM_COLS = 512;
constexpr int BAR_BYTES = 512;
constexpr int RING_BYTES = STAGES * STAGE_BYTES;
constexpr int SMEM_BYTES = RING_BYTES + NUM_EPI_WARPS * STG_BYTES + BAR_BYTES + 1024;
constexpr unsigned long long kTimeoutNs = 4000000000ull;

// instruction descriptor, kind::f16: D fp32, A/B bf16, both K-major, N, M
constexpr uint32_t IDESC_BASE = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BM >> 4) << 24);
__host__ __device__ constexpr uint32_t idesc_for(int n) { return IDESC_BASE | ((uint32_t)(n >> 3) << 17); }

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

// TMA store with an L2 evict-first policy: the output is streamed out and
// should not displace the operand tiles that other CTAs still read from L2
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, uint32_t src, int x, int y) {
    uint64_t policy;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(policy));
    asm volatile(
        "cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group.L2::cache_hint"
        " [%0, {%2, %3}], [%1], %4;" ::"l"(reinterpret_cast<uint64_t>(map)),
        "r"(src), "r"(x), "r"(y), "l"(policy)
        : "memory");
}
__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// the staging tile may be overwritten once the previous store has read it
__device__ __forceinline__ void bulk_wait_read0() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait0() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
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
                                          uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
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

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
        "%28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
        "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
        "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]),
        "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]),
        "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ---- CTA pairs (cluster of 2, cta_group::2)

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// the shared::cluster address of this CTA's shared-memory offset `saddr` in CTA `rank`
__device__ __forceinline__ uint32_t map_to_rank(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// arrive on a barrier of either CTA of the pair (after this warp's tensor-memory reads)
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cbar) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cbar)
                 : "memory");
}
// TMA load into this CTA's shared memory whose completion is counted on a
// barrier of either CTA of the pair
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap *map,
                                                 uint32_t cbar, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(cbar), "r"(x), "r"(y)
        : "memory");
}
// M = 256 (128 rows in each CTA's tensor memory), N = 256, K = 16 over the pair:
// A is each CTA's own 128 rows, B is each CTA's 128 of the 256 rows, at the
// same shared-memory offsets in both CTAs
__device__ __forceinline__ void umma_bf16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                               uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// arrive once on the barrier at offset `bar` in both CTAs of the pair when
// this thread's earlier MMAs complete
__device__ __forceinline__ void umma_commit_pair(uint32_t bar) {
    asm volatile(
        "{\n .reg .b16 mask;\n mov.b16 mask, 3;\n"
        " tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], mask;\n}\n" ::"r"(bar)
        : "memory");
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
    int32_t l1max[9][2];  // per-warp maxima of the row L1 norms (warps 1..9)
};
static_assert(sizeof(Smem) <= BAR_BYTES, "barrier block");

struct EpiArgs {
    const float *sx, *sw, *bias, *residual;
    const int32_t *x_l1, *w_l1;  // per-row sums of |code| (nullable)
    void *Y;
    int M, N;
    int tma_io;  // 1: TMA staging for Y (and the residual); 0: plain per-element I/O
    RequantOut rq;  // the requantising epilogue's outputs (kOutRequant kernels)
    // kOutRowMax kernels: per column n, (-s_next[n], RN(1/s_next[n]) or NaN),
    // two columns per float4; and the [M] running maxima they merge into
    const float4 *rm_pairs;
    float *row_amax;
    int rq_vec;     // 1: rows of the code arrays are 16-byte multiples (N % 16 == 0)
    int rq_fast;    // 1: scale >= 2^-70, so the reciprocal division may be used
    Schedule sched;     // work units (made on the host)
    int pair_plan;      // pair kernel: the cluster count its schedule is planned for
    int32_t *ws_cnt;    // split-K counters (zero between launches), or null
    int4 *ws_slots;     // split-K partial slots
};

// What the epilogue hands out: fp32 (or int32) Y; the next linear's
// Smooth-Static codes instead of Y; or Y plus each row's maximum of
// |fl(Y / s_next)| (the next linear's dynamic statistic, merged across the
// row's tiles by an integer atomicMax on the bit pattern).
constexpr int kOutPlain = 0, kOutRequant = 1, kOutRowMax = 2;

// Largest row L1 norm of int8 codes for which 127 * L1 < 2^24: then every
// partial sum of that row's products with any codes stays below 2^24 in
// magnitude and the whole K accumulates exactly in one fp32 pass.
constexpr int32_t kSinglePassL1 = 132104;

__device__ __forceinline__ float rcp_approx(float x) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}
__device__ __forceinline__ float ex2_approx(float x) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// GELU(t) = 0.5 t (1 + erf(t / sqrt 2)) on a pair.  erf by Abramowitz &
// Stegun, Handbook of Mathematical Functions, formula 7.1.26 (after Hastings):
// erf(x) = 1 - t (a1 + t (a2 + t (a3 + t (a4 + t a5)))) exp(-x^2),
// t = 1 / (1 + p x), x >= 0, odd extension for x < 0, absolute error <=
// 1.5e-7 (the hardware reciprocal and exp2 approximations add a few ulp).
// Branch-free, so a warp never splits across ranges.
__device__ __forceinline__ unsigned long long gelu2(unsigned long long t2) {
    const unsigned long long h2 = mul2(t2, pk(0.5f, 0.5f));
    const unsigned long long u2 = mul2(t2, pk(0.70710678118654752f, 0.70710678118654752f));
    float u0, u1;
    upk(u2, u0, u1);
    const unsigned long long a2 = pk(fabsf(u0), fabsf(u1));
    float d0, d1;
    upk(fma2(a2, pk(0.3275911f, 0.3275911f), pk(1.0f, 1.0f)), d0, d1);
    const unsigned long long tt = pk(rcp_approx(d0), rcp_approx(d1));
    // -poly(t) by Horner with negated coefficients, then 1 + (-poly) e
    unsigned long long p2 = fma2(pk(-1.061405429f, -1.061405429f), tt,
                                 pk(1.453152027f, 1.453152027f));
    p2 = fma2(p2, tt, pk(-1.421413741f, -1.421413741f));
    p2 = fma2(p2, tt, pk(0.284496736f, 0.284496736f));
    p2 = fma2(p2, tt, pk(-0.254829592f, -0.254829592f));
    p2 = mul2(p2, tt);
    float e0, e1;
    upk(mul2(mul2(a2, a2), pk(-1.4426950408889634f, -1.4426950408889634f)), e0, e1);
    float r0, r1;
    upk(fma2(p2, pk(ex2_approx(e0), ex2_approx(e1)), pk(1.0f, 1.0f)), r0, r1);
    return fma2(h2, pk(copysignf(r0, u0), copysignf(r1, u1)), h2);
}

// Per-column epilogue operands of one tile half, spread over the warp: lane j
// holds column (nb + 32 s + j) for slice s; a slice broadcasts them with
// shuffles.  Loaded before the accumulator wait, so their latency hides.
struct ColParams {
    float w[SLICES];
    float b[SLICES];
    float rs[SLICES], ry[SLICES];  // kOutRowMax: -s_next and RN(1/s_next) (or NaN)
};

template <int MODE, int OUT>
__device__ __forceinline__ void load_col_params(ColParams &cp, const EpiArgs &a, int nb,
                                                int lane) {
#pragma unroll
    for (int s = 0; s < SLICES; ++s) {
        const int n = nb + s * SLICE + lane;
        const bool ok = n < a.N;
        cp.w[s] = (MODE != SQ_EPI_RAW_I32 && ok) ? __ldg(a.sw + n) : 0.f;
        cp.b[s] = (MODE != SQ_EPI_RAW_I32 && MODE != SQ_EPI_NONE && ok) ? __ldg(a.bias + n) : 0.f;
        if (OUT == kOutRowMax) {
            // column n's pair alone (a float2: the table holds exactly N of them)
            const float2 c = ok ? __ldg(reinterpret_cast<const float2 *>(a.rm_pairs) + n)
                                : make_float2(-1.f, 1.f);
            cp.rs[s] = c.x;
            cp.ry[s] = c.y;
        }
    }
}

// The requantising epilogue's column parameters for this warp's 128 columns,
// (-s_next, RN(1/s_next)) per column -- NaN for the reciprocal where s_next is
// outside [2^-20, 2^20], which sends those columns to the exact path -- in the
// warp's staging area (unused by the requantising kernels), read back by every
// lane as broadcasts.
__device__ __forceinline__ void stage_next_smoothing(uint8_t *stg, const EpiArgs &a, int nb,
                                                     int lane) {
    float2 *sy = reinterpret_cast<float2 *>(stg);
#pragma unroll
    for (int s = 0; s < SLICES; ++s) {
        const int n = nb + s * SLICE + lane;
        const float sn = n < a.N ? __ldg(a.rq.s_next + n) : 1.f;
        const float as = fabsf(sn);
        const float yn = (as >= 0x1p-20f && as <= 0x1p20f) ? __frcp_rn(sn)
                                                           : __int_as_float(0x7fffffff);
        sy[s * SLICE + lane] = make_float2(-sn, yn);
    }
    __syncwarp();
}

// max that propagates NaN
__device__ __forceinline__ float max_nan(float a, float b) {
    float d;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
    return d;
}

// Requantising epilogue: the slice's fp32 values y (this thread's row m, 32
// columns from n) become the next linear's Smooth-Static codes,
// clamp(round_half_even(fl(fl(y / s_next[n]) / scale)), +-127), written as
// exact bf16 values and/or int8.  y / s_next takes the reciprocal division
// (div_smooth, exact where |y| >= 2^-100 and |y / s| <= 2^100; tinier y give
// code 0 either way since scale >= 2^-70), the code the 1.5 * 2^23 rounding;
// a thread whose slice holds a value outside that range, a smoothing factor
// outside [2^-20, 2^20] (NaN reciprocal) or a product within 2^-14 of a
// half-integer takes the IEEE divisions for that element (static_code).
__device__ __noinline__ float requant_exact(float y, float s, float scale, float rscale) {
    return static_code(__fdiv_rn(y, s), scale, rscale);
}

__device__ __forceinline__ void requant_slice(const uint32_t (&v)[32], int64_t m, int64_t n,
                                              const EpiArgs &a, const float4 *sy) {
    constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23
    const float lim = a.rq_fast ? 0.49993896484375f : -1.0f;  // 0.5 - 2^-14
    const unsigned long long r2 = pk(a.rq.rscale, a.rq.rscale);
    const unsigned long long mg2 = pk(kMagic, kMagic), nmg2 = pk(-kMagic, -kMagic);
    const unsigned long long neg1 = pk(-1.0f, -1.0f);
    float c[32];
    float dm = 0.0f, qm = 0.0f;  // largest |p - k| and |q0| (NaN kept) of the slice
#pragma unroll
    for (int j = 0; j < 32; j += 2) {
        // columns j, j+1: (-s, RN(1/s)) pairs, the same for every lane
        const float4 q = sy[j >> 1];
        const unsigned long long y2 = pk(__uint_as_float(v[j]), __uint_as_float(v[j + 1]));
        const unsigned long long yn2 = pk(q.y, q.w), ns2 = pk(q.x, q.z);
        const unsigned long long q0 = mul2(y2, yn2);
        const unsigned long long v2 = fma2(fma2(q0, ns2, y2), yn2, q0);  // div_smooth
        float p0, p1;
        upk(mul2(v2, r2), p0, p1);
        // clamping to +-127 before rounding yields the saturated code directly
        p0 = fminf(fmaxf(p0, -127.0f), 127.0f);
        p1 = fminf(fmaxf(p1, -127.0f), 127.0f);
        const unsigned long long pp = pk(p0, p1);
        const unsigned long long k2 = add2(add2(pp, mg2), nmg2);
        float k0, k1, d0, d1, qa, qb;
        upk(k2, k0, k1);
        upk(fma2(k2, neg1, pp), d0, d1);
        upk(q0, qa, qb);
        c[j] = k0;
        c[j + 1] = k1;
        dm = fmaxf(dm, fmaxf(fabsf(d0), fabsf(d1)));
        qm = max_nan(qm, max_nan(fabsf(qa), fabsf(qb)));
    }
    // a near-tie, a NaN or a |q0| above 2^100 somewhere in the slice: those
    // elements take the exact path (rare; one branch per slice)
    if (!(dm <= lim) || !(qm <= 0x1p100f)) {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const float2 q = reinterpret_cast<const float2 *>(sy)[j];
            const float y = __uint_as_float(v[j]);
            const float q0 = __fmul_rn(y, q.y);
            const float vv = __fmaf_rn(__fmaf_rn(q0, q.x, y), q.y, q0);
            const float p = fminf(fmaxf(__fmul_rn(vv, a.rq.rscale), -127.0f), 127.0f);
            const float k = __fsub_rn(__fadd_rn(p, kMagic), kMagic);
            if (!(fabsf(__fsub_rn(p, k)) <= lim) || !(fabsf(q0) <= 0x1p100f))
                c[j] = requant_exact(y, -q.x, a.rq.scale, a.rq.rscale);
        }
    }
    if (m >= a.M) return;
    const int64_t off = m * a.N + n;
    if (a.rq_vec && n + 31 < a.N) {
        if (a.rq.Yop) {
            uint4 *dst = reinterpret_cast<uint4 *>(a.rq.Yop + off);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e)  // integers |c| <= 127: the high halves are exact bf16
                    w[e] = __byte_perm(__float_as_uint(c[8 * q + 2 * e]),
                                       __float_as_uint(c[8 * q + 2 * e + 1]), 0x7632);
                dst[q] = make_uint4(w[0], w[1], w[2], w[3]);
            }
        }
        if (a.rq.Yq) {
            uint4 *dst = reinterpret_cast<uint4 *>(a.rq.Yq + off);
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int j = 16 * q + 4 * e;
                    w[e] = (uint32_t)(__float2int_rn(c[j]) & 0xff) |
                           ((uint32_t)(__float2int_rn(c[j + 1]) & 0xff) << 8) |
                           ((uint32_t)(__float2int_rn(c[j + 2]) & 0xff) << 16) |
                           ((uint32_t)(__float2int_rn(c[j + 3]) & 0xff) << 24);
                }
                dst[q] = make_uint4(w[0], w[1], w[2], w[3]);
            }
        }
    } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            if (n + j >= a.N) break;
            if (a.rq.Yop) a.rq.Yop[off + j] = __float2bfloat16_rn(c[j]);
            if (a.rq.Yq) a.rq.Yq[off + j] = (int8_t)__float2int_rn(c[j]);
        }
    }
}

// max over this thread's slice (row m, columns n..n+31 that are < N) of
// |fl(y / s_next[col])|, exactly: the corrected reciprocal division
// (div_smooth on f32x2 pairs) with the column pairs read as warp-uniform
// broadcasts.  It is the IEEE quotient wherever |s| is in [2^-20, 2^20] (else
// the table holds NaN), |y| >= 2^-100 and the quotient's first product is at
// most 2^100; a slice whose maximum is below 2^-70 may hold inexact tiny
// quotients, so it, a NaN or a product above 2^100 sends the slice to IEEE
// divisions (rare).  Partial slices take IEEE divisions too.
__device__ __forceinline__ float max3_nan_f(float a, float b, float c) {
    float d;
    asm("max.NaN.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

__device__ __noinline__ float slice_rowmax_exact(const float *y, const float4 *pairs, int64_t n,
                                                 int N) {
    float mx = 0.0f;
    for (int j = 0; j < 32 && n + j < N; ++j) {
        const float4 c = pairs[(n + j) >> 1];
        const float ns = ((n + j) & 1) ? c.z : c.x;
        mx = fmaxf(mx, fabsf(__fdiv_rn(y[j], -ns)));
    }
    return mx;
}

// rml: this lane's column (n + lane) pair (-s_next, RN(1/s_next)), shuffled out
// to every lane column by column (warp-uniform global loads here measured
// ~13 us slower per FFN up-projection: the L1 left beside the shared memory is
// small, so they wait on L2)
__device__ __forceinline__ float slice_rowmax(const uint32_t (&v)[32], int64_t n,
                                              const EpiArgs &a, float2 rml) {
    if (n + 31 < a.N) {
        float mx = 0.0f, qm = 0.0f;
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
            const float ns0 = __shfl_sync(0xffffffffu, rml.x, j);
            const float ns1 = __shfl_sync(0xffffffffu, rml.x, j + 1);
            const float yy0 = __shfl_sync(0xffffffffu, rml.y, j);
            const float yy1 = __shfl_sync(0xffffffffu, rml.y, j + 1);
            const unsigned long long y2 = pk(__uint_as_float(v[j]), __uint_as_float(v[j + 1]));
            const unsigned long long yn2 = pk(yy0, yy1);
            const unsigned long long q0 = mul2(y2, yn2);
            float a0, a1, b0, b1;
            upk(fma2(fma2(q0, pk(ns0, ns1), y2), yn2, q0), a0, a1);
            upk(q0, b0, b1);
            mx = max3_nan_f(mx, fabsf(a0), fabsf(a1));
            qm = max3_nan_f(qm, fabsf(b0), fabsf(b1));
        }
        if (qm <= 0x1p100f && mx >= 0x1p-70f) return mx;  // NaN fails both
    }
    // rare: the slice's values through memory (a stack copy), IEEE divisions
    float y[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) y[j] = __uint_as_float(v[j]);
    return slice_rowmax_exact(y, a.rm_pairs, n, a.N);
}

// The residual of one slice (the warp's 32 rows from m - lane, 32 columns
// from n).  A whole slice on the TMA output path (COAL) is read coalesced:
// r[c] = row 4 c + lane / 8, columns n + 4 (lane % 8) .. +3, four 128-byte
// lines per instruction (epilogue_slice transposes it through the staging
// tile); otherwise r holds this thread's own row segment.
template <bool COAL>
__device__ __forceinline__ void load_residual(float4 (&r)[8], const EpiArgs &a, int64_t m,
                                              int64_t n) {
    if (COAL && a.tma_io && n + 31 < a.N) {
        const int lane = threadIdx.x & 31;
        const int64_t r0 = m - lane + (lane >> 3);
        const float *base = a.residual + n + 4 * (lane & 7);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const int64_t rr = r0 + 4 * c;
            r[c] = rr < a.M ? *reinterpret_cast<const float4 *>(base + rr * (int64_t)a.N)
                            : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        return;
    }
    const bool row_ok = m < a.M;
    const float *rrow = a.residual + (row_ok ? m : 0) * (int64_t)a.N;
    const bool vec = a.tma_io && n + 31 < a.N;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const int64_t n4 = n + 4 * c;
        if (vec && row_ok) {
            r[c] = *reinterpret_cast<const float4 *>(rrow + n4);
        } else {
            r[c].x = (row_ok && n4 < a.N) ? rrow[n4] : 0.f;
            r[c].y = (row_ok && n4 + 1 < a.N) ? rrow[n4 + 1] : 0.f;
            r[c].z = (row_ok && n4 + 2 < a.N) ? rrow[n4 + 2] : 0.f;
            r[c].w = (row_ok && n4 + 3 < a.N) ? rrow[n4 + 3] : 0.f;
        }
    }
}

// L2 prefetch of this thread's residual row segment for the item's `nsl`
// slices (128-byte lines), issued before the accumulator wait: the per-slice
// loads then find it in L2 instead of waiting on DRAM one slice at a time
__device__ __forceinline__ void prefetch_residual(const EpiArgs &a, int64_t m, int64_t n,
                                                  int nsl) {
    if (m >= a.M) return;
    const float *rrow = a.residual + m * (int64_t)a.N;
    for (int s = 0; s < nsl; ++s) {
        if (n + s * SLICE >= a.N) break;
        asm volatile("prefetch.global.L2 [%0];" ::"l"(rrow + n + s * SLICE));
        if (n + s * SLICE + SLICE - 1 < a.N)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(rrow + n + s * SLICE + SLICE - 1));
    }
}

// Dequantise one 32 x 32 slice and store it: this thread's row m, the 32
// consecutive columns from n.  `v` holds the exact integer sums, as fp32
// (single-chunk accumulators straight from tensor memory) or as int32
// (INT_IN: the partial of multi-chunk shapes).  The wait for this warp's
// previous TMA store to release the staging tile comes after the arithmetic,
// so the store's latency hides behind it.  Staging tile row `lane` holds this
// thread's 32 values, 16-byte chunk c at c ^ (lane & 7) (the TMA 128-byte
// swizzle: conflict-free for the warp).
template <int MODE, bool INT_IN, int OUT>
__device__ __forceinline__ void epilogue_slice(uint32_t (&v)[32], int64_t m, int64_t n,
                                               int row0, int lane, const EpiArgs &a, float xs,
                                               float wl, float bl, float2 rml, int slice_index,
                                               const float4 (&r4)[8], const CUtensorMap *tmY,
                                               uint8_t *stg, float &rmax) {
    if (n >= a.N || row0 >= a.M) return;  // slice wholly outside Y
    float4 rrow[8];  // this thread's row of the residual slice
    if (MODE == SQ_EPI_BIAS_RESIDUAL) {
        if (OUT != kOutRequant && a.tma_io && n + 31 < a.N) {
            // r4 is in the coalesced layout (load_residual<true>): through the
            // staging tile (free once the previous store has read it), written
            // row 4 c + lane / 8, read back as row `lane`, both conflict-free
            // under the 128-byte swizzle
            if (lane == 0) bulk_wait_read0();
            __syncwarp();
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const int r = 4 * c + (lane >> 3), k = lane & 7;
                *reinterpret_cast<float4 *>(stg + r * 128 + ((k ^ (r & 7)) << 4)) = r4[c];
            }
            __syncwarp();
#pragma unroll
            for (int c = 0; c < 8; ++c)
                rrow[c] = *reinterpret_cast<const float4 *>(stg + lane * 128 +
                                                            ((c ^ (lane & 7)) << 4));
        } else {
#pragma unroll
            for (int c = 0; c < 8; ++c) rrow[c] = r4[c];
        }
    }
    if (MODE == SQ_EPI_RAW_I32) {
        if (!INT_IN) {
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = (uint32_t)__float2int_rn(__uint_as_float(v[j]));
        }
    } else {
        // two columns per step on packed fp32 pairs
        const unsigned long long xs2 = pk(xs, xs);
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
            const unsigned long long w2 =
                pk(__shfl_sync(0xffffffffu, wl, j), __shfl_sync(0xffffffffu, wl, j + 1));
            // the exact integer sums as fp32 (|acc| < 2^31: one rounding at most)
            const unsigned long long x2 =
                INT_IN ? pk(__int2float_rn((int32_t)v[j]), __int2float_rn((int32_t)v[j + 1]))
                       : pk(__uint_as_float(v[j]), __uint_as_float(v[j + 1]));
            const unsigned long long sc2 = mul2(xs2, w2);
            unsigned long long o2;
            if (MODE == SQ_EPI_NONE) {
                o2 = mul2(x2, sc2);
            } else {
                const unsigned long long b2 =
                    pk(__shfl_sync(0xffffffffu, bl, j), __shfl_sync(0xffffffffu, bl, j + 1));
                const unsigned long long t2 = fma2(x2, sc2, b2);
                if (MODE == SQ_EPI_BIAS) {
                    o2 = t2;
                } else if (MODE == SQ_EPI_BIAS_GELU) {
                    o2 = gelu2(t2);
                } else {
                    const float4 rq = rrow[j >> 2];
                    o2 = add2(t2, (j & 2) ? pk(rq.z, rq.w) : pk(rq.x, rq.y));
                }
            }
            float o0, o1;
            upk(o2, o0, o1);
            v[j] = __float_as_uint(o0);
            v[j + 1] = __float_as_uint(o1);
        }
    }
    if (OUT == kOutRowMax) rmax = fmaxf(rmax, slice_rowmax(v, n, a, rml));
    if (OUT == kOutRequant) {
        // this slice's columns in the warp's staging area (written per tile)
        requant_slice(v, m, n, a, reinterpret_cast<const float4 *>(stg) + 16 * slice_index);
        return;
    }
    if (a.tma_io) {
        // the previous TMA store of this warp must have finished reading the tile
        if (lane == 0) bulk_wait_read0();
        __syncwarp();
#pragma unroll
        for (int c = 0; c < 8; ++c)
            *reinterpret_cast<uint4 *>(stg + lane * 128 + ((c ^ (lane & 7)) << 4)) =
                make_uint4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            tma_store_2d(tmY, smem_u32(stg), (int)n, row0);
            bulk_commit();
        }
    } else if (m < a.M) {
        uint32_t *y = static_cast<uint32_t *>(a.Y) + m * a.N;
#pragma unroll
        for (int j = 0; j < 32; ++j)
            if (n + j < a.N) y[n + j] = v[j];
    }
}

// The first `nsl` slices of this warp's part of a tile (all four for a full
// tile, fewer for a column slice of one), reading tensor memory at `taddr`
// (fp32 sums, or int32 with INT_IN).
template <int MODE, bool INT_IN, int OUT>
__device__ __forceinline__ void epilogue_tile(uint32_t taddr, int64_t m, int nb, int row0,
                                              int lane, const EpiArgs &a, float xs,
                                              const ColParams &cp, float4 (&rnext)[8],
                                              const CUtensorMap *tmY, uint8_t *stg, int nsl) {
    float rmax = 0.0f;  // kOutRowMax: this row's maximum over the tile's columns
#pragma unroll 1
    for (int s = 0; s < nsl; ++s) {
        float4 rcur[8];
        if (MODE == SQ_EPI_BIAS_RESIDUAL) {
#pragma unroll
            for (int c = 0; c < 8; ++c) rcur[c] = rnext[c];
            if (s + 1 < nsl) load_residual<OUT != kOutRequant>(rnext, a, m, nb + (s + 1) * SLICE);
        }
        const float wl = s == 0 ? cp.w[0] : s == 1 ? cp.w[1] : s == 2 ? cp.w[2] : cp.w[3];
        const float bl = s == 0 ? cp.b[0] : s == 1 ? cp.b[1] : s == 2 ? cp.b[2] : cp.b[3];
        const float2 rml =
            OUT != kOutRowMax ? make_float2(0.f, 0.f)
            : s == 0          ? make_float2(cp.rs[0], cp.ry[0])
            : s == 1          ? make_float2(cp.rs[1], cp.ry[1])
            : s == 2          ? make_float2(cp.rs[2], cp.ry[2])
                              : make_float2(cp.rs[3], cp.ry[3]);
        uint32_t v[32];
        tmem_ld32(taddr + s * SLICE, v);
        epilogue_slice<MODE, INT_IN, OUT>(v, m, nb + s * SLICE, row0, lane, a, xs, wl, bl, rml, s,
                                          rcur, tmY, stg, rmax);
    }
    // non-negative floats order like their bit patterns
    if (OUT == kOutRowMax && m < a.M && rmax > 0.0f)
        atomicMax(reinterpret_cast<int *>(a.row_amax) + m, __float_as_int(rmax));
}

// Bounded wait until the counter at p reaches `target` (acquire).  The pieces
// it waits for have already finished their MMAs and only have stores left, so
// the wait is short; the limit guards against a corrupted workspace.
__device__ __noinline__ bool wait_count(const int32_t *p, int target, volatile int *abort_flag) {
    const uint64_t t0 = globaltimer();
    for (uint32_t it = 1;; ++it) {
        int32_t v;
        asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
        if (v >= target) return true;
        if ((it & 63u) == 0) {
            if (*abort_flag) return false;
            if (globaltimer() - t0 > kTimeoutNs) {
                *abort_flag = 1;
                atomicOr(&g_tc_error, 4u);
                return false;
            }
        }
    }
}

// This warp's 32 x 128 sub-block of the partial slot that CTA c uses for its
// piece of the split tile starting at K-block index tb: slot 0 when the
// tile is the first of c's share, else slot 1.  Layout (int4 units):
// [slice s][column quad j][lane], so that each warp access is 512 contiguous bytes.
__device__ __forceinline__ int4 *sk_slot(const EpiArgs &a, int c, long long tb, int ew) {
    const int e = sk_start(a.sched, c) >= tb ? 0 : 1;
    return a.ws_slots + (((long long)c * 2 + e) * NUM_EPI_WARPS + ew) * (kSlotWarpBytes / 16);
}

// Split-K fixup of one warp's 32 x 128 sub-block of a piece whose exact sums
// are in tensor memory at T (fp32 when fp32_in, else int32).  Every piece but
// the last to finish writes its sums to its slot; the last one waits until
// those writes are visible, adds them to its own, puts the int32 total back at
// T, resets the tile's counters and returns true (it then runs the epilogue).
__device__ __forceinline__ bool sk_fixup(uint32_t T, bool fp32_in, const Work &t, int ew,
                                         int lane, const EpiArgs &a, volatile int *abort_flag) {
    int32_t *cnt = a.ws_cnt + ((long long)t.skt * NUM_EPI_WARPS + ew) * 2;
    const long long tb = (long long)t.skt * a.sched.nkb;
    const int c0 = sk_cta_of(a.sched, tb), c1 = sk_cta_of(a.sched, tb + a.sched.nkb - 1);
    const int pieces = c1 - c0 + 1;
    int old = 0;
    if (lane == 0) old = atomicAdd(cnt, 1);
    old = __shfl_sync(0xffffffffu, old, 0);
    if (old < pieces - 1) {
        int4 *dst = sk_slot(a, blockIdx.x, tb, ew) + lane;
#pragma unroll 1
        for (int s = 0; s < SLICES; ++s) {
            uint32_t v[32];
            tmem_ld32(T + s * SLICE, v);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                int4 q;
                q.x = fp32_in ? __float2int_rn(__uint_as_float(v[4 * j])) : (int)v[4 * j];
                q.y = fp32_in ? __float2int_rn(__uint_as_float(v[4 * j + 1])) : (int)v[4 * j + 1];
                q.z = fp32_in ? __float2int_rn(__uint_as_float(v[4 * j + 2])) : (int)v[4 * j + 2];
                q.w = fp32_in ? __float2int_rn(__uint_as_float(v[4 * j + 3])) : (int)v[4 * j + 3];
                __stcg(dst + (s * 8 + j) * 32, q);
            }
        }
        __threadfence();
        __syncwarp();
        if (lane == 0) atomicAdd(cnt + 1, 1);
        return false;
    }
    int ok = 1;
    if (lane == 0) ok = wait_count(cnt + 1, pieces - 1, abort_flag);
    if (!__shfl_sync(0xffffffffu, ok, 0)) return false;
    __threadfence();
#pragma unroll 1
    for (int s = 0; s < SLICES; ++s) {
        uint32_t v[32];
        tmem_ld32(T + s * SLICE, v);
        if (fp32_in) {
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = (uint32_t)__float2int_rn(__uint_as_float(v[j]));
        }
        // peers two at a time: 16 loads of 16 bytes in flight per lane
#pragma unroll 1
        for (int c = c0; c <= c1; c += 2) {
            const bool has0 = c != (int)blockIdx.x;
            const bool has1 = c + 1 <= c1 && c + 1 != (int)blockIdx.x;
            const int4 *src0 = sk_slot(a, has0 ? c : c1, tb, ew) + lane + s * 256;
            const int4 *src1 = sk_slot(a, has1 ? c + 1 : c0, tb, ew) + lane + s * 256;
            int4 q0[8], q1[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                q0[j] = has0 ? __ldcg(src0 + j * 32) : make_int4(0, 0, 0, 0);
                q1[j] = has1 ? __ldcg(src1 + j * 32) : make_int4(0, 0, 0, 0);
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                v[4 * j] = (uint32_t)((int32_t)v[4 * j] + q0[j].x + q1[j].x);
                v[4 * j + 1] = (uint32_t)((int32_t)v[4 * j + 1] + q0[j].y + q1[j].y);
                v[4 * j + 2] = (uint32_t)((int32_t)v[4 * j + 2] + q0[j].z + q1[j].z);
                v[4 * j + 3] = (uint32_t)((int32_t)v[4 * j + 3] + q0[j].w + q1[j].w);
            }
        }
        tmem_st32(T + s * SLICE, v);
    }
    tmem_wait_st();
    __syncwarp();
    if (lane == 0) {
        cnt[0] = 0;
        cnt[1] = 0;
    }
    return true;
}

// K blocks per exact fp32 pass: 16 (K = 1024), or all of K when the row L1
// norms of either operand bound every partial sum below 2^24.  Decided by
// warps 1..9 (the MMA issuer and the epilogue) through named barrier 1; the
// producer (warp 0) does not need it and returns 16.
__device__ __forceinline__ int exact_pass_kb(const EpiArgs &args, int nkb, int warp, int lane,
                                             int32_t (*l1max)[2]) {
    if (warp == 0 || nkb <= KB_PER_CHUNK || !(args.x_l1 || args.w_l1)) return KB_PER_CHUNK;
    const int tid = threadIdx.x - 32;
    int32_t mx = args.x_l1 ? 0 : 0x7fffffff, mw = args.w_l1 ? 0 : 0x7fffffff;
    if (args.x_l1)
        for (int i = tid; i < args.M; i += THREADS - 32) mx = max(mx, __ldg(args.x_l1 + i));
    if (args.w_l1)
        for (int i = tid; i < args.N; i += THREADS - 32) mw = max(mw, __ldg(args.w_l1 + i));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        mw = max(mw, __shfl_xor_sync(0xffffffffu, mw, o));
    }
    if (lane == 0) {
        l1max[warp - 1][0] = mx;
        l1max[warp - 1][1] = mw;
    }
    asm volatile("bar.sync 1, %0;" ::"n"(THREADS - 32) : "memory");
    mx = 0;
    mw = 0;
    for (int w = 0; w < 9; ++w) {
        mx = max(mx, l1max[w][0]);
        mw = max(mw, l1max[w][1]);
    }
    return min(mx, mw) <= kSinglePassL1 ? nkb : KB_PER_CHUNK;
}

template <int MODE, int OUT>
__global__ void __launch_bounds__(THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmBs, const __grid_constant__ CUtensorMap tmY,
                   const EpiArgs args, int K) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *staging = smem + RING_BYTES;
    Smem &S = *reinterpret_cast<Smem *>(staging + NUM_EPI_WARPS * STG_BYTES);
    const uint32_t ring = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int M = args.M;

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
    pdl_launch_dependents();
    pdl_wait();  // every global-memory access below follows the previous kernel
    const uint32_t tmem_base = S.tmem_base;
    volatile int *abort_flag = &S.abort_flag;

    const Schedule &sched = args.sched;
    const int nkb = sched.nkb;
    // K per exact fp32 pass: 1024, or all of K when the row L1 norms of either
    // operand bound every partial sum below 2^24.  Decided by warps 1..9 (the
    // MMA issuer and the epilogue); the producer does not need it.
    const int chunk_kb = exact_pass_kb(args, nkb, warp, lane, S.l1max);
    const int nchunks = (nkb + chunk_kb - 1) / chunk_kb;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued = 0, fill_parity = 0;  // per-stage bits: loads in flight
            Cursor cu;
            cursor_init(sched, cu, blockIdx.x);
            Work t;
            while (next_work(sched, cu, t, gridDim.x)) {
                const bool slice = t.bn < BN;
                for (int kb = t.kb0; kb < t.kb1; ++kb) {
                    if (!mbar_wait(smem_u32(&S.empty[stage]), phase ^ 1, abort_flag)) goto done_p;
                    const uint32_t full = smem_u32(&S.full[stage]);
                    mbar_expect_tx(full, A_BYTES + t.bn * BK * 2);
                    const uint32_t sa = ring + stage * STAGE_BYTES;
                    tma_load_2d(sa, &tmA, full, kb * BK, t.m0);
                    tma_load_2d(sa + A_BYTES, slice ? &tmBs : &tmB, full, kb * BK, t.n0);
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
            uint32_t phase = 0, tph = 0;  // tph: per-buffer use parity bits
            bool issued_any = false;
            Cursor cu;
            cursor_init(sched, cu, blockIdx.x);
            Work t;
            for (int it = 0; next_work(sched, cu, t, gridDim.x); ++it) {
                const uint32_t idesc = idesc_for(t.bn);
                // exact fp32 passes: the unit's K blocks cut at multiples of chunk_kb
                for (int c = t.kb0 / chunk_kb; c * chunk_kb < t.kb1; ++c) {
                    const uint32_t b = nchunks == 1 ? (uint32_t)(it & 1) : 0u;
                    const uint32_t par = (tph >> b) & 1u;
                    if (!mbar_wait(smem_u32(&S.tempty[b]), par ^ 1, abort_flag)) goto done_m;
                    tph ^= 1u << b;
                    tc_fence_after();
                    const uint32_t d = tmem_base + b * BN;
                    const int kb0 = max(t.kb0, c * chunk_kb);
                    const int kb1 = min(t.kb1, (c + 1) * chunk_kb);
                    for (int kb = kb0; kb < kb1; ++kb) {
                        if (!mbar_wait(smem_u32(&S.full[stage]), phase, abort_flag)) goto done_m;
                        tc_fence_after();
                        const uint32_t sa = ring + stage * STAGE_BYTES;
                        const uint64_t adesc = sw128_desc(sa);
                        const uint64_t bdesc = sw128_desc(sa + A_BYTES);
#pragma unroll
                        for (int k = 0; k < BK / UMMA_K; ++k) {
                            // advance 16 bf16 = 32 bytes along K inside the swizzled row
                            umma_bf16(d, adesc + 2 * k, bdesc + 2 * k, idesc,
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
        const int ew = warp - 2;
        const int q = warp & 3;            // TMEM lane quarter this warp may access
        const int half = ew >> 2;          // which 128 of the 256 columns
        uint8_t *stg = staging + ew * STG_BYTES;
        uint32_t fph = 0;                  // accumulator-full parities
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        const uint32_t colP = BN;          // int32 partial (multi-chunk shapes)
        Cursor cu;
        cursor_init(sched, cu, blockIdx.x);
        Work t;
        for (int it = 0; next_work(sched, cu, t, gridDim.x); ++it) {
            const int row0 = t.m0 + q * 32;
            const int64_t m = (int64_t)row0 + lane;
            const int nb = t.n0 + half * COLS_PER_WARP;
            // 32-column slices of this warp's half that the unit covers (0..4)
            const int nsl = max(0, min(SLICES, (t.bn - half * COLS_PER_WARP) / SLICE));
            const bool piece = t.skt >= 0;
            // operands that do not depend on the accumulators: fetched before the
            // accumulator wait, so that their latency hides (a split-K piece
            // fetches them only once it is the one that finishes the tile)
            ColParams cp;
            float xs = 0.f;
            float4 rnext[8];
            auto fetch = [&]() {
                load_col_params<MODE, OUT>(cp, args, nb, lane);
                if (OUT == kOutRequant) stage_next_smoothing(stg, args, nb, lane);
                if (OUT == kOutRequant && args.rq.x_scale && t.n0 == 0 && half == 0 && m < M)
                    args.rq.x_scale[m] = args.rq.scale;  // the next linear's per-token scales
                xs = (MODE != SQ_EPI_RAW_I32 && m < M) ? __ldg(args.sx + m) : 0.f;
                if (MODE == SQ_EPI_BIAS_RESIDUAL && nsl > 0) {
                    prefetch_residual(args, m, nb, nsl);
                    load_residual<OUT != kOutRequant>(rnext, args, m, nb);
                }
            };
            if (!piece) fetch();
            // the unit's exact sums: fp32 in accumulator buffer b (one pass), or
            // int32 in the partial P (chunk passes)
            const uint32_t b = (uint32_t)(it & 1);
            uint32_t T;
            if (nchunks == 1) {
                if (!mbar_wait(smem_u32(&S.tfull[b]), (fph >> b) & 1u, abort_flag)) goto done_e;
                fph ^= 1u << b;
                tc_fence_after();
                T = tmem_base + lane_off + b * BN + half * COLS_PER_WARP;
            } else {
                const uint32_t tA = tmem_base + lane_off + half * COLS_PER_WARP;
                T = tmem_base + lane_off + colP + half * COLS_PER_WARP;
                const int cfirst = t.kb0 / chunk_kb;
                for (int c = cfirst; c * chunk_kb < t.kb1; ++c) {
                    if (!mbar_wait(smem_u32(&S.tfull[0]), fph & 1u, abort_flag)) goto done_e;
                    fph ^= 1u;
                    tc_fence_after();
#pragma unroll 1
                    for (int s = 0; s < nsl; ++s) {
                        uint32_t v[32];
                        tmem_ld32(tA + s * SLICE, v);
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            v[j] = (uint32_t)__float2int_rn(__uint_as_float(v[j]));
                        if (c > cfirst) {
                            uint32_t p[32];
                            tmem_ld32(T + s * SLICE, p);
#pragma unroll
                            for (int j = 0; j < 32; ++j) v[j] = (uint32_t)((int32_t)v[j] + (int32_t)p[j]);
                        }
                        tmem_st32(T + s * SLICE, v);
                    }
                    tmem_wait_st();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&S.tempty[0]));
                }
            }
            // epilogue (the int32 partial's final pass overlaps the next unit's MMAs)
            if (!piece) {
                if (nchunks == 1)
                    epilogue_tile<MODE, false, OUT>(T, m, nb, row0, lane, args, xs, cp, rnext,
                                                      &tmY, stg, nsl);
                else
                    epilogue_tile<MODE, true, OUT>(T, m, nb, row0, lane, args, xs, cp, rnext,
                                                     &tmY, stg, nsl);
            } else if (sk_fixup(T, nchunks == 1, t, ew, lane, args, abort_flag)) {
                fetch();
                epilogue_tile<MODE, true, OUT>(T, m, nb, row0, lane, args, xs, cp, rnext, &tmY,
                                                 stg, nsl);
            } else if (*abort_flag) {
                goto done_e;
            }
            if (nchunks == 1) {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&S.tempty[b]));
            }
        }
    done_e:
        if (lane == 0) bulk_wait0();  // stores complete before the CTA exits
        __syncwarp();
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

// ---------------------------------------------------------- pair kernel
//
// The same contraction and epilogue on CTA pairs (clusters of 2) with
// tcgen05.mma.cta_group::2, M = 256, N = 256: the pair's two SMs share one
// 256 x 256 output tile, each holding its 128 rows of A and 128 of the 256 rows
// of B in shared memory and its 128 x 256 accumulators in its own tensor
// memory.  Per K block an SM then takes in 32 KB instead of 48 KB, and its
// shared memory serves 32 KB to the tensor cores instead of 48 KB: the
// one-CTA kernel is bound by that shared-memory traffic (the TMA writing each
// stage and the MMA reading it), not by the tensor cores.  The 32 KB stage
// also lets the ring hold 6 stages.
//   both CTAs, warp 0 lane 0: load their halves into their own ring; the
//     copies complete on the leader's (rank 0) `full` barrier, which the
//     leader alone arms, locally, with both halves' bytes;
//   leader, warp 1 lane 0: the MMAs; their commits arrive on `empty`, `tfull`
//     and `mma_done` of both CTAs (multicast);
//   both CTAs, warps 2..9: the epilogue of their own 128 rows, as in the
//     one-CTA kernel; they release an accumulator on the leader's `tempty`.
constexpr int PAIR_STAGES = 6;
constexpr int PAIR_B_ROWS = BN / 2;
constexpr int PAIR_STAGE_BYTES = A_BYTES + PAIR_B_ROWS * BK * 2;
constexpr int PAIR_RING_BYTES = PAIR_STAGES * PAIR_STAGE_BYTES;
constexpr int PAIR_SMEM_BYTES = PAIR_RING_BYTES + NUM_EPI_WARPS * STG_BYTES + BAR_BYTES + 1024;
__host__ __device__ constexpr uint32_t idesc_pair(int n) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) |
           ((uint32_t)((2 * BM) >> 4) << 24);
}

struct PairSmem {
    uint64_t full[PAIR_STAGES];
    uint64_t empty[PAIR_STAGES];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t mma_done;
    uint32_t tmem_base;
    int abort_flag;
    int32_t l1max[9][2];
};
static_assert(sizeof(PairSmem) <= BAR_BYTES, "barrier block");

template <int MODE, int OUT>
__global__ void __launch_bounds__(THREADS, 1)
    gemm_tc_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmBq,
                        const __grid_constant__ CUtensorMap tmY, const EpiArgs args, int K) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *staging = smem + PAIR_RING_BYTES;
    PairSmem &S = *reinterpret_cast<PairSmem *>(staging + NUM_EPI_WARPS * STG_BYTES);
    const uint32_t ring = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int M = args.M, N = args.N;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < PAIR_STAGES; ++s) {
            mbar_init(smem_u32(&S.full[s]), 1);   // the leader's arming arrive (+ both halves' bytes)
            mbar_init(smem_u32(&S.empty[s]), 1);  // one multicast commit per phase
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&S.tfull[b]), 1);
            mbar_init(smem_u32(&S.tempty[b]), 2 * NUM_EPI_WARPS);  // both CTAs' epilogues
        }
        mbar_init(smem_u32(&S.mma_done), 1);
        S.abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&S.tmem_base)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // barriers of both CTAs initialised before any remote arrive
    tc_fence_after();
    pdl_wait();  // every global-memory access below follows the previous kernel
    const uint32_t tmem_base = S.tmem_base;
    volatile int *abort_flag = &S.abort_flag;

    const int cluster_id = blockIdx.x >> 1;
    const int num_clusters = gridDim.x >> 1;
    const PairSchedule sched =
        make_pair_schedule((M + 2 * BM - 1) / (2 * BM), (N + BN - 1) / BN, args.pair_plan);
    const int num_items = sched.items;
    const int nkb = (K + BK - 1) / BK;
    const int chunk_kb = exact_pass_kb(args, nkb, warp, lane, S.l1max);
    const int nchunks = (nkb + chunk_kb - 1) / chunk_kb;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer (both CTAs)
            int stage = 0;
            uint32_t phase = 0;
            for (int i = cluster_id; i < num_items; i += num_clusters) {
                int pm0, n0, bn;
                pair_item_at(sched, i, pm0, n0, bn);
                const int m0 = pm0 + (int)rank * BM;
                const int nB = n0 + (int)rank * (bn / 2);  // this CTA's rows of B
                const CUtensorMap *mapB = bn == BN ? &tmB : &tmBq;
                const uint32_t bytes = A_BYTES + (bn / 2) * BK * 2;
                for (int kb = 0; kb < nkb; ++kb) {
                    if (!mbar_wait(smem_u32(&S.empty[stage]), phase ^ 1, abort_flag)) goto done_p;
                    const uint32_t full_leader = map_to_rank(smem_u32(&S.full[stage]), 0);
                    if (leader) mbar_expect_tx(smem_u32(&S.full[stage]), 2 * bytes);
                    const uint32_t sa = ring + stage * PAIR_STAGE_BYTES;
                    tma_load_2d_pair(sa, &tmA, full_leader, kb * BK, m0);
                    tma_load_2d_pair(sa + A_BYTES, mapB, full_leader, kb * BK, nB);
                    if (++stage == PAIR_STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
            // the next kernel may be scheduled once every CTA has issued its last
            // copies (it still waits for this grid to complete before reading
            // memory): measured 784 -> 788 TOPS against triggering at the start
            pdl_launch_dependents();
        done_p:
            // every issued copy is consumed by the leader's MMAs, whose commits
            // complete this CTA's `empty` phases: wait (bounded) for the stages
            // still in use before the shared memory can go away
            for (int s = 0; s < PAIR_STAGES; ++s) {
                mbar_drain(smem_u32(&S.empty[stage]), phase ^ 1);
                if (++stage == PAIR_STAGES) {
                    stage = 0;
                    phase ^= 1;
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            // ------------------------------------------------ MMA issuer (leader)
            int stage = 0;
            uint32_t phase = 0, tph = 0;
            int it = 0;
            for (int i = cluster_id; i < num_items; i += num_clusters, ++it) {
                int pm0, n0, bn;
                pair_item_at(sched, i, pm0, n0, bn);
                const uint32_t idesc = idesc_pair(bn);
                for (int c = 0; c < nchunks; ++c) {
                    const uint32_t b = nchunks == 1 ? (uint32_t)(it & 1) : 0u;
                    const uint32_t par = (tph >> b) & 1u;
                    if (!mbar_wait(smem_u32(&S.tempty[b]), par ^ 1, abort_flag)) goto done_m;
                    tph ^= 1u << b;
                    tc_fence_after();
                    const uint32_t d = tmem_base + b * BN;
                    const int kb0 = c * chunk_kb;
                    const int kb1 = min(nkb, kb0 + chunk_kb);
                    for (int kb = kb0; kb < kb1; ++kb) {
                        if (!mbar_wait(smem_u32(&S.full[stage]), phase, abort_flag)) goto done_m;
                        tc_fence_after();
                        const uint32_t sa = ring + stage * PAIR_STAGE_BYTES;
                        const uint64_t adesc = sw128_desc(sa);
                        const uint64_t bdesc = sw128_desc(sa + A_BYTES);
#pragma unroll
                        for (int k = 0; k < BK / UMMA_K; ++k)
                            umma_bf16_pair(d, adesc + 2 * k, bdesc + 2 * k, idesc,
                                           (kb > kb0 || k > 0) ? 1u : 0u);
                        umma_commit_pair(smem_u32(&S.empty[stage]));
                        if (++stage == PAIR_STAGES) {
                            stage = 0;
                            phase ^= 1;
                        }
                    }
                    umma_commit_pair(smem_u32(&S.tfull[b]));
                }
            }
        done_m:
            // arrives on both CTAs once every MMA issued above has completed
            umma_commit_pair(smem_u32(&S.mma_done));
        }
        // no CTA frees its tensor memory while the pair's MMAs may still write it
        if (lane == 0) mbar_drain(smem_u32(&S.mma_done), 0);
        __syncwarp();
    } else {
        // ---------------------------------------------------- epilogue (both CTAs)
        const int ew = warp - 2;
        const int q = warp & 3;
        const int half = ew >> 2;
        uint8_t *stg = staging + ew * STG_BYTES;
        uint32_t fph = 0;
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        const uint32_t colP = BN;
        const uint32_t tempty_leader0 = map_to_rank(smem_u32(&S.tempty[0]), 0);
        const uint32_t tempty_leader1 = map_to_rank(smem_u32(&S.tempty[1]), 0);
        int it = 0;
        for (int i = cluster_id; i < num_items; i += num_clusters, ++it) {
            int pm0, n0, bn;
            pair_item_at(sched, i, pm0, n0, bn);
            const int m0 = pm0 + (int)rank * BM;
            const int row0 = m0 + q * 32;
            const int64_t m = (int64_t)row0 + lane;
            // the two warps of a lane quarter split the item's columns: 128 each
            // of a whole tile, 64 each of a half (all eight warps busy either way)
            const int wcols = bn / 2;
            const int nb = n0 + half * wcols;
            const int nsl = wcols / SLICE;  // 32-column slices of this warp (4 or 2)
            ColParams cp;
            load_col_params<MODE, OUT>(cp, args, nb, lane);
            if (OUT == kOutRequant) stage_next_smoothing(stg, args, nb, lane);
            if (OUT == kOutRequant && args.rq.x_scale && n0 == 0 && half == 0 && m < M)
                args.rq.x_scale[m] = args.rq.scale;
            const float xs = (MODE != SQ_EPI_RAW_I32 && m < M) ? __ldg(args.sx + m) : 0.f;
            float4 rnext[8];
            if (MODE == SQ_EPI_BIAS_RESIDUAL && nsl > 0) {
                prefetch_residual(args, m, nb, nsl);
                load_residual<OUT != kOutRequant>(rnext, args, m, nb);
            }
            if (nchunks == 1) {
                const uint32_t b = (uint32_t)(it & 1);
                if (!mbar_wait(smem_u32(&S.tfull[b]), (fph >> b) & 1u, abort_flag)) goto done_e;
                fph ^= 1u << b;
                tc_fence_after();
                const uint32_t tA = tmem_base + lane_off + b * BN + half * wcols;
                epilogue_tile<MODE, false, OUT>(tA, m, nb, row0, lane, args, xs, cp, rnext, &tmY,
                                                  stg, nsl);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(b ? tempty_leader1 : tempty_leader0);
            } else {
                const uint32_t tA = tmem_base + lane_off + half * wcols;
                // the int32 partial stays in this warp's own 128 columns whatever
                // the item's width: the quarter's other warp may still be reading
                // its partial of the previous item when this one starts the next
                const uint32_t tP = tmem_base + lane_off + colP + half * COLS_PER_WARP;
                for (int c = 0; c < nchunks; ++c) {
                    if (!mbar_wait(smem_u32(&S.tfull[0]), fph & 1u, abort_flag)) goto done_e;
                    fph ^= 1u;
                    tc_fence_after();
#pragma unroll 1
                    for (int s = 0; s < nsl; ++s) {
                        uint32_t v[32];
                        tmem_ld32(tA + s * SLICE, v);
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            v[j] = (uint32_t)__float2int_rn(__uint_as_float(v[j]));
                        if (c > 0) {
                            uint32_t p[32];
                            tmem_ld32(tP + s * SLICE, p);
#pragma unroll
                            for (int j = 0; j < 32; ++j) v[j] = (uint32_t)((int32_t)v[j] + (int32_t)p[j]);
                        }
                        tmem_st32(tP + s * SLICE, v);
                    }
                    tmem_wait_st();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster(tempty_leader0);
                }
                epilogue_tile<MODE, true, OUT>(tP, m, nb, row0, lane, args, xs, cp, rnext, &tmY,
                                                 stg, nsl);
            }
        }
    done_e:
        if (lane == 0) bulk_wait0();  // stores complete before the CTA exits
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // no remote arrive, copy or MMA touches either CTA after this
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
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

// 2-D row-major tensor of `rows` x `cols` elements, box box_rows x box_cols,
// 128-byte swizzle (the box's inner extent is 128 bytes).
sq_status make_map(CUtensorMap *map, CUtensorMapDataType dt, int esize, const void *base,
                   int64_t rows, int64_t cols, int box_rows, int box_cols) {
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * esize};
    cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, dt, 2, const_cast<void *>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? SQ_OK : SQ_ERR_CUDA;
}

// One-time set-up of a kernel on each device (its dynamic shared-memory
// attribute and, for the pair kernel, how many clusters fit at once), done
// under a lock so that host threads launching at once see it complete.
constexpr int kMaxDevices = 64;  // device_info rejects higher ordinals
struct KernelSetup {
    std::mutex mu;
    bool done[kMaxDevices] = {};
    int clusters[kMaxDevices] = {};
};

template <typename Kern>
sq_status setup_kernel(KernelSetup &ks, Kern kern, int smem_bytes, int device,
                       const cudaLaunchConfig_t *pair_cfg, int *clusters) {
    if (device < 0 || device >= kMaxDevices) return SQ_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(ks.mu);
    if (!ks.done[device]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 smem_bytes) != cudaSuccess)
            return SQ_ERR_CUDA;
        if (pair_cfg) {
            int n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, kern, pair_cfg) != cudaSuccess || n < 1)
                return SQ_ERR_CUDA;
            ks.clusters[device] = n;
        }
        ks.done[device] = true;
    }
    if (clusters) *clusters = ks.clusters[device];
    return SQ_OK;
}

template <int MODE, int OUT>
sq_status launch_kernel(const CUtensorMap &ta, const CUtensorMap &tb, const CUtensorMap &tbs,
                        const CUtensorMap &ty, const EpiArgs &args, int K, int grid, int device,
                        cudaStream_t st) {
    static KernelSetup ks;
    sq_status rc = setup_kernel(ks, gemm_tc_kernel<MODE, OUT>, SMEM_BYTES, device, nullptr,
                                nullptr);
    if (rc != SQ_OK) return rc;
    return launch_pdl(gemm_tc_kernel<MODE, OUT>, dim3(grid), dim3(THREADS), SMEM_BYTES, st, 1, ta,
                      tb, tbs, ty, args, K);
}

template <int MODE>
sq_status launch_mode(const CUtensorMap &ta, const CUtensorMap &tb, const CUtensorMap &tbs,
                      const CUtensorMap &ty, const EpiArgs &args, int K, int grid, int device,
                      int out, cudaStream_t st) {
    if (out == kOutRequant)
        return launch_kernel<MODE, kOutRequant>(ta, tb, tbs, ty, args, K, grid, device, st);
    if (out == kOutRowMax)
        return launch_kernel<MODE, kOutRowMax>(ta, tb, tbs, ty, args, K, grid, device, st);
    return launch_kernel<MODE, kOutPlain>(ta, tb, tbs, ty, args, K, grid, device, st);
}

// The pair kernel on clusters of 2: at most one cluster per pair tile and no
// more than can be resident at once (it is persistent).
template <int MODE, int OUT>
sq_status launch_pair_kernel(const CUtensorMap &ta, const CUtensorMap &tbp, const CUtensorMap &tbq,
                             const CUtensorMap &ty, const EpiArgs &args, int K, int device,
                             cudaStream_t st) {
    static KernelSetup ks;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(THREADS, 1, 1);
    cfg.dynamicSmemBytes = PAIR_SMEM_BYTES;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;  // the occupancy query: cluster shape only
    cfg.gridDim = dim3(2, 1, 1);
    int max_clusters = 0;
    sq_status rc = setup_kernel(ks, gemm_tc_pair_kernel<MODE, OUT>, PAIR_SMEM_BYTES, device,
                                &cfg, &max_clusters);
    if (rc != SQ_OK) return rc;
    // the schedule is planned for every cluster that fits; the grid holds no
    // more clusters than it has items (the kernel strides by the grid's count)
    EpiArgs a = args;
    a.pair_plan = max_clusters;
    const PairSchedule ps = make_pair_schedule((args.M + 2 * BM - 1) / (2 * BM),
                                               (args.N + BN - 1) / BN, max_clusters);
    const int clusters = std::min(ps.items, max_clusters);
    cfg.gridDim = dim3((unsigned)(2 * clusters), 1, 1);
    cfg.numAttrs = 2;  // the launch: cluster shape and programmatic serialisation
    return cuda_status(
        cudaLaunchKernelEx(&cfg, gemm_tc_pair_kernel<MODE, OUT>, ta, tbp, tbq, ty, a, K));
}

template <int MODE>
sq_status launch_pair_mode(const CUtensorMap &ta, const CUtensorMap &tbp, const CUtensorMap &tbq,
                           const CUtensorMap &ty, const EpiArgs &args, int K, int device,
                           int out, cudaStream_t st) {
    if (out == kOutRequant)
        return launch_pair_kernel<MODE, kOutRequant>(ta, tbp, tbq, ty, args, K, device,
                                                     st);
    if (out == kOutRowMax)
        return launch_pair_kernel<MODE, kOutRowMax>(ta, tbp, tbq, ty, args, K, device,
                                                    st);
    return launch_pair_kernel<MODE, kOutPlain>(ta, tbp, tbq, ty, args, K, device, st);
}

// Which kernel runs a launch: CTA pairs for every launch of at least one full
// 256-row pair tile that is not split over K.
bool use_pair(int64_t M, const Schedule &sched) {
    return sched.sk_tiles == 0 && M >= 2 * BM;
}

}  // namespace

static bool shape_ok(int64_t M, int64_t N, int64_t K) {
    if (M <= 0 || N <= 0 || K <= 0 || M > 0x7fffffff || N > 0x7fffffff || K > 0x7fffffff)
        return false;
    return ((M + BM - 1) / BM) * ((N + BN - 1) / BN) <= 0x7fffffff;
}

sq_status gemm_tc_workspace_bytes(int64_t M, int64_t N, int64_t K, size_t *bytes) {
    *bytes = 0;
    if (M == 0 || N == 0) return SQ_OK;
    if (!shape_ok(M, N, K)) return SQ_ERR_UNSUPPORTED;
    DeviceInfo di;
    sq_status rc = device_info(&di);
    if (rc != SQ_OK) return rc;
    int grid;
    *bytes = (size_t)sk_workspace_bytes(plan_launch(M, N, K, di.sms, true, &grid));
    return SQ_OK;
}

sq_status make_map_f32(void *map, const float *base, int64_t rows, int64_t cols, int box_rows,
                       int box_cols) {
    sq_status rc = get_encoder();
    if (rc != SQ_OK) return rc;
    return make_map(static_cast<CUtensorMap *>(map), CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, base,
                    rows, cols, box_rows, box_cols);
}

sq_status launch_gemm_tc(const __nv_bfloat16 *Xop, const float *sx, const int32_t *x_l1,
                         const __nv_bfloat16 *Wop, const float *sw, const int32_t *w_l1,
                         const float *bias, const float *residual, int64_t M, int64_t N,
                         int64_t K, int mode, void *Y, const RequantOut *rq, void *workspace,
                         size_t workspace_bytes, cudaStream_t st, const float *rm_pairs,
                         float *row_amax) {
    if (!shape_ok(M, N, K)) return SQ_ERR_UNSUPPORTED;
    if ((rq || row_amax) && mode == SQ_EPI_RAW_I32) return SQ_ERR_INVALID_ARG;
    if (rq && row_amax) return SQ_ERR_INVALID_ARG;
    sq_status rc = get_encoder();
    if (rc != SQ_OK) return rc;
    DeviceInfo di;
    if ((rc = device_info(&di)) != SQ_OK) return rc;
    EpiArgs args;
    args.sx = sx;
    args.sw = sw;
    args.bias = bias;
    args.residual = residual;
    args.x_l1 = x_l1;
    args.w_l1 = w_l1;
    args.Y = Y;
    args.M = (int)M;
    args.N = (int)N;
    // TMA staging for Y (and the residual) needs 16-byte rows and aligned bases;
    // the vector loads of the scales and bias need them aligned too
    args.tma_io = (N % 4 == 0) && (rq || aligned16(Y)) &&
                  (mode == SQ_EPI_RAW_I32 || aligned16(sw)) &&
                  (bias == nullptr || aligned16(bias)) &&
                  (residual == nullptr || aligned16(residual));
    args.rq = rq ? *rq : RequantOut{};
    args.rq_vec = rq && N % 16 == 0 && (!rq->Yq || aligned16(rq->Yq)) &&
                  (!rq->Yop || aligned16(rq->Yop));
    args.rq_fast = rq && rq->scale >= 0x1p-70f;
    args.rm_pairs = reinterpret_cast<const float4 *>(rm_pairs);
    args.row_amax = row_amax;
    CUtensorMap ta, tb, tbs, ty;
    if ((rc = make_map(&ta, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, Xop, M, K, BM, BK)) != SQ_OK)
        return rc;
    if ((rc = make_map(&tb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, Wop, N, K, BN, BK)) != SQ_OK)
        return rc;
    int grid;
    const Schedule sched = plan_launch(M, N, K, di.sms, workspace != nullptr, &grid);
    args.sched = sched;
    args.ws_cnt = nullptr;
    args.ws_slots = nullptr;
    if (sched.sk_tiles > 0) {
        const long long need = sk_workspace_bytes(sched);
        if ((long long)workspace_bytes < need || !aligned16(workspace)) return SQ_ERR_INVALID_ARG;
        args.ws_cnt = static_cast<int32_t *>(workspace);
        args.ws_slots = reinterpret_cast<int4 *>(static_cast<char *>(workspace) +
                                                 sk_counter_bytes(sched));
    }
    // B box of the column slices of the last wave's tiles (see make_schedule)
    tbs = tb;
    if (sched.sub > 1 &&
        (rc = make_map(&tbs, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, Wop, N, K, BN / sched.sub, BK)) !=
            SQ_OK)
        return rc;
    ty = ta;  // unused placeholder unless Y is stored through TMA
    if (args.tma_io && !rq) {
        const CUtensorMapDataType yt = mode == SQ_EPI_RAW_I32 ? CU_TENSOR_MAP_DATA_TYPE_INT32
                                                              : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
        if ((rc = make_map(&ty, yt, 4, Y, M, N, SLICE, SLICE)) != SQ_OK) return rc;
    }
    const int q = rq ? kOutRequant : row_amax ? kOutRowMax : kOutPlain;
    const int k = (int)K, dev = di.device;
    if (use_pair(M, sched)) {
        // B in 128-row halves, one per CTA of a pair; 64-row quarters for the
        // halves of a short last wave
        CUtensorMap tbp, tbq;
        if ((rc = make_map(&tbp, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, Wop, N, K, PAIR_B_ROWS, BK)) !=
                SQ_OK ||
            (rc = make_map(&tbq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, Wop, N, K, PAIR_B_ROWS / 2,
                           BK)) != SQ_OK)
            return rc;
        // the pair schedule counts its tiles (and twice that in halves) in int
        if (((M + 2 * BM - 1) / (2 * BM)) * ((N + BN - 1) / BN) > 0x3fffffff)
            return SQ_ERR_UNSUPPORTED;
        switch (mode) {
        case SQ_EPI_NONE:
            return launch_pair_mode<SQ_EPI_NONE>(ta, tbp, tbq, ty, args, k, dev, q, st);
        case SQ_EPI_BIAS:
            return launch_pair_mode<SQ_EPI_BIAS>(ta, tbp, tbq, ty, args, k, dev, q, st);
        case SQ_EPI_BIAS_GELU:
            return launch_pair_mode<SQ_EPI_BIAS_GELU>(ta, tbp, tbq, ty, args, k, dev, q, st);
        case SQ_EPI_BIAS_RESIDUAL:
            return launch_pair_mode<SQ_EPI_BIAS_RESIDUAL>(ta, tbp, tbq, ty, args, k, dev, q, st);
        default:
            return launch_pair_kernel<SQ_EPI_RAW_I32, kOutPlain>(ta, tbp, tbq, ty, args, k, dev,
                                                                 st);
        }
    }
    switch (mode) {
    case SQ_EPI_NONE: return launch_mode<SQ_EPI_NONE>(ta, tb, tbs, ty, args, k, grid, dev, q, st);
    case SQ_EPI_BIAS: return launch_mode<SQ_EPI_BIAS>(ta, tb, tbs, ty, args, k, grid, dev, q, st);
    case SQ_EPI_BIAS_GELU:
        return launch_mode<SQ_EPI_BIAS_GELU>(ta, tb, tbs, ty, args, k, grid, dev, q, st);
    case SQ_EPI_BIAS_RESIDUAL:
        return launch_mode<SQ_EPI_BIAS_RESIDUAL>(ta, tb, tbs, ty, args, k, grid, dev, q, st);
    default:
        return launch_kernel<SQ_EPI_RAW_I32, kOutPlain>(ta, tb, tbs, ty, args, k, grid, dev, st);
    }
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

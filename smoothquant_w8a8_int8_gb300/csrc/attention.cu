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
// Work unit: one (sequence, head, tile of 128 queries); S a multiple of 64, at
// most 448 (the logits of a query tile live in tensor memory: S columns, plus
// 64 for O).  Persistent: one CTA per SM (the shared memory allows no second)
// takes units blockIdx.x, + gridDim.x, ..., every barrier's phase running on
// across them; a unit's P V waits until the previous epilogue has read O
// (o_empty).  Roles (448 threads):
//   warps 0-3, 10-13  softmax and epilogue, two warps per tensor-memory lane
//              quarter (query rows), each taking 32 of every chunk's 64 keys:
//              the exact row maximum over all S logits (the two halves'
//              maxima combined through shared memory), then exp2((s - max) *
//              scale * log2 e) chunk by chunk as the split A operand of P V,
//              and finally O / sum (the two halves' sums added), each warp
//              storing half of O's columns;
//   warp 9     lane 0 copies the raw fp32 operands with TMA (64-row x 32-column
//              boxes, 128-byte swizzle): the Q tile and each K chunk (64 keys)
//              straight into the layout of their tf32 "hi" parts, each V chunk
//              into the "lo" half of its slot;
//   warps 4-7  split them into hi / lo tf32 parts in shared memory (K-major,
//              128-byte swizzle): Q and K in place (hi over the raw value, lo
//              beside it), V transposed so that keys run along K (every warp
//              reads its share of the raw chunk before any writes);
//   warp 8     tensor memory, and lane 0 issues the MMAs:
//              S[:, 64c..] = Q K_c^T, then O += P_c V_c.
// Where P lives (the template's TP):
//  * S <= 256 (TP): in tensor memory.  The softmax writes P's high part over
//    the S chunk it has just read and its low part into one of two 64-column
//    buffers (columns 320 and 384; O at 256), and the P V MMAs take A from
//    tensor memory.  Shared memory then holds only Q and four 32 KB chunk slots
//    that K and V chunks take in turn, so the next unit's Q tile is copied as
//    soon as this unit's logits are complete and its K chunks as slots free up
//    during this unit's P V: copies, splitting and logits of the next unit
//    overlap this unit's softmax (measured on GB300 at B = 32, S = 256, H = 16:
//    105 us, against 136 us with P in shared memory and 138 us with one CTA
//    per unit).  Slots 2p and 2p + 1 share a region in which their K chunks
//    form one 128-row operand, so the logits of two chunks take one N = 128
//    MMA group instead of two N = 64 ones (105 -> 97 us).
//  * S > 256: in shared memory, double-buffered: the first buffer over slots
//    2-3 (which take K chunks only, so that four are in flight), the second
//    over the Q tile (dead once the logits are complete); a unit's copies then
//    wait until the previous unit's P V products are complete (pv_done).
// A query tile that runs past its sequence (S % 128 == 64) copies the next
// rows of the input (or zeros past its end) into its unused query rows; their
// outputs are not stored and no other row reads them.
// Every wait is bounded (about 4 s); on expiry the CTA records an error for
// sq_device_status, lets its MMAs drain, frees tensor memory and exits.
#include "common.cuh"

#include <cuda.h>

#include <mutex>

namespace sq {
namespace {

constexpr int AD = 64;    // head dimension
constexpr int ABQ = 128;  // queries per CTA (the MMA's M)
constexpr int ACH = 64;   // keys per chunk (the first MMA's N, the second's K)
constexpr int AMAXS = 448;
constexpr int A_THREADS = 448;
constexpr int A_TMA_WARP = 9;
constexpr int Q_PART = ABQ * AD * 4;   // 32 KB: one tf32 part of the Q tile
constexpr int KV_PART = ACH * AD * 4;  // 16 KB: one part of a K or V^T chunk
constexpr int P_PART = ABQ * ACH * 4;  // 32 KB: one part of a P chunk
constexpr int OFF_QH = 0, OFF_QL = Q_PART;
constexpr int OFF_RING = 2 * Q_PART;  // 2 stages x (hi, lo)
constexpr int OFF_PH = OFF_RING + 4 * KV_PART, OFF_PL = OFF_PH + P_PART;
constexpr int OFF_BAR = OFF_PL + P_PART;
constexpr int OFF_XCH = OFF_BAR + 256;  // [2][128] row maxima, then [2][128] row sums
constexpr int SLOT_BYTES = 2 * KV_PART;  // hi + lo parts of one 64-row chunk
static_assert(OFF_QL == OFF_QH + SLOT_BYTES && OFF_PL == OFF_PH + SLOT_BYTES, "slot layout");
constexpr int A_SMEM = OFF_XCH + 2 * 2 * ABQ * 4 + 1024;  // + 1024-byte alignment slack
constexpr int TMEM_COLS = 512;                // S (<= 448) + O (64)
// P in tensor memory (sequences of at most 256): S in columns 0..S-1, P's tf32
// high part written over each S chunk once it is read, O at 256, and P's low
// part double-buffered at 320 and 384
constexpr int TP_MAXS = 256, TP_O = 256, TP_PLO = 320;
constexpr unsigned long long kAttnTimeoutNs = 4000000000ull;
constexpr float kLog2e = 1.4426950408889634f;

// instruction descriptor, kind::tf32: D fp32, A and B tf32, both K-major, N = 64, M = 128
constexpr uint32_t IDESC_TF32 =
    (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(64 >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
// the same with N = 128 (the logits of two K chunks at once)
constexpr uint32_t IDESC_TF32_N128 =
    (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(128 >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);

__device__ unsigned int g_attn_error;

struct AttnBars {
    uint64_t q_full, s_full, p_full[2], p_empty[2], o_full, mma_done, q_tma;
    uint64_t o_empty;  // the epilogue has read O: the next unit's P V may overwrite it
    uint64_t pv_done;  // a unit's P V MMAs are complete: its P buffers (Q, slots 2-3) are free
    uint64_t slot_tma[4], slot_full[4], slot_empty[4];  // copy landed / split / MMAs done
    uint64_t v_read;  // the splitters have read a V chunk's raw values
    uint64_t row_x;   // both softmax halves have posted their row maxima / sums
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
__device__ __forceinline__ void mma_tf32(uint32_t d, uint64_t a, uint64_t b, uint32_t acc,
                                         uint32_t idesc = IDESC_TF32) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}
// The same with A from tensor memory (lane = row of A, one 32-bit column per
// K element: K = 8 columns from taddr).
__device__ __forceinline__ void mma_tf32_ta(uint32_t d, uint32_t a_tmem, uint64_t b,
                                            uint32_t acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d),
        "r"(a_tmem), "l"(b), "r"(IDESC_TF32), "r"(acc)
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

// 32 columns of this warp's 32 lanes into tensor memory from registers; the
// caller waits (tmem_st_wait) before signalling that they are written.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, "
        "%10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, "
        "%27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
        "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
        "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
        "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
        "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
        "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
        : "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Byte offset of element (row, k), k < 64, of an operand part of `rows` rows:
// two 32-float K blocks of rows x 128 bytes, 16-byte chunk j of a row at
// j ^ (row & 7) (the 128-byte swizzle; every part starts 1024-byte aligned).
__device__ __forceinline__ uint32_t sw_off(int row, int k, int rows) {
    return (uint32_t)((k >> 5) * rows * 128 + row * 128 + ((((k & 31) >> 2) ^ (row & 7)) << 4) +
                      ((k & 3) << 2));
}

// With P in shared memory: slots 0, 1 of their own, 2, 3 the first P buffer;
// chunk n (K chunks first, then V) and the slot it uses; P buffer c % 2.
static_assert(OFF_PH == OFF_RING + 2 * SLOT_BYTES, "slots 2-3 over the first P buffer");
// Offset of K block kb (32 of the chunk's 64 columns) of part `part` (0: hi,
// 1: lo) of slot s, 64 rows x 128 bytes.  With P in shared memory a slot is
// [hi kb0 | hi kb1 | lo kb0 | lo kb1]; with P in tensor memory slots 2p and 2p + 1
// share a 64 KB region [hi kb0 | hi kb1 | lo kb0 | lo kb1] of 128 rows each,
// slot 2p in rows 0-63, so that two K chunks there form one 128-row operand.
template <bool TP>
__device__ __forceinline__ int piece_off(int s, int part, int kb) {
    return TP ? OFF_RING + (s >> 1) * 2 * SLOT_BYTES + part * 2 * KV_PART + kb * KV_PART +
                    (s & 1) * (KV_PART / 2)
              : OFF_RING + s * SLOT_BYTES + part * KV_PART + kb * (KV_PART / 2);
}
__device__ __forceinline__ int chunk_slot(int n, int nch) {
    return n < nch ? (n & 3) : ((n - nch) & 1);
}
__device__ __forceinline__ int p_off(int c) { return (c & 1) ? OFF_QH : OFF_PH; }

__device__ __forceinline__ void tma_box(uint32_t dst, const CUtensorMap *map, uint32_t bar, int x,
                                        int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
        : "memory");
}
__device__ __forceinline__ void arrive_expect(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

// exact split of x into a tf32 part and the fp32 remainder
__device__ __forceinline__ float hi_part(float x) {
    return __uint_as_float(__float_as_uint(x) & 0xffffe000u);
}

template <bool TP>
__global__ void __launch_bounds__(A_THREADS, 1)
    attention_kernel(const __grid_constant__ CUtensorMap tmQKV, int S, int H, int units,
                     float scale, float *__restrict__ O) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    AttnBars &B = *reinterpret_cast<AttnBars *>(smem + OFF_BAR);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int qtiles = (S + ABQ - 1) / ABQ;
    const int nch = S / ACH;
    // the slot of chunk n (K chunks first, then V): with P in tensor memory all
    // four slots take chunks in turn; otherwise slots 2-3 (the first P buffer)
    // take K chunks only
    auto slot_of = [&](int n) { return TP ? (n & 3) : chunk_slot(n, nch); };
    // unit u: query tile u % qtiles of head (u / qtiles) % H of sequence u / (qtiles H)
    auto unit_of = [&](int u, int &q0, int &h, int &row_b) {
        q0 = (u % qtiles) * ABQ;
        h = (u / qtiles) % H;
        row_b = (u / (qtiles * H)) * S;  // the sequence's first row of QKV
    };

    if (threadIdx.x == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 4;" ::"r"(su32(&B.q_full)));
        for (int i = 0; i < 4; ++i) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(su32(&B.slot_tma[i])));
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 4;" ::"r"(su32(&B.slot_full[i])));
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(su32(&B.slot_empty[i])));
        }
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 4;" ::"r"(su32(&B.v_read)));
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 8;" ::"r"(su32(&B.row_x)));
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(su32(&B.s_full)));
        for (int i = 0; i < 2; ++i) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 8;" ::"r"(su32(&B.p_full[i])));
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(su32(&B.p_empty[i])));
        }
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(su32(&B.o_full)));
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 8;" ::"r"(su32(&B.o_empty)));
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(su32(&B.pv_done)));
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(su32(&B.mma_done)));
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(su32(&B.q_tma)));
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

    if (warp == A_TMA_WARP) {
        // ------------------------------------------------------------ TMA copies
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmQKV))
                         : "memory");
            int uses[4] = {0, 0, 0, 0};
            int it = 0;
            for (int u = blockIdx.x; u < units; u += gridDim.x, ++it) {
                int q0, h, row_b;
                unit_of(u, q0, h, row_b);
                const int xq = h * AD, xk = H * AD + h * AD, xv = 2 * H * AD + h * AD;
                // the Q region is free: with P in tensor memory once the previous
                // unit's logits are complete, otherwise once its P V products are
                // (the Q region and slots 2-3 are its P buffers)
                if (it > 0 && !wait_bar(su32(TP ? &B.s_full : &B.pv_done), (uint32_t)(it - 1) & 1u,
                                        abort))
                    break;
                // the Q tile: four boxes (two 32-column K blocks x two 64-row halves)
                arrive_expect(su32(&B.q_tma), Q_PART);
                for (int kb = 0; kb < 2; ++kb)
                    for (int rh = 0; rh < 2; ++rh)
                        tma_box(sbase + OFF_QH + kb * (ABQ * 128) + rh * (64 * 128), &tmQKV,
                                su32(&B.q_tma), xq + 32 * kb, row_b + q0 + 64 * rh);
                // the V chunks (and any K chunks past the first four) into L2 now,
                // so that their copies, issued as slots free up, find them there
                for (int n = 4; n < 2 * nch; ++n) {
                    const bool kc = n < nch;
                    const int x = kc ? xk : xv, y = row_b + (kc ? n : n - nch) * ACH;
                    for (int kb = 0; kb < 2; ++kb)
                        asm volatile(
                            "cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                                reinterpret_cast<uint64_t>(&tmQKV)),
                            "r"(x + 32 * kb), "r"(y)
                            : "memory");
                }
                {
                    // this CTA's next unit's operands into L2, so that its first
                    // copies come from L2 rather than DRAM
                    const int fu = u + gridDim.x;
                    if (fu < units) {
                        int fq0, fh, frow;
                        unit_of(fu, fq0, fh, frow);
                        for (int kb = 0; kb < 2; ++kb) {
                            for (int rh = 0; rh < 2; ++rh)
                                if (fq0 + 64 * rh < S)  // its query rows inside its sequence
                                    asm volatile(
                                        "cp.async.bulk.prefetch.tensor.2d.L2.global.tile"
                                        " [%0, {%1, %2}];" ::"l"(
                                            reinterpret_cast<uint64_t>(&tmQKV)),
                                        "r"(fh * AD + 32 * kb), "r"(frow + fq0 + 64 * rh)
                                        : "memory");
                            for (int n = 0; n < nch; ++n)
                                for (int part = 1; part < 3; ++part)
                                    asm volatile(
                                        "cp.async.bulk.prefetch.tensor.2d.L2.global.tile"
                                        " [%0, {%1, %2}];" ::"l"(
                                            reinterpret_cast<uint64_t>(&tmQKV)),
                                        "r"(part * H * AD + fh * AD + 32 * kb), "r"(frow + n * ACH)
                                        : "memory");
                        }
                    }
                }
                bool ok = true;
                for (int n = 0; n < 2 * nch; ++n) {
                    const int sl = slot_of(n);
                    const int use = uses[sl];
                    // the slot's previous chunk is done with
                    if (use > 0 &&
                        !wait_bar(su32(&B.slot_empty[sl]), (uint32_t)(use - 1) & 1u, abort)) {
                        ok = false;
                        break;
                    }
                    ++uses[sl];
                    // K chunk n raw into the slot's hi part, V chunk n - nch into its lo part
                    const bool kc = n < nch;
                    const int x = kc ? xk : xv, y = row_b + (kc ? n : n - nch) * ACH;
                    arrive_expect(su32(&B.slot_tma[sl]), KV_PART);
                    for (int kb = 0; kb < 2; ++kb)
                        tma_box(sbase + piece_off<TP>(sl, kc ? 0 : 1, kb), &tmQKV,
                                su32(&B.slot_tma[sl]), x + 32 * kb, y);
                }
                if (!ok) {
                    ++it;  // its Q copy was issued
                    break;
                }
            }
            // every copy issued has landed before the shared memory can go away
            if (it > 0) drain_bar(su32(&B.q_tma), (uint32_t)(it - 1) & 1u);
            for (int sl = 0; sl < 4; ++sl)
                if (uses[sl] > 0) drain_bar(su32(&B.slot_tma[sl]), (uint32_t)(uses[sl] - 1) & 1u);
        }
        __syncwarp();
    } else if (warp >= 4 && warp < 8) {
        // ------------------------------------------------------------ splitters
        const int t = threadIdx.x - 128;
        int uses[4] = {0, 0, 0, 0};  // chunks taken per slot
        int vcount = 0;              // V chunks split so far (v_read phases)
        int it = 0;
        for (int u = blockIdx.x; u < units; u += gridDim.x, ++it) {
            {
                // the Q tile, in place: hi over the copied value, lo beside it
                if (!warp_wait(su32(&B.q_tma), (uint32_t)it & 1u, abort)) goto done_l;
                float4 *qh = reinterpret_cast<float4 *>(smem + OFF_QH);
                float4 *ql = reinterpret_cast<float4 *>(smem + OFF_QL);
#pragma unroll 4
                for (int i = 0; i < Q_PART / 16 / 128; ++i) {
                    const int f = i * 128 + t;
                    const float4 v = qh[f];
                    const float4 vh = make_float4(hi_part(v.x), hi_part(v.y), hi_part(v.z),
                                                  hi_part(v.w));
                    qh[f] = vh;
                    ql[f] = make_float4(v.x - vh.x, v.y - vh.y, v.z - vh.z, v.w - vh.w);
                }
                fence_async_smem();
                __syncwarp();
                if (lane == 0) bar_arrive(su32(&B.q_full));
            }
            for (int n = 0; n < 2 * nch; ++n) {
                const int sl = slot_of(n);
                const uint32_t ph = (uint32_t)uses[sl]++ & 1u;
                if (!warp_wait(su32(&B.slot_tma[sl]), ph, abort)) goto done_l;
                if (n < nch) {
                    // K chunk n, in place: hi over the copied value, lo beside it
#pragma unroll
                    for (int i = 0; i < KV_PART / 16 / 128; ++i) {
                        const int f = i * 128 + t;  // 512 float4 per K block
                        float4 *kh = reinterpret_cast<float4 *>(
                                         smem + piece_off<TP>(sl, 0, f >> 9)) + (f & 511);
                        float4 *kl = reinterpret_cast<float4 *>(
                                         smem + piece_off<TP>(sl, 1, f >> 9)) + (f & 511);
                        const float4 v = *kh;
                        const float4 vh = make_float4(hi_part(v.x), hi_part(v.y), hi_part(v.z),
                                                      hi_part(v.w));
                        *kh = vh;
                        *kl = make_float4(v.x - vh.x, v.y - vh.y, v.z - vh.z, v.w - vh.w);
                    }
                } else {
                    // V chunk (copied into the lo part as [key][dimension]), transposed
                    // into the hi / lo parts (rows: dimensions, K: keys): lane l takes
                    // key 32 kb + l and four dimensions per pass; the raw reads (a float4
                    // of one key row) and the part writes (32 consecutive keys of one
                    // dimension row) are conflict-free under the swizzle.  All four
                    // warps read their share before any warp overwrites the lo part.
                    const int w = warp - 4;
                    float4 v[8];
#pragma unroll
                    for (int k8 = 0; k8 < 8; ++k8) {
                        const int c = w * 8 + k8;  // 32 (key block, dimension group) pairs
                        const int key = 32 * (c >> 4) + lane, d = 4 * (c & 15);
                        v[k8] = *reinterpret_cast<const float4 *>(
                            smem + piece_off<TP>(sl, 1, d >> 5) + key * 128 +
                            ((((d & 31) >> 2) ^ (key & 7)) << 4));
                    }
                    __syncwarp();
                    if (lane == 0) bar_arrive(su32(&B.v_read));
                    if (!warp_wait(su32(&B.v_read), (uint32_t)vcount++ & 1u, abort)) goto done_l;
#pragma unroll
                    for (int k8 = 0; k8 < 8; ++k8) {
                        const int c = w * 8 + k8;
                        const int key = 32 * (c >> 4) + lane, d = 4 * (c & 15);
                        const float e[4] = {v[k8].x, v[k8].y, v[k8].z, v[k8].w};
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const float eh = hi_part(e[q]);
                            const uint32_t off = sw_off(d + q, key & 31, AD);
                            *reinterpret_cast<float *>(smem + piece_off<TP>(sl, 0, key >> 5) +
                                                       off) = eh;
                            *reinterpret_cast<float *>(smem + piece_off<TP>(sl, 1, key >> 5) +
                                                       off) = e[q] - eh;
                        }
                    }
                }
                fence_async_smem();
                __syncwarp();
                if (lane == 0) bar_arrive(su32(&B.slot_full[sl]));
            }
        }
    done_l:;
    } else if (warp == 8) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0) {
            int uses[4] = {0, 0, 0, 0};  // chunks taken per slot
            int pfill[2] = {0, 0};       // P chunks taken per buffer
            int it = 0;
            for (int u = blockIdx.x; u < units; u += gridDim.x, ++it) {
                if (!wait_bar(su32(&B.q_full), (uint32_t)it & 1u, abort)) goto done_m;
                tc_after();
                for (int c = 0; c < nch;) {
                    // with P in tensor memory two K chunks of one slot region form a
                    // 128-row operand: their logits in one N = 128 MMA group
                    const int sl = slot_of(c);
                    const bool two = TP && c + 1 < nch;
                    if (!wait_bar(su32(&B.slot_full[sl]), (uint32_t)uses[sl]++ & 1u, abort))
                        goto done_m;
                    if (two && !wait_bar(su32(&B.slot_full[sl + 1]), (uint32_t)uses[sl + 1]++ & 1u,
                                         abort))
                        goto done_m;
                    tc_after();
                    const uint32_t d = tmem + (uint32_t)(c * ACH);
#pragma unroll
                    for (int p = 0; p < 3; ++p) {
                        const uint32_t a = p == 2 ? sbase + OFF_QL : sbase + OFF_QH;
#pragma unroll
                        for (int kb = 0; kb < 2; ++kb) {
                            const uint64_t ad = desc_sw128(a + kb * ABQ * 128);
                            const uint64_t bd =
                                desc_sw128(sbase + piece_off<TP>(sl, p == 1 ? 1 : 0, kb));
#pragma unroll
                            for (int k = 0; k < 4; ++k)  // K = 8 tf32 = 32 bytes per MMA
                                mma_tf32(d, ad + 2 * k, bd + 2 * k, (p | kb | k) ? 1u : 0u,
                                         two ? IDESC_TF32_N128 : IDESC_TF32);
                        }
                    }
                    mma_commit(su32(&B.slot_empty[sl]));
                    if (two) mma_commit(su32(&B.slot_empty[sl + 1]));
                    c += two ? 2 : 1;
                }
                mma_commit(su32(&B.s_full));
                // the previous unit's epilogue has read O out of tensor memory
                if (it > 0 && !wait_bar(su32(&B.o_empty), (uint32_t)(it - 1) & 1u, abort))
                    goto done_m;
                for (int c = 0; c < nch; ++c) {
                    const int sl = slot_of(nch + c);
                    if (!wait_bar(su32(&B.slot_full[sl]), (uint32_t)uses[sl]++ & 1u, abort))
                        goto done_m;
                    if (!wait_bar(su32(&B.p_full[c & 1]), (uint32_t)pfill[c & 1]++ & 1u, abort))
                        goto done_m;
                    tc_after();
                    if (TP) {
                        // A = P from tensor memory: its high part over S chunk c, its
                        // low part in buffer c % 2
                        const uint32_t d = tmem + (uint32_t)TP_O;
                        const uint32_t phi = tmem + (uint32_t)(c * ACH);
                        const uint32_t plo = tmem + (uint32_t)(TP_PLO + (c & 1) * ACH);
#pragma unroll
                        for (int p = 0; p < 3; ++p) {
                            const uint32_t a = p == 2 ? plo : phi;
#pragma unroll
                            for (int kb = 0; kb < 2; ++kb) {
                                const uint64_t bd =
                                    desc_sw128(sbase + piece_off<TP>(sl, p == 1 ? 1 : 0, kb));
#pragma unroll
                                for (int k = 0; k < 4; ++k)
                                    mma_tf32_ta(d, a + (uint32_t)(32 * kb + 8 * k), bd + 2 * k,
                                                (c | p | kb | k) ? 1u : 0u);
                            }
                        }
                    } else {
                        const uint32_t pa = sbase + p_off(c);
                        const uint32_t d = tmem + (uint32_t)AMAXS;  // O after the logits' columns
#pragma unroll
                        for (int p = 0; p < 3; ++p) {
                            const uint32_t a = p == 2 ? pa + P_PART : pa;
#pragma unroll
                            for (int kb = 0; kb < 2; ++kb) {
                                const uint64_t ad = desc_sw128(a + kb * ABQ * 128);
                                const uint64_t bd =
                                    desc_sw128(sbase + piece_off<TP>(sl, p == 1 ? 1 : 0, kb));
#pragma unroll
                                for (int k = 0; k < 4; ++k)
                                    mma_tf32(d, ad + 2 * k, bd + 2 * k,
                                             (c | p | kb | k) ? 1u : 0u);
                            }
                        }
                    }
                    mma_commit(su32(&B.slot_empty[sl]));
                    mma_commit(su32(&B.p_empty[c & 1]));
                }
                mma_commit(su32(&B.o_full));
                if (!TP) mma_commit(su32(&B.pv_done));
            }
        done_m:
            // every MMA issued above completes before tensor memory is freed
            mma_commit(su32(&B.mma_done));
            drain_bar(su32(&B.mma_done), 0);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ softmax and epilogue
        const int qw = warp & 3;                // lane quarter: query rows 32 qw ..
        const int half = warp >= 8 ? 1 : 0;     // keys 32 half .. of every chunk
        const int r = 32 * qw + lane;           // query row of the tile, tensor-memory lane
        const uint32_t lane_addr = tmem + ((uint32_t)(32 * qw) << 16);
        const float cl2e = scale * kLog2e;
        float *xm = reinterpret_cast<float *>(smem + OFF_XCH);  // [half][row] maxima
        float *xs = xm + 2 * ABQ;                               // [half][row] sums
        int pfill[2] = {0, 0};  // P chunks written per buffer
        int it = 0;
        for (int u = blockIdx.x; u < units; u += gridDim.x, ++it) {
            int q0, h, row_b;
            unit_of(u, q0, h, row_b);
            if (!warp_wait(su32(&B.s_full), (uint32_t)it & 1u, abort)) goto done_s;
            tc_after();
            // the row maximum over all S logits: this half's columns, then the
            // other half's maximum from shared memory (row_x completes twice
            // per unit: maxima, then sums)
            float m = -INFINITY;
            for (int c = 0; c < nch; ++c) {
                float v[32];
                tmem_ld32(lane_addr + c * ACH + 32 * half, v);
#pragma unroll
                for (int j = 0; j < 32; ++j) m = fmaxf(m, v[j]);
            }
            xm[half * ABQ + r] = m;
            __syncwarp();
            if (lane == 0) bar_arrive(su32(&B.row_x));
            if (!warp_wait(su32(&B.row_x), 0, abort)) goto done_s;
            __syncwarp();
            m = fmaxf(xm[r], xm[ABQ + r]);
            const float mc = m * cl2e;
            float sum = 0.0f;
            for (int c = 0; c < nch; ++c) {
                // P buffer c % 2 is free once its previous chunk's MMAs are done
                if (!warp_wait(su32(&B.p_empty[c & 1]), ((uint32_t)pfill[c & 1]++ & 1u) ^ 1u,
                               abort))
                    goto done_s;
                float v[32];
                tmem_ld32(lane_addr + c * ACH + 32 * half, v);
                if (TP) {
                    // P's high part over the logits just read, its low part into
                    // buffer c % 2
                    float pl[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float pp = exp2f(__fmaf_rn(v[j], cl2e, -mc));
                        sum += pp;
                        v[j] = hi_part(pp);
                        pl[j] = pp - v[j];
                    }
                    tmem_st32(lane_addr + c * ACH + 32 * half, v);
                    tmem_st32(lane_addr + TP_PLO + (c & 1) * ACH + 32 * half, pl);
                    tmem_st_wait();
                } else {
                    uint8_t *pbuf = smem + p_off(c);
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
                        *reinterpret_cast<float4 *>(pbuf + off) =
                            make_float4(ph[0], ph[1], ph[2], ph[3]);
                        *reinterpret_cast<float4 *>(pbuf + P_PART + off) =
                            make_float4(pl[0], pl[1], pl[2], pl[3]);
                    }
                    fence_async_smem();
                }
                tc_before();
                __syncwarp();
                if (lane == 0) bar_arrive(su32(&B.p_full[c & 1]));
            }
            // the row sum: half 0's plus half 1's
            xs[half * ABQ + r] = sum;
            __syncwarp();
            if (lane == 0) bar_arrive(su32(&B.row_x));
            if (!warp_wait(su32(&B.row_x), 1, abort)) goto done_s;
            __syncwarp();
            sum = xs[r] + xs[ABQ + r];
            if (!warp_wait(su32(&B.o_full), (uint32_t)it & 1u, abort)) goto done_s;
            tc_after();
            const float inv = __frcp_rn(sum);
            float o[32];
            tmem_ld32(lane_addr + (TP ? TP_O : AMAXS) + 32 * half, o);
            // O is in registers: the next unit's P V may overwrite it
            tc_before();
            __syncwarp();
            if (lane == 0) bar_arrive(su32(&B.o_empty));
            if (q0 + r < S) {
                const int b = row_b / S;
                float4 *dst = reinterpret_cast<float4 *>(O + ((int64_t)b * S + q0 + r) * H * AD +
                                                         h * AD + 32 * half);
#pragma unroll
                for (int i = 0; i < 8; ++i)
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
            if (cudaFuncSetAttribute(attention_kernel<true>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     A_SMEM) != cudaSuccess ||
                cudaFuncSetAttribute(attention_kernel<false>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     A_SMEM) != cudaSuccess)
                return SQ_ERR_CUDA;
            attr[di.device & 63] = true;
        }
    }
    const int64_t units = B * H * ((S + ABQ - 1) / ABQ);
    if (units > 0x7fffffff || B * S > 0x7fffffff) return SQ_ERR_UNSUPPORTED;
    // persistent: one CTA per SM (the shared memory allows no second), each
    // taking units blockIdx.x, + grid, ...
    const int64_t grid = std::min<int64_t>(units, di.sms);
    // QKV as B*S rows of 3*H*64 floats, copied in boxes of 64 rows x 32 columns
    CUtensorMap map;
    if ((rc = make_map_f32(&map, QKV, B * S, 3 * H * AD, 64, 32)) != SQ_OK) return rc;
    return launch_pdl(S <= TP_MAXS ? attention_kernel<true> : attention_kernel<false>,
                      dim3((unsigned)grid), dim3(A_THREADS), A_SMEM, st, 1, map, (int)S, (int)H,
                      (int)units, scale, O);
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

// Self-check of the exact reciprocal division (div_smooth) that the
// requantising GEMM epilogue uses for y / s_next: the routine itself, run
// against IEEE division on significand pairs.
#include "common.cuh"

namespace sq {
namespace {

// Pairs (a, b) in [1, 2)^2, a = 1 + a_frac 2^-23, b = 1 + b_frac 2^-23.  Thread
// per b, loop over a.  With corrected == 0 the uncorrected RN(a RN(1/b)) is
// checked instead: the control that shows the check can fail.
// out[0] += mismatches; out[1] = 1 + (a_frac << 32 | b_frac) of one mismatch.
__global__ void check_division_kernel(uint32_t b_first, uint32_t b_count, uint32_t a_first,
                                      uint32_t a_count, int corrected,
                                      unsigned long long *out) {
    const uint32_t ib = blockIdx.x * blockDim.x + threadIdx.x;
    if (ib >= b_count) return;
    const uint32_t bf = b_first + ib;
    const float b = __uint_as_float(0x3f800000u | bf);
    const float y = __frcp_rn(b);
    unsigned long long bad = 0;
    uint32_t last = 0;
    for (uint32_t ia = 0; ia < a_count; ++ia) {
        const float a = __uint_as_float(0x3f800000u | (a_first + ia));
        const float got = corrected ? div_smooth(a, b, y) : __fmul_rn(a, y);
        if (got != __fdiv_rn(a, b)) {
            ++bad;
            last = a_first + ia;
        }
    }
    if (bad) {
        atomicAdd(out, bad);
        atomicExch(out + 1, 1ull + (((unsigned long long)last << 32) | bf));
    }
}

}  // namespace

sq_status launch_check_division(uint32_t b_first, uint32_t b_count, uint32_t a_first,
                                uint32_t a_count, int corrected, unsigned long long *out,
                                cudaStream_t st) {
    if (b_count == 0 || a_count == 0) return SQ_OK;
    const unsigned grid = (b_count + 255) / 256;
    check_division_kernel<<<grid, 256, 0, st>>>(b_first, b_count, a_first, a_count, corrected,
                                                out);
    return cuda_status(cudaGetLastError());
}

}  // namespace sq

// The linear block on host buffers (sq_linear_block_host): every layer's input
// copied to the device, quantised and multiplied there by the library's own
// entry points, and its output copied back, with the copies of neighbouring
// layers overlapping the kernels of the current one on three streams.
//
// Per layer i (slot i % 2 of two input and two output slots in the caller's
// scratch):
//   stream_h2d:      wait until layer i - 2's quantiser has read the input slot
//                    (x_free), copy X_host[i] in, record x_ready;
//   stream_compute:  wait for x_ready and for layer i - 2's output copy
//                    (y_free), quantise, record x_free, GEMM + epilogue into the
//                    output slot, record y_ready;
//   stream_d2h:      wait for y_ready, copy the slot out to Y_host[i], record
//                    y_free.
// A wait on an event takes its most recent record at the time it is enqueued,
// so four events per slot, recorded again for every layer that uses the slot,
// carry every dependency.  One cudaMemcpyAsync per copy.
#include "common.cuh"

#include <cstdint>

namespace {

constexpr int kSlots = 2;

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

// Byte offsets of the scratch parts for M tokens and the largest K and N.
struct ScratchLayout {
    size_t x_slot, y_slot, op, sx, total;
};

ScratchLayout layout_of(int64_t M, int64_t max_K, int64_t max_N) {
    ScratchLayout l;
    const size_t xs = round256((size_t)M * (size_t)max_K * 4);
    const size_t ys = round256((size_t)M * (size_t)max_N * 4);
    l.x_slot = xs;
    l.y_slot = ys;
    l.op = kSlots * xs + kSlots * ys;
    l.sx = l.op + round256((size_t)M * (size_t)max_K * 2);
    l.total = l.sx + round256((size_t)M * 4);
    return l;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// The checks of sq_quantize_act* / sq_linear_i8 for one layer, with the
// pipeline's own (aligned) scratch as X, operand, scales and Y.
sq_status check_layer(const sq_linear_layer &L, int64_t M, const float *X, void *op,
                      const float *sx, void *Y) {
    if (L.K <= 0 || L.N <= 0) return SQ_ERR_INVALID_ARG;
    if (L.mode < SQ_EPI_NONE || L.mode > SQ_EPI_BIAS_RESIDUAL) return SQ_ERR_INVALID_ARG;
    if (L.K % 16 != 0) return SQ_ERR_ALIGNMENT;
    if (!(L.static_scale >= 0.0f) || L.static_scale > 3.4028234663852886e38f)
        return SQ_ERR_INVALID_ARG;
    if (!L.s) return SQ_ERR_INVALID_ARG;
    if (!aligned(L.s, 16) || (L.s_table && !aligned(L.s_table, 16))) return SQ_ERR_ALIGNMENT;
    (void)X;
    return sq::validate_linear(op, sx, nullptr, L.Wop, L.w_scale, L.w_row_l1, L.bias, L.residual,
                               M, L.N, L.K, L.mode, Y);
}

}  // namespace

extern "C" {

sq_status sq_linear_block_host_scratch_bytes(int64_t M, int64_t max_K, int64_t max_N,
                                             size_t *bytes) {
    if (!bytes || M < 0 || max_K <= 0 || max_N <= 0) return SQ_ERR_INVALID_ARG;
    if (max_K > ((int64_t)1 << 30) || max_N > ((int64_t)1 << 30) || M > ((int64_t)1 << 31))
        return SQ_ERR_UNSUPPORTED;
    *bytes = layout_of(M, max_K, max_N).total;
    return SQ_OK;
}

sq_status sq_linear_block_host(const sq_linear_layer *layers, int64_t count, int64_t M,
                               const float *const *X_host, float *const *Y_host, void *scratch,
                               size_t scratch_bytes, void *stream_h2d, void *stream_compute,
                               void *stream_d2h) {
    if (count < 0 || M < 0) return SQ_ERR_INVALID_ARG;
    if (count == 0 || M == 0) return SQ_OK;
    if (!layers || !X_host || !Y_host || !scratch) return SQ_ERR_INVALID_ARG;
    if (!aligned(scratch, 256)) return SQ_ERR_ALIGNMENT;
    int64_t max_K = 0, max_N = 0;
    for (int64_t i = 0; i < count; ++i) {
        if (!X_host[i] || !Y_host[i]) return SQ_ERR_INVALID_ARG;
        if (layers[i].K <= 0 || layers[i].N <= 0) return SQ_ERR_INVALID_ARG;
        max_K = layers[i].K > max_K ? layers[i].K : max_K;
        max_N = layers[i].N > max_N ? layers[i].N : max_N;
    }
    size_t need = 0;
    sq_status rc = sq_linear_block_host_scratch_bytes(M, max_K, max_N, &need);
    if (rc != SQ_OK) return rc;
    if (scratch_bytes < need) return SQ_ERR_INVALID_ARG;
    const ScratchLayout lay = layout_of(M, max_K, max_N);
    uint8_t *base = static_cast<uint8_t *>(scratch);
    float *xs[kSlots], *ys[kSlots];
    for (int k = 0; k < kSlots; ++k) {
        xs[k] = reinterpret_cast<float *>(base + k * lay.x_slot);
        ys[k] = reinterpret_cast<float *>(base + kSlots * lay.x_slot + k * lay.y_slot);
    }
    void *op = base + lay.op;
    float *sx = reinterpret_cast<float *>(base + lay.sx);
    // every layer checked before anything is enqueued
    for (int64_t i = 0; i < count; ++i)
        if ((rc = check_layer(layers[i], M, xs[i % kSlots], op, sx, ys[i % kSlots])) != SQ_OK)
            return rc;
    if ((rc = sq::require_gb300()) != SQ_OK) return rc;

    cudaStream_t h2d = static_cast<cudaStream_t>(stream_h2d);
    cudaStream_t comp = static_cast<cudaStream_t>(stream_compute);
    cudaStream_t d2h = static_cast<cudaStream_t>(stream_d2h);
    // per slot: x_ready, x_free, y_ready, y_free
    cudaEvent_t ev[kSlots][4];
    int made = 0;
    for (int k = 0; k < kSlots && rc == SQ_OK; ++k)
        for (int e = 0; e < 4; ++e) {
            if (cudaEventCreateWithFlags(&ev[k][e], cudaEventDisableTiming) != cudaSuccess) {
                rc = SQ_ERR_CUDA;
                break;
            }
            ++made;
        }
    auto ok = [&](cudaError_t e) {
        if (e != cudaSuccess && rc == SQ_OK) rc = SQ_ERR_CUDA;
        return rc == SQ_OK;
    };
    for (int64_t i = 0; i < count && rc == SQ_OK; ++i) {
        const sq_linear_layer &L = layers[i];
        const int k = (int)(i % kSlots);
        const bool reuse = i >= kSlots;
        const size_t xbytes = (size_t)M * (size_t)L.K * 4, ybytes = (size_t)M * (size_t)L.N * 4;
        // host -> device
        if (reuse && !ok(cudaStreamWaitEvent(h2d, ev[k][1], 0))) break;
        if (!ok(cudaMemcpyAsync(xs[k], X_host[i], xbytes, cudaMemcpyHostToDevice, h2d))) break;
        if (!ok(cudaEventRecord(ev[k][0], h2d))) break;
        // the linear block
        if (!ok(cudaStreamWaitEvent(comp, ev[k][0], 0))) break;
        if (reuse && !ok(cudaStreamWaitEvent(comp, ev[k][3], 0))) break;
        if (L.static_scale > 0.0f)
            rc = sq_quantize_act_static(xs[k], L.s, M, L.K, L.static_scale, nullptr, sx, op,
                                        nullptr, comp);
        else if (L.s_table)
            rc = sq_quantize_act_table(xs[k], L.s, L.s_table, nullptr, M, L.K, nullptr, sx, op,
                                       nullptr, comp);
        else
            rc = sq_quantize_act(xs[k], L.s, M, L.K, nullptr, sx, op, nullptr, comp);
        if (rc != SQ_OK) break;
        if (!ok(cudaEventRecord(ev[k][1], comp))) break;
        rc = sq_linear_i8(op, sx, nullptr, L.Wop, L.w_scale, L.w_row_l1, L.bias, L.residual, M,
                          L.N, L.K, L.mode, ys[k], comp);
        if (rc != SQ_OK) break;
        if (!ok(cudaEventRecord(ev[k][2], comp))) break;
        // device -> host
        if (!ok(cudaStreamWaitEvent(d2h, ev[k][2], 0))) break;
        if (!ok(cudaMemcpyAsync(Y_host[i], ys[k], ybytes, cudaMemcpyDeviceToHost, d2h))) break;
        if (!ok(cudaEventRecord(ev[k][3], d2h))) break;
    }
    // the events are released once their pending records complete
    for (int n = 0; n < made; ++n) cudaEventDestroy(ev[n / 4][n % 4]);
    return rc;
}

}  // extern "C"

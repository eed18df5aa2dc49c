// sq_linear_i8_static_ws: sq_linear_i8_ws on a workspace the library holds in
// static device memory, for callers that may not allocate (or hand over) any
// device memory of their own.
//
// The scratch is one file-scope __device__ array of SQ_STATIC_WORKSPACE_BYTES,
// zero-filled when the module is loaded, which is what the split-K counters
// need; every completed launch leaves the counters at zero again, and after a
// launch whose bounded wait ran out, sq_device_status zero-fills them
// (static_ws_reset_counters).  The array's device address is looked up once
// per device (cudaGetSymbolAddress, checked) and cached for the life of the
// process, so a cudaDeviceReset while the library is loaded is not supported
// here.  A request larger than the array is rejected; nothing is allocated.
#include "common.cuh"
#include "schedule.cuh"

#include <mutex>

namespace {

static __device__ __align__(256) unsigned char g_static_ws[SQ_STATIC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;

std::mutex g_mu;
void *g_addr[kMaxDevices] = {};

// Device address of g_static_ws on the current device, looked up (and
// checked) once per device, with that device current, on its first call.
sq_status static_ws_address(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SQ_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return SQ_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_ws) != cudaSuccess || !p) {
            (void)cudaGetLastError();  // do not leave the failed lookup in the last-error slot
            return SQ_ERR_CUDA;
        }
        g_addr[dev] = p;
    }
    *out = g_addr[dev];
    return SQ_OK;
}

}  // namespace

namespace sq {

sq_status static_ws_reset_counters(cudaStream_t st) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SQ_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return SQ_OK;
    void *p = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        p = g_addr[dev];
    }
    if (!p) return SQ_OK;  // never used on this device: still zero from the module load
    DeviceInfo di;
    sq_status rc = device_info(&di);
    if (rc != SQ_OK) return rc;
    const size_t n = (size_t)sched::sk_counter_bytes_on(di.sms);
    if (cudaMemsetAsync(p, 0, n, st) != cudaSuccess || cudaStreamSynchronize(st) != cudaSuccess)
        return SQ_ERR_CUDA;
    return SQ_OK;
}

}  // namespace sq

extern "C" sq_status sq_linear_i8_static_ws(const void *Xop, const float *x_scale,
                                            const int32_t *x_row_l1, const void *Wop,
                                            const float *w_scale, const int32_t *w_row_l1,
                                            const float *bias, const float *residual, int64_t M,
                                            int64_t N, int64_t K, int mode, void *Y,
                                            void *stream) {
    // the checks of sq_linear_i8_ws first (same statuses), then the scratch
    sq_status rc = sq::validate_linear(Xop, x_scale, x_row_l1, Wop, w_scale, w_row_l1, bias,
                                       residual, M, N, K, mode, Y);
    if (rc != SQ_OK || M == 0 || N == 0) return rc;
    if ((rc = sq::require_gb300()) != SQ_OK) return rc;
    size_t need = 0;
    if ((rc = sq_linear_workspace_bytes(M, N, K, &need)) != SQ_OK) return rc;
    if (!sq::sched::fits_scratch((long long)need, (long long)SQ_STATIC_WORKSPACE_BYTES))
        return SQ_ERR_UNSUPPORTED;
    // looked up on every device's first call, split or not, so that later
    // calls (inside a stream capture, say) only launch
    void *ws = nullptr;
    if ((rc = static_ws_address(&ws)) != SQ_OK) return rc;
    return sq_linear_i8_ws(Xop, x_scale, x_row_l1, Wop, w_scale, w_row_l1, bias, residual, M, N,
                           K, mode, Y, need > 0 ? ws : nullptr, need, stream);
}

extern "C" sq_status sq_static_workspace(void **ptr, size_t *bytes) {
    if (!ptr || !bytes) return SQ_ERR_INVALID_ARG;
    sq_status rc = SQ_OK;
    {
        sq::DeviceInfo di;
        if ((rc = sq::device_info(&di)) != SQ_OK) return rc;
        if (di.major != 10 || di.minor != 3) return SQ_ERR_UNSUPPORTED;
    }
    void *p = nullptr;
    if ((rc = static_ws_address(&p)) != SQ_OK) return rc;
    *ptr = p;
    *bytes = SQ_STATIC_WORKSPACE_BYTES;
    return SQ_OK;
}

extern "C" sq_status sq_static_workspace_reset(void *stream) {
    return sq::static_ws_reset_counters(static_cast<cudaStream_t>(stream));
}

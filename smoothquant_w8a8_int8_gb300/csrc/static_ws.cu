// sq_linear_i8_static_ws: sq_linear_i8_ws on a workspace the library holds in
// static device memory, for callers that may not allocate (or hand over) any
// device memory of their own.
//
// The scratch is one file-scope __device__ array of SQ_STATIC_WORKSPACE_BYTES,
// zero-filled when the module is loaded, which is what the split-K counters
// need; every completed launch leaves the counters at zero again.  Its device
// address is looked up once per device (cudaGetSymbolAddress, checked) and
// cached; a request larger than the array is rejected, nothing is allocated.
#include "common.cuh"

#include <mutex>

namespace {

static __device__ __align__(256) unsigned char g_static_ws[SQ_STATIC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;

// Device address of g_static_ws on the current device (looked up once per device).
sq_status static_ws_address(void **out) {
    static std::mutex mu;
    static void *addr[kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SQ_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return SQ_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_ws) != cudaSuccess || !p) {
            (void)cudaGetLastError();  // do not leave the failed lookup in the last-error slot
            return SQ_ERR_CUDA;
        }
        addr[dev] = p;
    }
    *out = addr[dev];
    return SQ_OK;
}

}  // namespace

extern "C" sq_status sq_linear_i8_static_ws(const void *Xop, const float *x_scale,
                                            const int32_t *x_row_l1, const void *Wop,
                                            const float *w_scale, const int32_t *w_row_l1,
                                            const float *bias, const float *residual, int64_t M,
                                            int64_t N, int64_t K, int mode, void *Y,
                                            void *stream) {
    // empty calls: the argument checks of sq_linear_i8_ws, no launch, no device query
    if (M == 0 || N == 0)
        return sq_linear_i8_ws(Xop, x_scale, x_row_l1, Wop, w_scale, w_row_l1, bias, residual, M,
                               N, K, mode, Y, nullptr, 0, stream);
    size_t need = 0;
    sq_status rc = sq_linear_workspace_bytes(M, N, K, &need);
    if (rc != SQ_OK) return rc;
    if (need > (size_t)SQ_STATIC_WORKSPACE_BYTES) return SQ_ERR_UNSUPPORTED;
    // looked up on every device's first call, split or not, so that later calls
    // (inside a stream capture, say) only launch
    void *ws = nullptr;
    if ((rc = static_ws_address(&ws)) != SQ_OK) return rc;
    return sq_linear_i8_ws(Xop, x_scale, x_row_l1, Wop, w_scale, w_row_l1, bias, residual, M, N,
                           K, mode, Y, need > 0 ? ws : nullptr, need, stream);
}

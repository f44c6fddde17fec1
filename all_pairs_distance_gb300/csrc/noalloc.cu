// dbscan_fit_noalloc: the full DBSCAN with its workspace in static device
// memory, for callers that cannot allocate device memory (see dbscan.h).
// Nothing here calls cudaMalloc, cudaFree or any allocating routine; the
// pipeline itself is dbscan_fit_ex's, handed this file's array as workspace,
// with every kernel launched directly: it never captures or instantiates a
// CUDA graph, which would take device resources of its own.
#include "dbscan_internal.cuh"

#include <mutex>

namespace {

// The workspace of every dbscan_fit_noalloc call on a device.  In host code
// this name is only a stand-in for the device array: its device address comes
// from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[DBSCAN_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void *g_scratch_ptr[kMaxDevices] = {};   // device address per device, set on first use

// Device address of the array on the current device (looked up once per
// device, with that device current).
int scratch_address(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return DBSCAN_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return DBSCAN_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void *ptr = nullptr;
        cudaError_t e = cudaGetSymbolAddress((void **)&ptr, g_noalloc_scratch);
        if (e != cudaSuccess || ptr == nullptr) {
            cudaGetLastError();
            return DBSCAN_ERR_CUDA;
        }
        g_scratch_ptr[dev] = ptr;
    }
    *out = g_scratch_ptr[dev];
    return DBSCAN_OK;
}

}  // namespace

extern "C" int dbscan_fit_noalloc(const void *points, int32_t dtype, int64_t n, int32_t d,
                                  float eps, int32_t min_pts, int32_t *labels_out,
                                  uint8_t *is_core_out, void *stream) {
    const size_t need = dbscan_workspace_size(n, d, dtype);
    if (need == 0)   // shape rejected: report it as dbscan_fit_ex would
        return (n < 0 || d < 1 || (dtype != DBSCAN_F32 && dtype != DBSCAN_BF16))
                   ? DBSCAN_ERR_INVALID_ARG
                   : DBSCAN_ERR_UNSUPPORTED;
    if (need > (size_t)DBSCAN_NOALLOC_SCRATCH_BYTES) return DBSCAN_ERR_UNSUPPORTED;
    void *ws = nullptr;
    const int st = scratch_address(&ws);
    if (st != DBSCAN_OK) return st;
    // The pipeline clears its control block and counters at the start of
    // every call, so the previous call's contents of the array do no harm.
    return dbscan::fit_direct(points, dtype, n, d, eps, min_pts, labels_out, is_core_out, ws,
                              (size_t)DBSCAN_NOALLOC_SCRATCH_BYTES, stream);
}

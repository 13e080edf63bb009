// qdq_fused_static.cu -- fos_qdq_fused_static: the fused amax + QDQ list call
// for callers that cannot allocate device memory themselves.  The counters
// the fused launch needs live in one fixed array of this library instead of
// a caller-provided workspace.
#include <cstdint>
#include <mutex>

#include "../../include/fos.h"
#include "fos_launch.cuh"

namespace {

// Largest list served: one error word, then a counter and a running amax per
// tensor, i.e. 1 + 2 * 64 words, rounded up to whole 256-byte lines (768 B).
constexpr int kStaticMaxList = FOS_QDQ_MAX_LIST;
constexpr size_t kStaticWords = 192;
static_assert((1 + 2 * kStaticMaxList) <= (int)kStaticWords, "static workspace too small");

// The workspace itself: one copy per GPU that loads the library, held until
// the process exits.  In host code this name is only a stand-in for the
// device copy; its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) uint32_t g_qdq_fused_ws[kStaticWords];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {};  // last looked-up device address of g_qdq_fused_ws, per device

// Device of the first non-empty tensor (or of amax[0] when all are empty).
int list_device(int n, const void* const* x, const int64_t* rows, const int64_t* cols,
                float* const* amax) {
    const void* p = amax[0];
    for (int i = 0; i < n; ++i)
        if (rows[i] > 0 && cols[i] > 0 && x[i]) {
            p = x[i];
            break;
        }
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();
        return -1;
    }
    if (at.type != cudaMemoryTypeDevice && at.type != cudaMemoryTypeManaged) return -1;
    return at.device;
}

// True when `s` is being captured into a graph (or its state cannot be read).
bool capturing(cudaStream_t s) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) {
        cudaGetLastError();
        return true;
    }
    return cs != cudaStreamCaptureStatusNone;
}

// The array's device address on `dev`, looked up with that device current
// (the caller's current device is restored).  Outside stream capture the
// address is looked up again on every call, so a reset of the device's
// primary context between calls (which reloads the module and moves the
// array) is picked up; during capture the address of the last lookup on
// that device is used, so a device's first call must come before any
// capture.
void* workspace_on(int dev, cudaStream_t s) {
    if (dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> g(g_mu);
    if (g_addr[dev] && capturing(s)) return g_addr[dev];
    int prev = -1;
    if (cudaGetDevice(&prev) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    if (prev != dev && cudaSetDevice(dev) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    void* ptr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&ptr, g_qdq_fused_ws);
    if (e != cudaSuccess) {
        cudaGetLastError();
        ptr = nullptr;
    }
    if (prev != dev) cudaSetDevice(prev);
    g_addr[dev] = ptr;
    return ptr;
}

}  // namespace

extern "C" {

fos_status fos_qdq_fused_static(int n, const void* const* x, void* const* out,
                                const int64_t* rows, const int64_t* cols, float* const* amax,
                                fos_dtype dt, const fos_config* cfg, fos_stream_t stream) {
    // the same host-only checks, in the same order, as fos_qdq_fused, with
    // the fixed array's list limit; no CUDA call before they pass
    const fos_status st =
        fos::qdq_fused_host_checks(n, kStaticMaxList, x, out, rows, cols, amax, dt, cfg);
    if (st || n == 0) return st;
    const int dev = list_device(n, x, rows, cols, amax);
    if (dev < 0) return FOS_ERR_INVALID_ARG;
    void* ws = workspace_on(dev, reinterpret_cast<cudaStream_t>(stream));
    if (!ws) return FOS_ERR_CUDA;
    // fos_qdq_fused checks the devices of every pointer and clears the words
    // it uses (with cudaMemsetAsync on `stream`) before its launch.
    return fos_qdq_fused(n, x, out, rows, cols, amax, dt, cfg, ws,
                         kStaticWords * sizeof(uint32_t), stream);
}

}  // extern "C"

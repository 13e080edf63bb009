// fos_launch.cuh -- host-side launch helpers shared by the kernel
// translation units: persistent grid sizing and the per-family launchers.
#pragma once

#include <cuda_runtime.h>

#include <mutex>
#include <unordered_map>

#include "fos.h"
#include "fos_kernels.cuh"

namespace fos {

// Number of SMs of the current device (cached per device).
inline int sm_count() {
    static std::mutex mu;
    static std::unordered_map<int, int> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    std::lock_guard<std::mutex> g(mu);
    auto it = cache.find(dev);
    if (it != cache.end()) return it->second;
    int n = 1;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cache[dev] = n > 0 ? n : 1;
    return cache[dev];
}

// Resident CTAs per SM of a kernel at a dynamic shared-memory size (cached:
// the occupancy query costs host time on every launch otherwise).
inline int resident_ctas(const void* kernel, size_t dyn_smem) {
    struct Key {
        const void* k;
        size_t smem;
        int dev;
        bool operator==(const Key& o) const { return k == o.k && smem == o.smem && dev == o.dev; }
    };
    struct Hash {
        size_t operator()(const Key& k) const {
            return std::hash<const void*>()(k.k) ^ (k.smem * 1315423911u) ^ (size_t)k.dev;
        }
    };
    static std::mutex mu;
    static std::unordered_map<Key, int, Hash> cache;
    int dev = 0;
    cudaGetDevice(&dev);
    const Key key{kernel, dyn_smem, dev};
    {
        std::lock_guard<std::mutex> g(mu);
        auto it = cache.find(key);
        if (it != cache.end()) return it->second;
    }
    int occ = 1;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, kThreads, dyn_smem) !=
            cudaSuccess || occ < 1) {
        cudaGetLastError();
        occ = 1;
    }
    std::lock_guard<std::mutex> g(mu);
    cache[key] = occ;
    return occ;
}

// Persistent grid: as many CTAs as stay resident (SMs x occupancy), but no
// more than one warp per work unit needs.
template <class Kernel>
inline int persistent_grid(Kernel kernel, int64_t units, size_t dyn_smem) {
    const int occ = resident_ctas(reinterpret_cast<const void*>(kernel), dyn_smem);
    const int64_t full = (int64_t)sm_count() * occ;
    const int64_t need = (units + kWarps - 1) / kWarps;
    int64_t g = need < full ? need : full;
    return (int)(g < 1 ? 1 : g);
}

// Raises a kernel's dynamic shared-memory limit when it needs more than the
// default 48 KiB (once per kernel and size).
inline cudaError_t allow_smem(const void* kernel, size_t bytes) {
    if (bytes <= 48 * 1024) return cudaSuccess;
    static std::mutex mu;
    static std::unordered_map<const void*, size_t> done;
    std::lock_guard<std::mutex> g(mu);
    auto it = done.find(kernel);
    if (it != done.end() && it->second >= bytes) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)bytes);
    if (e == cudaSuccess) done[kernel] = bytes;
    return e;
}

template <class Kernel, class Args>
inline cudaError_t launch_persistent(Kernel kernel, const Args& a, int64_t units, size_t dyn_smem,
                                     cudaStream_t s) {
    cudaError_t e = allow_smem(reinterpret_cast<const void*>(kernel), dyn_smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)persistent_grid(kernel, units, dyn_smem));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = dyn_smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kernel, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_quant1x16_bf16(Err, Src, const EncArgs&, cudaStream_t);
cudaError_t launch_quant1x16_f16(Err, Src, const EncArgs&, cudaStream_t);
cudaError_t launch_quant1x16_f32(Err, Src, const EncArgs&, cudaStream_t);
cudaError_t launch_quant1x16_rowpass_bf16(Err, int k, const EncArgs&, cudaStream_t);
cudaError_t launch_quant1x16_rowpass_f16(Err, int k, const EncArgs&, cudaStream_t);
cudaError_t launch_quant1x16_rowpass_f32(Err, int k, const EncArgs&, cudaStream_t);
cudaError_t launch_quant16x16_bf16(Err, Src, const EncArgs&, cudaStream_t);
cudaError_t launch_quant16x16_f16(Err, Src, const EncArgs&, cudaStream_t);
cudaError_t launch_quant16x16_f32(Err, Src, const EncArgs&, cudaStream_t);
cudaError_t launch_qdq(In, Err, const QdqArgs&, cudaStream_t);
cudaError_t launch_qdq_fused(In, Err, const QdqFusedArgs&, cudaStream_t);
cudaError_t launch_colwise(In, Err, bool dual, const ColArgs&, cudaStream_t);
// the same kernels writing their block scales in the tiled GEMM layout
cudaError_t launch_quant1x16_tl_bf16(Err, Src, const EncArgs&, cudaStream_t);
cudaError_t launch_quant1x16_tl_f16(Err, Src, const EncArgs&, cudaStream_t);
cudaError_t launch_quant1x16_tl_f32(Err, Src, const EncArgs&, cudaStream_t);
cudaError_t launch_quant1x16_rowpass_tl_bf16(Err, int k, const EncArgs&, cudaStream_t);
cudaError_t launch_quant1x16_rowpass_tl_f16(Err, int k, const EncArgs&, cudaStream_t);
cudaError_t launch_quant1x16_rowpass_tl_f32(Err, int k, const EncArgs&, cudaStream_t);
cudaError_t launch_colwise_tl(In, Err, bool dual, const ColArgs&, cudaStream_t);
cudaError_t launch_pipe(In, Err, const PipeArgs&, cudaStream_t);
cudaError_t launch_pipe_tl(In, Err, const PipeArgs&, cudaStream_t);
cudaError_t launch_dequant(Out, bool b16, Src, const DeqArgs&, cudaStream_t);
cudaError_t launch_amax(In, Src, const AmaxArgs&, cudaStream_t);
cudaError_t launch_diag(int op, const void* in, void* out, int64_t n, cudaStream_t);
cudaError_t launch_wait_timeout(int which, uint32_t* word, cudaStream_t);
int run_mm(const uint8_t* a_codes, const uint8_t* a_scales, const float* a_amax, int a_row,
           const uint8_t* b_codes, const uint8_t* b_scales, const float* b_amax, int64_t M,
           int64_t N, int64_t K, float six_bound, float* out, cudaStream_t s);
cudaError_t launch_swizzle(const uint8_t* scales, int64_t rows, int64_t nb, uint8_t* out,
                           cudaStream_t);
cudaError_t launch_check_tile_amax(const float* amax, int64_t rows, int64_t* bad, cudaStream_t);

// Host-side argument checks shared by the two fused amax + QDQ entry points
// (fos_api.cu); no CUDA call.
fos_status qdq_fused_host_checks(int n, int max_n, const void* const* x, void* const* out,
                                 const int64_t* rows, const int64_t* cols, float* const* amax,
                                 fos_dtype dt, const fos_config* cfg);

}  // namespace fos

// Fused multi-tensor amax + QDQ (one persistent, cooperative launch).
#include "fos_launch.cuh"

namespace fos {

template <In IT, Err EM>
static cudaError_t go(const QdqFusedArgs& a, cudaStream_t s) {
    auto kernel = k_qdq_fused<IT, EM>;
    // every CTA must be resident at once (warps wait for one another): the
    // grid is the resident capacity and the launch is cooperative, so it
    // fails instead of starting when the CTAs cannot all be placed
    const int grid = sm_count() * resident_ctas(reinterpret_cast<const void*>(kernel), 0);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <In IT>
static cudaError_t by_err(Err em, const QdqFusedArgs& a, cudaStream_t s) {
    switch (em) {
        case Err::STD: return go<IT, Err::STD>(a, s);
        case Err::MAE: return go<IT, Err::MAE>(a, s);
        case Err::MSE: return go<IT, Err::MSE>(a, s);
        case Err::MAE_H: return go<IT, Err::MAE_H>(a, s);
        case Err::MSE_H: return go<IT, Err::MSE_H>(a, s);
        case Err::MAE_S: return go<IT, Err::MAE_S>(a, s);
        case Err::MSE_S: return go<IT, Err::MSE_S>(a, s);
        case Err::MAE_HS: return go<IT, Err::MAE_HS>(a, s);
        case Err::MSE_HS: return go<IT, Err::MSE_HS>(a, s);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_qdq_fused(In it, Err em, const QdqFusedArgs& a, cudaStream_t s) {
    switch (it) {
        case In::BF16: return by_err<In::BF16>(em, a, s);
        case In::F16: return by_err<In::F16>(em, a, s);
        case In::F32: break;
    }
    return cudaErrorInvalidValue;
}

}  // namespace fos

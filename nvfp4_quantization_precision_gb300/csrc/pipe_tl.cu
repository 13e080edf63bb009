// Instantiations of the list pipeline kernel that writes its block scales in
// the tiled GEMM layout.
#include "fos_launch.cuh"

namespace fos {

template <In IT>
static cudaError_t by_err(Err em, const PipeArgs& a, cudaStream_t s) {
    // every warp walks both tensors: the larger unit count sizes the grid
    const int64_t units = a.enc.units > a.aunits ? a.enc.units : a.aunits;
    switch (em) {
        case Err::STD: return launch_persistent(k_quant1x16_pipe<IT, Err::STD, true>, a, units, 0, s);
        case Err::MAE: return launch_persistent(k_quant1x16_pipe<IT, Err::MAE, true>, a, units, 0, s);
        case Err::MSE: return launch_persistent(k_quant1x16_pipe<IT, Err::MSE, true>, a, units, 0, s);
        case Err::MAE_H: return launch_persistent(k_quant1x16_pipe<IT, Err::MAE_H, true>, a, units, 0, s);
        case Err::MSE_H: return launch_persistent(k_quant1x16_pipe<IT, Err::MSE_H, true>, a, units, 0, s);
        case Err::MAE_S: return launch_persistent(k_quant1x16_pipe<IT, Err::MAE_S, true>, a, units, 0, s);
        case Err::MSE_S: return launch_persistent(k_quant1x16_pipe<IT, Err::MSE_S, true>, a, units, 0, s);
        case Err::MAE_HS: return launch_persistent(k_quant1x16_pipe<IT, Err::MAE_HS, true>, a, units, 0, s);
        case Err::MSE_HS: return launch_persistent(k_quant1x16_pipe<IT, Err::MSE_HS, true>, a, units, 0, s);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_pipe_tl(In it, Err em, const PipeArgs& a, cudaStream_t s) {
    switch (it) {
        case In::BF16: return by_err<In::BF16>(em, a, s);
        case In::F16: return by_err<In::F16>(em, a, s);
        case In::F32: return by_err<In::F32>(em, a, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace fos

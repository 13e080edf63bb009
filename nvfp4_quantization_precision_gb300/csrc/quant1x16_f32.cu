// Instantiations of the 1x16 quantize kernel for f32 input.
#include "fos_launch.cuh"

namespace fos {

template <Err EM, Src SRC>
static cudaError_t go(const EncArgs& a, cudaStream_t s) {
    if constexpr (SRC == Src::TENSOR) {
        return launch_persistent(k_quant1x16_tensor<In::F32, EM>, a, a.units, 0, s);
    } else {
        const size_t dyn = (SRC == Src::GROUP) ? sizeof(int32_t) * (size_t)a.G : 0;
        return launch_persistent(k_quant1x16<In::F32, EM, SRC>, a, a.units, dyn, s);
    }
}

template <Err EM>
static cudaError_t by_src(Src src, const EncArgs& a, cudaStream_t s) {
    switch (src) {
        case Src::TENSOR: return go<EM, Src::TENSOR>(a, s);
        case Src::ROW: return go<EM, Src::ROW>(a, s);
        case Src::GROUP: return go<EM, Src::GROUP>(a, s);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_quant1x16_f32(Err em, Src src, const EncArgs& a, cudaStream_t s) {
    switch (em) {
        case Err::STD: return by_src<Err::STD>(src, a, s);
        case Err::MAE: return by_src<Err::MAE>(src, a, s);
        case Err::MSE: return by_src<Err::MSE>(src, a, s);
        case Err::MAE_H: return by_src<Err::MAE_H>(src, a, s);
        case Err::MSE_H: return by_src<Err::MSE_H>(src, a, s);
        case Err::MAE_S: return by_src<Err::MAE_S>(src, a, s);
        case Err::MSE_S: return by_src<Err::MSE_S>(src, a, s);
        case Err::MAE_HS: return by_src<Err::MAE_HS>(src, a, s);
        case Err::MSE_HS: return by_src<Err::MSE_HS>(src, a, s);
    }
    return cudaErrorInvalidValue;
}

template <Err EM>
static cudaError_t rowpass(int k, const EncArgs& a, cudaStream_t s) {
    switch (k) {
        case 1: return launch_persistent(k_quant1x16_rowpass<In::F32, EM, 1>, a, a.rows * kWarps, 0, s);
        case 2: return launch_persistent(k_quant1x16_rowpass<In::F32, EM, 2>, a, a.rows * kWarps, 0, s);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_quant1x16_rowpass_f32(Err em, int k, const EncArgs& a, cudaStream_t s) {
    switch (em) {
        case Err::STD: return rowpass<Err::STD>(k, a, s);
        case Err::MAE: return rowpass<Err::MAE>(k, a, s);
        case Err::MSE: return rowpass<Err::MSE>(k, a, s);
        case Err::MAE_H: return rowpass<Err::MAE_H>(k, a, s);
        case Err::MSE_H: return rowpass<Err::MSE_H>(k, a, s);
        case Err::MAE_S: return rowpass<Err::MAE_S>(k, a, s);
        case Err::MSE_S: return rowpass<Err::MSE_S>(k, a, s);
        case Err::MAE_HS: return rowpass<Err::MAE_HS>(k, a, s);
        case Err::MSE_HS: return rowpass<Err::MSE_HS>(k, a, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace fos

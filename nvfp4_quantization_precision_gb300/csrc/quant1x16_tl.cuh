// Instantiations of the 1x16 quantize kernels that write their block scales
// in the tiled GEMM layout (per-tensor grid-stride, per-row walk, one-pass
// row kernel), for one input type IT; included by quant1x16_tl_*.cu.
#pragma once
#include "fos_launch.cuh"

namespace fos {
namespace tl {

template <In IT, Err EM>
cudaError_t go(Src src, const EncArgs& a, cudaStream_t s) {
    if (src == Src::TENSOR)
        return launch_persistent(k_quant1x16_tensor<IT, EM, true>, a, a.units, 0, s);
    if (src == Src::ROW)
        return launch_persistent(k_quant1x16<IT, EM, Src::ROW, true>, a, a.units, 0, s);
    return cudaErrorInvalidValue;  // grouped quantize writes plain scales only
}

template <In IT>
cudaError_t quant(Err em, Src src, const EncArgs& a, cudaStream_t s) {
    switch (em) {
        case Err::STD: return go<IT, Err::STD>(src, a, s);
        case Err::MAE: return go<IT, Err::MAE>(src, a, s);
        case Err::MSE: return go<IT, Err::MSE>(src, a, s);
        case Err::MAE_H: return go<IT, Err::MAE_H>(src, a, s);
        case Err::MSE_H: return go<IT, Err::MSE_H>(src, a, s);
        case Err::MAE_S: return go<IT, Err::MAE_S>(src, a, s);
        case Err::MSE_S: return go<IT, Err::MSE_S>(src, a, s);
        case Err::MAE_HS: return go<IT, Err::MAE_HS>(src, a, s);
        case Err::MSE_HS: return go<IT, Err::MSE_HS>(src, a, s);
    }
    return cudaErrorInvalidValue;
}

template <In IT, Err EM>
cudaError_t rowpass_go(int k, const EncArgs& a, cudaStream_t s) {
    if (k == 1)
        return launch_persistent(k_quant1x16_rowpass<IT, EM, 1, true>, a, a.rows * kWarps, 0, s);
    if (k == 2)
        return launch_persistent(k_quant1x16_rowpass<IT, EM, 2, true>, a, a.rows * kWarps, 0, s);
    return cudaErrorInvalidValue;
}

template <In IT>
cudaError_t rowpass(Err em, int k, const EncArgs& a, cudaStream_t s) {
    switch (em) {
        case Err::STD: return rowpass_go<IT, Err::STD>(k, a, s);
        case Err::MAE: return rowpass_go<IT, Err::MAE>(k, a, s);
        case Err::MSE: return rowpass_go<IT, Err::MSE>(k, a, s);
        case Err::MAE_H: return rowpass_go<IT, Err::MAE_H>(k, a, s);
        case Err::MSE_H: return rowpass_go<IT, Err::MSE_H>(k, a, s);
        case Err::MAE_S: return rowpass_go<IT, Err::MAE_S>(k, a, s);
        case Err::MSE_S: return rowpass_go<IT, Err::MSE_S>(k, a, s);
        case Err::MAE_HS: return rowpass_go<IT, Err::MAE_HS>(k, a, s);
        case Err::MSE_HS: return rowpass_go<IT, Err::MSE_HS>(k, a, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace tl
}  // namespace fos

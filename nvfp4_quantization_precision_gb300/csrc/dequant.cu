// Instantiations of the dequantize kernel.
#include "fos_launch.cuh"

namespace fos {

template <Out OT, bool B16>
static cudaError_t by_src(Src src, const DeqArgs& a, cudaStream_t s) {
    if (src == Src::ROW) return launch_persistent(k_dequant<OT, B16, Src::ROW>, a, a.units, 0, s);
    return launch_persistent(k_dequant<OT, B16, Src::TENSOR>, a, a.units, 0, s);
}

template <Out OT>
static cudaError_t by_block(bool b16, Src src, const DeqArgs& a, cudaStream_t s) {
    return b16 ? by_src<OT, true>(src, a, s) : by_src<OT, false>(src, a, s);
}

cudaError_t launch_dequant(Out ot, bool b16, Src src, const DeqArgs& a, cudaStream_t s) {
    switch (ot) {
        case Out::BF16: return by_block<Out::BF16>(b16, src, a, s);
        case Out::F16: return by_block<Out::F16>(b16, src, a, s);
        case Out::F32: return by_block<Out::F32>(b16, src, a, s);
        default: break;
    }
    return cudaErrorInvalidValue;
}

}  // namespace fos

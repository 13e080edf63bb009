// Instantiations of the 1x16 quantize kernels with tiled scales, f32 input.
#include "quant1x16_tl.cuh"

namespace fos {

cudaError_t launch_quant1x16_tl_f32(Err em, Src src, const EncArgs& a, cudaStream_t s) {
    return tl::quant<In::F32>(em, src, a, s);
}

cudaError_t launch_quant1x16_rowpass_tl_f32(Err em, int k, const EncArgs& a, cudaStream_t s) {
    return tl::rowpass<In::F32>(em, k, a, s);
}

}  // namespace fos

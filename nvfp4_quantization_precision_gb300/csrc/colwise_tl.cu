// Instantiations of the column-wise (x^T) quantize that write the block
// scales in the tiled GEMM layout, alone or with the row-wise result of the
// same read (DUAL).
#include "fos_launch.cuh"

namespace fos {

template <In IT, Err EM>
static cudaError_t go(bool dual, const ColArgs& a, cudaStream_t s) {
    constexpr size_t kSmem = 2 * (size_t)ColTile<IT>::kBytes + 128;  // two tiles, aligned
    const int64_t units = a.tiles * kWarps;  // one CTA per tile at most
    if (dual) return launch_persistent(k_quant_colwise<IT, EM, true, true>, a, units, kSmem, s);
    return launch_persistent(k_quant_colwise<IT, EM, false, true>, a, units, kSmem, s);
}

template <In IT>
static cudaError_t by_err(Err em, bool dual, const ColArgs& a, cudaStream_t s) {
    switch (em) {
        case Err::STD: return go<IT, Err::STD>(dual, a, s);
        case Err::MAE: return go<IT, Err::MAE>(dual, a, s);
        case Err::MSE: return go<IT, Err::MSE>(dual, a, s);
        case Err::MAE_H: return go<IT, Err::MAE_H>(dual, a, s);
        case Err::MSE_H: return go<IT, Err::MSE_H>(dual, a, s);
        case Err::MAE_S: return go<IT, Err::MAE_S>(dual, a, s);
        case Err::MSE_S: return go<IT, Err::MSE_S>(dual, a, s);
        case Err::MAE_HS: return go<IT, Err::MAE_HS>(dual, a, s);
        case Err::MSE_HS: return go<IT, Err::MSE_HS>(dual, a, s);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_colwise_tl(In it, Err em, bool dual, const ColArgs& a, cudaStream_t s) {
    switch (it) {
        case In::BF16: return by_err<In::BF16>(em, dual, a, s);
        case In::F16: return by_err<In::F16>(em, dual, a, s);
        case In::F32: return by_err<In::F32>(em, dual, a, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace fos

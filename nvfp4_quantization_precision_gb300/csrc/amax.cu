// Instantiations of the amax passes.
#include "fos_launch.cuh"

namespace fos {

template <In IT>
static cudaError_t by_scope(Src scope, const AmaxArgs& a, cudaStream_t s) {
    switch (scope) {
        case Src::TENSOR:
            return launch_persistent(k_amax_tensor<IT>, a, a.units, 0, s);
        case Src::ROW:
            return launch_persistent(k_amax_rows<IT>, a, (a.rows + 0), 0, s);
        case Src::GROUP:
            return launch_persistent(k_amax_groups<IT>, a, a.rows, sizeof(int32_t) * (size_t)a.G,
                                     s);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_amax(In it, Src scope, const AmaxArgs& a, cudaStream_t s) {
    switch (it) {
        case In::BF16: return by_scope<In::BF16>(scope, a, s);
        case In::F16: return by_scope<In::F16>(scope, a, s);
        case In::F32: return by_scope<In::F32>(scope, a, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace fos

// Instantiations of the fused quantize-dequantize list kernel.
#include "fos_launch.cuh"

namespace fos {

template <In IT>
static cudaError_t by_err(Err em, const QdqArgs& a, cudaStream_t s) {
    switch (em) {
        case Err::STD: return launch_persistent(k_qdq1x16<IT, Err::STD>, a, a.units, qdq_table_bytes(a.n), s);
        case Err::MAE: return launch_persistent(k_qdq1x16<IT, Err::MAE>, a, a.units, qdq_table_bytes(a.n), s);
        case Err::MSE: return launch_persistent(k_qdq1x16<IT, Err::MSE>, a, a.units, qdq_table_bytes(a.n), s);
        case Err::MAE_H: return launch_persistent(k_qdq1x16<IT, Err::MAE_H>, a, a.units, qdq_table_bytes(a.n), s);
        case Err::MSE_H: return launch_persistent(k_qdq1x16<IT, Err::MSE_H>, a, a.units, qdq_table_bytes(a.n), s);
        case Err::MAE_S: return launch_persistent(k_qdq1x16<IT, Err::MAE_S>, a, a.units, qdq_table_bytes(a.n), s);
        case Err::MSE_S: return launch_persistent(k_qdq1x16<IT, Err::MSE_S>, a, a.units, qdq_table_bytes(a.n), s);
        case Err::MAE_HS: return launch_persistent(k_qdq1x16<IT, Err::MAE_HS>, a, a.units, qdq_table_bytes(a.n), s);
        case Err::MSE_HS: return launch_persistent(k_qdq1x16<IT, Err::MSE_HS>, a, a.units, qdq_table_bytes(a.n), s);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_qdq(In it, Err em, const QdqArgs& a, cudaStream_t s) {
    if (it == In::BF16) return by_err<In::BF16>(em, a, s);
    if (it == In::F16) return by_err<In::F16>(em, a, s);
    return cudaErrorInvalidValue;
}

}  // namespace fos

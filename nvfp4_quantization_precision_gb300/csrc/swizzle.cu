// Block-scale bytes rearranged into the tiled layout that block-scaled FP4
// GEMMs read (128-row x 4-column tiles of scale bytes, 512 bytes each).
#include "fos_launch.cuh"

namespace fos {

// One thread per 4-byte group: row r, scale columns 4k .. 4k+3 of the padded
// [pr, pc] scale matrix (zeros outside [rows, nb]).  Tile (r / 128, k) is
// tile number (r / 128) * (pc / 4) + k; inside it, row r % 128 = 32 i + j
// sits at byte 16 j + 4 i.
__global__ void __launch_bounds__(kThreads) k_swizzle_scales(const uint8_t* scales, int64_t rows,
                                                             int64_t nb, int64_t pr, int64_t pc,
                                                             uint8_t* out) {
    chain_wait();
    chain_release();
    const int64_t groups = pr * (pc / 4);
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g < groups; g += stride) {
        const int64_t r = g / (pc / 4), k = g % (pc / 4);
        uint32_t w = 0;
        if (r < rows) {
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const int64_t c = 4 * k + t;
                if (c < nb) w |= (uint32_t)scales[r * nb + c] << (8 * t);
            }
        }
        const int64_t tile = (r / 128) * (pc / 4) + k;
        const int64_t rr = r % 128;
        *reinterpret_cast<uint32_t*>(out + tile * 512 + (rr % 32) * 16 + (rr / 32) * 4) = w;
    }
}

cudaError_t launch_swizzle(const uint8_t* scales, int64_t rows, int64_t nb, uint8_t* out,
                           cudaStream_t s) {
    const int64_t pr = (rows + 127) / 128 * 128, pc = (nb + 3) / 4 * 4;
    const int64_t groups = pr * (pc / 4);
    if (groups == 0) return cudaSuccess;
    int64_t blocks = (groups + kThreads - 1) / kThreads;
    const int64_t cap = (int64_t)sm_count() * 8;
    if (blocks > cap) blocks = cap;
    k_swizzle_scales<<<(unsigned)blocks, kThreads, 0, s>>>(scales, rows, nb, pr, pc, out);
    return cudaGetLastError();
}

}  // namespace fos

// Block-scale bytes rearranged into the tiled layout that block-scaled FP4
// GEMMs read (128-row x 4-column tiles of scale bytes, 512 bytes each).
#include "fos_launch.cuh"

namespace fos {

// One thread per 16-byte chunk of the output.  Tile (tr, k) of the padded
// [pr, pc] scale matrix (zeros outside [rows, nb]) is tile number
// tr * (pc / 4) + k; its chunk j (j < 32) holds, at bytes 4 i .. 4 i + 3
// (i < 4), the scales of columns 4k .. 4k + 3 of row 128 tr + 32 i + j.
// Consecutive threads write consecutive chunks, so a warp stores one whole
// tile.  WORD: nb % 4 == 0 and scales 4-byte aligned, so the four scales of
// a row come in one 32-bit load; VEC: out 16-byte aligned.
template <bool WORD, bool VEC>
__global__ void __launch_bounds__(kThreads) k_swizzle_scales(const uint8_t* scales, int64_t rows,
                                                             int64_t nb, int64_t pr, int64_t pc,
                                                             uint8_t* out) {
    chain_wait();
    chain_release();
    const int64_t kt = pc / 4;
    const int64_t chunks = (pr / 128) * kt * 32;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t q = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; q < chunks; q += stride) {
        const int64_t tile = q >> 5;
        const int j = (int)(q & 31);
        const int64_t tr = tile / kt, k = tile % kt;
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int64_t r = tr * 128 + 32 * i + j;
            w[i] = 0;
            if (r < rows) {
                const uint8_t* row = scales + r * nb + 4 * k;
                if constexpr (WORD) {
                    w[i] = __ldg(reinterpret_cast<const uint32_t*>(row));
                } else {
#pragma unroll
                    for (int t = 0; t < 4; ++t)
                        if (4 * k + t < nb) w[i] |= (uint32_t)__ldg(row + t) << (8 * t);
                }
            }
        }
        uint8_t* dst = out + tile * 512 + 16 * j;
        if constexpr (VEC) {
            st128(dst, w);
        } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) st32(dst + 4 * i, w[i]);
        }
    }
}

cudaError_t launch_swizzle(const uint8_t* scales, int64_t rows, int64_t nb, uint8_t* out,
                           cudaStream_t s) {
    const int64_t pr = (rows + 127) / 128 * 128, pc = (nb + 3) / 4 * 4;
    const int64_t chunks = (pr / 128) * (pc / 4) * 32;
    if (chunks == 0) return cudaSuccess;
    int64_t blocks = (chunks + kThreads - 1) / kThreads;
    const int64_t cap = (int64_t)sm_count() * 8;
    if (blocks > cap) blocks = cap;
    const bool word = nb % 4 == 0 && (reinterpret_cast<uintptr_t>(scales) & 3) == 0;
    const bool vec = (reinterpret_cast<uintptr_t>(out) & 15) == 0;
    const unsigned g = (unsigned)blocks;
    if (word && vec)
        k_swizzle_scales<true, true><<<g, kThreads, 0, s>>>(scales, rows, nb, pr, pc, out);
    else if (word)
        k_swizzle_scales<true, false><<<g, kThreads, 0, s>>>(scales, rows, nb, pr, pc, out);
    else if (vec)
        k_swizzle_scales<false, true><<<g, kThreads, 0, s>>>(scales, rows, nb, pr, pc, out);
    else
        k_swizzle_scales<false, false><<<g, kThreads, 0, s>>>(scales, rows, nb, pr, pc, out);
    return cudaGetLastError();
}

}  // namespace fos

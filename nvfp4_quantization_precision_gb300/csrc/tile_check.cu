// Validation of the tile-uniform per-row amax that 16x16 blocks with a
// row-scaled global scale require: the 16 rows of a tile must share one
// amax, hence one global scale.
#include "fos_launch.cuh"

namespace fos {

// One thread per 16-row tile, grid-stride: a tile is uniform when its 16
// amax words are bitwise equal.  Each warp adds its count of non-uniform
// tiles to *bad with one atomic.
__global__ void __launch_bounds__(kThreads) k_check_tile_amax(const uint32_t* amax, int64_t tiles,
                                                              unsigned long long* bad) {
    chain_wait();
    chain_release();
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    uint32_t mine = 0;
    for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < tiles; t += stride) {
        const uint32_t* a = amax + 16 * t;
        const uint32_t a0 = a[0];
        uint32_t diff = 0;
#pragma unroll
        for (int i = 1; i < 16; ++i) diff |= a[i] ^ a0;
        mine += diff != 0u;
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) mine += __shfl_down_sync(0xffffffffu, mine, o);
    if ((threadIdx.x & 31) == 0 && mine) atomicAdd(bad, (unsigned long long)mine);
}

cudaError_t launch_check_tile_amax(const float* amax, int64_t rows, int64_t* bad,
                                   cudaStream_t s) {
    cudaError_t e = cudaMemsetAsync(bad, 0, sizeof(int64_t), s);
    if (e != cudaSuccess) return e;
    const int64_t tiles = rows / 16;
    if (tiles == 0) return cudaSuccess;
    int64_t blocks = (tiles + kThreads - 1) / kThreads;
    const int64_t cap = (int64_t)sm_count() * 4;
    if (blocks > cap) blocks = cap;
    k_check_tile_amax<<<(unsigned)blocks, kThreads, 0, s>>>(
        reinterpret_cast<const uint32_t*>(amax), tiles, reinterpret_cast<unsigned long long*>(bad));
    return cudaGetLastError();
}

}  // namespace fos

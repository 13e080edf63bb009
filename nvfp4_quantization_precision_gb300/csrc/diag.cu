// Element-wise access to the conversion primitives (fos_diag.h).
#include "fos_launch.cuh"
#include "../../include/fos_diag.h"

namespace fos {

__global__ void k_diag(int op, const void* in, void* out, int64_t n) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
        const float* fi = static_cast<const float*>(in);
        const uint8_t* bi = static_cast<const uint8_t*>(in);
        switch (op) {
            case FOS_DIAG_E2M1_ENCODE:
                if ((i & 1) == 0 && i + 1 < n) {
                    const uint32_t q = e2m1x2(pk(fi[i], fi[i + 1]));
                    static_cast<uint8_t*>(out)[i] = q & 0xFu;
                    static_cast<uint8_t*>(out)[i + 1] = (q >> 4) & 0xFu;
                }
                break;
            case FOS_DIAG_E2M1_DECODE: {
                float lo, hi;
                upk(f16x2_f32x2(e2m1x2_f16x2(bi[i] & 0xFu)), lo, hi);
                static_cast<float*>(out)[i] = lo;
                break;
            }
            case FOS_DIAG_E4M3_ENCODE:
                if ((i & 1) == 0 && i + 1 < n) {
                    const uint32_t c = e4m3x2(fi[i], fi[i + 1]);
                    static_cast<uint8_t*>(out)[i] = c & 0xFFu;
                    static_cast<uint8_t*>(out)[i + 1] = c >> 8;
                }
                break;
            case FOS_DIAG_E4M3_DECODE:
                static_cast<float*>(out)[i] = e4m3_f32(bi[i]);
                break;
            case FOS_DIAG_F16_ROUND:
                if ((i & 1) == 0 && i + 1 < n) {
                    float lo, hi;
                    upk(f16x2_f32x2(f32x2_f16x2(pk(fi[i], fi[i + 1]))), lo, hi);
                    static_cast<float*>(out)[i] = lo;
                    static_cast<float*>(out)[i + 1] = hi;
                }
                break;
            case FOS_DIAG_BF16_BITS:
            case FOS_DIAG_F16_BITS:
                if ((i & 1) == 0 && i + 1 < n) {
                    const uint64_t p = pk(fi[i], fi[i + 1]);
                    const uint32_t w = (op == FOS_DIAG_BF16_BITS) ? f32x2_bf16x2(p) : f32x2_f16x2(p);
                    static_cast<uint16_t*>(out)[i] = w & 0xFFFFu;
                    static_cast<uint16_t*>(out)[i + 1] = w >> 16;
                }
                break;
            case FOS_DIAG_DIV6:
                static_cast<float*>(out)[i] = div6_rn(fi[i]);
                break;
            case FOS_DIAG_SCALE_CODES:
                static_cast<uint16_t*>(out)[i] = (uint16_t)scale_codes(fi[i], 1.0f);
                break;
            default:
                break;
        }
    }
}

cudaError_t launch_diag(int op, const void* in, void* out, int64_t n, cudaStream_t s) {
    int64_t blocks = (n + 255) / 256;
    const int64_t cap = (int64_t)sm_count() * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    k_diag<<<(int)blocks, 256, 0, s>>>(op, in, out, n);
    return cudaGetLastError();
}

// One of the library's bounded waits against a condition that never comes
// true: which = 0, the fused launch's CTA-counter wait (counter word[1],
// error word word[0]); which = 1, the column-wise kernel's mbarrier wait on
// a phase nothing completes (word[0] = 1 when it gave up).
__global__ void __launch_bounds__(kThreads) k_wait_timeout(int which, uint32_t* word) {
    __shared__ float s_amax;
    __shared__ __align__(8) uint64_t s_bar;
    if (which == 0) {
        fused_wait(&word[1], &word[1], 1u, &word[0], &s_amax);
    } else {
        if (threadIdx.x == 0) {
            mbar_init(&s_bar, 1);
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        }
        __syncthreads();
        const bool ok = mbar_wait(&s_bar, 0u);
        if (threadIdx.x == 0) word[0] = ok ? 0u : 1u;
    }
}

cudaError_t launch_wait_timeout(int which, uint32_t* word, cudaStream_t s) {
    cudaError_t e = cudaMemsetAsync(word, 0, 2 * sizeof(uint32_t), s);
    if (e != cudaSuccess) return e;
    k_wait_timeout<<<1, kThreads, 0, s>>>(which, word);
    return cudaGetLastError();
}

}  // namespace fos

// mm.cu -- A . B^T from quantized operands: the block-scaled product runs as
// a cuBLASLt NVFP4 GEMM (a library GEMM: fp32 accumulation, no workspace),
// then this library's epilogue applies the global decode scales per row.
#include <cublasLt.h>

#include <mutex>
#include <unordered_map>

#include "fos_launch.cuh"

namespace fos {

// out[m][n] = (D[m][n] * g_a(m)) * g_b, g = rn(1 / S) of the global scale S
// that quantization used (per row of a when row-scaled).  Four elements per
// thread (N is a multiple of 16).
__global__ void __launch_bounds__(kThreads) k_mm_epilogue(float* out, const float* a_amax,
                                                         int a_row, const float* b_amax,
                                                         int64_t M, int64_t N, float six_bound) {
    chain_wait();
    chain_release();
    const float gb = fdiv(1.0f, global_scale(b_amax[0], six_bound));
    const float ga0 = a_row ? 0.0f : fdiv(1.0f, global_scale(a_amax[0], six_bound));
    const int64_t quads = M * (N / 4);
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t q = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; q < quads; q += stride) {
        const int64_t m = q / (N / 4);
        const float ga = a_row ? fdiv(1.0f, global_scale(a_amax[m], six_bound)) : ga0;
        float4 v = reinterpret_cast<float4*>(out)[q];
        v.x = fmul(fmul(v.x, ga), gb);
        v.y = fmul(fmul(v.y, ga), gb);
        v.z = fmul(fmul(v.z, ga), gb);
        v.w = fmul(fmul(v.w, ga), gb);
        reinterpret_cast<float4*>(out)[q] = v;
    }
}

// One cuBLASLt handle per device (host-side object), created on first use.
static cublasLtHandle_t lt_handle(int dev) {
    static std::mutex mu;
    static std::unordered_map<int, cublasLtHandle_t> handles;
    std::lock_guard<std::mutex> g(mu);
    auto it = handles.find(dev);
    if (it != handles.end()) return it->second;
    cublasLtHandle_t h = nullptr;
    if (cublasLtCreate(&h) != CUBLAS_STATUS_SUCCESS) return nullptr;
    handles[dev] = h;
    return h;
}

// 0: done; 1: the library offers no algorithm for this shape; 2: a cuBLASLt
// or CUDA call failed.
int run_mm(const uint8_t* a_codes, const uint8_t* a_scales, const float* a_amax, int a_row,
           const uint8_t* b_codes, const uint8_t* b_scales, const float* b_amax, int64_t M,
           int64_t N, int64_t K, float six_bound, float* out, int dev, cudaStream_t s) {
    cublasLtHandle_t h = lt_handle(dev);
    if (!h) return 2;
    // Column-major view: D (N x M, ld N) = op(A') (N x K) * op(B') (K x M), with
    // A' = b's codes as K x N (each column one row of b, K contiguous; op = T)
    // and B' = a's codes as K x M (op = N); D column-major is out row-major.
    cublasLtMatmulDesc_t op = nullptr;
    cublasLtMatrixLayout_t la = nullptr, lb = nullptr, ld = nullptr;
    cublasLtMatmulPreference_t pref = nullptr;
    int rc = 2;
    do {
        if (cublasLtMatmulDescCreate(&op, CUBLAS_COMPUTE_32F, CUDA_R_32F) != CUBLAS_STATUS_SUCCESS)
            break;
        const cublasOperation_t ta = CUBLAS_OP_T, tb = CUBLAS_OP_N;
        const cublasLtMatmulMatrixScale_t mode = CUBLASLT_MATMUL_MATRIX_SCALE_VEC16_UE4M3;
        const void* sa = b_scales;  // scales of cuBLAS's A (our b)
        const void* sb = a_scales;  // scales of cuBLAS's B (our a)
        if (cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_TRANSA, &ta, sizeof(ta)) ||
            cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_TRANSB, &tb, sizeof(tb)) ||
            cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_A_SCALE_MODE, &mode,
                                           sizeof(mode)) ||
            cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_B_SCALE_MODE, &mode,
                                           sizeof(mode)) ||
            cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_A_SCALE_POINTER, &sa,
                                           sizeof(sa)) ||
            cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_B_SCALE_POINTER, &sb,
                                           sizeof(sb)))
            break;
        if (cublasLtMatrixLayoutCreate(&la, CUDA_R_4F_E2M1, K, N, K) ||
            cublasLtMatrixLayoutCreate(&lb, CUDA_R_4F_E2M1, K, M, K) ||
            cublasLtMatrixLayoutCreate(&ld, CUDA_R_32F, N, M, N))
            break;
        if (cublasLtMatmulPreferenceCreate(&pref)) break;
        const size_t ws = 0;
        if (cublasLtMatmulPreferenceSetAttribute(pref, CUBLASLT_MATMUL_PREF_MAX_WORKSPACE_BYTES,
                                                 &ws, sizeof(ws)))
            break;
        cublasLtMatmulHeuristicResult_t res = {};
        int found = 0;
        if (cublasLtMatmulAlgoGetHeuristic(h, op, la, lb, ld, ld, pref, 1, &res, &found) ||
            found < 1) {
            rc = 1;
            break;
        }
        const float alpha = 1.0f, beta = 0.0f;
        if (cublasLtMatmul(h, op, &alpha, b_codes, la, a_codes, lb, &beta, out, ld, out, ld,
                           &res.algo, nullptr, 0, s))
            break;
        int64_t quads = M * (N / 4);
        int64_t blocks = (quads + kThreads - 1) / kThreads;
        const int64_t cap = (int64_t)sm_count() * 8;
        if (blocks > cap) blocks = cap;
        k_mm_epilogue<<<(unsigned)blocks, kThreads, 0, s>>>(out, a_amax, a_row, b_amax, M, N,
                                                            six_bound);
        rc = cudaGetLastError() == cudaSuccess ? 0 : 2;
    } while (false);
    if (pref) cublasLtMatmulPreferenceDestroy(pref);
    if (ld) cublasLtMatrixLayoutDestroy(ld);
    if (lb) cublasLtMatrixLayoutDestroy(lb);
    if (la) cublasLtMatrixLayoutDestroy(la);
    if (op) cublasLtMatmulDescDestroy(op);
    return rc;
}

}  // namespace fos

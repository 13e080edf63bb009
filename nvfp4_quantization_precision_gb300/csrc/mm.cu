// mm.cu -- A . B^T from quantized operands: the block-scaled product runs as
// a cuBLASLt NVFP4 GEMM (a library GEMM: fp32 accumulation, no workspace),
// then this library's epilogue applies the global decode scales per row.
#include <cublasLt.h>

#include <mutex>
#include <unordered_map>

#include "fos_launch.cuh"

namespace fos {

// out[m][n] = (D[m][n] * g_a(m)) * g_b, g = rn(1 / S) of the global scale S
// that quantization used (per row of a when row-scaled).  A CTA takes whole
// rows (one g_a each), its threads four columns at a time (N is a multiple
// of 16).
__global__ void __launch_bounds__(kThreads) k_mm_epilogue(float* out, const float* a_amax,
                                                         int a_row, const float* b_amax,
                                                         int64_t M, int64_t N, float six_bound) {
    chain_wait();
    chain_release();
    const float gb = fdiv(1.0f, global_scale(b_amax[0], six_bound));
    const float ga0 = a_row ? 0.0f : fdiv(1.0f, global_scale(a_amax[0], six_bound));
    const int64_t nq = N / 4;
    for (int64_t m = blockIdx.x; m < M; m += gridDim.x) {
        const float ga = a_row ? fdiv(1.0f, global_scale(a_amax[m], six_bound)) : ga0;
        float4* row = reinterpret_cast<float4*>(out + m * N);
        for (int64_t q = threadIdx.x; q < nq; q += blockDim.x) {
            float4 v = row[q];
            v.x = fmul(fmul(v.x, ga), gb);
            v.y = fmul(fmul(v.y, ga), gb);
            v.z = fmul(fmul(v.z, ga), gb);
            v.w = fmul(fmul(v.w, ga), gb);
            row[q] = v;
        }
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

// Largest power of two (at most 256) that divides the address.
static uint32_t align_of(const void* p) {
    const uintptr_t v = reinterpret_cast<uintptr_t>(p);
    uint32_t a = 256;
    while (a > 1 && (v & (a - 1))) a >>= 1;
    return a;
}

// The cuBLASLt objects of one product, built once per call: the operation
// (our b as cuBLAS's A, our a as its B) and b's layout, and for each row-chunk
// height of a the layouts of the a chunk and of the output chunk with the
// algorithm the heuristic picks for them.  Column-major view of one chunk:
// D (N x rows, ld N) = op(A') (N x K) * op(B') (K x rows), with A' = b's codes
// as K x N (each column one row of b, K contiguous; op = T) and B' = the a
// chunk's codes as K x rows (op = N); D column-major is out row-major.
struct LtPlan {
    struct Shape {
        int64_t rows = -1;
        cublasLtMatrixLayout_t lb = nullptr, ld = nullptr;
        cublasLtMatmulAlgo_t algo;
    };
    cublasLtHandle_t h = nullptr;
    cublasLtMatmulDesc_t op = nullptr;
    cublasLtMatrixLayout_t la = nullptr;
    cublasLtMatmulPreference_t pref = nullptr;
    Shape sh[2];

    ~LtPlan() {
        for (Shape& x : sh) {
            if (x.ld) cublasLtMatrixLayoutDestroy(x.ld);
            if (x.lb) cublasLtMatrixLayoutDestroy(x.lb);
        }
        if (pref) cublasLtMatmulPreferenceDestroy(pref);
        if (la) cublasLtMatrixLayoutDestroy(la);
        if (op) cublasLtMatmulDescDestroy(op);
    }

    // 0: ready; 2: a call failed.  Chunks start on multiples of 256 rows, so
    // every chunk pointer has the alignment of its base pointer (capped at
    // 256 bytes, which the heuristic otherwise assumes).
    int init(const uint8_t* a_codes, const uint8_t* a_scales, const uint8_t* b_codes,
             const uint8_t* b_scales, const float* out, int64_t N, int64_t K) {
        if (cublasLtMatmulDescCreate(&op, CUBLAS_COMPUTE_32F, CUDA_R_32F) != CUBLAS_STATUS_SUCCESS)
            return 2;
        const cublasOperation_t ta = CUBLAS_OP_T, tb = CUBLAS_OP_N;
        const cublasLtMatmulMatrixScale_t mode = CUBLASLT_MATMUL_MATRIX_SCALE_VEC16_UE4M3;
        const void* sa = b_scales;  // scales of cuBLAS's A (our b)
        const void* sb = a_scales;  // scales of cuBLAS's B (our a; moved to each chunk's)
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
            return 2;
        if (cublasLtMatrixLayoutCreate(&la, CUDA_R_4F_E2M1, K, N, K)) return 2;
        if (cublasLtMatmulPreferenceCreate(&pref)) return 2;
        const size_t ws = 0;
        const uint32_t al_a = align_of(b_codes), al_b = align_of(a_codes), al_d = align_of(out);
        if (cublasLtMatmulPreferenceSetAttribute(pref, CUBLASLT_MATMUL_PREF_MAX_WORKSPACE_BYTES,
                                                 &ws, sizeof(ws)) ||
            cublasLtMatmulPreferenceSetAttribute(pref, CUBLASLT_MATMUL_PREF_MIN_ALIGNMENT_A_BYTES,
                                                 &al_a, sizeof(al_a)) ||
            cublasLtMatmulPreferenceSetAttribute(pref, CUBLASLT_MATMUL_PREF_MIN_ALIGNMENT_B_BYTES,
                                                 &al_b, sizeof(al_b)) ||
            cublasLtMatmulPreferenceSetAttribute(pref, CUBLASLT_MATMUL_PREF_MIN_ALIGNMENT_C_BYTES,
                                                 &al_d, sizeof(al_d)) ||
            cublasLtMatmulPreferenceSetAttribute(pref, CUBLASLT_MATMUL_PREF_MIN_ALIGNMENT_D_BYTES,
                                                 &al_d, sizeof(al_d)))
            return 2;
        return 0;
    }

    // Layouts and algorithm for chunks of `rows` rows into slot i.  0: ready;
    // 1: the library offers no algorithm; 2: a call failed.
    int shape(int i, int64_t rows, int64_t N, int64_t K) {
        Shape& x = sh[i];
        x.rows = rows;
        if (cublasLtMatrixLayoutCreate(&x.lb, CUDA_R_4F_E2M1, K, rows, K) ||
            cublasLtMatrixLayoutCreate(&x.ld, CUDA_R_32F, N, rows, N))
            return 2;
        cublasLtMatmulHeuristicResult_t res = {};
        int found = 0;
        if (cublasLtMatmulAlgoGetHeuristic(h, op, la, x.lb, x.ld, x.ld, pref, 1, &res, &found) ||
            found < 1)
            return 1;
        x.algo = res.algo;
        return 0;
    }

    // One chunk: its a codes and tiled scales against all of b.
    int run(const Shape& x, const uint8_t* a_codes, const uint8_t* a_scales,
            const uint8_t* b_codes, float* out, cudaStream_t s) {
        const void* sb = a_scales;  // scales of cuBLAS's B (our a chunk)
        if (cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_B_SCALE_POINTER, &sb,
                                           sizeof(sb)))
            return 2;
        const float alpha = 1.0f, beta = 0.0f;
        if (cublasLtMatmul(h, op, &alpha, b_codes, la, a_codes, x.lb, &beta, out, x.ld, out, x.ld,
                           &x.algo, nullptr, 0, s))
            return 2;
        return 0;
    }
};

// Rows of a per GEMM: a multiple of 256 whose fp32 output slice takes about
// half of the L2, so that the epilogue that follows each GEMM reads D back
// from L2 instead of HBM; all of M when it fits.
static int64_t chunk_rows(int64_t M, int64_t N, int dev) {
    int l2 = 0;
    if (cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev) != cudaSuccess) {
        cudaGetLastError();
        return M;
    }
    int64_t mc = (int64_t)l2 / 2 / (N * 4) / 256 * 256;
    if (mc < 256) mc = 256;
    return mc >= M ? M : mc;
}

// 0: done; 1: the library offers no algorithm for this shape; 2: a cuBLASLt
// or CUDA call failed.
int run_mm(const uint8_t* a_codes, const uint8_t* a_scales, const float* a_amax, int a_row,
           const uint8_t* b_codes, const uint8_t* b_scales, const float* b_amax, int64_t M,
           int64_t N, int64_t K, float six_bound, float* out, int dev, cudaStream_t s) {
    LtPlan plan;
    plan.h = lt_handle(dev);
    if (!plan.h) return 2;
    int rc = plan.init(a_codes, a_scales, b_codes, b_scales, out, N, K);
    if (rc) return rc;
    const int64_t mc = chunk_rows(M, N, dev);
    const int64_t tail = M % mc;
    if ((rc = plan.shape(0, mc, N, K))) return rc;
    if (tail && (rc = plan.shape(1, tail, N, K))) return rc;
    // a's tiled scales: 128-row tile rows of 128 * (K / 16) bytes (K % 64 == 0),
    // so a chunk that starts on a multiple of 128 rows starts at m0 * K / 16.
    for (int64_t m0 = 0; m0 < M; m0 += mc) {
        const int64_t rows = (M - m0 < mc) ? (M - m0) : mc;
        rc = plan.run(rows == mc ? plan.sh[0] : plan.sh[1], a_codes + m0 * (K / 2),
                      a_scales + m0 * (K / 16), b_codes, out + m0 * N, s);
        if (rc) return rc;
        int64_t blocks = rows;
        const int64_t cap = (int64_t)sm_count() * 8;
        if (blocks > cap) blocks = cap;
        k_mm_epilogue<<<(unsigned)blocks, kThreads, 0, s>>>(
            out + m0 * N, a_amax + (a_row ? m0 : 0), a_row, b_amax, rows, N, six_bound);
        if (cudaGetLastError() != cudaSuccess) return 2;
    }
    return 0;
}

}  // namespace fos

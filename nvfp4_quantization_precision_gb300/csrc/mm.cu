// mm.cu -- A . B^T from quantized operands on the tensor cores: the launch of
// the persistent block-scaled NVFP4 kernel (fos_mma.cuh) with its three TMA
// descriptors (a codes, b codes, out).
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

#include "fos_launch.cuh"
#include "fos_mma.cuh"

namespace fos {

namespace {

// Epilogue shape of the launch: warps and staging chunks per warp.
constexpr int kMmEpi = 4;
constexpr int kMmBufs = 2;

// cuTensorMapEncodeTiled is a driver function; its address comes from the
// runtime once (no link against the driver library).
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        else
            cudaGetLastError();
    });
    return fn;
}

// Codes [rows, K/2] bytes as a 2D tensor, box 128 bytes x box_rows rows with
// the 128-byte swizzle the MMA descriptors expect; rows past the end read 0.
bool code_map(CUtensorMap* map, const uint8_t* codes, int64_t rows, int64_t K, int box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)(K / 2), (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)(K / 2)};
    const cuuint32_t box[2] = {(cuuint32_t)mma::kKBytes, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(codes), dims, strides,
              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// out [M, N] fp32 as a 2D tensor, box 32 columns x 32 rows (one epilogue
// chunk, 128 bytes wide) with the 128-byte swizzle of the staging chunks.
// N % 16 == 0 makes the row pitch a multiple of 16 bytes.
bool out_map(CUtensorMap* map, float* out, int64_t M, int64_t N) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)N, (cuuint64_t)M};
    const cuuint64_t strides[1] = {(cuuint64_t)N * 4};
    const cuuint32_t box[2] = {32, 32};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, out, dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// 0: launched; 2: a descriptor or the launch failed.
int run_mm(const uint8_t* a_codes, const uint8_t* a_scales, const float* a_amax, int a_row,
           const uint8_t* b_codes, const uint8_t* b_scales, const float* b_amax, int64_t M,
           int64_t N, int64_t K, float six_bound, float* out, cudaStream_t s) {
    mma::MmArgs a;
    std::memset(&a, 0, sizeof(a));
    if (!code_map(&a.ta, a_codes, M, K, mma::BM) || !code_map(&a.tb, b_codes, N, K, mma::BN) ||
        !out_map(&a.to, out, M, N))
        return 2;
    a.sfa = a_scales;
    a.sfb = b_scales;
    a.a_amax = a_amax;
    a.b_amax = b_amax;
    a.out = out;
    a.M = M;
    a.N = N;
    a.K = K;
    a.tiles_m = (M + mma::BM - 1) / mma::BM;
    a.tiles_n = (N + mma::BN - 1) / mma::BN;
    a.a_row = a_row;
    a.six_bound = six_bound;
    const int64_t tiles = a.tiles_m * a.tiles_n;
    auto kernel = mma::k_mm_nvfp4<kMmEpi, kMmBufs>;
    constexpr int smem = mma::smem_bytes<kMmEpi, kMmBufs>();
    static std::once_flag once;
    static cudaError_t attr = cudaSuccess;
    std::call_once(once, [&] {
        attr = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    });
    if (attr != cudaSuccess) return 2;
    // persistent: one CTA per SM (the tensor memory and shared memory of a
    // CTA take an SM), never more CTAs than tiles
    const int64_t sms = sm_count();
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(tiles < sms ? tiles : sms));
    cfg.blockDim = dim3(mma::threads_mm(kMmEpi));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kernel, a) != cudaSuccess) {
        cudaGetLastError();
        return 2;
    }
    return cudaGetLastError() == cudaSuccess ? 0 : 2;
}

}  // namespace fos

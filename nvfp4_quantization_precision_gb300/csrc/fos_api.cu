// fos_api.cu -- host side of the C ABI declared in include/fos.h.
//
// Every entry point validates all arguments before touching the CUDA
// runtime, switches to the device that owns the data, enqueues its kernels on
// the caller's stream and restores the caller's current device (the
// Megatron fused-QDQ PR tests that the kernel "uses and restores" a
// non-current device).  Nothing here allocates device memory or synchronises
// the host.
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include <cudaTypedefs.h>

#include "../../include/fos.h"
#include "../../include/fos_diag.h"
#include "fos_launch.cuh"

using namespace fos;

namespace {

constexpr int kVersion = 10000;  // 1.0.0

bool valid_dtype(int dt) { return dt == FOS_BF16 || dt == FOS_FP16 || dt == FOS_FP32; }

fos_status check_config(const fos_config* cfg) {
    if (!cfg) return FOS_ERR_INVALID_ARG;
    if (cfg->block != FOS_BLOCK_1X16 && cfg->block != FOS_BLOCK_16X16) return FOS_ERR_INVALID_ARG;
    if (cfg->mode != FOS_MODE_STANDARD && cfg->mode != FOS_MODE_4OVER6) return FOS_ERR_INVALID_ARG;
    if (cfg->err_metric != FOS_MAE && cfg->err_metric != FOS_MSE) return FOS_ERR_INVALID_ARG;
    if (cfg->err_precision != FOS_ERR_EXACT_F32 && cfg->err_precision != FOS_ERR_F16)
        return FOS_ERR_INVALID_ARG;
    if (cfg->granularity != FOS_SCALE_TENSOR && cfg->granularity != FOS_SCALE_ROW)
        return FOS_ERR_INVALID_ARG;
    if (cfg->amax_is_input != 0 && cfg->amax_is_input != 1) return FOS_ERR_INVALID_ARG;
    if (cfg->err_order != FOS_ORDER_TREE && cfg->err_order != FOS_ORDER_SEQ)
        return FOS_ERR_INVALID_ARG;
    if (cfg->scale_layout != FOS_SCALES_PLAIN && cfg->scale_layout != FOS_SCALES_TILED)
        return FOS_ERR_INVALID_ARG;
    if (cfg->e4m3_bound != 448 && cfg->e4m3_bound != 256) return FOS_ERR_UNSUPPORTED;
    return FOS_OK;
}

bool tiled(const fos_config* cfg) { return cfg->scale_layout == FOS_SCALES_TILED; }

// Scales in the tiled GEMM layout are written for 1x16 blocks and fewer than
// 2^30 rows (the kernels keep block positions in 32 bits).
fos_status check_layout(const fos_config* cfg, int64_t rows) {
    if (tiled(cfg) && (cfg->block != FOS_BLOCK_1X16 || rows >= (INT64_C(1) << 30)))
        return FOS_ERR_UNSUPPORTED;
    return FOS_OK;
}

// 4-block tiles per tile-row of the tiled scale layout of [rows, cols].
int64_t tiled_pc4(int64_t cols) { return (cols / 16 + 3) / 4; }

// The tiled layout pads the scale matrix to whole 128 x 4 tiles; the padding
// must read as zero scales, so when there is any the buffer is cleared
// before the kernel writes the real scales.
cudaError_t clear_tiled_padding(uint8_t* scales, int64_t rows, int64_t cols, cudaStream_t s) {
    if (rows % 128 == 0 && (cols / 16) % 4 == 0) return cudaSuccess;
    const size_t bytes = (size_t)((rows + 127) / 128 * 128) * (size_t)(tiled_pc4(cols) * 4);
    return cudaMemsetAsync(scales, 0, bytes, s);
}

// The sequential term order is offered for 1x16 blocks (its source is a 1x16
// path); standard mode has no candidate errors, so the knob is moot there.
fos_status check_order(const fos_config* cfg) {
    if (cfg->err_order == FOS_ORDER_SEQ && cfg->block == FOS_BLOCK_16X16 &&
        cfg->mode == FOS_MODE_4OVER6)
        return FOS_ERR_UNSUPPORTED;
    return FOS_OK;
}

Err err_of(const fos_config* cfg) {
    if (cfg->mode == FOS_MODE_STANDARD) return Err::STD;
    const bool mse = cfg->err_metric == FOS_MSE, h = cfg->err_precision == FOS_ERR_F16;
    if (cfg->err_order == FOS_ORDER_SEQ) {
        if (mse) return h ? Err::MSE_HS : Err::MSE_S;
        return h ? Err::MAE_HS : Err::MAE_S;
    }
    if (mse) return h ? Err::MSE_H : Err::MSE;
    return h ? Err::MAE_H : Err::MAE;
}

fos_status check_shape(int64_t rows, int64_t cols, bool b16) {
    if (rows < 0 || cols < 0) return FOS_ERR_INVALID_ARG;
    if (cols % 16 != 0) return FOS_ERR_UNSUPPORTED;
    if (b16 && rows % 16 != 0) return FOS_ERR_UNSUPPORTED;
    // keeps every byte offset of the kernels inside int64
    if (cols > 0 && rows > (int64_t)(INT64_C(1) << 40) / cols) return FOS_ERR_UNSUPPORTED;
    return FOS_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Device that owns a pointer, or -1 when the pointer is not device memory.
int device_of(const void* p) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();
        return -1;
    }
    if (at.type != cudaMemoryTypeDevice && at.type != cudaMemoryTypeManaged) return -1;
    return at.device;
}

// Switches to the device owning the data for the lifetime of the object.
struct DeviceScope {
    int prev = -1;
    int dev = -1;
    bool switched = false;
    fos_status st = FOS_OK;
    explicit DeviceScope(int d) : dev(d) {
        if (cudaGetDevice(&prev) != cudaSuccess) {
            cudaGetLastError();
            st = FOS_ERR_CUDA;
            return;
        }
        if (prev != dev) {
            if (cudaSetDevice(dev) != cudaSuccess) {
                cudaGetLastError();
                st = FOS_ERR_CUDA;
                return;
            }
            switched = true;
        }
    }
    ~DeviceScope() {
        if (switched) cudaSetDevice(prev);
    }
};

// All listed device pointers must live on one device; returns it or -1.
int common_device(std::initializer_list<const void*> ptrs) {
    int dev = -1;
    for (const void* p : ptrs) {
        const int d = device_of(p);
        if (d < 0) return -1;
        if (dev >= 0 && d != dev) return -1;
        dev = d;
    }
    return dev;
}

fos_status cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return FOS_OK;
    cudaGetLastError();
    return FOS_ERR_CUDA;
}

In in_of(fos_dtype dt) { return dt == FOS_BF16 ? In::BF16 : (dt == FOS_FP16 ? In::F16 : In::F32); }

cudaError_t run_amax(const void* x, fos_dtype dt, int64_t rows, int64_t cols, Src scope,
                     float* amax, const int32_t* offs, int G, cudaStream_t s,
                     float* clear = nullptr) {
    AmaxArgs a{};
    a.x = x;
    a.amax = amax;
    a.clear = clear;
    a.offs = offs;
    a.G = G;
    a.rows = rows;
    a.nb = cols / 16;
    a.units = (rows * a.nb + 31) / 32;
    if (scope == Src::TENSOR || scope == Src::GROUP) {
        const size_t n = (scope == Src::TENSOR) ? 1 : (size_t)G;
        cudaError_t e = cudaMemsetAsync(amax, 0, sizeof(float) * n, s);
        if (e != cudaSuccess) return e;
        if (rows == 0 || cols == 0) return cudaSuccess;
    }
    if (rows == 0) return cudaSuccess;
    if (cols == 0) return cudaMemsetAsync(amax, 0, sizeof(float) * (size_t)rows, s);
    return launch_amax(in_of(dt), scope, a, s);
}

// Per-tensor amax into a buffer that is already +0 (no memset).
cudaError_t run_amax_cleared(const void* x, fos_dtype dt, int64_t rows, int64_t cols,
                             float* amax, cudaStream_t s, float* clear = nullptr) {
    AmaxArgs a{};
    a.x = x;
    a.amax = amax;
    a.clear = clear;
    a.rows = rows;
    a.nb = cols / 16;
    a.units = (rows * a.nb + 31) / 32;
    if (rows == 0 || cols == 0) {
        if (clear) return cudaMemsetAsync(clear, 0, sizeof(float), s);
        return cudaSuccess;
    }
    return launch_amax(in_of(dt), Src::TENSOR, a, s);
}

cudaError_t run_quant(const void* x, fos_dtype dt, int64_t rows, int64_t cols,
                      const fos_config* cfg, const float* amax, Src src, const int32_t* offs,
                      int G, uint8_t* codes, uint8_t* scales, cudaStream_t s) {
    if (rows == 0 || cols == 0) return cudaSuccess;
    EncArgs a{};
    a.x = x;
    a.codes = codes;
    a.scales = scales;
    a.amax = amax;
    a.offs = offs;
    a.G = G;
    a.rows = rows;
    a.nb = cols / 16;
    a.nblk = rows * a.nb;
    a.six_bound = 6.0f * (float)cfg->e4m3_bound;
    a.neg_zero = -0.0f;
    const Err em = err_of(cfg);
    const In it = in_of(dt);
    if (cfg->block == FOS_BLOCK_16X16) {
        a.cpr = (a.nb + 3) / 4;  // tile quads per 16-row band
        a.units = (rows / 16) * a.cpr;
        switch (it) {
            case In::BF16: return launch_quant16x16_bf16(em, src, a, s);
            case In::F16: return launch_quant16x16_f16(em, src, a, s);
            case In::F32: return launch_quant16x16_f32(em, src, a, s);
        }
    } else {
        a.cpr = (a.nb + 31) / 32;
        a.units = (src == Src::TENSOR) ? (a.nblk + 31) / 32 : rows * a.cpr;
        if (tiled(cfg) && src != Src::GROUP) {
            a.sc_pc4 = tiled_pc4(cols);
            switch (it) {
                case In::BF16: return launch_quant1x16_tl_bf16(em, src, a, s);
                case In::F16: return launch_quant1x16_tl_f16(em, src, a, s);
                case In::F32: return launch_quant1x16_tl_f32(em, src, a, s);
            }
        }
        switch (it) {
            case In::BF16: return launch_quant1x16_bf16(em, src, a, s);
            case In::F16: return launch_quant1x16_f16(em, src, a, s);
            case In::F32: return launch_quant1x16_f32(em, src, a, s);
        }
    }
    return cudaErrorInvalidValue;
}

// One-pass row-scaled 1x16 quantize: a CTA per row, each thread holding up to
// K = 2 blocks of the row in registers (rows of 2048 .. 8192 columns).
// Returns 0 outside that range; the two-pass path (row amax, then encode)
// is used there.
int rowpass_k(int64_t nb) {
    if (nb < 128) return 0;  // short rows would leave most of a CTA idle
    if (nb <= kThreads) return 1;
    if (nb <= 2 * kThreads) return 2;
    return 0;
}

cudaError_t run_rowpass(const void* x, fos_dtype dt, int64_t rows, int64_t cols,
                        const fos_config* cfg, float* amax, uint8_t* codes, uint8_t* scales,
                        int k, cudaStream_t s) {
    EncArgs a{};
    a.x = x;
    a.codes = codes;
    a.scales = scales;
    a.amax = amax;
    a.rows = rows;
    a.nb = cols / 16;
    a.nblk = rows * a.nb;
    a.six_bound = 6.0f * (float)cfg->e4m3_bound;
    a.neg_zero = -0.0f;
    a.amax_given = cfg->amax_is_input;
    const Err em = err_of(cfg);
    if (tiled(cfg)) {
        a.sc_pc4 = tiled_pc4(cols);
        switch (in_of(dt)) {
            case In::BF16: return launch_quant1x16_rowpass_tl_bf16(em, k, a, s);
            case In::F16: return launch_quant1x16_rowpass_tl_f16(em, k, a, s);
            case In::F32: return launch_quant1x16_rowpass_tl_f32(em, k, a, s);
        }
        return cudaErrorInvalidValue;
    }
    switch (in_of(dt)) {
        case In::BF16: return launch_quant1x16_rowpass_bf16(em, k, a, s);
        case In::F16: return launch_quant1x16_rowpass_f16(em, k, a, s);
        case In::F32: return launch_quant1x16_rowpass_f32(em, k, a, s);
    }
    return cudaErrorInvalidValue;
}

// Encode x (1x16, per-tensor amax given) and, in the same launch, the amax
// pass of x_next (cleared first).  Without x_next it is a plain encode.
// With next_cleared the caller guarantees amax_next is already +0 (the list
// clears it one stage earlier); clear_ahead, when set, is zeroed by this
// launch for a later stage.
fos_status overlap_one(const void* x, fos_dtype dt, int64_t rows, int64_t cols,
                       const fos_config* cfg, const float* amax, uint8_t* codes, uint8_t* scales,
                       const void* x_next, int64_t rows_next, int64_t cols_next, float* amax_next,
                       cudaStream_t s, bool next_cleared = false, float* clear_ahead = nullptr) {
    fos_status st = FOS_OK;
    const bool next = amax_next != nullptr;
    const bool next_live = next && rows_next > 0 && cols_next > 0;
    if (clear_ahead && !(next_live && rows > 0 && cols > 0)) {
        // this stage does not launch the overlapped kernel: clear directly
        st = cuda_status(cudaMemsetAsync(clear_ahead, 0, sizeof(float), s));
        if (st) return st;
        clear_ahead = nullptr;
    }
    if (next && !next_cleared) {
        st = cuda_status(cudaMemsetAsync(amax_next, 0, sizeof(float), s));
        if (st) return st;
    }
    if (rows == 0 || cols == 0) {
        if (next_live)
            return cuda_status(run_amax_cleared(x_next, dt, rows_next, cols_next, amax_next, s));
        return FOS_OK;
    }
    if (tiled(cfg)) {
        st = cuda_status(clear_tiled_padding(scales, rows, cols, s));
        if (st) return st;
    }
    if (!next_live)
        return cuda_status(run_quant(x, dt, rows, cols, cfg, amax, Src::TENSOR, nullptr, 0, codes,
                                     scales, s));
    PipeArgs p{};
    EncArgs& a = p.enc;
    a.x = x;
    a.codes = codes;
    a.scales = scales;
    a.amax = amax;
    a.rows = rows;
    a.nb = cols / 16;
    a.nblk = a.rows * a.nb;
    a.units = (a.nblk + 31) / 32;
    a.cpr = (a.nb + 31) / 32;
    a.six_bound = 6.0f * (float)cfg->e4m3_bound;
    a.neg_zero = -0.0f;
    p.clear = clear_ahead;
    p.ax = x_next;
    p.aamax = amax_next;
    p.aseg = rows_next * (cols_next / 16);
    p.aunits = (p.aseg + 31) / 32;
    if (tiled(cfg)) {
        a.sc_pc4 = tiled_pc4(cols);
        return cuda_status(launch_pipe_tl(in_of(dt), err_of(cfg), p, s));
    }
    return cuda_status(launch_pipe(in_of(dt), err_of(cfg), p, s));
}

// Shape / pointer / alignment checks of one quantize call (no CUDA calls).
fos_status check_quant_args(const void* x, int64_t rows, int64_t cols, const fos_config* cfg,
                            const float* amax, const uint8_t* codes, const uint8_t* scales) {
    fos_status st = check_shape(rows, cols, cfg->block == FOS_BLOCK_16X16);
    if (st) return st;
    st = check_order(cfg);
    if (st) return st;
    st = check_layout(cfg, rows);
    if (st) return st;
    if (rows == 0 || cols == 0) {
        if (!cfg->amax_is_input && !(cfg->granularity == FOS_SCALE_ROW && rows == 0) && !amax)
            return FOS_ERR_INVALID_ARG;
        return FOS_OK;
    }
    if (!x || !amax || !codes || !scales) return FOS_ERR_INVALID_ARG;
    if (!aligned(x, 32) || !aligned(codes, 8)) return FOS_ERR_MISALIGNED;
    return FOS_OK;
}

// 2D TMA descriptor of x [rows, cols] with the column-wise tile as its box.
// cuTensorMapEncodeTiled is a driver function; its address comes from the
// runtime once (no link against the driver library).
fos_status encode_tile_map(CUtensorMap* map, const void* x, fos_dtype dt, int64_t rows,
                           int64_t cols) {
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
    if (!fn) return FOS_ERR_CUDA;
    const bool f32 = dt == FOS_FP32;
    const CUtensorMapDataType ty = f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                       : (dt == FOS_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                         : CU_TENSOR_MAP_DATA_TYPE_FLOAT16);
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * (f32 ? 4 : 2)};
    const cuuint32_t box[2] = {(cuuint32_t)ColTile<In::BF16>::kC,
                               (cuuint32_t)(f32 ? ColTile<In::F32>::kR : ColTile<In::BF16>::kR)};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(map, ty, 2, const_cast<void*>(x), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? FOS_OK : FOS_ERR_CUDA;
}

// One quantize on the current device (arguments already validated).
fos_status quantize_one(const void* x, fos_dtype dt, int64_t rows, int64_t cols,
                        const fos_config* cfg, float* amax, uint8_t* codes, uint8_t* scales,
                        cudaStream_t s) {
    const Src src = cfg->granularity == FOS_SCALE_ROW ? Src::ROW : Src::TENSOR;
    if (rows == 0 || cols == 0) {  // nothing to encode; a computed amax is 0
        const size_t n = (src == Src::ROW) ? (size_t)rows : 1;
        return cuda_status(cudaMemsetAsync(amax, 0, sizeof(float) * n, s));
    }
    if (tiled(cfg)) {
        const fos_status st = cuda_status(clear_tiled_padding(scales, rows, cols, s));
        if (st) return st;
    }
    if (src == Src::ROW && cfg->block == FOS_BLOCK_1X16) {
        const int k = rowpass_k(cols / 16);
        if (k) return cuda_status(run_rowpass(x, dt, rows, cols, cfg, amax, codes, scales, k, s));
    }
    if (!cfg->amax_is_input) {
        fos_status st = cuda_status(run_amax(x, dt, rows, cols, src, amax, nullptr, 0, s));
        if (st) return st;
    }
    return cuda_status(run_quant(x, dt, rows, cols, cfg, amax, src, nullptr, 0, codes, scales, s));
}

}  // namespace

extern "C" {

const char* fos_status_string(fos_status s) {
    switch (s) {
        case FOS_OK: return "ok";
        case FOS_ERR_INVALID_ARG: return "invalid argument";
        case FOS_ERR_UNSUPPORTED: return "unsupported shape, knob or dtype";
        case FOS_ERR_MISALIGNED: return "misaligned pointer";
        case FOS_ERR_CUDA: return "CUDA runtime error";
        case FOS_ERR_NONUNIFORM_TILE_AMAX: return "per-row amax not uniform inside a 16-row tile";
    }
    return "unknown status";
}

int fos_version(void) { return kVersion; }

fos_status fos_amax(const void* x, fos_dtype dt, int64_t rows, int64_t cols, int granularity,
                    float* amax, fos_stream_t stream) {
    if (!valid_dtype(dt)) return FOS_ERR_INVALID_ARG;
    if (granularity != FOS_SCALE_TENSOR && granularity != FOS_SCALE_ROW) return FOS_ERR_INVALID_ARG;
    fos_status st = check_shape(rows, cols, false);
    if (st) return st;
    if (!x || !amax) return FOS_ERR_INVALID_ARG;
    if (!aligned(x, 32)) return FOS_ERR_MISALIGNED;
    const int dev = common_device({x, amax});
    if (dev < 0) return FOS_ERR_INVALID_ARG;
    DeviceScope scope(dev);
    if (scope.st) return scope.st;
    const Src sc = granularity == FOS_SCALE_ROW ? Src::ROW : Src::TENSOR;
    return cuda_status(run_amax(x, dt, rows, cols, sc, amax, nullptr, 0,
                                reinterpret_cast<cudaStream_t>(stream)));
}

fos_status fos_quantize(const void* x, fos_dtype dt, int64_t rows, int64_t cols,
                        const fos_config* cfg, float* amax, uint8_t* codes, uint8_t* scales,
                        fos_stream_t stream) {
    if (!valid_dtype(dt)) return FOS_ERR_INVALID_ARG;
    fos_status st = check_config(cfg);
    if (st) return st;
    st = check_quant_args(x, rows, cols, cfg, amax, codes, scales);
    if (st) return st;
    const bool empty = rows == 0 || cols == 0;
    if (empty && (cfg->amax_is_input || (cfg->granularity == FOS_SCALE_ROW && rows == 0)))
        return FOS_OK;  // nothing to read or write
    const int dev = empty ? device_of(amax) : common_device({x, amax, codes, scales});
    if (dev < 0) return FOS_ERR_INVALID_ARG;
    DeviceScope scope(dev);
    if (scope.st) return scope.st;
    return quantize_one(x, dt, rows, cols, cfg, amax, codes, scales,
                        reinterpret_cast<cudaStream_t>(stream));
}

fos_status fos_quantize_overlap(const void* x, fos_dtype dt, int64_t rows, int64_t cols,
                                const fos_config* cfg, const float* amax, uint8_t* codes,
                                uint8_t* scales, const void* x_next, int64_t rows_next,
                                int64_t cols_next, float* amax_next, fos_stream_t stream) {
    if (!valid_dtype(dt)) return FOS_ERR_INVALID_ARG;
    fos_status st = check_config(cfg);
    if (st) return st;
    if (cfg->block != FOS_BLOCK_1X16 || cfg->granularity != FOS_SCALE_TENSOR ||
        !cfg->amax_is_input)
        return FOS_ERR_UNSUPPORTED;
    st = check_quant_args(x, rows, cols, cfg, amax, codes, scales);
    if (st) return st;
    if (amax_next) {
        st = check_shape(rows_next, cols_next, false);
        if (st) return st;
        if (rows_next > 0 && cols_next > 0) {
            if (!x_next) return FOS_ERR_INVALID_ARG;
            if (!aligned(x_next, 32)) return FOS_ERR_MISALIGNED;
        }
    }
    const bool empty = rows == 0 || cols == 0;
    const bool next_live = amax_next && rows_next > 0 && cols_next > 0;
    int dev = -1;
    if (!empty) dev = common_device({x, amax, codes, scales});
    if (amax_next) {
        const int d = next_live ? common_device({x_next, amax_next}) : device_of(amax_next);
        if (d < 0 || (dev >= 0 && d != dev)) return FOS_ERR_INVALID_ARG;
        dev = d;
    }
    if (dev < 0) return empty ? FOS_OK : FOS_ERR_INVALID_ARG;
    DeviceScope scope(dev);
    if (scope.st) return scope.st;
    return overlap_one(x, dt, rows, cols, cfg, amax, codes, scales, x_next, rows_next, cols_next,
                       amax_next, reinterpret_cast<cudaStream_t>(stream));
}

fos_status fos_quantize_list(int n, const void* const* x, fos_dtype dt, const int64_t* rows,
                             const int64_t* cols, const fos_config* cfg, float* const* amax,
                             uint8_t* const* codes, uint8_t* const* scales,
                             fos_stream_t stream) {
    if (n < 0) return FOS_ERR_INVALID_ARG;
    if (!valid_dtype(dt)) return FOS_ERR_INVALID_ARG;
    fos_status st = check_config(cfg);
    if (st) return st;
    if (n == 0) return FOS_OK;
    if (!x || !rows || !cols || !amax || !codes || !scales) return FOS_ERR_INVALID_ARG;
    for (int i = 0; i < n; ++i) {  // host-side checks of every entry first
        st = check_quant_args(x[i], rows[i], cols[i], cfg, amax[i], codes[i], scales[i]);
        if (st) return st;
    }
    int dev = -1;
    for (int i = 0; i < n; ++i) {
        const bool empty = rows[i] == 0 || cols[i] == 0;
        if (empty && !amax[i]) continue;
        const int d = empty ? device_of(amax[i])
                            : common_device({x[i], amax[i], codes[i], scales[i]});
        if (d < 0 || (dev >= 0 && d != dev)) return FOS_ERR_INVALID_ARG;
        dev = d;
    }
    if (dev < 0) return FOS_OK;  // only empty tensors with nothing to write
    DeviceScope scope(dev);
    if (scope.st) return scope.st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const bool pipelined = cfg->block == FOS_BLOCK_1X16 && cfg->granularity == FOS_SCALE_TENSOR &&
                           !cfg->amax_is_input;
    if (!pipelined) {
        for (int i = 0; i < n; ++i) {
            const bool empty = rows[i] == 0 || cols[i] == 0;
            if (empty && (cfg->amax_is_input || (cfg->granularity == FOS_SCALE_ROW && rows[i] == 0)))
                continue;
            st = quantize_one(x[i], dt, rows[i], cols[i], cfg, amax[i], codes[i], scales[i], s);
            if (st) return st;
        }
        return FOS_OK;
    }
    // Pipelined per-tensor path: amax(0); then for each i one launch that
    // encodes tensor i and runs the amax pass of tensor i+1.  Every launch
    // clears the amax buffer of the stage after the next one, so only the
    // first buffer needs a memset and the launches chain back to back.
    st = cuda_status(cudaMemsetAsync(amax[0], 0, sizeof(float), s));
    if (st) return st;
    st = cuda_status(run_amax_cleared(x[0], dt, rows[0], cols[0], amax[0], s,
                                      n > 1 ? amax[1] : nullptr));
    if (st) return st;
    for (int i = 0; i < n; ++i) {
        const bool more = i + 1 < n;
        st = overlap_one(x[i], dt, rows[i], cols[i], cfg, amax[i], codes[i], scales[i],
                         more ? x[i + 1] : nullptr, more ? rows[i + 1] : 0,
                         more ? cols[i + 1] : 0, more ? amax[i + 1] : nullptr, s,
                         /*next_cleared=*/true, i + 2 < n ? amax[i + 2] : nullptr);
        if (st) return st;
    }
    return FOS_OK;
}

fos_status fos_quantize_grouped(const void* x, fos_dtype dt, int64_t rows, int64_t cols,
                                const int32_t* offs, int G, const fos_config* cfg,
                                float* group_amax, uint8_t* codes, uint8_t* scales,
                                fos_stream_t stream) {
    if (!valid_dtype(dt)) return FOS_ERR_INVALID_ARG;
    fos_status st = check_config(cfg);
    if (st) return st;
    st = check_shape(rows, cols, cfg->block == FOS_BLOCK_16X16);
    if (st) return st;
    st = check_order(cfg);
    if (st) return st;
    if (tiled(cfg)) return FOS_ERR_UNSUPPORTED;  // grouped scales are plain
    if (G < 1) return FOS_ERR_INVALID_ARG;
    if (G > FOS_GROUPED_MAX_GROUPS) return FOS_ERR_UNSUPPORTED;
    if (!x || !offs || !group_amax || !codes || !scales) return FOS_ERR_INVALID_ARG;
    if (!aligned(x, 32) || !aligned(codes, 8) || !aligned(offs, 4)) return FOS_ERR_MISALIGNED;
    const int dev = common_device({x, offs, group_amax, codes, scales});
    if (dev < 0) return FOS_ERR_INVALID_ARG;
    DeviceScope scope(dev);
    if (scope.st) return scope.st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (!cfg->amax_is_input) {
        st = cuda_status(run_amax(x, dt, rows, cols, Src::GROUP, group_amax, offs, G, s));
        if (st) return st;
    }
    return cuda_status(
        run_quant(x, dt, rows, cols, cfg, group_amax, Src::GROUP, offs, G, codes, scales, s));
}

fos_status fos_dequantize(const uint8_t* codes, const uint8_t* scales, const float* amax,
                          int64_t rows, int64_t cols, const fos_config* cfg, void* out,
                          fos_dtype out_dt, fos_stream_t stream) {
    if (!valid_dtype(out_dt)) return FOS_ERR_INVALID_ARG;
    fos_status st = check_config(cfg);
    if (st) return st;
    const bool b16 = cfg->block == FOS_BLOCK_16X16;
    st = check_shape(rows, cols, b16);
    if (st) return st;
    if (tiled(cfg)) return FOS_ERR_UNSUPPORTED;  // decodes plain scales
    if (!codes || !scales || !amax || !out) return FOS_ERR_INVALID_ARG;
    if (!aligned(out, 32) || !aligned(codes, 8)) return FOS_ERR_MISALIGNED;
    const int dev = common_device({codes, scales, amax, out});
    if (dev < 0) return FOS_ERR_INVALID_ARG;
    DeviceScope scope(dev);
    if (scope.st) return scope.st;
    if (rows == 0 || cols == 0) return FOS_OK;
    DeqArgs a{};
    a.codes = codes;
    a.scales = scales;
    a.amax = amax;
    a.out = out;
    a.rows = rows;
    a.nb = cols / 16;
    a.cpr = (a.nb + 31) / 32;
    a.units = rows * a.cpr;
    a.six_bound = 6.0f * (float)cfg->e4m3_bound;
    const Out ot = out_dt == FOS_BF16 ? Out::BF16 : (out_dt == FOS_FP16 ? Out::F16 : Out::F32);
    const Src src = cfg->granularity == FOS_SCALE_ROW ? Src::ROW : Src::TENSOR;
    return cuda_status(launch_dequant(ot, b16, src, a, reinterpret_cast<cudaStream_t>(stream)));
}

fos_status fos_qdq(int n, const void* const* x, void* const* out, const int64_t* rows,
                   const int64_t* cols, float* const* amax, fos_dtype dt,
                   const fos_config* cfg, fos_stream_t stream) {
    if (n < 0) return FOS_ERR_INVALID_ARG;
    if (dt != FOS_BF16 && dt != FOS_FP16) return valid_dtype(dt) ? FOS_ERR_UNSUPPORTED
                                                                  : FOS_ERR_INVALID_ARG;
    fos_status st = check_config(cfg);
    if (st) return st;
    if (cfg->block != FOS_BLOCK_1X16 || cfg->granularity != FOS_SCALE_TENSOR)
        return FOS_ERR_UNSUPPORTED;
    if (n == 0) return FOS_OK;
    if (!x || !out || !rows || !cols || !amax) return FOS_ERR_INVALID_ARG;
    for (int i = 0; i < n; ++i) {
        st = check_shape(rows[i], cols[i], false);
        if (st) return st;
        const bool empty = rows[i] == 0 || cols[i] == 0;  // data pointers may be null
        if (!amax[i] || (!empty && (!x[i] || !out[i]))) return FOS_ERR_INVALID_ARG;
        if (!empty && (!aligned(x[i], 32) || !aligned(out[i], 32))) return FOS_ERR_MISALIGNED;
    }
    int dev = -1;
    for (int i = 0; i < n; ++i) {
        const bool empty = rows[i] == 0 || cols[i] == 0;
        const int d = empty ? common_device({amax[i]}) : common_device({x[i], out[i], amax[i]});
        if (d < 0 || (dev >= 0 && d != dev)) return FOS_ERR_INVALID_ARG;
        dev = d;
    }
    DeviceScope scope(dev);
    if (scope.st) return scope.st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (!cfg->amax_is_input) {
        for (int i = 0; i < n; ++i) {
            st = cuda_status(run_amax(x[i], dt, rows[i], cols[i], Src::TENSOR, amax[i], nullptr,
                                      0, s));
            if (st) return st;
        }
    }
    const Err em = err_of(cfg);
    const In it = in_of(dt);
    for (int base = 0; base < n; base += kQdqMaxList) {
        const int m = (n - base < kQdqMaxList) ? n - base : kQdqMaxList;
        QdqArgs a;
        std::memset(&a, 0, sizeof(a));
        a.n = m;
        a.six_bound = 6.0f * (float)cfg->e4m3_bound;
        a.neg_zero = -0.0f;
        int64_t u = 0;
        for (int i = 0; i < m; ++i) {
            QdqTensor& t = a.t[i];
            t.x = x[base + i];
            t.out = out[base + i];
            t.amax = amax[base + i];
            t.nblk = rows[base + i] * (cols[base + i] / 16);
            t.unit_begin = u;
            u += (t.nblk + 31) / 32;
        }
        a.t[m].unit_begin = u;
        a.units = u;
        if (u == 0) continue;
        st = cuda_status(launch_qdq(it, em, a, s));
        if (st) return st;
    }
    return FOS_OK;
}

fos_status fos_diag_convert(int op, const void* in, void* out, int64_t n, fos_stream_t stream) {
    if (op < FOS_DIAG_E2M1_ENCODE || op > FOS_DIAG_SCALE_CODES) return FOS_ERR_INVALID_ARG;
    if (n < 0) return FOS_ERR_INVALID_ARG;
    if (n == 0) return FOS_OK;
    if (!in || !out) return FOS_ERR_INVALID_ARG;
    const int dev = common_device({in, out});
    if (dev < 0) return FOS_ERR_INVALID_ARG;
    DeviceScope scope(dev);
    if (scope.st) return scope.st;
    return cuda_status(launch_diag(op, in, out, n, reinterpret_cast<cudaStream_t>(stream)));
}

fos_status fos_diag_wait_timeout(int which, uint32_t* word, fos_stream_t stream) {
    if (which != 0 && which != 1) return FOS_ERR_INVALID_ARG;
    if (!word) return FOS_ERR_INVALID_ARG;
    if (!aligned(word, 4)) return FOS_ERR_MISALIGNED;
    const int dev = device_of(word);
    if (dev < 0) return FOS_ERR_INVALID_ARG;
    DeviceScope scope(dev);
    if (scope.st) return scope.st;
    return cuda_status(launch_wait_timeout(which, word, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"

// ------------------------------------------------------------ fused amax + QDQ
namespace fos {

// Host-only checks of a fused amax + QDQ list call, in the order both fused
// entry points report them: list length sign, dtype, configuration, the
// supported knobs, list length limit, then pointers, shapes and alignment of
// every tensor.  Makes no CUDA call.
fos_status qdq_fused_host_checks(int n, int max_n, const void* const* x, void* const* out,
                                 const int64_t* rows, const int64_t* cols, float* const* amax,
                                 fos_dtype dt, const fos_config* cfg) {
    if (n < 0) return FOS_ERR_INVALID_ARG;
    if (dt != FOS_BF16 && dt != FOS_FP16) return valid_dtype(dt) ? FOS_ERR_UNSUPPORTED
                                                                  : FOS_ERR_INVALID_ARG;
    fos_status st = check_config(cfg);
    if (st) return st;
    if (cfg->block != FOS_BLOCK_1X16 || cfg->granularity != FOS_SCALE_TENSOR ||
        cfg->amax_is_input)
        return FOS_ERR_UNSUPPORTED;
    if (n > max_n) return FOS_ERR_UNSUPPORTED;
    if (n == 0) return FOS_OK;
    if (!x || !out || !rows || !cols || !amax) return FOS_ERR_INVALID_ARG;
    for (int i = 0; i < n; ++i) {
        st = check_shape(rows[i], cols[i], false);
        if (st) return st;
        const bool empty = rows[i] == 0 || cols[i] == 0;
        if (!amax[i] || (!empty && (!x[i] || !out[i]))) return FOS_ERR_INVALID_ARG;
        if (!empty && (!aligned(x[i], 32) || !aligned(out[i], 32))) return FOS_ERR_MISALIGNED;
    }
    return FOS_OK;
}

}  // namespace fos

extern "C" {

size_t fos_qdq_fused_workspace_bytes(int n) {
    if (n <= 0) return 0;
    const size_t words = 1 + 2 * (size_t)n;  // error word, n counters, n running amaxes
    return (words * sizeof(uint32_t) + 255) / 256 * 256;
}

fos_status fos_qdq_fused(int n, const void* const* x, void* const* out, const int64_t* rows,
                         const int64_t* cols, float* const* amax, fos_dtype dt,
                         const fos_config* cfg, void* workspace, size_t workspace_bytes,
                         fos_stream_t stream) {
    fos_status st = qdq_fused_host_checks(n, kQdqMaxList, x, out, rows, cols, amax, dt, cfg);
    if (st || n == 0) return st;
    if (!workspace) return FOS_ERR_INVALID_ARG;
    const size_t need = fos_qdq_fused_workspace_bytes(n);
    if (workspace_bytes < need) return FOS_ERR_INVALID_ARG;
    if (!aligned(workspace, 256)) return FOS_ERR_MISALIGNED;
    int dev = device_of(workspace);
    if (dev < 0) return FOS_ERR_INVALID_ARG;
    for (int i = 0; i < n; ++i) {
        const bool empty = rows[i] == 0 || cols[i] == 0;
        const int d = empty ? common_device({amax[i]}) : common_device({x[i], out[i], amax[i]});
        if (d != dev) return FOS_ERR_INVALID_ARG;
    }
    DeviceScope scope(dev);
    if (scope.st) return scope.st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    QdqFusedArgs a;
    std::memset(&a, 0, sizeof(a));
    a.q.n = n;
    a.q.six_bound = 6.0f * (float)cfg->e4m3_bound;
    a.q.neg_zero = -0.0f;
    int64_t u = 0;
    for (int i = 0; i < n; ++i) {
        QdqTensor& t = a.q.t[i];
        t.x = x[i];
        t.out = out[i];
        t.nblk = rows[i] * (cols[i] / 16);
        t.unit_begin = u;
        u += (t.nblk + 31) / 32;
        a.amax_out[i] = amax[i];
    }
    a.q.t[n].unit_begin = u;
    a.q.units = u;
    uint32_t* w = static_cast<uint32_t*>(workspace);
    a.ws.err = w;
    a.ws.cnt = w + 1;
    a.ws.acc = w + 1 + n;
    st = cuda_status(cudaMemsetAsync(workspace, 0, need, s));
    if (st) return st;
    return cuda_status(launch_qdq_fused(in_of(dt), err_of(cfg), a, s));
}

fos_status fos_workspace_error(const void* workspace, fos_stream_t stream, int* code) {
    if (!workspace || !code) return FOS_ERR_INVALID_ARG;
    const int dev = device_of(workspace);
    if (dev < 0) return FOS_ERR_INVALID_ARG;
    DeviceScope scope(dev);
    if (scope.st) return scope.st;
    fos_status st = cuda_status(cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)));
    if (st) return st;
    uint32_t v = 0;
    st = cuda_status(cudaMemcpy(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost));
    if (st) return st;
    *code = (int)v;
    return FOS_OK;
}

}  // extern "C"

// ------------------------------------------------------------ column-wise quantize
extern "C" {

fos_status fos_quantize_colwise(const void* x, fos_dtype dt, int64_t rows, int64_t cols,
                                const fos_config* cfg, float* amax, uint8_t* codes_t,
                                uint8_t* scales_t, uint8_t* codes, uint8_t* scales,
                                fos_stream_t stream) {
    if (!valid_dtype(dt)) return FOS_ERR_INVALID_ARG;
    fos_status st = check_config(cfg);
    if (st) return st;
    if (cfg->block != FOS_BLOCK_1X16 || cfg->granularity != FOS_SCALE_TENSOR)
        return FOS_ERR_UNSUPPORTED;
    st = check_shape(rows, cols, false);
    if (st) return st;
    st = check_shape(cols, rows, false);  // x^T: blocks run down the rows
    if (st) return st;
    st = check_layout(cfg, rows > cols ? rows : cols);  // x^T has cols rows
    if (st) return st;
    if ((codes == nullptr) != (scales == nullptr)) return FOS_ERR_INVALID_ARG;
    const bool dual = codes != nullptr;
    if (!amax) return FOS_ERR_INVALID_ARG;
    if (rows == 0 || cols == 0) {
        if (cfg->amax_is_input) return FOS_OK;
        const int d = device_of(amax);
        if (d < 0) return FOS_ERR_INVALID_ARG;
        DeviceScope scope(d);
        if (scope.st) return scope.st;
        return cuda_status(cudaMemsetAsync(amax, 0, sizeof(float),
                                           reinterpret_cast<cudaStream_t>(stream)));
    }
    if (!x || !codes_t || !scales_t) return FOS_ERR_INVALID_ARG;
    if (!aligned(x, 32) || !aligned(codes_t, 8) || (dual && !aligned(codes, 8)))
        return FOS_ERR_MISALIGNED;
    if (rows >= (INT64_C(1) << 31) || cols >= (INT64_C(1) << 31))  // tile coordinates are int32
        return FOS_ERR_UNSUPPORTED;
    const int dev = dual ? common_device({x, amax, codes_t, scales_t, codes, scales})
                         : common_device({x, amax, codes_t, scales_t});
    if (dev < 0) return FOS_ERR_INVALID_ARG;
    DeviceScope scope(dev);
    if (scope.st) return scope.st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (!cfg->amax_is_input) {
        st = cuda_status(run_amax(x, dt, rows, cols, Src::TENSOR, amax, nullptr, 0, s));
        if (st) return st;
    }
    ColArgs a{};
    st = encode_tile_map(&a.tmap, x, dt, rows, cols);
    if (st) return st;
    a.codes_t = codes_t;
    a.scales_t = scales_t;
    a.codes = codes;
    a.scales = scales;
    a.amax = amax;
    a.rows = rows;
    a.cols = cols;
    const int tile_r = (dt == FOS_FP32) ? ColTile<In::F32>::kR : ColTile<In::BF16>::kR;
    const int tile_c = ColTile<In::BF16>::kC;
    a.tiles_c = (cols + tile_c - 1) / tile_c;
    a.tiles = ((rows + tile_r - 1) / tile_r) * a.tiles_c;
    a.six_bound = 6.0f * (float)cfg->e4m3_bound;
    a.neg_zero = -0.0f;
    if (tiled(cfg)) {
        // x^T is [cols, rows]: its scale matrix has cols rows of rows / 16 blocks
        a.pc4_t = tiled_pc4(rows);
        a.pc4 = tiled_pc4(cols);
        st = cuda_status(clear_tiled_padding(scales_t, cols, rows, s));
        if (st) return st;
        if (dual) {
            st = cuda_status(clear_tiled_padding(scales, rows, cols, s));
            if (st) return st;
        }
        return cuda_status(launch_colwise_tl(in_of(dt), err_of(cfg), dual, a, s));
    }
    return cuda_status(launch_colwise(in_of(dt), err_of(cfg), dual, a, s));
}

}  // extern "C"

// ------------------------------------------------------------ swizzled scales
extern "C" {

int64_t fos_swizzled_scales_bytes(int64_t rows, int64_t cols) {
    if (rows < 0 || cols < 0 || cols % 16 != 0) return -1;
    return (rows + 127) / 128 * 128 * ((cols / 16 + 3) / 4 * 4);
}

fos_status fos_swizzle_scales(const uint8_t* scales, int64_t rows, int64_t cols, uint8_t* out,
                              fos_stream_t stream) {
    fos_status st = check_shape(rows, cols, false);
    if (st) return st;
    if (rows == 0 || cols == 0) return FOS_OK;
    if (!scales || !out) return FOS_ERR_INVALID_ARG;
    if (!aligned(out, 4)) return FOS_ERR_MISALIGNED;
    const int dev = common_device({scales, out});
    if (dev < 0) return FOS_ERR_INVALID_ARG;
    DeviceScope scope(dev);
    if (scope.st) return scope.st;
    return cuda_status(launch_swizzle(scales, rows, cols / 16, out,
                                      reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"

// ------------------------------------------------------------ product of quantized operands
extern "C" {

fos_status fos_mm(const uint8_t* a_codes, const uint8_t* a_scales_tiled, const float* a_amax,
                  const uint8_t* b_codes, const uint8_t* b_scales_tiled, const float* b_amax,
                  int64_t M, int64_t N, int64_t K, const fos_config* cfg, float* out,
                  fos_stream_t stream) {
    fos_status st = check_config(cfg);
    if (st) return st;
    if (cfg->block != FOS_BLOCK_1X16) return FOS_ERR_UNSUPPORTED;
    if (M < 0 || N < 0 || K < 0) return FOS_ERR_INVALID_ARG;
    if (M % 16 || N % 16 || K % 64) return FOS_ERR_UNSUPPORTED;
    if (M >= (INT64_C(1) << 31) || N >= (INT64_C(1) << 31) || K >= (INT64_C(1) << 31))
        return FOS_ERR_UNSUPPORTED;
    if (M == 0 || N == 0) return FOS_OK;
    if (!a_codes || !a_scales_tiled || !a_amax || !b_codes || !b_scales_tiled || !b_amax || !out)
        return FOS_ERR_INVALID_ARG;
    if (!aligned(a_codes, 16) || !aligned(b_codes, 16) || !aligned(a_scales_tiled, 16) ||
        !aligned(b_scales_tiled, 16) || !aligned(out, 16))
        return FOS_ERR_MISALIGNED;
    const int dev = common_device({a_codes, a_scales_tiled, a_amax, b_codes, b_scales_tiled,
                                   b_amax, out});
    if (dev < 0) return FOS_ERR_INVALID_ARG;
    DeviceScope scope(dev);
    if (scope.st) return scope.st;
    if (K == 0) {  // empty sum
        return cuda_status(cudaMemsetAsync(out, 0, sizeof(float) * (size_t)(M * N),
                                           reinterpret_cast<cudaStream_t>(stream)));
    }
    const int rc = run_mm(a_codes, a_scales_tiled, a_amax, cfg->granularity == FOS_SCALE_ROW,
                          b_codes, b_scales_tiled, b_amax, M, N, K,
                          6.0f * (float)cfg->e4m3_bound, out,
                          reinterpret_cast<cudaStream_t>(stream));
    return rc == 0 ? FOS_OK : FOS_ERR_CUDA;
}

}  // extern "C"

// ------------------------------------------------------------ tile-uniform amax check
extern "C" {

fos_status fos_check_tile_amax(const float* amax, int64_t rows, int64_t* bad,
                               fos_stream_t stream) {
    if (rows < 0 || !bad) return FOS_ERR_INVALID_ARG;
    if (rows % 16 != 0) return FOS_ERR_UNSUPPORTED;
    if (rows > 0 && !amax) return FOS_ERR_INVALID_ARG;
    if (!aligned(bad, 8) || (amax && !aligned(amax, 4))) return FOS_ERR_MISALIGNED;
    const int dev = rows > 0 ? common_device({amax, bad}) : device_of(bad);
    if (dev < 0) return FOS_ERR_INVALID_ARG;
    DeviceScope scope(dev);
    if (scope.st) return scope.st;
    return cuda_status(launch_check_tile_amax(amax, rows, bad,
                                              reinterpret_cast<cudaStream_t>(stream)));
}

fos_status fos_tile_amax_status(const int64_t* bad, fos_stream_t stream) {
    if (!bad) return FOS_ERR_INVALID_ARG;
    const int dev = device_of(bad);
    if (dev < 0) return FOS_ERR_INVALID_ARG;
    DeviceScope scope(dev);
    if (scope.st) return scope.st;
    fos_status st = cuda_status(cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)));
    if (st) return st;
    int64_t v = 0;
    st = cuda_status(cudaMemcpy(&v, bad, sizeof(v), cudaMemcpyDeviceToHost));
    if (st) return st;
    return v == 0 ? FOS_OK : FOS_ERR_NONUNIFORM_TILE_AMAX;
}

}  // extern "C"

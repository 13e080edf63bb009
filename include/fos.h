/*
 * fos.h -- C ABI of the GB300 (sm_103a) NVFP4 four-over-six block quantizer.
 *
 * The method (torchao PR "Add the four-over-six grouped GEMM and dispatcher
 * wiring", description and first commit): every quantization block -- 1x16
 * elements along a row, or a 16x16 tile for weights -- is encoded twice under
 * an FP32 global scale, once as standard NVFP4 (block amax mapped to E2M1
 * value 6 by an E4M3 block scale) and once as a 1.5x-scale candidate (block
 * amax mapped to 4).  Both are rounded to E2M1 with correctly-rounded FP32
 * division, decoded exactly, and compared by MAE or MSE; the lower-error
 * candidate's packed E2M1 codes and E4M3 scale are stored (torchao PR "Add a
 * CuTe DSL fast-path kernel for four-over-six quantize": pinned rounding,
 * pinned width-16 error reduction, NaN-dropping block amax, NaN -> +6).
 *
 * Conventions shared by every entry point
 *   - Data pointers (x, out, codes, scales, amax, offs, workspaces) are
 *     DEVICE pointers owned by the caller; the library never allocates, frees
 *     or keeps them (fos_qdq_fused_static uses one fixed array of its
 *     own).  Host-side arrays (the pointer / size lists of the list calls)
 *     are read during the call only.
 *   - Tensors are row-major and contiguous: x is [rows, cols]; codes are
 *     [rows, cols/2] bytes, element 2j in the low nibble of byte j; scales are
 *     E4M3 bytes [rows, cols/16] (1x16) or [rows/16, cols/16] (16x16), plain
 *     row-major (fos_swizzle_scales gives the tiled GEMM layout).
 *   - cols % 16 == 0; with 16x16 blocks also rows % 16 == 0.
 *   - x / out must be 32-byte aligned, codes 8-byte aligned (any row slice of
 *     a tensor from the CUDA caching allocator satisfies this).
 *   - Work is enqueued on `stream` of the device that owns the data and the
 *     call returns without synchronising the host (fos_workspace_error and
 *     fos_tile_amax_status, which read a result back, are the exceptions).  The caller's current device is
 *     restored before return.
 *   - Every argument is validated on the host before anything is launched;
 *     a failed check returns an error status and launches nothing.  CUDA
 *     launch failures return FOS_ERR_CUDA.  Kernels never trap.  The only
 *     waits on other work are the bounded ones of fos_qdq_fused (between the
 *     CTAs of its cooperative launch) and of the column-wise kernel (on its
 *     own TMA loads); each gives up after about a second and reports it, so
 *     no call can hang the device.
 *   - Global scale (reading of "FP32 global scale"): S = (6 * bound) / A,
 *     correctly rounded, for a global amax A; S = 1 when A is zero, negative,
 *     NaN or Inf; S = FLT_MAX when the quotient overflows.
 */
#ifndef FOS_H
#define FOS_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define FOS_API __attribute__((visibility("default")))
#else
#define FOS_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Identical to cudaStream_t; 0 is the legacy default stream. */
typedef struct CUstream_st* fos_stream_t;

typedef enum {
    FOS_OK = 0,
    FOS_ERR_INVALID_ARG = 1, /* null pointer, negative size, bad enum value   */
    FOS_ERR_UNSUPPORTED = 2, /* shape / knob / dtype combination not offered  */
    FOS_ERR_MISALIGNED = 3,  /* pointer alignment rule above violated         */
    FOS_ERR_CUDA = 4,        /* a CUDA runtime call or launch failed          */
    FOS_ERR_NONUNIFORM_TILE_AMAX = 5 /* fos_tile_amax_status: a 16-row tile's
                                        per-row amax entries differ         */
} fos_status;

typedef enum { FOS_BF16 = 0, FOS_FP16 = 1, FOS_FP32 = 2 } fos_dtype;

enum { FOS_BLOCK_1X16 = 0, FOS_BLOCK_16X16 = 1 };
enum { FOS_MODE_STANDARD = 0, FOS_MODE_4OVER6 = 1 };
enum { FOS_MAE = 0, FOS_MSE = 1 };
enum { FOS_ERR_EXACT_F32 = 0, FOS_ERR_F16 = 1 };
enum { FOS_SCALE_TENSOR = 0, FOS_SCALE_ROW = 1 };
enum { FOS_ORDER_TREE = 0, FOS_ORDER_SEQ = 1 };
enum { FOS_SCALES_PLAIN = 0, FOS_SCALES_TILED = 1 };

/* The knobs the pages name (Megatron PR "Fuse NVFP4 fake-QAT quantize-
 * dequantize with CuTe DSL", numerical contract: standard NVFP4 plus 4over6
 * MAE/MSE, E4M3 256/448, exact-error / FP16-error; torchao PRs: 1x16 / 16x16
 * blocks, per-tensor or row-scaled global scale). */
typedef struct {
    int block;         /* FOS_BLOCK_1X16 | FOS_BLOCK_16X16                       */
    int mode;          /* FOS_MODE_STANDARD (map-to-6 only) | FOS_MODE_4OVER6    */
    int err_metric;    /* FOS_MAE | FOS_MSE                     (4over6 only)    */
    int err_precision; /* FOS_ERR_EXACT_F32 | FOS_ERR_F16       (4over6 only)    */
    int e4m3_bound;    /* 448 | 256: E4M3 value the global scale maps the amax to */
    int granularity;   /* FOS_SCALE_TENSOR | FOS_SCALE_ROW                       */
    int amax_is_input; /* 1: caller supplies amax; 0: library computes, writes it */
    int err_order;     /* how a block's 16 error terms are summed (4over6 only):
                        * FOS_ORDER_TREE (0): the pinned width-16 tree of the
                        *   torchao fast-path PR, for w = 8,4,2,1: t[i] += t[i+w];
                        * FOS_ORDER_SEQ (1): in element order, t0 + t1 + ... + t15
                        *   (the Transformer Engine term order the Megatron PR
                        *   keeps, "Packed pair arithmetic"); 1x16 blocks only,
                        *   FOS_ERR_UNSUPPORTED with 16x16 in 4over6 mode.     */
    int scale_layout;  /* where the quantize calls write the E4M3 block scales:
                        * FOS_SCALES_PLAIN (0): row-major [rows, cols/16]
                        *   ([rows/16, cols/16] for 16x16);
                        * FOS_SCALES_TILED (1): straight into the tiled layout
                        *   of block-scaled FP4 GEMMs that fos_swizzle_scales
                        *   produces (fos_swizzled_scales_bytes(rows, cols)
                        *   bytes, zero padding included), ready for fos_mm;
                        *   1x16 blocks and fewer than 2^30 rows (of x, and
                        *   of x^T for fos_quantize_colwise) only, else
                        *   FOS_ERR_UNSUPPORTED (fos_quantize, fos_quantize_list,
                        *   fos_quantize_overlap, fos_quantize_colwise); the
                        *   grouped quantize and fos_dequantize take plain
                        *   scales only and return FOS_ERR_UNSUPPORTED.     */
} fos_config;

/*
 * fos_amax -- global amax pass (Megatron PR, fused data path: FP32
 * per-tensor amax computed before the fused kernel).  NaN-dropping max|x|
 * with initial +0: a NaN never becomes the amax and an all-NaN or empty
 * scope gives 0.
 *   granularity FOS_SCALE_TENSOR: amax[0] = over all of x.
 *   granularity FOS_SCALE_ROW:    amax[r] = over row r, r < rows.
 * Errors: FOS_ERR_INVALID_ARG (null pointers with nonzero size, negative
 * sizes, bad enum), FOS_ERR_UNSUPPORTED (cols % 16 != 0), FOS_ERR_MISALIGNED.
 */
FOS_API fos_status fos_amax(const void* x, fos_dtype dt, int64_t rows, int64_t cols, int granularity,
                    float* amax, fos_stream_t stream);

/*
 * fos_quantize -- four-over-six (or standard) NVFP4 quantize of x [rows, cols]
 * of dtype bf16, fp16 or fp32 (torchao fast-path PR: the quantizer op;
 * grouped PR: per-tensor or row-scaled global scale, 1x16 / 16x16 blocks).
 *   amax   [1] (FOS_SCALE_TENSOR) or [rows] (FOS_SCALE_ROW): read when
 *          cfg->amax_is_input, otherwise computed first and written.
 *          With 16x16 blocks and FOS_SCALE_ROW the per-row amax must be
 *          uniform inside each 16-row tile (grouped PR, tile-uniform
 *          contract); each tile uses the amax of its first row.
 *   codes  [rows, cols/2] out; scales out (layout above).
 * Errors as for fos_amax, plus FOS_ERR_UNSUPPORTED for a bad bound, block,
 * mode or (16x16) rows % 16 != 0.
 */
FOS_API fos_status fos_quantize(const void* x, fos_dtype dt, int64_t rows, int64_t cols,
                        const fos_config* cfg, float* amax, uint8_t* codes, uint8_t* scales,
                        fos_stream_t stream);

/*
 * fos_check_tile_amax -- validation of the tile-uniform contract above
 * (grouped PR: with 16x16 blocks a row-scaled global scale must be the same
 * for the 16 rows of a tile, so the per-row amax must be): counts the 16-row
 * tiles of amax [rows] whose 16 entries are not all bitwise equal and writes
 * the count to *bad (device int64, cleared by the call).  rows % 16 == 0;
 * amax 4-byte aligned.  Asynchronous like every call; fos_quantize itself
 * never checks (it uses each tile's first-row amax), so a caller that wants
 * the check runs this first.  Errors: FOS_ERR_INVALID_ARG (null pointer with
 * rows > 0, negative rows), FOS_ERR_UNSUPPORTED (rows % 16 != 0),
 * FOS_ERR_MISALIGNED.
 */
FOS_API fos_status fos_check_tile_amax(const float* amax, int64_t rows, int64_t* bad,
                                       fos_stream_t stream);

/*
 * fos_tile_amax_status -- the validating read of that count: waits for
 * `stream`, reads *bad and returns FOS_OK when it is zero and
 * FOS_ERR_NONUNIFORM_TILE_AMAX otherwise (FOS_ERR_INVALID_ARG for a pointer
 * that is not device memory, FOS_ERR_CUDA when the wait fails).  This call
 * synchronises the host.
 */
FOS_API fos_status fos_tile_amax_status(const int64_t* bad, fos_stream_t stream);

/*
 * fos_quantize_list -- fos_quantize over a list of n tensors of one dtype
 * and one configuration; entry i reads x[i] (rows[i] x cols[i]) and writes
 * amax[i], codes[i], scales[i] exactly as fos_quantize would.  With 1x16
 * blocks, per-tensor scale and the amax computed by the library, the work is
 * pipelined: the launch that encodes tensor i also runs the amax pass of
 * tensor i+1 (every warp loads its next-tensor segment before encoding and
 * folds it into its max afterwards; the encode is bound by instruction
 * issue, the amax pass by HBM reads), so a list costs about one amax pass
 * plus n encodes.  Other configurations run the entries one after another.
 * Host arrays must hold n entries; errors as for fos_quantize (the first
 * failing entry's status, nothing launched).
 */
FOS_API fos_status fos_quantize_list(int n, const void* const* x, fos_dtype dt,
                                     const int64_t* rows, const int64_t* cols,
                                     const fos_config* cfg, float* const* amax,
                                     uint8_t* const* codes, uint8_t* const* scales,
                                     fos_stream_t stream);

/*
 * fos_quantize_overlap -- one stage of the list pipeline, for callers that
 * pipeline their own tensors: quantize x (1x16 blocks, per-tensor scale,
 * cfg->amax_is_input must be 1, amax given) and, in the same launch, compute
 * the per-tensor amax of x_next (same dtype, rows_next x cols_next) into
 * amax_next[0] (cleared first, written by the launch).  With amax_next NULL
 * it is fos_quantize.  Returns FOS_ERR_UNSUPPORTED for other configurations.
 */
FOS_API fos_status fos_quantize_overlap(const void* x, fos_dtype dt, int64_t rows, int64_t cols,
                                        const fos_config* cfg, const float* amax,
                                        uint8_t* codes, uint8_t* scales, const void* x_next,
                                        int64_t rows_next, int64_t cols_next,
                                        float* amax_next, fos_stream_t stream);

/*
 * fos_quantize_colwise -- the column-wise operand: fos_quantize applied to
 * x^T ([cols, rows]), computed from the row-major x [rows, cols] without
 * forming x^T.  Blocks are 16 consecutive rows of one column of x:
 *   codes_t [cols, rows/2], scales_t [cols, rows/16] (row c of x^T = column
 *   c of x, low nibble = the upper of two rows).
 * With codes and scales both non-NULL the row-wise result of x ([rows,
 * cols/2], [rows, cols/16], exactly fos_quantize's) is written by the same
 * launch from the same read of x; both NULL skips it.  1x16 blocks and a
 * per-tensor scale only (the amax of x and of x^T are the same value);
 * rows % 16 == 0 and cols % 16 == 0.  amax as in fos_quantize.  The pages
 * list transpose / column-wise output as a non-goal of their QDQ path (the
 * Megatron PR's deliberate non-goals); this is the layout a weight-gradient
 * GEMM reads, built with the same arithmetic.
 */
FOS_API fos_status fos_quantize_colwise(const void* x, fos_dtype dt, int64_t rows, int64_t cols,
                                        const fos_config* cfg, float* amax, uint8_t* codes_t,
                                        uint8_t* scales_t, uint8_t* codes, uint8_t* scales,
                                        fos_stream_t stream);

/*
 * fos_swizzle_scales -- the 1x16 block scales of a [rows, cols] tensor
 * (scales [rows, cols/16], as fos_quantize writes them) rearranged into the
 * tiled layout that block-scaled FP4 GEMMs read: the scale matrix is padded
 * with zero bytes to a multiple of 128 rows and 4 columns and cut into
 * 128 x 4 tiles of 512 bytes, stored tile-row by tile-row; inside a tile,
 * scale (32 i + j, k) (i < 4, j < 32, k < 4) is byte 16 j + 4 i + k.
 * out holds fos_swizzled_scales_bytes(rows, cols) bytes (4-byte aligned).
 * The pages pass plain scales to their GEMMs; this is the layout a GEMM
 * library's NVFP4 path takes, checked in the tests against such a GEMM.
 * fos_swizzled_scales_bytes returns -1 for negative sizes or cols % 16 != 0.
 * Errors: FOS_ERR_INVALID_ARG (negative sizes, null or non-device pointers
 * with a nonzero size), FOS_ERR_UNSUPPORTED (cols % 16 != 0),
 * FOS_ERR_MISALIGNED (out not 4-byte aligned).
 */
FOS_API int64_t fos_swizzled_scales_bytes(int64_t rows, int64_t cols);
FOS_API fos_status fos_swizzle_scales(const uint8_t* scales, int64_t rows, int64_t cols,
                                      uint8_t* out, fos_stream_t stream);

/*
 * fos_mm -- out = a . b^T from quantized operands, the forward product of
 * the grouped PR's four_over_six_mm: a [M, K] and b [N, K] were quantized
 * with 1x16 blocks (codes [M, K/2] and [N, K/2]) and their block scales put
 * into the tiled GEMM layout (fos_swizzle_scales, or written there directly
 * by the quantize call with scale_layout = FOS_SCALES_TILED); a_amax /
 * b_amax are the amaxes they were quantized with (a: [M] when
 * cfg->granularity is FOS_SCALE_ROW, else [1]; b: [1]).  One persistent
 * launch of this library's kernel on the tensor cores (tcgen05 block-scaled
 * E2M1 MMAs with UE4M3 scales, fp32 accumulation in tensor memory, one CTA
 * per SM walking 128 x 192 output tiles) forms the block-scaled product D
 * of each tile, and its epilogue applies the global decode scales before
 * the single store,
 *   out[m][n] = (D[m][n] * g_a(m)) * g_b,  g = rn(1 / S),
 * S the global scale fos_quantize used (cfg->e4m3_bound).  out: fp32
 * [M, N] row-major, 16-byte aligned, like all operands.  M and N multiples
 * of 16, K a multiple of 64.  The kernel's waits are bounded: a CTA whose
 * wait gave up (which takes about a second) writes NaN into the first
 * element of its first tile.  Nothing is allocated.
 */
FOS_API fos_status fos_mm(const uint8_t* a_codes, const uint8_t* a_scales_tiled,
                          const float* a_amax, const uint8_t* b_codes,
                          const uint8_t* b_scales_tiled, const float* b_amax, int64_t M,
                          int64_t N, int64_t K, const fos_config* cfg, float* out,
                          fos_stream_t stream);

/*
 * fos_dequantize -- standard NVFP4 decode (grouped PR, first commit:
 * "nvfp4_dequantize: the standard NVFP4 decode (recipe-agnostic)"):
 *   out = round_to(out_dt, e2m1(code) * (e4m3(scale) / S)),
 * with S recomputed from amax and cfg->e4m3_bound exactly as fos_quantize
 * does; the candidate choice need not be stored.  cfg->block and
 * cfg->granularity select the scale layout and the amax indexing;
 * mode / metric / precision are ignored.  out is [rows, cols] of out_dt.
 */
FOS_API fos_status fos_dequantize(const uint8_t* codes, const uint8_t* scales, const float* amax,
                          int64_t rows, int64_t cols, const fos_config* cfg, void* out,
                          fos_dtype out_dt, fos_stream_t stream);

/*
 * fos_qdq -- fused fake-QAT quantize-dequantize of a list of n discrete
 * rank-2 tensors (Megatron PR: "General list API" and "Fused data path":
 * codes and E4M3 scales stay in registers; only the dequantized BF16/FP16
 * result is written).  The whole list is processed in one kernel launch
 * (lists longer than FOS_QDQ_MAX_LIST are split into several launches).
 *   x[i], out[i]: device pointers, rows[i] x cols[i], dtype dt (bf16 or
 *   fp16; out has the same dtype).  amax[i]: device pointer to one float,
 *   the per-tensor amax: read when cfg->amax_is_input, else computed and
 *   written first.  Only 1x16 blocks and FOS_SCALE_TENSOR (the pages'
 *   non-goals exclude 2D blocks and row scaling for this path).
 * The host arrays x, out, rows, cols, amax must hold n entries each; the
 * data pointers of an empty tensor (rows or cols 0) may be null.
 * Result equals fos_dequantize(fos_quantize(x)) bit for bit.
 * Errors: FOS_ERR_INVALID_ARG (n < 0, null arrays or pointers, bad enum,
 * tensors on different devices), FOS_ERR_UNSUPPORTED (fp32, 16x16 blocks,
 * per-row scale, cols % 16 != 0), FOS_ERR_MISALIGNED (x or out not 32-byte
 * aligned).
 */
#define FOS_QDQ_MAX_LIST 64
FOS_API fos_status fos_qdq(int n, const void* const* x, void* const* out, const int64_t* rows,
                   const int64_t* cols, float* const* amax, fos_dtype dt,
                   const fos_config* cfg, fos_stream_t stream);

/*
 * fos_qdq_fused -- fos_qdq with the per-tensor amax computed, in ONE
 * persistent launch (the only other work on the stream is a clear of the
 * workspace): the launch runs the amax pass of tensor 0, then
 * quantize-dequantizes tensor i while it computes the amax of tensor i+1
 * (the Megatron PR, "Fused data path", computes each weight's amax with a
 * separate PyTorch reduction first and lists the per-weight launches among
 * its pending work).  Knobs, layouts and results are those of fos_qdq with
 * cfg->amax_is_input = 0, which this call requires; amax[i] receives tensor
 * i's amax.  n <= FOS_QDQ_MAX_LIST.
 *   workspace: the warps of the launch wait for one another (a tensor's QDQ
 *   starts once its amax is complete) and keep their counters here: device
 *   memory owned by the caller, on the tensors' device, 256-byte aligned, at
 *   least fos_qdq_fused_workspace_bytes(n) bytes.  The call clears it on
 *   `stream` before the launch; calls that may run at the same time need
 *   different workspaces.
 * The launch is cooperative (all of its CTAs resident at once); it returns
 * FOS_ERR_CUDA if the device cannot place them.  Every wait is bounded: one
 * that does not complete within about a second ends the launch with the
 * outputs incomplete and a nonzero code in the workspace, which
 * fos_workspace_error reads.
 */
FOS_API size_t fos_qdq_fused_workspace_bytes(int n);
FOS_API fos_status fos_qdq_fused(int n, const void* const* x, void* const* out,
                                 const int64_t* rows, const int64_t* cols, float* const* amax,
                                 fos_dtype dt, const fos_config* cfg, void* workspace,
                                 size_t workspace_bytes, fos_stream_t stream);

/*
 * fos_qdq_fused_static -- fos_qdq_fused without a workspace argument, for
 * callers that have no way to obtain device memory at the point of the call:
 * code that runs inside another framework's allocator and may not go around
 * it, or a runtime that forbids allocations after its start-up.  The pages
 * have no counterpart; this is a convenience of this library.
 * The counters live in one fixed array of the library (768 bytes on every
 * GPU that loads it, kept until the process exits), so lists are limited to
 * n <= FOS_QDQ_MAX_LIST (64); longer lists return FOS_ERR_UNSUPPORTED.
 * Nothing is allocated: no cudaMalloc, no cudaFree, no allocating library
 * call.  Each call looks up the array's device address on the data's device
 * (with that device current), so a reset of that device's primary context
 * between calls is harmless; while `stream` is being captured the address
 * of the previous lookup is reused instead, so make the first call on a
 * device before any stream capture.  Host-side argument checks are those of
 * fos_qdq_fused, in the same order, and come before any CUDA call.  Each
 * call clears the array on `stream` before its launch.
 * Every call on a device shares the one array: calls whose work may overlap
 * on the GPU (other streams, other threads) race and give wrong results;
 * order them on one stream.  A wait that runs out is recorded in the array
 * (not readable through this call); use fos_qdq_fused with a workspace of
 * your own when that must be checked.  Arguments, results and errors are
 * otherwise those of fos_qdq_fused.
 */
FOS_API fos_status fos_qdq_fused_static(int n, const void* const* x, void* const* out,
                                        const int64_t* rows, const int64_t* cols,
                                        float* const* amax, fos_dtype dt,
                                        const fos_config* cfg, fos_stream_t stream);

/*
 * fos_workspace_error -- waits for `stream` to finish, then stores in *code
 * the error word of a workspace used by fos_qdq_fused: 0 when no wait ran
 * out, 1 when one did.  The one call of this library that synchronises the
 * host (a diagnostic).
 */
FOS_API fos_status fos_workspace_error(const void* workspace, fos_stream_t stream, int* code);

/*
 * fos_quantize_grouped -- one call over a packed MoE token tensor (grouped
 * PR, third commit: "each token group's amax expands to a per-row vector so
 * the whole packed tensor quantizes in one call, bitwise identical to
 * quantizing each group separately"; expert weights flatten to one call).
 *   offs: device int32 [G], cumulative group ends.  Group g covers rows
 *   [end_{g-1}, end_g) with end_{-1} = 0 and end_g = clamp(offs[g],
 *   end_{g-1}, rows).  Rows at or past end_{G-1} (the over-allocated tail of
 *   a padded token dispatcher) are not read; their codes and scales are 0.
 *   With 16x16 blocks offs entries should be multiples of 16; a tile belongs
 *   to the group of its first row.
 *   group_amax: device float [G]; read when cfg->amax_is_input, otherwise
 *   computed (NaN-dropping, empty group -> 0) and written.
 *   cfg->granularity is ignored (the group amax is the global scale source).
 *   1 <= G <= FOS_GROUPED_MAX_GROUPS.
 * Errors: FOS_ERR_INVALID_ARG (G < 1, null pointers, bad enum, pointers on
 * different devices), FOS_ERR_UNSUPPORTED (G above the maximum, cols % 16,
 * 16x16 with rows % 16, a bad bound, the sequential order with 16x16),
 * FOS_ERR_MISALIGNED (x not 32-byte, codes not 8-byte, offs not 4-byte
 * aligned).
 */
#define FOS_GROUPED_MAX_GROUPS 8192
FOS_API fos_status fos_quantize_grouped(const void* x, fos_dtype dt, int64_t rows, int64_t cols,
                                const int32_t* offs, int G, const fos_config* cfg,
                                float* group_amax, uint8_t* codes, uint8_t* scales,
                                fos_stream_t stream);

/* Static, human-readable name of a status code. */
FOS_API const char* fos_status_string(fos_status s);

/* Library version as major * 10000 + minor * 100 + patch. */
FOS_API int fos_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FOS_H */

/*
 * fos_diag.h -- element-wise access to the device conversion primitives that
 * the quantizer kernels are built from, so that each rounding step can be
 * checked exhaustively against an independent implementation.  These are
 * the rounding-critical steps the fast-path PR pins ("correctly-rounded FP32
 * division, the FP4/E4M3 casts and their exact decodes").
 *
 * All pointers are device pointers owned by the caller; n elements are
 * processed (pairs for the E2M1 pair conversions); work is enqueued on
 * `stream` and the call does not synchronise the host.
 */
#ifndef FOS_DIAG_H
#define FOS_DIAG_H

#include "fos.h"

#ifdef __cplusplus
extern "C" {
#endif

enum {
    /* in f32[n] (n even) -> out u8[n]: element i's E2M1 code, computed two at a
     * time by the pair conversion the kernels use (RN, satfinite). */
    FOS_DIAG_E2M1_ENCODE = 0,
    /* in u8[n] codes (low 4 bits) -> out f32[n]: exact E2M1 decode. */
    FOS_DIAG_E2M1_DECODE = 1,
    /* in f32[n] (n even) -> out u8[n]: E4M3 code (RN, satfinite), pairwise. */
    FOS_DIAG_E4M3_ENCODE = 2,
    /* in u8[n] -> out f32[n]: exact E4M3 decode. */
    FOS_DIAG_E4M3_DECODE = 3,
    /* in f32[n] (n even) -> out f32[n]: round to binary16 and back, pairwise. */
    FOS_DIAG_F16_ROUND = 4,
    /* in f32[n] (n even) -> out u16[n]: bfloat16 bits (RN), pairwise. */
    FOS_DIAG_BF16_BITS = 5,
    /* in f32[n] (n even) -> out u16[n]: binary16 bits (RN), pairwise. */
    FOS_DIAG_F16_BITS = 6,
    /* in f32[n] -> out f32[n]: the block-scale quotient t / 6, correctly
     * rounded (Markstein's correction where the quotient is normal). */
    FOS_DIAG_DIV6 = 7,
    /* in f32[n] (t = block amax * S, t >= 0) -> out u16[n]: the two E4M3
     * block-scale codes the kernels derive from t, map-to-6 (E4M3 of t / 6)
     * in the low byte and map-to-4 (E4M3 of t / 4) in the high byte. */
    FOS_DIAG_SCALE_CODES = 8
};

/* fos_diag_convert -- applies `op` to n elements of the device buffer `in`
 * and writes `out` (device, caller-owned).  Pairwise ops leave the last
 * output element unwritten when n is odd.  Errors: FOS_ERR_INVALID_ARG (bad
 * op, n < 0, null or non-device pointers, buffers on different devices). */
FOS_API fos_status fos_diag_convert(int op, const void* in, void* out, int64_t n, fos_stream_t stream);

/*
 * fos_diag_wait_timeout -- runs one of the library's bounded waits against a
 * condition that never comes true, so that its time limit and its error
 * report can be checked without faulting or hanging the device:
 *   which = 0: the wait of fos_qdq_fused's CTAs on a counter (word[1],
 *              cleared by the call) that nothing increments; the wait gives
 *              up and stores the workspace error code 1 in word[0];
 *   which = 1: the column-wise kernel's wait on an mbarrier phase that no
 *              copy completes; word[0] = 1 when the wait gave up.
 * word: two uint32 of device memory owned by the caller.  One CTA runs for
 * about a second; the device stays usable afterwards.
 */
FOS_API fos_status fos_diag_wait_timeout(int which, uint32_t* word, fos_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FOS_DIAG_H */

// fos_kernels.cuh -- kernel templates of the four-over-six quantizer and the
// argument blocks the host passes to them.
//
// Work layout (all kernels are persistent: a grid of resident CTAs of 8
// warps; each warp takes one contiguous, balanced range of work units):
//   * 1x16 kernels, per-tensor scale: a unit is 32 consecutive blocks
//     (1 KiB of bf16 input), one block per lane; every warp-wide load is one
//     contiguous 256-bit-per-lane access.
//   * 1x16 kernels, per-row or per-group scale, and dequantize: a unit is
//     (row, 32-block chunk of that row), so the global scale is warp-uniform.
//   * 16x16 kernels: a unit is (16-row band, pair of tiles); each half-warp
//     owns one tile, each lane one row of it.
// The global scale S of the current unit selects a per-warp shared-memory
// table of the common scales of all 127 block-scale codes; it is rebuilt
// only when S changes (per tensor, row, group or list entry).  The next
// unit's input is loaded before the current one is encoded.
#pragma once

#include <cuda.h>

#include "fos_device.cuh"

namespace fos {

struct EncArgs {
    const void* x;
    uint8_t* codes;
    uint8_t* scales;
    const float* amax;     // TENSOR: [1]; ROW: [rows]; GROUP: [G]
    const int32_t* offs;   // GROUP: cumulative ends [G]
    int G;
    int64_t rows;
    int64_t nb;            // blocks (16-column segments) per row
    int64_t nblk;          // rows * nb
    int64_t units;
    int64_t cpr;           // 32-block chunks per row (ROW / GROUP)
    float six_bound;       // 6 * E4M3 bound
    float neg_zero;        // -0.0f (run-time operand of mul2_nc)
    int amax_given;        // row pass: amax is an input (else computed, written)
    int64_t sc_pc4;        // tiled scales: 4-block tiles per tile-row (kernels with TL)
};

// Scale byte index of block (row, j) = flat block b: the plain layout, or
// with TL the tiled layout of block-scaled FP4 GEMMs.
template <bool TL>
__device__ __forceinline__ int64_t scale_at(int64_t b, int64_t row, int64_t j, int64_t pc4) {
    if constexpr (TL) return tiled_scale_off((int32_t)row, (int32_t)j, (int32_t)pc4);
    else return b;
}

struct QdqTensor {
    const void* x;
    void* out;
    const float* amax;
    int64_t nblk;
    int64_t unit_begin;
};

constexpr int kQdqMaxList = 64;
constexpr int kQdqCtaTables = 16;  // QDQ lists up to this long keep all tables per CTA

// Dynamic shared memory of the QDQ list kernel: its common-scale tables.
inline size_t qdq_table_bytes(int n) {
    return (size_t)(n <= kQdqCtaTables ? n : kWarps) * 128 * 8;
}

struct QdqArgs {
    int n;
    int64_t units;
    float six_bound;
    float neg_zero;
    QdqTensor t[kQdqMaxList + 1];  // t[n].unit_begin == units
};

struct DeqArgs {
    const uint8_t* codes;
    const uint8_t* scales;
    const float* amax;
    void* out;
    int64_t rows, nb, units, cpr;
    float six_bound;
};

struct AmaxArgs {
    const void* x;
    float* amax;
    float* clear;          // optional: set to +0 by the launch (a later stage's amax)
    const int32_t* offs;
    int G;
    int64_t rows, nb, units;
};

__device__ __forceinline__ float warp_max_dev(float m) {
#pragma unroll
    for (int w = 16; w >= 1; w >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, w));
    return m;
}

// Position of a (row, chunk) walk.
struct RowChunk {
    int64_t row, chunk;
    __device__ __forceinline__ void next(int64_t cpr) {
        if (++chunk == cpr) { chunk = 0; ++row; }
    }
};

template <In IT, L2 H = L2::NORMAL>
__device__ __forceinline__ void load_if(Raw<IT>& r, const char* p, bool v) {
    if (v) load_seg<IT, H>(r, p);
}

// L2 priorities of the per-tensor paths.
constexpr L2 kEncHint = L2::FIRST;    // encode loads (read once)
constexpr L2 kAmaxHint = L2::NORMAL;  // amax-pass loads
constexpr L2 kQdqHint = L2::NORMAL;   // fused QDQ loads
// Minimum resident CTAs per SM the encode kernels are compiled for: caps
// their registers at 65536 / (256 * n).
constexpr int kStdMinCtas = 5;
constexpr int kFosMinCtas = 4;
template <Err EM>
constexpr int min_ctas() { return EM == Err::STD ? kStdMinCtas : kFosMinCtas; }
// 16x16 (two rows per lane and the next two in flight): up to 128 registers
// (2 CTAs per SM); measured faster than 80 registers at 3 CTAs per SM.
template <In IT>
constexpr int tile_min_ctas() { return 2; }

// ------------------------------------------------------------------------
// 1x16 quantize with a per-tensor scale.  Grid-stride over 32-block units:
// in each step the grid sweeps one contiguous window of the tensor; every
// lane loads its next block one step ahead.
// ------------------------------------------------------------------------
constexpr int kTensorBuf = 2;  // register buffers of the per-tensor encode (prefetch depth + 1)

template <In IT, Err EM, bool TL = false, int kBuf = kTensorBuf>
__global__ void __launch_bounds__(kThreads, min_ctas<EM>()) k_quant1x16_tensor(const EncArgs a) {
    chain_wait();
    chain_release();
    __shared__ float2 tbl[128];  // one common-scale table for the CTA
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint64_t nz = pk(a.neg_zero, a.neg_zero);
    const int64_t nw = (int64_t)gridDim.x * kWarps;
    const int64_t u = (int64_t)blockIdx.x * kWarps + warp;
    constexpr int64_t kBytes = (IT == In::F32) ? 64 : 32;
    const char* xb = static_cast<const char*>(a.x);
    // kBuf register buffers rotate over consecutive grid-stride units: unit i
    // lives in buffer i % kBuf and is loaded kBuf - 1 units before it is
    // encoded.  The loop body is unrolled over the buffers so every index is
    // static (no register copies, no local memory).
    const int64_t step = nw * 32;
    const int64_t b0 = u * 32 + lane;
    Raw<IT> buf[kBuf];
#pragma unroll
    for (int k = 0; k < kBuf - 1; ++k) {
        const int64_t bk = b0 + k * step;
        load_if<IT, kEncHint>(buf[k], xb + bk * kBytes, bk < a.nblk);
    }
    const float S = global_scale(a.amax[0], a.six_bound);
    fill_table_cta(tbl, S, threadIdx.x);
    __syncthreads();
    if (u >= a.units) return;
    uint32_t dummy[8];
    // TL: (row, column block) of the block encoded next, advanced by one grid
    // step per block
    BlockPos pos;
    int32_t srow = 0, scol = 0, nb32 = (int32_t)a.nb;
    if constexpr (TL) {
        pos.init(b0, a.nb);
        srow = (int32_t)(step / a.nb);
        scol = (int32_t)(step - (int64_t)srow * a.nb);
    }
    // Steady state: while every unit this step loads or encodes is whole
    // (the test is on the unit's first block, the same for the whole warp),
    // loads and encodes go without bounds checks or branches; the guarded
    // loop below finishes the tail.
    int64_t b = b0;
    for (; b - lane + (2 * kBuf - 2) * step + 31 < a.nblk; b += kBuf * step) {
#pragma unroll
        for (int k = 0; k < kBuf; ++k) {
            load_seg<IT, kEncHint>(buf[(k + kBuf - 1) % kBuf],
                                   xb + (b + (k + kBuf - 1) * step) * kBytes);
            uint64_t xp[8];
            widen<IT>(buf[k], xp);
            uint32_t code[2], scale;
            const int64_t bc = b + k * step;
            encode_block<EM, Out::NONE>(xp, S, tbl, nz, code, scale, dummy);
            st64(a.codes + bc * 8, code[0], code[1]);
            st8(a.scales + scale_at<TL>(bc, pos.row, pos.col, a.sc_pc4), scale);
            if constexpr (TL) pos.advance(srow, scol, nb32);
        }
    }
    for (; b < a.nblk + lane; b += kBuf * step) {  // b - lane: first block of unit
#pragma unroll
        for (int k = 0; k < kBuf; ++k) {
            const int64_t bl = b + (k + kBuf - 1) * step;  // unit loaded now
            load_if<IT, kEncHint>(buf[(k + kBuf - 1) % kBuf], xb + bl * kBytes, bl < a.nblk);
            const int64_t bc = b + k * step;  // unit encoded now
            if (bc < a.nblk) {
                uint64_t xp[8];
                widen<IT>(buf[k], xp);
                uint32_t code[2], scale;
                encode_block<EM, Out::NONE>(xp, S, tbl, nz, code, scale, dummy);
                st64(a.codes + bc * 8, code[0], code[1]);
                st8(a.scales + scale_at<TL>(bc, pos.row, pos.col, a.sc_pc4), scale);
            }
            if constexpr (TL) pos.advance(srow, scol, nb32);
        }
    }
}

// ------------------------------------------------------------------------
// 1x16 quantize with a per-row or per-group scale.  Each warp walks one
// contiguous range of (row, 32-block chunk) units so that the global scale
// (and its table) changes only at row / group boundaries.
// ------------------------------------------------------------------------
template <In IT, Err EM, Src SRC, bool TL = false>
__global__ void __launch_bounds__(kThreads, min_ctas<EM>()) k_quant1x16(const EncArgs a) {
    chain_wait();
    chain_release();
    extern __shared__ int32_t s_ends[];
    __shared__ float2 s_tbl[kWarps][128];
    if constexpr (SRC == Src::GROUP) load_group_ends(s_ends, a.offs, a.G, a.rows);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float2* tbl = s_tbl[warp];
    const uint64_t nz = pk(a.neg_zero, a.neg_zero);
    const int64_t nw = (int64_t)gridDim.x * kWarps, gw = (int64_t)blockIdx.x * kWarps + warp;
    const int64_t u0 = split_at(a.units, nw, gw), u1 = split_at(a.units, nw, gw + 1);
    if (u0 >= u1) return;
    constexpr int64_t kBytes = (IT == In::F32) ? 64 : 32;
    const char* xb = static_cast<const char*>(a.x);
    int64_t last_end = a.rows;
    if constexpr (SRC == Src::GROUP) last_end = s_ends[a.G - 1];
    RowChunk cc{u0 / a.cpr, u0 % a.cpr};
    int64_t j = cc.chunk * 32 + lane;
    Raw<IT> cur;
    load_if<IT, kEncHint>(cur, xb + (cc.row * a.nb + j) * kBytes, j < a.nb && cc.row < last_end);
    int g = 0;
    if constexpr (SRC == Src::GROUP)
        while (g < a.G && cc.row >= s_ends[g]) ++g;
    int64_t key = -1;
    float S = 1.0f;
    uint32_t dummy[8];
    const bool whole_chunks = (a.nb & 31) == 0;
    for (int64_t u = u0; u < u1; ++u) {
        int64_t k;
        if constexpr (SRC == Src::ROW) {
            k = cc.row;
        } else {
            while (g < a.G && cc.row >= s_ends[g]) ++g;
            k = g;  // g == G: tail past the last group end
        }
        if (k != key) {
            key = k;
            if (SRC == Src::ROW || k < a.G) {
                S = global_scale(a.amax[k], a.six_bound);
                build_table(tbl, S, lane);
            }
        }
        if (whole_chunks && (SRC == Src::ROW || k < a.G)) {
            // Steady state: the next unit is whole and under the same scale.
            // With whole chunks, unit v's block of this lane is v * 32 + lane
            // in the flat block order, so the walk just adds 32 (the row and
            // chunk are recovered once, when it ends).
            const int64_t seg_end = (SRC == Src::ROW) ? cc.row + 1 : (int64_t)s_ends[k];
            const int64_t u_end = min(u1, seg_end * a.cpr);  // past this warp's units of the segment
            if (u + 1 < u_end) {
                int64_t b = u * 32 + lane;
                BlockPos pos;
                if constexpr (TL) {
                    pos.row = (int32_t)cc.row;
                    pos.col = (int32_t)j;
                }
                const int32_t nb32 = (int32_t)a.nb;
                do {
                    Raw<IT> nxt;
                    load_seg<IT, kEncHint>(nxt, xb + (b + 32) * kBytes);
                    uint64_t xp[8];
                    widen<IT>(cur, xp);
                    uint32_t code[2], scale;
                    encode_block<EM, Out::NONE, SRC == Src::GROUP>(xp, S, tbl, nz, code, scale,
                                                                   dummy);
                    st64(a.codes + b * 8, code[0], code[1]);
                    st8(a.scales + scale_at<TL>(b, pos.row, pos.col, a.sc_pc4), scale);
                    if constexpr (TL) pos.advance(0, 32, nb32);
                    cur = nxt;
                    b += 32;
                    ++u;
                } while (u + 1 < u_end);
                cc.row = u / a.cpr;
                cc.chunk = u - cc.row * a.cpr;
                j = cc.chunk * 32 + lane;
            }
        }
        RowChunk nc = cc;
        nc.next(a.cpr);
        const int64_t jn = nc.chunk * 32 + lane;
        Raw<IT> nxt;
        load_if<IT, kEncHint>(nxt, xb + (nc.row * a.nb + jn) * kBytes,
                    u + 1 < u1 && jn < a.nb && nc.row < last_end);
        const int64_t b = cc.row * a.nb + j;
        if (j < a.nb) {
            if (cc.row < last_end) {
                uint64_t xp[8];
                widen<IT>(cur, xp);
                uint32_t code[2], scale;
                encode_block<EM, Out::NONE, SRC == Src::GROUP>(xp, S, tbl, nz, code, scale, dummy);
                st64(a.codes + b * 8, code[0], code[1]);
                st8(a.scales + scale_at<TL>(b, cc.row, j, a.sc_pc4), scale);
            } else {  // zero-extended tail of a padded grouped tensor
                st64(a.codes + b * 8, 0u, 0u);
                st8(a.scales + b, 0u);
            }
        }
        cur = nxt;
        cc = nc;
        j = jn;
    }
}

// ------------------------------------------------------------------------
// 1x16 quantize with a per-row scale in one pass: one CTA per row at a time
// (grid-stride over rows).  Each thread keeps its K blocks of the row in
// registers; the row amax (when it is not given) is a CTA max-reduction and
// is written out, the CTA builds the row's common-scale table (one division
// per thread), then encodes.  The next row is loaded before the current one
// is encoded.  The table is double-buffered by row parity: a buffer is
// rewritten two rows later, after every thread has passed the barrier of the
// row in between and so finished reading it.  One barrier per row (table
// ready) with the amax given, two with the amax computed (reduction, table).
// With the amax given, warp 0 computes the next row's global scale while the
// table of the current row is filled (the other warps read it from shared
// memory), and each block is widened once.
// ------------------------------------------------------------------------
template <In IT, Err EM, int K, bool TL = false>
__global__ void __launch_bounds__(kThreads) k_quant1x16_rowpass(const EncArgs a) {
    chain_wait();
    chain_release();
    __shared__ float2 s_tbl[2][128];
    __shared__ float s_red[kWarps];
    __shared__ float s_S[2];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint64_t nz = pk(a.neg_zero, a.neg_zero);
    constexpr int64_t kBytes = (IT == In::F32) ? 64 : 32;
    const char* xb = static_cast<const char*>(a.x);
    float* amax_out = const_cast<float*>(a.amax);
    int64_t row = blockIdx.x;
    if (row >= a.rows) return;
    Raw<IT> cur[K], nxt[K];
#pragma unroll
    for (int k = 0; k < K; ++k) {
        const int64_t j = tid + (int64_t)k * kThreads;
        load_if<IT, kEncHint>(cur[k], xb + (row * a.nb + j) * kBytes, j < a.nb);
    }
    uint32_t dummy[8];
    int par = 0;
    if (a.amax_given) {
        // The row's global scale is computed once per CTA, by warp 0 a row
        // ahead (into s_S, double-buffered like the table), and each block is
        // widened once: its amax comes out of the encode.
        float S = global_scale(a.amax[row], a.six_bound);
        for (; row < a.rows; row += gridDim.x, par ^= 1) {
            const int64_t rown = row + gridDim.x;
#pragma unroll
            for (int k = 0; k < K; ++k) {
                const int64_t j = tid + (int64_t)k * kThreads;
                load_if<IT, kEncHint>(nxt[k], xb + (rown * a.nb + j) * kBytes,
                                      rown < a.rows && j < a.nb);
            }
            fill_table_cta(s_tbl[par], S, tid);
            if (warp == 0 && rown < a.rows) {
                const float Sn = global_scale(a.amax[rown], a.six_bound);
                if (lane == 0) s_S[par] = Sn;
            }
            __syncthreads();
            const float Sn = s_S[par];  // read before the next barrier: rewritten two rows on
#pragma unroll
            for (int k = 0; k < K; ++k) {
                const int64_t j = tid + (int64_t)k * kThreads;
                if (j < a.nb) {
                    uint64_t xp[8];
                    widen<IT>(cur[k], xp);
                    uint32_t code[2], scale;
                    encode_block<EM, Out::NONE>(xp, S, s_tbl[par], nz, code, scale, dummy);
                    const int64_t b = row * a.nb + j;
                    st64(a.codes + b * 8, code[0], code[1]);
                    st8(a.scales + scale_at<TL>(b, row, j, a.sc_pc4), scale);
                }
                cur[k] = nxt[k];
            }
            S = Sn;
        }
        return;
    }
    for (; row < a.rows; row += gridDim.x, par ^= 1) {
        const int64_t rown = row + gridDim.x;
#pragma unroll
        for (int k = 0; k < K; ++k) {
            const int64_t j = tid + (int64_t)k * kThreads;
            load_if<IT, kEncHint>(nxt[k], xb + (rown * a.nb + j) * kBytes, rown < a.rows && j < a.nb);
        }
        float bam[K];
        float m = 0.0f;
#pragma unroll
        for (int k = 0; k < K; ++k) {
            uint64_t xp[8];
            widen<IT>(cur[k], xp);
            // blocks past the row end were not loaded and contribute nothing
            bam[k] = (tid + (int64_t)k * kThreads < a.nb) ? seg_amax(xp) : 0.0f;
            m = fmaxf(m, bam[k]);
        }
        m = warp_max_dev(m);
        if (lane == 0) s_red[warp] = m;
        __syncthreads();
        float A = 0.0f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) A = fmaxf(A, s_red[w]);
        if (tid == 0) amax_out[row] = A;
        const float S = global_scale(A, a.six_bound);
        fill_table_cta(s_tbl[par], S, tid);
        __syncthreads();
#pragma unroll
        for (int k = 0; k < K; ++k) {
            const int64_t j = tid + (int64_t)k * kThreads;
            if (j < a.nb) {
                uint64_t xp[8];
                widen<IT>(cur[k], xp);
                uint32_t code[2], scale;
                encode_block_amax<EM, Out::NONE>(xp, bam[k], S, s_tbl[par], nz, code, scale, dummy);
                const int64_t b = row * a.nb + j;
                st64(a.codes + b * 8, code[0], code[1]);
                st8(a.scales + scale_at<TL>(b, row, j, a.sc_pc4), scale);
            }
            cur[k] = nxt[k];
        }
    }
}

// ------------------------------------------------------------------------
// Fused quantize-dequantize over a list of tensors (per-tensor scale, 1x16),
// output dtype == input dtype (bf16 / fp16).  Codes and scales never leave
// registers.  Grid-stride over the concatenated 32-block units of the list
// (empty tensors own no units); the per-warp table is rebuilt whenever the
// warp's unit moves into the next tensor.
// ------------------------------------------------------------------------
template <In IT, Err EM>
__global__ void __launch_bounds__(kThreads, min_ctas<EM>()) k_qdq1x16(const __grid_constant__ QdqArgs a) {
    chain_wait();
    chain_release();
    static_assert(IT != In::F32, "fused QDQ is bf16 / fp16 only");
    constexpr Out OT = (IT == In::BF16) ? Out::BF16 : Out::F16;
    // Common-scale tables (dynamic shared memory, qdq_table_bytes): a list of
    // up to kQdqCtaTables tensors gets every tensor's table filled once per
    // CTA at the start (about n divisions per thread); a longer list keeps
    // one table per warp, rebuilt when the warp moves into the next tensor.
    extern __shared__ float2 s_tbls[];
    __shared__ float s_S[kQdqCtaTables];
    const bool cta_tables = a.n <= kQdqCtaTables;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint64_t nz = pk(a.neg_zero, a.neg_zero);
    const int64_t nw = (int64_t)gridDim.x * kWarps;
    int64_t u = (int64_t)blockIdx.x * kWarps + warp;
    int t = 0;
    while (t < a.n && a.t[t + 1].unit_begin <= u) ++t;
    int64_t b = (u - a.t[t].unit_begin) * 32 + lane;
    bool v = u < a.units && b < a.t[t].nblk;
    Raw<IT> cur;  // the first load goes out before the tables are filled
    load_if<IT, kQdqHint>(cur, static_cast<const char*>(a.t[t].x) + b * 32, v);
    if (cta_tables) {
        if ((int)threadIdx.x < a.n) s_S[threadIdx.x] = global_scale(*a.t[threadIdx.x].amax, a.six_bound);
        __syncthreads();
        for (int i = 0; i < a.n; ++i) fill_table_cta(s_tbls + 128 * i, s_S[i], threadIdx.x);
        __syncthreads();
    }
    float2* tbl = s_tbls + 128 * warp;
    if (u >= a.units) return;
    int ti = -1;
    float S = 1.0f;
    for (; u < a.units; u += nw) {
        if (t != ti) {
            ti = t;
            if (cta_tables) {
                S = s_S[t];
                tbl = s_tbls + 128 * t;
            } else {
                S = global_scale(*a.t[t].amax, a.six_bound);
                build_table(tbl, S, lane);
            }
        }
        if constexpr (EM != Err::STD) {
            // Steady state (4/6 modes): while the unit loaded next is whole
            // and in the same tensor, no tensor lookup and no bounds checks.
            // (In standard mode the same loop measured slower.)
            const int64_t ub = a.t[t].unit_begin;
            const int64_t t_end = ub + a.t[t].nblk / 32;  // first unit that is not whole
            const char* xt = static_cast<const char*>(a.t[t].x);
            char* ot = static_cast<char*>(a.t[t].out);
            while (u + nw < t_end) {
                const int64_t bn = (u + nw - ub) * 32 + lane;
                Raw<IT> nxt;
                load_seg<IT, kQdqHint>(nxt, xt + bn * 32);
                uint64_t xp[8];
                widen<IT>(cur, xp);
                uint32_t code[2], scale, out[8];
                encode_block<EM, OT, EM == Err::STD>(xp, S, tbl, nz, code, scale, out);
                st256(ot + b * 32, out);
                cur = nxt;
                b = bn;
                u += nw;
            }
        }
        const int64_t un = u + nw;
        int tn = t;
        while (tn < a.n && a.t[tn + 1].unit_begin <= un) ++tn;  // t[n] is a sentinel
        const int64_t bn = (un - a.t[tn].unit_begin) * 32 + lane;
        const bool vn = un < a.units && bn < a.t[tn].nblk;
        Raw<IT> nxt;
        load_if<IT, kQdqHint>(nxt, static_cast<const char*>(a.t[tn].x) + bn * 32, vn);
        if (v) {
            uint64_t xp[8];
            widen<IT>(cur, xp);
            uint32_t code[2], scale, out[8];
            encode_block<EM, OT, EM == Err::STD>(xp, S, tbl, nz, code, scale, out);
            st256(static_cast<char*>(a.t[t].out) + b * 32, out);
        }
        cur = nxt;
        t = tn;
        b = bn;
        v = vn;
    }
}

// ------------------------------------------------------------------------
// Column-wise quantize: the 1x16 quantization of x^T, computed from the
// row-major x without forming x^T (the operand layout a weight-gradient
// GEMM reads).  Each CTA walks tiles of kR rows x 256 columns grid-stride.
// A tile arrives in shared memory by one 2D TMA load (cp.async.bulk.tensor,
// completion on an mbarrier; elements past the tensor edge are filled with
// zeros) into one of two buffers, the next tile's load being issued before
// the current tile is worked on.  With DUAL, each thread first encodes four
// (two for fp32) 16-element row segments of the tile row-wise, so one read
// of x gives both layouts.  Then thread c encodes the kR/16 16-row blocks
// of tile column c and writes that part of row c of x^T.  The scale is per
// tensor (x and x^T have one amax).  The mbarrier waits are bounded: a wait
// that runs out sets the first scale byte of x^T to 0xFF (a code the
// quantizer never writes) after draining its own load, and ends the CTA.
// ------------------------------------------------------------------------
template <In IT>
struct ColTile {
    static constexpr int kR = (IT == In::F32) ? 32 : 64;  // tile rows
    static constexpr int kC = 256;                         // tile columns, one per thread
    static constexpr int kElt = (IT == In::F32) ? 4 : 2;
    static constexpr int kBytes = kR * kC * kElt;          // 32 KiB
};
constexpr uint32_t kMbarSpins = 1u << 20;  // tries of at most about 1 us each

struct ColArgs {
    CUtensorMap tmap;   // x as [rows, cols], box kR x 256 (2D TMA)
    uint8_t* codes_t;   // [cols, rows / 2]
    uint8_t* scales_t;  // [cols, rows / 16]
    uint8_t* codes;     // DUAL: [rows, cols / 2]
    uint8_t* scales;    // DUAL: [rows, cols / 16]
    const float* amax;  // [1]
    int64_t rows, cols;
    int64_t tiles_c;    // tiles across the columns
    int64_t tiles;
    float six_bound;
    float neg_zero;
    int64_t pc4_t;      // tiled scales of x^T (TL): 4-block tiles per tile-row
    int64_t pc4;        // tiled scales of x (TL, DUAL)
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes) : "memory");
}
// Bounded wait for the phase with the given parity to complete.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
    for (uint32_t i = 0; i < kMbarSpins; ++i) {
        uint32_t done;
        asm volatile("{\n\t.reg .pred p;\n\t"
                     "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, 1000;\n\t"
                     "selp.u32 %0, 1, 0, p;\n\t}"
                     : "=r"(done) : "r"(smem_u32(bar)), "r"(parity) : "memory");
        if (done) return true;
    }
    return false;
}
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int32_t x, int32_t y,
                                            uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];"
        ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y),
          "r"(smem_u32(bar)) : "memory");
}

// Elements (rb*16 .. rb*16+15, column c) of a staged tile as one segment.
template <In IT>
__device__ __forceinline__ void gather_col(const unsigned char* tile, int rb, int c, Raw<IT>& r) {
    constexpr int kC = ColTile<IT>::kC;
    if constexpr (IT == In::F32) {
        const uint32_t* t = reinterpret_cast<const uint32_t*>(tile);
#pragma unroll
        for (int i = 0; i < 16; ++i) r.w[i] = t[(rb * 16 + i) * kC + c];
    } else {
        const uint16_t* t = reinterpret_cast<const uint16_t*>(tile);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint32_t lo = t[(rb * 16 + 2 * j) * kC + c];
            const uint32_t hi = t[(rb * 16 + 2 * j + 1) * kC + c];
            r.w[j] = lo | (hi << 16);
        }
    }
}

template <In IT>
__device__ __forceinline__ void read_seg_smem(const unsigned char* p, Raw<IT>& r) {
    const uint4* q = reinterpret_cast<const uint4*>(p);
#pragma unroll
    for (int i = 0; i < InTraits<IT>::kWords / 4; ++i) {
        const uint4 v = q[i];
        r.w[4 * i] = v.x;
        r.w[4 * i + 1] = v.y;
        r.w[4 * i + 2] = v.z;
        r.w[4 * i + 3] = v.w;
    }
}

template <In IT, Err EM, bool DUAL, bool TL = false>
__global__ void __launch_bounds__(kThreads, min_ctas<EM>())
    k_quant_colwise(const __grid_constant__ ColArgs a) {
    using T = ColTile<IT>;
    chain_wait();
    chain_release();
    extern __shared__ __align__(128) unsigned char s_dyn[];  // two tiles of T::kBytes + 128
    // TMA destinations start on 128-byte boundaries: round the base up (the
    // launch reserves 128 spare bytes for this)
    unsigned char* s_buf = s_dyn + ((128u - (smem_u32(s_dyn) & 127u)) & 127u);
    __shared__ __align__(8) uint64_t s_bar[2];
    __shared__ float2 tbl[128];  // one common-scale table for the CTA
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint64_t nz = pk(a.neg_zero, a.neg_zero);
    const float S = global_scale(a.amax[0], a.six_bound);
    fill_table_cta(tbl, S, tid);  // ordered before use by the barrier below
    if (tid == 0) {
        mbar_init(&s_bar[0], 1);
        mbar_init(&s_bar[1], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    auto issue = [&](int64_t t, int b) {  // thread 0 only
        const int32_t r0 = (int32_t)((t / a.tiles_c) * T::kR);
        const int32_t c0 = (int32_t)((t % a.tiles_c) * T::kC);
        mbar_expect_tx(&s_bar[b], (uint32_t)T::kBytes);
        tma_load_2d(s_buf + b * T::kBytes, &a.tmap, c0, r0, &s_bar[b]);
    };
    if (tid == 0 && (int64_t)blockIdx.x < a.tiles) issue(blockIdx.x, 0);
    const int64_t nb_t = a.rows / 16;  // blocks per row of x^T
    // wide stores of a column's codes and scales need the row count to be a
    // multiple of the tile height and the output bases aligned to their size
    constexpr int kNBt = T::kR / 16;
    const bool full_rows = a.rows % T::kR == 0 &&
                           (reinterpret_cast<uintptr_t>(a.codes_t) % (8 * kNBt)) == 0 &&
                           (reinterpret_cast<uintptr_t>(a.scales_t) % kNBt) == 0;
    uint32_t dummy[8];
    int i = 0;
    for (int64_t tile = blockIdx.x; tile < a.tiles; tile += gridDim.x, ++i) {
        const int b = i & 1;
        const bool next = tile + gridDim.x < a.tiles;
        if (tid == 0 && next) {
            // buffer b^1 was last read in the previous tile, before the barrier
            // that ended it; order those reads before the asynchronous write
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            issue(tile + gridDim.x, b ^ 1);
        }
        const bool ok = mbar_wait(&s_bar[b], (uint32_t)((i >> 1) & 1));
        if (__syncthreads_or(!ok)) {
            if (tid == 0) {
                if (next) mbar_wait(&s_bar[b ^ 1], (uint32_t)(((i + 1) >> 1) & 1));  // drain
                a.scales_t[0] = 0xFF;
            }
            return;
        }
        const unsigned char* tb = s_buf + b * T::kBytes;
        const int64_t r0 = (tile / a.tiles_c) * T::kR, c0 = (tile % a.tiles_c) * T::kC;
        if constexpr (DUAL) {
#pragma unroll
            for (int k = 0; k < T::kR * T::kC / 16 / kThreads; ++k) {
                const int seg = tid + kThreads * k;
                const int tr = seg >> 4, ts = seg & 15;  // tile row, 16-column segment
                const int64_t row = r0 + tr, col = c0 + ts * 16;
                if (row < a.rows && col < a.cols) {
                    Raw<IT> raw;
                    read_seg_smem<IT>(tb + (tr * T::kC + ts * 16) * T::kElt, raw);
                    uint64_t xp[8];
                    widen<IT>(raw, xp);
                    uint32_t code[2], scale;
                    encode_block<EM, Out::NONE>(xp, S, tbl, nz, code, scale, dummy);
                    const int64_t blk = row * (a.cols / 16) + col / 16;
                    st64(a.codes + blk * 8, code[0], code[1]);
                    st8(a.scales + scale_at<TL>(blk, row, col / 16, a.pc4), scale);
                }
            }
        }
        const int64_t col = c0 + tid;  // one tile column per thread
        if (col < a.cols) {
            constexpr int kNB = T::kR / 16;  // blocks of the column in this tile
            // whole tile and rows a multiple of the tile height: the kNB
            // blocks' codes (8 * kNB bytes) and scales (kNB bytes) of row col
            // of x^T are contiguous and aligned, one store each
            const bool whole = full_rows && r0 + T::kR <= a.rows;
            uint32_t cw[2 * kNB], sw = 0;
#pragma unroll
            for (int rb = 0; rb < kNB; ++rb) {
                const int64_t row = r0 + rb * 16;  // rows % 16 == 0: a block is whole or absent
                if (row < a.rows) {
                    Raw<IT> raw;
                    gather_col<IT>(tb, rb, tid, raw);
                    uint64_t xp[8];
                    widen<IT>(raw, xp);
                    uint32_t code[2], scale;
                    encode_block<EM, Out::NONE>(xp, S, tbl, nz, code, scale, dummy);
                    cw[2 * rb] = code[0];
                    cw[2 * rb + 1] = code[1];
                    sw |= scale << (8 * rb);
                    if (!whole) {
                        const int64_t blk = col * nb_t + row / 16;
                        st64(a.codes_t + blk * 8, code[0], code[1]);
                        st8(a.scales_t + scale_at<TL>(blk, col, row / 16, a.pc4_t), scale);
                    }
                }
            }
            if (whole) {
                const int64_t blk = col * nb_t + r0 / 16;
                // tiled: the kNB scales (kNB | 4, r0 / 16 a multiple of kNB) are
                // consecutive bytes of one 4-byte group of the tile
                const int64_t sidx = scale_at<TL>(blk, col, r0 / 16, a.pc4_t);
                if constexpr (kNB == 4) {
                    st256(a.codes_t + blk * 8, cw);
                    st32(a.scales_t + sidx, sw);
                } else {
                    st128(a.codes_t + blk * 8, cw);
                    st16(a.scales_t + sidx, sw);
                }
            }
        }
        __syncthreads();  // buffer b is refilled two tiles on
    }
}

// ------------------------------------------------------------------------
// Fused multi-tensor amax + QDQ in one persistent launch.  The launch first
// runs the amax pass of tensor 0 with every warp; then, for each tensor i,
// it quantize-dequantizes tensor i while every warp folds one segment of
// tensor i+1 into its running max per step (as the list pipeline does).  A
// CTA starts the QDQ of tensor i once every CTA of the grid has finished its
// share of tensor i's amax: a CTA max-reduces its warps' maxima, atomicMax-es
// the result into the workspace and then adds 1 to the tensor's counter with
// release semantics; one thread per CTA polls the counter with acquire loads
// (backing off with nanosleep) until it holds the number of CTAs and hands
// the amax to the other threads through shared memory.  The launch is
// cooperative (all CTAs resident at once) and no CTA leaves early, so every
// counter fills; a wait still gives up after kWaitSpins polls (about a
// second), records kWsTimeout in the workspace and ends its CTA, and a CTA
// that sees a recorded failure stops waiting too.
// ------------------------------------------------------------------------
constexpr uint32_t kWaitSpins = 1u << 20;  // polls of up to about 1 us each
constexpr uint32_t kWsTimeout = 1u;        // workspace error code: a wait ran out

// Workspace of the fused launch (device memory, cleared before the launch):
// word 0 the error code, then n counters, then n running amaxes (float bits).
struct FusedWs {
    uint32_t* err;
    uint32_t* cnt;
    uint32_t* acc;
};

struct QdqFusedArgs {
    QdqArgs q;                       // t[i].amax unused; amax_out receives the amaxes
    float* amax_out[kQdqMaxList];
    FusedWs ws;
};

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void red_release_add_gpu(uint32_t* p, uint32_t v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// The CTA's share of one tensor's amax is done: max into the running amax,
// then count the CTA in (release orders the max before the count).  Every
// thread of the CTA calls it.
__device__ __forceinline__ void fused_arrive(float m, uint32_t* acc, uint32_t* cnt, float* s_red,
                                             int warp, int lane) {
    m = warp_max_dev(m);
    if (lane == 0) s_red[warp] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        float c = 0.0f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) c = fmaxf(c, s_red[w]);
        if (c > 0.0f) atomicMax(acc, __float_as_uint(c));
        red_release_add_gpu(cnt, 1u);
    }
}

// Wait until *cnt reaches target (every thread of the CTA calls it); returns
// the tensor's amax, or a negative value when the wait gave up (the error is
// then recorded).
__device__ __forceinline__ float fused_wait(const uint32_t* cnt, const uint32_t* acc,
                                            uint32_t target, uint32_t* err, float* s_amax) {
    if (threadIdx.x == 0) {
        float A = -1.0f;
        uint32_t spins = 0, sleep = 32;
        for (;;) {
            if (ld_acquire_gpu(cnt) >= target) {
                A = __uint_as_float(ld_acquire_gpu(acc));
                break;
            }
            if (ld_acquire_gpu(err) != 0u || ++spins > kWaitSpins) {
                atomicCAS(err, 0u, kWsTimeout);
                break;
            }
            __nanosleep(sleep);
            if (sleep < 1024) sleep *= 2;
        }
        *s_amax = A;
    }
    __syncthreads();
    return *s_amax;
}

template <In IT, Err EM>
__global__ void __launch_bounds__(kThreads, min_ctas<EM>())
    k_qdq_fused(const __grid_constant__ QdqFusedArgs a) {
    static_assert(IT != In::F32, "fused QDQ is bf16 / fp16 only");
    constexpr Out OT = (IT == In::BF16) ? Out::BF16 : Out::F16;
    constexpr int64_t kBytes = 32;
    __shared__ float2 tbl[128];  // the current tensor's common-scale table, one per CTA
    __shared__ float s_red[kWarps];
    __shared__ float s_amax;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint64_t nz = pk(a.q.neg_zero, a.q.neg_zero);
    const int64_t nw = (int64_t)gridDim.x * kWarps;
    const int64_t step = nw * 32;
    const int64_t b0 = ((int64_t)blockIdx.x * kWarps + warp) * 32 + lane;
    {  // amax pass of tensor 0
        const char* ab = static_cast<const char*>(a.q.t[0].x);
        const int64_t aseg = a.q.t[0].nblk;
        float m = 0.0f;
        for (int64_t b = b0; b < aseg + lane; b += step) {  // b - lane: first segment of unit
            Raw<IT> r;
            zero_seg<IT>(r);
            if (b < aseg) load_seg<IT, kAmaxHint>(r, ab + b * kBytes);
            uint64_t xq[8];
            widen<IT>(r, xq);
            m = fmaxf(m, seg_amax(xq));
        }
        fused_arrive(m, &a.ws.acc[0], &a.ws.cnt[0], s_red, warp, lane);
    }
    for (int s = 0; s < a.q.n; ++s) {
        const float A = fused_wait(&a.ws.cnt[s], &a.ws.acc[s], gridDim.x, a.ws.err, &s_amax);
        if (A < 0.0f) return;  // the wait gave up (the whole CTA leaves); failure recorded
        if (blockIdx.x == 0 && threadIdx.x == 0) *a.amax_out[s] = A;
        const float S = global_scale(A, a.q.six_bound);
        // every warp of the CTA is past the previous tensor (fused_wait ends
        // with a CTA barrier), so the one table can be refilled
        fill_table_cta(tbl, S, threadIdx.x);
        __syncthreads();
        const QdqTensor& T = a.q.t[s];
        const char* xb = static_cast<const char*>(T.x);
        char* ob = static_cast<char*>(T.out);
        const bool next = s + 1 < a.q.n;
        const char* ab = next ? static_cast<const char*>(a.q.t[s + 1].x) : nullptr;
        const int64_t aseg = next ? a.q.t[s + 1].nblk : 0;
        const int64_t nmax = T.nblk > aseg ? T.nblk : aseg;
        Raw<IT> buf[2];
        load_if<IT, kQdqHint>(buf[0], xb + b0 * kBytes, b0 < T.nblk);
        float m = 0.0f;
        for (int64_t b = b0; b < nmax + lane; b += 2 * step) {
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int64_t bl = b + (k + 1) * step;
                load_if<IT, kQdqHint>(buf[(k + 1) % 2], xb + bl * kBytes, bl < T.nblk);
                const int64_t bc = b + k * step;
                Raw<IT> ra;
                zero_seg<IT>(ra);
                if (bc < aseg) load_seg<IT, kAmaxHint>(ra, ab + bc * kBytes);
                if (bc < T.nblk) {
                    uint64_t xp[8];
                    widen<IT>(buf[k], xp);
                    uint32_t code[2], scale, out[8];
                    encode_block<EM, OT>(xp, S, tbl, nz, code, scale, out);
                    st256(ob + bc * kBytes, out);
                }
                uint64_t xq[8];
                widen<IT>(ra, xq);
                m = fmaxf(m, seg_amax(xq));
            }
        }
        if (next) fused_arrive(m, &a.ws.acc[s + 1], &a.ws.cnt[s + 1], s_red, warp, lane);
    }
}


// ------------------------------------------------------------------------
// 16x16 quantize.  Unit = (band of 16 rows, quad of four 16x16 tiles); lane l
// holds rows (l >> 2) and (l >> 2) + 8 of tile 4 * quad + (l & 3), so each
// warp load reads eight whole 4-tile row spans.  With a per-tensor scale the
// warps walk the units grid-stride; otherwise each CTA takes a contiguous
// range of units and its warps interleave inside it (neighbouring warps read
// neighbouring spans; the band, and with it a per-row or per-group scale,
// changes rarely for any one warp).  The next unit is loaded one step ahead.
// ------------------------------------------------------------------------
template <In IT, Err EM, Src SRC>
__global__ void __launch_bounds__(kThreads, tile_min_ctas<IT>()) k_quant16x16(const EncArgs a) {
    chain_wait();
    chain_release();
    extern __shared__ int32_t s_ends[];
    __shared__ float2 s_tbl[kWarps][128];
    if constexpr (SRC == Src::GROUP) load_group_ends(s_ends, a.offs, a.G, a.rows);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // per tensor: one table for the CTA; otherwise one per warp
    float2* tbl = (SRC == Src::TENSOR) ? s_tbl[0] : s_tbl[warp];
    const uint64_t nz = pk(a.neg_zero, a.neg_zero);
    if constexpr (SRC == Src::TENSOR) {  // filled before any warp can leave
        fill_table_cta(tbl, global_scale(a.amax[0], a.six_bound), threadIdx.x);
        __syncthreads();
    }
    // One table per tensor: a grid-stride walk (the whole grid sweeps one
    // window at a time).  Per-row / per-group scales: each CTA walks its own
    // contiguous range, warps interleaved, so a warp's scale changes rarely.
    constexpr bool kGrid = (SRC == Src::TENSOR);
    const int64_t ustep = kGrid ? (int64_t)gridDim.x * kWarps : kWarps;
    const int64_t c1 = kGrid ? a.units : split_at(a.units, gridDim.x, blockIdx.x + 1);
    const int64_t u0 = kGrid ? (int64_t)blockIdx.x * kWarps + warp
                             : split_at(a.units, gridDim.x, blockIdx.x) + warp;
    if (u0 >= c1) return;
    const int64_t step_rows = ustep / a.cpr, step_chunks = ustep % a.cpr;
    constexpr int64_t kElt = (IT == In::F32) ? 4 : 2;
    const char* xb = static_cast<const char*>(a.x);
    const int t = lane & 3, r = lane >> 2;
    const int64_t cols = a.nb * 16;
    int64_t last_end = a.rows;
    if constexpr (SRC == Src::GROUP) last_end = s_ends[a.G - 1];
    RowChunk cc{u0 / a.cpr, u0 % a.cpr};  // row = band, chunk = tile quad
    auto load_unit = [&](Raw<IT>& lo, Raw<IT>& hi, const RowChunk& p, bool in_range) {
        const int64_t J = p.chunk * 4 + t;
        zero_seg<IT>(lo);
        zero_seg<IT>(hi);
        if (in_range && J < a.nb && p.row * 16 < last_end) {
            const char* q = xb + ((p.row * 16 + r) * cols + J * 16) * kElt;
            load_seg<IT, kEncHint>(lo, q);
            load_seg<IT, kEncHint>(hi, q + 8 * cols * kElt);
        }
    };
    Raw<IT> cur0, cur1;
    load_unit(cur0, cur1, cc, true);
    int g = 0;
    if constexpr (SRC == Src::GROUP)
        while (g < a.G && cc.row * 16 >= s_ends[g]) ++g;
    int64_t key = -1;
    float S = 1.0f;
    if constexpr (SRC == Src::TENSOR) S = global_scale(a.amax[0], a.six_bound);
    int64_t u = u0;
    const bool quads_whole = (a.nb & 3) == 0;  // every band is whole tile quads
    for (; u < c1; u += ustep) {
        bool tail = false;
        int64_t seg_end = INT64_MAX;  // first band past the current scale's segment
        if constexpr (SRC != Src::TENSOR) {
            int64_t k;
            if constexpr (SRC == Src::ROW) {
                k = cc.row * 16;  // a tile uses the amax of its first row
                seg_end = cc.row + 1;
            } else {
                while (g < a.G && cc.row * 16 >= s_ends[g]) ++g;
                k = g;
                tail = (g >= a.G);
                if (!tail) seg_end = ((int64_t)s_ends[g] + 15) / 16;
            }
            if (k != key) {
                key = k;
                if (!tail) {
                    S = global_scale(a.amax[k], a.six_bound);
                    build_table(tbl, S, lane);
                }
            }
        }
        if (quads_whole && !tail) {
            // Steady state: while the next unit lies whole under the same
            // scale, loads and stores go without bounds checks or zero fill.
            while (u + ustep < c1) {
                RowChunk nc = cc;
                nc.row += step_rows;
                nc.chunk += step_chunks;
                if (nc.chunk >= a.cpr) {
                    nc.chunk -= a.cpr;
                    ++nc.row;
                }
                if (nc.row >= seg_end) break;
                const char* q = xb + ((nc.row * 16 + r) * cols + (nc.chunk * 4 + t) * 16) * kElt;
                Raw<IT> nxt0, nxt1;
                load_seg<IT, kEncHint>(nxt0, q);
                load_seg<IT, kEncHint>(nxt1, q + 8 * cols * kElt);
                const int64_t J = cc.chunk * 4 + t;
                uint8_t* c0 = a.codes + (cc.row * 16 + r) * (cols / 2) + J * 8;
                uint64_t x0[8], x1[8];
                widen<IT>(cur0, x0);
                widen<IT>(cur1, x1);
                uint32_t k0[2], k1[2], scale;
                encode_tile_rows<EM, SRC != Src::TENSOR>(x0, x1, S, tbl, nz, t, k0, k1, scale);
                st64(c0, k0[0], k0[1]);
                st64(c0 + 8 * (cols / 2), k1[0], k1[1]);
                if (r == 0) st8(a.scales + cc.row * a.nb + J, scale);
                cur0 = nxt0;
                cur1 = nxt1;
                cc = nc;
                u += ustep;
            }
        }
        RowChunk nc = cc;  // this warp's next unit, ustep units on
        nc.row += step_rows;
        nc.chunk += step_chunks;
        if (nc.chunk >= a.cpr) {
            nc.chunk -= a.cpr;
            ++nc.row;
        }
        Raw<IT> nxt0, nxt1;
        load_unit(nxt0, nxt1, nc, u + ustep < c1);
        const int64_t band = cc.row;
        const int64_t J = cc.chunk * 4 + t;
        uint8_t* c0 = a.codes + (band * 16 + r) * (cols / 2) + J * 8;
        uint8_t* c8 = c0 + 8 * (cols / 2);
        if (!tail) {
            uint64_t x0[8], x1[8];
            widen<IT>(cur0, x0);  // zeros past the last tile of the band
            widen<IT>(cur1, x1);
            uint32_t k0[2], k1[2], scale;
            encode_tile_rows<EM, SRC != Src::TENSOR>(x0, x1, S, tbl, nz, t, k0, k1, scale);  // all lanes take part
            if (J < a.nb) {
                st64(c0, k0[0], k0[1]);
                st64(c8, k1[0], k1[1]);
                if (r == 0) st8(a.scales + band * a.nb + J, scale);
            }
        } else if (J < a.nb) {
            st64(c0, 0u, 0u);
            st64(c8, 0u, 0u);
            if (r == 0) st8(a.scales + band * a.nb + J, 0u);
        }
        cur0 = nxt0;
        cur1 = nxt1;
        cc = nc;
    }
}

// ------------------------------------------------------------------------
// List pipeline: one launch encodes tensor i (per-tensor scale, 1x16) and
// runs the amax pass of tensor i+1.  Every warp walks both tensors with the
// same grid stride: in each step it loads one unit of tensor i+1, encodes
// its unit of tensor i (whose load went out a step earlier) and then folds
// the tensor i+1 unit into its running max, so that load's latency hides
// behind the encode.  The encode is bound by instruction issue and leaves
// HBM bandwidth idle; the extra read and max cost about 4 % more
// instructions.  The kernel boundary orders amax(i+1) before encode(i+1),
// so no grid-wide synchronisation is needed.  The amax target must be +0 on
// entry (the host clears it before the launch).
// ------------------------------------------------------------------------
struct PipeArgs {
    EncArgs enc;           // tensor i (amax given)
    float* clear;          // optional: set to +0 by the launch (amax of tensor i+2)
    const void* ax;        // tensor i+1: input
    float* aamax;          //             amax output (cleared)
    int64_t aseg;          //             16-element segments
    int64_t aunits;        //             32-segment units
};

template <In IT, Err EM, bool TL = false>
__global__ void __launch_bounds__(kThreads, min_ctas<EM>()) k_quant1x16_pipe(const PipeArgs p) {
    chain_wait();
    chain_release();
    if (p.clear && blockIdx.x == 0 && threadIdx.x == 0) *p.clear = 0.0f;
    __shared__ float2 tbl[128];  // one common-scale table for the CTA
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int64_t kBytes = (IT == In::F32) ? 64 : 32;
    const EncArgs& a = p.enc;
    const uint64_t nz = pk(a.neg_zero, a.neg_zero);
    const int64_t nw = (int64_t)gridDim.x * kWarps;
    const int64_t u = (int64_t)blockIdx.x * kWarps + warp;
    const char* xb = static_cast<const char*>(a.x);
    const char* ab = static_cast<const char*>(p.ax);
    const int64_t step = nw * 32;
    const int64_t b0 = u * 32 + lane;  // this lane's block of tensor i, segment of tensor i+1
    const int64_t nmax = a.nblk > p.aseg ? a.nblk : p.aseg;
    Raw<IT> buf[2];
    load_if<IT, kEncHint>(buf[0], xb + b0 * kBytes, b0 < a.nblk);
    const float S = global_scale(a.amax[0], a.six_bound);
    fill_table_cta(tbl, S, threadIdx.x);
    __syncthreads();
    uint32_t dummy[8];
    BlockPos pos;  // TL: (row, column block) of block b + k * step, advanced per step
    int32_t srow = 0, scol = 0, nb32 = (int32_t)a.nb;
    if constexpr (TL) {
        pos.init(b0, a.nb);
        srow = (int32_t)(step / a.nb);
        scol = (int32_t)(step - (int64_t)srow * a.nb);
    }
    float m = 0.0f;
    for (int64_t b = b0; b < nmax + lane; b += 2 * step) {  // b - lane: first block of unit
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int64_t bl = b + (k + 1) * step;
            load_if<IT, kEncHint>(buf[(k + 1) % 2], xb + bl * kBytes, bl < a.nblk);
            const int64_t bc = b + k * step;
            Raw<IT> ra;
            zero_seg<IT>(ra);
            if (bc < p.aseg) load_seg<IT, kAmaxHint>(ra, ab + bc * kBytes);
            if (bc < a.nblk) {
                uint64_t xp[8];
                widen<IT>(buf[k], xp);
                uint32_t code[2], scale;
                encode_block<EM, Out::NONE, true>(xp, S, tbl, nz, code, scale, dummy);
                st64(a.codes + bc * 8, code[0], code[1]);
                st8(a.scales + scale_at<TL>(bc, pos.row, pos.col, a.sc_pc4), scale);
            }
            if constexpr (TL) pos.advance(srow, scol, nb32);
            uint64_t xq[8];
            widen<IT>(ra, xq);
            m = fmaxf(m, seg_amax(xq));
        }
    }
    m = warp_max_dev(m);
    if (lane == 0 && m > 0.0f)
        atomicMax(reinterpret_cast<unsigned int*>(p.aamax), __float_as_uint(m));
}

// ------------------------------------------------------------------------
// Dequantize: out = round_to(OT, e2m1(code) * (sigma / S)).
// Unit = (row, 32-block chunk).  B16: 16x16 scale layout.
// ------------------------------------------------------------------------
template <Out OT, bool B16, Src SRC>
__global__ void __launch_bounds__(kThreads) k_dequant(const DeqArgs a) {
    chain_wait();
    chain_release();
    __shared__ float2 s_tbl[kWarps][128];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float2* tbl = s_tbl[warp];
    const int64_t nw = (int64_t)gridDim.x * kWarps, gw = (int64_t)blockIdx.x * kWarps + warp;
    const int64_t cols = a.nb * 16;
    char* ob = static_cast<char*>(a.out);
    if constexpr (SRC == Src::TENSOR) {
        // one scale for the tensor: the blocks are walked grid-stride as one
        // flat sequence (codes and outputs are block-major; a 1x16 scale is
        // per block, a 16x16 scale per (row / 16, block)), with the next
        // block's code word and scale byte loaded a step ahead; one table
        // for the CTA
        tbl = s_tbl[0];
        fill_table_cta(tbl, global_scale(a.amax[0], a.six_bound), threadIdx.x);
        __syncthreads();
        const int64_t nblk = a.rows * a.nb, step = nw * 32;
        int64_t b = gw * 32 + lane;
        // 16x16: (row, column block) of b, advanced by step each iteration
        int64_t brow = B16 ? b / a.nb : 0, bcol = B16 ? b % a.nb : 0;
        const int64_t srow = B16 ? step / a.nb : 0, scol = B16 ? step % a.nb : 0;
        auto scale_at = [&](int64_t blk, int64_t r, int64_t j) -> uint32_t {
            return B16 ? a.scales[(r >> 4) * a.nb + j] : a.scales[blk];
        };
        uint2 cw = make_uint2(0u, 0u);
        uint32_t sb = 0;
        if (b < nblk) {
            cw = *reinterpret_cast<const uint2*>(a.codes + b * 8);
            sb = scale_at(b, brow, bcol);
        }
        for (; b - lane < nblk; b += step) {
            const int64_t bn = b + step;
            if constexpr (B16) {
                brow += srow;
                bcol += scol;
                if (bcol >= a.nb) {
                    bcol -= a.nb;
                    ++brow;
                }
            }
            uint2 cwn = make_uint2(0u, 0u);
            uint32_t sbn = 0;
            if (bn < nblk) {
                cwn = *reinterpret_cast<const uint2*>(a.codes + bn * 8);
                sbn = scale_at(bn, brow, bcol);
            }
            if (b < nblk) {
                const float d = tbl[sb & 0x7Fu].y;
                // sigma / S is odd in sigma; a zero scale of either sign decodes by +0
                const float dsig = ((sb & 0x80u) && d != 0.0f) ? -d : d;
                const uint64_t dd = pk(dsig, dsig);
                uint32_t outw[16];
#pragma unroll
                for (int p = 0; p < 8; ++p) {
                    const uint32_t byte = ((p < 4 ? cw.x : cw.y) >> (8 * (p & 3))) & 0xFFu;
                    const uint64_t v = mul2(f16x2_f32x2(e2m1x2_f16x2(byte)), dd);
                    if constexpr (OT == Out::F32) {
                        float lo, hi;
                        upk(v, lo, hi);
                        outw[2 * p] = __float_as_uint(lo);
                        outw[2 * p + 1] = __float_as_uint(hi);
                    } else {
                        outw[p] = out_pair<OT>(v);
                    }
                }
                if constexpr (OT == Out::F32) {
                    st256(ob + b * 64, outw);
                    st256(ob + b * 64 + 32, outw + 8);
                } else {
                    st256(ob + b * 32, outw);
                }
            }
            cw = cwn;
            sb = sbn;
        }
        return;
    }
    const int64_t u0 = split_at(a.units, nw, gw), u1 = split_at(a.units, nw, gw + 1);
    if (u0 >= u1) return;
    int64_t row = u0 / a.cpr, chunk = u0 % a.cpr;
    int64_t key = -1;
    for (int64_t u = u0; u < u1; ++u) {
        const int64_t k = (SRC == Src::ROW) ? (B16 ? row - (row & 15) : row) : 0;
        if (k != key) {
            key = k;
            build_table(tbl, global_scale(a.amax[k], a.six_bound), lane);
        }
        const int64_t j = chunk * 32 + lane;
        if (j < a.nb) {
            const uint2 cw = *reinterpret_cast<const uint2*>(a.codes + row * (cols / 2) + j * 8);
            const int64_t sidx = (B16 ? (row >> 4) : row) * a.nb + j;
            const uint32_t sb = a.scales[sidx];
            const float d = tbl[sb & 0x7Fu].y;
            // sigma / S is odd in sigma; a zero scale of either sign decodes by +0
            const float dsig = ((sb & 0x80u) && d != 0.0f) ? -d : d;
            const uint64_t dd = pk(dsig, dsig);
            uint32_t outw[16];
#pragma unroll
            for (int p = 0; p < 8; ++p) {
                const uint32_t byte = ((p < 4 ? cw.x : cw.y) >> (8 * (p & 3))) & 0xFFu;
                const uint64_t v = mul2(f16x2_f32x2(e2m1x2_f16x2(byte)), dd);
                if constexpr (OT == Out::F32) {
                    float lo, hi;
                    upk(v, lo, hi);
                    outw[2 * p] = __float_as_uint(lo);
                    outw[2 * p + 1] = __float_as_uint(hi);
                } else {
                    outw[p] = out_pair<OT>(v);
                }
            }
            if constexpr (OT == Out::F32) {
                st256(ob + (row * cols + j * 16) * 4, outw);
                st256(ob + (row * cols + j * 16) * 4 + 32, outw + 8);
            } else {
                st256(ob + (row * cols + j * 16) * 2, outw);
            }
        }
        if (++chunk == a.cpr) { chunk = 0; ++row; }
    }
}

// ------------------------------------------------------------------------
// Amax passes (NaN-dropping max|x|, initial +0).
// ------------------------------------------------------------------------
__device__ __forceinline__ float warp_max(float m) {
#pragma unroll
    for (int w = 16; w >= 1; w >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, w));
    return m;
}

// Whole tensor: amax[0] must be +0 on entry (the host clears it); each CTA
// folds its maximum in with an unsigned atomic max, which orders
// non-negative floats like their values.
template <In IT>
__global__ void __launch_bounds__(kThreads) k_amax_tensor(const AmaxArgs a) {
    chain_wait();
    chain_release();
    if (a.clear && blockIdx.x == 0 && threadIdx.x == 0) *a.clear = 0.0f;
    __shared__ float s_m[kWarps];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t nw = (int64_t)gridDim.x * kWarps;
    constexpr int64_t kBytes = (IT == In::F32) ? 64 : 32;
    const char* xb = static_cast<const char*>(a.x);
    const int64_t nseg = a.rows * a.nb;
    float m = 0.0f;
    // grid-stride over 32-segment units, two units in flight per lane
    for (int64_t u = (int64_t)blockIdx.x * kWarps + warp; u < a.units; u += 2 * nw) {
        const int64_t s0 = u * 32 + lane, s1 = (u + nw) * 32 + lane;
        Raw<IT> r0, r1;
        zero_seg<IT>(r0);
        zero_seg<IT>(r1);
        if (s0 < nseg) load_seg<IT, kAmaxHint>(r0, xb + s0 * kBytes);
        if (u + nw < a.units && s1 < nseg) load_seg<IT, kAmaxHint>(r1, xb + s1 * kBytes);
        uint64_t xp[8];
        widen<IT>(r0, xp);
        m = fmaxf(m, seg_amax(xp));
        widen<IT>(r1, xp);
        m = fmaxf(m, seg_amax(xp));
    }
    m = warp_max(m);
    if (lane == 0) s_m[warp] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        float cm = 0.0f;
        for (int w = 0; w < kWarps; ++w) cm = fmaxf(cm, s_m[w]);
        if (cm > 0.0f) atomicMax(reinterpret_cast<unsigned int*>(a.amax), __float_as_uint(cm));
    }
}

// Per row: one warp per row at a time; amax[r] written directly.
template <In IT>
__global__ void __launch_bounds__(kThreads) k_amax_rows(const AmaxArgs a) {
    chain_wait();
    chain_release();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t nw = (int64_t)gridDim.x * kWarps, gw = (int64_t)blockIdx.x * kWarps + warp;
    constexpr int64_t kBytes = (IT == In::F32) ? 64 : 32;
    const char* xb = static_cast<const char*>(a.x);
    for (int64_t r = gw; r < a.rows; r += nw) {
        float m = 0.0f;
        for (int64_t j = lane; j < a.nb; j += 32) {
            Raw<IT> seg;
            load_seg<IT>(seg, xb + (r * a.nb + j) * kBytes);
            uint64_t xp[8];
            widen<IT>(seg, xp);
            m = fmaxf(m, seg_amax(xp));
        }
        m = warp_max(m);
        if (lane == 0) a.amax[r] = m;
    }
}

// Per group: each warp walks a contiguous row range; a running maximum is
// folded into amax[g] (cleared by the host) whenever the group changes.
template <In IT>
__global__ void __launch_bounds__(kThreads) k_amax_groups(const AmaxArgs a) {
    chain_wait();
    chain_release();
    extern __shared__ int32_t s_ends[];
    load_group_ends(s_ends, a.offs, a.G, a.rows);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t nw = (int64_t)gridDim.x * kWarps, gw = (int64_t)blockIdx.x * kWarps + warp;
    const int64_t last_end = s_ends[a.G - 1];
    const int64_t r0 = split_at(last_end, nw, gw), r1 = split_at(last_end, nw, gw + 1);
    constexpr int64_t kBytes = (IT == In::F32) ? 64 : 32;
    const char* xb = static_cast<const char*>(a.x);
    int g = 0;
    while (g < a.G && r0 >= s_ends[g]) ++g;
    float m = 0.0f;
    for (int64_t r = r0; r < r1; ++r) {
        while (g < a.G && r >= s_ends[g]) {
            if (lane == 0 && m > 0.0f)
                atomicMax(reinterpret_cast<unsigned int*>(a.amax + g), __float_as_uint(m));
            m = 0.0f;
            ++g;
        }
        float rm = 0.0f;
        for (int64_t j = lane; j < a.nb; j += 32) {
            Raw<IT> seg;
            load_seg<IT>(seg, xb + (r * a.nb + j) * kBytes);
            uint64_t xp[8];
            widen<IT>(seg, xp);
            rm = fmaxf(rm, seg_amax(xp));
        }
        m = fmaxf(m, warp_max(rm));
    }
    if (lane == 0 && m > 0.0f && g < a.G)
        atomicMax(reinterpret_cast<unsigned int*>(a.amax + g), __float_as_uint(m));
}

}  // namespace fos

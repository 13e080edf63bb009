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
};

struct QdqTensor {
    const void* x;
    void* out;
    const float* amax;
    int64_t nblk;
    int64_t unit_begin;
};

constexpr int kQdqMaxList = 64;

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
    const int32_t* offs;
    int G;
    int64_t rows, nb, units;
};

template <In IT>
using RingOf = LaneRing<(IT == In::F32) ? 4 : 2>;

// Shared memory of the encode kernels: the per-warp input rings, then (GROUP)
// the clamped group ends.
template <In IT>
__host__ __device__ constexpr size_t ring_smem_bytes() {
    return (size_t)kWarps * RingOf<IT>::kBytes;
}

// Position of a (row, 32-block chunk) walk.
struct RowChunk {
    int64_t row, chunk;
    __device__ __forceinline__ void next(int64_t cpr) {
        if (++chunk == cpr) { chunk = 0; ++row; }
    }
};

// ------------------------------------------------------------------------
// 1x16 quantize (codes + scales).
// ------------------------------------------------------------------------
template <In IT, Err EM, Src SRC>
__global__ void __launch_bounds__(kThreads) k_quant1x16(const EncArgs a) {
    extern __shared__ __align__(16) unsigned char s_dyn[];
    __shared__ float2 s_tbl[kWarps][128];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int32_t* s_ends = reinterpret_cast<int32_t*>(s_dyn + ring_smem_bytes<IT>());
    if constexpr (SRC == Src::GROUP) load_group_ends(s_ends, a.offs, a.G, a.rows);
    float2* tbl = s_tbl[warp];
    RingOf<IT> ring(s_dyn + warp * RingOf<IT>::kBytes, lane);
    const uint64_t nz = pk(a.neg_zero, a.neg_zero);
    const int64_t nw = (int64_t)gridDim.x * kWarps, gw = (int64_t)blockIdx.x * kWarps + warp;
    const int64_t u0 = split_at(a.units, nw, gw), u1 = split_at(a.units, nw, gw + 1);
    if (u0 >= u1) return;
    constexpr int64_t kBytes = (IT == In::F32) ? 64 : 32;
    const char* xb = static_cast<const char*>(a.x);
    uint32_t dummy[8];

    if constexpr (SRC == Src::TENSOR) {
        // issue the first kDepth-1 units before anything else
#pragma unroll
        for (int s = 0; s < kDepth - 1; ++s) {
            const int64_t b = (u0 + s) * 32 + lane;
            const bool v = (u0 + s < u1) && b < a.nblk;
            ring.issue(s, xb + (v ? b : 0) * kBytes, v);
        }
        const float S = global_scale(a.amax[0], a.six_bound);
        build_table(tbl, S, lane);
        int stage = 0;
        for (int64_t u = u0; u < u1; ++u) {
            const int64_t ui = u + kDepth - 1, bi = ui * 32 + lane;
            const bool vi = ui < u1 && bi < a.nblk;
            ring.issue((stage + kDepth - 1) % kDepth, xb + (vi ? bi : 0) * kBytes, vi);
            cp_async_wait<kDepth - 1>();
            const int64_t b = u * 32 + lane;
            if (b < a.nblk) {
                Raw<IT> cur;
                ring.read(stage, cur.w);
                uint64_t xp[8];
                widen<IT>(cur, xp);
                uint32_t code[2], scale;
                encode_block<EM, Out::NONE>(xp, S, tbl, nz, code, scale, dummy);
                st64(a.codes + b * 8, code[0], code[1]);
                st8(a.scales + b, scale);
            }
            stage = (stage + 1) % kDepth;
        }
    } else {
        // (row, chunk) walk; the key is the row (ROW) or its group (GROUP).
        int64_t last_end = a.rows;
        if constexpr (SRC == Src::GROUP) last_end = s_ends[a.G - 1];
        RowChunk cc{u0 / a.cpr, u0 % a.cpr}, ic = cc;
#pragma unroll
        for (int s = 0; s < kDepth - 1; ++s) {
            const int64_t j = ic.chunk * 32 + lane;
            const bool v = (u0 + s < u1) && j < a.nb && ic.row < last_end;
            ring.issue(s, xb + (v ? ic.row * a.nb + j : 0) * kBytes, v);
            ic.next(a.cpr);
        }
        int g = 0;
        if constexpr (SRC == Src::GROUP)
            while (g < a.G && cc.row >= s_ends[g]) ++g;
        int64_t key = -1;
        float S = 1.0f;
        int stage = 0;
        for (int64_t u = u0; u < u1; ++u) {
            {
                const int64_t j = ic.chunk * 32 + lane;
                const bool v = (u + kDepth - 1 < u1) && j < a.nb && ic.row < last_end;
                ring.issue((stage + kDepth - 1) % kDepth, xb + (v ? ic.row * a.nb + j : 0) * kBytes,
                           v);
                ic.next(a.cpr);
            }
            // global scale of this unit
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
            cp_async_wait<kDepth - 1>();
            const int64_t j = cc.chunk * 32 + lane;
            const int64_t b = cc.row * a.nb + j;
            if (j < a.nb) {
                if (cc.row < last_end) {
                    Raw<IT> cur;
                    ring.read(stage, cur.w);
                    uint64_t xp[8];
                    widen<IT>(cur, xp);
                    uint32_t code[2], scale;
                    encode_block<EM, Out::NONE>(xp, S, tbl, nz, code, scale, dummy);
                    st64(a.codes + b * 8, code[0], code[1]);
                    st8(a.scales + b, scale);
                } else {  // zero-extended tail of a padded grouped tensor
                    st64(a.codes + b * 8, 0u, 0u);
                    st8(a.scales + b, 0u);
                }
            }
            cc.next(a.cpr);
            stage = (stage + 1) % kDepth;
        }
    }
    cp_async_wait<0>();
}

// ------------------------------------------------------------------------
// Fused quantize-dequantize over a list of tensors (per-tensor scale, 1x16),
// output dtype == input dtype (bf16 / fp16).  Codes and scales never leave
// registers.  Units are 32-block chunks of one tensor; empty tensors own no
// units.
// ------------------------------------------------------------------------
struct ListPos {
    int t;
    int64_t u;  // global unit index
};

template <In IT, Err EM>
__global__ void __launch_bounds__(kThreads) k_qdq1x16(const __grid_constant__ QdqArgs a) {
    static_assert(IT != In::F32, "fused QDQ is bf16 / fp16 only");
    constexpr Out OT = (IT == In::BF16) ? Out::BF16 : Out::F16;
    extern __shared__ __align__(16) unsigned char s_dyn[];
    __shared__ float2 s_tbl[kWarps][128];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float2* tbl = s_tbl[warp];
    RingOf<IT> ring(s_dyn + warp * RingOf<IT>::kBytes, lane);
    const uint64_t nz = pk(a.neg_zero, a.neg_zero);
    const int64_t nw = (int64_t)gridDim.x * kWarps, gw = (int64_t)blockIdx.x * kWarps + warp;
    const int64_t u0 = split_at(a.units, nw, gw), u1 = split_at(a.units, nw, gw + 1);
    if (u0 >= u1) return;
    // tensor of a unit: advance while the next tensor starts at or before it
    auto seek = [&](ListPos& p) {
        while (p.t < a.n && a.t[p.t + 1].unit_begin <= p.u) ++p.t;
    };
    ListPos cp{0, u0};
    seek(cp);
    ListPos ip = cp;
#pragma unroll
    for (int s = 0; s < kDepth - 1; ++s) {
        const QdqTensor& T = a.t[ip.t];
        const int64_t b = (ip.u - T.unit_begin) * 32 + lane;
        const bool v = ip.u < u1 && b < T.nblk;
        ring.issue(s, static_cast<const char*>(v ? T.x : a.t[cp.t].x) + (v ? b : 0) * 32, v);
        ++ip.u;
        seek(ip);
    }
    int ti = -1;
    float S = 1.0f;
    int stage = 0;
    for (int64_t u = u0; u < u1; ++u) {
        {
            const QdqTensor& T = a.t[ip.t];
            const int64_t b = (ip.u - T.unit_begin) * 32 + lane;
            const bool v = ip.u < u1 && b < T.nblk;
            ring.issue((stage + kDepth - 1) % kDepth,
                       static_cast<const char*>(v ? T.x : a.t[cp.t].x) + (v ? b : 0) * 32, v);
            ++ip.u;
            seek(ip);
        }
        if (cp.t != ti) {
            ti = cp.t;
            S = global_scale(*a.t[ti].amax, a.six_bound);
            build_table(tbl, S, lane);
        }
        cp_async_wait<kDepth - 1>();
        const QdqTensor& T = a.t[cp.t];
        const int64_t b = (cp.u - T.unit_begin) * 32 + lane;
        if (b < T.nblk) {
            Raw<IT> cur;
            ring.read(stage, cur.w);
            uint64_t xp[8];
            widen<IT>(cur, xp);
            uint32_t code[2], scale, out[8];
            encode_block<EM, OT>(xp, S, tbl, nz, code, scale, out);
            st256(static_cast<char*>(T.out) + b * 32, out);
        }
        ++cp.u;
        seek(cp);
        stage = (stage + 1) % kDepth;
    }
    cp_async_wait<0>();
}

// ------------------------------------------------------------------------
// 16x16 quantize.  Unit = (band of 16 rows, pair of 16x16 tiles); lane l
// holds row (l & 15) of tile (2 * pair + (l >> 4)).
// ------------------------------------------------------------------------
template <In IT, Err EM, Src SRC>
__global__ void __launch_bounds__(kThreads) k_quant16x16(const EncArgs a) {
    extern __shared__ __align__(16) unsigned char s_dyn[];
    __shared__ float2 s_tbl[kWarps][128];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int32_t* s_ends = reinterpret_cast<int32_t*>(s_dyn + ring_smem_bytes<IT>());
    if constexpr (SRC == Src::GROUP) load_group_ends(s_ends, a.offs, a.G, a.rows);
    float2* tbl = s_tbl[warp];
    RingOf<IT> ring(s_dyn + warp * RingOf<IT>::kBytes, lane);
    const uint64_t nz = pk(a.neg_zero, a.neg_zero);
    const int64_t nw = (int64_t)gridDim.x * kWarps, gw = (int64_t)blockIdx.x * kWarps + warp;
    const int64_t u0 = split_at(a.units, nw, gw), u1 = split_at(a.units, nw, gw + 1);
    if (u0 >= u1) return;
    constexpr int64_t kElt = (IT == In::F32) ? 4 : 2;
    const char* xb = static_cast<const char*>(a.x);
    const int half = lane >> 4, r16 = lane & 15;
    const int64_t cols = a.nb * 16;
    int64_t last_end = a.rows;
    if constexpr (SRC == Src::GROUP) last_end = s_ends[a.G - 1];
    RowChunk cc{u0 / a.cpr, u0 % a.cpr}, ic = cc;  // row = band, chunk = tile pair
    auto src_of = [&](const RowChunk& p, bool& v) {
        const int64_t J = p.chunk * 2 + half;
        v = J < a.nb && p.row * 16 < last_end;
        return xb + (v ? ((p.row * 16 + r16) * cols + J * 16) * kElt : 0);
    };
#pragma unroll
    for (int s = 0; s < kDepth - 1; ++s) {
        bool v;
        const char* src = src_of(ic, v);
        ring.issue(s, src, v && (u0 + s < u1));
        ic.next(a.cpr);
    }
    int g = 0;
    if constexpr (SRC == Src::GROUP)
        while (g < a.G && cc.row * 16 >= s_ends[g]) ++g;
    int64_t key = -1;
    float S = 1.0f;
    if constexpr (SRC == Src::TENSOR) {
        S = global_scale(a.amax[0], a.six_bound);
        build_table(tbl, S, lane);
    }
    int stage = 0;
    for (int64_t u = u0; u < u1; ++u) {
        {
            bool v;
            const char* src = src_of(ic, v);
            ring.issue((stage + kDepth - 1) % kDepth, src, v && (u + kDepth - 1 < u1));
            ic.next(a.cpr);
        }
        const int64_t band = cc.row;
        bool tail = false;
        if constexpr (SRC != Src::TENSOR) {
            int64_t k;
            if constexpr (SRC == Src::ROW) {
                k = band * 16;  // a tile uses the amax of its first row
            } else {
                while (g < a.G && band * 16 >= s_ends[g]) ++g;
                k = g;
                tail = (g >= a.G);
            }
            if (k != key) {
                key = k;
                if (!tail) {
                    S = global_scale(a.amax[k], a.six_bound);
                    build_table(tbl, S, lane);
                }
            }
        }
        cp_async_wait<kDepth - 1>();
        const int64_t J = cc.chunk * 2 + half;
        const int64_t row = band * 16 + r16;
        if (!tail) {
            Raw<IT> cur;
            ring.read(stage, cur.w);  // zeros for a missing second tile
            uint64_t xp[8];
            widen<IT>(cur, xp);
            uint32_t code[2], scale;
            encode_tile_row<EM>(xp, S, tbl, nz, code, scale);  // all lanes take part
            if (J < a.nb) {
                st64(a.codes + row * (cols / 2) + J * 8, code[0], code[1]);
                if (r16 == 0) st8(a.scales + band * a.nb + J, scale);
            }
        } else if (J < a.nb) {
            st64(a.codes + row * (cols / 2) + J * 8, 0u, 0u);
            if (r16 == 0) st8(a.scales + band * a.nb + J, 0u);
        }
        cc.next(a.cpr);
        stage = (stage + 1) % kDepth;
    }
    cp_async_wait<0>();
}

// ------------------------------------------------------------------------
// Dequantize: out = round_to(OT, e2m1(code) * (sigma / S)).
// Unit = (row, 32-block chunk).  B16: 16x16 scale layout.
// ------------------------------------------------------------------------
template <Out OT, bool B16, Src SRC>
__global__ void __launch_bounds__(kThreads) k_dequant(const DeqArgs a) {
    __shared__ float2 s_tbl[kWarps][128];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float2* tbl = s_tbl[warp];
    const int64_t nw = (int64_t)gridDim.x * kWarps, gw = (int64_t)blockIdx.x * kWarps + warp;
    const int64_t u0 = split_at(a.units, nw, gw), u1 = split_at(a.units, nw, gw + 1);
    if (u0 >= u1) return;
    int64_t row = u0 / a.cpr, chunk = u0 % a.cpr;
    int64_t key = -1;
    const int64_t cols = a.nb * 16;
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
            char* ob = static_cast<char*>(a.out);
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
    extern __shared__ __align__(16) unsigned char s_dyn[];
    __shared__ float s_m[kWarps];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    RingOf<IT> ring(s_dyn + warp * RingOf<IT>::kBytes, lane);
    const int64_t nw = (int64_t)gridDim.x * kWarps, gw = (int64_t)blockIdx.x * kWarps + warp;
    const int64_t u0 = split_at(a.units, nw, gw), u1 = split_at(a.units, nw, gw + 1);
    constexpr int64_t kBytes = (IT == In::F32) ? 64 : 32;
    const char* xb = static_cast<const char*>(a.x);
    const int64_t nseg = a.rows * a.nb;
    float m = 0.0f;
    if (u0 < u1) {
#pragma unroll
        for (int s = 0; s < kDepth - 1; ++s) {
            const int64_t b = (u0 + s) * 32 + lane;
            const bool v = (u0 + s < u1) && b < nseg;
            ring.issue(s, xb + (v ? b : 0) * kBytes, v);
        }
        int stage = 0;
        for (int64_t u = u0; u < u1; ++u) {
            const int64_t ui = u + kDepth - 1, bi = ui * 32 + lane;
            const bool vi = ui < u1 && bi < nseg;
            ring.issue((stage + kDepth - 1) % kDepth, xb + (vi ? bi : 0) * kBytes, vi);
            cp_async_wait<kDepth - 1>();
            Raw<IT> cur;
            ring.read(stage, cur.w);  // zeros past the end leave the max unchanged
            uint64_t xp[8];
            widen<IT>(cur, xp);
            m = fmaxf(m, seg_amax(xp));
            stage = (stage + 1) % kDepth;
        }
        cp_async_wait<0>();
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

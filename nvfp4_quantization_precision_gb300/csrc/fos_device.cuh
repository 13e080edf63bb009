// fos_device.cuh -- device building blocks of the four-over-six NVFP4
// quantizer kernels for GB300 (sm_103a).
//
// Every rounding-critical step is one explicit instruction so that no
// compiler lowering choice can change a result (torchao fast-path PR,
// description: correctly-rounded FP32 division, RN casts to E2M1 / E4M3 with
// exact decodes, a pinned width-16 reduction order):
//   * products / sums / differences: mul/add/sub .rn (scalar or packed f32x2,
//     never contracted into an FMA);
//   * division: correctly rounded (div.rn semantics);
//   * E2M1 / E4M3 encode: cvt.rn.satfinite pair conversions; decode through
//     the exact cvt to f16x2 and a widening cvt to f32;
//   * FP16 rounding of the candidate decode (FP16-error mode): cvt.rn.f16x2.
// Adjacent elements travel as packed f32 pairs (low word = even element) and
// share one mul.rn.f32x2 by the block's common scale (Megatron fused-QDQ PR,
// "Packed pair arithmetic").
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace fos {

enum class In : int { BF16 = 0, F16 = 1, F32 = 2 };
// STD: standard NVFP4 (map-to-6 only).  The others are four-over-six with the
// given candidate-error metric; *_H compares candidates decoded to FP16.
enum class Err : int { STD = 0, MAE = 1, MSE = 2, MAE_H = 3, MSE_H = 4 };
enum class Src : int { TENSOR = 0, ROW = 1, GROUP = 2 };

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr float kFltMax = 3.402823466e38f;

__host__ __device__ constexpr bool err_is_mse(Err e) { return e == Err::MSE || e == Err::MSE_H; }
__host__ __device__ constexpr bool err_is_f16(Err e) { return e == Err::MAE_H || e == Err::MSE_H; }
template <In IT> struct InTraits;
template <> struct InTraits<In::BF16> { static constexpr int kWords = 8; };   // 16 x 2 B
template <> struct InTraits<In::F16> { static constexpr int kWords = 8; };
template <> struct InTraits<In::F32> { static constexpr int kWords = 16; };  // 16 x 4 B

// ------------------------------------------------------------ scalar / pairs
__device__ __forceinline__ float fmul(float a, float b) { return __fmul_rn(a, b); }
__device__ __forceinline__ float fadd(float a, float b) { return __fadd_rn(a, b); }
__device__ __forceinline__ float fdiv(float a, float b) { return __fdiv_rn(a, b); }

__device__ __forceinline__ uint64_t pk(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void upk(uint64_t p, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(p));
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t sub2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t abs2(uint64_t a) { return a & 0x7FFFFFFF7FFFFFFFull; }
// rn(a * b) per lane, written as fma(a, b, c) with c = (-0, -0) supplied at run
// time.  Adding -0 is exact and keeps the sign of a zero product, so the
// result is the correctly rounded product; because it is already a fused
// operation, the code generator cannot contract it with a following add or
// subtract into a single-rounding fma.  A plain mul.rn.f32x2 feeding a
// sub.rn.f32x2 was observed to be contracted, which changes e = x - v*d.
__device__ __forceinline__ uint64_t mul2_nc(uint64_t a, uint64_t b, uint64_t neg_zero) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(neg_zero));
    return r;
}

// ------------------------------------------------------------ conversions
// E2M1 pair encode (RN, satfinite): byte with the low element in the low nibble.
__device__ __forceinline__ uint32_t e2m1x2(uint64_t y) {
    uint32_t r;
    asm("{\n\t.reg .b8 q;\n\t.reg .f32 lo, hi;\n\tmov.b64 {lo, hi}, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 q, hi, lo;\n\tcvt.u32.u8 %0, q;\n\t}"
        : "=r"(r) : "l"(y));
    return r;
}
// Exact decode of an E2M1 pair byte to f16x2 (low half = low nibble).
__device__ __forceinline__ uint32_t e2m1x2_f16x2(uint32_t byte) {
    uint32_t r;
    asm("{\n\t.reg .b8 q;\n\tcvt.u8.u32 q, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, q;\n\t}"
        : "=r"(r) : "r"(byte));
    return r;
}
__device__ __forceinline__ uint64_t f16x2_f32x2(uint32_t h) {
    float lo, hi;
    asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\tcvt.f32.f16 %0, a;\n\t"
        "cvt.f32.f16 %1, b;\n\t}"
        : "=f"(lo), "=f"(hi) : "r"(h));
    return pk(lo, hi);
}
__device__ __forceinline__ uint32_t f32x2_f16x2(uint64_t p) {
    float lo, hi;
    upk(p, lo, hi);
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
__device__ __forceinline__ uint32_t f32x2_bf16x2(uint64_t p) {
    float lo, hi;
    upk(p, lo, hi);
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
// E4M3 pair encode (RN, satfinite): low byte = lo.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
    unsigned short r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}
// Exact decode of one E4M3 code (low byte of `code`).
__device__ __forceinline__ float e4m3_f32(uint32_t code) {
    uint32_t h;
    asm("{\n\t.reg .b16 c;\n\tcvt.u16.u32 c, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, c;\n\t}"
        : "=r"(h) : "r"(code & 0xFFu));
    float f;
    asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %1;\n\tcvt.f32.f16 %0, a;\n\t}" : "=f"(f) : "r"(h));
    return f;
}

// ------------------------------------------------------------ memory
__device__ __forceinline__ void ld256(const void* p, uint32_t* w) {
    asm volatile("ld.global.nc.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]),
                   "=r"(w[6]), "=r"(w[7])
                 : "l"(p));
}
__device__ __forceinline__ void st256(void* p, const uint32_t* w) {
    asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(w[0]),
                 "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
}
__device__ __forceinline__ void st64(void* p, uint32_t a, uint32_t b) {
    asm volatile("st.global.v2.b32 [%0], {%1,%2};" ::"l"(p), "r"(a), "r"(b) : "memory");
}
__device__ __forceinline__ void st8(void* p, uint32_t a) {
    asm volatile("st.global.u8 [%0], %1;" ::"l"(p), "r"(a) : "memory");
}

// ------------------------------------------------------------ per-lane ring
// Input staging through shared memory with cp.async: every lane copies its
// own 16-element segment (32 B, or 64 B for fp32) into a ring of kDepth
// stages and later reads back only what it copied itself, so no cross-lane
// synchronisation is needed; cp.async.wait_group is a hardware wait on the
// lane's own copies.  Keeping kDepth - 1 segments in flight per lane holds
// enough bytes in flight per SM to cover HBM latency without spending
// registers on prefetch buffers.  Within a stage the two (or four) 16-byte
// quarters of the lanes are laid out quarter-major so that each 128-bit
// shared load of a warp is conflict-free.
constexpr int kDepth = 4;

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
    // src-size 0 writes 16 zero bytes and reads nothing from global memory
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                 "r"(valid ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void lds128(uint32_t addr, uint32_t* w) {
    asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                 : "r"(addr));
}

template <int kQuarters>  // 16-byte pieces per lane segment: 2 (16-bit input) or 4 (fp32)
struct LaneRing {
    static constexpr int kStageBytes = kQuarters * 32 * 16;  // per warp
    static constexpr int kBytes = kStageBytes * kDepth;
    uint32_t base;  // shared address of this warp's ring
    int lane;
    __device__ __forceinline__ LaneRing(void* smem_warp, int l)
        : base((uint32_t)__cvta_generic_to_shared(smem_warp)), lane(l) {}
    __device__ __forceinline__ uint32_t at(int stage, int q) const {
        return base + stage * kStageBytes + q * 512 + lane * 16;
    }
    // Copies the lane's segment into `stage` -- or zeros when !valid, in which
    // case nothing is read and `src` only has to be a mapped address -- and
    // closes the commit group.
    __device__ __forceinline__ void issue(int stage, const void* src, bool valid) {
        const char* p = static_cast<const char*>(src);
#pragma unroll
        for (int q = 0; q < kQuarters; ++q) cp_async16(at(stage, q), p + (valid ? 16 * q : 0), valid);
        cp_async_commit();
    }
    __device__ __forceinline__ void read(int stage, uint32_t* w) const {
#pragma unroll
        for (int q = 0; q < kQuarters; ++q) lds128(at(stage, q), w + 4 * q);
    }
};

// Raw storage of one 16-element row segment.
template <In IT>
struct Raw {
    uint32_t w[InTraits<IT>::kWords];
};

template <In IT>
__device__ __forceinline__ void load_seg(Raw<IT>& r, const void* p) {
    ld256(p, r.w);
    if constexpr (IT == In::F32) ld256(static_cast<const char*>(p) + 32, r.w + 8);
}

template <In IT>
__device__ __forceinline__ void zero_seg(Raw<IT>& r) {
#pragma unroll
    for (int i = 0; i < InTraits<IT>::kWords; ++i) r.w[i] = 0u;
}

// Widen to 8 packed f32 pairs (exact).
template <In IT>
__device__ __forceinline__ void widen(const Raw<IT>& r, uint64_t (&xp)[8]) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        if constexpr (IT == In::BF16) {
            xp[j] = pk(__uint_as_float(r.w[j] << 16), __uint_as_float(r.w[j] & 0xFFFF0000u));
        } else if constexpr (IT == In::F16) {
            xp[j] = f16x2_f32x2(r.w[j]);
        } else {
            xp[j] = pk(__uint_as_float(r.w[2 * j]), __uint_as_float(r.w[2 * j + 1]));
        }
    }
}

// NaN-dropping max|x| over the 16 elements, initial +0 (max.f32 returns the
// non-NaN operand; the final max with +0 maps an all-NaN segment to 0).
__device__ __forceinline__ float seg_amax(const uint64_t (&xp)[8]) {
    float m = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        float a, b;
        upk(xp[j], a, b);
        m = fmaxf(m, fmaxf(fabsf(a), fabsf(b)));
    }
    return m;
}

// FP32 global encode scale from a global amax: S = (6 * bound) / A,
// correctly rounded; degenerate A -> 1; overflow -> FLT_MAX.
__device__ __forceinline__ float global_scale(float A, float six_bound) {
    if (!(A > 0.0f) || isinf(A)) return 1.0f;
    const float S = fdiv(six_bound, A);
    return isinf(S) ? kFltMax : S;
}

// Per-warp table of the common scales of every E4M3 block-scale code:
// tbl[c] = {r = S / sigma_c, d = sigma_c / S}, both 0 when sigma_c = 0.
// Codes 0x00..0x7E are the only ones a non-negative block scale produces.
__device__ __forceinline__ void build_table(float2* tbl, float S, int lane) {
    __syncwarp();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int c = lane + 32 * i;
        const float sig = e4m3_f32((uint32_t)c);
        float r = 0.0f, d = 0.0f;
        if (sig != 0.0f) {
            r = fdiv(S, sig);
            d = fdiv(sig, S);
        }
        tbl[c] = make_float2(r, d);
    }
    __syncwarp();
}

__device__ __forceinline__ uint32_t pack4(uint32_t b0, uint32_t b1, uint32_t b2, uint32_t b3) {
    return __byte_perm(__byte_perm(b0, b1, 0x0040), __byte_perm(b2, b3, 0x0040), 0x5410);
}

// Output element types of the decode paths.
enum class Out : int { NONE = 0, BF16 = 1, F16 = 2, F32 = 3 };

template <Out OT>
__device__ __forceinline__ uint32_t out_pair(uint64_t v) {
    if constexpr (OT == Out::BF16) return f32x2_bf16x2(v);
    else return f32x2_f16x2(v);
}

// One candidate of one 16-element row segment under common scales (r, d).
// Encodes y = x * r to E2M1, decodes exactly, and returns the segment's
// error reduced by the pinned tree (for w = 8,4,2,1: t[i] += t[i+w], i < w);
// element pairs (2j, 2j+1) sit in one packed register, so the first three
// tree levels are packed adds of pairs (j, j+4), (j, j+2), (0, 1).
// With OT != NONE it also returns the decode v * d rounded to the output type.
template <Err EM, Out OT>
__device__ __forceinline__ float candidate(const uint64_t (&xp)[8], float r, float d,
                                           uint64_t nz, uint32_t (&code)[2],
                                           uint32_t (&out)[8]) {
    const uint64_t rr = pk(r, r), dd = pk(d, d);
    uint32_t q[8];
    uint64_t term[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        q[j] = e2m1x2(mul2(xp[j], rr));
        if constexpr (EM != Err::STD) {
            uint64_t deq = mul2_nc(f16x2_f32x2(e2m1x2_f16x2(q[j])), dd, nz);
            if constexpr (OT != Out::NONE) out[j] = out_pair<OT>(deq);
            if constexpr (err_is_f16(EM)) {
                const uint32_t h = (OT == Out::F16) ? out[j] : f32x2_f16x2(deq);
                deq = f16x2_f32x2(h);
            }
            const uint64_t e = sub2(xp[j], deq);
            term[j] = err_is_mse(EM) ? mul2_nc(e, e, nz) : abs2(e);
        } else {
            if constexpr (OT != Out::NONE)
                out[j] = out_pair<OT>(mul2(f16x2_f32x2(e2m1x2_f16x2(q[j])), dd));
        }
    }
    code[0] = pack4(q[0], q[1], q[2], q[3]);
    code[1] = pack4(q[4], q[5], q[6], q[7]);
    if constexpr (EM == Err::STD) {
        return 0.0f;
    } else {
        const uint64_t t0 = add2(term[0], term[4]), t1 = add2(term[1], term[5]);
        const uint64_t t2 = add2(term[2], term[6]), t3 = add2(term[3], term[7]);
        const uint64_t u0 = add2(t0, t2), u1 = add2(t1, t3);
        float a, b;
        upk(add2(u0, u1), a, b);
        return fadd(a, b);
    }
}

// Block-scale codes of the two candidates for a block (tile) amax:
// s_k = (amax * S) / k, E4M3 RN satfinite.  Low byte: map-to-6, high byte:
// map-to-4 (t / 4 is the exact product t * 0.25).
__device__ __forceinline__ uint32_t scale_codes(float amax, float S) {
    const float t = fmul(amax, S);
    return e4m3x2(fdiv(t, 6.0f), fmul(t, 0.25f));
}

// Full 1x16 block: returns codes (2 words), the E4M3 scale byte, and with
// OT != NONE the 8 output words of the selected candidate's decode.
template <Err EM, Out OT>
__device__ __forceinline__ void encode_block(const uint64_t (&xp)[8], float S,
                                             const float2* tbl, uint64_t nz,
                                             uint32_t (&code)[2], uint32_t& scale,
                                             uint32_t (&out)[8]) {
    // Block scales are non-negative, so their codes are below 0x80; the mask
    // only keeps the table index in range by construction.
    const uint32_t sc = scale_codes(seg_amax(xp), S);
    const uint32_t c6 = sc & 0xFFu;
    const float2 rd6 = tbl[c6 & 0x7Fu];
    if constexpr (EM == Err::STD) {
        candidate<EM, OT>(xp, rd6.x, rd6.y, nz, code, out);
        scale = c6;
    } else {
        const uint32_t c4 = sc >> 8;
        const float2 rd4 = tbl[c4 & 0x7Fu];
        uint32_t code6[2], code4[2], out6[8], out4[8];
        const float e6 = candidate<EM, OT>(xp, rd6.x, rd6.y, nz, code6, out6);
        const float e4 = candidate<EM, OT>(xp, rd4.x, rd4.y, nz, code4, out4);
        const bool sel4 = e4 < e6;  // map-to-4 only when strictly better
        code[0] = sel4 ? code4[0] : code6[0];
        code[1] = sel4 ? code4[1] : code6[1];
        scale = sel4 ? c4 : c6;
        if constexpr (OT != Out::NONE) {
#pragma unroll
            for (int j = 0; j < 8; ++j) out[j] = sel4 ? out4[j] : out6[j];
        }
    }
}

// 16x16 tile: each of 16 lanes (a half-warp) holds one 16-element row of the
// tile.  The tile amax is a NaN-dropping max across the half-warp; each
// lane's row error is its width-16 tree, and the tile error runs the same
// tree over the 16 row partials (lane i adds lane i+w for w = 8,4,2,1).
__device__ __forceinline__ float half_max(float m) {
#pragma unroll
    for (int w = 8; w >= 1; w >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, w));
    return m;
}
__device__ __forceinline__ float half_tree(float p) {
#pragma unroll
    for (int w = 8; w >= 1; w >>= 1) p = fadd(p, __shfl_down_sync(0xFFFFFFFFu, p, w, 16));
    return __shfl_sync(0xFFFFFFFFu, p, 0, 16);
}

template <Err EM>
__device__ __forceinline__ void encode_tile_row(const uint64_t (&xp)[8], float S,
                                                const float2* tbl, uint64_t nz,
                                                uint32_t (&code)[2], uint32_t& scale) {
    const uint32_t sc = scale_codes(half_max(seg_amax(xp)), S);
    const uint32_t c6 = sc & 0xFFu;
    const float2 rd6 = tbl[c6 & 0x7Fu];
    uint32_t dummy[8];
    if constexpr (EM == Err::STD) {
        candidate<EM, Out::NONE>(xp, rd6.x, rd6.y, nz, code, dummy);
        scale = c6;
    } else {
        const uint32_t c4 = sc >> 8;
        const float2 rd4 = tbl[c4 & 0x7Fu];
        uint32_t code6[2], code4[2];
        const float e6 =
            half_tree(candidate<EM, Out::NONE>(xp, rd6.x, rd6.y, nz, code6, dummy));
        const float e4 =
            half_tree(candidate<EM, Out::NONE>(xp, rd4.x, rd4.y, nz, code4, dummy));
        const bool sel4 = e4 < e6;
        code[0] = sel4 ? code4[0] : code6[0];
        code[1] = sel4 ? code4[1] : code6[1];
        scale = sel4 ? c4 : c6;
    }
}

// Balanced contiguous split of `units` work units over `parts` workers.
__device__ __forceinline__ int64_t split_at(int64_t units, int64_t parts, int64_t i) {
    return (int64_t)(((unsigned __int128)units * (unsigned __int128)i) / (unsigned __int128)parts);
}

// Clamped cumulative group ends in shared memory:
// end_g = min(rows, max(0, offs[0], ..., offs[g])).  All threads of the CTA
// take part; ends must hold G entries.  Values fit int32 because the offs do.
__device__ __forceinline__ void load_group_ends(int32_t* ends, const int32_t* offs, int G,
                                                int64_t rows) {
    __shared__ int32_t s_part[kThreads];
    const int t = threadIdx.x;
    const int per = (G + kThreads - 1) / kThreads;
    const int lo = t * per, hi = min(G, lo + per);
    int32_t run = 0;
    for (int i = lo; i < hi; ++i) {
        run = max(run, offs[i]);
        ends[i] = run;
    }
    s_part[t] = run;
    __syncthreads();
    if (t == 0) {
        int32_t acc = 0;
        for (int i = 0; i < kThreads; ++i) {
            const int32_t v = s_part[i];
            s_part[i] = acc;  // exclusive prefix max
            acc = max(acc, v);
        }
    }
    __syncthreads();
    const int32_t before = s_part[t];
    for (int i = lo; i < hi; ++i) ends[i] = (int32_t)min(rows, (int64_t)max(before, ends[i]));
    __syncthreads();
}

}  // namespace fos

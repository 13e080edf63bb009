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
// given candidate-error metric; *_H compares candidates decoded to FP16; *_S
// sums a block's error terms in element order instead of the pinned tree.
enum class Err : int {
    STD = 0, MAE = 1, MSE = 2, MAE_H = 3, MSE_H = 4, MAE_S = 5, MSE_S = 6, MAE_HS = 7, MSE_HS = 8
};
enum class Src : int { TENSOR = 0, ROW = 1, GROUP = 2 };

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr float kFltMax = 3.402823466e38f;

__host__ __device__ constexpr bool err_is_mse(Err e) {
    return e == Err::MSE || e == Err::MSE_H || e == Err::MSE_S || e == Err::MSE_HS;
}
__host__ __device__ constexpr bool err_is_f16(Err e) {
    return e == Err::MAE_H || e == Err::MSE_H || e == Err::MAE_HS || e == Err::MSE_HS;
}
__host__ __device__ constexpr bool err_is_seq(Err e) {
    return e == Err::MAE_S || e == Err::MSE_S || e == Err::MAE_HS || e == Err::MSE_HS;
}
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
// Four pairs at once: encode y[0..3] to E2M1, return the four code bytes
// packed into one word (byte k = pair k, low nibble = low element) and, with
// DEC, the exact decodes as f16x2 (h[k] low half = low element of pair k).
template <bool DEC>
__device__ __forceinline__ void e2m1x8(const uint64_t* y, uint32_t& word, uint32_t* h) {
    if constexpr (DEC) {
        asm("{\n\t.reg .b8 q0, q1, q2, q3;\n\t.reg .f32 a0, b0, a1, b1, a2, b2, a3, b3;\n\t"
            "mov.b64 {a0, b0}, %5;\n\tmov.b64 {a1, b1}, %6;\n\t"
            "mov.b64 {a2, b2}, %7;\n\tmov.b64 {a3, b3}, %8;\n\t"
            "cvt.rn.satfinite.e2m1x2.f32 q0, b0, a0;\n\tcvt.rn.satfinite.e2m1x2.f32 q1, b1, a1;\n\t"
            "cvt.rn.satfinite.e2m1x2.f32 q2, b2, a2;\n\tcvt.rn.satfinite.e2m1x2.f32 q3, b3, a3;\n\t"
            "cvt.rn.f16x2.e2m1x2 %1, q0;\n\tcvt.rn.f16x2.e2m1x2 %2, q1;\n\t"
            "cvt.rn.f16x2.e2m1x2 %3, q2;\n\tcvt.rn.f16x2.e2m1x2 %4, q3;\n\t"
            "mov.b32 %0, {q0, q1, q2, q3};\n\t}"
            : "=r"(word), "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
            : "l"(y[0]), "l"(y[1]), "l"(y[2]), "l"(y[3]));
    } else {
        asm("{\n\t.reg .b8 q0, q1, q2, q3;\n\t.reg .f32 a0, b0, a1, b1, a2, b2, a3, b3;\n\t"
            "mov.b64 {a0, b0}, %1;\n\tmov.b64 {a1, b1}, %2;\n\t"
            "mov.b64 {a2, b2}, %3;\n\tmov.b64 {a3, b3}, %4;\n\t"
            "cvt.rn.satfinite.e2m1x2.f32 q0, b0, a0;\n\tcvt.rn.satfinite.e2m1x2.f32 q1, b1, a1;\n\t"
            "cvt.rn.satfinite.e2m1x2.f32 q2, b2, a2;\n\tcvt.rn.satfinite.e2m1x2.f32 q3, b3, a3;\n\t"
            "mov.b32 %0, {q0, q1, q2, q3};\n\t}"
            : "=r"(word) : "l"(y[0]), "l"(y[1]), "l"(y[2]), "l"(y[3]));
    }
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

// ------------------------------------------------------------ launch chaining
// Programmatic dependent launch: kernels are launched so that the next kernel
// in the stream may be placed on the SMs while this one drains.  Every kernel
// waits for the previous grid (completion and memory visibility) before its
// first global read, then lets its own dependents launch.  On a launch
// without the attribute both instructions have no effect.
__device__ __forceinline__ void chain_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void chain_release() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------ memory
__device__ __forceinline__ void ld256(const void* p, uint32_t* w) {
    asm volatile("ld.global.nc.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]),
                   "=r"(w[6]), "=r"(w[7])
                 : "l"(p));
}
// L2 eviction priority of a load: NORMAL, FIRST (streamed, last use) or LAST
// (read again soon).
enum class L2 : int { NORMAL = 0, FIRST = 1, LAST = 2 };
template <L2 H>
__device__ __forceinline__ uint64_t l2_policy() {
    uint64_t pol;
    if constexpr (H == L2::FIRST)
        asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    else
        asm("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
template <L2 H>
__device__ __forceinline__ void ld256h(const void* p, uint32_t* w) {
    if constexpr (H == L2::NORMAL) {
        ld256(p, w);
    } else {
        asm volatile(
            "ld.global.nc.L1::no_allocate.L2::cache_hint.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8], %9;"
            : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]), "=r"(w[6]),
              "=r"(w[7])
            : "l"(p), "l"(l2_policy<H>()));
    }
}
__device__ __forceinline__ void st256(void* p, const uint32_t* w) {
    asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(w[0]),
                 "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
}
__device__ __forceinline__ void st128(void* p, const uint32_t* w) {
    asm volatile("st.global.v4.b32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(w[0]), "r"(w[1]),
                 "r"(w[2]), "r"(w[3]) : "memory");
}
__device__ __forceinline__ void st32(void* p, uint32_t a) {
    asm volatile("st.global.b32 [%0], %1;" ::"l"(p), "r"(a) : "memory");
}
__device__ __forceinline__ void st16(void* p, uint32_t a) {
    asm volatile("st.global.b16 [%0], %1;" ::"l"(p), "h"((unsigned short)a) : "memory");
}
__device__ __forceinline__ void st64(void* p, uint32_t a, uint32_t b) {
    asm volatile("st.global.v2.b32 [%0], {%1,%2};" ::"l"(p), "r"(a), "r"(b) : "memory");
}
__device__ __forceinline__ void st8(void* p, uint32_t a) {
    asm volatile("st.global.u8 [%0], %1;" ::"l"(p), "r"(a) : "memory");
}

// Raw storage of one 16-element row segment.
template <In IT>
struct Raw {
    uint32_t w[InTraits<IT>::kWords];
};

template <In IT, L2 H = L2::NORMAL>
__device__ __forceinline__ void load_seg(Raw<IT>& r, const void* p) {
    ld256h<H>(p, r.w);
    if constexpr (IT == In::F32) ld256h<H>(static_cast<const char*>(p) + 32, r.w + 8);
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
__device__ __forceinline__ float max3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}
__device__ __forceinline__ float seg_amax(const uint64_t (&xp)[8]) {
    float m = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        float a, b;
        upk(xp[j], a, b);
        m = max3(m, fabsf(a), fabsf(b));
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

// The common-scale table filled by a whole CTA of kThreads = 256 threads,
// one division each: thread t < 128 writes r of code t, thread 128 + t
// writes d of code t.  One table per CTA costs a CTA barrier but an eighth
// of the divisions of per-warp tables (which also cost instruction issue
// at the start of every launch).
__device__ __forceinline__ void fill_table_cta(float2* tbl, float S, int tid) {
    const int c = tid & 127;
    const float sig = e4m3_f32((uint32_t)c);
    float v = 0.0f;
    if (sig != 0.0f) v = (tid < 128) ? fdiv(S, sig) : fdiv(sig, S);
    reinterpret_cast<float*>(tbl)[2 * c + (tid >> 7)] = v;
}


// Output element types of the decode paths.
enum class Out : int { NONE = 0, BF16 = 1, F16 = 2, F32 = 3 };

template <Out OT>
__device__ __forceinline__ uint32_t out_pair(uint64_t v) {
    if constexpr (OT == Out::BF16) return f32x2_bf16x2(v);
    else return f32x2_f16x2(v);
}

// e = h - x for an f16 pair h (widened exactly) and an f32 pair x: the
// negated FP16-mode error, which has the same magnitude and square.
__device__ __forceinline__ uint64_t sub2_f16(uint32_t h, uint64_t x) {
    float xl, xh, el, eh;
    upk(x, xl, xh);
    asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\t"
        "sub.rn.f32.f16 %0, a, %3;\n\tsub.rn.f32.f16 %1, b, %4;\n\t}"
        : "=f"(el), "=f"(eh) : "r"(h), "f"(xl), "f"(xh));
    return pk(el, eh);
}

// One candidate of one 16-element row segment under common scales (r, d).
// Encodes y = x * r to E2M1, decodes exactly, and returns the
// segment's error reduced by the pinned tree (for w = 8,4,2,1: t[i] +=
// t[i+w], i < w).  Element pairs (2j, 2j+1) sit in one packed register, so
// tree levels are packed adds of pairs (j, j+4), (j, j+2), (0, 1); for MAE
// the first level is done on scalars so that |e| folds into the add.
// With OT != NONE it also returns the decode v * d rounded to the output type.
template <Err EM, Out OT>
__device__ __forceinline__ float candidate(const uint64_t (&xp)[8], float r, float d,
                                           uint64_t nz, uint32_t (&code)[2],
                                           uint32_t (&out)[8]) {
    const uint64_t rr = pk(r, r), dd = pk(d, d);
    constexpr bool kDec = (EM != Err::STD) || (OT != Out::NONE);
    uint64_t term[8];
#pragma unroll
    for (int g = 0; g < 2; ++g) {
        uint64_t y[4];
        uint32_t h[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) y[k] = mul2(xp[4 * g + k], rr);
        e2m1x8<kDec>(y, code[g], h);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int j = 4 * g + k;
            if constexpr (EM != Err::STD) {
                const uint64_t deq = mul2_nc(f16x2_f32x2(h[k]), dd, nz);
                if constexpr (OT != Out::NONE) out[j] = out_pair<OT>(deq);
                uint64_t e;
                if constexpr (err_is_f16(EM)) {
                    e = sub2_f16((OT == Out::F16) ? out[j] : f32x2_f16x2(deq), xp[j]);
                } else {
                    e = sub2(xp[j], deq);
                }
                term[j] = err_is_mse(EM) ? mul2_nc(e, e, nz) : e;
            } else if constexpr (OT != Out::NONE) {
                out[j] = out_pair<OT>(mul2(f16x2_f32x2(h[k]), dd));
            }
        }
    }
    if constexpr (EM == Err::STD) {
        return 0.0f;
    } else if constexpr (err_is_seq(EM)) {
        // element order: ((t0 + t1) + t2) + ... + t15
        float acc = 0.0f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            float lo, hi;
            upk(term[j], lo, hi);
            if constexpr (!err_is_mse(EM)) {
                lo = fabsf(lo);
                hi = fabsf(hi);
            }
            acc = (j == 0) ? lo : fadd(acc, lo);
            acc = fadd(acc, hi);
        }
        return acc;
    } else {
        uint64_t t0, t1, t2, t3;
        if constexpr (err_is_mse(EM)) {
            t0 = add2(term[0], term[4]);
            t1 = add2(term[1], term[5]);
            t2 = add2(term[2], term[6]);
            t3 = add2(term[3], term[7]);
        } else {
            float s[8];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float al, ah, bl, bh;
                upk(term[j], al, ah);
                upk(term[j + 4], bl, bh);
                s[2 * j] = fadd(fabsf(al), fabsf(bl));
                s[2 * j + 1] = fadd(fabsf(ah), fabsf(bh));
            }
            t0 = pk(s[0], s[1]);
            t1 = pk(s[2], s[3]);
            t2 = pk(s[4], s[5]);
            t3 = pk(s[6], s[7]);
        }
        const uint64_t u0 = add2(t0, t2), u1 = add2(t1, t3);
        float a, b;
        upk(add2(u0, u1), a, b);
        return fadd(a, b);
    }
}

// Correctly rounded t / 6 for t >= 0.  In the range where the quotient is a
// normal number the division by the constant uses Markstein's correction:
// with c = rn(1/6), q = rn(t * c) is within an ulp of t / 6, the remainder
// r = t - 6q is exact in one fma, and rn(q + r * c) is the correctly rounded
// quotient (P. Markstein, "IA-64 and Elementary Functions", 2000, division
// by a correctly rounded reciprocal).  Subnormal quotients, Inf and NaN take
// the full division.  Checked against IEEE division for all 2^32 inputs.
__device__ __forceinline__ float div6_rn(float t) {
    constexpr float kInv6 = 0x1.555556p-3f;  // rn(1/6), bits 0x3E2AAAAB
    if (t >= 0x1.8p-124f && t <= kFltMax) {  // 6 * 2^-126 .. FLT_MAX
        const float q = fmul(t, kInv6);
        const float r = __fmaf_rn(-q, 6.0f, t);
        return __fmaf_rn(r, kInv6, q);
    }
    return fdiv(t, 6.0f);
}

// t / 6 where only its E4M3 code is used (the map-to-6 block scale), for
// t >= 0 or +Inf, without a branch: the same Markstein sequence as div6_rn,
// which is correctly rounded wherever the quotient is a normal number.  Below
// that (t < 6 * 2^-126) the quotient can be off in its last bits, but any
// value under 2^-10 encodes to the E4M3 code 0, so the code is unchanged;
// +Inf is clamped to FLT_MAX, whose quotient also saturates to 448.  (t is
// never NaN: the block amax drops NaN and S is finite.)  Checked against
// the code of the correctly rounded quotient for every non-negative float.
__device__ __forceinline__ float div6_for_code(float t) {
    constexpr float kInv6 = 0x1.555556p-3f;  // rn(1/6)
    const float c = fminf(t, kFltMax);
    const float q = fmul(c, kInv6);
    const float r = __fmaf_rn(-q, 6.0f, c);
    return __fmaf_rn(r, kInv6, q);
}

// Block-scale codes of the two candidates for a block (tile) amax:
// s_k = (amax * S) / k, E4M3 RN satfinite.  Low byte: map-to-6, high byte:
// map-to-4 (t / 4 is the exact product t * 0.25).  Both forms of t / 6 give
// the same codes for every t (checked exhaustively); which one a kernel uses
// is a code-generation choice made per kernel by measurement: DIV_BRANCH
// takes div6_rn (a branch to the full division outside the normal range),
// otherwise the branch-free div6_for_code.
template <bool DIV_BRANCH = false>
__device__ __forceinline__ uint32_t scale_codes(float amax, float S) {
    const float t = fmul(amax, S);
    if constexpr (DIV_BRANCH) return e4m3x2(div6_rn(t), fmul(t, 0.25f));
    else return e4m3x2(div6_for_code(t), fmul(t, 0.25f));
}

// Full 1x16 block: returns codes (2 words), the E4M3 scale byte, and with
// OT != NONE the 8 output words of the selected candidate's decode.
template <Err EM, Out OT, bool DB = false>
__device__ __forceinline__ void encode_block_amax(const uint64_t (&xp)[8], float block_amax,
                                                  float S, const float2* tbl, uint64_t nz,
                                                  uint32_t (&code)[2], uint32_t& scale,
                                                  uint32_t (&out)[8]);

template <Err EM, Out OT, bool DB = false>
__device__ __forceinline__ void encode_block(const uint64_t (&xp)[8], float S,
                                             const float2* tbl, uint64_t nz,
                                             uint32_t (&code)[2], uint32_t& scale,
                                             uint32_t (&out)[8]) {
    encode_block_amax<EM, OT, DB>(xp, seg_amax(xp), S, tbl, nz, code, scale, out);
}

template <Err EM, Out OT, bool DB>
__device__ __forceinline__ void encode_block_amax(const uint64_t (&xp)[8], float block_amax,
                                                  float S, const float2* tbl, uint64_t nz,
                                                  uint32_t (&code)[2], uint32_t& scale,
                                                  uint32_t (&out)[8]) {
    // Block scales are non-negative, so their codes are below 0x80; the mask
    // only keeps the table index in range by construction.
    const uint32_t sc = scale_codes<DB>(block_amax, S);
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

// 16x16 tile over lanes: lane l holds rows r = l >> 2 and r + 8 of tile
// t = l & 3, so the 16 rows of a tile sit in lanes t, t + 4, ..., t + 28.
// The tile amax is a NaN-dropping max over those lanes.  The tile error is
// the pinned tree over the 16 row partials (for w = 8,4,2,1: t[i] +=
// t[i+w]); level w = 8 pairs the two rows a lane holds, levels 4, 2, 1 pair
// lanes 16, 8 and 4 apart, and lane t ends with the tile's sum.
__device__ __forceinline__ float quad_max(float m) {
    m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 4));
    m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 8));
    return fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 16));
}
__device__ __forceinline__ float quad_tree(float p_r, float p_r8, int t) {
    float q = fadd(p_r, p_r8);
    q = fadd(q, __shfl_down_sync(0xFFFFFFFFu, q, 16));
    q = fadd(q, __shfl_down_sync(0xFFFFFFFFu, q, 8));
    q = fadd(q, __shfl_down_sync(0xFFFFFFFFu, q, 4));
    return __shfl_sync(0xFFFFFFFFu, q, t);
}

// Both rows (r, r + 8) a lane holds of one 16x16 tile: codes of each row and
// the tile's E4M3 scale byte.  Every lane of the warp must take part.
template <Err EM, bool DB = false>
__device__ __forceinline__ void encode_tile_rows(const uint64_t (&x0)[8], const uint64_t (&x1)[8],
                                                 float S, const float2* tbl, uint64_t nz, int t,
                                                 uint32_t (&k0)[2], uint32_t (&k1)[2],
                                                 uint32_t& scale) {
    const uint32_t sc = scale_codes<DB>(quad_max(fmaxf(seg_amax(x0), seg_amax(x1))), S);
    const uint32_t c6 = sc & 0xFFu;
    const float2 rd6 = tbl[c6 & 0x7Fu];
    uint32_t dummy[8];
    if constexpr (EM == Err::STD) {
        candidate<EM, Out::NONE>(x0, rd6.x, rd6.y, nz, k0, dummy);
        candidate<EM, Out::NONE>(x1, rd6.x, rd6.y, nz, k1, dummy);
        scale = c6;
    } else {
        const uint32_t c4 = sc >> 8;
        const float2 rd4 = tbl[c4 & 0x7Fu];
        uint32_t a0[2], a1[2], b0[2], b1[2];
        const float p6 = candidate<EM, Out::NONE>(x0, rd6.x, rd6.y, nz, a0, dummy);
        const float p6h = candidate<EM, Out::NONE>(x1, rd6.x, rd6.y, nz, a1, dummy);
        const float e6 = quad_tree(p6, p6h, t);
        const float p4 = candidate<EM, Out::NONE>(x0, rd4.x, rd4.y, nz, b0, dummy);
        const float p4h = candidate<EM, Out::NONE>(x1, rd4.x, rd4.y, nz, b1, dummy);
        const float e4 = quad_tree(p4, p4h, t);
        const bool sel4 = e4 < e6;
        k0[0] = sel4 ? b0[0] : a0[0];
        k0[1] = sel4 ? b0[1] : a0[1];
        k1[0] = sel4 ? b1[0] : a1[0];
        k1[1] = sel4 ? b1[1] : a1[1];
        scale = sel4 ? c4 : c6;
    }
}

// Byte offset of the scale of block (row, j) (j = 16-column block of the
// row) in the tiled layout block-scaled FP4 GEMMs read: the scale matrix
// padded to 128-row x 4-block tiles of 512 bytes stored tile-row by
// tile-row (pc4 tiles per tile-row), block (32 i + r, k) of a tile at byte
// 16 r + 4 i + k.  Rows and blocks fit 31 bits and the tile index 32 bits
// (the host admits tiled scales for rows < 2^30 only), so all but the final
// scaling by 512 is 32-bit arithmetic.
__device__ __forceinline__ int64_t tiled_scale_off(int32_t row, int32_t j, int32_t pc4) {
    const uint32_t tile = (uint32_t)(row >> 7) * (uint32_t)pc4 + (uint32_t)(j >> 2);
    return ((int64_t)tile << 9) + (int64_t)(((row & 31) << 4) | (((row >> 5) & 3) << 2) | (j & 3));
}

// Position (row, column block) of a block walked with a fixed stride in
// blocks, kept up to date without a division per block (tiled scales; rows
// below 2^30, so a position a few strides past the end still fits).
struct BlockPos {
    int32_t row = 0, col = 0;
    __device__ __forceinline__ void init(int64_t b, int64_t nb) {
        const int64_t r = b / nb;
        row = (int32_t)r;
        col = (int32_t)(b - r * nb);
    }
    __device__ __forceinline__ void advance(int32_t srow, int32_t scol, int32_t nb) {
        col += scol;
        row += srow;
        if (col >= nb) {
            col -= nb;
            ++row;
        }
    }
};

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

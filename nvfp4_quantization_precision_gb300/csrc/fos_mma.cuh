// fos_mma.cuh -- the block-scaled NVFP4 product on the 5th-generation tensor
// cores of sm_103a (tcgen05): out = a . b^T from 1x16 E2M1 codes and E4M3
// block scales in the tiled layout, with the FP32 global decode scales applied
// in the epilogue (grouped PR, the dense-recipe commit's four_over_six_mm
// forward; per row of a for a row-scaled a, the MoE commit's epilogue).
//
// One CTA computes one BM x BN tile of out.  Six warps:
//   warp 0   (one thread)  TMA producer: per K stage of 256 elements, the a and
//            b code tiles (2D TMA, 128-byte swizzle) and the stage's four
//            512-byte scale atoms of each operand (1D bulk copies) into a
//            ring of kStages shared-memory stages, completion on mbarriers;
//   warp 1   allocates the tensor memory; one thread copies each stage's scale
//            atoms into tensor memory (tcgen05.cp 32x128b.warpx4) and issues
//            four tcgen05.mma kind::mxf4nvf4 block_scale scale_vec::4X
//            (M = BM, N = BN, K = 64 each) accumulating in tensor memory,
//            then frees the stage (tcgen05.commit to its mbarrier);
//   warps 2-5 epilogue: wait for the last MMA, read the FP32 accumulator from
//            tensor memory (tcgen05.ld, warp w reads lanes 32 (w % 4) ..),
//            multiply by g_a(m) and then g_b, store.
// Operands are K-major: a row of a (or b) holds K/2 code bytes, element 2j in
// the low nibble of byte j, which is the element order of the E2M1 operand.
// The scale atom of rows [128 t, 128 t + 128) and K elements [64 c, 64 c + 64)
// is the 512-byte tile (t, c) of the tiled layout: byte 16 j + 4 i + k holds
// the scale of row 32 i + j, 16-element block k.  Copied with the warpx4
// shape, tensor-memory lane 32 q + j, column c0 + i then holds the four
// scales of row 32 i + j for every q, where the MMA reads them.
//
// Every mbarrier wait is bounded (about a second); a wait that gives up marks
// the CTA failed, the CTA still drains what it issued and frees its tensor
// memory, and the tile's first output element is set to NaN.
#pragma once

#include <cuda.h>

#include "fos_kernels.cuh"

namespace fos {
namespace mma {

constexpr int BM = 128, BN = 128;  // output tile
constexpr int kGroupM = 16;        // tile rows per band of the tile order
constexpr int kKBytes = 128;       // code bytes per row per stage (256 K elements)
constexpr int kThreadsMM = 192;
constexpr uint32_t kTmemCols = 256;  // accumulator BN columns + scale columns
constexpr int kABytes = BM * kKBytes, kBBytes = BN * kKBytes, kSfBytes = 4 * 512;

template <int kStages>
constexpr int smem_bytes() {
    return kStages * (kABytes + kBBytes + 2 * kSfBytes) + 1024;  // + alignment slack
}

struct MmArgs {
    CUtensorMap ta;      // a codes [M, K/2] u8, box 128 x BM, 128-byte swizzle
    CUtensorMap tb;      // b codes [N, K/2] u8, box 128 x BN, 128-byte swizzle
    const uint8_t* sfa;  // a scales, tiled layout
    const uint8_t* sfb;  // b scales, tiled layout
    const float* a_amax;
    const float* b_amax;
    float* out;          // [M, N] fp32
    int64_t M, N, K;
    int64_t tiles_m;     // tiles across M
    int64_t tiles_n;     // tiles across N
    int a_row;           // a_amax per row of a
    float six_bound;
};

template <int kStages>
struct __align__(8) MmShared {
    uint64_t full[kStages], empty[kStages], done;
    uint32_t tmem;
    int fail;
};

// Shared-memory matrix descriptors (tcgen05): start address >> 4 in bits
// 0-13, leading byte offset >> 4 in 16-29, stride byte offset >> 4 in 32-45,
// descriptor version 1 in 46-47, layout in 61-63.
// K-major, 128-byte swizzle: rows of 128 bytes, 8-row atoms 1024 bytes apart.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) |
           ((uint64_t)(1024 >> 4) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// No swizzle: 8-row x 16-byte core matrices 128 bytes apart (a scale atom).
__device__ __forceinline__ uint64_t desc_atom(uint32_t saddr) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)(128 >> 4) << 16) |
           ((uint64_t)(128 >> 4) << 32) | ((uint64_t)1 << 46);
}
// Instruction descriptor of kind::mxf4nvf4: A and B E2M1 (1 in bits 7-9 and
// 10-12), K-major, dense, UE4M3 scales (bit 23 = 0), N >> 3 in bits 17-22,
// M >> 4 in bits 24-28, scale-factor ids 0.
constexpr uint32_t kIdesc =
    (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);

__device__ __forceinline__ void bar_init(uint64_t* b, uint32_t n) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(b)), "r"(n) : "memory");
}
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                                 uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::
                     "r"(smem_u32(bar)) : "memory");
}

template <int kStages, int kMinCtas>
__global__ void __launch_bounds__(kThreadsMM, kMinCtas) k_mm_nvfp4(const __grid_constant__ MmArgs a) {
    chain_wait();
    chain_release();
    extern __shared__ __align__(1024) unsigned char s_raw[];
    __shared__ MmShared<kStages> sh;
    // TMA swizzle atoms need 1024-byte aligned stages: round the base up
    unsigned char* sA = s_raw + ((1024u - (smem_u32(s_raw) & 1023u)) & 1023u);
    unsigned char* sB = sA + kStages * kABytes;
    unsigned char* sSA = sB + kStages * kBBytes;
    unsigned char* sSB = sSA + kStages * kSfBytes;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Tile order: bands of kGroupM tile rows; inside a band the tiles run
    // down the rows first, so the CTAs resident at one time cover a compact
    // block of out (about 16 x 19 tiles) whose a and b tiles stay in L2.
    int64_t m0, n0;
    {
        const int64_t t = blockIdx.x;
        const int64_t band = t / (kGroupM * a.tiles_n);
        const int64_t rows_in_band = min((int64_t)kGroupM, a.tiles_m - band * kGroupM);
        const int64_t r = t - band * kGroupM * a.tiles_n;
        m0 = (band * kGroupM + r % rows_in_band) * BM;
        n0 = (r / rows_in_band) * BN;
    }
    const int kb64 = (int)(a.K / 64);  // MMA K steps
    const int nkb = (kb64 + 3) / 4;    // stages of up to four steps
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            bar_init(&sh.full[s], 1);
            bar_init(&sh.empty[s], 1);
        }
        bar_init(&sh.done, 1);
        sh.fail = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&sh.tmem)), "r"(kTmemCols) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sh.tmem;
    if (warp == 0 && lane == 0) {
        uint32_t issued[kStages] = {};  // uses of each stage issued
        for (int i = 0; i < nkb; ++i) {
            const int s = i % kStages;
            if (i >= kStages && !mbar_wait(&sh.empty[s], ((i / kStages) - 1) & 1)) {
                sh.fail = 1;
                break;
            }
            const int nk = min(4, kb64 - 4 * i);
            mbar_expect_tx(&sh.full[s], (uint32_t)(kABytes + kBBytes + 2 * nk * 512));
            tma_load_2d(sA + s * kABytes, &a.ta, i * kKBytes, (int32_t)m0, &sh.full[s]);
            tma_load_2d(sB + s * kBBytes, &a.tb, i * kKBytes, (int32_t)n0, &sh.full[s]);
            bulk_load(sSA + s * kSfBytes, a.sfa + ((m0 / 128) * kb64 + 4 * i) * 512,
                             (uint32_t)(nk * 512), &sh.full[s]);
            bulk_load(sSB + s * kSfBytes, a.sfb + ((n0 / 128) * kb64 + 4 * i) * 512,
                             (uint32_t)(nk * 512), &sh.full[s]);
            issued[s] = (uint32_t)(i / kStages + 1);
        }
        // every copy issued has landed before the CTA can leave
        for (int s = 0; s < kStages; ++s)
            if (issued[s] && !mbar_wait(&sh.full[s], (issued[s] - 1) & 1)) sh.fail = 1;
    } else if (warp == 1 && lane == 0) {
        for (int i = 0; i < nkb; ++i) {
            const int s = i % kStages;
            if (!mbar_wait(&sh.full[s], (i / kStages) & 1)) {
                sh.fail = 1;
                break;
            }
            tc_fence_after();
            const int nk = min(4, kb64 - 4 * i);
            // scale columns of this stage: a at +0, b at +16 (four steps of
            // four columns); alternate halves so a stage never overwrites
            // scales the previous stage's MMAs may still read
            const uint32_t sfc = tmem + BN + (uint32_t)((i & 1) * 32);
            for (int kk = 0; kk < nk; ++kk) {
                asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(sfc + kk * 4),
                             "l"(desc_atom(smem_u32(sSA + s * kSfBytes + kk * 512))) : "memory");
                asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(sfc + 16 + kk * 4),
                             "l"(desc_atom(smem_u32(sSB + s * kSfBytes + kk * 512))) : "memory");
            }
            const uint32_t a0 = smem_u32(sA + s * kABytes), b0 = smem_u32(sB + s * kBBytes);
            for (int kk = 0; kk < nk; ++kk) {
                // K step kk: 32 bytes into each 128-byte swizzled row
                const uint64_t ad = desc_sw128(a0 + kk * 32), bd = desc_sw128(b0 + kk * 32);
                const uint32_t accumulate = (i > 0 || kk > 0) ? 1u : 0u;
                asm volatile(
                    "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
                    "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, "
                    "%3, [%4], [%5], p;\n\t}" ::"r"(tmem),
                    "l"(ad), "l"(bd), "r"(kIdesc), "r"(sfc + kk * 4), "r"(sfc + 16 + kk * 4),
                    "r"(accumulate)
                    : "memory");
            }
            tc_commit(&sh.empty[s]);
        }
        tc_commit(&sh.done);  // arrives once every MMA issued above has completed
    } else if (warp >= 2) {
        const int q = warp & 3;  // tensor-memory lanes 32 q .. 32 q + 31
        const bool ok = mbar_wait(&sh.done, 0);
        __syncwarp();
        tc_fence_after();
        const int64_t m = m0 + 32 * q + lane;
        const float gb = fdiv(1.0f, global_scale(a.b_amax[0], a.six_bound));
        float ga = 0.0f;
        if (m < a.M) ga = fdiv(1.0f, global_scale(a.a_amax[a.a_row ? m : 0], a.six_bound));
        for (int c0 = 0; c0 < BN; c0 += 32) {
            uint32_t v[32];
            const uint32_t taddr = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)c0;
            asm volatile(
                "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
                "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
                : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
                  "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]),
                  "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]),
                  "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),
                  "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]),
                  "=r"(v[31])
                : "r"(taddr));
            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
            const int64_t n = n0 + c0;
            if (m < a.M && n < a.N) {
                float* dst = a.out + m * a.N + n;
#pragma unroll
                for (int j = 0; j < 32; j += 4) {
                    if (n + j < a.N) {  // N % 16 == 0: four columns are all in or all out
                        float4 o;
                        o.x = fmul(fmul(__uint_as_float(v[j]), ga), gb);
                        o.y = fmul(fmul(__uint_as_float(v[j + 1]), ga), gb);
                        o.z = fmul(fmul(__uint_as_float(v[j + 2]), ga), gb);
                        o.w = fmul(fmul(__uint_as_float(v[j + 3]), ga), gb);
                        // streamed (evict-first): out must not push the
                        // operand tiles out of L2
                        asm volatile("st.global.cs.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst + j),
                                     "f"(o.x), "f"(o.y), "f"(o.z), "f"(o.w) : "memory");
                    }
                }
            }
        }
        if (!ok) sh.fail = 1;
    }
    tc_fence_before();
    __syncthreads();
    if (sh.fail && threadIdx.x == 0 && m0 < a.M && n0 < a.N)
        a.out[m0 * a.N + n0] = __int_as_float(0x7FC00000);
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols) : "memory");
    }
}

}  // namespace mma
}  // namespace fos

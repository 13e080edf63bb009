// fos_mma.cuh -- the block-scaled NVFP4 product on the 5th-generation tensor
// cores of sm_103a (tcgen05): out = a . b^T from 1x16 E2M1 codes and E4M3
// block scales in the tiled layout, with the FP32 global decode scales applied
// in the epilogue (grouped PR, the dense-recipe commit's four_over_six_mm
// forward; per row of a for a row-scaled a, the MoE commit's epilogue).
//
// A persistent kernel: one CTA per SM walks BM x BN = 128 x 192 output tiles
// (tile t, t + grid, ...), with two accumulators in tensor memory so that
// the epilogue of one tile runs while the MMAs of the next fill the other.
// Warp roles:
//   warp 0      (one thread) TMA producer: per K stage of 256 elements, the a
//               and b code tiles (2D TMA, 128-byte swizzle) and the stage's
//               512-byte scale atoms (1D bulk copies: four for a, four for
//               each of the two 128-row scale tiles b's 192 rows touch) into
//               a ring of kStages shared-memory stages;
//   warp 1      allocates the tensor memory; one thread issues per stage four
//               tcgen05.mma kind::mxf4nvf4 block_scale scale_vec::4X
//               (M = 128, N = 192, K = 64 each) into the tile's accumulator,
//               then frees the stage (tcgen05.commit to its mbarrier) and,
//               after a tile's last stage, hands the accumulator to the
//               epilogue;
//   warps 2-5   scale warps: move each stage's scale atoms from shared to
//               tensor memory (ld.shared, two tcgen05.st of 16 and 32
//               columns), warp w into the lanes 32 (w % 4) .. 32 (w % 4) + 31
//               it may write;
//   warps 6-..  epilogue (kEpi warps, kEpi / 4 per lane quadrant): read the
//               FP32 accumulator (tcgen05.ld), multiply by g_a(m) and then
//               g_b, stage 32 x 32 chunks in shared memory in the 128-byte
//               swizzle and store them with TMA (cp.async.bulk.tensor), which
//               clips the rows and columns past the end of out.
// Two accumulators (192 columns each) and two scale buffers (48 columns
// each: a stage's scales are written while the previous stage's MMAs read
// theirs) take 480 of the 512 tensor-memory columns.
//
// Operands are K-major: a row of a (or b) holds K/2 code bytes, element 2j in
// the low nibble of byte j, which is the element order of the E2M1 operand.
// The scale atom of rows [128 t, 128 t + 128) and K elements [64 c, 64 c + 64)
// is the 512-byte tile (t, c) of the tiled layout: byte 16 j + 4 i + k holds
// the scale of row 32 i + j, 16-element block k.  The MMA reads the four
// scales of row r of its a (b) tile from tensor-memory lane 32 q + r % 32,
// column c0 + r / 32, for each quadrant q: a scale warp of quadrant q stores
// word i of 16-byte row j of the atom to its lane 32 q + j, column c0 + i.
// A b tile starts at n0 = 192 t, at row 0 or row 64 of a scale tile: its
// six 32-row groups are words 0-3 of the first atom and 0-1 of the next, or
// words 2-3 of the first and 0-3 of the next.
//
// Every mbarrier wait is bounded (about a second); a wait that gives up marks
// the CTA failed, the CTA still drains what it issued (copies, MMAs, stores)
// and frees its tensor memory, and the first element of its first tile is set
// to NaN.
#pragma once

#include <cuda.h>

#include "fos_kernels.cuh"

namespace fos {
namespace mma {

constexpr int BM = 128, BN = 192;  // output tile
constexpr int kGroupM = 16;        // tile rows per band of the tile order
constexpr int kKBytes = 128;       // code bytes per row per stage (256 K elements)
constexpr int kStages = 4;
constexpr int kSfWarps = 4;
constexpr uint32_t kTmemCols = 512;
constexpr int kABytes = BM * kKBytes, kBBytes = BN * kKBytes;
constexpr int kSfBytes = 4 * 512;                 // scale atoms of a stage, 128 rows
constexpr int kSfbBytes = 2 * kSfBytes;           // b's scale atoms of a stage (two tiles)
constexpr int kSfCols = 16 + 32;                  // scale columns of a stage: a 4, b 8 per K step
constexpr int kChunkBytes = 32 * 32 * 4;          // epilogue chunk: 32 rows x 32 fp32
constexpr int kAccCols = 2 * BN;                  // two accumulators
static_assert(kAccCols + 2 * kSfCols <= (int)kTmemCols, "tensor memory");

constexpr int threads_mm(int epi) { return 32 * (2 + kSfWarps + epi); }
template <int kEpi, int kBufs>
constexpr int smem_bytes() {
    return kStages * (kABytes + kBBytes + kSfBytes + kSfbBytes) + kEpi * kBufs * kChunkBytes +
           1024;  // + alignment slack
}

struct MmArgs {
    CUtensorMap ta;      // a codes [M, K/2] u8, box 128 x BM, 128-byte swizzle
    CUtensorMap tb;      // b codes [N, K/2] u8, box 128 x BN, 128-byte swizzle
    CUtensorMap to;      // out [M, N] fp32, box 32 x 32, 128-byte swizzle
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

struct __align__(8) MmShared {
    uint64_t full[kStages], empty[kStages], sf_ready[kStages], acc_full[2], acc_empty[2], mma_done;
    uint32_t tmem;
    int fail;
};

// Shared-memory matrix descriptor (tcgen05) of a K-major operand with the
// 128-byte swizzle: start address >> 4 in bits 0-13, leading byte offset 16
// (>> 4) in 16-29, 8-row atoms 1024 bytes apart (>> 4) in 32-45, descriptor
// version 1 in 46-47, layout 2 (128-byte swizzle) in 61-63.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) |
           ((uint64_t)(1024 >> 4) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// Instruction descriptor of kind::mxf4nvf4: A and B E2M1 (1 in bits 7-9 and
// 10-12), K-major, dense, UE4M3 scales (bit 23 = 0), N >> 3 in bits 17-22,
// M >> 4 in bits 24-28, scale-factor ids 0.
constexpr uint32_t kIdesc =
    (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);

__device__ __forceinline__ void bar_init(uint64_t* b, uint32_t n) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(b)), "r"(n) : "memory");
}
__device__ __forceinline__ void bar_arrive(uint64_t* b) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(b)) : "memory");
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
// tcgen05.st of 16 and 32 consecutive columns (32x32b shape: register c of
// lane l goes to lane 32 q + l, column taddr + c).
__device__ __forceinline__ void tmem_st_x16(uint32_t taddr, const uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
        "%13,%14,%15,%16};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
        "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
}
__device__ __forceinline__ void tmem_st_x32(uint32_t taddr, const uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
        "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(
            taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
        "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]),
        "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]),
        "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]),
        "r"(v[30]), "r"(v[31])
        : "memory");
}

// Tile order: bands of kGroupM tile rows; inside a band the tiles run down
// the rows first, so the tiles in flight at one time cover a compact block
// of out whose a and b tiles stay in L2.
__device__ __forceinline__ void tile_coords(const MmArgs& a, int64_t t, int64_t& m0, int64_t& n0) {
    const int64_t band = t / (kGroupM * a.tiles_n);
    const int64_t rows_in_band = min((int64_t)kGroupM, a.tiles_m - band * kGroupM);
    const int64_t r = t - band * kGroupM * a.tiles_n;
    m0 = (band * kGroupM + r % rows_in_band) * BM;
    n0 = (r / rows_in_band) * BN;
}

// kEpi epilogue warps (4 or 8), kBufs staging chunks per epilogue warp.
template <int kEpi, int kBufs>
__global__ void __launch_bounds__(threads_mm(kEpi), 1) k_mm_nvfp4(const __grid_constant__ MmArgs a) {
    static_assert(kEpi == 4 || kEpi == 8, "epilogue warps");
    static_assert(kBufs >= 1 && kBufs <= 3, "staging chunks");
    chain_wait();
    chain_release();
    extern __shared__ __align__(1024) unsigned char s_raw[];
    __shared__ MmShared sh;
    // TMA swizzle atoms need 1024-byte aligned stages: round the base up
    unsigned char* sA = s_raw + ((1024u - (smem_u32(s_raw) & 1023u)) & 1023u);
    unsigned char* sB = sA + kStages * kABytes;
    unsigned char* sSA = sB + kStages * kBBytes;
    unsigned char* sSB = sSA + kStages * kSfBytes;
    unsigned char* sOut = sSB + kStages * kSfbBytes;  // 1024-aligned chunks
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int kb64 = (int)(a.K / 64);  // MMA K steps
    const int nkb = (kb64 + 3) / 4;    // stages of up to four steps
    const int64_t tiles = a.tiles_m * a.tiles_n;
    const int64_t sf_tiles_n = (a.N + 127) / 128;  // 128-row scale tiles of b
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            bar_init(&sh.full[s], 1);
            bar_init(&sh.empty[s], 1);
            bar_init(&sh.sf_ready[s], kSfWarps);
        }
        for (int b = 0; b < 2; ++b) {
            bar_init(&sh.acc_full[b], 1);
            bar_init(&sh.acc_empty[b], kEpi);
        }
        bar_init(&sh.mma_done, 1);
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
    if (warp == 0) {
        if (lane == 0) {
            uint32_t g = 0;  // stages issued so far, over all tiles
            bool bad = false;
            for (int64_t t = blockIdx.x; t < tiles && !bad; t += gridDim.x) {
                int64_t m0, n0;
                tile_coords(a, t, m0, n0);
                const bool b1 = n0 / 128 + 1 < sf_tiles_n;  // b's second scale tile exists
                for (int i = 0; i < nkb; ++i, ++g) {
                    const int s = (int)(g % kStages);
                    if (g >= (uint32_t)kStages &&
                        !mbar_wait(&sh.empty[s], ((g / kStages) - 1) & 1)) {
                        bad = true;
                        break;
                    }
                    const int nk = min(4, kb64 - 4 * i);
                    mbar_expect_tx(&sh.full[s],
                                   (uint32_t)(kABytes + kBBytes + (b1 ? 3 : 2) * nk * 512));
                    tma_load_2d(sA + s * kABytes, &a.ta, i * kKBytes, (int32_t)m0, &sh.full[s]);
                    tma_load_2d(sB + s * kBBytes, &a.tb, i * kKBytes, (int32_t)n0, &sh.full[s]);
                    bulk_load(sSA + s * kSfBytes, a.sfa + ((m0 / 128) * kb64 + 4 * i) * 512,
                              (uint32_t)(nk * 512), &sh.full[s]);
                    bulk_load(sSB + s * kSfbBytes, a.sfb + ((n0 / 128) * kb64 + 4 * i) * 512,
                              (uint32_t)(nk * 512), &sh.full[s]);
                    if (b1)
                        bulk_load(sSB + s * kSfbBytes + kSfBytes,
                                  a.sfb + ((n0 / 128 + 1) * kb64 + 4 * i) * 512,
                                  (uint32_t)(nk * 512), &sh.full[s]);
                }
            }
            if (bad) sh.fail = 1;
            // every copy issued has landed before the CTA can leave
            for (uint32_t s = 0; s < (uint32_t)kStages; ++s)
                if (g > s && !mbar_wait(&sh.full[s], ((g - 1 - s) / kStages) & 1)) sh.fail = 1;
        }
    } else if (warp == 1) {
        if (lane == 0) {
            uint32_t g = 0;
            bool bad = false;
            int j = 0;
            for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x, ++j) {
                // the epilogue has read this accumulator's previous tile
                const int ab = j & 1;
                if (j >= 2 && !mbar_wait(&sh.acc_empty[ab], ((j >> 1) - 1) & 1)) {
                    bad = true;
                    break;
                }
                tc_fence_after();
                const uint32_t acc = tmem + (uint32_t)(ab * BN);
                for (int i = 0; i < nkb; ++i, ++g) {
                    const int s = (int)(g % kStages);
                    if (!mbar_wait(&sh.full[s], (g / kStages) & 1) ||
                        !mbar_wait(&sh.sf_ready[s], (g / kStages) & 1)) {
                        bad = true;
                        break;
                    }
                    tc_fence_after();
                    const int nk = min(4, kb64 - 4 * i);
                    // scales of this stage: a at +0 (4 columns per K step),
                    // b at +16 (8 per K step: 4 per 128 rows)
                    const uint32_t sfc = tmem + (uint32_t)(kAccCols + (g & 1) * kSfCols);
                    const uint32_t a0 = smem_u32(sA + s * kABytes), b0 = smem_u32(sB + s * kBBytes);
                    for (int kk = 0; kk < nk; ++kk) {
                        // K step kk: 32 bytes into each 128-byte swizzled row
                        const uint64_t ad = desc_sw128(a0 + kk * 32), bd = desc_sw128(b0 + kk * 32);
                        const uint32_t accumulate = (i > 0 || kk > 0) ? 1u : 0u;
                        asm volatile(
                            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
                            "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X "
                            "[%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(acc),
                            "l"(ad), "l"(bd), "r"(kIdesc), "r"(sfc + kk * 4),
                            "r"(sfc + 16 + kk * 8), "r"(accumulate)
                            : "memory");
                    }
                    tc_commit(&sh.empty[s]);
                }
                if (bad) break;
                tc_commit(&sh.acc_full[ab]);
            }
            if (bad) sh.fail = 1;
            // every MMA issued has completed before the tensor memory is freed
            tc_commit(&sh.mma_done);
            if (!mbar_wait(&sh.mma_done, 0)) sh.fail = 1;
        }
    } else if (warp < 2 + kSfWarps) {
        // scale warps: warp w writes tensor-memory lanes 32 q .. 32 q + 31,
        // q = w % 4; lane j takes 16-byte row j of each atom: a's four words
        // to columns +4 kk .. +4 kk + 3, b's six 32-row groups to columns
        // +16 + 8 kk .. (two more columns of zeros keep each K step's b
        // scales 8 columns apart)
        const int q = warp & 3;
        uint32_t g = 0;
        bool bad = false;
        for (int64_t t = blockIdx.x; t < tiles && !bad; t += gridDim.x) {
            int64_t m0, n0;
            tile_coords(a, t, m0, n0);
            const bool b1 = n0 / 128 + 1 < sf_tiles_n;
            const bool off2 = (n0 & 127) != 0;  // b's rows start half-way into a scale tile
            for (int i = 0; i < nkb; ++i, ++g) {
                const int s = (int)(g % kStages);
                if (!mbar_wait(&sh.full[s], (g / kStages) & 1) ||
                    (g >= 2 && !mbar_wait(&sh.empty[(g - 2) % kStages], ((g - 2) / kStages) & 1))) {
                    bad = true;
                    break;
                }
                tc_fence_after();
                const uint32_t sfc =
                    tmem + (uint32_t)(kAccCols + (g & 1) * kSfCols) + ((uint32_t)(32 * q) << 16);
                const unsigned char* pa = sSA + s * kSfBytes + 16 * lane;
                const unsigned char* pb = sSB + s * kSfbBytes + 16 * lane;
                uint32_t va[16], vb[32];
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint4 x = *reinterpret_cast<const uint4*>(pa + kk * 512);
                    va[4 * kk] = x.x; va[4 * kk + 1] = x.y; va[4 * kk + 2] = x.z; va[4 * kk + 3] = x.w;
                    const uint4 u0 = *reinterpret_cast<const uint4*>(pb + kk * 512);
                    uint4 u1 = make_uint4(0, 0, 0, 0);
                    if (b1) u1 = *reinterpret_cast<const uint4*>(pb + kSfBytes + kk * 512);
                    // column c holds row 32 c + lane of b's 192 rows
                    vb[8 * kk + 0] = off2 ? u0.z : u0.x;
                    vb[8 * kk + 1] = off2 ? u0.w : u0.y;
                    vb[8 * kk + 2] = off2 ? u1.x : u0.z;
                    vb[8 * kk + 3] = off2 ? u1.y : u0.w;
                    vb[8 * kk + 4] = off2 ? u1.z : u1.x;
                    vb[8 * kk + 5] = off2 ? u1.w : u1.y;
                    vb[8 * kk + 6] = 0;
                    vb[8 * kk + 7] = 0;
                }
                tmem_st_x16(sfc, va);
                tmem_st_x32(sfc + 16, vb);
                asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                tc_fence_before();
                __syncwarp();
                if (lane == 0) bar_arrive(&sh.sf_ready[s]);
            }
        }
        if (bad) sh.fail = 1;
    } else {
        // epilogue: warp e reads lanes 32 q .. of columns [c_beg, c_beg + kCols)
        const int q = warp & 3;
        const int e = warp - 2 - kSfWarps;
        constexpr int kCols = BN / (kEpi / 4);
        const int c_beg = (e / 4) * kCols;
        const float gb = fdiv(1.0f, global_scale(a.b_amax[0], a.six_bound));
        const float ga0 = a.a_row ? 0.0f : fdiv(1.0f, global_scale(a.a_amax[0], a.six_bound));
        int j = 0, chunk = 0;
        for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x, ++j) {
            const int ab = j & 1;
            if (!mbar_wait(&sh.acc_full[ab], (j >> 1) & 1)) {
                sh.fail = 1;
                break;
            }
            __syncwarp();
            tc_fence_after();
            int64_t m0, n0;
            tile_coords(a, t, m0, n0);
            const int64_t m = m0 + 32 * q + lane;
            float ga = ga0;
            if (a.a_row && m < a.M) ga = fdiv(1.0f, global_scale(a.a_amax[m], a.six_bound));
            for (int c0 = c_beg; c0 < c_beg + kCols; c0 += 32, ++chunk) {
                uint32_t v[32];
                const uint32_t taddr = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(ab * BN + c0);
                asm volatile(
                    "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,"
                    "%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,"
                    "%30,%31}, [%32];"
                    : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]),
                      "=r"(v[6]), "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]),
                      "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]),
                      "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]),
                      "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]), "=r"(v[26]),
                      "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
                    : "r"(taddr));
                asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
                if (c0 + 32 == c_beg + kCols) {  // this warp's columns read: the MMA may go on
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) bar_arrive(&sh.acc_empty[ab]);
                }
                // staging chunk of this warp: the store issued kBufs chunks
                // ago must have finished reading it
                unsigned char* buf = sOut + (e * kBufs + chunk % kBufs) * kChunkBytes;
                if (lane == 0) {
                    if constexpr (kBufs == 1)
                        asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
                    else if constexpr (kBufs == 2)
                        asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
                    else
                        asm volatile("cp.async.bulk.wait_group.read 2;" ::: "memory");
                }
                __syncwarp();
#pragma unroll
                for (int k = 0; k < 8; ++k) {  // 16-byte piece k of row `lane`, 128-byte swizzle
                    const uint32_t addr = smem_u32(buf) + lane * 128 + ((k ^ (lane & 7)) * 16);
                    asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr),
                                 "f"(fmul(fmul(__uint_as_float(v[4 * k]), ga), gb)),
                                 "f"(fmul(fmul(__uint_as_float(v[4 * k + 1]), ga), gb)),
                                 "f"(fmul(fmul(__uint_as_float(v[4 * k + 2]), ga), gb)),
                                 "f"(fmul(fmul(__uint_as_float(v[4 * k + 3]), ga), gb))
                                 : "memory");
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) {
                    asm volatile(
                        "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], "
                        "[%3];" ::"l"(&a.to),
                        "r"((int32_t)(n0 + c0)), "r"((int32_t)(m0 + 32 * q)), "r"(smem_u32(buf))
                        : "memory");
                    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
                }
            }
        }
        if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
        __syncwarp();
    }
    tc_fence_before();
    __syncthreads();
    if (sh.fail && threadIdx.x == 0 && (int64_t)blockIdx.x < tiles) {
        int64_t m0, n0;
        tile_coords(a, blockIdx.x, m0, n0);
        a.out[m0 * a.N + n0] = __int_as_float(0x7FC00000);
    }
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols) : "memory");
    }
}

}  // namespace mma
}  // namespace fos

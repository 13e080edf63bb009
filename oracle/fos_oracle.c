/*
 * fos_oracle.c -- CPU oracle for the NVFP4 four-over-six ("4/6") block quantizer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or call
 * this file; only the test suite, the smoke check and the benchmark's CPU
 * baseline use it.  It shares no code, header, table or helper with the CUDA
 * library: every format conversion below is written from the format
 * definitions, not taken from the GPU side.
 *
 * What it computes (sources are the three pages the method is described on):
 *   - torchao PR "Add the four-over-six grouped GEMM and dispatcher wiring",
 *     description, first commit: every 16-element block (1x16, or 16x16 for
 *     weights) is encoded twice under an FP32 global scale -- the standard
 *     map-to-6 encoding and a 1.5x-scale map-to-4 candidate -- and the
 *     lower-error candidate's packed E2M1 codes and E4M3 scale are stored;
 *     per-tensor or row-scaled global scales.
 *   - torchao PR "Add a CuTe DSL fast-path kernel for four-over-six quantize",
 *     description: correctly-rounded FP32 division, RN casts to FP4/E4M3 with
 *     exact decodes, a pinned width-16 clamped shuffle-down error reduction,
 *     NaN-dropping block amax with NaN elements encoded as +6.
 *   - Megatron-LM PR "Fuse NVFP4 fake-QAT quantize-dequantize with CuTe DSL",
 *     "What does this PR do?": caller FP32 per-tensor amax, MAE/MSE,
 *     E4M3 max 448/256, exact-FP32 or FP16 candidate error, FP32 error squares,
 *     one common per-block scale multiplied into adjacent values.
 *   - grouped PR, third commit: per-group amax expanded per row, grouped
 *     result bitwise equal to per-group calls, offs[-1] tail zero-extend,
 *     per-row amax with 16x16 blocks under a tile-uniform contract.
 *
 * Where the pages leave a step open, the reading taken is marked R<n> at the
 * point it is used; each R<n> is one constant or branch.
 *
 * Arithmetic: plain scalar IEEE binary32 (compile with -O2 -ffp-contract=off,
 * no fast-math) so that every *, -, + and / rounds once to nearest-even.
 * Format conversions use binary64 internally only where that is exact.
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------- */
/* Configuration mirror (the oracle's own; not the library's header).        */
/* ------------------------------------------------------------------------- */
typedef struct {
    int block16x16;     /* 0: 1x16 blocks, 1: 16x16 tiles                    */
    int four_over_six;  /* 0: standard map-to-6 only, 1: four-over-six       */
    int mse;            /* 0: MAE, 1: MSE                                    */
    int err_f16;        /* 0: exact-FP32 candidate error, 1: FP16 error      */
    int bound;          /* E4M3 bound used in the global scale: 448 or 256   */
    int row_scaled;     /* 0: per-tensor amax, 1: per-row amax               */
    int amax_is_input;  /* 1: amax given, 0: oracle computes and writes it   */
    int seq_order;      /* 0: pinned tree reduction, 1: sequential (R16)     */
} orc_config;

enum { ORC_OK = 0, ORC_BAD = 1 };
enum { ORC_OUT_F32 = 0, ORC_OUT_BF16 = 1, ORC_OUT_F16 = 2 };

/* ------------------------------------------------------------------------- */
/* E2M1 (OCP Microscaling Formats v1.0, FP4): sign, 2 exponent bits with     */
/* bias 1, 1 mantissa bit, no Inf/NaN.  Magnitudes 0,0.5,1,1.5,2,3,4,6.      */
/* ------------------------------------------------------------------------- */
float orc_e2m1_value(uint32_t code)
{
    uint32_t s = (code >> 3) & 1u, e = (code >> 1) & 3u, m = code & 1u;
    double mag = (e == 0) ? 0.5 * (double)m : ldexp(1.0 + 0.5 * (double)m, (int)e - 1);
    return (float)(s ? -mag : mag);
}

/* Round to nearest, ties to the even code; saturate to 6 (satfinite);
 * NaN encodes as +6 (0x7) -- the pages' documented NaN behaviour. */
uint32_t orc_e2m1_encode(float y)
{
    if (isnan(y)) return 0x7u;
    uint32_t sign = signbit(y) ? 0x8u : 0x0u;
    float a = fabsf(y);
    uint32_t best = 0x7u;
    for (uint32_t c = 0; c < 7u; ++c) {
        double mid = 0.5 * ((double)orc_e2m1_value(c) + (double)orc_e2m1_value(c + 1u));
        if ((double)a < mid) { best = c; break; }
        if ((double)a == mid) { best = (c & 1u) ? c + 1u : c; break; }
    }
    return sign | best;
}

/* ------------------------------------------------------------------------- */
/* E4M3 (OCP FP8 E4M3, "fn"): sign, 4 exponent bits bias 7, 3 mantissa bits; */
/* no Inf; S.1111.111 is NaN; largest finite 448 (0x7E).                     */
/* ------------------------------------------------------------------------- */
float orc_e4m3_value(uint32_t code)
{
    uint32_t s = (code >> 7) & 1u, e = (code >> 3) & 15u, m = code & 7u;
    if (e == 15u && m == 7u) return NAN;
    double mag = (e == 0) ? ldexp((double)m, -9) : ldexp(1.0 + (double)m / 8.0, (int)e - 7);
    return (float)(s ? -mag : mag);
}

/* RN-even with satfinite: magnitudes past 448 (including Inf) clamp to 448;
 * NaN stays NaN.  Scans the monotone code ladder 0x00..0x7E. */
uint32_t orc_e4m3_encode(float v)
{
    uint32_t sign = signbit(v) ? 0x80u : 0x00u;
    if (isnan(v)) return sign | 0x7Fu;
    float a = fabsf(v);
    uint32_t best = 0x7Eu;
    for (uint32_t c = 0; c < 0x7Eu; ++c) {
        double mid = 0.5 * ((double)orc_e4m3_value(c) + (double)orc_e4m3_value(c + 1u));
        if ((double)a < mid) { best = c; break; }
        if ((double)a == mid) { best = (c & 1u) ? c + 1u : c; break; }
    }
    return sign | best;
}

/* ------------------------------------------------------------------------- */
/* IEEE binary16 / bfloat16 round-to-nearest-even, from the definitions:     */
/* p-bit significand, minimum normal exponent emin; quantum of the binade    */
/* 2^(max(e,emin)-(p-1)).  Overflow rounds to Inf.                           */
/* ------------------------------------------------------------------------- */
static double rne_to_format(double a, int p, int emin, double maxfinite)
{
    /* a > 0, finite */
    int e2;
    (void)frexp(a, &e2);           /* a = f * 2^e2, f in [0.5, 1) */
    int e = e2 - 1;                 /* floor(log2 a) */
    if (e < emin) e = emin;
    double q = ldexp(1.0, e - (p - 1));
    double m = rint(a / q);         /* exact scaling, RNE to integer */
    double r = m * q;
    return (r > maxfinite) ? INFINITY : r;
}

float orc_f16_round(float v)
{
    if (isnan(v) || isinf(v) || v == 0.0f) return v;
    double r = rne_to_format(fabs((double)v), 11, -14, 65504.0);
    return (float)(signbit(v) ? -r : r);
}

float orc_bf16_round(float v)
{
    if (isnan(v) || isinf(v) || v == 0.0f) return v;
    double maxf = ldexp(255.0, 120);             /* (2 - 2^-7) * 2^127 */
    double r = rne_to_format(fabs((double)v), 8, -126, maxf);
    return (float)(signbit(v) ? -r : r);
}

/* Bit patterns of an already-rounded value.  Any NaN maps to 0x7FFF (R15:
 * the payload of a NaN result is not fixed by the pages). */
uint16_t orc_f16_bits(float v)
{
    uint16_t s = signbit(v) ? 0x8000u : 0u;
    if (isnan(v)) return 0x7FFFu;
    float r = orc_f16_round(v);
    if (isinf(r)) return s | 0x7C00u;
    double a = fabs((double)r);
    if (a == 0.0) return s;
    if (a < ldexp(1.0, -14)) return s | (uint16_t)(a / ldexp(1.0, -24));
    int e2;
    (void)frexp(a, &e2);
    int e = e2 - 1;
    uint32_t mant = (uint32_t)((a / ldexp(1.0, e) - 1.0) * 1024.0);
    return s | (uint16_t)((uint32_t)(e + 15) << 10) | (uint16_t)mant;
}

uint16_t orc_bf16_bits(float v)
{
    uint16_t s = signbit(v) ? 0x8000u : 0u;
    if (isnan(v)) return 0x7FFFu;
    float r = orc_bf16_round(v);
    if (isinf(r)) return s | 0x7F80u;
    double a = fabs((double)r);
    if (a == 0.0) return s;
    if (a < ldexp(1.0, -126)) return s | (uint16_t)(a / ldexp(1.0, -133));
    int e2;
    (void)frexp(a, &e2);
    int e = e2 - 1;
    uint32_t mant = (uint32_t)((a / ldexp(1.0, e) - 1.0) * 128.0);
    return s | (uint16_t)((uint32_t)(e + 127) << 7) | (uint16_t)mant;
}

/* ------------------------------------------------------------------------- */
/* Method steps                                                              */
/* ------------------------------------------------------------------------- */

/* NaN-dropping max|x| with initial +0 (fast-path PR: NaN-dropping block
 * amax).  R1: the same rule is used for tensor / row / group amaxes. */
static float amax_nan_dropping(const float* x, int64_t n, int64_t stride)
{
    float m = 0.0f;
    for (int64_t i = 0; i < n; ++i) {
        float v = fabsf(x[i * stride]);
        if (v > m) m = v;
    }
    return m;
}

/* R2: FP32 global encode scale S = (6 * bound) / A, correctly rounded.
 * Degenerate amax (zero, negative, NaN, Inf) gives S = 1; an overflowing
 * quotient (A tiny) gives FLT_MAX. */
float orc_global_scale(float A, int bound)
{
    if (!(A > 0.0f) || isinf(A)) return 1.0f;
    float S = (6.0f * (float)bound) / A;
    if (isinf(S)) S = FLT_MAX;
    return S;
}

/* Pinned width-16 reduction (clamped shuffle-down tree): for w = 8,4,2,1:
 * t[i] = t[i] + t[i+w] for i < w.  Returns t[0]. */
static float tree16(const float* in)
{
    float t[16];
    memcpy(t, in, sizeof(t));
    for (int w = 8; w >= 1; w /= 2)
        for (int i = 0; i < w; ++i) t[i] = t[i] + t[i + w];
    return t[0];
}

/* Sequential accumulation of the 16 terms in element order (R16): the
 * Transformer Engine term order the Megatron PR keeps for its sequential
 * error accumulation ("Packed pair arithmetic"): acc = t[0], then
 * acc = acc + t[i] for i = 1..15 (starting from +0 gives the same sums, the
 * terms being >= +0). */
static float seq16(const float* in)
{
    float acc = in[0];
    for (int i = 1; i < 16; ++i) acc = acc + in[i];
    return acc;
}

typedef struct {
    uint32_t sc_code;  /* E4M3 bits of the block scale          */
    float sigma;       /* its exact decode                      */
    float r, d;        /* encode / decode common scales         */
    float err;         /* reduced candidate error (sum, R9)     */
    uint8_t q[256];    /* E2M1 codes, element order of the block */
} orc_cand;

/* One candidate ("map-to-k", k = 6 or 4) for a block given as nrows rows of
 * 16 values (nrows = 1 or 16), row stride ld. */
static void candidate(const float* x, int nrows, int64_t ld, float a_b, float S, float k,
                      const orc_config* cfg, orc_cand* c)
{
    float t = a_b * S;               /* R3: amax times S, then divide by k  */
    float s = t / k;
    c->sc_code = orc_e4m3_encode(s); /* R4: RN satfinite, overflow -> 448    */
    c->sigma = orc_e4m3_value(c->sc_code);
    if (c->sigma == 0.0f) {          /* R5: zero scale -> zero common scales */
        c->r = 0.0f;
        c->d = 0.0f;
    } else {
        c->r = S / c->sigma;
        c->d = c->sigma / S;
    }
    float P[16];
    for (int rr = 0; rr < nrows; ++rr) {
        float terms[16];
        for (int i = 0; i < 16; ++i) {
            float xi = x[rr * ld + i];
            float y = xi * c->r;
            uint32_t q = orc_e2m1_encode(y);
            c->q[rr * 16 + i] = (uint8_t)q;
            float deq = orc_e2m1_value(q) * c->d;
            if (cfg->err_f16) deq = orc_f16_round(deq); /* R6 */
            float e = xi - deq;
            terms[i] = cfg->mse ? e * e : fabsf(e);
        }
        P[rr] = cfg->seq_order ? seq16(terms) : tree16(terms);
    }
    c->err = (nrows == 1) ? P[0] : tree16(P);        /* R8 */
}

/* Encode one block; returns the selected candidate (R10: map-to-4 only when
 * its error is strictly lower).  e6/e4 receive both errors when non-NULL. */
static const orc_cand* encode_block(const float* x, int nrows, int64_t ld, float S,
                                    const orc_config* cfg, orc_cand* c6, orc_cand* c4,
                                    float* e6, float* e4)
{
    float a_b = 0.0f;
    for (int rr = 0; rr < nrows; ++rr) {
        float m = amax_nan_dropping(x + rr * ld, 16, 1);
        if (m > a_b) a_b = m;
    }
    candidate(x, nrows, ld, a_b, S, 6.0f, cfg, c6);
    if (!cfg->four_over_six) {
        if (e6) *e6 = c6->err;
        if (e4) *e4 = NAN;
        return c6;
    }
    candidate(x, nrows, ld, a_b, S, 4.0f, cfg, c4);
    if (e6) *e6 = c6->err;
    if (e4) *e4 = c4->err;
    return (c4->err < c6->err) ? c4 : c6;
}

static void store_out(void* out, int out_kind, int64_t idx, float v)
{
    if (out_kind == ORC_OUT_F32) ((float*)out)[idx] = v;
    else if (out_kind == ORC_OUT_BF16) ((uint16_t*)out)[idx] = orc_bf16_bits(v);
    else ((uint16_t*)out)[idx] = orc_f16_bits(v);
}

/* ------------------------------------------------------------------------- */
/* Amax                                                                      */
/* ------------------------------------------------------------------------- */
void orc_amax_tensor(const float* x, int64_t n, float* out) { *out = amax_nan_dropping(x, n, 1); }

void orc_amax_rows(const float* x, int64_t rows, int64_t cols, float* out)
{
    for (int64_t r = 0; r < rows; ++r) out[r] = amax_nan_dropping(x + r * cols, cols, 1);
}

/* R12: offs are cumulative group ends; end_g = clamp(offs[g], end_{g-1}, rows). */
static void group_ends(const int32_t* offs, int G, int64_t rows, int64_t* ends)
{
    int64_t prev = 0;
    for (int g = 0; g < G; ++g) {
        int64_t e = offs[g];
        if (e < prev) e = prev;
        if (e > rows) e = rows;
        ends[g] = e;
        prev = e;
    }
}

void orc_amax_groups(const float* x, int64_t rows, int64_t cols, const int32_t* offs, int G,
                     float* out)
{
    int64_t* ends = (int64_t*)malloc(sizeof(int64_t) * (size_t)(G > 0 ? G : 1));
    group_ends(offs, G, rows, ends);
    int64_t lo = 0;
    for (int g = 0; g < G; ++g) {
        out[g] = amax_nan_dropping(x + lo * cols, (ends[g] - lo) * cols, 1);
        lo = ends[g];
    }
    free(ends);
}

/* ------------------------------------------------------------------------- */
/* Quantize / QDQ over a tensor whose rows each carry a global amax          */
/* (row_amax[r]); the public entry points below build that per-row view.    */
/* ------------------------------------------------------------------------- */
static void quantize_rows(const float* x, int64_t rows, int64_t cols, const orc_config* cfg,
                          const float* row_amax, const uint8_t* row_live, uint8_t* codes,
                          uint8_t* scales, float* err6, float* err4, void* qdq_out,
                          int out_kind)
{
    orc_cand* c6 = (orc_cand*)malloc(sizeof(orc_cand));
    orc_cand* c4 = (orc_cand*)malloc(sizeof(orc_cand));
    int64_t nb = cols / 16;
    int nrows = cfg->block16x16 ? 16 : 1;
    for (int64_t r0 = 0; r0 < rows; r0 += nrows) {
        /* 16x16 with a per-row amax: the tile uses its first row's amax (R14). */
        float S = orc_global_scale(row_amax[r0], cfg->bound);
        int live = row_live ? row_live[r0] : 1;
        for (int64_t j = 0; j < nb; ++j) {
            int64_t sidx = (r0 / nrows) * nb + j;
            if (!live) { /* grouped tail: zero codes and zero scales (R12) */
                if (scales) scales[sidx] = 0;
                for (int rr = 0; rr < nrows; ++rr) {
                    if (codes) memset(codes + (r0 + rr) * (cols / 2) + 8 * j, 0, 8);
                    if (qdq_out)
                        for (int i = 0; i < 16; ++i)
                            store_out(qdq_out, out_kind, (r0 + rr) * cols + 16 * j + i, 0.0f);
                }
                if (err6) err6[sidx] = 0.0f;
                if (err4) err4[sidx] = 0.0f;
                continue;
            }
            const float* xb = x + r0 * cols + 16 * j;
            const orc_cand* sel = encode_block(xb, nrows, cols, S, cfg, c6, c4,
                                               err6 ? err6 + sidx : NULL,
                                               err4 ? err4 + sidx : NULL);
            if (scales) scales[sidx] = (uint8_t)sel->sc_code;
            for (int rr = 0; rr < nrows; ++rr) {
                if (codes) {
                    uint8_t* cb = codes + (r0 + rr) * (cols / 2) + 8 * j;
                    for (int p = 0; p < 8; ++p) /* R11: even element in the low nibble */
                        cb[p] = (uint8_t)(sel->q[rr * 16 + 2 * p] | (sel->q[rr * 16 + 2 * p + 1] << 4));
                }
                if (qdq_out) {
                    for (int i = 0; i < 16; ++i) {
                        float v = orc_e2m1_value(sel->q[rr * 16 + i]) * sel->d;
                        store_out(qdq_out, out_kind, (r0 + rr) * cols + 16 * j + i, v);
                    }
                }
            }
        }
    }
    free(c6);
    free(c4);
}

static int check_shape(int64_t rows, int64_t cols, const orc_config* cfg)
{
    if (rows < 0 || cols < 0 || cols % 16 != 0) return ORC_BAD;
    if (cfg->block16x16 && rows % 16 != 0) return ORC_BAD;
    if (cfg->bound != 448 && cfg->bound != 256) return ORC_BAD;
    if (cfg->seq_order && cfg->block16x16) return ORC_BAD; /* R16: 1x16 only */
    return ORC_OK;
}

/* Expand the amax argument (tensor: [1], row-scaled: [rows]) to per-row,
 * computing and writing it first when it is not an input. */
static float* per_row_amax(const float* x, int64_t rows, int64_t cols, const orc_config* cfg,
                           float* amax)
{
    float* ra = (float*)malloc(sizeof(float) * (size_t)(rows > 0 ? rows : 1));
    if (cfg->row_scaled) {
        if (!cfg->amax_is_input) orc_amax_rows(x, rows, cols, amax);
        for (int64_t r = 0; r < rows; ++r) ra[r] = amax[r];
    } else {
        if (!cfg->amax_is_input) orc_amax_tensor(x, rows * cols, amax);
        for (int64_t r = 0; r < rows; ++r) ra[r] = amax[0];
    }
    return ra;
}

int orc_quantize(const float* x, int64_t rows, int64_t cols, const orc_config* cfg, float* amax,
                 uint8_t* codes, uint8_t* scales, float* err6, float* err4)
{
    if (check_shape(rows, cols, cfg)) return ORC_BAD;
    float* ra = per_row_amax(x, rows, cols, cfg, amax);
    quantize_rows(x, rows, cols, cfg, ra, NULL, codes, scales, err6, err4, NULL, 0);
    free(ra);
    return ORC_OK;
}

/* Fused quantize-dequantize: codes and scales are not stored; each value is
 * the selected candidate's decode v * d rounded once to the output type. */
int orc_qdq(const float* x, int64_t rows, int64_t cols, const orc_config* cfg, float* amax,
            void* out, int out_kind)
{
    if (check_shape(rows, cols, cfg)) return ORC_BAD;
    float* ra = per_row_amax(x, rows, cols, cfg, amax);
    quantize_rows(x, rows, cols, cfg, ra, NULL, NULL, NULL, NULL, NULL, out, out_kind);
    free(ra);
    return ORC_OK;
}

int orc_quantize_grouped(const float* x, int64_t rows, int64_t cols, const int32_t* offs, int G,
                         const orc_config* cfg, float* group_amax, uint8_t* codes,
                         uint8_t* scales)
{
    if (check_shape(rows, cols, cfg) || G < 0) return ORC_BAD;
    if (!cfg->amax_is_input) orc_amax_groups(x, rows, cols, offs, G, group_amax);
    int64_t* ends = (int64_t*)malloc(sizeof(int64_t) * (size_t)(G > 0 ? G : 1));
    group_ends(offs, G, rows, ends);
    float* ra = (float*)malloc(sizeof(float) * (size_t)(rows > 0 ? rows : 1));
    uint8_t* live = (uint8_t*)malloc((size_t)(rows > 0 ? rows : 1));
    int g = 0;
    for (int64_t r = 0; r < rows; ++r) {
        while (g < G && r >= ends[g]) ++g;
        live[r] = (g < G) ? 1 : 0;
        ra[r] = (g < G) ? group_amax[g] : 0.0f;
    }
    quantize_rows(x, rows, cols, cfg, ra, live, codes, scales, NULL, NULL, NULL, 0);
    free(live);
    free(ra);
    free(ends);
    return ORC_OK;
}

/* Standard NVFP4 decode (recipe-agnostic): out = v * (sigma / S), rounded to
 * the output type.  S is recomputed from amax and the bound as in quantize. */
int orc_dequantize(const uint8_t* codes, const uint8_t* scales, const float* amax, int64_t rows,
                   int64_t cols, const orc_config* cfg, void* out, int out_kind)
{
    if (check_shape(rows, cols, cfg)) return ORC_BAD;
    int64_t nb = cols / 16;
    int nrows = cfg->block16x16 ? 16 : 1;
    for (int64_t r = 0; r < rows; ++r) {
        int64_t r0 = r - (r % nrows);
        float S = orc_global_scale(cfg->row_scaled ? amax[r0] : amax[0], cfg->bound);
        for (int64_t j = 0; j < nb; ++j) {
            float sigma = orc_e4m3_value(scales[(r0 / nrows) * nb + j]);
            float d = (sigma == 0.0f) ? 0.0f : sigma / S;
            for (int i = 0; i < 16; ++i) {
                uint8_t byte = codes[r * (cols / 2) + 8 * j + i / 2];
                uint32_t q = (i & 1) ? (byte >> 4) : (byte & 0xFu);
                store_out(out, out_kind, r * cols + 16 * j + i, orc_e2m1_value(q) * d);
            }
        }
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------- */
/* Element-wise access to the format conversions, for the format pins.       */
/* ------------------------------------------------------------------------- */
void orc_e2m1_encode_array(const float* in, uint8_t* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = (uint8_t)orc_e2m1_encode(in[i]);
}
void orc_e4m3_encode_array(const float* in, uint8_t* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = (uint8_t)orc_e4m3_encode(in[i]);
}
void orc_f16_round_array(const float* in, float* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = orc_f16_round(in[i]);
}
void orc_bf16_round_array(const float* in, float* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = orc_bf16_round(in[i]);
}
void orc_f16_bits_array(const float* in, uint16_t* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = orc_f16_bits(in[i]);
}
void orc_bf16_bits_array(const float* in, uint16_t* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = orc_bf16_bits(in[i]);
}

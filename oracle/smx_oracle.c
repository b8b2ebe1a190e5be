/*
 * smx_oracle.c -- CPU oracle for the sparse MXFP4 attention decode step.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE: only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load or call it. It shares nothing with the CUDA
 * library. Build: gcc -O2 -std=c11 -fopenmp -ffp-contract=off (no fast-math, no FMA
 * contraction, so x86-64 and aarch64 hosts produce the same bits).
 *
 * Sources are named in smx_oracle.h. Each function cites the passage it follows and
 * lists the readings taken where the pages are silent.
 */
#define _GNU_SOURCE
#include "smx_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------------------
 * Element formats
 * ------------------------------------------------------------------------------------ */

/* [OCP-MX] E2M1: bit 3 = sign, bits 2..1 = exponent (bias 1), bit 0 = mantissa.
 * Magnitudes of codes 0..7, written out from the spec's value table. */
static const double E2M1_MAG[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

double orc_e2m1_value(int nibble) {
    double m = E2M1_MAG[nibble & 7];
    return (nibble & 8) ? -m : m;
}

/* [OCP-MX] E8M0 scale: 2^(e-127); 0xFF encodes NaN. */
double orc_e8m0_value(int byte) {
    byte &= 0xFF;
    if (byte == 0xFF) return NAN;
    return ldexp(1.0, byte - 127);
}

/* [OCP-FP8] E4M3 ("fn" variant): bias 7, exponent field 0 is subnormal (m * 2^-9),
 * S.1111.111 is NaN, no infinities; the largest finite magnitude is 448 (0x7E). */
double orc_e4m3_value(int byte) {
    byte &= 0xFF;
    int s = byte >> 7, e = (byte >> 3) & 15, m = byte & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m, -9);
    else v = ldexp(1.0 + m / 8.0, e - 7);
    return s ? -v : v;
}

/* bf16 = the upper 16 bits of an IEEE binary32. */
double orc_bf16_value(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* Nearest E2M1 magnitude to |v|, ties to the even code (mantissa bit 0), |v| >= 6
 * saturates to 6; the sign bit is the sign of v, so a negative value that rounds to zero
 * gives 0x8 (-0).
 * Reading: [ATOM-2812] writes pages with a round-to-nearest packed fp4 conversion; the
 * plainest reading of that and of [OCP-MX]'s conversion rules is RNE with saturation. The
 * thresholds are the midpoints between neighbouring magnitudes. */
uint8_t orc_e2m1_encode(double v) {
    uint8_t sign = signbit(v) ? 0x8 : 0x0;
    double a = fabs(v);
    int code;
    if (a <= 0.25) code = 0;        /* tie 0.25 -> 0 (even)   */
    else if (a < 0.75) code = 1;    /* 0.5                    */
    else if (a <= 1.25) code = 2;   /* 1.0; ties 0.75, 1.25   */
    else if (a < 1.75) code = 3;    /* 1.5                    */
    else if (a <= 2.5) code = 4;    /* 2.0; ties 1.75, 2.5    */
    else if (a < 3.5) code = 5;     /* 3.0                    */
    else if (a <= 5.0) code = 6;    /* 4.0; ties 3.5, 5.0     */
    else code = 7;                  /* 6.0, saturating        */
    return (uint8_t)(sign | code);
}

/* Nearest E4M3 value to a finite v with |v| <= 448, ties to the even mantissa.
 * The quantum of the binade [2^E, 2^(E+1)) is 2^(E-3) for normal numbers (E >= -6) and
 * 2^-9 below; v / quantum is exact in fp64 and nearbyint() rounds it half-to-even. */
uint8_t orc_e4m3_encode(double v) {
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs(v);
    int ex, E, qexp, m;
    double n, r;
    if (a == 0.0) return sign;
    frexp(a, &ex);
    E = ex - 1;
    qexp = (E < -6) ? -9 : E - 3;
    n = nearbyint(ldexp(a, -qexp));
    r = ldexp(n, qexp);
    if (r == 0.0) return sign;
    frexp(r, &ex);
    E = ex - 1;
    if (E < -6) return (uint8_t)(sign | (int)ldexp(r, 9));      /* subnormal: m * 2^-9 */
    m = (int)(ldexp(r, -E) * 8.0) - 8;                          /* 1.m * 2^E           */
    return (uint8_t)(sign | ((E + 7) << 3) | m);
}

/* ------------------------------------------------------------------------------------
 * Quantisers
 * ------------------------------------------------------------------------------------ */

/* One 128-element row to MXFP4: four groups of 32 elements, each with an E8M0 scale.
 * [ATOM-2812] commit "--index-cache-dtype mxfp4": the index-K row store (E8M0 group scale +
 * packed fp4 conversion); commit "MXFP4 main KV": K and V use the same row store.
 * Scale rule of the benchmark workloads: scale = 2^(floor(log2 amax) - 2).
 *   se = floor(log2 amax) - 2, clamped to the E8M0 range [-127, 127]; byte = se + 127.
 *   element code = E2M1 nearest to x / 2^se (x / 2^se is exact in fp64).
 * Readings (silent on the pages): amax == 0 -> se = 0 (byte 127); a group holding a NaN or
 * an infinity -> scale byte 0xFF (NaN) and all its nibbles 0. Nibble packing: element 2i in
 * the low nibble of byte i, element 2i+1 in the high nibble. */
void orc_mxfp4_quant_row(const float* x, uint8_t* nib64, uint8_t* scale4) {
    uint8_t codes[ORC_D];
    for (int g = 0; g < ORC_D / ORC_GROUP; ++g) {
        const float* xg = x + g * ORC_GROUP;
        int nonfinite = 0;
        double amax = 0.0;
        for (int i = 0; i < ORC_GROUP; ++i) {
            if (!isfinite(xg[i])) nonfinite = 1;
            else if (fabs((double)xg[i]) > amax) amax = fabs((double)xg[i]);
        }
        if (nonfinite) {
            scale4[g] = 0xFF;
            for (int i = 0; i < ORC_GROUP; ++i) codes[g * ORC_GROUP + i] = 0;
            continue;
        }
        int se = 0;
        if (amax > 0.0) {
            int ex;
            frexp(amax, &ex);          /* amax = f * 2^ex, f in [0.5, 1) */
            se = (ex - 1) - 2;         /* floor(log2 amax) - 2 */
            if (se < -127) se = -127;
            if (se > 127) se = 127;
        }
        scale4[g] = (uint8_t)(se + 127);
        for (int i = 0; i < ORC_GROUP; ++i)
            codes[g * ORC_GROUP + i] = orc_e2m1_encode(ldexp((double)xg[i], -se));
    }
    for (int i = 0; i < ORC_D / 2; ++i)
        nib64[i] = (uint8_t)(codes[2 * i] | (codes[2 * i + 1] << 4));
}

/* One 128-element row to e4m3 codes with one fp32 scale (FP8-KV workload: "one fp32 scale
 * per token row (scale = amax/448)"; [ATOM-2686] Summary: FP8 KV cache).
 *   s = fl32(amax / 448) (fp32 division); code_i = E4M3 nearest to fl32(x_i / s),
 *   saturated to +-448.
 * Readings: amax == 0 -> s = 1.0; a row holding a NaN or an infinity -> s = NaN and every
 * code 0x7F (NaN). */
void orc_e4m3rs_quant_row(const float* x, uint8_t* codes128, float* scale) {
    float amax = 0.0f;
    int nonfinite = 0;
    for (int i = 0; i < ORC_D; ++i) {
        if (!isfinite(x[i])) nonfinite = 1;
        else if (fabsf(x[i]) > amax) amax = fabsf(x[i]);
    }
    if (nonfinite) {
        *scale = NAN;
        for (int i = 0; i < ORC_D; ++i) codes128[i] = 0x7F;
        return;
    }
    float s = (amax == 0.0f) ? 1.0f : amax / 448.0f;
    for (int i = 0; i < ORC_D; ++i) {
        float y = x[i] / s;
        double yd = (double)y;
        if (yd > 448.0) yd = 448.0;
        if (yd < -448.0) yd = -448.0;
        codes128[i] = orc_e4m3_encode(yd);
    }
    *scale = s;
}

/* One 128-element row to NVFP4 with the per-tensor decode scale g ([NVFP4]): eight blocks of
 * 16 elements, each with an E4M3 scale byte; a value decodes as E2M1(code) x E4M3(byte) x g.
 * Readings (the pages name the format only):
 *   s = amax / (6 g), with 6 g and the quotient each rounded to fp32 (round to nearest even);
 *   byte = E4M3 nearest to min(s, 448), ties to even (0 when s rounds to zero);
 *   S = E4M3(byte) x g rounded to fp32; y_i = x_i / S rounded to fp32;
 *   code_i = E2M1 nearest to y_i (orc_e2m1_encode: ties to even, saturating at 6, sign kept).
 * The arithmetic is fp32 because the codes are decided by it: the quantiser of the kernel
 * computes in fp32 and the pages fix no other precision. A block whose scale byte is 0 (amax
 * 0, or below half the smallest E4M3 subnormal times 6 g) stores codes 0; a block holding a NaN
 * or an infinity stores byte 0x7F (E4M3 NaN) and codes 0. Nibble packing as MXFP4. */
void orc_nvfp4_quant_row(const float* x, float g, uint8_t* nib64, uint8_t* scale8) {
    uint8_t codes[ORC_D];
    volatile float six_g = 6.0f * g;   /* volatile: one fp32 rounding, no contraction */
    for (int blk = 0; blk < ORC_D / ORC_NV_BLOCK; ++blk) {
        const float* xb = x + blk * ORC_NV_BLOCK;
        int nonfinite = 0;
        float amax = 0.0f;
        for (int i = 0; i < ORC_NV_BLOCK; ++i) {
            if (!isfinite(xb[i])) nonfinite = 1;
            else if (fabsf(xb[i]) > amax) amax = fabsf(xb[i]);
        }
        if (nonfinite) {
            scale8[blk] = 0x7F;
            for (int i = 0; i < ORC_NV_BLOCK; ++i) codes[blk * ORC_NV_BLOCK + i] = 0;
            continue;
        }
        volatile float s = amax / six_g;
        double sc = (double)s;
        if (sc > 448.0) sc = 448.0;
        uint8_t byte = orc_e4m3_encode(sc);
        scale8[blk] = byte;
        volatile float S = (float)orc_e4m3_value(byte) * g;
        for (int i = 0; i < ORC_NV_BLOCK; ++i) {
            if (S == 0.0f) {
                codes[blk * ORC_NV_BLOCK + i] = 0;
                continue;
            }
            volatile float y = xb[i] / S;
            codes[blk * ORC_NV_BLOCK + i] = orc_e2m1_encode((double)y);
        }
    }
    for (int i = 0; i < ORC_D / 2; ++i)
        nib64[i] = (uint8_t)(codes[2 * i] | (codes[2 * i + 1] << 4));
}

/* q packing. [ATOM-2812] commit "e4m3 q_out convention": q is written as e4m3 at unit
 * scale, saturating, from the f32 elements; commit "pack_q_e4m3": in-range values are
 * torch's e4m3 cast, beyond +-448 (infinities too) saturate to +-448, NaN stays NaN.
 * Reading: the NaN byte is the canonical 0x7F whatever the input's sign. */
uint8_t orc_pack_q_one(float x) {
    double v = (double)x;
    if (isnan(v)) return 0x7F;
    if (v > 448.0) v = 448.0;
    if (v < -448.0) v = -448.0;
    return orc_e4m3_encode(v);
}

void orc_pack_q_e4m3(const float* q, uint8_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_pack_q_one(q[i]);
}

/* ------------------------------------------------------------------------------------
 * Page rows.
 * MXFP4 page (8704 B, [ATOM-2812] "8704 B MXFP4 page"; 68 B per 128-dim row):
 *   bytes [0, 8192)    : 128 token rows x 64 B of nibbles, token-major;
 *   bytes [8192, 8704) : 128 token rows x 4 E8M0 bytes; group g of slot s at 8192 + 4s + g.
 * Reading: the pages give the sizes and "a 16 B key load and a dword of e8m0 scales", not
 * the byte order; this split layout keeps the nibble rows 16-byte aligned.
 * E4M3 row-scale page (16896 B): 128 x 128 B codes, then 128 fp32 scales (little-endian).
 * ------------------------------------------------------------------------------------ */

void orc_mxfp4_store_row(uint8_t* page, int slot, const uint8_t* nib64, const uint8_t* scale4) {
    memcpy(page + (size_t)slot * 64, nib64, 64);
    memcpy(page + 8192 + (size_t)slot * 4, scale4, 4);
}

void orc_mxfp4_load_row(const uint8_t* page, int slot, double* out128) {
    const uint8_t* nib = page + (size_t)slot * 64;
    const uint8_t* sc = page + 8192 + (size_t)slot * 4;
    for (int d = 0; d < ORC_D; ++d) {
        int byte = nib[d / 2];
        int code = (d % 2 == 0) ? (byte & 0xF) : (byte >> 4);
        out128[d] = orc_e2m1_value(code) * orc_e8m0_value(sc[d / ORC_GROUP]);
    }
}

void orc_e4m3rs_store_row(uint8_t* page, int slot, const uint8_t* codes128, float scale) {
    memcpy(page + (size_t)slot * 128, codes128, 128);
    memcpy(page + 16384 + (size_t)slot * 4, &scale, 4);
}

void orc_e4m3rs_load_row(const uint8_t* page, int slot, double* out128) {
    float s;
    memcpy(&s, page + 16384 + (size_t)slot * 4, 4);
    for (int d = 0; d < ORC_D; ++d) out128[d] = orc_e4m3_value(page[(size_t)slot * 128 + d]) * (double)s;
}

/* NVFP4 page (9216 B; reading, the pages give none): bytes [0, 8192) the 128 token rows x 64 B
 * of nibbles as MXFP4; bytes [8192, 9216) the 128 token rows x 8 E4M3 block scales, block j of
 * slot s at 8192 + 8 s + j. The per-tensor scale g lives with the pool, not in its pages. */
void orc_nvfp4_store_row(uint8_t* page, int slot, const uint8_t* nib64, const uint8_t* scale8) {
    memcpy(page + (size_t)slot * 64, nib64, 64);
    memcpy(page + 8192 + (size_t)slot * 8, scale8, 8);
}

void orc_nvfp4_load_row(const uint8_t* page, int slot, float g, double* out128) {
    const uint8_t* nib = page + (size_t)slot * 64;
    const uint8_t* sc = page + 8192 + (size_t)slot * 8;
    for (int d = 0; d < ORC_D; ++d) {
        int byte = nib[d / 2];
        int code = (d % 2 == 0) ? (byte & 0xF) : (byte >> 4);
        out128[d] = orc_e2m1_value(code) * orc_e4m3_value(sc[d / ORC_NV_BLOCK]) * (double)g;
    }
}

static size_t kv_page_bytes(const orc_shape* sh) {
    if (sh->kv_format == ORC_KV_NVFP4) return ORC_NVFP4_PAGE_BYTES;
    return sh->kv_format == ORC_KV_E4M3_ROWSCALE ? ORC_E4M3RS_PAGE_BYTES : ORC_MXFP4_PAGE_BYTES;
}

static size_t idx_page_bytes(const orc_shape* sh) {
    return sh->idx_format == ORC_KV_NVFP4 ? ORC_NVFP4_PAGE_BYTES : ORC_MXFP4_PAGE_BYTES;
}

/* K/V pools hold [n_pool_pages][Hkv][page]; the index pool holds [n_pool_pages][page]. */
static uint8_t* kv_page(const orc_shape* sh, uint8_t* pool, int64_t phys, int kvh) {
    return pool + ((size_t)phys * sh->Hkv + kvh) * kv_page_bytes(sh);
}

/* g: the pool's NVFP4 scale (K or V). */
static void store_kv_row(const orc_shape* sh, uint8_t* page, int slot, const float* x, float g) {
    if (sh->kv_format == ORC_KV_E4M3_ROWSCALE) {
        uint8_t codes[ORC_D];
        float s;
        orc_e4m3rs_quant_row(x, codes, &s);
        orc_e4m3rs_store_row(page, slot, codes, s);
    } else if (sh->kv_format == ORC_KV_NVFP4) {
        uint8_t nib[64], sc[8];
        orc_nvfp4_quant_row(x, g, nib, sc);
        orc_nvfp4_store_row(page, slot, nib, sc);
    } else {
        uint8_t nib[64], sc[4];
        orc_mxfp4_quant_row(x, nib, sc);
        orc_mxfp4_store_row(page, slot, nib, sc);
    }
}

static void load_kv_row(const orc_shape* sh, const uint8_t* page, int slot, float g, double* out) {
    if (sh->kv_format == ORC_KV_E4M3_ROWSCALE) orc_e4m3rs_load_row(page, slot, out);
    else if (sh->kv_format == ORC_KV_NVFP4) orc_nvfp4_load_row(page, slot, g, out);
    else orc_mxfp4_load_row(page, slot, out);
}

/* The index pool's rows: MXFP4, or NVFP4 with the index scale. */
static void store_idx_row(const orc_shape* sh, uint8_t* idx_pool, int64_t phys, int slot, const float* x) {
    if (sh->idx_format == ORC_KV_NVFP4) {
        uint8_t nib[64], sc[8];
        orc_nvfp4_quant_row(x, sh->nv_scale_idx, nib, sc);
        orc_nvfp4_store_row(idx_pool + (size_t)phys * ORC_NVFP4_PAGE_BYTES, slot, nib, sc);
    } else {
        uint8_t nib[64], sc[4];
        orc_mxfp4_quant_row(x, nib, sc);
        orc_mxfp4_store_row(idx_pool + (size_t)phys * ORC_MXFP4_PAGE_BYTES, slot, nib, sc);
    }
}

/* Insert of token position pos of row b: index-K row, and K and V rows of every KV head. */
static void insert_token(const orc_shape* sh, int b, int64_t pos, const float* k_row,
                         const float* v_row, const float* kidx_row, const int32_t* page_table,
                         uint8_t* k_pool, uint8_t* v_pool, uint8_t* idx_pool) {
    int64_t p = pos / ORC_PAGE;
    int slot = (int)(pos % ORC_PAGE);
    int64_t phys;
    if (pos < 0 || p >= sh->max_pages) return;
    phys = page_table[(size_t)b * sh->max_pages + p];
    if (phys < 0 || phys >= sh->n_pool_pages) return;
    if (kidx_row && idx_pool)   /* a layer without an index cache writes K and V only */
        store_idx_row(sh, idx_pool, phys, slot, kidx_row);
    for (int h = 0; h < sh->Hkv; ++h) {
        store_kv_row(sh, kv_page(sh, k_pool, phys, h), slot, k_row + (size_t)h * ORC_D, sh->nv_scale_k);
        store_kv_row(sh, kv_page(sh, v_pool, phys, h), slot, v_row + (size_t)h * ORC_D, sh->nv_scale_v);
    }
}

/* a1: the Q new tokens of row b sit at positions ctx_len[b] - Q + t, t in [0, Q)
 * ([ATOM-2812] K1 index-K insert and K/V insert; ctx_len counts the new tokens).
 * k_new, v_new: [B][Q][Hkv][128]; kidx_new: [B][Q][128], or NULL (with idx_pool NULL) for a
 * layer without an index cache: K and V rows only. */
void orc_kv_insert(const orc_shape* sh, const float* k_new, const float* v_new,
                   const float* kidx_new, const int32_t* page_table, const int32_t* ctx_len,
                   uint8_t* k_pool, uint8_t* v_pool, uint8_t* idx_pool) {
    for (int b = 0; b < sh->B; ++b)
        for (int t = 0; t < sh->Q; ++t) {
            size_t r = (size_t)b * sh->Q + t;
            insert_token(sh, b, (int64_t)ctx_len[b] - sh->Q + t,
                         k_new + r * sh->Hkv * ORC_D, v_new + r * sh->Hkv * ORC_D,
                         kidx_new ? kidx_new + r * ORC_D : NULL, page_table, k_pool, v_pool, idx_pool);
        }
}

/* Bulk fill used to build test pools: positions [0, n_fill[b]) of row b from dense
 * k, v: [B][T][Hkv][128] and kidx: [B][T][128]. Same row store as the insert. */
void orc_kv_fill(const orc_shape* sh, const float* k, const float* v, const float* kidx,
                 int64_t T, const int32_t* page_table, const int32_t* n_fill,
                 uint8_t* k_pool, uint8_t* v_pool, uint8_t* idx_pool) {
    for (int b = 0; b < sh->B; ++b) {
        int64_t n = n_fill[b];
#pragma omp parallel for schedule(static)
        for (int64_t pos = 0; pos < n; ++pos) {
            size_t r = (size_t)b * T + pos;
            insert_token(sh, b, pos, k + r * sh->Hkv * ORC_D, v + r * sh->Hkv * ORC_D,
                         kidx + r * ORC_D, page_table, k_pool, v_pool, idx_pool);
        }
    }
}

/* ------------------------------------------------------------------------------------
 * a3 index score: [ATOM-2812] commit "--index-cache-dtype mxfp4": the scorer reads the MXFP4
 * index pages and scores blocks with the bf16 index query. Page score rule of the benchmark
 * workloads: max over the page's tokens of q_idx . k_idx (no softmax scale, no activation).
 * Readings: selection is per row, shared by the row's Q query tokens, so
 *   S_p = max over t in [0,Q), tokens j of page p with j < ctx_len and j <= pos_t,
 *         pos_t = ctx_len - Q + t (causal within the Q draft tokens),
 * of sum_d qidx[t][d] * deq(kidx[j][d]) in fp64. A token score that is NaN is left out of the
 * max. Pages p >= ceil(ctx_len/128) get -inf.
 * qidx: bf16 bits [B][Q][128]; scores: [B][max_pages].
 * ------------------------------------------------------------------------------------ */
static int64_t n_pages_of(const orc_shape* sh, int32_t ctx) {
    int64_t n = ((int64_t)ctx + ORC_PAGE - 1) / ORC_PAGE;
    if (n < 0) n = 0;
    if (n > sh->max_pages) n = sh->max_pages;
    return n;
}

void orc_index_scores(const orc_shape* sh, const uint16_t* qidx_bf16, const uint8_t* idx_pool,
                      const int32_t* page_table, const int32_t* ctx_len, double* scores) {
    int64_t total = (int64_t)sh->B * sh->max_pages;
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t bp = 0; bp < total; ++bp) {
        int b = (int)(bp / sh->max_pages);
        int64_t p = bp % sh->max_pages;
        int64_t ctx = ctx_len[b];
        double best = -INFINITY;
        double krow[ORC_D];
        if (p >= n_pages_of(sh, ctx_len[b])) {
            scores[bp] = -INFINITY;
            continue;
        }
        int64_t phys = page_table[bp];
        const uint8_t* page = idx_pool + (size_t)phys * idx_page_bytes(sh);
        for (int slot = 0; slot < ORC_PAGE; ++slot) {
            int64_t j = p * ORC_PAGE + slot;
            if (j >= ctx) break;
            if (sh->idx_format == ORC_KV_NVFP4) orc_nvfp4_load_row(page, slot, sh->nv_scale_idx, krow);
            else orc_mxfp4_load_row(page, slot, krow);
            for (int t = 0; t < sh->Q; ++t) {
                int64_t pos_t = ctx - sh->Q + t;
                if (j > pos_t) continue;
                const uint16_t* qt = qidx_bf16 + ((size_t)b * sh->Q + t) * ORC_D;
                double s = 0.0;
                for (int d = 0; d < ORC_D; ++d) s += orc_bf16_value(qt[d]) * krow[d];
                if (isnan(s)) continue;
                if (s > best) best = s;
            }
        }
        scores[bp] = best;
    }
}

/* a4 top-k: [ATOM-2812] commit "MXFP4 main KV": the selected blocks (one page-128 page each)
 * fill the row's sparse table. k_eff = min(k, ceil(ctx_len/128)) pages with the largest
 * score. Readings: ties go to the lower page id, NaN ranks below every number, no page is
 * forced in; the list is the logical page ids in ascending order, padded with -1.
 * Plain definition: page p is selected iff fewer than k_eff pages beat it. */
static int beats(double sa, int64_t a, double sb, int64_t b) {
    int na = isnan(sa), nb = isnan(sb);
    if (na || nb) {
        if (na && nb) return a < b;
        return nb;      /* a number beats NaN */
    }
    if (sa > sb) return 1;
    if (sa < sb) return 0;
    return a < b;
}

/* Pages per selected block ([ATOM-2812] commit "MXFP4 main KV": a selected block is one page of
 * the sparse table, PAGES_PER_BLOCK a build parameter). Reading for blocks of several pages: a
 * block's score is the max of its pages' scores (NaN left out, as for tokens), the top-k ranks
 * blocks with the same rule as pages, and the split stage takes every page of a selected block
 * that lies in the row. */
static int ppb_of(const orc_shape* sh) { return sh->pages_per_block > 1 ? sh->pages_per_block : 1; }

void orc_topk(const orc_shape* sh, const double* scores, const int32_t* ctx_len,
              int32_t* topk_pages, int32_t* topk_count) {
    const int ppb = ppb_of(sh);
    for (int b = 0; b < sh->B; ++b) {
        int64_t n = n_pages_of(sh, ctx_len[b]);
        int64_t nb = (n + ppb - 1) / ppb;
        int64_t k_eff = sh->topk < nb ? sh->topk : nb;
        const double* s = scores + (size_t)b * sh->max_pages;
        int32_t* out = topk_pages + (size_t)b * sh->topk;
        double* bs = (double*)malloc((size_t)(nb > 0 ? nb : 1) * sizeof(double));
        for (int64_t blk = 0; blk < nb; ++blk) {
            double m = NAN;
            for (int64_t p = blk * ppb; p < (blk + 1) * ppb && p < n; ++p)
                if (!isnan(s[p]) && (isnan(m) || s[p] > m)) m = s[p];
            bs[blk] = m;
        }
        int c = 0;
        for (int64_t p = 0; p < nb; ++p) {
            int64_t rank = 0;
            for (int64_t o = 0; o < nb; ++o)
                if (o != p && beats(bs[o], o, bs[p], p)) ++rank;
            if (rank < k_eff) out[c++] = (int32_t)p;
        }
        free(bs);
        for (int i = c; i < sh->topk; ++i) out[i] = -1;
        topk_count[b] = c;
    }
}

/* ------------------------------------------------------------------------------------
 * a5 split stage: [ATOM-2812] commit "MXFP4 main KV": per partition, QK over the selected
 * pages (K fp4 with its E8M0 group scale against the e4m3 q), softmax, PV, written as
 * (sp_o, sp_m, sp_l). For query (b, t, h): KV head h / (Hq / Hkv); tokens
 *   T = { j : page(j) selected, j < ctx_len, j <= pos_t };
 *   z_j = (sum_d q[d] K_j[d]) / sqrt(128), fp64.
 * Readings: partition s of S takes positions [floor(s k_eff / S), floor((s+1) k_eff / S)) of
 * the ascending list (S > k_eff gives empty partitions); with blocks of several pages an entry is
 * a block id and stands for the block's pages in the row; m is kept in the log2 domain,
 *   m_s = max_j z_j log2(e),  l_s = sum_j 2^(z_j log2(e) - m_s),
 *   o_s = sum_j 2^(z_j log2(e) - m_s) V_j      (unnormalised);
 * a partition with no token stores m = -inf, l = 0, o = 0.
 * q: e4m3 bytes [B][Q][Hq][128] for MXFP4 K/V, bf16 bits for the e4m3 row-scale K/V
 * ([ATOM-2812] commit "e4m3 q_out convention": fp8-KV keeps bf16 q).
 * part_o: [B][S][Q][Hq][128]; part_m, part_l: [B][S][Q][Hq].
 * ------------------------------------------------------------------------------------ */
static double q_elem(const orc_shape* sh, const void* q, size_t idx) {
    if (sh->kv_format == ORC_KV_E4M3_ROWSCALE) return orc_bf16_value(((const uint16_t*)q)[idx]);
    return orc_e4m3_value(((const uint8_t*)q)[idx]);
}

void orc_sparse_attn_split(const orc_shape* sh, const void* q, const uint8_t* k_pool,
                           const uint8_t* v_pool, const int32_t* page_table,
                           const int32_t* ctx_len, const int32_t* topk_pages,
                           const int32_t* topk_count, double* part_o, double* part_m,
                           double* part_l) {
    const int S = sh->num_splits, G = sh->Hq / sh->Hkv, ppb = ppb_of(sh);
    const double inv_sqrt_d = 1.0 / sqrt((double)ORC_D);
    int64_t total = (int64_t)sh->B * sh->Q * sh->Hq;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t bth = 0; bth < total; ++bth) {
        int b = (int)(bth / ((int64_t)sh->Q * sh->Hq));
        int t = (int)((bth / sh->Hq) % sh->Q);
        int h = (int)(bth % sh->Hq);
        int kvh = h / G;
        int64_t ctx = ctx_len[b], pos_t = ctx - sh->Q + t;
        int64_t n_row = n_pages_of(sh, ctx_len[b]);
        int k_eff = topk_count[b];
        double qv[ORC_D], krow[ORC_D], vrow[ORC_D];
        size_t qbase = (((size_t)b * sh->Q + t) * sh->Hq + h) * ORC_D;
        for (int d = 0; d < ORC_D; ++d) qv[d] = q_elem(sh, q, qbase + d);
        for (int s = 0; s < S; ++s) {
            int lo = (int)(((int64_t)s * k_eff) / S), hi = (int)(((int64_t)(s + 1) * k_eff) / S);
            size_t pi = (((size_t)b * S + s) * sh->Q + t) * sh->Hq + h;
            double* o = part_o + pi * ORC_D;
            double m = -INFINITY, l = 0.0;
            /* pass 1: the maximum */
            for (int64_t e = (int64_t)lo * ppb; e < (int64_t)hi * ppb; ++e) {
                int64_t p = (int64_t)topk_pages[(size_t)b * sh->topk + e / ppb] * ppb + e % ppb;
                if (p >= n_row) continue;   /* the row's last block may end past its pages */
                int64_t phys = page_table[(size_t)b * sh->max_pages + p];
                const uint8_t* kp = kv_page(sh, (uint8_t*)k_pool, phys, kvh);
                for (int slot = 0; slot < ORC_PAGE; ++slot) {
                    int64_t j = p * ORC_PAGE + slot;
                    if (j >= ctx || j > pos_t) continue;
                    load_kv_row(sh, kp, slot, sh->nv_scale_k, krow);
                    double dot = 0.0;
                    for (int d = 0; d < ORC_D; ++d) dot += qv[d] * krow[d];
                    double y = dot * inv_sqrt_d * M_LOG2E;
                    if (y > m) m = y;
                }
            }
            for (int d = 0; d < ORC_D; ++d) o[d] = 0.0;
            /* pass 2: weights and the weighted sum */
            if (m != -INFINITY) {
                for (int64_t e = (int64_t)lo * ppb; e < (int64_t)hi * ppb; ++e) {
                    int64_t p = (int64_t)topk_pages[(size_t)b * sh->topk + e / ppb] * ppb + e % ppb;
                    if (p >= n_row) continue;
                    int64_t phys = page_table[(size_t)b * sh->max_pages + p];
                    const uint8_t* kp = kv_page(sh, (uint8_t*)k_pool, phys, kvh);
                    const uint8_t* vp = kv_page(sh, (uint8_t*)v_pool, phys, kvh);
                    for (int slot = 0; slot < ORC_PAGE; ++slot) {
                        int64_t j = p * ORC_PAGE + slot;
                        if (j >= ctx || j > pos_t) continue;
                        load_kv_row(sh, kp, slot, sh->nv_scale_k, krow);
                        load_kv_row(sh, vp, slot, sh->nv_scale_v, vrow);
                        double dot = 0.0;
                        for (int d = 0; d < ORC_D; ++d) dot += qv[d] * krow[d];
                        double w = exp2(dot * inv_sqrt_d * M_LOG2E - m);
                        l += w;
                        for (int d = 0; d < ORC_D; ++d) o[d] += w * vrow[d];
                    }
                }
            }
            part_m[pi] = m;
            part_l[pi] = l;
        }
    }
}

/* a6 merge ([ATOM-2812] commit "MXFP4 main KV": sp_o / sp_m / sp_l and the merge):
 *   M = max_s m_s; out = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s; M = -inf -> out = 0.
 * A partition with m_s = -inf has weight 0; -inf - (-inf) is never formed. */
void orc_sparse_attn_merge(const orc_shape* sh, const double* part_o, const double* part_m,
                           const double* part_l, double* out) {
    const int S = sh->num_splits;
    for (int b = 0; b < sh->B; ++b)
        for (int t = 0; t < sh->Q; ++t)
            for (int h = 0; h < sh->Hq; ++h) {
                size_t oi = ((size_t)b * sh->Q + t) * sh->Hq + h;
                double M = -INFINITY;
                for (int s = 0; s < S; ++s) {
                    double m = part_m[(((size_t)b * S + s) * sh->Q + t) * sh->Hq + h];
                    if (m > M) M = m;
                }
                double* o = out + oi * ORC_D;
                for (int d = 0; d < ORC_D; ++d) o[d] = 0.0;
                if (M == -INFINITY) continue;
                double L = 0.0;
                for (int s = 0; s < S; ++s) {
                    size_t pi = (((size_t)b * S + s) * sh->Q + t) * sh->Hq + h;
                    if (part_m[pi] == -INFINITY) continue;
                    double w = exp2(part_m[pi] - M);
                    L += w * part_l[pi];
                    for (int d = 0; d < ORC_D; ++d) o[d] += w * part_o[pi * ORC_D + d];
                }
                for (int d = 0; d < ORC_D; ++d) o[d] /= L;
            }
}

/* The whole step in the pages' order: insert (a1), pack q (a2), index score (a3),
 * top-k (a4), split (a5), merge (a6). Pools are updated in place. q_f32 is used for MXFP4
 * K/V (packed to e4m3 into q_e4m3), q_bf16 for the e4m3 row-scale K/V. Partials may be NULL. */
void orc_decode_step(const orc_shape* sh, const float* q_f32, const uint16_t* q_bf16,
                     const uint16_t* qidx_bf16, const float* k_new, const float* v_new,
                     const float* kidx_new, const int32_t* page_table, const int32_t* ctx_len,
                     uint8_t* k_pool, uint8_t* v_pool, uint8_t* idx_pool, double* scores,
                     int32_t* topk_pages, int32_t* topk_count, uint8_t* q_e4m3,
                     double* part_o, double* part_m, double* part_l, double* out) {
    size_t nq = (size_t)sh->B * sh->Q * sh->Hq * ORC_D;
    size_t np = (size_t)sh->B * sh->num_splits * sh->Q * sh->Hq;
    double *po = part_o, *pm = part_m, *pl = part_l;
    const void* qa;
    orc_kv_insert(sh, k_new, v_new, kidx_new, page_table, ctx_len, k_pool, v_pool, idx_pool);
    if (sh->kv_format == ORC_KV_E4M3_ROWSCALE) {
        qa = q_bf16;
    } else {
        orc_pack_q_e4m3(q_f32, q_e4m3, (int64_t)nq);
        qa = q_e4m3;
    }
    orc_index_scores(sh, qidx_bf16, idx_pool, page_table, ctx_len, scores);
    orc_topk(sh, scores, ctx_len, topk_pages, topk_count);
    if (!po) po = (double*)malloc(np * ORC_D * sizeof(double));
    if (!pm) pm = (double*)malloc(np * sizeof(double));
    if (!pl) pl = (double*)malloc(np * sizeof(double));
    orc_sparse_attn_split(sh, qa, k_pool, v_pool, page_table, ctx_len, topk_pages, topk_count,
                          po, pm, pl);
    orc_sparse_attn_merge(sh, po, pm, pl, out);
    if (po != part_o) free(po);
    if (pm != part_m) free(pm);
    if (pl != part_l) free(pl);
}

/* The step of a layer that reuses an earlier layer's selection ([MiniMax-M3.1] "Enable Mono
 * decode with fixed DSpark verify", the dense_prefix_mono note: an index_topk_freq schedule gives
 * layers that run no indexer and attend over the sparse blocks a previous layer selected).
 * Readings: such a layer has no index cache, so only its K and V rows are inserted (a1 without
 * the index-K row); the selection arrives as the earlier layer's (topk_pages, topk_count): logical
 * page ids of the same rows, ascending, which this layer's page table maps to its own K/V pages;
 * q packing (a2), the split (a5) and the merge (a6) are those of the full step. */
void orc_decode_step_reuse(const orc_shape* sh, const float* q_f32, const uint16_t* q_bf16,
                           const float* k_new, const float* v_new, const int32_t* page_table,
                           const int32_t* ctx_len, uint8_t* k_pool, uint8_t* v_pool,
                           const int32_t* topk_pages, const int32_t* topk_count, uint8_t* q_e4m3,
                           double* part_o, double* part_m, double* part_l, double* out) {
    size_t nq = (size_t)sh->B * sh->Q * sh->Hq * ORC_D;
    size_t np = (size_t)sh->B * sh->num_splits * sh->Q * sh->Hq;
    double *po = part_o, *pm = part_m, *pl = part_l;
    const void* qa;
    orc_kv_insert(sh, k_new, v_new, NULL, page_table, ctx_len, k_pool, v_pool, NULL);
    if (sh->kv_format == ORC_KV_E4M3_ROWSCALE) {
        qa = q_bf16;
    } else {
        orc_pack_q_e4m3(q_f32, q_e4m3, (int64_t)nq);
        qa = q_e4m3;
    }
    if (!po) po = (double*)malloc(np * ORC_D * sizeof(double));
    if (!pm) pm = (double*)malloc(np * sizeof(double));
    if (!pl) pl = (double*)malloc(np * sizeof(double));
    orc_sparse_attn_split(sh, qa, k_pool, v_pool, page_table, ctx_len, topk_pages, topk_count,
                          po, pm, pl);
    orc_sparse_attn_merge(sh, po, pm, pl, out);
    if (po != part_o) free(po);
    if (pm != part_m) free(pm);
    if (pl != part_l) free(pl);
}

void orc_set_threads(int n) {
#ifdef _OPENMP
    omp_set_num_threads(n > 0 ? n : 1);
#else
    (void)n;
#endif
}

int orc_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

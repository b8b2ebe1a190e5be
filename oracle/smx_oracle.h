/*
 * smx_oracle.h -- CPU oracle for the sparse MXFP4 attention decode step.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE. Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load or call this library. The CUDA library shares no
 * code, header, table or helper with it, and neither includes the other.
 *
 * Everything is plain C11 with fp64 arithmetic, except where the method fixes fp32
 * (the e4m3 row-scale quantiser divides in fp32, as its scale rule states). Loops
 * follow the definitions in the order the method states them; OpenMP pragmas only
 * distribute independent outer iterations and never change the arithmetic.
 *
 * Sources (pages the method is described on):
 *   [ATOM-2812]  ROCm/ATOM PR 2812, "Mono decode over the MXFP4 KV and index caches":
 *                commit "--index-cache-dtype mxfp4" (index-K page writer, page scorer),
 *                commit "MXFP4 main KV" (K/V page writer, split stage, merge, PAGES_PER_BLOCK),
 *                commit "e4m3 q_out convention" and commit "pack_q_e4m3" (q packing).
 *   [ATOM-2686]  ROCm/ATOM PR 2686, "Enable Mono decode with fixed DSpark verify":
 *                Summary (fixed 7-draft verify: 8 query tokens per row; FP8 KV cache).
 *   [OCP-MX]     OCP Microscaling Formats (MX) v1.0 (E2M1 element, E8M0 scale).
 *   [OCP-FP8]    OCP 8-bit Floating Point (OFP8) v1.0 (E4M3: bias 7, max 448, no inf).
 *   [NVFP4]      NVIDIA's 4-bit format as the pages name it ([ATOM-2812] PR title "FP4 index
 *                cache and NVFP4 sparse KV cache"; commit "--index-cache-dtype mxfp4": "MXFP4 /
 *                NVFP4 main KV, NVFP4 index ... stay refused"): E2M1 elements, one E4M3 scale
 *                per 16 elements, one fp32 scale per tensor. The pages give no page layout or
 *                rounding rule; the readings are at orc_nvfp4_quant_row.
 * Readings the pages leave open are listed next to each function.
 */
#ifndef SMX_ORACLE_H
#define SMX_ORACLE_H
#include <stdint.h>

#define ORC_D 128            /* head_dim and index dim */
#define ORC_PAGE 128         /* tokens per page */
#define ORC_GROUP 32         /* MX block size */
#define ORC_MXFP4_PAGE_BYTES 8704   /* 128 x 64 B nibbles + 128 x 4 B E8M0 scales */
#define ORC_E4M3RS_PAGE_BYTES 16896 /* 128 x 128 B e4m3 codes + 128 x 4 B fp32 scales */
#define ORC_NV_BLOCK 16             /* NVFP4 block size */
#define ORC_NVFP4_PAGE_BYTES 9216   /* 128 x 64 B nibbles + 128 x 8 B E4M3 block scales */

enum { ORC_KV_MXFP4 = 0, ORC_KV_E4M3_ROWSCALE = 1, ORC_KV_NVFP4 = 2 };

typedef struct {
    int32_t B, Q, Hq, Hkv;
    int32_t max_pages;      /* page-table width per row */
    int64_t n_pool_pages;   /* physical pages in each pool */
    int32_t topk;           /* k (pages) */
    int32_t num_splits;     /* S partitions of the selected list */
    int32_t kv_format;      /* ORC_KV_* for the K/V pools */
    int32_t pages_per_block; /* pages per selected block (0 or 1: one page) */
    int32_t idx_format;     /* ORC_KV_MXFP4 or ORC_KV_NVFP4 for the index pool */
    float nv_scale_k;       /* NVFP4 per-tensor decode scales (fp32, > 0) of the K, V and */
    float nv_scale_v;       /* index pools; unused by the other formats */
    float nv_scale_idx;
} orc_shape;

/* ---- element formats ---- */
double orc_e2m1_value(int nibble);          /* [OCP-MX] 4-bit s.ee.m */
double orc_e8m0_value(int byte);            /* [OCP-MX] 2^(byte-127), 0xFF = NaN */
double orc_e4m3_value(int byte);            /* [OCP-FP8] */
double orc_bf16_value(uint16_t bits);
uint8_t orc_e2m1_encode(double v);          /* nearest E2M1, ties to even code, saturate at 6 */
uint8_t orc_e4m3_encode(double v);          /* nearest E4M3 for finite |v| <= 448, ties to even */

/* ---- quantisers ---- */
void orc_mxfp4_quant_row(const float* x, uint8_t* nib64, uint8_t* scale4);
void orc_e4m3rs_quant_row(const float* x, uint8_t* codes128, float* scale);
void orc_nvfp4_quant_row(const float* x, float g, uint8_t* nib64, uint8_t* scale8);
uint8_t orc_pack_q_one(float x);
void orc_pack_q_e4m3(const float* q, uint8_t* out, int64_t n);

/* ---- page rows ---- */
void orc_mxfp4_store_row(uint8_t* page, int slot, const uint8_t* nib64, const uint8_t* scale4);
void orc_mxfp4_load_row(const uint8_t* page, int slot, double* out128);
void orc_e4m3rs_store_row(uint8_t* page, int slot, const uint8_t* codes128, float scale);
void orc_e4m3rs_load_row(const uint8_t* page, int slot, double* out128);
void orc_nvfp4_store_row(uint8_t* page, int slot, const uint8_t* nib64, const uint8_t* scale8);
void orc_nvfp4_load_row(const uint8_t* page, int slot, float g, double* out128);

/* ---- insert ---- */
void orc_kv_insert(const orc_shape* sh, const float* k_new, const float* v_new,
                   const float* kidx_new, const int32_t* page_table, const int32_t* ctx_len,
                   uint8_t* k_pool, uint8_t* v_pool, uint8_t* idx_pool);
void orc_kv_fill(const orc_shape* sh, const float* k, const float* v, const float* kidx,
                 int64_t T, const int32_t* page_table, const int32_t* n_fill,
                 uint8_t* k_pool, uint8_t* v_pool, uint8_t* idx_pool);

/* ---- index score + top-k ---- */
void orc_index_scores(const orc_shape* sh, const uint16_t* qidx_bf16, const uint8_t* idx_pool,
                      const int32_t* page_table, const int32_t* ctx_len, double* scores);
void orc_topk(const orc_shape* sh, const double* scores, const int32_t* ctx_len,
              int32_t* topk_pages, int32_t* topk_count);

/* ---- split-K attention + merge ---- */
void orc_sparse_attn_split(const orc_shape* sh, const void* q, const uint8_t* k_pool,
                           const uint8_t* v_pool, const int32_t* page_table,
                           const int32_t* ctx_len, const int32_t* topk_pages,
                           const int32_t* topk_count, double* part_o, double* part_m,
                           double* part_l);
void orc_sparse_attn_merge(const orc_shape* sh, const double* part_o, const double* part_m,
                           const double* part_l, double* out);

/* ---- the whole step ---- */
void orc_decode_step(const orc_shape* sh, const float* q_f32, const uint16_t* q_bf16,
                     const uint16_t* qidx_bf16, const float* k_new, const float* v_new,
                     const float* kidx_new, const int32_t* page_table, const int32_t* ctx_len,
                     uint8_t* k_pool, uint8_t* v_pool, uint8_t* idx_pool, double* scores,
                     int32_t* topk_pages, int32_t* topk_count, uint8_t* q_e4m3,
                     double* part_o, double* part_m, double* part_l, double* out);

/* The step of a layer that reuses an earlier layer's selection: K/V insert (no index-K), q
 * packing, split over (topk_pages, topk_count) as given, merge. Same buffers as orc_decode_step. */
void orc_decode_step_reuse(const orc_shape* sh, const float* q_f32, const uint16_t* q_bf16,
                           const float* k_new, const float* v_new, const int32_t* page_table,
                           const int32_t* ctx_len, uint8_t* k_pool, uint8_t* v_pool,
                           const int32_t* topk_pages, const int32_t* topk_count, uint8_t* q_e4m3,
                           double* part_o, double* part_m, double* part_l, double* out);
void orc_set_threads(int n);
int orc_max_threads(void);

#endif

/*
 * smx.h -- C ABI of libsmx: the sparse MXFP4 attention decode step on GB300 (sm_103a).
 *
 * One decode step over a paged, block-scaled KV cache, as described on
 *   [ATOM-2812] ROCm/ATOM PR 2812 "Mono decode over the MXFP4 KV and index caches"
 *               (commit messages "--index-cache-dtype mxfp4", "MXFP4 main KV",
 *               "e4m3 q_out convention", "pack_q_e4m3");
 *   [ATOM-2686] ROCm/ATOM PR 2686 "Enable Mono decode with fixed DSpark verify" (Summary:
 *               fixed 7-draft verify = 8 query tokens per row, FP8 KV cache).
 * The step: insert the new tokens' index-K, K and V rows into their pages (a1); pack q to
 * saturating e4m3 (a2); score every page of each row with the index query (a3); select the
 * top-k pages (a4); split-K attention over the selected pages (a5); merge the partials (a6).
 *
 * Conventions for every entry point
 *  - All array pointers are DEVICE pointers owned by the caller; nothing is allocated, freed
 *    or synchronised. Work is enqueued on `stream` (NULL = the legacy default stream) and
 *    runs asynchronously; the return code reports argument checks and launch errors only.
 *  - Return 0 (SMX_OK) or a negative SMX_ERR_* code; nothing is launched when an argument
 *    check fails. Host-side checks never read device memory.
 *  - `dev_status` (nullable) is a device int32 that kernels OR SMX_DEV_* bits into when
 *    device-resident indices are out of range; the offending page/row is skipped (an index
 *    page scores -inf, an attention page contributes nothing), so a bad table can never make
 *    a kernel read or write outside the pools. The caller clears it.
 *  - D (head dim) = Di (index dim) = 128 and page_tokens = 128 are the only supported values.
 *  - Alignment: float and pool arrays 16-byte aligned; idx_pool 32-byte aligned for the calls that
 *    score it (it is read by tensor-map copies of a packed 4-bit type); otherwise
 *    SMX_ERR_INVALID_ARG.
 *
 * Shapes and layouts (row-major, C order):
 *   q_f32     [B][Q][Hq][128] float        q_bf16   [B][Q][Hq][128] bf16 bits (uint16)
 *   qidx_bf16 [B][Q][128] bf16 bits        k_new, v_new [B][Q][Hkv][128] float
 *   kidx_new  [B][Q][128] float            page_table [B][max_pages_per_row] int32 (physical ids)
 *   ctx_len   [B] int32: tokens of the row INCLUDING the Q new ones; query token t sits at
 *             position pos_t = ctx_len - Q + t (causal within the Q draft tokens).
 *   k_pool, v_pool [n_pool_pages][Hkv][kv_page_bytes] uint8; idx_pool [n_pool_pages][8704] uint8
 *   MXFP4 page (8704 B): bytes [0,8192) = 128 token rows x 64 B of E2M1 nibbles (element 2i
 *             in the low nibble of byte i); bytes [8192,8704) = 128 rows x 4 E8M0 group scales
 *             (group g of slot s at 8192 + 4s + g), one scale per 32 elements.
 *   E4M3 row-scale page (16896 B): 128 rows x 128 e4m3 codes, then 128 fp32 row scales.
 *   topk_pages [B][topk] int32: selected LOGICAL page ids, ascending, padded with -1;
 *   topk_count [B] int32: k_eff = min(topk, ceil(ctx_len/128)).
 *   part_o [B][S][Q][Hq][128] float (unnormalised), part_m, part_l [B][S][Q][Hq] float;
 *   m is a maximum of z*log2(e) (log2 domain), z = q.k / sqrt(128).
 *   out [B][Q][Hq][128] float.
 */
#ifndef SMX_H
#define SMX_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* smx_stream_t; /* the same type as cudaStream_t */

enum {
    SMX_OK = 0,
    SMX_ERR_INVALID_ARG = -1,  /* null pointer, non-positive size, Hq % Hkv != 0, ... */
    SMX_ERR_UNSUPPORTED = -2,  /* D, Di or page_tokens != 128, Q > 16, unknown kv_format, limits */
    SMX_ERR_CUDA = -3,         /* a kernel launch failed (cudaGetLastError) */
    SMX_ERR_WORKSPACE = -4     /* workspace pointer null or smaller than smx_workspace_bytes */
};

enum {
    SMX_KV_MXFP4 = 0,
    SMX_KV_E4M3_ROWSCALE = 1,
    SMX_KV_NVFP4 = 2   /* NVFP4 pages: the format [ATOM-2812] names (PR title "FP4 index cache and
                        * NVFP4 sparse KV cache") and its Mono path refuses ("--index-cache-dtype
                        * mxfp4": "MXFP4 / NVFP4 main KV, NVFP4 index ... stay refused"); built here
                        * from its plain reading: E2M1 codes packed as in an MXFP4 page, one E4M3
                        * scale byte per 16 elements, one fp32 per-tensor decode scale per pool
                        * (smx_shape_t.nv_scale_*). Page (9216 B): bytes [0, 8192) 128 token rows x
                        * 64 nibble bytes, bytes [8192, 9216) 128 token rows x 8 block scales. Row
                        * store: s = amax / (6 g) in fp32, byte = E4M3 nearest to min(s, 448),
                        * codes = nearest E2M1 to x / (E4M3(byte) g) in fp32 (ties to even,
                        * saturating, sign kept); a zero scale stores codes 0, a block holding
                        * NaN / Inf stores byte 0x7F and codes 0. Value = E2M1 x E4M3 x g. Valid as
                        * kv_format and as idx_format; steps with an NVFP4 pool run the standalone
                        * kernels in sequence (smx_decode_step_launches). */
};

/* device status bits */
enum {
    SMX_DEV_BAD_PAGE_ID = 1,   /* a page-table entry outside [0, n_pool_pages) was met */
    SMX_DEV_BAD_CTX = 2,       /* ctx_len outside [Q, max_pages_per_row * 128] (row clamped) */
    SMX_DEV_BAD_TOPK = 4,      /* a selected page id outside [0, ceil(ctx_len/128)) */
    SMX_DEV_TIMEOUT = 8        /* a bounded wait gave up: for another CTA (smx_set_wait_limit_ns), or for
                                * a page copy (the CTA stopped staging pages) */
};

#define SMX_MXFP4_PAGE_BYTES 8704
#define SMX_E4M3RS_PAGE_BYTES 16896
#define SMX_NVFP4_PAGE_BYTES 9216
#define SMX_MAX_Q 16
#define SMX_MAX_TOPK 4096
#define SMX_MAX_PAGES_PER_ROW 16384  /* 2M tokens per row */

typedef struct {
    int32_t B;                  /* rows (sequences) in the step */
    int32_t Q;                  /* query (draft) tokens per row, 1..16 ([ATOM-2812]: 16-token limit) */
    int32_t Hq;                 /* query heads */
    int32_t Hkv;                /* KV heads, Hq % Hkv == 0 */
    int32_t D;                  /* head dim, must be 128 */
    int32_t Di;                 /* index dim (one index head), must be 128 */
    int32_t page_tokens;        /* must be 128 (one selected block = one page) */
    int32_t max_pages_per_row;  /* page-table width */
    int64_t n_pool_pages;       /* physical pages in each pool */
    int32_t topk;               /* k pages selected per row */
    int32_t num_splits;         /* S partitions of the selected list for the split stage */
    int32_t kv_format;          /* SMX_KV_*: K/V page format */
    int32_t pages_per_block;    /* pages per selected block: 0 or 1 (one page), 2 or 4 ([ATOM-2812]
                                 * commit "MXFP4 main KV": PAGES_PER_BLOCK is a build parameter).
                                 * With 2 or 4, topk counts blocks: a block's score is its best page's,
                                 * topk_pages hold block ids (ascending), and the split stage takes
                                 * every page of a selected block inside the row. Only the fused
                                 * steps take 2 or 4; the standalone top-k and split stage refuse
                                 * them (SMX_ERR_UNSUPPORTED). topk * pages_per_block <= 4096. */
    int32_t idx_format;         /* index page format: SMX_KV_MXFP4 (0, [ATOM-2812] "--index-cache-dtype
                                 * mxfp4") or SMX_KV_NVFP4 */
    float nv_scale_k;           /* NVFP4 per-tensor decode scales of the K, V and index pools: finite */
    float nv_scale_v;           /* and > 0 where that pool is NVFP4, ignored otherwise (SMX_ERR_INVALID_ARG */
    float nv_scale_idx;         /* if not); with NVFP4, pages_per_block must be 0 or 1 */
} smx_shape_t;

/* Bytes of device workspace smx_decode_step needs for this shape (step counters, page scores,
 * split partials, packed q, alignment padding). Zero the workspace once before its first use: the
 * counters it holds must start at zero, and every call leaves them at zero again. One workspace
 * serves one shape; calls that share a workspace must not overlap on the GPU. Its last
 * B * Hkv * ceil(Q * Hq / Hkv / 128) * 16384 bytes are the packed q tiles of the tensor-core
 * attention units (e4m3 codes by smx_pack_q_e4m3's rule, 128 rows of 128 bytes per tile, the
 * 16-byte chunks of row i at ((chunk ^ i) & 7) * 16 within its 128 bytes, rows in 8-row atoms of
 * 1024 bytes), written by a step that takes that path; a caller may read them after the step. */
size_t smx_workspace_bytes(const smx_shape_t* shape);

/* a1 -- [ATOM-2812] "--index-cache-dtype mxfp4" (index-K row store: E8M0 group scale =
 * 2^(floor(log2 amax) - 2), E2M1 round-to-nearest-even, saturating at 6, sign kept on zero;
 * a group holding NaN/Inf gets scale 0xFF and zero nibbles) and "MXFP4 main KV" (K and V with
 * the same row store). With kv_format == SMX_KV_E4M3_ROWSCALE, K and V rows are written as
 * e4m3 codes of x / s with s = fl32(amax / 448) (s = 1 when amax = 0) and the index row stays
 * MXFP4. Writes the Q new tokens of every row at positions ctx_len - Q + t. */
int smx_kv_insert_mxfp4(const smx_shape_t* shape, const float* k_new, const float* v_new,
                        const float* kidx_new, const int32_t* page_table, const int32_t* ctx_len,
                        uint8_t* k_pool, uint8_t* v_pool, uint8_t* idx_pool, int32_t* dev_status,
                        smx_stream_t stream);

/* The same call under its shorter name (kept for existing callers). */
int smx_kv_insert(const smx_shape_t* shape, const float* k_new, const float* v_new,
                  const float* kidx_new, const int32_t* page_table, const int32_t* ctx_len,
                  uint8_t* k_pool, uint8_t* v_pool, uint8_t* idx_pool, int32_t* dev_status,
                  smx_stream_t stream);

/* Bulk form of smx_kv_insert for prompts: positions [0, n_fill[b]) of row b, read from dense
 * k, v [B][T][Hkv][128] and kidx [B][T][128] (T = token stride, n_fill[b] <= T). Same row
 * store as smx_kv_insert. shape->Q is ignored. */
int smx_kv_prefill(const smx_shape_t* shape, const float* k, const float* v, const float* kidx,
                   int64_t T, const int32_t* page_table, const int32_t* n_fill,
                   uint8_t* k_pool, uint8_t* v_pool, uint8_t* idx_pool, int32_t* dev_status,
                   smx_stream_t stream);

/* a2 -- [ATOM-2812] "e4m3 q_out convention" / "pack_q_e4m3": n floats to e4m3 bytes at unit
 * scale; in range = round to nearest even (torch's e4m3 cast), |x| > 448 and +-inf saturate to
 * +-448, NaN gives 0x7F. */
int smx_pack_q_e4m3(const float* q, uint8_t* q_e4m3, int64_t n, smx_stream_t stream);

/* a3 alone -- [ATOM-2812] "--index-cache-dtype mxfp4": the page scorer reads every MXFP4 index
 * page of the row (16 B key loads plus a dword of E8M0 scales per tile) against the bf16 index
 * query; the score of a page is the best dot product over its tokens and the row's query tokens
 * (page-score rule of the benchmark workloads: max over the page's tokens of q_idx . k_idx).
 * page_scores [B][max_pages_per_row] float as in smx_index_score_topk, without the selection.
 * Returns SMX_OK, SMX_ERR_INVALID_ARG (NULL or misaligned pointer), SMX_ERR_UNSUPPORTED (shape)
 * or SMX_ERR_CUDA. */
int smx_index_score(const smx_shape_t* shape, const uint16_t* qidx_bf16, const uint8_t* idx_pool,
                    const int32_t* page_table, const int32_t* ctx_len, float* page_scores,
                    int32_t* dev_status, smx_stream_t stream);

/* a3 + a4 -- [ATOM-2812] "--index-cache-dtype mxfp4" (the scorer reads the MXFP4 index pages
 * with the bf16 index query) and "MXFP4 main KV" (the selected blocks fill the sparse table).
 * page_scores[b][p] = max over query tokens t and tokens j of page p with j <= pos_t of
 * qidx[b][t] . kidx[j] (fp32 accumulation; -inf for p >= ceil(ctx_len/128); NaN token scores
 * are left out). Then the k_eff largest pages per row, ties to the lower page id, NaN last.
 * page_scores [B][max_pages_per_row] float is an output the caller provides. */
int smx_index_score_topk(const smx_shape_t* shape, const uint16_t* qidx_bf16,
                         const uint8_t* idx_pool, const int32_t* page_table,
                         const int32_t* ctx_len, float* page_scores, int32_t* topk_pages,
                         int32_t* topk_count, int32_t* dev_status, smx_stream_t stream);

/* a5 -- [ATOM-2812] "MXFP4 main KV": split stage. Partition s of S covers positions
 * [floor(s k_eff / S), floor((s+1) k_eff / S)) of the ascending selected list; for each query
 * (b, t, h) with KV head h / (Hq / Hkv) it keeps m = max z log2(e), l = sum 2^(z log2 e - m)
 * and o = sum 2^(z log2 e - m) V_j over tokens j of its pages with j <= pos_t. An empty
 * partition writes m = -inf, l = 0, o = 0. q is the packed e4m3 bytes (MXFP4 K/V) or bf16
 * bits (E4M3 row-scale K/V, [ATOM-2812] "e4m3 q_out convention": fp8-KV keeps bf16 q). */
int smx_sparse_attn_split(const smx_shape_t* shape, const void* q, const uint8_t* k_pool,
                          const uint8_t* v_pool, const int32_t* page_table,
                          const int32_t* ctx_len, const int32_t* topk_pages,
                          const int32_t* topk_count, float* part_o, float* part_m,
                          float* part_l, int32_t* dev_status, smx_stream_t stream);

/* a6 -- [ATOM-2812] "MXFP4 main KV": merge. out = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s
 * with M = max_s m_s; out = 0 when every partition is empty. */
int smx_sparse_attn_merge(const smx_shape_t* shape, const float* part_o, const float* part_m,
                          const float* part_l, float* out, smx_stream_t stream);

/* The whole step (a1..a6) on `stream`: [ATOM-2812] "--index-cache-dtype mxfp4" (index-K rows are
 * written, then every index page is scored and the top-k pages kept) and "MXFP4 main KV" (K/V rows
 * written, split stage over the selected pages, merge), in the fused single-launch form of
 * [ATOM-2686] Summary (the Mono decode path: one step per layer for the fixed 7-draft verify,
 * 8 query tokens per row). q_f32 is required for MXFP4 K/V, q_bf16 for E4M3
 * row-scale K/V (the other may be NULL). Pools are updated in place (the Q new rows).
 * topk_pages/topk_count are outputs; workspace holds ws_bytes >= smx_workspace_bytes(shape)
 * bytes of scratch (256-byte aligned, zeroed before its first use). One cooperative kernel of at
 * most one CTA per SM: inserts, q packing and page scores; then per attention unit the row's
 * selection, the split stage over one partition and the merge of a slice of rows, the phases
 * ordered by counters in the workspace (bounded waits: SMX_DEV_TIMEOUT in dev_status if one gives
 * up). Calls that share a workspace must not overlap on the GPU. The kernel is launched with
 * programmatic dependent launch: its CTAs may start their on-chip set-up while the previous kernel
 * on `stream` finishes, and wait for that kernel's completion before their first global access,
 * so stream order holds for every input and output. */
int smx_decode_step(const smx_shape_t* shape, const float* q_f32, const uint16_t* q_bf16,
                    const uint16_t* qidx_bf16, const float* k_new, const float* v_new,
                    const float* kidx_new, const int32_t* page_table, const int32_t* ctx_len,
                    uint8_t* k_pool, uint8_t* v_pool, uint8_t* idx_pool, int32_t* topk_pages,
                    int32_t* topk_count, float* out, void* workspace, size_t ws_bytes,
                    int32_t* dev_status, smx_stream_t stream);

/* The step of a layer that reuses an earlier layer's selection ([MiniMax-M3.1] "Enable Mono
 * decode with fixed DSpark verify": an index_topk_freq schedule gives layers that run no indexer
 * and attend over the sparse blocks a previous layer selected). On `stream`: the Q new K and V
 * rows of every row are inserted (no index cache: nothing is scored and no index row is
 * written), q is packed (MXFP4 K/V), and the split stage and the merge run over the given
 * selection: topk_count[b] in [0, min(topk, ceil(ctx_len[b] / 128))] and topk_pages[b][0 ..
 * count) the logical page ids, ascending, of row b ([B][topk] int32, device; e.g. an earlier
 * smx_decode_step's outputs), which this layer's page_table maps to its own K/V pages. Arguments
 * as smx_decode_step (same workspace size; q_f32 or q_bf16 by format; k_new/v_new/k_pool/v_pool
 * 16-byte aligned). A count outside that range is clamped and an id outside the row's pages
 * skipped (an empty page), both flagged SMX_DEV_BAD_TOPK in dev_status. One cooperative
 * kernel, as smx_decode_step without its scoring and selection. Returns SMX_OK,
 * SMX_ERR_INVALID_ARG (a NULL or misaligned pointer), SMX_ERR_UNSUPPORTED (shape),
 * SMX_ERR_WORKSPACE or SMX_ERR_CUDA. */
int smx_decode_step_reuse(const smx_shape_t* shape, const float* q_f32, const uint16_t* q_bf16,
                          const float* k_new, const float* v_new, const int32_t* page_table,
                          const int32_t* ctx_len, uint8_t* k_pool, uint8_t* v_pool,
                          const int32_t* topk_pages, const int32_t* topk_count, float* out,
                          void* workspace, size_t ws_bytes, int32_t* dev_status, smx_stream_t stream);

/* Bound, in nanoseconds of GPU global time, of every wait of the fused steps for other CTAs of
 * the same launch (a row's page scores, a group's partitions: the co-residency the pages' persistent
 * kernel assumed, [vLLM-60528] "Merge Danger"). A wait that runs out sets SMX_DEV_TIMEOUT in
 * dev_status and the CTA goes on with whatever it finds, reading and writing only inside the
 * caller's buffers: that step's outputs are then undefined but finite, and the step still leaves the
 * workspace counters at zero, so the next step is sound. ns = 0 restores the default (200 ms,
 * far above the longest step of the largest shapes). Process-wide; applies to launches enqueued
 * after the call. Returns the bound in force before the call. Meant for tests that make a wait give
 * up; waits for a CTA's own copies and MMAs are not affected. */
uint64_t smx_set_wait_limit_ns(uint64_t ns);

/* Static text for a status code. */
const char* smx_status_string(int status);

/* Number of kernel launches smx_decode_step enqueues for this shape. */
int smx_decode_step_launches(const smx_shape_t* shape);

/* Whether smx_decode_step runs its attention on the fifth-generation tensor cores (tcgen05,
 * 128-row tiles) for this shape on the CURRENT device: 1 yes, 0 no (mma.sync, up to 64-row
 * tiles), SMX_ERR_INVALID_ARG / SMX_ERR_UNSUPPORTED for a bad shape. The tensor-core path is taken
 * when the 64-row attention units (B x Hkv x row groups x S) would need more than one wave of the
 * device's SMs. Reads device attributes; launches nothing. */
int smx_decode_step_tensor_cores(const smx_shape_t* shape);

/* A partition count S for this shape on the CURRENT device (the pages leave S to the
 * implementation: any S >= 1 gives the same attention up to rounding). It is the largest S
 * whose split CTAs (B x Hkv x row groups of up to 64 query rows per partition) fill at most one
 * wave of the device's SMs, lowered so every partition holds the same number of selected pages.
 * For MXFP4 K/V with more than 64 query rows per KV head, when that leaves 3 or more selected
 * pages per partition, it is instead the same count for row groups of 128 rows: the fused step
 * then runs its attention on the tensor cores (smx_decode_step_tensor_cores), the standalone
 * split stage in two waves. shape->num_splits is ignored. Returns S >= 1, or 0 when the other
 * fields of the shape are invalid or a CUDA query fails. Reads device attributes; launches
 * nothing. */
int smx_suggest_num_splits(const smx_shape_t* shape);

/* Bytes of the static device scratch smx_decode_step_noalloc works in (16 MiB). */
#define SMX_NOALLOC_SCRATCH_BYTES (16u << 20)

/* smx_decode_step without a caller-provided workspace and without any device allocation. The
 * pages have no counterpart: it is an interface variant of the whole step above, with the same
 * arguments, results, launches and errors, minus workspace/ws_bytes.
 *
 * Its scratch is one module-scope device array of SMX_NOALLOC_SCRATCH_BYTES per device, placed
 * by the driver when the library's module is loaded. The call never calls cudaMalloc, cudaFree or
 * any other allocating routine. It is meant for callers that cannot allocate: a serving process
 * that reserves nearly all device memory for its KV pools at start-up (a later allocation could
 * fail, or fragment the reservation); code in a decode loop that must not run cudaFree, which can
 * synchronise the whole device; and plain C callers that have no device allocator of their own.
 *
 * The first call on each device (with that device current) looks up the array's address with
 * cudaGetSymbolAddress, which may load the module on that device: make that first call before any
 * stream capture. Every call clears the step counters at the head of the array (one memset of
 * smx_workspace_bytes' counter prefix, a few hundred bytes, on `stream`) and then launches the
 * step; the array keeps the rest of the last call's contents.
 *
 * Argument checks are smx_decode_step's and run first, before the device is touched; then
 * SMX_ERR_WORKSPACE when smx_workspace_bytes(shape) exceeds SMX_NOALLOC_SCRATCH_BYTES, and
 * SMX_ERR_CUDA if the address lookup or the memset fails. All calls on one device share the one
 * array: calls that overlap on the GPU (other streams, other host threads) race on it and give
 * undefined results. */
int smx_decode_step_noalloc(const smx_shape_t* shape, const float* q_f32, const uint16_t* q_bf16,
                            const uint16_t* qidx_bf16, const float* k_new, const float* v_new,
                            const float* kidx_new, const int32_t* page_table, const int32_t* ctx_len,
                            uint8_t* k_pool, uint8_t* v_pool, uint8_t* idx_pool, int32_t* topk_pages,
                            int32_t* topk_count, float* out, int32_t* dev_status, smx_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* SMX_H */

// smx_index.cu -- the standalone a3 (page scores from the MXFP4 index cache) and a4 (top-k pages
// per row) kernels of the C ABI. The per-tile scoring lives in smx_score.cuh and the selection in
// smx_select.cuh (both shared with the fused decode step).
//
// [ATOM-2812] "Mono decode over the MXFP4 KV and index caches", commit "--index-cache-dtype
// mxfp4": every page of the row is scored against the index query; commit "MXFP4 main KV": the
// selected blocks (one 128-token page each) fill the row's sparse table.
//
// Scorer: the tensor-map-fed tcgen05 scan of smx_scan.cuh, grid (CTAs per row, B), two CTAs of 8
// warps per SM; rows cut into very few pages per CTA take the mma.sync scorer.
#include <math.h>

#include <mutex>

#include "smx_device.cuh"
#include "smx_internal.h"
#include "smx_score.cuh"
#include "smx_scan.cuh"
#include "smx_select.cuh"

namespace smx {

struct IndexArgs {
    const uint16_t* qidx;     // [B][Q][128] bf16 bits
    const uint8_t* pool;      // [n_pool][8704]
    const int32_t* page_table;
    const int32_t* ctx_len;
    float* scores;            // [B][max_pages]
    int32_t* status;
    int64_t n_pool;
    int Q, max_pages, pages_per_cta;
    float nv_scale;   // NVFP4 index pages: the pool's per-tensor decode scale
};

constexpr int kIdxMaxPpc = 64;   // page-table entries of one CTA staged in shared memory
constexpr int kIdxScanMinPages = 3;   // pages per CTA from which the tensor-core scan is faster
// Shape of a scanning CTA with NQ query slots: with 8 slots two CTAs share an SM (6 page stages and
// 256 tensor-memory columns each); with 16 the epilogue needs all 255 registers a thread can hold,
// so one CTA takes the SM (12 stages, 512 columns).
template <int NQ>
struct IdxScanShape {
    static constexpr int kCtasPerSm = NQ <= 8 ? 2 : 1;
    static constexpr int kStages = 12 / kCtasPerSm;
    static constexpr int kTmemCols = 512 / kCtasPerSm;
    static constexpr int kAcc = scan_acc_stages(NQ, kTmemCols);
    // dynamic shared memory: the stages and query pieces, plus slack to align them to 1 KB
    static constexpr int kSmemBytes = scan_smem_bytes(kStages, kAcc, NQ) + 1024;
};

// Grid (CTAs per row, B), 256 threads: the CTA scans its range of the row's pages with the
// tensor-map-fed tensor-core pipeline of smx_scan.cuh.
template <int NQ>
__global__ void __launch_bounds__(256, IdxScanShape<NQ>::kCtasPerSm)
    index_scan_kernel(const IndexArgs a, const __grid_constant__ CUtensorMap map) {
    using Sh = IdxScanShape<NQ>;
    constexpr int kIdxStages = Sh::kStages, SA = Sh::kAcc;
    extern __shared__ __align__(1024) uint8_t dsm[];
    __shared__ int64_t phys_s[kIdxMaxPpc];
    __shared__ float gmax[16];
    __shared__ float red[kScanRedPages * 4];
    __shared__ __align__(8) uint64_t bars[scan_barriers(kIdxStages, SA)];
    __shared__ uint32_t tmem_slot;
    __shared__ int gave_up;

    uint8_t* base = dsm + ((1024u - (smem_u32(dsm) & 1023u)) & 1023u);
    ScanPipe sp;
    sp.tiles = base;
    sp.qt = base + kIdxStages * kScanTileBytes;
    sp.ring = sp.qt + scan_query_bytes(NQ);
    scan_bind<kIdxStages, SA>(sp, bars);
    sp.red = red;
    sp.gmax = gmax;
    sp.gave_up = &gave_up;
    sp.seq = 0;
    sp.ins_seq = 0;
    sp.q_seq = 0;
    const int b = blockIdx.y;
    const int warp = threadIdx.x >> 5;
    const int p_begin = blockIdx.x * a.pages_per_cta;
    const int p_end_all = min(p_begin + a.pages_per_cta, a.max_pages);
    // independent loads first: the row's length and this CTA's page-table entries
    const int ctx_raw = a.ctx_len[b];
    for (int i = threadIdx.x; i < p_end_all - p_begin; i += blockDim.x) {
        const int64_t ph = a.page_table[(int64_t)b * a.max_pages + p_begin + i];
        phys_s[i] = (ph < 0 || ph >= a.n_pool) ? -1 : ph;
    }
    if (threadIdx.x == 0) scan_init<kIdxStages, SA>(sp, 1);
    if (warp == 0) tmem_alloc(&tmem_slot, Sh::kTmemCols);
    tc_fence_before_sync();
    const int ctx = clamp_ctx(ctx_raw, a.Q, a.max_pages, (blockIdx.x == 0 && threadIdx.x == 0) ? a.status : nullptr);
    const int n_pages = (ctx + kPage - 1) / kPage;
    const int p_end = min(p_end_all, n_pages);
    for (int p = max(p_begin, n_pages) + threadIdx.x; p < p_end_all; p += blockDim.x)
        a.scores[(int64_t)b * a.max_pages + p] = -INFINITY;
    // phys_s, the barriers and the allocation published (the epilogue warps build the query pieces
    // inside the scan, while the first pages are in flight)
    __syncthreads();
    tc_fence_after_sync();
    sp.tmem = tmem_slot;
    const int np = max(0, p_end - p_begin);
    scan_pages<NQ, kIdxStages, SA>(sp, &map, phys_s, np, p_begin, np, ctx - a.Q, a.Q, a.qidx + (int64_t)b * a.Q * kD,
                                   a.scores + (int64_t)b * a.max_pages, a.status, [] {});
    __syncthreads();
    scan_finish<kIdxStages>(sp, a.status);
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after_sync();
        tmem_dealloc(sp.tmem, Sh::kTmemCols);
    }
}

// Rows cut into few pages per CTA: the mma.sync scorer of smx_score.cuh (8 warps walk the CTA's
// pages two at a time, a warp scoring two 16-token tiles of a page, the next tile's loads in flight
// while the current one is scored): one pass over a handful of pages finishes sooner than the
// tensor-core pipeline fills.
template <int NT, bool NV>
__global__ void __launch_bounds__(kIdxWarps * 32, 2) index_score_mma_kernel(IndexArgs a) {
    constexpr int kPageBytes = NV ? kNvPageBytes : kMxPageBytes;
    __shared__ __align__(16) uint32_t qh[16][64];  // f16x2 of q' per query, natural dim order
    __shared__ int sig[16];
    __shared__ float red[2][kIdxWarps];
    __shared__ int64_t phys_s[kIdxMaxPpc];

    const int b = blockIdx.y;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int p_begin = blockIdx.x * a.pages_per_cta;
    const int p_end_all = min(p_begin + a.pages_per_cta, a.max_pages);
    // independent loads first: the row's length and this CTA's page-table entries
    const int ctx_raw = a.ctx_len[b];
    for (int i = threadIdx.x; i < p_end_all - p_begin; i += blockDim.x) {
        const int64_t ph = a.page_table[(int64_t)b * a.max_pages + p_begin + i];
        phys_s[i] = (ph < 0 || ph >= a.n_pool) ? -1 : ph;
    }
    const int ctx = clamp_ctx(ctx_raw, a.Q, a.max_pages, (blockIdx.x == 0 && threadIdx.x == 0) ? a.status : nullptr);
    const int n_pages = (ctx + kPage - 1) / kPage;
    const int p_end = min(p_end_all, n_pages);
    for (int p = max(p_begin, n_pages) + threadIdx.x; p < p_end_all; p += blockDim.x)
        a.scores[(int64_t)b * a.max_pages + p] = -INFINITY;
    __syncthreads();   // page-table entries staged

    const int half = warp >> 2;          // which of the two pages of an iteration
    const int tile0 = (warp & 3) * 2;    // first of this warp's two tiles
    // tasks of this warp: (iteration it, tile k) -> page p_begin + 2 it + half, tile tile0 + k
    const int n_tasks = 2 * ((p_end - p_begin + 1) / 2);
    auto task_page = [&](int q) { return p_begin + 2 * (q >> 1) + half; };
    auto task_phys = [&](int q) {
        const int p = task_page(q);
        return p < p_end ? phys_s[p - p_begin] : (int64_t)-1;
    };
    // the first tile's loads go out before the query set-up
    TileFrag cur;
    if (n_tasks > 0) {
        const int64_t ph = task_phys(0);
        if (ph >= 0) load_tile<NV>(cur, a.pool + ph * kPageBytes, tile0, g, t);
    }
    uint32_t qf[NT][16];
    int sig_c[NT][2];
    setup_index_query<NT>(load_index_query(a.qidx + (int64_t)b * a.Q * kD, a.Q), a.Q, qh, sig, qf, sig_c);

    const int lim = ctx - a.Q;  // token j counts for query n iff j <= lim + n
    float best = -INFINITY;
#pragma unroll 1
    for (int q = 0; q < n_tasks; ++q) {
        const int p = task_page(q);
        const int64_t ph = task_phys(q);
        // next tile in flight while this one is scored
        TileFrag nxt;
        if (q + 1 < n_tasks) {
            const int64_t phn = task_phys(q + 1);
            if (phn >= 0) load_tile<NV>(nxt, a.pool + phn * kPageBytes, tile0 + ((q + 1) & 1), g, t);
        }
        if (ph >= 0) {
            if constexpr (NV) best = fmaxf(best, score_tile_nv<NT>(cur, qf, sig_c, p, tile0 + (q & 1), g, t, lim, a.Q, a.nv_scale));
            else best = fmaxf(best, score_tile<NT>(cur, qf, sig_c, p, tile0 + (q & 1), g, t, lim, a.Q));
        }
        else if (p < p_end && (q & 1) == 0 && lane == 0 && (warp & 3) == 0) flag_status(a.status, SMX_DEV_BAD_PAGE_ID);
        cur = nxt;
        if (q & 1) {   // both tiles of this iteration's page scored: combine the page's 4 warps
            const int it = q >> 1;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) best = fmaxf(best, __shfl_xor_sync(0xFFFFFFFFu, best, o));
            if (lane == 0) red[it & 1][warp] = best;
            best = -INFINITY;
            __syncthreads();
            if (threadIdx.x < 2) {
                const int pp = p_begin + 2 * it + threadIdx.x;
                if (pp < p_end) {
                    const float* r = red[it & 1] + 4 * threadIdx.x;
                    a.scores[(int64_t)b * a.max_pages + pp] = fmaxf(fmaxf(r[0], r[1]), fmaxf(r[2], r[3]));
                }
            }
        }
    }
}


// ---- standalone a4: one block per row ------------------------------------------------------------
__global__ void __launch_bounds__(kSelThreads) topk_kernel(const float* __restrict__ scores,
                                                           const int32_t* __restrict__ ctx_len,
                                                           int32_t* __restrict__ topk_pages,
                                                           int32_t* __restrict__ topk_count, int max_pages,
                                                           int topk) {
    extern __shared__ __align__(16) uint32_t keys[];
    __shared__ SelectSmem sm;
    const int b = blockIdx.x;
    const int ctx = max(0, min(ctx_len[b], max_pages * kPage));
    const int n = (ctx + kPage - 1) / kPage;
    const float* s = scores + (int64_t)b * max_pages;
    load_keys<false>(keys, s, n);
    __syncthreads();
    int32_t* outp = topk_pages + (int64_t)b * topk;
    const int k_eff = block_select(keys, n, topk, outp, sm);
    for (int i = k_eff + threadIdx.x; i < topk; i += blockDim.x) outp[i] = -1;
    if (threadIdx.x == 0) topk_count[b] = k_eff;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link against the driver
// library), looked up once.
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
        else
            (void)cudaGetLastError();
    });
    return fn;
}

cudaError_t encode_index_map(CUtensorMap* map, const uint8_t* idx_pool, int64_t n_pool) {
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return cudaErrorNotSupported;
    // [page][row][element]: a page is 136 rows of 128 fp4 elements (64 B): 128 token rows of
    // nibbles, then the 512 bytes of scale words as 8 more rows; pages 8704 B apart. One box = one
    // whole page, each 16-element chunk unpacked to 16 bytes, 128-byte swizzle.
    const cuuint64_t dims[3] = {128, (cuuint64_t)kScanRows, (cuuint64_t)n_pool};
    const cuuint64_t strides[2] = {64, (cuuint64_t)kMxPageBytes};
    const cuuint32_t box[3] = {128, (cuuint32_t)kScanRows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 3, const_cast<uint8_t*>(idx_pool), dims, strides,
                          box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

static int sm_count() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    if (cached[dev] == 0) {
        int n = 0;
        cached[dev] = (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && n > 0) ? n : 148;
    }
    return cached[dev];
}

// Pages per CTA for one wave of `per_sm` CTAs per SM over all rows (even for the mma.sync scorer,
// which walks pages in pairs), at most kIdxMaxPpc (longer rows take more waves).
static int index_pages_per_cta(const smx_shape_t& s, int per_sm, bool even) {
    const int64_t slots = per_sm * (int64_t)sm_count();
    const int64_t total = (int64_t)s.B * s.max_pages_per_row;
    int64_t ppc = (total + slots - 1) / slots;
    if (even) ppc = (ppc + 1) & ~(int64_t)1;
    if (ppc > kIdxMaxPpc) ppc = kIdxMaxPpc;
    return (int)(ppc < 2 ? 2 : ppc);
}

cudaError_t launch_index_scores(const smx_shape_t& s, const uint16_t* qidx, const uint8_t* idx_pool,
                                const int32_t* page_table, const int32_t* ctx_len, float* scores,
                                int32_t* status, cudaStream_t st) {
    IndexArgs a = {};
    a.qidx = qidx; a.pool = idx_pool; a.page_table = page_table; a.ctx_len = ctx_len; a.scores = scores;
    a.status = status; a.n_pool = s.n_pool_pages; a.Q = s.Q; a.max_pages = s.max_pages_per_row;
    a.nv_scale = s.nv_scale_idx;
    // the mma.sync scorer (two CTAs per SM) for rows cut into very few pages per CTA, else the scan
    a.pages_per_cta = index_pages_per_cta(s, 2, true);
    // NVFP4 index pages: always the mma.sync scorer
    const bool nv = s.idx_format == SMX_KV_NVFP4;
    const bool mma = nv || a.pages_per_cta < kIdxScanMinPages;
    if (mma) {
        const dim3 grid((s.max_pages_per_row + a.pages_per_cta - 1) / a.pages_per_cta, s.B);
        if (nv) {
            if (s.Q <= 8) index_score_mma_kernel<1, true><<<grid, kIdxWarps * 32, 0, st>>>(a);
            else index_score_mma_kernel<2, true><<<grid, kIdxWarps * 32, 0, st>>>(a);
        } else {
            if (s.Q <= 8) index_score_mma_kernel<1, false><<<grid, kIdxWarps * 32, 0, st>>>(a);
            else index_score_mma_kernel<2, false><<<grid, kIdxWarps * 32, 0, st>>>(a);
        }
        return cudaGetLastError();
    }
    CUtensorMap map;
    cudaError_t e = encode_index_map(&map, idx_pool, s.n_pool_pages);
    if (e != cudaSuccess) return e;
    auto scan = [&](auto kern, int per_sm, int smem) -> cudaError_t {
        a.pages_per_cta = index_pages_per_cta(s, per_sm, false);
        const dim3 grid((s.max_pages_per_row + a.pages_per_cta - 1) / a.pages_per_cta, s.B);
        const cudaError_t r = ensure_smem_attr(reinterpret_cast<const void*>(kern), smem);
        if (r != cudaSuccess) return r;
        kern<<<grid, 256, smem, st>>>(a, map);
        return cudaSuccess;
    };
    e = s.Q <= 8 ? scan(index_scan_kernel<8>, IdxScanShape<8>::kCtasPerSm, IdxScanShape<8>::kSmemBytes)
                 : scan(index_scan_kernel<16>, IdxScanShape<16>::kCtasPerSm, IdxScanShape<16>::kSmemBytes);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_topk(const smx_shape_t& s, const float* scores, const int32_t* ctx_len,
                        int32_t* topk_pages, int32_t* topk_count, cudaStream_t st) {
    const int smem = 4 * s.max_pages_per_row;
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(topk_kernel), smem);
    if (e != cudaSuccess) return e;
    topk_kernel<<<s.B, kSelThreads, smem, st>>>(scores, ctx_len, topk_pages, topk_count, s.max_pages_per_row,
                                                s.topk);
    return cudaGetLastError();
}

}  // namespace smx

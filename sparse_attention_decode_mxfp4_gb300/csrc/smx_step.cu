// smx_step.cu -- the whole decode step (a1..a6) as one cooperative kernel.
//
// [ATOM-2812] "Mono decode over the MXFP4 KV and index caches": the new token rows are written
// into the index, K and V pages before they are read ("--index-cache-dtype mxfp4", "MXFP4 main
// KV"), q is packed to saturating e4m3 ("pack_q_e4m3"), every page of the row is scored, the
// top-k pages are selected, the split stage runs over the selected pages only and the merge
// combines the partitions.
//
// The grid holds at most one CTA per SM and is launched cooperatively, so all of its CTAs are
// resident together and may wait for one another through counters in the workspace (never for a
// CTA that could still be waiting to start). Phases of every CTA:
//  A. Scoring. The B x max_pages page slots are cut into C chunks of P pages per row; chunk (b, j)
//     is taken by CTA (b C + j) mod grid. The chunk's CTA writes the new index-K rows that land
//     on its pages before it reads those pages (through L2), writes its share (j of C) of the
//     row's new K/V rows, scores its pages and counts itself on the row's counter.
//  B. Attention units (row b, KV head, row group, partition s), taken from the last CTA down. The
//     unit's CTA first loads what does not depend on phase A (its q fragments, packed from f32 for
//     MXFP4 K/V, and the row's page table), then waits for row b's C chunks, selects the row's
//     top-k pages itself from the row's scores (every unit of the row computes the same
//     selection, so no CTA waits for another to publish it), takes partition s of the ascending
//     list and runs the split stage over it, writes its partials and counts itself on the (row,
//     KV head, row group) counter.
//  C. Merge. Each unit's CTA waits for the S partitions of its group and merges slice s of the
//     group's query rows.
//  D. The last CTA to finish resets every counter to zero for the next step.
// Every wait is bounded (waits for other CTAs: 200 ms of global time by default, see
// smx_set_wait_limit_ns; waits for this CTA's own copies and MMAs: about a second); a wait that
// gives up sets SMX_DEV_TIMEOUT and the CTA goes on without reading or writing out of bounds.
#include <math.h>
#include <string.h>

#include <mutex>

#include "smx_attend.cuh"
#include "smx_attend_tc.cuh"
#include "smx_device.cuh"
#include "smx_internal.h"
#include "smx_scan.cuh"
#include "smx_score.cuh"
#include "smx_select.cuh"

namespace smx {

struct StepArgs {
    const float* q_f32;          // MXFP4 K/V: [B][Q][Hq][128], packed here
    const uint16_t* q_bf16;      // FP8-KV: [B][Q][Hq][128] bf16 bits
    const uint16_t* qidx;        // [B][Q][128] bf16 bits
    const float* k_new;          // [B][Q][Hkv][128]
    const float* v_new;
    const float* kidx_new;       // [B][Q][128]
    const int32_t* page_table;   // [B][max_pages]
    const int32_t* ctx_len;      // [B]
    uint8_t* idx_pool;
    uint8_t* k_pool;
    uint8_t* v_pool;
    int32_t* topk_out;           // [B][topk]
    int32_t* count_out;          // [B]
    float* out;                  // [B][Q][Hq][128]
    int32_t* status;
    uint32_t* row_cnt;           // [B] chunks scored
    uint32_t* grp_cnt;           // [B][Hkv][n_rg] partitions written
    uint32_t* done_cnt;          // [1] CTAs past their last wait
    float* scores;               // [B][max_pages]
    float* part_o;               // [B][S][Q][Hq][128]
    float* part_m;               // [B][S][Q][Hq]
    float* part_l;
    uint8_t* q_img;              // [B][Hkv][n_rg][kQImgBytes]: tensor-core units' packed q tiles
    int64_t n_pool;
    int B, Q, Hq, Hkv, G, max_pages, topk, S;
    int row_warps, rows_per_cta, n_rg, page_bytes;
    int chunk_pages, chunks_per_row;
    const int32_t* topk_in;      // REUSE: the given selection [B][topk], and its counts [B]
    const int32_t* count_in;
    int ppb_log2;                // log2 of the pages per selected block (0: one page)
    uint64_t wait_ns;            // bound of every wait for other CTAs (global-timer ns)
};

constexpr int kStepWarps = 8;
constexpr int kStepMaxChunk = 256;   // pages of one scoring chunk (page-table entries in smem)
constexpr int kPtCache = 2048;       // page-table entries of a unit's row kept in shared memory
constexpr int kCounterStride = 32;   // u32 words between counters: each on its own 128-byte line
constexpr int kStepScanStages = 9;   // page stages of the index scan (pages in flight per SM)
constexpr int kStepQFront = 32768;   // bytes ahead of the scan's stages: the first unit's q (staged or packed)
constexpr int kPlanRows = 256;       // rows up to which the scan's chunks follow the rows' real lengths
constexpr int kQImgBytes = kTcRows * kD;   // one unit's e4m3 q tile image (the shared-memory operand layout)


// Selection over blocks of 2^log2 pages: keys[0 .. n_pages) (page keys, shared memory) become
// keys[0 .. n_blocks), each block's best page key (score_key is order-preserving; NaN pages, key 0,
// lose to any number). In rounds of one block per thread: every read of a round comes before its
// writes (a barrier), and a round's writes land below the next rounds' reads. Every thread.
__device__ __forceinline__ int block_max_keys(uint32_t* keys, int n_pages, int log2) {
    const int ppb = 1 << log2, nb = (n_pages + ppb - 1) >> log2;
    for (int r0 = 0; r0 < nb; r0 += blockDim.x) {
        const int blk = r0 + (int)threadIdx.x;
        uint32_t m = 0u;
        if (blk < nb)
            for (int q = 0; q < ppb; ++q) {
                const int p = (blk << log2) + q;
                if (p < n_pages) m = max(m, keys[p]);
            }
        __syncthreads();
        if (blk < nb) keys[blk] = m;
    }
    __syncthreads();
    return nb;
}

// A reusing layer's selection for row b (entries [0, k_eff) of sel_all): the given count clamped
// to [0, min(topk, n_pages)], each id checked against the row's pages (an id outside them is
// flagged and becomes -1: an empty page). Every thread; ends with a barrier.
__device__ __forceinline__ int given_selection(const StepArgs& a, int b, int n_pages, int* sel_all) {
    const int raw = a.count_in[b];
    const int k_eff = max(0, min(raw, min(a.topk, n_pages)));
    if (threadIdx.x == 0 && raw != k_eff) flag_status(a.status, SMX_DEV_BAD_TOPK);
    for (int i = threadIdx.x; i < k_eff; i += blockDim.x) {
        int p = a.topk_in[(int64_t)b * a.topk + i];
        if (p < 0 || p >= n_pages) {
            flag_status(a.status, SMX_DEV_BAD_TOPK);
            p = -1;
        }
        sel_all[i] = p;
    }
    __syncthreads();
    return k_eff;
}

template <bool RS, int NT, bool TC, bool REUSE>
__global__ void __launch_bounds__(kStepWarps * 32, 1) decode_step_kernel(const StepArgs a,
                                                                       const __grid_constant__ CUtensorMap idx_map) {
    constexpr int NQ = 8 * NT;                   // query slots of the index scan
    constexpr int kStepScanAcc = scan_acc_stages(NQ, 384);   // its accumulator stages (of the 512 columns)
    constexpr bool kScan = !REUSE;               // phase A scans the index cache
    // the scanner: with the tensor-core attention (long rows, many pages per unit) the tensor-map
    // scan (smx_scan.cuh), which streams long chunks fastest; with the mma.sync attention the mma.sync
    // scorer (smx_score.cuh), which starts sooner on the short chunks those shapes give. One scanner
    // per kernel variant: two in one kernel measured slower on every workload.
    constexpr bool kScanTma = kScan && TC;
    constexpr bool kScanMma = kScan && !TC;
    constexpr bool kTmem = TC;                   // tensor memory: the scan's accumulators, the attention's
    constexpr bool kQImg = TC && !RS && kScan;   // q tiles packed by the scanning CTAs into the workspace
    extern __shared__ __align__(1024) uint8_t smem[];
    __shared__ int64_t phys_s[kStepMaxChunk];
    __shared__ float gmax[16];                   // the scan's query set-up
    __shared__ float scan_red[kScanRedPages * 4];
    __shared__ __align__(8) uint64_t scan_bars[scan_barriers(kStepScanStages, kStepScanAcc)];
    __shared__ int scan_gave_up;
    __shared__ int plan_c0[kPlanRows], plan_cn[kPlanRows];   // balanced chunk plan: row b's first chunk, count
    __shared__ int plan_total, plan_mine;
    __shared__ SelectSmem selsm;
    __shared__ __align__(8) uint64_t mbar[4];   // page copies (tensor-core MXFP4: K slot 0, 1, V slot 0, 1)
    __shared__ __align__(8) uint64_t mbar_q;   // the first unit's q rows
    __shared__ int stage_page[2];
    __shared__ int is_last;
    __shared__ int32_t pt_s[kPtCache];   // the unit's row of the page table (rows up to kPtCache pages)
    __shared__ __align__(8) uint64_t mbar_mma[2];   // tensor-core MMA completions (MXFP4: QK, PV)
    __shared__ uint32_t tmem_slot;
    __shared__ float xch_tc[kStepWarps * 32];    // row maxima / sums exchanged between the two halves

    // dynamic shared memory. Tensor-core path: the tiles of smx_attend_tc.cuh, then the
    // partition's lists; before the attention the K and V tiles hold the selection keys, the P
    // tile the selection and the V / P tiles the staged q rows. mma.sync path: the bf16 tiles of
    // smx_attend.cuh (also the keys), the page stages (also the staged q rows), then the lists.
    AttendSmem sm;
    uint32_t* keys;
    int* sel_all;
    uint8_t* q_stage;
    if constexpr (TC) {
        sm.raw = smem + (RS ? kTcRaw : kTcMxRaw);
        sm.mbar = mbar;
        sm.stage_page = stage_page;
        keys = reinterpret_cast<uint32_t*>(smem + kTcK);
        sel_all = reinterpret_cast<int*>(smem + kTcP);
        q_stage = smem + kTcV;
    } else {
        sm = attend_smem(smem, a.page_bytes, mbar, stage_page);
        keys = reinterpret_cast<uint32_t*>(smem);
        sel_all = reinterpret_cast<int*>(sm.raw + 4 * a.page_bytes) + 2 * (a.topk << a.ppb_log2);
        q_stage = sm.raw;   // the page stages (no copy lands there before the attention)
    }
    int* sel = reinterpret_cast<int*>(sm.raw + 4 * a.page_bytes);   // this partition's pages
    int* selph = sel + (a.topk << a.ppb_log2);                       // and their physical ids

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nC = gridDim.x, c = blockIdx.x;
    // the index scan's stages from the (1024-byte aligned) start of dynamic shared memory; they are
    // free again once phase A is done (the attention's tiles overlap them)
    ScanPipe sp;
    {
        uint8_t* base = smem + ((1024u - (smem_u32(smem) & 1023u)) & 1023u) + kStepQFront;
        sp.tiles = base;
        sp.qt = base + kStepScanStages * kScanTileBytes;
        sp.ring = sp.qt + scan_query_bytes(NQ);
        scan_bind<kStepScanStages, kStepScanAcc>(sp, scan_bars);
        sp.red = scan_red;
        sp.gmax = gmax;
        sp.q_seq = 0;
        sp.gave_up = &scan_gave_up;
        sp.seq = 0;
        sp.ins_seq = 0;
    }
    // one allocation of tensor memory for the whole kernel (one CTA per SM holds all 512 columns),
    // while warps 1 and 2 initialise the barriers: on-chip set-up that may run while the stream's
    // previous kernel finishes (the launch allows it to start early, programmatic dependent
    // launch); every global access comes after the wait for that kernel's completion
    if (kTmem && warp == 0) tmem_alloc(&tmem_slot, kTcCols);
    if (warp == 1 && lane < 7) {
        mbar_init(lane < 4 ? &mbar[lane] : lane == 4 ? &mbar_q : &mbar_mma[lane - 5], 1);
        mbar_fence_init();
    }
    if constexpr (kScan) {
        if (kScanTma && warp == 2) scan_init_warp<kStepScanStages, kStepScanAcc>(sp, 4, lane);   // insert hand-off: warps 4-7
    }
    pdl_wait();
    pdl_trigger();   // the next step may begin its own set-up once SMs free up
    // the set-up's global loads go out before anything waits: the rows' lengths for the balanced
    // plan (below), then the first attention unit's row length and row of the page table. The
    // balanced plan is the tensor-map scan's: its long chunks shrink by the rows' raggedness; the
    // mma.sync scan's short chunks gain less than the plan's round trip costs on rows of equal length.
    bool balanced = kScanTma && a.B <= kPlanRows && nC >= 2 * a.B;
    const int ctx_pre = (balanced && (int)threadIdx.x < a.B) ? a.ctx_len[threadIdx.x] : 0;
    const int kv_rows = a.Q * 2 * a.Hkv;
    const int M = a.G * a.Q;
    const int n_units = a.B * a.Hkv * a.n_rg * a.S;
    const int u0 = nC - 1 - c;   // this CTA's first attention unit
    const int R = a.rows_per_cta;
    const int ctx_u0 = u0 < n_units ? a.ctx_len[u0 / (a.S * a.n_rg * a.Hkv)] : 0;   // its row length
    // its row of the page table: loaded into registers now, stored to pt_s once the first chunk's
    // loads are out (a store right here would hold the warp for the round trip)
    constexpr int kPtPerThread = kPtCache / (kStepWarps * 32);
    int32_t pt_r[kPtPerThread];
    const int n_pt0 = u0 < n_units ? min(a.max_pages, kPtCache) : 0;
    {
        const int b = u0 < n_units ? u0 / (a.S * a.n_rg * a.Hkv) : 0;
#pragma unroll
        for (int k = 0; k < kPtPerThread; ++k) {
            const int i = threadIdx.x + k * kStepWarps * 32;
            pt_r[k] = i < n_pt0 ? a.page_table[(int64_t)b * a.max_pages + i] : 0;
        }
    }
    // The first unit's q rows: staged into shared memory by bulk copies (the mma.sync path: into the
    // page stages; a reusing layer on the tensor-core path: into the V and P tiles; both unused until
    // the attention), issued by the thread that initialised their barrier. The tensor-core path with
    // a scan packs the q tile images instead (MXFP4), or brings the FP8-KV q rows into L2 with the
    // evict-last priority, so that the index pages streaming through L2 during the scan, copied
    // with the evict-first one, leave them there.
    const bool q_stageable = !(TC && kScan) && (!RS || (reinterpret_cast<uintptr_t>(a.q_bf16) & 15u) == 0);
    if (TC && kScan && !kQImg && u0 < n_units) {
        const int rg = (u0 / a.S) % a.n_rg, kvh = (u0 / (a.S * a.n_rg)) % a.Hkv, b = u0 / (a.S * a.n_rg * a.Hkv);
        const int m_lo = rg * R, rows = min(M, m_lo + R) - m_lo;
        const int lines = RS ? 2 : 4;   // 128-byte lines of a q row (bf16 or f32)
        const uint8_t* q = RS ? reinterpret_cast<const uint8_t*>(a.q_bf16) : reinterpret_cast<const uint8_t*>(a.q_f32);
        for (int li = threadIdx.x; li < rows * lines; li += blockDim.x) {
            const int m = m_lo + li / lines;
            const int64_t row = ((int64_t)b * a.Q + m / a.G) * a.Hq + kvh * a.G + m % a.G;
            prefetch_l2_keep(q + row * (lines * 128) + (li % lines) * 128);
        }
    }
    if (q_stageable && u0 < n_units && warp == 1 && lane == 4) {
        const int rg = (u0 / a.S) % a.n_rg, kvh = (u0 / (a.S * a.n_rg)) % a.Hkv, b = u0 / (a.S * a.n_rg * a.Hkv);
        const int m_lo = rg * R, m_hi = min(M, m_lo + R);
        const uint32_t row_bytes = RS ? kD * 2 : kD * 4;
        const uint8_t* q = RS ? reinterpret_cast<const uint8_t*>(a.q_bf16) : reinterpret_cast<const uint8_t*>(a.q_f32);
        mbar_arrive_expect_tx(&mbar_q, (uint32_t)(m_hi - m_lo) * row_bytes);
        // rows of one draft token are consecutive heads: one copy per token
        for (int tq = m_lo / a.G; tq * a.G < m_hi; ++tq) {
            const int r0 = max(m_lo, tq * a.G), r1 = min(m_hi, (tq + 1) * a.G);
            const int64_t row = ((int64_t)b * a.Q + tq) * a.Hq + kvh * a.G + r0 % a.G;
            bulk_g2s(q_stage + (r0 - m_lo) * row_bytes, q + row * row_bytes, (uint32_t)(r1 - r0) * row_bytes, &mbar_q);
        }
    }
    tc_fence_before_sync();
    // Scoring chunks. Balanced plan (tensor-map scan, up to kPlanRows rows, at least two CTAs per row
    // and chunks of at most kStepMaxChunk pages): from the
    // rows' real page counts n_b (T in all), chunks of P = ceil(T / (grid - B)) pages, ceil(n_b / P)
    // of them (at least one) for row b -- at most one chunk per CTA, CTA c taking chunk c in row
    // order. Every CTA computes the same plan; plan_c0[b] / plan_cn[b] hold row b's first chunk and
    // chunk count (also the count its attention units wait for). Otherwise the host's plan: chunks of
    // a.chunk_pages over the page table's width, a.chunks_per_row per row, chunk ci on CTA ci mod grid.
    // (The plan's block barriers also publish the barriers' initialisation.)
    int P = a.chunk_pages, C = a.chunks_per_row;
    if (balanced) {
        int nb = 0;
        if ((int)threadIdx.x < a.B) {
            const int ctx_t = clamp_ctx(ctx_pre, a.Q, a.max_pages, nullptr);
            nb = (ctx_t + kPage - 1) / kPage;
        }
        const uint32_t tot = sel_block_incl_scan((uint32_t)nb, selsm, 0);
        if (threadIdx.x == blockDim.x - 1) plan_total = (int)tot;
        __syncthreads();
        P = max(1, (plan_total + (nC - a.B) - 1) / (nC - a.B));
        if (P > kStepMaxChunk) {
            // chunks longer than the page-table stage: the host's plan (every CTA sees the same total)
            balanced = false;
            P = a.chunk_pages;
        } else {
            const int cb = (int)threadIdx.x < a.B ? max(1, (nb + P - 1) / P) : 0;
            if (threadIdx.x == 0) plan_mine = -1;
            const uint32_t incl = sel_block_incl_scan((uint32_t)cb, selsm, 1);
            if ((int)threadIdx.x < a.B) {
                const int c0 = (int)incl - cb;
                plan_c0[threadIdx.x] = c0;
                plan_cn[threadIdx.x] = cb;
                if (c >= c0 && c < c0 + cb) plan_mine = threadIdx.x;   // the row of this CTA's chunk
            }
            __syncthreads();
        }
    } else {
        // the barriers are initialised before any thread polls one: a CTA with no chunk in phase A
        // reaches its attention unit's q wait without another barrier
        if (blockIdx.x >= a.B * a.chunks_per_row) __syncthreads();
    }
    // chunks per row b (the count of its row counter)
    auto row_chunks = [&](int b) { return balanced ? plan_cn[b] : C; };
    bool pt_stored = false;
    auto store_pt = [&]() {
#pragma unroll
        for (int k = 0; k < kPtPerThread; ++k) {
            const int i = threadIdx.x + k * kStepWarps * 32;
            if (i < n_pt0) pt_s[i] = pt_r[k];
        }
        pt_stored = true;
    };
    // ---------------- A. scoring chunks ----------------
    if constexpr (REUSE) {
        // a layer reusing an earlier layer's selection has no index cache: each chunk (b, j) writes
        // its warps' share of row b's new K/V rows (rows j + C w, j + C (w + 8), ...), then releases
        // the row counter
        for (int ci = c; ci < a.B * C; ci += nC) {
            const int b = ci / C, j = ci % C;
            const int ctx = clamp_ctx(a.ctx_len[b], a.Q, a.max_pages, (j == 0 && threadIdx.x == 0) ? a.status : nullptr);
            const int first_new = ctx - a.Q;
            for (int r = j + C * warp; r < kv_rows; r += C * kStepWarps) {
                const int tq = r / (2 * a.Hkv), kind = r % (2 * a.Hkv);   // kind < Hkv: K head, else V head
                const int pos = first_new + tq;
                if (pos < 0) continue;
                const int64_t tok = (int64_t)b * a.Q + tq;
                const float4 x = reinterpret_cast<const float4*>((kind < a.Hkv ? a.k_new : a.v_new) +
                                                                 (tok * a.Hkv + kind % a.Hkv) * kD)[lane];
                const int64_t phys = a.page_table[(int64_t)b * a.max_pages + pos / kPage];
                if (phys < 0 || phys >= a.n_pool) {
                    if (lane == 0) flag_status(a.status, SMX_DEV_BAD_PAGE_ID);
                    continue;
                }
                const int h = kind % a.Hkv, slot = pos % kPage;
                uint8_t* pool = kind < a.Hkv ? a.k_pool : a.v_pool;
                if (RS) {
                    uint8_t* page = pool + (phys * a.Hkv + h) * (int64_t)kRsPageBytes;
                    quant_row_e4m3rs_warp(x, page + slot * 128, reinterpret_cast<float*>(page + kRsScaleOff) + slot, lane);
                } else {
                    uint8_t* page = pool + (phys * a.Hkv + h) * (int64_t)kMxPageBytes;
                    quant_row_mxfp4_warp(x, page + slot * 64, page + kMxScaleOff + slot * 4, lane);
                }
            }
            if (!pt_stored) store_pt();
            __syncthreads();
            if (threadIdx.x == 0) red_release_add(&a.row_cnt[kCounterStride * b], 1u);
        }
    } else {
        // this CTA's chunks: balanced, chunk c (if any); else ci = c, c + grid, ...
        const int b_bal = balanced ? plan_mine : -1;
        const int n_chunks = balanced ? (b_bal >= 0 ? 1 : 0) : max(0, (a.B * C - c + nC - 1) / nC);
#pragma unroll 1
        for (int k = 0; k < n_chunks; ++k) {
            const int ci = c + k * nC;
            const int b = balanced ? b_bal : ci / C;
            const int j = balanced ? c - plan_c0[b_bal] : ci % C;
            const int Cb = row_chunks(b);
            const int p0 = j * P, np_max = max(0, min(P, a.max_pages - p0));
            // independent loads first: the row's length, this chunk's page-table entries
            const int ctx_raw = a.ctx_len[b];
            for (int i = threadIdx.x; i < np_max; i += blockDim.x) {
                const int64_t ph = a.page_table[(int64_t)b * a.max_pages + p0 + i];
                phys_s[i] = (ph < 0 || ph >= a.n_pool) ? -1 : ph;
            }
            if constexpr (kScanMma) {
                // the mma.sync scorer: all eight warps write the chunk's share of the new rows
                // (index-K rows on its pages, K/V rows), then score its pages four at a time: warp
                // 2q + h scores tiles 4h .. 4h + 3 of page i0 + q, the next group's tiles in flight;
                // the pages that take no new rows are loaded before the inserts. Scratch: the start
                // of the attention's K tile (free until the attention).
                const int g = lane >> 2, t = lane & 3;
                uint32_t(&qh)[16][64] = *reinterpret_cast<uint32_t(*)[16][64]>(smem);
                int* sig = reinterpret_cast<int*>(smem + 16 * 64 * 4);
                float(*red)[kStepWarps] = reinterpret_cast<float(*)[kStepWarps]>(smem + 16 * 64 * 4 + 64);
                const IndexQueryRaw qraw = load_index_query(a.qidx + (int64_t)b * a.Q * kD, a.Q);
                float4 kidx_x = make_float4(0.f, 0.f, 0.f, 0.f);
                if (warp < a.Q) kidx_x = reinterpret_cast<const float4*>(a.kidx_new + ((int64_t)b * a.Q + warp) * kD)[lane];
                const int kv_r0 = j + Cb * warp;   // this warp's K/V rows: kv_r0, kv_r0 + 8 Cb, ...
                auto kv_row_src = [&](int r) {
                    const int tq = r / (2 * a.Hkv), kind = r % (2 * a.Hkv);   // kind < Hkv: K head, else V head
                    const int64_t tok = (int64_t)b * a.Q + tq;
                    return reinterpret_cast<const float4*>((kind < a.Hkv ? a.k_new : a.v_new) + (tok * a.Hkv + kind % a.Hkv) * kD) + lane;
                };
                float4 kv_x = make_float4(0.f, 0.f, 0.f, 0.f);
                if (kv_r0 < kv_rows) kv_x = *kv_row_src(kv_r0);
                const int ctx = clamp_ctx(ctx_raw, a.Q, a.max_pages, (j == 0 && threadIdx.x == 0) ? a.status : nullptr);
                const int n_pages = (ctx + kPage - 1) / kPage;
                const int np = max(0, min(np_max, n_pages - p0));
                const int first_new = ctx - a.Q;
                // chunk pages [own_lo, own_hi) take new index-K rows (positions [lo_new, hi_new))
                const int lo_new = max(max(first_new, 0), p0 * kPage), hi_new = min(ctx, (p0 + np) * kPage);
                const bool owner = lo_new < hi_new;
                const int own_lo = owner ? lo_new / kPage - p0 : np, own_hi = owner ? (hi_new - 1) / kPage - p0 + 1 : np;
                __syncthreads();   // page-table entries staged (and the barriers initialised)
                const int pq = warp >> 1, tile0 = (warp & 1) * 4;
                TileFrag fa[4], fb[4];
                auto load_page = [&](TileFrag(&f)[4], int i, bool skip_own) {
                    if (i < np && phys_s[i] >= 0 && !(skip_own && i >= own_lo && i < own_hi)) {
                        const uint8_t* page = a.idx_pool + phys_s[i] * kMxPageBytes;
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) load_tile(f[kk], page, tile0 + kk, g, t);
                    }
                };
                load_page(fa, pq, true);
                if (!pt_stored) store_pt();
                if (owner) {
                    // the new index-K rows on this chunk's pages (one warp per row), then those pages' tiles
                    for (int tq = warp; tq < a.Q; tq += kStepWarps) {
                        const int pos = first_new + tq;
                        if (pos < lo_new || pos >= hi_new) continue;
                        const int64_t phys = phys_s[pos / kPage - p0];
                        if (phys < 0) {
                            if (lane == 0) flag_status(a.status, SMX_DEV_BAD_PAGE_ID);
                            continue;
                        }
                        const float4 x = tq == warp ? kidx_x : reinterpret_cast<const float4*>(a.kidx_new + ((int64_t)b * a.Q + tq) * kD)[lane];
                        uint8_t* page = a.idx_pool + phys * kMxPageBytes;
                        quant_row_mxfp4_warp(x, page + (pos % kPage) * 64, page + kMxScaleOff + (pos % kPage) * 4, lane);
                    }
                    __threadfence();
                    __syncthreads();
                    if (pq >= own_lo && pq < own_hi) load_page(fa, pq, false);
                }
                // this warp's new K/V rows (read only by the attention phase, after the row's counter),
                // while the index tiles are in flight
                for (int r = kv_r0; r < kv_rows; r += Cb * kStepWarps) {
                    const int tq = r / (2 * a.Hkv), kind = r % (2 * a.Hkv);
                    const int pos = first_new + tq;
                    if (pos < 0) continue;
                    const float4 x = r == kv_r0 ? kv_x : *kv_row_src(r);
                    const int64_t phys = a.page_table[(int64_t)b * a.max_pages + pos / kPage];
                    if (phys < 0 || phys >= a.n_pool) {
                        if (lane == 0) flag_status(a.status, SMX_DEV_BAD_PAGE_ID);
                        continue;
                    }
                    const int h = kind % a.Hkv, slot = pos % kPage;
                    uint8_t* pool = kind < a.Hkv ? a.k_pool : a.v_pool;
                    if (RS) {
                        uint8_t* page = pool + (phys * a.Hkv + h) * (int64_t)kRsPageBytes;
                        quant_row_e4m3rs_warp(x, page + slot * 128, reinterpret_cast<float*>(page + kRsScaleOff) + slot, lane);
                    } else {
                        uint8_t* page = pool + (phys * a.Hkv + h) * (int64_t)kMxPageBytes;
                        quant_row_mxfp4_warp(x, page + slot * 64, page + kMxScaleOff + slot * 4, lane);
                    }
                }
                uint32_t qf[NT][16];
                int sig_c[NT][2];
                setup_index_query<NT>(qraw, a.Q, qh, sig, qf, sig_c);
                const int lim = ctx - a.Q;   // token j counts for query n iff j <= lim + n
#pragma unroll 1
                for (int i0 = 0; i0 < np; i0 += 4) {
                    if (i0 + 4 < np) load_page(fb, i0 + 4 + pq, false);
                    const int i = i0 + pq;
                    if (i < np) {
                        float best = -INFINITY;
                        if (phys_s[i] >= 0) {
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk)
                                best = fmaxf(best, score_tile<NT>(fa[kk], qf, sig_c, p0 + i, tile0 + kk, g, t, lim, a.Q));
                        } else if ((warp & 1) == 0 && lane == 0) {
                            flag_status(a.status, SMX_DEV_BAD_PAGE_ID);
                        }
#pragma unroll
                        for (int o = 16; o > 0; o >>= 1) best = fmaxf(best, __shfl_xor_sync(0xFFFFFFFFu, best, o));
                        if (lane == 0) red[i % kScanRedPages][warp & 1] = best;
                    }
                    if ((i0 + 4) % kScanRedPages == 0 || i0 + 4 >= np) {   // page maxima of pages [base, i0 + 4)
                        __syncthreads();
                        const int base = (i0 / kScanRedPages) * kScanRedPages;
                        const int cnt = min(i0 + 4, np) - base;
                        if ((int)threadIdx.x < cnt)
                            a.scores[(int64_t)b * a.max_pages + p0 + base + threadIdx.x] =
                                fmaxf(red[threadIdx.x][0], red[threadIdx.x][1]);
                        __syncthreads();
                    }
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) fa[kk] = fb[kk];
                }
            } else {
                // the new rows are written by warps 4-7 (w = warp - 4) before they take the scan's epilogue
                const bool writer = warp >= 4;
                const int w4 = warp - 4;
                const int kv_r0 = j + Cb * w4;   // this writing warp's K/V rows: kv_r0, kv_r0 + 4 Cb, ...
                auto kv_row_src = [&](int r) {
                    const int tq = r / (2 * a.Hkv), kind = r % (2 * a.Hkv);   // kind < Hkv: K head, else V head
                    const int64_t tok = (int64_t)b * a.Q + tq;
                    return reinterpret_cast<const float4*>((kind < a.Hkv ? a.k_new : a.v_new) + (tok * a.Hkv + kind % a.Hkv) * kD) + lane;
                };
                float4 kidx_x = make_float4(0.f, 0.f, 0.f, 0.f), kv_x = kidx_x;
                if (writer) {
                    if (w4 < a.Q) kidx_x = reinterpret_cast<const float4*>(a.kidx_new + ((int64_t)b * a.Q + w4) * kD)[lane];
                    if (kv_r0 < kv_rows) kv_x = *kv_row_src(kv_r0);
                }
                const int ctx = clamp_ctx(ctx_raw, a.Q, a.max_pages, (j == 0 && threadIdx.x == 0) ? a.status : nullptr);
                const int n_pages = (ctx + kPage - 1) / kPage;
                const int np = max(0, min(np_max, n_pages - p0));
                const int first_new = ctx - a.Q;
                // chunk pages [own_lo, ..) take new index-K rows (positions [lo_new, hi_new))
                const int lo_new = max(max(first_new, 0), p0 * kPage), hi_new = min(ctx, (p0 + np) * kPage);
                const bool owner = lo_new < hi_new;
                const int own_lo = owner ? lo_new / kPage - p0 : np;
                // phys_s published (the epilogue warps build the row's query pieces inside the scan, while
                // the first pages are in flight)
                __syncthreads();
                if (!pt_stored) store_pt();
                auto write_rows = [&]() {   // warps 4-7, before the scan's epilogue
                    if (owner) {
                        // the new index-K rows on this chunk's pages (one warp per row), before the copiers
                        // read those pages (they wait for the four writing warps)
                        for (int tq = w4; tq < a.Q; tq += 4) {
                            const int pos = first_new + tq;
                            if (pos < lo_new || pos >= hi_new) continue;
                            const int64_t phys = phys_s[pos / kPage - p0];
                            if (phys < 0) {
                                if (lane == 0) flag_status(a.status, SMX_DEV_BAD_PAGE_ID);
                                continue;
                            }
                            const float4 x = tq == w4 ? kidx_x : reinterpret_cast<const float4*>(a.kidx_new + ((int64_t)b * a.Q + tq) * kD)[lane];
                            uint8_t* page = a.idx_pool + phys * kMxPageBytes;
                            quant_row_mxfp4_warp(x, page + (pos % kPage) * 64, page + kMxScaleOff + (pos % kPage) * 4, lane);
                        }
                        fence_proxy_async_global();
                        __threadfence();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(sp.ins);
                    }
                    // this warp's share of the row's new K/V rows (read only by the attention phase, after
                    // the row's counter)
                    for (int r = kv_r0; r < kv_rows; r += 4 * Cb) {
                        const int tq = r / (2 * a.Hkv), kind = r % (2 * a.Hkv);
                        const int pos = first_new + tq;
                        if (pos < 0) continue;
                        const float4 x = r == kv_r0 ? kv_x : *kv_row_src(r);
                        const int64_t phys = a.page_table[(int64_t)b * a.max_pages + pos / kPage];
                        if (phys < 0 || phys >= a.n_pool) {
                            if (lane == 0) flag_status(a.status, SMX_DEV_BAD_PAGE_ID);
                            continue;
                        }
                        const int h = kind % a.Hkv, slot = pos % kPage;
                        uint8_t* pool = kind < a.Hkv ? a.k_pool : a.v_pool;
                        if (RS) {
                            uint8_t* page = pool + (phys * a.Hkv + h) * (int64_t)kRsPageBytes;
                            quant_row_e4m3rs_warp(x, page + slot * 128, reinterpret_cast<float*>(page + kRsScaleOff) + slot, lane);
                        } else {
                            uint8_t* page = pool + (phys * a.Hkv + h) * (int64_t)kMxPageBytes;
                            quant_row_mxfp4_warp(x, page + slot * 64, page + kMxScaleOff + slot * 4, lane);
                        }
                    }
                    if constexpr (kQImg) {
                        // this chunk's share of the row's q rows (r = draft token x Hq + head, rows
                        // j + Cb w4 + 4 Cb k), by the q packing rule into the tensor-core units' q tile
                        // images: unit row m = token x G + head % G of KV head head / G, row group m / 128,
                        // in the operand layout the QK MMA reads (published by the row's counter)
                        const int QH = a.Q * a.Hq;
                        for (int r = j + Cb * w4; r < QH; r += 4 * Cb) {
                            const int tq = r / a.Hq, h = r % a.Hq, kvh = h / a.G, m = tq * a.G + h % a.G;
                            const float4 x = reinterpret_cast<const float4*>(a.q_f32 + ((int64_t)b * QH + r) * kD)[lane];
                            uint8_t* img = a.q_img + (((int64_t)b * a.Hkv + kvh) * a.n_rg + m / kTcRows) * kQImgBytes;
                            *reinterpret_cast<uint32_t*>(img + sw128_chunk(m % kTcRows, lane >> 2, kTcRows) + 4 * (lane & 3)) =
                                pack_q4(x);
                        }
                    }
                };
                if (kTmem) sp.tmem = tmem_slot;
                scan_pages<NQ, kStepScanStages, kStepScanAcc>(sp, &idx_map, phys_s, np, p0, owner ? own_lo : np,
                                                             ctx - a.Q, a.Q, a.qidx + (int64_t)b * a.Q * kD,
                                                             a.scores + (int64_t)b * a.max_pages,
                                                             a.status, write_rows);
            }
            __syncthreads();
            if (threadIdx.x == 0) red_release_add(&a.row_cnt[kCounterStride * b], 1u);
        }
    }

    // ---------------- B. attention units ----------------
    if constexpr (TC) {
        if (!pt_stored) store_pt();
        // tensor memory for this CTA's units (S at column 0, O at 128); the tiles need a
        // 1024-byte-aligned base (checked; a CTA without it stages nothing and flags a timeout)
        const bool has_units = u0 < n_units;
        const bool smem_ok = (smem_u32(smem) & 1023u) == 0;
        if (has_units && !smem_ok && threadIdx.x == 0) flag_status(a.status, SMX_DEV_TIMEOUT);
        // (tensor memory was allocated at the start; the scan's accumulators are all read)
        tc_fence_before_sync();
        __syncthreads();
        tc_fence_after_sync();
        const uint32_t tmem = tmem_slot;
        if (!RS && has_units && warp < 4) {   // unit scales for the e4m3 q (A) of the block-scaled QK
            tmem_st4(tmem + ((uint32_t)(32 * warp) << 16) + kTcColSFA, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
            tc_fence_before_sync();
        }
        uint32_t gp = 0;          // pages staged by this CTA so far (sets the stages' phase parity)
        uint32_t mma_ph = 0;      // MMA completions seen so far (MXFP4: QK completions)
        uint32_t pv_ph = 0;       // MXFP4: PV completions seen so far
        uint32_t q_img_ph = 0;    // q tile image copies waited for (the parity of mbar_q)
        bool copies_ok = smem_ok; // false after a copy or MMA that did not finish: stage nothing more
        for (int u = u0; u < n_units; u += nC) {
            const int s = u % a.S, rg = (u / a.S) % a.n_rg, kvh = (u / (a.S * a.n_rg)) % a.Hkv;
            const int b = u / (a.S * a.n_rg * a.Hkv);
            const bool first = u == u0;
            const int ctx = clamp_ctx(first ? ctx_u0 : a.ctx_len[b], a.Q, a.max_pages, nullptr);
            const int n_pages = (ctx + kPage - 1) / kPage;
            const bool pt_cached = n_pages <= kPtCache;
            const int m_lo = rg * R, rows = min(M - m_lo, R);
            TcLane L;
            L.r = threadIdx.x & 127;
            L.h = threadIdx.x >> 7;
            L.valid = L.r < rows;
            L.pos = ctx - a.Q + (L.valid ? (m_lo + L.r) / a.G : 0);
            // the q tile, before the wait: the first unit's rows were staged at the start (or, when the
            // scan took the staging area, brought into L2 at the start)
            if constexpr (!kQImg) {
                if (first && q_stageable) {
                    if (!mbar_wait_bounded(&mbar_q, 0)) flag_status(a.status, SMX_DEV_TIMEOUT);
                    pack_q_tile_tc<RS>(smem + kTcV, rows, smem + kTcQ);
                } else {
                    pack_q_tile_tc_global<RS>(RS ? (const void*)a.q_bf16 : (const void*)a.q_f32, b, kvh, m_lo, rows, a.Q,
                                              a.Hq, a.G, smem + kTcQ);
                }
            }
            if (!first && pt_cached) {
                __syncthreads();   // the previous unit is done with pt_s
                for (int base = 0; base < n_pages; base += kPtPerThread * kStepWarps * 32) {
                    int32_t v[kPtPerThread];
    #pragma unroll
                    for (int k = 0; k < kPtPerThread; ++k) {
                        const int i = base + threadIdx.x + k * kStepWarps * 32;
                        v[k] = i < n_pages ? a.page_table[(int64_t)b * a.max_pages + i] : 0;
                    }
    #pragma unroll
                    for (int k = 0; k < kPtPerThread; ++k) {
                        const int i = base + threadIdx.x + k * kStepWarps * 32;
                        if (i < n_pages) pt_s[i] = v[k];
                    }
                }
            }
            if (threadIdx.x == 0 && !wait_geq_bounded(&a.row_cnt[kCounterStride * b], (uint32_t)row_chunks(b), a.wait_ns))
                flag_status(a.status, SMX_DEV_TIMEOUT);
            __syncthreads();   // the row is scored; the staged q rows are packed (the V and P tiles are free)
            // the unit's q tile: one copy of its image (written by the row's scanning CTAs, acquired
            // with the row's counter), in flight during the selection
            const bool q_img_issued = kQImg && copies_ok;
            if (q_img_issued && threadIdx.x == 0) {
                fence_proxy_async_global();
                mbar_arrive_expect_tx(&mbar_q, (uint32_t)kQImgBytes);
                bulk_g2s(smem + kTcQ, a.q_img + (((int64_t)b * a.Hkv + kvh) * a.n_rg + rg) * kQImgBytes,
                         (uint32_t)kQImgBytes, &mbar_q);
            }
            const int n_blocks = (n_pages + (1 << a.ppb_log2) - 1) >> a.ppb_log2;
            int k_eff;
            if constexpr (REUSE) {
                k_eff = given_selection(a, b, n_blocks, sel_all);
            } else {
                load_keys<true>(keys, a.scores + (int64_t)b * a.max_pages, n_pages);
                __syncthreads();
                if (a.ppb_log2) block_max_keys(keys, n_pages, a.ppb_log2);
                k_eff = block_select(keys, n_blocks, a.topk, sel_all, selsm);
            }
            const int lo = (int)(((int64_t)s * k_eff) / a.S), hi = (int)(((int64_t)(s + 1) * k_eff) / a.S);
            const int npg = (hi - lo) << a.ppb_log2;   // the partition's blocks as pages (one block: one page)
            auto resolve = [&](int i) {   // entry i of this partition: logical and physical page
                const int blk = sel_all[lo + (i >> a.ppb_log2)];
                int p = blk < 0 ? -1 : (blk << a.ppb_log2) + (i & ((1 << a.ppb_log2) - 1));
                if (p >= n_pages) p = -1;   // past the row in its last block: an empty page
                int ph = -1;
                if (p >= 0) {   // (a reused selection's bad id is -1: an empty page, flagged)
                    const int64_t v = pt_cached ? pt_s[p] : a.page_table[(int64_t)b * a.max_pages + p];
                    if (v >= 0 && v < a.n_pool) ph = (int)v;
                    else flag_status(a.status, SMX_DEV_BAD_PAGE_ID);
                }
                sel[i] = max(p, 0);
                selph[i] = ph;
                return ph;
            };
            // the first two pages' copies go out first; the row's new K/V rows (other CTAs' writes,
            // acquired above) are ordered before them
            if (threadIdx.x == 0 && copies_ok) {
                fence_proxy_async_global();
                fence_proxy_async_smem();
                for (int i = 0; i < 2 && i < npg; ++i) {
                    if constexpr (RS) {
                        { const int ph = resolve(i); attend_issue(sm, i, sel[i], ph, gp, a.k_pool, a.v_pool, a.Hkv, kvh, a.page_bytes); }
                    } else {
                        const int ph = resolve(i);
                        mx_issue(sm.raw, mbar, i, false, ph, gp, a.k_pool, a.Hkv, kvh, a.page_bytes);
                        mx_issue(sm.raw, mbar, i, true, ph, gp, a.v_pool, a.Hkv, kvh, a.page_bytes);
                    }
                }
            }
            for (int i = 2 + threadIdx.x; i < npg; i += blockDim.x) resolve(i);
            if (!REUSE && kvh == 0 && rg == 0 && s == 0) {
                for (int i = threadIdx.x; i < a.topk; i += blockDim.x)
                    a.topk_out[(int64_t)b * a.topk + i] = i < k_eff ? sel_all[i] : -1;
                if (threadIdx.x == 0) a.count_out[b] = k_eff;
            }
            bool q_ok = true;   // the q tile landed (thread 0; issued before the selection)
            if (q_img_issued && threadIdx.x == 0) {
                q_ok = mbar_wait_bounded(&mbar_q, q_img_ph & 1u);
                if (!q_ok) flag_status(a.status, SMX_DEV_TIMEOUT);
            }
            if (q_img_issued) ++q_img_ph;
            if (__syncthreads_or(!q_ok)) copies_ok = false;   // stage nothing more

            float m_run = -INFINITY, l = 0.0f;
            const bool run = copies_ok && npg > 0;
            if (run) {
                if constexpr (RS)
                    copies_ok = attend_pages_tc<RS>(smem, sm, sel, selph, npg, a.k_pool, a.v_pool, a.Hkv, kvh,
                                                    a.page_bytes, ctx, tmem, &mbar_mma[0], mma_ph, L, xch_tc, gp, m_run, l,
                                                    a.status);
                else
                    copies_ok = attend_pages_tc_mx(smem, sm.raw, mbar, sel, selph, npg, a.k_pool, a.v_pool, a.Hkv,
                                                   kvh, a.page_bytes, ctx, tmem, mbar_mma, mma_ph, pv_ph, L, xch_tc, gp,
                                                   m_run, l, a.status);
            }
            finish_partials_tc(L, tmem, run, m_run, l, xch_tc, smem, a.part_o, a.part_m, a.part_l, b, s, kvh, a.S, a.Q,
                               a.Hq, a.G, m_lo, rows);
            __syncthreads();
            if (threadIdx.x == 0) red_release_add(&a.grp_cnt[kCounterStride * ((b * a.Hkv + kvh) * a.n_rg + rg)], 1u);
        }
        tc_fence_before_sync();
        __syncthreads();
        if (warp == 0) {
            tc_fence_after_sync();
            tmem_dealloc(tmem, kTcCols);
        }

    } else {
        if (!pt_stored) store_pt();
        uint32_t gp = 0;          // pages staged by this CTA so far (sets the stages' phase parity)
        bool copies_ok = true;    // false after a copy that did not land: stage nothing more
        for (int u = u0; u < n_units; u += nC) {
            const int s = u % a.S, rg = (u / a.S) % a.n_rg, kvh = (u / (a.S * a.n_rg)) % a.Hkv;
            const int b = u / (a.S * a.n_rg * a.Hkv);
            const bool first = u == u0;
            const int ctx = clamp_ctx(first ? ctx_u0 : a.ctx_len[b], a.Q, a.max_pages, nullptr);
            const int n_pages = (ctx + kPage - 1) / kPage;
            const bool pt_cached = n_pages <= kPtCache;
            const AttendLane L = attend_lane(rg, R, a.row_warps, M, a.G);
            uint32_t qa[8][4];
            if (!first || !q_stageable) {
                // later units: q and the page table from global memory, before the wait
                if (RS) load_qa_bf16<false>(qa, a.q_bf16, L, b, kvh, a.Q, a.Hq, a.G);
                else load_qa_f32_e4m3(qa, a.q_f32, L, b, kvh, a.Q, a.Hq, a.G);
            } else {
                // the first unit's q rows were staged at the start: unpack them before the wait
                if (!mbar_wait_bounded(&mbar_q, 0)) flag_status(a.status, SMX_DEV_TIMEOUT);
                pack_staged_q<RS>(q_stage, min(M - rg * R, R));
                load_qa_packed(qa, q_stage, rg * R, L);
            }
            if (!first && pt_cached) {
                __syncthreads();   // the previous unit is done with pt_s
                for (int base = 0; base < n_pages; base += kPtPerThread * kStepWarps * 32) {
                    int32_t v[kPtPerThread];
    #pragma unroll
                    for (int k = 0; k < kPtPerThread; ++k) {
                        const int i = base + threadIdx.x + k * kStepWarps * 32;
                        v[k] = i < n_pages ? a.page_table[(int64_t)b * a.max_pages + i] : 0;
                    }
    #pragma unroll
                    for (int k = 0; k < kPtPerThread; ++k) {
                        const int i = base + threadIdx.x + k * kStepWarps * 32;
                        if (i < n_pages) pt_s[i] = v[k];
                    }
                }
            }
            if (threadIdx.x == 0 && !wait_geq_bounded(&a.row_cnt[kCounterStride * b], (uint32_t)row_chunks(b), a.wait_ns))
                flag_status(a.status, SMX_DEV_TIMEOUT);
            __syncthreads();
            const int n_blocks = (n_pages + (1 << a.ppb_log2) - 1) >> a.ppb_log2;
            int k_eff;
            if constexpr (REUSE) {
                __syncthreads();   // the staged q rows read (the page stages are free)
                k_eff = given_selection(a, b, n_blocks, sel_all);
            } else {
                load_keys<true>(keys, a.scores + (int64_t)b * a.max_pages, n_pages);
                __syncthreads();   // keys in place; the staged q rows read (the page stages are free)
                if (a.ppb_log2) block_max_keys(keys, n_pages, a.ppb_log2);
                k_eff = block_select(keys, n_blocks, a.topk, sel_all, selsm);
            }
            const int lo = (int)(((int64_t)s * k_eff) / a.S), hi = (int)(((int64_t)(s + 1) * k_eff) / a.S);
            const int npg = (hi - lo) << a.ppb_log2;   // the partition's blocks as pages (one block: one page)
            auto resolve = [&](int i) {   // entry i of this partition: logical and physical page
                const int blk = sel_all[lo + (i >> a.ppb_log2)];
                int p = blk < 0 ? -1 : (blk << a.ppb_log2) + (i & ((1 << a.ppb_log2) - 1));
                if (p >= n_pages) p = -1;   // past the row in its last block: an empty page
                int ph = -1;
                if (p >= 0) {   // (a reused selection's bad id is -1: an empty page, flagged)
                    const int64_t v = pt_cached ? pt_s[p] : a.page_table[(int64_t)b * a.max_pages + p];
                    if (v >= 0 && v < a.n_pool) ph = (int)v;
                    else flag_status(a.status, SMX_DEV_BAD_PAGE_ID);
                }
                sel[i] = max(p, 0);
                selph[i] = ph;
                return ph;
            };
            // the first two pages' copies go out first; the row's new K/V rows (other CTAs' writes,
            // acquired above) are ordered before them
            if (threadIdx.x == 0 && copies_ok) {
                fence_proxy_async_global();
                fence_proxy_async_smem();   // the staged q rows were read from the page stages
                for (int i = 0; i < 2 && i < npg; ++i)
                    { const int ph = resolve(i); attend_issue(sm, i, sel[i], ph, gp, a.k_pool, a.v_pool, a.Hkv, kvh, a.page_bytes); }
            }
            for (int i = 2 + threadIdx.x; i < npg; i += blockDim.x) resolve(i);
            if (!REUSE && kvh == 0 && rg == 0 && s == 0) {
                for (int i = threadIdx.x; i < a.topk; i += blockDim.x)
                    a.topk_out[(int64_t)b * a.topk + i] = i < k_eff ? sel_all[i] : -1;
                if (threadIdx.x == 0) a.count_out[b] = k_eff;
            }
            __syncthreads();

            float o[16][4];
    #pragma unroll
            for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.0f;
            float mrow0 = -INFINITY, mrow1 = -INFINITY, l0 = 0.0f, l1 = 0.0f;
            const int pos0 = ctx - a.Q + L.t0, pos1 = ctx - a.Q + L.t1;
            if (copies_ok)
                copies_ok = attend_pages<RS>(sm, sel, selph, npg, a.k_pool, a.v_pool, a.Hkv, kvh, a.page_bytes, ctx,
                                             qa, L, pos0, pos1, gp, o, mrow0, mrow1, l0, l1, a.status, true);
            finish_partials(sm, L, o, mrow0, mrow1, l0, l1, a.part_o, a.part_m, a.part_l, b, s, kvh, a.S, a.Q, a.Hq, a.G);
            __syncthreads();
            if (threadIdx.x == 0) red_release_add(&a.grp_cnt[kCounterStride * ((b * a.Hkv + kvh) * a.n_rg + rg)], 1u);
        }

    }

    // ---------------- C. merge: slice s of each unit's group ----------------
    const int QH = a.Q * a.Hq;
    for (int u = u0; u < n_units; u += nC) {
        const int s = u % a.S, rg = (u / a.S) % a.n_rg, kvh = (u / (a.S * a.n_rg)) % a.Hkv;
        const int b = u / (a.S * a.n_rg * a.Hkv);
        if (threadIdx.x == 0 && !wait_geq_bounded(&a.grp_cnt[kCounterStride * ((b * a.Hkv + kvh) * a.n_rg + rg)], (uint32_t)a.S, a.wait_ns))
            flag_status(a.status, SMX_DEV_TIMEOUT);
        __syncthreads();
        const int r_end = min((s + 1) * R / a.S, M - rg * R);
        for (int lr = s * R / a.S + warp; lr < r_end; lr += kStepWarps) {
            const int m = rg * R + lr;
            const int r = (m / a.G) * a.Hq + kvh * a.G + m % a.G;   // draft token x Hq + head
            merge_row<true>(a.part_o, a.part_m, a.part_l, (int64_t)b * a.S * QH + r, QH, a.S,
                            a.out + ((int64_t)b * QH + r) * kD);
        }
    }

    // ---------------- D. the last CTA out clears the counters ----------------
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        is_last = atomicAdd(a.done_cnt, 1u) == (uint32_t)nC - 1;
        if (is_last) __threadfence();   // every other CTA's counter updates come before the reset
    }
    __syncthreads();
    if (is_last) {
        for (int i = threadIdx.x; i < a.B; i += blockDim.x) a.row_cnt[kCounterStride * i] = 0;
        for (int i = threadIdx.x; i < a.B * a.Hkv * a.n_rg; i += blockDim.x) a.grp_cnt[kCounterStride * i] = 0;
        if (threadIdx.x == 0) *a.done_cnt = 0;
    }
}

// ---- host side -------------------------------------------------------------------------------------
// Attention rows per unit: 128 on the tensor-core path, 16 x row warps (<= 64) on mma.sync.
static int unit_rows(const smx_shape_t& s, bool tc) {
    const int M = (s.Hq / s.Hkv) * s.Q;
    return tc ? kTcRows : 16 * min(kAttnMaxWarps / 2, (M + 15) / 16);
}

StepGeom step_geom(const smx_shape_t& s) { return step_geom(s, false); }

size_t step_q_image_bytes(const smx_shape_t& s) {
    const int M = (s.Hq / s.Hkv) * s.Q;
    return (size_t)s.B * s.Hkv * ((M + kTcRows - 1) / kTcRows) * kQImgBytes;
}

StepGeom step_geom(const smx_shape_t& s, bool tc) {
    StepGeom g;
    const int M = (s.Hq / s.Hkv) * s.Q;
    g.rows_per_cta = unit_rows(s, tc);
    g.row_warps = g.rows_per_cta / 16;
    g.n_rg = (M + g.rows_per_cta - 1) / g.rows_per_cta;
    g.page_bytes = s.kv_format == SMX_KV_E4M3_ROWSCALE ? kRsPageBytes : kMxPageBytes;
    const size_t ppb = s.pages_per_block > 1 ? (size_t)s.pages_per_block : 1;
    g.smem = tc ? attend_tc_smem_bytes(g.page_bytes) + 8 * ppb * (size_t)s.topk
                : attend_smem_bytes(g.page_bytes) + (8 * ppb + 4) * (size_t)s.topk;
    // the tensor-core path's index scan shares the space (plus slack to align it to 1 KB)
    const int nq = s.Q > 8 ? 16 : 8;
    const size_t scan = (size_t)kStepQFront + scan_smem_bytes(kStepScanStages, scan_acc_stages(nq, 384), nq) + 1024;
    if (tc && g.smem < scan) g.smem = scan;
    // counters for the larger (mma.sync) group count, so the workspace does not depend on the path
    const int rg64 = (M + unit_rows(s, false) - 1) / unit_rows(s, false);
    g.n_counters = kCounterStride * ((size_t)s.B + (size_t)s.B * s.Hkv * rg64 + 1);
    return g;
}

template <bool RS, int NT, bool TC, bool REUSE>
static const void* step_fn() {
    return reinterpret_cast<const void*>(decode_step_kernel<RS, NT, TC, REUSE>);
}

// The step kernel variant: FP8-KV pages (rs), 9..16 query tokens (nt2: two n-tiles in the
// scorer), tensor-core attention (tc), a reused selection (reuse: no scorer, so one n-tile form).
static const void* step_fn(bool rs, bool nt2, bool tc, bool reuse = false) {
    if (reuse) {
        if (tc) return rs ? step_fn<true, 1, true, true>() : step_fn<false, 1, true, true>();
        return rs ? step_fn<true, 1, false, true>() : step_fn<false, 1, false, true>();
    }
    if (tc) return rs ? (nt2 ? step_fn<true, 2, true, false>() : step_fn<true, 1, true, false>())
                      : (nt2 ? step_fn<false, 2, true, false>() : step_fn<false, 1, true, false>());
    return rs ? (nt2 ? step_fn<true, 2, false, false>() : step_fn<true, 1, false, false>())
              : (nt2 ? step_fn<false, 2, false, false>() : step_fn<false, 1, false, false>());
}

// Resident CTAs of the step kernel on the current device (cached per device, kernel and size).
static int step_max_ctas(const void* fn, size_t smem) {
    struct Entry { int dev; const void* fn; size_t smem; int n; };
    static std::mutex mu;
    static Entry seen[32];
    static int n_seen = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < n_seen; ++i)
        if (seen[i].dev == dev && seen[i].fn == fn && seen[i].smem == smem) return seen[i].n;
    int sms = 0, per_sm = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kStepWarps * 32, smem) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    const int n = sms * min(per_sm, 1);
    if (n_seen < 32) seen[n_seen++] = Entry{dev, fn, smem, n};
    return n;
}

// The tensor-core attention when the 64-row mma.sync units would need more than one wave of
// CTAs: per query row and page it does about 1.2x the work per SM of mma.sync (measured), but
// with half as many units; with one wave, twice the CTAs in flight win (the step is latency-bound).
static bool use_tc(const smx_shape_t& s, int max_ctas) {
    const int M = (s.Hq / s.Hkv) * s.Q;
    if (M <= 64 || max_ctas < 1) return false;
    const int64_t units64 = (int64_t)s.B * s.Hkv * ((M + 63) / 64) * s.num_splits;
    return units64 > max_ctas;
}

bool decode_step_uses_tc(const smx_shape_t& s) {
    const StepGeom geo = step_geom(s, true);
    const void* fn = step_fn(s.kv_format == SMX_KV_E4M3_ROWSCALE, s.Q > 8, true);
    if (ensure_smem_attr(fn, (int)geo.smem) != cudaSuccess) {
        (void)cudaGetLastError();
        return false;
    }
    return use_tc(s, step_max_ctas(fn, geo.smem));
}

// One cooperative launch of a step kernel variant (every CTA resident, at most one per SM).
static cudaError_t launch_step_kernel(const void* fn, int n_ctas, size_t smem, cudaStream_t st, StepArgs a,
                                      const CUtensorMap& map) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(n_ctas);
    cfg.blockDim = dim3(kStepWarps * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    // programmatic dependent launch: the kernel's on-chip set-up may overlap the previous kernel's
    // tail; it waits for that kernel's completion before its first global access
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    static bool pdl_ok = true;   // cleared if the runtime refuses the pair of attributes
    cfg.numAttrs = pdl_ok ? 2 : 1;
    auto kernel = reinterpret_cast<void (*)(StepArgs, CUtensorMap)>(const_cast<void*>(fn));
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, a, map);
    if (e != cudaSuccess && pdl_ok && e != cudaErrorStreamCaptureInvalidated && e != cudaErrorStreamCaptureUnsupported) {
        (void)cudaGetLastError();
        pdl_ok = false;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, kernel, a, map);
    }
    return e;
}

cudaError_t launch_decode_step(const smx_shape_t& s, const StepIO& io, cudaStream_t st, bool reuse) {
    const bool rs = s.kv_format == SMX_KV_E4M3_ROWSCALE;
    const bool nt2 = s.Q > 8;
    const bool tc = decode_step_uses_tc(s);
    const StepGeom geo = step_geom(s, tc);
    const void* fn = step_fn(rs, nt2, tc, reuse);
    cudaError_t e = ensure_smem_attr(fn, (int)geo.smem);
    if (e != cudaSuccess) return e;
    const int max_ctas = step_max_ctas(fn, geo.smem);
    if (max_ctas < 1) return cudaErrorCooperativeLaunchTooLarge;

    StepArgs a = {};
    a.q_f32 = io.q_f32; a.q_bf16 = io.q_bf16; a.qidx = io.qidx;
    a.k_new = io.k_new; a.v_new = io.v_new; a.kidx_new = io.kidx_new;
    a.page_table = io.page_table; a.ctx_len = io.ctx_len;
    a.idx_pool = io.idx_pool; a.k_pool = io.k_pool; a.v_pool = io.v_pool;
    a.topk_out = io.topk_out; a.count_out = io.count_out; a.out = io.out; a.status = io.status;
    a.row_cnt = io.counters;
    a.grp_cnt = io.counters + kCounterStride * s.B;
    a.done_cnt = io.counters + kCounterStride * (s.B + (size_t)s.B * s.Hkv * geo.n_rg);
    a.scores = io.scores; a.part_o = io.part_o; a.part_m = io.part_m; a.part_l = io.part_l; a.q_img = io.q_img;
    a.n_pool = s.n_pool_pages;
    a.B = s.B; a.Q = s.Q; a.Hq = s.Hq; a.Hkv = s.Hkv; a.G = s.Hq / s.Hkv; a.max_pages = s.max_pages_per_row;
    a.topk = s.topk; a.S = s.num_splits;
    a.row_warps = geo.row_warps; a.rows_per_cta = geo.rows_per_cta; a.n_rg = geo.n_rg; a.page_bytes = geo.page_bytes;
    a.topk_in = io.topk_in; a.count_in = io.count_in;
    a.ppb_log2 = s.pages_per_block == 4 ? 2 : s.pages_per_block == 2 ? 1 : 0;
    a.wait_ns = wait_limit_ns();

    // grid: enough CTAs for every attention unit and for two pages each, at most one per SM
    const int64_t n_units = (int64_t)s.B * s.Hkv * geo.n_rg * s.num_splits;
    const int64_t slots = (int64_t)s.B * s.max_pages_per_row;
    CUtensorMap map;   // the index pool for the scan (unused by a reusing layer)
    memset(&map, 0, sizeof(map));
    if (!reuse) {
        e = encode_index_map(&map, io.idx_pool, s.n_pool_pages);
        if (e != cudaSuccess) return e;
    }
    if (reuse) {
        // no scoring: chunks of a row only write its new K/V rows, one row per warp
        const int kv_rows = s.Q * 2 * s.Hkv;
        const int C = (kv_rows + kStepWarps - 1) / kStepWarps;
        const int64_t want = n_units > (int64_t)s.B * C ? n_units : (int64_t)s.B * C;
        a.chunk_pages = 0;
        a.chunks_per_row = C;
        const int n_ctas = (int)(want < max_ctas ? want : max_ctas);
        return launch_step_kernel(fn, n_ctas, geo.smem, st, a, map);
    }
    const int64_t want = n_units > (slots + 1) / 2 ? n_units : (slots + 1) / 2;
    const int n_ctas = (int)(want < max_ctas ? want : max_ctas);
    int64_t P = (slots + n_ctas - 1) / n_ctas;
    if (P > kStepMaxChunk) P = kStepMaxChunk;
    a.chunk_pages = (int)P;
    a.chunks_per_row = (int)((s.max_pages_per_row + P - 1) / P);
    return launch_step_kernel(fn, n_ctas, geo.smem, st, a, map);
}

}  // namespace smx

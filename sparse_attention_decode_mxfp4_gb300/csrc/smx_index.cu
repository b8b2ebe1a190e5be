// smx_index.cu -- a3 (page scores from the MXFP4 index cache), optionally with a1 fused in, and
// the standalone a4 (top-k pages per row).
//
// [ATOM-2812] "Mono decode over the MXFP4 KV and index caches", commit "--index-cache-dtype
// mxfp4": the scorer reads each index page as 16 B key loads plus a dword of E8M0 scales and
// widens the fp4 keys for a 16-bit MMA against the index query; K1 writes the new index-K rows
// before the scorer reads them; commit "MXFP4 main KV": the selected blocks (one 128-token page
// each) fill the row's sparse table.
//
// GB300 form of the scorer. A CTA of 8 warps walks a range of pages of one row, two pages at a
// time; a warp scores 32 tokens (two 16-token tiles) of a page. Lane (g, t) of the m16n8k16 MMA
// loads 16 B (= 32 elements of scale group t) of token rows g and g+8 of each tile straight
// into registers (a warp instruction covers 512 contiguous bytes), converts byte pairs with the
// hardware E2M1 -> f16x2 conversion, and multiplies group t by 2^(s_t - max_g s_g) so that one
// fp32 accumulator serves the whole row; the row's common factor 2^(max_g s_g) and the query's
// power-of-two factor are applied to the fp32 result. The index query is held in f16 after a
// per-query power-of-two rescale that puts its largest element in [2^14, 2^15): every bf16
// element within 2^31 of that maximum is exact in f16, so products are exact and only the fp32
// accumulation rounds. The K permutation of the MMA is chosen so that each lane's 16 contiguous
// bytes are its A fragment: k-step s takes bytes 2s and 2s+1 of every lane's group.
//
// Fused insert: a CTA whose page range holds some of the row's new token positions quantises
// those index-K rows (and, for the rows it owns, the K and V rows) before scoring, fences, and
// then reads its pages through L2 so that it sees its own writes.
#include <math.h>

#include "smx_device.cuh"
#include "smx_internal.h"
#include "smx_select.cuh"

namespace smx {

struct IndexArgs {
    const uint16_t* qidx;     // [B][Q][128] bf16 bits
    uint8_t* pool;            // [n_pool][8704]
    const int32_t* page_table;
    const int32_t* ctx_len;
    float* scores;            // [B][max_pages]
    int32_t* status;
    int64_t n_pool;
    int Q, max_pages, pages_per_cta;
    // fused insert (k_new == nullptr: none)
    const float* k_new;       // [B][Q][Hkv][128]
    const float* v_new;
    const float* kidx_new;    // [B][Q][128]
    uint8_t* k_pool;
    uint8_t* v_pool;
    int Hkv, kv_format;
    int pdl;                  // wait for the preceding grid before touching memory
    // fused step: q packed once for the split stage, and the row's selection made once by the
    // last CTA of the row to finish (sel_pages == nullptr: none)
    const float* q_f32;       // MXFP4 K/V: [B][Q][Hq][128] to pack (nullptr: nothing to pack)
    uint16_t* qbf;            // [B][Q][Hq][128] bf16 of the packed q (exact)
    int q_row_elems;          // Q * Hq * 128
    int32_t* arrivals;        // [B] CTAs of the row that have finished; the last one resets it to 0
    int32_t* sel_pages;       // [B][topk] selected logical page ids, ascending, -1 padded
    int32_t* sel_phys;        // [B][topk] their physical ids (-1: none or out of range)
    int32_t* sel_count;       // [B] k_eff
    int32_t* topk_out;        // [B][topk] (the caller's output)
    int32_t* count_out;       // [B]
    int topk;
};

constexpr int kIdxWarps = 8;

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t h16) { return __uint_as_float(h16 << 16); }

// x * 2^k for any k a float exponent difference can take (two exact power-of-two steps).
__device__ __forceinline__ float mul_exp2(float x, int k) {
    const int k1 = max(-126, min(127, k / 2));
    const int k2 = max(-126, min(127, k - k1));
    return x * exp2i_normal(k1) * exp2i_normal(k2);
}

// One lane's share of one 16-token tile: 16 B of nibbles of token rows g and g+8 and the rows'
// scale words. Pages are read through L2 (a CTA that inserted rows must see its own writes).
struct TileFrag {
    uint4 c0, c1;
    uint32_t sw0, sw1;
};

__device__ __forceinline__ void load_tile(TileFrag& f, const uint8_t* page, int tile, int g, int t) {
    const int r0 = tile * 16 + g, r1 = r0 + 8;
    f.c0 = ldg_cg_v4(page + r0 * 64 + 16 * t);
    f.c1 = ldg_cg_v4(page + r1 * 64 + 16 * t);
    f.sw0 = ldg_cg_u32(page + kMxScaleOff + 4 * r0);
    f.sw1 = ldg_cg_u32(page + kMxScaleOff + 4 * r1);
}

// Max over this lane's scores of one tile (two token rows x its query columns).
template <int NT>
__device__ __forceinline__ float score_tile(const TileFrag& f, const uint32_t (&qf)[NT][16], const int (&sig_c)[NT][2],
                                            int p, int tile, int g, int t, int lim, int Q) {
    const int r0 = tile * 16 + g, r1 = r0 + 8;
    uint32_t f0, f1;   // f16x2 of 2^(s_t - max s) per row
    int e0, e1;        // max scale byte per row (0xFF marks a NaN scale)
    {
        const uint32_t a0 = f.sw0, a1 = f.sw1;
        const uint32_t m0 = max(max(a0 & 0xFF, (a0 >> 8) & 0xFF), max((a0 >> 16) & 0xFF, a0 >> 24));
        const uint32_t m1 = max(max(a1 & 0xFF, (a1 >> 8) & 0xFF), max((a1 >> 16) & 0xFF, a1 >> 24));
        const int rel0 = (int)((a0 >> (8 * t)) & 0xFF) - (int)m0;
        const int rel1 = (int)((a1 >> (8 * t)) & 0xFF) - (int)m1;
        const __half h0 = rel0 >= -22 ? __float2half_rn(exp2i_normal(rel0)) : __float2half_rn(0.0f);
        const __half h1 = rel1 >= -22 ? __float2half_rn(exp2i_normal(rel1)) : __float2half_rn(0.0f);
        const __half2 hh0 = __halves2half2(h0, h0), hh1 = __halves2half2(h1, h1);
        f0 = *reinterpret_cast<const uint32_t*>(&hh0);
        f1 = *reinterpret_cast<const uint32_t*>(&hh1);
        e0 = (int)m0;
        e1 = (int)m1;
    }
    // two accumulator chains per n-tile (even and odd k-steps) for more parallel MMAs
    float acc[NT][2][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int h = 0; h < 2; ++h) acc[nt][h][0] = acc[nt][h][1] = acc[nt][h][2] = acc[nt][h][3] = 0.0f;
    const uint32_t w0[4] = {f.c0.x, f.c0.y, f.c0.z, f.c0.w};
    const uint32_t w1[4] = {f.c1.x, f.c1.y, f.c1.z, f.c1.w};
#pragma unroll
    for (int wi = 0; wi < 4; ++wi) {
        uint32_t x0, x1, x2, x3, y0, y1, y2, y3;
        e2m1x8_to_f16x2(w0[wi], x0, x1, x2, x3);
        e2m1x8_to_f16x2(w1[wi], y0, y1, y2, y3);
        x0 = hmul2_u32(x0, f0); x1 = hmul2_u32(x1, f0); x2 = hmul2_u32(x2, f0); x3 = hmul2_u32(x3, f0);
        y0 = hmul2_u32(y0, f1); y1 = hmul2_u32(y1, f1); y2 = hmul2_u32(y2, f1); y3 = hmul2_u32(y3, f1);
        const int s0 = 2 * wi, s1 = 2 * wi + 1;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            mma_f16_16816(acc[nt][0], x0, y0, x1, y1, qf[nt][2 * s0], qf[nt][2 * s0 + 1]);
            mma_f16_16816(acc[nt][1], x2, y2, x3, y3, qf[nt][2 * s1], qf[nt][2 * s1 + 1]);
        }
    }
    const int j0 = p * kPage + r0, j1 = p * kPage + r1;
    float best = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int col = c & 1;
            const int n = nt * 8 + 2 * t + col;
            const int j = (c < 2) ? j0 : j1;
            const int e = (c < 2) ? e0 : e1;
            const bool valid = (n < Q) && (j <= lim + n) && (e != 0xFF);
            const float v = mul_exp2(acc[nt][0][c] + acc[nt][1][c], (e - 127) - sig_c[nt][col]);
            best = valid ? fmaxf(best, v) : best;
        }
    }
    return best;
}

constexpr int kIdxMaxPpc = 64;   // page-table entries of one CTA staged in shared memory

template <int NT>
__global__ void __launch_bounds__(kIdxWarps * 32, 2) index_score_kernel(IndexArgs a) {
    __shared__ __align__(16) uint32_t qh[16][64];  // f16x2 of q' per query, natural dim order
    __shared__ int sig[16];
    __shared__ float red[2][kIdxWarps];
    __shared__ int64_t phys_s[kIdxMaxPpc];

    const int b = blockIdx.y;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, t = lane & 3;
    if (a.pdl) pdl_wait();
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

    // ---- fused insert. The index-K rows of the new tokens are written by the CTA that scores
    // their page (before it reads the page); the K and V rows, read only by the split stage, are
    // spread over all CTAs of the row.
    const int first_new = ctx - a.Q;
    const bool wrote = a.k_new != nullptr && p_begin < p_end && first_new / kPage < p_end &&
                       (ctx - 1) / kPage >= p_begin;
    if (a.k_new != nullptr) {
        const int kv_rows = a.Q * 2 * a.Hkv;
        // index-K rows of this CTA's pages: one warp per row
        if (wrote && warp < a.Q) {
            for (int tq = warp; tq < a.Q; tq += kIdxWarps) {
                const int pos = first_new + tq, pg = pos / kPage;
                if (pos < 0 || pg < p_begin || pg >= p_end) continue;
                const int64_t phys = a.page_table[(int64_t)b * a.max_pages + pg];
                if (phys < 0 || phys >= a.n_pool) {
                    if (lane == 0) flag_status(a.status, SMX_DEV_BAD_PAGE_ID);
                    continue;
                }
                const float4 x = reinterpret_cast<const float4*>(a.kidx_new + ((int64_t)b * a.Q + tq) * kD)[lane];
                uint8_t* page = a.pool + phys * kMxPageBytes;
                quant_row_mxfp4_warp(x, page + (pos % kPage) * 64, page + kMxScaleOff + (pos % kPage) * 4, lane);
            }
        }
                // K/V rows: row r of the row's Q x 2 x Hkv goes to CTA r % gridDim.x, warp (r / gridDim.x) % 8
        for (int r = blockIdx.x + gridDim.x * warp; r < kv_rows; r += gridDim.x * kIdxWarps) {
            const int tq = r / (2 * a.Hkv), kind = r % (2 * a.Hkv);   // kind < Hkv: K head, else V head
            const int pos = first_new + tq;
            if (pos < 0) continue;
            const int64_t phys = a.page_table[(int64_t)b * a.max_pages + pos / kPage];
            if (phys < 0 || phys >= a.n_pool) {
                if (lane == 0) flag_status(a.status, SMX_DEV_BAD_PAGE_ID);
                continue;
            }
            const int h = kind % a.Hkv, slot = pos % kPage;
            const int64_t tok = (int64_t)b * a.Q + tq;
            const float4 x = reinterpret_cast<const float4*>((kind < a.Hkv ? a.k_new : a.v_new) + (tok * a.Hkv + h) * kD)[lane];
            uint8_t* pool = kind < a.Hkv ? a.k_pool : a.v_pool;
            if (a.kv_format == SMX_KV_E4M3_ROWSCALE) {
                uint8_t* page = pool + (phys * a.Hkv + h) * (int64_t)kRsPageBytes;
                quant_row_e4m3rs_warp(x, page + slot * 128, reinterpret_cast<float*>(page + kRsScaleOff) + slot, lane);
            } else {
                uint8_t* page = pool + (phys * a.Hkv + h) * (int64_t)kMxPageBytes;
                quant_row_mxfp4_warp(x, page + slot * 64, page + kMxScaleOff + slot * 4, lane);
            }
        }
        if (wrote) __threadfence();
    }
    __syncthreads();   // page-table entries staged; inserted rows written and fenced

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
        if (ph >= 0) load_tile(cur, a.pool + ph * kMxPageBytes, tile0, g, t);
    }

    // ---- index query: f16 with a per-query power-of-two factor 2^sigma, staged in smem ----
    for (int n = warp; n < a.Q; n += kIdxWarps) {
        const uint2 v = reinterpret_cast<const uint2*>(a.qidx + ((int64_t)b * a.Q + n) * kD)[lane];  // dims 4l..4l+3
        uint32_t mx = max(max(v.x & 0x7FFFu, (v.x >> 16) & 0x7FFFu), max(v.y & 0x7FFFu, (v.y >> 16) & 0x7FFFu));
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
        int sigma = 0;
        if (mx != 0) {
            const int e = (int)(mx >> 7);
            const int E = e ? e - 127 : -133 + (31 - __clz((int)(mx & 0x7F)));
            sigma = 14 - E;
        }
        const __half2 h0 = __floats2half2_rn(mul_exp2(bf16_bits_to_f32(v.x & 0xFFFFu), sigma),
                                             mul_exp2(bf16_bits_to_f32(v.x >> 16), sigma));
        const __half2 h1 = __floats2half2_rn(mul_exp2(bf16_bits_to_f32(v.y & 0xFFFFu), sigma),
                                             mul_exp2(bf16_bits_to_f32(v.y >> 16), sigma));
        qh[n][2 * lane] = *reinterpret_cast<const uint32_t*>(&h0);
        qh[n][2 * lane + 1] = *reinterpret_cast<const uint32_t*>(&h1);
        if (lane == 0) sig[n] = sigma;
    }
    for (int n = a.Q + warp; n < 8 * NT; n += kIdxWarps) {
        qh[n][2 * lane] = 0;
        qh[n][2 * lane + 1] = 0;
        if (lane == 0) sig[n] = 0;
    }
    __syncthreads();
    // B fragments: lane (g, t) of n-tile nt holds q'[nt*8+g][32t .. 32t+31]
    uint32_t qf[NT][16];
    int sig_c[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const uint4* src = reinterpret_cast<const uint4*>(&qh[nt * 8 + g][16 * t]);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint4 v = src[i];
            qf[nt][4 * i] = v.x; qf[nt][4 * i + 1] = v.y; qf[nt][4 * i + 2] = v.z; qf[nt][4 * i + 3] = v.w;
        }
        sig_c[nt][0] = sig[nt * 8 + 2 * t];
        sig_c[nt][1] = sig[nt * 8 + 2 * t + 1];
    }

    // fused step: this CTA's slice of q[b] packed to e4m3 and stored as (exact) bf16
    if (a.q_f32 != nullptr) {
        const int n4 = a.q_row_elems / 4;
        const int per = (n4 + gridDim.x - 1) / gridDim.x;
        const int i_end = min(n4, (int)(blockIdx.x + 1) * per);
        const float4* src = reinterpret_cast<const float4*>(a.q_f32 + (int64_t)b * a.q_row_elems);
        uint2* dst = reinterpret_cast<uint2*>(a.qbf + (int64_t)b * a.q_row_elems);
        for (int i = blockIdx.x * per + threadIdx.x; i < i_end; i += blockDim.x) {
            const uint32_t w = pack_q4(src[i]);
            const float2 lo = f16x2_to_f32x2(e4m3x2_to_f16x2(w & 0xFFFF));
            const float2 hi = f16x2_to_f32x2(e4m3x2_to_f16x2(w >> 16));
            dst[i] = make_uint2(f32x2_to_bf16x2(lo.x, lo.y), f32x2_to_bf16x2(hi.x, hi.y));
        }
    }

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
            if (phn >= 0) load_tile(nxt, a.pool + phn * kMxPageBytes, tile0 + ((q + 1) & 1), g, t);
        }
        if (ph >= 0) best = fmaxf(best, score_tile<NT>(cur, qf, sig_c, p, tile0 + (q & 1), g, t, lim, a.Q));
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
    // the split stage's CTAs may launch now onto the SMs this grid leaves idle; they still wait
    // for this whole grid (the selection included) before reading anything it writes
    pdl_trigger();
    if (a.sel_pages != nullptr) {
        __shared__ int is_last;
        __threadfence();   // this thread's page scores are visible device-wide
        __syncthreads();
        if (threadIdx.x == 0) {
            is_last = atomicAdd(&a.arrivals[b], 1) == (int)gridDim.x - 1;
        }
        __syncthreads();
        if (is_last) {
            // every CTA of the row fenced its scores before arriving: read them through L2
            __threadfence();
            extern __shared__ __align__(16) uint32_t dyn[];
            uint32_t* keys = dyn;
            int* sel = reinterpret_cast<int*>(dyn + a.max_pages);
            __shared__ SelectSmem selsm;
            const float* srow = a.scores + (int64_t)b * a.max_pages;
            for (int i = threadIdx.x; i < n_pages; i += blockDim.x) keys[i] = score_key(ldg_cg_f32(srow + i));
            __syncthreads();
            const int k_eff = block_select(keys, n_pages, a.topk, sel, selsm);
            for (int i = threadIdx.x; i < a.topk; i += blockDim.x) {
                const int pg = i < k_eff ? sel[i] : -1;
                int32_t ph = -1;
                if (pg >= 0) {
                    const int64_t v = a.page_table[(int64_t)b * a.max_pages + pg];
                    if (v >= 0 && v < a.n_pool) ph = (int32_t)v;
                    else flag_status(a.status, SMX_DEV_BAD_PAGE_ID);
                }
                a.sel_pages[(int64_t)b * a.topk + i] = pg;
                a.sel_phys[(int64_t)b * a.topk + i] = ph;
                a.topk_out[(int64_t)b * a.topk + i] = pg;
            }
            if (threadIdx.x == 0) {
                a.sel_count[b] = k_eff;
                a.count_out[b] = k_eff;
                a.arrivals[b] = 0;
            }
        }
    }
}

// ---- standalone a4: one block per row ------------------------------------------------------------
constexpr int kTopkThreads = 512;

__global__ void __launch_bounds__(kTopkThreads) topk_kernel(const float* __restrict__ scores,
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
    for (int i = threadIdx.x; i < n; i += blockDim.x) keys[i] = score_key(s[i]);
    __syncthreads();
    int32_t* outp = topk_pages + (int64_t)b * topk;
    const int k_eff = block_select(keys, n, topk, outp, sm);
    for (int i = k_eff + threadIdx.x; i < topk; i += blockDim.x) outp[i] = -1;
    if (threadIdx.x == 0) topk_count[b] = k_eff;
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

static int index_pages_per_cta(const smx_shape_t& s) {
    // one wave: two CTAs of 8 warps per SM (their registers allow two) over all rows, an even
    // number of pages each
    const int64_t target = 2 * (int64_t)sm_count();
    int64_t ppc = ((int64_t)s.max_pages_per_row * s.B + target - 1) / target;
    ppc = (ppc + 1) & ~1LL;
    if (ppc > kIdxMaxPpc) ppc = kIdxMaxPpc;
    return (int)(ppc < 2 ? 2 : ppc);
}

cudaError_t launch_index(const smx_shape_t& s, const uint16_t* qidx, uint8_t* idx_pool,
                         const int32_t* page_table, const int32_t* ctx_len, float* scores, int32_t* status,
                         const float* k_new, const float* v_new, const float* kidx_new, uint8_t* k_pool,
                         uint8_t* v_pool, bool pdl, cudaStream_t st, const FusedSelect* fs) {
    IndexArgs a = {};
    if (fs) {
        a.q_f32 = fs->q_f32; a.qbf = fs->qbf; a.q_row_elems = s.Q * s.Hq * 128; a.arrivals = fs->arrivals;
        a.sel_pages = fs->sel_pages; a.sel_phys = fs->sel_phys; a.sel_count = fs->sel_count;
        a.topk_out = fs->topk_out; a.count_out = fs->count_out;
    }
    a.topk = s.topk;
    a.qidx = qidx; a.pool = idx_pool; a.page_table = page_table; a.ctx_len = ctx_len; a.scores = scores;
    a.status = status; a.n_pool = s.n_pool_pages; a.Q = s.Q; a.max_pages = s.max_pages_per_row;
    a.pages_per_cta = index_pages_per_cta(s);
    a.k_new = k_new; a.v_new = v_new; a.kidx_new = kidx_new; a.k_pool = k_pool; a.v_pool = v_pool;
    a.Hkv = s.Hkv; a.kv_format = s.kv_format; a.pdl = pdl ? 1 : 0;
    dim3 grid((s.max_pages_per_row + a.pages_per_cta - 1) / a.pages_per_cta, s.B);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kIdxWarps * 32);
    cfg.dynamicSmemBytes = fs ? 4 * ((size_t)s.max_pages_per_row + s.topk) : 0;
    cfg.stream = st;
    if (fs) {
        const void* kfn = s.Q <= 8 ? reinterpret_cast<const void*>(index_score_kernel<1>)
                                   : reinterpret_cast<const void*>(index_score_kernel<2>);
        cudaError_t e = ensure_smem_attr(kfn, (int)cfg.dynamicSmemBytes);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    if (s.Q <= 8) return cudaLaunchKernelEx(&cfg, index_score_kernel<1>, a);
    return cudaLaunchKernelEx(&cfg, index_score_kernel<2>, a);
}

cudaError_t launch_index_scores(const smx_shape_t& s, const uint16_t* qidx, const uint8_t* idx_pool,
                                const int32_t* page_table, const int32_t* ctx_len, float* scores,
                                int32_t* status, cudaStream_t st) {
    return launch_index(s, qidx, const_cast<uint8_t*>(idx_pool), page_table, ctx_len, scores, status, nullptr,
                        nullptr, nullptr, nullptr, nullptr, false, st, nullptr);
}

cudaError_t launch_topk(const smx_shape_t& s, const float* scores, const int32_t* ctx_len,
                        int32_t* topk_pages, int32_t* topk_count, cudaStream_t st) {
    const int smem = 4 * s.max_pages_per_row;
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(topk_kernel), smem);
    if (e != cudaSuccess) return e;
    topk_kernel<<<s.B, kTopkThreads, smem, st>>>(scores, ctx_len, topk_pages, topk_count, s.max_pages_per_row,
                                                  s.topk);
    return cudaGetLastError();
}

}  // namespace smx

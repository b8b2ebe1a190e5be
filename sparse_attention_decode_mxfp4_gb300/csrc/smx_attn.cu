// smx_attn.cu -- the standalone a5 (split-K attention over given selected pages) and a6 (merge)
// kernels of the C ABI. The per-page attention, the partial store and the row merge live in
// smx_attend.cuh (shared with the fused decode step).
//
// [ATOM-2812] "Mono decode over the MXFP4 KV and index caches", commit "MXFP4 main KV": one
// partition of the selected pages per split CTA, (sp_o, sp_m, sp_l) per partition, then the merge.
#include <math.h>

#include "smx_attend.cuh"
#include "smx_device.cuh"
#include "smx_internal.h"

namespace smx {

struct AttnArgs {
    const void* q;            // e4m3 bytes (MXFP4 K/V) or bf16 bits (FP8-KV), [B][Q][Hq][128]
    const uint8_t* k_pool;
    const uint8_t* v_pool;
    const int32_t* page_table;
    const int32_t* ctx_len;
    const int32_t* topk_pages;
    const int32_t* topk_count;
    float* part_o;
    float* part_m;
    float* part_l;
    int32_t* status;
    int64_t n_pool;
    int B, Q, Hq, Hkv, G, max_pages, topk, S, rows_per_cta, n_row_groups, page_bytes;
    int nv;            // NVFP4 K/V pages
    float qk_scale;    // log2(e) / sqrt(128), times the K pool's NVFP4 scale
    float o_scale;     // 1, or the V pool's NVFP4 scale
};

// grid (S, B, Hkv x row groups), 2 x row_warps warps
template <bool RS>
__global__ void __launch_bounds__(kAttnMaxWarps * 32, 1) attn_split_kernel(AttnArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t mbar[2];
    __shared__ int stage_page[2];
    const AttendSmem sm = attend_smem(smem, a.page_bytes, mbar, stage_page);
    int* sel = reinterpret_cast<int*>(sm.raw + 4 * a.page_bytes);   // this partition's pages
    int* selph = sel + a.topk;                                       // and their physical ids

    const int s = blockIdx.x, b = blockIdx.y;
    const int kvh = blockIdx.z / a.n_row_groups, rg = blockIdx.z % a.n_row_groups;
    const int row_warps = (blockDim.x >> 5) >> 1;
    const int M = a.G * a.Q;
    const AttendLane L = attend_lane(rg, a.rows_per_cta, row_warps, M, a.G);
    const int ctx = clamp_ctx(a.ctx_len[b], a.Q, a.max_pages, nullptr);
    const int n_pages = (ctx + kPage - 1) / kPage;
    const int pos0 = ctx - a.Q + L.t0, pos1 = ctx - a.Q + L.t1;

    uint32_t qa[8][4];
    if (RS) {
        load_qa_bf16<false>(qa, reinterpret_cast<const uint16_t*>(a.q), L, b, kvh, a.Q, a.Hq, a.G);
    } else {
        // e4m3 q widened to bf16 (exact)
        const uint8_t* q8 = reinterpret_cast<const uint8_t*>(a.q);
        const int mc0 = L.v0 ? L.m0 : 0, mc1 = L.v1 ? L.m1 : 0;
        const int64_t base0 = (((int64_t)b * a.Q + mc0 / a.G) * a.Hq + kvh * a.G + mc0 % a.G) * kD + 2 * L.t;
        const int64_t base1 = (((int64_t)b * a.Q + mc1 / a.G) * a.Hq + kvh * a.G + mc1 % a.G) * kD + 2 * L.t;
        uint32_t w0[16], w1[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            w0[k] = *reinterpret_cast<const uint16_t*>(q8 + base0 + 8 * k);
            w1[k] = *reinterpret_cast<const uint16_t*>(q8 + base1 + 8 * k);
        }
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            const float2 g0 = f16x2_to_f32x2(e4m3x2_to_f16x2(w0[k])), g1 = f16x2_to_f32x2(e4m3x2_to_f16x2(w1[k]));
            qa[k >> 1][(k & 1) * 2 + 0] = f32x2_to_bf16x2(g0.x, g0.y);
            qa[k >> 1][(k & 1) * 2 + 1] = f32x2_to_bf16x2(g1.x, g1.y);
        }
    }
    // this partition's entries of the row's selection, checked against the context and the pool
    const int k_eff = max(0, min(a.topk_count[b], min(a.topk, n_pages)));
    const int lo = (int)(((int64_t)s * k_eff) / a.S), hi = (int)(((int64_t)(s + 1) * k_eff) / a.S);
    for (int i = threadIdx.x; i < hi - lo; i += blockDim.x) {
        const int p = a.topk_pages[(int64_t)b * a.topk + lo + i];
        int ph = -1;
        if (p < 0 || p >= n_pages) {
            flag_status(a.status, SMX_DEV_BAD_TOPK);
        } else {
            const int64_t v = a.page_table[(int64_t)b * a.max_pages + p];
            if (v >= 0 && v < a.n_pool) ph = (int)v;
            else flag_status(a.status, SMX_DEV_BAD_PAGE_ID);
        }
        sel[i] = p;
        selph[i] = ph;
    }
    if (threadIdx.x == 0) {
        mbar_init(&mbar[0], 1);
        mbar_init(&mbar[1], 1);
        mbar_fence_init();
    }
    __syncthreads();

    float o[16][4];
#pragma unroll
    for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.0f;
    float mrow0 = -INFINITY, mrow1 = -INFINITY, l0 = 0.0f, l1 = 0.0f;
    uint32_t gp = 0;
    attend_pages<RS>(sm, sel, selph, hi - lo, a.k_pool, a.v_pool, a.Hkv, kvh, a.page_bytes, ctx, qa, L, pos0, pos1,
                     gp, o, mrow0, mrow1, l0, l1, a.status, false, a.qk_scale, a.nv != 0);
    finish_partials(sm, L, o, mrow0, mrow1, l0, l1, a.part_o, a.part_m, a.part_l, b, s, kvh, a.S, a.Q, a.Hq, a.G,
                    a.o_scale);
}

// a6: one warp per (b, t, h) row
constexpr int kMergeWarps = 4;

__global__ void __launch_bounds__(kMergeWarps * 32) attn_merge_kernel(const float* __restrict__ part_o,
                                                                      const float* __restrict__ part_m,
                                                                      const float* __restrict__ part_l,
                                                                      float* __restrict__ out, int S, int QH,
                                                                      int rows) {
    const int row = blockIdx.x * kMergeWarps + (threadIdx.x >> 5);   // b * Q * Hq + t * Hq + h
    if (row >= rows) return;
    const int b = row / QH, r = row % QH;
    merge_row<false>(part_o, part_m, part_l, (int64_t)b * S * QH + r, QH, S, out + (int64_t)row * kD);
}

// The largest S whose units of up to `rows` query rows (B x Hkv x row groups per partition) fill at
// most one wave of `sms` CTAs, lowered so every partition holds the same number of selected pages.
static int one_wave_splits(const smx_shape_t& s, int rows, int sms) {
    const int M = (s.Hq / s.Hkv) * s.Q;
    const int per_split = s.B * s.Hkv * ((M + rows - 1) / rows);
    const int s_max = max(1, sms / max(1, per_split));
    const int pages_per_split = (s.topk + s_max - 1) / s_max;
    return max(1, (s.topk + pages_per_split - 1) / pages_per_split);
}

int suggest_num_splits(const smx_shape_t& s) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    // one CTA per SM: one wave of 64-row (mma.sync) units
    const int M = (s.Hq / s.Hkv) * s.Q;
    const int rows64 = 16 * min(kAttnMaxWarps / 2, (M + 15) / 16);
    const int s_mma = one_wave_splits(s, rows64, sms);
    // MXFP4 K/V with more than 64 query rows per KV head: when that wave leaves 3 or more selected
    // pages per partition, one wave of 128-row tensor-core units (which the fused step then takes,
    // the 64-row units needing more than one wave) is faster. Measured on GB300, whole step: 4 to 8
    // pages per 64-row unit 10 to 26 % faster; at 2 pages about even, at 1 page mma.sync ahead.
    const int ppb = s.pages_per_block > 1 ? s.pages_per_block : 1;   // pages per selected block
    if (s.kv_format == SMX_KV_MXFP4 && M > 64 && (s.topk + s_mma - 1) / s_mma * ppb >= 3) return one_wave_splits(s, 128, sms);
    return s_mma;
}

cudaError_t launch_attn_split(const smx_shape_t& s, const void* q, const uint8_t* k_pool,
                              const uint8_t* v_pool, const int32_t* page_table, const int32_t* ctx_len,
                              const int32_t* topk_pages, const int32_t* topk_count, float* part_o,
                              float* part_m, float* part_l, int32_t* status, cudaStream_t st) {
    AttnArgs a = {};
    a.q = q; a.k_pool = k_pool; a.v_pool = v_pool; a.page_table = page_table; a.ctx_len = ctx_len;
    a.topk_pages = topk_pages; a.topk_count = topk_count; a.part_o = part_o; a.part_m = part_m;
    a.part_l = part_l; a.status = status;
    a.n_pool = s.n_pool_pages; a.B = s.B; a.Q = s.Q; a.Hq = s.Hq;
    a.Hkv = s.Hkv; a.G = s.Hq / s.Hkv; a.max_pages = s.max_pages_per_row; a.topk = s.topk; a.S = s.num_splits;
    const int M = a.G * a.Q;
    // warps = 2 token halves x up to 4 groups of 16 query rows
    const int row_warps = min(kAttnMaxWarps / 2, (M + 15) / 16);
    a.rows_per_cta = row_warps * 16;
    a.n_row_groups = (M + a.rows_per_cta - 1) / a.rows_per_cta;
    const bool rs = s.kv_format == SMX_KV_E4M3_ROWSCALE;
    a.page_bytes = kv_page_bytes(s);
    a.nv = s.kv_format == SMX_KV_NVFP4;
    // NVFP4: the pool's per-tensor scales, on the scores (folded into the softmax scale) and on O
    a.qk_scale = a.nv ? kLog2eOverSqrtD * s.nv_scale_k : kLog2eOverSqrtD;
    a.o_scale = a.nv ? s.nv_scale_v : 1.0f;
    const size_t smem = attend_smem_bytes(a.page_bytes) + 8 * (size_t)s.topk;
    const void* kfn = rs ? reinterpret_cast<const void*>(attn_split_kernel<true>)
                         : reinterpret_cast<const void*>(attn_split_kernel<false>);
    cudaError_t e = ensure_smem_attr(kfn, (int)smem);
    if (e != cudaSuccess) return e;
    const dim3 grid(s.num_splits, s.B, s.Hkv * a.n_row_groups), block(2 * row_warps * 32);
    if (rs) attn_split_kernel<true><<<grid, block, smem, st>>>(a);
    else attn_split_kernel<false><<<grid, block, smem, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_attn_merge(const smx_shape_t& s, const float* part_o, const float* part_m,
                              const float* part_l, float* out, cudaStream_t st) {
    const int rows = s.B * s.Q * s.Hq;
    attn_merge_kernel<<<(rows + kMergeWarps - 1) / kMergeWarps, kMergeWarps * 32, 0, st>>>(
        part_o, part_m, part_l, out, s.num_splits, s.Q * s.Hq, rows);
    return cudaGetLastError();
}

}  // namespace smx

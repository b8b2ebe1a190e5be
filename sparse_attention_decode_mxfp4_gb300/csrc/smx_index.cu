// smx_index.cu -- a3 (page scores from the MXFP4 index cache) and a4 (top-k pages per row).
//
// [ATOM-2812] "Mono decode over the MXFP4 KV and index caches", commit "--index-cache-dtype
// mxfp4": the scorer reads each index page as 16 B key loads plus a dword of E8M0 scales and
// widens the fp4 keys for a 16-bit MMA against the index query; commit "MXFP4 main KV": the
// selected blocks (one 128-token page each) fill the row's sparse table.
//
// GB300 form of the scorer: one warp scores one page. Lane (g, t) of the m16n8k16 MMA loads
// 16 B (= 32 elements of group t) of token rows g and g+8 of each 16-token tile straight into
// registers (a warp instruction covers 512 contiguous bytes), converts byte pairs with the
// hardware E2M1 -> f16x2 conversion, and multiplies group t by 2^(s_t - max_g s_g) so that
// one fp32 accumulator serves the whole row; the row's common factor 2^max_g s_g and the
// query's own power-of-two factor are applied to the fp32 result. The query is held in f16
// after a per-query power-of-two rescale that puts its largest element in [2^14, 2^15): every
// bf16 element within 2^31 of that maximum is exact in f16, so products are exact and only
// the fp32 accumulation rounds. The K permutation of the MMA is chosen so that each lane's 16
// contiguous bytes are its A fragment: k-step s takes bytes 2s and 2s+1 of every lane's group.
#include <math.h>

#include "smx_device.cuh"
#include "smx_internal.h"

namespace smx {

struct IndexArgs {
    const uint16_t* qidx;     // [B][Q][128] bf16 bits
    const uint8_t* pool;      // [n_pool][8704]
    const int32_t* page_table;
    const int32_t* ctx_len;
    float* scores;            // [B][max_pages]
    int32_t* status;
    int64_t n_pool;
    int Q, max_pages;
};

constexpr int kIdxWarps = 4;

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t h16) { return __uint_as_float(h16 << 16); }

template <int NT>
__global__ void __launch_bounds__(kIdxWarps * 32, (NT == 1 ? 4 : 3)) index_score_kernel(IndexArgs a) {
    const int b = blockIdx.y;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int p = blockIdx.x * kIdxWarps + warp;
    if (p >= a.max_pages) return;
    const int ctx = clamp_ctx(a.ctx_len[b], a.Q, a.max_pages, (p == 0 && lane == 0) ? a.status : nullptr);
    const int n_pages = (ctx + kPage - 1) / kPage;
    float* out = a.scores + (int64_t)b * a.max_pages + p;
    if (p >= n_pages) {
        if (lane == 0) *out = -INFINITY;
        return;
    }
    const int64_t phys = a.page_table[(int64_t)b * a.max_pages + p];
    if (phys < 0 || phys >= a.n_pool) {
        if (lane == 0) {
            *out = -INFINITY;
            flag_status(a.status, SMX_DEV_BAD_PAGE_ID);
        }
        return;
    }

    // ---- index query: f16 B fragments with a per-query power-of-two factor 2^sigma ----
    uint32_t qf[NT][16];
    int sig_c[NT][2];  // sigma of the two query columns this lane's accumulators hold
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int n = nt * 8 + g;
        uint32_t w[16];
        if (n < a.Q) {
            const uint4* src = reinterpret_cast<const uint4*>(a.qidx + ((int64_t)b * a.Q + n) * kD + 32 * t);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                uint4 v = src[i];
                w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
            }
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) w[i] = 0;
        }
        uint32_t mx = 0;
#pragma unroll
        for (int i = 0; i < 16; ++i) mx = max(mx, max(w[i] & 0x7FFFu, (w[i] >> 16) & 0x7FFFu));
        mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 1));
        mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 2));
        int sigma = 0;
        if (mx != 0) {
            const int e = (int)(mx >> 7);
            const int E = e ? e - 127 : -133 + (31 - __clz((int)(mx & 0x7F)));
            sigma = 14 - E;
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            float lo = scalbnf(bf16_bits_to_f32(w[i] & 0xFFFFu), sigma);
            float hi = scalbnf(bf16_bits_to_f32(w[i] >> 16), sigma);
            __half2 h = __floats2half2_rn(lo, hi);
            qf[nt][i] = *reinterpret_cast<uint32_t*>(&h);
        }
        sig_c[nt][0] = __shfl_sync(0xFFFFFFFFu, sigma, (2 * t) << 2);
        sig_c[nt][1] = __shfl_sync(0xFFFFFFFFu, sigma, (2 * t + 1) << 2);
    }

    const uint8_t* page = a.pool + phys * kMxPageBytes;
    const int lim = ctx - a.Q;  // token j counts for query n iff j <= lim + n
    float best = -INFINITY;

    // the whole page in flight at once: 16 x 16 B of nibbles and 16 scale words per lane
    uint4 c0[8], c1[8];
    uint32_t sw0[8], sw1[8];
#pragma unroll
    for (int tile = 0; tile < 8; ++tile) {
        const int r0 = tile * 16 + g, r1 = r0 + 8;
        c0[tile] = ldg_nc_v4(page + r0 * 64 + 16 * t);
        c1[tile] = ldg_nc_v4(page + r1 * 64 + 16 * t);
        sw0[tile] = __ldg(reinterpret_cast<const uint32_t*>(page + kMxScaleOff) + r0);
        sw1[tile] = __ldg(reinterpret_cast<const uint32_t*>(page + kMxScaleOff) + r1);
    }

#pragma unroll
    for (int tile = 0; tile < 8; ++tile) {
        const int r0 = tile * 16 + g, r1 = r0 + 8;
        uint32_t f0, f1;   // f16x2 of 2^(s_t - max s) per row
        int e0, e1;        // max scale byte per row (0xFF marks a NaN scale)
        {
            const uint32_t a0 = sw0[tile], a1 = sw1[tile];
            uint32_t m0 = max(max(a0 & 0xFF, (a0 >> 8) & 0xFF), max((a0 >> 16) & 0xFF, a0 >> 24));
            uint32_t m1 = max(max(a1 & 0xFF, (a1 >> 8) & 0xFF), max((a1 >> 16) & 0xFF, a1 >> 24));
            int rel0 = (int)((a0 >> (8 * t)) & 0xFF) - (int)m0;
            int rel1 = (int)((a1 >> (8 * t)) & 0xFF) - (int)m1;
            __half h0 = rel0 >= -22 ? __float2half_rn(exp2i_normal(rel0)) : __float2half_rn(0.0f);
            __half h1 = rel1 >= -22 ? __float2half_rn(exp2i_normal(rel1)) : __float2half_rn(0.0f);
            __half2 hh0 = __halves2half2(h0, h0), hh1 = __halves2half2(h1, h1);
            f0 = *reinterpret_cast<uint32_t*>(&hh0);
            f1 = *reinterpret_cast<uint32_t*>(&hh1);
            e0 = (int)m0;
            e1 = (int)m1;
        }
        float acc[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.0f;
        const uint32_t w0[4] = {c0[tile].x, c0[tile].y, c0[tile].z, c0[tile].w};
        const uint32_t w1[4] = {c1[tile].x, c1[tile].y, c1[tile].z, c1[tile].w};
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
                mma_f16_16816(acc[nt], x0, y0, x1, y1, qf[nt][2 * s0], qf[nt][2 * s0 + 1]);
                mma_f16_16816(acc[nt], x2, y2, x3, y3, qf[nt][2 * s1], qf[nt][2 * s1 + 1]);
            }
        }
        const int j0 = p * kPage + r0, j1 = p * kPage + r1;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int col = c & 1;
                const int n = nt * 8 + 2 * t + col;
                const int j = (c < 2) ? j0 : j1;
                const int e = (c < 2) ? e0 : e1;
                const bool valid = (n < a.Q) && (j <= lim + n) && (e != 0xFF);
                const float v = scalbnf(acc[nt][c], (e - 127) - sig_c[nt][col]);
                best = valid ? fmaxf(best, v) : best;
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) best = fmaxf(best, __shfl_xor_sync(0xFFFFFFFFu, best, o));
    if (lane == 0) *out = best;
}

// ---- a4: radix select of the k_eff best pages, then an id-ordered compaction --------------------
constexpr int kTopkThreads = 512;

// Block-wide exclusive scan of two counters at once; returns the block totals.
__device__ __forceinline__ void block_scan2(int a, int b, int& ea, int& eb, int& ta, int& tb, int* sm) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    int ia = a, ib = b;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int xa = __shfl_up_sync(0xFFFFFFFFu, ia, o), xb = __shfl_up_sync(0xFFFFFFFFu, ib, o);
        if (lane >= o) { ia += xa; ib += xb; }
    }
    if (lane == 31) { sm[warp] = ia; sm[32 + warp] = ib; }
    __syncthreads();
    if (warp == 0) {
        int va = lane < nw ? sm[lane] : 0, vb = lane < nw ? sm[32 + lane] : 0;
        int sa = va, sb = vb;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int xa = __shfl_up_sync(0xFFFFFFFFu, sa, o), xb = __shfl_up_sync(0xFFFFFFFFu, sb, o);
            if (lane >= o) { sa += xa; sb += xb; }
        }
        if (lane < nw) { sm[64 + lane] = sa - va; sm[96 + lane] = sb - vb; }
        if (lane == 31) { sm[128] = sa; sm[129] = sb; }
    }
    __syncthreads();
    ea = sm[64 + warp] + ia - a;
    eb = sm[96 + warp] + ib - b;
    ta = sm[128];
    tb = sm[129];
    __syncthreads();
}

__global__ void __launch_bounds__(kTopkThreads) topk_kernel(const float* __restrict__ scores,
                                                            const int32_t* __restrict__ ctx_len,
                                                            int32_t* __restrict__ topk_pages,
                                                            int32_t* __restrict__ topk_count, int max_pages,
                                                            int topk) {
    __shared__ uint32_t hist[256];
    __shared__ int sm[136];
    __shared__ uint32_t sh_digit, sh_above;
    const int b = blockIdx.x;
    const int ctx = max(0, min(ctx_len[b], max_pages * kPage));
    const int n = (ctx + kPage - 1) / kPage;
    const int k_eff = min(topk, n);
    const float* s = scores + (int64_t)b * max_pages;
    int32_t* outp = topk_pages + (int64_t)b * topk;
    const bool all = (k_eff >= n);

    uint32_t prefix = 0, mask = 0;
    int k_rem = k_eff;
    if (!all && k_eff > 0) {
#pragma unroll 1
        for (int pass = 0; pass < 4; ++pass) {
            const int shift = 24 - 8 * pass;
            for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0;
            __syncthreads();
            for (int i = threadIdx.x; i < n; i += blockDim.x) {
                const uint32_t key = score_key(s[i]);
                if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 0xFF], 1u);
            }
            __syncthreads();
            if (threadIdx.x < 32) {
                const int lane = threadIdx.x;
                // lane covers bins 255-8*lane .. 248-8*lane (descending)
                uint32_t c[8];
                uint32_t lsum = 0;
#pragma unroll
                for (int i = 0; i < 8; ++i) { c[i] = hist[255 - 8 * lane - i]; lsum += c[i]; }
                uint32_t incl = lsum;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    uint32_t x = __shfl_up_sync(0xFFFFFFFFu, incl, o);
                    if (lane >= o) incl += x;
                }
                const uint32_t excl = incl - lsum;
                const bool here = (excl < (uint32_t)k_rem) && (incl >= (uint32_t)k_rem);
                if (here) {
                    uint32_t run = excl;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        if (run + c[i] >= (uint32_t)k_rem) {
                            sh_digit = 255 - 8 * lane - i;
                            sh_above = run;
                            break;
                        }
                        run += c[i];
                    }
                }
            }
            __syncthreads();
            prefix |= sh_digit << shift;
            mask |= 0xFFu << shift;
            k_rem -= (int)sh_above;
            __syncthreads();
        }
    }
    // compaction in page-id order: every key > T, then the first k_rem pages with key == T
    const uint32_t T = prefix;
    int base_sel = 0, base_eq = 0;
    for (int start = 0; start < n; start += blockDim.x) {
        const int i = start + threadIdx.x;
        int gt = 0, eq = 0;
        if (i < n) {
            if (all) {
                gt = 1;
            } else if (k_eff > 0) {
                const uint32_t key = score_key(s[i]);
                gt = key > T;
                eq = key == T;
            }
        }
        int e_eq, t_eq, dummy_e, dummy_t;
        block_scan2(eq, 0, e_eq, dummy_e, t_eq, dummy_t, sm);
        const int sel = gt || (eq && (base_eq + e_eq) < k_rem);
        int e_sel, t_sel;
        block_scan2(sel, 0, e_sel, dummy_e, t_sel, dummy_t, sm);
        if (sel) outp[base_sel + e_sel] = i;
        base_sel += t_sel;
        base_eq += t_eq;
    }
    for (int i = k_eff + threadIdx.x; i < topk; i += blockDim.x) outp[i] = -1;
    if (threadIdx.x == 0) topk_count[b] = k_eff;
}

cudaError_t launch_index_scores(const smx_shape_t& s, const uint16_t* qidx, const uint8_t* idx_pool,
                                const int32_t* page_table, const int32_t* ctx_len, float* scores,
                                int32_t* status, cudaStream_t st) {
    IndexArgs a;
    a.qidx = qidx; a.pool = idx_pool; a.page_table = page_table; a.ctx_len = ctx_len; a.scores = scores;
    a.status = status; a.n_pool = s.n_pool_pages; a.Q = s.Q; a.max_pages = s.max_pages_per_row;
    dim3 grid((s.max_pages_per_row + kIdxWarps - 1) / kIdxWarps, s.B);
    if (s.Q <= 8) index_score_kernel<1><<<grid, kIdxWarps * 32, 0, st>>>(a);
    else index_score_kernel<2><<<grid, kIdxWarps * 32, 0, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_topk(const smx_shape_t& s, const float* scores, const int32_t* ctx_len,
                        int32_t* topk_pages, int32_t* topk_count, cudaStream_t st) {
    topk_kernel<<<s.B, kTopkThreads, 0, st>>>(scores, ctx_len, topk_pages, topk_count, s.max_pages_per_row,
                                              s.topk);
    return cudaGetLastError();
}

}  // namespace smx

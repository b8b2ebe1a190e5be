// smx_attn.cu -- a5 (split-K attention over the selected pages) and a6 (merge).
//
// [ATOM-2812] "Mono decode over the MXFP4 KV and index caches", commit "MXFP4 main KV": the
// split stage runs QK against the K page (fp4 with E8M0 group scales) and the e4m3 q, softmax
// with P in bf16 registers, PV against V widened to bf16 in on-chip memory, and writes
// (sp_o, sp_m, sp_l) per partition; the merge combines the partitions.
//
// GB300 form: one CTA per (row b, partition s, KV head, group of up to 128 query rows); rows
// are (draft token t, head of the KV group) pairs, so QK and PV are dense 16-row tiles for
// the m16n8k16 bf16 MMA. Per selected page the CTA widens K and V to bf16 in shared memory
// (E2M1 x 2^e and e4m3 codes are exact in bf16), zeroing token rows past the context so
// poisoned slots never reach an MMA, with a 16-byte XOR swizzle that keeps ldmatrix
// conflict-free. Each warp owns 16 rows and walks the page in two 64-token chunks: QK (fp32),
// mask, online softmax in the log2 domain, then the weights (times the V row scale for the
// FP8-KV format) split into a bf16 high part and a bf16 low part, both multiplied into V, so the
// weights keep ~16 significant bits (the accumulator layout of QK is the A layout of PV).
#include <math.h>

#include "smx_device.cuh"
#include "smx_internal.h"

namespace smx {

struct AttnArgs {
    const void* q;            // e4m3 bytes or bf16 bits, [B][Q][Hq][128]
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
    int B, Q, Hq, Hkv, G, max_pages, topk, S, kv_format, rows_per_cta, n_row_groups;
    // fused step: q as bf16 (packed by the scorer for MXFP4, the caller's for FP8-KV) and the
    // row's selection staged by the scorer's last CTA
    const uint16_t* qbf;      // [B][Q][Hq][128]
    const int32_t* sel_pages; // [B][topk]
    const int32_t* sel_phys;  // [B][topk]
    const int32_t* sel_count; // [B]
    int region_bytes;         // shared bytes of the K/V tiles (also holds the selection keys)
    int page_bytes;           // bytes of one K or V page (one KV head)
    int pdl;
};

constexpr int kAttnMaxWarps = 8;   // 2 token halves x 4 row groups
constexpr float kLog2eOverSqrtD = (float)(1.4426950408889634 / 11.313708498984761);

// bf16 tile [128 tokens][128 dims], 256 B rows, 16-B chunk c of row r stored at c ^ (r & 7).
__device__ __forceinline__ uint32_t swz(int row, int chunk) { return row * 256 + ((chunk ^ (row & 7)) << 4); }

// Widen one staged page (K or V of one KV head, raw bytes in shared memory) to bf16 tiles in
// shared memory (exact in both formats). For the e4m3 row-scale pages the codes are widened
// unscaled and the row scales go to rscale[]: K's scale multiplies the scores, V's multiplies
// the softmax weights. Token rows at or past valid_rows are zero.
template <bool RS>
__device__ __forceinline__ void widen_page(const uint8_t* raw, int valid_rows, uint8_t* tile, float* rscale) {
    if constexpr (RS) {
        // 128 rows x 8 chunks of 16 codes
        for (int it = threadIdx.x; it < 128 * 8; it += blockDim.x) {
            const int r = it >> 3, c = it & 7;
            uint4 o0 = make_uint4(0, 0, 0, 0), o1 = o0;
            if (r < valid_rows) {
                const uint4 w = *reinterpret_cast<const uint4*>(raw + r * 128 + c * 16);
                const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
                uint32_t ob[8];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float2 lo = f16x2_to_f32x2(e4m3x2_to_f16x2(ws[i] & 0xFFFF));
                    const float2 hi = f16x2_to_f32x2(e4m3x2_to_f16x2(ws[i] >> 16));
                    ob[2 * i] = f32x2_to_bf16x2(lo.x, lo.y);
                    ob[2 * i + 1] = f32x2_to_bf16x2(hi.x, hi.y);
                }
                o0 = make_uint4(ob[0], ob[1], ob[2], ob[3]);
                o1 = make_uint4(ob[4], ob[5], ob[6], ob[7]);
            }
            if (c == 0) rscale[r] = r < valid_rows ? reinterpret_cast<const float*>(raw + kRsScaleOff)[r] : 0.0f;
            *reinterpret_cast<uint4*>(tile + swz(r, 2 * c)) = o0;
            *reinterpret_cast<uint4*>(tile + swz(r, 2 * c + 1)) = o1;
        }
        return;
    }
    // MXFP4: 128 rows x 4 chunks of 16 nibble bytes (32 elements = one scale group)
    for (int it = threadIdx.x; it < 128 * 4; it += blockDim.x) {
        const int r = it >> 2, c = it & 3;
        uint32_t ob[16];
        if (r < valid_rows) {
            const uint4 w = *reinterpret_cast<const uint4*>(raw + r * 64 + c * 16);
            const float sc = e8m0_to_f32(raw[kMxScaleOff + r * 4 + c]);
            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                uint32_t h0, h1, h2, h3;
                e2m1x8_to_f16x2(ws[i], h0, h1, h2, h3);
                const float2 f0 = f16x2_to_f32x2(h0), f1 = f16x2_to_f32x2(h1);
                const float2 f2 = f16x2_to_f32x2(h2), f3 = f16x2_to_f32x2(h3);
                ob[4 * i + 0] = f32x2_to_bf16x2(f0.x * sc, f0.y * sc);
                ob[4 * i + 1] = f32x2_to_bf16x2(f1.x * sc, f1.y * sc);
                ob[4 * i + 2] = f32x2_to_bf16x2(f2.x * sc, f2.y * sc);
                ob[4 * i + 3] = f32x2_to_bf16x2(f3.x * sc, f3.y * sc);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) ob[i] = 0;
        }
#pragma unroll
        for (int k = 0; k < 4; ++k)
            *reinterpret_cast<uint4*>(tile + swz(r, 4 * c + k)) =
                make_uint4(ob[4 * k], ob[4 * k + 1], ob[4 * k + 2], ob[4 * k + 3]);
    }
}

template <bool RS, bool FUSED>
__global__ void __launch_bounds__(kAttnMaxWarps * 32, 1) attn_split_kernel(AttnArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t mbar[2];
    __shared__ int stage_page[2];
    uint8_t* Ks = smem;                  // 32 KB
    uint8_t* Vs = smem + 32768;          // 32 KB
    float* xch = reinterpret_cast<float*>(smem);                                 // after the pages
    float* kscale = reinterpret_cast<float*>(smem + a.region_bytes);             // 128 floats (FP8-KV K)
    float* vscale = reinterpret_cast<float*>(smem + a.region_bytes + 512);       // 128 floats (FP8-KV V)
    uint8_t* raw = smem + a.region_bytes + 1024;                                 // 2 stages x (K, V) page
    int* sel = reinterpret_cast<int*>(raw + 4 * a.page_bytes);                  // this partition's pages
    int* selph = sel + a.topk;                                                   // and their physical ids

    const int s = blockIdx.x, b = blockIdx.y;
    const int kvh = blockIdx.z / a.n_row_groups, rg = blockIdx.z % a.n_row_groups;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int row_warps = (blockDim.x >> 5) >> 1;   // warps per token half
    const int wr = warp % row_warps;                // this warp's 16-row group
    const int th = warp / row_warps;                // this warp's 64-token half of every page
    const int M = a.G * a.Q;

    // this lane's two rows
    const int m0 = rg * a.rows_per_cta + wr * 16 + g, m1 = m0 + 8;
    const bool v0 = m0 < M, v1 = m1 < M;
    const int t0 = v0 ? m0 / a.G : 0, t1 = v1 ? m1 / a.G : 0;
    const bool warp_active = rg * a.rows_per_cta + wr * 16 < M;

    const int ctx = clamp_ctx(a.ctx_len[b], a.Q, a.max_pages, nullptr);
    const int n_pages = (ctx + kPage - 1) / kPage;
    const int pos0 = ctx - a.Q + t0, pos1 = ctx - a.Q + t1;
    if (FUSED && a.pdl) pdl_wait();
    pdl_trigger();
    // q A fragments (bf16, exact) for 8 k-steps: a0/a2 row m0, a1/a3 row m1; lane (g, t) holds
    // dims 16 ks + 8 h + 2t, +1. All loads in flight together.
    uint32_t qa[8][4];
    {
        // padding rows (past the KV group's rows) read row 0: their scores are masked and their
        // outputs never written
        const int mc0 = v0 ? m0 : 0, mc1 = v1 ? m1 : 0;
        const int64_t base0 = (((int64_t)b * a.Q + mc0 / a.G) * a.Hq + kvh * a.G + mc0 % a.G) * kD + 2 * t;
        const int64_t base1 = (((int64_t)b * a.Q + mc1 / a.G) * a.Hq + kvh * a.G + mc1 % a.G) * kD + 2 * t;
        if (RS || FUSED) {
            const uint16_t* qb = FUSED && !RS ? a.qbf : reinterpret_cast<const uint16_t*>(a.q);
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                qa[k >> 1][(k & 1) * 2 + 0] = *reinterpret_cast<const uint32_t*>(qb + base0 + 8 * k);
                qa[k >> 1][(k & 1) * 2 + 1] = *reinterpret_cast<const uint32_t*>(qb + base1 + 8 * k);
            }
        } else {
            const uint8_t* q8 = reinterpret_cast<const uint8_t*>(a.q);
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
    }
    // this partition's pages; the first two page copies go out before anything else
    const int k_eff = FUSED ? max(0, min(a.sel_count[b], min(a.topk, n_pages)))
                            : max(0, min(a.topk_count[b], min(a.topk, n_pages)));
    const int lo = (int)(((int64_t)s * k_eff) / a.S), hi = (int)(((int64_t)(s + 1) * k_eff) / a.S);
    const int page_bytes = a.page_bytes;
    auto resolve = [&](int i, int& p, int& ph) {   // entry i of the row's selection
        const int64_t at = (int64_t)b * a.topk + i;
        p = FUSED ? a.sel_pages[at] : a.topk_pages[at];
        ph = -1;
        if (p < 0 || p >= n_pages) {
            flag_status(a.status, SMX_DEV_BAD_TOPK);
        } else if (FUSED) {
            ph = a.sel_phys[at];
        } else {
            const int64_t v = a.page_table[(int64_t)b * a.max_pages + p];
            if (v >= 0 && v < a.n_pool) ph = (int)v;
            else flag_status(a.status, SMX_DEV_BAD_PAGE_ID);
        }
    };
    auto issue = [&](int st, int p, int64_t phys) {  // thread 0 only
        if (phys < 0) {
            stage_page[st] = -1;
            mbar_arrive(&mbar[st]);
            return;
        }
        stage_page[st] = p;
        const int64_t off = (phys * a.Hkv + kvh) * (int64_t)page_bytes;
        mbar_arrive_expect_tx(&mbar[st], 2u * page_bytes);
        bulk_g2s(raw + st * 2 * page_bytes, a.k_pool + off, page_bytes, &mbar[st]);
        bulk_g2s(raw + st * 2 * page_bytes + page_bytes, a.v_pool + off, page_bytes, &mbar[st]);
    };
    if (threadIdx.x == 0) {
        mbar_init(&mbar[0], 1);
        mbar_init(&mbar[1], 1);
        mbar_fence_init();
        for (int st = 0; st < 2 && lo + st < hi; ++st) {
            int p, ph;
            resolve(lo + st, p, ph);
            issue(st, p, ph);
        }
    }
    // entries of the later pages, for their copies
    for (int i = threadIdx.x + 2; i < hi - lo; i += blockDim.x) resolve(lo + i, sel[i], selph[i]);

    __syncthreads();

    float o[16][4];
#pragma unroll
    for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.0f;
    float mrow0 = -INFINITY, mrow1 = -INFINITY, l0 = 0.0f, l1 = 0.0f;

    bool timed_out = false;
    int to_stage = 0;
    uint32_t to_parity = 0;
#pragma unroll 1
    for (int i = lo; i < hi; ++i) {
        const int st = (i - lo) & 1;
        const uint32_t parity = ((i - lo) >> 1) & 1;
        const bool ok = mbar_wait_bounded(&mbar[st], parity);
        if (__syncthreads_or(!ok)) {
            timed_out = true;
            to_stage = st;
            to_parity = parity;
            break;
        }
        const int p = stage_page[st];
        const int valid_rows = p >= 0 ? min(kPage, ctx - p * kPage) : 0;
        if (p >= 0) {
            const uint8_t* rk = raw + st * 2 * page_bytes;
            widen_page<RS>(rk, valid_rows, Ks, kscale);
            widen_page<RS>(rk + page_bytes, valid_rows, Vs, vscale);
        }
        __syncthreads();   // tiles ready; this stage's raw bytes are consumed
        if (threadIdx.x == 0 && i + 2 < hi) {
            fence_proxy_async_smem();
            issue(st, sel[i + 2 - lo], selph[i + 2 - lo]);
        }
        // this warp's half of the page in 16-token units: QK, online softmax, one PV k-step
        const int units = (p >= 0 && warp_active) ? max(0, min(4, (valid_rows - th * 64 + 15) / 16)) : 0;
        const int jpage = p * kPage;
#pragma unroll 1
        for (int u = 0; u < units; ++u) {
            const int tok0 = th * 64 + u * 16;
            float sc[2][4];
#pragma unroll
            for (int nb = 0; nb < 2; ++nb) sc[nb][0] = sc[nb][1] = sc[nb][2] = sc[nb][3] = 0.0f;
#pragma unroll
            for (int ks = 0; ks < 8; ks += 2) {
                uint32_t b0, b1, b2, b3, c0, c1, c2, c3;
                ldmatrix_x4(b0, b1, b2, b3, Ks + swz(tok0 + (lane & 7), 2 * ks + (lane >> 3)));
                ldmatrix_x4(c0, c1, c2, c3, Ks + swz(tok0 + 8 + (lane & 7), 2 * ks + (lane >> 3)));
                mma_bf16_16816(sc[0], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b0, b1);
                mma_bf16_16816(sc[1], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], c0, c1);
                mma_bf16_16816(sc[0], qa[ks + 1][0], qa[ks + 1][1], qa[ks + 1][2], qa[ks + 1][3], b2, b3);
                mma_bf16_16816(sc[1], qa[ks + 1][0], qa[ks + 1][1], qa[ks + 1][2], qa[ks + 1][3], c2, c3);
            }
            // scale, mask, row max (a query token sees tokens j <= pos_t)
            float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
            for (int nb = 0; nb < 2; ++nb) {
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int tok = tok0 + nb * 8 + 2 * t + (c & 1);
                    const int j = jpage + tok;
                    float z = sc[nb][c] * kLog2eOverSqrtD;
                    if (RS) z *= kscale[tok];
                    const bool ok2 = (c < 2) ? (v0 && j <= pos0) : (v1 && j <= pos1);
                    z = ok2 ? z : -INFINITY;
                    sc[nb][c] = z;
                    if (c < 2) mx0 = fmaxf(mx0, z);
                    else mx1 = fmaxf(mx1, z);
                }
            }
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xFFFFFFFFu, mx0, 1));
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xFFFFFFFFu, mx0, 2));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xFFFFFFFFu, mx1, 1));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xFFFFFFFFu, mx1, 2));
            const float mn0 = fmaxf(mrow0, mx0), mn1 = fmaxf(mrow1, mx1);
            if (__any_sync(0xFFFFFFFFu, mn0 > mrow0 || mn1 > mrow1)) {   // a row's maximum grew
                const float al0 = (mn0 == -INFINITY) ? 1.0f : exp2f(mrow0 - mn0);
                const float al1 = (mn1 == -INFINITY) ? 1.0f : exp2f(mrow1 - mn1);
                l0 *= al0;
                l1 *= al1;
#pragma unroll
                for (int db = 0; db < 16; ++db) {
                    o[db][0] *= al0; o[db][1] *= al0;
                    o[db][2] *= al1; o[db][3] *= al1;
                }
                mrow0 = mn0;
                mrow1 = mn1;
            }
            // weights. MXFP4: P in bf16 (as the pages do). FP8-KV: P' = p x V row scale as a bf16
            // high part plus a bf16 low part (its x50 rows need ~16 bits). l (per lane, reduced at
            // the end) sums the weights the PV product uses.
            uint32_t ph[2][2], pl[2][2];
#pragma unroll
            for (int nb = 0; nb < 2; ++nb) {
                float e[4];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const float mn = (c < 2) ? mrow0 : mrow1;
                    e[c] = (mn == -INFINITY) ? 0.0f : exp2f(sc[nb][c] - mn);
                }
                if (RS) {
                    l0 += e[0] + e[1];
                    l1 += e[2] + e[3];
                    const int tok = tok0 + nb * 8 + 2 * t;
                    const float s0 = vscale[tok], s1 = vscale[tok + 1];
                    e[0] *= s0; e[1] *= s1; e[2] *= s0; e[3] *= s1;
                }
                const __nv_bfloat162 h01 = __floats2bfloat162_rn(e[0], e[1]), h23 = __floats2bfloat162_rn(e[2], e[3]);
                const float2 r01 = __bfloat1622float2(h01), r23 = __bfloat1622float2(h23);
                if (!RS) {
                    l0 += r01.x + r01.y;
                    l1 += r23.x + r23.y;
                }
                ph[nb][0] = *reinterpret_cast<const uint32_t*>(&h01);
                ph[nb][1] = *reinterpret_cast<const uint32_t*>(&h23);
                if (RS) {
                    const __nv_bfloat162 l01 = __floats2bfloat162_rn(e[0] - r01.x, e[1] - r01.y);
                    const __nv_bfloat162 l23 = __floats2bfloat162_rn(e[2] - r23.x, e[3] - r23.y);
                    pl[nb][0] = *reinterpret_cast<const uint32_t*>(&l01);
                    pl[nb][1] = *reinterpret_cast<const uint32_t*>(&l23);
                }
            }
            // O += P V for these 16 tokens (the QK accumulator layout is PV's A layout)
#pragma unroll
            for (int db = 0; db < 16; db += 2) {
                uint32_t b0, b1, b2, b3;
                ldmatrix_x4_trans(b0, b1, b2, b3, Vs + swz(tok0 + ((lane >> 3) & 1) * 8 + (lane & 7), db + (lane >> 4)));
                mma_bf16_16816(o[db], ph[0][0], ph[0][1], ph[1][0], ph[1][1], b0, b1);
                mma_bf16_16816(o[db + 1], ph[0][0], ph[0][1], ph[1][0], ph[1][1], b2, b3);
                if (RS) {
                    mma_bf16_16816(o[db], pl[0][0], pl[0][1], pl[1][0], pl[1][1], b0, b1);
                    mma_bf16_16816(o[db + 1], pl[0][0], pl[0][1], pl[1][0], pl[1][1], b2, b3);
                }
            }
        }
        __syncthreads();   // before the next page overwrites the tiles
    }
    if (timed_out) {
        // give the copies still in flight a bounded chance to land before the CTA exits
        if (threadIdx.x == 0) {
            flag_status(a.status, SMX_DEV_TIMEOUT);
            mbar_wait_bounded(&mbar[to_stage], to_parity);
        }
        __syncthreads();
    }
    l0 += __shfl_xor_sync(0xFFFFFFFFu, l0, 1);
    l0 += __shfl_xor_sync(0xFFFFFFFFu, l0, 2);
    l1 += __shfl_xor_sync(0xFFFFFFFFu, l1, 1);
    l1 += __shfl_xor_sync(0xFFFFFFFFu, l1, 2);

    // ---- combine the two token halves: warps of half 1 hand (m, l, O) to half 0 ----
    __syncthreads();
    {
        float* slot = xch + wr * (32 * 68);     // per row group: 32 lanes x (64 O + m0, m1, l0, l1)
        if (th == 1) {
            float* me = slot + lane * 68;
#pragma unroll
            for (int db = 0; db < 16; ++db) {
                me[4 * db + 0] = o[db][0]; me[4 * db + 1] = o[db][1];
                me[4 * db + 2] = o[db][2]; me[4 * db + 3] = o[db][3];
            }
            me[64] = mrow0; me[65] = mrow1; me[66] = l0; me[67] = l1;
        }
        __syncthreads();
        if (th == 0) {
            const float* ot = slot + lane * 68;
            const float mo0 = ot[64], mo1 = ot[65], lo0 = ot[66], lo1 = ot[67];
            const float n0 = fmaxf(mrow0, mo0), n1 = fmaxf(mrow1, mo1);
            const float wa0 = n0 == -INFINITY ? 0.0f : exp2f(mrow0 - n0), wb0 = n0 == -INFINITY ? 0.0f : exp2f(mo0 - n0);
            const float wa1 = n1 == -INFINITY ? 0.0f : exp2f(mrow1 - n1), wb1 = n1 == -INFINITY ? 0.0f : exp2f(mo1 - n1);
#pragma unroll
            for (int db = 0; db < 16; ++db) {
                o[db][0] = o[db][0] * wa0 + ot[4 * db + 0] * wb0;
                o[db][1] = o[db][1] * wa0 + ot[4 * db + 1] * wb0;
                o[db][2] = o[db][2] * wa1 + ot[4 * db + 2] * wb1;
                o[db][3] = o[db][3] * wa1 + ot[4 * db + 3] * wb1;
            }
            l0 = l0 * wa0 + lo0 * wb0;
            l1 = l1 * wa1 + lo1 * wb1;
            mrow0 = n0;
            mrow1 = n1;
        }
    }

    // ---- write the partials of real rows ----
    if (th == 0 && (v0 || v1)) {
        const int h0 = kvh * a.G + m0 % a.G, h1 = kvh * a.G + m1 % a.G;
        const int64_t r0 = (((int64_t)b * a.S + s) * a.Q + t0) * a.Hq + h0;
        const int64_t r1 = (((int64_t)b * a.S + s) * a.Q + t1) * a.Hq + h1;
#pragma unroll
        for (int db = 0; db < 16; ++db) {
            const int d = db * 8 + 2 * t;
            if (v0) *reinterpret_cast<float2*>(a.part_o + r0 * kD + d) = make_float2(o[db][0], o[db][1]);
            if (v1) *reinterpret_cast<float2*>(a.part_o + r1 * kD + d) = make_float2(o[db][2], o[db][3]);
        }
        if (t == 0) {
            if (v0) { a.part_m[r0] = mrow0; a.part_l[r0] = l0; }
            if (v1) { a.part_m[r1] = mrow1; a.part_l[r1] = l1; }
        }
    }
}

// ---- a6 merge: one warp per (b, t, h) row; lane l owns dims 4l..4l+3 and partitions l, l+32, ...
constexpr int kMergeWarps = 4;

__global__ void __launch_bounds__(kMergeWarps * 32) attn_merge_kernel(const float* __restrict__ part_o,
                                                                      const float* __restrict__ part_m,
                                                                      const float* __restrict__ part_l,
                                                                      float* __restrict__ out, int S, int QH,
                                                                      int rows, int pdl) {
    if (pdl) pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * kMergeWarps + (threadIdx.x >> 5);   // b * Q * Hq + t * Hq + h
    if (row >= rows) return;
    const int b = row / QH, r = row % QH;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float M = -INFINITY, L = 0.0f;
    // 16 partitions per pass: lane l reads m, l of partition s0 + (l & 15) and dims 4l..4l+3 of all
    // 16 partial outputs, every load of the pass in flight together
    for (int s0 = 0; s0 < S; s0 += 16) {
        const int n = min(16, S - s0);
        const int sl = s0 + (lane & 15);
        float m = -INFINITY, lv = 0.0f;
        if ((lane & 15) < n) {
            const int64_t pi = ((int64_t)b * S + sl) * QH + r;
            m = part_m[pi];
            lv = part_l[pi];
        }
        float4 v[16];
#pragma unroll
        for (int k = 0; k < 16; ++k)
            v[k] = k < n ? reinterpret_cast<const float4*>(part_o + (((int64_t)b * S + s0 + k) * QH + r) * kD)[lane]
                         : make_float4(0.f, 0.f, 0.f, 0.f);
        float mp = m;
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) mp = fmaxf(mp, __shfl_xor_sync(0xFFFFFFFFu, mp, o));
        const float Mn = fmaxf(M, mp);
        if (Mn != -INFINITY) {
            const float al = (M == -INFINITY) ? 0.0f : exp2f(M - Mn);
            acc.x *= al; acc.y *= al; acc.z *= al; acc.w *= al;
            L *= al;
            const float w = (m == -INFINITY) ? 0.0f : exp2f(m - Mn);
            // both 16-lane halves hold the same partitions: each half sums its own copy
            float lw = w * lv;
#pragma unroll
            for (int o = 8; o > 0; o >>= 1) lw += __shfl_xor_sync(0xFFFFFFFFu, lw, o);
            L += lw;
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                const float wk = __shfl_sync(0xFFFFFFFFu, w, k);
                acc.x += wk * v[k].x; acc.y += wk * v[k].y; acc.z += wk * v[k].z; acc.w += wk * v[k].w;
            }
            M = Mn;
        }
    }
    if (M != -INFINITY) {
        acc.x /= L; acc.y /= L; acc.z /= L; acc.w /= L;
    }
    reinterpret_cast<float4*>(out + (int64_t)row * kD)[lane] = acc;
}

int suggest_num_splits(const smx_shape_t& s) {
    const int M = (s.Hq / s.Hkv) * s.Q;
    const int row_warps = min(kAttnMaxWarps / 2, (M + 15) / 16);
    const int rows_per_cta = row_warps * 16;
    const int ctas_per_split = s.B * s.Hkv * ((M + rows_per_cta - 1) / rows_per_cta);
    const int page_bytes = s.kv_format == SMX_KV_E4M3_ROWSCALE ? kRsPageBytes : kMxPageBytes;
    const size_t smem = (size_t)65536 + 1024 + 4 * (size_t)page_bytes + 8 * (size_t)s.topk;
    const void* kfn = s.kv_format == SMX_KV_E4M3_ROWSCALE ? reinterpret_cast<const void*>(attn_split_kernel<true, true>)
                                                          : reinterpret_cast<const void*>(attn_split_kernel<false, true>);
    int dev = 0, sms = 0, per_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        ensure_smem_attr(kfn, (int)smem) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kfn, 2 * row_warps * 32, smem) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    // one wave of split CTAs, then equal page counts per partition
    const int s_max = max(1, (sms * max(1, per_sm)) / max(1, ctas_per_split));
    const int pages_per_split = (s.topk + s_max - 1) / s_max;
    return max(1, (s.topk + pages_per_split - 1) / pages_per_split);
}

static cudaError_t launch_split_impl(const smx_shape_t& s, AttnArgs& a, bool fused, cudaStream_t st) {
    a.n_pool = s.n_pool_pages; a.B = s.B; a.Q = s.Q; a.Hq = s.Hq;
    a.Hkv = s.Hkv; a.G = s.Hq / s.Hkv; a.max_pages = s.max_pages_per_row; a.topk = s.topk; a.S = s.num_splits;
    a.kv_format = s.kv_format; a.pdl = fused ? 1 : 0;
    const int M = a.G * a.Q;
    // warps = 2 token halves x up to 4 groups of 16 query rows
    const int row_warps = min(kAttnMaxWarps / 2, (M + 15) / 16);
    const int warps = 2 * row_warps;
    a.rows_per_cta = row_warps * 16;
    a.n_row_groups = (M + a.rows_per_cta - 1) / a.rows_per_cta;
    a.region_bytes = 65536;
    a.page_bytes = s.kv_format == SMX_KV_E4M3_ROWSCALE ? kRsPageBytes : kMxPageBytes;
    const size_t smem = (size_t)a.region_bytes + 1024 + 4 * (size_t)a.page_bytes + 8 * (size_t)s.topk;
    const bool rs = s.kv_format == SMX_KV_E4M3_ROWSCALE;
    const void* kfn = rs ? (fused ? reinterpret_cast<const void*>(attn_split_kernel<true, true>)
                                  : reinterpret_cast<const void*>(attn_split_kernel<true, false>))
                         : (fused ? reinterpret_cast<const void*>(attn_split_kernel<false, true>)
                                  : reinterpret_cast<const void*>(attn_split_kernel<false, false>));
    cudaError_t e = ensure_smem_attr(kfn, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(s.num_splits, s.B, s.Hkv * a.n_row_groups);
    cfg.blockDim = dim3(warps * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = fused ? 1 : 0;
    if (rs) return fused ? cudaLaunchKernelEx(&cfg, attn_split_kernel<true, true>, a)
                         : cudaLaunchKernelEx(&cfg, attn_split_kernel<true, false>, a);
    return fused ? cudaLaunchKernelEx(&cfg, attn_split_kernel<false, true>, a)
                 : cudaLaunchKernelEx(&cfg, attn_split_kernel<false, false>, a);
}

cudaError_t launch_attn_split(const smx_shape_t& s, const void* q, const uint8_t* k_pool,
                              const uint8_t* v_pool, const int32_t* page_table, const int32_t* ctx_len,
                              const int32_t* topk_pages, const int32_t* topk_count, float* part_o,
                              float* part_m, float* part_l, int32_t* status, cudaStream_t st) {
    AttnArgs a = {};
    a.q = q; a.k_pool = k_pool; a.v_pool = v_pool; a.page_table = page_table; a.ctx_len = ctx_len;
    a.topk_pages = topk_pages; a.topk_count = topk_count; a.part_o = part_o; a.part_m = part_m;
    a.part_l = part_l; a.status = status;
    return launch_split_impl(s, a, false, st);
}

cudaError_t launch_attn_fused_split(const smx_shape_t& s, const uint16_t* qbf, const uint8_t* k_pool,
                                    const uint8_t* v_pool, const int32_t* ctx_len, const int32_t* sel_pages,
                                    const int32_t* sel_phys, const int32_t* sel_count, float* part_o,
                                    float* part_m, float* part_l, int32_t* status, cudaStream_t st) {
    AttnArgs a = {};
    a.q = qbf; a.qbf = qbf; a.k_pool = k_pool; a.v_pool = v_pool; a.ctx_len = ctx_len;
    a.sel_pages = sel_pages; a.sel_phys = sel_phys; a.sel_count = sel_count;
    a.part_o = part_o; a.part_m = part_m; a.part_l = part_l; a.status = status;
    return launch_split_impl(s, a, true, st);
}

cudaError_t launch_attn_merge(const smx_shape_t& s, const float* part_o, const float* part_m,
                              const float* part_l, float* out, bool pdl, cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    const int rows = s.B * s.Q * s.Hq;
    cfg.gridDim = dim3((rows + kMergeWarps - 1) / kMergeWarps);
    cfg.blockDim = dim3(kMergeWarps * 32);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, attn_merge_kernel, part_o, part_m, part_l, out, s.num_splits, s.Q * s.Hq, rows,
                              pdl ? 1 : 0);
}

}  // namespace smx

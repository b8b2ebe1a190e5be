// smx_attend_tc.cuh -- the split stage (a5) of one partition on the fifth-generation tensor cores:
// QK and PV as 128 x 128 x 128 bf16 tcgen05 MMAs with fp32 accumulators in tensor memory.
//
// [ATOM-2812] "Mono decode over the MXFP4 KV and index caches", commit "MXFP4 main KV": QK against
// the K page (fp4 with E8M0 group scales) and the e4m3 q, softmax with P in bf16, PV against V
// widened to bf16 on chip, (sp_o, sp_m, sp_l) per partition.
//
// One CTA (8 warps) serves up to 128 query rows of one KV head; rows are (draft token, head)
// pairs. Per selected page, staged by bulk copies (two pages in flight):
//  1. K is widened to bf16 as a [128 tokens][128 dims] tile and V transposed into a
//     [128 dims][128 tokens] tile (E2M1 x 2^e and e4m3 are exact in bf16; token rows past the
//     context are zero, so poisoned slots never reach an MMA); both are K-major, 128-byte swizzle.
//  2. One thread issues S = q K^T (8 MMA steps of K = 16) into tensor-memory columns 0..127.
//  3. Thread (warp w, lane l) owns query row 32 (w % 4) + l and token / dim half w / 4: it reads
//     its 64 scores (tcgen05.ld), scales, masks, takes the online softmax in the log2 domain (the
//     row maximum is exchanged with its partner thread through shared memory) and writes its
//     half of P as bf16 (FP8-KV: p times the V row scale as a bf16 high part and low part, the low
//     part in the K tile, which S no longer needs).
//  4. One thread issues O_page = P V^T (and P_lo V^T) into columns 128..255; every thread reads
//     its 64 output columns and adds them to its running O after the softmax rescale.
#pragma once

#include <math.h>

#include "smx_attend.cuh"
#include "smx_device.cuh"
#include "smx_tc.cuh"

namespace smx {

// Dynamic shared memory of the tensor-core attention (base 1024-byte aligned).
constexpr int kTcQ = 0;             // q tile, bf16 [128 rows][128 dims]
constexpr int kTcK = 32768;         // K tile [128 tokens][128 dims]; P low part (FP8-KV) after QK
constexpr int kTcV = 65536;         // V^T tile [128 dims][128 tokens]
constexpr int kTcP = 98304;         // P tile [128 rows][128 tokens]
constexpr int kTcScale = 131072;    // 128 K row scales, 128 V row scales (FP8-KV)
constexpr int kTcRaw = 132096;      // two stages of (K page, V page)
constexpr uint32_t kTcCols = 256;   // tensor-memory columns: S at 0, O at 128
constexpr int kTcRows = 128;        // query rows per CTA

__host__ __device__ constexpr size_t attend_tc_smem_bytes(int page_bytes) {
    return (size_t)kTcRaw + 4 * (size_t)page_bytes;
}

// The q tile from `rows` query rows (rows past them are zero). Staged rows at src (shared memory,
// 512-byte f32 rows for MXFP4 K/V, packed here to e4m3 by the q packing rule and widened to bf16;
// 256-byte bf16 rows for FP8-KV). One (row, half) piece per thread of the 256-thread block.
template <bool RS>
__device__ __forceinline__ void pack_q_tile_tc(const uint8_t* src, int rows, uint8_t* tile) {
    const int r = threadIdx.x >> 1, h = threadIdx.x & 1;
#pragma unroll 1
    for (int c = 0; c < 8; ++c) {   // chunk c of the half: dims 64 h + 8 c .. + 7
        uint4 v = make_uint4(0, 0, 0, 0);
        if (r < rows) {
            if (RS) {
                v = *reinterpret_cast<const uint4*>(src + r * 256 + (8 * h + c) * 16);
            } else {
                const float4* f = reinterpret_cast<const float4*>(src + r * 512 + (8 * h + c) * 32);
                const float4 f0 = f[0], f1 = f[1];
                const float2 g0 = f16x2_to_f32x2(e4m3x2_to_f16x2(pack_q2(f0.x, f0.y)));
                const float2 g1 = f16x2_to_f32x2(e4m3x2_to_f16x2(pack_q2(f0.z, f0.w)));
                const float2 g2 = f16x2_to_f32x2(e4m3x2_to_f16x2(pack_q2(f1.x, f1.y)));
                const float2 g3 = f16x2_to_f32x2(e4m3x2_to_f16x2(pack_q2(f1.z, f1.w)));
                v = make_uint4(f32x2_to_bf16x2(g0.x, g0.y), f32x2_to_bf16x2(g1.x, g1.y), f32x2_to_bf16x2(g2.x, g2.y),
                               f32x2_to_bf16x2(g3.x, g3.y));
            }
        }
        *reinterpret_cast<uint4*>(tile + sw128_chunk(r, 8 * h + c, kTcRows)) = v;
    }
}

// The same from global q rows: row i of the unit is q row (b, i / G ... ) given by qrow(i).
template <bool RS>
__device__ __forceinline__ void pack_q_tile_tc_global(const void* q, int b, int kvh, int m_lo, int rows, int Q, int Hq,
                                                      int G, uint8_t* tile) {
    const int r = threadIdx.x >> 1, h = threadIdx.x & 1;
    const int m = m_lo + r;
    const int64_t row = ((int64_t)b * Q + (r < rows ? m / G : 0)) * Hq + kvh * G + (r < rows ? m % G : 0);
#pragma unroll 1
    for (int c = 0; c < 8; ++c) {
        uint4 v = make_uint4(0, 0, 0, 0);
        if (r < rows) {
            if (RS) {
                v = *reinterpret_cast<const uint4*>(reinterpret_cast<const uint8_t*>(q) + row * 256 + (8 * h + c) * 16);
            } else {
                const float4* f = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(q) + row * kD + (8 * h + c) * 8);
                const float4 f0 = f[0], f1 = f[1];
                const float2 g0 = f16x2_to_f32x2(e4m3x2_to_f16x2(pack_q2(f0.x, f0.y)));
                const float2 g1 = f16x2_to_f32x2(e4m3x2_to_f16x2(pack_q2(f0.z, f0.w)));
                const float2 g2 = f16x2_to_f32x2(e4m3x2_to_f16x2(pack_q2(f1.x, f1.y)));
                const float2 g3 = f16x2_to_f32x2(e4m3x2_to_f16x2(pack_q2(f1.z, f1.w)));
                v = make_uint4(f32x2_to_bf16x2(g0.x, g0.y), f32x2_to_bf16x2(g1.x, g1.y), f32x2_to_bf16x2(g2.x, g2.y),
                               f32x2_to_bf16x2(g3.x, g3.y));
            }
        }
        *reinterpret_cast<uint4*>(tile + sw128_chunk(r, 8 * h + c, kTcRows)) = v;
    }
}

// K page (raw, shared memory) -> K tile [token][dim]; FP8-KV row scales -> rscale.
template <bool RS>
__device__ __forceinline__ void widen_k_tc(const uint8_t* raw, int valid_rows, uint8_t* tile, float* rscale) {
    if constexpr (RS) {
        // 128 tokens x 8 chunks of 16 codes (two output chunks each)
#pragma unroll 1
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
            *reinterpret_cast<uint4*>(tile + sw128_chunk(r, 2 * c, kTcRows)) = o0;
            *reinterpret_cast<uint4*>(tile + sw128_chunk(r, 2 * c + 1, kTcRows)) = o1;
        }
    } else {
        // 128 tokens x 4 scale groups of 16 nibble bytes (four output chunks each)
#pragma unroll 1
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
                *reinterpret_cast<uint4*>(tile + sw128_chunk(r, 4 * c + k, kTcRows)) =
                    make_uint4(ob[4 * k], ob[4 * k + 1], ob[4 * k + 2], ob[4 * k + 3]);
        }
    }
}

// V page (raw, shared memory) -> V^T tile [dim][token]; FP8-KV row scales -> rscale. Thread t
// widens the 8 x 8 block of dims 8 (t % 16) .. + 7 and tokens 8 (t / 16) .. + 7 (256 threads):
// the 16 threads of a half-warp read consecutive words of the same token rows.
template <bool RS>
__device__ __forceinline__ void widen_vt_tc(const uint8_t* raw, int valid_rows, uint8_t* tile, float* rscale) {
    const int d0 = 8 * (threadIdx.x & 15), t0 = 8 * (threadIdx.x >> 4);
    float v[8][8];   // [token][dim]
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int r = t0 + i;
        if (r < valid_rows) {
            if (RS) {
                const uint2 w = *reinterpret_cast<const uint2*>(raw + r * 128 + d0);
                const float2 a = f16x2_to_f32x2(e4m3x2_to_f16x2(w.x & 0xFFFF)), b = f16x2_to_f32x2(e4m3x2_to_f16x2(w.x >> 16));
                const float2 c = f16x2_to_f32x2(e4m3x2_to_f16x2(w.y & 0xFFFF)), d = f16x2_to_f32x2(e4m3x2_to_f16x2(w.y >> 16));
                v[i][0] = a.x; v[i][1] = a.y; v[i][2] = b.x; v[i][3] = b.y;
                v[i][4] = c.x; v[i][5] = c.y; v[i][6] = d.x; v[i][7] = d.y;
            } else {
                const uint32_t w = *reinterpret_cast<const uint32_t*>(raw + r * 64 + d0 / 2);
                const float sc = e8m0_to_f32(raw[kMxScaleOff + r * 4 + d0 / 32]);
                uint32_t h0, h1, h2, h3;
                e2m1x8_to_f16x2(w, h0, h1, h2, h3);
                const float2 f0 = f16x2_to_f32x2(h0), f1 = f16x2_to_f32x2(h1);
                const float2 f2 = f16x2_to_f32x2(h2), f3 = f16x2_to_f32x2(h3);
                v[i][0] = f0.x * sc; v[i][1] = f0.y * sc; v[i][2] = f1.x * sc; v[i][3] = f1.y * sc;
                v[i][4] = f2.x * sc; v[i][5] = f2.y * sc; v[i][6] = f3.x * sc; v[i][7] = f3.y * sc;
            }
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) v[i][j] = 0.0f;
        }
    }
    if (RS && threadIdx.x < 128)
        rscale[threadIdx.x] = (int)threadIdx.x < valid_rows ? reinterpret_cast<const float*>(raw + kRsScaleOff)[threadIdx.x] : 0.0f;
#pragma unroll
    for (int j = 0; j < 8; ++j)
        *reinterpret_cast<uint4*>(tile + sw128_chunk(d0 + j, t0 >> 3, kTcRows)) =
            make_uint4(f32x2_to_bf16x2(v[0][j], v[1][j]), f32x2_to_bf16x2(v[2][j], v[3][j]),
                       f32x2_to_bf16x2(v[4][j], v[5][j]), f32x2_to_bf16x2(v[6][j], v[7][j]));
}

// Per-thread state of the tensor-core attention: query row r (TMEM lane) and half h.
struct TcLane {
    int r, h;
    bool valid;   // the row is a real query row
    int pos;      // the last token position the row may see
};

// After a copy that did not land: flag the timeout and give the copies still in flight (stage st,
// and the other stage if `other`) a bounded chance to land before the CTA goes on. One thread.
__device__ __noinline__ void attend_drain(const AttendSmem& sm, int st, uint32_t parity, bool other,
                                         uint32_t other_parity, int32_t* status) {
    flag_status(status, SMX_DEV_TIMEOUT);
    mbar_wait_bounded(&sm.mbar[st], parity);
    if (other) mbar_wait_bounded(&sm.mbar[st ^ 1], other_parity);
}

// Bounded wait on an mbarrier phase by every thread; false if it gave up.
__device__ __forceinline__ bool tc_wait(uint64_t* bar, uint32_t parity) { return mbar_wait_bounded(bar, parity); }

// Scaled, masked log2-domain scores of 16 columns of this thread's row (from S in tensor memory).
template <bool RS>
__device__ __forceinline__ void tc_scores16(uint32_t taddr, int col0, int jpage, int valid_rows, const TcLane& L,
                                           const float* kscale, float (&z)[16]) {
    tmem_ld16(taddr, z);
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const int tok = col0 + j;
        float s = z[j] * kLog2eOverSqrtD;
        if (RS) s *= kscale[tok];
        z[j] = (L.valid && tok < valid_rows && jpage + tok <= L.pos) ? s : -INFINITY;
    }
}

// The pages sel[0..np) / selph[0..np) of this CTA's partition (shared memory); pages 0 and 1 were
// issued by the caller's thread 0 (attend_issue, stage area sm.raw). tmem: the CTA's kTcCols
// columns; the output O of this CTA's rows accumulates in columns 128..255 across the pages
// (rescaled in place when a row's maximum grows). mma_bar counts MMA completions (mma_ph = phases
// seen). m: the row's running maximum (log2 domain); l: this half's share of the row's weight
// sum. Returns false if a copy or an MMA did not finish within the bounded wait (status gets
// SMX_DEV_TIMEOUT); O is then incomplete.
template <bool RS>
__device__ __forceinline__ bool attend_pages_tc(uint8_t* smem, const AttendSmem& sm, const int* sel, const int* selph,
                                                int np, const uint8_t* k_pool, const uint8_t* v_pool, int Hkv, int kvh,
                                                int page_bytes, int ctx, uint32_t tmem, uint64_t* mma_bar,
                                                uint32_t& mma_ph, const TcLane& L, float* xch, uint32_t& gp, float& m,
                                                float& l, int32_t* status) {
    uint8_t* q_tile = smem + kTcQ;
    uint8_t* k_tile = smem + kTcK;
    uint8_t* vt_tile = smem + kTcV;
    uint8_t* p_tile = smem + kTcP;
    float* kscale = reinterpret_cast<float*>(smem + kTcScale);
    float* vscale = kscale + 128;
    const uint32_t s_cols = tmem + ((uint32_t)(L.r & ~31) << 16) + 64 * L.h;   // this warp's lanes, its half
    const uint32_t o_cols = s_cols + 128;
    constexpr uint32_t kIdesc = idesc_bf16(128, 128);
    bool ok_all = true;
#pragma unroll 1
    for (int i = 0; i < np; ++i) {
        const int st = (int)((gp + i) & 1);
        const uint32_t parity = (uint32_t)(((gp + i) >> 1) & 1);
        const bool ok = mbar_wait_bounded(&sm.mbar[st], parity);
        if (__syncthreads_or(!ok)) {
            if (threadIdx.x == 0) attend_drain(sm, st, parity, i + 1 < np, (uint32_t)(((gp + i + 1) >> 1) & 1), status);
            __syncthreads();
            ok_all = false;
            break;
        }
        const int p = sm.stage_page[st];
        const int valid_rows = p >= 0 ? min(kPage, ctx - p * kPage) : 0;
        const int jpage = p >= 0 ? p * kPage : 0;
        const uint8_t* rk = sm.raw + st * 2 * page_bytes;
        widen_k_tc<RS>(rk, valid_rows, k_tile, kscale);
        widen_vt_tc<RS>(rk + page_bytes, valid_rows, vt_tile, vscale);
        fence_proxy_async_smem();   // the tiles (generic writes) before the MMAs read them
        __syncthreads();            // tiles ready; this stage's raw bytes are consumed
        if (threadIdx.x == 0) {
            if (i + 2 < np) attend_issue(sm, i + 2, sel[i + 2], selph[i + 2], gp, k_pool, v_pool, Hkv, kvh, page_bytes);
            tc_fence_after_sync();
            tc_mma_tile(tmem, smem_u32(q_tile), smem_u32(k_tile), kTcRows, kTcRows, kIdesc, false, mma_bar);
        }
        bool mma_ok = tc_wait(mma_bar, mma_ph & 1);
        ++mma_ph;
        tc_fence_after_sync();
        // the row maximum over this half (S is read twice from tensor memory rather than kept)
        float mx = -INFINITY;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
            float z[16];
            tc_scores16<RS>(s_cols + 16 * c, 64 * L.h + 16 * c, jpage, valid_rows, L, kscale, z);
#pragma unroll
            for (int j = 0; j < 16; ++j) mx = fmaxf(mx, z[j]);
        }
        xch[threadIdx.x] = mx;
        __syncthreads();
        mx = fmaxf(mx, xch[threadIdx.x ^ 128]);   // the partner thread holds the other half of the row
        const float m_new = fmaxf(m, mx);
        const float alpha = (m_new == -INFINITY) ? 1.0f : exp2f(m - m_new);
        m = m_new;
        l *= alpha;
        if (i > 0 && __any_sync(0xFFFFFFFFu, alpha != 1.0f)) {
            // a row's maximum grew: rescale the warp's output columns in place (the last PV is
            // done); the whole warp takes part (alpha is 1 for the other rows)
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
                float ov[16];
                tmem_ld16(o_cols + 16 * c, ov);
#pragma unroll
                for (int j = 0; j < 16; ++j) ov[j] *= alpha;
                tmem_st16(o_cols + 16 * c, ov);
            }
        }
        // weights of this half: bf16 (MXFP4); FP8-KV: p x V row scale as high + low bf16 parts,
        // the low part in the K tile (S is computed, the K tile is free)
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
            float z[16];
            tc_scores16<RS>(s_cols + 16 * c, 64 * L.h + 16 * c, jpage, valid_rows, L, kscale, z);
            uint32_t hw[8], lw[8];
#pragma unroll
            for (int q2 = 0; q2 < 8; ++q2) {
                float e0 = (m_new == -INFINITY) ? 0.0f : exp2f(z[2 * q2] - m_new);
                float e1 = (m_new == -INFINITY) ? 0.0f : exp2f(z[2 * q2 + 1] - m_new);
                if (RS) {
                    const int tok = 64 * L.h + 16 * c + 2 * q2;
                    l += e0 + e1;
                    e0 *= vscale[tok];
                    e1 *= vscale[tok + 1];
                }
                const __nv_bfloat162 hb = __floats2bfloat162_rn(e0, e1);
                const float2 hr = __bfloat1622float2(hb);
                if (!RS) l += hr.x + hr.y;
                hw[q2] = *reinterpret_cast<const uint32_t*>(&hb);
                if (RS) {
                    const __nv_bfloat162 lb = __floats2bfloat162_rn(e0 - hr.x, e1 - hr.y);
                    lw[q2] = *reinterpret_cast<const uint32_t*>(&lb);
                }
            }
            const int ch = 8 * L.h + 2 * c;   // 16-byte chunks ch, ch + 1 of the row
            *reinterpret_cast<uint4*>(p_tile + sw128_chunk(L.r, ch, kTcRows)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            *reinterpret_cast<uint4*>(p_tile + sw128_chunk(L.r, ch + 1, kTcRows)) = make_uint4(hw[4], hw[5], hw[6], hw[7]);
            if (RS) {
                *reinterpret_cast<uint4*>(k_tile + sw128_chunk(L.r, ch, kTcRows)) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
                *reinterpret_cast<uint4*>(k_tile + sw128_chunk(L.r, ch + 1, kTcRows)) = make_uint4(lw[4], lw[5], lw[6], lw[7]);
            }
        }
        fence_proxy_async_smem();   // P (generic writes) before the MMA reads it
        tc_fence_before_sync();
        __syncthreads();
        if (threadIdx.x == 0) {
            tc_fence_after_sync();
            if (RS) {
                // O (+)= P_hi V^T + P_lo V^T, one commit after both
                tc_mma_tile(tmem + 128, smem_u32(p_tile), smem_u32(vt_tile), kTcRows, kTcRows, kIdesc, i > 0, nullptr);
                tc_mma_tile(tmem + 128, smem_u32(k_tile), smem_u32(vt_tile), kTcRows, kTcRows, kIdesc, true, mma_bar);
            } else {
                tc_mma_tile(tmem + 128, smem_u32(p_tile), smem_u32(vt_tile), kTcRows, kTcRows, kIdesc, i > 0, mma_bar);
            }
        }
        mma_ok = tc_wait(mma_bar, mma_ph & 1) && mma_ok;
        ++mma_ph;
        tc_fence_after_sync();
        if (__syncthreads_or(!mma_ok)) {   // the tiles are free for the next page
            if (threadIdx.x == 0) flag_status(status, SMX_DEV_TIMEOUT);
            ok_all = false;
            break;
        }
    }
    gp += (uint32_t)np;
    return ok_all;
}

// Partials of this CTA's real rows for partition s: O from tensor-memory columns 128..255 (zero
// if the partition had no page), the row's l this half's plus the partner's (exchanged through
// xch); half h writes dims 64 h .. 64 h + 63. part_o [B][S][Q][Hq][128], part_m / part_l
// [B][S][Q][Hq]; unit row i is query row m_lo + i. Every thread calls it.
__device__ __forceinline__ void finish_partials_tc(const TcLane& L, uint32_t tmem, bool have_o, float m, float l,
                                                   float* xch, float* part_o, float* part_m, float* part_l, int b, int s,
                                                   int kvh, int S, int Q, int Hq, int G, int m_lo) {
    __syncthreads();   // xch free (its last readers passed the page loop's final barrier)
    xch[threadIdx.x] = l;
    __syncthreads();
    const float l_row = l + xch[threadIdx.x ^ 128];
    const int mq = m_lo + L.r;
    const int64_t row = (((int64_t)b * S + s) * Q + (L.valid ? mq / G : 0)) * Hq + kvh * G + (L.valid ? mq % G : 0);
    float4* dst = reinterpret_cast<float4*>(part_o + row * kD + 64 * L.h);
    const uint32_t o_cols = tmem + ((uint32_t)(L.r & ~31) << 16) + 128 + 64 * L.h;
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
        float ov[16];
        if (have_o) {
            tmem_ld16(o_cols + 16 * c, ov);   // every lane of the warp takes part
        } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) ov[j] = 0.0f;
        }
        if (L.valid) {
#pragma unroll
            for (int j = 0; j < 4; ++j) dst[4 * c + j] = make_float4(ov[4 * j], ov[4 * j + 1], ov[4 * j + 2], ov[4 * j + 3]);
        }
    }
    if (L.valid && L.h == 0) {
        part_m[row] = m;
        part_l[row] = l_row;
    }
}

}  // namespace smx

// smx_attend_tc.cuh -- the split stage (a5) of one partition on the fifth-generation tensor cores:
// QK and PV as 128 x 128 x 128 tcgen05 MMAs with fp32 accumulators in tensor memory.
//
// [ATOM-2812] "Mono decode over the MXFP4 KV and index caches", commit "MXFP4 main KV": QK against
// the K page (fp4 with E8M0 group scales) and the e4m3 q, softmax with P in bf16, PV against V
// widened to bf16 on chip, (sp_o, sp_m, sp_l) per partition.
//
// One CTA (8 warps) serves up to 128 query rows of one KV head; rows are (draft token, head)
// pairs. Thread (warp w, lane l) owns query row 32 (w % 4) + l and token / dim half w / 4. Per
// selected page, staged by bulk copies (two pages in flight):
//
// MXFP4 K/V (attend_pages_tc_mx):
//  1. The K page's nibbles are copied into the fp4 operand layout (no conversion) and its E8M0
//     scale words into the B scale block in tensor memory; one thread issues S = q K^T as four
//     block-scaled MMAs (kind::mxf8f6f4, e4m3 q with unit scales, one per 32-dim group).
//  2. Meanwhile V is widened to bf16 row by row ([token][dim], read by the PV MMA as an MN-major
//     operand; token rows past the context are zero, so poisoned slots never reach an MMA).
//  3. Each thread reads its 64 scores with one tensor-memory load, masks them, exchanges the half
//     maximum with its partner thread, and writes its half of P as a bf16 high part and a bf16
//     low part (~16 significant bits; two PV passes; the PV MMAs also sum the weights they use,
//     against a column of ones appended to V: N = 144). The running maximum
//     follows the row maximum exactly, so the largest weight is exactly 1 (a maximum that lags by
//     up to 8 would leave every weight rounded: on rows scaled x50 that alone breaks the output
//     bound); O is rescaled in tensor memory when a row's maximum grows.
//  4. One thread issues O += P_hi V + P_lo V (sixteen MMAs) into columns 128..271; the next
//     page's K copy and QK go ahead while it runs, and V / P are rewritten only after it
//     completes.
//
// FP8-KV (attend_pages_tc): K widened to bf16 and V transposed into [dim][token] tiles, both
// K-major; QK and PV as bf16 MMAs; p times the V row scale as a bf16 high part and low part.
#pragma once

#include <math.h>

#include "smx_attend.cuh"
#include "smx_device.cuh"
#include "smx_tc.cuh"

namespace smx {

// Dynamic shared memory of the tensor-core attention (base 1024-byte aligned).
constexpr int kTcQ = 0;             // q tile [128 rows][128 dims]: e4m3 (MXFP4), bf16 (FP8-KV)
constexpr int kTcK = 32768;         // K tile [128 tokens][128 dims]: fp4 operand (MXFP4), bf16 (FP8-KV,
                                    // then the P low part)
constexpr int kTcV = 65536;         // V tile, bf16: [token][dim] (MXFP4), [dim][token] (FP8-KV)
constexpr int kTcP = 98304;         // P tile [128 rows][128 tokens] (FP8-KV); MXFP4: V's third block
constexpr int kTcMxP0 = 16384;      // MXFP4 P tile, tokens 0..63 [128 rows][64] (after the e4m3 q tile)
constexpr int kTcMxP1 = 49152;      // MXFP4 P tile, tokens 64..127 (after the fp4 K tile)
constexpr int kTcScale = 131072;    // 128 K row scales, 128 V row scales (FP8-KV)
constexpr int kTcRaw = 132096;      // two stages of (K page, V page) (FP8-KV)
constexpr int kTcMxPL0 = 114688;    // MXFP4 P low part, tokens 0..63 (after V's third block)
constexpr int kTcMxPL1 = 131072;    // MXFP4 P low part, tokens 64..127
constexpr int kTcMxRaw = 147456;    // MXFP4: two stages of (K page, V page)
constexpr uint32_t kTcCols = 512;   // tensor-memory columns allocated
constexpr uint32_t kTcColO = 128;   // S at column 0, O at 128 (MXFP4: 144 columns, the last 16 from
                                    // V's column of ones: column 256 is the row's weight sum l)
constexpr uint32_t kTcColSFA = 288; // the A (q) scale block: 0x7F (2^0) in every byte
constexpr uint32_t kTcColSFB = 296; // the B (K page) scale block
constexpr int kTcMxN = 144;         // MXFP4 PV: 128 V dims + 16 (a column of ones, then zeros)
constexpr int kTcRows = 128;        // query rows per CTA

__host__ __device__ constexpr size_t attend_tc_smem_bytes(int page_bytes) {
    return (size_t)(page_bytes == kMxPageBytes ? kTcMxRaw : kTcRaw) + 4 * (size_t)page_bytes;
}

// The q tile from `rows` query rows (rows past them are zero). MXFP4 K/V: e4m3 codes by the q
// packing rule, 128-byte rows; FP8-KV: bf16, 256-byte rows. Staged rows at src (shared memory):
// 512-byte f32 rows (MXFP4), 256-byte bf16 rows (FP8-KV). Every thread of the 256-thread block.
template <bool RS>
__device__ __forceinline__ void pack_q_tile_tc(const uint8_t* src, int rows, uint8_t* tile) {
    if constexpr (RS) {
        const int r = threadIdx.x >> 1, h = threadIdx.x & 1;
#pragma unroll 1
        for (int c = 0; c < 8; ++c) {   // chunk c of the half: dims 64 h + 8 c .. + 7
            uint4 v = make_uint4(0, 0, 0, 0);
            if (r < rows) v = *reinterpret_cast<const uint4*>(src + r * 256 + (8 * h + c) * 16);
            *reinterpret_cast<uint4*>(tile + sw128_chunk(r, 8 * h + c, kTcRows)) = v;
        }
    } else {
        // warp w packs rows w, w + 8, ...; lane l dims 4 l .. 4 l + 3 (one 512-byte row per warp)
        const int lane = threadIdx.x & 31;
#pragma unroll 4
        for (int r = threadIdx.x >> 5; r < kTcRows; r += 8) {   // 8 warps
            uint32_t w = 0;
            if (r < rows) {
                const float4 f = *reinterpret_cast<const float4*>(src + r * 512 + lane * 16);
                w = pack_q2(f.x, f.y) | (pack_q2(f.z, f.w) << 16);
            }
            *reinterpret_cast<uint32_t*>(tile + sw128_chunk(r, lane >> 2, kTcRows) + 4 * (lane & 3)) = w;
        }
    }
}

// The same from global q rows: unit row i is q row (b, (m_lo + i) / G, kvh G + (m_lo + i) % G).
template <bool RS>
__device__ __forceinline__ void pack_q_tile_tc_global(const void* q, int b, int kvh, int m_lo, int rows, int Q, int Hq,
                                                      int G, uint8_t* tile) {
    auto q_row = [&](int i) {   // global row of unit row i < rows
        const int m = m_lo + i;
        return ((int64_t)b * Q + m / G) * Hq + kvh * G + m % G;
    };
    if constexpr (RS) {
        const int r = threadIdx.x >> 1, h = threadIdx.x & 1;
        const int64_t row = q_row(r < rows ? r : 0);
#pragma unroll 1
        for (int c = 0; c < 8; ++c) {
            uint4 v = make_uint4(0, 0, 0, 0);
            if (r < rows) v = *reinterpret_cast<const uint4*>(reinterpret_cast<const uint8_t*>(q) + row * 256 + (8 * h + c) * 16);
            *reinterpret_cast<uint4*>(tile + sw128_chunk(r, 8 * h + c, kTcRows)) = v;
        }
    } else {
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
        constexpr int kPer = kTcRows / 8;   // rows per warp
        float4 f[kPer];
#pragma unroll
        for (int k = 0; k < kPer; ++k) {   // all loads in flight together
            const int r = warp + 8 * k;
            f[k] = r < rows ? *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(q) + q_row(r) * kD + 4 * lane)
                            : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        }
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            const int r = warp + 8 * k;
            const uint32_t w = pack_q2(f[k].x, f[k].y) | (pack_q2(f[k].z, f[k].w) << 16);
            *reinterpret_cast<uint32_t*>(tile + sw128_chunk(r, lane >> 2, kTcRows) + 4 * (lane & 3)) = w;
        }
    }
}

// A K or V page (raw, shared memory) -> bf16 tile [token][dim] (K-major for the token as the
// row); FP8-KV row scales -> rscale. Token rows at or past valid_rows are zero.
template <bool RS>
__device__ __forceinline__ void widen_rows_tc(const uint8_t* raw, int valid_rows, uint8_t* tile, float* rscale) {
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

// MXFP4 K page (raw, shared memory) -> the fp4 operand tile [token][128 dims] (each 16-dim chunk:
// its 8 nibble bytes, then 8 zero bytes) and its E8M0 scale words -> the B scale block (token t's
// word, byte g = group g, in lane t % 32 of column t / 32, every quadrant: warp w < 4 writes
// quadrant w). Token rows past the context keep whatever the page holds: their scores are masked.
__device__ __forceinline__ void repack_k_mx_tc(const uint8_t* raw, uint8_t* tile, uint32_t tmem) {
    uint2 w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {   // 128 tokens x 8 chunks over the 256 threads
        const int it = (int)threadIdx.x + 256 * k;
        w[k] = *reinterpret_cast<const uint2*>(raw + (it >> 3) * 64 + (it & 7) * 8);
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int it = (int)threadIdx.x + 256 * k;
        *reinterpret_cast<uint4*>(tile + sw128_chunk(it >> 3, it & 7, kTcRows)) = make_uint4(w[k].x, w[k].y, 0u, 0u);
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp < 4) {
        const uint32_t* sc = reinterpret_cast<const uint32_t*>(raw + kMxScaleOff);
        tmem_st4(tmem + ((uint32_t)(32 * warp) << 16) + kTcColSFB, sc[lane], sc[32 + lane], sc[64 + lane], sc[96 + lane]);
    }
}

// 2^x for the softmax weights (x <= 0; -inf gives 0): the hardware base-2 exponential.
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
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
        widen_rows_tc<RS>(rk, valid_rows, k_tile, kscale);
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

// MXFP4 K/V copies: the K or V page of entry i into slot (gp + i) % 2 of the stage area
// (slot s: K page at raw + 2 s page_bytes, V page right after it), completing on cbar[slot] (K)
// or cbar[2 + slot] (V). phys < 0: no copy, the barrier's phase completes at once. One thread.
__device__ __forceinline__ void mx_issue(uint8_t* raw, uint64_t* cbar, int i, bool v, int64_t phys, uint32_t gp,
                                         const uint8_t* pool, int Hkv, int kvh, int page_bytes) {
    const int st = (int)((gp + i) & 1);
    uint64_t* bar = &cbar[(v ? 2 : 0) + st];
    if (phys < 0) {
        mbar_arrive(bar);
        return;
    }
    mbar_arrive_expect_tx(bar, (uint32_t)page_bytes);
    bulk_g2s(raw + st * 2 * page_bytes + (v ? page_bytes : 0), pool + (phys * Hkv + kvh) * (int64_t)page_bytes,
             (uint32_t)page_bytes, bar);
}

// bf16x2 product (round to nearest even; exact here: powers of two times codes).
__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// The two bf16x2 factors whose product is 2^(b - 15) for an E8M0 byte b (each a power of two in
// bf16's normal range for every b < 255; b = 255 gives NaN, as the E8M0 NaN code).
__device__ __forceinline__ void v_scale_factors(uint32_t b, uint32_t& s1, uint32_t& s2) {
    const int k = (int)b - 15, k1 = k >> 1, k2 = k - k1;
    const uint32_t e1 = (uint32_t)(k1 + 127) << 7, e2 = (uint32_t)(k2 + 127) << 7;
    s1 = b == 0xFFu ? 0x7FC07FC0u : (e1 | (e1 << 16));
    s2 = e2 | (e2 << 16);
}

// One 16-byte chunk of the V tile: 8 E2M1 codes (w) times 2^(b - 127) as bf16 (exact). Each code's
// f16 (exact) with its exponent and mantissa bits shifted down by 3 is a bf16 holding the code
// times 2^-112 (zero stays zero); two power-of-two multiplies (s1 s2 = 2^(b - 15)) finish it.
// No conversion-pipe work past the E2M1 -> f16 conversion.
__device__ __forceinline__ uint4 widen_v_chunk(uint32_t w, uint32_t s1, uint32_t s2) {
    uint32_t h[4], o[4];
    e2m1x8_to_f16x2(w, h[0], h[1], h[2], h[3]);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const uint32_t t = ((h[q] & 0x7FFF7FFFu) >> 3) | (h[q] & 0x80008000u);
        o[q] = bf16x2_mul(bf16x2_mul(t, s1), s2);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// MXFP4 K/V: the pages sel[0..np) / selph[0..np) of this CTA's partition. The caller issued the
// K and V copies of entries 0 and 1 (mx_issue, in that order: K 0, V 0, K 1, V 1); the q tile
// holds e4m3 codes; the A scale block (column kTcColSFA) holds 0x7F in every byte. cbar: copy
// barriers [K slot 0, K slot 1, V slot 0, V slot 1]; bars[0] counts QK completions (qk_ph phases
// seen), bars[1] PV completions (pv_ph). Per page i, with two CTA barriers:
//   (QK i was issued during page i - 1) K i + 1 is repacked (QK i is done, so the K tile and B
//   scale block are free; PV i - 1 may still run) and S i is read and masked; barrier B; thread 0 issues QK i + 1 and the
//   K copy of page i + 3; the row maxima are combined, PV i - 1 is waited for, O is rescaled,
//   and P i (ex2) is written interleaved with the widening of V i (ALU and conversion pipes);
//   the PV MMA (N = 144) also sums the bf16 weights, against V's column of ones;
//   barrier C; thread 224 issues PV i, thread 32 the V copy of page i + 2.
// m: the row's running maximum (log2 domain). l: on return, the row's weight sum relative to 2^m
// (column 128 of O, from V's column of ones) in the h = 0 thread, 0 in the other (as the FP8-KV
// loop's halves, which the partials add). Returns false (every thread alike) if a copy or an MMA did not finish within the bounded wait
// (status gets SMX_DEV_TIMEOUT); O is then incomplete.
__device__ __forceinline__ bool attend_pages_tc_mx(uint8_t* smem, uint8_t* raw, uint64_t* cbar, const int* sel,
                                                   const int* selph, int np, const uint8_t* k_pool,
                                                   const uint8_t* v_pool, int Hkv, int kvh, int page_bytes, int ctx,
                                                   uint32_t tmem, uint64_t* bars, uint32_t& qk_ph, uint32_t& pv_ph,
                                                   const TcLane& L, float* xch, uint32_t& gp, float& m, float& l,
                                                   int32_t* status) {
    uint8_t* q_tile = smem + kTcQ;
    uint8_t* k_tile = smem + kTcK;
    uint8_t* v_tile = smem + kTcV;
    uint8_t* p_half = smem + (L.h ? kTcMxP1 : kTcMxP0);    // this thread's half of the P tile
    uint8_t* pl_half = smem + (L.h ? kTcMxPL1 : kTcMxPL0); // and of its low part
    const uint32_t lane_base = tmem + ((uint32_t)(L.r & ~31) << 16);   // this warp's 32 lanes
    const uint32_t s_cols = lane_base + 64 * L.h;
    const uint32_t o_cols = lane_base + kTcColO + 64 * L.h;
    const uint32_t l_col = lane_base + kTcColO + 128;   // O's column 128: the row's weight sum
    // V's third 64-dim block: dim 128 is 1 for every token, dims 129..143 are 0 (read by the PV
    // MMA as N = 144, so the MMA sums the bf16 weights it multiplies)
    {
        const int t = threadIdx.x >> 1, j = threadIdx.x & 1;
        *reinterpret_cast<uint4*>(v_tile + sw128_chunk(t, 16 + j, kTcRows)) =
            make_uint4(j == 0 ? 0x3F80u : 0u, 0u, 0u, 0u);
    }
    auto slot = [&](int i) { return (int)((gp + i) & 1); };
    auto par = [&](int i) { return (uint32_t)(((gp + i) >> 1) & 1); };
    auto k_raw = [&](int i) { return raw + slot(i) * 2 * page_bytes; };
    // copies issued / waited for (pages), MMA commits issued: the same in every thread
    int k_iss = min(np, 2), v_iss = min(np, 2), k_done = 0, v_done = 0;
    uint32_t qk_iss = qk_ph, pv_iss = pv_ph;
    bool ok_all = true;

    // K 0 and QK 0
    bool ok = mbar_wait_bounded(&cbar[slot(0)], par(0));
    if (ok) k_done = 1;
    repack_k_mx_tc(k_raw(0), k_tile, tmem);
    fence_proxy_async_smem();
    tc_fence_before_sync();
    if (__syncthreads_or(!ok)) {
        ok_all = false;
    } else {
        if (threadIdx.x == 0) {
            tc_fence_after_sync();
            tc_mma_mx_tile(tmem, smem_u32(q_tile), smem_u32(k_tile), tmem + kTcColSFA, tmem + kTcColSFB);
            tc_commit(&bars[0]);
            if (np > 2) mx_issue(raw, cbar, 2, false, selph[2], gp, k_pool, Hkv, kvh, page_bytes);
        }
        ++qk_iss;
        if (np > 2) ++k_iss;
    }

#pragma unroll 1
    for (int i = 0; ok_all && i < np; ++i) {
        const int p = selph[i] >= 0 ? sel[i] : -1;
        const int valid_rows = p >= 0 ? min(kPage, ctx - p * kPage) : 0;
        const int jpage = p >= 0 ? p * kPage : 0;
        ok = tc_wait(&bars[0], qk_ph & 1);   // QK i
        ++qk_ph;
        tc_fence_after_sync();
        // K i + 1 first (QK i is done: the K tile and the B scale block are free): it needs no
        // tensor-memory read, so it runs while PV i - 1 still occupies tensor memory
        if (i + 1 < np) {
            if (mbar_wait_bounded(&cbar[slot(i + 1)], par(i + 1))) k_done = i + 2;
            else ok = false;
            repack_k_mx_tc(k_raw(i + 1), k_tile, tmem);
        }
        // S i: scaled to the log2 domain, masked past the context and causally
        float z[64];   // raw q.k; the log2-domain scale is applied with the maximum below
        tmem_ld64(s_cols, z);
        const int lim = L.valid ? min(valid_rows, L.pos - jpage + 1) - 64 * L.h : 0;
        float mx = -INFINITY;
#pragma unroll
        for (int j = 0; j < 64; ++j) {
            z[j] = j < lim ? z[j] : -INFINITY;
            mx = fmaxf(mx, z[j]);
        }
        mx *= kLog2eOverSqrtD;
        xch[threadIdx.x] = mx;
        fence_proxy_async_smem();
        tc_fence_before_sync();   // S i read; the B scale block written
        if (__syncthreads_or(!ok)) {
            ok_all = false;
            break;
        }
        if (threadIdx.x == 0) {
            if (i + 1 < np) {
                tc_fence_after_sync();
                tc_mma_mx_tile(tmem, smem_u32(q_tile), smem_u32(k_tile), tmem + kTcColSFA, tmem + kTcColSFB);
                tc_commit(&bars[0]);
            }
            if (i + 3 < np) mx_issue(raw, cbar, i + 3, false, selph[i + 3], gp, k_pool, Hkv, kvh, page_bytes);
        }
        if (i + 1 < np) ++qk_iss;
        if (i + 3 < np) ++k_iss;

        mx = fmaxf(mx, xch[threadIdx.x ^ 128]);   // the partner thread holds the other half of the row
        const bool raise = mx > m;   // false while the row has seen nothing (mx = -inf)
        const float alpha = raise ? ex2_approx(m - mx) : 1.0f;   // m = -inf: 0
        if (raise) m = mx;
        // PV i - 1 done: O, the P tile and the V tile are free
        bool ok2 = true;
        if (pv_iss != pv_ph) {
            ok2 = tc_wait(&bars[1], pv_ph & 1);
            ++pv_ph;
            tc_fence_after_sync();
        }
        if (i > 0 && __any_sync(0xFFFFFFFFu, raise)) {
            float ov[64];
            tmem_ld64(o_cols, ov);
#pragma unroll
            for (int j = 0; j < 64; ++j) ov[j] *= alpha;
            tmem_st64(o_cols, ov);
            if (L.h) tmem_st1(l_col, tmem_ld1(l_col) * alpha);   // warp-uniform: h is the warp's half
        }
        if (mbar_wait_bounded(&cbar[2 + slot(i)], par(i))) v_done = i + 1;
        else ok2 = false;
        // this half of P as bf16 (l sums the rounded weights the MMA uses), interleaved with this
        // thread's two (token, 32-dim group) items of V: item t + 256 k is token (t + 256 k) / 4,
        // group t % 4; chunk q of an item is dims 32 g + 8 q .. + 7
        const uint8_t* vr = k_raw(i) + page_bytes;
        uint4 vw[2];
        uint32_t vs1[2], vs2[2];
        int vrow[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int it = (int)threadIdx.x + 256 * k;
            vrow[k] = it >> 2;
            vw[k] = *reinterpret_cast<const uint4*>(vr + vrow[k] * 64 + (it & 3) * 16);
            v_scale_factors(vr[kMxScaleOff + it], vs1[k], vs2[k]);
        }
        const float nmb = m == -INFINITY ? 0.0f : -m;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            uint32_t hw[4], lw[4];
#pragma unroll
            for (int q2 = 0; q2 < 4; ++q2) {
                const float e0 = ex2_approx(fmaf(z[8 * c + 2 * q2], kLog2eOverSqrtD, nmb));
                const float e1 = ex2_approx(fmaf(z[8 * c + 2 * q2 + 1], kLog2eOverSqrtD, nmb));
                hw[q2] = f32x2_to_bf16x2(e0, e1);
                lw[q2] = f32x2_to_bf16x2(e0 - __uint_as_float(hw[q2] << 16), e1 - __uint_as_float(hw[q2] & 0xFFFF0000u));
            }
            *reinterpret_cast<uint4*>(p_half + sw128_chunk(L.r, c, kTcRows)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            *reinterpret_cast<uint4*>(pl_half + sw128_chunk(L.r, c, kTcRows)) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
            const int k = c >> 2, q = c & 3;
            const int g = ((int)threadIdx.x + 256 * k) & 3;
            const uint32_t w = q == 0 ? vw[k].x : q == 1 ? vw[k].y : q == 2 ? vw[k].z : vw[k].w;
            const uint4 o = vrow[k] < valid_rows ? widen_v_chunk(w, vs1[k], vs2[k]) : make_uint4(0u, 0u, 0u, 0u);
            *reinterpret_cast<uint4*>(v_tile + sw128_chunk(vrow[k], 4 * g + q, kTcRows)) = o;
        }
        fence_proxy_async_smem();   // P and V (generic writes) before the MMA reads them
        tc_fence_before_sync();     // the O accesses before the next MMAs
        if (__syncthreads_or(!ok2)) {
            ok_all = false;
            break;
        }
        if (threadIdx.x == 224) {
            tc_fence_after_sync();
            tc_mma_tile_bmn(tmem + kTcColO, smem_u32(smem + kTcMxP0), smem_u32(smem + kTcMxP1), smem_u32(v_tile), kTcMxN,
                            i > 0);
            tc_mma_tile_bmn(tmem + kTcColO, smem_u32(smem + kTcMxPL0), smem_u32(smem + kTcMxPL1), smem_u32(v_tile), kTcMxN,
                            true);
            tc_commit(&bars[1]);
        }
        if (threadIdx.x == 32 && i + 2 < np)
            mx_issue(raw, cbar, i + 2, true, selph[i + 2], gp, v_pool, Hkv, kvh, page_bytes);
        ++pv_iss;
        if (i + 2 < np) ++v_iss;
    }

    // drain: every MMA committed and every copy issued completes before the tiles, the stage area
    // or tensor memory are used again (bounded waits; a timeout is flagged)
    bool ok3 = true;
    while (pv_ph != pv_iss) {
        ok3 = tc_wait(&bars[1], pv_ph & 1) && ok3;
        ++pv_ph;
    }
    while (qk_ph != qk_iss) {
        ok3 = tc_wait(&bars[0], qk_ph & 1) && ok3;
        ++qk_ph;
    }
    tc_fence_after_sync();
    if (!ok_all && threadIdx.x == 0) {
        for (int j = k_done; j < k_iss; ++j) mbar_wait_bounded(&cbar[slot(j)], par(j));
        for (int j = v_done; j < v_iss; ++j) mbar_wait_bounded(&cbar[2 + slot(j)], par(j));
    }
    if ((!ok_all || !ok3) && threadIdx.x == 0) flag_status(status, SMX_DEV_TIMEOUT);
    // the row's weight sum, from the MMA: held by the h = 0 thread (the partner's share is 0)
    const float l_row = tmem_ld1(l_col);
    l = L.h ? 0.0f : l_row;
    gp += (uint32_t)np;
    return __syncthreads_and(ok_all && ok3) != 0;
}

// Partials of this CTA's real rows for partition s: O from tensor-memory columns 128..255 (zero
// if the partition had no page), the row's l this half's plus the partner's (exchanged through
// xch). part_o [B][S][Q][Hq][128], part_m / part_l [B][S][Q][Hq]; unit row i is query row
// m_lo + i. O goes through `stage` (64 KB of free shared memory, 16-byte aligned: 128 rows of
// 512 bytes, the 16-byte chunk q of row i at chunk q ^ (i % 32)), so that each warp writes whole
// 512-byte rows of part_o (a thread's own half row would scatter 16-byte pieces over 32 rows).
// Every thread calls it, after the page loop drained (the tiles are free).
__device__ __forceinline__ void finish_partials_tc(const TcLane& L, uint32_t tmem, bool have_o, float m, float l,
                                                   float* xch, uint8_t* stage, float* part_o, float* part_m,
                                                   float* part_l, int b, int s, int kvh, int S, int Q, int Hq, int G,
                                                   int m_lo, int rows) {
    __syncthreads();   // xch and the stage free (their last readers passed the page loop's final barrier)
    xch[threadIdx.x] = l;
    const uint32_t o_cols = tmem + ((uint32_t)(L.r & ~31) << 16) + 128 + 64 * L.h;
    uint4* srow = reinterpret_cast<uint4*>(stage) + L.r * 32;
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
        float ov[16];
        if (have_o) {
            tmem_ld16(o_cols + 16 * c, ov);   // every lane of the warp takes part
        } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) ov[j] = 0.0f;
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int q = 16 * L.h + 4 * c + k;   // logical chunk: dims 4 q .. 4 q + 3
            srow[q ^ (L.r & 31)] = make_uint4(__float_as_uint(ov[4 * k]), __float_as_uint(ov[4 * k + 1]),
                                              __float_as_uint(ov[4 * k + 2]), __float_as_uint(ov[4 * k + 3]));
        }
    }
    __syncthreads();
    const int mq = m_lo + L.r;
    if (L.valid && L.h == 0) {
        const int64_t row = (((int64_t)b * S + s) * Q + mq / G) * Hq + kvh * G + mq % G;
        part_m[row] = m;
        part_l[row] = l + xch[threadIdx.x ^ 128];
    }
    // whole rows: warp w writes unit rows w, w + 8, ..., lane j the dims 4 j .. 4 j + 3
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint4* st4 = reinterpret_cast<const uint4*>(stage);
#pragma unroll 4
    for (int i = warp; i < rows; i += 8) {
        const int mi = m_lo + i;
        const int64_t row = (((int64_t)b * S + s) * Q + mi / G) * Hq + kvh * G + mi % G;
        reinterpret_cast<uint4*>(part_o + row * kD)[lane] = st4[i * 32 + (lane ^ (i & 31))];
    }
}

}  // namespace smx

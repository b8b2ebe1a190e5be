// smx_attend.cuh -- split-K attention over one partition's selected pages (a5) and the merge of
// one output row (a6), shared by the standalone kernels and the fused decode step.
//
// [ATOM-2812] "Mono decode over the MXFP4 KV and index caches", commit "MXFP4 main KV": the
// split stage runs QK against the K page (fp4 with E8M0 group scales) and the e4m3 q, softmax
// with P in bf16 registers, PV against V widened to bf16 in on-chip memory, and writes
// (sp_o, sp_m, sp_l) per partition; the merge combines the partitions.
//
// A CTA serves one (row b, KV head, group of up to 64 query rows); rows are (draft token t, head
// of the KV group) pairs, so QK and PV are dense 16-row tiles for the m16n8k16 bf16 MMA. Per
// selected page the CTA stages K and V with 1-D bulk copies (two pages in flight), widens them to
// bf16 in shared memory (E2M1 x 2^e and e4m3 codes are exact in bf16), zeroing token rows past
// the context so poisoned slots never reach an MMA, with a 16-byte XOR swizzle that keeps
// ldmatrix conflict-free. Warp (half h, group w) owns 16 rows and 64 tokens of every page, in
// 16-token units: QK (fp32), mask, online softmax in the log2 domain (rescale only when a row's
// maximum grows), then the weights -- p (FP8-KV: p times the V row scale) as a bf16 high part
// plus a bf16 low part, so they keep ~16 significant bits -- multiplied into V (the accumulator
// layout of QK is the A layout of PV). The pages keep P in bf16 alone; that is the reading kept
// here only for the high part: when a few tokens share a row's mass, one bf16 rounding of their
// weights moves outputs near zero by ~2^-9 |v_i - v_j|, the size of the output bound. The two
// token halves are combined in shared memory at the end.
#pragma once

#include <math.h>

#include "smx_device.cuh"

namespace smx {

constexpr int kAttnMaxWarps = 8;   // 2 token halves x 4 row groups
constexpr int kAttnRegionBytes = 65536;
constexpr float kLog2eOverSqrtD = (float)(1.4426950408889634 / 11.313708498984761);

// bf16 tile [128 tokens][128 dims], 256 B rows, 16-B chunk c of row r stored at c ^ (r & 7).
__device__ __forceinline__ uint32_t swz(int row, int chunk) { return row * 256 + ((chunk ^ (row & 7)) << 4); }

// Widen one staged page (K or V of one KV head, raw bytes in shared memory) to bf16 tiles in
// shared memory (exact in both formats). For the e4m3 row-scale pages the codes are widened
// unscaled and the row scales go to rscale[]: K's scale multiplies the scores, V's multiplies
// the softmax weights. Token rows at or past valid_rows are zero.
template <bool RS>
__device__ __forceinline__ void widen_page(const uint8_t* raw, int valid_rows, uint8_t* tile, float* rscale,
                                           bool nv = false) {
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
    } else {
        // MXFP4: 128 rows x 4 chunks of 16 nibble bytes (32 elements = one scale group). NVFP4 (nv):
        // the chunk is blocks 2c (words 0, 1) and 2c + 1 (words 2, 3), each with an E4M3 scale; the
        // product E2M1 x E4M3 (at most 6 significant bits) is exact in bf16, and the pool's
        // per-tensor scale is applied by the caller (to the scores and to O)
        for (int it = threadIdx.x; it < 128 * 4; it += blockDim.x) {
            const int r = it >> 2, c = it & 3;
            uint32_t ob[16];
            if (r < valid_rows) {
                const uint4 w = *reinterpret_cast<const uint4*>(raw + r * 64 + c * 16);
                float sc_lo, sc_hi;
                if (nv) {
                    const uint32_t b2 = *reinterpret_cast<const uint16_t*>(raw + kNvScaleOff + r * 8 + 2 * c);
                    const float2 f = f16x2_to_f32x2(e4m3x2_to_f16x2(b2));
                    sc_lo = f.x;
                    sc_hi = f.y;
                } else {
                    sc_lo = sc_hi = e8m0_to_f32(raw[kMxScaleOff + r * 4 + c]);
                }
                const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float sc = i < 2 ? sc_lo : sc_hi;
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
}

// Shared memory of the attention: bf16 K and V tiles (64 KB, also the half-exchange buffer),
// the FP8-KV row scales, two stages of raw (K, V) pages, and the stages' barriers.
struct AttendSmem {
    uint8_t* Ks;
    uint8_t* Vs;
    float* xch;
    float* kscale;
    float* vscale;
    uint8_t* raw;
    uint64_t* mbar;       // [2]
    int* stage_page;      // [2]
};

__device__ __forceinline__ AttendSmem attend_smem(uint8_t* base, int page_bytes, uint64_t* mbar, int* stage_page) {
    AttendSmem sm;
    sm.Ks = base;
    sm.Vs = base + 32768;
    sm.xch = reinterpret_cast<float*>(base);
    sm.kscale = reinterpret_cast<float*>(base + kAttnRegionBytes);
    sm.vscale = reinterpret_cast<float*>(base + kAttnRegionBytes + 512);
    sm.raw = base + kAttnRegionBytes + 1024;
    sm.mbar = mbar;
    sm.stage_page = stage_page;
    (void)page_bytes;
    return sm;
}

// Dynamic shared bytes of the attention (tiles, scales, two stages of K and V pages).
__host__ __device__ constexpr size_t attend_smem_bytes(int page_bytes) {
    return (size_t)kAttnRegionBytes + 1024 + 4 * (size_t)page_bytes;
}

// This lane's place in the attention of one (row, KV head, row group). Warps at or past
// 2 x row_warps take no rows (they still widen pages and pass every barrier).
struct AttendLane {
    int lane, g, t, wr, th;
    int m0, m1, t0, t1;
    bool v0, v1, active;
};

__device__ __forceinline__ AttendLane attend_lane(int rg, int rows_per_cta, int row_warps, int M, int G) {
    AttendLane L;
    const int warp = threadIdx.x >> 5;
    L.lane = threadIdx.x & 31;
    L.g = L.lane >> 2;
    L.t = L.lane & 3;
    L.wr = warp % row_warps;
    L.th = warp / row_warps;
    L.m0 = rg * rows_per_cta + L.wr * 16 + L.g;
    L.m1 = L.m0 + 8;
    L.v0 = L.th < 2 && L.m0 < M;
    L.v1 = L.th < 2 && L.m1 < M;
    L.t0 = L.v0 ? L.m0 / G : 0;
    L.t1 = L.v1 ? L.m1 / G : 0;
    L.active = L.th < 2 && rg * rows_per_cta + L.wr * 16 < M;
    return L;
}

// q A fragments (bf16, exact) for 8 k-steps from bf16 q [B][Q][Hq][128]: a0/a2 row m0, a1/a3
// row m1; lane (g, t) holds dims 16 ks + 8 h + 2t, +1. Padding rows read row 0 (their scores are
// masked and their outputs never written). CG: read through L2 (data written by other CTAs of
// the running grid).
template <bool CG>
__device__ __forceinline__ void load_qa_bf16(uint32_t (&qa)[8][4], const uint16_t* q, const AttendLane& L, int b, int kvh,
                                             int Q, int Hq, int G) {
    const int mc0 = L.v0 ? L.m0 : 0, mc1 = L.v1 ? L.m1 : 0;
    const int64_t base0 = (((int64_t)b * Q + mc0 / G) * Hq + kvh * G + mc0 % G) * kD + 2 * L.t;
    const int64_t base1 = (((int64_t)b * Q + mc1 / G) * Hq + kvh * G + mc1 % G) * kD + 2 * L.t;
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        if (CG) {
            qa[k >> 1][(k & 1) * 2 + 0] = ldg_cg_u32(q + base0 + 8 * k);
            qa[k >> 1][(k & 1) * 2 + 1] = ldg_cg_u32(q + base1 + 8 * k);
        } else {
            qa[k >> 1][(k & 1) * 2 + 0] = *reinterpret_cast<const uint32_t*>(q + base0 + 8 * k);
            qa[k >> 1][(k & 1) * 2 + 1] = *reinterpret_cast<const uint32_t*>(q + base1 + 8 * k);
        }
    }
}

// q A fragments from f32 q [B][Q][Hq][128], packed to saturating e4m3 with the q packing rule and
// widened to bf16 (exact); same lane layout as load_qa_bf16.
__device__ __forceinline__ void load_qa_f32_e4m3(uint32_t (&qa)[8][4], const float* q, const AttendLane& L, int b, int kvh,
                                                 int Q, int Hq, int G) {
    const int mc0 = L.v0 ? L.m0 : 0, mc1 = L.v1 ? L.m1 : 0;
    const int64_t base0 = (((int64_t)b * Q + mc0 / G) * Hq + kvh * G + mc0 % G) * kD + 2 * L.t;
    const int64_t base1 = (((int64_t)b * Q + mc1 / G) * Hq + kvh * G + mc1 % G) * kD + 2 * L.t;
    float2 f0[16], f1[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        f0[k] = *reinterpret_cast<const float2*>(q + base0 + 8 * k);
        f1[k] = *reinterpret_cast<const float2*>(q + base1 + 8 * k);
    }
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        const float2 g0 = f16x2_to_f32x2(e4m3x2_to_f16x2(pack_q2(f0[k].x, f0[k].y)));
        const float2 g1 = f16x2_to_f32x2(e4m3x2_to_f16x2(pack_q2(f1[k].x, f1[k].y)));
        qa[k >> 1][(k & 1) * 2 + 0] = f32x2_to_bf16x2(g0.x, g0.y);
        qa[k >> 1][(k & 1) * 2 + 1] = f32x2_to_bf16x2(g1.x, g1.y);
    }
}

// q A fragments from rows staged in shared memory: q_s holds query rows [m_lo, ...) of the unit,
// f32 (MXFP4 K/V, packed here to e4m3 and widened to bf16) or bf16 bits (RS), 512 or 256 bytes
// per row; same lane layout as load_qa_bf16.
template <bool RS>
__device__ __forceinline__ void load_qa_staged(uint32_t (&qa)[8][4], const uint8_t* q_s, int m_lo, const AttendLane& L) {
    const int lr0 = L.v0 ? L.m0 - m_lo : 0, lr1 = L.v1 ? L.m1 - m_lo : 0;
    if (RS) {
        const uint16_t* r0 = reinterpret_cast<const uint16_t*>(q_s + lr0 * 256) + 2 * L.t;
        const uint16_t* r1 = reinterpret_cast<const uint16_t*>(q_s + lr1 * 256) + 2 * L.t;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            qa[k >> 1][(k & 1) * 2 + 0] = *reinterpret_cast<const uint32_t*>(r0 + 8 * k);
            qa[k >> 1][(k & 1) * 2 + 1] = *reinterpret_cast<const uint32_t*>(r1 + 8 * k);
        }
    } else {
        const float* r0 = reinterpret_cast<const float*>(q_s + lr0 * 512) + 2 * L.t;
        const float* r1 = reinterpret_cast<const float*>(q_s + lr1 * 512) + 2 * L.t;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            const float2 f0 = *reinterpret_cast<const float2*>(r0 + 8 * k);
            const float2 f1 = *reinterpret_cast<const float2*>(r1 + 8 * k);
            const float2 g0 = f16x2_to_f32x2(e4m3x2_to_f16x2(pack_q2(f0.x, f0.y)));
            const float2 g1 = f16x2_to_f32x2(e4m3x2_to_f16x2(pack_q2(f1.x, f1.y)));
            qa[k >> 1][(k & 1) * 2 + 0] = f32x2_to_bf16x2(g0.x, g0.y);
            qa[k >> 1][(k & 1) * 2 + 1] = f32x2_to_bf16x2(g1.x, g1.y);
        }
    }
}

// Rewrite `rows` query rows staged at q_s (f32 rows of 512 B for MXFP4 K/V, packed here to e4m3
// with the q packing rule; bf16 rows of 256 B for RS) in place as bf16 rows of 256 B in the
// swizzled tile layout (swz), zero-filling rows up to 64. Every thread calls it (two barriers).
template <bool RS>
__device__ __forceinline__ void pack_staged_q(uint8_t* q_s, int rows) {
    const int tid = threadIdx.x, nthr = blockDim.x;
    // each 64-byte piece of bf16 output = 4 chunks: piece p = (row p / 4, chunks 4 (p % 4) .. + 3)
    constexpr int kPieces = 64 * 4;
    uint32_t w[16];
    const int p = tid;   // one piece per thread (blockDim is 256)
    const int r = p >> 2, c0 = (p & 3) * 4;
    if (p < kPieces) {
        if (r < rows) {
            if (RS) {
                const uint4* src = reinterpret_cast<const uint4*>(q_s + r * 256 + c0 * 16);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const uint4 v = src[k];
                    w[4 * k] = v.x; w[4 * k + 1] = v.y; w[4 * k + 2] = v.z; w[4 * k + 3] = v.w;
                }
            } else {
                const float4* src = reinterpret_cast<const float4*>(q_s + r * 512 + c0 * 32);
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const float4 f = src[k];
                    const float2 g0 = f16x2_to_f32x2(e4m3x2_to_f16x2(pack_q2(f.x, f.y)));
                    const float2 g1 = f16x2_to_f32x2(e4m3x2_to_f16x2(pack_q2(f.z, f.w)));
                    w[2 * k] = f32x2_to_bf16x2(g0.x, g0.y);
                    w[2 * k + 1] = f32x2_to_bf16x2(g1.x, g1.y);
                }
            }
        } else {
#pragma unroll
            for (int k = 0; k < 16; ++k) w[k] = 0;
        }
    }
    (void)nthr;
    __syncthreads();   // every staged row read
    if (p < kPieces) {
#pragma unroll
        for (int k = 0; k < 4; ++k)
            *reinterpret_cast<uint4*>(q_s + swz(r, c0 + k)) = make_uint4(w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
    }
    __syncthreads();
}

// q A fragments by ldmatrix from the packed, swizzled rows of pack_staged_q (row m - m_lo).
__device__ __forceinline__ void load_qa_packed(uint32_t (&qa)[8][4], const uint8_t* q_s, int m_lo, const AttendLane& L) {
    // lanes 0-7: rows r0..r0+7 of chunk 2 ks, 8-15: rows r0+8.., 16-23: chunk 2 ks + 1, rows r0..; 24-31
    const int lane = L.lane;
    const int rb = L.active ? L.m0 - L.g - m_lo : 0;   // first row of this warp's 16
    const int row = rb + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks)
        ldmatrix_x4(qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], q_s + swz(row, 2 * ks + (lane >> 4)));
}

// Stage page i of a partition's list (logical id p, physical id phys; phys < 0: nothing to copy)
// into stage (gp + i) & 1: one thread issues the K and V bulk copies, completing on that stage's
// barrier.
__device__ __forceinline__ void attend_issue(const AttendSmem& sm, int i, int p, int64_t phys, uint32_t gp,
                                             const uint8_t* k_pool, const uint8_t* v_pool, int Hkv, int kvh,
                                             int page_bytes) {
    const int st = (int)((gp + i) & 1);
    if (phys < 0) {
        sm.stage_page[st] = -1;
        mbar_arrive(&sm.mbar[st]);
        return;
    }
    sm.stage_page[st] = p;
    const int64_t off = (phys * Hkv + kvh) * (int64_t)page_bytes;
    mbar_arrive_expect_tx(&sm.mbar[st], 2u * page_bytes);
    bulk_g2s(sm.raw + st * 2 * page_bytes, k_pool + off, page_bytes, &sm.mbar[st]);
    bulk_g2s(sm.raw + st * 2 * page_bytes + page_bytes, v_pool + off, page_bytes, &sm.mbar[st]);
}

// Attention of this CTA's rows over np selected pages: sel[i] logical page ids and selph[i]
// physical ids (-1: skip) in shared memory. The caller initialised sm.mbar[0..1] (count 1) once;
// gp counts the pages this CTA has staged so far (it sets each stage's phase parity) and is
// advanced by np. first_issued: the caller's thread 0 already issued pages 0 and 1 (attend_issue).
// Accumulates into (o, mrow, l) (per lane, l not yet reduced over the quad). Returns false if a
// copy did not land within the bounded wait (status gets SMX_DEV_TIMEOUT); the CTA must then
// issue no more copies.
template <bool RS>
__device__ __forceinline__ bool attend_pages(const AttendSmem& sm, const int* sel, const int* selph, int np,
                                             const uint8_t* k_pool, const uint8_t* v_pool, int Hkv, int kvh,
                                             int page_bytes, int ctx, const uint32_t (&qa)[8][4], const AttendLane& L,
                                             int pos0, int pos1, uint32_t& gp, float (&o)[16][4], float& mrow0,
                                             float& mrow1, float& l0, float& l1, int32_t* status, bool first_issued,
                                             float qk_scale = kLog2eOverSqrtD, bool nv = false) {
    const int lane = L.lane, t = L.t, th = L.th;
    auto issue = [&](int i) { attend_issue(sm, i, sel[i], selph[i], gp, k_pool, v_pool, Hkv, kvh, page_bytes); };
    if (threadIdx.x == 0 && !first_issued)
        for (int i = 0; i < 2 && i < np; ++i) issue(i);

    bool ok_all = true;
#pragma unroll 1
    for (int i = 0; i < np; ++i) {
        const int st = (int)((gp + i) & 1);
        const uint32_t parity = (uint32_t)(((gp + i) >> 1) & 1);
        const bool ok = mbar_wait_bounded(&sm.mbar[st], parity);
        if (__syncthreads_or(!ok)) {
            // give the copies still in flight a bounded chance to land before going on
            if (threadIdx.x == 0) {
                flag_status(status, SMX_DEV_TIMEOUT);
                mbar_wait_bounded(&sm.mbar[st], parity);
                if (i + 1 < np) mbar_wait_bounded(&sm.mbar[st ^ 1], (uint32_t)(((gp + i + 1) >> 1) & 1));
            }
            __syncthreads();
            ok_all = false;
            break;
        }
        const int p = sm.stage_page[st];
        const int valid_rows = p >= 0 ? min(kPage, ctx - p * kPage) : 0;
        if (p >= 0) {
            const uint8_t* rk = sm.raw + st * 2 * page_bytes;
            widen_page<RS>(rk, valid_rows, sm.Ks, sm.kscale, nv);
            widen_page<RS>(rk + page_bytes, valid_rows, sm.Vs, sm.vscale, nv);
        }
        __syncthreads();   // tiles ready; this stage's raw bytes are consumed
        if (threadIdx.x == 0 && i + 2 < np) {
            fence_proxy_async_smem();
            issue(i + 2);
        }
        // this warp's half of the page in 16-token units: QK, online softmax, one PV k-step
        const int units = (p >= 0 && L.active) ? max(0, min(4, (valid_rows - th * 64 + 15) / 16)) : 0;
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
                ldmatrix_x4(b0, b1, b2, b3, sm.Ks + swz(tok0 + (lane & 7), 2 * ks + (lane >> 3)));
                ldmatrix_x4(c0, c1, c2, c3, sm.Ks + swz(tok0 + 8 + (lane & 7), 2 * ks + (lane >> 3)));
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
                    float z = sc[nb][c] * qk_scale;
                    if (RS) z *= sm.kscale[tok];
                    const bool ok2 = (c < 2) ? (L.v0 && j <= pos0) : (L.v1 && j <= pos1);
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
            // weights as a bf16 high part plus a bf16 low part (~16 significant bits: bf16 alone
            // moves outputs near zero by up to ~2^-9 |v_i - v_j| when a few tokens share the
            // mass, the size of the output bound); l (per lane, reduced at the end) sums them
            uint32_t ph[2][2], pl[2][2];
#pragma unroll
            for (int nb = 0; nb < 2; ++nb) {
                float e[4];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const float mn = (c < 2) ? mrow0 : mrow1;
                    e[c] = (mn == -INFINITY) ? 0.0f : exp2f(sc[nb][c] - mn);
                }
                l0 += e[0] + e[1];
                l1 += e[2] + e[3];
                if (RS) {
                    const int tok = tok0 + nb * 8 + 2 * t;
                    const float s0 = sm.vscale[tok], s1 = sm.vscale[tok + 1];
                    e[0] *= s0; e[1] *= s1; e[2] *= s0; e[3] *= s1;
                }
                const __nv_bfloat162 h01 = __floats2bfloat162_rn(e[0], e[1]), h23 = __floats2bfloat162_rn(e[2], e[3]);
                const float2 r01 = __bfloat1622float2(h01), r23 = __bfloat1622float2(h23);
                ph[nb][0] = *reinterpret_cast<const uint32_t*>(&h01);
                ph[nb][1] = *reinterpret_cast<const uint32_t*>(&h23);
                const __nv_bfloat162 l01 = __floats2bfloat162_rn(e[0] - r01.x, e[1] - r01.y);
                const __nv_bfloat162 l23 = __floats2bfloat162_rn(e[2] - r23.x, e[3] - r23.y);
                pl[nb][0] = *reinterpret_cast<const uint32_t*>(&l01);
                pl[nb][1] = *reinterpret_cast<const uint32_t*>(&l23);
            }
            // O += P V for these 16 tokens
#pragma unroll
            for (int db = 0; db < 16; db += 2) {
                uint32_t b0, b1, b2, b3;
                ldmatrix_x4_trans(b0, b1, b2, b3, sm.Vs + swz(tok0 + ((lane >> 3) & 1) * 8 + (lane & 7), db + (lane >> 4)));
                mma_bf16_16816(o[db], ph[0][0], ph[0][1], ph[1][0], ph[1][1], b0, b1);
                mma_bf16_16816(o[db + 1], ph[0][0], ph[0][1], ph[1][0], ph[1][1], b2, b3);
                mma_bf16_16816(o[db], pl[0][0], pl[0][1], pl[1][0], pl[1][1], b0, b1);
                mma_bf16_16816(o[db + 1], pl[0][0], pl[0][1], pl[1][0], pl[1][1], b2, b3);
            }
        }
        __syncthreads();   // before the next page overwrites the tiles
    }
    gp += (uint32_t)np;
    return ok_all;
}

// Reduce l over the quad, combine the two token halves (half 1 hands (m, l, O) to half 0
// through sm.xch), and write the partials of this CTA's real rows for partition s:
// part_o [B][S][Q][Hq][128], part_m / part_l [B][S][Q][Hq]. Every thread calls it (barriers).
__device__ __forceinline__ void finish_partials(const AttendSmem& sm, const AttendLane& L, float (&o)[16][4], float mrow0,
                                                float mrow1, float l0, float l1, float* part_o, float* part_m,
                                                float* part_l, int b, int s, int kvh, int S, int Q, int Hq, int G,
                                                float o_scale = 1.0f) {
    const int lane = L.lane, t = L.t;
    l0 += __shfl_xor_sync(0xFFFFFFFFu, l0, 1);
    l0 += __shfl_xor_sync(0xFFFFFFFFu, l0, 2);
    l1 += __shfl_xor_sync(0xFFFFFFFFu, l1, 1);
    l1 += __shfl_xor_sync(0xFFFFFFFFu, l1, 2);
    __syncthreads();
    // per row group: 17 float4 per lane (16 of O, then m0, m1, l0, l1), lane-contiguous
    float4* slot = reinterpret_cast<float4*>(sm.xch) + L.wr * (17 * 32) + lane;
    if (L.th == 1) {
#pragma unroll
        for (int db = 0; db < 16; ++db) slot[db * 32] = make_float4(o[db][0], o[db][1], o[db][2], o[db][3]);
        slot[16 * 32] = make_float4(mrow0, mrow1, l0, l1);
    }
    __syncthreads();
    if (L.th == 0) {
        const float4 ml = slot[16 * 32];
        const float mo0 = ml.x, mo1 = ml.y, lo0 = ml.z, lo1 = ml.w;
        const float n0 = fmaxf(mrow0, mo0), n1 = fmaxf(mrow1, mo1);
        const float wa0 = n0 == -INFINITY ? 0.0f : exp2f(mrow0 - n0), wb0 = n0 == -INFINITY ? 0.0f : exp2f(mo0 - n0);
        const float wa1 = n1 == -INFINITY ? 0.0f : exp2f(mrow1 - n1), wb1 = n1 == -INFINITY ? 0.0f : exp2f(mo1 - n1);
#pragma unroll
        for (int db = 0; db < 16; ++db) {
            const float4 ot = slot[db * 32];
            o[db][0] = o[db][0] * wa0 + ot.x * wb0;
            o[db][1] = o[db][1] * wa0 + ot.y * wb0;
            o[db][2] = o[db][2] * wa1 + ot.z * wb1;
            o[db][3] = o[db][3] * wa1 + ot.w * wb1;
        }
        l0 = l0 * wa0 + lo0 * wb0;
        l1 = l1 * wa1 + lo1 * wb1;
        mrow0 = n0;
        mrow1 = n1;
        if (L.v0 || L.v1) {
            const int h0 = kvh * G + L.m0 % G, h1 = kvh * G + L.m1 % G;
            const int64_t r0 = (((int64_t)b * S + s) * Q + L.t0) * Hq + h0;
            const int64_t r1 = (((int64_t)b * S + s) * Q + L.t1) * Hq + h1;
#pragma unroll
            for (int db = 0; db < 16; ++db) {
                const int d = db * 8 + 2 * t;
                if (L.v0) *reinterpret_cast<float2*>(part_o + r0 * kD + d) = make_float2(o[db][0] * o_scale, o[db][1] * o_scale);
                if (L.v1) *reinterpret_cast<float2*>(part_o + r1 * kD + d) = make_float2(o[db][2] * o_scale, o[db][3] * o_scale);
            }
            if (t == 0) {
                if (L.v0) { part_m[r0] = mrow0; part_l[r0] = l0; }
                if (L.v1) { part_m[r1] = mrow1; part_l[r1] = l1; }
            }
        }
    }
}

// One output row from S partitions: out = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s with
// M = max_s m_s (zero when every partition is empty). One warp; lane l owns dims 4l..4l+3 and
// reads 16 partitions per pass with every load of the pass in flight. pi0 = index of the row's
// partition-0 entry in part_m / part_l; partition s is at pi0 + s * stride. CG: read through L2.
template <bool CG>
__device__ __forceinline__ void merge_row(const float* part_o, const float* part_m, const float* part_l, int64_t pi0,
                                          int64_t stride, int S, float* out_row) {
    const int lane = threadIdx.x & 31;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float M = -INFINITY, L = 0.0f;
    for (int s0 = 0; s0 < S; s0 += 16) {
        const int n = min(16, S - s0);
        const int sl = s0 + (lane & 15);
        float m = -INFINITY, lv = 0.0f;
        if ((lane & 15) < n) {
            const int64_t pi = pi0 + sl * stride;
            m = CG ? ldg_cg_f32(part_m + pi) : part_m[pi];
            lv = CG ? ldg_cg_f32(part_l + pi) : part_l[pi];
        }
        float4 v[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            v[k] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (k < n) {
                const float* src = part_o + (pi0 + (s0 + k) * stride) * kD + 4 * lane;
                if (CG) {
                    const uint4 u = ldg_cg_v4(src);
                    v[k] = make_float4(__uint_as_float(u.x), __uint_as_float(u.y), __uint_as_float(u.z), __uint_as_float(u.w));
                } else {
                    v[k] = *reinterpret_cast<const float4*>(src);
                }
            }
        }
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
        if (L == 0.0f) {
            // a partition with a maximum but no weight is never written by a completed split stage
            // (its largest weight is 1); it can be read only after a wait gave up: write zeros
            acc = make_float4(0.f, 0.f, 0.f, 0.f);
        } else {
            acc.x /= L; acc.y /= L; acc.z /= L; acc.w /= L;
        }
    }
    reinterpret_cast<float4*>(out_row)[lane] = acc;
}

}  // namespace smx

// smx_scan.cuh -- the index scan (a3) as a tensor-map-fed pipeline on the fifth-generation tensor
// cores: every page of the MXFP4 index cache against the row's index queries, with no SIMT work
// on the fp4 keys.
//
// [ATOM-2812] "Mono decode over the MXFP4 KV and index caches", commit "--index-cache-dtype
// mxfp4": every page of the row is scored; S_p = max over its tokens j and the draft queries t
// (j <= pos_t) of q_idx[t] . k_idx[j], the keys being E2M1 codes times the E8M0 scale of their
// 32-element group; the scorer reads a 16 B key load plus a dword of scales per tile.
//
// Per page:
//  * ONE tensor-map copy (cp.async.bulk.tensor, data type 16U4_ALIGN16B, 128-byte swizzle) takes
//    the whole 8704-byte page as 136 rows of 64 bytes: rows 0..127 are the tokens' packed nibbles,
//    rows 128..135 the tokens' E8M0 scale words (16 tokens a row). Shared memory receives each
//    16-element chunk as its 8 bytes followed by an 8-byte gap: rows 0..127 form the K-major
//    [128 tokens][128] fp4 operand the MMA reads, and token t's scale word sits in row 128 + t/16.
//    The copy counts the 8704 bytes it reads.
//  * An MMA-issuing warp copies the page's 128 scale words into a small ring (the tile is then the
//    MMA's alone) and its lane 0 issues four tcgen05.mma kind::f8f6f4 (A = the page's E2M1 codes,
//    M = 128 tokens; B = the query pieces in e4m3, N = 2 NQ; K = 32 = one scale group each) into
//    four fp32 accumulators in tensor memory, unscaled.
//  * The epilogue (thread = token) weighs group g's accumulator by 2^(e_g - 127 - sigma_g), adds
//    the two query pieces, masks by the causal rule and takes the max over queries, then over the
//    page's tokens. A NaN group scale (0xFF) makes the token's score NaN, which the max leaves out.
// The queries (scan_setup_query): each bf16 element times 2^sigma_g (the group's largest
// magnitude in (224, 448]) split exactly into two e4m3 pieces (rows n and NQ + n): exact for every
// element within 2^9.8 of its group's maximum (e4m3 keeps 4 significant bits per piece), a
// smaller one off by at most half the e4m3 subnormal step, 2^-17.8 of the group maximum. The
// products are exact; only the MMA's and the epilogue's fp32 additions round.
// Roles (8 warps): lane 0 of warps 0 and 3 issue the copies of the even and the odd pages (one
// thread issues at most one copy per ~600 cycles: two issuers reach the copy engines' rate);
// warps 1 and 2 take the MMAs of the even and the odd pages (the scale copy by the whole warp, the
// MMA issue by lane 0, which an issue holds about a hundred cycles); warps 4-7 first run the
// query set-up and the caller's work (the fused step writes the new rows there: they would idle
// until the first accumulator anyway), then take the epilogue (warp 4 + q reaches tensor-memory lanes 32 q ..), two
// pages an iteration. Nothing waits on the epilogue but the reuse of an accumulator stage, so the
// copies and the MMAs run as the data lands. Every wait is bounded; once one gives up the CTA's
// later waits return at once and SMX_DEV_TIMEOUT is set.
#pragma once

#include <cuda.h>

#include "smx_device.cuh"
#include "smx_tc.cuh"

namespace smx {

// The query pieces of NQ query slots: rows [0, NQ) the high pieces, [NQ, 2 NQ) the low pieces,
// [2 NQ, 3 NQ) zero (so that rows [NQ, 3 NQ) are a second N = 2 NQ operand whose first NQ rows are
// the low pieces); at least 32 rows.
__host__ __device__ constexpr int scan_query_bytes(int nq) { return (3 * nq > 32 ? 3 * nq : 32) * 128; }

// Byte offset of 16-byte chunk c of row r of a K-major tile with the 128-byte swizzle (8-row atoms
// of 1024 bytes).
__host__ __device__ __forceinline__ uint32_t sc_chunk(int r, int c) {
    return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + (((c ^ r) & 7) << 4));
}

__device__ __forceinline__ float2 e4m3x2_to_f32x2(uint32_t w16) { return f16x2_to_f32x2(e4m3x2_to_f16x2(w16)); }

constexpr int kScanRows = 136;                    // one page as rows of 64 bytes
constexpr int kScanTileBytes = kScanRows * 128;   // unpacked: 128 bytes a row (17 x 1 KB)
constexpr uint32_t kScanTxBytes = kMxPageBytes;   // completion bytes of one page's copy
constexpr int kScanRedPages = 32;                 // page maxima combined per flush
constexpr int kScanScaleBytes = 512;              // one page's scale words in the ring
// Accumulator stages of a scan with NQ query slots in `cols` tensor-memory columns (four groups x
// 2 NQ columns a stage).
__host__ __device__ constexpr int scan_acc_stages(int nq, int cols) { return cols / (8 * nq); }

// Shared-memory bytes of a scan of NQ query slots with `stages` page stages (then the query
// pieces and the scale ring of `sa` pages), from a 1024-byte-aligned base.
__host__ __device__ constexpr int scan_smem_bytes(int stages, int sa, int nq) {
    return stages * kScanTileBytes + scan_query_bytes(nq) + sa * kScanScaleBytes;
}

struct ScanPipe {
    uint8_t* tiles;       // [ST][kScanTileBytes], 1024-byte aligned
    uint8_t* qt;          // the query pieces (scan_setup_query), 1024-byte aligned
    uint8_t* ring;        // [SA][kScanScaleBytes]: the scale words of the page in accumulator stage a
    uint64_t* full;       // [ST] page copy landed (1 arrival + transaction bytes)
    uint64_t* empty;      // [ST] stage free: the page's MMAs are done (commit)
    uint64_t* afull;      // [SA] accumulators written (commit) and the ring slot filled (1 arrival)
    uint64_t* aempty;     // [SA] accumulators and ring slot read (4 epilogue warps)
    uint64_t* ins;        // the caller's new index rows are written (insert_arrivals arrivals)
    uint64_t* qready;     // the query pieces are in qt (4 arrivals: the epilogue warps)
    float* red;           // [kScanRedPages][4] warp maxima (as order-preserving keys)
    float* gmax;          // [4][4] per-warp group maxima of the query set-up (shared)
    int* gave_up;         // shared flag
    uint32_t tmem;        // base column of the scan's tensor memory
    uint32_t seq;         // pages this CTA has scanned so far (sets every barrier's phase)
    uint32_t ins_seq;     // insert hand-offs so far (the parity of `ins`)
    uint32_t q_seq;       // query set-ups so far (the parity of `qready`)
};

// Barriers a ScanPipe needs: 2 ST + 2 SA + 2.
__host__ __device__ constexpr int scan_barriers(int st, int sa) { return 2 * st + 2 * sa + 2; }

// Points the pipe's barriers into bars[scan_barriers(ST, SA)].
template <int ST, int SA>
__device__ __forceinline__ void scan_bind(ScanPipe& sp, uint64_t* bars) {
    sp.full = bars;
    sp.empty = bars + ST;
    sp.afull = bars + 2 * ST;
    sp.aempty = sp.afull + SA;
    sp.ins = sp.aempty + SA;
    sp.qready = sp.ins + 1;
}

// One warp: the barriers, one per lane (before the first use, behind a block barrier).
template <int ST, int SA>
__device__ __forceinline__ void scan_init_warp(ScanPipe& sp, uint32_t insert_arrivals, int lane) {
    constexpr int kN = 2 * ST + 2 * SA + 2;
    for (int j = lane; j < kN; j += 32) {
        if (j < ST) mbar_init(&sp.full[j], 1);
        else if (j < 2 * ST) mbar_init(&sp.empty[j - ST], 1);
        else if (j < 2 * ST + SA) mbar_init(&sp.afull[j - 2 * ST], 2);
        else if (j < 2 * ST + 2 * SA) mbar_init(&sp.aempty[j - 2 * ST - SA], 4);
        else if (j == 2 * ST + 2 * SA) mbar_init(sp.ins, insert_arrivals);
        else mbar_init(sp.qready, 4);
    }
    if (lane == 0) *sp.gave_up = 0;
    mbar_fence_init();
}

// One thread: the barriers (before the first use, behind a block barrier).
template <int ST, int SA>
__device__ __forceinline__ void scan_init(ScanPipe& sp, uint32_t insert_arrivals) {
#pragma unroll
    for (int s = 0; s < ST; ++s) {
        mbar_init(&sp.full[s], 1);
        mbar_init(&sp.empty[s], 1);
    }
#pragma unroll
    for (int s = 0; s < SA; ++s) {
        mbar_init(&sp.afull[s], 2);
        mbar_init(&sp.aempty[s], 4);
    }
    mbar_init(sp.ins, insert_arrivals);
    mbar_init(sp.qready, 4);
    *sp.gave_up = 0;
    mbar_fence_init();
}

__device__ __forceinline__ bool scan_wait(const ScanPipe& sp, uint64_t* bar, uint32_t parity, int32_t* status) {
    if (*(volatile int*)sp.gave_up) return false;
    if (mbar_wait_spin(bar, parity)) return true;
    *(volatile int*)sp.gave_up = 1;
    flag_status(status, SMX_DEV_TIMEOUT);
    return false;
}

// L2 policy for the index pages: each is read once a step, so evict it first.
__device__ __forceinline__ uint64_t scan_l2_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// The whole page `phys` (tensor map over the index pool: [pages][136 rows][128 fp4]) into `dst`,
// completing on bar, with L2 policy pol.
__device__ __forceinline__ void scan_tma_page(void* dst, const CUtensorMap* map, int phys, uint64_t* bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;"
        ::"r"(smem_u32(dst)), "l"(map), "r"(0), "r"(0), "r"(phys), "r"(smem_u32(bar)), "l"(pol)
        : "memory");
}

// kind::f8f6f4 instruction descriptor: fp32 D, A E2M1, B E4M3 (both K-major), M = 128, N.
__host__ __device__ constexpr uint32_t idesc_scan(int N) {
    return (1u << 4) | (5u << 7) | (0u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}

// NQ consecutive fp32 columns of this thread's lane (no wait).
template <int NQ>
__device__ __forceinline__ void scan_ld(uint32_t taddr, uint32_t (&r)[NQ]) {
    if constexpr (NQ == 8) {
        asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                     : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                     : "r"(taddr)
                     : "memory");
    } else {
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
            : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
              "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
            : "r"(taddr)
            : "memory");
    }
}

// A token's score for one page from its scale word and its four group accumulators (group g at
// columns taddr + 2 NQ g; column n holds D_g[n], the high and the low query piece of query n
// summed by the two MMAs): with x_g = e_g - sigma_g and X = max_g x_g,
// t_n = sum_g 2^(x_g - X) D_g[n] (weights exact powers of two, at most 1; a group more than 2^126
// below the largest is dropped) and the score is the max over queries n < Q with j <= lim + n of
// t_n, times 2^(X - 127): -inf if no query counts, NaN if a group scale is NaN. One wait for the
// four groups' loads.
template <int NQ>
__device__ __forceinline__ float scan_token_score(uint32_t taddr, uint32_t sw, const int (&sig)[4], int j, int lim,
                                                  int Q) {
    uint32_t r[4][NQ];
#pragma unroll
    for (int g = 0; g < 4; ++g) scan_ld<NQ>(taddr + (uint32_t)(g * 2 * NQ), r[g]);
    int x[4];
    int X = -1000;
    bool nan = false;
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        const int e = (int)((sw >> (8 * g)) & 0xFFu);
        nan |= e == 0xFF;
        x[g] = e - sig[g];
        X = max(X, x[g]);
    }
    float f[4];
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        const int d = x[g] - X;   // <= 0
        f[g] = d >= -126 ? __uint_as_float((uint32_t)(d + 127) << 23) : 0.0f;
    }
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
    float t[NQ];
#pragma unroll
    for (int n = 0; n < NQ; ++n) {
        t[n] = f[0] * __uint_as_float(r[0][n]);
#pragma unroll
        for (int g = 1; g < 4; ++g) t[n] = fmaf(f[g], __uint_as_float(r[g][n]), t[n]);
    }
    float best = -INFINITY;
#pragma unroll
    for (int n = 0; n < NQ; ++n) {
        const bool ok = n < Q && j <= lim + n;
        best = ok ? fmaxf(best, t[n]) : best;
    }
    if (nan) return __uint_as_float(0x7FC00000u);
    return best == -INFINITY ? best : mul_exp2(best, X - 127);
}

// Order-preserving u32 key of a float (NaN lowest) and back, for one-instruction warp maxima.
__device__ __forceinline__ uint32_t scan_key(float v) {
    if (v != v) return 0u;
    const uint32_t u = __float_as_uint(v);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float scan_unkey(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}
__device__ __forceinline__ uint32_t warp_max_u32(uint32_t v) {
    uint32_t r;
    asm volatile("redux.sync.max.u32 %0, %1, 0xffffffff;" : "=r"(r) : "r"(v));
    return r;
}

// Scores pages phys[0 .. np) (physical ids in shared memory; -1 = a bad id: flagged, scored -inf)
// of one row, logical pages p_first .., into score_row[p_first + i]. Warps 4-7 call pre() first;
// the new index rows of pages [wait_from, np) are written there: pre() arrives on sp.ins (one arrival
// per warp, after a proxy fence) and the copiers wait for those arrivals before copying those pages
// (wait_from >= np: no wait). Every thread of the 8-warp block calls it. Every thread must reach a
// block barrier after the call before the next one (or before reusing the query pieces);
// scan_finish then retires the last stages.
// The query pieces of one row (bf16 bits [Q][128], Q <= NQ) built by the 128 threads of warps 4-7
// while the first pages are in flight (per 32-dim group g a
// power-of-two scale 2^sig[g] that brings the group's largest |q| into (224, 448] where it fits;
// each scaled value as an e4m3 high piece plus an e4m3 low piece of the remainder), item
// it = t, t + 128 being query slot it / 16 and 8-dim slice it % 16. Writes the pieces to qt, makes
// them visible to the tensor cores, arrives on qready (one arrival per warp) and returns sig.
template <int NQ>
__device__ __forceinline__ void scan_setup_query(const ScanPipe& sp, const uint16_t* qrow, int Q, int (&sig)[4]) {
    const int t = (int)threadIdx.x - 128, lane = t & 31, qd = t >> 5;
    constexpr int kItems = NQ / 8;   // 16 slices per query slot over 128 threads
    float x[kItems][8];
    float m = 0.0f;
#pragma unroll
    for (int k = 0; k < kItems; ++k) {
        const int it = t + 128 * k, n = it >> 4, c8 = it & 15;
        uint2 r0 = make_uint2(0, 0), r1 = r0;
        if (n < Q) {
            const uint2* src = reinterpret_cast<const uint2*>(qrow + (int64_t)n * kD + 8 * c8);
            r0 = src[0];
            r1 = src[1];
        }
        const uint32_t w[4] = {r0.x, r0.y, r1.x, r1.y};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            x[k][2 * i] = __uint_as_float(w[i] << 16);
            x[k][2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(x[k][i]));   // (NaN ignored, as the scorer's)
    }
    // lanes of one group within the warp differ in lane bits 0, 1 (slice) and 4 (query); item k's
    // group is the same as item 0's (it differs by 128)
    m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
    m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
    m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 16));
    if ((lane & 3) == 0 && lane < 16) sp.gmax[qd * 4 + (lane >> 2)] = m;
    asm volatile("bar.sync 1, 128;" ::: "memory");
#pragma unroll
    for (int gg = 0; gg < 4; ++gg) {
        const float mx = fmaxf(fmaxf(sp.gmax[gg], sp.gmax[4 + gg]), fmaxf(sp.gmax[8 + gg], sp.gmax[12 + gg]));
        int s = 0;
        if (mx > 0.0f && mx == mx) {
            const int E = floor_log2_pos(mx);            // mx in [2^E, 2^(E+1))
            s = 7 - E;                                    // scaled max in [128, 256)
            if (mul_exp2(mx, s + 1) <= 448.0f) s += 1;   // in (224, 448] where it fits
        }
        sig[gg] = s;
    }
    const int g = (lane & 15) >> 2;
    const int s_mine = g == 0 ? sig[0] : g == 1 ? sig[1] : g == 2 ? sig[2] : sig[3];
#pragma unroll
    for (int k = 0; k < kItems; ++k) {
        const int it = t + 128 * k, n = it >> 4, c8 = it & 15;
        uint32_t b0[2] = {0, 0}, b1[2] = {0, 0};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float y0 = mul_exp2(x[k][2 * i], s_mine), y1 = mul_exp2(x[k][2 * i + 1], s_mine);
            const uint32_t q0 = e4m3x2_rn_sat(y0, y1);
            const float2 f0 = e4m3x2_to_f32x2(q0);
            const uint32_t q1 = e4m3x2_rn_sat(y0 - f0.x, y1 - f0.y);
            b0[i >> 1] |= q0 << (16 * (i & 1));
            b1[i >> 1] |= q1 << (16 * (i & 1));
        }
        *reinterpret_cast<uint2*>(sp.qt + sc_chunk(n, c8 >> 1) + 8 * (c8 & 1)) = make_uint2(b0[0], b0[1]);
        *reinterpret_cast<uint2*>(sp.qt + sc_chunk(NQ + n, c8 >> 1) + 8 * (c8 & 1)) = make_uint2(b1[0], b1[1]);
        *reinterpret_cast<uint2*>(sp.qt + sc_chunk(2 * NQ + n, c8 >> 1) + 8 * (c8 & 1)) = make_uint2(0u, 0u);
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(sp.qready);
}

template <int NQ, int ST, int SA, class Pre>
__device__ __forceinline__ void scan_pages(ScanPipe& sp, const CUtensorMap* map, const int64_t* phys, int np,
                                           int p_first, int wait_from, int lim, int Q, const uint16_t* qrow,
                                           float* score_row, int32_t* status, Pre pre) {
    constexpr int N = 2 * NQ;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t seq = sp.seq;
    if (warp == 0 || warp == 3) {
        // ---- page copies: warp 0 the even pages, warp 3 the odd ones ----
        if (lane == 0) {
            bool waited = false;
            const uint64_t pol = scan_l2_policy();
#pragma unroll 1
            for (int i = warp == 0 ? 0 : 1; i < np; i += 2) {
                const uint32_t g = seq + (uint32_t)i, st = g % ST, use = g / ST;
                if (use > 0) scan_wait(sp, &sp.empty[st], (use - 1) & 1u, status);
                if (i >= wait_from && !waited) {
                    scan_wait(sp, sp.ins, sp.ins_seq & 1u, status);
                    fence_proxy_async_global();
                    waited = true;
                }
                const int64_t ph = phys[i];
                if (ph >= 0 && !*(volatile int*)sp.gave_up) {
                    mbar_arrive_expect_tx(&sp.full[st], kScanTxBytes);
                    scan_tma_page(sp.tiles + st * kScanTileBytes, map, (int)ph, &sp.full[st], pol);
                } else {
                    mbar_arrive(&sp.full[st]);   // a bad page id: nothing to copy (scored -inf)
                }
            }
        }
        __syncwarp();
    } else if (warp == 1 || warp == 2) {
        // ---- scale copy and MMA issue: warp 1 the even pages, warp 2 the odd ones ----
        constexpr uint32_t idesc = idesc_scan(N);
        const uint32_t qt_s = smem_u32(sp.qt);
        // the query pieces (written by the epilogue warps while the first pages are in flight)
        if (np > warp - 1) scan_wait(sp, sp.qready, sp.q_seq & 1u, status);
#pragma unroll 1
        for (int i = warp - 1; i < np; i += 2) {
            const uint32_t g = seq + (uint32_t)i, st = g % ST, as = g % SA;
            // the accumulator stage and its ring slot are free (the epilogue read page g - SA)
            if (g >= (uint32_t)SA) scan_wait(sp, &sp.aempty[as], ((g / SA) - 1) & 1u, status);
            const bool ok = scan_wait(sp, &sp.full[st], (g / ST) & 1u, status);
            // tokens 4 lane .. 4 lane + 3: two 8-byte halves of the scale rows, one 16-byte store
            const uint8_t* srow = sp.tiles + st * kScanTileBytes + 128 * 128;
            {
                const int t0 = 4 * lane, r = t0 >> 4, c0 = (t0 & 15) >> 1;
                const uint2 w01 = *reinterpret_cast<const uint2*>(srow + r * 128 + (((c0 ^ r) & 7) << 4));
                const uint2 w23 = *reinterpret_cast<const uint2*>(srow + r * 128 + ((((c0 + 1) ^ r) & 7) << 4));
                *reinterpret_cast<uint4*>(sp.ring + as * kScanScaleBytes + 16 * lane) = make_uint4(w01.x, w01.y, w23.x, w23.y);
            }
            __syncwarp();
            if (lane == 0) {
                tc_fence_after_sync();
                if (ok && phys[i] >= 0 && !*(volatile int*)sp.gave_up) {
                    const uint32_t tile_s = smem_u32(sp.tiles + st * kScanTileBytes);
                    const uint32_t d = sp.tmem + as * 4 * N;
                    // per group two MMAs into one accumulator: B = query rows [0, N) (high pieces,
                    // then low), then rows [NQ, NQ + N) (low pieces, then zeros), so that column n <
                    // NQ sums both pieces of query n (columns NQ.. are not read)
#pragma unroll
                    for (int gg = 0; gg < 4; ++gg) {
                        const uint64_t ad = sw128_desc(tile_s + 32 * gg);
#pragma unroll
                        for (int pc = 0; pc < 2; ++pc) {
                            const uint64_t bd = sw128_desc(qt_s + pc * NQ * 128 + 32 * gg);
                            asm volatile("{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n"
                                         " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}" ::"r"(d + gg * N),
                                         "l"(ad), "l"(bd), "r"(idesc), "r"((uint32_t)pc)
                                         : "memory");
                        }
                    }
                }
                tc_commit(&sp.afull[as]);
                tc_commit(&sp.empty[st]);
                mbar_arrive(&sp.afull[as]);   // the ring slot is written (release)
            }
            __syncwarp();
        }
    } else if (warp >= 4) {
        int sig[4];
        scan_setup_query<NQ>(sp, qrow, Q, sig);
        pre();
        // ---- epilogue: thread = token, two pages an iteration ----
        const int qd = warp - 4, tok = 32 * qd + lane;
        const uint32_t lane_base = sp.tmem + ((uint32_t)(32 * qd) << 16);
#pragma unroll 1
        for (int i = 0; i < np; i += 2) {
            const bool two = i + 1 < np;
            const uint32_t g0 = seq + (uint32_t)i, g1 = g0 + 1u;
            scan_wait(sp, &sp.afull[g0 % SA], (g0 / SA) & 1u, status);
            if (two) scan_wait(sp, &sp.afull[g1 % SA], (g1 / SA) & 1u, status);
            tc_fence_after_sync();
            // warp-uniform (the tensor-memory loads are warp-collective)
            const bool gave = *(volatile int*)sp.gave_up != 0;
            const bool good0 = __all_sync(0xFFFFFFFFu, phys[i] >= 0 && !gave);
            const bool good1 = two && __all_sync(0xFFFFFFFFu, phys[i + 1] >= 0 && !gave);
            const uint32_t sw0 = reinterpret_cast<const uint32_t*>(sp.ring + (g0 % SA) * kScanScaleBytes)[tok];
            const uint32_t sw1 = two ? reinterpret_cast<const uint32_t*>(sp.ring + (g1 % SA) * kScanScaleBytes)[tok] : 0u;
            const int j0 = (p_first + i) * kPage + tok;
            const float s0 = good0 ? scan_token_score<NQ>(lane_base + (g0 % SA) * 4 * N, sw0, sig, j0, lim, Q) : -INFINITY;
            const float s1 = good1 ? scan_token_score<NQ>(lane_base + (g1 % SA) * 4 * N, sw1, sig, j0 + kPage, lim, Q)
                                   : -INFINITY;
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&sp.aempty[g0 % SA]);
                if (two) mbar_arrive(&sp.aempty[g1 % SA]);
            }
            // NaN tokens rank lowest
            const uint32_t k0 = warp_max_u32(scan_key(s0)), k1 = warp_max_u32(scan_key(s1));
            if (lane == 0) {
                reinterpret_cast<uint32_t*>(sp.red)[(i % kScanRedPages) * 4 + qd] = k0;
                if (two) reinterpret_cast<uint32_t*>(sp.red)[((i + 1) % kScanRedPages) * 4 + qd] = k1;
            }
            const int last = two ? i + 1 : i;
            if ((last + 1) % kScanRedPages == 0 || last + 1 == np) {
                asm volatile("bar.sync 1, 128;" ::: "memory");
                const int base = (last / kScanRedPages) * kScanRedPages, cnt = last + 1 - base;
                const int t = threadIdx.x - 128;
                if (t < cnt) {
                    const uint32_t* m = reinterpret_cast<const uint32_t*>(sp.red) + 4 * t;
                    const bool ok_page = phys[base + t] >= 0;
                    const uint32_t k = max(max(m[0], m[1]), max(m[2], m[3]));
                    // a page whose every token is NaN or masked scores -inf
                    score_row[p_first + base + t] = (ok_page && k != 0u) ? scan_unkey(k) : -INFINITY;
                    if (!ok_page) flag_status(status, SMX_DEV_BAD_PAGE_ID);
                }
                asm volatile("bar.sync 1, 128;" ::: "memory");
            }
        }
    }
    sp.seq = seq + (uint32_t)np;
    if (wait_from < np) sp.ins_seq += 1;
    sp.q_seq += 1;
}

// After the block barrier that follows the last scan_pages of a CTA (or before its barriers or
// columns are used for anything else): thread 0 waits until the last stages' MMA commits have
// arrived.
template <int ST>
__device__ __forceinline__ void scan_finish(ScanPipe& sp, int32_t* status) {
    if (threadIdx.x == 0) {
        const uint32_t end = sp.seq;
        for (uint32_t g = end > (uint32_t)ST ? end - ST : 0u; g < end; ++g)
            scan_wait(sp, &sp.empty[g % ST], (g / ST) & 1u, status);
    }
}

}  // namespace smx

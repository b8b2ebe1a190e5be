// smx_score_tc.cuh -- the index scorer (a3) on the fifth-generation tensor cores: one page of the
// MXFP4 index cache against the row's index queries, with no conversion of the fp4 keys.
//
// [ATOM-2812] "Mono decode over the MXFP4 KV and index caches", commit "--index-cache-dtype
// mxfp4": every page of the row is scored, S_p = max over its tokens and the draft queries of
// q_idx . k_idx, the keys being E2M1 codes times the E8M0 scale of their 32-element group.
//
// The MMA is tcgen05 kind::mxf8f6f4 with block scaling (one E8M0 scale per 32 elements of K):
// A = the page's E2M1 codes (M = 128 tokens, K = 128 dims), B = the queries (N = 2 NQ rows: two
// pieces of NQ = 8 or 16 query slots), one MMA per 32-dim group g (K = 32) with scale-factor id g,
// all four accumulating into one fp32 accumulator in tensor memory (lane r = token r).
//  * A in shared memory: K-major, 128-byte swizzle, each 16-element chunk of a row as its 8 bytes
//    of packed nibbles (element 2i in the low nibble of byte i) followed by 8 bytes of padding --
//    the form the MMA reads fp4 operands in. A row of the page (64 B) becomes eight such chunks.
//  * A's scale factors in tensor memory: token r's word sits in lane r of column base + r / 32,
//    byte g = the scale of group g -- the page's own scale word of the token, each byte lowered
//    by sigma_g - sigma_min (below).
//  * B: each bf16 query element x, times a power of two 2^sigma_g per group (the group's largest
//    |x| over the queries lands in (224, 448]), is split into two e4m3 pieces p0 = e4m3(x),
//    p1 = e4m3(x - p0) (round to nearest even): rows n and NQ + n. The split is exact for every
//    element of magnitude >= 1/4 after scaling, i.e. within 2^9.8 of its group's maximum (e4m3
//    keeps 4 significant bits per piece); a smaller element is off by at most half the e4m3
//    subnormal step, 2^-10, i.e. 2^-17.8 of the group maximum. B's scale factors are 2^0.
//  * So D[r][n] + D[r][NQ + n] = 2^sigma_min * q_n . k_r exactly up to the fp32 accumulation;
//    the epilogue masks by the causal rule and takes the max over n, then over the page's tokens,
//    and scales by 2^-sigma_min once per page. A NaN group scale (0xFF) makes the token's sums
//    NaN, which the max skips: such a token takes no part.
// Measured on this part: one narrow MMA costs about 17 + 3 N cycles of the tensor pipe (about 100
// with block scaling at N = 16) and holds its issuing thread for about as long, so the pieces go
// side by side in N, the groups share one accumulator (four MMAs per page), and the pipeline below
// gives the issue to a warp of its own.
#pragma once

#include <math.h>

#include "smx_device.cuh"
#include "smx_tc.cuh"

namespace smx {

constexpr int kScTileBytes = 128 * 128;     // one page as the A operand
constexpr int kScQueryBytes = 32 * 128;     // B: up to 32 rows (two pieces x 16 query slots)
constexpr int kScChunksPerThread = 4;       // 1024 8-byte chunks of a page over 256 threads
// tensor-memory columns of a scorer: accumulator stage d at 32 d (d < 3), the A scale factors of
// tile stage t at 96 + 4 t (t < 4), B's scale factors at 120
constexpr uint32_t kScColD = 0, kScColSFA = 96, kScColSFB = 120;
constexpr int kScTmemCols = 128;
constexpr int kScMaxTileStages = 4, kScMaxAccStages = 3;

// Byte offset of the 16-byte chunk c of row r of a [rows][128 B] K-major 128-byte-swizzled tile.
__host__ __device__ __forceinline__ uint32_t sc_chunk(int r, int c) {
    return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + (((c ^ r) & 7) << 4));
}

__device__ __forceinline__ float2 e4m3x2_to_f32x2(uint32_t w16) { return f16x2_to_f32x2(e4m3x2_to_f16x2(w16)); }

// The per-row query state: sigma_min and the per-group offsets sigma_g - sigma_min.
struct ScQuery {
    int sig_min;
    int rel[4];
};

// Builds the two B pieces of one row's queries (bf16 bits [Q][128], Q <= NQ) in qt (shared,
// 1024-byte aligned, kScQueryBytes) and the row's scale exponents. Every thread of the block calls
// it (threads 0..255 do the work, any others only pass the barriers); gmax is [8][4] shared
// scratch. Ends with the pieces visible to the tensor cores.
template <int NQ>
__device__ __forceinline__ ScQuery sc_setup_query(const uint16_t* qrow, int Q, uint8_t* qt, float (*gmax)[4]) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n = tid >> 4, c8 = tid & 15, g = c8 >> 2;   // query slot, 8-dim slice, its group
    uint2 r0 = make_uint2(0, 0), r1 = r0;
    if (n < Q) {
        const uint2* src = reinterpret_cast<const uint2*>(qrow + (int64_t)n * kD + 8 * c8);
        r0 = src[0];
        r1 = src[1];
    }
    const uint32_t w[4] = {r0.x, r0.y, r1.x, r1.y};
    float x[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        x[2 * i] = __uint_as_float(w[i] << 16);
        x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(x[i]));
    // lanes of one group within the warp differ in lane bits 0, 1 (slice) and 4 (query)
    m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
    m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
    m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 16));
    if ((lane & 3) == 0 && lane < 16 && warp < 8) gmax[warp][lane >> 2] = m;
    __syncthreads();
    ScQuery sq;
    int sig[4];
#pragma unroll
    for (int gg = 0; gg < 4; ++gg) {
        float mx = 0.0f;
#pragma unroll
        for (int ww = 0; ww < 8; ++ww) mx = fmaxf(mx, gmax[ww][gg]);
        int s = 0;
        if (mx > 0.0f && mx == mx) {
            const int E = floor_log2_pos(mx);            // mx in [2^E, 2^(E+1))
            s = 7 - E;                                    // scaled max in [128, 256)
            if (mul_exp2(mx, s + 1) <= 448.0f) s += 1;   // in (224, 448] where it fits
        }
        sig[gg] = s;
    }
    sq.sig_min = min(min(sig[0], sig[1]), min(sig[2], sig[3]));
#pragma unroll
    for (int gg = 0; gg < 4; ++gg) sq.rel[gg] = sig[gg] - sq.sig_min;
    const int s_mine = g == 0 ? sig[0] : g == 1 ? sig[1] : g == 2 ? sig[2] : sig[3];
    uint32_t b0[2] = {0, 0}, b1[2] = {0, 0};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float y0 = mul_exp2(x[2 * i], s_mine), y1 = mul_exp2(x[2 * i + 1], s_mine);
        const uint32_t q0 = e4m3x2_rn_sat(y0, y1);
        const float2 f0 = e4m3x2_to_f32x2(q0);
        const uint32_t q1 = e4m3x2_rn_sat(y0 - f0.x, y1 - f0.y);
        b0[i >> 1] |= q0 << (16 * (i & 1));
        b1[i >> 1] |= q1 << (16 * (i & 1));
    }
    if (n < NQ && warp < 8) {
        *reinterpret_cast<uint2*>(qt + sc_chunk(n, c8 >> 1) + 8 * (c8 & 1)) = make_uint2(b0[0], b0[1]);
        *reinterpret_cast<uint2*>(qt + sc_chunk(NQ + n, c8 >> 1) + 8 * (c8 & 1)) = make_uint2(b1[0], b1[1]);
    }
    fence_proxy_async_smem();
    __syncthreads();
    return sq;
}

// B's scale factors (2^0 everywhere): warps 0..3 fill their lane quadrant of four columns. The
// caller orders it before the first MMA (tcgen05 fences around a barrier).
__device__ __forceinline__ void sc_init_sfb(uint32_t tmem) {
    const int warp = threadIdx.x >> 5;
    if (warp < 4) {
        const uint32_t one = 0x7F7F7F7Fu;
        asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                         tmem + ((uint32_t)(32 * warp) << 16) + kScColSFB),
                     "r"(one), "r"(one), "r"(one), "r"(one)
                     : "memory");
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
    }
}

// This thread's share of one page: chunks tid + 256 i (8 bytes of nibbles each; row = chunk / 8).
// Read through L2 (rows inserted earlier in the same grid must be seen).
struct ScPage {
    uint2 w[kScChunksPerThread];
};

__device__ __forceinline__ uint2 ldg_cg_v2(const void* p) {
    uint2 r;
    asm volatile("ld.global.cg.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p) : "memory");
    return r;
}

__device__ __forceinline__ void sc_load_page(ScPage& pg, const uint8_t* page) {
#pragma unroll
    for (int i = 0; i < kScChunksPerThread; ++i) pg.w[i] = ldg_cg_v2(page + 8 * (threadIdx.x + 256 * i));
}

// Token r's scale word of a page.
__device__ __forceinline__ uint32_t sc_load_scales(const uint8_t* page, int r) {
    return ldg_cg_u32(page + kMxScaleOff + 4 * r);
}

__device__ __forceinline__ void sc_store_tile(const ScPage& pg, uint8_t* tile) {
#pragma unroll
    for (int i = 0; i < kScChunksPerThread; ++i) {
        const int ch = threadIdx.x + 256 * i, r = ch >> 3, c = ch & 7;
        *reinterpret_cast<uint4*>(tile + sc_chunk(r, c)) = make_uint4(pg.w[i].x, pg.w[i].y, 0u, 0u);
    }
}

// The calling warp's tokens' A scale factors into the four columns at sfa_col (warp w holds tokens
// 32 (w % 4) + lane; token r's word goes to column sfa_col + r / 32): byte g = e_g - (sigma_g -
// sigma_min), clamped at 0; a NaN scale (0xFF) stays NaN. Waits for the store.
__device__ __forceinline__ void sc_store_sfa(uint32_t tmem, uint32_t sfa_col, uint32_t sw, const ScQuery& sq) {
    uint32_t out = 0;
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        const int e = (int)((sw >> (8 * g)) & 0xFFu);
        const int a = e == 0xFF ? 0xFF : max(0, e - sq.rel[g]);
        out |= (uint32_t)a << (8 * g);
    }
    const int q = (threadIdx.x >> 5) & 3;
    const uint32_t addr = tmem + ((uint32_t)(32 * q) << 16) + sfa_col + q;
    asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(addr), "r"(out) : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// One thread: the 4 MMAs of one page (tile_s, shared address; A scale factors at sfa_col) against
// the query pieces (qt_s) into the accumulator columns at d_col.
template <int NQ>
__device__ __forceinline__ void sc_issue_page(uint32_t tmem, uint32_t d_col, uint32_t sfa_col, uint32_t tile_s,
                                              uint32_t qt_s) {
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        // block-scaled kind::mxf8f6f4: B scale id 0 (bits 4-5), A E2M1 (5, bits 7-9), B E4M3 (0, bits
        // 10-12), N >> 3 (bits 17-22), E8M0 scales (bit 23), M >> 4 (bits 24-28), A scale id g (bits 29-30)
        const uint32_t idesc = (5u << 7) | (0u << 10) | (((uint32_t)(2 * NQ) >> 3) << 17) | (1u << 23) |
                               ((128u >> 4) << 24) | ((uint32_t)g << 29);
        const uint64_t ad = sw128_desc(tile_s + 32 * g);
        const uint64_t bd = sw128_desc(qt_s + 32 * g);
        const uint32_t acc = g > 0 ? 1u : 0u;
        asm volatile("{\n .reg .pred p;\n setp.ne.u32 p, %6, 0;\n"
                     " tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n}"
                     ::"r"(tmem + d_col), "l"(ad), "l"(bd), "r"(idesc), "r"(tmem + sfa_col), "r"(tmem + kScColSFB),
                     "r"(acc)
                     : "memory");
    }
}

// Epilogue of one page for the calling thread's token (TMEM lane = 32 (warp % 4) + lane; the
// page's accumulator at d_col): the max over query slots n < Q with token j <= lim + n (j = the
// token's position) of D[n] + D[NQ + n] (the score times 2^sigma_min), -inf if none.
template <int NQ>
__device__ __forceinline__ float sc_token_max(uint32_t tmem, uint32_t d_col, int j, int lim, int Q) {
    const uint32_t addr = tmem + ((uint32_t)(32 * ((threadIdx.x >> 5) & 3)) << 16) + d_col;
    uint32_t r[2 * NQ];
    if constexpr (NQ == 8) {
        asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
                     "tcgen05.wait::ld.sync.aligned;"
                     : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                       "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
                     : "r"(addr)
                     : "memory");
    } else {
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
            "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
            "tcgen05.wait::ld.sync.aligned;"
            : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
              "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
              "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
              "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
            : "r"(addr)
            : "memory");
    }
    float best = -INFINITY;
#pragma unroll
    for (int n = 0; n < NQ; ++n) {
        const float s = __uint_as_float(r[n]) + __uint_as_float(r[NQ + n]);
        const bool ok = n < Q && j <= lim + n;
        best = ok ? fmaxf(best, s) : best;
    }
    return best;
}

// ---- the pipelined scorer ----------------------------------------------------------------------
// Whole pages stream into a ring of SR raw stages by 1-D bulk copies (lane 0 of warp 9 issues them
// as the stages free up). Warps 0-3 produce: repack a landed page's nibbles into a tile stage, store the
// adjusted scale factors and signal the stage full (and the raw stage free). Lane 0 of warp 8 issues
// the MMAs (an MMA issue holds its thread for about a hundred cycles, so the issuer does nothing
// else); warps 4-7 take the epilogue (one token per thread), combine the four warp maxima at a
// named barrier and free the accumulator stage. Every
// wait is bounded; once one gives up, the CTA's later waits return at once and the status records it.
struct ScPipe {
    uint8_t* raw;        // kMxPageBytes per raw stage (whole pages, bulk-copied), 16-byte aligned
    uint64_t* rfull;     // [raw stages] the page landed (transaction count)
    uint64_t* rfree;     // [raw stages] the producers have read it (4 arrivals)
    uint8_t* tiles;      // kScTileBytes per tile stage, 1024-byte aligned
    uint8_t* qt;         // the query pieces
    uint64_t* full;      // [tile stages] producers done (4 arrivals: one per producer warp)
    uint64_t* tfree;     // [tile stages] the stage's MMAs done (commit)
    uint64_t* afull;     // [accumulator stages] MMAs done (commit)
    uint64_t* afree;     // [accumulator stages] epilogue done (1 arrival)
    float* red;          // [accumulator stages][4] warp maxima
    int* gave_up;        // shared flag
    uint32_t tmem;
    uint32_t seq;        // pages this CTA has scored so far (sets every barrier's phase)
};

// One thread: initialise the pipeline's barriers (before the first use, behind a barrier).
template <int SR, int ST, int SD>
__device__ __forceinline__ void sc_pipe_init(ScPipe& pp) {
#pragma unroll
    for (int r = 0; r < SR; ++r) {
        mbar_init(&pp.rfull[r], 1);
        mbar_init(&pp.rfree[r], 4);
    }
#pragma unroll
    for (int t = 0; t < ST; ++t) {
        mbar_init(&pp.full[t], 4);
        mbar_init(&pp.tfree[t], 1);
    }
#pragma unroll
    for (int d = 0; d < SD; ++d) {
        mbar_init(&pp.afull[d], 1);
        mbar_init(&pp.afree[d], 1);
    }
    *pp.gave_up = 0;
    mbar_fence_init();
}

__device__ __forceinline__ bool sc_wait(ScPipe& pp, uint64_t* bar, uint32_t parity, int32_t* status) {
    if (*(volatile int*)pp.gave_up) return false;
    if (mbar_wait_spin(bar, parity)) return true;
    *(volatile int*)pp.gave_up = 1;
    flag_status(status, SMX_DEV_TIMEOUT);
    return false;
}

// Producer thread t (0..127): repack chunks t + 128 i (8 bytes of nibbles each; row = chunk / 8) of
// a raw page in shared memory into a tile.
__device__ __forceinline__ void sc_repack(const uint8_t* raw, uint8_t* tile, int t) {
    uint2 w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = *reinterpret_cast<const uint2*>(raw + 8 * (t + 128 * i));
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int ch = t + 128 * i, r = ch >> 3, c = ch & 7;
        *reinterpret_cast<uint4*>(tile + sc_chunk(r, c)) = make_uint4(w[i].x, w[i].y, 0u, 0u);
    }
}

// Scores pages phys[0 .. np) (physical ids in shared memory, -1 = a bad id: flagged, scored -inf)
// of one row, logical pages p_first .., into score_row[p_first + i] (times 2^-sigma_min). Every
// thread of the 320-thread block (10 warps) calls it after sc_setup_query; it ends with a block
// barrier.
template <int NQ, int SR, int ST, int SD>
__device__ __forceinline__ void sc_score_pages(ScPipe& pp, const uint8_t* pool, const int64_t* phys, int np,
                                               int p_first, int lim, int Q, const ScQuery& sq, float* score_row,
                                               int32_t* status) {
    static_assert(SR >= 2 && ST >= 2 && ST <= kScMaxTileStages && SD >= 2 && SD <= kScMaxAccStages, "pipeline stages");
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t seq = pp.seq;
    if (warp == 9) {
        // ---- page copies ----
        if (lane == 0) {
#pragma unroll 1
            for (int i = 0; i < np; ++i) {
                const uint32_t g = seq + (uint32_t)i, rs = g % SR, use = g / SR;
                if (use > 0) sc_wait(pp, &pp.rfree[rs], (use - 1) & 1u, status);
                if (phys[i] >= 0) {
                    mbar_arrive_expect_tx(&pp.rfull[rs], (uint32_t)kMxPageBytes);
                    bulk_g2s(pp.raw + rs * kMxPageBytes, pool + phys[i] * kMxPageBytes, (uint32_t)kMxPageBytes,
                             &pp.rfull[rs]);
                } else {
                    mbar_arrive(&pp.rfull[rs]);   // a bad page id: nothing to copy (scored -inf)
                }
            }
        }
        __syncwarp();
    } else if (warp < 4) {
        // ---- producers ----
        const int t = threadIdx.x;
#pragma unroll 1
        for (int i = 0; i < np; ++i) {
            const uint32_t g = seq + (uint32_t)i, rs = g % SR, st = g % ST, use = g / ST;
            sc_wait(pp, &pp.rfull[rs], (g / SR) & 1u, status);
            if (use > 0) sc_wait(pp, &pp.tfree[st], (use - 1) & 1u, status);
            const uint8_t* raw = pp.raw + rs * kMxPageBytes;
            sc_repack(raw, pp.tiles + st * kScTileBytes, t);
            const uint32_t sw = *reinterpret_cast<const uint32_t*>(raw + kMxScaleOff + 4 * t);
            sc_store_sfa(pp.tmem, kScColSFA + 4 * st, sw, sq);
            fence_proxy_async_smem();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&pp.full[st]);
                mbar_arrive(&pp.rfree[rs]);
            }
        }
    } else if (warp == 8) {
        // ---- MMA issue ----
        if (lane == 0) {
#pragma unroll 1
            for (int i = 0; i < np; ++i) {
                const uint32_t g = seq + (uint32_t)i, st = g % ST, ds = g % SD;
                bool ok = sc_wait(pp, &pp.full[st], (g / ST) & 1u, status);
                if (g >= (uint32_t)SD) ok = sc_wait(pp, &pp.afree[ds], ((g / SD) - 1) & 1u, status) && ok;
                tc_fence_after_sync();
                if (ok)
                    sc_issue_page<NQ>(pp.tmem, kScColD + 32 * ds, kScColSFA + 4 * st,
                                      smem_u32(pp.tiles + st * kScTileBytes), smem_u32(pp.qt));
                tc_commit(&pp.afull[ds]);
                tc_commit(&pp.tfree[st]);
            }
        }
        __syncwarp();
    } else if (warp < 8) {
        // ---- epilogue (warps 4-7) ----
        const int tok = threadIdx.x - 128;
#pragma unroll 1
        for (int i = 0; i < np; ++i) {
            const uint32_t g = seq + (uint32_t)i, ds = g % SD;
            sc_wait(pp, &pp.afull[ds], (g / SD) & 1u, status);
            tc_fence_after_sync();
            float best = -INFINITY;
            const bool good = phys[i] >= 0;
            if (good) best = sc_token_max<NQ>(pp.tmem, kScColD + 32 * ds, (p_first + i) * kPage + tok, lim, Q);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) best = fmaxf(best, __shfl_xor_sync(0xFFFFFFFFu, best, o));
            if (lane == 0) pp.red[4 * ds + (warp - 4)] = best;
            tc_fence_before_sync();
            asm volatile("bar.sync 1, 128;" ::: "memory");
            if (warp == 4 && lane == 0) {
                const float* r = pp.red + 4 * ds;
                score_row[p_first + i] = good ? mul_exp2(fmaxf(fmaxf(r[0], r[1]), fmaxf(r[2], r[3])), -sq.sig_min) : -INFINITY;
                if (!good) flag_status(status, SMX_DEV_BAD_PAGE_ID);
                mbar_arrive(&pp.afree[ds]);
            }
        }
    }
    // every stage's last commit has arrived before the barriers or the columns are used again
    if (threadIdx.x == 0) {
        for (int k = max(0, np - ST); k < np; ++k) {
            const uint32_t g = seq + (uint32_t)k;
            sc_wait(pp, &pp.tfree[g % ST], (g / ST) & 1u, status);
        }
    }
    pp.seq = seq + (uint32_t)np;
    __syncthreads();
}

}  // namespace smx

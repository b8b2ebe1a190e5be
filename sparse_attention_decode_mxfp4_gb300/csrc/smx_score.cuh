// smx_score.cuh -- the index scorer's per-tile work (a3), shared by the standalone scorer and the
// fused decode step.
//
// [ATOM-2812] "Mono decode over the MXFP4 KV and index caches", commit "--index-cache-dtype
// mxfp4": each index page is read as 16 B key loads plus a dword of E8M0 scales and the fp4 keys
// are widened for a 16-bit MMA against the index query.
//
// Lane (g, t) of the m16n8k16 MMA loads 16 B (= 32 elements of scale group t) of token rows g and
// g+8 of a 16-token tile straight into registers (a warp instruction covers 512 contiguous
// bytes), converts byte pairs with the hardware E2M1 -> f16x2 conversion, and multiplies group t
// by 2^(s_t - max_g s_g) so that one fp32 accumulator serves the whole row; the row's common
// factor 2^(max_g s_g) and the query's power-of-two factor are applied to the fp32 result. The
// index query is held in f16 after a per-query power-of-two rescale that puts its largest element
// in [2^14, 2^15): every bf16 element within 2^31 of that maximum is exact in f16, so products are
// exact and only the fp32 accumulation rounds. The K permutation of the MMA is chosen so that each
// lane's 16 contiguous bytes are its A fragment: k-step s takes bytes 2s and 2s+1 of every lane's
// group.
#pragma once

#include "smx_device.cuh"

namespace smx {

constexpr int kIdxWarps = 8;

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t h16) { return __uint_as_float(h16 << 16); }

// One lane's share of one 16-token tile: 16 B of nibbles of token rows g and g+8 and the rows'
// scale words. Pages are read through L2 (a CTA that inserted rows must see its own writes).
// NVFP4 pages (NV): the lane's 32 elements are blocks 2t and 2t + 1, whose two E4M3 scale bytes
// are the low (t even) or high (t odd) half of the row's scale word 4 (t / 2).
struct TileFrag {
    uint4 c0, c1;
    uint32_t sw0, sw1;
};

template <bool NV = false>
__device__ __forceinline__ void load_tile(TileFrag& f, const uint8_t* page, int tile, int g, int t) {
    const int r0 = tile * 16 + g, r1 = r0 + 8;
    f.c0 = ldg_cg_v4(page + r0 * 64 + 16 * t);
    f.c1 = ldg_cg_v4(page + r1 * 64 + 16 * t);
    if constexpr (NV) {
        const int sh = 16 * (t & 1);
        f.sw0 = (ldg_cg_u32(page + kNvScaleOff + 8 * r0 + 4 * (t >> 1)) >> sh) & 0xFFFFu;
        f.sw1 = (ldg_cg_u32(page + kNvScaleOff + 8 * r1 + 4 * (t >> 1)) >> sh) & 0xFFFFu;
    } else {
        f.sw0 = ldg_cg_u32(page + kMxScaleOff + 4 * r0);
        f.sw1 = ldg_cg_u32(page + kMxScaleOff + 4 * r1);
    }
}

// NVFP4: the max over this lane's scores of one tile. Each E2M1 pair is widened to f16x2 and
// multiplied by its block's E4M3 scale (as f16; the product, at most 6 significant bits between
// 2^-10 and 2688, is exact), so one fp32 accumulator per row serves the whole row; the query's
// power-of-two factor and the per-tensor scale g are applied to the fp32 result. A NaN scale
// makes the token's score NaN, which the maximum leaves out.
template <int NT>
__device__ __forceinline__ float score_tile_nv(const TileFrag& f, const uint32_t (&qf)[NT][16], const int (&sig_c)[NT][2],
                                               int p, int tile, int g, int t, int lim, int Q, float g_idx) {
    const int r0 = tile * 16 + g, r1 = r0 + 8;
    // f16x2 splats of the scales of blocks 2t (words 0, 1) and 2t + 1 (words 2, 3), rows r0, r1
    uint32_t fa[2], fb[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const uint32_t b0 = (f.sw0 >> (8 * k)) & 0xFFu, b1 = (f.sw1 >> (8 * k)) & 0xFFu;
        fa[k] = e4m3x2_to_f16x2(b0 | (b0 << 8));
        fb[k] = e4m3x2_to_f16x2(b1 | (b1 << 8));
    }
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
        const uint32_t s0 = fa[wi >> 1], s1 = fb[wi >> 1];
        x0 = hmul2_u32(x0, s0); x1 = hmul2_u32(x1, s0); x2 = hmul2_u32(x2, s0); x3 = hmul2_u32(x3, s0);
        y0 = hmul2_u32(y0, s1); y1 = hmul2_u32(y1, s1); y2 = hmul2_u32(y2, s1); y3 = hmul2_u32(y3, s1);
        const int k0 = 2 * wi, k1 = 2 * wi + 1;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            mma_f16_16816(acc[nt][0], x0, y0, x1, y1, qf[nt][2 * k0], qf[nt][2 * k0 + 1]);
            mma_f16_16816(acc[nt][1], x2, y2, x3, y3, qf[nt][2 * k1], qf[nt][2 * k1 + 1]);
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
            const bool valid = (n < Q) && (j <= lim + n);
            const float v = __fmul_rn(mul_exp2(acc[nt][0][c] + acc[nt][1][c], -sig_c[nt][col]), g_idx);
            best = valid ? fmaxf(best, v) : best;
        }
    }
    return best;
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

// The raw index-query words a warp needs for setup_index_query (rows warp and warp + 8 of the
// row's [Q][128] bf16 bits, dims 4 lane .. 4 lane + 3), loaded ahead so their latency overlaps
// other work.
struct IndexQueryRaw {
    uint2 v[2];
};

__device__ __forceinline__ IndexQueryRaw load_index_query(const uint16_t* qrow, int Q) {
    IndexQueryRaw r;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int n = warp + kIdxWarps * k;
        r.v[k] = n < Q ? reinterpret_cast<const uint2*>(qrow + (int64_t)n * kD)[lane] : make_uint2(0, 0);
    }
    return r;
}

// Index queries of one row as f16 with a per-query power-of-two factor 2^sigma, staged in shared
// memory (qh, sig), then this lane's B fragments: lane (g, t) of n-tile nt holds
// q'[nt*8+g][32t .. 32t+31]. Every thread of the (kIdxWarps-warp) block calls it; it holds one
// barrier. Q <= 16.
template <int NT>
__device__ __forceinline__ void setup_index_query(const IndexQueryRaw& raw, int Q, uint32_t (&qh)[16][64], int* sig,
                                                  uint32_t (&qf)[NT][16], int (&sig_c)[NT][2]) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int n = warp + kIdxWarps * k;
        if (n >= 8 * NT) continue;
        const uint2 v = raw.v[k];
        int sigma = 0;
        if (n < Q) {
            uint32_t mx = max(max(v.x & 0x7FFFu, (v.x >> 16) & 0x7FFFu), max(v.y & 0x7FFFu, (v.y >> 16) & 0x7FFFu));
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
            if (mx != 0) {
                const int e = (int)(mx >> 7);
                const int E = e ? e - 127 : -133 + (31 - __clz((int)(mx & 0x7F)));
                sigma = 14 - E;
            }
        }
        // rows past Q are zero
        const __half2 h0 = __floats2half2_rn(mul_exp2(bf16_bits_to_f32(v.x & 0xFFFFu), sigma),
                                             mul_exp2(bf16_bits_to_f32(v.x >> 16), sigma));
        const __half2 h1 = __floats2half2_rn(mul_exp2(bf16_bits_to_f32(v.y & 0xFFFFu), sigma),
                                             mul_exp2(bf16_bits_to_f32(v.y >> 16), sigma));
        qh[n][2 * lane] = *reinterpret_cast<const uint32_t*>(&h0);
        qh[n][2 * lane + 1] = *reinterpret_cast<const uint32_t*>(&h1);
        if (lane == 0) sig[n] = sigma;
    }
    __syncthreads();
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
}

}  // namespace smx

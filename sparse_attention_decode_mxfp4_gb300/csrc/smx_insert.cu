// smx_insert.cu -- a1 (page row store) and a2 (q packing).
//
// [ATOM-2812] "Mono decode over the MXFP4 KV and index caches", commit "--index-cache-dtype
// mxfp4": K1 writes each new token's index-K row into its 8704 B MXFP4 page (E8M0 group scale
// + packed fp4 conversion); commit "MXFP4 main KV": K and V rows use the same row store;
// commits "e4m3 q_out convention" / "pack_q_e4m3": q as saturating e4m3 at unit scale.
// One warp quantises one 128-element row: lane l owns elements 4l..4l+3 (one float4 load,
// coalesced 512 B per warp) and writes 2 nibble bytes; lane 0 writes the 4 scale bytes (MXFP4)
// or the 8 block scale bytes (NVFP4, the format the pages name: E2M1 with an E4M3 scale per 16
// elements and the pool's per-tensor fp32 scale).
#include "smx_device.cuh"
#include "smx_internal.h"

namespace smx {

struct InsertArgs {
    const float* k;        // [B][T][Hkv][128]
    const float* v;
    const float* kidx;     // [B][T][128]
    const int32_t* page_table;
    const int32_t* ctx_len;   // insert: positions ctx - Q + t; prefill: unused
    const int32_t* n_fill;    // prefill: positions [0, n_fill[b])
    uint8_t* k_pool;
    uint8_t* v_pool;
    uint8_t* idx_pool;
    int32_t* status;
    int64_t T;             // token stride of the dense inputs
    int64_t n_pool;
    int B, Q, Hkv, max_pages, kv_format, idx_format;
    float nv_k, nv_v, nv_idx;  // NVFP4 per-tensor decode scales
    int prefill;
};

__device__ __forceinline__ void store_row(const InsertArgs& a, int kind, int64_t phys, int slot,
                                          const float* src, int lane) {
    const float4 x = reinterpret_cast<const float4*>(src)[lane];
    if (kind == 0) {
        if (a.idx_format == SMX_KV_NVFP4) {
            uint8_t* page = a.idx_pool + phys * kNvPageBytes;
            quant_row_nvfp4_warp(x, a.nv_idx, page + slot * 64, page + kNvScaleOff + slot * 8, lane);
        } else {
            uint8_t* page = a.idx_pool + phys * kMxPageBytes;
            quant_row_mxfp4_warp(x, page + slot * 64, page + kMxScaleOff + slot * 4, lane);
        }
        return;
    }
    const int h = (kind - 1) % a.Hkv;
    uint8_t* pool = (kind <= a.Hkv) ? a.k_pool : a.v_pool;
    if (a.kv_format == SMX_KV_NVFP4) {
        uint8_t* page = pool + (phys * a.Hkv + h) * (int64_t)kNvPageBytes;
        quant_row_nvfp4_warp(x, kind <= a.Hkv ? a.nv_k : a.nv_v, page + slot * 64, page + kNvScaleOff + slot * 8, lane);
    } else if (a.kv_format == SMX_KV_E4M3_ROWSCALE) {
        uint8_t* page = pool + (phys * a.Hkv + h) * (int64_t)kRsPageBytes;
        quant_row_e4m3rs_warp(x, page + slot * 128, reinterpret_cast<float*>(page + kRsScaleOff) + slot, lane);
    } else {
        uint8_t* page = pool + (phys * a.Hkv + h) * (int64_t)kMxPageBytes;
        quant_row_mxfp4_warp(x, page + slot * 64, page + kMxScaleOff + slot * 4, lane);
    }
}

// One warp per (row b, token, kind) with kind 0 = index-K (skipped without an index input),
// 1..Hkv = K heads, Hkv+1..2Hkv = V.
__global__ void __launch_bounds__(256) kv_insert_kernel(InsertArgs a) {
    const int lane = threadIdx.x & 31;
    const int kinds = 1 + 2 * a.Hkv;
    const int64_t per_row = a.prefill ? a.T : (int64_t)a.Q;
    const int64_t total = (int64_t)a.B * per_row * kinds;
    const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t w = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); w < total; w += nwarps) {
        const int kind = (int)(w % kinds);
        if (kind == 0 && a.kidx == nullptr) continue;
        const int64_t tok = w / kinds;
        const int b = (int)(tok / per_row);
        const int64_t i = tok % per_row;
        int64_t pos, src_tok;
        if (a.prefill) {
            const int64_t n = a.n_fill[b];
            if (i >= n) continue;
            if (n > (int64_t)a.max_pages * kPage || n > a.T) {
                if (lane == 0 && i == 0) flag_status(a.status, SMX_DEV_BAD_CTX);
                continue;
            }
            pos = i;
            src_tok = (int64_t)b * a.T + i;
        } else {
            const int ctx = a.ctx_len[b];
            if (ctx < a.Q || ctx > a.max_pages * kPage) {
                if (lane == 0 && kind == 1) flag_status(a.status, SMX_DEV_BAD_CTX);
                continue;
            }
            pos = (int64_t)ctx - a.Q + i;
            src_tok = (int64_t)b * a.Q + i;
        }
        const int64_t phys = a.page_table[(int64_t)b * a.max_pages + pos / kPage];
        if (phys < 0 || phys >= a.n_pool) {
            if (lane == 0 && kind == 1) flag_status(a.status, SMX_DEV_BAD_PAGE_ID);
            continue;
        }
        const int slot = (int)(pos % kPage);
        const float* src;
        if (kind == 0) src = a.kidx + src_tok * kD;
        else if (kind <= a.Hkv) src = a.k + (src_tok * a.Hkv + (kind - 1)) * kD;
        else src = a.v + (src_tok * a.Hkv + (kind - 1 - a.Hkv)) * kD;
        store_row(a, kind, phys, slot, src, lane);
    }
}

__global__ void __launch_bounds__(256) pack_q_kernel(const float* __restrict__ q, uint8_t* __restrict__ out, int64_t n) {
    const int64_t n4 = n / 4;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += stride) {
        const float4 x = reinterpret_cast<const float4*>(q)[i];
        reinterpret_cast<uint32_t*>(out)[i] = pack_q4(x);
    }
    for (int64_t i = n4 * 4 + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
        const float4 x = make_float4(q[i], 0.f, 0.f, 0.f);
        out[i] = (uint8_t)(pack_q4(x) & 0xFF);
    }
}

cudaError_t launch_kv_insert(const smx_shape_t& s, const float* k, const float* v, const float* kidx,
                             int64_t T, const int32_t* page_table, const int32_t* ctx_len,
                             const int32_t* n_fill, uint8_t* k_pool, uint8_t* v_pool, uint8_t* idx_pool,
                             int32_t* status, bool prefill, cudaStream_t st) {
    InsertArgs a;
    a.k = k; a.v = v; a.kidx = kidx; a.page_table = page_table; a.ctx_len = ctx_len; a.n_fill = n_fill;
    a.k_pool = k_pool; a.v_pool = v_pool; a.idx_pool = idx_pool; a.status = status;
    a.T = T; a.n_pool = s.n_pool_pages; a.B = s.B; a.Q = s.Q; a.Hkv = s.Hkv;
    a.max_pages = s.max_pages_per_row; a.kv_format = s.kv_format; a.idx_format = s.idx_format;
    a.nv_k = s.nv_scale_k; a.nv_v = s.nv_scale_v; a.nv_idx = s.nv_scale_idx; a.prefill = prefill ? 1 : 0;
    const int64_t rows = (int64_t)s.B * (prefill ? T : s.Q) * (1 + 2 * s.Hkv);
    int64_t blocks = (rows + 7) / 8;
    if (blocks > 152 * 32) blocks = 152 * 32;
    if (blocks < 1) blocks = 1;
    kv_insert_kernel<<<(unsigned)blocks, 256, 0, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_pack_q(const float* q, uint8_t* out, int64_t n, cudaStream_t st) {
    int64_t blocks = (n / 4 + 255) / 256;
    if (blocks > 152 * 16) blocks = 152 * 16;
    if (blocks < 1) blocks = 1;
    pack_q_kernel<<<(unsigned)blocks, 256, 0, st>>>(q, out, n);
    return cudaGetLastError();
}

}  // namespace smx

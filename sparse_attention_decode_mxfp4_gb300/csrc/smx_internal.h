// smx_internal.h -- launchers shared between the kernel translation units and the C ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/smx.h"

namespace smx {

// Raise a kernel's dynamic shared-memory limit once per device (the first launch on a device
// does it, so that launch should come before any stream capture).
cudaError_t ensure_smem_attr(const void* kernel, int bytes);

cudaError_t launch_kv_insert(const smx_shape_t& s, const float* k, const float* v, const float* kidx,
                             int64_t T, const int32_t* page_table, const int32_t* ctx_len,
                             const int32_t* n_fill, uint8_t* k_pool, uint8_t* v_pool, uint8_t* idx_pool,
                             int32_t* status, bool prefill, cudaStream_t st);

cudaError_t launch_pack_q(const float* q, uint8_t* out, int64_t n, cudaStream_t st);

cudaError_t launch_index_scores(const smx_shape_t& s, const uint16_t* qidx, const uint8_t* idx_pool,
                                const int32_t* page_table, const int32_t* ctx_len, float* scores,
                                int32_t* status, cudaStream_t st);

// Tensor map of an MXFP4 index pool ([n_pool][8704] bytes, 32-byte aligned) for the scan: one box
// = one whole page (128 token rows of nibbles, then its scale words), unpacked for the fp4 MMA
// operand, 128-byte swizzle.
cudaError_t encode_index_map(CUtensorMap* map, const uint8_t* idx_pool, int64_t n_pool);

cudaError_t launch_topk(const smx_shape_t& s, const float* scores, const int32_t* ctx_len,
                        int32_t* topk_pages, int32_t* topk_count, cudaStream_t st);

cudaError_t launch_attn_split(const smx_shape_t& s, const void* q, const uint8_t* k_pool,
                              const uint8_t* v_pool, const int32_t* page_table, const int32_t* ctx_len,
                              const int32_t* topk_pages, const int32_t* topk_count, float* part_o,
                              float* part_m, float* part_l, int32_t* status, cudaStream_t st);

cudaError_t launch_attn_merge(const smx_shape_t& s, const float* part_o, const float* part_m,
                              const float* part_l, float* out, cudaStream_t st);

// Partition count that fills one wave of the device's SMs with split CTAs (0 on a CUDA error).
int suggest_num_splits(const smx_shape_t& s);

// Steps with an NVFP4 pool run the standalone kernels in sequence instead of the fused kernel.
inline bool nvfp4_chain(const smx_shape_t& s) { return s.kv_format == SMX_KV_NVFP4 || s.idx_format == SMX_KV_NVFP4; }
// Bytes of one K or V page of one KV head, and of one index page.
inline int kv_page_bytes(const smx_shape_t& s) {
    return s.kv_format == SMX_KV_E4M3_ROWSCALE ? SMX_E4M3RS_PAGE_BYTES
         : s.kv_format == SMX_KV_NVFP4 ? SMX_NVFP4_PAGE_BYTES : SMX_MXFP4_PAGE_BYTES;
}
inline int idx_page_bytes(const smx_shape_t& s) {
    return s.idx_format == SMX_KV_NVFP4 ? SMX_NVFP4_PAGE_BYTES : SMX_MXFP4_PAGE_BYTES;
}

// ---- the fused decode step (one cooperative kernel, smx_step.cu) ----
struct StepGeom {
    int row_warps;        // warps per token half of the attention (16 query rows each)
    int rows_per_cta;     // 16 x row_warps
    int n_rg;             // row groups per KV head
    int page_bytes;       // bytes of one K or V page of one KV head
    size_t smem;          // dynamic shared bytes of the kernel
    size_t n_counters;    // u32 counters in the workspace: B rows, B x Hkv x n_rg groups, 1
};
StepGeom step_geom(const smx_shape_t& s);                // the workspace's geometry (either path)
StepGeom step_geom(const smx_shape_t& s, bool tc);       // tc: the tensor-core attention path
// Whether the fused step runs its attention on the tensor-core path for this shape (current device).
bool decode_step_uses_tc(const smx_shape_t& s);

struct StepIO {
    const float* q_f32;
    const uint16_t* q_bf16;
    const uint16_t* qidx;
    const float* k_new;
    const float* v_new;
    const float* kidx_new;
    const int32_t* page_table;
    const int32_t* ctx_len;
    uint8_t* idx_pool;
    uint8_t* k_pool;
    uint8_t* v_pool;
    int32_t* topk_out;
    int32_t* count_out;
    const int32_t* topk_in;    // a reused selection (launch_decode_step with reuse), else null
    const int32_t* count_in;
    float* out;
    int32_t* status;
    uint32_t* counters;   // n_counters, zero before the first step; every step leaves them zero
    float* scores;        // [B][max_pages]
    float* part_o;        // [B][S][Q][Hq][128]
    float* part_m;        // [B][S][Q][Hq]
    float* part_l;
    uint8_t* q_img;       // [B][Hkv][tc row groups][16384]: the tensor-core units' packed q tiles
};
// Bytes of the packed q tile images of the fused step's tensor-core units (either path reserves them).
size_t step_q_image_bytes(const smx_shape_t& s);
cudaError_t launch_decode_step(const smx_shape_t& s, const StepIO& io, cudaStream_t st, bool reuse = false);

// The argument checks of smx_decode_step (shape, pointers, alignment; not the workspace): SMX_OK
// or the status smx_decode_step returns for them. Reads no device memory.
int check_step_args(const smx_shape_t* s, const float* q_f32, const uint16_t* q_bf16, const uint16_t* qidx_bf16,
                    const float* k_new, const float* v_new, const float* kidx_new, const int32_t* page_table,
                    const int32_t* ctx_len, const uint8_t* k_pool, const uint8_t* v_pool, const uint8_t* idx_pool,
                    const int32_t* topk_pages, const int32_t* topk_count, const float* out);

// Bound of the step kernels' waits for other CTAs (ns), as set by smx_set_wait_limit_ns.
uint64_t wait_limit_ns();

// Bytes at the head of the decode-step workspace that must be zero before a step (the counters).
size_t workspace_counter_bytes(const smx_shape_t& s);

}  // namespace smx

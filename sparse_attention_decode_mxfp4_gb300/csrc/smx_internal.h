// smx_internal.h -- launchers shared between the kernel translation units and the C ABI.
#pragma once

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

cudaError_t launch_topk(const smx_shape_t& s, const float* scores, const int32_t* ctx_len,
                        int32_t* topk_pages, int32_t* topk_count, cudaStream_t st);

cudaError_t launch_attn_split(const smx_shape_t& s, const void* q, const uint8_t* k_pool,
                              const uint8_t* v_pool, const int32_t* page_table, const int32_t* ctx_len,
                              const int32_t* topk_pages, const int32_t* topk_count, float* part_o,
                              float* part_m, float* part_l, int32_t* status, cudaStream_t st);

cudaError_t launch_attn_merge(const smx_shape_t& s, const float* part_o, const float* part_m,
                              const float* part_l, float* out, bool pdl, cudaStream_t st);

// The fused step's kernels: a1 + a2 + a3 + a4 in one launch (the scorer with the insert, the q
// packing and, in the last CTA of each row, the selection), then a5 (split stage from the staged
// selection); each may be launched as a programmatic dependent of the preceding kernel.
// Workspace pieces through which the fused scorer hands the split stage the packed q and the
// row's selection.
struct FusedSelect {
    const float* q_f32;   // MXFP4 K/V: q to pack (nullptr for the e4m3 row-scale format)
    uint16_t* qbf;
    int32_t* arrivals;
    int32_t* sel_pages;
    int32_t* sel_phys;
    int32_t* sel_count;
    int32_t* topk_out;
    int32_t* count_out;
};

cudaError_t launch_index(const smx_shape_t& s, const uint16_t* qidx, uint8_t* idx_pool,
                         const int32_t* page_table, const int32_t* ctx_len, float* scores, int32_t* status,
                         const float* k_new, const float* v_new, const float* kidx_new, uint8_t* k_pool,
                         uint8_t* v_pool, bool pdl, cudaStream_t st, const FusedSelect* fs);

// Partition count that fills one wave of the device's SMs with split CTAs (0 on a CUDA error).
int suggest_num_splits(const smx_shape_t& s);
cudaError_t launch_attn_fused_split(const smx_shape_t& s, const uint16_t* qbf, const uint8_t* k_pool,
                                    const uint8_t* v_pool, const int32_t* ctx_len, const int32_t* sel_pages,
                                    const int32_t* sel_phys, const int32_t* sel_count, float* part_o,
                                    float* part_m, float* part_l, int32_t* status, cudaStream_t st);

}  // namespace smx

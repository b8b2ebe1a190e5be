// smx_api.cu -- the C ABI of libsmx (declared in include/smx.h): argument checks, workspace
// layout and the order of launches. No device memory is read, allocated or synchronised here.
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "smx_device.cuh"
#include "smx_internal.h"

namespace smx {

cudaError_t ensure_smem_attr(const void* kernel, int bytes) {
    constexpr int kMaxDev = 64, kMaxKernels = 16;
    static std::mutex mu;
    static const void* seen_kernel[kMaxKernels] = {};
    static int seen_bytes[kMaxKernels][kMaxDev] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDev) return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    std::lock_guard<std::mutex> lock(mu);
    int slot = -1;
    for (int i = 0; i < kMaxKernels; ++i) {
        if (seen_kernel[i] == kernel || seen_kernel[i] == nullptr) {
            slot = i;
            break;
        }
    }
    if (slot < 0) return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    seen_kernel[slot] = kernel;
    if (seen_bytes[slot][dev] >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) seen_bytes[slot][dev] = bytes;
    return e;
}

size_t workspace_counter_bytes(const smx_shape_t& s) { return step_geom(s).n_counters * sizeof(uint32_t); }

static std::atomic<uint64_t> g_wait_limit_ns{0};   // 0: the default bound

uint64_t wait_limit_ns() {
    const uint64_t v = g_wait_limit_ns.load(std::memory_order_relaxed);
    return v ? v : kDefaultWaitNs;
}

}  // namespace smx

namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t x) { return (x + kAlign - 1) & ~(kAlign - 1); }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The index pool is read by tensor-map copies of a packed 4-bit type: 32-byte aligned.
bool aligned32(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; }

int check_shape(const smx_shape_t* s) {
    if (!s) return SMX_ERR_INVALID_ARG;
    if (s->B < 1 || s->Q < 1 || s->Hq < 1 || s->Hkv < 1 || s->max_pages_per_row < 1 ||
        s->n_pool_pages < 1 || s->topk < 1 || s->num_splits < 1)
        return SMX_ERR_INVALID_ARG;
    if (s->Hq % s->Hkv != 0) return SMX_ERR_INVALID_ARG;
    if (s->D != 128 || s->Di != 128 || s->page_tokens != 128) return SMX_ERR_UNSUPPORTED;
    if (s->Q > SMX_MAX_Q) return SMX_ERR_UNSUPPORTED;
    if (s->kv_format != SMX_KV_MXFP4 && s->kv_format != SMX_KV_E4M3_ROWSCALE && s->kv_format != SMX_KV_NVFP4)
        return SMX_ERR_UNSUPPORTED;
    if (s->idx_format != SMX_KV_MXFP4 && s->idx_format != SMX_KV_NVFP4) return SMX_ERR_UNSUPPORTED;
    auto scale_ok = [](float g) { return g > 0.0f && g <= 3.0e38f; };   // finite, positive (NaN fails)
    if (s->kv_format == SMX_KV_NVFP4 && !(scale_ok(s->nv_scale_k) && scale_ok(s->nv_scale_v))) return SMX_ERR_INVALID_ARG;
    if (s->idx_format == SMX_KV_NVFP4 && !scale_ok(s->nv_scale_idx)) return SMX_ERR_INVALID_ARG;
    if (smx::nvfp4_chain(*s) && s->pages_per_block > 1) return SMX_ERR_UNSUPPORTED;
    if (s->topk > SMX_MAX_TOPK || s->max_pages_per_row > SMX_MAX_PAGES_PER_ROW) return SMX_ERR_UNSUPPORTED;
    if (s->n_pool_pages > 0x7FFFFFFF) return SMX_ERR_UNSUPPORTED;
    if (s->B > 65535 || s->num_splits > 65535 || (int64_t)s->Hkv * s->Hq * s->Q > 65535)
        return SMX_ERR_UNSUPPORTED;
    const int ppb = s->pages_per_block;
    if (ppb != 0 && ppb != 1 && ppb != 2 && ppb != 4) return SMX_ERR_UNSUPPORTED;
    if ((int64_t)s->topk * (ppb > 1 ? ppb : 1) > SMX_MAX_TOPK) return SMX_ERR_UNSUPPORTED;
    return SMX_OK;
}

// The standalone top-k and split stage take one page per selected block only.
static int check_page_blocks(const smx_shape_t* s) { return s->pages_per_block > 1 ? SMX_ERR_UNSUPPORTED : SMX_OK; }

int cuda_status(cudaError_t e) { return e == cudaSuccess ? SMX_OK : SMX_ERR_CUDA; }

struct Workspace {
    uint32_t* counters;   // step counters (zero between calls)
    float* scores;        // [B][max_pages]
    float* part_o;
    float* part_m;
    float* part_l;
    uint8_t* q_img;
    size_t bytes;
};

Workspace layout(const smx_shape_t* s, void* base) {
    Workspace w;
    const uintptr_t p = reinterpret_cast<uintptr_t>(base);
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const uintptr_t at = p + off;
        off = align_up(off + bytes);
        return at;
    };
    const size_t rows = (size_t)s->B * s->num_splits * s->Q * s->Hq;
    // the counters come first so that a zeroed prefix is easy to keep
    w.counters = reinterpret_cast<uint32_t*>(take(smx::step_geom(*s).n_counters * sizeof(uint32_t)));
    w.scores = reinterpret_cast<float*>(take((size_t)s->B * s->max_pages_per_row * sizeof(float)));
    w.part_o = reinterpret_cast<float*>(take(rows * 128 * sizeof(float)));
    w.part_m = reinterpret_cast<float*>(take(rows * sizeof(float)));
    w.part_l = reinterpret_cast<float*>(take(rows * sizeof(float)));
    w.q_img = reinterpret_cast<uint8_t*>(take(smx::step_q_image_bytes(*s)));
    w.bytes = off;
    return w;
}

}  // namespace

namespace smx {

int check_step_args(const smx_shape_t* s, const float* q_f32, const uint16_t* q_bf16, const uint16_t* qidx_bf16,
                    const float* k_new, const float* v_new, const float* kidx_new, const int32_t* page_table,
                    const int32_t* ctx_len, const uint8_t* k_pool, const uint8_t* v_pool, const uint8_t* idx_pool,
                    const int32_t* topk_pages, const int32_t* topk_count, const float* out) {
    const int rc = check_shape(s);
    if (rc) return rc;
    const bool rs = s->kv_format == SMX_KV_E4M3_ROWSCALE;
    if ((rs ? (const void*)q_bf16 : (const void*)q_f32) == nullptr) return SMX_ERR_INVALID_ARG;
    if (!qidx_bf16 || !k_new || !v_new || !kidx_new || !page_table || !ctx_len || !k_pool || !v_pool ||
        !idx_pool || !topk_pages || !topk_count || !out)
        return SMX_ERR_INVALID_ARG;
    if (!rs && !aligned16(q_f32)) return SMX_ERR_INVALID_ARG;
    if (rs && (reinterpret_cast<uintptr_t>(q_bf16) & 3u)) return SMX_ERR_INVALID_ARG;
    if (!aligned16(qidx_bf16) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(kidx_new) ||
        !aligned16(k_pool) || !aligned16(v_pool) || !aligned32(idx_pool))
        return SMX_ERR_INVALID_ARG;
    return SMX_OK;
}

}  // namespace smx

extern "C" {

size_t smx_workspace_bytes(const smx_shape_t* shape) {
    if (check_shape(shape) != SMX_OK) return 0;
    return layout(shape, nullptr).bytes;
}

int smx_kv_insert_mxfp4(const smx_shape_t* s, const float* k_new, const float* v_new, const float* kidx_new,
                        const int32_t* page_table, const int32_t* ctx_len, uint8_t* k_pool, uint8_t* v_pool,
                        uint8_t* idx_pool, int32_t* dev_status, smx_stream_t stream) {
    int rc = check_shape(s);
    if (rc) return rc;
    if (!k_new || !v_new || !kidx_new || !page_table || !ctx_len || !k_pool || !v_pool || !idx_pool)
        return SMX_ERR_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(kidx_new) || !aligned16(k_pool) ||
        !aligned16(v_pool) || !aligned16(idx_pool))
        return SMX_ERR_INVALID_ARG;
    return cuda_status(smx::launch_kv_insert(*s, k_new, v_new, kidx_new, s->Q, page_table, ctx_len, nullptr,
                                             k_pool, v_pool, idx_pool, dev_status, false, (cudaStream_t)stream));
}

int smx_kv_insert(const smx_shape_t* s, const float* k_new, const float* v_new, const float* kidx_new,
                  const int32_t* page_table, const int32_t* ctx_len, uint8_t* k_pool, uint8_t* v_pool,
                  uint8_t* idx_pool, int32_t* dev_status, smx_stream_t stream) {
    return smx_kv_insert_mxfp4(s, k_new, v_new, kidx_new, page_table, ctx_len, k_pool, v_pool, idx_pool, dev_status,
                               stream);
}

int smx_kv_prefill(const smx_shape_t* s, const float* k, const float* v, const float* kidx, int64_t T,
                   const int32_t* page_table, const int32_t* n_fill, uint8_t* k_pool, uint8_t* v_pool,
                   uint8_t* idx_pool, int32_t* dev_status, smx_stream_t stream) {
    int rc = check_shape(s);
    if (rc) return rc;
    if (!k || !v || !kidx || !page_table || !n_fill || !k_pool || !v_pool || !idx_pool || T < 1)
        return SMX_ERR_INVALID_ARG;
    if (!aligned16(k) || !aligned16(v) || !aligned16(kidx) || !aligned16(k_pool) || !aligned16(v_pool) ||
        !aligned16(idx_pool))
        return SMX_ERR_INVALID_ARG;
    return cuda_status(smx::launch_kv_insert(*s, k, v, kidx, T, page_table, nullptr, n_fill, k_pool, v_pool,
                                             idx_pool, dev_status, true, (cudaStream_t)stream));
}

int smx_pack_q_e4m3(const float* q, uint8_t* q_e4m3, int64_t n, smx_stream_t stream) {
    if (!q || !q_e4m3 || n < 1) return SMX_ERR_INVALID_ARG;
    if (!aligned16(q) || (reinterpret_cast<uintptr_t>(q_e4m3) & 3u)) return SMX_ERR_INVALID_ARG;
    return cuda_status(smx::launch_pack_q(q, q_e4m3, n, (cudaStream_t)stream));
}

int smx_index_score(const smx_shape_t* s, const uint16_t* qidx_bf16, const uint8_t* idx_pool,
                    const int32_t* page_table, const int32_t* ctx_len, float* page_scores, int32_t* dev_status,
                    smx_stream_t stream) {
    int rc = check_shape(s);
    if (rc) return rc;
    if (!qidx_bf16 || !idx_pool || !page_table || !ctx_len || !page_scores) return SMX_ERR_INVALID_ARG;
    if (!aligned16(qidx_bf16) || !aligned32(idx_pool)) return SMX_ERR_INVALID_ARG;
    return cuda_status(smx::launch_index_scores(*s, qidx_bf16, idx_pool, page_table, ctx_len, page_scores,
                                                dev_status, (cudaStream_t)stream));
}

int smx_index_score_topk(const smx_shape_t* s, const uint16_t* qidx_bf16, const uint8_t* idx_pool,
                         const int32_t* page_table, const int32_t* ctx_len, float* page_scores,
                         int32_t* topk_pages, int32_t* topk_count, int32_t* dev_status, smx_stream_t stream) {
    int rc = check_shape(s);
    if (rc) return rc;
    if ((rc = check_page_blocks(s))) return rc;
    if (!qidx_bf16 || !idx_pool || !page_table || !ctx_len || !page_scores || !topk_pages || !topk_count)
        return SMX_ERR_INVALID_ARG;
    if (!aligned16(qidx_bf16) || !aligned32(idx_pool)) return SMX_ERR_INVALID_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    cudaError_t e = smx::launch_index_scores(*s, qidx_bf16, idx_pool, page_table, ctx_len, page_scores,
                                             dev_status, st);
    if (e != cudaSuccess) return SMX_ERR_CUDA;
    return cuda_status(smx::launch_topk(*s, page_scores, ctx_len, topk_pages, topk_count, st));
}

int smx_sparse_attn_split(const smx_shape_t* s, const void* q, const uint8_t* k_pool, const uint8_t* v_pool,
                          const int32_t* page_table, const int32_t* ctx_len, const int32_t* topk_pages,
                          const int32_t* topk_count, float* part_o, float* part_m, float* part_l,
                          int32_t* dev_status, smx_stream_t stream) {
    int rc = check_shape(s);
    if (rc) return rc;
    if ((rc = check_page_blocks(s))) return rc;
    if (!q || !k_pool || !v_pool || !page_table || !ctx_len || !topk_pages || !topk_count || !part_o ||
        !part_m || !part_l)
        return SMX_ERR_INVALID_ARG;
    if (!aligned16(k_pool) || !aligned16(v_pool) || (reinterpret_cast<uintptr_t>(q) & 3u) ||
        (reinterpret_cast<uintptr_t>(part_o) & 7u))
        return SMX_ERR_INVALID_ARG;
    return cuda_status(smx::launch_attn_split(*s, q, k_pool, v_pool, page_table, ctx_len, topk_pages, topk_count,
                                              part_o, part_m, part_l, dev_status, (cudaStream_t)stream));
}

int smx_sparse_attn_merge(const smx_shape_t* s, const float* part_o, const float* part_m, const float* part_l,
                          float* out, smx_stream_t stream) {
    int rc = check_shape(s);
    if (rc) return rc;
    if (!part_o || !part_m || !part_l || !out) return SMX_ERR_INVALID_ARG;
    return cuda_status(smx::launch_attn_merge(*s, part_o, part_m, part_l, out, (cudaStream_t)stream));
}

int smx_decode_step(const smx_shape_t* s, const float* q_f32, const uint16_t* q_bf16, const uint16_t* qidx_bf16,
                    const float* k_new, const float* v_new, const float* kidx_new, const int32_t* page_table,
                    const int32_t* ctx_len, uint8_t* k_pool, uint8_t* v_pool, uint8_t* idx_pool,
                    int32_t* topk_pages, int32_t* topk_count, float* out, void* workspace, size_t ws_bytes,
                    int32_t* dev_status, smx_stream_t stream) {
    const int rc = smx::check_step_args(s, q_f32, q_bf16, qidx_bf16, k_new, v_new, kidx_new, page_table, ctx_len,
                                        k_pool, v_pool, idx_pool, topk_pages, topk_count, out);
    if (rc) return rc;
    const bool rs = s->kv_format == SMX_KV_E4M3_ROWSCALE;
    const size_t need = layout(s, nullptr).bytes;
    if (!workspace || ws_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)))
        return SMX_ERR_WORKSPACE;
    const Workspace w = layout(s, workspace);
    if (smx::nvfp4_chain(*s)) {
        // NVFP4 pages: the standalone kernels in the step's order (the packed q goes to the
        // workspace's q tile region, which holds B x Q x Hq x 128 bytes)
        const cudaStream_t st = (cudaStream_t)stream;
        cudaError_t e = smx::launch_kv_insert(*s, k_new, v_new, kidx_new, s->Q, page_table, ctx_len, nullptr, k_pool,
                                              v_pool, idx_pool, dev_status, false, st);
        if (e == cudaSuccess && !rs) e = smx::launch_pack_q(q_f32, w.q_img, (int64_t)s->B * s->Q * s->Hq * 128, st);
        if (e == cudaSuccess)
            e = smx::launch_index_scores(*s, qidx_bf16, idx_pool, page_table, ctx_len, w.scores, dev_status, st);
        if (e == cudaSuccess) e = smx::launch_topk(*s, w.scores, ctx_len, topk_pages, topk_count, st);
        if (e == cudaSuccess)
            e = smx::launch_attn_split(*s, rs ? (const void*)q_bf16 : (const void*)w.q_img, k_pool, v_pool, page_table,
                                       ctx_len, topk_pages, topk_count, w.part_o, w.part_m, w.part_l, dev_status, st);
        if (e == cudaSuccess) e = smx::launch_attn_merge(*s, w.part_o, w.part_m, w.part_l, out, st);
        return cuda_status(e);
    }
    smx::StepIO io = {};
    io.q_f32 = rs ? nullptr : q_f32;
    io.q_bf16 = rs ? q_bf16 : nullptr;
    io.qidx = qidx_bf16;
    io.k_new = k_new; io.v_new = v_new; io.kidx_new = kidx_new;
    io.page_table = page_table; io.ctx_len = ctx_len;
    io.idx_pool = idx_pool; io.k_pool = k_pool; io.v_pool = v_pool;
    io.topk_out = topk_pages; io.count_out = topk_count; io.out = out; io.status = dev_status;
    io.counters = w.counters; io.scores = w.scores;
    io.part_o = w.part_o; io.part_m = w.part_m; io.part_l = w.part_l; io.q_img = w.q_img;
    return cuda_status(smx::launch_decode_step(*s, io, (cudaStream_t)stream));
}

int smx_decode_step_reuse(const smx_shape_t* s, const float* q_f32, const uint16_t* q_bf16, const float* k_new,
                          const float* v_new, const int32_t* page_table, const int32_t* ctx_len, uint8_t* k_pool,
                          uint8_t* v_pool, const int32_t* topk_pages, const int32_t* topk_count, float* out,
                          void* workspace, size_t ws_bytes, int32_t* dev_status, smx_stream_t stream) {
    int rc = check_shape(s);
    if (rc) return rc;
    const bool rs = s->kv_format == SMX_KV_E4M3_ROWSCALE;
    if ((rs ? (const void*)q_bf16 : (const void*)q_f32) == nullptr) return SMX_ERR_INVALID_ARG;
    if (!k_new || !v_new || !page_table || !ctx_len || !k_pool || !v_pool || !topk_pages || !topk_count || !out)
        return SMX_ERR_INVALID_ARG;
    if (!rs && !aligned16(q_f32)) return SMX_ERR_INVALID_ARG;
    if (rs && (reinterpret_cast<uintptr_t>(q_bf16) & 3u)) return SMX_ERR_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_pool) || !aligned16(v_pool)) return SMX_ERR_INVALID_ARG;
    const size_t need = layout(s, nullptr).bytes;
    if (!workspace || ws_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)))
        return SMX_ERR_WORKSPACE;
    const Workspace w = layout(s, workspace);
    if (smx::nvfp4_chain(*s)) {
        // NVFP4 K/V: insert (K and V rows only), pack q, the split over the given selection, merge
        const cudaStream_t st = (cudaStream_t)stream;
        cudaError_t e = smx::launch_kv_insert(*s, k_new, v_new, nullptr, s->Q, page_table, ctx_len, nullptr, k_pool,
                                              v_pool, nullptr, dev_status, false, st);
        if (e == cudaSuccess && !rs) e = smx::launch_pack_q(q_f32, w.q_img, (int64_t)s->B * s->Q * s->Hq * 128, st);
        if (e == cudaSuccess)
            e = smx::launch_attn_split(*s, rs ? (const void*)q_bf16 : (const void*)w.q_img, k_pool, v_pool, page_table,
                                       ctx_len, topk_pages, topk_count, w.part_o, w.part_m, w.part_l, dev_status, st);
        if (e == cudaSuccess) e = smx::launch_attn_merge(*s, w.part_o, w.part_m, w.part_l, out, st);
        return cuda_status(e);
    }
    smx::StepIO io = {};
    io.q_f32 = rs ? nullptr : q_f32;
    io.q_bf16 = rs ? q_bf16 : nullptr;
    io.k_new = k_new; io.v_new = v_new;
    io.page_table = page_table; io.ctx_len = ctx_len;
    io.k_pool = k_pool; io.v_pool = v_pool;
    io.topk_in = topk_pages; io.count_in = topk_count; io.out = out; io.status = dev_status;
    io.counters = w.counters; io.scores = w.scores;
    io.part_o = w.part_o; io.part_m = w.part_m; io.part_l = w.part_l; io.q_img = w.q_img;
    return cuda_status(smx::launch_decode_step(*s, io, (cudaStream_t)stream, true));
}

int smx_decode_step_launches(const smx_shape_t* s) {
    if (check_shape(s) != SMX_OK) return 0;
    if (smx::nvfp4_chain(*s)) return s->kv_format == SMX_KV_E4M3_ROWSCALE ? 5 : 6;
    return 1;
}

int smx_decode_step_tensor_cores(const smx_shape_t* s) {
    const int rc = check_shape(s);
    if (rc) return rc;
    if (smx::nvfp4_chain(*s)) return 0;
    return smx::decode_step_uses_tc(*s) ? 1 : 0;
}

int smx_suggest_num_splits(const smx_shape_t* s) {
    if (s == nullptr) return 0;
    smx_shape_t t = *s;
    t.num_splits = 1;
    if (check_shape(&t) != SMX_OK) return 0;
    return smx::suggest_num_splits(t);
}

uint64_t smx_set_wait_limit_ns(uint64_t ns) {
    const uint64_t before = smx::wait_limit_ns();
    smx::g_wait_limit_ns.store(ns, std::memory_order_relaxed);
    return before;
}

const char* smx_status_string(int status) {
    switch (status) {
        case SMX_OK: return "ok";
        case SMX_ERR_INVALID_ARG: return "invalid argument";
        case SMX_ERR_UNSUPPORTED: return "unsupported shape or format";
        case SMX_ERR_CUDA: return "CUDA launch error";
        case SMX_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
        default: return "unknown status";
    }
}

}  // extern "C"

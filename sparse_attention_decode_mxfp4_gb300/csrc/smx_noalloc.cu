// smx_noalloc.cu -- smx_decode_step_noalloc: the decode step with its scratch held in a static
// device array of SMX_NOALLOC_SCRATCH_BYTES, so that no call allocates device memory.
//
// The array is a module-scope device variable: the driver places it when the module is loaded,
// and the first call on each device looks up its address once. Later calls launch the step into
// it (plus a memset of the step counters when a shape needs more of them than the previous call
// left zero). All calls on one device share the array.
#include <mutex>

#include "smx_internal.h"

static __device__ __align__(256) unsigned char smx_noalloc_scratch[SMX_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
void* g_scratch[kMaxDevices] = {};
size_t g_zero_prefix[kMaxDevices] = {};   // leading bytes of the array known to be zero

// Address of the scratch array on the current device, with its first counter_bytes zero. The first
// call on a device resolves it (cudaGetSymbolAddress, which also loads the module there if it is
// not loaded yet) and clears the counters on `st`. The step leaves its counters zero but may write
// its other data right after them, so a later call whose counters reach past the zero prefix the
// previous call left clears them again (one memset on `st`).
int scratch_on_current_device(void** out, size_t counter_bytes, cudaStream_t st) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SMX_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return SMX_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_setup_mu);
    if (g_scratch[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, smx_noalloc_scratch) != cudaSuccess || p == nullptr) {
            (void)cudaGetLastError();
            return SMX_ERR_CUDA;
        }
        g_scratch[dev] = p;
        g_zero_prefix[dev] = 0;
    }
    if (counter_bytes > g_zero_prefix[dev] && cudaMemsetAsync(g_scratch[dev], 0, counter_bytes, st) != cudaSuccess)
        return SMX_ERR_CUDA;
    g_zero_prefix[dev] = counter_bytes;
    *out = g_scratch[dev];
    return SMX_OK;
}

}  // namespace

extern "C" int smx_decode_step_noalloc(const smx_shape_t* s, const float* q_f32, const uint16_t* q_bf16,
                                       const uint16_t* qidx_bf16, const float* k_new, const float* v_new,
                                       const float* kidx_new, const int32_t* page_table, const int32_t* ctx_len,
                                       uint8_t* k_pool, uint8_t* v_pool, uint8_t* idx_pool, int32_t* topk_pages,
                                       int32_t* topk_count, float* out, int32_t* dev_status, smx_stream_t stream) {
    const size_t need = smx_workspace_bytes(s);
    if (need == 0) {
        // an invalid shape: smx_decode_step checks the shape before anything else and returns
        // its status without touching the device
        return smx_decode_step(s, q_f32, q_bf16, qidx_bf16, k_new, v_new, kidx_new, page_table, ctx_len, k_pool,
                               v_pool, idx_pool, topk_pages, topk_count, out, nullptr, 0, dev_status, stream);
    }
    if (need > (size_t)SMX_NOALLOC_SCRATCH_BYTES) return SMX_ERR_WORKSPACE;
    void* scratch = nullptr;
    // the step's counters open the workspace layout
    const int rc = scratch_on_current_device(&scratch, smx::workspace_counter_bytes(*s), (cudaStream_t)stream);
    if (rc != SMX_OK) return rc;
    return smx_decode_step(s, q_f32, q_bf16, qidx_bf16, k_new, v_new, kidx_new, page_table, ctx_len, k_pool, v_pool,
                           idx_pool, topk_pages, topk_count, out, scratch, (size_t)SMX_NOALLOC_SCRATCH_BYTES,
                           dev_status, stream);
}

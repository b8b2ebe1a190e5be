// smx_noalloc.cu -- smx_decode_step_noalloc: the decode step with its scratch held in a static
// device array of SMX_NOALLOC_SCRATCH_BYTES, so that no call allocates device memory.
//
// The array is a module-scope device variable: the driver places it when the module is loaded,
// and the first call on each device looks up its address once. Every call then clears the step
// counters at the head of the array (one memset of a few hundred bytes on the caller's stream)
// and launches the step into it. All calls on one device share the array.
#include <mutex>

#include "smx_internal.h"

static __device__ __align__(256) unsigned char smx_noalloc_scratch[SMX_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
void* g_scratch[kMaxDevices] = {};

// Address of the scratch array on the current device. The first call on a device resolves it
// (cudaGetSymbolAddress, which also loads the module there if it is not loaded yet); host code
// only ever passes this address to kernels, never the array's host-side name.
int scratch_on_current_device(void** out) {
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
    }
    *out = g_scratch[dev];
    return SMX_OK;
}

}  // namespace

extern "C" int smx_decode_step_noalloc(const smx_shape_t* s, const float* q_f32, const uint16_t* q_bf16,
                                       const uint16_t* qidx_bf16, const float* k_new, const float* v_new,
                                       const float* kidx_new, const int32_t* page_table, const int32_t* ctx_len,
                                       uint8_t* k_pool, uint8_t* v_pool, uint8_t* idx_pool, int32_t* topk_pages,
                                       int32_t* topk_count, float* out, int32_t* dev_status, smx_stream_t stream) {
    // the same argument checks as smx_decode_step, before the device is touched
    int rc = smx::check_step_args(s, q_f32, q_bf16, qidx_bf16, k_new, v_new, kidx_new, page_table, ctx_len, k_pool,
                                  v_pool, idx_pool, topk_pages, topk_count, out);
    if (rc != SMX_OK) return rc;
    if (smx_workspace_bytes(s) > (size_t)SMX_NOALLOC_SCRATCH_BYTES) return SMX_ERR_WORKSPACE;
    void* scratch = nullptr;
    if ((rc = scratch_on_current_device(&scratch)) != SMX_OK) return rc;
    // The step's counters open the workspace layout and must be zero when it starts. A step leaves
    // them zero, but a call of another shape may have written other data over that range since,
    // so every call clears them, on the same stream, just before the launch.
    if (cudaMemsetAsync(scratch, 0, smx::workspace_counter_bytes(*s), (cudaStream_t)stream) != cudaSuccess) {
        (void)cudaGetLastError();
        return SMX_ERR_CUDA;
    }
    return smx_decode_step(s, q_f32, q_bf16, qidx_bf16, k_new, v_new, kidx_new, page_table, ctx_len, k_pool, v_pool,
                           idx_pool, topk_pages, topk_count, out, scratch, (size_t)SMX_NOALLOC_SCRATCH_BYTES,
                           dev_status, stream);
}

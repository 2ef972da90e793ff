// rad_attn_paged_noalloc: the same op as rad_attn_paged for callers that
// cannot allocate device memory, with the split-combine scratch held in a
// fixed, library-owned device array instead of a caller-provided workspace.
//
// Who needs it: a runtime that plans all of its device memory once, at load
// time (an arena owned by its own allocator, or by a framework's caching
// allocator), and code that is handed only the tensors of the call (a plugin
// given inputs and outputs but no scratch buffer).  Neither may call cudaMalloc
// per call: it would fail once the arena has reserved the device, or break the
// one-time memory plan.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "rad_attn.h"

namespace {

constexpr int kMaxDevices = 64;

// The scratch every call of this entry point shares.  Each GPU that loads the
// library holds RAD_NOALLOC_SCRATCH_BYTES of it until the process exits.  In
// host code `g_noalloc_scratch` names a host-side stand-in, never a device
// address: the device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[RAD_NOALLOC_SCRATCH_BYTES];

using CtxGetCurrentFn = CUresult (*)(CUcontext*);

std::mutex g_setup_mutex;
CtxGetCurrentFn g_ctx_get_current = nullptr;
// Per device: the context the address was looked up in, and the address.  A
// device reset (or a released and re-created primary context) loads the
// module again, possibly elsewhere, so a changed context means a new lookup.
CUcontext g_scratch_ctx[kMaxDevices] = {};
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array in the current device's current
// context, looked up (with that device current) the first time and again
// whenever the context has changed.  Returns RAD_OK or RAD_E_CUDA.
int scratch_address(void** addr) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return RAD_E_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return RAD_E_DEVICE;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (g_ctx_get_current == nullptr) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || fn == nullptr)
            return RAD_E_CUDA;
        g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(fn);
    }
    // no current context yet (the runtime has not touched the device): the
    // lookup below makes the device's primary context current
    CUcontext ctx = nullptr;
    if (g_ctx_get_current(&ctx) != CUDA_SUCCESS) return RAD_E_CUDA;
    if (ctx == nullptr || g_scratch_addr[dev] == nullptr || g_scratch_ctx[dev] != ctx) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return RAD_E_CUDA;
        if (g_ctx_get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return RAD_E_CUDA;
        g_scratch_addr[dev] = p;
        g_scratch_ctx[dev] = ctx;
    }
    *addr = g_scratch_addr[dev];
    return RAD_OK;
}

}  // namespace

extern "C" int rad_attn_paged_noalloc(const void* q, const void* k_pool, const void* v_pool,
                                      const int32_t* page_table, const int32_t* seq_lens, int32_t groups,
                                      int32_t rows, int32_t n_head, int32_t n_head_kv, int32_t head_dim,
                                      int32_t page_size, int32_t pages_per_seq, int32_t num_pages,
                                      float scale, int32_t kv_dtype, const float* k_scales,
                                      const float* v_scales, void* out, uint32_t* err_word,
                                      rad_stream_t stream) {
    // Shapes the workspace entry point refuses are refused the same way (a zero
    // workspace need is also what it reports for them).
    const size_t need = rad_attn_paged_workspace_bytes(groups, rows, n_head, n_head_kv, head_dim, page_size,
                                                       pages_per_seq, kv_dtype);
    if (need > (size_t)RAD_NOALLOC_SCRATCH_BYTES) return RAD_E_WORKSPACE;
    void* scratch = nullptr;
    if (need > 0) {
        const int rc = scratch_address(&scratch);
        if (rc != RAD_OK) return rc;
    }
    // The scratch needs no initialisation: the combine reads only partials
    // written earlier in the same call.
    return rad_attn_paged(q, k_pool, v_pool, page_table, seq_lens, groups, rows, n_head, n_head_kv, head_dim,
                          page_size, pages_per_seq, num_pages, scale, kv_dtype, k_scales, v_scales, out, scratch,
                          need > 0 ? (size_t)RAD_NOALLOC_SCRATCH_BYTES : 0, err_word, stream);
}

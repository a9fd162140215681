// spec_attn_run_noalloc: the same attention call as spec_attn_run, for
// callers that cannot allocate device memory.
//
// spec_attn_run needs a caller-provided workspace for the split-KV partials
// (and the device-status word).  Some callers have no way to provide one:
// code that runs where cudaMalloc is off limits (inside a host callback or
// a custom allocator's own hook, under a memory pool that is already full or
// locked by a framework, or in a plugin that is handed only its input and
// output buffers).  For them this entry point takes its scratch from a
// fixed-size array that lives in the library's own device memory.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds its 32 MiB until the process exits, and every call on a
// device shares the same array.  Calls that may overlap on the GPU (two
// streams, or two host threads) race on it and must be serialised by the
// caller.  The array keeps whatever the last call left; the only part that
// must start at zero (the device-status word) is cleared by every call.
// Plans that need more scratch than the array holds are rejected with
// SPEC_ATTN_E_WORKSPACE_TOO_SMALL.
//
// Host code can not use the array's name as a device address, so the first
// call on each device looks the address up (cudaGetSymbolAddress, with that
// device current) and caches it with the unique id of the context it belongs
// to; make that first call before any stream capture begins.  A later call
// whose current context has another id (the device was reset, and its
// primary context created anew) looks the address up again.
//
// Each call clears the status word only after its host checks have passed,
// so a rejected call writes nothing.  spec_attn_noalloc_check_device_status
// reads (and clears) the word the last call on the device left.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/spec_attn.h"
#include "spec_attn_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = SPEC_ATTN_NOALLOC_SCRATCH_BYTES;  // 32 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_setup_mutex;
void* g_scratch_addr[kMaxDevices] = {};
unsigned long long g_scratch_ctx[kMaxDevices] = {};   // id of the context the address belongs to

template <class F>
F driver_fn(const char* name, int version) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    const bool ok = cudaGetDriverEntryPointByVersion(name, &ptr, version, cudaEnableDefault, &q) == cudaSuccess &&
                    q == cudaDriverEntryPointSuccess;
    return ok ? reinterpret_cast<F>(ptr) : nullptr;
}

// Unique id of this thread's current context, 0 when none is current yet.
unsigned long long current_context_id() {
    static const PFN_cuCtxGetCurrent_v4000 get_current = driver_fn<PFN_cuCtxGetCurrent_v4000>("cuCtxGetCurrent", 4000);
    static const PFN_cuCtxGetId_v12000 get_id = driver_fn<PFN_cuCtxGetId_v12000>("cuCtxGetId", 12000);
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current && get_id && get_current(&ctx) == CUDA_SUCCESS && ctx && get_id(ctx, &id) == CUDA_SUCCESS)
        return id;
    return 0;
}

// The array's address on the current device (looked up again whenever the
// current context is not the one the cached address came from); nullptr on
// a CUDA error.  Called with g_setup_mutex held.
void* scratch_for(int dev) {
    const unsigned long long id = current_context_id();
    if (!g_scratch_addr[dev] || id == 0 || id != g_scratch_ctx[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return nullptr;
        g_scratch_addr[dev] = ptr;
        g_scratch_ctx[dev] = current_context_id();   // the lookup made the context current
    }
    return g_scratch_addr[dev];
}

}  // namespace

extern "C" int spec_attn_run_noalloc(const spec_attn_plan* plan, const void* q, const void* k_pool,
                                     const void* v_pool, const void* k_scales, const void* v_scales,
                                     float k_gscale, float v_gscale, const int32_t* block_table,
                                     const int32_t* seq_lens, const int32_t* q_indptr, void* o,
                                     float* lse, spec_attn_stream_t stream) {
    if (!plan) return SPEC_ATTN_E_INVALID_ARG;
    spec_attn_plan_info info;
    int st = spec_attn_plan_get_info(plan, &info);
    if (st != SPEC_ATTN_OK) return st;
    if (info.workspace_bytes > kNoAllocScratchBytes) return SPEC_ATTN_E_WORKSPACE_TOO_SMALL;

    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SPEC_ATTN_E_CUDA;
    void* scratch = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_setup_mutex);
        scratch = scratch_for(dev);
    }
    if (!scratch) return SPEC_ATTN_E_CUDA;
    // the device-status word at the head of the scratch starts each call at zero
    return spec_attn::run_clearing_status(plan, q, k_pool, v_pool, k_scales, v_scales, k_gscale, v_gscale,
                                          block_table, seq_lens, q_indptr, o, lse, scratch, kNoAllocScratchBytes,
                                          stream);
}

extern "C" int spec_attn_noalloc_check_device_status(spec_attn_stream_t stream, uint32_t* bits) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SPEC_ATTN_E_CUDA;
    void* scratch = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_setup_mutex);
        if (!g_scratch_addr[dev]) {   // no call has run on this device: nothing to report
            if (bits) *bits = 0;
            return SPEC_ATTN_OK;
        }
        scratch = scratch_for(dev);
    }
    if (!scratch) return SPEC_ATTN_E_CUDA;
    return spec_attn_check_device_status(scratch, stream, bits);
}

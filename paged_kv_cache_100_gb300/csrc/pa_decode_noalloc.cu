// pa_decode_static_scratch: paged decode attention for callers that cannot
// allocate device memory.
//
// pa_decode needs caller-provided scratch (the split-K partials) whenever a
// context spans more than one partition.  Some callers have no way to provide
// it: their device memory is entirely reserved up front by another allocator
// (so a cudaMalloc would fail or break that allocator's accounting), or they
// run in a loop where the implicit device synchronisation of cudaMalloc /
// cudaFree is not acceptable, or they sit behind an interface that hands them
// only the inputs and outputs.  This entry point serves them: its scratch is a
// fixed-size array in device global memory that belongs to this library, so a
// call allocates nothing.  The array exists on every device that loads the
// library and stays there until the process exits.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "pa_internal.h"

namespace pa {
namespace {

// The library's own scratch for pa_decode_static_scratch (PA_STATIC_SCRATCH_BYTES).
static __device__ __align__(256) unsigned char g_static_scratch[PA_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
struct ScratchEntry {
    unsigned long long context_id;   // context the address belongs to (0: none cached)
    void *ptr;
};
ScratchEntry g_scratch[kMaxDevices] = {};

// Process-unique identifier of the calling thread's current CUDA context (a
// context made after cudaDeviceReset gets a new one), or 0 when there is no
// current context or it cannot be read.
unsigned long long current_context_id() {
    static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current == nullptr || get_id == nullptr || get_current(&ctx) != CUDA_SUCCESS ||
        ctx == nullptr || get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

// Device address of g_static_scratch on the current device.  In host code the
// array's name is only a host-side stand-in, so the address is looked up with
// the device current (cudaGetSymbolAddress) and cached per device together with
// the context it belongs to: after a cudaDeviceReset the module is loaded again
// in a new context, the cached address is stale, and it is looked up again.
pa_status scratch_address(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_failure(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return PA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    const unsigned long long ctx = current_context_id();
    if (ctx != 0 && g_scratch[dev].context_id == ctx) {
        *out = g_scratch[dev].ptr;
        return PA_OK;
    }
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess || p == nullptr)
        return cuda_failure(e == cudaSuccess ? cudaErrorInvalidSymbol : e, "cudaGetSymbolAddress");
    // the lookup made the device's context current if it was not yet
    g_scratch[dev].context_id = current_context_id();
    g_scratch[dev].ptr = p;
    *out = p;
    return PA_OK;
}

}  // namespace
}  // namespace pa

using namespace pa;

extern "C" pa_status pa_decode_static_scratch(void *out, const void *query, const void *key_cache,
                                              const void *value_cache, const int32_t *block_tables,
                                              const int32_t *context_lens, int num_seqs,
                                              int num_q_heads, int num_kv_heads, int head_dim,
                                              int block_size, int max_blocks_per_seq,
                                              int num_blocks, float scale, pa_dtype dtype,
                                              int partition_size, int32_t *device_status,
                                              void *stream) {
    const size_t need = pa_decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                                  max_blocks_per_seq, block_size, partition_size,
                                                  dtype);
    if (need == (size_t)-1 || need > (size_t)PA_STATIC_SCRATCH_BYTES) {
        // pa_decode's own checks decide these calls, so that every argument error
        // is reported as pa_decode reports it: given no workspace, it returns
        // its error for invalid arguments and PA_ERR_WORKSPACE for valid ones
        // that need scratch, before anything is enqueued.
        return pa_decode(out, query, key_cache, value_cache, block_tables, context_lens, num_seqs,
                         num_q_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq,
                         num_blocks, scale, dtype, partition_size, nullptr, 0, device_status,
                         stream);
    }
    void *scratch = nullptr;
    if (need > 0) {
        pa_status s = scratch_address(&scratch);
        if (s != PA_OK) return s;
    }
    // The partials are written before they are read within one call, so no part
    // of the array has to start at zero.
    return pa_decode(out, query, key_cache, value_cache, block_tables, context_lens, num_seqs,
                     num_q_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq,
                     num_blocks, scale, dtype, partition_size, scratch,
                     need > 0 ? (size_t)PA_STATIC_SCRATCH_BYTES : 0, device_status, stream);
}

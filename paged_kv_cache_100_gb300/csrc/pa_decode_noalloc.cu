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
#include <cuda_runtime.h>

#include <mutex>

#include "pa_internal.h"

namespace pa {
namespace {

// The library's own scratch for pa_decode_static_scratch (PA_STATIC_SCRATCH_BYTES).
static __device__ __align__(256) unsigned char g_static_scratch[PA_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of g_static_scratch on the current device.  In host code the
// array's name is only a host-side stand-in, so the address is looked up once
// per device, with that device current, and cached.
pa_status scratch_address(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_failure(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return PA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_ptr[dev] == nullptr) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess || p == nullptr)
            return cuda_failure(e == cudaSuccess ? cudaErrorInvalidSymbol : e, "cudaGetSymbolAddress");
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
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
    if (need == (size_t)-1) return PA_ERR_INVALID_ARG;
    if (need > (size_t)PA_STATIC_SCRATCH_BYTES) return PA_ERR_WORKSPACE;
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

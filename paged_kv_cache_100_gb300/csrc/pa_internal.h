// Host-side declarations shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "pagedkv.h"

namespace pa {

constexpr int kBlockSize = 16;            // tokens per physical block
constexpr int kMaxPartition = 16384;      // largest partition (its table slice lives in smem)

// Adds n to the process-wide launch counter returned by pa_launch_count().
void count_launches(uint64_t n);

// Records the message of a failed CUDA call for pa_last_error() and returns PA_ERR_CUDA.
pa_status cuda_failure(cudaError_t err, const char *where);

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Launches a kernel with programmatic stream serialisation: it may be scheduled
// while the previous kernel in the stream is still running.  Every kernel of
// this library starts with griddepcontrol.wait (nothing before it reads global
// memory), so ordering with earlier work is kept; what overlaps is only the
// launch and CTA set-up of one kernel with the tail of the one before.  The
// one exception is the suffix decode of pa_decode_shared_prefix, which follows
// the prefix kernel and runs beside it (DecodeArgs::defer_wait).
template <typename... KArgs, typename... Args>
cudaError_t launch_chained(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                           cudaStream_t stream, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Shared prefix of a decode batch on the tensor cores (pa_prefill.cu): split-K
// partials (max, sum, unnormalised output) of every (sequence, query head) row
// against each chunk of the prefix blocks, written to partial index = chunk.
// staged: key_cache / value_cache are a bf16 copy of the prefix blocks' E4M3
// code values, block j of the prefix at index j (num_blocks = prefix_blocks),
// with per-KV-head scales k_scales / v_scales (else both nullptr).
bool prefix_tc_supported(int head_dim, int num_q_heads, int num_kv_heads);
int prefix_tc_chunk_blocks(int num_seqs, int num_q_heads, int num_kv_heads, int prefix_blocks,
                           int sm_count);
pa_status launch_prefix_tc(const void *query, const void *key_cache, const void *value_cache,
                           const int32_t *block_tables, const int32_t *context_lens, int num_seqs,
                           int num_q_heads, int num_kv_heads, int max_blocks, int num_blocks,
                           float scale_log2, int prefix_blocks, int chunk_blocks, int chunks,
                           float *part_o, float2 *part_ml, int max_parts, bool staged,
                           const float *k_scales, const float *v_scales, int32_t *status,
                           cudaStream_t stream);

}  // namespace pa

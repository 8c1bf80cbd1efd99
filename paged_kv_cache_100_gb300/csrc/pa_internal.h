// Host-side declarations shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "pagedkv.h"

namespace pa {

constexpr int kBlockSize = 16;            // tokens per physical block
constexpr int kDefaultPartition = 512;    // tokens per split-K partition by default
constexpr int kMaxPartition = 16384;      // largest partition (its table slice lives in smem)

// Adds n to the process-wide launch counter returned by pa_launch_count().
void count_launches(uint64_t n);

// Records the message of a failed CUDA call for pa_last_error() and returns PA_ERR_CUDA.
pa_status cuda_failure(cudaError_t err, const char *where);

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace pa

// Cache write and copy-on-write block copy, plus the library's small ABI helpers.
//
// Cache write ("PagedAttention por dentro", section "La tabla de páginas
// (block table)"): the new token of a sequence goes into the free slot of its
// last block, or into the first slot of a freshly appended block; the host
// block manager turns that rule into one slot per token, and this kernel
// scatters each token's K/V rows there.
//
// Block copy (same page, section "Copy-on-write para sampling paralelo"): when
// a sequence is about to modify a block it shares, only that block is copied.
//
// Both are pure bandwidth kernels: 16-byte vector loads and stores, one thread
// per 16-byte chunk, index checks before every access.  They are launched
// chained to the previous kernel of the stream (programmatic dependent launch)
// and wait for it before touching memory.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdio>
#include <cstring>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

namespace {

std::atomic<uint64_t> g_launches{0};
thread_local char g_last_error[256] = "";

// One thread per 16-byte chunk of one (token, KV head) row of K and of V.
__global__ void __launch_bounds__(256)
pa_cache_write_kernel(uint4 *__restrict__ kc, uint4 *__restrict__ vc,
                      const uint4 *__restrict__ key, const uint4 *__restrict__ value,
                      const int64_t *__restrict__ slot_mapping, int num_tokens, int num_kv_heads,
                      int chunks_per_row, int num_blocks, int32_t *status) {
    grid_dependency_wait();
    grid_dependents_launch();
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t per_token = (int64_t)num_kv_heads * chunks_per_row;
    if (idx >= (int64_t)num_tokens * per_token) return;
    const int64_t i = idx / per_token;
    const int64_t rem = idx - i * per_token;          // kvh * chunks_per_row + chunk
    const int64_t slot = slot_mapping[i];
    if (slot < 0) return;
    if (slot >= (int64_t)num_blocks * kBlockSize) {
        if (rem == 0) report(status, PA_DEV_BAD_SLOT);
        return;
    }
    const int64_t blk = slot / kBlockSize;
    const int64_t off = slot - blk * kBlockSize;
    const int64_t kvh = rem / chunks_per_row;
    const int64_t ch = rem - kvh * chunks_per_row;
    const int64_t dst = ((blk * num_kv_heads + kvh) * kBlockSize + off) * chunks_per_row + ch;
    kc[dst] = key[idx];
    vc[dst] = value[idx];
}

// Quantising cache write into FP8 pools: one thread per 16 codes (16 bytes) of
// one (token, KV head) row of K and of V.  Each element x of the bf16 row
// becomes the E4M3 code of the float32 quotient x / scale[kv_head] (IEEE
// division, round to nearest even, saturating at +-448).
__global__ void __launch_bounds__(256)
pa_cache_write_fp8_kernel(uint4 *__restrict__ kc, uint4 *__restrict__ vc,
                          const uint4 *__restrict__ key, const uint4 *__restrict__ value,
                          const int64_t *__restrict__ slot_mapping,
                          const float *__restrict__ k_scales, const float *__restrict__ v_scales,
                          int num_tokens, int num_kv_heads, int chunks_per_row, int num_blocks,
                          int32_t *status) {
    grid_dependency_wait();
    grid_dependents_launch();
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t per_token = (int64_t)num_kv_heads * chunks_per_row;
    if (idx >= (int64_t)num_tokens * per_token) return;
    const int64_t i = idx / per_token;
    const int64_t rem = idx - i * per_token;
    const int64_t slot = slot_mapping[i];
    if (slot < 0) return;
    if (slot >= (int64_t)num_blocks * kBlockSize) {
        if (rem == 0) report(status, PA_DEV_BAD_SLOT);
        return;
    }
    const int64_t blk = slot / kBlockSize;
    const int64_t off = slot - blk * kBlockSize;
    const int64_t kvh = rem / chunks_per_row;
    const int64_t ch = rem - kvh * chunks_per_row;
    const int64_t dst = ((blk * num_kv_heads + kvh) * kBlockSize + off) * chunks_per_row + ch;
    const float ks = k_scales[kvh], vs = v_scales[kvh];
    // 16 bf16 inputs (two uint4) per 16 output codes
    const uint4 *ksrc = key + 2 * idx;
    const uint4 *vsrc = value + 2 * idx;
    const uint4 k0 = ksrc[0], k1 = ksrc[1], v0 = vsrc[0], v1 = vsrc[1];
    const uint32_t kw[8] = {k0.x, k0.y, k0.z, k0.w, k1.x, k1.y, k1.z, k1.w};
    const uint32_t vw[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    uint32_t ko[4], vo[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t klo = f32x2_to_e4m3x2(__fdiv_rn(bf16lo(kw[2 * j]), ks),
                                             __fdiv_rn(bf16hi(kw[2 * j]), ks));
        const uint32_t khi = f32x2_to_e4m3x2(__fdiv_rn(bf16lo(kw[2 * j + 1]), ks),
                                             __fdiv_rn(bf16hi(kw[2 * j + 1]), ks));
        const uint32_t vlo = f32x2_to_e4m3x2(__fdiv_rn(bf16lo(vw[2 * j]), vs),
                                             __fdiv_rn(bf16hi(vw[2 * j]), vs));
        const uint32_t vhi = f32x2_to_e4m3x2(__fdiv_rn(bf16lo(vw[2 * j + 1]), vs),
                                             __fdiv_rn(bf16hi(vw[2 * j + 1]), vs));
        ko[j] = klo | (khi << 16);
        vo[j] = vlo | (vhi << 16);
    }
    kc[dst] = make_uint4(ko[0], ko[1], ko[2], ko[3]);
    vc[dst] = make_uint4(vo[0], vo[1], vo[2], vo[3]);
}

// grid.x = pair, grid.y = slice of the block; every thread copies up to
// kChunksPerThread 16-byte chunks of K and of V.
//
// The pairs of one list are independent copies into fresh blocks (every
// copy-on-write takes its destination from the pool), so they run
// concurrently.  A pair is "live" when both indices are in the pool and
// src != dst; a live pair whose dst is the src or the dst of another live
// pair would race with it and is skipped and flagged.  Each CTA checks its
// own pair against the whole list (num_pairs reads of 8 bytes, spread over the
// CTA's threads).
constexpr int kCopyThreads = 256;
constexpr int kChunksPerThread = 4;

__global__ void __launch_bounds__(kCopyThreads)
pa_block_copy_kernel(uint4 *__restrict__ kc, uint4 *__restrict__ vc,
                     const int32_t *__restrict__ src_dst, int num_pairs, int64_t chunks_per_block,
                     int num_blocks, int32_t *status) {
    grid_dependency_wait();
    grid_dependents_launch();
    const int32_t src = src_dst[2 * blockIdx.x];
    const int32_t dst = src_dst[2 * blockIdx.x + 1];
    if ((unsigned)src >= (unsigned)num_blocks || (unsigned)dst >= (unsigned)num_blocks) {
        if (blockIdx.y == 0 && threadIdx.x == 0) report(status, PA_DEV_BAD_COPY_PAIR);
        return;
    }
    if (src == dst) return;
    bool clash = false;
    for (int q = threadIdx.x; q < num_pairs; q += kCopyThreads) {
        if (q == (int)blockIdx.x) continue;
        const int2 o = reinterpret_cast<const int2 *>(src_dst)[q];
        const bool live = (unsigned)o.x < (unsigned)num_blocks &&
                          (unsigned)o.y < (unsigned)num_blocks && o.x != o.y;
        clash |= live && (o.x == dst || o.y == dst);
    }
    if (__syncthreads_or(clash)) {
        if (blockIdx.y == 0 && threadIdx.x == 0) report(status, PA_DEV_BAD_COPY_PAIR);
        return;
    }
    const int64_t first = (int64_t)blockIdx.y * kCopyThreads * kChunksPerThread + threadIdx.x;
    const uint4 *ks = kc + (int64_t)src * chunks_per_block;
    const uint4 *vs = vc + (int64_t)src * chunks_per_block;
    uint4 *kd = kc + (int64_t)dst * chunks_per_block;
    uint4 *vd = vc + (int64_t)dst * chunks_per_block;
    uint4 kb[kChunksPerThread], vb[kChunksPerThread];
#pragma unroll
    for (int u = 0; u < kChunksPerThread; ++u) {
        const int64_t c = first + (int64_t)u * kCopyThreads;
        if (c < chunks_per_block) {
            kb[u] = ks[c];
            vb[u] = vs[c];
        }
    }
#pragma unroll
    for (int u = 0; u < kChunksPerThread; ++u) {
        const int64_t c = first + (int64_t)u * kCopyThreads;
        if (c < chunks_per_block) {
            kd[c] = kb[u];
            vd[c] = vb[u];
        }
    }
}

// Swap between the pools and a staging buffer laid out [id][K, V][block
// bytes]: CTA (i, slice, kv) moves one slice of block_ids[i]'s K or V tile.
// The staging side may be page-locked host memory reached over the
// CPU-GPU link, so each thread keeps kChunksPerThread 16-byte loads in
// flight before it stores.
template <bool kOut>
__global__ void __launch_bounds__(kCopyThreads)
pa_swap_kernel(uint4 *__restrict__ kc, uint4 *__restrict__ vc, uint4 *__restrict__ stage,
               const int32_t *__restrict__ block_ids, int64_t chunks_per_block, int num_blocks,
               int32_t *status) {
    grid_dependency_wait();
    grid_dependents_launch();
    const int32_t id = block_ids[blockIdx.x];
    if ((unsigned)id >= (unsigned)num_blocks) {
        if (blockIdx.y == 0 && blockIdx.z == 0 && threadIdx.x == 0)
            report(status, PA_DEV_BAD_BLOCK_ID);
        return;
    }
    uint4 *pool = (blockIdx.z == 0 ? kc : vc) + (int64_t)id * chunks_per_block;
    uint4 *st = stage + ((int64_t)blockIdx.x * 2 + blockIdx.z) * chunks_per_block;
    const uint4 *from = kOut ? pool : st;
    uint4 *to = kOut ? st : pool;
    const int64_t first = (int64_t)blockIdx.y * kCopyThreads * kChunksPerThread + threadIdx.x;
    uint4 buf[kChunksPerThread];
#pragma unroll
    for (int u = 0; u < kChunksPerThread; ++u) {
        const int64_t c = first + (int64_t)u * kCopyThreads;
        if (c < chunks_per_block) buf[u] = from[c];
    }
#pragma unroll
    for (int u = 0; u < kChunksPerThread; ++u) {
        const int64_t c = first + (int64_t)u * kCopyThreads;
        if (c < chunks_per_block) to[c] = buf[u];
    }
}

int elem_bytes(pa_dtype dtype) {
    return dtype == PA_DTYPE_F32 ? 4 : (dtype == PA_DTYPE_BF16 ? 2 : 1);
}

}  // namespace

void count_launches(uint64_t n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

pa_status cuda_failure(cudaError_t err, const char *where) {
    std::snprintf(g_last_error, sizeof g_last_error, "%s: %s (%d)", where, cudaGetErrorString(err),
                  (int)err);
    return PA_ERR_CUDA;
}

}  // namespace pa

using namespace pa;

extern "C" const char *pa_status_string(pa_status status) {
    switch (status) {
    case PA_OK: return "PA_OK";
    case PA_ERR_INVALID_ARG: return "PA_ERR_INVALID_ARG";
    case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED";
    case PA_ERR_CUDA: return "PA_ERR_CUDA";
    case PA_ERR_NO_BLOCKS: return "PA_ERR_NO_BLOCKS";
    case PA_ERR_WORKSPACE: return "PA_ERR_WORKSPACE";
    case PA_ERR_NOT_FOUND: return "PA_ERR_NOT_FOUND";
    default: return "PA_ERR_UNKNOWN";
    }
}

extern "C" const char *pa_last_error(void) { return g_last_error; }

extern "C" int pa_version(void) { return 100; }

extern "C" uint64_t pa_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

extern "C" pa_status pa_cache_write(void *key_cache, void *value_cache, const void *key,
                                    const void *value, const int64_t *slot_mapping, int num_tokens,
                                    int num_kv_heads, int head_dim, int block_size, int num_blocks,
                                    pa_dtype dtype, int32_t *device_status, void *stream) {
    if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size != kBlockSize ||
        num_blocks <= 0)
        return PA_ERR_INVALID_ARG;
    if (dtype != PA_DTYPE_F32 && dtype != PA_DTYPE_BF16) return PA_ERR_INVALID_ARG;
    const int row_bytes = head_dim * elem_bytes(dtype);
    if (row_bytes % 16 != 0) return PA_ERR_UNSUPPORTED;
    if (num_tokens == 0) return PA_OK;
    if (!key_cache || !value_cache || !key || !value || !slot_mapping) return PA_ERR_INVALID_ARG;
    if (!aligned16(key_cache) || !aligned16(value_cache) || !aligned16(key) || !aligned16(value) ||
        (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
        return PA_ERR_INVALID_ARG;
    const int chunks = row_bytes / 16;
    const int64_t total = (int64_t)num_tokens * num_kv_heads * chunks;
    const int64_t grid = (total + 255) / 256;
    if (grid >= ((int64_t)1 << 31)) return PA_ERR_UNSUPPORTED;
    cudaError_t e = launch_chained(
        pa_cache_write_kernel, dim3((unsigned)grid), dim3(256), 0, static_cast<cudaStream_t>(stream),
        static_cast<uint4 *>(key_cache), static_cast<uint4 *>(value_cache),
        static_cast<const uint4 *>(key), static_cast<const uint4 *>(value), slot_mapping,
        num_tokens, num_kv_heads, chunks, num_blocks, device_status);
    if (e != cudaSuccess) return cuda_failure(e, "pa_cache_write_kernel launch");
    count_launches(1);
    return PA_OK;
}

extern "C" pa_status pa_block_copy(void *key_cache, void *value_cache, const int32_t *src_dst,
                                   int num_pairs, int num_kv_heads, int head_dim, int block_size,
                                   int num_blocks, pa_dtype dtype, int32_t *device_status,
                                   void *stream) {
    if (num_pairs < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size != kBlockSize ||
        num_blocks <= 0)
        return PA_ERR_INVALID_ARG;
    if (dtype != PA_DTYPE_F32 && dtype != PA_DTYPE_BF16 && dtype != PA_DTYPE_FP8_E4M3)
        return PA_ERR_INVALID_ARG;
    const int64_t block_bytes = (int64_t)num_kv_heads * kBlockSize * head_dim * elem_bytes(dtype);
    if (block_bytes % 16 != 0) return PA_ERR_UNSUPPORTED;
    if (num_pairs == 0) return PA_OK;
    if (!key_cache || !value_cache || !src_dst) return PA_ERR_INVALID_ARG;
    if (!aligned16(key_cache) || !aligned16(value_cache) ||
        (reinterpret_cast<uintptr_t>(src_dst) & 7u))
        return PA_ERR_INVALID_ARG;
    const int64_t chunks = block_bytes / 16;
    const int64_t per_cta = (int64_t)kCopyThreads * kChunksPerThread;
    const int64_t slices = (chunks + per_cta - 1) / per_cta;
    if (slices > 65535) return PA_ERR_UNSUPPORTED;
    dim3 grid((unsigned)num_pairs, (unsigned)slices);
    cudaError_t e = launch_chained(
        pa_block_copy_kernel, grid, dim3(kCopyThreads), 0, static_cast<cudaStream_t>(stream),
        static_cast<uint4 *>(key_cache), static_cast<uint4 *>(value_cache), src_dst, num_pairs,
        chunks, num_blocks, device_status);
    if (e != cudaSuccess) return cuda_failure(e, "pa_block_copy_kernel launch");
    count_launches(1);
    return PA_OK;
}

extern "C" pa_status pa_cache_write_fp8(void *key_cache, void *value_cache, const void *key,
                                        const void *value, const int64_t *slot_mapping,
                                        const float *k_scales, const float *v_scales,
                                        int num_tokens, int num_kv_heads, int head_dim,
                                        int block_size, int num_blocks, int32_t *device_status,
                                        void *stream) {
    if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size != kBlockSize ||
        num_blocks <= 0)
        return PA_ERR_INVALID_ARG;
    if (head_dim % 16 != 0) return PA_ERR_UNSUPPORTED;
    if (num_tokens == 0) return PA_OK;
    if (!key_cache || !value_cache || !key || !value || !slot_mapping || !k_scales || !v_scales)
        return PA_ERR_INVALID_ARG;
    if (!aligned16(key_cache) || !aligned16(value_cache) || !aligned16(key) || !aligned16(value) ||
        (reinterpret_cast<uintptr_t>(slot_mapping) & 7u) ||
        (reinterpret_cast<uintptr_t>(k_scales) & 3u) || (reinterpret_cast<uintptr_t>(v_scales) & 3u))
        return PA_ERR_INVALID_ARG;
    const int chunks = head_dim / 16;
    const int64_t total = (int64_t)num_tokens * num_kv_heads * chunks;
    const int64_t grid = (total + 255) / 256;
    if (grid >= ((int64_t)1 << 31)) return PA_ERR_UNSUPPORTED;
    cudaError_t e = launch_chained(
        pa_cache_write_fp8_kernel, dim3((unsigned)grid), dim3(256), 0,
        static_cast<cudaStream_t>(stream), static_cast<uint4 *>(key_cache),
        static_cast<uint4 *>(value_cache), static_cast<const uint4 *>(key),
        static_cast<const uint4 *>(value), slot_mapping, k_scales, v_scales, num_tokens,
        num_kv_heads, chunks, num_blocks, device_status);
    if (e != cudaSuccess) return cuda_failure(e, "pa_cache_write_fp8_kernel launch");
    count_launches(1);
    return PA_OK;
}

namespace {

// The address a kernel on the current device uses for p: device memory of this
// device and managed memory as they are, page-locked host memory through its
// mapping.  Anything else (pageable host memory, another device's memory) is
// refused, so that no kernel dereferences an address it cannot reach.
pa_status device_address(const void *p, void **dev) {
    cudaPointerAttributes at;
    cudaError_t e = cudaPointerGetAttributes(&at, p);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return PA_ERR_INVALID_ARG;
    }
    int cur = 0;
    e = cudaGetDevice(&cur);
    if (e != cudaSuccess) return cuda_failure(e, "cudaGetDevice");
    switch (at.type) {
    case cudaMemoryTypeDevice:
        if (at.device != cur) return PA_ERR_INVALID_ARG;
        *dev = const_cast<void *>(p);
        return PA_OK;
    case cudaMemoryTypeManaged:
        *dev = const_cast<void *>(p);
        return PA_OK;
    case cudaMemoryTypeHost:
        if (at.devicePointer == nullptr) return PA_ERR_INVALID_ARG;
        *dev = at.devicePointer;
        return PA_OK;
    default:
        return PA_ERR_INVALID_ARG;
    }
}

pa_status swap_common(bool out, void *key_cache, void *value_cache, const int32_t *block_ids,
                      int num_ids, void *staging, int num_kv_heads, int head_dim, int block_size,
                      int num_blocks, pa_dtype dtype, int32_t *device_status, void *stream) {
    if (num_ids < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size != kBlockSize ||
        num_blocks <= 0)
        return PA_ERR_INVALID_ARG;
    if (dtype != PA_DTYPE_F32 && dtype != PA_DTYPE_BF16 && dtype != PA_DTYPE_FP8_E4M3)
        return PA_ERR_INVALID_ARG;
    const int64_t block_bytes = (int64_t)num_kv_heads * kBlockSize * head_dim * elem_bytes(dtype);
    if (block_bytes % 16 != 0) return PA_ERR_UNSUPPORTED;
    if (num_ids == 0) return PA_OK;
    if (!key_cache || !value_cache || !block_ids || !staging) return PA_ERR_INVALID_ARG;
    if (!aligned16(key_cache) || !aligned16(value_cache) || !aligned16(staging) ||
        (reinterpret_cast<uintptr_t>(block_ids) & 3u))
        return PA_ERR_INVALID_ARG;
    void *stage = nullptr;
    pa_status st = device_address(staging, &stage);
    if (st != PA_OK) return st;
    if (!aligned16(stage)) return PA_ERR_INVALID_ARG;
    const int64_t chunks = block_bytes / 16;
    const int64_t per_cta = (int64_t)kCopyThreads * kChunksPerThread;
    const int64_t slices = (chunks + per_cta - 1) / per_cta;
    if (slices > 65535) return PA_ERR_UNSUPPORTED;
    dim3 grid((unsigned)num_ids, (unsigned)slices, 2);
    auto kernel = out ? pa_swap_kernel<true> : pa_swap_kernel<false>;
    cudaError_t e = launch_chained(kernel, grid, dim3(kCopyThreads), 0,
                                   static_cast<cudaStream_t>(stream),
                                   static_cast<uint4 *>(key_cache), static_cast<uint4 *>(value_cache),
                                   static_cast<uint4 *>(stage), block_ids, chunks, num_blocks,
                                   device_status);
    if (e != cudaSuccess) return cuda_failure(e, "pa_swap_kernel launch");
    count_launches(1);
    return PA_OK;
}

}  // namespace

extern "C" size_t pa_swap_bytes(int num_ids, int num_kv_heads, int head_dim, pa_dtype dtype) {
    if (num_ids < 0 || num_kv_heads <= 0 || head_dim <= 0 ||
        (dtype != PA_DTYPE_F32 && dtype != PA_DTYPE_BF16 && dtype != PA_DTYPE_FP8_E4M3))
        return (size_t)-1;
    return (size_t)num_ids * 2 * num_kv_heads * kBlockSize * head_dim * elem_bytes(dtype);
}

extern "C" pa_status pa_swap_out(const void *key_cache, const void *value_cache,
                                 const int32_t *block_ids, int num_ids, void *staging,
                                 int num_kv_heads, int head_dim, int block_size, int num_blocks,
                                 pa_dtype dtype, int32_t *device_status, void *stream) {
    return swap_common(true, const_cast<void *>(key_cache), const_cast<void *>(value_cache),
                       block_ids, num_ids, staging, num_kv_heads, head_dim, block_size,
                       num_blocks, dtype, device_status, stream);
}

extern "C" pa_status pa_swap_in(void *key_cache, void *value_cache, const int32_t *block_ids,
                                int num_ids, const void *staging, int num_kv_heads, int head_dim,
                                int block_size, int num_blocks, pa_dtype dtype,
                                int32_t *device_status, void *stream) {
    return swap_common(false, key_cache, value_cache, block_ids, num_ids,
                       const_cast<void *>(staging), num_kv_heads, head_dim, block_size,
                       num_blocks, dtype, device_status, stream);
}

/*
 * pagedkv.h - C ABI of the paged KV-cache decode library for GB300 (sm_103a).
 *
 * The library implements the decode hot path of PagedAttention as described in
 * "PagedAttention por dentro: bloques, tabla de páginas, evicción y el estado
 * del arte del KV cache en 2026" (sections "El modelo de bloques", "La tabla de
 * páginas (block table)", "El pool de bloques", "Copy-on-write para sampling
 * paralelo", "El kernel CUDA"): the K/V of every sequence live in fixed
 * 16-token physical blocks scattered through a pool, and a per-sequence block
 * table maps logical block j (tokens 16j .. 16j+15) to its physical block.
 *
 * Conventions shared by every entry point
 * --------------------------------------
 *  - Memory: the caller owns all memory.  Pointers documented as "device" must
 *    point to CUDA device memory of the current device; the library allocates
 *    nothing and keeps no pointer after a call returns.
 *  - Streams: `stream` is a cudaStream_t passed as void* (NULL = the legacy
 *    default stream).  Kernels are enqueued asynchronously on it; a PA_OK
 *    return means the work was enqueued, not that it finished.
 *  - Layouts (row-major, no padding):
 *      key_cache, value_cache : [num_blocks][num_kv_heads][block_size][head_dim]
 *      query, out             : [num_seqs][num_q_heads][head_dim]
 *      block_tables           : int32 [num_seqs][max_blocks_per_seq]; only the
 *                               first ceil(context_len / block_size) entries of
 *                               a row are read
 *      context_lens           : int32 [num_seqs]
 *      key, value (new rows)  : [num_tokens][num_kv_heads][head_dim]
 *      slot_mapping           : int64 [num_tokens]; slot = block * block_size + offset
 *  - block_size must be 16 (the block size the pages use).
 *  - GQA: query head h reads KV head h / (num_q_heads / num_kv_heads)
 *    ("KV cache: la memoria de trabajo que sostiene la inferencia LLM",
 *    section "Trucos para que el cuaderno sea más fino").
 *  - Argument errors are detected synchronously on the host and returned as a
 *    status; nothing is enqueued then.  Index values held in device memory
 *    (table entries, context lengths, slots, copy pairs) are checked by the
 *    kernels: an out-of-range value is never dereferenced; it is replaced as
 *    each entry point documents and, when `device_status` is not NULL, the
 *    matching PA_DEV_* bit is OR-ed into that device int32 (zero it first).
 *  - Kernels never trap.  Every wait inside a kernel is bounded (about one
 *    second); if one gives up, PA_DEV_TIMEOUT is set and the kernel returns.
 */
#ifndef PAGEDKV_H_
#define PAGEDKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pa_status {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = 1,  /* null pointer, bad size, misaligned pointer, ... */
    PA_ERR_UNSUPPORTED = 2,  /* valid arguments the library has no kernel for */
    PA_ERR_CUDA = 3,         /* a CUDA call failed; see pa_last_error() */
    PA_ERR_NO_BLOCKS = 4,    /* block manager: the pool has no free block */
    PA_ERR_WORKSPACE = 5,    /* workspace missing or smaller than required */
    PA_ERR_NOT_FOUND = 6     /* block manager: unknown or duplicate sequence id */
} pa_status;

typedef enum pa_dtype {
    PA_DTYPE_F32 = 0,        /* IEEE binary32 */
    PA_DTYPE_BF16 = 1,       /* bfloat16 */
    PA_DTYPE_FP8_E4M3 = 2    /* FP8 E4M3 codes (pools only; see pa_decode_fp8) */
} pa_dtype;

/* Bits OR-ed into the optional device status word. */
#define PA_DEV_BAD_BLOCK_ID    1  /* a table entry outside [0, num_blocks) */
#define PA_DEV_BAD_CONTEXT_LEN 2  /* context_len < 0 or > max_blocks_per_seq * block_size */
#define PA_DEV_BAD_SLOT        4  /* slot >= num_blocks * block_size */
#define PA_DEV_BAD_COPY_PAIR   8  /* a copy pair index outside [0, num_blocks) */
#define PA_DEV_TIMEOUT        16  /* a bounded in-kernel wait gave up */
#define PA_DEV_PREFIX_MISMATCH 32 /* pa_decode_shared_prefix: tables do not share the prefix */
#define PA_DEV_BAD_QUERY_LEN  64  /* pa_prefill: a chunk longer than max_query_len */
#define PA_DEV_SMEM_ALIGN    128  /* pa_prefill: shared memory not 1024-byte aligned (nothing computed) */
#define PA_DEV_RANGE         256  /* a value outside f16's finite range (|x| >= 65536, or infinite)
                                     reached an f16 operand; see the entry points that stage in f16 */

/* Human-readable name of a status. Never NULL. */
const char *pa_status_string(pa_status status);

/* Message of the last PA_ERR_CUDA on the calling thread ("" if none). */
const char *pa_last_error(void);

/* ABI version (major * 100 + minor). */
int pa_version(void);

/* Number of kernels this library has launched in this process (all threads). */
uint64_t pa_launch_count(void);

/*
 * Partition size pa_decode uses when it is given partition_size = 0: the
 * largest of 4096, 2048, 1024, 512, 256, 128 tokens for which
 * num_seqs * heads * ceil(max_blocks_per_seq * 16 / size) reaches four CTAs
 * per SM of the current device (heads = num_kv_heads for bf16 and FP8 pools,
 * num_q_heads for f32).  Returns -1 for invalid arguments.
 */
int pa_decode_partition_size(int num_seqs, int num_q_heads, int num_kv_heads,
                             int max_blocks_per_seq, pa_dtype dtype);

/*
 * Bytes of workspace pa_decode needs for the split-K partials.  Returns 0 when
 * no sequence can span more than one partition (no workspace needed).
 * max_blocks_per_seq bounds the context length (max_blocks_per_seq * block_size).
 * partition_size: 0 = library choice (pa_decode_partition_size), else a
 * multiple of 16 in [16, 16384].  Returns (size_t)-1 for invalid arguments.
 */
size_t pa_decode_workspace_bytes(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                 int max_blocks_per_seq, int block_size, int partition_size,
                                 pa_dtype dtype);

/*
 * Paged decode attention: for every sequence b and query head h,
 *   out[b][h] = sum_t softmax_t(scale * <query[b][h], K_t>) * V_t
 * over the context_lens[b] tokens of sequence b, where token t's K/V row is
 * key_cache/value_cache[block_tables[b][t / 16]][h / group][t % 16].
 * Source: "KV cache: la memoria de trabajo que sostiene la inferencia LLM",
 * section "El mecanismo en sí (en cristiano)" (the attention of one new token),
 * and "PagedAttention por dentro", sections "La tabla de páginas (block table)"
 * and "El kernel CUDA" (the block-table indirection, processed block by block).
 *
 *  out, query        device, dtype elements, [num_seqs][num_q_heads][head_dim]
 *  key_cache,
 *  value_cache       device, dtype elements, 16-byte aligned
 *  block_tables      device int32 [num_seqs][max_blocks_per_seq]
 *  context_lens      device int32 [num_seqs]
 *  head_dim          bf16: 64 or 128; f32: 32, 64, 128 or 256
 *  num_q_heads       a multiple of num_kv_heads; bf16 needs the group
 *                    (num_q_heads / num_kv_heads) in {1, ..., 8, 12, 16}
 *  scale             the softmax scale (usually 1/sqrt(head_dim))
 *  partition_size    tokens per split-K partition: 0 = library choice
 *                    (pa_decode_partition_size), else a
 *                    multiple of 16 in [16, 16384].  A sequence longer than
 *                    one partition is processed by several CTAs whose partial
 *                    (max, sum, output) are merged by a second kernel.
 *  workspace         device scratch of at least pa_decode_workspace_bytes(...)
 *                    bytes (may be NULL when that is 0), 16-byte aligned
 *  device_status     device int32 or NULL (see PA_DEV_*)
 * Arithmetic: fp32 accumulation; bf16 output rounded to nearest even.
 * context_len 0 gives a zero output row.  A table entry out of range is read
 * as block 0 and flagged; a context length out of range is clamped to
 * [0, max_blocks_per_seq * 16] and flagged.
 */
pa_status pa_decode(void *out, const void *query, const void *key_cache, const void *value_cache,
                    const int32_t *block_tables, const int32_t *context_lens, int num_seqs,
                    int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                    int max_blocks_per_seq, int num_blocks, float scale, pa_dtype dtype,
                    int partition_size, void *workspace, size_t workspace_bytes,
                    int32_t *device_status, void *stream);

/*
 * Paged decode attention for a batch whose block tables all begin with the same
 * num_prefix_blocks physical blocks (a shared prefix: "PagedAttention por
 * dentro", section "Copy-on-write para sampling paralelo" and "Prefix caching
 * cross-session" - several sequences reading the same blocks).  The result of
 * pa_decode with the same arguments, within pa_decode's tolerance; the shared
 * blocks are read once per KV head for all sequences instead of once per
 * sequence.
 * Precision: at head_dim 128 and groups 1, 2, 4, 8 or 16 the prefix runs on
 * the tensor-core kernel of pa_prefill, whose P.V takes f16 operands (see
 * pa_prefill): the softmax weights are rounded to f16 and each prefix V value
 * is converted to f16, exact for |v| in [2^-14, 65504].  A prefix V value of
 * magnitude 65536 or more (or infinite) saturates to +-65504 and the call
 * flags PA_DEV_RANGE; such results are not those of pa_decode.  Other shapes
 * run the prefix on bf16 tensor-core tiles without that limit.
 *  num_prefix_blocks  length of the shared prefix in blocks; the blocks are
 *                     taken from the first row of block_tables and every row
 *                     must list the same ones (a row that does not is flagged
 *                     PA_DEV_PREFIX_MISMATCH and its result is undefined).
 *                     Contexts shorter than the prefix are handled (their
 *                     positions past the context are masked).  0 = pa_decode.
 *  partition_size     split-K partition of the part past the prefix (0 = the
 *                     library's choice for max_blocks_per_seq - num_prefix_blocks)
 *  workspace          at least pa_decode_shared_prefix_workspace_bytes(...)
 * bf16 only; head_dim 64 or 128; group as in pa_decode.  Launches three kernels
 * on the caller's stream: the prefix kernel first (it takes part of the SMs),
 * the suffix decode beside it, then the merge of both.
 */
size_t pa_decode_shared_prefix_workspace_bytes(int num_seqs, int num_q_heads, int num_kv_heads,
                                               int head_dim, int max_blocks_per_seq,
                                               int num_prefix_blocks, int partition_size);
pa_status pa_decode_shared_prefix(void *out, const void *query, const void *key_cache,
                                  const void *value_cache, const int32_t *block_tables,
                                  const int32_t *context_lens, int num_seqs, int num_q_heads,
                                  int num_kv_heads, int head_dim, int block_size,
                                  int max_blocks_per_seq, int num_blocks, float scale,
                                  pa_dtype dtype, int num_prefix_blocks, int partition_size,
                                  void *workspace, size_t workspace_bytes, int32_t *device_status,
                                  void *stream);

/*
 * The shared-prefix decode over FP8 (E4M3) pools with per-KV-head scales, as
 * pa_decode_fp8 computes it: same arguments as pa_decode_fp8 plus
 * num_prefix_blocks.  The prefix blocks' codes are first widened to bf16 code
 * values (exact) in the workspace, then the tensor-core prefix kernel reads
 * that copy once per KV head for all sequences, with the K scale folded into
 * the softmax scale and the V scale into its partial outputs; the rest of every
 * context runs through the FP8 decode kernel.  head_dim 128; groups 1, 2, 4, 8
 * take this path, and with num_prefix_blocks 0 the call is pa_decode_fp8.
 *  workspace  at least pa_decode_shared_prefix_fp8_workspace_bytes(...) bytes
 * Launches four kernels on the caller's stream (widen, prefix, suffix, merge).
 */
size_t pa_decode_shared_prefix_fp8_workspace_bytes(int num_seqs, int num_q_heads,
                                                   int num_kv_heads, int head_dim,
                                                   int max_blocks_per_seq, int num_prefix_blocks,
                                                   int partition_size);
pa_status pa_decode_shared_prefix_fp8(void *out, const void *query, const void *key_cache,
                                      const void *value_cache, const float *k_scales,
                                      const float *v_scales, const int32_t *block_tables,
                                      const int32_t *context_lens, int num_seqs, int num_q_heads,
                                      int num_kv_heads, int head_dim, int block_size,
                                      int max_blocks_per_seq, int num_blocks, float scale,
                                      int num_prefix_blocks, int partition_size, void *workspace,
                                      size_t workspace_bytes, int32_t *device_status,
                                      void *stream);

/*
 * Paged decode attention over FP8 pools.  The pages name quantising the KV
 * cache to FP8 as halving it ("KV cache: la memoria de trabajo que sostiene la
 * inferencia LLM", section "Trucos para que el cuaderno sea más fino"); the
 * code format is E4M3 ("E4M3FN" of the OCP 8-bit floating point
 * specification: 1 sign, 4 exponent bits with bias 7, 3 mantissa bits, no
 * infinities, largest finite 448).
 *  key_cache,
 *  value_cache       device E4M3 codes [num_blocks][num_kv_heads][16][head_dim]
 *  k_scales,
 *  v_scales          device float [num_kv_heads]: the value a code stands for
 *                    is code_value * scale of its KV head
 *  query, out        device bfloat16, as in pa_decode
 * Everything else is as in pa_decode (partition_size, workspace with
 * pa_decode_workspace_bytes(..., PA_DTYPE_FP8_E4M3), device_status, stream).
 * Supported: head_dim 128, group (num_q_heads / num_kv_heads) 1..8.
 * Arithmetic: codes are widened exactly; the query is rounded to f16 once
 * (exact for |q| in [2^-14, 65504]; a query element of magnitude 65536 or
 * more, or infinite, becomes infinite and the call flags PA_DEV_RANGE); the
 * softmax weights enter P.V as f16 (an output moves by at most 2^-11 of the
 * largest |v| it weighs); accumulation is fp32.
 */
pa_status pa_decode_fp8(void *out, const void *query, const void *key_cache,
                        const void *value_cache, const float *k_scales, const float *v_scales,
                        const int32_t *block_tables, const int32_t *context_lens, int num_seqs,
                        int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                        int max_blocks_per_seq, int num_blocks, float scale, int partition_size,
                        void *workspace, size_t workspace_bytes, int32_t *device_status,
                        void *stream);

/*
 * Paged decode attention with a sliding window of `window` positions ("PagedAttention
 * por dentro", section "Sliding window attention": a model with a window of W
 * tokens attends only to the last W tokens of its context).  For a context of
 * L = context_lens[b] tokens, the softmax and the weighted sum of pa_decode run
 * over positions [max(L - window, 0), L) only; blocks wholly before the window
 * are never read, so their table entries may be anything (a block manager may
 * already have released them: pa_bm_trim_window).
 *  k_scales, v_scales  FP8 pools only (dtype PA_DTYPE_FP8_E4M3, as in
 *                      pa_decode_fp8); ignored otherwise (may be NULL)
 *  dtype               PA_DTYPE_F32, PA_DTYPE_BF16 or PA_DTYPE_FP8_E4M3 with
 *                      the limits of pa_decode / pa_decode_fp8
 *  window              > 0 (PA_ERR_INVALID_ARG otherwise)
 *  workspace           at least pa_decode_sliding_window_workspace_bytes(...)
 *                      with the same window; the split-K partitions cover the
 *                      window, at most ceil(window / 16) + 1 blocks
 * Everything else, results for window >= L included, is as in pa_decode.
 */
size_t pa_decode_sliding_window_workspace_bytes(int num_seqs, int num_q_heads, int num_kv_heads,
                                                int head_dim, int max_blocks_per_seq,
                                                int block_size, int window, int partition_size,
                                                pa_dtype dtype);
pa_status pa_decode_sliding_window(void *out, const void *query, const void *key_cache,
                                   const void *value_cache, const float *k_scales,
                                   const float *v_scales, const int32_t *block_tables,
                                   const int32_t *context_lens, int num_seqs, int num_q_heads,
                                   int num_kv_heads, int head_dim, int block_size,
                                   int max_blocks_per_seq, int num_blocks, float scale,
                                   pa_dtype dtype, int window, int partition_size, void *workspace,
                                   size_t workspace_bytes, int32_t *device_status, void *stream);

/*
 * Cache write into FP8 pools: as pa_cache_write, but each element x of the
 * new bfloat16 rows is stored as the E4M3 code of the float32 quotient
 * x / scale[kv_head] (IEEE single-precision division, then rounding to the
 * nearest E4M3 value with ties to an even mantissa; magnitudes of 448 or more
 * saturate to +-448; NaN stays NaN).
 *  key, value        device bfloat16 [num_tokens][num_kv_heads][head_dim]
 *  k_scales,
 *  v_scales          device float [num_kv_heads]
 *  head_dim          a multiple of 16
 */
pa_status pa_cache_write_fp8(void *key_cache, void *value_cache, const void *key,
                             const void *value, const int64_t *slot_mapping,
                             const float *k_scales, const float *v_scales, int num_tokens,
                             int num_kv_heads, int head_dim, int block_size, int num_blocks,
                             int32_t *device_status, void *stream);

/*
 * Size of the library-owned scratch array used by pa_decode_static_scratch
 * (32 MiB of device global memory on every device that loads the library).
 */
#define PA_STATIC_SCRATCH_BYTES (32u << 20)

/*
 * pa_decode without caller scratch.  The pages have no counterpart: this is an
 * interface addition for callers that cannot allocate device memory at call
 * time - their device memory is reserved up front by another allocator, or a
 * cudaMalloc / cudaFree (with its implicit device synchronisation) is not
 * acceptable where they run, or they are handed only inputs and outputs.
 * Arguments, layouts, results and error behaviour are those of pa_decode;
 * the split-K partials go to a fixed library-owned device array of
 * PA_STATIC_SCRATCH_BYTES instead of a workspace.  Nothing is allocated.
 *  - Size limit: when pa_decode_workspace_bytes(...) for these arguments
 *    exceeds PA_STATIC_SCRATCH_BYTES the call returns PA_ERR_WORKSPACE and
 *    enqueues nothing (use pa_decode with a workspace, or a larger
 *    partition_size, then).  Invalid arguments are reported first, with the
 *    status pa_decode gives them.
 *  - Set-up: the first call on a device that needs scratch looks up the
 *    array's device address (cudaGetSymbolAddress) with that device current;
 *    make that first call before any stream capture.  The address is kept
 *    with the context it belongs to; a call in a new context of the device
 *    (after cudaDeviceReset) looks it up again, so make the first call after
 *    a reset before any stream capture too.
 *  - Sharing: every call on a device uses the same array and leaves its last
 *    contents there.  No part of it has to start at zero.  Calls that overlap
 *    on the GPU (other streams, other host threads) race on it; serialise them.
 */
pa_status pa_decode_static_scratch(void *out, const void *query, const void *key_cache,
                                   const void *value_cache, const int32_t *block_tables,
                                   const int32_t *context_lens, int num_seqs, int num_q_heads,
                                   int num_kv_heads, int head_dim, int block_size,
                                   int max_blocks_per_seq, int num_blocks, float scale,
                                   pa_dtype dtype, int partition_size, int32_t *device_status,
                                   void *stream);

/*
 * Cache write: for every new token i with slot_mapping[i] >= 0, copies its K
 * and V rows (all KV heads) into offset slot % 16 of physical block slot / 16:
 *   key_cache[slot / 16][kvh][slot % 16][:] = key[i][kvh][:]   (same for V)
 * Source: "PagedAttention por dentro", section "La tabla de páginas (block
 * table)" (a new token is written into the free slot of its block).
 *  key, value      device [num_tokens][num_kv_heads][head_dim], 16-byte aligned
 *  slot_mapping    device int64 [num_tokens]; negative = skip (padding)
 *  head_dim        head_dim * element size must be a multiple of 16 bytes
 * Bit-exact copy.  Two tokens with the same slot race (one of them wins).
 * A slot >= num_blocks * 16 is skipped and flagged.
 */
pa_status pa_cache_write(void *key_cache, void *value_cache, const void *key, const void *value,
                         const int64_t *slot_mapping, int num_tokens, int num_kv_heads,
                         int head_dim, int block_size, int num_blocks, pa_dtype dtype,
                         int32_t *device_status, void *stream);

/*
 * Block copy for copy-on-write: for every pair p, physical block dst becomes a
 * bit-exact copy of block src in both pools (all KV heads, all 16 slots).
 * Source: "PagedAttention por dentro", section "Copy-on-write para sampling
 * paralelo" (on divergence only the last shared block is copied).
 *  src_dst     device int32 [num_pairs][2] = (src, dst), 8-byte aligned
 * The pairs are independent copies into fresh blocks (on the pages every copy
 * goes into a block just taken from the pool), so they run concurrently and
 * each copies block src as it was before the call:
 *  - a pair with an index outside [0, num_blocks) is skipped and flagged
 *    PA_DEV_BAD_COPY_PAIR;
 *  - a pair with src == dst changes nothing;
 *  - a pair (src != dst) whose dst is the src or the dst of another pair
 *    (both indices in range, src != dst) is skipped and flagged
 *    PA_DEV_BAD_COPY_PAIR: a chained list such as (a, b), (b, c) copies only
 *    (b, c), and two pairs with one dst both stay undone.
 * Every other pair is copied.  The host block manager never emits a skipped
 * pair.  Each CTA checks its pair against the whole list, so the kernel reads
 * the list num_pairs times (from L2).
 */
pa_status pa_block_copy(void *key_cache, void *value_cache, const int32_t *src_dst, int num_pairs,
                        int num_kv_heads, int head_dim, int block_size, int num_blocks,
                        pa_dtype dtype, int32_t *device_status, void *stream);

/*
 * Chunked (paged) prefill attention ("PagedAttention por dentro", section
 * "Chunked prefill integrado con paged KV": prefill is cut into chunks that run
 * over the same paged KV cache as decode).  Sequence b brings a chunk of
 * T_b = query_start[b+1] - query_start[b] new tokens whose K/V are already in
 * the pools (pa_cache_write); its context then holds L_b = context_lens[b]
 * tokens, the chunk being the last T_b of them.  Query row i of the chunk sits
 * at position p = L_b - T_b + i and attends causally to positions [0, p]
 * ("KV cache: la memoria de trabajo que sostiene la inferencia LLM", "El
 * mecanismo en sí (en cristiano)"); with window > 0, to [p + 1 - window, p]
 * ("PagedAttention por dentro", "Sliding window attention").
 *  out, query        device bfloat16 [num_query_tokens][num_q_heads][head_dim];
 *                    rows query_start[b] .. query_start[b+1]-1 are sequence b's
 *  query_start       device int32 [num_seqs + 1], non-decreasing, [0] = 0,
 *                    [num_seqs] = num_query_tokens
 *  context_lens      device int32 [num_seqs], L_b >= T_b
 *  max_query_len     host int, at least every T_b (sizes the grid); rows of a
 *                    longer chunk past max_query_len are not computed and the
 *                    call flags PA_DEV_BAD_QUERY_LEN
 *  window            0 = causal over the whole context
 * Pools, block tables, scale, device_status and stream as in pa_decode; table
 * entries of blocks wholly before every row's window are not read.
 *  workspace         device scratch of at least pa_prefill_workspace_bytes()
 *                    bytes, 16-byte aligned: the work counter of the CTAs
 *                    (set to zero on the stream by each call; calls that run
 *                    at the same time need their own)
 * Supported: bf16, head_dim 128, group (num_q_heads / num_kv_heads) 1, 2, 4, 8
 * or 16.  Arithmetic: S = QK^T and O = PV on tcgen05 tensor cores with fp32
 * accumulation in tensor memory.  The second product runs on f16 operands: P
 * rounded to f16 (2^-11 relative, so an output moves by at most 2^-11 of the
 * largest |v| it weighs), each V tile converted to f16 in shared memory, which
 * is exact for |v| in [2^-14, 65504]; smaller magnitudes lose at most 2^-25
 * absolute, larger ones (|v| >= 65536, or infinite) saturate to +-65504 and
 * the call flags PA_DEV_RANGE (V beyond f16's range is not supported; the
 * flag says the result is not the attention of the given values).  A memset
 * of the work counter,
 * then one kernel launch: one CTA per SM, each taking (256-row tile, KV head,
 * sequence) items in turn.
 */
size_t pa_prefill_workspace_bytes(void);
pa_status pa_prefill(void *out, const void *query, const void *key_cache, const void *value_cache,
                     const int32_t *block_tables, const int32_t *context_lens,
                     const int32_t *query_start, int num_seqs, int num_q_heads, int num_kv_heads,
                     int head_dim, int block_size, int max_blocks_per_seq, int num_blocks,
                     int num_query_tokens, int max_query_len, float scale, pa_dtype dtype,
                     int window, void *workspace, size_t workspace_bytes, int32_t *device_status,
                     void *stream);

/*
 * Swap of blocks between the pools and a staging buffer ("PagedAttention por
 * dentro", section "Evicción y preemption", strategy 2 "swap": the blocks of
 * a preempted sequence move to CPU memory, freeing device memory, and come
 * back when it is scheduled again).
 *  block_ids    device int32 [num_ids]: physical blocks, in staging order
 *  staging      [num_ids][2][num_kv_heads][16][head_dim] elements of dtype:
 *               entry i holds block_ids[i]'s K tile, then its V tile (all KV
 *               heads), pa_swap_bytes(num_ids, ...) bytes in all.  Any
 *               device-accessible address, 16-byte aligned: device memory of
 *               the current device, managed memory, or page-locked host memory
 *               (cudaHostAlloc / cudaMallocHost / cudaHostRegister; the host
 *               pointer is passed and the library uses its device mapping),
 *               which the kernel reads or writes directly over the CPU-GPU
 *               link.  Other addresses (pageable host memory, another device's
 *               memory) return PA_ERR_INVALID_ARG.
 * pa_swap_out copies the listed blocks (both pools) into staging; pa_swap_in
 * copies staging into the listed blocks.  Bit copies.  For pa_swap_in the ids
 * must be distinct.  An id outside [0, num_blocks) is skipped and flagged
 * PA_DEV_BAD_BLOCK_ID.  One kernel launch each; the caller owns both sides and
 * orders them with the stream (the staging buffer is complete once the stream
 * reaches the point after pa_swap_out).
 */
size_t pa_swap_bytes(int num_ids, int num_kv_heads, int head_dim, pa_dtype dtype);
pa_status pa_swap_out(const void *key_cache, const void *value_cache, const int32_t *block_ids,
                      int num_ids, void *staging, int num_kv_heads, int head_dim, int block_size,
                      int num_blocks, pa_dtype dtype, int32_t *device_status, void *stream);
pa_status pa_swap_in(void *key_cache, void *value_cache, const int32_t *block_ids, int num_ids,
                     const void *staging, int num_kv_heads, int head_dim, int block_size,
                     int num_blocks, pa_dtype dtype, int32_t *device_status, void *stream);

/*
 * Host block manager: one pool of num_blocks blocks of block_size tokens,
 * per-sequence block tables, reference counts and copy-on-write.
 * Source: "PagedAttention por dentro", sections "La tabla de páginas (block
 * table)" (growth rule: a sequence holding N tokens writes its next token into
 * its last block when N mod 16 != 0, otherwise it appends a new block taken
 * from the pool), "El pool de bloques" (one global pool) and "Copy-on-write
 * para sampling paralelo" (forked sequences share blocks; only the shared
 * block about to change is copied).
 * Allocation order is deterministic: the free list is a stack that first hands
 * out 0, 1, 2, ...; a freed block is the next one handed out; pa_bm_free_seq
 * releases a table from its last entry to its first.
 * Host memory only; no CUDA call.  A handle is not thread-safe.
 * Operations that fail change nothing.
 */
typedef struct pa_bm pa_bm;

pa_bm *pa_bm_create(int num_blocks, int block_size);   /* NULL on bad arguments */
void pa_bm_destroy(pa_bm *bm);
/* New sequence with room for num_tokens tokens (all or nothing). */
pa_status pa_bm_alloc_seq(pa_bm *bm, int seq, int num_tokens);
/* child shares every block of parent (reference counts + 1). */
pa_status pa_bm_fork(pa_bm *bm, int parent, int child);
/* Room for one more token: *slot receives its slot; when the last block was
 * shared it is first copied: *cow_src / *cow_dst receive the pair, else -1. */
pa_status pa_bm_append_slot(pa_bm *bm, int seq, int64_t *slot, int32_t *cow_src, int32_t *cow_dst);
/* Copy-on-write of one logical block; the pair is (-1, -1) if it was private. */
pa_status pa_bm_make_private(pa_bm *bm, int seq, int logical_block, int32_t *cow_src,
                             int32_t *cow_dst);
pa_status pa_bm_free_seq(pa_bm *bm, int seq);
int pa_bm_num_free(const pa_bm *bm);
/* Released blocks kept for the prefix cache (handed out once the free list is empty). */
int pa_bm_num_evictable(const pa_bm *bm);
/* Prefix caching ("PagedAttention por dentro", section "Prefix caching
 * cross-session"; "Cómo funciona realmente vLLM", section "Automatic Prefix
 * Caching").  A full block whose K/V are written can be indexed by
 *   key_j = FNV1a64(le64(key_{j-1}) || le32(tokens of block j)), key_{-1} = 0
 * (a hash of its content and of everything before it).  A new sequence that
 * begins with the same tokens reuses the indexed blocks (reference counts + 1;
 * a lookup also compares the block's own tokens) and only the rest is newly
 * allocated; *num_cached_tokens receives the number of leading tokens whose
 * K/V are already in the pool (a multiple of block_size).  All or nothing. */
pa_status pa_bm_alloc_seq_cached(pa_bm *bm, int seq, const int32_t *tokens, int num_tokens,
                                 int *num_cached_tokens);
/* Index seq's full blocks (over its first num_tokens tokens) once their K/V are
 * written; returns how many blocks were newly indexed, -1 for an unknown seq.
 * A key already indexed keeps its block; a block is indexed once. */
int pa_bm_register_prefix(pa_bm *bm, int seq, const int32_t *tokens, int num_tokens);
/* Sliding window ("PagedAttention por dentro", section "Sliding window
 * attention": only the blocks of the active window are kept, older ones are
 * freed).  For a sequence of N tokens attending to its last `window` tokens,
 * releases every block whose positions all lie before N - window (the last
 * such entry first) and sets its table entry to -1; returns how many blocks
 * were released (0 when none), -1 for an unknown seq or window <= 0.  Such a
 * sequence is decoded with pa_decode_sliding_window with the same window or a
 * smaller one; forks share only its remaining blocks, and pa_bm_make_private
 * of a released entry returns PA_ERR_INVALID_ARG. */
int pa_bm_trim_window(pa_bm *bm, int seq, int window);
/* Swap bookkeeping ("PagedAttention por dentro", section "Evicción y
 * preemption", strategy "swap").  pa_bm_swap_out lists seq's blocks in table
 * order (skipping entries released by pa_bm_trim_window) into block_ids (cap
 * entries; *num_ids receives the count), releases them (last entry first) and
 * marks seq swapped: its live entries read -2.  A swapped sequence can only be
 * swapped in, freed or queried.  pa_bm_swap_in takes fresh blocks for its -2
 * entries in table order (all or nothing: PA_ERR_NO_BLOCKS) and writes them,
 * in that order, to block_ids - the order pa_swap_out's staging holds them
 * in.  Sharing with other sequences is not restored: every block swapped in
 * is private.  PA_ERR_INVALID_ARG for a sequence in the wrong state or a cap
 * that is too small (nothing changes then). */
pa_status pa_bm_swap_out(pa_bm *bm, int seq, int32_t *block_ids, int cap, int *num_ids);
pa_status pa_bm_swap_in(pa_bm *bm, int seq, int32_t *block_ids, int cap, int *num_ids);
int pa_bm_num_tokens(const pa_bm *bm, int seq);       /* -1 if unknown */
int pa_bm_ref_count(const pa_bm *bm, int block);      /* -1 if out of range */
/* Copies up to cap entries of seq's table to out; returns its length, -1 if unknown. */
int pa_bm_table(const pa_bm *bm, int seq, int32_t *out, int cap);
/* One decode step for n sequences: appends a slot to each, in order.
 * slots [n]; cow_pairs receives up to n (src, dst) pairs, *num_cow their count.
 * Stops at the first failure: *num_done = sequences appended before it. */
pa_status pa_bm_append_slots(pa_bm *bm, const int32_t *seqs, int n, int64_t *slots,
                             int32_t *cow_pairs, int *num_cow, int *num_done);
/* Dense host block tables [n][max_blocks] (-1 past each table's end) and
 * context lengths [n] for the listed sequences. */
pa_status pa_bm_fill_tables(const pa_bm *bm, const int32_t *seqs, int n, int32_t *tables,
                            int max_blocks, int32_t *context_lens);
/* Occupancy of the pool and its internal fragmentation ("Cómo funciona
 * realmente vLLM", section "La sobre-reserva estática y los tres tipos de
 * desperdicio": slots reserved for a sequence that never receive a token;
 * "PagedAttention por dentro", opening section: paging keeps that waste under
 * 4 %, since only a sequence's last block can be partly empty).  A block's
 * filled slots are the most tokens any table entry pointing at it holds (an
 * entry fills its block from offset 0 up, and shared entries fill it alike). */
typedef struct pa_bm_stats_t {
    int64_t num_blocks;        /* pool size */
    int64_t free_blocks;       /* on the free list */
    int64_t evictable_blocks;  /* released but kept for the prefix cache */
    int64_t used_blocks;       /* reference count >= 1 */
    int64_t shared_blocks;     /* reference count >= 2 */
    int64_t reserved_slots;    /* used_blocks * block_size */
    int64_t filled_slots;      /* slots of used blocks holding a token */
    int64_t logical_tokens;    /* tokens of all sequences held in blocks, a shared
                                  block counted once per sequence */
    double internal_fragmentation; /* (reserved - filled) / reserved; 0 if nothing is used */
} pa_bm_stats_t;
pa_status pa_bm_stats(const pa_bm *bm, pa_bm_stats_t *out);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H_ */

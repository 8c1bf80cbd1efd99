// Chunked (paged) prefill attention on 5th-generation tensor cores.
//
// "PagedAttention por dentro: bloques, tabla de páginas, evicción y el estado
// del arte del KV cache en 2026", section "Chunked prefill integrado con paged
// KV": prefill is cut into chunks that run over the same paged KV cache as
// decode.  Sequence b brings T_b new tokens (their K/V already written into the
// pools); its context then holds L_b tokens, the chunk being the last T_b.  Row
// i of the chunk (position p = L_b - T_b + i) attends causally to positions
// [0, p] ("KV cache: la memoria de trabajo que sostiene la inferencia LLM",
// "El mecanismo en sí (en cristiano)"), or to its last W positions with a
// sliding window ("PagedAttention por dentro", "Sliding window attention").
//
// One CTA computes two 128-row tiles (A, then B) of (token, query head of the
// group) rows of one sequence and one KV head, flash-attention style over
// 128-position K/V tiles gathered block by block through the block table.
// Each K/V tile loaded serves 256 rows.
//   warp 0       TMA producer: both Q tiles once, then K and V tiles (eight
//                16-row blocks each) into kStages-deep rings;
//   warp 1       MMA issuer, ping-pong between the tiles:
//                  S_A(0) S_B(0) | PV_A(j) S_A(j+1) PV_B(j) S_B(j+1) | ...
//                S = Q K^T lands in tensor memory; O += P V reads P from tensor
//                memory (written over its own S) and accumulates in tensor
//                memory; owns the TMEM allocation (S_A, S_B, O_A, O_B);
//   warps 2..9   softmax of tile A, warps 10..17 softmax of tile B: two threads
//                per row (= TMEM lane), each owning 64 of the 128 columns of S
//                and of O.  In one pass over S per K/V tile they write P (f16)
//                over the S columns they read, against an integer reference
//                that rises only when a chunk's weights would grow past 2^15;
//                they agree on the row's reference through shared memory once
//                per K/V tile, keep their part of the running sum, rescale
//                their part of O (by a power of two) only when the reference
//                rose, and write their part of the output row;
//   warps 18..19 convert each landed V tile to f16 in place (P.V runs on f16
//                operands: bf16 weights would be too coarse for the output
//                tolerance) and zero the rows of positions outside the tile's
//                range.
// While one tile's softmax runs, the tensor cores work on the other tile.  The
// MMAs of one thread execute in issue order: S_X(j+1), issued after PV_X(j),
// cannot overwrite the P that PV_X(j) reads.
// The same kernel, in prefix mode, computes the shared prefix of a decode
// batch whose tables all start with the same blocks ("PagedAttention por
// dentro", "Copy-on-write para sampling paralelo" and "Prefix caching
// cross-session"): its rows are (sequence, query head) pairs across the batch,
// its K/V the shared blocks, and it leaves split-K partials that the decode's
// merge combines with the rest of each context.
// Every wait is bounded (about a second); a wait that gives up sets
// PA_DEV_TIMEOUT and the CTA drains its tensor-core work and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <math.h>

#include <algorithm>
#include <climits>
#include <mutex>

#include "pa_device.cuh"
#include "pa_internal.h"
#include "pa_tc.cuh"

namespace pa {
namespace {

constexpr int kRows = 128;               // rows per Q tile (M of every MMA)
constexpr int kQT = 2;                   // Q tiles per CTA
constexpr int kKv = 128;                 // N: K/V positions per step (8 blocks)
constexpr int kD = 128;                  // head_dim
constexpr int kHalf = 16384;             // one 64-column swizzled region of a tile
constexpr int kTile = 2 * kHalf;         // 128 rows x 256 bytes
constexpr int kSplit = 2;                // softmax threads per row
constexpr int kCols = kKv / kSplit;      // S / O columns per softmax thread
constexpr int kGroup = kRows * kSplit;   // softmax threads per Q tile
constexpr int kConvWarp0 = 2 + kQT * kGroup / 32;   // first V-conversion warp
constexpr int kConvThreads = 64;                     // V-conversion threads
constexpr int kThreads = 64 + kQT * kGroup + kConvThreads;
#ifndef PA_PREFILL_STAGES
#define PA_PREFILL_STAGES 2
#endif
constexpr int kStages = PA_PREFILL_STAGES;   // depth of the K and V rings
constexpr float kChunkSumMax = 32768.f;  // largest weight sum of a 32-column chunk kept as computed
constexpr size_t kPrefillWorkspaceBytes = 256;   // the ticket counter (rounded up)

// shared memory map (offsets from the 1024-byte aligned dynamic base)
constexpr int kOffQ = 0;                          // kQT tiles
constexpr int kOffK = kOffQ + kQT * kTile;        // kStages tiles
constexpr int kOffV = kOffK + kStages * kTile;    // kStages tiles
constexpr int kOffBar = kOffV + kStages * kTile;
constexpr int kNumBars = 5 * kStages + 15;
constexpr int kOffRed = kOffBar + 256;            // [kQT][2 parities][kSplit][128] floats
constexpr int kPermMax = 64;                      // prefill: sequences ordered by length (at most)
constexpr int kOffPerm = kOffRed + kQT * 2 * kSplit * kRows * 4;   // int [kPermMax]
constexpr int kSmemBytes = kOffPerm + kPermMax * 4;
// The tiles need 1024-byte alignment; the dynamic shared memory of a kernel
// without static shared memory starts on such a boundary, and the kernel
// checks it (PA_DEV_SMEM_ALIGN) instead of reserving slack.

// barrier indices
constexpr int kQFull = 0, kKFull = 1, kKEmpty = kKFull + kStages, kVFull = kKEmpty + kStages,
              kVEmpty = kVFull + kStages, kVConv = kVEmpty + kStages, kSFull = kVConv + kStages,
              kPFull = kSFull + kQT,
              kPvDone = kPFull + kQT, kOFree = kPvDone + kQT, kItemFull = kOFree + kQT,
              kItemEmpty = kItemFull + 2, kQFree = kItemEmpty + 2, kDrain = kQFree + 1;
static_assert(kDrain + 1 == kNumBars, "barrier count");
// barriers, then the TMEM slot, the failure flag, the prefix-mode context bound
// and the two-entry item queue
static_assert(kNumBars * 8 + 20 <= 256, "barrier block");
static_assert(kSmemBytes <= 227 * 1024, "shared memory");
static_assert(kQT * kRows * kD * 4 <= 2 * kStages * kTile, "prefix partials staged over the K/V rings");

// TMEM columns: S_A, S_B, then O_A, O_B.
constexpr uint32_t kTmemCols = 512;
__device__ __forceinline__ uint32_t col_s(int x) { return (uint32_t)(x * kKv); }
__device__ __forceinline__ uint32_t col_o(int x) { return (uint32_t)(kQT * kKv + x * kD); }

}  // namespace

struct PrefillArgs {
    void *out;                    // prefill: bf16 [tokens][Hq][D]
    const int32_t *block_tables;
    const int32_t *context_lens;
    const int32_t *query_start;   // prefill only
    int32_t *status;
    int num_seqs;
    int num_q_heads;
    int num_kv_heads;
    int group;
    int max_blocks;
    int num_blocks;
    int max_query_len;            // prefill only
    int window;                   // prefill only
    float scale_log2;
    // shared-prefix mode: split-K partials of the prefix, one per chunk
    float *part_o;                // [rows * max_parts][D], rows = (b * Hq + h)
    float2 *part_ml;              // [rows * max_parts]: (max, sum), log2 domain
    int max_parts;
    int prefix_blocks;
    int chunk_blocks;
    // shared prefix of FP8 pools: the K/V tensors are a staging copy of the
    // prefix blocks' code values in bf16, block j at index j (no table), and
    // the stored values are code * scale of the KV head (nullptr: bf16 pools)
    int staged;
    const float *k_scales;
    const float *v_scales;
    // items: n_mt pair tiles per (sequence or prefix chunk, KV head); prefill
    // CTAs take them from *work_counter (zero at launch) up to num_items
    int n_mt;
    int num_items;
    unsigned int *work_counter;
};

namespace {

__device__ __forceinline__ bool wait_or_fail(uint64_t *bar, uint32_t parity, volatile int *fail,
                                             int32_t *status) {
    if (*fail) return false;
    if (mbar_wait_bounded(bar, parity)) return true;
    *fail = 1;
    report(status, PA_DEV_TIMEOUT);
    return false;
}

// A bounded wait whose outcome is the same for every lane of the warp, so
// that the .sync.aligned tensor-memory instructions after it stay convergent.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, volatile int *fail,
                                          int32_t *status) {
    return __all_sync(0xffffffffu, wait_or_fail(bar, parity, fail, status));
}

// 2^x (ex2.approx.ftz: about 2 ulp; 2^-inf = +0)
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Packed pairs of floats for the f32x2 arithmetic of sm_100 and later (one
// instruction for two lanes of work): x = (lo, hi).
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t x, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(x));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

// 2^(a - b) for references a <= b that are integers or -inf (b may be +inf
// after infinite scores): exact, 0 when a is -inf or far below b.
__device__ __forceinline__ float pow2_diff(float a, float b) {
    if (a == b) return 1.f;
    if (!(a > -INFINITY) || !(b - a < 256.f)) return 0.f;
    return ldexpf(1.f, (int)(a - b));
}

__device__ __forceinline__ uint32_t pack2_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// two floats as an f16 pair, `lo` in the low half (round to nearest even)
__device__ __forceinline__ uint32_t pack2_f16(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// The softmax's rare paths, kept out of line so that the registers of the
// common path stay free.  Both are called by all lanes of a warp together
// (their tensor-memory accesses are warp-wide).

// Weights of the 32-column chunk of S at taddr (its first column is position
// kc) written over it as 16 f16 pairs: P = 2^(s * sl2k - ref).  A lane whose
// first attempt summed past the limit (over) first raises its reference ref to
// the next integer at or above the chunk's largest scaled attended score.
// Returns (weight sum, reference).
__device__ __noinline__ float2 chunk_weights_again(uint32_t taddr, float sl2k, float ref, bool over,
                                                   bool masked, int kc, int qpos, int wlo) {
    uint32_t v[32];
    tmem_ld32(taddr, v);
    tmem_wait_ld();
    if (over) {
        float rmax = -INFINITY;
#pragma unroll
        for (int i = 0; i < 32; ++i)
            if (!masked || (kc + i <= qpos && kc + i >= wlo))
                rmax = fmaxf(rmax, __uint_as_float(v[i]) * sl2k);
        const float nref = ceilf(rmax);
        if (nref > ref) ref = nref;   // else non-finite scores: as computed before
    }
    uint32_t pp[16];
    float sum = 0.f;
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
        float p0 = ex2_approx(__uint_as_float(v[i]) * sl2k - ref);
        float p1 = ex2_approx(__uint_as_float(v[i + 1]) * sl2k - ref);
        if (masked) {
            if (!(kc + i <= qpos && kc + i >= wlo)) p0 = 0.f;
            if (!(kc + i + 1 <= qpos && kc + i + 1 >= wlo)) p1 = 0.f;
        }
        sum += p0 + p1;
        pp[i >> 1] = pack2_f16(p0, p1);
    }
    tmem_st16(taddr, pp);
    return make_float2(sum, ref);
}

// Scales the f16 weights of this thread's two 32-column chunks (first 16
// columns of each, from taddr) by f0 and f1.
__device__ __noinline__ void scale_chunk_weights(uint32_t taddr, float f0, float f1) {
#pragma unroll 1
    for (int c = 0; c < 64; c += 32) {
        const float f = c == 0 ? f0 : f1;
        uint32_t w[32];
        tmem_ld32(taddr + c, w);
        tmem_wait_ld();
        uint32_t q[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) q[i] = pack2_f16(f16lo(w[i]) * f, f16hi(w[i]) * f);
        tmem_st16(taddr + c, q);
    }
    tmem_wait_st();
}

// Eight bf16 values (a 16-byte chunk) as eight f16 values in place order:
// exact for magnitudes in [2^-14, 65504], smaller ones become f16 subnormals
// (absolute error below 2^-25), larger ones saturate to +-65504.
__device__ __forceinline__ uint4 bf16x8_to_f16x8(uint4 w) {
    uint32_t o[4];
    const uint32_t in[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
        asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;"
            : "=r"(o[i])
            : "f"(__uint_as_float(in[i] & 0xffff0000u)), "f"(__uint_as_float(in[i] << 16)));
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// |x| of both halves of an f16 pair (the sign bits cleared)
__device__ __forceinline__ __half2 abs_f16x2(uint32_t w) {
    const uint32_t m = w & 0x7fff7fffu;
    return *reinterpret_cast<const __half2 *>(&m);
}

__device__ __forceinline__ void named_sync(int id) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "n"(kGroup) : "memory");
}

// The two warps of a softmax group that hold the same 32 rows (one warp per
// half of the columns) meet here: barriers 5 .. 5 + 4 kQT - 1, 64 threads each.
__device__ __forceinline__ void pair_sync(int x, int quarter) {
    asm volatile("bar.sync %0, 64;" ::"r"(5 + 4 * x + quarter) : "memory");
}

// The work of one CTA step ("item"): two 128-row Q tiles of one KV head
// against a range of positions.
struct Item {
    int b;          // sequence whose table (and chunk, prefill) the item reads
    int kvh;
    int q0, T, C;   // first query row of the chunk, its tokens, context before it
    int t0;         // first token (prefix mode: sequence) of tile A
    int kv_lo, kv_hi, blk_lo, blk_hi, n_tiles;
    int zidx;       // prefix mode: chunk index (partial row)
    bool has_b;
};

// kPrefix = false: chunked prefill.  Item (pair tile, KV head, sequence): 256
// (token, head) rows of one sequence's chunk, causal over its own table.
// Items are numbered pair-tile fastest (the last, longest tile of a (sequence,
// KV head) first), so that CTAs working at the same time share K/V in L2.
// kPrefix = true: the shared prefix of a decode batch.  Item (pair tile, KV
// head, prefix chunk): 256 (sequence, head) rows across sequences against one
// chunk of the blocks every table starts with (read from the first table);
// each row sees the chunk's positions below its own context length, and the
// CTA writes split-K partials instead of outputs.
template <bool kPrefix>
__device__ __forceinline__ bool describe_item(const PrefillArgs &a, int item, int kv_hi_cap,
                                              bool report_errors, Item &d,
                                              const int *perm = nullptr) {
    const int g = a.group;
    const int tok_per_tile = kRows / g;
    const int lmax = a.max_blocks * kBlockSize;
    if constexpr (!kPrefix) {
        // kv_hi_cap (prefill): 0 = a (sequence, KV head) group's tiles
        // together, longest first; 1 = every group's longest tile, then every
        // group's next one, ...
        const int groups = a.num_seqs * a.num_kv_heads;
        const int x = kv_hi_cap ? item / groups : item % a.n_mt;
        const int rest = kv_hi_cap ? item - x * groups : item / a.n_mt;
        d.kvh = rest % a.num_kv_heads;
        d.b = rest / a.num_kv_heads;
        if (perm != nullptr) d.b = perm[d.b];   // sequences longest first
        const int mt = a.n_mt - 1 - x;
        d.q0 = a.query_start[d.b];
        d.T = a.query_start[d.b + 1] - d.q0;
        const int L = a.context_lens[d.b];
        if (d.T < 0 || d.T > L || L > lmax) {
            if (report_errors && x == 0 && d.kvh == 0) report(a.status, PA_DEV_BAD_CONTEXT_LEN);
            return false;
        }
        if (report_errors && d.T > a.max_query_len && x == 0 && d.kvh == 0)
            report(a.status, PA_DEV_BAD_QUERY_LEN);
        d.t0 = mt * kQT * tok_per_tile;
        if (d.t0 >= d.T) return false;
        d.C = L - d.T;
        const int last_tok = min(d.T, d.t0 + kQT * tok_per_tile) - 1;
        d.kv_hi = d.C + last_tok + 1;
        d.kv_lo = a.window > 0 ? max(0, d.C + d.t0 + 1 - a.window) : 0;
        d.blk_lo = d.kv_lo / kBlockSize;
        d.blk_hi = (d.kv_hi + kBlockSize - 1) / kBlockSize;
        d.zidx = 0;
    } else {
        const int x = item % a.n_mt;
        const int rest = item / a.n_mt;
        d.kvh = rest % a.num_kv_heads;
        d.zidx = rest / a.num_kv_heads;
        d.b = 0;                                          // the shared blocks: first table
        d.q0 = 0;
        d.T = a.num_seqs;                                 // "tokens" are the sequences
        d.C = 0;
        d.t0 = x * kQT * tok_per_tile;
        d.blk_lo = d.zidx * a.chunk_blocks;
        d.blk_hi = min(a.prefix_blocks, d.blk_lo + a.chunk_blocks);
        d.kv_lo = d.blk_lo * kBlockSize;
        // positions past every row's context are never attended: their V rows
        // are zeroed like a context's tail
        d.kv_hi = max(d.kv_lo, min(d.blk_hi * kBlockSize, kv_hi_cap));
    }
    d.has_b = d.t0 + tok_per_tile < d.T;
    d.n_tiles = (d.blk_hi - d.blk_lo + 7) / 8;
    return true;
}

// AND of `v` over the kGroup threads of softmax group x (named barrier 3 + x).
__device__ __forceinline__ bool group_all(int x, bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v), "r"(3 + x), "n"(kGroup)
        : "memory");
    return r != 0;
}

// A persistent CTA (one per SM) works through items.  Prefill takes them in
// order from a ticket counter (a.work_counter, zero at launch), so CTAs that
// finish early take more; prefix mode has one item per CTA (its block index,
// known to every warp).  In prefill the producer warp fetches the next item
// while the current one runs and passes it to the other warps through a
// two-entry queue in shared memory;
// every barrier phase is counted across items, so the next item's Q and K/V
// loads and its first QK^T products start while the last P.V products and the
// output of the item before are still in flight.
template <bool kPrefix>
__global__ void __launch_bounds__(kThreads, 1)
    pa_attn_tc_kernel(const __grid_constant__ CUtensorMap qmap,
                      const __grid_constant__ CUtensorMap kmap,
                      const __grid_constant__ CUtensorMap vmap, const PrefillArgs a) {
    // Prefix mode lets the suffix decode launched after it start once all of
    // its CTAs have started.  Normally that comes after its own wait for the
    // kernels before it, since the suffix reads what they wrote without waiting
    // itself.  With FP8 pools the kernel before it is the prefix widening,
    // every CTA of which waited for all earlier kernels before this kernel
    // could start, so the suffix is released at once and only this kernel
    // waits for the widened prefix.
    const bool early_release = kPrefix && a.staged;
    if (early_release) grid_dependents_launch();
    grid_dependency_wait();
    if (!early_release) grid_dependents_launch();
    const int g = a.group;
    const int tok_per_tile = kRows / g;
    const int lmax = a.max_blocks * kBlockSize;

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    if (smem_u32(smem_raw) & 1023u) {
        if (threadIdx.x == 0) report(a.status, PA_DEV_SMEM_ALIGN);
        return;
    }
    uint8_t *base = smem_raw;
    uint8_t *sQ = base + kOffQ;
    uint8_t *sK = base + kOffK;
    uint8_t *sV = base + kOffV;
    uint64_t *bars = reinterpret_cast<uint64_t *>(base + kOffBar);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(base + kOffBar + kNumBars * 8);
    volatile int *fail = reinterpret_cast<volatile int *>(base + kOffBar + kNumBars * 8 + 4);
    int *s_maxl = reinterpret_cast<int *>(base + kOffBar + kNumBars * 8 + 8);
    volatile int *s_item = reinterpret_cast<volatile int *>(base + kOffBar + kNumBars * 8 + 12);  // [2]

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        mbar_init(&bars[kQFull], 1);
        mbar_init(&bars[kQFree], 1);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&bars[kKFull + s], 1);
            mbar_init(&bars[kKEmpty + s], 1);
            mbar_init(&bars[kVFull + s], 1);
            mbar_init(&bars[kVEmpty + s], 1);
            mbar_init(&bars[kVConv + s], kConvThreads);
        }
        for (int x = 0; x < kQT; ++x) {
            mbar_init(&bars[kSFull + x], 1);
            mbar_init(&bars[kPFull + x], kGroup);
            mbar_init(&bars[kPvDone + x], 1);
            mbar_init(&bars[kOFree + x], kGroup);
        }
        for (int q = 0; q < 2; ++q) {
            mbar_init(&bars[kItemFull + q], 1);
            mbar_init(&bars[kItemEmpty + q], 1 + kQT * kGroup + kConvThreads);
        }
        mbar_init(&bars[kDrain], 1);
        *fail = 0;
        *s_maxl = 0;
        fence_mbar_init();
        tma_prefetch_desc(&qmap);
        tma_prefetch_desc(&kmap);
        tma_prefetch_desc(&vmap);
    }
    __syncthreads();   // s_maxl is zero
    if constexpr (kPrefix) {
        // this CTA's one item: the longest context among its rows bounds the
        // positions attended, and (KV head 0) every sequence of these rows
        // must list the chunk's blocks
        const int kvh = blockIdx.y;
        const int t0 = blockIdx.x * kQT * tok_per_tile;
        const int nseq = min(a.num_seqs - t0, kQT * tok_per_tile);
        for (int i = threadIdx.x; i < nseq; i += kThreads) {
            int L = a.context_lens[t0 + i];
            L = L < 0 ? 0 : (L > lmax ? lmax : L);
            atomicMax(s_maxl, L);
        }
        if (kvh == 0) {
            const int blk_lo = blockIdx.z * a.chunk_blocks;
            const int nblk = min(a.prefix_blocks, blk_lo + a.chunk_blocks) - blk_lo;
            for (int i = threadIdx.x; i < nseq * nblk; i += kThreads) {
                const int sq = t0 + i / nblk, jb = blk_lo + i % nblk;
                if (a.block_tables[(size_t)sq * a.max_blocks + jb] != a.block_tables[jb])
                    report(a.status, PA_DEV_PREFIX_MISMATCH);
            }
        }
    } else if (warp == 2) {
        // Item order for this call: when the chunks bring more tokens than the
        // contexts held before them (fresh prompts), a group's causal tiles
        // range from short to long and the tiles go longest first across all
        // groups; otherwise a group's tiles stay together (their K/V shared in
        // L2 by the CTAs working at the same time).
        long long cached = 0, fresh = 0;
        for (int i = lane; i < a.num_seqs; i += 32) {
            const int T = a.query_start[i + 1] - a.query_start[i];
            const int L = a.context_lens[i];
            fresh += T > 0 ? T : 0;
            cached += L - T > 0 ? L - T : 0;
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
            cached += __shfl_xor_sync(0xffffffffu, cached, o);
            fresh += __shfl_xor_sync(0xffffffffu, fresh, o);
        }
        if (lane == 0) *s_maxl = cached < fresh ? 1 : 0;
        // sequences longest context first (ties by index), so that the call
        // ends on the shortest ones
        if (a.num_seqs <= kPermMax) {
            int *perm = reinterpret_cast<int *>(base + kOffPerm);
            for (int i = lane; i < a.num_seqs; i += 32) {
                const int li = a.context_lens[i];
                int r = 0;
                for (int j = 0; j < a.num_seqs; ++j) {
                    const int lj = a.context_lens[j];
                    r += (lj > li) | ((lj == li) & (j < i));
                }
                perm[r] = i;
            }
        }
    }
    if (warp == 1) tmem_alloc(tslot, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    // prefix mode: the longest context of the CTA's rows; prefill: the item order
    const int kv_hi_cap = *s_maxl;
    const int *perm = (!kPrefix && a.num_seqs <= kPermMax) ? reinterpret_cast<const int *>(base + kOffPerm)
                                                           : nullptr;

    if (warp == 0) {
        // ---------------- TMA producer (and item fetch) ----------------
        if (lane == 0) {
            int item_issued = -1;                   // items whose Q load was issued
            uint32_t issued_k = 0, issued_v = 0;    // K/V steps issued (global count)
            uint32_t gstep = 0;                     // K/V steps of earlier items
            bool ok = true;
            bool first = true;
            for (int it = 0;; ++it) {
                // next non-empty item, or -1
                int item = -1;
                Item d;
                if constexpr (kPrefix) {
                    if (first) {
                        item = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
                        describe_item<true>(a, item, kv_hi_cap, true, d);
                    }
                } else {
                    for (;;) {
                        const int t = (int)atomicAdd(a.work_counter, 1u);
                        if (t >= a.num_items) break;
                        if (describe_item<false>(a, t, kv_hi_cap, true, d, perm)) {
                            item = t;
                            break;
                        }
                    }
                }
                first = false;
                if (!ok) item = -1;
                if constexpr (!kPrefix) {
                    // prefix mode has no queue: every warp knows its one item
                    const int slot = it & 1;
                    if (it >= 2 && !wait_or_fail(&bars[kItemEmpty + slot], ((it >> 1) - 1) & 1, fail, a.status))
                        item = -1;
                    s_item[slot] = item;
                    mbar_arrive(&bars[kItemFull + slot]);
                }
                if (item < 0) break;
                // Q (both tiles) once the last QK^T of the item before has run
                if (it >= 1 && !wait_or_fail(&bars[kQFree], (it - 1) & 1, fail, a.status)) {
                    ok = false;
                    continue;
                }
                const int nq = d.has_b ? kQT : 1;
                mbar_arrive_expect_tx(&bars[kQFull], nq * kTile);
                for (int x = 0; x < nq; ++x) {
                    const int row0 = d.q0 + d.t0 + x * tok_per_tile;
                    tma_load_4d(sQ + x * kTile, &qmap, 0, 0, d.kvh, row0, &bars[kQFull]);
                    tma_load_4d(sQ + x * kTile + kHalf, &qmap, 64, 0, d.kvh, row0, &bars[kQFull]);
                }
                item_issued = it;
                const int32_t *trow = a.block_tables + (size_t)d.b * a.max_blocks;
                // K/V step j of this item, as rows of the pool maps (8 blocks at most)
                auto step_rows = [&](int j, int (&rows)[8]) {
                    const int blk0 = d.blk_lo + 8 * j;
                    const int nb = min(8, d.blk_hi - blk0);
                    for (int i = 0; i < nb; ++i) {
                        int phys = a.staged ? blk0 + i : trow[blk0 + i];
                        if ((unsigned)phys >= (unsigned)a.num_blocks) {
                            report(a.status, PA_DEV_BAD_BLOCK_ID);
                            phys = 0;
                        }
                        rows[i] = (phys * a.num_kv_heads + d.kvh) * kBlockSize;
                    }
                    return nb;
                };
                for (int j = 0; ok && j < d.n_tiles; ++j) {
                    const uint32_t gs = gstep + j;
                    const int s = gs % kStages;
                    const uint32_t ph = (gs / kStages) & 1u;   // this use of stage s
                    int rows[8];
                    const int nb = step_rows(j, rows);
                    if (gs >= kStages && !wait_or_fail(&bars[kKEmpty + s], ph ^ 1u, fail, a.status)) {
                        ok = false;
                        break;
                    }
                    uint8_t *kd = sK + s * kTile;
                    mbar_arrive_expect_tx(&bars[kKFull + s], nb * 4096);
                    for (int i = 0; i < nb; ++i) {
                        tma_load_2d(kd + i * 2048, &kmap, 0, rows[i], &bars[kKFull + s]);
                        tma_load_2d(kd + kHalf + i * 2048, &kmap, 64, rows[i], &bars[kKFull + s]);
                    }
                    issued_k = gs + 1;
                    if (gs >= kStages && !wait_or_fail(&bars[kVEmpty + s], ph ^ 1u, fail, a.status)) {
                        ok = false;
                        break;
                    }
                    uint8_t *vd = sV + s * kTile;
                    mbar_arrive_expect_tx(&bars[kVFull + s], nb * 4096);
                    for (int i = 0; i < nb; ++i) {
                        tma_load_2d(vd + i * 2048, &vmap, 0, rows[i], &bars[kVFull + s]);
                        tma_load_2d(vd + kHalf + i * 2048, &vmap, 64, rows[i], &bars[kVFull + s]);
                    }
                    issued_v = gs + 1;
                }
                gstep += d.n_tiles;
            }
            // drain: no copy of ours may still be landing when the CTA leaves
            if (item_issued >= 0) (void)mbar_wait_bounded(&bars[kQFull], item_issued & 1);
            for (uint32_t j = issued_k > kStages ? issued_k - kStages : 0; j < issued_k; ++j)
                (void)mbar_wait_bounded(&bars[kKFull + j % kStages], (j / kStages) & 1);
            for (uint32_t j = issued_v > kStages ? issued_v - kStages : 0; j < issued_v; ++j)
                (void)mbar_wait_bounded(&bars[kVFull + j % kStages], (j / kStages) & 1);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            constexpr uint32_t idS = idesc_bf16_f32(kRows, kKv, false);
            constexpr uint32_t idPV = idesc_f16_f32(kRows, kD, true);
            const uint32_t q_u = smem_u32(sQ), k_u = smem_u32(sK), v_u = smem_u32(sV);
            uint32_t gstep = 0;
            uint32_t pcount[kQT] = {0, 0};   // P phases per Q tile (global)
            bool ok = true;
            auto issue_s = [&](int x, uint32_t gs) {
                const uint32_t qb = q_u + x * kTile;
                const uint32_t kb = k_u + (gs % kStages) * kTile;
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const uint32_t o = (k >> 2) * kHalf + (k & 3) * 32;
                    umma_bf16(tmem + col_s(x), sw128_desc(qb + o, 16, 1024),
                              sw128_desc(kb + o, 16, 1024), idS, k > 0 ? 1u : 0u);
                }
                umma_commit(&bars[kSFull + x]);
            };
            // P (f16 pairs) of tokens [16k, 16k + 16) sits in the 32-column
            // chunk k / 2 of the S buffer, from column 32 (k / 2) + 8 (k % 2)
            auto issue_pv = [&](int x, uint32_t gs, int j, int it) -> bool {
                if (!wait_or_fail(&bars[kPFull + x], pcount[x] & 1, fail, a.status)) return false;
                ++pcount[x];
                // the first P.V of an item overwrites O: the item before must
                // have read it out
                if (j == 0 && it >= 1 && !wait_or_fail(&bars[kOFree + x], (it - 1) & 1, fail, a.status))
                    return false;
                tc_fence_after();
                const uint32_t vb = v_u + (gs % kStages) * kTile;
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const uint32_t pc = tmem + col_s(x) + 32 * (k >> 1) + 8 * (k & 1);
                    const uint64_t vdesc = sw128_desc(vb + k * 2048, kHalf, 1024);
                    umma_bf16_tmem_a(tmem + col_o(x), pc, vdesc, idPV, (j > 0 || k > 0) ? 1u : 0u);
                }
                umma_commit(&bars[kPvDone + x]);
                return true;
            };
            for (int it = 0; ok; ++it) {
                int item;
                if constexpr (kPrefix) {
                    item = it == 0 ? (int)(blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z)) : -1;
                } else {
                    const int slot = it & 1;
                    if (!wait_or_fail(&bars[kItemFull + slot], (it >> 1) & 1, fail, a.status)) break;
                    item = s_item[slot];
                    mbar_arrive(&bars[kItemEmpty + slot]);
                }
                if (item < 0) break;
                Item d;
                describe_item<kPrefix>(a, item, kv_hi_cap, false, d, perm);
                const int n = d.n_tiles;
                if (!wait_or_fail(&bars[kQFull], it & 1, fail, a.status) ||
                    !wait_or_fail(&bars[kKFull + gstep % kStages], (gstep / kStages) & 1, fail, a.status))
                    break;
                tc_fence_after();
                issue_s(0, gstep);
                if (d.has_b) issue_s(1, gstep);
                umma_commit(&bars[kKEmpty + gstep % kStages]);
                if (n == 1) umma_commit(&bars[kQFree]);
                for (int j = 0; ok && j < n; ++j) {
                    const uint32_t gs = gstep + j, gk = gs + 1;
                    const bool more = j + 1 < n;
                    if (!wait_or_fail(&bars[kVConv + gs % kStages], (gs / kStages) & 1, fail, a.status) ||
                        !issue_pv(0, gs, j, it)) {
                        ok = false;
                        break;
                    }
                    if (more) {
                        if (!wait_or_fail(&bars[kKFull + gk % kStages], (gk / kStages) & 1, fail, a.status)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        issue_s(0, gk);
                    }
                    if (d.has_b && !issue_pv(1, gs, j, it)) {
                        ok = false;
                        break;
                    }
                    umma_commit(&bars[kVEmpty + gs % kStages]);
                    if (more) {
                        if (d.has_b) issue_s(1, gk);
                        umma_commit(&bars[kKEmpty + gk % kStages]);
                        if (j + 2 == n) umma_commit(&bars[kQFree]);   // the item's last QK^T is issued
                    }
                }
                // every MMA of this item has completed once kDrain flips
                umma_commit(&bars[kDrain]);
                gstep += n;
            }
        }
    } else if (warp >= kConvWarp0) {
        // ---------------- V conversion ----------------
        // Each landed V tile becomes f16 in place before its P.V products:
        // rows of positions outside [kv_lo, kv_hi) may hold anything (NaN
        // included) and are zeroed instead, so that 0 * row stays 0.  Thread t
        // takes the 16-byte chunks t, t + kConvThreads, ... (a chunk's row is
        // its offset within the 64-column half over 128 bytes; the swizzle only
        // permutes chunks within a row).
        const int ct = threadIdx.x - kConvWarp0 * 32;
        uint32_t gstep = 0;
        // running maximum of |f16 value| written (NaN ignored): 65504 is no bf16
        // value, so a maximum of 65504 means an input outside f16's range saturated
        __half2 vmax = __float2half2_rn(0.f);
        bool ok = true;
        for (int it = 0;; ++it) {
            int item;
            if constexpr (kPrefix) {
                item = it == 0 ? (int)(blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z)) : -1;
            } else {
                const int slot = it & 1;
                const bool got_item = wait_or_fail(&bars[kItemFull + slot], (it >> 1) & 1, fail, a.status);
                item = got_item ? s_item[slot] : -1;
                mbar_arrive(&bars[kItemEmpty + slot]);
            }
            if (item < 0) break;
            Item d;
            describe_item<kPrefix>(a, item, kv_hi_cap, false, d, perm);
            for (int j = 0; ok && j < d.n_tiles; ++j) {
                const uint32_t gs = gstep + j;
                const int st = gs % kStages;
                if (!wait_or_fail(&bars[kVFull + st], (gs / kStages) & 1, fail, a.status)) {
                    ok = false;
                    break;
                }
                const int k0_tile = (d.blk_lo + 8 * j) * kBlockSize;
                const bool edge = k0_tile < d.kv_lo || k0_tile + kKv > d.kv_hi;
                uint4 *vt = reinterpret_cast<uint4 *>(sV + st * kTile);
#pragma unroll 8
                for (int i = 0; i < kTile / 16 / kConvThreads; ++i) {
                    const int c = ct + i * kConvThreads;
                    const int kp = k0_tile + (c % (kHalf / 16)) / 8;
                    const uint4 w = vt[c];
                    const uint4 h = (edge && (kp < d.kv_lo || kp >= d.kv_hi)) ? make_uint4(0, 0, 0, 0)
                                                                              : bf16x8_to_f16x8(w);
                    vt[c] = h;
                    vmax = __hmax2(__hmax2(vmax, abs_f16x2(h.x)),
                                   __hmax2(__hmax2(abs_f16x2(h.y), abs_f16x2(h.z)), abs_f16x2(h.w)));
                }
                fence_proxy_async_smem();
                mbar_arrive(&bars[kVConv + st]);
            }
            gstep += d.n_tiles;
        }
        const uint32_t vm = *reinterpret_cast<const uint32_t *>(&vmax);
        if ((vm & 0xffffu) == 0x7bffu || (vm >> 16) == 0x7bffu) report(a.status, PA_DEV_RANGE);
    } else {
        // ---------------- softmax groups ----------------
        const int x = (warp - 2) / (kGroup / 32);     // Q tile of this group
        const int gw = (warp - 2) % (kGroup / 32);    // warp within the group
        const int quarter = warp & 3;
        const int part = gw >> 2;                     // columns [kCols * part, + kCols)
        const int r = quarter * 32 + lane;            // tile row = TMEM lane
        const int tr = r / g;
        const uint32_t lane_off = ((uint32_t)(quarter * 32) << 16) + part * kCols;
        const uint32_t s_base = tmem + col_s(x) + lane_off;
        const uint32_t o_base = tmem + col_o(x) + lane_off;
        float *red = reinterpret_cast<float *>(base + kOffRed) + x * 2 * kSplit * kRows;
        uint32_t sc = 0;      // S / P / P.V phases of this group (global)
        uint32_t ex = 0;      // exchanges through `red` (their slot alternates)
        uint32_t gstep = 0;   // K/V steps of earlier items
        bool ok = true;
        for (int it = 0;; ++it) {
            int item;
            if constexpr (kPrefix) {
                item = it == 0 ? (int)(blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z)) : -1;
            } else {
                const int slot = it & 1;
                const bool got_item = warp_wait(&bars[kItemFull + slot], (it >> 1) & 1, fail, a.status);
                item = got_item ? s_item[slot] : -1;
                mbar_arrive(&bars[kItemEmpty + slot]);
            }
            // every thread of the group takes the same decision, so that all of
            // them reach the group's named barriers equally often
            if (!group_all(x, item >= 0 && ok && !*fail)) break;
            Item d;
            describe_item<kPrefix>(a, item, kv_hi_cap, false, d, perm);
            const int n_tiles = d.n_tiles;
            if (x == 0 || d.has_b) {
                const float sl2k = a.k_scales != nullptr ? a.scale_log2 * a.k_scales[d.kvh] : a.scale_log2;
                const int tx0 = d.t0 + x * tok_per_tile;      // first token (sequence) of this tile
                const int ntok = max(0, min(tok_per_tile, d.T - tx0));
                const bool real = tr < ntok;
                // this row attends to positions [wlo, qpos]; a 32-column chunk
                // needs no mask when it lies inside [qpos_lo_win, qpos_lo] for
                // every row of the tile
                int qpos, qpos_lo, qpos_hi, wlo;
                if constexpr (!kPrefix) {
                    qpos = d.C + tx0 + min(tr, max(ntok, 1) - 1);
                    qpos_lo = d.C + tx0;
                    qpos_hi = d.C + tx0 + max(ntok, 1) - 1;
                    wlo = a.window > 0 ? qpos + 1 - a.window : INT_MIN;
                } else {
                    int L = real ? a.context_lens[tx0 + tr] : 0;
                    L = L < 0 ? 0 : (L > lmax ? lmax : L);
                    qpos = min(L, d.blk_hi * kBlockSize) - 1;   // last attended position
                    qpos_lo = -1;                                // decided per warp below
                    qpos_hi = 0;
                    wlo = INT_MIN;
                }
                // Whether the 32 columns from position kc need the per-element
                // mask: in prefill, unless they lie inside every row's range of
                // the tile; in prefix mode (rows of many sequences), unless they
                // lie inside every row's range of this warp (one vote per chunk).
                auto chunk_masked = [&](int kc) -> bool {
                    if constexpr (kPrefix) return __any_sync(0xffffffffu, kc + 31 > qpos);
                    return (kc + 31 > qpos_lo) || (a.window > 0 && kc < qpos_hi + 1 - a.window);
                };
                // The row's reference (log2 units): an integer, or -inf before the
                // row has seen a position; O and l are relative to it.
                float m_used = -INFINITY, l = 0.f;
                // Every thread of the group runs every iteration and reaches the
                // named barrier the same number of times, even after a wait gave
                // up (then it only skips the work), so that no barrier waits forever.
                for (int j = 0; j < n_tiles; ++j) {
                    const bool got = ok && warp_wait(&bars[kSFull + x], sc & 1, fail, a.status);
                    const int k0 = (d.blk_lo + 8 * j) * kBlockSize + part * kCols;   // column 0's position
                    // One pass over S: each 32-column chunk's weights P = 2^(s *
                    // scale_log2 - ref) are computed against this thread's current
                    // reference ref and written over the chunk in f16, unless they
                    // sum to more than 2^15 (a weight could leave f16's range, or
                    // there is no reference yet and the sum is infinite): then ref
                    // rises to the next integer at or above the chunk's largest
                    // scaled score and the chunk is computed again.  Each chunk keeps
                    // the reference it was written with (cref) and its weight sum.
                    float mref = m_used;
                    float cref0 = m_used, cref1 = m_used, csum0 = 0.f, csum1 = 0.f;
                    static_assert(kCols == 64, "two 32-column chunks per softmax thread");
                    if (got) {
                        tc_fence_after();
                        const uint64_t k2 = f2_pack(sl2k, sl2k);
#pragma unroll 1
                        for (int c = 0; c < kCols; c += 32) {
                            const int kc = k0 + c;
                            const bool masked = chunk_masked(kc);
                            uint32_t pp[16];
                            float sum;
                            {
                                uint32_t v[32];
                                tmem_ld32(s_base + c, v);
                                tmem_wait_ld();
                                // pairs of columns on f32x2 arithmetic: one FMA and
                                // one add instruction for two weights; 11 significant
                                // bits (f16) keep the weights within the output
                                // tolerance, where bf16's 8 bits do not
                                const uint64_t nm2 = f2_pack(-mref, -mref);
                                uint64_t ps2[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
#pragma unroll
                                for (int i = 0; i < 32; i += 2) {
                                    float x0, x1;
                                    f2_unpack(f2_fma(f2_pack(__uint_as_float(v[i]), __uint_as_float(v[i + 1])), k2, nm2), x0, x1);
                                    float p0 = ex2_approx(x0);
                                    float p1 = ex2_approx(x1);
                                    if (masked) {
                                        if (!(kc + i <= qpos && kc + i >= wlo)) p0 = 0.f;
                                        if (!(kc + i + 1 <= qpos && kc + i + 1 >= wlo)) p1 = 0.f;
                                    }
                                    ps2[(i >> 1) & 1] = f2_add(ps2[(i >> 1) & 1], f2_pack(p0, p1));
                                    pp[i >> 1] = pack2_f16(p0, p1);
                                }
                                float a0, a1, b0, b1;
                                f2_unpack(ps2[0], a0, a1);
                                f2_unpack(ps2[1], b0, b1);
                                sum = (a0 + b0) + (a1 + b1);
                            }
                            const bool over = !(sum <= kChunkSumMax);
                            if (__any_sync(0xffffffffu, over)) {
                                // the whole warp (warp-wide tensor-memory access); S is
                                // still in place, P not yet written
                                const float2 r2 = chunk_weights_again(s_base + c, sl2k, mref, over, masked,
                                                                      kc, qpos, wlo);
                                sum = r2.x;
                                mref = r2.y;
                            } else {
                                tmem_st16(s_base + c, pp);
                            }
                            if (c == 0) {
                                cref0 = mref;
                                csum0 = sum;
                            } else {
                                cref1 = mref;
                                csum1 = sum;
                            }
                        }
                        tmem_wait_st();
                    }
                    // the two threads of the row agree on the larger reference
                    const int rp = ex & 1;
                    ++ex;
                    red[(rp * kSplit + part) * kRows + r] = mref;
                    pair_sync(x, quarter);
                    float rref = mref;
#pragma unroll
                    for (int o = 1; o < kSplit; ++o)
                        rref = fmaxf(rref, red[(rp * kSplit + ((part + o) % kSplit)) * kRows + r]);
                    const uint32_t my_sc = sc++;
                    if (!got) {
                        ok = false;
                        continue;
                    }
                    // chunks written against a smaller reference than the row's are
                    // scaled by the exact power of two between them (0 when their
                    // reference was -inf: all their weights are 0); the warp does it
                    // together (warp-wide tensor-memory access, factor 1 elsewhere)
                    const float f0 = pow2_diff(cref0, rref);
                    const float f1 = pow2_diff(cref1, rref);
                    if (__any_sync(0xffffffffu, f0 != 1.f || f1 != 1.f)) scale_chunk_weights(s_base, f0, f1);
                    const float psum = csum0 * f0 + csum1 * f1;
                    // O and l follow when the row's reference moved; the warp
                    // rescales O together once every PV of this tile issued so far
                    // has landed
                    const bool need = rref > m_used;
                    const float alpha = need ? pow2_diff(m_used, rref) : 1.f;   // 0 while m_used is -inf
                    if (j >= 1 && __any_sync(0xffffffffu, need)) {
                        if (!warp_wait(&bars[kPvDone + x], (my_sc - 1) & 1, fail, a.status)) {
                            ok = false;
                            continue;
                        }
                        tc_fence_after();
#pragma unroll 1
                        for (int c = 0; c < kCols; c += 32) {
                            uint32_t o[32];
                            tmem_ld32(o_base + c, o);
                            tmem_wait_ld();
                            const uint64_t a2 = f2_pack(alpha, alpha);
#pragma unroll
                            for (int i = 0; i < 32; i += 2) {
                                float r0, r1;
                                f2_unpack(f2_mul(f2_pack(__uint_as_float(o[i]), __uint_as_float(o[i + 1])), a2), r0, r1);
                                o[i] = __float_as_uint(r0);
                                o[i + 1] = __float_as_uint(r1);
                            }
                            tmem_st32(o_base + c, o);
                        }
                        tmem_wait_st();
                    }
                    if (need) {
                        l *= alpha;
                        m_used = rref;
                    }
                    l += psum;
                    tc_fence_before();
                    mbar_arrive(&bars[kPFull + x]);
                }
                // the row sum is the parts' sums (all against the row's reference),
                // exchanged in the slots of the other parity
                const int sx = ex & 1;
                ++ex;
                red[(sx * kSplit + part) * kRows + r] = l;
                pair_sync(x, quarter);
                float l_row = l;
#pragma unroll
                for (int o = 1; o < kSplit; ++o) l_row += red[(sx * kSplit + ((part + o) % kSplit)) * kRows + r];
                const bool drained = warp_wait(&bars[kDrain], it & 1, fail, a.status);
                if constexpr (kPrefix) {
                    // split-K partial of this chunk: (max, sum) and the unnormalised
                    // output, in the partial row of (sequence, head, chunk).  The
                    // rows pass through shared memory (the K/V rings are idle once
                    // the CTA's one item has drained) so that each 512-byte row
                    // leaves in one coalesced store; a thread's own columns would
                    // scatter over 32 rows per store.  Chunk c of tile row rr sits
                    // at c ^ (rr % 32) of the row (fewest bank conflicts both ways).
                    const bool go = group_all(x, __all_sync(0xffffffffu, ok) && drained);
                    float4 *stage = reinterpret_cast<float4 *>(sK) + (size_t)x * kRows * (kD / 4);
                    const float vs = a.v_scales != nullptr ? a.v_scales[d.kvh] : 1.f;
                    if (go) {
                        tc_fence_after();
                        float4 *srow = stage + (size_t)r * (kD / 4);
#pragma unroll 1
                        for (int c = 0; c < kCols; c += 32) {
                            uint32_t o[32];
                            tmem_ld32(o_base + c, o);
                            tmem_wait_ld();
#pragma unroll
                            for (int q = 0; q < 8; ++q)
                                srow[((part * kCols + c) / 4 + q) ^ (r & 31)] =
                                    make_float4(__uint_as_float(o[4 * q]) * vs, __uint_as_float(o[4 * q + 1]) * vs,
                                                __uint_as_float(o[4 * q + 2]) * vs,
                                                __uint_as_float(o[4 * q + 3]) * vs);
                        }
                        if (real && part == 0) {
                            const size_t prow = ((size_t)(tx0 + tr) * a.num_q_heads + d.kvh * g + (r % g)) *
                                                    a.max_parts + d.zidx;
                            a.part_ml[prow] = make_float2(l_row > 0.f ? m_used : -INFINITY, l_row);
                        }
                    }
                    named_sync(1 + x);
                    if (go) {
                        // warp gw of the group writes tile rows [16 gw, 16 gw + 16)
                        for (int rr = gw * (kRows / (kGroup / 32)); rr < (gw + 1) * (kRows / (kGroup / 32)); ++rr) {
                            const int trr = rr / g;
                            if (trr >= ntok) continue;
                            const size_t prow = ((size_t)(tx0 + trr) * a.num_q_heads + d.kvh * g + (rr % g)) *
                                                    a.max_parts + d.zidx;
                            reinterpret_cast<float4 *>(a.part_o + prow * kD)[lane] =
                                stage[(size_t)rr * (kD / 4) + (lane ^ (rr & 31))];
                        }
                    }
                } else if (__all_sync(0xffffffffu, ok) && drained) {
                    tc_fence_after();
                    const float inv = l_row > 0.f ? 1.f / l_row : 0.f;
                    __nv_bfloat16 *orow = static_cast<__nv_bfloat16 *>(a.out) +
                                          ((size_t)(d.q0 + tx0 + tr) * a.num_q_heads + d.kvh * g + (r % g)) * kD +
                                          part * kCols;
#pragma unroll 1
                    for (int c = 0; c < kCols; c += 32) {
                        uint32_t o[32];
                        tmem_ld32(o_base + c, o);
                        tmem_wait_ld();
                        if (real) {
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                uint4 w;
                                w.x = pack2_bf16(__uint_as_float(o[8 * q + 0]) * inv, __uint_as_float(o[8 * q + 1]) * inv);
                                w.y = pack2_bf16(__uint_as_float(o[8 * q + 2]) * inv, __uint_as_float(o[8 * q + 3]) * inv);
                                w.z = pack2_bf16(__uint_as_float(o[8 * q + 4]) * inv, __uint_as_float(o[8 * q + 5]) * inv);
                                w.w = pack2_bf16(__uint_as_float(o[8 * q + 6]) * inv, __uint_as_float(o[8 * q + 7]) * inv);
                                *reinterpret_cast<uint4 *>(orow + c + 8 * q) = w;
                            }
                        }
                    }
                }
                if (!drained) ok = false;
            } else {
                // tile B has no rows in this item: keep the drain phase in step
                if (!warp_wait(&bars[kDrain], it & 1, fail, a.status)) ok = false;
            }
            // O of this tile has been read: the next item's first P.V may overwrite it
            tc_fence_before();
            mbar_arrive(&bars[kOFree + x]);
            gstep += n_tiles;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// Tensor maps of one call: the query as [rows][KV head][head of the group]
// [head_dim] (a box of 128 / group rows x group heads x 64 elements is one
// 128-row tile), and each pool as [num_blocks * num_kv_heads * 16 rows]
// [head_dim] with 16-row boxes.
pa_status encode_maps(const void *query, int query_rows, int num_q_heads, int num_kv_heads,
                      const void *key_cache, const void *value_cache, int64_t pool_rows,
                      CUtensorMap *qmap, CUtensorMap *kmap, CUtensorMap *vmap) {
    auto enc = encoder();
    if (enc == nullptr) return cuda_failure(cudaErrorInvalidValue, "cuTensorMapEncodeTiled lookup");
    const int group = num_q_heads / num_kv_heads;
    {
        cuuint64_t dims[4] = {(cuuint64_t)kD, (cuuint64_t)group, (cuuint64_t)num_kv_heads,
                              (cuuint64_t)query_rows};
        cuuint64_t strides[3] = {(cuuint64_t)kD * 2, (cuuint64_t)group * kD * 2,
                                 (cuuint64_t)num_q_heads * kD * 2};
        cuuint32_t box[4] = {64, (cuuint32_t)group, 1, (cuuint32_t)(kRows / group)};
        cuuint32_t estr[4] = {1, 1, 1, 1};
        if (enc(qmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(query), dims, strides,
                box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cuda_failure(cudaErrorInvalidValue, "cuTensorMapEncodeTiled(query)");
    }
    for (int which = 0; which < 2; ++which) {
        cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)pool_rows};
        cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
        cuuint32_t box[2] = {64, (cuuint32_t)kBlockSize};
        cuuint32_t estr[2] = {1, 1};
        CUtensorMap *m = which == 0 ? kmap : vmap;
        const void *pool = which == 0 ? key_cache : value_cache;
        if (enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(pool), dims, strides,
                box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cuda_failure(cudaErrorInvalidValue, "cuTensorMapEncodeTiled(pool)");
    }
    return PA_OK;
}

template <bool kPrefix>
pa_status launch_tc(const CUtensorMap &qmap, const CUtensorMap &kmap, const CUtensorMap &vmap,
                    const PrefillArgs &a, dim3 grid, cudaStream_t stream) {
    auto kernel = pa_attn_tc_kernel<kPrefix>;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSmemBytes);
    if (e != cudaSuccess) return cuda_failure(e, "cudaFuncSetAttribute(tensor-core attention)");
    e = launch_chained(kernel, grid, dim3(kThreads), (size_t)kSmemBytes, stream, qmap, kmap, vmap, a);
    if (e != cudaSuccess) return cuda_failure(e, "pa_attn_tc_kernel launch");
    count_launches(1);
    return PA_OK;
}

// Streaming multiprocessors of the current device (152 when the runtime
// cannot tell).
int prefill_sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
        (void)cudaGetLastError();
        return 152;
    }
    return n;
}

bool group_ok(int group) {
    return group == 1 || group == 2 || group == 4 || group == 8 || group == 16;
}

}  // namespace

bool prefix_tc_supported(int head_dim, int num_q_heads, int num_kv_heads) {
    return head_dim == kD && num_kv_heads > 0 && num_q_heads % num_kv_heads == 0 &&
           group_ok(num_q_heads / num_kv_heads);
}

// Prefix chunk (in blocks, whole 8-block K/V tiles) that gives about
// PA_PREFIX_TC_CTAS_PER_100_SM / 100 CTAs per SM over (256-row tiles x KV heads
// x chunks).  The prefix runs beside the suffix decode, so it takes only part
// of the GPU: on the 128-sequence mix (63 shared blocks, 8 KV heads) a sixth
// of the SMs (two chunks, 32 CTAs) gave the shortest call; 16 CTAs made the
// prefix the longer of the two, 48 or more slowed the suffix.
#ifndef PA_PREFIX_TC_CTAS_PER_100_SM
#define PA_PREFIX_TC_CTAS_PER_100_SM 15
#endif
int prefix_tc_chunk_blocks(int num_seqs, int num_q_heads, int num_kv_heads, int prefix_blocks,
                           int sm_count) {
    const int group = num_q_heads / num_kv_heads;
    const int64_t tiles = ((int64_t)num_seqs * group + kQT * kRows - 1) / (kQT * kRows);
    const int64_t per_chunk = std::max<int64_t>(1, tiles * num_kv_heads);
    const int64_t target = std::max<int64_t>(1, (int64_t)sm_count * PA_PREFIX_TC_CTAS_PER_100_SM / 100);
    const int64_t want = std::max<int64_t>(1, (target + per_chunk - 1) / per_chunk);
    int cb = (int)((prefix_blocks + want - 1) / want);
    cb = ((cb + 7) / 8) * 8;
    return std::max(8, std::min(cb, ((prefix_blocks + 7) / 8) * 8));
}

pa_status launch_prefix_tc(const void *query, const void *key_cache, const void *value_cache,
                           const int32_t *block_tables, const int32_t *context_lens, int num_seqs,
                           int num_q_heads, int num_kv_heads, int max_blocks, int num_blocks,
                           float scale_log2, int prefix_blocks, int chunk_blocks, int chunks,
                           float *part_o, float2 *part_ml, int max_parts, bool staged,
                           const float *k_scales, const float *v_scales, int32_t *status,
                           cudaStream_t stream) {
    const int group = num_q_heads / num_kv_heads;
    const int64_t pool_rows = (int64_t)num_blocks * num_kv_heads * kBlockSize;
    const int64_t tiles = ((int64_t)num_seqs * group + kQT * kRows - 1) / (kQT * kRows);
    if (tiles > 0x7fffffff || num_kv_heads > 65535 || chunks > 65535) return PA_ERR_UNSUPPORTED;
    CUtensorMap qmap, kmap, vmap;
    pa_status st = encode_maps(query, num_seqs, num_q_heads, num_kv_heads, key_cache, value_cache,
                               pool_rows, &qmap, &kmap, &vmap);
    if (st != PA_OK) return st;
    PrefillArgs a = {};
    a.block_tables = block_tables;
    a.context_lens = context_lens;
    a.status = status;
    a.num_seqs = num_seqs;
    a.num_q_heads = num_q_heads;
    a.num_kv_heads = num_kv_heads;
    a.group = group;
    a.max_blocks = max_blocks;
    a.num_blocks = num_blocks;
    a.scale_log2 = scale_log2;
    a.part_o = part_o;
    a.part_ml = part_ml;
    a.max_parts = max_parts;
    a.prefix_blocks = prefix_blocks;
    a.chunk_blocks = chunk_blocks;
    a.staged = staged ? 1 : 0;
    a.k_scales = k_scales;
    a.v_scales = v_scales;
    a.n_mt = (int)tiles;                 // one item per CTA: its block index
    a.num_items = (int)(tiles * num_kv_heads * chunks);
    return launch_tc<true>(qmap, kmap, vmap, a, dim3((unsigned)tiles, (unsigned)num_kv_heads,
                                                      (unsigned)chunks),
                           stream);
}

}  // namespace pa

using namespace pa;

extern "C" size_t pa_prefill_workspace_bytes(void) { return kPrefillWorkspaceBytes; }

extern "C" pa_status pa_prefill(void *out, const void *query, const void *key_cache,
                                const void *value_cache, const int32_t *block_tables,
                                const int32_t *context_lens, const int32_t *query_start,
                                int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                int block_size, int max_blocks_per_seq, int num_blocks,
                                int num_query_tokens, int max_query_len, float scale,
                                pa_dtype dtype, int window, void *workspace, size_t workspace_bytes,
                                int32_t *device_status, void *stream) {
    if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || block_size != kBlockSize ||
        max_blocks_per_seq < 0 || num_blocks <= 0 || num_q_heads % num_kv_heads != 0 ||
        num_query_tokens < 0 || max_query_len < 0 || window < 0 || !(scale == scale))
        return PA_ERR_INVALID_ARG;
    if (dtype != PA_DTYPE_BF16) return PA_ERR_UNSUPPORTED;
    if (!prefix_tc_supported(head_dim, num_q_heads, num_kv_heads)) return PA_ERR_UNSUPPORTED;
    const int group = num_q_heads / num_kv_heads;
    if (num_seqs == 0 || num_query_tokens == 0 || max_query_len == 0) return PA_OK;
    if (!out || !query || !key_cache || !value_cache || !block_tables || !context_lens ||
        !query_start)
        return PA_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(query) || !aligned16(key_cache) || !aligned16(value_cache))
        return PA_ERR_INVALID_ARG;
    if (workspace == nullptr || workspace_bytes < kPrefillWorkspaceBytes || !aligned16(workspace))
        return PA_ERR_WORKSPACE;
    const int64_t rows = (int64_t)num_blocks * num_kv_heads * kBlockSize;
    if (rows >= ((int64_t)1 << 31)) return PA_ERR_UNSUPPORTED;
    const int64_t tiles = ((int64_t)max_query_len * group + kQT * kRows - 1) / (kQT * kRows);
    const int64_t items = tiles * num_kv_heads * num_seqs;
    if (items >= ((int64_t)1 << 31) - kThreads) return PA_ERR_UNSUPPORTED;
    CUtensorMap qmap, kmap, vmap;
    pa_status st = encode_maps(query, num_query_tokens, num_q_heads, num_kv_heads, key_cache,
                               value_cache, rows, &qmap, &kmap, &vmap);
    if (st != PA_OK) return st;
    PrefillArgs a = {};
    a.out = out;
    a.block_tables = block_tables;
    a.context_lens = context_lens;
    a.query_start = query_start;
    a.status = device_status;
    a.num_seqs = num_seqs;
    a.num_q_heads = num_q_heads;
    a.num_kv_heads = num_kv_heads;
    a.group = group;
    a.max_blocks = max_blocks_per_seq;
    a.num_blocks = num_blocks;
    a.max_query_len = max_query_len;
    a.window = window;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.n_mt = (int)tiles;
    a.num_items = (int)items;
    a.work_counter = static_cast<unsigned int *>(workspace);
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    // the ticket counter starts at zero on every call
    cudaError_t e = cudaMemsetAsync(workspace, 0, sizeof(unsigned int), cs);
    if (e != cudaSuccess) return cuda_failure(e, "cudaMemsetAsync(prefill ticket)");
    // persistent: one CTA per SM (each holds a whole SM), at most one per item
    const int64_t grid = std::min<int64_t>(items, prefill_sm_count());
    return launch_tc<false>(qmap, kmap, vmap, a, dim3((unsigned)grid), cs);
}

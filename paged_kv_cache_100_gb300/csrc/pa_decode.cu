// Paged decode attention for GB300 (sm_103a).
//
// What is computed ("KV cache: la memoria de trabajo que sostiene la inferencia
// LLM", section "El mecanismo en sí (en cristiano)"): the new token's query is
// multiplied against the keys of every context token, normalised with a
// softmax and used to weight the values.  Where the keys and values live
// ("PagedAttention por dentro", sections "La tabla de páginas (block table)"
// and "El kernel CUDA"): in 16-token physical blocks found through the
// sequence's block table, processed block by block.
//
// Work decomposition.  One CTA handles one (sequence, KV head, partition),
// where a partition is a run of `partition_size` logical tokens (split-K).
// Each warp of the CTA owns every NW-th block of the partition and runs its
// own TMA pipeline: lane 0 issues tiled tensor loads of the block's K and V
// tiles (16 rows x head_dim, 128-byte swizzled) into a ring of STAGES shared
// memory slots, completion is tracked by one mbarrier per slot, and the warp
// consumes the slots in order with an online (running max / running sum)
// softmax in fp32.  At the end the warps' states are merged in shared memory;
// a sequence that fits in one partition is written directly, otherwise the
// partition's (max, sum, unnormalised output) go to the workspace and a second
// kernel merges the partitions.
//
// Consumers:
//   * MHA (one query head per KV head): CUDA-core fp32 FMAs.  Each lane owns
//     8 head-dim elements of half (D=128) or a quarter (D=64) of the block's
//     rows; dot products are finished with a butterfly reduction that leaves
//     one row's score per lane pair.
//   * GQA (2..16 query heads share a KV head): the group makes Q.K^T and P.V
//     dense tiles, so they run on the tensor cores (mma.sync m16n8k16, bf16
//     in, fp32 accumulate).  Groups of up to 8 use the transposed form (the
//     block's 16 tokens are the M rows, the heads the 8 N columns); groups of
//     9..16 put the heads on the M rows.  One K/V pass serves the group
//     ("Trucos para que el cuaderno sea más fino": query heads share K/V).
//   * fp32 caches: a plain CUDA-core kernel, one query head per CTA.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <math.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

namespace {

constexpr uint32_t kFull = 0xffffffffu;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLazyRescaleLog2 = 8.f;   // FP8 consumers: rescale when the maximum grows by > 2^8

struct DecodeArgs {
    void *out;
    const void *query;
    const int32_t *block_tables;
    const int32_t *context_lens;
    float *part_o;      // [rows][head_dim], rows = (b * Hq + h) * max_parts + part
    float2 *part_ml;    // [rows] = (running max in log2 units, running sum)
    int32_t *status;
    const float *k_scales;  // FP8 pools: per-KV-head scales (stored value = code * scale)
    const float *v_scales;
    int num_seqs;
    int num_q_heads;
    int num_kv_heads;
    int max_blocks;     // block-table row length
    int num_blocks;     // pool size
    int part_blocks;    // partition size in blocks
    int max_parts;      // partition rows per (sequence, query head) in the workspace
    float scale_log2;   // softmax scale * log2(e)
    // Shared-prefix (cascade) mode; all zero for plain decode.
    int token_offset;   // tokens of every context handled elsewhere (a multiple of 16)
    int part_base;      // workspace partition rows used before this kernel's partitions
    int always_partial; // write (max, sum, output) partials even for one partition
    int prefix_blocks;  // shared prefix length in blocks (prefix kernel)
    int prefix_chunk_blocks;
    int prefix_chunks;
    int window;         // > 0: attend only to the last `window` positions
    // 1: only the grid's last CTA waits for the kernel before it in the stream
    // (the shared-prefix kernel), so that the others stream the suffix beside
    // it.  Safe because every kernel before that one had completed when it let
    // this one launch: all of its CTAs had waited for them first, or (FP8
    // pools) all CTAs of the prefix-widening kernel before it had done so
    // before it could start.  The last CTA's wait keeps this grid from
    // completing before the shared-prefix kernel (and what it waits for).  The last CTA is
    // dispatched last, when the prefix kernel is nearly done, so its wait is
    // short (CTA 0 would hold its SM idle for the whole prefix kernel).
    int defer_wait;
};

// The (sequence, head, partition) a CTA works on, with its token range.
struct Work {
    int b, head, part;
    int L;          // context length (clamped)
    int start;      // first position attended (sliding window), else 0
    int nparts;     // partitions of this sequence (1 when L == 0)
    int blk0;       // first logical block of the partition
    int nblk;       // blocks in the partition
};

// CTAs are numbered partition-major: every sequence's first partition comes
// first and the shorter trailing partitions (and the empty ones of short
// sequences) last, so the grid's tail is made of the smallest pieces.
// The (sequence, head, partition) of this CTA, from its index alone.
__device__ __forceinline__ void cta_coords(const DecodeArgs &a, int heads_axis, Work &w) {
    int idx = blockIdx.x;
    const int per_part = a.num_seqs * heads_axis;
    w.part = idx / per_part;
    idx -= w.part * per_part;
    w.b = idx / heads_axis;
    w.head = idx - w.b * heads_axis;
}

// The token range of the CTA's partition given its sequence's context length
// L as read from context_lens (clamped and flagged when out of range); false
// when the partition lies past the context.
__device__ __forceinline__ bool cta_range(const DecodeArgs &a, int L, Work &w) {
    const int lmax = a.max_blocks * kBlockSize;
    if (L < 0 || L > lmax) {
        if (threadIdx.x == 0 && w.part == 0 && w.head == 0) report(a.status, PA_DEV_BAD_CONTEXT_LEN);
        L = L < 0 ? 0 : lmax;
    }
    L = max(L - a.token_offset, 0);   // the part of the context this kernel covers
    w.L = L;
    // sliding window: positions [L - window, L); whole blocks before it are skipped
    w.start = (a.window > 0 && L > a.window) ? L - a.window : 0;
    const int first_blk = w.start / kBlockSize;
    const int seq_blocks = (L + kBlockSize - 1) / kBlockSize;
    const int range = seq_blocks - first_blk;
    w.nparts = range <= 0 ? 1 : (range + a.part_blocks - 1) / a.part_blocks;
    if (w.part >= w.nparts) return false;
    w.blk0 = first_blk + w.part * a.part_blocks;
    const int end = min(w.blk0 + a.part_blocks, seq_blocks);
    w.nblk = max(end - w.blk0, 0);
    return true;
}

__device__ __forceinline__ bool cta_work(const DecodeArgs &a, int heads_axis, Work &w) {
    cta_coords(a, heads_axis, w);
    return cta_range(a, a.context_lens[w.b], w);
}

template <typename T>
__device__ __forceinline__ void store_out(T *p, float v);
template <>
__device__ __forceinline__ void store_out<float>(float *p, float v) { *p = v; }
template <>
__device__ __forceinline__ void store_out<__nv_bfloat16>(__nv_bfloat16 *p, float v) {
    *p = __float2bfloat16_rn(v);
}

// Merges the NW per-warp states of a CTA (rows x D accumulators in shared
// memory, one (max, sum) per row and warp) and writes either the final output
// (single partition) or the partition's partial state.
template <typename OutT, int NW>
__device__ __forceinline__ void merge_and_store(const DecodeArgs &a, const Work &w, int first_head,
                                                int rows, int D, const float *acc_base,
                                                int acc_warp_stride, const float *s_m,
                                                const float *s_l, int row_stride) {
    for (int idx = threadIdx.x; idx < rows * D; idx += NW * 32) {
        const int r = idx / D;
        const int d = idx - r * D;
        float M = -INFINITY;
#pragma unroll
        for (int k = 0; k < NW; ++k) M = fmaxf(M, s_m[k * row_stride + r]);
        float O = 0.f, Lsum = 0.f;
#pragma unroll
        for (int k = 0; k < NW; ++k) {
            const float mk = s_m[k * row_stride + r];
            const float wk = (mk == -INFINITY) ? 0.f : exp2f(mk - M);
            Lsum += wk * s_l[k * row_stride + r];
            O += wk * acc_base[k * acc_warp_stride + r * D + d];
        }
        const int h = first_head + r;
        if (w.nparts == 1 && !a.always_partial) {
            OutT *out = static_cast<OutT *>(a.out) + ((size_t)w.b * a.num_q_heads + h) * D + d;
            store_out<OutT>(out, Lsum > 0.f ? O / Lsum : 0.f);
        } else {
            const size_t row = ((size_t)w.b * a.num_q_heads + h) * a.max_parts + a.part_base + w.part;
            a.part_o[row * D + d] = O;
            if (d == 0) a.part_ml[row] = make_float2(M, Lsum);
        }
    }
}

// ---------------------------------------------------------------------------
// Consumers for bf16 tiles staged by TMA with 128-byte swizzle.  A tile of one
// block is 16 rows x D bf16, stored as D/64 sub-tiles of [16][64] (2 KiB each);
// 16-byte chunk c of row r of a sub-tile sits at chunk (c ^ (r & 7)).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t swz(uint32_t tile, int row, int chunk) {
    return tile + (uint32_t)((chunk >> 3) * 2048 + row * 128 + (((chunk & 7) ^ (row & 7)) << 4));
}

// Zeroes the rows outside [nlo, nvalid) of a 16-row bf16 tile of D/64 swizzled
// sub-tiles (whole rows, so the swizzle does not matter).
template <int D>
__device__ __forceinline__ void zero_rows_outside(uint32_t tile, int nlo, int nvalid, int lane) {
    constexpr int kChunks = D / 8;          // 16-byte chunks per row
    const int zrows = 16 - (nvalid - nlo);
    for (int i = lane; i < zrows * kChunks; i += 32) {
        int r = i / kChunks;
        r = r < nlo ? r : r - nlo + nvalid;
        const int ch = i % kChunks;
        asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(swz(tile, r, ch)), "r"(0u)
                     : "memory");
    }
    __syncwarp();
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

__device__ __forceinline__ float dot8(const float (&q)[8], uint4 k) {
    float s = q[0] * bf16lo(k.x);
    s = fmaf(q[1], bf16hi(k.x), s);
    s = fmaf(q[2], bf16lo(k.y), s);
    s = fmaf(q[3], bf16hi(k.y), s);
    s = fmaf(q[4], bf16lo(k.z), s);
    s = fmaf(q[5], bf16hi(k.z), s);
    s = fmaf(q[6], bf16lo(k.w), s);
    s = fmaf(q[7], bf16hi(k.w), s);
    return s;
}

__device__ __forceinline__ void axpy8(float (&acc)[8], float p, uint4 v) {
    acc[0] = fmaf(p, bf16lo(v.x), acc[0]);
    acc[1] = fmaf(p, bf16hi(v.x), acc[1]);
    acc[2] = fmaf(p, bf16lo(v.y), acc[2]);
    acc[3] = fmaf(p, bf16hi(v.y), acc[3]);
    acc[4] = fmaf(p, bf16lo(v.z), acc[4]);
    acc[5] = fmaf(p, bf16hi(v.z), acc[5]);
    acc[6] = fmaf(p, bf16lo(v.w), acc[6]);
    acc[7] = fmaf(p, bf16hi(v.w), acc[7]);
}

// One query head per KV head.  Lane layout: chunk c = lane % CH owns head-dim
// elements [8c, 8c+8); row group rg = lane / CH owns rows [rg*RPL, rg*RPL+RPL).
template <int D>
struct MhaConsumer {
    static constexpr int CH = D / 8;
    static constexpr int RG = 32 / CH;
    static constexpr int RPL = 16 / RG;
    static constexpr int ROWS = 1;     // query heads per warp state
    static constexpr int kElemBytes = 2;
    static constexpr bool kEarlyLoads = true;   // table and query loaded beside the length
    static_assert(RPL * 2 == CH, "lane layout");

    float q[8];
    float acc[8];
    float m, l;
    int lane, c, rg;

    __device__ __forceinline__ void init(const DecodeArgs &a, const Work &w, int lane_) {
        lane = lane_;
        c = lane & (CH - 1);
        rg = lane / CH;
        const __nv_bfloat16 *qrow =
            static_cast<const __nv_bfloat16 *>(a.query) + ((size_t)w.b * a.num_q_heads + w.head) * D;
        const uint4 raw = *reinterpret_cast<const uint4 *>(qrow + 8 * c);
        const uint32_t words[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            q[2 * e] = bf16lo(words[e]) * a.scale_log2;
            q[2 * e + 1] = bf16hi(words[e]) * a.scale_log2;
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = 0.f;
        m = -INFINITY;
        l = 0.f;
    }

    __device__ __forceinline__ void block(uint32_t ktile, uint32_t vtile, int nlo, int nvalid) {
        float v[RPL];
#pragma unroll
        for (int i = 0; i < RPL; ++i) v[i] = dot8(q, lds128(swz(ktile, rg * RPL + i, c)));
        // Butterfly: after the step with mask M a lane keeps the half of its
        // values selected by (lane & M); the last step (mask 1) completes the sum.
#pragma unroll
        for (int M = CH / 2, n = RPL; M >= 2; M >>= 1, n >>= 1) {
            const bool upper = (lane & M) != 0;
#pragma unroll
            for (int k = 0; k < n / 2; ++k) {
                const float send = upper ? v[k] : v[k + n / 2];
                const float keep = upper ? v[k + n / 2] : v[k];
                v[k] = keep + __shfl_xor_sync(kFull, send, M);
            }
        }
        float s = v[0] + __shfl_xor_sync(kFull, v[0], 1);
        const int row = rg * RPL + ((lane & (CH - 1)) >> 1);
        s = (row >= nlo && row < nvalid) ? s : -INFINITY;
        float bmax = s;
#pragma unroll
        for (int M = 2; M < 32; M <<= 1) bmax = fmaxf(bmax, __shfl_xor_sync(kFull, bmax, M));
        const float m_new = fmaxf(m, bmax);
        const float alpha = exp2f(m - m_new);
        const float p = ex2_fast(s - m_new);
        l = l * alpha + ((lane & 1) ? 0.f : p);
        m = m_new;
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] *= alpha;
#pragma unroll
        for (int i = 0; i < RPL; ++i) {
            const int r = rg * RPL + i;
            const float pr = __shfl_sync(kFull, p, rg * CH + 2 * i);
            const uint4 vv = lds128(swz(vtile, r, c));
            if (r >= nlo && r < nvalid) axpy8(acc, pr, vv);
        }
    }

    // Writes this warp's state: acc[ROWS][D] floats at `acc_out`, (m, l) per row.
    __device__ __forceinline__ void finish(float *acc_out, float *m_out, float *l_out) {
#pragma unroll
        for (int M = CH; M < 32; M <<= 1)
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] += __shfl_xor_sync(kFull, acc[e], M);
#pragma unroll
        for (int M = 1; M < 32; M <<= 1) l += __shfl_xor_sync(kFull, l, M);
        if (lane < CH) {
            float4 *dst = reinterpret_cast<float4 *>(acc_out + 8 * c);
            dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
            dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
        }
        if (lane == 0) {
            m_out[0] = m;
            l_out[0] = l;
        }
    }
};

// 2..16 query heads per KV head on the tensor cores.  Fragment owner:
// g = lane / 4 (query-head row g and g + 8), t = lane % 4.
template <int D, int G>
struct GqaConsumer {
    static constexpr int KS = D / 16;   // k-steps of Q.K^T
    static constexpr int NT = D / 8;    // n-tiles of P.V
    static constexpr bool HI = G > 8;   // rows 8..15 hold real heads
    static constexpr int ROWS = G;
    static constexpr int kElemBytes = 2;
    static constexpr bool kEarlyLoads = true;   // table and query loaded beside the length

    uint32_t qa[KS][4];
    float o[NT][4];
    float m0, m1, l0, l1;
    float scale_log2;
    int lane, g, t;

    __device__ __forceinline__ void init(const DecodeArgs &a, const Work &w, int lane_) {
        lane = lane_;
        g = lane >> 2;
        t = lane & 3;
        scale_log2 = a.scale_log2;
        const __nv_bfloat16 *qg = static_cast<const __nv_bfloat16 *>(a.query) +
                                  ((size_t)w.b * a.num_q_heads + (size_t)w.head * G) * D;
        const uint32_t *q0 = reinterpret_cast<const uint32_t *>(qg + (size_t)g * D);
        const uint32_t *q1 = reinterpret_cast<const uint32_t *>(qg + (size_t)(g + 8) * D);
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            const bool r0 = g < G, r1 = HI && (g + 8 < G);
            qa[ks][0] = r0 ? q0[(16 * ks + 2 * t) / 2] : 0u;
            qa[ks][2] = r0 ? q0[(16 * ks + 8 + 2 * t) / 2] : 0u;
            qa[ks][1] = r1 ? q1[(16 * ks + 2 * t) / 2] : 0u;
            qa[ks][3] = r1 ? q1[(16 * ks + 8 + 2 * t) / 2] : 0u;
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
        m0 = m1 = -INFINITY;
        l0 = l1 = 0.f;
    }

    __device__ __forceinline__ void block(uint32_t ktile, uint32_t vtile, int nlo, int nvalid) {
        float s[2][4];
#pragma unroll
        for (int j = 0; j < 2; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
        const int mi = lane >> 3, rr = lane & 7;
#pragma unroll
        for (int kk = 0; kk < D / 32; ++kk) {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                uint32_t b[4];
                ldsm_x4(b, swz(ktile, 8 * j + rr, 4 * kk + mi));
                mma_bf16_16816(s[j], qa[2 * kk], b[0], b[1]);
                mma_bf16_16816(s[j], qa[2 * kk + 1], b[2], b[3]);
            }
        }
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int tok = 8 * j + 2 * t + (e & 1);
                s[j][e] = (tok >= nlo && tok < nvalid) ? s[j][e] * scale_log2 : -INFINITY;
            }
        float mx0 = fmaxf(fmaxf(s[0][0], s[0][1]), fmaxf(s[1][0], s[1][1]));
        mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, 2));
        const float mn0 = fmaxf(m0, mx0);
        const float a0 = exp2f(m0 - mn0);
        m0 = mn0;
        float mn1 = 0.f, a1 = 1.f;
        if (HI) {
            float mx1 = fmaxf(fmaxf(s[0][2], s[0][3]), fmaxf(s[1][2], s[1][3]));
            mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, 1));
            mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, 2));
            mn1 = fmaxf(m1, mx1);
            a1 = exp2f(m1 - mn1);
            m1 = mn1;
        }
        float p[2][4];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            p[j][0] = ex2_fast(s[j][0] - mn0);
            p[j][1] = ex2_fast(s[j][1] - mn0);
            p[j][2] = HI ? ex2_fast(s[j][2] - mn1) : 0.f;
            p[j][3] = HI ? ex2_fast(s[j][3] - mn1) : 0.f;
        }
        l0 = l0 * a0 + (p[0][0] + p[0][1]) + (p[1][0] + p[1][1]);
        if (HI) l1 = l1 * a1 + (p[0][2] + p[0][3]) + (p[1][2] + p[1][3]);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            o[nt][0] *= a0;
            o[nt][1] *= a0;
            if (HI) {
                o[nt][2] *= a1;
                o[nt][3] *= a1;
            }
        }
        // P enters the tensor cores as bf16; a single rounding would perturb each
        // weight by up to 2^-9, so P is split into a bf16 head and a bf16 residual
        // (P = hi + lo up to 2^-18 relative) and both are multiplied by V.
        uint32_t pa[4], pl[4];
        split_bf16x2(p[0][0], p[0][1], pa[0], pl[0]);
        split_bf16x2(p[1][0], p[1][1], pa[2], pl[2]);
        if (HI) {
            split_bf16x2(p[0][2], p[0][3], pa[1], pl[1]);
            split_bf16x2(p[1][2], p[1][3], pa[3], pl[3]);
        } else {
            pa[1] = pa[3] = pl[1] = pl[3] = 0u;
        }
        // Rows outside the context may hold anything (even NaN): zero them so
        // that 0 * row stays 0 in the tensor-core sum.
        if (nlo > 0 || nvalid < 16) zero_rows_outside<D>(vtile, nlo, nvalid, lane);
#pragma unroll
        for (int dd = 0; dd < D / 16; ++dd) {
            uint32_t b[4];
            ldsm_x4_trans(b, swz(vtile, (mi & 1) * 8 + rr, 2 * dd + (mi >> 1)));
            mma_bf16_16816(o[2 * dd], pa, b[0], b[1]);
            mma_bf16_16816(o[2 * dd + 1], pa, b[2], b[3]);
            mma_bf16_16816(o[2 * dd], pl, b[0], b[1]);
            mma_bf16_16816(o[2 * dd + 1], pl, b[2], b[3]);
        }
    }

    __device__ __forceinline__ void finish(float *acc_out, float *m_out, float *l_out) {
        l0 += __shfl_xor_sync(kFull, l0, 1);
        l0 += __shfl_xor_sync(kFull, l0, 2);
        if (HI) {
            l1 += __shfl_xor_sync(kFull, l1, 1);
            l1 += __shfl_xor_sync(kFull, l1, 2);
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int d = 8 * nt + 2 * t;
            if (g < G) *reinterpret_cast<float2 *>(acc_out + g * D + d) = make_float2(o[nt][0], o[nt][1]);
            if (HI && g + 8 < G)
                *reinterpret_cast<float2 *>(acc_out + (g + 8) * D + d) = make_float2(o[nt][2], o[nt][3]);
        }
        if (t == 0) {
            if (g < G) {
                m_out[g] = m0;
                l_out[g] = l0;
            }
            if (HI && g + 8 < G) {
                m_out[g + 8] = m1;
                l_out[g + 8] = l1;
            }
        }
    }
};

// 2..8 query heads per KV head on the tensor cores, transposed: the block's 16
// tokens are the M rows and the query heads the N = 8 columns, so
//   S^T[16 tok x 8 heads] = K[16 x D] . Q^T[D x 8]        (D/16 mma)
//   O^T[D x 8 heads]     += V^T[D x 16 tok] . P^T[16 x 8]  (D/16 m-tiles, x2 for hi/lo)
// and no M row is padding.  The S^T accumulators become the B operand of the
// second product after a warp-wide 8x8 transpose (movmatrix).  Fragment
// owner: g = lane / 4, t = lane % 4; this lane holds tokens g and g + 8 for
// query heads 2t and 2t + 1.
template <int D, int G>
struct GqaTConsumer {
    static_assert(G >= 2 && G <= 8, "one n-tile of query heads");
    static constexpr int KS = D / 16;   // k-steps of S^T and m-tiles of O^T
    static constexpr int ROWS = G;
    static constexpr int kElemBytes = 2;
    static constexpr bool kEarlyLoads = true;   // table and query loaded beside the length

    uint32_t qb[KS][2];
    float o[KS][4];
    float m0, m1, l0, l1;               // heads 2t and 2t + 1
    float scale_log2;
    int lane, g, t;

    __device__ __forceinline__ void init(const DecodeArgs &a, const Work &w, int lane_) {
        lane = lane_;
        g = lane >> 2;
        t = lane & 3;
        scale_log2 = a.scale_log2;
        const __nv_bfloat16 *qg = static_cast<const __nv_bfloat16 *>(a.query) +
                                  ((size_t)w.b * a.num_q_heads + (size_t)w.head * G) * D;
        const uint32_t *qrow = reinterpret_cast<const uint32_t *>(qg + (size_t)g * D);
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            qb[ks][0] = g < G ? qrow[(16 * ks + 2 * t) / 2] : 0u;
            qb[ks][1] = g < G ? qrow[(16 * ks + 8 + 2 * t) / 2] : 0u;
        }
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
        m0 = m1 = -INFINITY;
        l0 = l1 = 0.f;
    }

    __device__ __forceinline__ void block(uint32_t ktile, uint32_t vtile, int nlo, int nvalid) {
        const int mi = lane >> 3, rr = lane & 7;
        float s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            uint32_t a[4];
            ldsm_x4(a, swz(ktile, (mi & 1) * 8 + rr, 2 * ks + (mi >> 1)));
            mma_bf16_16816(s, a, qb[ks][0], qb[ks][1]);
        }
        const bool v0 = g >= nlo && g < nvalid, v1 = g + 8 >= nlo && g + 8 < nvalid;
        s[0] = v0 ? s[0] * scale_log2 : -INFINITY;
        s[1] = v0 ? s[1] * scale_log2 : -INFINITY;
        s[2] = v1 ? s[2] * scale_log2 : -INFINITY;
        s[3] = v1 ? s[3] * scale_log2 : -INFINITY;
        float mx0 = fmaxf(s[0], s[2]), mx1 = fmaxf(s[1], s[3]);
#pragma unroll
        for (int M = 4; M < 32; M <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, M));
            mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, M));
        }
        const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
        const float a0 = exp2f(m0 - mn0), a1 = exp2f(m1 - mn1);
        m0 = mn0;
        m1 = mn1;
        const float p0 = ex2_fast(s[0] - mn0), p1 = ex2_fast(s[1] - mn1);
        const float p2 = ex2_fast(s[2] - mn0), p3 = ex2_fast(s[3] - mn1);
        l0 = l0 * a0 + (p0 + p2);
        l1 = l1 * a1 + (p1 + p3);
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
            o[mt][0] *= a0;
            o[mt][1] *= a1;
            o[mt][2] *= a0;
            o[mt][3] *= a1;
        }
        // P enters the tensor cores as bf16 head + bf16 residual (see GqaConsumer).
        uint32_t top_hi, top_lo, bot_hi, bot_lo;
        split_bf16x2(p0, p1, top_hi, top_lo);   // token g
        split_bf16x2(p2, p3, bot_hi, bot_lo);   // token g + 8
        const uint32_t bh0 = movmatrix_trans(top_hi), bh1 = movmatrix_trans(bot_hi);
        const uint32_t bl0 = movmatrix_trans(top_lo), bl1 = movmatrix_trans(bot_lo);
        if (nlo > 0 || nvalid < 16) zero_rows_outside<D>(vtile, nlo, nvalid, lane);
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
            uint32_t a[4];
            ldsm_x4_trans(a, swz(vtile, (mi >> 1) * 8 + rr, 2 * mt + (mi & 1)));
            mma_bf16_16816(o[mt], a, bh0, bh1);
            mma_bf16_16816(o[mt], a, bl0, bl1);
        }
    }

    __device__ __forceinline__ void finish(float *acc_out, float *m_out, float *l_out) {
#pragma unroll
        for (int M = 4; M < 32; M <<= 1) {
            l0 += __shfl_xor_sync(kFull, l0, M);
            l1 += __shfl_xor_sync(kFull, l1, M);
        }
        const int h0 = 2 * t, h1 = 2 * t + 1;
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
            const int d = 16 * mt + g;
            if (h0 < G) {
                acc_out[h0 * D + d] = o[mt][0];
                acc_out[h0 * D + d + 8] = o[mt][2];
            }
            if (h1 < G) {
                acc_out[h1 * D + d] = o[mt][1];
                acc_out[h1 * D + d + 8] = o[mt][3];
            }
        }
        if (g == 0) {
            if (h0 < G) {
                m_out[h0] = m0;
                l_out[h0] = l0;
            }
            if (h1 < G) {
                m_out[h1] = m1;
                l_out[h1] = l1;
            }
        }
    }
};

// ---------------------------------------------------------------------------
// FP8 (E4M3) pools.  A tile is 16 rows x D codes (D bytes per row, one 128-byte
// swizzle row at D = 128); the stored value of a code is code_value * scale of
// its KV head, and the scales are applied once per score (K) and once per
// output (V).  E4M3 values are exact in f16, so the kernels widen codes to f16
// and keep fp32 accumulation.  The query is rounded to f16 once (exact for
// |q| in [2^-14, 65504]).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t fp8_addr(uint32_t tile, int row, int byte) {
    return tile + (uint32_t)(row * 128 + ((((byte >> 4) ^ (row & 7))) << 4) + (byte & 15));
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint2 lds64(uint32_t addr) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
    return v;
}

// Zeroes the rows outside [nlo, nvalid) of a 16 x 128-byte tile (values
// outside the context may be anything, NaN codes included, and must not reach
// a tensor-core sum).
__device__ __forceinline__ void zero_rows_outside_128(uint32_t tile, int nlo, int nvalid, int lane) {
    const int zrows = 16 - (nvalid - nlo);
    for (int i = lane; i < zrows * 8; i += 32) {
        int r = i / 8;
        r = r < nlo ? r : r - nlo + nvalid;
        const uint32_t addr = tile + (uint32_t)(r * 128 + (i % 8) * 16);
        asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(0u) : "memory");
    }
    __syncwarp();
}

// One query head per KV head, FP8 pools, D = 128.  Lane layout: chunk c =
// lane % 8 owns head-dim elements [16c, 16c+16) (one 16-byte chunk of codes);
// row group rg = lane / 8 owns rows [4rg, 4rg+4).
template <int D>
struct MhaFp8Consumer {
    static_assert(D == 128, "one 128-byte swizzle row per tile row");
    static constexpr int CH = D / 16;
    static constexpr int RG = 32 / CH;
    static constexpr int RPL = 16 / RG;
    static constexpr int ROWS = 1;
    static constexpr int kElemBytes = 1;
    // table entries and query loaded after the length (as one chain): loaded
    // beside it they gain nothing on the 7B-shaped FP8 batch (92.1 us either
    // way; 2 % slower with an earlier form of this consumer)
    static constexpr bool kEarlyLoads = false;

    uint32_t q[8];       // f16x2: elements 16c + 2i, 16c + 2i + 1
    float acc[16];
    float m, l;
    float ck;            // softmax scale * log2(e) * k scale
    float vs;
    int lane, c, rg;
    // byte offsets of this lane's 16-byte chunk c in rows 4rg .. 4rg + 3 of a
    // swizzled tile (the same for K and V tiles)
    uint32_t off[RPL];

    __device__ __forceinline__ void init(const DecodeArgs &a, const Work &w, int lane_) {
        lane = lane_;
        c = lane & (CH - 1);
        rg = lane / CH;
#pragma unroll
        for (int i = 0; i < RPL; ++i) off[i] = swz(0u, rg * RPL + i, c);
        const __nv_bfloat16 *qrow =
            static_cast<const __nv_bfloat16 *>(a.query) + ((size_t)w.b * a.num_q_heads + w.head) * D;
        const uint4 r0 = *reinterpret_cast<const uint4 *>(qrow + 16 * c);
        const uint4 r1 = *reinterpret_cast<const uint4 *>(qrow + 16 * c + 8);
        const uint32_t words[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
        bool beyond = false;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            q[i] = pack_f16x2(bf16lo(words[i]), bf16hi(words[i]));
            beyond |= bf16x2_beyond_f16(words[i]);
        }
        if (beyond) report(a.status, PA_DEV_RANGE);   // the f16 query is not q
#pragma unroll
        for (int e = 0; e < 16; ++e) acc[e] = 0.f;
        m = -INFINITY;
        l = 0.f;
        ck = a.scale_log2 * a.k_scales[w.head];
        vs = a.v_scales[w.head];
    }

    __device__ __forceinline__ void block(uint32_t ktile, uint32_t vtile, int nlo, int nvalid) {
        float v[RPL];
#pragma unroll
        for (int i = 0; i < RPL; ++i) {
            const uint4 kw = lds128(ktile + off[i]);
            const uint32_t w4[4] = {kw.x, kw.y, kw.z, kw.w};
            float dot = 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uint32_t k01, k23;
                e4m3x4_to_f16x2x2(w4[j], k01, k23);
                dot = dot2_f16_f32(q[2 * j], k01, dot);
                dot = dot2_f16_f32(q[2 * j + 1], k23, dot);
            }
            v[i] = dot;
        }
#pragma unroll
        for (int M = CH / 2, n = RPL; M >= 2; M >>= 1, n >>= 1) {
            const bool upper = (lane & M) != 0;
#pragma unroll
            for (int k = 0; k < n / 2; ++k) {
                const float send = upper ? v[k] : v[k + n / 2];
                const float keep = upper ? v[k + n / 2] : v[k];
                v[k] = keep + __shfl_xor_sync(kFull, send, M);
            }
        }
        float s = (v[0] + __shfl_xor_sync(kFull, v[0], 1)) * ck;
        const int row = rg * RPL + ((lane & (CH - 1)) >> 1);
        s = (row >= nlo && row < nvalid) ? s : -INFINITY;
        float bmax = s;
#pragma unroll
        for (int M = 2; M < 32; M <<= 1) bmax = fmaxf(bmax, __shfl_xor_sync(kFull, bmax, M));
        // Lazy rescale: the reference maximum m moves (and acc, l are rescaled)
        // only when the block's maximum exceeds it by more than 2^8, so the
        // weights stay in [0, 256].  The decision is warp-uniform.
        if (bmax > m + kLazyRescaleLog2) {
            const float alpha = exp2f(m - bmax);   // 0 while m is -inf
            l *= alpha;
#pragma unroll
            for (int e = 0; e < 16; ++e) acc[e] *= alpha;
            m = bmax;
        }
        const float p = ex2_fast(s - m);
        l += (lane & 1) ? 0.f : p;
        // rows outside [nlo, nvalid) may hold anything (NaN included), so their
        // products are skipped; a full block (the common case) needs no test
        const bool full = nlo == 0 && nvalid == 16;
#pragma unroll
        for (int i = 0; i < RPL; ++i) {
            const int r = rg * RPL + i;
            // the weight enters the products as f16 (relative error <= 2^-11)
            const uint32_t p16 = pack_f16x2(__shfl_sync(kFull, p, rg * CH + 2 * i), 0.f);
            const uint4 vw = lds128(vtile + off[i]);
            if (full || (r >= nlo && r < nvalid)) {
                const uint32_t w4[4] = {vw.x, vw.y, vw.z, vw.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    uint32_t v01, v23;
                    e4m3x4_to_f16x2x2(w4[j], v01, v23);
                    fma2_f16_f32(p16, v01, acc[4 * j + 0], acc[4 * j + 1]);
                    fma2_f16_f32(p16, v23, acc[4 * j + 2], acc[4 * j + 3]);
                }
            }
        }
    }

    __device__ __forceinline__ void finish(float *acc_out, float *m_out, float *l_out) {
#pragma unroll
        for (int M = CH; M < 32; M <<= 1)
#pragma unroll
            for (int e = 0; e < 16; ++e) acc[e] += __shfl_xor_sync(kFull, acc[e], M);
#pragma unroll
        for (int M = 1; M < 32; M <<= 1) l += __shfl_xor_sync(kFull, l, M);
        if (lane < CH) {
            float4 *dst = reinterpret_cast<float4 *>(acc_out + 16 * c);
#pragma unroll
            for (int k = 0; k < 4; ++k)
                dst[k] = make_float4(acc[4 * k] * vs, acc[4 * k + 1] * vs, acc[4 * k + 2] * vs,
                                     acc[4 * k + 3] * vs);
        }
        if (lane == 0) {
            m_out[0] = m;
            l_out[0] = l;
        }
    }
};

// 2..8 query heads per KV head, FP8 pools, D = 128, on f16 tensor cores in the
// transposed form of GqaTConsumer (tokens on M, heads on N).
//  * S^T = K.Q^T: the contraction over the head dimension may visit it in any
//    order as long as K and Q agree, so lane (g, t) loads 8 consecutive codes
//    of rows g and g + 8 (bytes 32kk + 8t .. +8) and the Q fragments are laid
//    out to match: k-step 2kk + hh covers head-dim elements
//    32kk + 8t + 4hh + {0, 1} (k = 2t, 2t+1) and + {2, 3} (k = 2t+8, 2t+9).
//  * O^T += V^T.P^T: the A operand needs two tokens of one head-dim element
//    per register, so lane (g, t) loads 4 codes (bytes 32c + 4g ..) of token
//    rows 2t, 2t+1, 2t+8, 2t+9 and pairs them with byte permutes; output rows
//    are head-dim elements 32c + 4g + 2jp (row g) and + 1 (row g + 8) of m-tile
//    2c + jp.
template <int D, int G>
struct GqaTFp8Consumer {
    static_assert(D == 128, "one 128-byte swizzle row per tile row");
    static_assert(G >= 1 && G <= 8, "one n-tile of query heads");
    static constexpr int KS = D / 16;
    static constexpr int ROWS = G;
    static constexpr int kElemBytes = 1;
    static constexpr bool kEarlyLoads = true;   // table and query loaded beside the length

    uint32_t qb[KS][2];
    float o[KS][4];
    float m0, m1, l0, l1;
    float ck, vs;
    int lane, g, t;
    // This lane's swizzled byte offsets in a tile (fp8_addr with the lane's
    // rows and columns folded in): K rows g (+ 1024 for row g + 8) at column
    // 32kk + 8t; V rows 2t (+ 1024: 2t + 8) and 2t + 1 (+ 1024: 2t + 9) at
    // column 32c + 4g.
    uint32_t koff[D / 32], voff_a[D / 32], voff_b[D / 32];

    __device__ __forceinline__ void init(const DecodeArgs &a, const Work &w, int lane_) {
        lane = lane_;
        g = lane >> 2;
        t = lane & 3;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
            koff[c] = fp8_addr(0u, g, 32 * c + 8 * t);
            voff_a[c] = fp8_addr(0u, 2 * t, 32 * c + 4 * g);
            voff_b[c] = fp8_addr(0u, 2 * t + 1, 32 * c + 4 * g);
        }
        ck = a.scale_log2 * a.k_scales[w.head];
        vs = a.v_scales[w.head];
        const __nv_bfloat16 *qg = static_cast<const __nv_bfloat16 *>(a.query) +
                                  ((size_t)w.b * a.num_q_heads + (size_t)w.head * G) * D;
        const uint32_t *qrow = reinterpret_cast<const uint32_t *>(qg + (size_t)g * D);
        bool beyond = false;
#pragma unroll
        for (int kk = 0; kk < D / 32; ++kk)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int d = 32 * kk + 8 * t + 4 * hh;
                const uint32_t w0 = g < G ? qrow[d / 2] : 0u;
                const uint32_t w1 = g < G ? qrow[d / 2 + 1] : 0u;
                qb[2 * kk + hh][0] = pack_f16x2(bf16lo(w0), bf16hi(w0));
                qb[2 * kk + hh][1] = pack_f16x2(bf16lo(w1), bf16hi(w1));
                beyond |= bf16x2_beyond_f16(w0) | bf16x2_beyond_f16(w1);
            }
        if (beyond) report(a.status, PA_DEV_RANGE);   // the f16 query is not q
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
        m0 = m1 = -INFINITY;
        l0 = l1 = 0.f;
    }

    __device__ __forceinline__ void block(uint32_t ktile, uint32_t vtile, int nlo, int nvalid) {
        float s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kk = 0; kk < D / 32; ++kk) {
            const uint32_t ka = ktile + koff[kk];
            const uint2 r0 = lds64(ka);
            const uint2 r1 = lds64(ka + 1024);   // row g + 8: same swizzle phase
            uint32_t a[4];
            e4m3x4_to_f16x2x2(r0.x, a[0], a[2]);
            e4m3x4_to_f16x2x2(r1.x, a[1], a[3]);
            mma_f16_16816(s, a, qb[2 * kk][0], qb[2 * kk][1]);
            e4m3x4_to_f16x2x2(r0.y, a[0], a[2]);
            e4m3x4_to_f16x2x2(r1.y, a[1], a[3]);
            mma_f16_16816(s, a, qb[2 * kk + 1][0], qb[2 * kk + 1][1]);
        }
        const bool v0 = g >= nlo && g < nvalid, v1 = g + 8 >= nlo && g + 8 < nvalid;
        s[0] = v0 ? s[0] * ck : -INFINITY;
        s[1] = v0 ? s[1] * ck : -INFINITY;
        s[2] = v1 ? s[2] * ck : -INFINITY;
        s[3] = v1 ? s[3] * ck : -INFINITY;
        float mx0 = fmaxf(s[0], s[2]), mx1 = fmaxf(s[1], s[3]);
#pragma unroll
        for (int M = 4; M < 32; M <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, M));
            mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, M));
        }
        // Lazy rescale: a head's reference maximum moves (and its O and sum
        // are rescaled) only when the block's maximum exceeds it by more than
        // 2^8, so the weights stay in [0, 256] (f16 holds them); the warp skips
        // the rescale when no head of it needs one.
        const bool need0 = mx0 > m0 + kLazyRescaleLog2, need1 = mx1 > m1 + kLazyRescaleLog2;
        if (__any_sync(kFull, need0 || need1)) {
            const float a0 = need0 ? exp2f(m0 - mx0) : 1.f;   // 0 while m0 is -inf
            const float a1 = need1 ? exp2f(m1 - mx1) : 1.f;
            m0 = need0 ? mx0 : m0;
            m1 = need1 ? mx1 : m1;
            l0 *= a0;
            l1 *= a1;
#pragma unroll
            for (int mt = 0; mt < KS; ++mt) {
                o[mt][0] *= a0;
                o[mt][1] *= a1;
                o[mt][2] *= a0;
                o[mt][3] *= a1;
            }
        }
        const float p0 = ex2_fast(s[0] - m0), p1 = ex2_fast(s[1] - m1);
        const float p2 = ex2_fast(s[2] - m0), p3 = ex2_fast(s[3] - m1);
        l0 += p0 + p2;
        l1 += p1 + p3;
        // P in f16, rounded once: 11 significant bits move an output by at most
        // 2^-11 of the largest |v| it weighs (no residual product needed, unlike
        // bf16 weights)
        const uint32_t bh0 = movmatrix_trans(pack_f16x2(p0, p1));
        const uint32_t bh1 = movmatrix_trans(pack_f16x2(p2, p3));
        if (nlo > 0 || nvalid < 16) zero_rows_outside_128(vtile, nlo, nvalid, lane);
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
            const uint32_t va = vtile + voff_a[c], vb = vtile + voff_b[c];
            const uint32_t wa = lds32(va);
            const uint32_t wb = lds32(vb);
            const uint32_t wc = lds32(va + 1024);   // rows + 8: same swizzle phase
            const uint32_t wd = lds32(vb + 1024);
#pragma unroll
            for (int jp = 0; jp < 2; ++jp) {
                const uint32_t sel = jp == 0 ? 0x5140u : 0x7362u;
                const uint32_t x0 = __byte_perm(wa, wb, sel);   // tokens 2t, 2t+1
                const uint32_t x1 = __byte_perm(wc, wd, sel);   // tokens 2t+8, 2t+9
                uint32_t a[4];
                e4m3x4_to_f16x2x2(x0, a[0], a[1]);
                e4m3x4_to_f16x2x2(x1, a[2], a[3]);
                mma_f16_16816(o[2 * c + jp], a, bh0, bh1);
            }
        }
    }

    __device__ __forceinline__ void finish(float *acc_out, float *m_out, float *l_out) {
#pragma unroll
        for (int M = 4; M < 32; M <<= 1) {
            l0 += __shfl_xor_sync(kFull, l0, M);
            l1 += __shfl_xor_sync(kFull, l1, M);
        }
        const int h0 = 2 * t, h1 = 2 * t + 1;
#pragma unroll
        for (int c = 0; c < D / 32; ++c)
#pragma unroll
            for (int jp = 0; jp < 2; ++jp) {
                const int d = 32 * c + 4 * g + 2 * jp;
                const float *oo = o[2 * c + jp];
                if (h0 < G) {
                    acc_out[h0 * D + d] = oo[0] * vs;
                    acc_out[h0 * D + d + 1] = oo[2] * vs;
                }
                if (h1 < G) {
                    acc_out[h1 * D + d] = oo[1] * vs;
                    acc_out[h1 * D + d + 1] = oo[3] * vs;
                }
            }
        if (g == 0) {
            if (h0 < G) {
                m_out[h0] = m0;
                l_out[h0] = l0;
            }
            if (h1 < G) {
                m_out[h1] = m1;
                l_out[h1] = l1;
            }
        }
    }
};

template <int D, int ELEM, int NW, int STAGES>
struct TmaLayout {
    static constexpr int kTileBytes = 16 * D * ELEM;
    static constexpr int kBoxElems = 128 / ELEM;     // one 128-byte swizzle row per box row
    static constexpr int kStageBytes = 2 * kTileBytes;
    static constexpr int kStagesBytes = NW * STAGES * kStageBytes;
    static constexpr int kRowsMax = 16;   // rows of the merge state per warp
    static size_t smem_bytes(int part_blocks) {
        return 1024 /* alignment slack */ + kStagesBytes + NW * STAGES * sizeof(uint64_t) +
               (size_t)part_blocks * sizeof(int32_t) + 2 * NW * kRowsMax * sizeof(float) + 16;
    }
};

// bf16 kernel: one CTA per (sequence, KV head, partition); NW warps, each with
// its own STAGES-deep TMA ring.
template <int D, class Consumer, int NW, int STAGES>
__global__ void __launch_bounds__(NW * 32)
pa_decode_bf16_kernel(const __grid_constant__ CUtensorMap kmap,
                      const __grid_constant__ CUtensorMap vmap, const DecodeArgs a) {
    using Lay = TmaLayout<D, Consumer::kElemBytes, NW, STAGES>;
    if (!a.defer_wait || blockIdx.x == gridDim.x - 1) grid_dependency_wait();
    grid_dependents_launch();
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    Work w;
    cta_coords(a, a.num_kv_heads, w);
    // The loads that depend only on the CTA's index go out together, so that a
    // CTA waits one memory round trip before its first K/V tile is requested
    // instead of three in a row: the context length, the partition's first
    // table entries (when no sliding window moves the partition with the
    // length) and the query.
    const int len = a.context_lens[w.b];
    constexpr int kPre = 2;   // table entries per thread fetched ahead
    const int tab0 = a.token_offset / kBlockSize + w.part * a.part_blocks;
    const bool use_ahead = Consumer::kEarlyLoads && a.window == 0;
    const int ahead = use_ahead ? min(a.part_blocks, a.max_blocks - tab0) : 0;
    const int32_t *trow_ahead = a.block_tables + (size_t)w.b * a.max_blocks + tab0;
    int32_t pre[kPre];
#pragma unroll
    for (int k = 0; k < kPre; ++k) {
        const int i = threadIdx.x + k * NW * 32;
        pre[k] = i < ahead ? trow_ahead[i] : -1;
    }
    Consumer cons;
    if constexpr (Consumer::kEarlyLoads) cons.init(a, w, lane);
    if (!cta_range(a, len, w)) return;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~uintptr_t(1023));
    uint8_t *stages = smem;
    uint64_t *bars = reinterpret_cast<uint64_t *>(stages + Lay::kStagesBytes);
    int32_t *s_table = reinterpret_cast<int32_t *>(bars + NW * STAGES);
    float *s_m = reinterpret_cast<float *>(s_table + a.part_blocks);
    float *s_l = s_m + NW * Lay::kRowsMax;
    __shared__ int s_fail;

    if (threadIdx.x == 0) {
        s_fail = 0;
        tma_prefetch_desc(&kmap);
        tma_prefetch_desc(&vmap);
    }
    const int32_t *trow =
        a.block_tables + (size_t)w.b * a.max_blocks + a.token_offset / kBlockSize + w.blk0;
    auto put_entry = [&](int i, int phys) {
        if ((unsigned)phys >= (unsigned)a.num_blocks) {
            report(a.status, PA_DEV_BAD_BLOCK_ID);
            phys = 0;
        }
        s_table[i] = phys;
    };
    // without a window the partition starts at tab0, so the entries fetched
    // ahead are its first ones (all it has, up to kPre * NW * 32)
#pragma unroll
    for (int k = 0; k < kPre; ++k) {
        const int i = threadIdx.x + k * NW * 32;
        if (i < w.nblk) put_entry(i, use_ahead ? pre[k] : trow[i]);
    }
    for (int i = threadIdx.x + kPre * NW * 32; i < w.nblk; i += NW * 32) put_entry(i, trow[i]);
    uint64_t *my_bars = bars + warp * STAGES;
    uint8_t *my_stages = stages + warp * STAGES * Lay::kStageBytes;
    if (lane == 0) {
#pragma unroll
        for (int s = 0; s < STAGES; ++s) mbar_init(&my_bars[s], 1);
        fence_mbar_init();
    }
    __syncthreads();
    if constexpr (!Consumer::kEarlyLoads) cons.init(a, w, lane);

    const int my_count = w.nblk > warp ? (w.nblk - warp + NW - 1) / NW : 0;
    const int row_base = w.head * kBlockSize;   // + phys * Hkv * 16

    // Each K/V tile is read once per call: it leaves L2 first, so that what is
    // read again (tables, queries, partials, a shared prefix) stays.
    const uint64_t stream_policy = l2_policy_evict_first();
    auto issue = [&](int it) {
        const int s = it % STAGES;
        const int phys = s_table[warp + it * NW];
        const int y = phys * a.num_kv_heads * kBlockSize + row_base;
        uint8_t *kt = my_stages + s * Lay::kStageBytes;
        uint8_t *vt = kt + Lay::kTileBytes;
        mbar_arrive_expect_tx(&my_bars[s], Lay::kStageBytes);
#pragma unroll
        for (int x = 0; x < D; x += Lay::kBoxElems) {
            tma_load_2d_hint(kt + (x / Lay::kBoxElems) * 2048, &kmap, x, y, &my_bars[s], stream_policy);
            tma_load_2d_hint(vt + (x / Lay::kBoxElems) * 2048, &vmap, x, y, &my_bars[s], stream_policy);
        }
    };

    if (lane == 0)
        for (int it = 0; it < STAGES && it < my_count; ++it) issue(it);

    bool ok = true;
    int it = 0;
    for (; it < my_count; ++it) {
        const int s = it % STAGES;
        const bool done = mbar_wait_bounded(&my_bars[s], (it / STAGES) & 1);
        if (!__all_sync(kFull, done)) {
            ok = false;
            break;
        }
        const int tok0 = (w.blk0 + warp + it * NW) * kBlockSize;
        const int nvalid = min(kBlockSize, w.L - tok0);
        const int nlo = max(0, w.start - tok0);
        const uint32_t kt = smem_u32(my_stages + s * Lay::kStageBytes);
        cons.block(kt, kt + Lay::kTileBytes, nlo, nvalid);
        __syncwarp();
        if (lane == 0 && it + STAGES < my_count) {
            fence_proxy_async_smem();
            issue(it + STAGES);
        }
    }
    if (!ok) {
        // Give every copy still in flight a bounded chance to land before the
        // CTA's shared memory is released, then drop this CTA's result.
        for (int k = it; k < my_count && k < it + STAGES; ++k)
            (void)mbar_wait_bounded(&my_bars[k % STAGES], (k / STAGES) & 1);
        if (lane == 0) {
            report(a.status, PA_DEV_TIMEOUT);
            s_fail = 1;
        }
    }

    float *acc_out = reinterpret_cast<float *>(my_stages);   // the ring is idle now
    cons.finish(acc_out, s_m + warp * Lay::kRowsMax, s_l + warp * Lay::kRowsMax);
    if (my_count == 0 && lane == 0) {
        for (int r = 0; r < Consumer::ROWS; ++r) {
            s_m[warp * Lay::kRowsMax + r] = -INFINITY;
            s_l[warp * Lay::kRowsMax + r] = 0.f;
        }
    }
    __syncthreads();
    if (s_fail) return;
    merge_and_store<__nv_bfloat16, NW>(a, w, w.head * Consumer::ROWS, Consumer::ROWS, D,
                                       reinterpret_cast<const float *>(stages),
                                       STAGES * Lay::kStageBytes / 4, s_m, s_l, Lay::kRowsMax);
}

// ---------------------------------------------------------------------------
// Shared-prefix (cascade) attention.  When every block table of the batch
// starts with the same physical blocks, those blocks' K/V are the same for all
// sequences: instead of each sequence streaming them, the prefix is streamed
// once per KV head for query rows taken across sequences.  Head dimension 128
// with groups the tcgen05 kernel supports runs it there (pa_prefill.cu, prefix
// mode: 256 rows per K/V tile); other shapes use the kernel below, where one
// CTA streams a chunk of the prefix for 64 query rows (16 per warp) as dense
// 16-row mma.sync tiles (query rows on M, tokens and head-dim elements on N/K;
// P.V with P split into bf16 head and residual).  Each (row, prefix chunk)
// leaves a partial (max, sum, output) in the workspace; the suffix of every
// context runs through the decode kernel in partial mode, and the merge kernel
// combines both.  The attention arithmetic is unchanged: the softmax over the
// whole context is the merge of softmaxes over its parts.
// ---------------------------------------------------------------------------
template <int D>
struct PrefixWarp {
    static constexpr int KS = D / 16;
    static constexpr int NT = D / 8;

    uint32_t qa[KS][4];
    float o[NT][4];
    float m0, m1, l0, l1;
    int lim0, lim1;     // tokens of the rows' contexts (positions >= limit are masked)
    float scale_log2;
    int lane, g, t;

    // rows r0 + g and r0 + g + 8 of this KV head's query rows (row = b * G + j)
    __device__ __forceinline__ void init(const DecodeArgs &a, int kvh, int group, int rows_total,
                                         int r0, int lane_) {
        lane = lane_;
        g = lane >> 2;
        t = lane & 3;
        scale_log2 = a.scale_log2;
        const int lmax = a.max_blocks * kBlockSize;
        int lims[2];
        const uint32_t *qr[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int r = r0 + g + 8 * k;
            if (r < rows_total) {
                const int b = r / group, j = r - b * group;
                const int L = a.context_lens[b];
                lims[k] = L < 0 ? 0 : (L > lmax ? lmax : L);
                qr[k] = reinterpret_cast<const uint32_t *>(
                    static_cast<const __nv_bfloat16 *>(a.query) +
                    ((size_t)b * a.num_q_heads + (size_t)kvh * group + j) * D);
            } else {
                lims[k] = 0;
                qr[k] = nullptr;
            }
        }
        lim0 = lims[0];
        lim1 = lims[1];
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            qa[ks][0] = qr[0] ? qr[0][(16 * ks + 2 * t) / 2] : 0u;
            qa[ks][2] = qr[0] ? qr[0][(16 * ks + 8 + 2 * t) / 2] : 0u;
            qa[ks][1] = qr[1] ? qr[1][(16 * ks + 2 * t) / 2] : 0u;
            qa[ks][3] = qr[1] ? qr[1][(16 * ks + 8 + 2 * t) / 2] : 0u;
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
        m0 = m1 = -INFINITY;
        l0 = l1 = 0.f;
    }

    // One full 16-token block whose first token has context position tok0.
    __device__ __forceinline__ void block(uint32_t ktile, uint32_t vtile, int tok0) {
        // two independent accumulation chains per n-tile halve the dependent
        // mma chain of Q.K^T
        float s[2][4], u[2][4];
#pragma unroll
        for (int j = 0; j < 2; ++j)
            s[j][0] = s[j][1] = s[j][2] = s[j][3] = u[j][0] = u[j][1] = u[j][2] = u[j][3] = 0.f;
        const int mi = lane >> 3, rr = lane & 7;
#pragma unroll
        for (int kk = 0; kk < D / 32; ++kk) {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                uint32_t b[4];
                ldsm_x4(b, swz(ktile, 8 * j + rr, 4 * kk + mi));
                mma_bf16_16816(s[j], qa[2 * kk], b[0], b[1]);
                mma_bf16_16816(u[j], qa[2 * kk + 1], b[2], b[3]);
            }
        }
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) s[j][e] += u[j][e];
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int tok = tok0 + 8 * j + 2 * t + (e & 1);
                const int lim = e < 2 ? lim0 : lim1;
                s[j][e] = tok < lim ? s[j][e] * scale_log2 : -INFINITY;
            }
        float mx0 = fmaxf(fmaxf(s[0][0], s[0][1]), fmaxf(s[1][0], s[1][1]));
        float mx1 = fmaxf(fmaxf(s[0][2], s[0][3]), fmaxf(s[1][2], s[1][3]));
        mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, 2));
        // a row may have no valid token yet (all -inf): keep its state at zero
        const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
        const float ref0 = mn0 == -INFINITY ? 0.f : mn0, ref1 = mn1 == -INFINITY ? 0.f : mn1;
        const float a0 = exp2f(m0 - ref0), a1 = exp2f(m1 - ref1);
        m0 = mn0;
        m1 = mn1;
        float p[2][4];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            p[j][0] = ex2_fast(s[j][0] - ref0);
            p[j][1] = ex2_fast(s[j][1] - ref0);
            p[j][2] = ex2_fast(s[j][2] - ref1);
            p[j][3] = ex2_fast(s[j][3] - ref1);
        }
        l0 = l0 * a0 + (p[0][0] + p[0][1]) + (p[1][0] + p[1][1]);
        l1 = l1 * a1 + (p[0][2] + p[0][3]) + (p[1][2] + p[1][3]);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            o[nt][0] *= a0;
            o[nt][1] *= a0;
            o[nt][2] *= a1;
            o[nt][3] *= a1;
        }
        uint32_t pa[4], pl[4];
        split_bf16x2(p[0][0], p[0][1], pa[0], pl[0]);
        split_bf16x2(p[0][2], p[0][3], pa[1], pl[1]);
        split_bf16x2(p[1][0], p[1][1], pa[2], pl[2]);
        split_bf16x2(p[1][2], p[1][3], pa[3], pl[3]);
#pragma unroll
        for (int dd = 0; dd < D / 16; ++dd) {
            uint32_t b[4];
            ldsm_x4_trans(b, swz(vtile, (mi & 1) * 8 + rr, 2 * dd + (mi >> 1)));
            mma_bf16_16816(o[2 * dd], pa, b[0], b[1]);
            mma_bf16_16816(o[2 * dd + 1], pa, b[2], b[3]);
            mma_bf16_16816(o[2 * dd], pl, b[0], b[1]);
            mma_bf16_16816(o[2 * dd + 1], pl, b[2], b[3]);
        }
    }

    // Partial state of rows r0 + g and r0 + g + 8 into workspace partition `part`.
    __device__ __forceinline__ void store(const DecodeArgs &a, int kvh, int group, int rows_total,
                                          int r0, int part) {
        l0 += __shfl_xor_sync(kFull, l0, 1);
        l0 += __shfl_xor_sync(kFull, l0, 2);
        l1 += __shfl_xor_sync(kFull, l1, 1);
        l1 += __shfl_xor_sync(kFull, l1, 2);
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int r = r0 + g + 8 * k;
            if (r >= rows_total) continue;
            const int b = r / group, j = r - b * group;
            const size_t row =
                ((size_t)b * a.num_q_heads + (size_t)kvh * group + j) * a.max_parts + part;
            float *dst = a.part_o + row * D;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
                *reinterpret_cast<float2 *>(dst + 8 * nt + 2 * t) =
                    k == 0 ? make_float2(o[nt][0], o[nt][1]) : make_float2(o[nt][2], o[nt][3]);
            if (t == 0) a.part_ml[row] = k == 0 ? make_float2(m0, l0) : make_float2(m1, l1);
        }
    }
};

constexpr int kPrefixWarps = 4;     // consumer warps; one more warp issues the TMA loads
constexpr int kPrefixRows = 16 * kPrefixWarps;

template <int D, int STAGES>
__global__ void __launch_bounds__((kPrefixWarps + 1) * 32)
pa_prefix_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                 const DecodeArgs a) {
    constexpr int kTile = 16 * D * 2;
    constexpr int kStage = 2 * kTile;
    grid_dependency_wait();
    grid_dependents_launch();
    const int group = a.num_q_heads / a.num_kv_heads;
    const int rows_total = a.num_seqs * group;
    const int row_chunks = (rows_total + kPrefixRows - 1) / kPrefixRows;
    int idx = blockIdx.x;
    const int pc = idx % a.prefix_chunks;
    idx /= a.prefix_chunks;
    const int rc = idx % row_chunks;
    const int kvh = idx / row_chunks;
    const int blk0 = pc * a.prefix_chunk_blocks;
    const int nblk = min(a.prefix_blocks - blk0, a.prefix_chunk_blocks);

    extern __shared__ uint8_t smem_raw[];
    uint8_t *stages = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                  ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(stages + STAGES * kStage);
    uint64_t *empty = full + STAGES;
    int32_t *s_table = reinterpret_cast<int32_t *>(empty + STAGES);
    __shared__ int s_fail;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        s_fail = 0;
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kPrefixWarps);
        }
        fence_mbar_init();
        tma_prefetch_desc(&kmap);
        tma_prefetch_desc(&vmap);
    }
    // the shared blocks, from the first sequence's table
    for (int i = threadIdx.x; i < nblk; i += blockDim.x) {
        int phys = a.block_tables[blk0 + i];
        if ((unsigned)phys >= (unsigned)a.num_blocks) {
            report(a.status, PA_DEV_BAD_BLOCK_ID);
            phys = 0;
        }
        s_table[i] = phys;
    }
    // every sequence of this row chunk must list the same blocks (checked once,
    // by the CTAs of KV head 0)
    if (kvh == 0) {
        const int b_first = rc * kPrefixRows / group;
        const int b_last = min(a.num_seqs, ((rc + 1) * kPrefixRows + group - 1) / group);
        for (int i = threadIdx.x; i < (b_last - b_first) * nblk; i += blockDim.x) {
            const int b = b_first + i / nblk, j = blk0 + i % nblk;
            if (a.block_tables[(size_t)b * a.max_blocks + j] != a.block_tables[j])
                report(a.status, PA_DEV_PREFIX_MISMATCH);
        }
    }
    __syncthreads();

    if (warp == kPrefixWarps) {          // producer
        if (lane == 0) {
            for (int it = 0; it < nblk; ++it) {
                const int s = it % STAGES;
                if (it >= STAGES && !mbar_wait_bounded(&empty[s], ((it / STAGES) - 1) & 1)) {
                    report(a.status, PA_DEV_TIMEOUT);
                    s_fail = 1;
                    break;
                }
                const int y = (s_table[it] * a.num_kv_heads + kvh) * kBlockSize;
                uint8_t *kt = stages + s * kStage;
                uint8_t *vt = kt + kTile;
                mbar_arrive_expect_tx(&full[s], kStage);
#pragma unroll
                for (int x = 0; x < D; x += 64) {
                    tma_load_2d(kt + (x / 64) * 2048, &kmap, x, y, &full[s]);
                    tma_load_2d(vt + (x / 64) * 2048, &vmap, x, y, &full[s]);
                }
            }
        }
        return;
    }

    PrefixWarp<D> pw;
    const int r0 = rc * kPrefixRows + warp * 16;
    pw.init(a, kvh, group, rows_total, r0, lane);
    bool ok = true;
    int it = 0;
    for (; it < nblk; ++it) {
        const int s = it % STAGES;
        const bool done = mbar_wait_bounded(&full[s], (it / STAGES) & 1);
        if (!__all_sync(kFull, done)) {
            ok = false;
            break;
        }
        const uint32_t kt = smem_u32(stages + s * kStage);
        pw.block(kt, kt + kTile, (blk0 + it) * kBlockSize);
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }
    if (!ok) {
        // give copies that may still be in flight a bounded chance to land first
        for (int k = it; k < nblk && k < it + STAGES; ++k)
            (void)mbar_wait_bounded(&full[k % STAGES], (k / STAGES) & 1);
        if (lane == 0) report(a.status, PA_DEV_TIMEOUT);
        return;
    }
    pw.store(a, kvh, group, rows_total, r0, pc);
}

// fp32 kernel: one CTA per (sequence, query head, partition); lane owns
// head-dim elements lane + 32 e.  Plain loads; online softmax per token.
template <int D, int NW>
__global__ void __launch_bounds__(NW * 32) pa_decode_f32_kernel(const float *__restrict__ kc,
                                                                const float *__restrict__ vc,
                                                                const DecodeArgs a) {
    constexpr int EPL = D / 32;
    grid_dependency_wait();
    grid_dependents_launch();
    Work w;
    if (!cta_work(a, a.num_q_heads, w)) return;
    __shared__ float s_acc[NW][D];
    __shared__ float s_m[NW], s_l[NW];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int group = a.num_q_heads / a.num_kv_heads;
    const int kvh = w.head / group;
    const float *qrow = static_cast<const float *>(a.query) + ((size_t)w.b * a.num_q_heads + w.head) * D;
    float q[EPL], acc[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
        q[e] = qrow[lane + 32 * e] * a.scale_log2;
        acc[e] = 0.f;
    }
    float m = -INFINITY, l = 0.f;
    const int32_t *trow =
        a.block_tables + (size_t)w.b * a.max_blocks + a.token_offset / kBlockSize + w.blk0;
    for (int j = warp; j < w.nblk; j += NW) {
        int phys = trow[j];
        if ((unsigned)phys >= (unsigned)a.num_blocks) {
            if (lane == 0) report(a.status, PA_DEV_BAD_BLOCK_ID);
            phys = 0;
        }
        const int tok0 = (w.blk0 + j) * kBlockSize;
        const int nvalid = min(kBlockSize, w.L - tok0);
        const int nlo = max(0, w.start - tok0);
        const size_t base = (((size_t)phys * a.num_kv_heads + kvh) * kBlockSize) * D;
        for (int r = nlo; r < nvalid; ++r) {
            const float *krow = kc + base + (size_t)r * D;
            const float *vrow = vc + base + (size_t)r * D;
            float s = 0.f;
#pragma unroll
            for (int e = 0; e < EPL; ++e) s = fmaf(q[e], krow[lane + 32 * e], s);
#pragma unroll
            for (int M = 16; M >= 1; M >>= 1) s += __shfl_xor_sync(kFull, s, M);
            const float m_new = fmaxf(m, s);
            const float alpha = exp2f(m - m_new);
            const float p = ex2_fast(s - m_new);
            l = l * alpha + p;
#pragma unroll
            for (int e = 0; e < EPL; ++e) acc[e] = fmaf(p, vrow[lane + 32 * e], acc[e] * alpha);
            m = m_new;
        }
    }
#pragma unroll
    for (int e = 0; e < EPL; ++e) s_acc[warp][lane + 32 * e] = acc[e];
    if (lane == 0) {
        s_m[warp] = m;
        s_l[warp] = l;
    }
    __syncthreads();
    merge_and_store<float, NW>(a, w, w.head, 1, D, &s_acc[0][0], D, s_m, s_l, 1);
}

// Merges the partitions of every (sequence, query head) that has more than one.
// Merge of the split-K partials: one warp per (sequence, query head) row, four
// rows per CTA.  Every lane owns D/128 float4 columns of the output; the
// partials' (max, sum) pairs are read by the lanes in parallel, and the
// partial rows are loaded eight at a time so that their L2 latencies overlap.
constexpr int kReduceRows = 4;
constexpr int kReduceSpec = 8;   // shared-prefix merge: partial rows read in the first round

template <typename OutT>
__global__ void __launch_bounds__(32 * kReduceRows) pa_reduce_kernel(const DecodeArgs a, int D) {
    grid_dependency_wait();
    grid_dependents_launch();
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * kReduceRows + (threadIdx.x >> 5);
    if (row >= a.num_seqs * a.num_q_heads) return;
    const int b = row / a.num_q_heads;
    const int q4 = D >> 2;                         // float4 columns per row
    if (a.always_partial && a.part_base < kReduceSpec && q4 <= 32) {
        // Shared-prefix merge: every row has the prefix chunks' partials and at
        // least one suffix partial, so those kSpec = part_base + 1 rows are read
        // at once with the context length (one round of L2 latency); only a
        // context with several suffix partitions reads more.
        const int kSpec = a.part_base + 1;
        const size_t row0 = (size_t)row * a.max_parts;
        const float2 *ml = a.part_ml + row0;
        const float4 *po = reinterpret_cast<const float4 *>(a.part_o + row0 * D);
        int L = a.context_lens[b];
        float2 m_l[kReduceSpec];
        float4 v[kReduceSpec];
#pragma unroll
        for (int i = 0; i < kReduceSpec; ++i) {
            if (i < kSpec) {
                m_l[i] = ml[i];
                v[i] = lane < q4 ? po[(size_t)i * q4 + lane] : make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
        const int lmax = a.max_blocks * kBlockSize;
        L = L < 0 ? 0 : (L > lmax ? lmax : L);
        L = max(L - a.token_offset, 0);
        const int range = (L + kBlockSize - 1) / kBlockSize;
        const int nparts = a.part_base + (range <= 0 ? 1 : (range + a.part_blocks - 1) / a.part_blocks);
        float M = -INFINITY;
#pragma unroll
        for (int i = 0; i < kReduceSpec; ++i)
            if (i < kSpec) M = fmaxf(M, m_l[i].x);
        for (int p = kSpec; p < nparts; ++p) M = fmaxf(M, ml[p].x);
        float Lsum = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        auto add = [&](float2 mlp, float4 o) {
            const float w = mlp.x == -INFINITY ? 0.f : exp2f(mlp.x - M);
            Lsum = fmaf(w, mlp.y, Lsum);
            acc.x = fmaf(w, o.x, acc.x);
            acc.y = fmaf(w, o.y, acc.y);
            acc.z = fmaf(w, o.z, acc.z);
            acc.w = fmaf(w, o.w, acc.w);
        };
#pragma unroll
        for (int i = 0; i < kReduceSpec; ++i)
            if (i < kSpec) add(m_l[i], v[i]);
        for (int p = kSpec; p < nparts; ++p)
            add(ml[p], lane < q4 ? po[(size_t)p * q4 + lane] : make_float4(0.f, 0.f, 0.f, 0.f));
        if (lane < q4) {
            const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
            OutT *out = static_cast<OutT *>(a.out) + (size_t)row * D + 4 * lane;
            store_out<OutT>(out + 0, acc.x * inv);
            store_out<OutT>(out + 1, acc.y * inv);
            store_out<OutT>(out + 2, acc.z * inv);
            store_out<OutT>(out + 3, acc.w * inv);
        }
        return;
    }
    int L = a.context_lens[b];
    const int lmax = a.max_blocks * kBlockSize;
    L = L < 0 ? 0 : (L > lmax ? lmax : L);
    L = max(L - a.token_offset, 0);
    const int start = (a.window > 0 && L > a.window) ? L - a.window : 0;
    const int range = (L + kBlockSize - 1) / kBlockSize - start / kBlockSize;
    const int nparts =
        a.part_base + (range <= 0 ? 1 : (range + a.part_blocks - 1) / a.part_blocks);
    if (nparts <= 1 && !a.always_partial) return;
    const size_t row0 = (size_t)row * a.max_parts;
    const float2 *ml = a.part_ml + row0;
    float M = -INFINITY;
    for (int p = lane; p < nparts; p += 32) M = fmaxf(M, ml[p].x);
#pragma unroll
    for (int k = 16; k >= 1; k >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, k));
    float Lsum = 0.f;
    for (int p = lane; p < nparts; p += 32) {
        const float2 v = ml[p];
        Lsum += v.x == -INFINITY ? 0.f : exp2f(v.x - M) * v.y;
    }
#pragma unroll
    for (int k = 16; k >= 1; k >>= 1) Lsum += __shfl_xor_sync(kFull, Lsum, k);
    const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
    const float4 *po = reinterpret_cast<const float4 *>(a.part_o + row0 * D);
    OutT *out = static_cast<OutT *>(a.out) + (size_t)row * D;
    for (int q = lane; q < q4; q += 32) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int p0 = 0; p0 < nparts; p0 += 8) {
            float4 v[8];
            float w[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                if (p0 + i < nparts) {
                    v[i] = po[(size_t)(p0 + i) * q4 + q];
                    const float mi = ml[p0 + i].x;
                    w[i] = mi == -INFINITY ? 0.f : exp2f(mi - M);
                } else {
                    v[i] = make_float4(0.f, 0.f, 0.f, 0.f);
                    w[i] = 0.f;
                }
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                acc.x = fmaf(w[i], v[i].x, acc.x);
                acc.y = fmaf(w[i], v[i].y, acc.y);
                acc.z = fmaf(w[i], v[i].z, acc.z);
                acc.w = fmaf(w[i], v[i].w, acc.w);
            }
        }
        store_out<OutT>(out + 4 * q + 0, acc.x * inv);
        store_out<OutT>(out + 4 * q + 1, acc.y * inv);
        store_out<OutT>(out + 4 * q + 2, acc.z * inv);
        store_out<OutT>(out + 4 * q + 3, acc.w * inv);
    }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
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

// 2-D view of a pool as [num_blocks * num_kv_heads * 16 rows][head_dim]
// elements, loaded as boxes of 16 rows x 128 bytes with 128-byte swizzle.
bool encode_pool_map(CUtensorMap *map, const void *pool, int64_t rows, int D, int elem_bytes) {
    auto enc = tensor_map_encoder();
    if (enc == nullptr) return false;
    cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)D * elem_bytes};
    cuuint32_t box[2] = {(cuuint32_t)(128 / elem_bytes), 16};
    cuuint32_t estr[2] = {1, 1};
    const CUtensorMapDataType type =
        elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    CUresult r = enc(map, type, 2, const_cast<void *>(pool), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <typename K>
cudaError_t allow_smem(K kernel, size_t bytes) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

// Warps per CTA and TMA stages per warp of the bf16 kernels (compile-time
// tunables, one pair per consumer).  What sets the speed on GB300 is the
// number of consumer warps resident per SM, not the depth of each ring:
//  * MHA (72 registers): 8 warps x 1 stage x 8 KiB = 64 KiB, three CTAs and 24
//    warps per SM;
//  * GQA groups of 9..16 (heads-as-rows consumer, about 140 registers, so at
//    most ~14 warps per SM): 4 warps x 2 stages, three CTAs, 12 warps per SM;
//  * GQA groups of 2..8 (transposed consumer): PA_GQA_WARPS x PA_GQA_STAGES.
// (Measured alternatives at head_dim 128: 4x1, 2x2, 3x2, 4x3, 4x4, 8x2, 8x3,
// 2x6 all streamed slower for the consumer they were tried on.)
#ifndef PA_MHA_WARPS
#define PA_MHA_WARPS 8
#endif
#ifndef PA_MHA_STAGES
#define PA_MHA_STAGES 1
#endif
#ifndef PA_GQA_WARPS
#define PA_GQA_WARPS 4
#endif
#ifndef PA_GQA_STAGES
#define PA_GQA_STAGES 2
#endif
#ifndef PA_GQA16_WARPS
#define PA_GQA16_WARPS 4
#endif
#ifndef PA_GQA16_STAGES
#define PA_GQA16_STAGES 2
#endif
// FP8 pools (4 KiB per block): MHA 8 warps x 2 stages (64 KiB, three CTAs per
// SM); GQA 6 warps x 3 stages (72 KiB, three CTAs per SM).  Measured
// alternatives: MHA 8x3, 12x2, 6x3, 4x4 (7B-shaped batch 92.3 us at 8x2 against
// 94.5-105.1 us); GQA 8x3, 8x2, 4x4, 12x2 (70B-shaped batch 198.2 us at 6x3
// against 200.9-244.0 us).
#ifndef PA_MHA8_WARPS
#define PA_MHA8_WARPS 8
#endif
#ifndef PA_MHA8_STAGES
#define PA_MHA8_STAGES 2
#endif
#ifndef PA_GQA8_WARPS
#define PA_GQA8_WARPS 6
#endif
#ifndef PA_GQA8_STAGES
#define PA_GQA8_STAGES 3
#endif
// FP8 GQA CTAs that stream at most PA_GQA8S_MAX_BLOCKS blocks (short contexts,
// e.g. the part of a context past a shared prefix, or a sliding window):
// 2 warps x 2 stages, many small CTAs per SM so that one CTA's fixed latency
// (length, table, first tile; merge and store) overlaps the others' streaming.
// Shared-prefix FP8 call 41.7 us (4 x 2: 43.1, 8 x 2: 54.3, 1 x 3: 50.0);
// 70B-shaped batch with a 512-token window 57.5 us (4 x 2: 59.9), 1024-token
// window 91.9 us (4 x 2: 92.8).
#ifndef PA_GQA8S_WARPS
#define PA_GQA8S_WARPS 2
#endif
#ifndef PA_GQA8S_STAGES
#define PA_GQA8S_STAGES 2
#endif
#ifndef PA_GQA8S_MAX_BLOCKS
#define PA_GQA8S_MAX_BLOCKS 128
#endif
#ifndef PA_MHA8T_MAX_BLOCKS
#define PA_MHA8T_MAX_BLOCKS 64
#endif
constexpr int kNW = 4;   // fp32 kernel

template <int D, class Consumer, int NW, int STAGES>
pa_status launch_bf16(const DecodeArgs &a, const void *kc, const void *vc, int64_t rows,
                      cudaStream_t stream) {
    CUtensorMap kmap, vmap;
    if (!encode_pool_map(&kmap, kc, rows, D, Consumer::kElemBytes) ||
        !encode_pool_map(&vmap, vc, rows, D, Consumer::kElemBytes))
        return cuda_failure(cudaErrorInvalidValue, "cuTensorMapEncodeTiled");
    const size_t smem = TmaLayout<D, Consumer::kElemBytes, NW, STAGES>::smem_bytes(a.part_blocks);
    auto kernel = pa_decode_bf16_kernel<D, Consumer, NW, STAGES>;
    cudaError_t e = allow_smem(kernel, smem);
    if (e != cudaSuccess) return cuda_failure(e, "cudaFuncSetAttribute(decode)");
    // partitions this kernel owns (the workspace rows before part_base belong to
    // the shared-prefix kernel)
    const int64_t grid = (int64_t)a.num_seqs * a.num_kv_heads * (a.max_parts - a.part_base);
    e = launch_chained(kernel, dim3((unsigned)grid), dim3(NW * 32), smem, stream, kmap, vmap, a);
    if (e != cudaSuccess) return cuda_failure(e, "pa_decode_bf16_kernel launch");
    count_launches(1);
    return PA_OK;
}

template <int D, int G>
pa_status launch_gqa(const DecodeArgs &a, const void *kc, const void *vc, int64_t rows,
                     cudaStream_t stream) {
    if constexpr (G <= 8)
        return launch_bf16<D, GqaTConsumer<D, G>, PA_GQA_WARPS, PA_GQA_STAGES>(a, kc, vc, rows,
                                                                             stream);
    else
        return launch_bf16<D, GqaConsumer<D, G>, PA_GQA16_WARPS, PA_GQA16_STAGES>(a, kc, vc, rows,
                                                                                stream);
}

template <int D>
pa_status dispatch_bf16(int group, const DecodeArgs &a, const void *kc, const void *vc,
                        int64_t rows, cudaStream_t stream) {
    switch (group) {
    case 1: return launch_bf16<D, MhaConsumer<D>, PA_MHA_WARPS, PA_MHA_STAGES>(a, kc, vc, rows, stream);
    case 2: return launch_gqa<D, 2>(a, kc, vc, rows, stream);
    case 3: return launch_gqa<D, 3>(a, kc, vc, rows, stream);
    case 4: return launch_gqa<D, 4>(a, kc, vc, rows, stream);
    case 5: return launch_gqa<D, 5>(a, kc, vc, rows, stream);
    case 6: return launch_gqa<D, 6>(a, kc, vc, rows, stream);
    case 7: return launch_gqa<D, 7>(a, kc, vc, rows, stream);
    case 8: return launch_gqa<D, 8>(a, kc, vc, rows, stream);
    case 12: return launch_gqa<D, 12>(a, kc, vc, rows, stream);
    case 16: return launch_gqa<D, 16>(a, kc, vc, rows, stream);
    default: return PA_ERR_UNSUPPORTED;
    }
}

template <int G>
pa_status launch_gqa_fp8(bool short_span, const DecodeArgs &a, const void *kc, const void *vc,
                         int64_t rows, cudaStream_t stream) {
    constexpr int D = 128;
    if (short_span)
        return launch_bf16<D, GqaTFp8Consumer<D, G>, PA_GQA8S_WARPS, PA_GQA8S_STAGES>(a, kc, vc, rows,
                                                                                    stream);
    return launch_bf16<D, GqaTFp8Consumer<D, G>, PA_GQA8_WARPS, PA_GQA8_STAGES>(a, kc, vc, rows,
                                                                              stream);
}

pa_status dispatch_fp8(int group, const DecodeArgs &a, const void *kc, const void *vc,
                       int64_t rows, cudaStream_t stream) {
    constexpr int D = 128;
    // blocks one CTA streams at most: short spans take the narrower GQA CTA
    int span = std::min(a.part_blocks, std::max(0, a.max_blocks - a.token_offset / kBlockSize));
    if (a.window > 0) span = std::min(span, a.window / kBlockSize + 1);
    const bool short_span = span <= PA_GQA8S_MAX_BLOCKS;
    switch (group) {
    case 1:
        // CTAs of at most PA_MHA8T_MAX_BLOCKS blocks (e.g. 512-token partitions
        // of long contexts) take the tensor-core consumer with one real query
        // head of its eight n-tile columns: fewer instructions per block than
        // the CUDA-core consumer (long_splitk 32k contexts: 327.8 against
        // 337.0 us); longer spans keep the CUDA-core consumer (7B-shaped batch:
        // 93.3 against 96.7 us).
        if (span <= PA_MHA8T_MAX_BLOCKS)
            return launch_bf16<D, GqaTFp8Consumer<D, 1>, PA_GQA8S_WARPS, PA_GQA8S_STAGES>(a, kc, vc, rows,
                                                                                        stream);
        return launch_bf16<D, MhaFp8Consumer<D>, PA_MHA8_WARPS, PA_MHA8_STAGES>(a, kc, vc, rows, stream);
    case 2: return launch_gqa_fp8<2>(short_span, a, kc, vc, rows, stream);
    case 3: return launch_gqa_fp8<3>(short_span, a, kc, vc, rows, stream);
    case 4: return launch_gqa_fp8<4>(short_span, a, kc, vc, rows, stream);
    case 5: return launch_gqa_fp8<5>(short_span, a, kc, vc, rows, stream);
    case 6: return launch_gqa_fp8<6>(short_span, a, kc, vc, rows, stream);
    case 7: return launch_gqa_fp8<7>(short_span, a, kc, vc, rows, stream);
    case 8: return launch_gqa_fp8<8>(short_span, a, kc, vc, rows, stream);
    default: return PA_ERR_UNSUPPORTED;
    }
}

template <int D>
pa_status launch_f32(const DecodeArgs &a, const void *kc, const void *vc, cudaStream_t stream) {
    const int64_t grid = (int64_t)a.num_seqs * a.num_q_heads * a.max_parts;
    cudaError_t e = launch_chained(pa_decode_f32_kernel<D, kNW>, dim3((unsigned)grid),
                                   dim3(kNW * 32), 0, stream, static_cast<const float *>(kc),
                                   static_cast<const float *>(vc), a);
    if (e != cudaSuccess) return cuda_failure(e, "pa_decode_f32_kernel launch");
    count_launches(1);
    return PA_OK;
}

template <typename OutT>
pa_status launch_reduce(const DecodeArgs &a, int D, cudaStream_t stream) {
    auto kernel = pa_reduce_kernel<OutT>;
    const int64_t rows = (int64_t)a.num_seqs * a.num_q_heads;
    const unsigned grid = (unsigned)((rows + kReduceRows - 1) / kReduceRows);
    cudaError_t e = launch_chained(kernel, dim3(grid), dim3(32 * kReduceRows), 0, stream, a, D);
    if (e != cudaSuccess) return cuda_failure(e, "pa_reduce_kernel launch");
    count_launches(1);
    return PA_OK;
}

// Streaming multiprocessors of the current device (GB300's 152 when the
// runtime cannot tell, e.g. in a process without a GPU).
int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
        (void)cudaGetLastError();
        return 152;
    }
    return n;
}

// Partition size for partition_size == 0: the largest of kAutoPartitionMax
// .. 128 tokens that still gives at least four CTAs per SM when every
// sequence is as long as the table allows.  Long partitions amortise each
// CTA's fixed cost (table slice, pipeline fill, merge) and need fewer
// partials; enough CTAs keep every SM streaming to the end.
#ifndef PA_AUTO_PARTITION_MAX
#define PA_AUTO_PARTITION_MAX 4096
#endif
int auto_partition(int num_seqs, int heads_axis, int max_blocks) {
    const int64_t target = 4LL * sm_count();
    for (int p = PA_AUTO_PARTITION_MAX; p > 128; p /= 2) {
        const int pb = p / kBlockSize;
        const int64_t parts = std::max(1, (max_blocks + pb - 1) / pb);
        if ((int64_t)num_seqs * heads_axis * parts >= target) return p;
    }
    return 128;
}

int resolve_partition(int partition_size, int num_seqs, int heads_axis, int max_blocks) {
    const int p = partition_size == 0 ? auto_partition(num_seqs, heads_axis, max_blocks)
                                      : partition_size;
    if (p < kBlockSize || p > kMaxPartition || p % kBlockSize != 0) return -1;
    return p;
}

size_t workspace_for(int num_seqs, int num_q_heads, int head_dim, int max_parts) {
    if (max_parts <= 1) return 0;
    const size_t rows = (size_t)num_seqs * num_q_heads * max_parts;
    const size_t o_bytes = (rows * head_dim * sizeof(float) + 255) & ~size_t(255);
    return o_bytes + rows * sizeof(float2);
}

}  // namespace
}  // namespace pa

using namespace pa;

extern "C" int pa_decode_partition_size(int num_seqs, int num_q_heads, int num_kv_heads,
                                        int max_blocks_per_seq, pa_dtype dtype) {
    if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || max_blocks_per_seq < 0 ||
        (dtype != PA_DTYPE_F32 && dtype != PA_DTYPE_BF16 && dtype != PA_DTYPE_FP8_E4M3))
        return -1;
    const int heads_axis = dtype == PA_DTYPE_F32 ? num_q_heads : num_kv_heads;
    return auto_partition(num_seqs, heads_axis, max_blocks_per_seq);
}

namespace pa {
namespace {

bool kv_dtype_ok(pa_dtype d) {
    return d == PA_DTYPE_F32 || d == PA_DTYPE_BF16 || d == PA_DTYPE_FP8_E4M3;
}

// Blocks one sequence's decode can touch: the whole table, or for a sliding
// window of W positions at most ceil(W / 16) + 1 blocks (the window's first
// position need not start a block).
int span_blocks(int max_blocks, int window) {
    if (window <= 0) return max_blocks;
    return std::min(max_blocks, (window + kBlockSize - 1) / kBlockSize + 1);
}

// Partition size and partition count of a decode call; false on a bad size.
bool plan_decode(int num_seqs, int num_q_heads, int num_kv_heads, int max_blocks, pa_dtype dtype,
                 int window, int partition_size, int *part_blocks, int *max_parts) {
    const int heads_axis = dtype == PA_DTYPE_F32 ? num_q_heads : num_kv_heads;
    const int span = span_blocks(max_blocks, window);
    const int p = resolve_partition(partition_size, num_seqs, heads_axis, span);
    if (p < 0) return false;
    *part_blocks = p / kBlockSize;
    *max_parts = std::max(1, (span + *part_blocks - 1) / *part_blocks);
    // Every sequence longer than a window covers the same number of blocks
    // (span or span - 1): spread them evenly over the partitions instead of
    // leaving a last partition of a block or two.
    if (window > 0 && partition_size == 0 && *max_parts > 1)
        *part_blocks = (span + *max_parts - 1) / *max_parts;
    return true;
}

size_t decode_workspace(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                        int max_blocks, int block_size, int window, int partition_size,
                        pa_dtype dtype) {
    if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
        max_blocks < 0 || block_size != kBlockSize || window < 0 || !kv_dtype_ok(dtype))
        return (size_t)-1;
    int part_blocks, max_parts;
    if (!plan_decode(num_seqs, num_q_heads, num_kv_heads, max_blocks, dtype, window,
                     partition_size, &part_blocks, &max_parts))
        return (size_t)-1;
    return workspace_for(num_seqs, num_q_heads, head_dim, max_parts);
}

// The one decode path behind pa_decode, pa_decode_fp8 and
// pa_decode_sliding_window: validation, planning, kernel and merge launches.
pa_status decode_common(void *out, const void *query, const void *key_cache,
                        const void *value_cache, const float *k_scales, const float *v_scales,
                        const int32_t *block_tables, const int32_t *context_lens, int num_seqs,
                        int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                        int max_blocks_per_seq, int num_blocks, float scale, pa_dtype dtype,
                        int window, int partition_size, void *workspace, size_t workspace_bytes,
                        int32_t *device_status, void *stream) {
    if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || block_size != kBlockSize ||
        max_blocks_per_seq < 0 || num_blocks <= 0 || num_q_heads % num_kv_heads != 0 ||
        !(scale == scale) || window < 0 || !kv_dtype_ok(dtype))
        return PA_ERR_INVALID_ARG;
    if (partition_size != 0 &&
        (partition_size < kBlockSize || partition_size > kMaxPartition || partition_size % kBlockSize))
        return PA_ERR_INVALID_ARG;
    if (num_seqs == 0) return PA_OK;
    const bool fp8 = dtype == PA_DTYPE_FP8_E4M3;
    if (!out || !query || !key_cache || !value_cache || !block_tables || !context_lens)
        return PA_ERR_INVALID_ARG;
    if (fp8 && (!k_scales || !v_scales)) return PA_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(query) || !aligned16(key_cache) || !aligned16(value_cache))
        return PA_ERR_INVALID_ARG;
    if (fp8 && ((reinterpret_cast<uintptr_t>(k_scales) & 3u) ||
                (reinterpret_cast<uintptr_t>(v_scales) & 3u)))
        return PA_ERR_INVALID_ARG;
    const int group = num_q_heads / num_kv_heads;
    if (dtype == PA_DTYPE_BF16) {
        if (head_dim != 64 && head_dim != 128) return PA_ERR_UNSUPPORTED;
        if (group > 16) return PA_ERR_UNSUPPORTED;
    } else if (fp8) {
        if (head_dim != 128 || group > 8) return PA_ERR_UNSUPPORTED;
    } else {
        if (head_dim != 32 && head_dim != 64 && head_dim != 128 && head_dim != 256)
            return PA_ERR_UNSUPPORTED;
    }
    const int64_t rows = (int64_t)num_blocks * num_kv_heads * kBlockSize;
    if (rows >= ((int64_t)1 << 31)) return PA_ERR_UNSUPPORTED;
    int part_blocks, max_parts;
    if (!plan_decode(num_seqs, num_q_heads, num_kv_heads, max_blocks_per_seq, dtype, window,
                     partition_size, &part_blocks, &max_parts))
        return PA_ERR_INVALID_ARG;
    const int heads_axis = dtype == PA_DTYPE_F32 ? num_q_heads : num_kv_heads;
    if ((int64_t)num_seqs * heads_axis * max_parts >= ((int64_t)1 << 31)) return PA_ERR_UNSUPPORTED;
    const size_t need = workspace_for(num_seqs, num_q_heads, head_dim, max_parts);
    if (need > 0 && (workspace == nullptr || workspace_bytes < need || !aligned16(workspace)))
        return PA_ERR_WORKSPACE;

    DecodeArgs a;
    a.out = out;
    a.query = query;
    a.block_tables = block_tables;
    a.context_lens = context_lens;
    a.part_o = static_cast<float *>(workspace);
    a.part_ml = need > 0 ? reinterpret_cast<float2 *>(
                               static_cast<uint8_t *>(workspace) +
                               (((size_t)num_seqs * num_q_heads * max_parts * head_dim * sizeof(float) +
                                 255) & ~size_t(255)))
                         : nullptr;
    a.status = device_status;
    a.k_scales = fp8 ? k_scales : nullptr;
    a.v_scales = fp8 ? v_scales : nullptr;
    a.num_seqs = num_seqs;
    a.num_q_heads = num_q_heads;
    a.num_kv_heads = num_kv_heads;
    a.max_blocks = max_blocks_per_seq;
    a.num_blocks = num_blocks;
    a.part_blocks = part_blocks;
    a.max_parts = max_parts;
    a.scale_log2 = scale * kLog2e;
    a.token_offset = a.part_base = a.always_partial = 0;
    a.prefix_blocks = a.prefix_chunk_blocks = a.prefix_chunks = 0;
    a.window = window;
    a.defer_wait = 0;
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    pa_status s;
    if (fp8) {
        s = dispatch_fp8(group, a, key_cache, value_cache, rows, st);
    } else if (dtype == PA_DTYPE_BF16) {
        s = head_dim == 64 ? dispatch_bf16<64>(group, a, key_cache, value_cache, rows, st)
                           : dispatch_bf16<128>(group, a, key_cache, value_cache, rows, st);
    } else {
        switch (head_dim) {
        case 32: s = launch_f32<32>(a, key_cache, value_cache, st); break;
        case 64: s = launch_f32<64>(a, key_cache, value_cache, st); break;
        case 128: s = launch_f32<128>(a, key_cache, value_cache, st); break;
        default: s = launch_f32<256>(a, key_cache, value_cache, st); break;
        }
    }
    if (s != PA_OK || max_parts <= 1) return s;
    return dtype == PA_DTYPE_F32 ? launch_reduce<float>(a, head_dim, st)
                                 : launch_reduce<__nv_bfloat16>(a, head_dim, st);
}

}  // namespace
}  // namespace pa

extern "C" size_t pa_decode_workspace_bytes(int num_seqs, int num_q_heads, int num_kv_heads,
                                            int head_dim, int max_blocks_per_seq, int block_size,
                                            int partition_size, pa_dtype dtype) {
    return decode_workspace(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                            block_size, 0, partition_size, dtype);
}

extern "C" pa_status pa_decode(void *out, const void *query, const void *key_cache,
                               const void *value_cache, const int32_t *block_tables,
                               const int32_t *context_lens, int num_seqs, int num_q_heads,
                               int num_kv_heads, int head_dim, int block_size,
                               int max_blocks_per_seq, int num_blocks, float scale, pa_dtype dtype,
                               int partition_size, void *workspace, size_t workspace_bytes,
                               int32_t *device_status, void *stream) {
    if (dtype != PA_DTYPE_F32 && dtype != PA_DTYPE_BF16) return PA_ERR_INVALID_ARG;
    return decode_common(out, query, key_cache, value_cache, nullptr, nullptr, block_tables,
                         context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                         max_blocks_per_seq, num_blocks, scale, dtype, 0, partition_size,
                         workspace, workspace_bytes, device_status, stream);
}

extern "C" pa_status pa_decode_fp8(void *out, const void *query, const void *key_cache,
                                   const void *value_cache, const float *k_scales,
                                   const float *v_scales, const int32_t *block_tables,
                                   const int32_t *context_lens, int num_seqs, int num_q_heads,
                                   int num_kv_heads, int head_dim, int block_size,
                                   int max_blocks_per_seq, int num_blocks, float scale,
                                   int partition_size, void *workspace, size_t workspace_bytes,
                                   int32_t *device_status, void *stream) {
    return decode_common(out, query, key_cache, value_cache, k_scales, v_scales, block_tables,
                         context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                         max_blocks_per_seq, num_blocks, scale, PA_DTYPE_FP8_E4M3, 0,
                         partition_size, workspace, workspace_bytes, device_status, stream);
}

extern "C" size_t pa_decode_sliding_window_workspace_bytes(int num_seqs, int num_q_heads,
                                                           int num_kv_heads, int head_dim,
                                                           int max_blocks_per_seq, int block_size,
                                                           int window, int partition_size,
                                                           pa_dtype dtype) {
    if (window <= 0) return (size_t)-1;
    return decode_workspace(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                            block_size, window, partition_size, dtype);
}

extern "C" pa_status pa_decode_sliding_window(
    void *out, const void *query, const void *key_cache, const void *value_cache,
    const float *k_scales, const float *v_scales, const int32_t *block_tables,
    const int32_t *context_lens, int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
    int block_size, int max_blocks_per_seq, int num_blocks, float scale, pa_dtype dtype, int window,
    int partition_size, void *workspace, size_t workspace_bytes, int32_t *device_status,
    void *stream) {
    if (window <= 0) return PA_ERR_INVALID_ARG;
    return decode_common(out, query, key_cache, value_cache, k_scales, v_scales, block_tables,
                         context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                         max_blocks_per_seq, num_blocks, scale, dtype, window, partition_size,
                         workspace, workspace_bytes, device_status, stream);
}

namespace pa {
namespace {

constexpr int kPrefixStages = 4;

// Chunks of the shared prefix: about three CTAs per SM (each CTA works through
// its chunk block after block, so short chunks finish sooner), at least 4
// blocks per chunk.
void prefix_chunking(int prefix_blocks, int kv_heads, int row_chunks, int *chunk_blocks,
                     int *chunks) {
    const int64_t per_chunk_ctas = (int64_t)kv_heads * row_chunks;
    int want = (int)std::max<int64_t>(1, (3LL * sm_count() + per_chunk_ctas - 1) / per_chunk_ctas);
    int cb = std::max(4, (prefix_blocks + want - 1) / std::max(1, want));
    cb = std::min(cb, std::max(prefix_blocks, 1));
    *chunk_blocks = cb;
    *chunks = prefix_blocks == 0 ? 0 : (prefix_blocks + cb - 1) / cb;
}

struct SharedPlan {
    int suffix_part_blocks, suffix_max_parts, prefix_chunk_blocks, prefix_chunks, max_parts;
};

bool plan_shared(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                 int max_blocks_per_seq, int num_prefix_blocks, int partition_size,
                 SharedPlan *p) {
    if (num_prefix_blocks < 0 || num_prefix_blocks > max_blocks_per_seq) return false;
    const int suffix_blocks = max_blocks_per_seq - num_prefix_blocks;
    int ps = resolve_partition(partition_size, num_seqs, num_kv_heads, suffix_blocks);
    if (ps < 0) return false;
    // The suffix CTAs are short and many, and one holding a long suffix that
    // starts late sets the end of the call.  When the library's choice covers
    // every suffix with one partition, suffixes longer than three quarters of
    // the longest possible one are split in two instead (128-sequence mix:
    // 59.7 -> 58.0 us bf16, 49.1 -> 46.1 us FP8; halves or 1/1.02 measured slower).
    if (partition_size == 0 && ps / kBlockSize >= suffix_blocks && suffix_blocks >= 8)
        ps = kBlockSize * ((3 * suffix_blocks + 3) / 4);
    p->suffix_part_blocks = ps / kBlockSize;
    p->suffix_max_parts = std::max(1, (suffix_blocks + p->suffix_part_blocks - 1) / p->suffix_part_blocks);
    const int group = num_q_heads / num_kv_heads;
    if (prefix_tc_supported(head_dim, num_q_heads, num_kv_heads)) {
        // tensor-core prefix: whole 8-block K/V tiles, about one CTA per SM
        p->prefix_chunk_blocks =
            prefix_tc_chunk_blocks(num_seqs, num_q_heads, num_kv_heads, num_prefix_blocks, sm_count());
        p->prefix_chunks = num_prefix_blocks == 0
                               ? 0
                               : (num_prefix_blocks + p->prefix_chunk_blocks - 1) / p->prefix_chunk_blocks;
    } else {
        const int row_chunks = (num_seqs * group + kPrefixRows - 1) / kPrefixRows;
        prefix_chunking(num_prefix_blocks, num_kv_heads, row_chunks, &p->prefix_chunk_blocks,
                        &p->prefix_chunks);
    }
    p->max_parts = p->prefix_chunks + p->suffix_max_parts;
    return true;
}

}  // namespace
}  // namespace pa

namespace pa {
namespace {

// Widens the E4M3 codes of the shared prefix (the first prefix_blocks entries
// of the first block table, every KV head, K and V) to their bf16 code values
// (exact: every E4M3 value is a bf16 value) in a staging pool
// [prefix_blocks][Hkv][16][D], block j of the prefix at index j.  The
// tensor-core prefix kernel reads it and applies the per-head scales.  CTA
// (prefix block, KV head, K or V): 128 threads, 16 codes each per step.
__global__ void __launch_bounds__(128)
    pa_widen_prefix_kernel(const uint8_t *__restrict__ kc, const uint8_t *__restrict__ vc,
                           const int32_t *__restrict__ table0, int num_kv_heads, int num_blocks,
                           int D, __nv_bfloat16 *__restrict__ sk, __nv_bfloat16 *__restrict__ sv,
                           int32_t *status) {
    grid_dependency_wait();
    grid_dependents_launch();
    const int j = blockIdx.x / num_kv_heads;
    const int kvh = blockIdx.x - j * num_kv_heads;
    int phys = table0[j];
    if ((unsigned)phys >= (unsigned)num_blocks) {
        if (threadIdx.x == 0) report(status, PA_DEV_BAD_BLOCK_ID);
        phys = 0;
    }
    const size_t tile = (size_t)kBlockSize * D;
    const uint4 *src = reinterpret_cast<const uint4 *>((blockIdx.y ? vc : kc) +
                                                       ((size_t)phys * num_kv_heads + kvh) * tile);
    uint4 *dst = reinterpret_cast<uint4 *>((blockIdx.y ? sv : sk) +
                                           ((size_t)j * num_kv_heads + kvh) * tile);
    for (int i = threadIdx.x; i < (int)(tile / 16); i += 128) {
        const uint4 c = src[i];
        const uint32_t words[4] = {c.x, c.y, c.z, c.w};
        uint32_t o[8];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t lo = e4m3x2_to_f16x2(words[k] & 0xffffu);
            const uint32_t hi = e4m3x2_to_f16x2(words[k] >> 16);
            o[2 * k] = pack_bf16x2(f16lo(lo), f16hi(lo));
            o[2 * k + 1] = pack_bf16x2(f16lo(hi), f16hi(hi));
        }
        dst[2 * i] = make_uint4(o[0], o[1], o[2], o[3]);
        dst[2 * i + 1] = make_uint4(o[4], o[5], o[6], o[7]);
    }
}

bool partition_ok(int partition_size) {
    return partition_size == 0 || (partition_size >= kBlockSize && partition_size <= kMaxPartition &&
                                   partition_size % kBlockSize == 0);
}

// FP8 pools take the cascade where the tensor-core prefix kernel takes the
// shape (head_dim 128, groups 1, 2, 4, 8); elsewhere the call is pa_decode_fp8.
bool fp8_cascade(int head_dim, int num_q_heads, int num_kv_heads, int num_prefix_blocks) {
    return num_prefix_blocks > 0 && prefix_tc_supported(head_dim, num_q_heads, num_kv_heads) &&
           num_q_heads / num_kv_heads <= 8;
}

// Workspace of the shared-prefix decode: partial outputs and (max, sum) pairs,
// then (FP8 pools) the staging copies of the prefix's K and V; every part
// 256-byte aligned.
struct SharedLayout {
    size_t ml_offset, staged_k_offset, staged_v_offset, total;
};
SharedLayout shared_layout(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                           int max_parts, int staged_blocks) {
    auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
    const size_t rows = (size_t)num_seqs * num_q_heads * max_parts;
    const size_t staged = (size_t)staged_blocks * num_kv_heads * kBlockSize * head_dim * 2;
    SharedLayout l;
    l.ml_offset = up(rows * head_dim * sizeof(float));
    l.staged_k_offset = l.ml_offset + up(rows * sizeof(float2));
    l.staged_v_offset = l.staged_k_offset + up(staged);
    l.total = staged_blocks > 0 ? l.staged_v_offset + staged : l.ml_offset + rows * sizeof(float2);
    return l;
}

size_t shared_workspace(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                        int max_blocks_per_seq, int num_prefix_blocks, int partition_size,
                        bool fp8) {
    if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
        num_q_heads % num_kv_heads != 0 || !partition_ok(partition_size))
        return (size_t)-1;
    if (fp8 && !fp8_cascade(head_dim, num_q_heads, num_kv_heads, num_prefix_blocks))
        return decode_workspace(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                                kBlockSize, 0, partition_size, PA_DTYPE_FP8_E4M3);
    SharedPlan p;
    if (!plan_shared(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                     num_prefix_blocks, partition_size, &p))
        return (size_t)-1;
    return shared_layout(num_seqs, num_q_heads, num_kv_heads, head_dim, p.max_parts,
                         fp8 ? num_prefix_blocks : 0)
        .total;
}

// The path behind pa_decode_shared_prefix (bf16 pools) and
// pa_decode_shared_prefix_fp8 (E4M3 pools with per-head scales).
pa_status shared_prefix_common(void *out, const void *query, const void *key_cache,
                               const void *value_cache, const float *k_scales,
                               const float *v_scales, const int32_t *block_tables,
                               const int32_t *context_lens, int num_seqs, int num_q_heads,
                               int num_kv_heads, int head_dim, int block_size,
                               int max_blocks_per_seq, int num_blocks, float scale, pa_dtype dtype,
                               int num_prefix_blocks, int partition_size, void *workspace,
                               size_t workspace_bytes, int32_t *device_status, void *stream) {
    const bool fp8 = dtype == PA_DTYPE_FP8_E4M3;
    if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || block_size != kBlockSize ||
        max_blocks_per_seq < 0 || num_blocks <= 0 || num_q_heads % num_kv_heads != 0 ||
        !(scale == scale) || num_prefix_blocks < 0 || num_prefix_blocks > max_blocks_per_seq)
        return PA_ERR_INVALID_ARG;
    if (!partition_ok(partition_size)) return PA_ERR_INVALID_ARG;
    if (num_seqs == 0) return PA_OK;
    if (!out || !query || !key_cache || !value_cache || !block_tables || !context_lens)
        return PA_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(query) || !aligned16(key_cache) || !aligned16(value_cache))
        return PA_ERR_INVALID_ARG;
    const int group = num_q_heads / num_kv_heads;
    if (fp8) {
        if (!k_scales || !v_scales) return PA_ERR_INVALID_ARG;
        if (head_dim != 128 || group > 8) return PA_ERR_UNSUPPORTED;
        if (!fp8_cascade(head_dim, num_q_heads, num_kv_heads, num_prefix_blocks))
            return decode_common(out, query, key_cache, value_cache, k_scales, v_scales,
                                 block_tables, context_lens, num_seqs, num_q_heads, num_kv_heads,
                                 head_dim, block_size, max_blocks_per_seq, num_blocks, scale, dtype,
                                 0, partition_size, workspace, workspace_bytes, device_status,
                                 stream);
    } else {
        if (head_dim != 64 && head_dim != 128) return PA_ERR_UNSUPPORTED;
        if (group > 16) return PA_ERR_UNSUPPORTED;
        if (num_prefix_blocks == 0)
            return decode_common(out, query, key_cache, value_cache, nullptr, nullptr, block_tables,
                                 context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim,
                                 block_size, max_blocks_per_seq, num_blocks, scale, dtype, 0,
                                 partition_size, workspace, workspace_bytes, device_status, stream);
    }
    const int64_t rows = (int64_t)num_blocks * num_kv_heads * kBlockSize;
    if (rows >= ((int64_t)1 << 31)) return PA_ERR_UNSUPPORTED;
    SharedPlan p;
    if (!plan_shared(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                     num_prefix_blocks, partition_size, &p))
        return PA_ERR_INVALID_ARG;
    const SharedLayout lay = shared_layout(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                           p.max_parts, fp8 ? num_prefix_blocks : 0);
    if (workspace == nullptr || workspace_bytes < lay.total || !aligned16(workspace))
        return PA_ERR_WORKSPACE;
    const int row_chunks = (num_seqs * group + kPrefixRows - 1) / kPrefixRows;
    if ((int64_t)num_seqs * num_kv_heads * p.suffix_max_parts >= ((int64_t)1 << 31) ||
        (int64_t)num_kv_heads * row_chunks * p.prefix_chunks >= ((int64_t)1 << 31) ||
        (int64_t)num_prefix_blocks * num_kv_heads >= ((int64_t)1 << 31))
        return PA_ERR_UNSUPPORTED;

    const bool tc_prefix = prefix_tc_supported(head_dim, num_q_heads, num_kv_heads);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    DecodeArgs a;
    a.out = out;
    a.query = query;
    a.block_tables = block_tables;
    a.context_lens = context_lens;
    a.part_o = reinterpret_cast<float *>(ws);
    a.part_ml = reinterpret_cast<float2 *>(ws + lay.ml_offset);
    a.status = device_status;
    a.k_scales = fp8 ? k_scales : nullptr;
    a.v_scales = fp8 ? v_scales : nullptr;
    a.num_seqs = num_seqs;
    a.num_q_heads = num_q_heads;
    a.num_kv_heads = num_kv_heads;
    a.max_blocks = max_blocks_per_seq;
    a.num_blocks = num_blocks;
    a.part_blocks = p.suffix_part_blocks;
    a.max_parts = p.max_parts;
    a.scale_log2 = scale * kLog2e;
    a.token_offset = num_prefix_blocks * kBlockSize;
    a.part_base = p.prefix_chunks;
    a.always_partial = 1;
    a.prefix_blocks = num_prefix_blocks;
    a.prefix_chunk_blocks = p.prefix_chunk_blocks;
    a.prefix_chunks = p.prefix_chunks;
    a.window = 0;
    a.defer_wait = 1;
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    // 0. FP8 pools: the prefix blocks' codes widened to bf16 for the tensor cores
    if (fp8) {
        cudaError_t e = launch_chained(
            pa_widen_prefix_kernel, dim3((unsigned)(num_prefix_blocks * num_kv_heads), 2), dim3(128),
            0, st, static_cast<const uint8_t *>(key_cache), static_cast<const uint8_t *>(value_cache),
            block_tables, num_kv_heads, num_blocks, head_dim,
            reinterpret_cast<__nv_bfloat16 *>(ws + lay.staged_k_offset),
            reinterpret_cast<__nv_bfloat16 *>(ws + lay.staged_v_offset), device_status);
        if (e != cudaSuccess) return cuda_failure(e, "pa_widen_prefix_kernel launch");
        count_launches(1);
    }
    // 1. the shared prefix, once per KV head for all sequences: on the tensor
    //    cores (256 rows per K/V tile) where the shape allows, else 64 query
    //    rows at a time on mma.sync tiles.  It takes part of the SMs (one CTA
    //    each) and lets the suffix kernel launch as soon as all of its CTAs
    //    have started.
    if (tc_prefix) {
        pa_status ps =
            fp8 ? launch_prefix_tc(query, ws + lay.staged_k_offset, ws + lay.staged_v_offset,
                                   block_tables, context_lens, num_seqs, num_q_heads, num_kv_heads,
                                   max_blocks_per_seq, num_prefix_blocks, a.scale_log2,
                                   num_prefix_blocks, p.prefix_chunk_blocks, p.prefix_chunks,
                                   a.part_o, a.part_ml, p.max_parts, true, k_scales, v_scales,
                                   device_status, st)
                : launch_prefix_tc(query, key_cache, value_cache, block_tables, context_lens,
                                   num_seqs, num_q_heads, num_kv_heads, max_blocks_per_seq,
                                   num_blocks, a.scale_log2, num_prefix_blocks,
                                   p.prefix_chunk_blocks, p.prefix_chunks, a.part_o, a.part_ml,
                                   p.max_parts, false, nullptr, nullptr, device_status, st);
        if (ps != PA_OK) return ps;
    } else {
        CUtensorMap kmap, vmap;
        if (!encode_pool_map(&kmap, key_cache, rows, head_dim, 2) ||
            !encode_pool_map(&vmap, value_cache, rows, head_dim, 2))
            return cuda_failure(cudaErrorInvalidValue, "cuTensorMapEncodeTiled");
        const size_t smem = 1024 + (size_t)kPrefixStages * 2 * 16 * head_dim * 2 +
                            2 * kPrefixStages * sizeof(uint64_t) +
                            (size_t)p.prefix_chunk_blocks * sizeof(int32_t) + 16;
        const unsigned grid = (unsigned)((int64_t)num_kv_heads * row_chunks * p.prefix_chunks);
        cudaError_t e;
        if (head_dim == 128) {
            auto kernel = pa_prefix_kernel<128, kPrefixStages>;
            e = allow_smem(kernel, smem);
            if (e == cudaSuccess)
                e = launch_chained(kernel, dim3(grid), dim3((kPrefixWarps + 1) * 32), smem, st,
                                   kmap, vmap, a);
        } else {
            auto kernel = pa_prefix_kernel<64, kPrefixStages>;
            e = allow_smem(kernel, smem);
            if (e == cudaSuccess)
                e = launch_chained(kernel, dim3(grid), dim3((kPrefixWarps + 1) * 32), smem, st,
                                   kmap, vmap, a);
        }
        if (e != cudaSuccess) return cuda_failure(e, "pa_prefix_kernel launch");
        count_launches(1);
    }
    // 2. every context past the prefix, as partials, beside the prefix kernel
    //    (defer_wait: only its last CTA waits for the prefix kernel to finish)
    pa_status s = fp8 ? dispatch_fp8(group, a, key_cache, value_cache, rows, st)
                : head_dim == 64 ? dispatch_bf16<64>(group, a, key_cache, value_cache, rows, st)
                                 : dispatch_bf16<128>(group, a, key_cache, value_cache, rows, st);
    if (s != PA_OK) return s;
    // 3. merge prefix and suffix partials
    return launch_reduce<__nv_bfloat16>(a, head_dim, st);
}

}  // namespace
}  // namespace pa

extern "C" size_t pa_decode_shared_prefix_workspace_bytes(int num_seqs, int num_q_heads,
                                                          int num_kv_heads, int head_dim,
                                                          int max_blocks_per_seq,
                                                          int num_prefix_blocks,
                                                          int partition_size) {
    return shared_workspace(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                            num_prefix_blocks, partition_size, false);
}

extern "C" pa_status pa_decode_shared_prefix(
    void *out, const void *query, const void *key_cache, const void *value_cache,
    const int32_t *block_tables, const int32_t *context_lens, int num_seqs, int num_q_heads,
    int num_kv_heads, int head_dim, int block_size, int max_blocks_per_seq, int num_blocks,
    float scale, pa_dtype dtype, int num_prefix_blocks, int partition_size, void *workspace,
    size_t workspace_bytes, int32_t *device_status, void *stream) {
    if (dtype != PA_DTYPE_BF16) return PA_ERR_UNSUPPORTED;
    return shared_prefix_common(out, query, key_cache, value_cache, nullptr, nullptr, block_tables,
                                context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim,
                                block_size, max_blocks_per_seq, num_blocks, scale, dtype,
                                num_prefix_blocks, partition_size, workspace, workspace_bytes,
                                device_status, stream);
}

extern "C" size_t pa_decode_shared_prefix_fp8_workspace_bytes(int num_seqs, int num_q_heads,
                                                              int num_kv_heads, int head_dim,
                                                              int max_blocks_per_seq,
                                                              int num_prefix_blocks,
                                                              int partition_size) {
    return shared_workspace(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                            num_prefix_blocks, partition_size, true);
}

extern "C" pa_status pa_decode_shared_prefix_fp8(
    void *out, const void *query, const void *key_cache, const void *value_cache,
    const float *k_scales, const float *v_scales, const int32_t *block_tables,
    const int32_t *context_lens, int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
    int block_size, int max_blocks_per_seq, int num_blocks, float scale, int num_prefix_blocks,
    int partition_size, void *workspace, size_t workspace_bytes, int32_t *device_status,
    void *stream) {
    if ((reinterpret_cast<uintptr_t>(k_scales) & 3u) || (reinterpret_cast<uintptr_t>(v_scales) & 3u))
        return PA_ERR_INVALID_ARG;
    return shared_prefix_common(out, query, key_cache, value_cache, k_scales, v_scales,
                                block_tables, context_lens, num_seqs, num_q_heads, num_kv_heads,
                                head_dim, block_size, max_blocks_per_seq, num_blocks, scale,
                                PA_DTYPE_FP8_E4M3, num_prefix_blocks, partition_size, workspace,
                                workspace_bytes, device_status, stream);
}

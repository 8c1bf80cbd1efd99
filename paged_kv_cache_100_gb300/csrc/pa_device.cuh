// Device-side helpers for the sm_103a kernels: mbarriers, TMA tensor loads,
// ldmatrix / mma.sync, bf16 unpacking and the bounded wait.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "pa_internal.h"

namespace pa {

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void report(int32_t *status, int32_t bits) {
    if (status != nullptr) atomicOr(status, bits);
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Waits for the phase with the given parity to complete.  Gives up after
// kWaitLimitNs of wall time and returns false (the caller reports it).
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // one second

__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 63u) == 0 && globaltimer_ns() - t0 > kWaitLimitNs) return false;
    }
}

// Orders this thread's earlier generic-proxy shared-memory accesses before
// later async-proxy (TMA) accesses to the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------------------
// TMA (tiled tensor copy global -> shared, completion on an mbarrier)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tma_load_2d(void *smem_dst, const CUtensorMap *map, int x, int y,
                                            uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// The same load with an L2 eviction-priority hint (a policy from
// l2_policy_evict_first: streamed data that no one reads again leaves L2 first).
__device__ __forceinline__ void tma_load_2d_hint(void *smem_dst, const CUtensorMap *map, int x, int y,
                                                 uint64_t *bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
// ---------------------------------------------------------------------------
// Programmatic dependent launch
// ---------------------------------------------------------------------------
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_dependents_launch() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Tensor-core fragments (legacy warp-level mma; used only for GQA tiles)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

// Transposes an 8x8 b16 matrix held in the warp's fragment layout (thread T
// holds row T/4, columns 2(T%4), 2(T%4)+1).
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

// D = A * B + D, A 16x16 bf16 (row), B 16x8 bf16 (col), D 16x8 fp32.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// D = A * B + D with f16 inputs, fp32 accumulation.
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                              uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// ---------------------------------------------------------------------------
// FP8 E4M3 helpers
// ---------------------------------------------------------------------------
// Two E4M3 codes (low byte = first element) to f16x2; exact (every E4M3 value,
// subnormals included, is an f16 value).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_codes) {
    uint32_t r;
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, lo;\n\t}"
        : "=r"(r)
        : "r"(two_codes));
    return r;
}

// Four E4M3 codes (byte k = element k) to two f16x2 words: elements 0, 1 in
// *lo and 2, 3 in *hi; exact.  Both halves come straight from the 32-bit
// word's 16-bit halves (no shift).
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t four_codes, uint32_t &lo, uint32_t &hi) {
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(four_codes));
}

// acc0 += p * v.lo, acc1 += p * v.hi with an f16 weight p (low half of the
// 32-bit p16), an f16x2 pair v and fp32 accumulators (each product is exact in
// fp32).
__device__ __forceinline__ void fma2_f16_f32(uint32_t p16, uint32_t v, float &acc0, float &acc1) {
    asm("{\n\t.reg .b16 pl, ph, vl, vh;\n\t"
        "mov.b32 {pl, ph}, %2;\n\tmov.b32 {vl, vh}, %3;\n\t"
        "fma.rn.f32.f16 %0, pl, vl, %0;\n\t"
        "fma.rn.f32.f16 %1, pl, vh, %1;\n\t}"
        : "+f"(acc0), "+f"(acc1)
        : "r"(p16), "r"(v));
}

// E4M3 codes of two floats, round to nearest even, saturating at +-448
// (first element in the low byte).
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float first, float second) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(second), "f"(first));
    return r;
}

// c + a.lo * b.lo + a.hi * b.hi with f16x2 a, b and fp32 accumulation
// (each f16 product is exact in fp32).
__device__ __forceinline__ float dot2_f16_f32(uint32_t a, uint32_t b, float c) {
    float d;
    asm("{\n\t.reg .b16 al, ah, bl, bh;\n\t"
        "mov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
        "fma.rn.f32.f16 %0, al, bl, %3;\n\t"
        "fma.rn.f32.f16 %0, ah, bh, %0;\n\t}"
        : "=f"(d)
        : "r"(a), "r"(b), "f"(c));
    return d;
}

__device__ __forceinline__ float f16lo(uint32_t w) {
    return __half2float(__ushort_as_half((unsigned short)(w & 0xffffu)));
}
__device__ __forceinline__ float f16hi(uint32_t w) {
    return __half2float(__ushort_as_half((unsigned short)(w >> 16)));
}

// True when either bfloat16 of the pair lies outside f16's finite range:
// |x| >= 65536 (the largest bf16 below that, 65280, is an f16 value) or
// infinite; NaN is not counted.
__device__ __forceinline__ bool bf16x2_beyond_f16(uint32_t w) {
    const uint32_t lo = w & 0x7fffu, hi = (w >> 16) & 0x7fffu;
    return (lo - 0x4780u <= 0x7f80u - 0x4780u) | (hi - 0x4780u <= 0x7f80u - 0x4780u);
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// 2^x with the single-instruction approximation (ex2.approx.ftz: a relative
// error of about 2^-22; results below 2^-126 flush to +0, and 2^-inf = +0).
// Used for the softmax weights, whose rounding to f16 or bf16 afterwards is far
// coarser.
__device__ __forceinline__ float ex2_fast(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ---------------------------------------------------------------------------
// bf16 helpers (bfloat16 is the upper half of a binary32, so widening is exact)
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// x = head + residual: head is x rounded to bf16, residual is the exact fp32
// remainder rounded to bf16 (relative error of the pair about 2^-18).
__device__ __forceinline__ void split_bf16x2(float x0, float x1, uint32_t &head, uint32_t &rest) {
    head = pack_bf16x2(x0, x1);
    const float r0 = x0 - bf16lo(head);
    const float r1 = x1 - bf16hi(head);
    rest = pack_bf16x2(r0, r1);
}

}  // namespace pa

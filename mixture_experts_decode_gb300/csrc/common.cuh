// common.cuh -- device helpers shared by the libmoedec kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moedec.h"

namespace moedec {

constexpr unsigned FULL_MASK = 0xffffffffu;

struct U256 {
    uint32_t v[8];
};

// 32-byte streaming load of weight bytes read exactly once per call: skip L1
// and mark the L2 lines evict-first, so L2 keeps the small reused tensors
// (activations, intermediates) rather than weight rows.
__device__ __forceinline__ U256 ld_stream_256(const void* p) {
    U256 r;
    asm volatile(
        "ld.global.nc.L1::no_allocate.L2::evict_first.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
        : "=r"(r.v[0]), "=r"(r.v[1]), "=r"(r.v[2]), "=r"(r.v[3]), "=r"(r.v[4]), "=r"(r.v[5]),
          "=r"(r.v[6]), "=r"(r.v[7])
        : "l"(p));
    return r;
}

// 32-byte load through L1 (activations / intermediates reused across warps).
__device__ __forceinline__ U256 ld_cached_256(const void* p) {
    U256 r;
    asm volatile("ld.global.nc.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r.v[0]), "=r"(r.v[1]), "=r"(r.v[2]), "=r"(r.v[3]), "=r"(r.v[4]),
                   "=r"(r.v[5]), "=r"(r.v[6]), "=r"(r.v[7])
                 : "l"(p));
    return r;
}

__device__ __forceinline__ uint8_t ld_stream_u8(const uint8_t* p) {
    uint16_t v;
    asm volatile("ld.global.nc.L1::no_allocate.u8 %0, [%1];" : "=h"(v) : "l"(p));
    return (uint8_t)v;
}

// Two E4M3 codes (low byte = lower K index) -> two floats, exact
// (E4M3 -> F16 is exact; F16 -> F32 is exact).
__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t two) {
    uint32_t h2;
    uint16_t q = (uint16_t)(two & 0xffffu);
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(q));
    __half2 hh;
    memcpy(&hh, &h2, 4);
    return __half22float2(hh);
}

// Four E4M3 codes (one 32-bit word, lowest byte = lowest K index) -> four
// floats, exact.
__device__ __forceinline__ void e4m3x4_to_float(uint32_t w, float2& lo, float2& hi) {
    uint32_t a, b;
    asm("{ .reg .b16 l, h;\n\t mov.b32 {l, h}, %2;\n\t cvt.rn.f16x2.e4m3x2 %0, l;\n\t cvt.rn.f16x2.e4m3x2 %1, h; }"
        : "=r"(a), "=r"(b)
        : "r"(w));
    __half2 ha, hb;
    memcpy(&ha, &a, 4);
    memcpy(&hb, &b, 4);
    lo = __half22float2(ha);
    hi = __half22float2(hb);
}

// One 32-bit word of codes (four bytes, each an E2M1 pair with the lower K
// index in the low nibble) -> four float2 (x = lower K index), exact.
__device__ __forceinline__ void e2m1x8_to_float(uint32_t w, float2 (&f)[4]) {
    uint32_t h[4];
    asm("{ .reg .b8 b0, b1, b2, b3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, b3; }"
        : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
        : "r"(w));
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __half2 hh;
        memcpy(&hh, &h[i], 4);
        f[i] = __half22float2(hh);
    }
}

// E8M0 scale byte -> 2^(s-127) as float (s = 0 gives the subnormal 2^-127;
// s = 255, NaN in the format, is a precondition violation and yields inf).
__device__ __forceinline__ float e8m0_to_float(uint32_t s) {
    // s >= 1 gives bits s << 23 >= 0x00800000, above the subnormal 2^-127 (0x00400000) of s = 0
    return __uint_as_float(max(s << 23, 0x00400000u));
}

// Two BF16 values packed in one 32-bit word -> float2 (low half first).
__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

__device__ __forceinline__ float warp_sum_group(float v, int L) {
    for (int off = L >> 1; off >= 1; off >>= 1) v += __shfl_xor_sync(FULL_MASK, v, off);
    return v;
}

__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

}  // namespace moedec

namespace moedec {

// ---- asynchronous global -> shared copies (per thread, 16 or 4 bytes) ----

__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// 16 bytes, L2 only, evict-first; src_bytes = 0 fills the destination with zeros.
__device__ __forceinline__ void cp_async_16(void* smem, const void* gmem, int src_bytes, uint64_t pol) {
    const uint32_t a = (uint32_t)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2, %3;" ::"r"(a), "l"(gmem),
                 "r"(src_bytes), "l"(pol)
                 : "memory");
}

__device__ __forceinline__ void cp_async_4(void* smem, const void* gmem, int src_bytes) {
    const uint32_t a = (uint32_t)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(a), "l"(gmem), "r"(src_bytes) : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ uint4 ld_cached_128(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// Reduce N values across the 32 lanes of a warp in log2(N) exchange rounds
// that each halve the values a lane holds (a butterfly reduce-scatter), then
// finish with plain butterfly rounds.  Afterwards every lane holds the full
// sum of value idx = (lane >> (5 - log2 N)) & (N - 1).  N is a power of two
// <= 32.
template <int N>
__device__ __forceinline__ float warp_reduce_scatter(float (&v)[N], int lane) {
    int o = 16;
#pragma unroll
    for (int cnt = N; cnt > 1; cnt >>= 1, o >>= 1) {
        const bool upper = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < cnt / 2; ++i) {
            const float send = upper ? v[i] : v[i + cnt / 2];
            const float keep = upper ? v[i + cnt / 2] : v[i];
            v[i] = keep + __shfl_xor_sync(FULL_MASK, send, o);
        }
    }
    float r = v[0];
#pragma unroll
    for (; o >= 1; o >>= 1) r += __shfl_xor_sync(FULL_MASK, r, o);
    return r;
}

}  // namespace moedec

namespace moedec {

// ---- mbarrier + bulk (TMA) copies --------------------------------------

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Wait for the phase with the given parity to complete.  Each try_wait
// suspends the thread (until the phase completes or a ~0.5 ms hint runs
// out) instead of spinning, so waiting warps take no issue slots.  Bounded:
// gives up after ~2^32 SM cycles (about two seconds), returning false.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
    const uint32_t a = smem_addr(bar);
    uint32_t ok = 0;
    const long long t0 = clock64();
    do {
        asm volatile(
            "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3; selp.u32 %0, 1, 0, p; }"
            : "=r"(ok)
            : "r"(a), "r"(parity), "r"(500000u)
            : "memory");
        if (ok) return true;
    } while (clock64() - t0 < (1ll << 32));
    return false;
}

// 1D bulk copy global -> shared, completion counted on `bar`.  dst, src
// 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                         uint64_t pol) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(pol)
        : "memory");
}

__device__ __forceinline__ void bulk_g2s_keep(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_addr(dst)),
                 "l"(src), "r"(bytes), "r"(smem_addr(bar))
                 : "memory");
}

__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

}  // namespace moedec

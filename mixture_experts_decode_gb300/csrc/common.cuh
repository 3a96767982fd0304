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

// E8M0 scale byte -> 2^(s-127) as float (s = 0 gives the subnormal 2^-127;
// s = 255, NaN in the format, is a precondition violation and yields inf).
__device__ __forceinline__ float e8m0_to_float(uint32_t s) {
    return __uint_as_float(s ? (s << 23) : 0x00400000u);
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

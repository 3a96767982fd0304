// requant.cu -- the activation round trip of the conventional expert-centric
// MoE path: BF16 -> MXFP8 -> BF16 ("Warp decode", section "準確度改進": the
// conventional path converts the BF16 activations to MXFP8 and back before
// each grouped GEMM, a rounding floor that warp decode avoids).  The rule is
// OCP MX v1.0's, the format the page names for its weights: per block of 32
// consecutive values along K the shared exponent is
// X = floor(log2(max |v|)) - 8, clamped to [-127, 127]; each element becomes
// the E4M3 value nearest v / 2^X (ties to even, saturating at 448) and comes
// back as that value times 2^X, rounded to BF16 (exact unless below BF16's
// subnormal range).
//
// Memory-bound: two threads per block with one 32-byte load and store each
// (four with 16 bytes when a buffer is only 16-byte aligned), the block
// maximum by shuffles, CTAs in address order (as the copy kernel).  The
// E4M3 rounding is the hardware conversion (cvt.rn.satfinite.e4m3x2.f32:
// nearest even, saturating to the largest finite value), and v / 2^X and
// e4m3 * 2^X are exact in FP32, so every output is bit-identical to the rule
// applied in exact arithmetic.  The loads are coherent (no .nc, no restrict):
// out may be in itself.
#include <algorithm>
#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "internal.h"

namespace moedec {

// Two BF16 (low half first) through E4M3 at the block's exponent and back.
__device__ __forceinline__ uint32_t mx_round_pair(uint32_t w, float down, float up) {
    const float lo = __uint_as_float(w << 16) * down;          // exact: a power-of-two scaling
    const float hi = __uint_as_float(w & 0xffff0000u) * down;
    uint16_t e2;  // upper byte <- hi, lower byte <- lo
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(e2) : "f"(hi), "f"(lo));
    uint32_t f2;  // upper half <- upper byte, lower half <- lower byte
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(f2) : "h"(e2));
    __half2 h2;
    memcpy(&h2, &f2, 4);
    const float2 r = __half22float2(h2);                       // exact: E4M3 values are F16 values
    const __nv_bfloat162 b = __floats2bfloat162_rn(r.x * up, r.y * up);  // .x is the low half
    uint32_t out;
    memcpy(&out, &b, 4);
    return out;
}

// A thread takes V 32-bit words (2V values): V = 8 (32-byte accesses, two
// threads per 32-value block) when both buffers are 32-byte aligned, else
// V = 4 (16-byte accesses, four threads per block).  nunits = rows * K / (2V);
// a block is 16 / V consecutive units and never straddles a warp
// (K % 32 == 0).  32 bytes per thread keep twice the bytes in flight per SM.
template <int V>
__global__ void __launch_bounds__(256) mx_requant_kernel(const uint32_t* in, uint32_t* out, int64_t nunits) {
    constexpr int TPB = 16 / V;  // threads per block
    const int lane = threadIdx.x & 31;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    // warp-uniform loop: every lane reaches the shuffles on every pass
    for (int64_t base = (int64_t)blockIdx.x * blockDim.x + (threadIdx.x & ~31); base < nunits; base += stride) {
        const int64_t g = base + lane;
        const bool ok = g < nunits;
        uint32_t w[V];
#pragma unroll
        for (int i = 0; i < V; ++i) w[i] = 0u;
        if (ok) {
            if constexpr (V == 8) {
                asm volatile("ld.global.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                             : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]),
                               "=r"(w[6]), "=r"(w[7])
                             : "l"(in + g * 8));
            } else {
                asm volatile("ld.global.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                             : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                             : "l"(in + g * 4));
            }
        }
        // |v| as FP32 bit patterns (a BF16 is the upper half of an FP32)
        uint32_t m = 0;
#pragma unroll
        for (int i = 0; i < V; ++i) m = max(m, max((w[i] << 16) & 0x7fff0000u, w[i] & 0x7fff0000u));
#pragma unroll
        for (int o = 1; o < TPB; o <<= 1) m = max(m, __shfl_xor_sync(FULL_MASK, m, o));
        // X = floor(log2 amax) - 8 in [-127, 127]; a block of zeros keeps any X
        int X = -127;
        if (m) {
            const int ef = (int)(m >> 23);
            const int fl = ef ? ef - 127 : (31 - __clz((int)m)) - 149;  // subnormal amax
            X = min(max(fl - 8, -127), 127);
        }
        const float down = ldexpf(1.0f, -X), up = ldexpf(1.0f, X);
#pragma unroll
        for (int i = 0; i < V; ++i) w[i] = mx_round_pair(w[i], down, up);
        if (ok) {
            if constexpr (V == 8) {
                asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(out + g * 8), "r"(w[0]),
                             "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                             : "memory");
            } else {
                asm volatile("st.global.v4.b32 [%0], {%1,%2,%3,%4};" ::"l"(out + g * 4), "r"(w[0]), "r"(w[1]),
                             "r"(w[2]), "r"(w[3])
                             : "memory");
            }
        }
    }
}

cudaError_t launch_mx_requant(const void* in, void* out, int64_t rows, int K, cudaStream_t st) {
    const bool wide = (reinterpret_cast<uintptr_t>(in) % 32 == 0) && (reinterpret_cast<uintptr_t>(out) % 32 == 0);
    const int64_t nunits = rows * (int64_t)K / (wide ? 16 : 8);
    if (nunits == 0) return cudaSuccess;
    const int64_t grid = std::min<int64_t>((nunits + 255) / 256, (int64_t)INT32_MAX);
    const uint32_t* src = static_cast<const uint32_t*>(in);
    uint32_t* dst = static_cast<uint32_t*>(out);
    if (wide)
        mx_requant_kernel<8><<<(unsigned)grid, 256, 0, st>>>(src, dst, nunits);
    else
        mx_requant_kernel<4><<<(unsigned)grid, 256, 0, st>>>(src, dst, nunits);
    return cudaGetLastError();
}

}  // namespace moedec

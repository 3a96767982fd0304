// decode_fp4.cu -- the decode layer with MXFP4 weights: E2M1 codes, two per
// byte with the lower K index in the low nibble, one E8M0 scale per 32
// consecutive elements along K (OCP MX v1.0; the GC-MoE page names FP8/FP4
// MoE operators).  Activations BF16, products and sums FP32, h BF16, y BF16,
// exactly as for the MXFP8 weights.
//
// This file holds the fallback FP4 kernels, organised as the "Warp decode"
// page describes its two kernels (section "兩個 kernel 的運作方式"): one warp
// per output value.  Shapes that the grouped kernels take (gate_up.cu,
// down.cu: d % 512 == 0 and I % 16 == 0 for gate/up with B >= 2, I % 256 ==
// 0 for down, 16-byte aligned weights) run there instead, streaming each
// distinct expert's rows once per call.
//   gate/up: a warp owns one (token, slot, neuron) and streams the gate and
//     up rows of the slot's expert once; lanes take 16-byte chunks (32 codes
//     = one scale block) and the matching 32 values of x, loaded for each
//     projection (the second load hits L1); a __shfl_xor_sync butterfly sums
//     the lanes; lane 0 applies SiLU(g) * u and stores BF16.
//   down: a warp owns one (token, output), walks the token's experts and adds
//     each chunk's partial dot, scaled by the block scale times the routing
//     weight, into one FP32 accumulator per lane; one butterfly at the end.
// Tokens that share an expert each stream its rows (there is no grouping by
// expert), so at B > 1 this path moves more bytes than the MXFP8 kernels.
// An expert id outside [0, E) sets MOE_DEVERR_EXPERT_ID; its slot
// contributes nothing (h is written as zero, down skips it).
#include <algorithm>
#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "internal.h"

namespace moedec {

constexpr int F4_WARPS = 8;  // output values (warps) per CTA

__device__ __forceinline__ uint4 ld_nc_128(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

// Partial dot of one 32-element chunk: 16 code bytes against 32 BF16 values.
__device__ __forceinline__ float2 chunk_dot(const uint4& w4, const uint16_t* v) {
    float2 p = make_float2(0.f, 0.f);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const uint4 xv = ld_nc_128(v + q * 8);  // K pairs 4q .. 4q+3 of the chunk
        float2 f[4];
        e2m1x8_to_float((&w4.x)[q], f);
#pragma unroll
        for (int i = 0; i < 4; ++i) p = __ffma2_rn(bf16x2_to_float2((&xv.x)[i]), f[i], p);
    }
    return p;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(FULL_MASK, v, off);
    return v;
}

struct F4Args {
    DecodeShape s;
    const uint16_t* x;    // gate/up: BF16 [B][d]
    const uint16_t* h;    // down: BF16 [B][k+S][I]
    const int32_t* ids;   // [B][k]
    const float* w;       // down: [B][k]
    MXView wg, wu, wd;    // routed experts
    MXView shg, shu, shd; // shared expert (S = 1)
    uint16_t* out;        // gate/up: h; down: y
    int* err;
};

__global__ void __launch_bounds__(F4_WARPS * 32) gate_up_fp4_kernel(F4Args a) {
    const DecodeShape s = a.s;
    const int lane = threadIdx.x & 31;
    const int KS = s.k + s.S;
    const int64_t item = (int64_t)blockIdx.x * F4_WARPS + (threadIdx.x >> 5);
    if (item >= (int64_t)s.B * KS * s.I) return;  // the whole warp
    const int n = (int)(item % s.I);
    const int64_t slot = item / s.I;  // b * KS + j
    const int b = (int)(slot / KS), j = (int)(slot % KS);
    MXView vg = a.shg, vu = a.shu;
    int64_t e = 0;
    if (j < s.k) {
        e = a.ids[(int64_t)b * s.k + j];
        if (e < 0 || e >= s.E) {
            if (lane == 0) {
                atomicOr(a.err, MOE_DEVERR_EXPERT_ID);
                a.out[slot * s.I + n] = 0;
            }
            return;
        }
        vg = a.wg;
        vu = a.wu;
    }
    const int64_t row = e * s.I + n;
    const uint8_t* wgr = vg.w + row * (s.d / 2);
    const uint8_t* wur = vu.w + row * (s.d / 2);
    const uint8_t* sgr = vg.s + row * (s.d / 32);
    const uint8_t* sur = vu.s + row * (s.d / 32);
    const uint16_t* xr = a.x + (int64_t)b * s.d;
    float2 g2 = make_float2(0.f, 0.f), u2 = make_float2(0.f, 0.f);
    for (int c = lane; c < s.d / 32; c += 32) {
        const uint4 wg4 = ld_nc_128(wgr + c * 16), wu4 = ld_nc_128(wur + c * 16);
        const float gs = e8m0_to_float(ld_stream_u8(sgr + c)), us = e8m0_to_float(ld_stream_u8(sur + c));
        const float2 pg = chunk_dot(wg4, xr + c * 32), pu = chunk_dot(wu4, xr + c * 32);
        g2 = __ffma2_rn(pg, make_float2(gs, gs), g2);
        u2 = __ffma2_rn(pu, make_float2(us, us), u2);
    }
    const float g = warp_sum(g2.x + g2.y), u = warp_sum(u2.x + u2.y);
    if (lane == 0) {
        const float hv = g / (1.0f + expf(-g)) * u;
        a.out[slot * s.I + n] = __bfloat16_as_ushort(__float2bfloat16_rn(hv));
    }
}

__global__ void __launch_bounds__(F4_WARPS * 32) down_fp4_kernel(F4Args a) {
    const DecodeShape s = a.s;
    const int lane = threadIdx.x & 31;
    const int KS = s.k + s.S;
    const int64_t item = (int64_t)blockIdx.x * F4_WARPS + (threadIdx.x >> 5);
    if (item >= (int64_t)s.B * s.d) return;  // the whole warp
    const int o = (int)(item % s.d);
    const int b = (int)(item / s.d);
    float2 acc = make_float2(0.f, 0.f);  // one FP32 accumulator over all experts
    for (int j = 0; j < KS; ++j) {
        MXView vd = a.shd;
        int64_t e = 0;
        float wt = 1.0f;  // the shared expert's weight
        if (j < s.k) {
            e = a.ids[(int64_t)b * s.k + j];
            if (e < 0 || e >= s.E) {
                if (lane == 0 && o == 0) atomicOr(a.err, MOE_DEVERR_EXPERT_ID);
                continue;
            }
            vd = a.wd;
            wt = a.w[(int64_t)b * s.k + j];
        }
        const int64_t row = e * s.d + o;
        const uint8_t* wdr = vd.w + row * (s.I / 2);
        const uint8_t* sdr = vd.s + row * (s.I / 32);
        const uint16_t* hr = a.h + ((int64_t)b * KS + j) * s.I;
        // the block scale multiplies each chunk's partial sum (exact, a power
        // of two, while the product stays in FP32's normal range); the
        // routing weight multiplies the expert's whole dot once, as the
        // grouped kernels do
        float2 ex = make_float2(0.f, 0.f);
        for (int c = lane; c < s.I / 32; c += 32) {
            const uint4 w4 = ld_nc_128(wdr + c * 16);
            const float sc = e8m0_to_float(ld_stream_u8(sdr + c));
            ex = __ffma2_rn(chunk_dot(w4, hr + c * 32), make_float2(sc, sc), ex);
        }
        acc = __ffma2_rn(ex, make_float2(wt, wt), acc);
    }
    const float v = warp_sum(acc.x + acc.y);
    if (lane == 0) a.out[(int64_t)b * s.d + o] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
}

static cudaError_t launch_fp4(void (*kernel)(F4Args), const F4Args& a, int64_t items, cudaStream_t st) {
    if (items == 0) return cudaSuccess;
    const int64_t grid = (items + F4_WARPS - 1) / F4_WARPS;
    if (grid > INT32_MAX) return cudaErrorInvalidValue;
    kernel<<<(unsigned)grid, F4_WARPS * 32, 0, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_gate_up_fp4(const DecodeShape& s, const void* x, const int32_t* ids, MXView wg, MXView wu,
                               MXView shg, MXView shu, void* h, cudaStream_t st) {
    cudaError_t err = cudaSuccess;
    // the grouped kernel (each distinct expert's rows streamed once) when it applies
    if (launch_gate_up_grouped_fp4(s, x, ids, wg, wu, shg, shu, h, st, &err)) return err;
    DeviceInfo di;
    err = device_info(&di);
    if (err != cudaSuccess) return err;
    F4Args a{};
    a.s = s;
    a.x = static_cast<const uint16_t*>(x);
    a.ids = ids;
    a.wg = wg;
    a.wu = wu;
    a.shg = shg;
    a.shu = shu;
    a.out = static_cast<uint16_t*>(h);
    a.err = di.err_word;
    return launch_fp4(gate_up_fp4_kernel, a, (int64_t)s.B * (s.k + s.S) * s.I, st);
}

cudaError_t launch_down_fp4(const DecodeShape& s, const void* h, const int32_t* ids, const float* w, MXView wd,
                            MXView shd, void* y, cudaStream_t st) {
    cudaError_t err = cudaSuccess;
    if (launch_down_grouped_fp4(s, h, ids, w, wd, shd, y, st, &err)) return err;
    DeviceInfo di;
    err = device_info(&di);
    if (err != cudaSuccess) return err;
    F4Args a{};
    a.s = s;
    a.h = static_cast<const uint16_t*>(h);
    a.ids = ids;
    a.w = w;
    a.wd = wd;
    a.shd = shd;
    a.out = static_cast<uint16_t*>(y);
    a.err = di.err_word;
    return launch_fp4(down_fp4_kernel, a, (int64_t)s.B * s.d, st);
}

}  // namespace moedec

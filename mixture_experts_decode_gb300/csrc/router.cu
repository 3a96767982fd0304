// router.cu -- the routing step in front of the decode layer: per token, the
// k largest of E router logits (ties: the lower expert index first), in
// descending order, with weights either renormalised softmax probabilities
// (FasterTransformer's fused topk_gating_softmax, named on the MoE Align &
// Sort page, section "MoE Align & Sort CUDA算法在其他开源平台的实现") or
// sigmoid scores normalised over the k and multiplied by a scale (the
// DeepSeek-V3-style gate).  One warp per token: the row's logits sit in
// registers (E / 32 per lane), k passes of a warp arg-max pick the experts,
// and the weights come from the k chosen logits alone (the softmax
// denominator over all E cancels in the renormalisation).
#include "common.cuh"
#include "internal.h"

namespace moedec {

constexpr int RTR_WARPS = 8;  // tokens per CTA

template <int NV>  // logits per lane (E <= 32 * NV)
__global__ void __launch_bounds__(RTR_WARPS * 32)
    router_topk_kernel(const float* __restrict__ logits, int B, int E, int k, int score, float scale,
                       int32_t* __restrict__ ids, float* __restrict__ w, int* err) {
    const int lane = threadIdx.x & 31;
    const int b = blockIdx.x * RTR_WARPS + (threadIdx.x >> 5);
    if (b >= B) return;
    const float* row = logits + (size_t)b * E;
    float v[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        const int e = i * 32 + lane;
        v[i] = e < E ? row[e] : -INFINITY;
    }
    float sel_v = 0.f;
    int sel_i = -1;
    bool short_row = false;
    for (int j = 0; j < k; ++j) {
        // this lane's largest remaining logit (lowest index first on ties) ...
        float bv = -INFINITY;
        int bi = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < NV; ++i)
            if (v[i] > bv) {
                bv = v[i];
                bi = i * 32 + lane;
            }
        // ... then the warp's
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float ov = __shfl_xor_sync(FULL_MASK, bv, off);
            const int oi = __shfl_xor_sync(FULL_MASK, bi, off);
            if (ov > bv || (ov == bv && oi < bi)) {
                bv = ov;
                bi = oi;
            }
        }
        if (bi == 0x7fffffff) {  // fewer than k logits above -inf (NaN or -inf rows)
            short_row = true;
            break;
        }
        if (lane == j) {
            sel_v = bv;
            sel_i = bi;
        }
        if ((bi & 31) == lane) {
#pragma unroll
            for (int i = 0; i < NV; ++i)
                if (i == (bi >> 5)) v[i] = -INFINITY;
        }
    }
    const bool mine = lane < k && sel_i >= 0;
    float t;
    if (score == MOE_ROUTER_SOFTMAX) {
        const float m = __shfl_sync(FULL_MASK, sel_v, 0);  // the first pick is the largest
        t = mine ? expf(sel_v - m) : 0.f;
    } else {
        t = mine ? 1.0f / (1.0f + expf(-sel_v)) : 0.f;
    }
    float tot = t;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) tot += __shfl_xor_sync(FULL_MASK, tot, off);
    if (lane < k) {
        ids[(size_t)b * k + lane] = mine ? sel_i : -1;
        w[(size_t)b * k + lane] = mine ? scale * t / tot : 0.f;
    }
    if (short_row && lane == 0) atomicOr(err, MOE_DEVERR_LOGIT);
}

template <int NV>
static cudaError_t launch_router_nv(const float* logits, int B, int E, int k, int score, float scale, int32_t* ids,
                                    float* w, int* err, cudaStream_t st) {
    const int grid = (B + RTR_WARPS - 1) / RTR_WARPS;
    router_topk_kernel<NV><<<grid, RTR_WARPS * 32, 0, st>>>(logits, B, E, k, score, scale, ids, w, err);
    return cudaGetLastError();
}

cudaError_t launch_router(const float* logits, int B, int E, int k, int score, float scale, int32_t* ids, float* w,
                          cudaStream_t st) {
    DeviceInfo di;
    cudaError_t e = device_info(&di);
    if (e != cudaSuccess) return e;
    if (E <= 128) return launch_router_nv<4>(logits, B, E, k, score, scale, ids, w, di.err_word, st);
    if (E <= 256) return launch_router_nv<8>(logits, B, E, k, score, scale, ids, w, di.err_word, st);
    if (E <= 512) return launch_router_nv<16>(logits, B, E, k, score, scale, ids, w, di.err_word, st);
    return launch_router_nv<32>(logits, B, E, k, score, scale, ids, w, di.err_word, st);
}

}  // namespace moedec

// decode.cu -- the MoE expert-FFN decode layer on sm_103a.
//
// Two kernels, as in "Warp decode" (section on how the two kernels work):
//   gate_up : one FP32 dot pair (gate, up) per (token, routed expert,
//             intermediate neuron); lanes split K in 32-element MXFP8 blocks,
//             dequantise in registers, reduce with a shfl.xor butterfly,
//             apply SiLU(gate) * up and store one BF16 value.
//   down    : one FP32 accumulator per output value (token, hidden dim) that
//             takes every routed expert's contribution already multiplied by
//             its routing weight -- no per-expert output buffer, no combine.
//
// What differs from the page's mapping (one warp per output scalar, each
// warp reading its own weight row): here a warp owns a weight ROW of a
// DISTINCT expert and serves every token routed to that expert, so each
// weight byte leaves HBM once per call even when several tokens share an
// expert.  The token -> distinct-expert map is built in shared memory by
// every CTA from topk_ids (no extra launch, no global buffer).
#include <algorithm>
#include <mutex>
#include <map>

#include "common.cuh"
#include "internal.h"

namespace moedec {

constexpr int DEC_THREADS = 256;
constexpr int DEC_WARPS = DEC_THREADS / 32;
constexpr int TC = 4;  // tokens served per pass over a weight row

struct GateUpArgs {
    DecodeShape s;
    const uint16_t* x;
    const int32_t* ids;
    MXView wg, wu, shg, shu;
    uint16_t* h;
    int* err;
};

struct DownArgs {
    DecodeShape s;
    const uint16_t* h;
    const int32_t* ids;
    const float* w;
    MXView wd, shd;
    uint16_t* y;
    int* err;
    int es;  // expert splits per CTA (1, 2, 4 or 8)
};

// ------------------------------------------------------ routing map ------
// Per CTA, in shared memory: the distinct experts of this call in increasing
// id order (the shared expert, when present, last with id E), and for each
// the slots routed to it in increasing flat-slot order.

struct RouteMap {
    int* hdr;   // [0] distinct experts incl. shared, [1] routed distinct, [2] routed slots
    int* uexp;  // [max_unique] expert id (E = the shared expert)
    int* uoff;  // [max_unique + 1] slot range of each distinct expert
    int* hrow;  // [slots] row of h: b * (k + S) + j
    float* wt;  // [slots] routing weight (down only)
    int* cnt;   // [E] per-expert counts, then fill cursors
    int* sid;   // [B * k] expert id of each slot (-1 if out of range)
    int* wtot;  // [DEC_WARPS] scan scratch
};

__host__ __device__ inline int max_unique(const DecodeShape& s) {
    const int r = s.B * s.k;
    return (s.E < r ? s.E : r) + s.S;
}
__host__ __device__ inline int n_slots(const DecodeShape& s) { return s.B * s.k + s.S * s.B; }

__host__ __device__ inline size_t map_ints(const DecodeShape& s, bool with_w) {
    const size_t mu = (size_t)max_unique(s);
    size_t ints = 4 + mu + (mu + 1) + n_slots(s) + (with_w ? n_slots(s) : 0) + s.E +
                  (size_t)s.B * s.k + DEC_WARPS;
    return (ints + 3) / 4 * 4;  // keep what follows 16-byte aligned
}

__device__ RouteMap carve_map(int* p, const DecodeShape& s, bool with_w) {
    RouteMap m;
    const int mu = max_unique(s);
    m.hdr = p;
    p += 4;
    m.uexp = p;
    p += mu;
    m.uoff = p;
    p += mu + 1;
    m.hrow = p;
    p += n_slots(s);
    if (with_w) {
        m.wt = reinterpret_cast<float*>(p);
        p += n_slots(s);
    } else {
        m.wt = nullptr;
    }
    m.cnt = p;
    p += s.E;
    m.sid = p;
    p += s.B * s.k;
    m.wtot = p;
    return m;
}

__device__ void build_route_map(const RouteMap& m, const int32_t* __restrict__ ids,
                                const float* __restrict__ w, const DecodeShape& s, int* err) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n = s.B * s.k;
    for (int e = tid; e < s.E; e += DEC_THREADS) m.cnt[e] = 0;
    __syncthreads();
    int bad = 0;
    for (int f = tid; f < n; f += DEC_THREADS) {
        int e = ids[f];
        if ((unsigned)e < (unsigned)s.E) {
            atomicAdd(&m.cnt[e], 1);
        } else {
            e = -1;
            bad = 1;
        }
        m.sid[f] = e;
    }
    if (bad) atomicOr(err, MOE_DEVERR_EXPERT_ID);
    __syncthreads();

    // Exclusive scan over experts of (count << 16 | present): gives each
    // present expert its distinct index (low half) and slot offset (high).
    const int per = (s.E + DEC_THREADS - 1) / DEC_THREADS;
    const int e0 = min(tid * per, s.E), e1 = min(e0 + per, s.E);
    int local = 0;
    for (int e = e0; e < e1; ++e) {
        const int c = m.cnt[e];
        local += (c << 16) | (c > 0 ? 1 : 0);
    }
    int incl = local;
    for (int off = 1; off < 32; off <<= 1) {
        const int v = __shfl_up_sync(FULL_MASK, incl, off);
        if (lane >= off) incl += v;
    }
    if (lane == 31) m.wtot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int v = lane < DEC_WARPS ? m.wtot[lane] : 0;
        int sc = v;
        for (int off = 1; off < 32; off <<= 1) {
            const int t = __shfl_up_sync(FULL_MASK, sc, off);
            if (lane >= off) sc += t;
        }
        if (lane < DEC_WARPS) m.wtot[lane] = sc - v;
        if (lane == DEC_WARPS - 1) {
            m.hdr[1] = sc & 0xffff;
            m.hdr[2] = sc >> 16;
        }
    }
    __syncthreads();
    int run = m.wtot[warp] + incl - local;
    for (int e = e0; e < e1; ++e) {
        const int c = m.cnt[e];
        if (c > 0) {
            const int uid = run & 0xffff, off = run >> 16;
            m.uexp[uid] = e;
            m.uoff[uid] = off;
            m.cnt[e] = off;
            run += (c << 16) | 1;
        }
    }
    __syncthreads();

    // Stable placement of slots into their expert's range (one warp; the
    // order inside an expert is increasing flat slot index).
    const int nu = m.hdr[1], tot = m.hdr[2];
    const int KS = s.k + s.S;
    if (warp == 0) {
        for (int f0 = 0; f0 < n; f0 += 32) {
            const int f = f0 + lane;
            const int e = f < n ? m.sid[f] : -1;
            const unsigned grp = __match_any_sync(FULL_MASK, e);
            const int base = e >= 0 ? m.cnt[e] : 0;
            __syncwarp();
            if (e >= 0) {
                const int pos = base + __popc(grp & lanemask_lt());
                const int b = f / s.k, j = f - b * s.k;
                m.hrow[pos] = b * KS + j;
                if (m.wt) m.wt[pos] = w[f];
                if ((grp & lanemask_lt()) == 0) m.cnt[e] = base + __popc(grp);
            }
            __syncwarp();
        }
    }
    if (tid == 0) {
        m.uoff[nu] = tot;
        m.hdr[0] = nu + s.S;
        if (s.S) {
            m.uexp[nu] = s.E;
            m.uoff[nu + 1] = tot + s.B;
        }
    }
    if (s.S) {
        for (int b = tid; b < s.B; b += DEC_THREADS) {
            m.hrow[tot + b] = b * KS + s.k;
            if (m.wt) m.wt[tot + b] = 1.0f;
        }
    }
    __syncthreads();
}

template <int L>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
    for (int off = L >> 1; off >= 1; off >>= 1) v += __shfl_xor_sync(FULL_MASK, v, off);
    return v;
}

// ------------------------------------------------------------ gate/up ----

template <int L, int NT>
__device__ __forceinline__ void gate_up_rows(const uint8_t* __restrict__ wg_row,
                                             const uint8_t* __restrict__ sg_row,
                                             const uint8_t* __restrict__ wu_row,
                                             const uint8_t* __restrict__ su_row,
                                             const uint16_t* __restrict__ x, int d,
                                             const int* __restrict__ hrow_s, int KS, int cpl,
                                             int li, bool row_ok, int n, int I,
                                             uint16_t* __restrict__ h) {
    const char* xr[NT];
    int hr[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        hr[t] = hrow_s[t];
        xr[t] = reinterpret_cast<const char*>(x + (size_t)(hr[t] / KS) * d);
    }
    float2 ag[NT], au[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) ag[t] = au[t] = make_float2(0.f, 0.f);

#pragma unroll 2
    for (int i = 0; i < cpl; ++i) {
        const int blk = li + i * L;
        const U256 wgv = ld_stream_256(wg_row + (size_t)blk * 32);
        const U256 wuv = ld_stream_256(wu_row + (size_t)blk * 32);
        const float gs = e8m0_to_float(ld_stream_u8(sg_row + blk));
        const float us = e8m0_to_float(ld_stream_u8(su_row + blk));
        const float2 gs2 = make_float2(gs, gs), us2 = make_float2(us, us);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            U256 xv[NT];
#pragma unroll
            for (int t = 0; t < NT; ++t) xv[t] = ld_cached_256(xr[t] + (size_t)blk * 64 + half * 32);
#pragma unroll
            for (int p = 0; p < 8; ++p) {
                const int pp = half * 8 + p;
                const float2 gq = __fmul2_rn(e4m3x2_to_float2(wgv.v[pp >> 1] >> ((pp & 1) * 16)), gs2);
                const float2 uq = __fmul2_rn(e4m3x2_to_float2(wuv.v[pp >> 1] >> ((pp & 1) * 16)), us2);
#pragma unroll
                for (int t = 0; t < NT; ++t) {
                    const float2 xf = bf16x2_to_float2(xv[t].v[p]);
                    ag[t] = __ffma2_rn(xf, gq, ag[t]);
                    au[t] = __ffma2_rn(xf, uq, au[t]);
                }
            }
        }
    }
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        const float g = group_sum<L>(ag[t].x + ag[t].y);
        const float u = group_sum<L>(au[t].x + au[t].y);
        if (row_ok && li == (t % L)) {
            const float hv = g / (1.0f + expf(-g)) * u;
            h[(size_t)hr[t] * I + n] = __bfloat16_as_ushort(__float2bfloat16_rn(hv));
        }
    }
}

template <int L>
__global__ void __launch_bounds__(DEC_THREADS) gate_up_kernel(GateUpArgs a) {
    extern __shared__ __align__(16) int smem_i[];
    const DecodeShape s = a.s;
    const RouteMap m = carve_map(smem_i, s, false);
    build_route_map(m, a.ids, nullptr, s, a.err);
    // the down pass may start its own (independent) prologue now
    asm volatile("griddepcontrol.launch_dependents;");

    constexpr int G = 32 / L;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int grp = lane / L, li = lane % L;
    const int nu = m.hdr[0];
    const int tiles = (s.I + G - 1) / G;
    const int items = nu * tiles;
    const int cpl = s.d / 32 / L;
    const int KS = s.k + s.S;
    const size_t rowsK = (size_t)s.I * s.d;

    for (int item = blockIdx.x * DEC_WARPS + warp; item < items; item += gridDim.x * DEC_WARPS) {
        const int u = item / tiles;
        const int n = (item - u * tiles) * G + grp;
        const bool row_ok = n < s.I;
        const int nr = row_ok ? n : s.I - 1;
        const int e = m.uexp[u];
        const bool sh = e >= s.E;
        const size_t eo = sh ? 0 : (size_t)e;
        const MXView vg = sh ? a.shg : a.wg, vu = sh ? a.shu : a.wu;
        const uint8_t* wg_row = vg.w + eo * rowsK + (size_t)nr * s.d;
        const uint8_t* wu_row = vu.w + eo * rowsK + (size_t)nr * s.d;
        const uint8_t* sg_row = vg.s + (eo * rowsK + (size_t)nr * s.d) / 32;
        const uint8_t* su_row = vu.s + (eo * rowsK + (size_t)nr * s.d) / 32;
        const int s0 = m.uoff[u], s1 = m.uoff[u + 1];
        for (int t0 = s0; t0 < s1; t0 += TC) {
            const int nt = min(TC, s1 - t0);
            const int* hs = m.hrow + t0;
            switch (nt) {
                case 1: gate_up_rows<L, 1>(wg_row, sg_row, wu_row, su_row, a.x, s.d, hs, KS, cpl, li, row_ok, n, s.I, a.h); break;
                case 2: gate_up_rows<L, 2>(wg_row, sg_row, wu_row, su_row, a.x, s.d, hs, KS, cpl, li, row_ok, n, s.I, a.h); break;
                case 3: gate_up_rows<L, 3>(wg_row, sg_row, wu_row, su_row, a.x, s.d, hs, KS, cpl, li, row_ok, n, s.I, a.h); break;
                default: gate_up_rows<L, 4>(wg_row, sg_row, wu_row, su_row, a.x, s.d, hs, KS, cpl, li, row_ok, n, s.I, a.h); break;
            }
        }
    }
}

// --------------------------------------------------------------- down ----

template <int L, int NT>
__device__ __forceinline__ void down_rows(const uint8_t* __restrict__ wd_row,
                                          const uint8_t* __restrict__ sd_row,
                                          const uint16_t* __restrict__ h,
                                          const int* __restrict__ hrow_s, int I, int cpl, int li,
                                          float* out) {
    const char* hp[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) hp[t] = reinterpret_cast<const char*>(h + (size_t)hrow_s[t] * I);
    float2 acc[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) acc[t] = make_float2(0.f, 0.f);
#pragma unroll 2
    for (int i = 0; i < cpl; ++i) {
        const int blk = li + i * L;
        const U256 wv = ld_stream_256(wd_row + (size_t)blk * 32);
        const float sc = e8m0_to_float(ld_stream_u8(sd_row + blk));
        const float2 sc2 = make_float2(sc, sc);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            U256 hv[NT];
#pragma unroll
            for (int t = 0; t < NT; ++t) hv[t] = ld_cached_256(hp[t] + (size_t)blk * 64 + half * 32);
#pragma unroll
            for (int p = 0; p < 8; ++p) {
                const int pp = half * 8 + p;
                const float2 wq = __fmul2_rn(e4m3x2_to_float2(wv.v[pp >> 1] >> ((pp & 1) * 16)), sc2);
#pragma unroll
                for (int t = 0; t < NT; ++t) acc[t] = __ffma2_rn(bf16x2_to_float2(hv[t].v[p]), wq, acc[t]);
            }
        }
    }
#pragma unroll
    for (int t = 0; t < NT; ++t) out[t] = group_sum<L>(acc[t].x + acc[t].y);
}

template <int L>
__global__ void __launch_bounds__(DEC_THREADS) down_kernel(DownArgs a) {
    extern __shared__ __align__(16) int smem_i[];
    const DecodeShape s = a.s;
    const RouteMap m = carve_map(smem_i, s, true);
    float* acc = reinterpret_cast<float*>(smem_i + map_ints(s, true));

    constexpr int G = 32 / L;
    const int RS = DEC_WARPS / a.es;
    const int rows_cta = RS * G;
    build_route_map(m, a.ids, a.w, s, a.err);
    for (int i = threadIdx.x; i < DEC_WARPS * G * s.B; i += DEC_THREADS) acc[i] = 0.f;
    __syncthreads();
    // h comes from the gate/up pass: wait for it (no-op when this grid was
    // not launched as a programmatic dependent).
    asm volatile("griddepcontrol.wait;" ::: "memory");

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int grp = lane / L, li = lane % L;
    const int rs = warp % RS, es = warp / RS;
    const int r_local = rs * G + grp;
    const int o = blockIdx.x * rows_cta + r_local;
    const bool row_ok = o < s.d;
    const int orow = row_ok ? o : s.d - 1;
    const int nu = m.hdr[0];
    const int cpl = s.I / 32 / L;
    const int KS = s.k + s.S;
    const size_t rowsK = (size_t)s.d * s.I;
    float* my_acc = acc + (size_t)(es * rows_cta + r_local) * s.B;

    for (int u = es; u < nu; u += a.es) {
        const int e = m.uexp[u];
        const bool sh = e >= s.E;
        const size_t eo = sh ? 0 : (size_t)e;
        const MXView vd = sh ? a.shd : a.wd;
        const uint8_t* wd_row = vd.w + eo * rowsK + (size_t)orow * s.I;
        const uint8_t* sd_row = vd.s + (eo * rowsK + (size_t)orow * s.I) / 32;
        const int s0 = m.uoff[u], s1 = m.uoff[u + 1];
        for (int t0 = s0; t0 < s1; t0 += TC) {
            const int nt = min(TC, s1 - t0);
            float dots[TC];
            const int* hs = m.hrow + t0;
            switch (nt) {
                case 1: down_rows<L, 1>(wd_row, sd_row, a.h, hs, s.I, cpl, li, dots); break;
                case 2: down_rows<L, 2>(wd_row, sd_row, a.h, hs, s.I, cpl, li, dots); break;
                case 3: down_rows<L, 3>(wd_row, sd_row, a.h, hs, s.I, cpl, li, dots); break;
                default: down_rows<L, 4>(wd_row, sd_row, a.h, hs, s.I, cpl, li, dots); break;
            }
            if (li == 0 && row_ok) {
                for (int t = 0; t < nt; ++t) my_acc[hs[t] / KS] += m.wt[t0 + t] * dots[t];
            }
        }
    }
    __syncthreads();
    // add the expert splits in a fixed order, round once to BF16
    for (int i = threadIdx.x; i < rows_cta * s.B; i += DEC_THREADS) {
        const int r = i % rows_cta, b = i / rows_cta;
        const int oo = blockIdx.x * rows_cta + r;
        if (oo < s.d) {
            float sum = 0.f;
            for (int q = 0; q < a.es; ++q) sum += acc[(size_t)(q * rows_cta + r) * s.B + b];
            a.y[(size_t)b * s.d + oo] = __bfloat16_as_ushort(__float2bfloat16_rn(sum));
        }
    }
}

// -------------------------------------------------------------- host -----

// Lanes per weight row: the largest power of two <= 32 that divides the
// number of 32-element blocks along K, so every lane of a row group gets
// the same number of blocks.
static int lanes_per_row(int K) {
    const int nb = K / 32;
    int L = 32;
    while (L > 1 && nb % L) L >>= 1;
    return L;
}

size_t gate_up_smem_bytes(const DecodeShape& s) { return map_ints(s, false) * 4; }

size_t down_smem_bytes(const DecodeShape& s) {
    const int G = 32 / lanes_per_row(s.I);
    return map_ints(s, true) * 4 + (size_t)DEC_WARPS * G * s.B * 4;
}

template <typename F>
static cudaError_t prepare(F* fn, size_t smem, int dev, int* blocks_per_sm) {
    static std::mutex mu;
    static std::map<std::pair<const void*, int>, std::pair<size_t, int>> cache;
    std::lock_guard<std::mutex> lock(mu);
    auto key = std::make_pair((const void*)fn, dev);
    auto it = cache.find(key);
    if (it != cache.end() && it->second.first >= smem) {
        *blocks_per_sm = it->second.second;
        return cudaSuccess;
    }
    cudaError_t err = cudaSuccess;
    if (smem > 48 * 1024) {
        err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (err != cudaSuccess) return err;
    }
    int nb = 0;
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, fn, DEC_THREADS, smem);
    if (err != cudaSuccess) return err;
    if (nb < 1) nb = 1;
    cache[key] = std::make_pair(smem, nb);
    *blocks_per_sm = nb;
    return cudaSuccess;
}

template <int L>
static cudaError_t launch_gate_up_L(const GateUpArgs& a, size_t smem, const DeviceInfo& di, int dev,
                                    cudaStream_t st) {
    int bps = 1;
    cudaError_t err = prepare(gate_up_kernel<L>, smem, dev, &bps);
    if (err != cudaSuccess) return err;
    constexpr int G = 32 / L;
    const long items = (long)max_unique(a.s) * ((a.s.I + G - 1) / G);
    long grid = std::min<long>((long)di.sm_count * bps, (items + DEC_WARPS - 1) / DEC_WARPS);
    if (grid < 1) grid = 1;
    gate_up_kernel<L><<<(unsigned)grid, DEC_THREADS, smem, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_gate_up(const DecodeShape& s, const void* x, const int32_t* ids, MXView wg,
                           MXView wu, MXView shg, MXView shu, void* h, cudaStream_t st) {
    DeviceInfo di;
    cudaError_t err = device_info(&di);
    if (err != cudaSuccess) return err;
    int dev = 0;
    cudaGetDevice(&dev);
    GateUpArgs a{s, (const uint16_t*)x, ids, wg, wu, shg, shu, (uint16_t*)h, di.err_word};
    const size_t smem = gate_up_smem_bytes(s);
    switch (lanes_per_row(s.d)) {
        case 32: return launch_gate_up_L<32>(a, smem, di, dev, st);
        case 16: return launch_gate_up_L<16>(a, smem, di, dev, st);
        case 8: return launch_gate_up_L<8>(a, smem, di, dev, st);
        case 4: return launch_gate_up_L<4>(a, smem, di, dev, st);
        case 2: return launch_gate_up_L<2>(a, smem, di, dev, st);
        default: return launch_gate_up_L<1>(a, smem, di, dev, st);
    }
}

template <int L>
static cudaError_t launch_down_L(DownArgs a, size_t smem, const DeviceInfo& di, int dev,
                                 cudaStream_t st, bool pdl) {
    int bps = 1;
    cudaError_t err = prepare(down_kernel<L>, smem, dev, &bps);
    if (err != cudaSuccess) return err;
    constexpr int G = 32 / L;
    // expert splits: enough warps to cover the GPU, never more splits than
    // distinct experts a call can have
    const long target_warps = (long)di.sm_count * 16;
    const int mu = max_unique(a.s);
    int es = 1;
    while (es < DEC_WARPS && es * 2 <= mu) {
        const long rows_cta = (long)(DEC_WARPS / es) * G;
        const long warps = (a.s.d + rows_cta - 1) / rows_cta * DEC_WARPS;
        if (warps >= target_warps) break;
        es *= 2;
    }
    a.es = es;
    const int rows_cta = (DEC_WARPS / es) * G;
    const unsigned grid = (unsigned)((a.s.d + rows_cta - 1) / rows_cta);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(DEC_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, down_kernel<L>, a);
}

cudaError_t launch_down(const DecodeShape& s, const void* h, const int32_t* ids, const float* w,
                        MXView wd, MXView shd, void* y, cudaStream_t st, bool after_gate_up) {
    DeviceInfo di;
    cudaError_t err = device_info(&di);
    if (err != cudaSuccess) return err;
    int dev = 0;
    cudaGetDevice(&dev);
    DownArgs a{s, (const uint16_t*)h, ids, w, wd, shd, (uint16_t*)y, di.err_word, 1};
    const size_t smem = down_smem_bytes(s);
    switch (lanes_per_row(s.I)) {
        case 32: return launch_down_L<32>(a, smem, di, dev, st, after_gate_up);
        case 16: return launch_down_L<16>(a, smem, di, dev, st, after_gate_up);
        case 8: return launch_down_L<8>(a, smem, di, dev, st, after_gate_up);
        case 4: return launch_down_L<4>(a, smem, di, dev, st, after_gate_up);
        case 2: return launch_down_L<2>(a, smem, di, dev, st, after_gate_up);
        default: return launch_down_L<1>(a, smem, di, dev, st, after_gate_up);
    }
}

}  // namespace moedec

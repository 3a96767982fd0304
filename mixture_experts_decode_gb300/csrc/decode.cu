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
#include <cuda.h>

#include <algorithm>
#include <map>
#include <mutex>
#include <tuple>

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
    int* ucnt;  // [max_unique] slots per distinct expert after merging duplicates (down)
    int* tok;   // [slots] token of each entry (down)
};

__host__ __device__ inline int max_unique(const DecodeShape& s) {
    const int r = s.B * s.k;
    return (s.E < r ? s.E : r) + s.S;
}
__host__ __device__ inline int n_slots(const DecodeShape& s) { return s.B * s.k + s.S * s.B; }

__host__ __device__ inline size_t map_ints(const DecodeShape& s, bool with_w) {
    const size_t mu = (size_t)max_unique(s);
    size_t ints = 4 + mu + (mu + 1) + n_slots(s) + (with_w ? 2 * n_slots(s) + mu : 0) + s.E +
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
    p += DEC_WARPS;
    m.ucnt = with_w ? p : nullptr;
    if (with_w) p += mu;
    m.tok = with_w ? p : nullptr;
    return m;
}

__device__ void build_route_map(const RouteMap& m, const int32_t* __restrict__ ids,
                                const float* __restrict__ w, const DecodeShape& s, int* err,
                                bool merge = false, int* scratch = nullptr, int scratch_ints = 0) {
    // The first PT = min(blockDim.x, DEC_THREADS) threads (whole warps) build
    // the map; any further threads only take part in the barriers.
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int PT = min((int)blockDim.x, DEC_THREADS) & ~31, PW = PT >> 5;
    const bool part = tid < PT;
    const int n = s.B * s.k;
    // Parallel placement (32 < n <= PT, with a PW x E scratch table, e.g. the
    // idle copy ring; one warp's worth of slots is placed as fast serially):
    // thread f holds slot f; its position inside its expert's
    // range is the number of earlier slots with the same expert, i.e. the
    // slots of earlier warps (per-warp counts, scanned over warps) plus the
    // earlier lanes of its own warp (a match mask).
    const bool fast = n > 32 && n <= PT && scratch != nullptr && scratch_ints >= s.E * PW;
    int my_e = -1, my_rank = 0;
    float my_w = 0.f;
    if (fast) {
        if (tid < n) {
            my_e = ids[tid];
            if (w) my_w = w[tid];
        }
        for (int i = tid; i < s.E * PW; i += blockDim.x) scratch[i] = 0;
        if (tid < n && (unsigned)my_e >= (unsigned)s.E) {
            my_e = -1;
            atomicOr(err, MOE_DEVERR_EXPERT_ID);
        }
        __syncthreads();
        if (part) {
            const unsigned mask = __match_any_sync(FULL_MASK, my_e);
            my_rank = __popc(mask & lanemask_lt());
            if (my_e >= 0 && my_rank == 0) scratch[my_e * PW + warp] = __popc(mask);
        }
        __syncthreads();
        // per expert: counts of the earlier warps (exclusive) and the total
        if (part)
            for (int e = tid; e < s.E; e += PT) {
                int c = 0;
                for (int q = 0; q < PW; ++q) {
                    const int t = scratch[e * PW + q];
                    scratch[e * PW + q] = c;
                    c += t;
                }
                m.cnt[e] = c;
            }
    } else {
        if (part)
            for (int e = tid; e < s.E; e += PT) m.cnt[e] = 0;
        __syncthreads();
        if (part) {
            int bad = 0;
            for (int f = tid; f < n; f += PT) {
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
        }
    }
    __syncthreads();

    // Exclusive scan over experts of (count << 16 | present): gives each
    // present expert its distinct index (low half) and slot offset (high).
    const int per = (s.E + PT - 1) / PT;
    const int e0 = part ? min(tid * per, s.E) : s.E, e1 = part ? min(e0 + per, s.E) : s.E;
    int local = 0, incl = 0;
    if (part) {
        for (int e = e0; e < e1; ++e) {
            const int c = m.cnt[e];
            local += (c << 16) | (c > 0 ? 1 : 0);
        }
        incl = local;
        for (int off = 1; off < 32; off <<= 1) {
            const int v = __shfl_up_sync(FULL_MASK, incl, off);
            if (lane >= off) incl += v;
        }
        if (lane == 31) m.wtot[warp] = incl;
    }
    __syncthreads();
    if (warp == 0) {
        const int v = lane < PW ? m.wtot[lane] : 0;
        int sc = v;
        for (int off = 1; off < 32; off <<= 1) {
            const int t = __shfl_up_sync(FULL_MASK, sc, off);
            if (lane >= off) sc += t;
        }
        if (lane < PW) m.wtot[lane] = sc - v;
        if (lane == PW - 1) {
            m.hdr[1] = sc & 0xffff;
            m.hdr[2] = sc >> 16;
        }
    }
    __syncthreads();
    if (part) {
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
    }
    __syncthreads();

    // Stable placement of slots into their expert's range (the order inside
    // an expert is increasing flat slot index).
    const int nu = m.hdr[1], tot = m.hdr[2];
    const int KS = s.k + s.S;
    if (fast) {
        if (my_e >= 0) {
            const int pos = m.cnt[my_e] + scratch[my_e * PW + warp] + my_rank;
            const int b = tid / s.k, j = tid - b * s.k;
            m.hrow[pos] = b * KS + j;
            if (m.wt) m.wt[pos] = my_w;
        }
    } else if (warp == 0) {
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
    if (s.S && part) {
        for (int b = tid; b < s.B; b += PT) {
            m.hrow[tot + b] = b * KS + s.k;
            if (m.wt) m.wt[tot + b] = 1.0f;
        }
    }
    __syncthreads();
    if (merge) {
        // A token that picked the same expert twice gets one entry with the
        // summed routing weight (its two h rows are equal); entries of one
        // token are adjacent because placement follows the flat slot order.
        const int ntot = m.hdr[0];
        if (part) {
            for (int u = tid; u < ntot; u += PT) {
                const int i0 = m.uoff[u], i1 = m.uoff[u + 1];
                int wpos = i0;
                for (int i = i0; i < i1; ++i) {
                    const int hr = m.hrow[i];
                    const int b = hr / KS;
                    if (wpos > i0 && b == m.tok[wpos - 1]) {
                        m.wt[wpos - 1] += m.wt[i];
                    } else {
                        m.hrow[wpos] = hr;
                        m.wt[wpos] = m.wt[i];
                        m.tok[wpos] = b;
                        ++wpos;
                    }
                }
                m.ucnt[u] = wpos - i0;
            }
        }
        __syncthreads();
    }
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

// --------------------------------------------------------- gate/up v2 ----
// Each warp owns (distinct expert, pair of rows) items.  A lane handles
// 16-byte K chunks (16 E4M3 codes, all inside one 32-element scale block) of
// both rows and both projections, so one BF16->FP32 conversion of x serves
// four weight rows.  Chunks are prefetched into a per-warp shared-memory ring
// with cp.async (each lane reads back only the bytes it copied, so no warp
// barrier is needed); x comes through L1, where the CTA's warps, which walk
// adjacent rows of the same expert, share it.  The E8M0 scale multiplies each
// chunk's partial sums once; the 4 x NT results of an item are reduced across
// the warp in one reduce-scatter.  Needs d % 128 == 0 (4-byte scale words).

constexpr int GU2_STAGES = 4;
constexpr int GU2_PARTS = 4;  // (row 0 gate, row 1 gate, row 0 up, row 1 up)
constexpr int GU2_CHUNK = 512;  // K bytes per warp per part per step (32 lanes x 16)

struct GU2Ring {
    uint4 w[GU2_STAGES][GU2_PARTS][32];
    uint32_t s[GU2_STAGES][GU2_PARTS][32];
};

struct GU2Warp {
    int first, stride, end;  // this warp's items: first, first + stride, ... < end
    int tiles;               // row pairs per expert
    int nch;                 // chunks per row
};

struct GU2Cursor {
    int m, g, c;  // item ordinal of this warp, token group, chunk
};

__device__ __forceinline__ int gu2_groups(const RouteMap& m, int u) {
    return (m.uoff[u + 1] - m.uoff[u] + TC - 1) / TC;
}

// Issue the copies of the step under the cursor into ring slot `slot` and
// advance the cursor; always commits one group (empty past the end).
__device__ __forceinline__ void gu2_issue(const GateUpArgs& a, const RouteMap& m, const GU2Warp& wi,
                                          GU2Cursor& pc, GU2Ring* ring, int slot, int lane,
                                          uint64_t pol) {
    const int item = wi.first + pc.m * wi.stride;
    if (item < wi.end) {
        const DecodeShape& s = a.s;
        const int u = item / wi.tiles;
        const int n0 = (item - u * wi.tiles) * 2;
        const int e = m.uexp[u];
        const bool sh = e >= s.E;
        const size_t eo = sh ? 0 : (size_t)e;
        const MXView vg = sh ? a.shg : a.wg, vu = sh ? a.shu : a.wu;
        const size_t r0 = eo * s.I + n0;
        const int kofs = pc.c * GU2_CHUNK + lane * 16;
        const bool ok = kofs < s.d;
        const int kk = ok ? kofs : 0;
        const int nb = s.d / 32;
        const int sw = ok ? (((pc.c * 16 + (lane >> 1)) >> 2) << 2) : 0;
        const uint8_t* wrow[GU2_PARTS] = {vg.w + r0 * s.d, vg.w + (r0 + 1) * s.d, vu.w + r0 * s.d,
                                          vu.w + (r0 + 1) * s.d};
        const uint8_t* srow[GU2_PARTS] = {vg.s + r0 * nb, vg.s + (r0 + 1) * nb, vu.s + r0 * nb,
                                          vu.s + (r0 + 1) * nb};
#pragma unroll
        for (int p = 0; p < GU2_PARTS; ++p) {
            cp_async_16(&ring->w[slot][p][lane], wrow[p] + kk, ok ? 16 : 0, pol);
            cp_async_4(&ring->s[slot][p][lane], srow[p] + sw, ok ? 4 : 0);
        }
        if (++pc.c == wi.nch) {
            pc.c = 0;
            if (++pc.g == gu2_groups(m, u)) {
                pc.g = 0;
                ++pc.m;
            }
        }
    }
    cp_async_commit();
}

template <int NT, bool FOLD>
__device__ __forceinline__ void gu2_group(const GateUpArgs& a, const RouteMap& m, const GU2Warp& wi,
                                          GU2Cursor& pc, GU2Ring* ring, int& slot, int lane,
                                          uint64_t pol, int n0, const int* hs, int nt) {
    constexpr int NTP = NT == 3 ? 4 : NT;  // padded to a power of two for the reduction
    const DecodeShape& s = a.s;
    const int KS = s.k + s.S;
    const char* xr[NT];
    int hr[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        hr[t] = hs[t];
        xr[t] = reinterpret_cast<const char*>(a.x + (size_t)(hr[t] / KS) * s.d);
    }
    float2 acc[GU2_PARTS][NT];
#pragma unroll
    for (int p = 0; p < GU2_PARTS; ++p)
#pragma unroll
        for (int t = 0; t < NT; ++t) acc[p][t] = make_float2(0.f, 0.f);
    const int bsh = ((lane >> 1) & 3) * 8;  // this lane's scale byte inside its 4-byte word

    for (int c = 0; c < wi.nch; ++c) {
        gu2_issue(a, m, wi, pc, ring, (slot + GU2_STAGES - 1) % GU2_STAGES, lane, pol);
        cp_async_wait<GU2_STAGES - 1>();
        const int kofs = c * GU2_CHUNK + lane * 16;
        const bool kin = kofs < s.d;
        uint4 wv[GU2_PARTS];
        float sc[GU2_PARTS];
#pragma unroll
        for (int p = 0; p < GU2_PARTS; ++p) {
            wv[p] = ring->w[slot][p][lane];
            sc[p] = e8m0_to_float((ring->s[slot][p][lane] >> bsh) & 0xffu);
        }
        float2 part[GU2_PARTS][NT];
#pragma unroll
        for (int p = 0; p < GU2_PARTS; ++p)
#pragma unroll
            for (int t = 0; t < NT; ++t) part[p][t] = make_float2(0.f, 0.f);
        uint4 xv[NT];
#pragma unroll
        for (int q = 0; q < 8; ++q) {  // pairs of K elements
            if ((q & 3) == 0) {        // next 8 activations of every token
#pragma unroll
                for (int t = 0; t < NT; ++t)
                    xv[t] = kin ? ld_cached_128(xr[t] + (size_t)kofs * 2 + (q >> 2) * 16) : make_uint4(0, 0, 0, 0);
            }
            float2 wq[GU2_PARTS];
#pragma unroll
            for (int p = 0; p < GU2_PARTS; ++p) {
                const uint32_t word = (&wv[p].x)[q >> 1];
                wq[p] = e4m3x2_to_float2(word >> ((q & 1) * 16));
                if (!FOLD) wq[p] = __fmul2_rn(wq[p], make_float2(sc[p], sc[p]));
            }
#pragma unroll
            for (int t = 0; t < NT; ++t) {
                const uint32_t xw = (&xv[t].x)[q & 3];
                const float2 xf = bf16x2_to_float2(xw);
#pragma unroll
                for (int p = 0; p < GU2_PARTS; ++p) {
                    if (FOLD)
                        part[p][t] = __ffma2_rn(xf, wq[p], part[p][t]);
                    else
                        acc[p][t] = __ffma2_rn(xf, wq[p], acc[p][t]);
                }
            }
        }
        if (FOLD) {
#pragma unroll
            for (int p = 0; p < GU2_PARTS; ++p)
#pragma unroll
                for (int t = 0; t < NT; ++t)
                    acc[p][t] = __ffma2_rn(part[p][t], make_float2(sc[p], sc[p]), acc[p][t]);
        }
        slot = (slot + 1) % GU2_STAGES;
    }

    // value index = proj * 2NTP + row * NTP + token
    constexpr int N = 4 * NTP;
    float v[N];
#pragma unroll
    for (int p = 0; p < GU2_PARTS; ++p) {
        const int proj = p >> 1, rr = p & 1;
#pragma unroll
        for (int t = 0; t < NTP; ++t)
            v[proj * 2 * NTP + rr * NTP + t] = t < NT ? acc[p][t < NT ? t : 0].x + acc[p][t < NT ? t : 0].y : 0.f;
    }
    const float r = warp_reduce_scatter<N>(v, lane);
    const float up = __shfl_xor_sync(FULL_MASK, r, 16);
    constexpr int LOGN = N == 4 ? 2 : (N == 8 ? 3 : 4);
    const int idx = (lane >> (5 - LOGN)) & (N - 1);
    const int proj = idx / (2 * NTP), rr = (idx / NTP) & 1, t = idx % NTP;
    const bool lead = (lane & ((1 << (5 - LOGN)) - 1)) == 0;
    if (proj == 0 && lead && t < nt) {
        const float hv = r / (1.0f + expf(-r)) * up;
        int hrow = hs[0];
#pragma unroll
        for (int tt = 1; tt < NT; ++tt)
            if (tt == t) hrow = hr[tt];
        a.h[(size_t)hrow * s.I + n0 + rr] = __bfloat16_as_ushort(__float2bfloat16_rn(hv));
    }
}

#ifndef MOEDEC_GU2_MINB
#define MOEDEC_GU2_MINB 2
#endif

template <bool FOLD>
__global__ void __launch_bounds__(DEC_THREADS, MOEDEC_GU2_MINB) gate_up_v2_kernel(GateUpArgs a) {
    extern __shared__ __align__(16) int smem_i[];
    const DecodeShape s = a.s;
    const RouteMap m = carve_map(smem_i, s, false);
    GU2Ring* rings = reinterpret_cast<GU2Ring*>(smem_i + map_ints(s, false));
    build_route_map(m, a.ids, nullptr, s, a.err);
    asm volatile("griddepcontrol.launch_dependents;");

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    GU2Ring* ring = rings + warp;
    const int nu = m.hdr[0];
    GU2Warp wi;
    wi.tiles = s.I / 2;
    wi.nch = (s.d + GU2_CHUNK - 1) / GU2_CHUNK;
    // items round-robin over every warp of the grid: consecutive items (rows
    // of one expert) run at the same time on the warps of one CTA, and a hot
    // expert's items spread over the whole GPU
    wi.end = nu * wi.tiles;
    wi.first = blockIdx.x * DEC_WARPS + warp;
    wi.stride = gridDim.x * DEC_WARPS;
    const uint64_t pol = l2_evict_first_policy();

    GU2Cursor pc{0, 0, 0};
    int slot = 0;
#pragma unroll
    for (int i = 0; i < GU2_STAGES - 1; ++i) gu2_issue(a, m, wi, pc, ring, i, lane, pol);

    for (int item = wi.first; item < wi.end; item += wi.stride) {
        const int u = item / wi.tiles;
        const int n0 = (item - u * wi.tiles) * 2;
        const int s0 = m.uoff[u], s1 = m.uoff[u + 1];
        for (int t0 = s0; t0 < s1; t0 += TC) {
            const int nt = min(TC, s1 - t0);
            const int* hs = m.hrow + t0;
            switch (nt) {
                case 1: gu2_group<1, FOLD>(a, m, wi, pc, ring, slot, lane, pol, n0, hs, nt); break;
                case 2: gu2_group<2, FOLD>(a, m, wi, pc, ring, slot, lane, pol, n0, hs, nt); break;
                case 3: gu2_group<3, FOLD>(a, m, wi, pc, ring, slot, lane, pol, n0, hs, nt); break;
                default: gu2_group<4, FOLD>(a, m, wi, pc, ring, slot, lane, pol, n0, hs, nt); break;
            }
        }
    }
    cp_async_wait<0>();
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

// --------------------------------------------------------- gate/up v3 ----
// Warp-specialised: one producer warp streams, per stage, a 16-row x 512-byte
// K slice of the gate and up weights of one distinct expert (one 1D bulk
// copy per row and projection, plus the matching E8M0 scale bytes) and the
// same K slice of x for up to TC tokens into a 4-stage shared-memory ring,
// completion counted on an mbarrier; eight consumer warps each own two of the
// 16 rows, lanes take 16 bytes of the slice, and compute as in v2.  A tile =
// (distinct expert, 16 rows); tiles are dealt round-robin to persistent CTAs,
// and a tile with more than TC tokens streams its slices once per token
// group (the repeat hits L2).  Every wait is bounded.  Needs d % 512 == 0.

constexpr int GU3_CW = 8;                       // consumer warps
constexpr int GU3_THREADS = (GU3_CW + 1) * 32;  // + one producer warp
constexpr int GU3_ROWS = 2 * GU3_CW;            // weight rows per tile
constexpr int GU3_KT = 512;                     // K bytes per stage
constexpr int GU3_S = 4;                        // ring stages
#ifndef MOEDEC_GU3_MINB
#define MOEDEC_GU3_MINB 2
#endif
#ifndef MOEDEC_GU3_FOLD
#define MOEDEC_GU3_FOLD 0
#endif

constexpr int GU3_BOX = 256;                    // inner box of a 2D tensor copy (bytes)

struct __align__(128) GU3Stage {
    uint8_t w[2][GU3_KT / GU3_BOX][GU3_ROWS][GU3_BOX];  // [proj][half][row][k]
    uint8_t sc[2][GU3_ROWS][16];                        // E8M0 scales of the slice
    uint16_t x[TC][GU3_KT];                             // BF16 activations of the slice
};

struct GU3Smem {
    GU3Stage st[GU3_S];
    uint64_t full[GU3_S];
    uint64_t empty[GU3_S];
};

// 2D tensor maps (uint8, [rows][cols]) of the weight codes and scales.
struct GU3Maps {
    CUtensorMap w[2][2];  // [routed / shared][gate / up], box 16 rows x 256 B
    CUtensorMap s[2][2];  // the same for the scales, box 16 rows x 16 B
};

__device__ __forceinline__ void tma_3d(void* dst, const CUtensorMap* map, int x, int y, int z, uint64_t* bar,
                                       uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar)), "l"(pol)
        : "memory");
}

__device__ __forceinline__ void tma_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar,
                                       uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar)), "l"(pol)
        : "memory");
}

template <int NT>
__device__ __forceinline__ bool gu3_group(const GateUpArgs& a, GU3Smem* sm, uint32_t& it, int nkt,
                                          int cw, int lane, int n0, const int* hs, int nt) {
    constexpr int NTP = NT == 3 ? 4 : NT;
    const DecodeShape& s = a.s;
    float2 acc[GU2_PARTS][NT];
#pragma unroll
    for (int p = 0; p < GU2_PARTS; ++p)
#pragma unroll
        for (int t = 0; t < NT; ++t) acc[p][t] = make_float2(0.f, 0.f);

    for (int kt = 0; kt < nkt; ++kt, ++it) {
        const int slot = it % GU3_S;
        if (!mbar_wait(&sm->full[slot], (it / GU3_S) & 1)) return false;
        const GU3Stage& st = sm->st[slot];
        uint4 wv[GU2_PARTS];
        float sc[GU2_PARTS];
#pragma unroll
        for (int p = 0; p < GU2_PARTS; ++p) {  // part = proj * 2 + row
            const int proj = p >> 1, row = 2 * cw + (p & 1);
            wv[p] = *reinterpret_cast<const uint4*>(&st.w[proj][lane >> 4][row][(lane & 15) * 16]);
            sc[p] = e8m0_to_float(st.sc[proj][row][lane >> 1]);
        }
#if MOEDEC_GU3_FOLD
        float2 part[GU2_PARTS][NT];
#endif
        uint4 xv[NT];
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {  // groups of four K elements
            if ((q4 & 1) == 0) {
#pragma unroll
                for (int t = 0; t < NT; ++t)
                    xv[t] = *reinterpret_cast<const uint4*>(&st.x[t][lane * 16 + (q4 >> 1) * 8]);
            }
            float2 wq[GU2_PARTS][2];
#pragma unroll
            for (int p = 0; p < GU2_PARTS; ++p) {
                e4m3x4_to_float((&wv[p].x)[q4], wq[p][0], wq[p][1]);
#if !MOEDEC_GU3_FOLD
                wq[p][0] = __fmul2_rn(wq[p][0], make_float2(sc[p], sc[p]));
                wq[p][1] = __fmul2_rn(wq[p][1], make_float2(sc[p], sc[p]));
#endif
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
#pragma unroll
                for (int t = 0; t < NT; ++t) {
                    const float2 xf = bf16x2_to_float2((&xv[t].x)[(q4 & 1) * 2 + h]);
#pragma unroll
                    for (int p = 0; p < GU2_PARTS; ++p) {
#if MOEDEC_GU3_FOLD
                        if (q4 == 0 && h == 0)
                            part[p][t] = __fmul2_rn(xf, wq[p][h]);
                        else
                            part[p][t] = __ffma2_rn(xf, wq[p][h], part[p][t]);
#else
                        acc[p][t] = __ffma2_rn(xf, wq[p][h], acc[p][t]);
#endif
                    }
                }
            }
        }
#if MOEDEC_GU3_FOLD
#pragma unroll
        for (int p = 0; p < GU2_PARTS; ++p)
#pragma unroll
            for (int t = 0; t < NT; ++t) acc[p][t] = __ffma2_rn(part[p][t], make_float2(sc[p], sc[p]), acc[p][t]);
#endif
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm->empty[slot]);
    }

    constexpr int N = 4 * NTP;  // value index = proj * 2NTP + row * NTP + token
    float v[N];
#pragma unroll
    for (int p = 0; p < GU2_PARTS; ++p) {
        const int proj = p >> 1, rr = p & 1;
#pragma unroll
        for (int t = 0; t < NTP; ++t)
            v[proj * 2 * NTP + rr * NTP + t] = t < NT ? acc[p][t < NT ? t : 0].x + acc[p][t < NT ? t : 0].y : 0.f;
    }
    const float r = warp_reduce_scatter<N>(v, lane);
    const float up = __shfl_xor_sync(FULL_MASK, r, 16);
    constexpr int LOGN = N == 4 ? 2 : (N == 8 ? 3 : 4);
    const int idx = (lane >> (5 - LOGN)) & (N - 1);
    const int proj = idx / (2 * NTP), rr = (idx / NTP) & 1, t = idx % NTP;
    const bool lead = (lane & ((1 << (5 - LOGN)) - 1)) == 0;
    if (proj == 0 && lead && t < nt) {
        const float hv = r / (1.0f + expf(-r)) * up;
        int hrow = hs[0];
#pragma unroll
        for (int tt = 1; tt < NT; ++tt)
            if (tt == t) hrow = hs[tt];
        a.h[(size_t)hrow * s.I + n0 + 2 * cw + rr] = __bfloat16_as_ushort(__float2bfloat16_rn(hv));
    }
    return true;
}

__host__ __device__ inline size_t gu3_smem_offset(const DecodeShape& s) {
    return (map_ints(s, false) * 4 + 127) / 128 * 128;
}

__global__ void __launch_bounds__(GU3_THREADS, MOEDEC_GU3_MINB)
    gate_up_v3_kernel(GateUpArgs a, const __grid_constant__ GU3Maps maps) {
    extern __shared__ __align__(128) int smem_i[];
    const DecodeShape s = a.s;
    const RouteMap m = carve_map(smem_i, s, false);
    // tensor copies want 128-byte aligned destinations: align at run time
    // (the launch reserves 128 spare bytes)
    const uintptr_t raw = reinterpret_cast<uintptr_t>(smem_i) + gu3_smem_offset(s);
    GU3Smem* sm = reinterpret_cast<GU3Smem*>((raw + 127) & ~uintptr_t(127));
    if (threadIdx.x == 0) {
        for (int i = 0; i < GU3_S; ++i) {
            mbar_init(&sm->full[i], 1);
            mbar_init(&sm->empty[i], GU3_CW);
        }
        mbar_init_fence();
    }
    // the copy ring is idle until the map is built: it serves as the map's scratch
    build_route_map(m, a.ids, nullptr, s, a.err, false, reinterpret_cast<int*>(sm->st),
                    (int)(sizeof(sm->st) / 4));  // ends with __syncthreads
    asm volatile("griddepcontrol.launch_dependents;");

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int KS = s.k + s.S;
    const int rbs = s.I / GU3_ROWS;
    const int tiles = m.hdr[0] * rbs;
    const int nkt = s.d / GU3_KT;
    bool ok = true;
    uint32_t it = 0;  // stages produced / consumed by this thread so far

    if (warp == GU3_CW) {
        // ---------------- producer ----------------
        const uint64_t pol = l2_evict_first_policy();
        for (int tile = blockIdx.x; tile < tiles && ok; tile += gridDim.x) {
            const int u = tile / rbs;
            const int n0 = (tile - u * rbs) * GU3_ROWS;
            const int e = m.uexp[u];
            const int sh = e >= s.E ? 1 : 0;
            const int row0 = (sh ? 0 : e) * s.I + n0;
            const int s0 = m.uoff[u], s1 = m.uoff[u + 1];
            for (int t0 = s0; t0 < s1 && ok; t0 += TC) {
                const int nt = min(TC, s1 - t0);
                const uint16_t* xrow = a.x + (size_t)(lane < nt ? m.hrow[t0 + lane] / KS : 0) * s.d;
                for (int kt = 0; kt < nkt; ++kt, ++it) {
                    const int slot = it % GU3_S;
                    if (it >= GU3_S && !mbar_wait(&sm->empty[slot], ((it / GU3_S) - 1) & 1)) {
                        ok = false;
                        break;
                    }
                    GU3Stage& st = sm->st[slot];
                    if (lane == 0) {
                        mbar_arrive_expect_tx(&sm->full[slot],
                                              2 * GU3_ROWS * (GU3_KT + 16) + nt * GU3_KT * 2);
                        fence_proxy_async();
#pragma unroll
                        for (int p = 0; p < 2; ++p) {
#pragma unroll
                            for (int hf = 0; hf < GU3_KT / GU3_BOX; ++hf)
                                tma_2d(st.w[p][hf], &maps.w[sh][p], kt * GU3_KT + hf * GU3_BOX, row0,
                                       &sm->full[slot], pol);
                            tma_2d(st.sc[p], &maps.s[sh][p], kt * 16, row0, &sm->full[slot], pol);
                        }
                    }
                    __syncwarp();
                    if (lane < nt) {
                        fence_proxy_async();
                        bulk_g2s_keep(st.x[lane], xrow + (size_t)kt * GU3_KT, GU3_KT * 2, &sm->full[slot]);
                    }
                }
            }
        }
        // never leave the CTA with a copy in flight: wait for the last stages
        for (uint32_t j = it > GU3_S ? it - GU3_S : 0; j < it; ++j)
            mbar_wait(&sm->full[j % GU3_S], (j / GU3_S) & 1);
    } else {
        // ---------------- consumers ----------------
        for (int tile = blockIdx.x; tile < tiles && ok; tile += gridDim.x) {
            const int u = tile / rbs;
            const int n0 = (tile - u * rbs) * GU3_ROWS;
            const int s0 = m.uoff[u], s1 = m.uoff[u + 1];
            for (int t0 = s0; t0 < s1 && ok; t0 += TC) {
                const int nt = min(TC, s1 - t0);
                const int* hs = m.hrow + t0;
                switch (nt) {
                    case 1: ok = gu3_group<1>(a, sm, it, nkt, warp, lane, n0, hs, nt); break;
                    case 2: ok = gu3_group<2>(a, sm, it, nkt, warp, lane, n0, hs, nt); break;
                    case 3: ok = gu3_group<3>(a, sm, it, nkt, warp, lane, n0, hs, nt); break;
                    default: ok = gu3_group<4>(a, sm, it, nkt, warp, lane, n0, hs, nt); break;
                }
            }
        }
    }
    if (!ok && lane == 0) atomicOr(a.err, MOE_DEVERR_TIMEOUT);
}

// --------------------------------------------------------- gate/up v4 ----
// Lane per weight row.  A tile = (distinct expert, RT rows of I); LPR = 32 /
// RT lanes of every consumer warp own row n0 + r of both W_gate and W_up,
// each lane a different 32-element scale block of it, so a lane sums whole
// scale blocks by itself and scales each block's partial sum once.  The CW
// consumer warps split every 512-element K stage into its 16 scale blocks,
// warp w taking blocks w * LPR .. w * LPR + LPR - 1: per stage the warp
// converts those blocks of each token's x to FP32 once, into its own small
// buffer, and its lanes read them back as broadcasts.  The producer warp
// brings each stage's RT x 512 code bytes of both projections as RT-row x
// 128-byte tensor boxes stored in the 128-byte swizzled layout (chunk j of
// row r lands at chunk j ^ (r & 7)), so lanes reading the same chunk of
// consecutive rows hit distinct banks; plus the scale bytes and the tokens'
// x slices.  After a tile's last stage the lanes of a row add their halves
// by a shuffle, the warps' partial dots go through shared memory (double
// buffered by token-group parity, one barrier per group) and 2 x RT x nt
// threads, a pair per (token, row), add the CW warps in a fixed order,
// apply SiLU(g) * u and store h.  Every wait is bounded; a wait that runs
// out raises a CTA-wide abort flag so that all warps still pass every
// barrier.  Two geometries: RT = 32 with 16 consumer warps and one CTA per
// SM, RT = 16 with 8 consumer warps and two CTAs per SM.

#ifndef MOEDEC_GU4_ORDER
#define MOEDEC_GU4_ORDER 1
#endif
constexpr int GU4_KT = 512;   // K elements per stage (16 scale blocks)
constexpr int GU4_BOX = 128;  // inner box of a weight tensor copy (bytes)
constexpr int GU4_S = 4;      // ring stages

template <int RT>
struct __align__(1024) GU4Stage {
    uint8_t w[2][GU4_KT / GU4_BOX][RT][GU4_BOX];  // [proj][box][row][128 B, swizzled]
    uint8_t sc[2][RT][GU4_KT / 32];               // [proj][row][block] E8M0
    uint16_t x[TC][GU4_KT];                       // BF16 activations of the slice
};

// A warp's FP32 copy of x keeps each 32-element block at a stride of 36
// floats: the two blocks that the two halves of the warp broadcast from then
// sit in different banks.
constexpr int GU4_XH = 36;

template <int RT, int CW>
struct GU4Shared {
    float xf[CW][TC][(GU4_KT / CW / 32) * GU4_XH];  // per warp: its blocks of x, FP32
    float part[2][CW][2][TC][RT];         // [group parity][warp][proj][token][row] partial dots
    uint64_t full[GU4_S];
    uint64_t empty[GU4_S];
    int abort;
    int perm[256];  // distinct experts by descending token count (when at most 256)
};

struct GU4Maps {
    CUtensorMap w[2][2];  // [routed / shared][gate / up]: 128-byte swizzle; 2D box RT rows x 128 B,
                          // or (w3d) 3D box of the stage's 4 column blocks x RT rows x 128 B
    CUtensorMap s[2][2];  // the same for the scales, box RT rows x 16 B
    int w3d;
};

// Bounded wait that also gives up as soon as another warp raised `abort`;
// a wait that runs out (~2^32 cycles) raises it.
__device__ __forceinline__ bool mbar_wait_abort(uint64_t* bar, uint32_t parity, volatile int* abort) {
    const uint32_t a = smem_addr(bar);
    const long long t0 = clock64();
    for (;;) {
        uint32_t ok;
        asm volatile(
            "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3; selp.u32 %0, 1, 0, p; }"
            : "=r"(ok)
            : "r"(a), "r"(parity), "r"(20000u)
            : "memory");
        if (ok) return true;
        if (*abort) return false;
        if (clock64() - t0 > (1ll << 32)) {
            *abort = 1;
            return false;
        }
    }
}

template <int NTHREADS>
__device__ __forceinline__ void consumer_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(NTHREADS) : "memory");
}

// Ring position of a thread: slot and the parity of the phase it waits for.
struct RingPos {
    int slot;
    uint32_t par;
    __device__ __forceinline__ void next(int S) {
        if (++slot == S) {
            slot = 0;
            par ^= 1u;
        }
    }
};

__host__ __device__ inline size_t gu4_ring_offset(const DecodeShape& s) { return map_ints(s, false) * 4; }

template <int RT, int CW, int NT>
__device__ __forceinline__ void gu4_group(const GateUpArgs& a, GU4Stage<RT>* ring, GU4Shared<RT, CW>* sh,
                                          RingPos& rp, int grp, int nkt, int warp, int lane, int n0,
                                          const int* hs) {
    constexpr int LPR = 32 / RT;       // lanes per row
    constexpr int KW = GU4_KT / CW;    // K elements of a warp per stage (= 32 * LPR)
    static_assert(KW == 32 * LPR, "one scale block per lane");
    constexpr int XS = LPR * GU4_XH;   // floats per token in the warp's x copy
    const DecodeShape& s = a.s;
    float2 acc[2][NT];
#pragma unroll
    for (int p = 0; p < 2; ++p)
#pragma unroll
        for (int t = 0; t < NT; ++t) acc[p][t] = make_float2(0.f, 0.f);
    const int r = lane % RT, hb = lane / RT;   // row, which of the warp's blocks
    const int blk = warp * LPR + hb;           // scale block within the stage
    const int box = blk >> 2, c0 = (blk & 3) * 2, sw = r & 7;
    float* xf = &sh->xf[warp][0][0];
    for (int kt = 0; kt < nkt; ++kt, rp.next(GU4_S)) {
        const int slot = rp.slot;
        if (!mbar_wait_abort(&sh->full[slot], rp.par, &sh->abort)) continue;
        const GU4Stage<RT>& st = ring[slot];
        {  // this warp's blocks of x -> FP32: lane = (token, four K elements of each block)
            const int t = lane >> 3, k = (lane & 7) * 4;
            if (t < NT) {
                const uint16_t* xs = &st.x[t][warp * KW + k];
                float* xd = xf + t * XS + k;
#pragma unroll
                for (int q = 0; q < LPR; ++q) {
                    const uint2 xv = *reinterpret_cast<const uint2*>(xs + q * 32);
                    const float2 lo = bf16x2_to_float2(xv.x), hi = bf16x2_to_float2(xv.y);
                    *reinterpret_cast<float4*>(xd + q * GU4_XH) = make_float4(lo.x, lo.y, hi.x, hi.y);
                }
            }
        }
        __syncwarp();
        const float* xl = xf + hb * GU4_XH;
        float2 part[2][NT];
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2) {  // two 16-byte chunks = this lane's 32 K elements
            uint4 wv[2];
#pragma unroll
            for (int p = 0; p < 2; ++p)
                wv[p] = *reinterpret_cast<const uint4*>(&st.w[p][box][r][((c0 + c2) ^ sw) * 16]);
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                float2 wq[2][2];
#pragma unroll
                for (int p = 0; p < 2; ++p) e4m3x4_to_float((&wv[p].x)[q4], wq[p][0], wq[p][1]);
#pragma unroll
                for (int t = 0; t < NT; ++t) {
                    const float4 xv = *reinterpret_cast<const float4*>(xl + t * XS + c2 * 16 + q4 * 4);
#pragma unroll
                    for (int p = 0; p < 2; ++p) {
                        if (c2 == 0 && q4 == 0)
                            part[p][t] = __fmul2_rn(make_float2(xv.x, xv.y), wq[p][0]);
                        else
                            part[p][t] = __ffma2_rn(make_float2(xv.x, xv.y), wq[p][0], part[p][t]);
                        part[p][t] = __ffma2_rn(make_float2(xv.z, xv.w), wq[p][1], part[p][t]);
                    }
                }
            }
        }
#pragma unroll
        for (int p = 0; p < 2; ++p) {
            const float sc = e8m0_to_float(st.sc[p][r][blk]);
#pragma unroll
            for (int t = 0; t < NT; ++t) acc[p][t] = __ffma2_rn(part[p][t], make_float2(sc, sc), acc[p][t]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh->empty[slot]);
    }
    // this warp's partial dots (the lanes of a row add theirs, lower block
    // first) -> shared memory, double-buffered by group parity so one
    // barrier per group suffices; then two threads per (token, row) add the
    // warps' gate and up partials in a fixed order
    float(*part)[2][TC][RT] = sh->part[grp & 1];
#pragma unroll
    for (int p = 0; p < 2; ++p)
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            float v = acc[p][t].x + acc[p][t].y;
            if (LPR == 2) {
                const float o = __shfl_xor_sync(FULL_MASK, v, 16);
                v = hb ? o + v : v + o;
            }
            if (lane < RT) part[warp][p][t][lane] = v;
        }
    consumer_sync<CW * 32>();
    const int idx = warp * 32 + lane;
    if (warp < (2 * RT * NT + 31) / 32) {
        const int pj = idx & 1, rr = (idx >> 1) % RT, t = (idx >> 1) / RT;
        float v = 0.f;
        if (t < NT) {
#pragma unroll
            for (int w = 0; w < CW; ++w) v += part[w][pj][t][rr];
        }
        const float up = __shfl_xor_sync(FULL_MASK, v, 1);
        if (pj == 0 && t < NT && !sh->abort) {
            const float hv = v / (1.0f + expf(-v)) * up;
            int hrow = hs[0];
#pragma unroll
            for (int tt = 1; tt < NT; ++tt)
                if (tt == t) hrow = hs[tt];
            a.h[(size_t)hrow * s.I + n0 + rr] = __bfloat16_as_ushort(__float2bfloat16_rn(hv));
        }
    }
}

// The distinct experts u < nu (nu <= 256) ordered by descending slot count,
// the lower index first on ties, into perm[]: a bitonic sort of packed
// (255 - count, u) keys by the first 256 threads (shuffles below a distance
// of 32, `scratch` (256 words) above).  Every thread of the CTA must call it.
__device__ void order_experts_by_count(const RouteMap& m, int nu, int* perm, uint32_t* scratch) {
    const int tid = threadIdx.x;
    const bool part = tid < 256;
    uint32_t key = 0xffffffffu;
    if (part && tid < nu) {
        const int n = m.uoff[tid + 1] - m.uoff[tid];
        const int c = min(n, 255);
        key = ((uint32_t)(255 - c) << 16) | (uint32_t)tid;
    }
    for (int k = 2; k <= 256; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            uint32_t other = key;
            if (j >= 32) {
                if (part) scratch[tid] = key;
                __syncthreads();
                if (part) other = scratch[tid ^ j];
                __syncthreads();
            } else {
                other = __shfl_xor_sync(FULL_MASK, key, j);
            }
            const bool asc = (tid & k) == 0, low = (tid & j) == 0;
            if (part) key = low == asc ? min(key, other) : max(key, other);
        }
    }
    if (part && tid < nu) perm[tid] = (int)(key & 0xffffu);
    __syncthreads();
}

// Tile of round r for this CTA when tiles are dealt in snake order (round r
// goes over the CTAs forwards when r is even, backwards when odd).
__device__ __forceinline__ int snake_tile(int r) {
    return r * (int)gridDim.x + ((r & 1) ? (int)gridDim.x - 1 - (int)blockIdx.x : (int)blockIdx.x);
}

template <int RT, int CW>
__global__ void __launch_bounds__((CW + 1) * 32, RT == 32 ? 1 : 2)
    gate_up_v4_kernel(GateUpArgs a, const __grid_constant__ GU4Maps maps) {
    constexpr int S = GU4_S;
    extern __shared__ __align__(128) int smem_i[];
    const DecodeShape s = a.s;
    const RouteMap m = carve_map(smem_i, s, false);
    // swizzled tensor copies want 1024-byte aligned boxes: align at run time
    // (the launch reserves 1024 spare bytes)
    const uintptr_t raw = reinterpret_cast<uintptr_t>(smem_i) + gu4_ring_offset(s);
    GU4Stage<RT>* ring = reinterpret_cast<GU4Stage<RT>*>((raw + 1023) & ~uintptr_t(1023));
    GU4Shared<RT, CW>* sh = reinterpret_cast<GU4Shared<RT, CW>*>(ring + S);
    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(&sh->full[i], 1);
            mbar_init(&sh->empty[i], CW);
        }
        sh->abort = 0;
        mbar_init_fence();
    }
    // the copy ring is idle until the map is built: it serves as the map's scratch
    build_route_map(m, a.ids, nullptr, s, a.err, false, reinterpret_cast<int*>(ring),
                    (int)(S * sizeof(GU4Stage<RT>) / 4));  // ends with __syncthreads
    asm volatile("griddepcontrol.launch_dependents;");

    const int nu = m.hdr[0];
    const int rbs = s.I / RT;
    const int tiles = nu * rbs;
    // With few tiles per CTA and some expert needing more than one pass over
    // its rows, deal the heaviest experts' tiles first, in snake order over
    // the CTAs, so that the CTAs' loads even out; otherwise plain round robin.
    // (The order never changes a result.)
    bool ordered = (CW + 1) * 32 >= 256 && MOEDEC_GU4_ORDER && nu <= 256 && tiles <= 32 * (int)gridDim.x;
    if (ordered)  // uniform over the CTA: the map is shared
        ordered = __syncthreads_or((int)threadIdx.x < nu && m.uoff[threadIdx.x + 1] - m.uoff[threadIdx.x] > TC);
    if (ordered) order_experts_by_count(m, nu, sh->perm, reinterpret_cast<uint32_t*>(ring));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int KS = s.k + s.S;
    const int nkt = s.d / GU4_KT;

    if (warp == CW) {
        // ---------------- producer ----------------
        const uint64_t pol = l2_evict_first_policy();
        uint32_t it = 0;  // stages issued so far
        bool ok = true;
        for (int rr = 0; ok; ++rr) {
            const int tile = ordered ? snake_tile(rr) : rr * (int)gridDim.x + (int)blockIdx.x;
            if (tile >= tiles) break;
            const int q = tile / rbs;
            const int u = ordered ? sh->perm[q] : q;
            const int n0 = (tile - q * rbs) * RT;
            const int e = m.uexp[u];
            const int shx = e >= s.E ? 1 : 0;
            const int row0 = (shx ? 0 : e) * s.I + n0;
            const int s0 = m.uoff[u], s1 = m.uoff[u + 1];
            for (int t0 = s0; t0 < s1 && ok; t0 += TC) {
                const int nt = min(TC, s1 - t0);
                const uint16_t* xrow = a.x + (size_t)(lane < nt ? m.hrow[t0 + lane] / KS : 0) * s.d;
                for (int kt = 0; kt < nkt; ++kt, ++it) {
                    const int slot = it % S;
                    if (it >= (uint32_t)S &&
                        !mbar_wait_abort(&sh->empty[slot], ((it / S) - 1) & 1, &sh->abort)) {
                        ok = false;
                        break;
                    }
                    GU4Stage<RT>& st = ring[slot];
                    if (lane == 0) {
                        mbar_arrive_expect_tx(&sh->full[slot], 2 * RT * (GU4_KT + GU4_KT / 32) + nt * GU4_KT * 2);
                        fence_proxy_async();
#pragma unroll
                        for (int p = 0; p < 2; ++p) {
                            if (maps.w3d) {
                                tma_3d(st.w[p][0], &maps.w[shx][p], 0, row0, kt * (GU4_KT / GU4_BOX), &sh->full[slot],
                                       pol);
                            } else {
#pragma unroll
                                for (int b = 0; b < GU4_KT / GU4_BOX; ++b)
                                    tma_2d(st.w[p][b], &maps.w[shx][p], kt * GU4_KT + b * GU4_BOX, row0,
                                           &sh->full[slot], pol);
                            }
                            tma_2d(st.sc[p], &maps.s[shx][p], kt * (GU4_KT / 32), row0, &sh->full[slot], pol);
                        }
                    }
                    __syncwarp();
                    if (lane < nt) {
                        fence_proxy_async();
                        bulk_g2s_keep(st.x[lane], xrow + (size_t)kt * GU4_KT, GU4_KT * 2, &sh->full[slot]);
                    }
                }
            }
        }
        // never leave the CTA with a copy in flight: wait for the last stages
        for (uint32_t j = it > (uint32_t)S ? it - S : 0; j < it; ++j) mbar_wait(&sh->full[j % S], (j / S) & 1);
    } else {
        // ---------------- consumers ----------------
        RingPos rp{0, 0u};
        int grp = 0;
        for (int rr = 0;; ++rr) {
            const int tile = ordered ? snake_tile(rr) : rr * (int)gridDim.x + (int)blockIdx.x;
            if (tile >= tiles) break;
            const int q = tile / rbs;
            const int u = ordered ? sh->perm[q] : q;
            const int n0 = (tile - q * rbs) * RT;
            const int s0 = m.uoff[u], s1 = m.uoff[u + 1];
            for (int t0 = s0; t0 < s1; t0 += TC, ++grp) {
                const int nt = min(TC, s1 - t0);
                const int* hs = m.hrow + t0;
                switch (nt) {
                    case 1: gu4_group<RT, CW, 1>(a, ring, sh, rp, grp, nkt, warp, lane, n0, hs); break;
                    case 2: gu4_group<RT, CW, 2>(a, ring, sh, rp, grp, nkt, warp, lane, n0, hs); break;
                    case 3: gu4_group<RT, CW, 3>(a, ring, sh, rp, grp, nkt, warp, lane, n0, hs); break;
                    default: gu4_group<RT, CW, 4>(a, ring, sh, rp, grp, nkt, warp, lane, n0, hs); break;
                }
            }
        }
    }
    if (lane == 0 && sh->abort) atomicOr(a.err, MOE_DEVERR_TIMEOUT);
}

// ------------------------------------------------------------ down v2 ----
// The CTA owns RT output rows and keeps one FP32 accumulator per (row,
// token) in shared memory.  Its warps split the rows and the distinct
// experts; a lane group of L lanes covers L x 16 bytes of I per step for two
// rows at once (one h load serves both).  Weight chunks stream through a
// per-warp cp.async ring; the first ones are issued before waiting for the
// gate/up pass, since they do not depend on it.  After each (expert, token
// group) a reduce-scatter inside the lane group leaves each (row, token)
// dot in one lane, which adds w * dot to the accumulator.  Needs I % 128 == 0.

constexpr int DN2_STAGES = 4;
constexpr int DN2_R = 2;  // rows per lane

struct DN2Ring {
    uint4 w[DN2_STAGES][DN2_R][32];
    uint32_t s[DN2_STAGES][DN2_R][32];
};

struct DN2Warp {
    int es, ES, nu, nstep, rbase;
};

template <int N, int L>
__device__ __forceinline__ float group_reduce_scatter(float (&v)[N], int li) {
    int o = L / 2;
#pragma unroll
    for (int cnt = N; cnt > 1; cnt >>= 1, o >>= 1) {
        const bool upper = (li & o) != 0;
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

template <int L>
__device__ __forceinline__ void dn2_issue(const DownArgs& a, const RouteMap& m, const DN2Warp& wi,
                                          GU2Cursor& pc, DN2Ring* ring, int slot, int lane,
                                          uint64_t pol) {
    const int u = wi.es + pc.m * wi.ES;
    if (u < wi.nu) {
        const DecodeShape& s = a.s;
        const int e = m.uexp[u];
        const bool sh = e >= s.E;
        const MXView vd = sh ? a.shd : a.wd;
        const size_t eo = sh ? 0 : (size_t)e;
        const int kofs = pc.c * (L * 16) + (lane % L) * 16;
        const int nb = s.I / 32;
        const int sw = ((kofs >> 5) >> 2) << 2;
#pragma unroll
        for (int rr = 0; rr < DN2_R; ++rr) {
            const int row = min(wi.rbase + rr, s.d - 1);
            const size_t r = eo * s.d + row;
            cp_async_16(&ring->w[slot][rr][lane], vd.w + r * s.I + kofs, 16, pol);
            cp_async_4(&ring->s[slot][rr][lane], vd.s + r * nb + sw, 4);
        }
        if (++pc.c == wi.nstep) {
            pc.c = 0;
            if (++pc.g == (m.ucnt[u] + TC - 1) / TC) {
                pc.g = 0;
                ++pc.m;
            }
        }
    }
    cp_async_commit();
}

template <int L, int NT>
__device__ __forceinline__ void dn2_group(const DownArgs& a, const RouteMap& m, const DN2Warp& wi,
                                          GU2Cursor& pc, DN2Ring* ring, int& slot, int lane,
                                          uint64_t pol, const int* hs, const float* ws, int nt,
                                          float* acc_rows, int RT) {
    constexpr int NTP = NT == 3 ? 4 : NT;
    const DecodeShape& s = a.s;
    const int KS = s.k + s.S;
    const int li = lane % L;
    const char* hp[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) hp[t] = reinterpret_cast<const char*>(a.h + (size_t)hs[t] * s.I);
    float2 acc[DN2_R][NT];
#pragma unroll
    for (int r = 0; r < DN2_R; ++r)
#pragma unroll
        for (int t = 0; t < NT; ++t) acc[r][t] = make_float2(0.f, 0.f);
    const int bsh = ((li >> 1) & 3) * 8;

    for (int c = 0; c < wi.nstep; ++c) {
        dn2_issue<L>(a, m, wi, pc, ring, (slot + DN2_STAGES - 1) % DN2_STAGES, lane, pol);
        cp_async_wait<DN2_STAGES - 1>();
        const int kofs = c * (L * 16) + li * 16;
        uint4 wv[DN2_R];
        float sc[DN2_R];
#pragma unroll
        for (int r = 0; r < DN2_R; ++r) {
            wv[r] = ring->w[slot][r][lane];
            sc[r] = e8m0_to_float((ring->s[slot][r][lane] >> bsh) & 0xffu);
        }
        uint4 hv[NT];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            if ((q & 3) == 0) {
#pragma unroll
                for (int t = 0; t < NT; ++t) hv[t] = ld_cached_128(hp[t] + (size_t)kofs * 2 + (q >> 2) * 16);
            }
            float2 wq[DN2_R];
#pragma unroll
            for (int r = 0; r < DN2_R; ++r)
                wq[r] = __fmul2_rn(e4m3x2_to_float2((&wv[r].x)[q >> 1] >> ((q & 1) * 16)),
                                   make_float2(sc[r], sc[r]));
#pragma unroll
            for (int t = 0; t < NT; ++t) {
                const float2 hf = bf16x2_to_float2((&hv[t].x)[q & 3]);
#pragma unroll
                for (int r = 0; r < DN2_R; ++r) acc[r][t] = __ffma2_rn(hf, wq[r], acc[r][t]);
            }
        }
        slot = (slot + 1) % DN2_STAGES;
    }
    constexpr int N = DN2_R * NTP;  // value index = row * NTP + token
    float v[N];
#pragma unroll
    for (int r = 0; r < DN2_R; ++r)
#pragma unroll
        for (int t = 0; t < NTP; ++t)
            v[r * NTP + t] = t < NT ? acc[r][t < NT ? t : 0].x + acc[r][t < NT ? t : 0].y : 0.f;
    const float dot = group_reduce_scatter<N, L>(v, li);
    constexpr int LOGN = N == 2 ? 1 : (N == 4 ? 2 : 3);
    constexpr int LOGL = L == 8 ? 3 : (L == 16 ? 4 : 5);
    const int idx = (li >> (LOGL - LOGN)) & (N - 1);
    const int rr = idx / NTP, t = idx % NTP;
    if ((li & ((1 << (LOGL - LOGN)) - 1)) == 0 && t < nt && wi.rbase + rr < s.d) {
        int hrow = hs[0];
        float wt = ws[0];
#pragma unroll
        for (int tt = 1; tt < NT; ++tt)
            if (tt == t) {
                hrow = hs[tt];
                wt = ws[tt];
            }
        acc_rows[rr * s.B + hrow / KS] += wt * dot;
    }
}

template <int L>
__global__ void __launch_bounds__(DEC_THREADS, 2) down_v2_kernel(DownArgs a) {
    extern __shared__ __align__(16) int smem_i[];
    const DecodeShape s = a.s;
    const RouteMap m = carve_map(smem_i, s, true);
    constexpr int G = 32 / L;
    const int RS = DEC_WARPS / a.es;
    const int RT = RS * G * DN2_R;
    float* acc = reinterpret_cast<float*>(smem_i + map_ints(s, true));
    const int acc_n = DEC_WARPS * G * DN2_R * s.B;  // = ES * RT * B
    DN2Ring* rings = reinterpret_cast<DN2Ring*>(acc + (acc_n + 3) / 4 * 4);
    build_route_map(m, a.ids, a.w, s, a.err, true);
    for (int i = threadIdx.x; i < acc_n; i += DEC_THREADS) acc[i] = 0.f;

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int grp = lane / L;
    const int rs = warp % RS, es = warp / RS;
    DN2Warp wi;
    wi.es = es;
    wi.ES = a.es;
    wi.nu = m.hdr[0];
    wi.nstep = s.I / (L * 16);
    const int rloc = (rs * G + grp) * DN2_R;
    wi.rbase = blockIdx.x * RT + rloc;
    DN2Ring* ring = rings + warp;
    const uint64_t pol = l2_evict_first_policy();
    GU2Cursor pc{0, 0, 0};
    int slot = 0;
    // weight prefetch does not depend on the gate/up pass
#pragma unroll
    for (int i = 0; i < DN2_STAGES - 1; ++i) dn2_issue<L>(a, m, wi, pc, ring, i, lane, pol);
    __syncthreads();
    asm volatile("griddepcontrol.wait;" ::: "memory");

    float* acc_rows = acc + (size_t)(es * RT + rloc) * s.B;
    for (int u = es; u < wi.nu; u += a.es) {
        const int s0 = m.uoff[u], cnt = m.ucnt[u];
        for (int t0 = 0; t0 < cnt; t0 += TC) {
            const int nt = min(TC, cnt - t0);
            const int* hs = m.hrow + s0 + t0;
            const float* ws = m.wt + s0 + t0;
            switch (nt) {
                case 1: dn2_group<L, 1>(a, m, wi, pc, ring, slot, lane, pol, hs, ws, nt, acc_rows, RT); break;
                case 2: dn2_group<L, 2>(a, m, wi, pc, ring, slot, lane, pol, hs, ws, nt, acc_rows, RT); break;
                case 3: dn2_group<L, 3>(a, m, wi, pc, ring, slot, lane, pol, hs, ws, nt, acc_rows, RT); break;
                default: dn2_group<L, 4>(a, m, wi, pc, ring, slot, lane, pol, hs, ws, nt, acc_rows, RT); break;
            }
        }
    }
    cp_async_wait<0>();
    __syncthreads();
    for (int i = threadIdx.x; i < RT * s.B; i += DEC_THREADS) {
        const int r = i % RT, b = i / RT;
        const int oo = blockIdx.x * RT + r;
        if (oo < s.d) {
            float sum = 0.f;
            for (int q = 0; q < a.es; ++q) sum += acc[(size_t)(q * RT + r) * s.B + b];
            a.y[(size_t)b * s.d + oo] = __bfloat16_as_ushort(__float2bfloat16_rn(sum));
        }
    }
}

// ------------------------------------------------------------ down v3 ----
// Warp-specialised like gate/up v3.  A CTA owns DN3_RT = 8 output rows; the
// stages are the (distinct expert, group of up to TC tokens) pairs in order,
// and stage j holds the expert's contiguous [8 rows x I] block of Wd, its
// scale block and the tokens' h rows, brought in by three kinds of 1D bulk
// copies (the weight copies of the first stages go out before waiting for
// the gate/up pass).  Eight consumer warps form RW expert splits of 8/RW
// warps; split j % RW takes stage j, each of its warps owning RW rows (one h
// load serves RW rows), lanes taking 8-byte K chunks (eight E4M3 codes in
// one scale block, whose partial sums are scaled once).  Each split has its
// own ring slots, so every barrier phase is consumed in order.  After each
// stage a reduce-scatter leaves each (row, token) dot in one lane, which adds
// w * dot to the split's FP32 accumulator in shared memory; the splits are
// added in a fixed order at the end.  Needs I % 256 == 0.

constexpr int DN3_CW = 8;                       // consumer warps
constexpr int DN3_THREADS = (DN3_CW + 1) * 32;  // + producer warp
constexpr int DN3_RT = 8;                       // rows per CTA
constexpr int DN3_SMAX = 8;                     // ring slots (all splits)
#ifndef MOEDEC_DN3_RING
#define MOEDEC_DN3_RING (80 * 1024)
#endif
#ifndef MOEDEC_DN3_MINS
#define MOEDEC_DN3_MINS 1
#endif
constexpr int DN3_RING_BYTES = MOEDEC_DN3_RING;  // two CTAs per SM

struct DN3Layout {
    int stage_bytes, w_off, s_off, h_off, S;  // S = slots per split
};

__host__ __device__ inline DN3Layout dn3_layout(const DecodeShape& s, int RW) {
    DN3Layout L;
    L.w_off = 0;
    L.s_off = DN3_RT * s.I;  // multiple of 16
    L.h_off = (L.s_off + DN3_RT * (s.I / 32) + 127) / 128 * 128;
    L.stage_bytes = (L.h_off + TC * s.I * 2 + 127) / 128 * 128;
    int S = DN3_RING_BYTES / (RW * L.stage_bytes);
    const int smax = DN3_SMAX / RW;
    L.S = S > smax ? smax : S;  // >= 2 is checked by the launcher
    return L;
}

__host__ __device__ inline size_t dn3_smem_offset(const DecodeShape& s, int RW) {
    const size_t acc = (size_t)RW * DN3_RT * s.B * 4;
    return (map_ints(s, true) * 4 + acc + 127) / 128 * 128;
}

// Rows per warp (= expert splits) for a given I: at least ~48 weight bytes
// per lane per stage, and at least two ring slots per split.
#ifndef MOEDEC_DN3_RWSMALL
#define MOEDEC_DN3_RWSMALL 4
#endif
__host__ __device__ inline int dn3_rw(int I) { return I >= 2048 ? 1 : MOEDEC_DN3_RWSMALL; }

template <int RW, int NT, int NCH = 0>
__device__ __forceinline__ bool dn3_group(const DownArgs& a, const DN3Layout& L, const char* st, uint64_t* full,
                                          uint64_t* empty, uint32_t parity, int cw, int lane, const int* toks,
                                          const float* ws, int nt, float* acc_rows) {
    constexpr int NTP = NT == 3 ? 4 : NT;
    const DecodeShape& s = a.s;
    if (!mbar_wait(full, parity)) return false;
    const uint8_t* wb = reinterpret_cast<const uint8_t*>(st + L.w_off) + (size_t)cw * RW * s.I;
    const uint8_t* sb = reinterpret_cast<const uint8_t*>(st + L.s_off) + cw * RW * (s.I / 32);
    const uint16_t* hb = reinterpret_cast<const uint16_t*>(st + L.h_off);
    float2 acc[RW][NT];
#pragma unroll
    for (int r = 0; r < RW; ++r)
#pragma unroll
        for (int t = 0; t < NT; ++t) acc[r][t] = make_float2(0.f, 0.f);
    const int nch = NCH ? NCH : s.I / 256;  // 8-byte chunks per lane
#pragma unroll(NCH ? NCH : 1)
    for (int i = 0; i < nch; ++i) {
        const int k0 = (lane + 32 * i) * 8;  // first K element of this chunk
        float2 hf[NT][4];  // the tokens' eight activations, converted once for all rows
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            const uint4 hv = *reinterpret_cast<const uint4*>(hb + (size_t)t * s.I + k0);
#pragma unroll
            for (int q = 0; q < 4; ++q) hf[t][q] = bf16x2_to_float2((&hv.x)[q]);
        }
#pragma unroll
        for (int r = 0; r < RW; ++r) {
            const uint2 wv = *reinterpret_cast<const uint2*>(wb + (size_t)r * s.I + k0);
            const float sc = e8m0_to_float(sb[r * (s.I / 32) + (k0 >> 5)]);
            float2 wq[4];
            e4m3x4_to_float(wv.x, wq[0], wq[1]);
            e4m3x4_to_float(wv.y, wq[2], wq[3]);
            // the chunk lies inside one scale block: scale its partial sum once
#pragma unroll
            for (int t = 0; t < NT; ++t) {
                float2 part = __fmul2_rn(hf[t][0], wq[0]);
#pragma unroll
                for (int q = 1; q < 4; ++q) part = __ffma2_rn(hf[t][q], wq[q], part);
                acc[r][t] = __ffma2_rn(part, make_float2(sc, sc), acc[r][t]);
            }
        }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty);

    constexpr int N = RW * NTP;  // value index = row * NTP + token
    float v[N];
#pragma unroll
    for (int r = 0; r < RW; ++r)
#pragma unroll
        for (int t = 0; t < NTP; ++t)
            v[r * NTP + t] = t < NT ? acc[r][t < NT ? t : 0].x + acc[r][t < NT ? t : 0].y : 0.f;
    const float dot = warp_reduce_scatter<N>(v, lane);
    constexpr int LOGN = N == 1 ? 0 : (N == 2 ? 1 : (N == 4 ? 2 : (N == 8 ? 3 : 4)));
    const int idx = (lane >> (5 - LOGN)) & (N - 1);
    const int rr = idx / NTP, t = idx % NTP;
    if ((lane & ((1 << (5 - LOGN)) - 1)) == 0 && t < nt) {
        int b = toks[0];
        float wt = ws[0];
#pragma unroll
        for (int tt = 1; tt < NT; ++tt)
            if (tt == t) {
                b = toks[tt];
                wt = ws[tt];
            }
        acc_rows[rr * s.B + b] += wt * dot;
    }
    return true;
}

template <int RW>
__global__ void __launch_bounds__(DN3_THREADS, 2) down_v3_kernel(DownArgs a) {
    constexpr int ES = RW;              // expert splits
    constexpr int SW = DN3_CW / ES;     // warps per split
    static_assert(SW * RW == DN3_RT, "8 rows per CTA");
    extern __shared__ __align__(128) int smem_i[];
    const DecodeShape s = a.s;
    const RouteMap m = carve_map(smem_i, s, true);
    float* acc = reinterpret_cast<float*>(smem_i + map_ints(s, true));  // [ES][DN3_RT][B]
    const uintptr_t raw = reinterpret_cast<uintptr_t>(smem_i) + dn3_smem_offset(s, RW);
    char* ring = reinterpret_cast<char*>((raw + 127) & ~uintptr_t(127));
    const DN3Layout L = dn3_layout(s, RW);
    // slot (split h, k) = h * L.S + k
    uint64_t* full = reinterpret_cast<uint64_t*>(ring + (size_t)ES * L.S * L.stage_bytes);
    uint64_t* empty = full + DN3_SMAX;
    if (threadIdx.x == 0) {
        for (int i = 0; i < ES * L.S; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], SW);
        }
        mbar_init_fence();
    }
    build_route_map(m, a.ids, a.w, s, a.err, true);  // ends with __syncthreads

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int o0 = blockIdx.x * DN3_RT;
    const int nu = m.hdr[0];
    bool ok = true;

    if (warp == DN3_CW) {
        // ---------------- producer ----------------
        const uint64_t pol = l2_evict_first_policy();
        const int nb = s.I / 32;
        const uint32_t wbytes = DN3_RT * s.I, sbytes = DN3_RT * nb;
        // stage j -> split j % ES, its n = j / ES-th stage, slot n % S, use n / S
        auto slot_of = [&](uint32_t j) { return (int)((j % ES) * L.S + (j / ES) % L.S); };
        auto issue_w = [&](int u, int t0, uint32_t j) {
            const int nt = min(TC, m.ucnt[u] - t0);
            const int e = m.uexp[u];
            const bool sh = e >= s.E;
            const MXView vd = sh ? a.shd : a.wd;
            const size_t r0 = (sh ? 0 : (size_t)e) * s.d + o0;
            const int slot = slot_of(j);
            char* st = ring + (size_t)slot * L.stage_bytes;
            if (lane == 0) {
                mbar_arrive_expect_tx(&full[slot], wbytes + sbytes + nt * s.I * 2);
                fence_proxy_async();
                bulk_g2s(st + L.w_off, vd.w + r0 * s.I, wbytes, &full[slot], pol);
                bulk_g2s(st + L.s_off, vd.s + r0 * nb, sbytes, &full[slot], pol);
            }
        };
        auto issue_h = [&](int u, int t0, uint32_t j) {
            const int nt = min(TC, m.ucnt[u] - t0);
            const int slot = slot_of(j);
            char* st = ring + (size_t)slot * L.stage_bytes;
            if (lane < nt) {
                fence_proxy_async();
                bulk_g2s_keep(st + L.h_off + (size_t)lane * s.I * 2,
                              a.h + (size_t)m.hrow[m.uoff[u] + t0 + lane] * s.I, s.I * 2, &full[slot]);
            }
        };
        auto advance = [&](int& u, int& t0) {
            t0 += TC;
            if (t0 >= m.ucnt[u]) {
                t0 = 0;
                ++u;
            }
        };
        // the first ES * S stages fill fresh slots; their weights do not
        // depend on the gate/up pass
        int pu = 0, pt = 0;
        uint32_t j = 0;
        for (; j < (uint32_t)(ES * L.S) && pu < nu; ++j) {
            issue_w(pu, pt, j);
            advance(pu, pt);
        }
        asm volatile("griddepcontrol.wait;" ::: "memory");
        int hu = 0, ht = 0;
        for (uint32_t i = 0; i < j; ++i) {
            issue_h(hu, ht, i);
            advance(hu, ht);
        }
        for (; pu < nu; ++j) {
            const uint32_t n = j / ES;
            if (!mbar_wait(&empty[slot_of(j)], ((n / L.S) - 1) & 1)) {
                ok = false;
                break;
            }
            issue_w(pu, pt, j);
            __syncwarp();
            issue_h(pu, pt, j);
            advance(pu, pt);
        }
        // never leave the CTA with a copy in flight
        for (uint32_t i = j > (uint32_t)(ES * L.S) ? j - ES * L.S : 0; i < j; ++i)
            mbar_wait(&full[slot_of(i)], ((i / ES) / L.S) & 1);
    } else {
        // ---------------- consumers ----------------
        const int split = warp / SW, cw = warp % SW;
        float* acc_rows = acc + (size_t)(split * DN3_RT + cw * RW) * s.B;
        for (int i = lane; i < RW * s.B; i += 32) acc_rows[i] = 0.f;
        __syncwarp();
        uint32_t j0 = 0;  // global index of u's first stage
        int k = 0;        // ring slot of this split's next stage
        uint32_t par = 0; // its phase parity
        for (int u = 0; u < nu && ok; ++u) {
            const int cnt = m.ucnt[u], s0 = m.uoff[u];
            const int groups = (cnt + TC - 1) / TC;
            // u's stages are j0 .. j0 + groups - 1; this split takes j % ES == split
            for (int g = (split - (int)(j0 % ES) + ES) % ES; g < groups && ok; g += ES) {
                const int t0 = g * TC;
                const int nt = min(TC, cnt - t0);
                const int slot = split * L.S + k;
                const char* st = ring + (size_t)slot * L.stage_bytes;
                const int* tk = m.tok + s0 + t0;
                const float* wsp = m.wt + s0 + t0;
                switch (nt) {
                    case 1: ok = dn3_group<RW, 1>(a, L, st, &full[slot], &empty[slot], par, cw, lane, tk, wsp, nt, acc_rows); break;
                    case 2: ok = dn3_group<RW, 2>(a, L, st, &full[slot], &empty[slot], par, cw, lane, tk, wsp, nt, acc_rows); break;
                    case 3: ok = dn3_group<RW, 3>(a, L, st, &full[slot], &empty[slot], par, cw, lane, tk, wsp, nt, acc_rows); break;
                    default: ok = dn3_group<RW, 4>(a, L, st, &full[slot], &empty[slot], par, cw, lane, tk, wsp, nt, acc_rows); break;
                }
                if (++k == L.S) {
                    k = 0;
                    par ^= 1;
                }
            }
            j0 += groups;
        }
    }
    // add the expert splits in a fixed order and round once to BF16
    __syncthreads();
    for (int i = threadIdx.x; i < DN3_RT * s.B; i += blockDim.x) {
        const int r = i / s.B, b = i - r * s.B;
        float sum = 0.f;
#pragma unroll
        for (int q = 0; q < ES; ++q) sum += acc[(size_t)q * DN3_RT * s.B + i];
        a.y[(size_t)b * s.d + o0 + r] = __bfloat16_as_ushort(__float2bfloat16_rn(sum));
    }
    if (!ok && lane == 0) atomicOr(a.err, MOE_DEVERR_TIMEOUT);
}

// ------------------------------------------------------------ down v4 ----
// Like down v3, but every consumer warp takes every stage, in order (one
// ring, so no barrier phase is ever skipped), each warp owning RW rows of a
// block of RT = 8 * RW output rows; and a thread-block cluster of CL CTAs
// shares one row block, CTA rank r taking the distinct experts u with
// u % CL == r.  At the end the CL partial accumulators are added through
// distributed shared memory, in rank order, each CTA rounding and storing
// RT / CL of the rows.  Larger blocks mean bigger bulk copies and fewer h
// reads; the cluster split keeps enough CTAs.

constexpr int DN4_SMAX = 8;
constexpr int DN4_RING_BYTES = 96 * 1024;  // two CTAs per SM

__host__ __device__ inline DN3Layout dn4_layout(const DecodeShape& s, int RT) {
    DN3Layout L;
    L.w_off = 0;
    L.s_off = RT * s.I;
    L.h_off = (L.s_off + RT * (s.I / 32) + 127) / 128 * 128;
    L.stage_bytes = (L.h_off + TC * s.I * 2 + 127) / 128 * 128;
    const int S = DN4_RING_BYTES / L.stage_bytes;
    L.S = S > DN4_SMAX ? DN4_SMAX : S;
    return L;
}

__host__ __device__ inline size_t dn4_smem_offset(const DecodeShape& s, int RT) {
    const size_t acc = (size_t)RT * s.B * 4;
    return (map_ints(s, true) * 4 + acc + 127) / 128 * 128;
}

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ float ld_cluster_f32(const float* local, uint32_t rank) {
    uint32_t ra;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(smem_addr(local)), "r"(rank));
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(ra) : "memory");
    return v;
}

template <int RW, int CL, int NCH, int CW>
__global__ void __launch_bounds__((CW + 1) * 32, 2) down_v4_kernel(DownArgs a) {
    constexpr int RT = CW * RW;
    extern __shared__ __align__(128) int smem_i[];
    const DecodeShape s = a.s;
    const RouteMap m = carve_map(smem_i, s, true);
    float* acc = reinterpret_cast<float*>(smem_i + map_ints(s, true));  // [RT][B]
    const uintptr_t raw = reinterpret_cast<uintptr_t>(smem_i) + dn4_smem_offset(s, RT);
    char* ring = reinterpret_cast<char*>((raw + 127) & ~uintptr_t(127));
    const DN3Layout L = dn4_layout(s, RT);
    uint64_t* full = reinterpret_cast<uint64_t*>(ring + (size_t)L.S * L.stage_bytes);
    uint64_t* empty = full + DN4_SMAX;
    if (threadIdx.x == 0) {
        for (int i = 0; i < L.S; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], CW);
        }
        mbar_init_fence();
    }
    // the copy ring is idle until the map is built: it serves as the map's scratch
    build_route_map(m, a.ids, a.w, s, a.err, true, reinterpret_cast<int*>(ring),
                    L.S * L.stage_bytes / 4);  // ends with __syncthreads

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rank = CL > 1 ? (int)cluster_rank() : 0;
    const int o0 = (blockIdx.x / CL) * RT;
    const int rows = min(RT, s.d - o0);  // the last block may be partial (rows is even)
    const int nu = m.hdr[0];
    bool ok = true;

    if (warp == CW) {
        // ---------------- producer ----------------
        const uint64_t pol = l2_evict_first_policy();
        const int nb = s.I / 32;
        const uint32_t wbytes = rows * s.I, sbytes = rows * nb;
        auto issue_w = [&](int u, int t0, int slot) {
            const int nt = min(TC, m.ucnt[u] - t0);
            const int e = m.uexp[u];
            const bool sh = e >= s.E;
            const MXView vd = sh ? a.shd : a.wd;
            const size_t r0 = (sh ? 0 : (size_t)e) * s.d + o0;
            char* st = ring + (size_t)slot * L.stage_bytes;
            if (lane == 0) {
                mbar_arrive_expect_tx(&full[slot], wbytes + sbytes + nt * s.I * 2);
                fence_proxy_async();
                bulk_g2s(st + L.w_off, vd.w + r0 * s.I, wbytes, &full[slot], pol);
                bulk_g2s(st + L.s_off, vd.s + r0 * nb, sbytes, &full[slot], pol);
            }
        };
        auto issue_h = [&](int u, int t0, int slot) {
            const int nt = min(TC, m.ucnt[u] - t0);
            char* st = ring + (size_t)slot * L.stage_bytes;
            if (lane < nt) {
                fence_proxy_async();
                bulk_g2s_keep(st + L.h_off + (size_t)lane * s.I * 2,
                              a.h + (size_t)m.hrow[m.uoff[u] + t0 + lane] * s.I, s.I * 2, &full[slot]);
            }
        };
        // this CTA's stages: experts u = rank, rank + CL, ..., each in groups of TC tokens
        auto advance = [&](int& u, int& t0) {
            t0 += TC;
            if (t0 >= m.ucnt[u]) {
                t0 = 0;
                u += CL;
            }
        };
        int pu = rank, pt = 0, npro = 0;
        for (; npro < L.S && pu < nu; ++npro) {
            issue_w(pu, pt, npro);
            advance(pu, pt);
        }
        asm volatile("griddepcontrol.wait;" ::: "memory");
        {
            int hu = rank, ht = 0;
            for (int i = 0; i < npro; ++i) {
                issue_h(hu, ht, i);
                advance(hu, ht);
            }
        }
        uint32_t j = npro;
        int slot = npro % L.S;
        uint32_t par = 0;  // parity of the empty phase to wait for at `slot`
        if (npro == L.S) slot = 0;
        while (pu < nu) {
            if (!mbar_wait(&empty[slot], par)) {
                ok = false;
                break;
            }
            issue_w(pu, pt, slot);
            __syncwarp();
            issue_h(pu, pt, slot);
            advance(pu, pt);
            ++j;
            if (++slot == L.S) {
                slot = 0;
                par ^= 1;
            }
        }
        for (uint32_t i = j > (uint32_t)L.S ? j - L.S : 0; i < j; ++i) mbar_wait(&full[i % L.S], (i / L.S) & 1);
    } else {
        // ---------------- consumers ----------------
        float* acc_rows = acc + (size_t)(warp * RW) * s.B;
        for (int i = lane; i < RW * s.B; i += 32) acc_rows[i] = 0.f;
        __syncwarp();
        int slot = 0;
        uint32_t par = 0;
        for (int u = rank; u < nu && ok; u += CL) {
            const int cnt = m.ucnt[u], s0 = m.uoff[u];
            for (int t0 = 0; t0 < cnt && ok; t0 += TC) {
                const int nt = min(TC, cnt - t0);
                const char* st = ring + (size_t)slot * L.stage_bytes;
                const int* tk = m.tok + s0 + t0;
                const float* wsp = m.wt + s0 + t0;
                switch (nt) {
                    case 1: ok = dn3_group<RW, 1, NCH>(a, L, st, &full[slot], &empty[slot], par, warp, lane, tk, wsp, nt, acc_rows); break;
                    case 2: ok = dn3_group<RW, 2, NCH>(a, L, st, &full[slot], &empty[slot], par, warp, lane, tk, wsp, nt, acc_rows); break;
                    case 3: ok = dn3_group<RW, 3, NCH>(a, L, st, &full[slot], &empty[slot], par, warp, lane, tk, wsp, nt, acc_rows); break;
                    default: ok = dn3_group<RW, 4, NCH>(a, L, st, &full[slot], &empty[slot], par, warp, lane, tk, wsp, nt, acc_rows); break;
                }
                if (++slot == L.S) {
                    slot = 0;
                    par ^= 1;
                }
            }
        }
    }
    // add the cluster's partial sums in rank order; CTA `rank` stores rows
    // [rank * RT / CL, (rank + 1) * RT / CL) of the block
    __syncthreads();
    if (CL > 1) cluster_sync_all();
    constexpr int RR = RT / CL;
    for (int i = threadIdx.x; i < RR * s.B; i += blockDim.x) {
        const int rl = rank * RR + i / s.B, b = i % s.B;
        const float* p = acc + (size_t)rl * s.B + b;
        float sum = 0.f;
#pragma unroll
        for (int q = 0; q < CL; ++q) sum += CL > 1 ? ld_cluster_f32(p, q) : *p;
        if (rl < rows) a.y[(size_t)b * s.d + o0 + rl] = __bfloat16_as_ushort(__float2bfloat16_rn(sum));
    }
    if (CL > 1) cluster_sync_all();  // keep this CTA's accumulators alive for its peers
    if (!ok && lane == 0) atomicOr(a.err, MOE_DEVERR_TIMEOUT);
}

// ------------------------------------------------------------ down v5 ----
// Lane per output row.  A CTA owns a block of RT <= 16 output rows; the
// stages are (distinct expert, group of up to TC tokens, K slab of KSLAB
// elements) in order, each holding the expert's RT x KSLAB code block of
// W_down as 128-byte tensor boxes in the 128-byte swizzled layout, its
// scale bytes, and the tokens' KSLAB-long slices of h.  The eight consumer
// warps split each slab evenly (warp w takes its w-th eighth), and in a
// warp the two lanes r and r + 16 share row r, each taking half of the
// warp's 16-byte chunks: a lane dequantises its chunk of its row, takes
// the tokens' h values of that chunk from a per-warp FP32 copy (converted
// once per stage) as broadcasts, and scales each chunk's partial sum once.
// After an expert's last slab the two lanes of a row add their halves by a
// shuffle and the row's lane adds w * dot into the warp's own FP32 partial
// outputs [token][row] in shared memory, in stage order.  When the block is
// done the eight warps' partials are added in a fixed order (and, for a
// two-CTA cluster that splits the experts, the two CTAs' sums in rank
// order through distributed shared memory) and rounded once to BF16.  With
// CL = 1 a CTA may own several row blocks in turn.  Every wait is bounded;
// a wait that runs out raises a CTA-wide abort flag so that all warps still
// pass every barrier.

constexpr int DN5_CW = 8;
constexpr int DN5_THREADS = (DN5_CW + 1) * 32;
constexpr int DN5_RTMAX = 16;
constexpr int DN5_SMAX = 6;

struct DN5Maps {
    CUtensorMap w[2];  // [routed / shared]: 3D block view, box 128 B x RT rows x KSLAB / 128 blocks, 128-byte swizzle
    CUtensorMap s[2];  // scales, box RT rows x 16 B (used when the slab is shorter than I)
};

struct DN5Params {
    int RT;           // rows per block (even, <= 16)
    int KSLAB;        // K elements per stage: I itself (<= 768) or 512
    int S;            // ring stages
    int nblk;         // row blocks
    int scale2d;      // 1: scales by a 2D tensor copy (KSLAB = 512 < I); 0: one 1D copy (KSLAB = I)
    int stage_bytes;  // stage layout: weights at 0 (KSLAB / 128 box slots of 2 KB), scales, h
    int sc_off, h_off;
};

template <int KSLAB, int NT>
__device__ __forceinline__ void dn5_group(const DN5Params& P, const char* ring, uint64_t* full, uint64_t* empty,
                                          int* abortf, RingPos& rp, int nslab, int warp, int lane, float* xf,
                                          float* yp, const int* tok, const float* wt, int rows) {
    constexpr int KW = KSLAB / 8;     // K elements of a warp per stage
    constexpr int CPL = KSLAB / 256;  // 16-byte chunks of a lane per stage
    const int r = lane & 15, hb = lane >> 4;
    const int RT = P.RT;
    float2 acc[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) acc[t] = make_float2(0.f, 0.f);
    for (int sl = 0; sl < nslab; ++sl, rp.next(P.S)) {
        if (!mbar_wait_abort(&full[rp.slot], rp.par, abortf)) continue;
        const char* st = ring + (size_t)rp.slot * P.stage_bytes;
        {  // this warp's part of the tokens' h -> FP32: lane = (token, KW / 8 elements)
            const uint16_t* hst = reinterpret_cast<const uint16_t*>(st + P.h_off);
            const int t = lane >> 3, k = (lane & 7) * (KW / 8);
            if (t < NT) {
#pragma unroll
                for (int q = 0; q < KW / 32; ++q) {
                    const uint2 hv = *reinterpret_cast<const uint2*>(hst + t * KSLAB + warp * KW + k + 4 * q);
                    const float2 lo = bf16x2_to_float2(hv.x), hi = bf16x2_to_float2(hv.y);
                    *reinterpret_cast<float4*>(xf + t * KW + k + 4 * q) = make_float4(lo.x, lo.y, hi.x, hi.y);
                }
            }
        }
        __syncwarp();
        const uint8_t* scs = reinterpret_cast<const uint8_t*>(st + P.sc_off) + r * (KSLAB / 32);
        const int c0 = warp * (KSLAB / 128) + hb * CPL;  // this lane's first chunk in the slab
#pragma unroll
        for (int q = 0; q < CPL; ++q) {
            // the slab's 128-byte column blocks are consecutive [RT][128] tiles in
            // the 128-byte swizzled layout: chunk j of tile row y sits at chunk
            // j ^ (y & 7), y counted from the (1024-byte aligned) stage start
            const int c = c0 + q;
            const int y = (c >> 3) * RT + r;
            const uint4 wv = *reinterpret_cast<const uint4*>(st + y * 128 + (((c & 7) ^ (y & 7)) << 4));
            const float sc = e8m0_to_float(scs[c >> 1]);
            const float* xl = xf + (hb * CPL + q) * 16;
            float2 part[NT];
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                float2 wq[2];
                e4m3x4_to_float((&wv.x)[q4], wq[0], wq[1]);
#pragma unroll
                for (int t = 0; t < NT; ++t) {
                    const float4 xv = *reinterpret_cast<const float4*>(xl + t * KW + q4 * 4);
                    if (q4 == 0)
                        part[t] = __fmul2_rn(make_float2(xv.x, xv.y), wq[0]);
                    else
                        part[t] = __ffma2_rn(make_float2(xv.x, xv.y), wq[0], part[t]);
                    part[t] = __ffma2_rn(make_float2(xv.z, xv.w), wq[1], part[t]);
                }
            }
#pragma unroll
            for (int t = 0; t < NT; ++t) acc[t] = __ffma2_rn(part[t], make_float2(sc, sc), acc[t]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[rp.slot]);
    }
    // the expert's dots (lower half of K first) times the routing weights
    // into this warp's partial outputs
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        float v = acc[t].x + acc[t].y;
        const float o = __shfl_xor_sync(FULL_MASK, v, 16);
        v = hb ? o + v : v + o;
        if (hb == 0 && r < rows) yp[tok[t] * DN5_RTMAX + r] += wt[t] * v;
    }
}

template <int CL, int KSLAB>
__global__ void __launch_bounds__(DN5_THREADS, 2)
    down_v5_kernel(DownArgs a, const __grid_constant__ DN5Maps maps, const DN5Params P) {
    extern __shared__ __align__(128) int smem_i[];
    const DecodeShape s = a.s;
    const RouteMap m = carve_map(smem_i, s, true);
    const uintptr_t raw = reinterpret_cast<uintptr_t>(smem_i) + map_ints(s, true) * 4;
    char* ring = reinterpret_cast<char*>((raw + 1023) & ~uintptr_t(1023));
    const int S = P.S, RT = P.RT;
    float* xfa = reinterpret_cast<float*>(ring + (size_t)S * P.stage_bytes);  // [CW][TC][KSLAB / 8]
    float* ypa = xfa + DN5_CW * TC * (KSLAB / 8);                               // [CW][B][RTMAX]
    uint64_t* full = reinterpret_cast<uint64_t*>(ypa + (size_t)DN5_CW * s.B * DN5_RTMAX);
    uint64_t* empty = full + S;
    int* abortf = reinterpret_cast<int*>(empty + S);
    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], DN5_CW);
        }
        *abortf = 0;
        mbar_init_fence();
    }
    // the copy ring is idle until the map is built: it serves as the map's scratch
    build_route_map(m, a.ids, a.w, s, a.err, true, reinterpret_cast<int*>(ring),
                    S * P.stage_bytes / 4);  // ends with __syncthreads

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rank = CL > 1 ? (int)cluster_rank() : 0;
    const int nu = m.hdr[0];
    const int nslab = s.I / KSLAB;
    const int cl_idx = blockIdx.x / CL;
    const int step = CL > 1 ? P.nblk : (int)gridDim.x;  // row blocks advance (CL > 1: one block)

    if (warp == DN5_CW) {
        // ---------------- producer ----------------
        const uint64_t pol = l2_evict_first_policy();
        struct Cur {
            int rb, u, g0, sl;
        };
        auto settle = [&](Cur& c) {  // skip row blocks with no expert for this rank
            while (c.rb < P.nblk && c.u >= nu) {
                c.rb += step;
                c.u = rank;
            }
        };
        auto advance = [&](Cur& c) {
            if (++c.sl < nslab) return;
            c.sl = 0;
            c.g0 += TC;
            if (c.g0 < m.ucnt[c.u]) return;
            c.g0 = 0;
            c.u += CL;
            if (c.u >= nu) {
                c.rb += step;
                c.u = rank;
            }
            settle(c);
        };
        auto issue_w = [&](const Cur& c, int slot) {
            const int e = m.uexp[c.u];
            const int shx = e >= s.E ? 1 : 0;
            const int o0 = c.rb * RT, rows = min(RT, s.d - o0);
            const int row0 = (shx ? 0 : e) * s.d + o0;
            const int nt = min(TC, m.ucnt[c.u] - c.g0);
            char* st = ring + (size_t)slot * P.stage_bytes;
            if (lane == 0) {
                const uint32_t sbytes = P.scale2d ? (uint32_t)RT * 16 : (uint32_t)rows * (s.I / 32);
                mbar_arrive_expect_tx(&full[slot], (uint32_t)RT * KSLAB + sbytes + nt * KSLAB * 2);
                fence_proxy_async();
                tma_3d(st, &maps.w[shx], 0, row0, c.sl * (KSLAB / 128), &full[slot], pol);
                if (P.scale2d)
                    tma_2d(st + P.sc_off, &maps.s[shx], c.sl * (KSLAB / 32), row0, &full[slot], pol);
                else
                    bulk_g2s(st + P.sc_off, (shx ? a.shd.s : a.wd.s) + (size_t)row0 * (s.I / 32), sbytes, &full[slot],
                             pol);
            }
        };
        auto issue_h = [&](const Cur& c, int slot) {
            const int nt = min(TC, m.ucnt[c.u] - c.g0);
            char* st = ring + (size_t)slot * P.stage_bytes;
            if (lane < nt) {
                fence_proxy_async();
                bulk_g2s_keep(st + P.h_off + (size_t)lane * KSLAB * 2,
                              a.h + (size_t)m.hrow[m.uoff[c.u] + c.g0 + lane] * s.I + (size_t)c.sl * KSLAB,
                              KSLAB * 2, &full[slot]);
            }
        };
        // the weights of the first S stages go out before waiting for the
        // gate/up pass (they do not depend on it), their h after
        Cur pw{cl_idx, rank, 0, 0};
        settle(pw);
        int npro = 0;
        for (; npro < S && pw.rb < P.nblk; ++npro) {
            issue_w(pw, npro);
            advance(pw);
        }
        asm volatile("griddepcontrol.wait;" ::: "memory");
        {
            Cur ph{cl_idx, rank, 0, 0};
            settle(ph);
            for (int i = 0; i < npro; ++i) {
                issue_h(ph, i);
                advance(ph);
            }
        }
        uint32_t issued = npro;
        RingPos rp{0, 0u};  // reached only when npro == S
        while (pw.rb < P.nblk) {
            if (!mbar_wait_abort(&empty[rp.slot], rp.par, abortf)) break;
            issue_w(pw, rp.slot);
            __syncwarp();
            issue_h(pw, rp.slot);
            advance(pw);
            ++issued;
            rp.next(S);
        }
        // never leave the CTA with a copy in flight
        for (uint32_t j = issued > (uint32_t)S ? issued - S : 0; j < issued; ++j)
            mbar_wait(&full[j % S], (j / S) & 1);
    } else {
        // ---------------- consumers ----------------
        float* yp = ypa + (size_t)warp * s.B * DN5_RTMAX;
        float* xf = xfa + warp * TC * (KSLAB / 8);
        RingPos rp{0, 0u};
        for (int rb = cl_idx; rb < P.nblk; rb += step) {
            const int o0 = rb * RT, rows = min(RT, s.d - o0);
            for (int i = lane; i < s.B * DN5_RTMAX; i += 32) yp[i] = 0.f;
            __syncwarp();
            for (int u = rank; u < nu; u += CL) {
                const int cnt = m.ucnt[u], s0 = m.uoff[u];
                for (int g0 = 0; g0 < cnt; g0 += TC) {
                    const int nt = min(TC, cnt - g0);
                    const int* tk = m.tok + s0 + g0;
                    const float* wsp = m.wt + s0 + g0;
                    switch (nt) {
                        case 1: dn5_group<KSLAB, 1>(P, ring, full, empty, abortf, rp, nslab, warp, lane, xf, yp, tk, wsp, rows); break;
                        case 2: dn5_group<KSLAB, 2>(P, ring, full, empty, abortf, rp, nslab, warp, lane, xf, yp, tk, wsp, rows); break;
                        case 3: dn5_group<KSLAB, 3>(P, ring, full, empty, abortf, rp, nslab, warp, lane, xf, yp, tk, wsp, rows); break;
                        default: dn5_group<KSLAB, 4>(P, ring, full, empty, abortf, rp, nslab, warp, lane, xf, yp, tk, wsp, rows); break;
                    }
                }
            }
            if (CL == 1) {
                // add the warps' partials in a fixed order, round once to BF16
                consumer_sync<DN5_CW * 32>();
                for (int i = threadIdx.x; i < s.B * RT; i += DN5_CW * 32) {
                    const int b = i / RT, rr = i - b * RT;
                    if (rr < rows) {
                        float v = 0.f;
#pragma unroll
                        for (int w = 0; w < DN5_CW; ++w) v += ypa[((size_t)w * s.B + b) * DN5_RTMAX + rr];
                        a.y[(size_t)b * s.d + o0 + rr] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
                    }
                }
                consumer_sync<DN5_CW * 32>();
            }
        }
    }
    if (CL > 1) {
        // one row block per cluster: the warps' partials, then the ranks' sums
        // in rank order; CTA `rank` stores rows [rank * RT / CL, (rank + 1) * RT / CL)
        __syncthreads();
        const int o0 = cl_idx * RT, rows = min(RT, s.d - o0);
        for (int i = threadIdx.x; i < s.B * DN5_RTMAX; i += DN5_THREADS) {
            float v = 0.f;
#pragma unroll
            for (int w = 0; w < DN5_CW; ++w) v += ypa[(size_t)w * s.B * DN5_RTMAX + i];
            ypa[i] = v;
        }
        cluster_sync_all();
        const int RR = RT / CL;
        for (int i = threadIdx.x; i < s.B * RR; i += DN5_THREADS) {
            const int b = i / RR, rl = rank * RR + (i - b * RR);
            if (rl < rows) {
                const float* p = ypa + (size_t)b * DN5_RTMAX + rl;
                float v = 0.f;
#pragma unroll
                for (int q = 0; q < CL; ++q) v += ld_cluster_f32(p, q);
                a.y[(size_t)b * s.d + o0 + rl] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
            }
        }
        cluster_sync_all();  // keep this CTA's sums alive for its peer
    }
    if (lane == 0 && *abortf) atomicOr(a.err, MOE_DEVERR_TIMEOUT);
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

#ifndef MOEDEC_GU2_FOLD
#define MOEDEC_GU2_FOLD 0
#endif

static bool gate_up_v2_ok(const DecodeShape& s) { return s.d % 128 == 0; }

static size_t gate_up_v2_smem(const DecodeShape& s) {
    return map_ints(s, false) * 4 + (size_t)DEC_WARPS * sizeof(GU2Ring);
}

static cudaError_t launch_gate_up_v2(const GateUpArgs& a, const DeviceInfo& di, int dev, cudaStream_t st) {
    const size_t smem = gate_up_v2_smem(a.s);
    int bps = 1;
    cudaError_t err = prepare(gate_up_v2_kernel<MOEDEC_GU2_FOLD != 0>, smem, dev, &bps);
    if (err != cudaSuccess) return err;
    const long items = (long)max_unique(a.s) * (a.s.I / 2);
    long grid = std::min<long>((long)di.sm_count * bps, (items + DEC_WARPS - 1) / DEC_WARPS);
    if (grid < 1) grid = 1;
    gate_up_v2_kernel<MOEDEC_GU2_FOLD != 0><<<(unsigned)grid, DEC_THREADS, smem, st>>>(a);
    return cudaGetLastError();
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// Bulk copies need 16-byte aligned sources: weight and x rows are (d % 512),
// the scale rows are too when the scale arrays themselves are.
static bool gate_up_v3_ok(const GateUpArgs& a) {
    const DecodeShape& s = a.s;
    if (s.d % GU3_KT || s.I % GU3_ROWS) return false;
    if (!aligned16(a.wg.s) || !aligned16(a.wu.s)) return false;
    if (s.S && (!aligned16(a.shg.s) || !aligned16(a.shu.s))) return false;
    return true;
}

static size_t gate_up_v3_smem(const DecodeShape& s) { return gu3_smem_offset(s) + sizeof(GU3Smem) + 128; }

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_tiled() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// 2D uint8 tensor map over [rows][cols] (row stride = cols bytes); cached by
// (address, rows, cols, box) so repeated calls on the same weights do not
// re-encode.
static bool map_2d_u8(CUtensorMap* out, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows,
                      uint32_t box_cols, bool swizzle128 = false) {
    static std::mutex mu;
    static std::map<std::tuple<const void*, uint64_t, uint64_t, uint32_t, uint32_t, bool>, CUtensorMap> cache;
    const auto key = std::make_tuple(base, rows, cols, box_rows, box_cols, swizzle128);
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) {
        *out = it->second;
        return true;
    }
    EncodeTiledFn fn = encode_tiled();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t es[2] = {1, 1};
    CUtensorMap m;
    if (fn(&m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
           CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    if (cache.size() > 1024) cache.clear();
    cache[key] = m;
    *out = m;
    return true;
}

// 3D uint8 tensor map viewing a [rows][cols] matrix as [cols / 128][rows][128]
// (128-byte column blocks): one copy of a box (128, box_rows, nblk) brings
// box_rows rows x nblk * 128 bytes as nblk consecutive [box_rows][128] tiles,
// each in the 128-byte swizzled layout.  Cached like map_2d_u8.
static bool map_3d_u8_blocks(CUtensorMap* out, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows,
                             uint32_t nblk) {
    static std::mutex mu;
    static std::map<std::tuple<const void*, uint64_t, uint64_t, uint32_t, uint32_t>, CUtensorMap> cache;
    const auto key = std::make_tuple(base, rows, cols, box_rows, nblk);
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) {
        *out = it->second;
        return true;
    }
    EncodeTiledFn fn = encode_tiled();
    if (!fn || cols % 128) return false;
    const cuuint64_t dims[3] = {128, rows, cols / 128};
    const cuuint64_t strides[2] = {cols, 128};
    const cuuint32_t box[3] = {128, box_rows, nblk};
    const cuuint32_t es[3] = {1, 1, 1};
    CUtensorMap m;
    if (fn(&m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, es,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    if (cache.size() > 1024) cache.clear();
    cache[key] = m;
    *out = m;
    return true;
}

static bool gate_up_v3_maps(const GateUpArgs& a, GU3Maps* maps) {
    const DecodeShape& s = a.s;
    const MXView v[2][2] = {{a.wg, a.wu}, {a.shg, a.shu}};
    for (int sh = 0; sh < 2; ++sh) {
        const uint64_t rows = (uint64_t)(sh ? 1 : s.E) * s.I;
        for (int p = 0; p < 2; ++p) {
            const MXView& m = sh && !s.S ? v[0][p] : v[sh][p];  // no shared expert: any valid map
            const uint64_t r = sh && !s.S ? (uint64_t)s.E * s.I : rows;
            if (!map_2d_u8(&maps->w[sh][p], m.w, r, s.d, GU3_ROWS, GU3_BOX)) return false;
            if (!map_2d_u8(&maps->s[sh][p], m.s, r, s.d / 32, GU3_ROWS, 16)) return false;
        }
    }
    return true;
}

static cudaError_t launch_gate_up_v3(const GateUpArgs& a, const GU3Maps& maps, const DeviceInfo& di, int dev,
                                     cudaStream_t st) {
    const size_t smem = gate_up_v3_smem(a.s);
    static std::mutex mu;
    static int bps_cache[64] = {0};
    static size_t smem_cache[64] = {0};
    int bps = 1;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (dev < 64 && bps_cache[dev] && smem_cache[dev] >= smem) {
            bps = bps_cache[dev];
        } else {
            cudaError_t err = cudaFuncSetAttribute(gate_up_v3_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   (int)std::max<size_t>(smem, 48 * 1024));
            if (err != cudaSuccess) return err;
            err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bps, gate_up_v3_kernel, GU3_THREADS, smem);
            if (err != cudaSuccess) return err;
            if (bps < 1) bps = 1;
            if (dev < 64) {
                bps_cache[dev] = bps;
                smem_cache[dev] = smem;
            }
        }
    }
    const long tiles = (long)max_unique(a.s) * (a.s.I / GU3_ROWS);
    long grid = std::min<long>((long)di.sm_count * bps, tiles);
    if (grid < 1) grid = 1;
    gate_up_v3_kernel<<<(unsigned)grid, GU3_THREADS, smem, st>>>(a, maps);
    return cudaGetLastError();
}

// gate/up v4: K in 512-element stages, RT-row tiles, the whole scale row of
// a stage in one 16-byte box; scale and weight bases 16-byte aligned.
#ifndef MOEDEC_GU4_RT
#define MOEDEC_GU4_RT 16
#endif
constexpr int GU4_HOST_RT = MOEDEC_GU4_RT;
constexpr int GU4_HOST_CW = GU4_HOST_RT == 32 ? 16 : 8;

static bool gate_up_v4_ok(const GateUpArgs& a) {
    const DecodeShape& s = a.s;
    if (s.d % GU4_KT || s.I % GU4_HOST_RT) return false;
    if (!aligned16(a.wg.w) || !aligned16(a.wu.w) || !aligned16(a.wg.s) || !aligned16(a.wu.s)) return false;
    if (s.S && (!aligned16(a.shg.w) || !aligned16(a.shu.w) || !aligned16(a.shg.s) || !aligned16(a.shu.s)))
        return false;
    return true;
}

static size_t gate_up_v4_smem(const DecodeShape& s) {
    return gu4_ring_offset(s) + 1024 + (size_t)GU4_S * sizeof(GU4Stage<GU4_HOST_RT>) +
           sizeof(GU4Shared<GU4_HOST_RT, GU4_HOST_CW>);
}

#ifndef MOEDEC_GU4_W3D
#define MOEDEC_GU4_W3D 1
#endif

static bool gate_up_v4_maps(const GateUpArgs& a, GU4Maps* maps) {
    const DecodeShape& s = a.s;
    const MXView v[2][2] = {{a.wg, a.wu}, {a.shg, a.shu}};
    // one 3D copy per projection and stage when the driver takes the block
    // view, else four 2D copies
    maps->w3d = MOEDEC_GU4_W3D;
    for (int pass = 0; pass < 2; ++pass) {
        bool ok = true;
        for (int sh = 0; sh < 2 && ok; ++sh) {
            for (int p = 0; p < 2 && ok; ++p) {
                const MXView& m = sh && !s.S ? v[0][p] : v[sh][p];  // no shared expert: any valid map
                const uint64_t r = (uint64_t)(sh && s.S ? 1 : s.E) * s.I;
                ok = maps->w3d ? map_3d_u8_blocks(&maps->w[sh][p], m.w, r, s.d, GU4_HOST_RT, GU4_KT / GU4_BOX)
                               : map_2d_u8(&maps->w[sh][p], m.w, r, s.d, GU4_HOST_RT, GU4_BOX, true);
                ok = ok && map_2d_u8(&maps->s[sh][p], m.s, r, s.d / 32, GU4_HOST_RT, GU4_KT / 32);
            }
        }
        if (ok) return true;
        if (!maps->w3d) return false;
        maps->w3d = 0;
    }
    return false;
}

// Resident CTAs per SM (0 when the kernel cannot be resident).
static int gate_up_v4_occupancy(size_t smem, int dev) {
    static std::mutex mu;
    static int occ_cache[64] = {0};
    static size_t smem_cache[64] = {0};
    std::lock_guard<std::mutex> lock(mu);
    if (dev < 64 && smem_cache[dev] == smem) return occ_cache[dev];
    auto* fn = gate_up_v4_kernel<GU4_HOST_RT, GU4_HOST_CW>;
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    int bps = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bps, fn, (GU4_HOST_CW + 1) * 32, smem) != cudaSuccess) {
        cudaGetLastError();
        bps = 0;
    }
    if (dev < 64) {
        occ_cache[dev] = bps;
        smem_cache[dev] = smem;
    }
    return bps;
}

static cudaError_t launch_gate_up_v4(const GateUpArgs& a, const GU4Maps& maps, size_t smem, int bps,
                                     const DeviceInfo& di, cudaStream_t st) {
    const long tiles = (long)max_unique(a.s) * (a.s.I / GU4_HOST_RT);
    long grid = std::min<long>((long)di.sm_count * bps, tiles);
    if (grid < 1) grid = 1;
    gate_up_v4_kernel<GU4_HOST_RT, GU4_HOST_CW><<<(unsigned)grid, (GU4_HOST_CW + 1) * 32, smem, st>>>(a, maps);
    return cudaGetLastError();
}

#ifndef MOEDEC_GU4_MIN_TOKENS
#define MOEDEC_GU4_MIN_TOKENS 2
#endif

cudaError_t launch_gate_up(const DecodeShape& s, const void* x, const int32_t* ids, MXView wg,
                           MXView wu, MXView shg, MXView shu, void* h, cudaStream_t st) {
    DeviceInfo di;
    cudaError_t err = device_info(&di);
    if (err != cudaSuccess) return err;
    int dev = 0;
    cudaGetDevice(&dev);
    GateUpArgs a{s, (const uint16_t*)x, ids, wg, wu, shg, shu, (uint16_t*)h, di.err_word};
#ifndef MOEDEC_NO_GU4
    if (s.B >= MOEDEC_GU4_MIN_TOKENS && gate_up_v4_ok(a)) {
        const size_t smem = gate_up_v4_smem(s);
        GU4Maps maps;
        const int bps = smem <= (size_t)di.max_smem_optin ? gate_up_v4_occupancy(smem, dev) : 0;
        if (bps >= 1 && gate_up_v4_maps(a, &maps)) return launch_gate_up_v4(a, maps, smem, bps, di, st);
    }
#endif
#ifndef MOEDEC_NO_GU3
    if (gate_up_v3_ok(a) && gate_up_v3_smem(s) <= (size_t)di.max_smem_optin) {
        GU3Maps maps;
        if (gate_up_v3_maps(a, &maps)) return launch_gate_up_v3(a, maps, di, dev, st);
    }
#endif
    if (gate_up_v2_ok(s) && gate_up_v2_smem(s) <= (size_t)di.max_smem_optin)
        return launch_gate_up_v2(a, di, dev, st);
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

static int down_v2_lanes(const DecodeShape& s) {
    if (s.I % 512 == 0) return 32;
    if (s.I % 256 == 0) return 16;
    if (s.I % 128 == 0) return 8;
    return 0;
}

static size_t down_v2_smem(const DecodeShape& s, int L) {
    const int G = 32 / L;
    const size_t acc_n = (size_t)DEC_WARPS * G * DN2_R * s.B;
    return map_ints(s, true) * 4 + (acc_n + 3) / 4 * 4 * 4 + (size_t)DEC_WARPS * sizeof(DN2Ring);
}

template <int L>
static cudaError_t launch_down_v2_L(DownArgs a, size_t smem, const DeviceInfo& di, int dev,
                                    cudaStream_t st, bool pdl) {
    int bps = 1;
    cudaError_t err = prepare(down_v2_kernel<L>, smem, dev, &bps);
    if (err != cudaSuccess) return err;
    constexpr int G = 32 / L;
    const long target_warps = (long)di.sm_count * 16;
    const int mu = max_unique(a.s);
    int es = 1;
    while (es < DEC_WARPS && es * 2 <= mu) {
        const long rt = (long)(DEC_WARPS / es) * G * DN2_R;
        const long warps = (a.s.d + rt - 1) / rt * DEC_WARPS;
        if (warps >= target_warps) break;
        es *= 2;
    }
    a.es = es;
    const int RT = (DEC_WARPS / es) * G * DN2_R;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((a.s.d + RT - 1) / RT));
    cfg.blockDim = dim3(DEC_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, down_v2_kernel<L>, a);
}

// Bulk copies: the [8 rows x I] weight block and its scale block must start
// on 16-byte boundaries (I % 256 == 0 keeps them there when the arrays do).
static bool down_v3_ok(const DecodeShape& s, MXView wd, MXView shd) {
    if (s.I % 256 || s.d % DN3_RT) return false;
    if (!aligned16(wd.s) || (s.S && !aligned16(shd.s))) return false;
    return true;
}

static size_t down_v3_smem(const DecodeShape& s) {
    const int RW = dn3_rw(s.I);
    const DN3Layout L = dn3_layout(s, RW);
    if (L.S < MOEDEC_DN3_MINS) return ~(size_t)0;  // ring too small for this shape
    return dn3_smem_offset(s, RW) + (size_t)RW * L.S * L.stage_bytes + 2 * DN3_SMAX * sizeof(uint64_t) + 128;
}

template <int RW>
static cudaError_t launch_down_v3_rw(const DownArgs& a, size_t smem, int dev, cudaStream_t st, bool pdl) {
    static std::mutex mu;
    static size_t attr_smem[64] = {0};
    {
        std::lock_guard<std::mutex> lock(mu);
        if (dev >= 64 || attr_smem[dev] < smem) {
            cudaError_t err = cudaFuncSetAttribute(down_v3_kernel<RW>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   (int)std::max<size_t>(smem, 48 * 1024));
            if (err != cudaSuccess) return err;
            if (dev < 64) attr_smem[dev] = smem;
        }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(a.s.d / DN3_RT));
    cfg.blockDim = dim3(DN3_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, down_v3_kernel<RW>, a);
}

static cudaError_t launch_down_v3(const DownArgs& a, size_t smem, int dev, cudaStream_t st, bool pdl) {
    switch (dn3_rw(a.s.I)) {
        case 1: return launch_down_v3_rw<1>(a, smem, dev, st, pdl);
#if MOEDEC_DN3_RWSMALL == 4
        default: return launch_down_v3_rw<4>(a, smem, dev, st, pdl);
#else
        default: return launch_down_v3_rw<2>(a, smem, dev, st, pdl);
#endif
    }
}

// Rows per warp for down v4: ~96 weight bytes per lane per stage.
#ifndef MOEDEC_DN4_RWSMALL
#define MOEDEC_DN4_RWSMALL 2
#endif
static int dn4_rw(int I) { return I >= 2048 ? 1 : (I >= 1024 ? 2 : MOEDEC_DN4_RWSMALL); }

static size_t down_v4_smem(const DecodeShape& s, int RT) {
    const DN3Layout L = dn4_layout(s, RT);
    if (L.S < 2) return ~(size_t)0;
    return dn4_smem_offset(s, RT) + (size_t)L.S * L.stage_bytes + 2 * DN4_SMAX * sizeof(uint64_t) + 128;
}

template <int RW, int CL, int NCH, int CW>
static cudaError_t launch_down_v4_k(const DownArgs& a, size_t smem, int dev, cudaStream_t st, bool pdl) {
    static std::mutex mu;
    static size_t attr_smem[64] = {0};
    {
        std::lock_guard<std::mutex> lock(mu);
        if (dev >= 64 || attr_smem[dev] < smem) {
            cudaError_t err = cudaFuncSetAttribute(down_v4_kernel<RW, CL, NCH, CW>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   (int)std::max<size_t>(smem, 48 * 1024));
            if (err != cudaSuccess) return err;
            if (dev < 64) attr_smem[dev] = smem;
        }
    }
    constexpr int RT = CW * RW;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((a.s.d + RT - 1) / RT * CL));
    cfg.blockDim = dim3((CW + 1) * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (CL > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = CL;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    if (pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, down_v4_kernel<RW, CL, NCH, CW>, a);
}

// Consumer warps per CTA (8, or 7 = 14-row blocks with two rows per warp)
// and cluster size: the fewest rows per CTA over the waves the grid needs at
// two CTAs per SM, never a cluster larger than the distinct experts a call
// can have; ties go to 8 warps, then to the smaller cluster.
struct DN4Geom {
    int cw, cl;
};

#ifndef MOEDEC_DN4_CW7
#define MOEDEC_DN4_CW7 1
#endif

static DN4Geom dn4_geom(const DecodeShape& s, int RW, int sm_count) {
    const long slots = 2L * sm_count;
    DN4Geom best{8, 1};
    long best_cost = -1;
    for (int cw = 8; cw >= 7; --cw) {
        if (cw == 7 && (RW == 1 || !MOEDEC_DN4_CW7)) continue;
        if (cw == 8 && RW == 4 && MOEDEC_DN4_CW7) continue;  // four rows per warp want the 128-register CTA
        const int RT = cw * RW;
        const long nblk = (s.d + RT - 1) / RT;
        for (int cl = 1; cl <= 4; cl *= 2) {
            if (cl > 1 && cl > max_unique(s)) break;
            if (RT % cl) continue;
            const long waves = (nblk * cl + slots - 1) / slots;
            const long cost = waves * RT * 64 / cl;
            if (best_cost < 0 || cost < best_cost) {
                best_cost = cost;
                best = DN4Geom{cw, cl};
            }
        }
    }
    return best;
}

template <int RW, int NCH, int CW>
static cudaError_t launch_down_v4_cl(const DownArgs& a, int cl, size_t smem, int dev, cudaStream_t st, bool pdl) {
    switch (cl) {
        case 1: return launch_down_v4_k<RW, 1, NCH, CW>(a, smem, dev, st, pdl);
        case 2: return launch_down_v4_k<RW, 2, NCH, CW>(a, smem, dev, st, pdl);
        default:
            if constexpr ((CW * RW) % 4 == 0) return launch_down_v4_k<RW, 4, NCH, CW>(a, smem, dev, st, pdl);
            return cudaErrorInvalidValue;
    }
}

template <int RW, int NCH>
static cudaError_t launch_down_v4_cw(const DownArgs& a, const DN4Geom& g, size_t smem, int dev, cudaStream_t st,
                                     bool pdl) {
    if constexpr (RW >= 2) {
        if (g.cw == 7) return launch_down_v4_cl<RW, NCH, 7>(a, g.cl, smem, dev, st, pdl);
    }
    return launch_down_v4_cl<RW, NCH, 8>(a, g.cl, smem, dev, st, pdl);
}

// The chunk loop is unrolled for the common lengths (I = 768 at two rows per
// warp, I = 2048 at one), a run-time loop otherwise.
template <int RW>
static cudaError_t launch_down_v4_rw(const DownArgs& a, const DN4Geom& g, size_t smem, int dev, cudaStream_t st,
                                     bool pdl) {
    const int nch = a.s.I / 256;
    if constexpr (RW >= 2) {
        if (nch == 3) return launch_down_v4_cw<RW, 3>(a, g, smem, dev, st, pdl);
    }
    if constexpr (RW == 1) {
        if (nch == 8) return launch_down_v4_cw<RW, 8>(a, g, smem, dev, st, pdl);
    }
    return launch_down_v4_cw<RW, 0>(a, g, smem, dev, st, pdl);
}

// ---- down v5 plan: slab, stage layout, ring depth, row block and cluster
#ifndef MOEDEC_DN5_MAXB
#define MOEDEC_DN5_MAXB 64
#endif

struct DN5Plan {
    DN5Params P;
    int CL, grid;
    size_t smem;
};

static int smem_per_sm(int dev) {
    static std::mutex mu;
    static int cache[64] = {0};
    std::lock_guard<std::mutex> lock(mu);
    if (dev < 64 && cache[dev]) return cache[dev];
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess) {
        cudaGetLastError();
        v = 0;
    }
    if (dev < 64) cache[dev] = v;
    return v;
}

static bool down_v5_plan(const DownArgs& a, const DeviceInfo& di, int dev, DN5Plan* out) {
    const DecodeShape& s = a.s;
    if (s.B > MOEDEC_DN5_MAXB || s.I % 256 || s.d % 2) return false;
    DN5Params P{};
    if (s.I == 256 || s.I == 512 || s.I == 768) {
        P.KSLAB = s.I;
        P.scale2d = 0;
    } else if (s.I % 512 == 0) {
        P.KSLAB = 512;
        P.scale2d = 1;
    } else {
        return false;
    }
    if (!aligned16(a.wd.w) || !aligned16(a.wd.s)) return false;
    if (s.S && (!aligned16(a.shd.w) || !aligned16(a.shd.s))) return false;
    auto r128 = [](size_t v) { return (v + 127) / 128 * 128; };
    auto r1024 = [](size_t v) { return (v + 1023) / 1024 * 1024; };
    P.sc_off = P.KSLAB * 16;
    P.h_off = (int)(P.sc_off + r128((size_t)DN5_RTMAX * (P.KSLAB / 32)));
    P.stage_bytes = (int)r1024((size_t)P.h_off + (size_t)TC * P.KSLAB * 2);
    const size_t fixed = map_ints(s, true) * 4 + 1024 + (size_t)DN5_CW * TC * (P.KSLAB / 8) * 4 +
                         (size_t)DN5_CW * s.B * DN5_RTMAX * 4 + 2 * DN5_SMAX * 8 + 16;
    // two CTAs per SM
    const int per_sm = smem_per_sm(dev);
    const size_t limit = per_sm > 0 ? (size_t)per_sm / 2 - 1024 : 0;
    if (limit <= fixed) return false;
    P.S = (int)std::min<size_t>(DN5_SMAX, (limit - fixed) / P.stage_bytes);
    if (P.S < 3) return false;
    const size_t smem = fixed + (size_t)P.S * P.stage_bytes;
    if (smem > (size_t)di.max_smem_optin) return false;
    // row block and cluster: the fewest rows per CTA over the waves the
    // grid needs (two CTAs per SM), preferring larger blocks on ties
    const int slots = 2 * di.sm_count;
    const int nu_max = max_unique(s);
    int best_cost = 1 << 30, bRT = 0, bCL = 0;
    for (int CL = 2; CL >= 1; --CL) {
        if (CL > nu_max) continue;
        for (int RT = DN5_RTMAX; RT >= 8; RT -= 2) {
            const int nblk = (s.d + RT - 1) / RT;
            int cost;
            if (CL > 1) {
                if (nblk * CL > slots) continue;
                cost = RT * 64 / CL;
            } else {
                const int ctas = std::min(nblk, slots);
                const int waves = (nblk + ctas - 1) / ctas;
                cost = waves * RT * 64;
            }
            if (cost < best_cost) {
                best_cost = cost;
                bRT = RT;
                bCL = CL;
            }
        }
    }
    if (!bRT) return false;
    P.RT = bRT;
    P.nblk = (s.d + bRT - 1) / bRT;
    out->P = P;
    out->CL = bCL;
    out->grid = bCL > 1 ? P.nblk * bCL : std::min(P.nblk, slots);
    out->smem = smem;
    return true;
}

static bool down_v5_maps(const DownArgs& a, const DN5Params& P, DN5Maps* maps) {
    const DecodeShape& s = a.s;
    const MXView v[2] = {a.wd, a.shd};
    for (int sh = 0; sh < 2; ++sh) {
        const MXView& m = sh && !s.S ? v[0] : v[sh];  // no shared expert: any valid map
        const uint64_t rows = (uint64_t)(sh && s.S ? 1 : s.E) * s.d;
        if (!map_3d_u8_blocks(&maps->w[sh], m.w, rows, s.I, P.RT, P.KSLAB / 128)) return false;
        if (P.scale2d && !map_2d_u8(&maps->s[sh], m.s, rows, s.I / 32, P.RT, 16)) return false;
        if (!P.scale2d) maps->s[sh] = maps->w[sh];  // unused
    }
    return true;
}

template <int CL, int KSLAB>
static cudaError_t launch_down_v5_k(const DownArgs& a, const DN5Maps& maps, const DN5Plan& pl, int dev,
                                    cudaStream_t st, bool pdl) {
    static std::mutex mu;
    static size_t attr_smem[64] = {0};
    {
        std::lock_guard<std::mutex> lock(mu);
        if (dev >= 64 || attr_smem[dev] < pl.smem) {
            cudaError_t err = cudaFuncSetAttribute(down_v5_kernel<CL, KSLAB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   (int)std::max<size_t>(pl.smem, 48 * 1024));
            if (err != cudaSuccess) return err;
            if (dev < 64) attr_smem[dev] = pl.smem;
        }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)pl.grid);
    cfg.blockDim = dim3(DN5_THREADS);
    cfg.dynamicSmemBytes = pl.smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (CL > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = CL;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    if (pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, down_v5_kernel<CL, KSLAB>, a, maps, pl.P);
}

cudaError_t launch_down(const DecodeShape& s, const void* h, const int32_t* ids, const float* w,
                        MXView wd, MXView shd, void* y, cudaStream_t st, bool after_gate_up) {
    DeviceInfo di;
    cudaError_t err = device_info(&di);
    if (err != cudaSuccess) return err;
    int dev = 0;
    cudaGetDevice(&dev);
    DownArgs a{s, (const uint16_t*)h, ids, w, wd, shd, (uint16_t*)y, di.err_word, 1};
#ifdef MOEDEC_DN5
    {
        DN5Plan pl;
        DN5Maps maps;
        if (down_v5_plan(a, di, dev, &pl) && down_v5_maps(a, pl.P, &maps)) {
            const int ks = pl.P.KSLAB;
            if (pl.CL > 1) {
                if (ks == 768) return launch_down_v5_k<2, 768>(a, maps, pl, dev, st, after_gate_up);
                if (ks == 512) return launch_down_v5_k<2, 512>(a, maps, pl, dev, st, after_gate_up);
                return launch_down_v5_k<2, 256>(a, maps, pl, dev, st, after_gate_up);
            }
            if (ks == 768) return launch_down_v5_k<1, 768>(a, maps, pl, dev, st, after_gate_up);
            if (ks == 512) return launch_down_v5_k<1, 512>(a, maps, pl, dev, st, after_gate_up);
            return launch_down_v5_k<1, 256>(a, maps, pl, dev, st, after_gate_up);
        }
    }
#endif
#ifndef MOEDEC_NO_DN4
    if (down_v3_ok(s, wd, shd)) {
        // rows per block and s.d even: every block's scale bytes are a multiple of 16
        const int RW = dn4_rw(s.I);
        const DN4Geom g = dn4_geom(s, RW, di.sm_count);
        const size_t smem4 = down_v4_smem(s, g.cw * RW);
        if (s.d % 2 == 0 && smem4 <= (size_t)di.max_smem_optin) {
            switch (RW) {
                case 1: return launch_down_v4_rw<1>(a, g, smem4, dev, st, after_gate_up);
                case 2: return launch_down_v4_rw<2>(a, g, smem4, dev, st, after_gate_up);
                default: return launch_down_v4_rw<4>(a, g, smem4, dev, st, after_gate_up);
            }
        }
    }
#endif
#ifndef MOEDEC_NO_DN3
    if (down_v3_ok(s, wd, shd)) {
        const size_t smem3 = down_v3_smem(s);
        if (smem3 <= (size_t)di.max_smem_optin) return launch_down_v3(a, smem3, dev, st, after_gate_up);
    }
#endif
    const int L2 = down_v2_lanes(s);
    if (L2) {
        const size_t smem2 = down_v2_smem(s, L2);
        if (smem2 <= (size_t)di.max_smem_optin) {
            switch (L2) {
                case 32: return launch_down_v2_L<32>(a, smem2, di, dev, st, after_gate_up);
                case 16: return launch_down_v2_L<16>(a, smem2, di, dev, st, after_gate_up);
                default: return launch_down_v2_L<8>(a, smem2, di, dev, st, after_gate_up);
            }
        }
    }
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

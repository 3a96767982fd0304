// gate_up.cu -- the MoE expert-FFN decode layer on sm_103a.
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
#include "decode_common.cuh"

namespace moedec {

// ------------------------------------------------------------ gate/up ----

template <int L, int NT>
__device__ __forceinline__ void gate_up_rows(const uint8_t* __restrict__ wg_row,
                                             const uint8_t* __restrict__ sg_row,
                                             const uint8_t* __restrict__ wu_row,
                                             const uint8_t* __restrict__ su_row,
                                             const uint16_t* __restrict__ x, int d,
                                             const int* __restrict__ hrow_s, int KS, int cpl,
                                             int li, bool row_ok, int n, const GateUpArgs& a) {
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
            store_h(a, hr[t], n, hv);
        }
    }
}

template <int L>
__global__ void __launch_bounds__(DEC_THREADS) gate_up_kernel(GateUpArgs a) {
    extern __shared__ __align__(128) int smem_i[];
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
                case 1: gate_up_rows<L, 1>(wg_row, sg_row, wu_row, su_row, a.x, s.d, hs, KS, cpl, li, row_ok, n, a); break;
                case 2: gate_up_rows<L, 2>(wg_row, sg_row, wu_row, su_row, a.x, s.d, hs, KS, cpl, li, row_ok, n, a); break;
                case 3: gate_up_rows<L, 3>(wg_row, sg_row, wu_row, su_row, a.x, s.d, hs, KS, cpl, li, row_ok, n, a); break;
                default: gate_up_rows<L, 4>(wg_row, sg_row, wu_row, su_row, a.x, s.d, hs, KS, cpl, li, row_ok, n, a); break;
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

template <int NT>
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
                wq[p] = __fmul2_rn(wq[p], make_float2(sc[p], sc[p]));
            }
#pragma unroll
            for (int t = 0; t < NT; ++t) {
                const uint32_t xw = (&xv[t].x)[q & 3];
                const float2 xf = bf16x2_to_float2(xw);
#pragma unroll
                for (int p = 0; p < GU2_PARTS; ++p) acc[p][t] = __ffma2_rn(xf, wq[p], acc[p][t]);
            }
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
        store_h(a, hrow, n0 + rr, hv);
    }
}


__global__ void __launch_bounds__(DEC_THREADS, 2) gate_up_v2_kernel(GateUpArgs a) {
    extern __shared__ __align__(128) int smem_i[];
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
                case 1: gu2_group<1>(a, m, wi, pc, ring, slot, lane, pol, n0, hs, nt); break;
                case 2: gu2_group<2>(a, m, wi, pc, ring, slot, lane, pol, n0, hs, nt); break;
                case 3: gu2_group<3>(a, m, wi, pc, ring, slot, lane, pol, n0, hs, nt); break;
                default: gu2_group<4>(a, m, wi, pc, ring, slot, lane, pol, n0, hs, nt); break;
            }
        }
    }
    cp_async_wait<0>();
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
                wq[p][0] = __fmul2_rn(wq[p][0], make_float2(sc[p], sc[p]));
                wq[p][1] = __fmul2_rn(wq[p][1], make_float2(sc[p], sc[p]));
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
#pragma unroll
                for (int t = 0; t < NT; ++t) {
                    const float2 xf = bf16x2_to_float2((&xv[t].x)[(q4 & 1) * 2 + h]);
#pragma unroll
                    for (int p = 0; p < GU2_PARTS; ++p) {
                        acc[p][t] = __ffma2_rn(xf, wq[p][h], acc[p][t]);
                    }
                }
            }
        }
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
        store_h(a, hrow, n0 + 2 * cw + rr, hv);
    }
    return true;
}

__host__ __device__ inline size_t gu3_smem_offset(const DecodeShape& s) {
    return (map_ints(s, false) * 4 + 127) / 128 * 128;
}

__global__ void __launch_bounds__(GU3_THREADS, 2)
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

constexpr int GU4_KT = 512;   // K elements per stage (16 scale blocks)
constexpr int GU4_BOX = 128;  // inner box of a weight tensor copy (bytes)
constexpr int GU4_S = 4;      // ring stages

// FP4: MXFP4 weights, two E2M1 codes per byte, so a stage's code bytes
// per row are half those of MXFP8.
template <int RT, bool FP4 = false>
struct __align__(1024) GU4Stage {
    static constexpr int BOXES = GU4_KT / (FP4 ? 2 : 1) / GU4_BOX;
    uint8_t w[2][BOXES][RT][GU4_BOX];             // [proj][box][row][128 B, swizzled]
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
__host__ __device__ inline size_t gu4_ring_offset(const DecodeShape& s) { return map_ints(s, false) * 4; }

template <int RT, int CW, int NT, bool FP4>
__device__ __forceinline__ void gu4_group(const GateUpArgs& a, GU4Stage<RT, FP4>* ring, GU4Shared<RT, CW>* sh,
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
        const GU4Stage<RT, FP4>& st = ring[slot];
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
        if constexpr (FP4) {
            // one 16-byte chunk holds the lane's whole 32-element block
            uint4 wv[2];
#pragma unroll
            for (int p = 0; p < 2; ++p)
                wv[p] = *reinterpret_cast<const uint4*>(&st.w[p][blk >> 3][r][((blk & 7) ^ sw) * 16]);
#pragma unroll
            for (int q8 = 0; q8 < 4; ++q8) {  // eight K elements per code word
                float2 wq[2][4];
#pragma unroll
                for (int p = 0; p < 2; ++p) e2m1x8_to_float((&wv[p].x)[q8], wq[p]);
#pragma unroll
                for (int t = 0; t < NT; ++t) {
                    const float4 x0 = *reinterpret_cast<const float4*>(xl + t * XS + q8 * 8);
                    const float4 x1 = *reinterpret_cast<const float4*>(xl + t * XS + q8 * 8 + 4);
#pragma unroll
                    for (int p = 0; p < 2; ++p) {
                        if (q8 == 0)
                            part[p][t] = __fmul2_rn(make_float2(x0.x, x0.y), wq[p][0]);
                        else
                            part[p][t] = __ffma2_rn(make_float2(x0.x, x0.y), wq[p][0], part[p][t]);
                        part[p][t] = __ffma2_rn(make_float2(x0.z, x0.w), wq[p][1], part[p][t]);
                        part[p][t] = __ffma2_rn(make_float2(x1.x, x1.y), wq[p][2], part[p][t]);
                        part[p][t] = __ffma2_rn(make_float2(x1.z, x1.w), wq[p][3], part[p][t]);
                    }
                }
            }
        } else {
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
            store_h(a, hrow, n0 + rr, hv);
        }
    }
}

template <int RT, int CW, bool FP4>
__global__ void __launch_bounds__((CW + 1) * 32, RT == 32 ? 1 : 2)
    gate_up_v4_kernel(GateUpArgs a, const __grid_constant__ GU4Maps maps) {
    constexpr int S = GU4_S;
    extern __shared__ __align__(128) int smem_i[];
    const DecodeShape s = a.s;
    const RouteMap m = carve_map(smem_i, s, false);
    // swizzled tensor copies want 1024-byte aligned boxes: align at run time
    // (the launch reserves 1024 spare bytes)
    const uintptr_t raw = reinterpret_cast<uintptr_t>(smem_i) + gu4_ring_offset(s);
    using Stage = GU4Stage<RT, FP4>;
    Stage* ring = reinterpret_cast<Stage*>((raw + 1023) & ~uintptr_t(1023));
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
                    (int)(S * sizeof(Stage) / 4));  // ends with __syncthreads
    asm volatile("griddepcontrol.launch_dependents;");

    const int nu = m.hdr[0];
    const int rbs = s.I / RT;
    const int tiles = nu * rbs;
    // With few tiles per CTA and some expert needing more than one pass over
    // its rows, deal the heaviest experts' tiles first, in snake order over
    // the CTAs, so that the CTAs' loads even out; otherwise plain round robin.
    // (The order never changes a result.)
    bool ordered = (CW + 1) * 32 >= 256 && nu <= 256 && tiles <= 32 * (int)gridDim.x;
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
                    Stage& st = ring[slot];
                    if (lane == 0) {
                        mbar_arrive_expect_tx(&sh->full[slot], 2 * RT * (Stage::BOXES * GU4_BOX + GU4_KT / 32) +
                                                                   nt * GU4_KT * 2);
                        fence_proxy_async();
#pragma unroll
                        for (int p = 0; p < 2; ++p) {
                            if (maps.w3d) {
                                tma_3d(st.w[p][0], &maps.w[shx][p], 0, row0, kt * Stage::BOXES, &sh->full[slot],
                                       pol);
                            } else {
#pragma unroll
                                for (int b = 0; b < Stage::BOXES; ++b)
                                    tma_2d(st.w[p][b], &maps.w[shx][p], (kt * Stage::BOXES + b) * GU4_BOX, row0,
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
                    case 1: gu4_group<RT, CW, 1, FP4>(a, ring, sh, rp, grp, nkt, warp, lane, n0, hs); break;
                    case 2: gu4_group<RT, CW, 2, FP4>(a, ring, sh, rp, grp, nkt, warp, lane, n0, hs); break;
                    case 3: gu4_group<RT, CW, 3, FP4>(a, ring, sh, rp, grp, nkt, warp, lane, n0, hs); break;
                    default: gu4_group<RT, CW, 4, FP4>(a, ring, sh, rp, grp, nkt, warp, lane, n0, hs); break;
                }
            }
        }
    }
    if (lane == 0 && sh->abort) atomicOr(a.err, MOE_DEVERR_TIMEOUT);
}

// -------------------------------------------------------------- host -----

size_t gate_up_smem_bytes(const DecodeShape& s) { return map_ints(s, false) * 4; }

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


static bool gate_up_v2_ok(const DecodeShape& s) { return s.d % 128 == 0; }

static size_t gate_up_v2_smem(const DecodeShape& s) {
    return map_ints(s, false) * 4 + (size_t)DEC_WARPS * sizeof(GU2Ring);
}

static cudaError_t launch_gate_up_v2(const GateUpArgs& a, const DeviceInfo& di, int dev, cudaStream_t st) {
    const size_t smem = gate_up_v2_smem(a.s);
    int bps = 1;
    cudaError_t err = prepare(gate_up_v2_kernel, smem, dev, &bps);
    if (err != cudaSuccess) return err;
    const long items = (long)max_unique(a.s) * (a.s.I / 2);
    long grid = std::min<long>((long)di.sm_count * bps, (items + DEC_WARPS - 1) / DEC_WARPS);
    if (grid < 1) grid = 1;
    gate_up_v2_kernel<<<(unsigned)grid, DEC_THREADS, smem, st>>>(a);
    return cudaGetLastError();
}

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
constexpr int GU4_HOST_RT = 16;
constexpr int GU4_HOST_CW = 8;

static bool gate_up_v4_ok(const GateUpArgs& a) {
    const DecodeShape& s = a.s;
    if (s.d % GU4_KT || s.I % GU4_HOST_RT) return false;  // (MXFP4: 256-byte code stages, 128-byte boxes)
    if (!aligned16(a.wg.w) || !aligned16(a.wu.w) || !aligned16(a.wg.s) || !aligned16(a.wu.s)) return false;
    if (s.S && (!aligned16(a.shg.w) || !aligned16(a.shu.w) || !aligned16(a.shg.s) || !aligned16(a.shu.s)))
        return false;
    return true;
}

static size_t gate_up_v4_smem(const DecodeShape& s, bool fp4) {
    const size_t stage = fp4 ? sizeof(GU4Stage<GU4_HOST_RT, true>) : sizeof(GU4Stage<GU4_HOST_RT, false>);
    return gu4_ring_offset(s) + 1024 + (size_t)GU4_S * stage + sizeof(GU4Shared<GU4_HOST_RT, GU4_HOST_CW>);
}


static bool gate_up_v4_maps(const GateUpArgs& a, bool fp4, GU4Maps* maps) {
    const DecodeShape& s = a.s;
    const uint64_t cols = fp4 ? s.d / 2 : s.d;  // code bytes per row
    const uint32_t nblk = (uint32_t)(GU4_KT / (fp4 ? 2 : 1) / GU4_BOX);
    const MXView v[2][2] = {{a.wg, a.wu}, {a.shg, a.shu}};
    // one 3D copy per projection and stage when the driver takes the block
    // view, else four 2D copies
    maps->w3d = 1;
    for (int pass = 0; pass < 2; ++pass) {
        bool ok = true;
        for (int sh = 0; sh < 2 && ok; ++sh) {
            for (int p = 0; p < 2 && ok; ++p) {
                const MXView& m = sh && !s.S ? v[0][p] : v[sh][p];  // no shared expert: any valid map
                const uint64_t r = (uint64_t)(sh && s.S ? 1 : s.E) * s.I;
                ok = maps->w3d ? map_3d_u8_blocks(&maps->w[sh][p], m.w, r, cols, GU4_HOST_RT, nblk)
                               : map_2d_u8(&maps->w[sh][p], m.w, r, cols, GU4_HOST_RT, GU4_BOX, true);
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
static int gate_up_v4_occupancy(size_t smem, int dev, bool fp4) {
    static std::mutex mu;
    static int occ_cache[2][64] = {{0}};
    static size_t smem_cache[2][64] = {{0}};
    std::lock_guard<std::mutex> lock(mu);
    if (dev < 0 || dev >= 64) return 0;
    if (smem_cache[fp4][dev] == smem) return occ_cache[fp4][dev];
    auto* fn = fp4 ? gate_up_v4_kernel<GU4_HOST_RT, GU4_HOST_CW, true> : gate_up_v4_kernel<GU4_HOST_RT, GU4_HOST_CW, false>;
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    int bps = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bps, fn, (GU4_HOST_CW + 1) * 32, smem) != cudaSuccess) {
        cudaGetLastError();
        bps = 0;
    }
    occ_cache[fp4][dev] = bps;
    smem_cache[fp4][dev] = smem;
    return bps;
}

static cudaError_t launch_gate_up_v4(const GateUpArgs& a, const GU4Maps& maps, size_t smem, int bps,
                                     const DeviceInfo& di, cudaStream_t st, bool fp4) {
    const long tiles = (long)max_unique(a.s) * (a.s.I / GU4_HOST_RT);
    long grid = std::min<long>((long)di.sm_count * bps, tiles);
    if (grid < 1) grid = 1;
    if (fp4)
        gate_up_v4_kernel<GU4_HOST_RT, GU4_HOST_CW, true><<<(unsigned)grid, (GU4_HOST_CW + 1) * 32, smem, st>>>(a, maps);
    else
        gate_up_v4_kernel<GU4_HOST_RT, GU4_HOST_CW, false><<<(unsigned)grid, (GU4_HOST_CW + 1) * 32, smem, st>>>(a, maps);
    return cudaGetLastError();
}

// The grouped gate/up kernel with MXFP4 weights (moe_gate_up_fp4); returns
// false when the shape or alignment does not suit it (the caller then uses
// the one-warp-per-output kernel).
bool launch_gate_up_grouped_fp4(const DecodeShape& s, const void* x, const int32_t* ids, MXView wg, MXView wu,
                                MXView shg, MXView shu, void* h, cudaStream_t st, cudaError_t* err) {
    DeviceInfo di;
    if ((*err = device_info(&di)) != cudaSuccess) return true;
    int dev = 0;
    if ((*err = cudaGetDevice(&dev)) != cudaSuccess) return true;
    GateUpArgs a{s, (const uint16_t*)x, ids, wg, wu, shg, shu, (uint16_t*)h, di.err_word, nullptr};
    if (s.B < 2 || !gate_up_v4_ok(a)) return false;
    const size_t smem = gate_up_v4_smem(s, true);
    const int bps = smem <= (size_t)di.max_smem_optin ? gate_up_v4_occupancy(smem, dev, true) : 0;
    GU4Maps maps;
    if (bps < 1 || !gate_up_v4_maps(a, true, &maps)) return false;
    *err = launch_gate_up_v4(a, maps, smem, bps, di, st, true);
    return true;
}



cudaError_t launch_gate_up(const DecodeShape& s, const void* x, const int32_t* ids, MXView wg,
                           MXView wu, MXView shg, MXView shu, void* h, bool h32, cudaStream_t st) {
    DeviceInfo di;
    cudaError_t err = device_info(&di);
    if (err != cudaSuccess) return err;
    int dev = 0;
    if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
    GateUpArgs a{s, (const uint16_t*)x, ids, wg, wu, shg, shu, h32 ? nullptr : (uint16_t*)h, di.err_word,
                 h32 ? (float*)h : nullptr};
    if (s.B >= 2 && gate_up_v4_ok(a)) {
        const size_t smem = gate_up_v4_smem(s, false);
        GU4Maps maps;
        const int bps = smem <= (size_t)di.max_smem_optin ? gate_up_v4_occupancy(smem, dev, false) : 0;
        if (bps >= 1 && gate_up_v4_maps(a, false, &maps)) return launch_gate_up_v4(a, maps, smem, bps, di, st, false);
    }
    if (gate_up_v3_ok(a) && gate_up_v3_smem(s) <= (size_t)di.max_smem_optin) {
        GU3Maps maps;
        if (gate_up_v3_maps(a, &maps)) return launch_gate_up_v3(a, maps, di, dev, st);
    }
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

}  // namespace moedec

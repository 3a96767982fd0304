// down.cu -- the down pass of the MoE expert-FFN decode layer on sm_103a.
#include "decode_common.cuh"

namespace moedec {

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
    extern __shared__ __align__(128) int smem_i[];
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
    extern __shared__ __align__(128) int smem_i[];
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

struct DN3Layout {
    int stage_bytes, w_off, s_off, h_off, S;  // S = slots per split
};


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

// ------------------------------------------------------- down, row tiles ----
// Output-stationary down pass.  A cluster of CL CTAs owns a block of RT =
// 8 * CW output rows; the block's work items are (distinct expert u, group g
// of up to DT_TC of its tokens), dealt round robin to the cluster's CTAs.  An
// item streams I / 256 stages; a stage holds the expert's RT x 256 code block
// (one 3D tensor copy: two 128-byte column blocks, 128-byte swizzled), its
// RT x 8 scale bytes (8-byte cp.async per row, completion counted on the
// same mbarrier) and the item's tokens' 256 intermediate values.
//
// Each of the CW consumer warps owns 8 rows; lane (kr, rr) takes the rows
// rr and rr + 4 of its warp's eight and the 32-element scale block kr of
// every stage, so a lane dequantises each code of its two rows once, uses
// each activation it loads for both rows, and scales each block's partial
// sum once.  Per lane and stage the block's partial sums go into FP32
// accumulators per (row, token); after the item's last stage the eight
// K-lanes of a row reduce them by shuffles and the lane left holding a
// (row, token) sum adds w * sum to that output's FP32 accumulator in shared
// memory, which no other thread writes.  At the end the cluster's CTAs add
// their accumulators in rank order through distributed shared memory and
// round once to BF16: no combine buffer, deterministic.
//
// The intermediate comes either as FP32 in h32_pos order (the layer's own
// gate/up pass writes it so: each lane's four values of one step are one
// conflict-free 16-byte load) or as the BF16 h of the interface, converted
// by each lane.  The weights and scales of the first stages are issued
// before the wait for the gate/up pass (programmatic dependent launch).
// Every mbarrier wait is bounded; a wait that runs out sets
// MOE_DEVERR_TIMEOUT and ends the CTA's work (every thread still reaches the
// cluster barriers).

constexpr int DT_KS = 256;   // K elements per stage: 8 lanes x one 32-element block
constexpr int DT_TC = 4;     // tokens per item
constexpr int DT_SMAX = 8;   // most ring stages
constexpr int DT_RL = 2;     // rows per lane

struct DTLayout {
    int S;             // ring stages
    int stage_bytes;   // multiple of 1024
    int sc_off, h_off; // offsets of the scale bytes and the intermediate inside a stage
    int ring_off;      // offset of the ring (before aligning to 1024) from the dynamic smem base
    int smem;          // dynamic shared memory bytes
};

struct DTMaps {
    CUtensorMap w[2];  // [routed / shared] codes viewed as [I / 128][rows][128], box 128 x RT x 2
};

__host__ __device__ inline DTLayout dt_layout(const DecodeShape& s, int RT, bool hf32, int budget) {
    DTLayout L;
    L.sc_off = 256 * RT;
    L.h_off = (L.sc_off + 8 * RT + 127) / 128 * 128;
    L.stage_bytes = (L.h_off + DT_TC * DT_KS * (hf32 ? 4 : 2) + 1023) / 1024 * 1024;
    L.ring_off = (int)(map_ints(s, true) * 4 + (size_t)RT * s.B * 4);
    const int fixed = L.ring_off + 1024 + 2 * DT_SMAX * 8;
    int S = (budget - fixed) / L.stage_bytes;
    L.S = S > DT_SMAX ? DT_SMAX : S;
    L.smem = fixed + (L.S > 0 ? L.S : 0) * L.stage_bytes;
    return L;
}

// This CTA's next item: items (u, g) are numbered in order of u then g, and
// the CTA of cluster rank `rank` takes the numbers congruent to it mod CL.
struct DTCursor {
    int u, g, it, ks;
};

__device__ __forceinline__ void dt_seek(DTCursor& c, const RouteMap& m, int ntot, int CL, int rank) {
    while (c.u < ntot) {
        const int ng = (m.ucnt[c.u] + DT_TC - 1) / DT_TC;
        if (c.g >= ng) {
            ++c.u;
            c.g = 0;
            continue;
        }
        if (c.it % CL == rank) return;
        ++c.g;
        ++c.it;
    }
}

__device__ __forceinline__ void dt_advance(DTCursor& c, const RouteMap& m, int ntot, int nks, int CL, int rank) {
    if (++c.ks < nks) return;
    c.ks = 0;
    ++c.g;
    ++c.it;
    dt_seek(c, m, ntot, CL, rank);
}

// Sum N values (one per (row, token)) over the eight K-lanes of a row (lane
// bits 3, 1, 0): reduce-scatter while a lane holds more than one value,
// then plain butterfly steps.  Returns the sum of value `idx`; `owner` is
// true in exactly one of the eight lanes for each value.
template <int N>
__device__ __forceinline__ float klane_reduce(float (&v)[N], int lane, int& idx, bool& owner) {
    idx = 0;
    owner = true;
    int cnt = N;
#pragma unroll
    for (int l = 0; l < 3; ++l) {
        const int o = l == 0 ? 8 : (l == 1 ? 2 : 1);
        if (cnt > 1) {
            const bool up = (lane & o) != 0;
#pragma unroll
            for (int i = 0; i < N / 2; ++i) {
                if (i < cnt / 2) {
                    const float send = up ? v[i] : v[i + cnt / 2];
                    const float keep = up ? v[i + cnt / 2] : v[i];
                    v[i] = keep + __shfl_xor_sync(FULL_MASK, send, o);
                }
            }
            if (up) idx += cnt / 2;
            cnt >>= 1;
        } else {
            v[0] += __shfl_xor_sync(FULL_MASK, v[0], o);
            if (lane & o) owner = false;
        }
    }
    return v[0];
}

// One item (u, g) of NT tokens for a consumer warp: its I / 256 stages, then
// the reduction and the accumulator update.  Returns false if a wait ran out.
template <bool HF32, int NT>
__device__ __forceinline__ bool dt_item(const DownArgs& a, const DTLayout& L, const char* ring, uint64_t* full,
                                        uint64_t* empty, int& slot, uint32_t& par, int nks, int RT, int lane,
                                        int rw0, const int* tok, const float* wt, int rows, float* acc) {
    constexpr int NTP = NT == 3 ? 4 : NT;
    const int kr = (lane & 3) | ((lane >> 1) & 4);
    const int rr = ((lane >> 2) & 1) | ((lane >> 3) & 2);
    int r[DT_RL];
#pragma unroll
    for (int i = 0; i < DT_RL; ++i) r[i] = rw0 + 4 * i + rr;
    const int half = kr >> 2, ch = (kr & 3) * 2;
    float2 accv[DT_RL][NT];
#pragma unroll
    for (int i = 0; i < DT_RL; ++i)
#pragma unroll
        for (int t = 0; t < NT; ++t) accv[i][t] = make_float2(0.f, 0.f);
    for (int ks = 0; ks < nks; ++ks) {
        if (!mbar_wait(&full[slot], par)) return false;
        const char* st = ring + (size_t)slot * L.stage_bytes;
        uint4 cw[DT_RL][2];
        float sc[DT_RL];
#pragma unroll
        for (int i = 0; i < DT_RL; ++i) {
            const char* rowp = st + (size_t)half * RT * 128 + r[i] * 128;
#pragma unroll
            for (int c = 0; c < 2; ++c)
                cw[i][c] = *reinterpret_cast<const uint4*>(rowp + (((ch + c) ^ (r[i] & 7)) << 4));
            sc[i] = e8m0_to_float(*reinterpret_cast<const uint8_t*>(st + L.sc_off + r[i] * 8 + kr));
        }
        float2 part[DT_RL][NT];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            float4 hv[NT];
#pragma unroll
            for (int t = 0; t < NT; ++t) {
                if (HF32) {
                    hv[t] = *reinterpret_cast<const float4*>(st + L.h_off + t * (DT_KS * 4) + (q * 8 + kr) * 16);
                } else {
                    const uint2 b = *reinterpret_cast<const uint2*>(st + L.h_off + t * (DT_KS * 2) +
                                                                    (kr * 32 + q * 4) * 2);
                    const float2 lo = bf16x2_to_float2(b.x), hi = bf16x2_to_float2(b.y);
                    hv[t] = make_float4(lo.x, lo.y, hi.x, hi.y);
                }
            }
#pragma unroll
            for (int i = 0; i < DT_RL; ++i) {
                float2 w01, w23;
                e4m3x4_to_float((&cw[i][q >> 2].x)[q & 3], w01, w23);
#pragma unroll
                for (int t = 0; t < NT; ++t) {
                    const float2 h01 = make_float2(hv[t].x, hv[t].y), h23 = make_float2(hv[t].z, hv[t].w);
                    part[i][t] = q == 0 ? __fmul2_rn(h01, w01) : __ffma2_rn(h01, w01, part[i][t]);
                    part[i][t] = __ffma2_rn(h23, w23, part[i][t]);
                }
            }
        }
#pragma unroll
        for (int i = 0; i < DT_RL; ++i)
#pragma unroll
            for (int t = 0; t < NT; ++t) accv[i][t] = __ffma2_rn(part[i][t], make_float2(sc[i], sc[i]), accv[i][t]);
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
        if (++slot == L.S) {
            slot = 0;
            par ^= 1u;
        }
    }
    constexpr int N = DT_RL * NTP;  // value index = row slot * NTP + token
    float v[N];
#pragma unroll
    for (int i = 0; i < DT_RL; ++i)
#pragma unroll
        for (int t = 0; t < NTP; ++t) v[i * NTP + t] = t < NT ? accv[i][t < NT ? t : 0].x + accv[i][t < NT ? t : 0].y : 0.f;
    int idx;
    bool owner;
    const float dot = klane_reduce<N>(v, lane, idx, owner);
    const int i = idx / NTP, t = idx % NTP;
    int row = r[0];
#pragma unroll
    for (int ii = 1; ii < DT_RL; ++ii)
        if (ii == i) row = r[ii];
    if (owner && t < NT && row < rows) {
        int b = tok[0];
        float w = wt[0];
#pragma unroll
        for (int tt = 1; tt < NT; ++tt)
            if (tt == t) {
                b = tok[tt];
                w = wt[tt];
            }
        acc[row * a.s.B + b] += w * dot;
    }
    __syncwarp();
    return true;
}

template <bool HF32, int CW>
__global__ void __launch_bounds__((CW + 1) * 32, 2)
    down_tile_kernel(DownArgs a, const __grid_constant__ DTMaps maps, DTLayout L) {
    constexpr int RT = 8 * CW;
    extern __shared__ __align__(128) int smem_i[];
    const DecodeShape s = a.s;
    const RouteMap m = carve_map(smem_i, s, true);
    float* acc = reinterpret_cast<float*>(smem_i + map_ints(s, true));  // [RT][B]
    const uintptr_t raw = reinterpret_cast<uintptr_t>(smem_i) + L.ring_off;
    char* ring = reinterpret_cast<char*>((raw + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(ring + (size_t)L.S * L.stage_bytes);
    uint64_t* empty = full + DT_SMAX;
    if (threadIdx.x == 0) {
        for (int i = 0; i < L.S; ++i) {
            mbar_init(&full[i], 1 + 32);  // the producer's expect_tx arrival + one cp.async arrival per lane
            mbar_init(&empty[i], CW);
        }
        mbar_init_fence();
    }
    for (int i = threadIdx.x; i < RT * s.B; i += blockDim.x) acc[i] = 0.f;
    // the copy ring is idle until the map is built: it serves as the map's scratch
    build_route_map(m, a.ids, a.w, s, a.err, true, reinterpret_cast<int*>(ring),
                    L.S * L.stage_bytes / 4);  // ends with __syncthreads

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint32_t CL, rank;
    asm("mov.u32 %0, %%cluster_nctarank;" : "=r"(CL));
    asm("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
    const int o0 = (int)(blockIdx.x / CL) * RT;
    const int rows = min(RT, s.d - o0);
    const int ntot = m.hdr[0];
    const int nks = s.I / DT_KS;
    bool ok = true;

    if (warp == CW) {
        // ---------------- producer ----------------
        const uint64_t pol = l2_evict_first_policy();
        const int nb = s.I / 32;  // scale bytes per row
        const int hb = DT_KS * (HF32 ? 4 : 2);
        auto issue_w = [&](const DTCursor& c, int slot) {
            const int nt = min(DT_TC, m.ucnt[c.u] - c.g * DT_TC);
            const int e = m.uexp[c.u];
            const int sh = e >= s.E ? 1 : 0;
            const MXView vd = sh ? a.shd : a.wd;
            const size_t r0 = (size_t)(sh ? 0 : e) * s.d + o0;
            char* st = ring + (size_t)slot * L.stage_bytes;
            if (lane == 0) {
                mbar_arrive_expect_tx(&full[slot], 256 * RT + nt * hb);
                fence_proxy_async();
                tma_3d(st, &maps.w[sh], 0, (int)r0, c.ks * 2, &full[slot], pol);
            }
            const uint8_t* src = vd.s + r0 * nb + c.ks * 8;
            for (int rr = lane; rr < rows; rr += 32) cp_async_8(st + L.sc_off + rr * 8, src + (size_t)rr * nb);
            cp_async_mbar_arrive_noinc(&full[slot]);
        };
        auto issue_h = [&](const DTCursor& c, int slot) {
            const int nt = min(DT_TC, m.ucnt[c.u] - c.g * DT_TC);
            char* st = ring + (size_t)slot * L.stage_bytes;
            if (lane < nt) {
                const size_t hr = (size_t)m.hrow[m.uoff[c.u] + c.g * DT_TC + lane];
                const char* src = HF32 ? reinterpret_cast<const char*>(a.h32 + hr * s.I + c.ks * DT_KS)
                                       : reinterpret_cast<const char*>(a.h + hr * s.I + c.ks * DT_KS);
                fence_proxy_async();
                bulk_g2s_keep(st + L.h_off + lane * hb, src, hb, &full[slot]);
            }
        };
        DTCursor c{0, 0, 0, 0};
        dt_seek(c, m, ntot, (int)CL, (int)rank);
        DTCursor hc = c;
        uint32_t j = 0;  // stages issued
        // the first stages' weights do not depend on the gate/up pass
        for (; j < (uint32_t)L.S && c.u < ntot; ++j) {
            issue_w(c, (int)j);
            dt_advance(c, m, ntot, nks, (int)CL, (int)rank);
        }
        asm volatile("griddepcontrol.wait;" ::: "memory");
        for (uint32_t i = 0; i < j; ++i) {
            issue_h(hc, (int)i);
            dt_advance(hc, m, ntot, nks, (int)CL, (int)rank);
        }
        while (c.u < ntot) {
            const int slot = (int)(j % L.S);
            if (!mbar_wait(&empty[slot], ((j / L.S) - 1) & 1)) {
                ok = false;
                break;
            }
            issue_w(c, slot);
            __syncwarp();
            issue_h(c, slot);
            dt_advance(c, m, ntot, nks, (int)CL, (int)rank);
            ++j;
        }
        // never leave the CTA with a copy in flight
        for (uint32_t i = j > (uint32_t)L.S ? j - L.S : 0; i < j; ++i) mbar_wait(&full[i % L.S], (i / L.S) & 1);
    } else {
        // ---------------- consumers ----------------
        DTCursor c{0, 0, 0, 0};
        dt_seek(c, m, ntot, (int)CL, (int)rank);
        int slot = 0;
        uint32_t par = 0;
        const int rw0 = warp * 8;
        while (c.u < ntot && ok) {
            const int e0 = m.uoff[c.u] + c.g * DT_TC;
            const int nt = min(DT_TC, m.ucnt[c.u] - c.g * DT_TC);
            const int* tk = m.tok + e0;
            const float* wp = m.wt + e0;
            switch (nt) {
                case 1: ok = dt_item<HF32, 1>(a, L, ring, full, empty, slot, par, nks, RT, lane, rw0, tk, wp, rows, acc); break;
                case 2: ok = dt_item<HF32, 2>(a, L, ring, full, empty, slot, par, nks, RT, lane, rw0, tk, wp, rows, acc); break;
                case 3: ok = dt_item<HF32, 3>(a, L, ring, full, empty, slot, par, nks, RT, lane, rw0, tk, wp, rows, acc); break;
                default: ok = dt_item<HF32, 4>(a, L, ring, full, empty, slot, par, nks, RT, lane, rw0, tk, wp, rows, acc); break;
            }
            c.ks = nks - 1;
            dt_advance(c, m, ntot, nks, (int)CL, (int)rank);
        }
    }
    // add the cluster's partial sums in rank order; CTA `rank` stores rows
    // [rank * RR, (rank + 1) * RR) of the block
    __syncthreads();
    if (CL > 1) cluster_sync_all();
    const int RR = (RT + (int)CL - 1) / (int)CL;
    for (int i = threadIdx.x; i < RR * s.B; i += blockDim.x) {
        const int rl = (int)rank * RR + i % RR, b = i / RR;
        if (rl < rows) {
            const float* p = acc + (size_t)rl * s.B + b;
            float sum = 0.f;
            for (uint32_t q = 0; q < CL; ++q) sum += CL > 1 ? ld_cluster_f32(p, q) : *p;
            a.y[(size_t)b * s.d + o0 + rl] = __bfloat16_as_ushort(__float2bfloat16_rn(sum));
        }
    }
    if (CL > 1) cluster_sync_all();  // keep this CTA's accumulators alive for its peers
    if (!ok && lane == 0) atomicOr(a.err, MOE_DEVERR_TIMEOUT);
}

// -------------------------------------------------------------- host -----

size_t down_smem_bytes(const DecodeShape& s) {
    const int G = 32 / lanes_per_row(s.I);
    return map_ints(s, true) * 4 + (size_t)DEC_WARPS * G * s.B * 4;
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

// Bulk copies: the [rows x I] weight block and its scale block must start
// on 16-byte boundaries (I % 256 == 0 keeps them there when the arrays do).
static bool down_v4_ok(const DecodeShape& s, MXView wd, MXView shd) {
    if (s.I % 256 || s.d % 2) return false;
    if (!aligned16(wd.s) || (s.S && !aligned16(shd.s))) return false;
    return true;
}

// Rows per warp for down v4: ~96 weight bytes per lane per stage.
static int dn4_rw(int I) { return I >= 2048 ? 1 : 2; }

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

static DN4Geom dn4_geom(const DecodeShape& s, int RW, int sm_count) {
    const long slots = 2L * sm_count;
    DN4Geom best{8, 1};
    long best_cost = -1;
    for (int cw = 8; cw >= 7; --cw) {
        if (cw == 7 && RW == 1) continue;
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


// ---- down, row tiles: plan and launch -----------------------------------

// Preconditions of the row-tile kernel: whole 256-element slabs; the code
// arrays 16-byte aligned (tensor copies), the scale arrays 8-byte aligned
// (8-byte copies of a slab's scale bytes; I % 256 == 0 keeps every row's
// scales 8-byte aligned when the array is).
static bool down_tile_ok(const DecodeShape& s, MXView wd, MXView shd) {
    if (s.I % DT_KS) return false;
    if (!aligned16(wd.w) || (reinterpret_cast<uintptr_t>(wd.s) & 7)) return false;
    if (s.S && (!aligned16(shd.w) || (reinterpret_cast<uintptr_t>(shd.s) & 7))) return false;
    return true;
}

struct DTPlan {
    int cw, cl, bps;
    DTLayout L;
};

// Consumer warps (8, 7 or 6: 64-, 56- or 48-row blocks), CTAs per SM (two
// with at least three ring stages, else one with at least two) and cluster
// size: the least estimated work of the busiest CTA slot, i.e. waves x rows
// x items per CTA, with items estimated as the distinct experts the call can
// have plus the shared expert's token groups.  Cluster sizes are at most 8
// (portable) and never above the item estimate.
static bool dt_plan(const DecodeShape& s, bool hf32, const DeviceInfo& di, DTPlan* out) {
    const long items = std::min<long>((long)s.B * s.k, s.E) + (long)s.S * ((s.B + DT_TC - 1) / DT_TC);
    long best = -1;
    for (int cw = 8; cw >= 6; --cw) {
        const int RT = 8 * cw;
        DTLayout L{};
        int bps = 0;
        const int two = std::min(di.max_smem_optin, di.smem_per_sm / 2 - 1024);
        L = dt_layout(s, RT, hf32, two);
        if (L.S >= 3) {
            bps = 2;
        } else {
            L = dt_layout(s, RT, hf32, di.max_smem_optin);
            if (L.S >= 2) bps = 1;
        }
        if (!bps) continue;
        const long nblk = (s.d + RT - 1) / RT, slots = (long)bps * di.sm_count;
        for (int cl = 1; cl <= 8; ++cl) {
            if (cl > 1 && cl > items) break;
            const long waves = (nblk * cl + slots - 1) / slots;
            const long cost = waves * RT * ((items + cl - 1) / cl);
            if (best < 0 || cost < best) {
                best = cost;
                *out = DTPlan{cw, cl, bps, L};
            }
        }
    }
    return best >= 0;
}

static bool dt_maps(const DownArgs& a, int RT, DTMaps* maps) {
    const DecodeShape& s = a.s;
    if (!map_3d_u8_blocks(&maps->w[0], a.wd.w, (uint64_t)s.E * s.d, s.I, RT, 2)) return false;
    if (s.S) return map_3d_u8_blocks(&maps->w[1], a.shd.w, (uint64_t)s.d, s.I, RT, 2);
    maps->w[1] = maps->w[0];  // no shared expert: any valid map
    return true;
}

template <bool HF32, int CW>
static cudaError_t launch_down_tile_k(const DownArgs& a, const DTPlan& pl, const DTMaps& maps, int dev,
                                      cudaStream_t st, bool pdl) {
    auto* fn = down_tile_kernel<HF32, CW>;
    static std::mutex mu;
    static int attr_smem[64] = {0};
    {
        std::lock_guard<std::mutex> lock(mu);
        if (dev >= 64 || attr_smem[dev] < pl.L.smem) {
            cudaError_t err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   std::max(pl.L.smem, 48 * 1024));
            if (err != cudaSuccess) return err;
            if (dev < 64) attr_smem[dev] = pl.L.smem;
        }
    }
    constexpr int RT = 8 * CW;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((a.s.d + RT - 1) / RT * pl.cl));
    cfg.blockDim = dim3((CW + 1) * 32);
    cfg.dynamicSmemBytes = (size_t)pl.L.smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (pl.cl > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = (unsigned)pl.cl;
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
    return cudaLaunchKernelEx(&cfg, fn, a, maps, pl.L);
}

template <bool HF32>
static cudaError_t launch_down_tile(const DownArgs& a, const DTPlan& pl, const DTMaps& maps, int dev,
                                    cudaStream_t st, bool pdl) {
    switch (pl.cw) {
        case 8: return launch_down_tile_k<HF32, 8>(a, pl, maps, dev, st, pdl);
        case 7: return launch_down_tile_k<HF32, 7>(a, pl, maps, dev, st, pdl);
        default: return launch_down_tile_k<HF32, 6>(a, pl, maps, dev, st, pdl);
    }
}

bool down_reads_h32(const DecodeShape& s, MXView wd, MXView shd) {
    DeviceInfo di;
    DTPlan pl;
    return device_info(&di) == cudaSuccess && down_tile_ok(s, wd, shd) && dt_plan(s, true, di, &pl);
}

cudaError_t launch_down(const DecodeShape& s, const void* h, bool h32, const int32_t* ids, const float* w,
                        MXView wd, MXView shd, void* y, cudaStream_t st, bool after_gate_up) {
    DeviceInfo di;
    cudaError_t err = device_info(&di);
    if (err != cudaSuccess) return err;
    int dev = 0;
    if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
    DownArgs a{s, (const uint16_t*)h, ids, w, wd, shd, (uint16_t*)y, di.err_word, 1, nullptr};
    if (h32) {  // only ever set when down_reads_h32() said the row-tile kernel takes this call
        a.h = nullptr;
        a.h32 = static_cast<const float*>(h);
    }
    if (down_tile_ok(s, wd, shd)) {
        DTPlan pl;
        if (dt_plan(s, h32, di, &pl)) {
            DTMaps maps;
            if (dt_maps(a, 8 * pl.cw, &maps))
                return h32 ? launch_down_tile<true>(a, pl, maps, dev, st, after_gate_up)
                           : launch_down_tile<false>(a, pl, maps, dev, st, after_gate_up);
        }
    }
    if (h32) return cudaErrorInvalidValue;
    if (down_v4_ok(s, wd, shd)) {
        // rows per block and s.d even: every block's scale bytes are a multiple of 16
        const int RW = dn4_rw(s.I);
        const DN4Geom g = dn4_geom(s, RW, di.sm_count);
        const size_t smem4 = down_v4_smem(s, g.cw * RW);
        if (s.d % 2 == 0 && smem4 <= (size_t)di.max_smem_optin) {
            switch (RW) {
                case 1: return launch_down_v4_rw<1>(a, g, smem4, dev, st, after_gate_up);
                default: return launch_down_v4_rw<2>(a, g, smem4, dev, st, after_gate_up);
            }
        }
    }
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
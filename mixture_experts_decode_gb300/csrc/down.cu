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


template <int RW, int NT, int NCH = 0, bool HF32 = false, bool FP4 = false>
__device__ __forceinline__ bool dn3_group(const DownArgs& a, const DN3Layout& L, const char* st, uint64_t* full,
                                          uint64_t* empty, uint32_t parity, int cw, int lane, const int* toks,
                                          const float* ws, int nt, float* acc_rows) {
    constexpr int NTP = NT == 3 ? 4 : NT;
    const DecodeShape& s = a.s;
    if (!mbar_wait(full, parity)) return false;
    constexpr int CB = FP4 ? 2 : 1;  // K elements per code byte
    const uint8_t* wb = reinterpret_cast<const uint8_t*>(st + L.w_off) + (size_t)cw * RW * (s.I / CB);
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
        float2 hf[NT][4];  // the tokens' eight activations as FP32, for all rows
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            if (HF32) {  // already FP32, in h32_pos order: two contiguous 16-byte loads
                const float* hr = reinterpret_cast<const float*>(hb) + (size_t)t * s.I + (k0 & ~255) + lane * 4;
                const float4 u0 = *reinterpret_cast<const float4*>(hr);
                const float4 u1 = *reinterpret_cast<const float4*>(hr + 128);
                hf[t][0] = make_float2(u0.x, u0.y);
                hf[t][1] = make_float2(u0.z, u0.w);
                hf[t][2] = make_float2(u1.x, u1.y);
                hf[t][3] = make_float2(u1.z, u1.w);
            } else {
                const uint4 hv = *reinterpret_cast<const uint4*>(hb + (size_t)t * s.I + k0);
#pragma unroll
                for (int q = 0; q < 4; ++q) hf[t][q] = bf16x2_to_float2((&hv.x)[q]);
            }
        }
#pragma unroll
        for (int r = 0; r < RW; ++r) {
            const float sc = e8m0_to_float(sb[r * (s.I / 32) + (k0 >> 5)]);
            float2 wq[4];
            if (FP4) {  // eight E2M1 codes in one 32-bit word
                e2m1x8_to_float(*reinterpret_cast<const uint32_t*>(wb + (size_t)r * (s.I / 2) + k0 / 2), wq);
            } else {
                const uint2 wv = *reinterpret_cast<const uint2*>(wb + (size_t)r * s.I + k0);
                e4m3x4_to_float(wv.x, wq[0], wq[1]);
                e4m3x4_to_float(wv.y, wq[2], wq[3]);
            }
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

// hf32: the intermediate arrives as FP32 (h32_pos order), else BF16.
__host__ __device__ inline DN3Layout dn4_layout(const DecodeShape& s, int RT, bool hf32, bool fp4 = false) {
    DN3Layout L;
    L.w_off = 0;
    L.s_off = RT * (fp4 ? s.I / 2 : s.I);
    L.h_off = (L.s_off + RT * (s.I / 32) + 127) / 128 * 128;
    L.stage_bytes = (L.h_off + TC * s.I * (hf32 ? 4 : 2) + 127) / 128 * 128;
    const int S = DN4_RING_BYTES / L.stage_bytes;
    L.S = S > DN4_SMAX ? DN4_SMAX : S;
    return L;
}

__host__ __device__ inline size_t dn4_smem_offset(const DecodeShape& s, int RT) {
    const size_t acc = (size_t)RT * s.B * 4;
    return (map_ints(s, true) * 4 + acc + 127) / 128 * 128;
}

template <int RW, int CL, int NCH, int CW, bool HF32, bool FP4>
__global__ void __launch_bounds__((CW + 1) * 32, 2) down_v4_kernel(DownArgs a) {
    constexpr int RT = CW * RW;
    extern __shared__ __align__(128) int smem_i[];
    const DecodeShape s = a.s;
    const RouteMap m = carve_map(smem_i, s, true);
    float* acc = reinterpret_cast<float*>(smem_i + map_ints(s, true));  // [RT][B]
    const uintptr_t raw = reinterpret_cast<uintptr_t>(smem_i) + dn4_smem_offset(s, RT);
    char* ring = reinterpret_cast<char*>((raw + 127) & ~uintptr_t(127));
    const DN3Layout L = dn4_layout(s, RT, HF32, FP4);
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
    // (the one-warp map for small B is left out here: in this kernel it
    // measured slower at B = 32 through register allocation)
    build_route_map(m, a.ids, a.w, s, a.err, true, reinterpret_cast<int*>(ring),
                    L.S * L.stage_bytes / 4, false);  // ends with __syncthreads

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
        const int cbytes = FP4 ? s.I / 2 : s.I;  // code bytes per row
        const uint32_t wbytes = rows * cbytes, sbytes = rows * nb, hbytes = s.I * (HF32 ? 4 : 2);
        auto issue_w = [&](int u, int t0, int slot) {
            const int nt = min(TC, m.ucnt[u] - t0);
            const int e = m.uexp[u];
            const bool sh = e >= s.E;
            const MXView vd = sh ? a.shd : a.wd;
            const size_t r0 = (sh ? 0 : (size_t)e) * s.d + o0;
            char* st = ring + (size_t)slot * L.stage_bytes;
            if (lane == 0) {
                mbar_arrive_expect_tx(&full[slot], wbytes + sbytes + nt * hbytes);
                fence_proxy_async();
                bulk_g2s(st + L.w_off, vd.w + r0 * cbytes, wbytes, &full[slot], pol);
                bulk_g2s(st + L.s_off, vd.s + r0 * nb, sbytes, &full[slot], pol);
            }
        };
        auto issue_h = [&](int u, int t0, int slot) {
            const int nt = min(TC, m.ucnt[u] - t0);
            char* st = ring + (size_t)slot * L.stage_bytes;
            if (lane < nt) {
                fence_proxy_async();
                const size_t hr = (size_t)m.hrow[m.uoff[u] + t0 + lane];
                const void* src = HF32 ? static_cast<const void*>(a.h32 + hr * s.I)
                                       : static_cast<const void*>(a.h + hr * s.I);
                bulk_g2s_keep(st + L.h_off + (size_t)lane * hbytes, src, hbytes, &full[slot]);
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
                    case 1: ok = dn3_group<RW, 1, NCH, HF32, FP4>(a, L, st, &full[slot], &empty[slot], par, warp, lane, tk, wsp, nt, acc_rows); break;
                    case 2: ok = dn3_group<RW, 2, NCH, HF32, FP4>(a, L, st, &full[slot], &empty[slot], par, warp, lane, tk, wsp, nt, acc_rows); break;
                    case 3: ok = dn3_group<RW, 3, NCH, HF32, FP4>(a, L, st, &full[slot], &empty[slot], par, warp, lane, tk, wsp, nt, acc_rows); break;
                    default: ok = dn3_group<RW, 4, NCH, HF32, FP4>(a, L, st, &full[slot], &empty[slot], par, warp, lane, tk, wsp, nt, acc_rows); break;
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

static size_t down_v4_smem(const DecodeShape& s, int RT, bool hf32, bool fp4 = false) {
    const DN3Layout L = dn4_layout(s, RT, hf32, fp4);
    if (L.S < 2) return ~(size_t)0;
    return dn4_smem_offset(s, RT) + (size_t)L.S * L.stage_bytes + 2 * DN4_SMAX * sizeof(uint64_t) + 128;
}

template <int RW, int CL, int NCH, int CW, bool HF32, bool FP4>
static cudaError_t launch_down_v4_k(const DownArgs& a, size_t smem, int dev, cudaStream_t st, bool pdl) {
    static std::mutex mu;
    static size_t attr_smem[64] = {0};
    {
        std::lock_guard<std::mutex> lock(mu);
        if (dev >= 64 || attr_smem[dev] < smem) {
            cudaError_t err = cudaFuncSetAttribute(down_v4_kernel<RW, CL, NCH, CW, HF32, FP4>,
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
    return cudaLaunchKernelEx(&cfg, down_v4_kernel<RW, CL, NCH, CW, HF32, FP4>, a);
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

template <int RW, int NCH, int CW, bool HF32, bool FP4>
static cudaError_t launch_down_v4_cl(const DownArgs& a, int cl, size_t smem, int dev, cudaStream_t st, bool pdl) {
    switch (cl) {
        case 1: return launch_down_v4_k<RW, 1, NCH, CW, HF32, FP4>(a, smem, dev, st, pdl);
        case 2: return launch_down_v4_k<RW, 2, NCH, CW, HF32, FP4>(a, smem, dev, st, pdl);
        default:
            if constexpr ((CW * RW) % 4 == 0) return launch_down_v4_k<RW, 4, NCH, CW, HF32, FP4>(a, smem, dev, st, pdl);
            return cudaErrorInvalidValue;
    }
}

template <int RW, int NCH, bool HF32, bool FP4>
static cudaError_t launch_down_v4_cw(const DownArgs& a, const DN4Geom& g, size_t smem, int dev, cudaStream_t st,
                                     bool pdl) {
    if constexpr (RW >= 2) {
        if (g.cw == 7) return launch_down_v4_cl<RW, NCH, 7, HF32, FP4>(a, g.cl, smem, dev, st, pdl);
    }
    return launch_down_v4_cl<RW, NCH, 8, HF32, FP4>(a, g.cl, smem, dev, st, pdl);
}

// The chunk loop is unrolled for the common lengths (I = 768 at two rows per
// warp, I = 2048 at one), a run-time loop otherwise.
template <int RW, bool HF32, bool FP4 = false>
static cudaError_t launch_down_v4_rw(const DownArgs& a, const DN4Geom& g, size_t smem, int dev, cudaStream_t st,
                                     bool pdl) {
    const int nch = a.s.I / 256;
    if constexpr (RW >= 2) {
        if (nch == 3) return launch_down_v4_cw<RW, 3, HF32, FP4>(a, g, smem, dev, st, pdl);
    }
    if constexpr (RW == 1) {
        if (nch == 8) return launch_down_v4_cw<RW, 8, HF32, FP4>(a, g, smem, dev, st, pdl);
    }
    return launch_down_v4_cw<RW, 0, HF32, FP4>(a, g, smem, dev, st, pdl);
}

// The v4 kernel takes the call (and can read the FP32 intermediate).
static bool down_v4_takes(const DecodeShape& s, MXView wd, MXView shd, const DeviceInfo& di, bool hf32) {
    if (!down_v4_ok(s, wd, shd)) return false;
    const DN4Geom g = dn4_geom(s, dn4_rw(s.I), di.sm_count);
    return down_v4_smem(s, g.cw * dn4_rw(s.I), hf32) <= (size_t)di.max_smem_optin;
}

bool launch_down_grouped_fp4(const DecodeShape& s, const void* h, const int32_t* ids, const float* w, MXView wd,
                             MXView shd, void* y, cudaStream_t st, cudaError_t* err) {
    DeviceInfo di;
    if ((*err = device_info(&di)) != cudaSuccess) return true;
    int dev = 0;
    if ((*err = cudaGetDevice(&dev)) != cudaSuccess) return true;
    if (!down_v4_ok(s, wd, shd)) return false;
    const int RW = dn4_rw(s.I);
    const DN4Geom g = dn4_geom(s, RW, di.sm_count);
    const size_t smem4 = down_v4_smem(s, g.cw * RW, false, true);
    if (smem4 > (size_t)di.max_smem_optin) return false;
    DownArgs a{s, (const uint16_t*)h, ids, w, wd, shd, (uint16_t*)y, di.err_word, 1, nullptr};
    *err = RW == 1 ? launch_down_v4_rw<1, false, true>(a, g, smem4, dev, st, false)
                   : launch_down_v4_rw<2, false, true>(a, g, smem4, dev, st, false);
    return true;
}

bool down_reads_h32(const DecodeShape& s, MXView wd, MXView shd) {
    DeviceInfo di;
    return device_info(&di) == cudaSuccess && down_v4_takes(s, wd, shd, di, true);
}

cudaError_t launch_down(const DecodeShape& s, const void* h, bool h32, const int32_t* ids, const float* w,
                        MXView wd, MXView shd, void* y, cudaStream_t st, bool after_gate_up) {
    DeviceInfo di;
    cudaError_t err = device_info(&di);
    if (err != cudaSuccess) return err;
    int dev = 0;
    if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
    DownArgs a{s, (const uint16_t*)h, ids, w, wd, shd, (uint16_t*)y, di.err_word, 1, nullptr};
    if (h32) {  // only ever set when down_reads_h32() said the v4 kernel takes this call
        a.h = nullptr;
        a.h32 = static_cast<const float*>(h);
    }
    if (down_v4_takes(s, wd, shd, di, h32)) {
        const int RW = dn4_rw(s.I);
        const DN4Geom g = dn4_geom(s, RW, di.sm_count);
        const size_t smem4 = down_v4_smem(s, g.cw * RW, h32);
        if (RW == 1)
            return h32 ? launch_down_v4_rw<1, true>(a, g, smem4, dev, st, after_gate_up)
                       : launch_down_v4_rw<1, false>(a, g, smem4, dev, st, after_gate_up);
        return h32 ? launch_down_v4_rw<2, true>(a, g, smem4, dev, st, after_gate_up)
                   : launch_down_v4_rw<2, false>(a, g, smem4, dev, st, after_gate_up);
    }
    if (h32) return cudaErrorInvalidValue;
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
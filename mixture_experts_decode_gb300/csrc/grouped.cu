// grouped.cu -- the expert-centric path of the MoE expert-FFN layer, for
// large batches and prefill: moe_align_block_size sorts the (token, slot)
// pairs by expert into blocks of GR_BM rows of one expert each, then two
// grouped GEMMs run on the 5th-generation tensor cores and a combine step
// adds each token's k rows with their routing weights ("Warp decode",
// section "Warp decode 與 Composer 訓練": prefill and large batches keep
// expert-centric packing; the align page's MoE Align & Sort feeds exactly
// such grouped GEMMs).
//
//   gemm1 (gate/up): one CTA per (block of GR_BM sorted slots, GR_BN rows of
//     I).  A = the slots' token rows of x (BF16; the pad slots zero), B = the
//     block's expert's W_gate and W_up rows, dequantised from MXFP8 to BF16
//     in shared memory by the CTA's threads (exact: an E4M3 value times a
//     power of two has at most four significant bits), D = two FP32
//     accumulators in tensor memory.  Epilogue: h = bf16(SiLU(g) * u) per
//     sorted slot.
//   gemm2 (down): A = h of the block's slots, B = the expert's W_down rows,
//     D = FP32 in tensor memory; the epilogue stores each real slot's row
//     of partial outputs (FP32) at its flat slot index.
//   combine: y[t][o] = bf16( sum_j w[t][j] * out[t*k + j][o] ), the k slots
//     in order.
// Each MMA is tcgen05.mma kind::f16 (BF16 x BF16 -> FP32), M = 128, N =
// 128, K = 16, issued by one thread from K-major 128-byte-swizzled shared
// memory tiles; completion is signalled to an mbarrier by tcgen05.commit.
// K advances in chunks of 64 through a two-stage ring: the copies of chunk
// c + 1 (cp.async into the swizzled positions) and its dequantisation
// overlap the MMAs of chunk c.  The products are those of the MX values
// exactly; sums are FP32 (the tensor core's order).  With act_mx set, x and
// h are first rounded through MXFP8 (moe_mx_requant): the conventional
// path's activations.
#include <cstdint>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace moedec {

constexpr int GR_BM = GROUPED_BLOCK;  // sorted slots per block (the MMA's M)
constexpr int GR_BN = 128;   // weight rows per CTA (the MMA's N)
constexpr int GR_KC = 64;    // K elements per chunk (one 128-byte swizzle row of BF16)
constexpr int GR_THREADS = 128;

struct GRArgs {
    const uint16_t* a_src;     // gemm1: x [T][d] (rows by token); gemm2: h_sorted [n_sorted][I]
    const int32_t* sorted;     // flat slot of each sorted row (T*k = pad)
    const int32_t* expert_ids; // expert of each block
    const int32_t* ntpp;       // rows used (a multiple of GR_BM)
    const uint8_t *w0, *s0;    // gemm1: W_gate; gemm2: W_down (codes, E8M0 scales)
    const uint8_t *w1, *s1;    // gemm1: W_up
    uint16_t* h_sorted;        // gemm1 output [n_sorted][I] BF16
    float* out;                // gemm2 output [T*k][d] FP32 by flat slot
    int T, k, E, d, I;
    int* err;
};

// One stage: the A tile and each B matrix's raw codes and BF16 tile.
template <int NB>
struct __align__(1024) GRStage {
    uint16_t a[GR_BM * GR_KC];        // [row][64] BF16, 128-byte swizzle (8-row atoms of 1024 B)
    uint16_t b[NB][GR_BN * GR_KC];    // [row][64] BF16, same layout
    uint8_t raw[NB][GR_BN * GR_KC];   // [row][64] E4M3 codes as copied
};

// 16 bytes global -> shared (L2 only); src_bytes = 0 writes zeros.
__device__ __forceinline__ void cp_async_16_plain(void* smem, const void* gmem, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_addr(smem)), "l"(gmem), "r"(src_bytes)
                 : "memory");
}

__device__ __forceinline__ uint32_t swz128(int row, int chunk16) {
    return (uint32_t)(row * 128 + ((chunk16 ^ (row & 7)) << 4));
}

// Shared-memory matrix descriptor of a K-major tile in the 128-byte swizzle
// layout: start address >> 4 in bits [0, 14), leading-dimension offset
// (unused for swizzled K-major tiles; 1) in [16, 30), stride between
// 8-row groups (1024 B) >> 4 in [32, 46), descriptor version 1 in [46, 48),
// layout 128-byte swizzle (2) in [61, 64).
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t saddr) {
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | (1ull << 16) | ((uint64_t)(1024 >> 4) << 32) | (1ull << 46) |
           (2ull << 61);
}

// Instruction descriptor of tcgen05.mma kind::f16: D FP32 (bits [4,6) = 1),
// A and B BF16 ([7,10) = [10,13) = 1), both K-major (bits 15, 16 = 0),
// N >> 3 in [17, 23), M >> 4 in [24, 29).
__host__ __device__ constexpr uint32_t gr_idesc(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{ .reg .pred p; setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void umma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 consecutive FP32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// NB = 2: gemm1 (gate, up; K = d, N over I); NB = 1: gemm2 (down; K = I, N over d).
template <int NB>
__global__ void __launch_bounds__(GR_THREADS, 1) grouped_mma_kernel(GRArgs a) {
    const int blk = blockIdx.x;
    if (blk * GR_BM >= *a.ntpp) return;  // a block past the used rows: nothing to do (uniform exit)
    extern __shared__ __align__(128) unsigned char gr_smem[];
    const uintptr_t base = (reinterpret_cast<uintptr_t>(gr_smem) + 1023) & ~uintptr_t(1023);
    GRStage<NB>* stage = reinterpret_cast<GRStage<NB>*>(base);
    const int K = NB == 2 ? a.d : a.I;         // contraction length
    const int NK = K / GR_KC;
    const int nsc = K / 32;                    // scale bytes per weight row
    uint8_t* scales = reinterpret_cast<uint8_t*>(stage + 2);  // [NB][GR_BN][nsc]
    uint64_t* bars = reinterpret_cast<uint64_t*>(scales + ((NB * GR_BN * nsc + 15) & ~15));
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int e = a.expert_ids[blk];
    const int n0 = blockIdx.y * GR_BN;
    const int rows_w = NB == 2 ? a.I : a.d;    // weight rows per expert
    const int64_t pad = (int64_t)a.T * a.k;

    if (tid == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        mbar_init_fence();
    }
    if (warp == 0) {  // tensor memory: NB x 128 FP32 columns
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                     "r"(NB * 128)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    // this CTA's weight rows' scale bytes (32-bit loads: K % 128 == 0 keeps rows 4-byte aligned)
    for (int p = 0; p < NB; ++p) {
        const uint8_t* sp = (p ? a.s1 : a.s0) + ((int64_t)e * rows_w + n0) * nsc;
        const int words = GR_BN * nsc / 4;
        for (int i = tid; i < words; i += GR_THREADS)
            reinterpret_cast<uint32_t*>(scales + p * GR_BN * nsc)[i] = reinterpret_cast<const uint32_t*>(sp)[i];
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // source row of each of this thread's A rows (8 chunks of 16 B per row, 8 threads per row)
    auto issue_chunk = [&](int kc, int st) {
        GRStage<NB>& S = stage[st];
        for (int q = tid; q < GR_BM * 8; q += GR_THREADS) {
            const int row = q >> 3, c = q & 7;
            const char* src;
            int bytes = 16;
            if (NB == 2) {
                const int64_t f = a.sorted[(int64_t)blk * GR_BM + row];
                const int64_t t = f < pad ? f / a.k : 0;
                if (f >= pad) bytes = 0;  // pad slot: zero row
                src = reinterpret_cast<const char*>(a.a_src + t * a.d + (int64_t)kc * GR_KC) + c * 16;
            } else {
                src = reinterpret_cast<const char*>(a.a_src + ((int64_t)blk * GR_BM + row) * a.I +
                                                    (int64_t)kc * GR_KC) + c * 16;
            }
            cp_async_16_plain(reinterpret_cast<char*>(S.a) + swz128(row, c), src, bytes);
        }
        for (int p = 0; p < NB; ++p) {
            const uint8_t* wp = (p ? a.w1 : a.w0) + ((int64_t)e * rows_w + n0) * K + (int64_t)kc * GR_KC;
            for (int q = tid; q < GR_BN * 4; q += GR_THREADS) {
                const int row = q >> 2, c = q & 3;
                cp_async_16_plain(S.raw[p] + row * GR_KC + c * 16, wp + (int64_t)row * K + c * 16, 16);
            }
        }
        cp_async_commit();
    };

    constexpr uint32_t IDESC = gr_idesc(GR_BM, GR_BN);
    issue_chunk(0, 0);
    bool ok = true;
    for (int kc = 0; kc < NK; ++kc) {
        const int st = kc & 1;
        if (kc + 1 < NK) {
            // the MMAs of chunk kc - 1 read the other stage: wait before refilling it
            const bool done = kc < 1 || mbar_wait(&bars[(kc + 1) & 1], ((kc - 1) >> 1) & 1);
            if (__syncthreads_or(!done)) {  // a wait gave up: every thread leaves together
                ok = false;
                break;
            }
            issue_chunk(kc + 1, (kc + 1) & 1);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        // dequantise this chunk's weight rows: item = (row, 16 codes)
        GRStage<NB>& S = stage[st];
        for (int p = 0; p < NB; ++p) {
            for (int q = tid; q < GR_BN * 4; q += GR_THREADS) {
                const int row = q >> 2, c = q & 3;
                const uint4 w4 = *reinterpret_cast<const uint4*>(S.raw[p] + row * GR_KC + c * 16);
                const float sc = e8m0_to_float(scales[p * GR_BN * nsc + row * nsc + kc * 2 + (c >> 1)]);
                uint32_t o[8];
#pragma unroll
                for (int wq = 0; wq < 4; ++wq) {
                    float2 lo, hi;
                    e4m3x4_to_float((&w4.x)[wq], lo, hi);
                    const __nv_bfloat162 b0 = __floats2bfloat162_rn(lo.x * sc, lo.y * sc);
                    const __nv_bfloat162 b1 = __floats2bfloat162_rn(hi.x * sc, hi.y * sc);
                    memcpy(&o[wq * 2], &b0, 4);
                    memcpy(&o[wq * 2 + 1], &b1, 4);
                }
                char* dst = reinterpret_cast<char*>(S.b[p]);
                *reinterpret_cast<uint4*>(dst + swz128(row, 2 * c)) = make_uint4(o[0], o[1], o[2], o[3]);
                *reinterpret_cast<uint4*>(dst + swz128(row, 2 * c + 1)) = make_uint4(o[4], o[5], o[6], o[7]);
            }
        }
        fence_proxy_async();  // the tiles' generic-proxy writes, before the tensor cores read them
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            const uint32_t a0 = smem_addr(S.a);
#pragma unroll
            for (int p = 0; p < NB; ++p) {
                const uint32_t b0 = smem_addr(S.b[p]);
#pragma unroll
                for (int kk = 0; kk < GR_KC / 16; ++kk)
                    umma_bf16(tmem + p * 128, umma_desc_sw128(a0 + kk * 32), umma_desc_sw128(b0 + kk * 32), IDESC,
                              (kc > 0 || kk > 0) ? 1u : 0u);
            }
            umma_commit(&bars[st]);
        }
    }
    cp_async_wait<0>();  // no copy still in flight on any exit from the loop
    // all MMAs done (they complete in order: the last commit covers them)
    const bool done = ok && mbar_wait(&bars[(NK - 1) & 1], ((NK - 1) >> 1) & 1);
    const bool failed = __syncthreads_or(!done);
    tc_fence_after();

    if (!failed) {
        const int m = warp * 32 + lane;                      // this thread's accumulator row
        const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
        const int64_t srow = (int64_t)blk * GR_BM + m;
        const int64_t f = a.sorted[srow];
        if (NB == 2) {
            for (int c0 = 0; c0 < GR_BN; c0 += 32) {
                float g[32], u[32];
                tmem_ld32(lane_base + c0, g);
                tmem_ld32(lane_base + 128 + c0, u);
                uint32_t o[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    float h0 = g[2 * i] / (1.0f + expf(-g[2 * i])) * u[2 * i];
                    float h1 = g[2 * i + 1] / (1.0f + expf(-g[2 * i + 1])) * u[2 * i + 1];
                    if (f >= pad) h0 = h1 = 0.f;
                    const __nv_bfloat162 hb = __floats2bfloat162_rn(h0, h1);
                    memcpy(&o[i], &hb, 4);
                }
                uint4* dst = reinterpret_cast<uint4*>(a.h_sorted + srow * a.I + n0 + c0);
#pragma unroll
                for (int i = 0; i < 4; ++i) dst[i] = make_uint4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
            }
        } else {
            for (int c0 = 0; c0 < GR_BN; c0 += 32) {
                float v[32];
                tmem_ld32(lane_base + c0, v);
                if (f < pad) {
                    float4* dst = reinterpret_cast<float4*>(a.out + f * a.d + n0 + c0);
#pragma unroll
                    for (int i = 0; i < 8; ++i) dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(NB * 128) : "memory");
    }
    if (tid == 0 && failed) atomicOr(a.err, MOE_DEVERR_TIMEOUT);
}

// y[t][o] = bf16( sum_j w[t][j] * out[t*k + j][o] ), j in order; a slot
// whose expert id is outside [0, E) (never placed by the sort) adds nothing.
__global__ void grouped_combine_kernel(const float* __restrict__ out, const float* __restrict__ w,
                                       const int32_t* __restrict__ ids, int T, int k, int E, int d,
                                       uint16_t* __restrict__ y) {
    const int64_t n = (int64_t)T * d;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t t = i / d, o = i - t * d;
        float acc = 0.f;
        for (int j = 0; j < k; ++j)
            if ((unsigned)ids[t * k + j] < (unsigned)E) acc = fmaf(w[t * k + j], out[(t * k + j) * d + o], acc);
        y[i] = __bfloat16_as_ushort(__float2bfloat16_rn(acc));
    }
}

template <int NB>
static size_t grouped_smem(int K) {
    return 1024 + 2 * sizeof(GRStage<NB>) + ((NB * GR_BN * (K / 32) + 15) & ~15) + 2 * sizeof(uint64_t) + 8;
}

template <int NB>
static cudaError_t launch_grouped_mma(const GRArgs& a, int64_t n_blocks, int ntile, size_t smem, int dev,
                                      cudaStream_t st) {
    static std::mutex mu;
    static size_t attr[64] = {0};
    {
        std::lock_guard<std::mutex> lock(mu);
        if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
        if (attr[dev] < smem) {
            cudaError_t err =
                cudaFuncSetAttribute(grouped_mma_kernel<NB>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (err != cudaSuccess) return err;
            attr[dev] = smem;
        }
    }
    grouped_mma_kernel<NB><<<dim3((unsigned)n_blocks, (unsigned)ntile), GR_THREADS, smem, st>>>(a);
    return cudaGetLastError();
}

bool grouped_shape_ok(int d, int I) { return d % GR_BN == 0 && I % GR_BN == 0 && d % 128 == 0 && I % 128 == 0; }

size_t grouped_smem_bytes(int d, int I) { return std::max(grouped_smem<2>(d), grouped_smem<1>(I)); }

cudaError_t launch_grouped(const uint16_t* x, int T, int d, const int32_t* ids, const float* w, int k, MXView wg,
                           MXView wu, MXView wd, int E, int I, bool act_mx, const GroupedWorkspace& ws, uint16_t* y,
                           cudaStream_t st) {
    DeviceInfo di;
    cudaError_t err = device_info(&di);
    if (err != cudaSuccess) return err;
    int dev = 0;
    if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
    err = launch_align(ids, T, k, E, GR_BM, ws.sorted, ws.n_sorted, ws.expert_ids, ws.n_blocks, ws.ntpp, ws.align_ws,
                       st);
    if (err != cudaSuccess) return err;
    const uint16_t* xa = x;
    if (act_mx) {
        if ((err = launch_mx_requant(x, ws.x_mx, T, d, st)) != cudaSuccess) return err;
        xa = ws.x_mx;
    }
    GRArgs a{};
    a.sorted = ws.sorted;
    a.expert_ids = ws.expert_ids;
    a.ntpp = ws.ntpp;
    a.h_sorted = ws.h_sorted;
    a.out = ws.out;
    a.T = T;
    a.k = k;
    a.E = E;
    a.d = d;
    a.I = I;
    a.err = di.err_word;
    a.a_src = xa;
    a.w0 = wg.w;
    a.s0 = wg.s;
    a.w1 = wu.w;
    a.s1 = wu.s;
    if ((err = launch_grouped_mma<2>(a, ws.n_blocks, I / GR_BN, grouped_smem<2>(d), dev, st)) != cudaSuccess)
        return err;
    if (act_mx && (err = launch_mx_requant(ws.h_sorted, ws.h_sorted, ws.n_sorted, I, st)) != cudaSuccess) return err;
    a.a_src = ws.h_sorted;
    a.w0 = wd.w;
    a.s0 = wd.s;
    a.w1 = nullptr;
    a.s1 = nullptr;
    if ((err = launch_grouped_mma<1>(a, ws.n_blocks, d / GR_BN, grouped_smem<1>(I), dev, st)) != cudaSuccess)
        return err;
    const int64_t n = (int64_t)T * d;
    const int64_t grid = std::min<int64_t>((n + 255) / 256, (int64_t)di.sm_count * 8);
    grouped_combine_kernel<<<(unsigned)std::max<int64_t>(grid, 1), 256, 0, st>>>(ws.out, w, ids, T, k, E, d, y);
    return cudaGetLastError();
}

}  // namespace moedec

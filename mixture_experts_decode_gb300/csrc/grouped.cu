// grouped.cu -- the expert-centric path of the MoE expert-FFN layer, for
// large batches and prefill: moe_align_block_size sorts the (token, slot)
// pairs by expert into blocks of GR_BM rows of one expert each, then two
// grouped GEMMs run on the 5th-generation tensor cores and a combine step
// adds each token's k rows with their routing weights ("Warp decode",
// section "Warp decode 與 Composer 訓練": prefill and large batches keep
// expert-centric packing; the align page's MoE Align & Sort feeds exactly
// such grouped GEMMs).
//
//   gemm1 (gate/up): per tile (block of GR_BM sorted slots, GR_BN rows of
//     I), the block's expert's W_gate and W_up rows, dequantised from MXFP8
//     to BF16 in shared memory (exact for scale bytes >= 3: an E4M3 value
//     times a power of two has at most four significant bits and stays a
//     BF16 normal), times the block's real slots' token rows of x (BF16),
//     into two FP32 accumulators in tensor memory.  Epilogue:
//     h = bf16(SiLU(g) * u) per real slot, into h_sorted.
//   gemm2 (down): the expert's W_down rows times the real slots' rows of
//     h_sorted, FP32 in tensor memory; the epilogue stores each real slot's
//     row of partial outputs (FP32) at its flat slot index.
//   shared expert (when given): the same two passes as a one-expert layer
//     over every token in order.
//   combine: y[t][o] = bf16( sum_j w[t][j] * out[t*k + j][o] + shared[t][o] ),
//     the k slots in order, the shared row last.
// Each MMA is tcgen05.mma kind::f16 (BF16 x BF16 -> FP32) with the weight
// tile as its M = 128 operand and the block's slot rows as N (the real rows
// rounded up to 16), K = 16, issued by one thread from K-major 128-byte-
// swizzled shared memory tiles; tcgen05.commit signals completion to an
// mbarrier.  The pad rows of a block's slot tile are never written: they
// only feed accumulator columns that no epilogue reads.  The products are
// those of the MX values exactly; sums are FP32 in the tensor core's order.
// With act_mx set, x and h are first rounded through MXFP8
// (moe_mx_requant): the conventional path's activations.
#include <cstdint>
#include <mutex>

#include "common.cuh"
#include "decode_common.cuh"
#include "internal.h"

namespace moedec {

constexpr int GR_BM = GROUPED_BLOCK;       // sorted slots per block (at most the MMA's N)
constexpr int GR_BN = 128;                 // weight rows per tile (the MMA's M)
constexpr int GR_KC = 64;                  // K elements per chunk (one 128-byte swizzle row of BF16)
constexpr int GR_RC = 128;                 // K elements per raw-code stage (two chunks: 128 B per row)
constexpr int GR_RAW = GR_BN * GR_RC;      // raw-code bytes per matrix and stage
constexpr int GR_CW = 8;                   // dequantising (consumer) warps: 0 .. 7
constexpr int GR_PW = GR_CW;               // the copy warp
constexpr int GR_MW = GR_CW + 1;           // the MMA warp
constexpr int GR_THREADS = (GR_CW + 6) * 32;  // + four epilogue warps (10 .. 13: TMEM lane quadrants 2, 3, 0, 1)
constexpr int GR_MAXR = 8;                 // deepest ring of raw code stages
constexpr int GR_AROWS = GR_CW * 32 / 8;   // A rows the consumers copy per pass (8 pieces of 16 B per row)
constexpr int GR_IROWS = GR_CW * 32 / 4;   // weight rows the consumers dequantise per pass (4 items per row)
constexpr int GR_ITEMS = GR_BN / GR_IROWS; // dequantisation items per thread and matrix
static_assert(GR_BN % GR_IROWS == 0, "whole passes of items");
constexpr int GR_APASS = (GR_BM + GR_AROWS - 1) / GR_AROWS;

struct GRArgs {
    const uint16_t* a_src;     // gate/up: x [T][d] (rows by token); down: h_sorted [n_sorted][I]
    const int32_t* sorted;     // flat slot of each sorted row (T*k = pad)
    const int32_t* expert_ids; // expert of each block
    const int32_t* ntpp;       // rows used (a multiple of GR_BM)
    const uint8_t *s0, *s1;    // E8M0 scales: gate/up: W_gate, W_up; down: W_down
    uint16_t* h_sorted;        // gate/up output [n_sorted][I] BF16 (real rows only)
    float* out;                // down output [T*k][d] FP32 by flat slot
    int T, k, E, d, I;
    int NR;                    // raw code stages in the ring
    int TB;                    // per-tile buffers (scales + sorted rows): 1 or 2
    int* err;
};

// The weight codes' tensor maps: [E * rows][K] bytes, boxes of 64 x 128.
struct GRMaps {
    CUtensorMap w0, w1;
};

// Shared memory, byte offsets from a 1024-aligned base.
struct GRLayout {
    uint32_t a, bf, raw, tile, tile_bytes, bars, tmem_slot, abort, total;
};

__host__ __device__ inline GRLayout gr_layout(int NB, int K, int NR, int TB) {
    GRLayout L;
    uint32_t off = 0;
    L.a = off;          off += 2 * 16384;                              // A tile per BF16 stage
    L.bf = off;         off += 2 * NB * 16384;                         // dequantised B tiles
    L.raw = off;        off += NR * NB * GR_RAW;                       // raw E4M3 codes (TMA ring)
    L.tile_bytes = NB * GR_BN * (K / 32) + GR_BM * 4;                  // a tile's scales + sorted rows
    L.tile = off;       off += TB * L.tile_bytes;
    L.bars = off;       off += (2 * GR_MAXR + 12) * 8;
    L.tmem_slot = off;  off += 8;
    L.abort = off;      off += 8;
    L.total = off;
    return L;
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

// 16 bytes global -> shared (L2 only).
__device__ __forceinline__ void cp_async_16_plain(void* smem, const void* gmem) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(smem)), "l"(gmem) : "memory");
}

// Real rows of a block: its sorted slots below the pad value form a prefix
// (the sort pads each expert's run at its end); binary search.
__device__ __forceinline__ int real_rows(const void* srt_bytes, int pad) {
    const int32_t* srt = reinterpret_cast<const int32_t*>(srt_bytes);
    int lo = 0, hi = GR_BM;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (srt[mid] < pad)
            lo = mid + 1;
        else
            hi = mid;
    }
    return lo;
}

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

// A persistent CTA works through tiles t = blockIdx.x, + gridDim.x, ...; a
// tile is (block of GR_BM sorted slots of one expert, GR_BN weight rows).
// NB = 2: the gate/up GEMMs (K = d, N over I); NB = 1: the down GEMM (K = I,
// N over d).  Roles, all overlapped across tiles:
//   copy warp      per tile: the tile's scale rows and sorted slots (1D bulk
//                  copies); per 128 K elements (two chunks): the raw codes
//                  (2D TMA, 128-byte swizzled rows) into an NR-stage ring;
//   warps 0..7     per chunk: the real rows of A (cp.async into the 128-byte
//                  swizzle) and the dequantisation of the codes into BF16
//                  tiles (two stages);
//   MMA warp       per chunk: NB x 4 tcgen05.mma into one of two TMEM
//                  accumulators (alternating by tile);
//   warps 10..13   per tile: the epilogue from TMEM (one lane quadrant each).
// Barriers: raw_full/raw_empty (ring), bf_full/bf_empty (BF16 stages; empty
// by tcgen05.commit), tile_full/tile_empty (per-tile buffers), acc_full
// (commit) / acc_empty (epilogue done with an accumulator).  Every wait is
// bounded; one that gives up raises `abort` and every role skips to the end
// (copies drained, MMAs finished, TMEM freed).
template <int NB>
__global__ void __launch_bounds__(GR_THREADS, NB == 1 ? 2 : 1) grouped_mma_kernel(GRArgs a, const __grid_constant__ GRMaps maps) {
    const int ntile = (NB == 2 ? a.I : a.d) / GR_BN;
    const int n_tiles = (*a.ntpp / GR_BM) * ntile;
    if ((int)blockIdx.x >= n_tiles) return;  // uniform: no tile for this CTA
    extern __shared__ __align__(1024) unsigned char gr_smem[];
    unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(gr_smem) + 1023) &
                                                           ~uintptr_t(1023));
    const int K = NB == 2 ? a.d : a.I;  // contraction length
    const int NK = K / GR_KC;
    const int nsc = K / 32;             // scale bytes per weight row
    const int NR = a.NR, TB = a.TB;
    const GRLayout L = gr_layout(NB, K, NR, TB);
    uint64_t* bars = reinterpret_cast<uint64_t*>(base + L.bars);
    uint64_t* raw_full = bars;
    uint64_t* raw_empty = bars + GR_MAXR;
    uint64_t* bf_full = bars + 2 * GR_MAXR;
    uint64_t* bf_empty = bf_full + 2;
    uint64_t* tile_full = bf_full + 4;
    uint64_t* tile_empty = bf_full + 6;
    uint64_t* acc_full = bf_full + 8;
    uint64_t* acc_empty = bf_full + 10;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + L.tmem_slot);
    volatile int* abort = reinterpret_cast<volatile int*>(base + L.abort);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rows_w = NB == 2 ? a.I : a.d;  // weight rows per expert
    const int pad = a.T * a.k;
    const int n_my = (n_tiles - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;  // tiles of this CTA

    if (tid == 0) {
        for (int i = 0; i < NR; ++i) {
            mbar_init(&raw_full[i], 1);
            mbar_init(&raw_empty[i], GR_CW);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bf_full[i], GR_CW);
            mbar_init(&bf_empty[i], 1);
            mbar_init(&tile_full[i], 1);
            mbar_init(&tile_empty[i], GR_CW + 4);
            mbar_init(&acc_full[i], 1);
            mbar_init(&acc_empty[i], 4);
        }
        *abort = 0;
        mbar_init_fence();
    }
    if (warp == 0) {  // tensor memory: two accumulators of NB x 128 FP32 columns
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                     "r"(2 * NB * 128)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == GR_PW) {
        // ---------------- copy warp ----------------
        if (lane == 0) {
            const uint64_t pol = l2_evict_first_policy();
            int g = 0, li = 0;  // raw stages and tiles issued
            bool ok = true;
            for (; li < n_my && ok; ++li) {
                const int t = (int)blockIdx.x + li * (int)gridDim.x;
                const int blk = t / ntile, n0 = (t - blk * ntile) * GR_BN;
                const int e = a.expert_ids[blk];
                const int wrow = e * rows_w + n0;
                const int tb = li % TB;
                if (li >= TB && !mbar_wait_abort(&tile_empty[tb], ((li / TB) - 1) & 1, abort)) break;
                unsigned char* tbuf = base + L.tile + tb * L.tile_bytes;
                mbar_arrive_expect_tx(&tile_full[tb], L.tile_bytes);
                for (int p = 0; p < NB; ++p)
                    bulk_g2s_keep(tbuf + p * GR_BN * nsc, (p ? a.s1 : a.s0) + (int64_t)wrow * nsc, GR_BN * nsc,
                                  &tile_full[tb]);
                bulk_g2s_keep(tbuf + NB * GR_BN * nsc, a.sorted + (int64_t)blk * GR_BM, GR_BM * 4, &tile_full[tb]);
                for (int kr = 0; kr < K / GR_RC; ++kr, ++g) {
                    const int r = g % NR;
                    if (g >= NR && !mbar_wait_abort(&raw_empty[r], ((g / NR) - 1) & 1, abort)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&raw_full[r], NB * GR_RAW);
#pragma unroll
                    for (int p = 0; p < NB; ++p)
                        tma_2d(base + L.raw + (r * NB + p) * GR_RAW, p ? &maps.w1 : &maps.w0, kr * GR_RC, wrow,
                               &raw_full[r], pol);
                }
            }
            // never leave the CTA with a copy in flight (the last ring stages and tile buffers issued)
            for (int j = g > NR ? g - NR : 0; j < g; ++j) mbar_wait(&raw_full[j % NR], (j / NR) & 1);
            for (int j = li > TB ? li - TB : 0; j < li; ++j) mbar_wait(&tile_full[j % TB], (j / TB) & 1);
        }
    } else if (warp == GR_MW) {
        // ---------------- MMA warp ----------------
        // D^T = W_tile x A^T: the weight tile is the MMA's A operand (M = 128
        // rows in TMEM lanes), the block's slot rows its B operand with N =
        // the real rows rounded up to 16, so a block with few real slots
        // costs few tensor-core cycles.
        if (lane == 0) {
            int g = 0;  // chunks issued
            bool ok = true;
            for (int li = 0; li < n_my && ok; ++li) {
                const int ab = li & 1, tb = li % TB;
                if (li >= 2 && !mbar_wait_abort(&acc_empty[ab], ((li >> 1) - 1) & 1, abort)) break;
                if (!mbar_wait_abort(&tile_full[tb], (li / TB) & 1, abort)) break;
                const int nreal = real_rows(base + L.tile + tb * L.tile_bytes + NB * GR_BN * nsc, pad);
                const uint32_t idesc = gr_idesc(GR_BN, max(16, (nreal + 15) & ~15));
                tc_fence_after();
                const uint32_t acc = tmem + ab * NB * 128;
                for (int kc = 0; kc < NK; ++kc, ++g) {
                    const int b = g & 1;
                    if (!mbar_wait_abort(&bf_full[b], (g >> 1) & 1, abort)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = smem_addr(base + L.a + b * 16384);
#pragma unroll
                    for (int p = 0; p < NB; ++p) {
                        const uint32_t b0 = smem_addr(base + L.bf + (b * NB + p) * 16384);
#pragma unroll
                        for (int kk = 0; kk < GR_KC / 16; ++kk)
                            umma_bf16(acc + p * 128, umma_desc_sw128(b0 + kk * 32), umma_desc_sw128(a0 + kk * 32),
                                      idesc, (kc > 0 || kk > 0) ? 1u : 0u);
                    }
                    umma_commit(&bf_empty[b]);
                }
                if (ok) umma_commit(&acc_full[ab]);
            }
            // let the MMAs already issued finish before TMEM is freed
            if (g > 0) mbar_wait(&bf_empty[(g - 1) & 1], ((g - 1) >> 1) & 1);
        }
    } else if (warp < GR_CW) {
        // ---------------- consumers: A rows + dequantisation ----------------
        const int ct = tid;  // 0 .. GR_CW*32-1
        // this thread's dequantisation items: rows row0 + GR_IROWS i, 16 codes at c * 16 of each 64-code half
        const int row0 = ct >> 2, c = ct & 3, sw = row0 & 7;
        const uint32_t raw_off0 = row0 * 128 + ((c ^ sw) << 4), raw_off1 = row0 * 128 + (((4 + c) ^ sw) << 4);
        const uint32_t dst_off0 = row0 * 128 + (((2 * c) ^ sw) << 4), dst_off1 = row0 * 128 + (((2 * c + 1) ^ sw) << 4);
        const int sc_off = row0 * nsc + (c >> 1);
        int g = 0;
        bool ok = true;
        for (int li = 0; li < n_my && ok; ++li) {
            const int t = (int)blockIdx.x + li * (int)gridDim.x;
            const int blk = t / ntile;
            const int tb = li % TB;
            if (!__all_sync(FULL_MASK, mbar_wait_abort(&tile_full[tb], (li / TB) & 1, abort))) break;
            const unsigned char* tbuf = base + L.tile + tb * L.tile_bytes;
            const int32_t* srt = reinterpret_cast<const int32_t*>(tbuf + NB * GR_BN * nsc);
            // this thread's A rows: ct/8 + GR_AROWS i, 16-byte piece ct % 8
            const uint16_t* src[GR_APASS];
            int nsrc = 0;
#pragma unroll
            for (int i = 0; i < GR_APASS; ++i) {
                const int row = (ct >> 3) + GR_AROWS * i;
                const int f = row < GR_BM ? srt[row] : pad;
                if (f < pad) {
                    const int64_t srow = NB == 2 ? (int64_t)(f / a.k) : (int64_t)blk * GR_BM + row;
                    src[i] = a.a_src + srow * K + (ct & 7) * 8;
                    nsrc = i + 1;  // real rows are a prefix of the block
                }
            }
            for (int kc = 0; kc < NK; ++kc, ++g) {
                const int b = g & 1, r = (g >> 1) % NR;  // two chunks per raw stage
                // the MMAs that read stage b two chunks ago must be done
                if (g >= 2 && !__all_sync(FULL_MASK, mbar_wait_abort(&bf_empty[b], ((g >> 1) - 1) & 1, abort))) {
                    ok = false;
                    break;
                }
                unsigned char* As = base + L.a + b * 16384;
#pragma unroll
                for (int i = 0; i < GR_APASS; ++i)
                    if (i < nsrc) cp_async_16_plain(As + swz128((ct >> 3) + GR_AROWS * i, ct & 7), src[i] + kc * GR_KC);
                cp_async_commit();
                if (!__all_sync(FULL_MASK, mbar_wait_abort(&raw_full[r], ((g >> 1) / NR) & 1, abort))) {
                    ok = false;
                    break;
                }
#pragma unroll
                for (int p = 0; p < NB; ++p) {
                    const uint8_t* raw = base + L.raw + (r * NB + p) * GR_RAW + ((g & 1) ? raw_off1 : raw_off0);  // swizzled rows
                    char* dst = reinterpret_cast<char*>(base + L.bf + (b * NB + p) * 16384);
                    const uint8_t* scp = tbuf + p * GR_BN * nsc + sc_off + kc * 2;
#pragma unroll
                    for (int i = 0; i < GR_ITEMS; ++i) {  // rows row0 + GR_IROWS * i
                        const uint4 w4 = *reinterpret_cast<const uint4*>(raw + i * GR_IROWS * 128);
                        const float sc = e8m0_to_float(scp[i * GR_IROWS * nsc]);
                        uint32_t o[8];
#pragma unroll
                        for (int wq = 0; wq < 4; ++wq) {
                            float2 lo, hi;
                            e4m3x4_to_float((&w4.x)[wq], lo, hi);
                            lo = __fmul2_rn(lo, make_float2(sc, sc));
                            hi = __fmul2_rn(hi, make_float2(sc, sc));
                            const __nv_bfloat162 b0 = __floats2bfloat162_rn(lo.x, lo.y);
                            const __nv_bfloat162 b1 = __floats2bfloat162_rn(hi.x, hi.y);
                            memcpy(&o[wq * 2], &b0, 4);
                            memcpy(&o[wq * 2 + 1], &b1, 4);
                        }
                        char* d = dst + i * GR_IROWS * 128;
                        *reinterpret_cast<uint4*>(d + dst_off0) = make_uint4(o[0], o[1], o[2], o[3]);
                        *reinterpret_cast<uint4*>(d + dst_off1) = make_uint4(o[4], o[5], o[6], o[7]);
                    }
                }
                __syncwarp();
                if (lane == 0 && (g & 1)) mbar_arrive(&raw_empty[r]);  // both chunks of the stage read
                cp_async_wait<0>();
                fence_proxy_async();  // this thread's tile writes, before the tensor cores read them
                __syncwarp();
                if (lane == 0) mbar_arrive(&bf_full[b]);
            }
            if (!ok) break;
            __syncwarp();
            if (lane == 0) mbar_arrive(&tile_empty[tb]);
        }
        cp_async_wait<0>();  // no copy still in flight on any exit
    } else {
        // ---------------- epilogue warps: TMEM -> h (gate/up) or the slots' partial outputs (down) ----------------
        // TMEM lane = weight row n of the tile, column = slot row m of the block.
        const int quad = warp & 3;                        // TMEM lanes 32 quad .. 32 quad + 31
        const int n = quad * 32 + lane;                   // weight row within the tile
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        for (int li = 0; li < n_my; ++li) {
            const int t = (int)blockIdx.x + li * (int)gridDim.x;
            const int blk = t / ntile, n0 = (t - blk * ntile) * GR_BN;
            const int tb = li % TB, ab = li & 1;
            if (!__all_sync(FULL_MASK, mbar_wait_abort(&acc_full[ab], (li >> 1) & 1, abort))) break;
            if (!__all_sync(FULL_MASK, mbar_wait_abort(&tile_full[tb], (li / TB) & 1, abort))) break;
            tc_fence_after();
            const int32_t* srt = reinterpret_cast<const int32_t*>(base + L.tile + tb * L.tile_bytes + NB * GR_BN * nsc);
            const int nreal = real_rows(srt, pad);
            const uint32_t acc = tmem + lane_off + ab * NB * 128;
#pragma unroll 1
            for (int c0 = 0; c0 < nreal; c0 += 32) {
                if (NB == 2) {
                    float gv[32], uv[32];
                    tmem_ld32(acc + c0, gv);
                    tmem_ld32(acc + 128 + c0, uv);
                    uint16_t* hp = a.h_sorted + ((int64_t)blk * GR_BM + c0) * a.I + n0 + n;
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (c0 + i < nreal) {
                            const float hv = gv[i] / (1.0f + expf(-gv[i])) * uv[i];
                            hp[(int64_t)i * a.I] = __bfloat16_as_ushort(__float2bfloat16_rn(hv));
                        }
                } else {
                    float v[32];
                    tmem_ld32(acc + c0, v);
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (c0 + i < nreal) a.out[(int64_t)srt[c0 + i] * a.d + n0 + n] = v[i];
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&acc_empty[ab]);
                mbar_arrive(&tile_empty[tb]);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(2 * NB * 128)
                     : "memory");
    }
    if (tid == 0 && *abort) atomicOr(a.err, MOE_DEVERR_TIMEOUT);
}

// y[t][o] = bf16( sum_j w[t][j] * out[t*k + j][o] + sh[t][o] ), j in order,
// then the shared expert's row (weight 1; sh null without one); a slot whose
// expert id is outside [0, E) (never placed by the sort) adds nothing.  Four
// consecutive outputs per thread (d % 4 == 0).
__global__ void grouped_combine_kernel(const float* __restrict__ out, const float* __restrict__ w,
                                       const int32_t* __restrict__ ids, const float* __restrict__ sh, int T, int k,
                                       int E, int d, uint16_t* __restrict__ y) {
    const int64_t n4 = (int64_t)T * d / 4;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t t = i * 4 / d, o = i * 4 - t * d;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int j = 0; j < k; ++j) {
            if ((unsigned)ids[t * k + j] >= (unsigned)E) continue;
            const float wt = w[t * k + j];
            const float4 v = *reinterpret_cast<const float4*>(out + (t * k + j) * d + o);
            acc.x = fmaf(wt, v.x, acc.x);
            acc.y = fmaf(wt, v.y, acc.y);
            acc.z = fmaf(wt, v.z, acc.z);
            acc.w = fmaf(wt, v.w, acc.w);
        }
        if (sh) {
            const float4 v = *reinterpret_cast<const float4*>(sh + t * d + o);
            acc.x += v.x;
            acc.y += v.y;
            acc.z += v.z;
            acc.w += v.w;
        }
        const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y), hi = __floats2bfloat162_rn(acc.z, acc.w);
        uint2 pk;
        memcpy(&pk.x, &lo, 4);
        memcpy(&pk.y, &hi, 4);
        *reinterpret_cast<uint2*>(y + i * 4) = pk;
    }
}

// The shared expert's sort: every token in order, padded to whole blocks of
// GR_BM rows, all of expert 0 (of the one-expert shared arrays).
__global__ void grouped_shared_sort_kernel(int32_t* __restrict__ sorted, int32_t* __restrict__ expert, int32_t* ntpp,
                                           int T, int64_t n_sh) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_sh; i += (int64_t)gridDim.x * blockDim.x) {
        sorted[i] = i < T ? (int32_t)i : T;
        if (i % GR_BM == 0) expert[i / GR_BM] = 0;
        if (i == 0) *ntpp = (int32_t)n_sh;
    }
}

// Ring depth NR and per-tile buffers TB for a pass: the deepest ring (up to
// 4 stages of 128 K elements) with two tile buffers that fits `budget`
// bytes, else with one.
static bool grouped_plan(int NB, int K, size_t budget, int* NR, int* TB) {
    for (int tb = 2; tb >= 1; --tb)
        for (int nr = 4; nr >= 2; --nr)
            if (gr_layout(NB, K, nr, tb).total + 1024 <= budget) {
                *NR = nr;
                *TB = tb;
                return true;
            }
    return false;
}

template <int NB>
static cudaError_t launch_grouped_mma(GRArgs a, const GRMaps& maps, int64_t n_blocks, const DeviceInfo& di, int dev,
                                      cudaStream_t st) {
    static std::mutex mu;
    static size_t attr[64] = {0};
    const int K = NB == 2 ? a.d : a.I;
    // the down pass keeps two CTAs per SM (half the SM's shared memory each) when it can
    size_t budget = (size_t)di.max_smem_optin;
    if (NB == 1 && grouped_plan(NB, K, (size_t)di.smem_per_sm / 2 - 1024, &a.NR, &a.TB))
        budget = (size_t)di.smem_per_sm / 2 - 1024;
    if (!grouped_plan(NB, K, budget, &a.NR, &a.TB)) return cudaErrorInvalidValue;
    const size_t smem = gr_layout(NB, K, a.NR, a.TB).total + 1024;
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
    const int per_sm = (NB == 1 && smem <= (size_t)di.smem_per_sm / 2 - 1024) ? 2 : 1;
    const int64_t tiles_max = n_blocks * ((NB == 2 ? a.I : a.d) / GR_BN);
    const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(tiles_max, (int64_t)di.sm_count * per_sm));
    grouped_mma_kernel<NB><<<(unsigned)grid, GR_THREADS, smem, st>>>(a, maps);
    return cudaGetLastError();
}

bool grouped_shape_ok(int d, int I) { return d % 128 == 0 && I % 128 == 0; }

size_t grouped_smem_bytes(int d, int I) {
    return std::max(gr_layout(2, d, 2, 1).total, gr_layout(1, I, 2, 1).total) + 1024;
}

cudaError_t launch_grouped(const uint16_t* x, int T, int d, const int32_t* ids, const float* w, int k, MXView wg,
                           MXView wu, MXView wd, MXView shg, MXView shu, MXView shd, int E, int I, bool act_mx,
                           const GroupedWorkspace& ws, uint16_t* y, cudaStream_t st) {
    DeviceInfo di;
    cudaError_t err = device_info(&di);
    if (err != cudaSuccess) return err;
    int dev = 0;
    if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
    const bool shared = shg.w != nullptr;
    GRMaps m1{}, m2{}, s1{}, s2{};
    if (!map_2d_u8(&m1.w0, wg.w, (uint64_t)E * I, d, GR_BN, GR_RC, true) ||
        !map_2d_u8(&m1.w1, wu.w, (uint64_t)E * I, d, GR_BN, GR_RC, true) ||
        !map_2d_u8(&m2.w0, wd.w, (uint64_t)E * d, I, GR_BN, GR_RC, true))
        return cudaErrorInvalidValue;
    m2.w1 = m2.w0;
    if (shared) {
        if (!map_2d_u8(&s1.w0, shg.w, (uint64_t)I, d, GR_BN, GR_RC, true) ||
            !map_2d_u8(&s1.w1, shu.w, (uint64_t)I, d, GR_BN, GR_RC, true) ||
            !map_2d_u8(&s2.w0, shd.w, (uint64_t)d, I, GR_BN, GR_RC, true))
            return cudaErrorInvalidValue;
        s2.w1 = s2.w0;
    }
    err = launch_align(ids, T, k, E, GR_BM, ws.sorted, ws.n_sorted, ws.expert_ids, ws.n_blocks, ws.ntpp, ws.align_ws,
                       st);
    if (err != cudaSuccess) return err;
    const uint16_t* xa = x;
    if (act_mx) {
        if ((err = launch_mx_requant(x, ws.x_mx, T, d, st)) != cudaSuccess) return err;
        xa = ws.x_mx;
    }
    // the routed experts, then (as a one-expert layer over every token) the shared one
    for (int pass = 0; pass < (shared ? 2 : 1); ++pass) {
        GRArgs a{};
        const bool sp = pass == 1;
        if (sp) {
            const int64_t g = std::min<int64_t>((ws.n_sh + 255) / 256, (int64_t)di.sm_count * 4);
            grouped_shared_sort_kernel<<<(unsigned)g, 256, 0, st>>>(ws.sh_sorted, ws.sh_expert, ws.sh_ntpp, T,
                                                                   ws.n_sh);
            if ((err = cudaGetLastError()) != cudaSuccess) return err;
        }
        a.sorted = sp ? ws.sh_sorted : ws.sorted;
        a.expert_ids = sp ? ws.sh_expert : ws.expert_ids;
        a.ntpp = sp ? ws.sh_ntpp : ws.ntpp;
        a.h_sorted = sp ? ws.sh_h : ws.h_sorted;
        a.out = sp ? ws.sh_out : ws.out;
        a.T = T;
        a.k = sp ? 1 : k;
        a.E = sp ? 1 : E;
        a.d = d;
        a.I = I;
        a.err = di.err_word;
        a.a_src = xa;
        a.s0 = sp ? shg.s : wg.s;
        a.s1 = sp ? shu.s : wu.s;
        const int64_t nb = sp ? ws.n_sh / GR_BM : ws.n_blocks;
        const int64_t nrows = sp ? ws.n_sh : ws.n_sorted;
        if ((err = launch_grouped_mma<2>(a, sp ? s1 : m1, nb, di, dev, st)) != cudaSuccess) return err;
        // only the real rows of h were written: round those (and harmless pad-row bits) through MXFP8
        if (act_mx && (err = launch_mx_requant(a.h_sorted, a.h_sorted, nrows, I, st)) != cudaSuccess) return err;
        a.a_src = a.h_sorted;
        a.s0 = sp ? shd.s : wd.s;
        a.s1 = nullptr;
        if ((err = launch_grouped_mma<1>(a, sp ? s2 : m2, nb, di, dev, st)) != cudaSuccess) return err;
    }
    const int64_t n = (int64_t)T * d / 4;
    const int64_t grid = std::min<int64_t>((n + 255) / 256, (int64_t)di.sm_count * 8);
    grouped_combine_kernel<<<(unsigned)std::max<int64_t>(grid, 1), 256, 0, st>>>(ws.out, w, ids,
                                                                                 shared ? ws.sh_out : nullptr, T, k,
                                                                                 E, d, y);
    return cudaGetLastError();
}

}  // namespace moedec

// decode_common.cuh -- pieces shared by the gate/up and down passes of the
// MoE expert-FFN decode layer: the argument blocks, the per-CTA routing map
// (token -> distinct expert, built in shared memory from topk_ids by every
// CTA: no extra launch, no global buffer), tensor-copy and mbarrier helpers,
// cluster helpers, and the host-side tensor-map encoders.
#pragma once
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
    float* h32;  // when set, h goes here instead: FP32, in the down pass's K-slab order (h32_pos)
};

struct DownArgs {
    DecodeShape s;
    const uint16_t* h;
    const int32_t* ids;
    const float* w;
    MXView wd, shd;
    uint16_t* y;
    int* err;
    int es;            // expert splits per CTA (1, 2, 4 or 8)
    const float* h32;  // when set, the intermediate is read from here (FP32, h32_pos order)
};

// Position of intermediate neuron n inside a row of the FP32 intermediate
// that the gate/up pass writes for the down pass (I % 256 == 0).  The down
// pass's lane l takes elements 8 l .. 8 l + 7 of each 256-element group;
// the group is stored as [2 halves][32 lanes][4], so that lane's two
// 16-byte loads are contiguous across the warp (bank-conflict free).
__host__ __device__ inline int h32_pos(int n) {
    const int w = n & 255, l = w >> 3, e = w & 7;
    return (n & ~255) | ((e >> 2) << 7) | (l << 2) | (e & 3);
}

// Store one intermediate value: BF16 round to nearest even, then either the
// BF16 bits at [hrow][n] of h or the same value as FP32 at h32_pos(n).
__device__ __forceinline__ void store_h(const GateUpArgs& a, int hrow, int n, float hv) {
    const __nv_bfloat16 hb = __float2bfloat16_rn(hv);
    if (a.h32)
        a.h32[(size_t)hrow * a.s.I + h32_pos(n)] = __bfloat162float(hb);
    else
        a.h[(size_t)hrow * a.s.I + n] = __bfloat16_as_ushort(hb);
}

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

// Position of a warp in its sequence of (item, token group, chunk) steps.
struct GU2Cursor {
    int m, g, c;  // item ordinal of this warp, token group, chunk
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

__device__ inline RouteMap carve_map(int* p, const DecodeShape& s, bool with_w) {
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

__device__ inline void build_route_map(const RouteMap& m, const int32_t* __restrict__ ids,
                                const float* __restrict__ w, const DecodeShape& s, int* err,
                                bool merge = false, int* scratch = nullptr, int scratch_ints = 0,
                                bool small = true) {
    // The first PT = min(blockDim.x, DEC_THREADS) threads (whole warps) build
    // the map; any further threads only take part in the barriers.
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int PT = min((int)blockDim.x, DEC_THREADS) & ~31, PW = PT >> 5;
    const bool part = tid < PT;
    const int n = s.B * s.k;
    const int KS = s.k + s.S;
    if (small && n <= 32) {
        // Few slots (B * k <= 32): one warp builds the map.  A slot's expert
        // group is its __match_any_sync mask; the distinct experts are
        // numbered, and their slot ranges laid out, in increasing expert id
        // (as the general path does), slots inside a range in flat order.
        if (warp == 0) {
            int e = -1;
            float wv = 0.f;
            if (lane < n) {
                e = ids[lane];
                if (w) wv = w[lane];
                if ((unsigned)e >= (unsigned)s.E) {
                    e = -1;
                    atomicOr(err, MOE_DEVERR_EXPERT_ID);
                }
            }
            const unsigned grp = __match_any_sync(FULL_MASK, e);
            const unsigned below = grp & lanemask_lt();
            const bool lead = e >= 0 && below == 0;
            const int cnt = __popc(grp);
            const unsigned leaders = __ballot_sync(FULL_MASK, lead);
            int uid = 0, off = 0;  // distinct experts with a smaller id and their slots
            for (unsigned rest = leaders; rest; rest &= rest - 1) {
                const int q = __ffs(rest) - 1;
                const int eq = __shfl_sync(FULL_MASK, e, q), cq = __shfl_sync(FULL_MASK, cnt, q);
                if (e >= 0 && eq < e) {
                    ++uid;
                    off += cq;
                }
            }
            if (lead) {
                m.uexp[uid] = e;
                m.uoff[uid] = off;
            }
            if (e >= 0) {
                const int pos = off + __popc(below);
                const int b = lane / s.k, j = lane - b * s.k;
                m.hrow[pos] = b * KS + j;
                if (m.wt) m.wt[pos] = wv;
            }
            const int tot_r = __popc(__ballot_sync(FULL_MASK, e >= 0));
            if (lane == 0) {
                m.hdr[1] = __popc(leaders);
                m.hdr[2] = tot_r;
            }
        }
        __syncthreads();
    } else {
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
    }
    const int nu = m.hdr[1], tot = m.hdr[2];
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

// The distinct experts u < nu (nu <= 256) ordered by descending slot count,
// the lower index first on ties, into perm[]: a bitonic sort of packed
// (255 - count, u) keys by the first 256 threads (shuffles below a distance
// of 32, `scratch` (256 words) above).  Every thread of the CTA must call it.
__device__ inline void order_experts_by_count(const RouteMap& m, int nu, int* perm, uint32_t* scratch) {
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

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

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

}  // namespace moedec

// align.cu -- moe_align_block_size on sm_103a: a stable, multi-block
// counting sort of flat (token, slot) indices by expert id, each expert's
// run padded to a multiple of block_size.
//
// Follows the count / cumsum / placement (D-C-P) split of the MoE Align &
// Sort page ("编写对AMD设备友好的CUDA实现"), rebuilt for one GB300:
//   align_count  : every block builds a shared-memory histogram of its
//                  contiguous chunk of ids and stores it to the workspace.
//   align_place  : every block reads all chunk histograms (a few KB, L2
//                  resident) and derives what it needs itself -- per-expert
//                  totals, its own prefix over earlier chunks, the padded
//                  exclusive scan over experts -- so no third launch, grid
//                  barrier or atomic counter is needed; it then writes its
//                  share of expert_ids / pad sentinels and places its chunk.
// Stability inside a chunk: tiles of blockDim ids in order; inside a warp
// the rank comes from __match_any_sync + popc, across warps from a per-tile
// scan over warps of per-warp expert counts.
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace moedec {

constexpr int ALIGN_CHUNK = 2048;     // target ids per block
constexpr int ALIGN_MAX_BLOCKS = 256;

struct AlignPlan {
    int N, NB, CH, W;
};

static AlignPlan align_plan(int64_t n, int E) {
    AlignPlan p;
    p.N = (int)n;
    long nb = (n + ALIGN_CHUNK - 1) / ALIGN_CHUNK;
    nb = std::max(1L, std::min<long>(nb, ALIGN_MAX_BLOCKS));
    long ch = (n + nb - 1) / nb;
    ch = (ch + 3) / 4 * 4;
    if (ch < 4) ch = 4;
    p.NB = (int)nb;
    p.CH = (int)ch;
    // warps per placement block: the per-warp tables (2 * W * E ints) stay
    // within 160 KB of shared memory
    p.W = std::max(1, std::min(32, 20480 / E));
    return p;
}

size_t align_workspace_bytes(int64_t n, int E) {
    const AlignPlan p = align_plan(n, E);
    return (size_t)p.NB * E * sizeof(int);
}

size_t align_smem_bytes(int E) {
    const AlignPlan p = align_plan(1, E);
    // start, run, tot | wc, wp | scan scratch
    return ((size_t)3 * E + (size_t)2 * p.W * E + 64) * sizeof(int);
}

__global__ void __launch_bounds__(1024) align_count_kernel(const int32_t* __restrict__ ids, int N,
                                                           int E, int CH, int* __restrict__ cnt,
                                                           int* err) {
    extern __shared__ int hist[];
    for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
    __syncthreads();
    const int f0 = blockIdx.x * CH;
    const int f1 = min(N, f0 + CH);
    int bad = 0;
    for (int f = f0 + threadIdx.x; f < f1; f += blockDim.x) {
        const int e = ids[f];
        if ((unsigned)e < (unsigned)E)
            atomicAdd(&hist[e], 1);
        else
            bad = 1;
    }
    if (bad) atomicOr(err, MOE_DEVERR_EXPERT_ID);
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[(size_t)blockIdx.x * E + e] = hist[e];
}

// Block-wide exclusive scan of one int per thread; returns the exclusive
// prefix and writes the block total to *total (all threads see it).
__device__ int block_exclusive_scan(int v, int* scratch, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    int incl = v;
    for (int off = 1; off < 32; off <<= 1) {
        const int t = __shfl_up_sync(FULL_MASK, incl, off);
        if (lane >= off) incl += t;
    }
    if (lane == 31) scratch[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int w = lane < nw ? scratch[lane] : 0;
        int sc = w;
        for (int off = 1; off < 32; off <<= 1) {
            const int t = __shfl_up_sync(FULL_MASK, sc, off);
            if (lane >= off) sc += t;
        }
        if (lane < nw) scratch[lane] = sc - w;
        if (lane == 31) scratch[32] = sc;
    }
    __syncthreads();
    const int r = scratch[warp] + incl - v;
    *total = scratch[32];
    __syncthreads();
    return r;
}

__global__ void __launch_bounds__(1024) align_place_kernel(
    const int32_t* __restrict__ ids, int N, int E, int bs, int CH, int NB,
    const int* __restrict__ cnt, int32_t* __restrict__ sorted, int n_sorted,
    int32_t* __restrict__ expert_ids, int n_blocks, int32_t* __restrict__ ntpp) {
    extern __shared__ int sm[];
    const int W = blockDim.x >> 5;
    int* start = sm;             // [E]
    int* run = start + E;        // [E] fill cursor
    int* tot = run + E;          // [E]
    int* wc = tot + E;           // [W][E] per-warp counts of the current tile
    int* wp = wc + W * E;        // [W][E] per-warp base positions
    int* scratch = wp + W * E;   // [33]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    for (int i = tid; i < W * E; i += blockDim.x) wc[i] = 0;
    // (C) per-expert totals and this block's prefix over earlier chunks
    for (int e = tid; e < E; e += blockDim.x) {
        int t = 0, pre = 0;
        for (int b = 0; b < NB; ++b) {
            const int c = cnt[(size_t)b * E + e];
            t += c;
            pre += (b < (int)blockIdx.x) ? c : 0;
        }
        tot[e] = t;
        run[e] = pre;
    }
    __syncthreads();
    // padded exclusive scan over experts: each thread a contiguous segment
    const int per = (E + blockDim.x - 1) / blockDim.x;
    const int e0 = min(tid * per, E), e1 = min(e0 + per, E);
    int local = 0;
    for (int e = e0; e < e1; ++e) local += (tot[e] + bs - 1) / bs * bs;
    int total = 0;
    int r = block_exclusive_scan(local, scratch, &total);
    for (int e = e0; e < e1; ++e) {
        start[e] = r;
        run[e] += r;
        r += (tot[e] + bs - 1) / bs * bs;
    }
    __syncthreads();
    if (blockIdx.x == 0 && tid == 0) *ntpp = total;

    // expert_ids and pad sentinels of experts e = blockIdx.x (mod NB), one
    // warp per expert
    for (int e = blockIdx.x + NB * warp; e < E; e += NB * W) {
        const int s = start[e], t = tot[e];
        const int p = (t + bs - 1) / bs * bs;
        for (int i = s + t + lane; i < s + p; i += 32) sorted[i] = N;
        for (int q = s / bs + lane; q < (s + p) / bs; q += 32) expert_ids[q] = e;
    }
    // tail past num_tokens_post_pad, spread over all blocks
    {
        const int gt = blockIdx.x * blockDim.x + tid, gs = NB * blockDim.x;
        for (int i = total + gt; i < n_sorted; i += gs) sorted[i] = N;
        for (int q = total / bs + gt; q < n_blocks; q += gs) expert_ids[q] = -1;
    }

    // (P) stable placement of this block's chunk, tile by tile
    const int f0 = blockIdx.x * CH;
    const int f1 = min(N, f0 + CH);
    for (int base = f0; base < f1; base += blockDim.x) {
        const int f = base + tid;
        int e = f < f1 ? ids[f] : -1;
        if ((unsigned)e >= (unsigned)E) e = -1;
        const unsigned grp = __match_any_sync(FULL_MASK, e);
        const unsigned below = grp & lanemask_lt();
        if (e >= 0 && below == 0) wc[warp * E + e] = __popc(grp);
        __syncthreads();
        for (int x = tid; x < E; x += blockDim.x) {
            int c0 = run[x];
            for (int w = 0; w < W; ++w) {
                const int c = wc[w * E + x];
                if (c) {
                    wp[w * E + x] = c0;
                    c0 += c;
                    wc[w * E + x] = 0;
                }
            }
            run[x] = c0;
        }
        __syncthreads();
        if (e >= 0) sorted[wp[warp * E + e] + __popc(below)] = f;
    }
}

cudaError_t launch_align(const int32_t* ids, int T, int k, int E, int block_size, int32_t* sorted,
                         int64_t n_sorted, int32_t* expert_ids, int64_t n_blocks, int32_t* ntpp,
                         void* ws, cudaStream_t st) {
    DeviceInfo di;
    cudaError_t err = device_info(&di);
    if (err != cudaSuccess) return err;
    const int64_t n = (int64_t)T * k;
    const AlignPlan p = align_plan(n, E);
    int* cnt = static_cast<int*>(ws);
    const size_t smem = align_smem_bytes(E);
    // once per device: allow the placement kernel all the opt-in shared
    // memory (entry points may be called from several host threads)
    static std::mutex attr_mu;
    static bool attr_done[64] = {false};
    int dev = 0;
    if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    {
        std::lock_guard<std::mutex> lock(attr_mu);
        if (!attr_done[dev]) {
            err = cudaFuncSetAttribute(align_place_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)(di.max_smem_optin));
            if (err != cudaSuccess) return err;
            attr_done[dev] = true;
        }
    }
    if (n > 0) {
        align_count_kernel<<<p.NB, 1024, E * sizeof(int), st>>>(ids, p.N, E, p.CH, cnt, di.err_word);
        err = cudaGetLastError();
        if (err != cudaSuccess) return err;
    } else {
        err = cudaMemsetAsync(cnt, 0, (size_t)p.NB * E * sizeof(int), st);
        if (err != cudaSuccess) return err;
    }
    align_place_kernel<<<p.NB, p.W * 32, smem, st>>>(ids, p.N, E, block_size, p.CH, p.NB, cnt,
                                                     sorted, (int)n_sorted, expert_ids,
                                                     (int)n_blocks, ntpp);
    return cudaGetLastError();
}

// ------------------------------------------- fixed-scratch variant -----
// For callers that cannot supply device scratch: the per-block histogram
// table lives in this file-scope array.  Host code must not pass the
// symbol itself to a kernel (on the host it names a stand-in, not device
// memory); it looks up the device address once per device instead.

static __device__ __align__(256) int g_align_scratch[MOE_ALIGN_STATIC_SCRATCH_BYTES / sizeof(int)];

cudaError_t align_static_scratch(void** out) {
    static std::mutex mu;
    static void* addr[64] = {nullptr};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void* p = nullptr;
        err = cudaGetSymbolAddress(&p, g_align_scratch);
        if (err != cudaSuccess) return err;
        addr[dev] = p;
    }
    *out = addr[dev];
    return cudaSuccess;
}

}  // namespace moedec

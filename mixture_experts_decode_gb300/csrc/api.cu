// api.cu -- the extern "C" boundary of libmoedec.so: argument checks,
// workspace carving and launches.  No allocation anywhere in the library.
#include <algorithm>
#include <cstdint>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace moedec {

// Sticky device error bits, one word per device (set by kernels that meet
// bad input; read and cleared by moe_device_error).
__device__ int g_err_word;

cudaError_t device_info(DeviceInfo* out) {
    static std::mutex mu;
    static DeviceInfo cache[64];
    static bool have[64] = {false};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!have[dev]) {
        DeviceInfo di;
        err = cudaDeviceGetAttribute(&di.sm_count, cudaDevAttrMultiProcessorCount, dev);
        if (err != cudaSuccess) return err;
        err = cudaDeviceGetAttribute(&di.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (err != cudaSuccess) return err;
        err = cudaDeviceGetAttribute(&di.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
        if (err != cudaSuccess) return err;
        void* p = nullptr;
        err = cudaGetSymbolAddress(&p, g_err_word);
        if (err != cudaSuccess) return err;
        di.err_word = static_cast<int*>(p);
        cache[dev] = di;
        have[dev] = true;
    }
    *out = cache[dev];
    return cudaSuccess;
}

// One 32-byte element per thread, CTAs in address order: each CTA moves one
// contiguous 8 KB span and the CTAs in flight at any time cover neighbouring
// spans.  On GB300 this streams 7.1 TB/s (1-2 GiB, read + write counted),
// faster than a grid-stride loop over a resident grid (6.4 TB/s) and than the
// runtime's device-to-device copy (6.8 TB/s).  The loop only runs again when
// the buffer needs more CTAs than one launch can have.
__global__ void __launch_bounds__(256) copy_kernel(const U256* __restrict__ src, U256* __restrict__ dst,
                                                   size_t n) {
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
        const U256 v = ld_stream_256(src + i);
        asm volatile("st.global.L1::no_allocate.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(dst + i),
                     "r"(v.v[0]), "r"(v.v[1]), "r"(v.v[2]), "r"(v.v[3]), "r"(v.v[4]), "r"(v.v[5]),
                     "r"(v.v[6]), "r"(v.v[7])
                     : "memory");
    }
}

cudaError_t launch_copy(void* dst, const void* src, size_t bytes, cudaStream_t st) {
    const size_t n = bytes / 32;
    if (n == 0) return cudaSuccess;
    const size_t grid = std::min<size_t>((n + 255) / 256, (size_t)INT32_MAX);
    copy_kernel<<<(unsigned)grid, 256, 0, st>>>(static_cast<const U256*>(src), static_cast<U256*>(dst), n);
    return cudaGetLastError();
}

}  // namespace moedec

using namespace moedec;

namespace {

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

int check_mx(const moe_mx_t& m) {
    if (!m.w || !m.s) return MOE_ERR_ARG;
    if (!aligned(m.w, 32)) return MOE_ERR_ALIGN;
    return MOE_OK;
}

// Shared checks of the decode entry points.
int check_decode_shape(int B, int k, int E, int d, int I) {
    if (B < 0 || k < 0 || E < 0 || d < 0 || I < 0) return MOE_ERR_ARG;
    if (d == 0 || I == 0 || E == 0 || k == 0) return MOE_ERR_SHAPE;
    if (d % 32 || I % 32 || k > E) return MOE_ERR_SHAPE;
    if (B > MOE_MAX_TOKENS || E > MOE_MAX_EXPERTS || (long)B * k > MOE_MAX_SLOTS) return MOE_ERR_LIMIT;
    return MOE_OK;
}

int check_smem(size_t need) {
    DeviceInfo di;
    if (device_info(&di) != cudaSuccess) return MOE_ERR_CUDA;
    return need <= (size_t)di.max_smem_optin ? MOE_OK : MOE_ERR_LIMIT;
}

MXView view(const moe_mx_t* m) { return m ? MXView{m->w, m->s} : MXView{nullptr, nullptr}; }

// The layer keeps its intermediate in FP32 (BF16-rounded values) when the
// row-tile down pass takes it, else in BF16: room for the larger.
size_t h_bytes(int B, int k, int I, int S) { return (size_t)B * (k + S) * I * 4; }

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

int gate_up_checked(const void* x, int B, int d, const int32_t* ids, int k, moe_mx_t wg, moe_mx_t wu,
                    int E, int I, const moe_mx_t* sg, const moe_mx_t* su, void* h, bool h32,
                    cudaStream_t st) {
    int rc = check_decode_shape(B, k, E, d, I);
    if (rc) return rc;
    if ((sg == nullptr) != (su == nullptr)) return MOE_ERR_ARG;
    if (B == 0) return MOE_OK;
    if (!x || !ids || !h) return MOE_ERR_ARG;
    if ((rc = check_mx(wg)) || (rc = check_mx(wu))) return rc;
    if (sg && ((rc = check_mx(*sg)) || (rc = check_mx(*su)))) return rc;
    if (!aligned(x, 32) || !aligned(h, 32) || !aligned(ids, 4)) return MOE_ERR_ALIGN;
    const DecodeShape s{B, k, E, d, I, sg ? 1 : 0};
    if ((rc = check_smem(gate_up_smem_bytes(s)))) return rc;
    return cuda_status(launch_gate_up(s, x, ids, view(&wg), view(&wu), view(sg), view(su), h, h32, st));
}

int down_checked(const void* h, bool h32, int B, int k, const int32_t* ids, const float* w, moe_mx_t wd, int E,
                 int d, int I, const moe_mx_t* sd, void* y, cudaStream_t st, bool pdl) {
    int rc = check_decode_shape(B, k, E, d, I);
    if (rc) return rc;
    if (B == 0) return MOE_OK;
    if (!h || !ids || !w || !y) return MOE_ERR_ARG;
    if ((rc = check_mx(wd))) return rc;
    if (sd && (rc = check_mx(*sd))) return rc;
    if (!aligned(h, 32) || !aligned(ids, 4) || !aligned(w, 4) || !aligned(y, 2)) return MOE_ERR_ALIGN;
    const DecodeShape s{B, k, E, d, I, sd ? 1 : 0};
    if ((rc = check_smem(down_smem_bytes(s)))) return rc;
    return cuda_status(launch_down(s, h, h32, ids, w, view(&wd), view(sd), y, st, pdl));
}

// Carves the grouped layer's buffers out of one workspace (256-byte aligned
// pieces); returns the bytes used.  ws == nullptr only measures.
size_t grouped_carve(int T, int k, int E, int d, int I, bool shared, char* base, GroupedWorkspace* ws) {
    const int64_t ns = (int64_t)T * k + (int64_t)E * (GROUPED_BLOCK - 1);
    const int64_t nb = (ns + GROUPED_BLOCK - 1) / GROUPED_BLOCK;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        char* p = base ? base + off : nullptr;
        off += round_up(bytes, 256);
        return p;
    };
    char* sorted = take((size_t)ns * 4);
    char* eids = take((size_t)nb * 4);
    char* ntpp = take(4);
    char* aws = take(align_workspace_bytes((int64_t)T * k, E));
    char* xmx = take((size_t)T * d * 2);
    char* hs = take((size_t)ns * I * 2);
    char* out = take((size_t)T * k * d * 4);
    const int64_t nsh = shared ? ((int64_t)T + GROUPED_BLOCK - 1) / GROUPED_BLOCK * GROUPED_BLOCK : 0;
    char* sh_sorted = shared ? take((size_t)nsh * 4) : nullptr;
    char* sh_expert = shared ? take((size_t)nsh / GROUPED_BLOCK * 4) : nullptr;
    char* sh_ntpp = shared ? take(4) : nullptr;
    char* sh_h = shared ? take((size_t)nsh * I * 2) : nullptr;
    char* sh_out = shared ? take((size_t)T * d * 4) : nullptr;
    if (ws) {
        ws->sh_sorted = reinterpret_cast<int32_t*>(sh_sorted);
        ws->sh_expert = reinterpret_cast<int32_t*>(sh_expert);
        ws->sh_ntpp = reinterpret_cast<int32_t*>(sh_ntpp);
        ws->n_sh = nsh;
        ws->sh_h = reinterpret_cast<uint16_t*>(sh_h);
        ws->sh_out = reinterpret_cast<float*>(sh_out);
        ws->sorted = reinterpret_cast<int32_t*>(sorted);
        ws->n_sorted = ns;
        ws->expert_ids = reinterpret_cast<int32_t*>(eids);
        ws->n_blocks = nb;
        ws->ntpp = reinterpret_cast<int32_t*>(ntpp);
        ws->align_ws = aws;
        ws->x_mx = reinterpret_cast<uint16_t*>(xmx);
        ws->h_sorted = reinterpret_cast<uint16_t*>(hs);
        ws->out = reinterpret_cast<float*>(out);
    }
    return off;
}

int check_grouped_shape(int T, int k, int E, int d, int I) {
    if (T < 0 || k < 0 || E < 0 || d < 0 || I < 0) return MOE_ERR_ARG;
    if (d == 0 || I == 0 || E == 0 || k == 0 || k > E) return MOE_ERR_SHAPE;
    if (!grouped_shape_ok(d, I)) return MOE_ERR_SHAPE;
    if (E > MOE_ALIGN_MAX_EXPERTS) return MOE_ERR_LIMIT;
    const int64_t ns = (int64_t)T * k + (int64_t)E * (GROUPED_BLOCK - 1);
    if (ns > 0x7fffffffLL || (int64_t)T * k * d > ((int64_t)1 << 40)) return MOE_ERR_LIMIT;
    return MOE_OK;
}

}  // namespace

extern "C" {

int moe_version(void) { return 100; }

const char* moe_strerror(int status) {
    switch (status) {
        case MOE_OK: return "ok";
        case MOE_ERR_ARG: return "invalid argument (NULL pointer or negative size)";
        case MOE_ERR_SHAPE: return "invalid shape (d and I must be multiples of 32, 1 <= k <= E)";
        case MOE_ERR_LIMIT: return "shape beyond a documented limit of the kernels";
        case MOE_ERR_WORKSPACE: return "workspace missing or too small";
        case MOE_ERR_ALIGN: return "pointer not aligned as documented";
        case MOE_ERR_CUDA: return "CUDA runtime error";
        case MOE_ERR_DEVICE: return "a kernel flagged bad input (expert id out of range)";
        default: return "unknown status";
    }
}

int moe_gate_up(const void* x, int B, int d, const int32_t* topk_ids, int k, moe_mx_t w_gate,
                moe_mx_t w_up, int E, int I, const moe_mx_t* shared_gate,
                const moe_mx_t* shared_up, void* h, moe_stream_t stream) {
    return gate_up_checked(x, B, d, topk_ids, k, w_gate, w_up, E, I, shared_gate, shared_up, h, false,
                           (cudaStream_t)stream);
}

int moe_down(const void* h, int B, int k, const int32_t* topk_ids, const float* topk_w,
             moe_mx_t w_down, int E, int d, int I, const moe_mx_t* shared_down, void* y,
             moe_stream_t stream) {
    return down_checked(h, false, B, k, topk_ids, topk_w, w_down, E, d, I, shared_down, y,
                        (cudaStream_t)stream, false);
}

int moe_gate_up_fp4(const void* x, int B, int d, const int32_t* topk_ids, int k, moe_mx_t w_gate,
                    moe_mx_t w_up, int E, int I, const moe_mx_t* shared_gate,
                    const moe_mx_t* shared_up, void* h, moe_stream_t stream) {
    int rc = check_decode_shape(B, k, E, d, I);
    if (rc) return rc;
    if ((shared_gate == nullptr) != (shared_up == nullptr)) return MOE_ERR_ARG;
    if (B == 0) return MOE_OK;
    if (!x || !topk_ids || !h) return MOE_ERR_ARG;
    if ((rc = check_mx(w_gate)) || (rc = check_mx(w_up))) return rc;
    if (shared_gate && ((rc = check_mx(*shared_gate)) || (rc = check_mx(*shared_up)))) return rc;
    if (!aligned(x, 16) || !aligned(h, 16) || !aligned(topk_ids, 4)) return MOE_ERR_ALIGN;
    const DecodeShape s{B, k, E, d, I, shared_gate ? 1 : 0};
    return cuda_status(launch_gate_up_fp4(s, x, topk_ids, view(&w_gate), view(&w_up), view(shared_gate),
                                          view(shared_up), h, (cudaStream_t)stream));
}

int moe_down_fp4(const void* h, int B, int k, const int32_t* topk_ids, const float* topk_w,
                 moe_mx_t w_down, int E, int d, int I, const moe_mx_t* shared_down, void* y,
                 moe_stream_t stream) {
    int rc = check_decode_shape(B, k, E, d, I);
    if (rc) return rc;
    if (B == 0) return MOE_OK;
    if (!h || !topk_ids || !topk_w || !y) return MOE_ERR_ARG;
    if ((rc = check_mx(w_down))) return rc;
    if (shared_down && (rc = check_mx(*shared_down))) return rc;
    if (!aligned(h, 16) || !aligned(topk_ids, 4) || !aligned(topk_w, 4) || !aligned(y, 2)) return MOE_ERR_ALIGN;
    const DecodeShape s{B, k, E, d, I, shared_down ? 1 : 0};
    return cuda_status(launch_down_fp4(s, h, topk_ids, topk_w, view(&w_down), view(shared_down), y,
                                       (cudaStream_t)stream));
}

int moe_layer_workspace_bytes(int B, int k, int I, int has_shared, size_t* bytes) {
    if (!bytes || B < 0 || k < 0 || I < 0) return MOE_ERR_ARG;
    *bytes = round_up(h_bytes(B, k, I, has_shared ? 1 : 0), 256);
    return MOE_OK;
}

int moe_layer(const void* x, int B, int d, const int32_t* topk_ids, const float* topk_w, int k,
              moe_mx_t w_gate, moe_mx_t w_up, moe_mx_t w_down, int E, int I,
              const moe_mx_t* shared_gate, const moe_mx_t* shared_up,
              const moe_mx_t* shared_down, void* workspace, size_t workspace_bytes, void* y,
              moe_stream_t stream) {
    int rc = check_decode_shape(B, k, E, d, I);
    if (rc) return rc;
    const int ns = (shared_gate != nullptr) + (shared_up != nullptr) + (shared_down != nullptr);
    if (ns != 0 && ns != 3) return MOE_ERR_ARG;
    if (B == 0) return MOE_OK;
    size_t need = 0;
    moe_layer_workspace_bytes(B, k, I, ns == 3, &need);
    if (!workspace || workspace_bytes < need) return MOE_ERR_WORKSPACE;
    if (!aligned(workspace, 256)) return MOE_ERR_ALIGN;
    // validate the down pass's arguments too before the first launch
    if (!topk_w || !y) return MOE_ERR_ARG;
    if ((rc = check_mx(w_down))) return rc;
    if (shared_down && (rc = check_mx(*shared_down))) return rc;
    if (!aligned(topk_w, 4) || !aligned(y, 2)) return MOE_ERR_ALIGN;
    const DecodeShape s{B, k, E, d, I, ns == 3 ? 1 : 0};
    if ((rc = check_smem(down_smem_bytes(s)))) return rc;
    cudaStream_t st = (cudaStream_t)stream;
    const bool h32 = down_reads_h32(s, view(&w_down), view(shared_down));
    rc = gate_up_checked(x, B, d, topk_ids, k, w_gate, w_up, E, I, shared_gate, shared_up,
                         workspace, h32, st);
    if (rc) return rc;
    return down_checked(workspace, h32, B, k, topk_ids, topk_w, w_down, E, d, I, shared_down, y, st, true);
}

int moe_layer_host_workspace_bytes(int B, int d, int k, int I, int has_shared, size_t* bytes) {
    if (!bytes || B < 0 || d < 0 || k < 0 || I < 0) return MOE_ERR_ARG;
    size_t hb = 0;
    moe_layer_workspace_bytes(B, k, I, has_shared, &hb);
    const size_t xb = round_up((size_t)B * d * 2, 256);
    const size_t ib = round_up((size_t)B * k * 4, 256);
    const size_t yb = round_up((size_t)B * d * 2, 256);
    *bytes = hb + xb + 2 * ib + yb;
    return MOE_OK;
}

int moe_layer_host(const void* x_host, int B, int d, const int32_t* topk_ids_host,
                   const float* topk_w_host, int k, moe_mx_t w_gate, moe_mx_t w_up,
                   moe_mx_t w_down, int E, int I, const moe_mx_t* shared_gate,
                   const moe_mx_t* shared_up, const moe_mx_t* shared_down, void* workspace,
                   size_t workspace_bytes, void* y_host, moe_stream_t stream) {
    int rc = check_decode_shape(B, k, E, d, I);
    if (rc) return rc;
    const int ns = (shared_gate != nullptr) + (shared_up != nullptr) + (shared_down != nullptr);
    if (ns != 0 && ns != 3) return MOE_ERR_ARG;
    if (B == 0) return MOE_OK;
    if (!x_host || !topk_ids_host || !topk_w_host || !y_host) return MOE_ERR_ARG;
    size_t need = 0, hb = 0;
    moe_layer_host_workspace_bytes(B, d, k, I, ns == 3, &need);
    moe_layer_workspace_bytes(B, k, I, ns == 3, &hb);
    if (!workspace || workspace_bytes < need) return MOE_ERR_WORKSPACE;
    if (!aligned(workspace, 256)) return MOE_ERR_ALIGN;
    char* p = static_cast<char*>(workspace) + hb;
    void* xd = p;
    p += round_up((size_t)B * d * 2, 256);
    int32_t* idd = reinterpret_cast<int32_t*>(p);
    p += round_up((size_t)B * k * 4, 256);
    float* wdv = reinterpret_cast<float*>(p);
    p += round_up((size_t)B * k * 4, 256);
    void* yd = p;
    cudaStream_t st = (cudaStream_t)stream;
    cudaError_t err;
    if ((err = cudaMemcpyAsync(xd, x_host, (size_t)B * d * 2, cudaMemcpyHostToDevice, st)) ||
        (err = cudaMemcpyAsync(idd, topk_ids_host, (size_t)B * k * 4, cudaMemcpyHostToDevice, st)) ||
        (err = cudaMemcpyAsync(wdv, topk_w_host, (size_t)B * k * 4, cudaMemcpyHostToDevice, st)))
        return MOE_ERR_CUDA;
    rc = moe_layer(xd, B, d, idd, wdv, k, w_gate, w_up, w_down, E, I, shared_gate, shared_up,
                   shared_down, workspace, hb, yd, stream);
    if (rc) return rc;
    if (cudaMemcpyAsync(y_host, yd, (size_t)B * d * 2, cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}

int moe_layer_grouped_workspace_bytes(int T, int k, int E, int d, int I, int has_shared, size_t* bytes) {
    if (!bytes) return MOE_ERR_ARG;
    const int rc = check_grouped_shape(T, k, E, d, I);
    if (rc) return rc;
    *bytes = grouped_carve(T, k, E, d, I, has_shared != 0, nullptr, nullptr);
    return MOE_OK;
}

int moe_layer_grouped(const void* x, int T, int d, const int32_t* topk_ids, const float* topk_w, int k,
                      moe_mx_t w_gate, moe_mx_t w_up, moe_mx_t w_down, int E, int I,
                      const moe_mx_t* shared_gate, const moe_mx_t* shared_up, const moe_mx_t* shared_down,
                      int act_mx, void* workspace, size_t workspace_bytes, void* y, moe_stream_t stream) {
    int rc = check_grouped_shape(T, k, E, d, I);
    if (rc) return rc;
    if (act_mx != 0 && act_mx != 1) return MOE_ERR_ARG;
    const int ns = (shared_gate != nullptr) + (shared_up != nullptr) + (shared_down != nullptr);
    if (ns != 0 && ns != 3) return MOE_ERR_ARG;
    if (T == 0) return MOE_OK;
    if (!x || !topk_ids || !topk_w || !y) return MOE_ERR_ARG;
    if ((rc = check_mx(w_gate)) || (rc = check_mx(w_up)) || (rc = check_mx(w_down))) return rc;
    if (!aligned(w_gate.s, 16) || !aligned(w_up.s, 16) || !aligned(w_down.s, 16)) return MOE_ERR_ALIGN;
    if (ns == 3) {
        if ((rc = check_mx(*shared_gate)) || (rc = check_mx(*shared_up)) || (rc = check_mx(*shared_down))) return rc;
        if (!aligned(shared_gate->s, 16) || !aligned(shared_up->s, 16) || !aligned(shared_down->s, 16))
            return MOE_ERR_ALIGN;
    }
    if (!aligned(x, 32) || !aligned(topk_ids, 4) || !aligned(topk_w, 4) || !aligned(y, 8)) return MOE_ERR_ALIGN;
    const size_t need = grouped_carve(T, k, E, d, I, ns == 3, nullptr, nullptr);
    if (!workspace || workspace_bytes < need) return MOE_ERR_WORKSPACE;
    if (!aligned(workspace, 256)) return MOE_ERR_ALIGN;
    DeviceInfo di;
    if (device_info(&di) != cudaSuccess) return MOE_ERR_CUDA;
    if (align_smem_bytes(E) > (size_t)di.max_smem_optin || grouped_smem_bytes(d, I) > (size_t)di.max_smem_optin)
        return MOE_ERR_LIMIT;
    GroupedWorkspace ws{};
    grouped_carve(T, k, E, d, I, ns == 3, static_cast<char*>(workspace), &ws);
    return cuda_status(launch_grouped(static_cast<const uint16_t*>(x), T, d, topk_ids, topk_w, k, view(&w_gate),
                                      view(&w_up), view(&w_down), view(shared_gate), view(shared_up),
                                      view(shared_down), E, I, act_mx != 0, ws, static_cast<uint16_t*>(y),
                                      (cudaStream_t)stream));
}

int moe_router_topk(const float* logits, int B, int E, int k, int score, float scale, int32_t* topk_ids,
                    float* topk_w, moe_stream_t stream) {
    if (B < 0 || E < 1 || k < 1 || (score != MOE_ROUTER_SOFTMAX && score != MOE_ROUTER_SIGMOID))
        return MOE_ERR_ARG;
    if (k > E) return MOE_ERR_SHAPE;
    if (E > MOE_ROUTER_MAX_EXPERTS || k > MOE_ROUTER_MAX_K) return MOE_ERR_LIMIT;
    if (B == 0) return MOE_OK;
    if (!logits || !topk_ids || !topk_w) return MOE_ERR_ARG;
    if (!aligned(logits, 4) || !aligned(topk_ids, 4) || !aligned(topk_w, 4)) return MOE_ERR_ALIGN;
    return cuda_status(launch_router(logits, B, E, k, score, scale, topk_ids, topk_w, (cudaStream_t)stream));
}

int moe_mx_requant(const void* in, void* out, int64_t rows, int K, moe_stream_t stream) {
    if (rows < 0) return MOE_ERR_ARG;
    if (K <= 0 || K % 32) return MOE_ERR_SHAPE;
    if (rows > INT64_MAX / K) return MOE_ERR_LIMIT;
    if (rows == 0) return MOE_OK;
    if (!in || !out) return MOE_ERR_ARG;
    if (!aligned(in, 16) || !aligned(out, 16)) return MOE_ERR_ALIGN;
    return cuda_status(launch_mx_requant(in, out, rows, K, (cudaStream_t)stream));
}

int moe_align_sizes(int T, int k, int E, int block_size, int64_t* n_sorted, int64_t* n_blocks,
                    size_t* ws_bytes) {
    if (T < 0 || k < 1 || E < 1 || block_size < 1) return MOE_ERR_ARG;
    if (E > MOE_ALIGN_MAX_EXPERTS) return MOE_ERR_LIMIT;
    const int64_t ns = (int64_t)T * k + (int64_t)E * (block_size - 1);
    if (ns > 0x7fffffffLL) return MOE_ERR_LIMIT;
    if (n_sorted) *n_sorted = ns;
    if (n_blocks) *n_blocks = (ns + block_size - 1) / block_size;
    if (ws_bytes) *ws_bytes = align_workspace_bytes((int64_t)T * k, E);
    return MOE_OK;
}

int moe_align_block_size(const int32_t* topk_ids, int T, int k, int E, int block_size,
                         int32_t* sorted_token_ids, int32_t* expert_ids,
                         int32_t* num_tokens_post_pad, void* workspace, size_t workspace_bytes,
                         moe_stream_t stream) {
    int64_t ns = 0, nb = 0;
    size_t wsb = 0;
    int rc = moe_align_sizes(T, k, E, block_size, &ns, &nb, &wsb);
    if (rc) return rc;
    if (!sorted_token_ids || !expert_ids || !num_tokens_post_pad) return MOE_ERR_ARG;
    if (T > 0 && !topk_ids) return MOE_ERR_ARG;
    if (!workspace || workspace_bytes < wsb) return MOE_ERR_WORKSPACE;
    if (!aligned(workspace, 16) || !aligned(sorted_token_ids, 4) || !aligned(expert_ids, 4) ||
        !aligned(num_tokens_post_pad, 4) || (topk_ids && !aligned(topk_ids, 4)))
        return MOE_ERR_ALIGN;
    DeviceInfo di;
    if (device_info(&di) != cudaSuccess) return MOE_ERR_CUDA;
    if (align_smem_bytes(E) > (size_t)di.max_smem_optin) return MOE_ERR_LIMIT;
    return cuda_status(launch_align(topk_ids, T, k, E, block_size, sorted_token_ids, ns, expert_ids,
                                    nb, num_tokens_post_pad, workspace, (cudaStream_t)stream));
}

int moe_align_static_fits(int T, int k, int E) {
    size_t wsb = 0;
    if (moe_align_sizes(T, k, E, 1, nullptr, nullptr, &wsb) != MOE_OK) return 0;
    return wsb <= MOE_ALIGN_STATIC_SCRATCH_BYTES ? 1 : 0;
}

int moe_align_block_size_static(const int32_t* topk_ids, int T, int k, int E, int block_size,
                                int32_t* sorted_token_ids, int32_t* expert_ids,
                                int32_t* num_tokens_post_pad, moe_stream_t stream) {
    int64_t ns = 0, nb = 0;
    size_t wsb = 0;
    int rc = moe_align_sizes(T, k, E, block_size, &ns, &nb, &wsb);
    if (rc) return rc;
    if (wsb > MOE_ALIGN_STATIC_SCRATCH_BYTES) return MOE_ERR_LIMIT;
    void* scratch = nullptr;
    if (align_static_scratch(&scratch) != cudaSuccess) return MOE_ERR_CUDA;
    return moe_align_block_size(topk_ids, T, k, E, block_size, sorted_token_ids, expert_ids,
                                num_tokens_post_pad, scratch, MOE_ALIGN_STATIC_SCRATCH_BYTES, stream);
}

int moe_copy(void* dst, const void* src, size_t bytes, moe_stream_t stream) {
    if (!dst || !src) return MOE_ERR_ARG;
    if (!aligned(dst, 32) || !aligned(src, 32) || bytes % 32) return MOE_ERR_ALIGN;
    return cuda_status(launch_copy(dst, src, bytes, (cudaStream_t)stream));
}

int moe_device_error(moe_stream_t stream, int* bits) {
    if (!bits) return MOE_ERR_ARG;
    DeviceInfo di;
    if (device_info(&di) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return MOE_ERR_CUDA;
    int v = 0;
    if (cudaMemcpy(&v, di.err_word, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (v) {
        const int zero = 0;
        if (cudaMemcpy(di.err_word, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
            return MOE_ERR_CUDA;
    }
    *bits = v;
    return v ? MOE_ERR_DEVICE : MOE_OK;
}

}  // extern "C"

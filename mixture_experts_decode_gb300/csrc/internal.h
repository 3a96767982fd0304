// internal.h -- launch interfaces between the C-ABI layer and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace moedec {

struct MXView {
    const uint8_t* w;
    const uint8_t* s;
};

struct DecodeShape {
    int B, k, E, d, I, S;  // S = 1 with a shared expert
};

// Device properties cached per device (SM count, shared memory per block).
struct DeviceInfo {
    int sm_count;
    int max_smem_optin;
    int smem_per_sm;
    int* err_word;  // sticky device error bits (MOE_DEVERR_*)
};
cudaError_t device_info(DeviceInfo* out);

// h32: the intermediate is FP32 in the row-tile down pass's order (h32_pos)
// instead of the interface's BF16 [B][k+S][I]; the layer uses it when
// down_reads_h32() holds for its shape and weights.
cudaError_t launch_gate_up(const DecodeShape& s, const void* x, const int32_t* ids, MXView wg,
                           MXView wu, MXView shg, MXView shu, void* h, bool h32, cudaStream_t st);
cudaError_t launch_down(const DecodeShape& s, const void* h, bool h32, const int32_t* ids, const float* w,
                        MXView wd, MXView shd, void* y, cudaStream_t st, bool after_gate_up);
bool down_reads_h32(const DecodeShape& s, MXView wd, MXView shd);
cudaError_t launch_router(const float* logits, int B, int E, int k, int score, float scale, int32_t* ids, float* w,
                          cudaStream_t st);
cudaError_t launch_mx_requant(const void* in, void* out, int64_t rows, int K, cudaStream_t st);
cudaError_t launch_gate_up_fp4(const DecodeShape& s, const void* x, const int32_t* ids, MXView wg, MXView wu,
                               MXView shg, MXView shu, void* h, cudaStream_t st);
// The grouped (one pass over each distinct expert's rows) kernels with MXFP4
// weights: return false, launching nothing, when the shape or alignment
// does not suit them; else launch and set *err.
bool launch_gate_up_grouped_fp4(const DecodeShape& s, const void* x, const int32_t* ids, MXView wg, MXView wu,
                                MXView shg, MXView shu, void* h, cudaStream_t st, cudaError_t* err);
bool launch_down_grouped_fp4(const DecodeShape& s, const void* h, const int32_t* ids, const float* w, MXView wd,
                             MXView shd, void* y, cudaStream_t st, cudaError_t* err);
cudaError_t launch_down_fp4(const DecodeShape& s, const void* h, const int32_t* ids, const float* w, MXView wd,
                            MXView shd, void* y, cudaStream_t st);
// Shared-memory bytes the decode kernels need; 0 if the shape is beyond the
// supported limits.
size_t gate_up_smem_bytes(const DecodeShape& s);
size_t down_smem_bytes(const DecodeShape& s);

cudaError_t launch_align(const int32_t* ids, int T, int k, int E, int block_size, int32_t* sorted,
                         int64_t n_sorted, int32_t* expert_ids, int64_t n_blocks, int32_t* ntpp,
                         void* ws, cudaStream_t st);
size_t align_workspace_bytes(int64_t n, int E);
size_t align_smem_bytes(int E);
// Device address of the library's fixed align scratch on the current device.
cudaError_t align_static_scratch(void** out);

cudaError_t launch_copy(void* dst, const void* src, size_t bytes, cudaStream_t st);

// The expert-centric (grouped GEMM) layer's device buffers, carved from the
// caller's workspace.
struct GroupedWorkspace {
    int32_t* sorted;      // [n_sorted] flat slot of each sorted row (T*k = pad)
    int64_t n_sorted;
    int32_t* expert_ids;  // [n_blocks]
    int64_t n_blocks;
    int32_t* ntpp;        // rows used, a multiple of the block size
    void* align_ws;
    uint16_t* x_mx;       // [T][d] x rounded through MXFP8 (act_mx only)
    uint16_t* h_sorted;   // [n_sorted][I] BF16
    float* out;           // [T*k][d] FP32 per-slot partial outputs
    // the shared expert's pass (null without one): every token, in order
    int32_t* sh_sorted;   // [n_sh] token of each row (T = pad)
    int32_t* sh_expert;   // [n_sh / 128] all 0
    int32_t* sh_ntpp;     // n_sh
    int64_t n_sh;         // T rounded up to a multiple of 128
    uint16_t* sh_h;       // [n_sh][I] BF16
    float* sh_out;        // [T][d] FP32
};
constexpr int GROUPED_BLOCK = 128;  // sorted rows per block
bool grouped_shape_ok(int d, int I);
size_t grouped_smem_bytes(int d, int I);
// shg / shu / shd: the shared expert's matrices ([1][rows][K]) or all null.
cudaError_t launch_grouped(const uint16_t* x, int T, int d, const int32_t* ids, const float* w, int k, MXView wg,
                           MXView wu, MXView wd, MXView shg, MXView shu, MXView shd, int E, int I, bool act_mx,
                           const GroupedWorkspace& ws, uint16_t* y, cudaStream_t st);

}  // namespace moedec

/*
 * moedec.h -- C ABI of libmoedec.so, a GB300 (sm_103a) small-batch
 * mixture-of-experts expert-FFN decode layer with MXFP8 weights, plus the
 * expert-centric align-and-sort bookkeeping.
 *
 * Sources (web pages; cited by title and section):
 *   [WD] "Warp decode" (cursor.com blog): the decode layer as two passes --
 *        a fused gate/up pass (section "兩個 kernel 的運作方式", how the two
 *        kernels work) and a down pass that folds every routed expert's
 *        routing weight into one FP32 accumulator per output value, with no
 *        gather buffer, per-expert output buffer or separate combine
 *        (sections "消除緩衝區" eliminating buffers, "準確度改進" accuracy).
 *   [AS] "AMD GPU性能暴涨7倍 ... 高效MoE支持任意专家数量" (aizws.net): MoE
 *        Align & Sort and its multi-block count / cumsum / placement
 *        algorithm (section "编写对AMD设备友好的CUDA实现").
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers unless the name says _host.
 *     The caller owns every buffer; the library never allocates device or
 *     host memory and never frees anything.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream).  Host-side argument checks happen before any launch;
 *     a call that returns an error has launched nothing.
 *   - Return value: MOE_OK (0) or a negative MOE_ERR_* code; moe_strerror()
 *     names it.
 *   - BF16 tensors are passed as `void*` (raw 16-bit patterns).
 *   - MXFP8 weights: one byte per element holding an E4M3 code (OCP OFP8,
 *     no infinities), row-major with K innermost, plus one E8M0 scale byte
 *     per 32 consecutive elements along K (value 2^(s-127)); the scale
 *     array is row-major [rows][K/32].  K must be a multiple of 32.
 *   - Device-side input checks: an expert id outside [0, E) never causes
 *     an out-of-bounds access; the slot is skipped and a sticky device error
 *     bit is set, which moe_device_error() reports.
 */
#ifndef MOEDEC_H
#define MOEDEC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* moe_stream_t; /* identical to cudaStream_t */

enum moe_status {
    MOE_OK = 0,
    MOE_ERR_ARG = -1,       /* NULL pointer where one is required, negative size */
    MOE_ERR_SHAPE = -2,     /* d or I not a multiple of 32, k > E, ... */
    MOE_ERR_LIMIT = -3,     /* beyond a documented limit of the decode kernels */
    MOE_ERR_WORKSPACE = -4, /* workspace missing or smaller than required */
    MOE_ERR_ALIGN = -5,     /* pointer not aligned as documented */
    MOE_ERR_CUDA = -6,      /* a CUDA runtime call or launch failed */
    MOE_ERR_DEVICE = -7     /* a kernel flagged bad input (see moe_device_error) */
};

/* Device error bits reported by moe_device_error(). */
#define MOE_DEVERR_EXPERT_ID 0x1 /* an expert id outside [0, E) was skipped */
#define MOE_DEVERR_TIMEOUT 0x2   /* a kernel's bounded wait gave up (never expected) */
#define MOE_DEVERR_LOGIT 0x4     /* a router row had fewer than k logits above -inf */

/* Limits of the decode kernels (moe_gate_up, moe_down, moe_layer*). */
#define MOE_MAX_EXPERTS 1024  /* E */
#define MOE_MAX_TOKENS 256    /* B */
#define MOE_MAX_SLOTS 2048    /* B * k */
/* Limits of moe_align_block_size. */
#define MOE_ALIGN_MAX_EXPERTS 1024
/* Limits and score kinds of moe_router_topk. */
#define MOE_ROUTER_MAX_EXPERTS 1024
#define MOE_ROUTER_MAX_K 32
#define MOE_ROUTER_SOFTMAX 0
#define MOE_ROUTER_SIGMOID 1

/* One MXFP8 weight tensor: codes [E][rows][K] and scales [E][rows][K/32].
 * Both device pointers; `w` must be 32-byte aligned (K % 32 == 0 then keeps
 * every row 32-byte aligned). */
typedef struct {
    const uint8_t* w;
    const uint8_t* s;
} moe_mx_t;

/* Library version: major*10000 + minor*100 + patch. */
int moe_version(void);

/* Human-readable name of a status code (static string, never NULL). */
const char* moe_strerror(int status);

/*
 * moe_gate_up -- fused gate/up pass [WD, how the two kernels work].
 *   For each token b < B, routed slot j < k (expert e = topk_ids[b*k+j])
 *   and, when a shared expert is given, slot j = k (the shared expert),
 *   and each intermediate neuron n < I:
 *     g = sum_c x[b,c] * deq(Wg[e,n,c]),  u = sum_c x[b,c] * deq(Wu[e,n,c])
 *     h[b,j,n] = bf16_rn( g * sigmoid(g) * u )
 *   with deq() the MXFP8 dequantisation, FP32 products and accumulation.
 *   x reads once per distinct expert; each weight row is streamed once.
 * Arguments
 *   x         BF16 [B][d], 16-byte aligned.
 *   topk_ids  int32 [B][k].
 *   w_gate    MXFP8 [E][I][d];  w_up  MXFP8 [E][I][d].
 *   shared_gate, shared_up: NULL for no shared expert, else MXFP8 [1][I][d]
 *             (both or neither).
 *   h         BF16 [B][k+S][I] output (S = 1 with a shared expert), 4-byte
 *             aligned.  Every element is written.
 * Limits: B <= MOE_MAX_TOKENS, B*k <= MOE_MAX_SLOTS, E <= MOE_MAX_EXPERTS,
 *   1 <= k <= E, d and I multiples of 32.  B == 0 is a no-op.
 */
int moe_gate_up(const void* x, int B, int d, const int32_t* topk_ids, int k, moe_mx_t w_gate,
                moe_mx_t w_up, int E, int I, const moe_mx_t* shared_gate,
                const moe_mx_t* shared_up, void* h, moe_stream_t stream);

/*
 * moe_down -- down pass with the routing-weighted combine folded in
 * [WD, how the two kernels work; eliminating buffers]:
 *   y[b,o] = bf16_rn( sum_{j<k} topk_w[b,j] * sum_i h[b,j,i] * deq(Wd[e_j,o,i])
 *                     + S * 1.0 * sum_i h[b,k,i] * deq(Wsd[o,i]) )
 *   one FP32 accumulator per output value across all routed experts; no
 *   per-expert output buffer and no separate combine step.
 * Arguments
 *   h         BF16 [B][k+S][I] (as written by moe_gate_up), 16-byte aligned.
 *   topk_ids  int32 [B][k];  topk_w  float32 [B][k].
 *   w_down    MXFP8 [E][d][I];  shared_down NULL or MXFP8 [1][d][I].
 *   y         BF16 [B][d] output; every element is written.
 * Limits as for moe_gate_up.
 */
int moe_down(const void* h, int B, int k, const int32_t* topk_ids, const float* topk_w,
             moe_mx_t w_down, int E, int d, int I, const moe_mx_t* shared_down, void* y,
             moe_stream_t stream);

/*
 * moe_gate_up_fp4, moe_down_fp4 -- the two passes with MXFP4 weights: the
 * formulas, arguments, limits and outputs of moe_gate_up / moe_down, except
 * that each moe_mx_t's codes are E2M1 (OCP MX v1.0 FP4: 1 sign, 2 exponent
 * bits with bias 1, 1 mantissa bit), two per byte with the lower K index in
 * the low nibble: gate/up codes [E][I][d/2] bytes, down codes [E][d][I/2];
 * the E8M0 scales stay one per 32 elements along K ([E][I][d/32],
 * [E][d][I/32]).  The GC-MoE page names FP8/FP4 MoE operators; MXFP4 halves
 * the weight bytes of MXFP8.  x and h 16-byte aligned, codes 32-byte aligned.
 * For B >= 2 (and d % 512 == 0, I % 256 == 0, 16-byte aligned scales) the
 * passes run on the same row-tile kernels as MXFP8, each distinct expert's
 * rows streamed once per call; otherwise one warp computes one output value
 * ([WD, how the two kernels work]).  An expert id outside [0, E) sets
 * MOE_DEVERR_EXPERT_ID, its h is written as zero and down skips the slot.
 */
int moe_gate_up_fp4(const void* x, int B, int d, const int32_t* topk_ids, int k, moe_mx_t w_gate,
                    moe_mx_t w_up, int E, int I, const moe_mx_t* shared_gate,
                    const moe_mx_t* shared_up, void* h, moe_stream_t stream);
int moe_down_fp4(const void* h, int B, int k, const int32_t* topk_ids, const float* topk_w,
                 moe_mx_t w_down, int E, int d, int I, const moe_mx_t* shared_down, void* y,
                 moe_stream_t stream);

/* Bytes of workspace moe_layer needs: B*(k+S)*I*4, room for the
 * intermediate h held as FP32. */
int moe_layer_workspace_bytes(int B, int k, int I, int has_shared, size_t* bytes);

/*
 * moe_layer -- the whole decode layer: the gate/up pass then the down pass on
 * the same stream, with the results of moe_gate_up followed by moe_down.
 * The intermediate h lives at the start of `workspace` (>=
 * moe_layer_workspace_bytes, 256-byte aligned); its layout there is internal:
 * when I % 256 == 0 (and the weight arrays are aligned for tensor copies) it
 * is kept as FP32 (the same BF16-rounded values) in the order the down pass
 * reads, so that pass loads it without conversion; otherwise as the BF16
 * [B][k+S][I] of moe_gate_up.  Shared expert: all three shared pointers or
 * none.
 */
int moe_layer(const void* x, int B, int d, const int32_t* topk_ids, const float* topk_w, int k,
              moe_mx_t w_gate, moe_mx_t w_up, moe_mx_t w_down, int E, int I,
              const moe_mx_t* shared_gate, const moe_mx_t* shared_up,
              const moe_mx_t* shared_down, void* workspace, size_t workspace_bytes, void* y,
              moe_stream_t stream);

/* Bytes of device workspace moe_layer_host needs. */
int moe_layer_host_workspace_bytes(int B, int d, int k, int I, int has_shared, size_t* bytes);

/*
 * moe_layer_host -- moe_layer with the per-step activations in HOST memory:
 * copies x_host (BF16 [B][d]), topk_ids_host (int32 [B][k]) and topk_w_host
 * (float32 [B][k]) to device staging inside `workspace`, runs the layer, and
 * copies y back to y_host (BF16 [B][d]), all asynchronously on `stream`.
 * Host buffers should be pinned (page-locked) for the copies to be
 * asynchronous; the caller synchronises the stream before reading y_host.
 * Weights stay device pointers.  workspace >= moe_layer_host_workspace_bytes,
 * 256-byte aligned.
 */
int moe_layer_host(const void* x_host, int B, int d, const int32_t* topk_ids_host,
                   const float* topk_w_host, int k, moe_mx_t w_gate, moe_mx_t w_up,
                   moe_mx_t w_down, int E, int I, const moe_mx_t* shared_gate,
                   const moe_mx_t* shared_up, const moe_mx_t* shared_down, void* workspace,
                   size_t workspace_bytes, void* y_host, moe_stream_t stream);

/*
 * moe_layer_grouped -- the same layer computed expert-centrically, the way
 * prefill and large batches are served [WD, section "Warp decode 與 Composer
 * 訓練": expert-centric packing stays the right choice there; AS: the sorted
 * blocks feed grouped GEMMs].  Steps, all on `stream`:
 *   1. moe_align_block_size with block_size 128 (into the workspace);
 *   2. if act_mx, x is rounded through MXFP8 (moe_mx_requant) first;
 *   3. per block of 128 sorted slots and expert e:
 *        g, u = the slots' x rows times deq(Wg[e]), deq(Wu[e]) (tensor
 *        cores, BF16 operands -- exact for MXFP8 values with scale bytes
 *        >= 3 -- FP32 sums),
 *        h = bf16_rn( g * sigmoid(g) * u )  per slot;
 *   4. if act_mx, h is rounded through MXFP8;
 *   5. out[slot] = h[slot] times deq(Wd[e]) (FP32);
 *   6. y[t,o] = bf16_rn( sum_j topk_w[t,j] * out[t*k+j, o] ), j in order.
 * With a shared expert (all three shared pointers, [1][rows][K] each) steps
 * 3-5 also run as a one-expert layer over every token in order, and step 6
 * adds its row with weight 1.0 after the k routed slots.  The sums run in
 * the tensor cores' order, not the decode layer's, so the results agree with
 * moe_layer to FP32 rounding, not bit for bit.
 * Arguments
 *   x         BF16 [T][d], 32-byte aligned.  topk_ids int32 [T][k]; an id
 *             outside [0, E) adds nothing and sets MOE_DEVERR_EXPERT_ID.
 *   topk_w    float32 [T][k].  weights as for moe_layer; each scale array
 *             16-byte aligned.
 *   shared_gate, shared_up, shared_down: NULL for no shared expert, else
 *             MXFP8 [1][I][d], [1][I][d], [1][d][I] (all three or none).
 *   d, I      multiples of 128.  E <= MOE_ALIGN_MAX_EXPERTS; T*k +
 *             E*127 < 2^31.  No limit on T beyond that.
 *   act_mx    0: activations as given (the decode layer's numerics);
 *             1: x and h rounded through MXFP8, the conventional path.
 *   workspace >= moe_layer_grouped_workspace_bytes(..., has_shared, ...),
 *             256-byte aligned; its layout is internal.
 *   y         BF16 [T][d], 8-byte aligned.
 * Errors: MOE_ERR_SHAPE (d or I not a multiple of 128, k > E),
 * MOE_ERR_LIMIT, MOE_ERR_WORKSPACE, MOE_ERR_ALIGN, MOE_ERR_CUDA.
 */
int moe_layer_grouped_workspace_bytes(int T, int k, int E, int d, int I, int has_shared, size_t* bytes);
int moe_layer_grouped(const void* x, int T, int d, const int32_t* topk_ids, const float* topk_w, int k,
                      moe_mx_t w_gate, moe_mx_t w_up, moe_mx_t w_down, int E, int I,
                      const moe_mx_t* shared_gate, const moe_mx_t* shared_up, const moe_mx_t* shared_down,
                      int act_mx, void* workspace, size_t workspace_bytes, void* y, moe_stream_t stream);

/*
 * moe_align_sizes -- output and workspace sizes for moe_align_block_size:
 *   n_sorted = T*k + E*(block_size-1)  (every expert's run padded at worst)
 *   n_blocks = ceil(n_sorted / block_size)
 *   ws_bytes = device workspace moe_align_block_size needs.
 * Any of the output pointers may be NULL.
 */
int moe_align_sizes(int T, int k, int E, int block_size, int64_t* n_sorted, int64_t* n_blocks,
                    size_t* ws_bytes);

/*
 * moe_align_block_size -- expert-centric bookkeeping [AS]: a stable
 * counting sort of the flat slot indices f = t*k + j by expert id
 * topk_ids[f], each expert's run padded to a multiple of block_size.
 * Multi-block: per-block shared-memory histograms (count), a prefix over
 * blocks and experts with padding (cumsum), then parallel placement.
 * Outputs (device, int32):
 *   sorted_token_ids [n_sorted]: expert e's flat indices in increasing f
 *     order starting at start[e] = sum_{e'<e} pad(e'), followed by sentinel
 *     T*k up to the padded length; entries past num_tokens_post_pad hold
 *     T*k too.
 *   expert_ids [n_blocks]: owning expert of each block_size block; -1 for
 *     blocks past num_tokens_post_pad / block_size.
 *   num_tokens_post_pad [1]: sum over experts of the padded run lengths.
 * Every output element is written.  Ties are broken by flat index, so the
 * result is unique and bit-exact.  workspace >= ws_bytes of
 * moe_align_sizes, 16-byte aligned.  T*k must fit in int32.
 * Limits: 1 <= E <= MOE_ALIGN_MAX_EXPERTS, block_size >= 1, k >= 1.
 */
int moe_align_block_size(const int32_t* topk_ids, int T, int k, int E, int block_size,
                         int32_t* sorted_token_ids, int32_t* expert_ids,
                         int32_t* num_tokens_post_pad, void* workspace, size_t workspace_bytes,
                         moe_stream_t stream);

/*
 * moe_align_block_size_static -- moe_align_block_size for callers that
 * cannot provide device scratch memory.  (No counterpart in the source
 * pages; this is a convenience of this library.)
 * Some callers can only hand over their inputs and outputs: an engine that
 * forbids device allocation after start-up, a plugin or custom-op host that
 * owns all device memory and passes no workspace, or code that must not call
 * cudaMalloc because it may run while a stream is being captured.  This
 * variant needs no workspace argument: its scratch is a fixed array inside
 * the library (MOE_ALIGN_STATIC_SCRATCH_BYTES, held on every GPU that loads
 * the library until the process exits).  It never calls cudaMalloc,
 * cudaFree or any other allocating routine.
 * Arguments and outputs are those of moe_align_block_size, minus workspace.
 * Returns MOE_ERR_LIMIT when the problem needs more scratch than the array
 * holds (see moe_align_static_fits).  The first call on each device looks up
 * the array's device address; make that first call before any stream
 * capture on that device.  Every call shares the one array: each call
 * overwrites the part it uses before reading it, but calls whose executions
 * overlap on the GPU (different streams, or graphs replayed concurrently)
 * race on it and must be serialised by the caller.
 */
#define MOE_ALIGN_STATIC_SCRATCH_BYTES (256u * 1024u)
int moe_align_block_size_static(const int32_t* topk_ids, int T, int k, int E, int block_size,
                                int32_t* sorted_token_ids, int32_t* expert_ids,
                                int32_t* num_tokens_post_pad, moe_stream_t stream);

/* 1 if moe_align_block_size_static can serve (T, k, E), else 0. */
int moe_align_static_fits(int T, int k, int E);

/*
 * moe_copy -- device-to-device copy kernel used as the HBM bandwidth
 * reference (contiguous 32-byte loads and stores).  dst and src 32-byte
 * aligned; bytes a multiple of 32.
 */
int moe_copy(void* dst, const void* src, size_t bytes, moe_stream_t stream);

/*
 * moe_router_topk -- the routing step in front of the decode layer: for each
 * token b, the k largest of its E router logits, in descending order (ties:
 * the lower expert index first), with their routing weights [AS, section
 * "MoE Align & Sort CUDA算法在其他开源平台的实现": FasterTransformer's fused
 * topk_gating_softmax].
 *   score MOE_ROUTER_SOFTMAX: w_j = scale * p_j / (sum of the k chosen p),
 *     p = softmax over all E logits (renormalised top-k; scale 1 for the
 *     plain renormalisation);
 *   score MOE_ROUTER_SIGMOID: w_j = scale * s_j / (sum of the k chosen s),
 *     s = 1 / (1 + exp(-logit)) (e.g. scale 2.5 for the DeepSeek-V3 gate).
 * Both score maps are increasing, so the choice is the k largest logits.
 *   logits    float32 [B][E], row-major; finite values expected.  A row with
 *             fewer than k logits above -inf (NaN counts as absent) gets id
 *             -1 and weight 0 in the missing places and sets
 *             MOE_DEVERR_LOGIT.
 *   topk_ids  int32 [B][k] out; topk_w float32 [B][k] out.  4-byte aligned.
 * Limits: 1 <= E <= MOE_ROUTER_MAX_EXPERTS, 1 <= k <= min(E, MOE_ROUTER_MAX_K),
 * B >= 0 (B = 0 launches nothing).  Weights are FP32 (expf), within a few
 * ulps of the exact values.
 */
int moe_router_topk(const float* logits, int B, int E, int k, int score, float scale, int32_t* topk_ids,
                    float* topk_w, moe_stream_t stream);

/*
 * moe_mx_requant -- BF16 -> MXFP8 -> BF16, the activation round trip of the
 * conventional expert-centric path [WD, section "準確度改進": that path
 * converts the BF16 activations to MXFP8 and back before each grouped GEMM,
 * which warp decode avoids].  It lets a caller build that path's numerics
 * around moe_gate_up / moe_down (x before gate/up, h before down) and
 * measure both against a full-precision reference.  The rule is OCP MX
 * v1.0's: for each block of 32 consecutive values of a row, the shared
 * exponent X = floor(log2(max |v|)) - 8 (clamped to [-127, 127]); each
 * element becomes the E4M3 value nearest v / 2^X (ties to even, magnitudes
 * above 448 saturated to 448), times 2^X, rounded to BF16 (exact unless it
 * falls below BF16's subnormal range).  Blocks of zeros are unchanged.
 *   in, out  BF16 [rows][K], row-major, 16-byte aligned; out may equal in
 *            (in place); other overlap is undefined.  Values must be finite.
 *   rows >= 0 (0 launches nothing); K > 0 and a multiple of 32.
 * Errors: MOE_ERR_ARG (rows < 0, NULL with rows > 0), MOE_ERR_SHAPE (K),
 * MOE_ERR_LIMIT (rows * K overflows), MOE_ERR_ALIGN.  Bit-exact: the result
 * is unique.
 */
int moe_mx_requant(const void* in, void* out, int64_t rows, int K, moe_stream_t stream);

/*
 * moe_device_error -- synchronise `stream`, then read and clear the sticky
 * device error bits (MOE_DEVERR_*) of the current device into *bits.
 * Returns MOE_ERR_DEVICE when any bit was set, MOE_OK otherwise.
 */
int moe_device_error(moe_stream_t stream, int* bits);

#ifdef __cplusplus
}
#endif

#endif /* MOEDEC_H */

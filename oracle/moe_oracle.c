/*
 * moe_oracle.c -- plain, slow, single-threaded CPU oracle for the MoE
 * expert-FFN decode layer and for moe_align_block_size.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, calls or
 * includes this file; only tests/, __graft_entry__.smoke() and bench.py's
 * cpu_baseline / reference legs load it.  It shares no code, header, table
 * or constant with the CUDA path.
 *
 * Everything floating-point is FP64.  Each function names the passage of the
 * source pages it follows:
 *   [WD]  "Warp decode" (cursor.com blog, zh-Hant), sections
 *         "兩個 kernel 的運作方式" (how the two kernels work) and
 *         "準確度改進" (accuracy: BF16 activations, FP32 accumulation).
 *   [AS]  "AMD GPU性能暴涨7倍 ... 高效MoE支持任意专家数量" (aizws.net), sections
 *         on MoE Align & Sort and "编写对AMD设备友好的CUDA实现" (the D-C-P
 *         counting / cumsum / placement algorithm).
 *   [MX]  MXFP8 as the decode page names it: E4M3 elements with one E8M0
 *         scale per 32 consecutive elements along K (OCP MX v1.0 / OFP8);
 *         the conversion of BF16 values to it (shared-exponent rule, nearest
 *         E4M3 with ties to even and saturation) is that standard's.  FP4
 *         weights (the GC-MoE page names FP8/FP4 MoE operators) are read as
 *         the same standard's MXFP4: E2M1 elements with an E8M0 scale per 32.
 *
 * Parity status: every function here is pinned by tests/test_oracle_pins.py
 * (exhaustive code tables, library cross-checks, a dense SwiGLU reduction,
 * invariants, brute force).  The pages print no worked numeric example of a
 * layer output, so the FFN is pinned by those reductions, not by page values.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_ERR_ARG (-1)

/* ---------------------------------------------------------------- [MX] --- */

/* OCP OFP8 E4M3 ("fn" variant: no infinities, S.1111.111 is NaN).
 * Bias 7; exponent field 0 is subnormal: (-1)^s * 2^-6 * m/8. */
double oracle_e4m3_decode(uint8_t q) {
    int s = (q >> 7) & 1;
    int e = (q >> 3) & 15;
    int m = q & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -v : v;
}

/* OCP MX E8M0 shared scale: 2^(s-127); 0xFF is NaN. */
double oracle_e8m0_decode(uint8_t s) {
    if (s == 0xFF) return NAN;
    return ldexp(1.0, (int)s - 127);
}

/* OCP FP4 E2M1 (MX v1.0): sign, 2 exponent bits (bias 1), 1 mantissa bit,
 * no infinities or NaN; exponent field 0 is subnormal: (-1)^s * m/2. */
double oracle_e2m1_decode(uint8_t q) {
    int s = (q >> 3) & 1;
    int e = (q >> 1) & 3;
    int m = q & 1;
    double v = (e == 0) ? (double)m / 2.0 : ldexp(1.0 + (double)m / 2.0, e - 1);
    return s ? -v : v;
}

/* Weight formats: MXFP8 (one E4M3 code per byte, [rows][K]) and MXFP4 (two
 * E2M1 codes per byte, [rows][K/2], the lower K index in the low nibble);
 * both with one E8M0 scale per 32 consecutive elements along K [MX]. */
enum { WFMT_MXFP8 = 0, WFMT_MXFP4 = 1 };

/* dequantised weight element: code(row, col) * 2^(scale-127) [MX] */
static double deq(int fmt, const uint8_t* w, const uint8_t* sc, int64_t K, int64_t row, int64_t col) {
    double c;
    if (fmt == WFMT_MXFP4) {
        uint8_t byte = w[row * (K / 2) + col / 2];
        c = oracle_e2m1_decode((col & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 15));
    } else {
        c = oracle_e4m3_decode(w[row * K + col]);
    }
    return c * oracle_e8m0_decode(sc[row * (K / 32) + col / 32]);
}

/* bytes of one expert's [rows][K] weight codes */
static int64_t wbytes(int fmt, int64_t rows, int64_t K) { return fmt == WFMT_MXFP4 ? rows * K / 2 : rows * K; }

/* ------------------------------------------------------- BF16 helpers --- */

double oracle_bf16_to_double(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* Round a double to the nearest BF16 (ties to even), in one rounding step.
 * bf16 keeps 8 significant bits; its exponent range is that of binary32
 * (normal down to 2^-126, subnormal step 2^-133).  The quantum for |v| in
 * [2^e, 2^(e+1)) is 2^(e-7), floored at 2^-133; rint() is round-half-even
 * under the default rounding mode and v/quantum is exact in binary64. */
uint16_t oracle_bf16_round(double v) {
    if (isnan(v)) return 0x7FC0;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (isinf(a)) return sign | 0x7F80;
    if (a == 0.0) return sign;
    int e;
    frexp(a, &e);           /* a = f * 2^e, f in [0.5, 1) -> floor(log2 a) = e-1 */
    int lead = e - 1;
    if (lead < -126) lead = -126;
    double quantum = ldexp(1.0, lead - 7);
    double r = rint(a / quantum) * quantum;
    /* largest finite bf16 = (2 - 2^-7) * 2^127 */
    if (r > ldexp(2.0 - ldexp(1.0, -7), 127)) return sign | 0x7F80;
    float rf = (float)r;    /* exact: r has <= 8 significant bits */
    uint32_t u;
    memcpy(&u, &rf, 4);
    return sign | (uint16_t)((u >> 16) & 0x7FFF);
}

/* -------------------------------------------- MXFP8 activation round trip --- */

/* The E4M3 value nearest q (finite), ties to the even code, magnitudes
 * beyond the largest finite value 448 saturated to 448 [MX].  E4M3 has four
 * significant bits: for |q| in [2^e, 2^(e+1)) the spacing is 2^(e-3), and
 * below the smallest normal 2^-6 it stays 2^-9 (subnormals).  q / spacing is
 * exact in binary64 and rint() rounds half to even, which on this grid is
 * the code with an even last mantissa bit. */
double oracle_e4m3_round(double q) {
    double a = fabs(q);
    if (a == 0.0) return q;
    if (a >= 448.0) return copysign(448.0, q);
    int e;
    frexp(a, &e);           /* floor(log2 a) = e - 1 */
    int lead = e - 1;
    if (lead < -6) lead = -6;
    double spacing = ldexp(1.0, lead - 3);
    return copysign(rint(a / spacing) * spacing, q);
}

/*
 * BF16 -> MXFP8 -> BF16, the activation round trip of the conventional
 * expert-centric path ("Warp decode", section "準確度改進": it converts the
 * BF16 activations to MXFP8 and back before each grouped GEMM, a rounding
 * floor that warp decode avoids).  The conversion is the OCP MX v1.0 one,
 * the format the page names for its weights: for each block of 32
 * consecutive values along K, the shared exponent is
 *     X = floor(log2(max |v|)) - 8        (8: the exponent of E4M3's largest
 *                                          power of two, 256),
 * clamped to the E8M0 range [-127, 127]; each element becomes the E4M3 value
 * nearest v / 2^X (ties to even, saturating at 448), and the result is that
 * value times 2^X, returned as BF16 (exact unless it falls below BF16's
 * subnormal range, then rounded to nearest even).  A block of zeros stays as
 * it is.  in and out hold rows * K BF16 bit patterns, rows major; inputs are
 * finite.  Returns ORACLE_ERR_ARG unless K is a positive multiple of 32.
 */
int oracle_mx_requant(const uint16_t* in, int64_t rows, int64_t K, uint16_t* out) {
    if (rows < 0 || K <= 0 || K % 32) return ORACLE_ERR_ARG;
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t b0 = 0; b0 < K; b0 += 32) {
            const uint16_t* v = in + r * K + b0;
            uint16_t* o = out + r * K + b0;
            double amax = 0.0;
            for (int i = 0; i < 32; ++i) {
                double a = fabs(oracle_bf16_to_double(v[i]));
                if (a > amax) amax = a;
            }
            if (amax == 0.0) {
                for (int i = 0; i < 32; ++i) o[i] = v[i];
                continue;
            }
            int e;
            frexp(amax, &e);
            int X = (e - 1) - 8;
            if (X < -127) X = -127;
            if (X > 127) X = 127;
            for (int i = 0; i < 32; ++i) {
                double q = ldexp(oracle_bf16_to_double(v[i]), -X);
                o[i] = oracle_bf16_round(ldexp(oracle_e4m3_round(q), X));
            }
        }
    }
    return ORACLE_OK;
}

/* ---------------------------------------------------------------- [WD] --- */

static double silu(double g) { return g / (1.0 + exp(-g)); }

/* One expert's gate/up pass for one token.
 *  [WD] gate/up kernel: the routed expert's gate row and up row are both
 *  dotted with the same activation vector, then SiLU(gate) * up gives one
 *  intermediate value per (token, expert, neuron); the intermediate is
 *  BF16 (the pages keep activations in BF16 throughout).
 *  hf_out (optional) receives the unrounded FP64 value. */
static void gate_up_one(int fmt, const uint16_t* xb, int64_t d, const uint8_t* wg, const uint8_t* sg,
                        const uint8_t* wu, const uint8_t* su, int64_t I, int64_t e,
                        uint16_t* h_out, double* hf_out, double* g_out, double* u_out) {
    const uint8_t* wge = wg + e * wbytes(fmt, I, d);
    const uint8_t* sge = sg + e * I * (d / 32);
    const uint8_t* wue = wu + e * wbytes(fmt, I, d);
    const uint8_t* sue = su + e * I * (d / 32);
    for (int64_t n = 0; n < I; ++n) {
        double g = 0.0, u = 0.0;
        for (int64_t c = 0; c < d; ++c) {
            double xv = oracle_bf16_to_double(xb[c]);
            g += xv * deq(fmt, wge, sge, d, n, c);
            u += xv * deq(fmt, wue, sue, d, n, c);
        }
        double hf = silu(g) * u;
        if (g_out) g_out[n] = g;
        if (u_out) u_out[n] = u;
        if (hf_out) hf_out[n] = hf;
        if (h_out) h_out[n] = oracle_bf16_round(hf);
    }
}

/* One expert's down projection of one intermediate vector, FP64. */
static void down_one(int fmt, const double* hv, int64_t I, const uint8_t* wd, const uint8_t* sd, int64_t d,
                     int64_t e, double scale, double* y) {
    const uint8_t* wde = wd + e * wbytes(fmt, d, I);
    const uint8_t* sde = sd + e * d * (I / 32);
    for (int64_t o = 0; o < d; ++o) {
        double acc = 0.0;
        for (int64_t i = 0; i < I; ++i) acc += hv[i] * deq(fmt, wde, sde, I, o, i);
        y[o] += scale * acc;
    }
}

/*
 * The whole decode layer [WD]:
 *   for each token b and routed slot j (e = topk_ids[b,j]):
 *       h[b,j,:] = bf16( SiLU(Wg[e] x_b) * (Wu[e] x_b) )
 *   y64[b,:] = sum_j topk_w[b,j] * Wd[e_j] h[b,j,:]
 *              + (shared expert present) 1.0 * Wsd h[b,k,:]
 * with h[b,k,:] the shared expert's intermediate.  y64 is left unrounded.
 * truth64 (optional) is the same computation with h kept in FP64.
 * h_bf16 (optional) receives the BF16 intermediates, layout [B][k+S][I];
 * h64 (optional) the same intermediates before rounding; g64 and u64
 * (optional) the gate and up dot products they come from.
 * Shared-expert arrays are NULL when there is no shared expert; the shared
 * expert has the same I and d as the routed ones.
 * Returns ORACLE_ERR_ARG on a bad shape or an expert id outside [0, E).
 */
static int layer_impl(const uint16_t* x, int B, int d, const int32_t* topk_ids, const float* topk_w,
                      int k, const uint8_t* wg, const uint8_t* sg, const uint8_t* wu,
                      const uint8_t* su, const uint8_t* wd, const uint8_t* sd, int E, int I,
                      const uint8_t* shg, const uint8_t* shsg, const uint8_t* shu,
                      const uint8_t* shsu, const uint8_t* shd, const uint8_t* shsd,
                      uint16_t* h_bf16, double* h64, double* g64, double* u64, double* y64,
                      double* truth64, int mx_act, int fmt) {
    if (B < 0 || d <= 0 || I <= 0 || k < 0 || E <= 0 || d % 32 || I % 32) return ORACLE_ERR_ARG;
    int S = (shg != NULL) ? 1 : 0;
    int slots = k + S;
    uint16_t* hb = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)I);
    uint16_t* hq = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)I);
    uint16_t* xq = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)d);
    double* hf = (double*)malloc(sizeof(double) * (size_t)I);
    double* hr = (double*)malloc(sizeof(double) * (size_t)I);
    if (!hb || !hq || !xq || !hf || !hr) {
        free(hb); free(hq); free(xq); free(hf); free(hr);
        return ORACLE_ERR_ARG;
    }
    int rc = ORACLE_OK;
    for (int b = 0; b < B && rc == ORACLE_OK; ++b) {
        const uint16_t* xb = x + (int64_t)b * d;
        if (mx_act) {  /* the conventional path's x before the gate/up GEMM */
            oracle_mx_requant(xb, 1, d, xq);
            xb = xq;
        }
        double* yb = y64 + (int64_t)b * d;
        double* tb = truth64 ? truth64 + (int64_t)b * d : NULL;
        for (int o = 0; o < d; ++o) {
            yb[o] = 0.0;
            if (tb) tb[o] = 0.0;
        }
        for (int j = 0; j < slots; ++j) {
            int shared = (j == k);
            int64_t e = shared ? 0 : topk_ids[(int64_t)b * k + j];
            if (!shared && (e < 0 || e >= E)) { rc = ORACLE_ERR_ARG; break; }
            double wt = shared ? 1.0 : (double)topk_w[(int64_t)b * k + j];
            const int64_t row0 = ((int64_t)b * slots + j) * I;
            gate_up_one(fmt, xb, d, shared ? shg : wg, shared ? shsg : sg, shared ? shu : wu,
                        shared ? shsu : su, I, e, hb, hf, g64 ? g64 + row0 : NULL,
                        u64 ? u64 + row0 : NULL);
            if (mx_act) {  /* ... and its h before the down GEMM */
                oracle_mx_requant(hb, 1, I, hq);
                for (int i = 0; i < I; ++i) hr[i] = oracle_bf16_to_double(hq[i]);
            } else {
                for (int i = 0; i < I; ++i) hr[i] = oracle_bf16_to_double(hb[i]);
            }
            if (h_bf16) memcpy(h_bf16 + ((int64_t)b * slots + j) * I, hb, sizeof(uint16_t) * (size_t)I);
            if (h64) memcpy(h64 + ((int64_t)b * slots + j) * I, hf, sizeof(double) * (size_t)I);
            down_one(fmt, hr, I, shared ? shd : wd, shared ? shsd : sd, d, e, wt, yb);
            if (tb) down_one(fmt, hf, I, shared ? shd : wd, shared ? shsd : sd, d, e, wt, tb);
        }
    }
    free(hb); free(hq); free(xq); free(hf); free(hr);
    return rc;
}

int oracle_moe_layer(const uint16_t* x, int B, int d, const int32_t* topk_ids, const float* topk_w,
                     int k, const uint8_t* wg, const uint8_t* sg, const uint8_t* wu,
                     const uint8_t* su, const uint8_t* wd, const uint8_t* sd, int E, int I,
                     const uint8_t* shg, const uint8_t* shsg, const uint8_t* shu,
                     const uint8_t* shsu, const uint8_t* shd, const uint8_t* shsd,
                     uint16_t* h_bf16, double* h64, double* g64, double* u64, double* y64,
                     double* truth64) {
    return layer_impl(x, B, d, topk_ids, topk_w, k, wg, sg, wu, su, wd, sd, E, I, shg, shsg, shu, shsu,
                      shd, shsd, h_bf16, h64, g64, u64, y64, truth64, 0, WFMT_MXFP8);
}

/*
 * The same layer with MXFP4 weights (E2M1 codes, two per byte, the lower K
 * index in the low nibble; one E8M0 scale per 32 along K): wg, wu are
 * [E][I][d/2] bytes, wd [E][d][I/2], the scales as for MXFP8.  Activations,
 * accumulation and every output are as in oracle_moe_layer.
 */
int oracle_moe_layer_mx4(const uint16_t* x, int B, int d, const int32_t* topk_ids, const float* topk_w,
                         int k, const uint8_t* wg, const uint8_t* sg, const uint8_t* wu,
                         const uint8_t* su, const uint8_t* wd, const uint8_t* sd, int E, int I,
                         const uint8_t* shg, const uint8_t* shsg, const uint8_t* shu,
                         const uint8_t* shsu, const uint8_t* shd, const uint8_t* shsd,
                         uint16_t* h_bf16, double* h64, double* g64, double* u64, double* y64,
                         double* truth64) {
    return layer_impl(x, B, d, topk_ids, topk_w, k, wg, sg, wu, su, wd, sd, E, I, shg, shsg, shu, shsu,
                      shd, shsd, h_bf16, h64, g64, u64, y64, truth64, 0, WFMT_MXFP4);
}

/*
 * The conventional expert-centric path's numerics ("Warp decode", section
 * "準確度改進"): the same layer with x converted to MXFP8 and back before
 * the gate/up GEMM and h (already BF16) converted the same way before the
 * down GEMM (oracle_mx_requant, blocks of 32 along d and along I).  h_bf16,
 * h64, g64 and u64 are those of the gate/up pass on the converted x (h_bf16
 * before its own conversion); y64 is unrounded.  The full-precision truth
 * to compare both paths with is oracle_moe_layer's truth64 on the original
 * x (h kept in FP64, nothing converted).
 */
int oracle_moe_layer_mx_act(const uint16_t* x, int B, int d, const int32_t* topk_ids,
                            const float* topk_w, int k, const uint8_t* wg, const uint8_t* sg,
                            const uint8_t* wu, const uint8_t* su, const uint8_t* wd,
                            const uint8_t* sd, int E, int I, const uint8_t* shg,
                            const uint8_t* shsg, const uint8_t* shu, const uint8_t* shsu,
                            const uint8_t* shd, const uint8_t* shsd, uint16_t* h_bf16, double* h64,
                            double* g64, double* u64, double* y64) {
    return layer_impl(x, B, d, topk_ids, topk_w, k, wg, sg, wu, su, wd, sd, E, I, shg, shsg, shu, shsu,
                      shd, shsd, h_bf16, h64, g64, u64, y64, NULL, 1, WFMT_MXFP8);
}

/* ---------------------------------------------------------------- [AS] --- */

/* Sizes of the align outputs: the padded buffer is the worst case in which
 * every expert's segment needs block_size-1 pad entries. */
int oracle_align_sizes(int T, int k, int E, int block_size, int64_t* n_sorted, int64_t* n_blocks) {
    if (T < 0 || k < 0 || E <= 0 || block_size <= 0) return ORACLE_ERR_ARG;
    int64_t n = (int64_t)T * k + (int64_t)E * (block_size - 1);
    *n_sorted = n;
    *n_blocks = (n + block_size - 1) / block_size;
    return ORACLE_OK;
}

/*
 * moe_align_block_size [AS]: sort the flat (token, slot) indices f = t*k + j
 * by expert id, pad each expert's run up to a multiple of block_size with the
 * sentinel T*k, and record which expert owns each block_size-sized block.
 * Step by step, in the page's D-C-P order, done serially:
 *   count   cnt[e] = #{f : ids[f] == e}
 *   cumsum  pad[e] = ceil(cnt[e]/bs)*bs ; start = exclusive prefix of pad
 *   place   walk f in increasing order: sorted[start[e] + pos[e]++] = f
 * Ties are therefore broken by flat index (a stable counting sort).
 * Entries past num_tokens_post_pad hold the sentinel; expert_ids past
 * num_tokens_post_pad/bs hold -1.
 */
int oracle_align(const int32_t* ids, int T, int k, int E, int block_size, int32_t* sorted,
                 int64_t n_sorted, int32_t* expert_ids, int64_t n_blocks, int32_t* ntpp) {
    int64_t need_sorted, need_blocks;
    if (oracle_align_sizes(T, k, E, block_size, &need_sorted, &need_blocks) != ORACLE_OK)
        return ORACLE_ERR_ARG;
    if (n_sorted < need_sorted || n_blocks < need_blocks) return ORACLE_ERR_ARG;
    int64_t N = (int64_t)T * k;
    int64_t* cnt = (int64_t*)calloc((size_t)E, sizeof(int64_t));
    int64_t* start = (int64_t*)calloc((size_t)E + 1, sizeof(int64_t));
    int64_t* pos = (int64_t*)calloc((size_t)E, sizeof(int64_t));
    if (!cnt || !start || !pos) {
        free(cnt); free(start); free(pos);
        return ORACLE_ERR_ARG;
    }
    int rc = ORACLE_OK;
    for (int64_t f = 0; f < N; ++f) {
        int32_t e = ids[f];
        if (e < 0 || e >= E) { rc = ORACLE_ERR_ARG; break; }
        cnt[e] += 1;
    }
    if (rc == ORACLE_OK) {
        for (int e = 0; e < E; ++e) {
            int64_t padded = (cnt[e] + block_size - 1) / block_size * block_size;
            start[e + 1] = start[e] + padded;
        }
        for (int64_t i = 0; i < n_sorted; ++i) sorted[i] = (int32_t)N;
        for (int64_t f = 0; f < N; ++f) {
            int32_t e = ids[f];
            sorted[start[e] + pos[e]] = (int32_t)f;
            pos[e] += 1;
        }
        for (int64_t blk = 0; blk < n_blocks; ++blk) expert_ids[blk] = -1;
        for (int e = 0; e < E; ++e)
            for (int64_t p = start[e]; p < start[e + 1]; p += block_size)
                expert_ids[p / block_size] = e;
        *ntpp = (int32_t)start[E];
    }
    free(cnt); free(start); free(pos);
    return rc;
}

/* ---------------------------------------------------------- router [AS] --- */

/* The routing step in front of the decode layer ([AS], section
 * "MoE Align & Sort CUDA算法在其他开源平台的实现": FasterTransformer's fused
 * topk_gating_softmax), per token b, by definition:
 *   score 0 (softmax): p = softmax over all E logits; the k largest p (ties:
 *     lower expert index first), in descending order; w_j = scale * p_j /
 *     (sum of the k chosen p);
 *   score 1 (sigmoid): s = 1 / (1 + exp(-logit)) for all E; the k largest s,
 *     same order; w_j = scale * s_j / (sum of the k chosen s).
 * Selection is k passes of "largest remaining, lowest index on ties", taken
 * on the FP32 logits themselves: both score maps are strictly increasing, so
 * this is the exact score order (FP64 sigmoid scores can tie where the exact
 * ones do not, e.g. all logits above ~37 round to 1.0).  Weights are FP64. */
int oracle_router_topk(const float* logits, int B, int E, int k, int score, double scale, int32_t* ids,
                       double* w) {
    if (B < 0 || E < 1 || k < 1 || k > E || (score != 0 && score != 1)) return ORACLE_ERR_ARG;
    double* sc = (double*)malloc(sizeof(double) * (size_t)E);
    char* used = (char*)malloc((size_t)E);
    if (!sc || !used) {
        free(sc);
        free(used);
        return ORACLE_ERR_ARG;
    }
    for (int b = 0; b < B; ++b) {
        const float* l = logits + (size_t)b * E;
        if (score == 0) {
            double m = l[0];
            for (int e = 1; e < E; ++e)
                if (l[e] > m) m = l[e];
            double z = 0.0;
            for (int e = 0; e < E; ++e) {
                sc[e] = exp((double)l[e] - m);
                z += sc[e];
            }
            for (int e = 0; e < E; ++e) sc[e] /= z;
        } else {
            for (int e = 0; e < E; ++e) sc[e] = 1.0 / (1.0 + exp(-(double)l[e]));
        }
        memset(used, 0, (size_t)E);
        double tot = 0.0;
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e)
                if (!used[e] && (best < 0 || l[e] > l[best])) best = e;
            used[best] = 1;
            ids[(size_t)b * k + j] = best;
            w[(size_t)b * k + j] = sc[best];
            tot += sc[best];
        }
        for (int j = 0; j < k; ++j) w[(size_t)b * k + j] = scale * w[(size_t)b * k + j] / tot;
    }
    free(sc);
    free(used);
    return ORACLE_OK;
}

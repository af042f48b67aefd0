/*
 * Oracle for MoE token dispatch / combine -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, single-threaded C99 restatement of what the hot path
 * computes. Only the tests, the smoke check and the bench's CPU-baseline leg
 * may load this library; the product path never does. It shares no code,
 * header, table or helper with the CUDA library.
 *
 * Build: gcc -O2 -std=c99 -ffp-contract=off -fno-fast-math -shared -fPIC
 * (no SIMD intrinsics, no threads; float arithmetic is IEEE binary32 with
 * round-to-nearest-even, and fmaf is the correctly rounded fused multiply-add).
 *
 * Sources (page title, then section):
 *  - "nccl_ep.cc" (NCCL EP host code mirrored in TheRock/rccl contrib),
 *    struct ncclEpHandle: is_token_in_rank is the outbound [token, rank] mask;
 *    num_tokens_for_experts counts a token once however many local experts it
 *    reaches; sparse_to_dense_map uses -1 for "not routed".
 *    ncclEpCreateHandle: topk_idx is int64 [T, K]; num_experts % num_ranks == 0;
 *    experts per rank = num_experts / num_ranks.
 *    ncclEpDispatch (low-latency branch): fp8 scales are fp32, one per 128
 *    hidden channels, laid out [rows, hidden/128].
 *    ncclEpCombine (low-latency branch): combine is weighted by fp32
 *    topk_weights [T, K] and writes out [T, hidden] in the input's dtype.
 *  - DeepEP API docs: "dispatch()" (do_expand: one received row per
 *    (token, expert) pair) and "Prefix Sum Interpretation for Expert Token
 *    Counts" (per-expert row ranges come from a prefix sum of counts).
 *  - NeMo fused_a2a (HybridEPDispatch / HybridEPCombine): -1 marks an unused
 *    top-k slot; combine returns rows in the original token order.
 *
 * Readings where the pages leave a step open (each also listed in the design
 * notes): expert e belongs to rank e / (E/R); offsets are the exclusive scan
 * [E+1]; rows inside one expert keep (token, k) order; an id outside [-1, E)
 * is an error and its slot is treated as dropped; fp8 uses
 * scale = amax / 448 and q = e4m3_rne_satfinite(x / scale), with an all-zero
 * block giving scale 0 and zero bytes; combine accumulates fp32 fmaf in
 * ascending k from +0 and rounds once to bf16 (nearest-even).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_ERR_ARG 1
#define ORC_ERR_EXPERT 2

/* ---------------------------------------------------------------- formats */

/* bf16 -> fp32: a bf16 value is the top half of the fp32 with the same bits. */
float orc_bf16_to_f32(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* fp32 -> bf16, round to nearest, ties to even. bf16 keeps fp32's sign and
 * 8-bit exponent and the top 7 mantissa bits, so rounding acts on the low 16
 * bits: above half goes up, below half goes down, exactly half goes to the
 * neighbour whose last kept bit is 0. A carry out of the mantissa correctly
 * bumps the exponent (up to infinity). NaN stays a quiet NaN. */
uint16_t orc_f32_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if (isnan(f)) return (uint16_t)(((u >> 16) & 0x8000u) | 0x7FC0u);
    uint32_t hi = u >> 16, lo = u & 0xFFFFu;
    if (lo > 0x8000u || (lo == 0x8000u && (hi & 1u))) hi += 1u;
    return (uint16_t)hi;
}

/* OCP FP8 E4M3 ("e4m3fn"): 1 sign, 4 exponent (bias 7), 3 mantissa bits; no
 * infinities; S.1111.111 is NaN, so the largest finite is S.1111.110 = 448.
 * Normal values (exponent field 1..15): 2^(e-7) * (1 + m/8).
 * Subnormals (exponent field 0): m * 2^-9.
 * Encoding rounds to nearest, ties to even, and saturates anything beyond 448
 * to +-448 ("satfinite"). Zero keeps its sign. */
uint8_t orc_f32_to_e4m3(float f) {
    if (isnan(f)) return 0x7F;
    uint8_t sign = signbit(f) ? 0x80 : 0x00;
    double a = fabs((double)f);
    if (a >= 448.0) return (uint8_t)(sign | 0x7E);
    if (a < ldexp(1.0, -6)) {
        /* subnormal range: count steps of 2^-9; rint rounds half to even.
         * 8 steps is 2^-6, the smallest normal, whose code is 0x08. */
        double m = rint(a * 512.0);
        return (uint8_t)(sign | (uint8_t)m);
    }
    int ex;
    (void)frexp(a, &ex);            /* a = fr * 2^ex, fr in [0.5, 1) */
    int E = ex - 1;                 /* a in [2^E, 2^(E+1)) */
    double m = rint(ldexp(a, 3 - E)); /* 8..16 mantissa steps of 2^(E-3) */
    if (m >= 16.0) { m = 8.0; E += 1; }
    int field = E + 7;
    int code = (field << 3) | ((int)m - 8);
    if (code > 0x7E) code = 0x7E;   /* rounding up past 448 saturates */
    return (uint8_t)(sign | code);
}

/* E4M3 byte -> value (used by tests for dequantisation bounds). */
float orc_e4m3_to_f32(uint8_t q) {
    int s = q >> 7, field = (q >> 3) & 0xF, m = q & 7;
    double v;
    if (field == 0xF && m == 7) return NAN;
    if (field == 0) v = ldexp((double)m, -9);
    else v = ldexp(1.0 + m / 8.0, field - 7);
    return (float)(s ? -v : v);
}

/* OCP FP8 E5M2: 1 sign, 5 exponent (bias 15), 2 mantissa bits, laid out
 * like an IEEE format: exponent field 31 holds infinity (mantissa 0) and NaN,
 * so the largest finite is S.11110.11 = 1.75 * 2^15 = 57344.
 * Normal values (exponent field 1..30): 2^(e-15) * (1 + m/4).
 * Subnormals (exponent field 0): m * 2^-16.
 * Encoding rounds to nearest, ties to even, and saturates anything beyond
 * 57344 to +-57344 (satfinite, as for e4m3). Zero keeps its sign.
 * nccl_ep.cc (ncclTypeSize, ncclEpDispatch) accepts it beside e4m3 as a
 * one-byte fp8 token type. */
uint8_t orc_f32_to_e5m2(float f) {
    if (isnan(f)) return 0x7F;
    uint8_t sign = signbit(f) ? 0x80 : 0x00;
    double a = fabs((double)f);
    if (a >= 57344.0) return (uint8_t)(sign | 0x7B);
    if (a < ldexp(1.0, -14)) {
        /* subnormal range: steps of 2^-16, half to even; 4 steps is 2^-14,
         * the smallest normal, whose code is 0x04 */
        double m = rint(a * 65536.0);
        return (uint8_t)(sign | (uint8_t)m);
    }
    int ex;
    (void)frexp(a, &ex);
    int E = ex - 1;                    /* a in [2^E, 2^(E+1)) */
    double m = rint(ldexp(a, 2 - E));  /* 4..8 mantissa steps of 2^(E-2) */
    if (m >= 8.0) { m = 4.0; E += 1; }
    int code = ((E + 15) << 2) | ((int)m - 4);
    if (code > 0x7B) code = 0x7B;
    return (uint8_t)(sign | code);
}

/* E5M2 byte -> value. */
float orc_e5m2_to_f32(uint8_t q) {
    int s = q >> 7, field = (q >> 2) & 0x1F, m = q & 3;
    double v;
    if (field == 0x1F) {
        if (m != 0) return NAN;
        v = INFINITY;
    } else if (field == 0) {
        v = ldexp((double)m, -16);
    } else {
        v = ldexp(1.0 + m / 4.0, field - 15);
    }
    return (float)(s ? -v : v);
}

/* ---------------------------------------------------------------- layout */

/* Routing layout from topk_idx [T, K] (int64, -1 = unused slot).
 *   num_tokens_per_expert[e] = number of slots naming e
 *   is_token_in_rank[t, r]   = 1 if any slot of t names an expert of rank r
 *   num_tokens_per_rank[r]   = number of tokens t with is_token_in_rank[t, r]
 *   expert_offsets[E + 1]    = exclusive prefix sum of the expert counts
 *   row_of_slot[t, k]        = receive row of slot (t, k), -1 if unused;
 *                              rows of expert e are expert_offsets[e] .. in
 *                              (t, k) order (a counting sort keyed by expert).
 * Returns ORC_ERR_EXPERT if any id lies outside [-1, E) (that slot is then
 * treated as unused), ORC_ERR_ARG for bad sizes. */
int orc_layout(const int64_t* topk_idx, int64_t T, int K, int E, int R,
               int32_t* num_tokens_per_expert, int32_t* num_tokens_per_rank,
               uint8_t* is_token_in_rank, int32_t* expert_offsets,
               int32_t* row_of_slot) {
    if (T < 0 || K <= 0 || E <= 0 || R <= 0 || E % R != 0) return ORC_ERR_ARG;
    int L = E / R;
    int status = ORC_OK;
    int64_t* cnt64 = (int64_t*)calloc((size_t)E, sizeof(int64_t));
    int64_t* next = (int64_t*)calloc((size_t)E, sizeof(int64_t));
    if (!cnt64 || !next) { free(cnt64); free(next); return ORC_ERR_ARG; }
    for (int r = 0; r < R; ++r) num_tokens_per_rank[r] = 0;

    for (int64_t t = 0; t < T; ++t) {
        uint8_t* mask = is_token_in_rank + t * R;
        for (int r = 0; r < R; ++r) mask[r] = 0;
        for (int k = 0; k < K; ++k) {
            int64_t e = topk_idx[t * K + k];
            if (e == -1) continue;
            if (e < -1 || e >= E) { status = ORC_ERR_EXPERT; continue; }
            cnt64[e] += 1;
            mask[e / L] = 1;
        }
        for (int r = 0; r < R; ++r) num_tokens_per_rank[r] += mask[r];
    }

    int64_t run = 0;
    for (int e = 0; e < E; ++e) {
        expert_offsets[e] = (int32_t)run;
        num_tokens_per_expert[e] = (int32_t)cnt64[e];
        next[e] = run;
        run += cnt64[e];
    }
    if (run > INT32_MAX) { free(cnt64); free(next); return ORC_ERR_ARG; }
    expert_offsets[E] = (int32_t)run;

    for (int64_t t = 0; t < T; ++t) {
        for (int k = 0; k < K; ++k) {
            int64_t e = topk_idx[t * K + k];
            if (e < 0 || e >= E) { row_of_slot[t * K + k] = -1; continue; }
            row_of_slot[t * K + k] = (int32_t)next[e]++;
        }
    }
    free(cnt64);
    free(next);
    return status;
}

/* ---------------------------------------------------------------- dispatch */

/* bf16 permute: recv_x[row_of_slot[t, k]] = x[t] for every used slot.
 * Optional outputs (NULL = skip): recv_src_token[row] = t and
 * recv_weights[row] = topk_weights[t, k]. */
void orc_dispatch_bf16(const uint16_t* x, int64_t T, int H, const int32_t* row_of_slot,
                       int K, const float* topk_weights, uint16_t* recv_x,
                       int32_t* recv_src_token, float* recv_weights) {
    for (int64_t t = 0; t < T; ++t) {
        for (int k = 0; k < K; ++k) {
            int32_t row = row_of_slot[t * K + k];
            if (row < 0) continue;
            memcpy(recv_x + (int64_t)row * H, x + t * H, (size_t)H * sizeof(uint16_t));
            if (recv_src_token) recv_src_token[row] = (int32_t)t;
            if (recv_weights && topk_weights) recv_weights[row] = topk_weights[t * K + k];
        }
    }
}

/* Quantise one token row to e4m3 with one fp32 scale per 128 channels:
 *   amax  = max |x| over the block (exact, in fp32)
 *   scale = amax / 448            (fp32 division, nearest-even)
 *   q     = e4m3(x / scale)       (fp32 division, then nearest-even, satfinite)
 * An all-zero block gives scale 0 and all-zero bytes. */
void orc_quant_row_e4m3(const uint16_t* xrow, int H, uint8_t* qrow, float* srow) {
    for (int b = 0; b < H / 128; ++b) {
        float amax = 0.0f;
        for (int i = 0; i < 128; ++i) {
            float v = fabsf(orc_bf16_to_f32(xrow[b * 128 + i]));
            if (v > amax) amax = v;
        }
        if (amax == 0.0f) {
            srow[b] = 0.0f;
            for (int i = 0; i < 128; ++i) qrow[b * 128 + i] = 0x00;
            continue;
        }
        float scale = amax / 448.0f;
        srow[b] = scale;
        for (int i = 0; i < 128; ++i) {
            float v = orc_bf16_to_f32(xrow[b * 128 + i]) / scale;
            qrow[b * 128 + i] = orc_f32_to_e4m3(v);
        }
    }
}

/* fp8 permute: each used slot's row receives its token's e4m3 bytes [H] and
 * scales [H/128]. */
void orc_dispatch_e4m3(const uint16_t* x, int64_t T, int H, const int32_t* row_of_slot,
                       int K, const float* topk_weights, uint8_t* recv_q, float* recv_scales,
                       int32_t* recv_src_token, float* recv_weights) {
    int nb = H / 128;
    uint8_t* q = (uint8_t*)malloc((size_t)(H > 0 ? H : 1));
    float* s = (float*)malloc((size_t)(nb > 0 ? nb : 1) * sizeof(float));
    if (!q || !s) { free(q); free(s); return; }
    for (int64_t t = 0; t < T; ++t) {
        int any = 0;
        for (int k = 0; k < K; ++k) any |= row_of_slot[t * K + k] >= 0;
        if (!any) continue;
        orc_quant_row_e4m3(x + t * H, H, q, s);
        for (int k = 0; k < K; ++k) {
            int32_t row = row_of_slot[t * K + k];
            if (row < 0) continue;
            memcpy(recv_q + (int64_t)row * H, q, (size_t)H);
            memcpy(recv_scales + (int64_t)row * nb, s, (size_t)nb * sizeof(float));
            if (recv_src_token) recv_src_token[row] = (int32_t)t;
            if (recv_weights && topk_weights) recv_weights[row] = topk_weights[t * K + k];
        }
    }
    free(q);
    free(s);
}

/* ---------------------------------------------------------------- combine */

/* One output row: out[h] = bf16( sum over k ascending with row >= 0 of
 * w[k] * y[row_k, h] ), accumulated in fp32 with fmaf from +0.
 * w == NULL means every weight is 1. */
void orc_combine_row(const uint16_t* y, int H, const int32_t* rows, const float* w, int K,
                     uint16_t* out_row) {
    for (int h = 0; h < H; ++h) {
        float acc = 0.0f;
        for (int k = 0; k < K; ++k) {
            int32_t row = rows[k];
            if (row < 0) continue;
            float wk = w ? w[k] : 1.0f;
            acc = fmaf(wk, orc_bf16_to_f32(y[(int64_t)row * H + h]), acc);
        }
        out_row[h] = orc_f32_to_bf16(acc);
    }
}

void orc_combine(const uint16_t* y, int H, const int32_t* row_of_slot, int64_t T, int K,
                 const float* topk_weights, uint16_t* out) {
    for (int64_t t = 0; t < T; ++t)
        orc_combine_row(y, H, row_of_slot + t * K, topk_weights ? topk_weights + t * K : 0, K,
                        out + t * H);
}

/* ---------------------------------------------------------------- arrays */

/* Element-wise encoders over arrays, for exhaustive format sweeps. */
void orc_f32_to_bf16_array(const float* in, int64_t n, uint16_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_f32_to_bf16(in[i]);
}

void orc_f32_to_e4m3_array(const float* in, int64_t n, uint8_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_f32_to_e4m3(in[i]);
}

/* Sweep fp32 bit patterns [lo, hi) through the e4m3 encoder (no input array). */
void orc_e4m3_sweep(uint32_t lo, uint32_t hi, uint8_t* out) {
    for (uint64_t u = lo; u < hi; ++u) {
        uint32_t b = (uint32_t)u;
        float f;
        memcpy(&f, &b, sizeof f);
        out[u - lo] = orc_f32_to_e4m3(f);
    }
}

/* ---------------------------------------------------------------- alignment */

/* Routing layout with per-expert row alignment A >= 1 (DeepEP API docs,
 * "dispatch()" expert_alignment and "Prefix Sum Interpretation for Expert
 * Token Counts": in expand mode expert i's rows start at the previous
 * expert's end rounded up to a multiple of the alignment).
 *   expert_offsets[e] = sum over e' < e of roundup(count[e'], A)
 *   expert_offsets[E] = padded row total
 * Expert e's real rows are expert_offsets[e] .. + count[e] - 1 in (t, k)
 * order; the rest of its range up to expert_offsets[e+1] are pad rows.
 * Counts, masks and per-rank tokens are those of orc_layout. */
int orc_layout_aligned(const int64_t* topk_idx, int64_t T, int K, int E, int R, int A,
                       int32_t* num_tokens_per_expert, int32_t* num_tokens_per_rank,
                       uint8_t* is_token_in_rank, int32_t* expert_offsets,
                       int32_t* row_of_slot) {
    if (A < 1) return ORC_ERR_ARG;
    int32_t* plain_offsets = (int32_t*)malloc(sizeof(int32_t) * (size_t)(E + 1));
    if (!plain_offsets) return ORC_ERR_ARG;
    int status = orc_layout(topk_idx, T, K, E, R, num_tokens_per_expert, num_tokens_per_rank,
                            is_token_in_rank, plain_offsets, row_of_slot);
    if (status == ORC_ERR_ARG) { free(plain_offsets); return status; }
    int64_t run = 0;
    for (int e = 0; e < E; ++e) {
        expert_offsets[e] = (int32_t)run;
        int64_t c = num_tokens_per_expert[e];
        run += (c + A - 1) / A * A;
    }
    if (run > INT32_MAX) { free(plain_offsets); return ORC_ERR_ARG; }
    expert_offsets[E] = (int32_t)run;
    /* move every real row from its packed position to the aligned range */
    for (int64_t s = 0; s < T * (int64_t)K; ++s) {
        int64_t e = topk_idx[s];
        if (row_of_slot[s] < 0) continue;
        row_of_slot[s] = row_of_slot[s] - plain_offsets[e] + expert_offsets[e];
    }
    free(plain_offsets);
    return status;
}

/* Pad rows of an aligned layout: every receive row of expert e from
 * expert_offsets[e] + count[e] up to expert_offsets[e+1] is zero (row_bytes
 * zero bytes), has scale 0 in each of its nb scale slots (if scales), source
 * token -1 (if src) and weight 0 (if weights). */
void orc_fill_pad_rows(const int32_t* num_tokens_per_expert, const int32_t* expert_offsets, int E,
                       int64_t row_bytes, uint8_t* recv, float* scales, int nb, int32_t* src,
                       float* weights) {
    for (int e = 0; e < E; ++e) {
        for (int64_t r = (int64_t)expert_offsets[e] + num_tokens_per_expert[e]; r < expert_offsets[e + 1]; ++r) {
            memset(recv + r * row_bytes, 0, (size_t)row_bytes);
            if (scales) for (int b = 0; b < nb; ++b) scales[r * nb + b] = 0.0f;
            if (src) src[r] = -1;
            if (weights) weights[r] = 0.0f;
        }
    }
}

/* ---------------------------------------------------------------- backward */

/* Backward of the weighted combine out[t] = sum_k w[t,k] * y[row(t,k)]
 * (DeepEP API docs, README training snippet: the backward of combine is a
 * dispatch; nccl_ep.cc, ncclEpCombine: the high-throughput backward mode also
 * reduces the probabilities):
 *   grad_y[row(t,k), h] = bf16( w[t,k] * grad_out[t, h] )   (fp32 product, one round)
 *   grad_w[t, k]        = sum_h grad_out[t, h] * y[row(t,k), h]   (in double here)
 * Dropped slots get grad_w = 0 and write no row. w == NULL means all ones. */
void orc_combine_backward(const uint16_t* grad_out, const uint16_t* y, int H, const int32_t* row_of_slot,
                          int64_t T, int K, const float* w, uint16_t* grad_y, double* grad_w) {
    for (int64_t t = 0; t < T; ++t) {
        for (int k = 0; k < K; ++k) {
            int32_t row = row_of_slot[t * K + k];
            double dot = 0.0;
            if (row >= 0) {
                float wk = w ? w[t * K + k] : 1.0f;
                for (int h = 0; h < H; ++h) {
                    float g = orc_bf16_to_f32(grad_out[t * H + h]);
                    if (grad_y) grad_y[(int64_t)row * H + h] = orc_f32_to_bf16(wk * g);
                    dot += (double)g * (double)orc_bf16_to_f32(y[(int64_t)row * H + h]);
                }
            }
            if (grad_w) grad_w[t * K + k] = dot;
        }
    }
}

/* Backward of dispatch: grad_x[t] = bf16( sum over valid k of grad_recv[row(t,k)] )
 * (fp32 adds in ascending k from +0, one round; the unweighted combine), and
 * grad_topk_weights[t, k] = grad_recv_weights[row(t,k)], 0 for dropped slots. */
void orc_dispatch_backward(const uint16_t* grad_recv, const float* grad_recv_weights, int H,
                           const int32_t* row_of_slot, int64_t T, int K, uint16_t* grad_x,
                           float* grad_topk_weights) {
    orc_combine(grad_recv, H, row_of_slot, T, K, 0, grad_x);
    if (grad_topk_weights) {
        for (int64_t s = 0; s < T * (int64_t)K; ++s) {
            int32_t row = row_of_slot[s];
            grad_topk_weights[s] = row >= 0 ? grad_recv_weights[row] : 0.0f;
        }
    }
}

/* ---------------------------------------------------------------- fp8 variants */

/* Smallest power of two >= s (s > 0, finite fp32), found by exponent
 * arithmetic on the exact value: frexp gives s = fr * 2^ex, fr in [0.5, 1);
 * s is itself a power of two iff fr == 0.5. */
float orc_pow2_ceil(float s) {
    int ex;
    double fr = frexp((double)s, &ex);
    return (float)ldexp(1.0, fr == 0.5 ? ex - 1 : ex);
}

/* Quantise one row with power-of-two block scales (nccl_ep.cc, ncclEpDispatch:
 * round_scales; DeepEP API docs: use_ue8m0 scale factors):
 *   s = amax / 448 (fp32 division), scale = smallest power of two >= s,
 *   q = e4m3_rne_satfinite(x / scale).
 * ue8m0 != 0: the scale is stored as its biased exponent byte (value
 * 2^(byte - 127)); powers below 2^-127 are raised to 2^-127 (byte 0) before
 * quantising. An all-zero block gives zero codes and scale 0 (byte 0).
 * Scales go to srow[b] as fp32, or to sbytes[b] as bytes when ue8m0. */
void orc_quant_row_e4m3_pow2(const uint16_t* xrow, int H, int ue8m0, uint8_t* qrow, float* srow,
                             uint8_t* sbytes) {
    for (int b = 0; b < H / 128; ++b) {
        float amax = 0.0f;
        for (int i = 0; i < 128; ++i) {
            float v = fabsf(orc_bf16_to_f32(xrow[b * 128 + i]));
            if (v > amax) amax = v;
        }
        if (amax == 0.0f) {
            if (ue8m0) sbytes[b] = 0; else srow[b] = 0.0f;
            for (int i = 0; i < 128; ++i) qrow[b * 128 + i] = 0x00;
            continue;
        }
        float scale = orc_pow2_ceil(amax / 448.0f);
        if (ue8m0) {
            if (scale < ldexpf(1.0f, -127)) scale = ldexpf(1.0f, -127);
            int ex;
            (void)frexpf(scale, &ex);          /* scale = 0.5 * 2^ex = 2^(ex-1) */
            sbytes[b] = (uint8_t)(ex - 1 + 127);
        } else {
            srow[b] = scale;
        }
        for (int i = 0; i < 128; ++i)
            qrow[b * 128 + i] = orc_f32_to_e4m3(orc_bf16_to_f32(xrow[b * 128 + i]) / scale);
    }
}

/* Quantise one row to e5m2 with one scale per 128 channels, the e4m3 recipe
 * with e5m2's largest finite value in place of 448:
 *   s = amax / 57344 (fp32 division);
 *   scale_mode 0: scale = s, stored as fp32;
 *   scale_mode 1: scale = smallest power of two >= s, stored as fp32;
 *   scale_mode 2: that power raised to at least 2^-127, stored as its biased
 *                 exponent byte in sbytes[b];
 *   q = e5m2_rne_satfinite(x / scale).
 * An all-zero block gives zero codes and scale 0 (byte 0). */
void orc_quant_row_e5m2(const uint16_t* xrow, int H, int scale_mode, uint8_t* qrow, float* srow,
                        uint8_t* sbytes) {
    for (int b = 0; b < H / 128; ++b) {
        float amax = 0.0f;
        for (int i = 0; i < 128; ++i) {
            float v = fabsf(orc_bf16_to_f32(xrow[b * 128 + i]));
            if (v > amax) amax = v;
        }
        if (amax == 0.0f) {
            if (scale_mode == 2) sbytes[b] = 0; else srow[b] = 0.0f;
            for (int i = 0; i < 128; ++i) qrow[b * 128 + i] = 0x00;
            continue;
        }
        float scale = amax / 57344.0f;
        if (scale_mode != 0) scale = orc_pow2_ceil(scale);
        if (scale_mode == 2) {
            if (scale < ldexpf(1.0f, -127)) scale = ldexpf(1.0f, -127);
            int ex;
            (void)frexpf(scale, &ex);          /* scale = 2^(ex-1) */
            sbytes[b] = (uint8_t)(ex - 1 + 127);
        } else {
            srow[b] = scale;
        }
        for (int i = 0; i < 128; ++i)
            qrow[b * 128 + i] = orc_f32_to_e5m2(orc_bf16_to_f32(xrow[b * 128 + i]) / scale);
    }
}

void orc_f32_to_e5m2_array(const float* in, int64_t n, uint8_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_f32_to_e5m2(in[i]);
}

/* Sweep fp32 bit patterns [lo, hi) through the e5m2 encoder (no input array). */
void orc_e5m2_sweep(uint32_t lo, uint32_t hi, uint8_t* out) {
    for (uint32_t u = lo; u < hi; ++u) {
        float f;
        memcpy(&f, &u, sizeof f);
        out[u - lo] = orc_f32_to_e5m2(f);
    }
}

/* Byte permute of whole rows: recv[row_of_slot[t,k]] = src[t] (row_bytes
 * each) for every used slot -- fp8 input pass-through of codes and of scale
 * rows (DeepEP API docs, dispatch(): x may be an (fp8 data, scales) tuple). */
void orc_dispatch_rows(const uint8_t* src, int64_t T, int64_t row_bytes, const int32_t* row_of_slot, int K,
                       uint8_t* recv) {
    for (int64_t t = 0; t < T; ++t)
        for (int k = 0; k < K; ++k) {
            int32_t row = row_of_slot[t * K + k];
            if (row >= 0) memcpy(recv + (int64_t)row * row_bytes, src + t * row_bytes, (size_t)row_bytes);
        }
}

/* ---------------------------------------------------------------- dense maps */

/* Sparse top-k routing -> dense routing map and probabilities (nccl_ep.cc,
 * ncclEpCreateHandle: convert_topk_to_routing_map; ncclEpDispatch:
 * sparse_to_dense_prob; NeMo fused_a2a HybridEPDispatch: routing_map [T, E]
 * bool with probs [T, E]):
 *   routing_map[t, e] = 1 if some slot of t names e, else 0
 *   probs[t, e]       = sum over those slots, ascending k, of w[t, k] (fp32), else 0
 * Ids outside [0, E) are skipped. Returns ORC_ERR_EXPERT if any id lies
 * outside [-1, E). */
int orc_topk_to_routing_map(const int64_t* topk_idx, const float* w, int64_t T, int K, int E,
                            uint8_t* routing_map, float* probs) {
    int status = ORC_OK;
    for (int64_t t = 0; t < T; ++t) {
        for (int e = 0; e < E; ++e) {
            routing_map[t * E + e] = 0;
            if (probs) probs[t * E + e] = 0.0f;
        }
        for (int k = 0; k < K; ++k) {
            int64_t e = topk_idx[t * K + k];
            if (e == -1) continue;
            if (e < -1 || e >= E) { status = ORC_ERR_EXPERT; continue; }
            routing_map[t * E + e] = 1;
            if (probs && w) probs[t * E + e] += w[t * K + k];
        }
    }
    return status;
}

/* Dense routing map -> sparse top-k (nccl_ep.cc: dense_to_sparse_prob): the
 * experts of token t with routing_map[t, e] != 0, in ascending e, fill slots
 * 0, 1, ...; the remaining slots are -1 with weight 0; topk_weights take
 * probs[t, e] (or 1 if probs is NULL). Returns ORC_ERR_ARG (and keeps the
 * first K experts) if a token has more than K experts. */
int orc_routing_map_to_topk(const uint8_t* routing_map, const float* probs, int64_t T, int E, int K,
                            int64_t* topk_idx, float* topk_weights) {
    int status = ORC_OK;
    for (int64_t t = 0; t < T; ++t) {
        int k = 0;
        for (int e = 0; e < E; ++e) {
            if (!routing_map[t * E + e]) continue;
            if (k < K) {
                topk_idx[t * K + k] = e;
                if (topk_weights) topk_weights[t * K + k] = probs ? probs[t * E + e] : 1.0f;
            } else {
                status = ORC_ERR_ARG;
            }
            ++k;
        }
        for (; k < K; ++k) {
            topk_idx[t * K + k] = -1;
            if (topk_weights) topk_weights[t * K + k] = 0.0f;
        }
    }
    return status;
}

/* ---------------------------------------------------------------- strided layout */

#define ORC_ERR_CAPACITY 3

/* Routing layout with a fixed row stride per expert: the padded 3-D receive
 * buffer [E, cap, H] of nccl_ep.cc's low-latency dispatch (recv_x
 * [num_local_experts, num_ranks * max_tokens_per_rank, hidden] with
 * per-expert receive counts). expert_offsets[e] = e * cap,
 * expert_offsets[E] = E * cap; expert e's slots take rows e * cap + 0, 1, ...
 * in (t, k) order. A slot whose rank inside its expert reaches cap is dropped
 * (row -1) and the call returns ORC_ERR_CAPACITY; the counts stay the full
 * counts. Rows past an expert's count are not part of the layout. */
int orc_layout_strided(const int64_t* topk_idx, int64_t T, int K, int E, int R, int cap,
                       int32_t* num_tokens_per_expert, int32_t* num_tokens_per_rank,
                       uint8_t* is_token_in_rank, int32_t* expert_offsets, int32_t* row_of_slot) {
    if (cap < 1) return ORC_ERR_ARG;
    int32_t* packed = (int32_t*)malloc(sizeof(int32_t) * (size_t)(E + 1));
    if (!packed) return ORC_ERR_ARG;
    int status = orc_layout(topk_idx, T, K, E, R, num_tokens_per_expert, num_tokens_per_rank,
                            is_token_in_rank, packed, row_of_slot);
    if (status == ORC_ERR_ARG) { free(packed); return status; }
    if ((int64_t)E * cap > INT32_MAX) { free(packed); return ORC_ERR_ARG; }
    for (int e = 0; e <= E; ++e) expert_offsets[e] = e * cap;
    for (int64_t s = 0; s < T * (int64_t)K; ++s) {
        if (row_of_slot[s] < 0) continue;
        int64_t e = topk_idx[s];
        int32_t rank_in_expert = row_of_slot[s] - packed[e];
        if (rank_in_expert >= cap) {
            row_of_slot[s] = -1;
            if (status == ORC_OK) status = ORC_ERR_CAPACITY;
        } else {
            row_of_slot[s] = (int32_t)(e * cap) + rank_in_expert;
        }
    }
    free(packed);
    return status;
}

/* ---------------------------------------------------------------- non-expand */

/* Non-expand layout: one receive row per (token, rank) pair (DeepEP API
 * docs, "Prefix Sum Interpretation for Expert Token Counts", non-expand mode;
 * nccl_ep.cc, struct ncclEpHandle: sparse_to_dense_map [tokens, ranks] with -1
 * for "not routed"). Rows are grouped by rank, tokens ascending inside a rank:
 *   rank_offsets[R + 1] = exclusive prefix sum of num_tokens_per_rank
 *   row_of_slot[t, k]   = the row of (t, rank(e)) for the FIRST slot of token
 *                         t on that rank (lowest k), -1 for its other slots on
 *                         the same rank and for unused slots.
 * num_tokens_per_expert, num_tokens_per_rank and is_token_in_rank are those of
 * orc_layout. */
int orc_layout_nonexpand(const int64_t* topk_idx, int64_t T, int K, int E, int R,
                         int32_t* num_tokens_per_expert, int32_t* num_tokens_per_rank,
                         uint8_t* is_token_in_rank, int32_t* rank_offsets, int32_t* row_of_slot) {
    int32_t* expert_offsets = (int32_t*)malloc(sizeof(int32_t) * (size_t)(E + 1));
    if (!expert_offsets) return ORC_ERR_ARG;
    int status = orc_layout(topk_idx, T, K, E, R, num_tokens_per_expert, num_tokens_per_rank,
                            is_token_in_rank, expert_offsets, row_of_slot);
    free(expert_offsets);
    if (status == ORC_ERR_ARG) return status;
    int L = E / R;
    int64_t run = 0;
    for (int r = 0; r < R; ++r) { rank_offsets[r] = (int32_t)run; run += num_tokens_per_rank[r]; }
    rank_offsets[R] = (int32_t)run;
    int64_t* next = (int64_t*)malloc(sizeof(int64_t) * (size_t)R);
    if (!next) return ORC_ERR_ARG;
    for (int r = 0; r < R; ++r) next[r] = rank_offsets[r];
    for (int64_t t = 0; t < T; ++t) {
        for (int k = 0; k < K; ++k) {
            int64_t e = topk_idx[t * K + k];
            row_of_slot[t * K + k] = -1;
            if (e < 0 || e >= E) continue;
            int64_t r = e / L;
            int first = 1;
            for (int j = 0; j < k; ++j) {
                int64_t ej = topk_idx[t * K + j];
                if (ej >= 0 && ej < E && ej / L == r) { first = 0; break; }
            }
            if (first) row_of_slot[t * K + k] = (int32_t)next[r]++;
        }
    }
    free(next);
    return status;
}

/* What each non-expand receive row carries for its rank's experts (DeepEP API
 * docs, "dispatch()": recv_topk_idx / recv_topk_weights): for the row of
 * (t, r), entry k is the rank-local expert id e - r * (E/R) if slot k of t
 * names an expert of rank r, else -1 (weight w[t, k], else 0). */
void orc_nonexpand_recv_topk(const int64_t* topk_idx, const float* w, const int32_t* row_of_slot,
                             int64_t T, int K, int E, int R, int64_t* recv_topk_idx,
                             float* recv_topk_weights) {
    int L = E / R;
    for (int64_t t = 0; t < T; ++t) {
        for (int k = 0; k < K; ++k) {
            int32_t row = row_of_slot[t * K + k];
            if (row < 0) continue;
            int64_t r = topk_idx[t * K + k] / L;
            for (int j = 0; j < K; ++j) {
                int64_t ej = topk_idx[t * K + j];
                int on = ej >= 0 && ej < E && ej / L == r;
                recv_topk_idx[(int64_t)row * K + j] = on ? ej - r * L : -1;
                if (recv_topk_weights) recv_topk_weights[(int64_t)row * K + j] = on && w ? w[t * K + j] : 0.0f;
            }
        }
    }
}

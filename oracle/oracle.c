/*
 * oracle.c -- CPU oracle for the W8A8 quantised mixture-of-experts layer.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the tests, the smoke check and
 * the benchmark's CPU-baseline leg load this library.  The CUDA library never
 * links, loads or calls it, and the two share no source, header, table or
 * helper.
 *
 * Every function is the method's definition written out as plain loops, in
 * the order the pages state it, with no blocking, fusion or reordering:
 *
 *   symmetric INT8 quantisation  q = clamp(round(x / s), -128, 127),
 *   s = amax / 127, weights per output channel, activations per token
 *     -- "W8A8 quantisation of MiniMax-M3 on K100AI" (mhpn.cn), section 2.1
 *   INT8 GEMM [A,K]x[K,N] with the activation scale [A,1] and the weight
 *   scale [1,N] applied as an outer product on the output
 *     -- same page, section 2.1
 *   low-precision operands, FP32 accumulator/epilogue, re-quantise the
 *   output to 8 bits for the next operator
 *     -- "DeepSeek V4 950 FP8 inference on H100" (lpnh.cn), section 2.3
 *   router kept in FP32, never quantised
 *     -- same page, section 4.1
 *   gate -> top-k -> per-expert contiguous slots -> expert GEMMs -> weighted
 *   combine back to token order
 *     -- "Tencent Hunyuan AI Infra on Hopper" (pnsm.cn), section 1.3
 *   SmoothQuant-folded activations with per-expert factors (last section)
 *     -- "W8A8 quantisation of MiniMax-M3 on K100AI", section 2.2
 *
 * Precision.  Wherever a floating-point value decides an integer (a
 * quantised code) the oracle works in IEEE binary32 with the operation order
 * written below, because the GPU takes the same decision in binary32.  The
 * router logits are summed in binary64 and rounded once to binary32 (the
 * best binary32 value of the dot product).  Integer GEMMs accumulate in
 * int64 and report overflow of int32.  Build with -ffp-contract=off and no
 * fast-math so that every multiply and add is a separately rounded
 * binary32 operation.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   round()      -> round half to even (rintf in the default rounding mode)
 *   s            -> amax / 127.0f, one correctly rounded binary32 division;
 *                   x / s likewise (not x * (1/s))
 *   amax == 0    -> s = 0 and every code 0
 *   epilogue     -> (float(acc) * s_act) * s_w, two rounded multiplies
 *   SiLU gate    -> h = (g / (1 + expf(-g))) * u, w13 rows = gate then up
 *   requant      -> per (token, expert) slot row of h, over its I columns
 *   top-k        -> k largest logits, ties to the lower expert index, in
 *                   descending order; weights = softmax over the selected
 *                   logits (equal to the renormalised full softmax)
 *   router bias  -> optional, added to the logits before selection
 *   slot order   -> experts ascending; inside an expert, tokens ascending
 *   combine      -> y = bf16_rne(sum_j w_j * o_j), j = 0..k-1 in top-k
 *                   order, binary32 multiply then add
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_ERR_ARG -1
#define ORACLE_ERR_OVERFLOW -2
#define ORACLE_ERR_NOMEM -3

/* ---- bfloat16 <-> binary32 (bf16 = the upper 16 bits of a binary32) ---- */

static float bf16_to_f32(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* Round a binary32 to the nearest bf16, ties to even; NaN stays NaN. */
static uint16_t f32_to_bf16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0u)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb;
    return (uint16_t)(u >> 16);
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int oracle_bf16_to_f32(const uint16_t* in, int64_t n, float* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = bf16_to_f32(in[i]);
    return ORACLE_OK;
}

int oracle_f32_to_bf16(const float* in, int64_t n, uint16_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = f32_to_bf16_rne(in[i]);
    return ORACLE_OK;
}

/* ---- symmetric per-row INT8 quantisation --------------------------------
 * One scale per row of length K:  amax = max_k |x[k]|,  s = amax / 127,
 * q[k] = clamp(round_half_even(x[k] / s), -128, 127).  A row of zeros gets
 * s = 0 and q = 0.  This is the weight quantiser (rows = output channels),
 * the activation quantiser (rows = tokens) and the requantiser (rows =
 * slots of h): "W8A8 quantisation of MiniMax-M3 on K100AI", section 2.1.
 */
static void quantize_row(const float* x, int64_t K, int8_t* q, float* s_out) {
    float amax = 0.0f;
    for (int64_t k = 0; k < K; ++k) {
        float a = fabsf(x[k]);
        if (a > amax) amax = a;
    }
    float s = amax / 127.0f;
    *s_out = s;
    for (int64_t k = 0; k < K; ++k) {
        if (s == 0.0f) {
            q[k] = 0;
            continue;
        }
        float r = rintf(x[k] / s);
        if (r > 127.0f) r = 127.0f;
        if (r < -128.0f) r = -128.0f;
        q[k] = (int8_t)r;
    }
}

int oracle_quantize_rows(const float* x, int64_t rows, int64_t K, int8_t* q, float* s) {
    if (rows < 0 || K <= 0) return ORACLE_ERR_ARG;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) quantize_row(x + r * K, K, q + r * K, s + r);
    return ORACLE_OK;
}

/* Per-token quantisation of bf16 activations: the bf16 value widened to
 * binary32 (exact), then the quantiser above. */
int oracle_quantize_rows_bf16(const uint16_t* x, int64_t rows, int64_t K, int8_t* q, float* s) {
    if (rows < 0 || K <= 0) return ORACLE_ERR_ARG;
    int err = 0;
#pragma omp parallel
    {
        float* row = (float*)malloc((size_t)K * sizeof(float));
        if (!row) {
#pragma omp atomic write
            err = 1;
        }
#pragma omp for schedule(static)
        for (int64_t r = 0; r < rows; ++r) {
            if (!row) continue;
            for (int64_t k = 0; k < K; ++k) row[k] = bf16_to_f32(x[r * K + k]);
            quantize_row(row, K, q + r * K, s + r);
        }
        free(row);
    }
    return err ? ORACLE_ERR_NOMEM : ORACLE_OK;
}

/* ---- router: FP32 logits, top-k, softmax over the selected ---------------
 * logit[t][e] = sum_h x[t][h] * Wr[h][e] (+ bias[e]), summed in binary64 and
 * rounded once to binary32 ("keep the router in FP32": "DeepSeek V4 950 FP8
 * inference on H100", section 4.1).  The k largest logits are selected,
 * ties to the lower expert index, listed in descending order; their weights
 * are exp(l_j - l_max) / sum_i exp(l_i - l_max) over the selected ones,
 * computed in binary64 and rounded to binary32.  Gate -> top-k is the first
 * stage of the fused MoE pipeline in "Tencent Hunyuan AI Infra on Hopper",
 * section 1.3.
 */
int oracle_router(const uint16_t* x, const float* Wr, const float* bias, int64_t T, int64_t H,
                  int64_t E, int64_t k, int32_t* topk_ids, float* topk_w, float* logits_out) {
    if (T < 0 || H <= 0 || E <= 0 || k <= 0 || k > E) return ORACLE_ERR_ARG;
    int err = 0;
#pragma omp parallel
    {
        float* logit = (float*)malloc((size_t)E * sizeof(float));
        unsigned char* taken = (unsigned char*)malloc((size_t)E);
        if (!logit || !taken) {
#pragma omp atomic write
            err = 1;
        }
#pragma omp for schedule(static)
        for (int64_t t = 0; t < T; ++t) {
            if (!logit || !taken) continue;
            for (int64_t e = 0; e < E; ++e) {
                double acc = 0.0;
                for (int64_t h = 0; h < H; ++h)
                    acc += (double)bf16_to_f32(x[t * H + h]) * (double)Wr[h * E + e];
                if (bias) acc += (double)bias[e];
                logit[e] = (float)acc;
                taken[e] = 0;
                if (logits_out) logits_out[t * E + e] = logit[e];
            }
            /* selection: repeatedly take the largest remaining logit; a
             * strictly larger value wins, so equal values keep the lower
             * index. */
            for (int64_t j = 0; j < k; ++j) {
                int64_t best = -1;
                for (int64_t e = 0; e < E; ++e) {
                    if (taken[e]) continue;
                    if (best < 0 || logit[e] > logit[best]) best = e;
                }
                taken[best] = 1;
                topk_ids[t * k + j] = (int32_t)best;
            }
            double lmax = (double)logit[topk_ids[t * k + 0]];
            double denom = 0.0;
            for (int64_t j = 0; j < k; ++j) denom += exp((double)logit[topk_ids[t * k + j]] - lmax);
            for (int64_t j = 0; j < k; ++j)
                topk_w[t * k + j] = (float)(exp((double)logit[topk_ids[t * k + j]] - lmax) / denom);
        }
        free(logit);
        free(taken);
    }
    return err ? ORACLE_ERR_NOMEM : ORACLE_OK;
}

/* ---- permutation into contiguous per-expert slots -----------------------
 * counts[e] = number of (t, j) routed to e; offsets = exclusive prefix sum
 * (offsets[E] = T*k); expert e owns slots [offsets[e], offsets[e+1]) and
 * fills them with its tokens in ascending token order.  slot_of[t][j] is the
 * slot of (t, j) and slot_token[s] the token held by slot s.  "Reserve a
 * contiguous output region for every expert during routing pre-processing":
 * "Tencent Hunyuan AI Infra on Hopper", section 1.3.
 */
int oracle_permute(const int32_t* topk_ids, int64_t T, int64_t E, int64_t k, int32_t* counts,
                   int32_t* offsets, int32_t* slot_of, int32_t* slot_token) {
    if (T < 0 || E <= 0 || k <= 0) return ORACLE_ERR_ARG;
    for (int64_t e = 0; e < E; ++e) counts[e] = 0;
    for (int64_t i = 0; i < T * k; ++i) {
        int32_t e = topk_ids[i];
        if (e < 0 || e >= E) return ORACLE_ERR_ARG;
        counts[e] += 1;
    }
    offsets[0] = 0;
    for (int64_t e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
    int32_t* next = (int32_t*)malloc((size_t)E * sizeof(int32_t));
    if (!next) return ORACLE_ERR_NOMEM;
    for (int64_t e = 0; e < E; ++e) next[e] = offsets[e];
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t j = 0; j < k; ++j) {
            int32_t e = topk_ids[t * k + j];
            int32_t s = next[e]++;
            slot_of[t * k + j] = s;
            slot_token[s] = (int32_t)t;
        }
    }
    free(next);
    return ORACLE_OK;
}

/* ---- exact INT8 GEMM ------------------------------------------------------
 * acc[m][n] = sum_k a[m][k] * b[n][k] (both operands K-contiguous, i.e.
 * Y = A * B^T), accumulated in int64; returns ORACLE_ERR_OVERFLOW if a
 * result does not fit int32.  The integer matmul of "W8A8 quantisation of
 * MiniMax-M3 on K100AI", section 2.1.
 */
int oracle_gemm_s8(const int8_t* a, const int8_t* b, int64_t M, int64_t N, int64_t K, int32_t* acc) {
    if (M < 0 || N < 0 || K <= 0) return ORACLE_ERR_ARG;
    int overflow = 0;
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            int64_t sum = 0;
            for (int64_t kk = 0; kk < K; ++kk) sum += (int64_t)a[m * K + kk] * (int64_t)b[n * K + kk];
            if (sum > INT32_MAX || sum < INT32_MIN) {
#pragma omp atomic write
                overflow = 1;
            }
            acc[m * N + n] = (int32_t)sum;
        }
    }
    return overflow ? ORACLE_ERR_OVERFLOW : ORACLE_OK;
}

/* ---- epilogues (binary32, fixed operation order) -------------------------
 * Scale outer product: value = (float(acc) * s_act[row]) * s_w[col].
 * "W8A8 quantisation of MiniMax-M3 on K100AI", section 2.1.
 */
static float dequant(int32_t acc, float s_act, float s_w) {
    float v = (float)acc;
    v = v * s_act;
    v = v * s_w;
    return v;
}

static float silu(float g) {
    float d = 1.0f + expf(-g);
    return g / d;
}

/* Gate/up epilogue of the first expert GEMM for S rows of one expert.
 * acc1 is [S][2I] (gate columns 0..I-1, up columns I..2I-1), s_act[S] the
 * per-row activation scales, s_w13[2I] the expert's channel scales:
 * h[s][n] = silu(g) * u with g = dequant(acc1[s][n]), u = dequant(acc1[s][I+n]).
 */
int oracle_epilogue_gate_up(const int32_t* acc1, const float* s_act, const float* s_w13, int64_t S,
                            int64_t I, float* h) {
    if (S < 0 || I <= 0) return ORACLE_ERR_ARG;
#pragma omp parallel for schedule(static)
    for (int64_t s = 0; s < S; ++s) {
        for (int64_t n = 0; n < I; ++n) {
            float g = dequant(acc1[s * 2 * I + n], s_act[s], s_w13[n]);
            float u = dequant(acc1[s * 2 * I + I + n], s_act[s], s_w13[I + n]);
            h[s * I + n] = silu(g) * u;
        }
    }
    return ORACLE_OK;
}

/* Output epilogue of a GEMM: out[s][c] = dequant(acc[s][c], s_act[s], s_w[c]). */
int oracle_epilogue_scale(const int32_t* acc, const float* s_act, const float* s_w, int64_t S,
                          int64_t N, float* out) {
    if (S < 0 || N <= 0) return ORACLE_ERR_ARG;
#pragma omp parallel for schedule(static)
    for (int64_t s = 0; s < S; ++s)
        for (int64_t c = 0; c < N; ++c) out[s * N + c] = dequant(acc[s * N + c], s_act[s], s_w[c]);
    return ORACLE_OK;
}

/* ---- weighted top-k combine ------------------------------------------------
 * y[t][c] = bf16_rne( sum_{j=0}^{k-1} w[t][j] * o[slot_of[t][j]][c] ), the
 * sum in binary32, one multiply and one add per term, j in top-k order.
 * "Weighted aggregation at the end of the pipeline": "Tencent Hunyuan AI
 * Infra on Hopper", section 1.3.
 */
int oracle_combine(const float* o, const int32_t* slot_of, const float* topk_w, int64_t T, int64_t k,
                   int64_t H, uint16_t* y) {
    if (T < 0 || k <= 0 || H <= 0) return ORACLE_ERR_ARG;
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t c = 0; c < H; ++c) {
            float acc = 0.0f;
            for (int64_t j = 0; j < k; ++j) {
                float term = topk_w[t * k + j] * o[(int64_t)slot_of[t * k + j] * H + c];
                acc = acc + term;
            }
            y[t * H + c] = f32_to_bf16_rne(acc);
        }
    }
    return ORACLE_OK;
}

/* ---- the whole layer, sparse path ----------------------------------------
 * x bf16 [T][H]; Wr fp32 [H][E]; bias fp32 [E] or NULL;
 * w13_q int8 [E][2I][H], s_w13 fp32 [E][2I]; w2_q int8 [E][H][I],
 * s_w2 fp32 [E][H]; y bf16 [T][H].  The optional dump pointers receive the
 * intermediates (NULL = skip):
 *   topk_ids [T][k], topk_w [T][k], offsets [E+1], slot_of [T][k],
 *   slot_token [S], s_x [T], q_x [T][H], acc1 [S][2I], h [S][I], s_h [S],
 *   q_h [S][I], acc2 [S][H], o [S][H]       with S = T*k.
 */
typedef struct {
    int32_t* topk_ids;
    float* topk_w;
    int32_t* offsets;
    int32_t* slot_of;
    int32_t* slot_token;
    float* s_x;
    int8_t* q_x;
    int32_t* acc1;
    float* h;
    float* s_h;
    int8_t* q_h;
    int32_t* acc2;
    float* o;
} oracle_dump_t;

static void* xmalloc(size_t n) { return malloc(n ? n : 1); }

static void quantize_row_bf16_smoothed(const uint16_t* x, const float* sm, int64_t H, float* tmp, int8_t* q,
                                       float* s_out);

/* smooth: NULL, or the per-expert smoothing factors [E][H] of the section on
 * SmoothQuant below (each slot's row is then its token's row times the
 * reciprocal factors of the slot's expert, quantised per slot). */
static int moe_forward_impl(const uint16_t* x, const float* Wr, const float* bias, const float* smooth,
                            const int8_t* w13_q, const float* s_w13, const int8_t* w2_q, const float* s_w2,
                            int64_t T, int64_t H, int64_t I, int64_t E, int64_t k, uint16_t* y,
                            const oracle_dump_t* dump, float* s_slot_dump, int8_t* q_slot_dump) {
    if (T < 0 || H <= 0 || I <= 0 || E <= 0 || k <= 0 || k > E) return ORACLE_ERR_ARG;
    const int64_t S = T * k;
    int rc = ORACLE_OK;
    int32_t* topk_ids = (int32_t*)xmalloc((size_t)S * 4);
    float* topk_w = (float*)xmalloc((size_t)S * 4);
    int32_t* counts = (int32_t*)xmalloc((size_t)E * 4);
    int32_t* offsets = (int32_t*)xmalloc((size_t)(E + 1) * 4);
    int32_t* slot_of = (int32_t*)xmalloc((size_t)S * 4);
    int32_t* slot_token = (int32_t*)xmalloc((size_t)S * 4);
    float* s_x = (float*)xmalloc((size_t)T * 4);
    int8_t* q_x = (int8_t*)xmalloc((size_t)(T * H));
    float* s_slot = (float*)xmalloc((size_t)S * 4);
    int8_t* q_slot = (int8_t*)xmalloc((size_t)(S * H));
    int32_t* acc1 = (int32_t*)xmalloc((size_t)(S * 2 * I) * 4);
    float* h = (float*)xmalloc((size_t)(S * I) * 4);
    float* s_h = (float*)xmalloc((size_t)S * 4);
    int8_t* q_h = (int8_t*)xmalloc((size_t)(S * I));
    int32_t* acc2 = (int32_t*)xmalloc((size_t)(S * H) * 4);
    float* o = (float*)xmalloc((size_t)(S * H) * 4);
    if (!topk_ids || !topk_w || !counts || !offsets || !slot_of || !slot_token || !s_x || !q_x ||
        !s_slot || !q_slot || !acc1 || !h || !s_h || !q_h || !acc2 || !o) {
        rc = ORACLE_ERR_NOMEM;
        goto done;
    }

    /* router, top-k */
    rc = oracle_router(x, Wr, bias, T, H, E, k, topk_ids, topk_w, NULL);
    if (rc) goto done;
    /* contiguous per-expert slots */
    rc = oracle_permute(topk_ids, T, E, k, counts, offsets, slot_of, slot_token);
    if (rc) goto done;
    /* per-token dynamic activation quantisation */
    rc = oracle_quantize_rows_bf16(x, T, H, q_x, s_x);
    if (rc) goto done;
    if (!smooth) {
        /* every slot holds a copy of its token's quantised row and scale */
        for (int64_t s = 0; s < S; ++s) {
            int64_t t = slot_token[s];
            memcpy(q_slot + s * H, q_x + t * H, (size_t)H);
            s_slot[s] = s_x[t];
        }
    } else {
        /* every slot quantises its token's row smoothed by its expert's factors */
        float* tmp = (float*)xmalloc((size_t)H * 4);
        if (!tmp) {
            rc = ORACLE_ERR_NOMEM;
            goto done;
        }
        for (int64_t e = 0; e < E; ++e)
            for (int64_t s = offsets[e]; s < offsets[e + 1]; ++s)
                quantize_row_bf16_smoothed(x + (int64_t)slot_token[s] * H, smooth + e * H, H, tmp,
                                           q_slot + s * H, s_slot + s);
        free(tmp);
        /* a token's own scale and row are those of its first choice */
        for (int64_t t = 0; t < T; ++t) {
            s_x[t] = s_slot[slot_of[t * k]];
            memcpy(q_x + t * H, q_slot + (int64_t)slot_of[t * k] * H, (size_t)H);
        }
    }
    /* per expert: GEMM1, gate/up epilogue, requant, GEMM2, output epilogue */
    for (int64_t e = 0; e < E; ++e) {
        int64_t s0 = offsets[e], n = offsets[e + 1] - offsets[e];
        if (n == 0) continue;
        rc = oracle_gemm_s8(q_slot + s0 * H, w13_q + e * 2 * I * H, n, 2 * I, H, acc1 + s0 * 2 * I);
        if (rc) goto done;
        rc = oracle_epilogue_gate_up(acc1 + s0 * 2 * I, s_slot + s0, s_w13 + e * 2 * I, n, I, h + s0 * I);
        if (rc) goto done;
        rc = oracle_quantize_rows(h + s0 * I, n, I, q_h + s0 * I, s_h + s0);
        if (rc) goto done;
        rc = oracle_gemm_s8(q_h + s0 * I, w2_q + e * H * I, n, H, I, acc2 + s0 * H);
        if (rc) goto done;
        rc = oracle_epilogue_scale(acc2 + s0 * H, s_h + s0, s_w2 + e * H, n, H, o + s0 * H);
        if (rc) goto done;
    }
    /* weighted combine back to token order */
    rc = oracle_combine(o, slot_of, topk_w, T, k, H, y);
    if (rc) goto done;

    if (dump) {
        if (dump->topk_ids) memcpy(dump->topk_ids, topk_ids, (size_t)S * 4);
        if (dump->topk_w) memcpy(dump->topk_w, topk_w, (size_t)S * 4);
        if (dump->offsets) memcpy(dump->offsets, offsets, (size_t)(E + 1) * 4);
        if (dump->slot_of) memcpy(dump->slot_of, slot_of, (size_t)S * 4);
        if (dump->slot_token) memcpy(dump->slot_token, slot_token, (size_t)S * 4);
        if (dump->s_x) memcpy(dump->s_x, s_x, (size_t)T * 4);
        if (dump->q_x) memcpy(dump->q_x, q_x, (size_t)(T * H));
        if (dump->acc1) memcpy(dump->acc1, acc1, (size_t)(S * 2 * I) * 4);
        if (dump->h) memcpy(dump->h, h, (size_t)(S * I) * 4);
        if (dump->s_h) memcpy(dump->s_h, s_h, (size_t)S * 4);
        if (dump->q_h) memcpy(dump->q_h, q_h, (size_t)(S * I));
        if (dump->acc2) memcpy(dump->acc2, acc2, (size_t)(S * H) * 4);
        if (dump->o) memcpy(dump->o, o, (size_t)(S * H) * 4);
    }
    if (s_slot_dump) memcpy(s_slot_dump, s_slot, (size_t)S * 4);
    if (q_slot_dump) memcpy(q_slot_dump, q_slot, (size_t)(S * H));
done:
    free(topk_ids); free(topk_w); free(counts); free(offsets); free(slot_of); free(slot_token);
    free(s_x); free(q_x); free(s_slot); free(q_slot); free(acc1); free(h); free(s_h); free(q_h);
    free(acc2); free(o);
    return rc;
}

int oracle_moe_forward(const uint16_t* x, const float* Wr, const float* bias, const int8_t* w13_q,
                       const float* s_w13, const int8_t* w2_q, const float* s_w2, int64_t T,
                       int64_t H, int64_t I, int64_t E, int64_t k, uint16_t* y,
                       const oracle_dump_t* dump) {
    return moe_forward_impl(x, Wr, bias, NULL, w13_q, s_w13, w2_q, s_w2, T, H, I, E, k, y, dump, NULL, NULL);
}

/* ---- the whole layer, brute force -----------------------------------------
 * Evaluates every expert on every token with no routing structure at all
 * (no counts, offsets or slots): for each (t, e) the expert output row
 * o_te = epilogue(GEMM2(requant(epilogue(GEMM1(q_x[t]))))), then
 * y[t] = bf16_rne(sum_j w[t][j] * o_{t, e_j}).  Only for tiny shapes; it
 * must agree with the sparse path bit for bit.
 */
int oracle_moe_forward_dense(const uint16_t* x, const float* Wr, const float* bias,
                             const int8_t* w13_q, const float* s_w13, const int8_t* w2_q,
                             const float* s_w2, int64_t T, int64_t H, int64_t I, int64_t E,
                             int64_t k, uint16_t* y) {
    if (T < 0 || H <= 0 || I <= 0 || E <= 0 || k <= 0 || k > E) return ORACLE_ERR_ARG;
    int rc = ORACLE_OK;
    int32_t* topk_ids = (int32_t*)xmalloc((size_t)(T * k) * 4);
    float* topk_w = (float*)xmalloc((size_t)(T * k) * 4);
    float* s_x = (float*)xmalloc((size_t)T * 4);
    int8_t* q_x = (int8_t*)xmalloc((size_t)(T * H));
    float* o_all = (float*)xmalloc((size_t)(T * E * H) * 4);
    int32_t* acc1 = (int32_t*)xmalloc((size_t)(2 * I) * 4);
    float* h = (float*)xmalloc((size_t)I * 4);
    int8_t* q_h = (int8_t*)xmalloc((size_t)I);
    int32_t* acc2 = (int32_t*)xmalloc((size_t)H * 4);
    if (!topk_ids || !topk_w || !s_x || !q_x || !o_all || !acc1 || !h || !q_h || !acc2) {
        rc = ORACLE_ERR_NOMEM;
        goto done;
    }
    rc = oracle_router(x, Wr, bias, T, H, E, k, topk_ids, topk_w, NULL);
    if (rc) goto done;
    rc = oracle_quantize_rows_bf16(x, T, H, q_x, s_x);
    if (rc) goto done;
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t e = 0; e < E; ++e) {
            float s_h;
            rc = oracle_gemm_s8(q_x + t * H, w13_q + e * 2 * I * H, 1, 2 * I, H, acc1);
            if (rc) goto done;
            rc = oracle_epilogue_gate_up(acc1, s_x + t, s_w13 + e * 2 * I, 1, I, h);
            if (rc) goto done;
            rc = oracle_quantize_rows(h, 1, I, q_h, &s_h);
            if (rc) goto done;
            rc = oracle_gemm_s8(q_h, w2_q + e * H * I, 1, H, I, acc2);
            if (rc) goto done;
            rc = oracle_epilogue_scale(acc2, &s_h, s_w2 + e * H, 1, H, o_all + (t * E + e) * H);
            if (rc) goto done;
        }
    }
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t c = 0; c < H; ++c) {
            float acc = 0.0f;
            for (int64_t j = 0; j < k; ++j) {
                int64_t e = topk_ids[t * k + j];
                float term = topk_w[t * k + j] * o_all[(t * E + e) * H + c];
                acc = acc + term;
            }
            y[t * H + c] = f32_to_bf16_rne(acc);
        }
    }
done:
    free(topk_ids); free(topk_w); free(s_x); free(q_x); free(o_all); free(acc1); free(h); free(q_h);
    free(acc2);
    return rc;
}

/* ---- single W8A8 linear layer (the dense form of the expert GEMM) --------
 * x bf16 [M][K] quantised per token, w_q int8 [N][K] with per-channel scales
 * s_w [N]:  y[m][n] = bf16_rne((float(acc[m][n]) * s_x[m]) * s_w[n]).
 * "W8A8 quantisation of MiniMax-M3 on K100AI", section 2.1.
 */
int oracle_linear(const uint16_t* x, const int8_t* w_q, const float* s_w, int64_t M, int64_t N,
                  int64_t K, uint16_t* y, int8_t* q_x_out, float* s_x_out, int32_t* acc_out) {
    if (M < 0 || N <= 0 || K <= 0) return ORACLE_ERR_ARG;
    int rc = ORACLE_OK;
    int8_t* q_x = (int8_t*)xmalloc((size_t)(M * K));
    float* s_x = (float*)xmalloc((size_t)M * 4);
    int32_t* acc = (int32_t*)xmalloc((size_t)(M * N) * 4);
    if (!q_x || !s_x || !acc) {
        rc = ORACLE_ERR_NOMEM;
        goto done;
    }
    rc = oracle_quantize_rows_bf16(x, M, K, q_x, s_x);
    if (rc) goto done;
    rc = oracle_gemm_s8(q_x, w_q, M, N, K, acc);
    if (rc) goto done;
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) y[m * N + n] = f32_to_bf16_rne(dequant(acc[m * N + n], s_x[m], s_w[n]));
    if (q_x_out) memcpy(q_x_out, q_x, (size_t)(M * K));
    if (s_x_out) memcpy(s_x_out, s_x, (size_t)M * 4);
    if (acc_out) memcpy(acc_out, acc, (size_t)(M * N) * 4);
done:
    free(q_x); free(s_x); free(acc);
    return rc;
}

/* ==== FP8 (E4M3) variant of the layer =====================================
 * "DeepSeek V4 950 FP8 inference on H100" (lpnh.cn): weights and activations
 * of the forward pass in E4M3 (4 exponent bits, 3 mantissa bits, largest
 * finite magnitude 448; section 2.1), FP8 operands with an FP32 accumulator
 * whose result is re-quantised to FP8 for the next operator (section 2.3),
 * one scale per weight output channel and per token for the activations,
 * computed dynamically (section 2.4), weight scales from the absolute
 * maximum (section 3.1).  The rest of the layer (router, slots, SiLU gate,
 * combine) is the INT8 layer's.
 *
 * Readings where the page is silent (each is listed in the design notes):
 *   scale        -> s = amax / 448.0f, one correctly rounded binary32 division
 *   code         -> the E4M3 value nearest to the binary32 quotient x / s,
 *                   ties to the code with an even mantissa, magnitudes above
 *                   448 saturated to 448 (the quotient exceeds 448 only through
 *                   its own rounding); the sign of a zero quotient is kept
 *   amax == 0    -> s = 0 and every code +0
 *   accumulator  -> the exact sum of the exact E4M3 products, rounded once to
 *                   binary32 (the best binary32 value of the FP32 accumulator's
 *                   dot product).  Every E4M3 value is an integer multiple of
 *                   2^-9 below 2^18 * 2^-9 in magnitude, so every product is an
 *                   integer multiple of 2^-18 below 2^18 in magnitude and the
 *                   binary64 sum of K < 2^17 of them is exact.
 */

/* Value of an E4M3 code: sign bit 7, exponent bits 6..3 (bias 7), mantissa
 * bits 2..0; exponent 0 is subnormal (m * 2^-9); S.1111.111 is NaN and there
 * is no infinity. */
static float e4m3_value(uint8_t b) {
    const int e = (b >> 3) & 15, m = b & 7;
    float v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexpf((float)m, -9);
    else v = ldexpf((float)(8 + m), e - 10);
    return (b & 0x80) ? -v : v;
}

/* Nearest E4M3 code (see the readings above).  The non-negative finite
 * codes 0x00..0x7E are increasing in value, so the nearest one is found by
 * bisection and a comparison with its two neighbours. */
static uint8_t e4m3_code(float v) {
    const uint8_t sign = signbit(v) ? 0x80 : 0x00;
    const float a = fabsf(v);
    if (a >= 448.0f) return (uint8_t)(sign | 0x7E);
    int lo = 0, hi = 0x7E;  /* invariant: value(lo) <= a < value(hi) */
    while (hi - lo > 1) {
        const int mid = (lo + hi) / 2;
        if (e4m3_value((uint8_t)mid) <= a) lo = mid; else hi = mid;
    }
    const double dlo = (double)a - (double)e4m3_value((uint8_t)lo);
    const double dhi = (double)e4m3_value((uint8_t)hi) - (double)a;
    int c;
    if (dlo < dhi) c = lo;
    else if (dhi < dlo) c = hi;
    else c = (lo % 2 == 0) ? lo : hi;  /* tie: the even mantissa */
    return (uint8_t)(sign | c);
}

int oracle_e4m3_encode(const float* in, int64_t n, uint8_t* out) {
    if (n < 0) return ORACLE_ERR_ARG;
    for (int64_t i = 0; i < n; ++i) out[i] = e4m3_code(in[i]);
    return ORACLE_OK;
}

int oracle_e4m3_decode(const uint8_t* in, int64_t n, float* out) {
    if (n < 0) return ORACLE_ERR_ARG;
    for (int64_t i = 0; i < n; ++i) out[i] = e4m3_value(in[i]);
    return ORACLE_OK;
}

/* One scale per row: amax = max_k |x[k]|, s = amax / 448, q[k] = code(x[k] / s). */
static void quantize_row_fp8(const float* x, int64_t K, uint8_t* q, float* s_out) {
    float amax = 0.0f;
    for (int64_t k = 0; k < K; ++k) {
        float a = fabsf(x[k]);
        if (a > amax) amax = a;
    }
    float s = amax / 448.0f;
    *s_out = s;
    for (int64_t k = 0; k < K; ++k) q[k] = (s == 0.0f) ? 0 : e4m3_code(x[k] / s);
}

int oracle_quantize_rows_fp8(const float* x, int64_t rows, int64_t K, uint8_t* q, float* s) {
    if (rows < 0 || K <= 0) return ORACLE_ERR_ARG;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) quantize_row_fp8(x + r * K, K, q + r * K, s + r);
    return ORACLE_OK;
}

int oracle_quantize_rows_bf16_fp8(const uint16_t* x, int64_t rows, int64_t K, uint8_t* q, float* s) {
    if (rows < 0 || K <= 0) return ORACLE_ERR_ARG;
    int err = 0;
#pragma omp parallel
    {
        float* row = (float*)malloc((size_t)K * sizeof(float));
        if (!row) {
#pragma omp atomic write
            err = 1;
        }
#pragma omp for schedule(static)
        for (int64_t r = 0; r < rows; ++r) {
            if (!row) continue;
            for (int64_t k = 0; k < K; ++k) row[k] = bf16_to_f32(x[r * K + k]);
            quantize_row_fp8(row, K, q + r * K, s + r);
        }
        free(row);
    }
    return err ? ORACLE_ERR_NOMEM : ORACLE_OK;
}

/* acc[m][n] = binary32( sum_k value(a[m][k]) * value(b[n][k]) ), the sum exact
 * in binary64 (K < 2^17); a [M][K], b [N][K] (both K-contiguous). */
int oracle_gemm_fp8(const uint8_t* a, const uint8_t* b, int64_t M, int64_t N, int64_t K, float* acc) {
    if (M < 0 || N < 0 || K <= 0 || K >= (1 << 17)) return ORACLE_ERR_ARG;
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            double sum = 0.0;
            for (int64_t k = 0; k < K; ++k)
                sum += (double)e4m3_value(a[m * K + k]) * (double)e4m3_value(b[n * K + k]);
            acc[m * N + n] = (float)sum;
        }
    }
    return ORACLE_OK;
}

/* The epilogues of the FP8 layer: those of the INT8 layer on a binary32
 * accumulator, value = (acc * s_act) * s_w. */
static float dequant_f(float acc, float s_act, float s_w) {
    float v = acc * s_act;
    v = v * s_w;
    return v;
}

int oracle_epilogue_gate_up_f32(const float* acc1, const float* s_act, const float* s_w13, int64_t S,
                                int64_t I, float* h) {
    if (S < 0 || I <= 0) return ORACLE_ERR_ARG;
#pragma omp parallel for schedule(static)
    for (int64_t s = 0; s < S; ++s) {
        for (int64_t n = 0; n < I; ++n) {
            float g = dequant_f(acc1[s * 2 * I + n], s_act[s], s_w13[n]);
            float u = dequant_f(acc1[s * 2 * I + I + n], s_act[s], s_w13[I + n]);
            h[s * I + n] = silu(g) * u;
        }
    }
    return ORACLE_OK;
}

int oracle_epilogue_scale_f32(const float* acc, const float* s_act, const float* s_w, int64_t S, int64_t N,
                              float* out) {
    if (S < 0 || N <= 0) return ORACLE_ERR_ARG;
#pragma omp parallel for schedule(static)
    for (int64_t s = 0; s < S; ++s)
        for (int64_t c = 0; c < N; ++c) out[s * N + c] = dequant_f(acc[s * N + c], s_act[s], s_w[c]);
    return ORACLE_OK;
}

/* The whole FP8 layer, sparse path: the INT8 layer's steps with the E4M3
 * quantisers and GEMMs.  w13_q E4M3 [E][2I][H], w2_q E4M3 [E][H][I]; the dump
 * fields q_x and q_h receive E4M3 codes, acc1 and acc2 binary32 values (as
 * their bit patterns in the int32 fields). */
int oracle_moe_forward_fp8(const uint16_t* x, const float* Wr, const float* bias, const uint8_t* w13_q,
                           const float* s_w13, const uint8_t* w2_q, const float* s_w2, int64_t T, int64_t H,
                           int64_t I, int64_t E, int64_t k, uint16_t* y, const oracle_dump_t* dump) {
    if (T < 0 || H <= 0 || I <= 0 || E <= 0 || k <= 0 || k > E) return ORACLE_ERR_ARG;
    const int64_t S = T * k;
    int rc = ORACLE_OK;
    int32_t* topk_ids = (int32_t*)xmalloc((size_t)S * 4);
    float* topk_w = (float*)xmalloc((size_t)S * 4);
    int32_t* counts = (int32_t*)xmalloc((size_t)E * 4);
    int32_t* offsets = (int32_t*)xmalloc((size_t)(E + 1) * 4);
    int32_t* slot_of = (int32_t*)xmalloc((size_t)S * 4);
    int32_t* slot_token = (int32_t*)xmalloc((size_t)S * 4);
    float* s_x = (float*)xmalloc((size_t)T * 4);
    uint8_t* q_x = (uint8_t*)xmalloc((size_t)(T * H));
    float* s_slot = (float*)xmalloc((size_t)S * 4);
    uint8_t* q_slot = (uint8_t*)xmalloc((size_t)(S * H));
    float* acc1 = (float*)xmalloc((size_t)(S * 2 * I) * 4);
    float* h = (float*)xmalloc((size_t)(S * I) * 4);
    float* s_h = (float*)xmalloc((size_t)S * 4);
    uint8_t* q_h = (uint8_t*)xmalloc((size_t)(S * I));
    float* acc2 = (float*)xmalloc((size_t)(S * H) * 4);
    float* o = (float*)xmalloc((size_t)(S * H) * 4);
    if (!topk_ids || !topk_w || !counts || !offsets || !slot_of || !slot_token || !s_x || !q_x ||
        !s_slot || !q_slot || !acc1 || !h || !s_h || !q_h || !acc2 || !o) {
        rc = ORACLE_ERR_NOMEM;
        goto done;
    }
    rc = oracle_router(x, Wr, bias, T, H, E, k, topk_ids, topk_w, NULL);
    if (rc) goto done;
    rc = oracle_permute(topk_ids, T, E, k, counts, offsets, slot_of, slot_token);
    if (rc) goto done;
    rc = oracle_quantize_rows_bf16_fp8(x, T, H, q_x, s_x);
    if (rc) goto done;
    for (int64_t s = 0; s < S; ++s) {  /* each slot holds its token's codes and scale */
        memcpy(q_slot + s * H, q_x + (int64_t)slot_token[s] * H, (size_t)H);
        s_slot[s] = s_x[slot_token[s]];
    }
    for (int64_t e = 0; e < E; ++e) {
        int64_t s0 = offsets[e], n = offsets[e + 1] - offsets[e];
        if (n == 0) continue;
        rc = oracle_gemm_fp8(q_slot + s0 * H, w13_q + e * 2 * I * H, n, 2 * I, H, acc1 + s0 * 2 * I);
        if (rc) goto done;
        rc = oracle_epilogue_gate_up_f32(acc1 + s0 * 2 * I, s_slot + s0, s_w13 + e * 2 * I, n, I, h + s0 * I);
        if (rc) goto done;
        rc = oracle_quantize_rows_fp8(h + s0 * I, n, I, q_h + s0 * I, s_h + s0);
        if (rc) goto done;
        rc = oracle_gemm_fp8(q_h + s0 * I, w2_q + e * H * I, n, H, I, acc2 + s0 * H);
        if (rc) goto done;
        rc = oracle_epilogue_scale_f32(acc2 + s0 * H, s_h + s0, s_w2 + e * H, n, H, o + s0 * H);
        if (rc) goto done;
    }
    rc = oracle_combine(o, slot_of, topk_w, T, k, H, y);
    if (rc) goto done;
    if (dump) {
        if (dump->topk_ids) memcpy(dump->topk_ids, topk_ids, (size_t)S * 4);
        if (dump->topk_w) memcpy(dump->topk_w, topk_w, (size_t)S * 4);
        if (dump->offsets) memcpy(dump->offsets, offsets, (size_t)(E + 1) * 4);
        if (dump->slot_of) memcpy(dump->slot_of, slot_of, (size_t)S * 4);
        if (dump->slot_token) memcpy(dump->slot_token, slot_token, (size_t)S * 4);
        if (dump->s_x) memcpy(dump->s_x, s_x, (size_t)T * 4);
        if (dump->q_x) memcpy(dump->q_x, q_x, (size_t)(T * H));
        if (dump->acc1) memcpy(dump->acc1, acc1, (size_t)(S * 2 * I) * 4);
        if (dump->h) memcpy(dump->h, h, (size_t)(S * I) * 4);
        if (dump->s_h) memcpy(dump->s_h, s_h, (size_t)S * 4);
        if (dump->q_h) memcpy(dump->q_h, q_h, (size_t)(S * I));
        if (dump->acc2) memcpy(dump->acc2, acc2, (size_t)(S * H) * 4);
        if (dump->o) memcpy(dump->o, o, (size_t)(S * H) * 4);
    }
done:
    free(topk_ids); free(topk_w); free(counts); free(offsets); free(slot_of); free(slot_token);
    free(s_x); free(q_x); free(s_slot); free(q_slot); free(acc1); free(h); free(s_h); free(q_h);
    free(acc2); free(o);
    return rc;
}

/* ==== SmoothQuant-folded activations, calibrated per expert ================
 * "W8A8 quantisation of MiniMax-M3 on K100AI" (mhpn.cn), section 2.2: the
 * activations are hard to quantise because a few channels hold large values;
 * a per-channel factor moves part of that difficulty onto the weights (the
 * activation channel is scaled down, the weights' input channel up by the
 * same factor, which leaves x W^T unchanged in exact arithmetic), with alpha
 * setting the balance and the statistics gathered per expert (each expert's
 * calibration tokens are those the router sends to it).
 * Readings (listed in the design notes): the factor s_e[h] of expert e and
 * channel h follows SmoothQuant's balance
 *     s = max|X_e[:,h]|^alpha / max|W_e[:,h]|^(1 - alpha)
 * (binary64 powers, rounded once to binary32; a channel whose activation or
 * weight statistic is 0 gets s = 1); the folded weight is w[n][h] * s[h] (one
 * binary32 multiply) before the per-channel quantiser; the activation of a
 * slot of expert e is x[t][h] * (1 / s_e[h]) with 1 / s the correctly
 * rounded binary32 reciprocal (one multiply), quantised per slot.  The page's
 * alpha sweep on calibration data and its percentile statistics need data
 * this project does not have.
 */
int oracle_smooth_factors(const float* x_absmax, const float* w_absmax, int64_t n, double alpha, float* s) {
    if (n < 0 || alpha < 0.0 || alpha > 1.0) return ORACLE_ERR_ARG;
    for (int64_t i = 0; i < n; ++i) {
        double a = x_absmax[i], b = w_absmax[i];
        s[i] = (a > 0.0 && b > 0.0) ? (float)(pow(a, alpha) / pow(b, 1.0 - alpha)) : 1.0f;
    }
    return ORACLE_OK;
}

/* Per-output-channel quantisation of the folded weights w[r][k] * s[k]. */
int oracle_quantize_rows_smoothed(const float* w, const float* s, int64_t rows, int64_t K, int8_t* q,
                                  float* scale) {
    if (rows < 0 || K <= 0) return ORACLE_ERR_ARG;
    int err = 0;
#pragma omp parallel
    {
        float* row = (float*)malloc((size_t)K * sizeof(float));
        if (!row) {
#pragma omp atomic write
            err = 1;
        }
#pragma omp for schedule(static)
        for (int64_t r = 0; r < rows; ++r) {
            if (!row) continue;
            for (int64_t k = 0; k < K; ++k) row[k] = w[r * K + k] * s[k];
            quantize_row(row, K, q + r * K, scale + r);
        }
        free(row);
    }
    return err ? ORACLE_ERR_NOMEM : ORACLE_OK;
}

/* One activation row smoothed by one expert's factors, then quantised. */
static void quantize_row_bf16_smoothed(const uint16_t* x, const float* sm, int64_t H, float* tmp, int8_t* q,
                                       float* s_out) {
    for (int64_t h = 0; h < H; ++h) {
        float r = 1.0f / sm[h];
        tmp[h] = bf16_to_f32(x[h]) * r;
    }
    quantize_row(tmp, H, q, s_out);
}

/* The layer with per-expert smoothing factors smooth [E][H] and w13_q folded
 * with them; s_slot [S] and q_slot [S][H] (optional) receive each slot's
 * scale and codes.  Everything else is the sparse layer above. */
int oracle_moe_forward_smooth(const uint16_t* x, const float* Wr, const float* bias, const float* smooth,
                              const int8_t* w13_q, const float* s_w13, const int8_t* w2_q, const float* s_w2,
                              int64_t T, int64_t H, int64_t I, int64_t E, int64_t k, uint16_t* y,
                              const oracle_dump_t* dump, float* s_slot, int8_t* q_slot) {
    if (!smooth) return ORACLE_ERR_ARG;
    return moe_forward_impl(x, Wr, bias, smooth, w13_q, s_w13, w2_q, s_w2, T, H, I, E, k, y, dump, s_slot,
                            q_slot);
}

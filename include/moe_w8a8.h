/*
 * moe_w8a8.h -- C ABI of the W8A8 quantised mixture-of-experts layer for
 * NVIDIA GB300 (sm_103a).
 *
 * The layer (one MoE feed-forward block of an LLM, serving-time forward):
 *
 *   router logits  l[t][e] = sum_h x[t][h] * Wr[h][e] (+ bias[e]), FP32
 *   top-k          k largest logits per token (ties -> lower expert index),
 *                  weights w = softmax over the selected logits
 *   permutation    every (token, choice) gets a slot; expert e owns the
 *                  contiguous slots [offsets[e], offsets[e+1]), tokens in
 *                  ascending order
 *   quantise       per token: s_x = amax_h |x| / 127,
 *                  q_x = clamp(round_half_even(x / s_x), -128, 127)
 *   GEMM1          acc1[s][n] = sum_h q_x[t(s)][h] * w13_q[e(s)][n][h]  (exact int32)
 *   epilogue 1     g = (acc1[s][n] * s_x) * s_w13[e][n], u likewise at n + I,
 *                  h = silu(g) * u = (g / (1 + exp(-g))) * u           (FP32)
 *   requantise     per slot: s_h = amax_n |h| / 127, q_h = round(h / s_h)
 *   GEMM2          acc2[s][c] = sum_n q_h[s][n] * w2_q[e(s)][c][n]      (exact int32)
 *   epilogue 2     o[s][c] = (acc2[s][c] * s_h[s]) * s_w2[e][c]         (FP32)
 *   combine        y[t][c] = bf16_rne(sum_j w[t][j] * o[slot(t, j)][c])
 *
 * Sources: the quantisation formula, per-channel weight scales, per-token
 * dynamic activation scales and the scale outer product applied in the GEMM
 * epilogue -- "W8A8 quantisation of MiniMax-M3 on K100AI" (mhpn.cn), section
 * 2.1; FP32 accumulation with re-quantisation between operators -- "DeepSeek
 * V4 950 FP8 inference on H100" (lpnh.cn), section 2.3; the FP32 router --
 * same page, section 4.1; the gate -> top-k -> contiguous per-expert slots
 * -> expert GEMMs -> weighted combine pipeline -- "Tencent Hunyuan AI Infra
 * on Hopper" (pnsm.cn), section 1.3.
 *
 * Conventions for every call
 *   - All data pointers are DEVICE pointers owned by the caller; the library
 *     allocates and frees nothing.  bf16 tensors are passed as uint16_t bit
 *     patterns.  Every pointer must be 16-byte aligned; tensors are dense and
 *     row-major (last index contiguous).
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls
 *     only enqueue work on it and never synchronise, except
 *     moe_w8a8_device_error.
 *   - Arguments are checked on the host before anything is launched; a
 *     failed check returns an error status and launches nothing.
 *   - Calls on different streams are safe when their workspaces differ.
 *   - The calls are deterministic: the same inputs give bit-identical
 *     outputs.
 *   - Fault injection for tests of the error paths: the environment variable
 *     MOE_INJECT (read at every call; a comma-separated list) fakes faults.
 *     On the host, reaching no GPU: "ws_short": the workspace check fails as
 *     if the workspace were one byte short (MOE_ERR_WORKSPACE_TOO_SMALL);
 *     "bad_ptr": the pointer check fails as if a data pointer were null
 *     (MOE_ERR_INVALID_ARG); "launch_fail": every kernel launch fails before
 *     anything is queued (MOE_ERR_CUDA).  On the GPU: "stall": every
 *     tensor-core expert or linear GEMM launch starts with its producer
 *     waiting, within the wait limit (moe_w8a8_set_wait_timeout_ns), on a
 *     barrier that nothing completes, so that the limit runs out and the
 *     kernel takes its abort path (MOE_ERR_DEVICE_TIMEOUT from
 *     moe_w8a8_device_error; outputs undefined).  "bad_slot", honoured only
 *     by the checked build below: after the quantiser the first slot index
 *     is overwritten with an out-of-range value, which the combine's check
 *     reports (MOE_ERR_DEVICE; that token's output undefined).  Unset in
 *     normal use.
 *
 *   Checked build.  Compiled with -DMOE_CHECKED=1 (libmoe_w8a8_checked.so,
 *     `python -m w8a8_quantised_moe_gb300.build --checked`), the kernels
 *     range-check every index they take from data rather than from their
 *     launch shape (expert ids, slots, expert offsets, exact-path lists,
 *     gathered rows).  An index out of range sets the device error word
 *     (MOE_ERR_DEVICE from moe_w8a8_device_error) and the access is skipped,
 *     where the normal build would read or write out of bounds.  The same
 *     entry points and results; a debugging aid, not the fast path.
 */
#ifndef MOE_W8A8_H
#define MOE_W8A8_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_W8A8_API __attribute__((visibility("default")))
#else
#define MOE_W8A8_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = -1,        /* null or misaligned pointer, bad count */
    MOE_ERR_UNSUPPORTED_SHAPE = -2,  /* a dimension outside the supported set */
    MOE_ERR_WORKSPACE_TOO_SMALL = -3,
    MOE_ERR_CUDA = -4,               /* a CUDA runtime call or launch failed */
    MOE_ERR_DEVICE_TIMEOUT = -5,     /* a device-side wait ran out of time */
    MOE_ERR_NOT_IMPLEMENTED = -6,
    MOE_ERR_DEVICE = -7              /* a device-side consistency check failed */
} moe_status_t;

/* Human-readable name of a status code (static string, never NULL). */
MOE_W8A8_API const char* moe_w8a8_status_string(moe_status_t status);

/* Library version as an integer major*10000 + minor*100 + patch. */
MOE_W8A8_API int moe_w8a8_version(void);

/* ---------------------------------------------------------------------------
 * moe_w8a8_quantize_weights -- offline per-output-channel weight quantisation.
 *
 * For each of `rows` rows of length K:  s = max_k |w[k]| / 127 (binary32
 * division), w_q[k] = clamp(round_half_even(w[k] / s), -128, 127); a row of
 * zeros gives s = 0 and codes 0.  Weight scales are per output channel and
 * computed once, offline ("W8A8 quantisation of MiniMax-M3 on K100AI",
 * section 2.1).  Call it once per expert tensor: rows = E * 2I for w13
 * (row order: expert, then gate rows 0..I-1, then up rows I..2I-1) and
 * rows = E * H for w2.
 *
 *   w        fp32 [rows][K]  input
 *   w_q      int8 [rows][K]  output
 *   w_scale  fp32 [rows]     output
 * Requirements: rows >= 0, 1 <= K <= 2^20.  rows == 0 is a no-op.
 * ------------------------------------------------------------------------- */
MOE_W8A8_API moe_status_t moe_w8a8_quantize_weights(const float* w, int64_t rows, int64_t K, int8_t* w_q,
                                       float* w_scale, void* stream);

/* ---------------------------------------------------------------------------
 * Workspace of moe_w8a8_forward / moe_w8a8_forward_debug, in bytes, for the
 * given shape.  Returns 0 for shapes the forward rejects.  The workspace is
 * caller-owned device memory (256-byte aligned) that the forward uses for
 * its intermediates (routing tables, quantised activations, the FP32 gate/up
 * output, its requantised form and the per-slot expert outputs).  Its first
 * 256 bytes hold the sticky device error word read by moe_w8a8_device_error
 * and a routing counter that every call leaves at zero; zero them once before
 * the first call on a new workspace.  Calls that share a workspace must not
 * overlap on the GPU.
 * ------------------------------------------------------------------------- */
MOE_W8A8_API size_t moe_w8a8_workspace_size(int64_t T, int64_t H, int64_t I, int64_t E, int64_t top_k);

/* ---------------------------------------------------------------------------
 * moe_w8a8_forward -- the whole MoE layer (see the top of this file).
 *
 *   x           bf16 [T][H]       activations
 *   router_w    fp32 [H][E]       router weights (never quantised)
 *   router_bias fp32 [E] or NULL  added to the logits before top-k
 *   w13_q       int8 [E][2I][H]   gate rows 0..I-1 then up rows I..2I-1
 *   w13_scale   fp32 [E][2I]
 *   w2_q        int8 [E][H][I]    down projection
 *   w2_scale    fp32 [E][H]
 *   y           bf16 [T][H]       output
 *   workspace   >= moe_w8a8_workspace_size(T, H, I, E, top_k) bytes
 *
 * Supported shapes: 0 <= T <= 2^20; H and I multiples of 128 with
 * 128 <= H, I <= 16384; 1 <= E <= 256; 1 <= top_k <= min(E, 8).  T == 0 is a
 * no-op that reads no pointer (NULL is accepted).  Integer results (routing, quantised codes, int32 accumulators)
 * are exact; the router's binary32 sums can order two logits differently
 * from an exact evaluation only when they differ by less than about 1e-6.
 * Errors: MOE_ERR_INVALID_ARG (null/misaligned pointer), _UNSUPPORTED_SHAPE,
 * _WORKSPACE_TOO_SMALL, _CUDA (launch failure).  Device-side timeouts are
 * reported later through moe_w8a8_device_error.
 * Launches: all on `stream`, no host synchronisation.  Every kernel after
 * the first is launched with programmatic dependent launch (its set-up
 * overlaps the previous kernel's tail; it reads nothing before that kernel
 * has completed); the first serialises with earlier work on the stream as a
 * plain launch does.  MOE_W8A8_NO_PDL=1 in the environment turns this off.
 * ------------------------------------------------------------------------- */
MOE_W8A8_API moe_status_t moe_w8a8_forward(const uint16_t* x, const float* router_w, const float* router_bias,
                              const int8_t* w13_q, const float* w13_scale, const int8_t* w2_q,
                              const float* w2_scale, int64_t T, int64_t H, int64_t I, int64_t E,
                              int64_t top_k, uint16_t* y, void* workspace, size_t workspace_bytes,
                              void* stream);

/* Device buffers that moe_w8a8_forward_debug fills with the intermediates
 * (S = T * top_k).  Any field may be NULL (skipped).  The raw accumulators
 * cost a full extra GEMM output each; use them on small shapes. */
typedef struct {
    int32_t* topk_ids;    /* [T][top_k]  selected experts, descending logit */
    float* topk_w;        /* [T][top_k]  their weights */
    int32_t* offsets;     /* [E+1]       slot offsets per expert */
    int32_t* slot_of;     /* [T][top_k]  slot of each (token, choice) */
    int32_t* slot_token;  /* [S]         token held by each slot */
    float* s_x;           /* [T]         activation scales */
    int8_t* q_x;          /* [T][H]      quantised activations */
    int32_t* acc1;        /* [S][2I]     GEMM1 accumulators (gate | up) */
    float* h;             /* [S][I]      FP32 gate/up output */
    float* s_h;           /* [S]         requantisation scales */
    int8_t* q_h;          /* [S][I]      requantised h */
    int32_t* acc2;        /* [S][H]      GEMM2 accumulators */
    float* o;             /* [S][H]      per-slot expert outputs */
    float* s_slot;        /* [S]         activation scale of each slot */
    int8_t* q_slot;       /* [S][H]      quantised activation row of each slot */
} moe_w8a8_debug_t;

/* moe_w8a8_forward plus copies of the intermediates into `dbg` (same
 * arguments and errors; `dbg` may be NULL). */
MOE_W8A8_API moe_status_t moe_w8a8_forward_debug(const uint16_t* x, const float* router_w,
                                    const float* router_bias, const int8_t* w13_q,
                                    const float* w13_scale, const int8_t* w2_q,
                                    const float* w2_scale, int64_t T, int64_t H, int64_t I,
                                    int64_t E, int64_t top_k, uint16_t* y, void* workspace,
                                    size_t workspace_bytes, void* stream,
                                    const moe_w8a8_debug_t* dbg);

/* ---------------------------------------------------------------------------
 * moe_w8a8_forward_fused -- the same layer for few tokens as ONE persistent
 * kernel ("Tencent Hunyuan AI Infra on Hopper", section 1.3: gate, top-k,
 * routing pre-processing, both expert GEMMs and the weighted aggregation in
 * one fused operator).  Router, top-k and routing tables, per-token
 * quantisation, gate/up GEMM with its epilogue, requantisation, down GEMM and
 * combine run as phases of one cooperative launch separated by grid-wide
 * barriers, with the arithmetic of moe_w8a8_forward: y and every
 * intermediate equal moe_w8a8_forward's bit for bit.
 *
 * Arguments, workspace (moe_w8a8_workspace_size) and errors as
 * moe_w8a8_forward_debug; `dbg` may be NULL.  Shapes: those of
 * moe_w8a8_forward with T <= 128 (moe_w8a8_fused_supported returns 1); others
 * return MOE_ERR_UNSUPPORTED_SHAPE.  One launch on `stream` (plus the copies into
 * `dbg`); it occupies every SM until it ends.  Every barrier wait is bounded
 * by moe_w8a8_set_wait_timeout_ns: one that runs out makes every CTA skip the
 * remaining phases (y is then undefined) and is reported by
 * moe_w8a8_device_error as MOE_ERR_DEVICE_TIMEOUT.  MOE_INJECT=stall makes
 * one CTA skip a barrier arrival, so that the limit runs out.
 * ------------------------------------------------------------------------- */
MOE_W8A8_API moe_status_t moe_w8a8_forward_fused(const uint16_t* x, const float* router_w,
                                    const float* router_bias, const int8_t* w13_q,
                                    const float* w13_scale, const int8_t* w2_q,
                                    const float* w2_scale, int64_t T, int64_t H, int64_t I,
                                    int64_t E, int64_t top_k, uint16_t* y, void* workspace,
                                    size_t workspace_bytes, void* stream,
                                    const moe_w8a8_debug_t* dbg);

/* 1 if moe_w8a8_forward_fused takes the shape, else 0. */
MOE_W8A8_API int moe_w8a8_fused_supported(int64_t T, int64_t H, int64_t I, int64_t E, int64_t top_k);

/* ---------------------------------------------------------------------------
 * moe_w8a8_linear -- one W8A8 linear layer, the dense form of the expert
 * GEMM: per-token dynamic quantisation of x, exact INT8 GEMM, and the
 * per-token x per-channel scale outer product in the epilogue
 * ("W8A8 quantisation of MiniMax-M3 on K100AI", section 2.1):
 *   y[m][n] = bf16_rne((acc[m][n] * s_x[m]) * w_scale[n]).
 *
 *   x        bf16 [M][K]
 *   w_q      int8 [N][K]     per-output-channel quantised weights
 *   w_scale  fp32 [N]
 *   y        bf16 [M][N]
 *   workspace >= moe_w8a8_linear_workspace_size(M, N, K) bytes
 * Supported: 0 <= M <= 2^20; N, K multiples of 128 in [128, 65536].  M == 0
 * is a no-op that reads no pointer.
 * ------------------------------------------------------------------------- */
MOE_W8A8_API size_t moe_w8a8_linear_workspace_size(int64_t M, int64_t N, int64_t K);
MOE_W8A8_API moe_status_t moe_w8a8_linear(const uint16_t* x, const int8_t* w_q, const float* w_scale, int64_t M,
                             int64_t N, int64_t K, uint16_t* y, void* workspace,
                             size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * moe_w8a8_linear_static -- moe_w8a8_linear for callers that cannot
 * allocate device memory.  The method's pages have no counterpart to it.
 *
 * Some callers cannot allocate when they run the layer: a plugin whose host
 * framework gives it no allocator, or a serving loop that reserved all
 * device memory for its own pool at start-up (a fresh cudaMalloc would fail,
 * fragment the pool, or synchronise the device).  This entry point needs no
 * workspace and allocates nothing, neither itself nor through a library
 * routine: its scratch is a static device array of 8 MiB inside the library,
 * which every GPU that loads the library holds until the process exits.
 *
 *   x, w_q, w_scale, y, M, N, K, stream: as for moe_w8a8_linear; the caller
 *   still provides the inputs and the output.
 * Limit: the scratch of a call, moe_w8a8_linear_workspace_size(M, N, K)
 *   bytes (about 2*M*K + 12*M + 1 KiB; e.g. up to 1022 tokens at K = 4096), must
 *   fit the 8 MiB; a larger shape is rejected with MOE_ERR_UNSUPPORTED_SHAPE
 *   before anything is launched.
 * Set-up: the first call on each device looks up that device's address of
 *   the array (with the device current) and caches it; make that first call
 *   before any stream capture.  The cached address belongs to the device's
 *   primary context: after cudaDeviceReset (or anything else that destroys
 *   that context) this entry point must not be called again in the process.
 * Sharing: every call on a device uses the same array, which keeps the last
 *   call's contents (the call clears what must start at zero).  Calls that
 *   overlap on the GPU -- on different streams, or from several host threads
 *   -- race on the array and give undefined results; serialise them.
 * Waits: the kernels' spin-waits use the limit of
 *   moe_w8a8_set_wait_timeout_ns, like every other entry point.
 * Errors: as moe_w8a8_linear.  A device-side timeout sets the array's own
 *   sticky error word (the output is then undefined); read it with
 *   moe_w8a8_linear_static_error.
 * ------------------------------------------------------------------------- */
MOE_W8A8_API moe_status_t moe_w8a8_linear_static(const uint16_t* x, const int8_t* w_q, const float* w_scale,
                                                 int64_t M, int64_t N, int64_t K, uint16_t* y, void* stream);

/* moe_w8a8_linear_static_error -- synchronise `stream`, then read and clear
 * the sticky device error word of moe_w8a8_linear_static's static scratch on
 * the current device (set by any earlier call on that device since it was
 * last read).  Returns MOE_OK, MOE_ERR_DEVICE_TIMEOUT, MOE_ERR_DEVICE, or
 * MOE_ERR_CUDA if the synchronisation or the read failed.  Allocates
 * nothing; like the entry point, it must not overlap a call on the GPU. */
MOE_W8A8_API moe_status_t moe_w8a8_linear_static_error(void* stream);

/* ---------------------------------------------------------------------------
 * The FP8 (E4M3) layer.  "DeepSeek V4 950 FP8 inference on H100" (lpnh.cn):
 * weights and activations in E4M3 (section 2.1), FP8 operands with an FP32
 * accumulator whose result is re-quantised to FP8 for the next operator
 * (2.3), per-channel weight scales and per-token dynamic activation scales
 * (2.4), weight scales from the absolute maximum (3.1).  A row's scale is
 * s = amax / 448 (binary32 division) and its codes are the E4M3 values
 * nearest to the binary32 quotients x / s, ties to even, saturated at +-448;
 * a row of zeros gives s = 0 and codes 0.  E4M3 codes are bytes (sign bit 7,
 * exponent bits 6..3 with bias 7, mantissa bits 2..0).
 *
 * moe_w8a8_fp8_quantize_weights: the weight quantiser.  w fp32 [rows][K]
 * (K a multiple of 4), w_q E4M3 [rows][K], w_scale fp32 [rows]; call it once
 * per expert tensor as moe_w8a8_quantize_weights.  Errors as that function.
 * ------------------------------------------------------------------------- */
MOE_W8A8_API moe_status_t moe_w8a8_fp8_quantize_weights(const float* w, int64_t rows, int64_t K, uint8_t* w_q,
                                                        float* w_scale, void* stream);

/* moe_w8a8_fp8_forward: the whole FP8 layer.  Arguments, shapes, workspace
 * (moe_w8a8_workspace_size), launches and errors as moe_w8a8_forward, with
 * w13_q and w2_q holding E4M3 codes.  Router, top-k, slots, SiLU gate and
 * combine are those of the INT8 layer; the expert GEMMs run on the
 * tcgen05.mma kind::f8f6f4 tensor cores.  The E4M3 products are exact and
 * their sum is an fp32 accumulation, so the GEMM results agree with the
 * exact dot product within fp32 accumulation error (not bit for bit). */
MOE_W8A8_API moe_status_t moe_w8a8_fp8_forward(const uint16_t* x, const float* router_w, const float* router_bias,
                                               const uint8_t* w13_q, const float* w13_scale, const uint8_t* w2_q,
                                               const float* w2_scale, int64_t T, int64_t H, int64_t I, int64_t E,
                                               int64_t top_k, uint16_t* y, void* workspace, size_t workspace_bytes,
                                               void* stream);

/* moe_w8a8_fp8_forward plus copies of the intermediates into `dbg`, as
 * moe_w8a8_forward_debug; q_x and q_h receive E4M3 codes and acc1, acc2 the
 * fp32 accumulators (their bit patterns in the int32 fields). */
MOE_W8A8_API moe_status_t moe_w8a8_fp8_forward_debug(const uint16_t* x, const float* router_w,
                                                     const float* router_bias, const uint8_t* w13_q,
                                                     const float* w13_scale, const uint8_t* w2_q,
                                                     const float* w2_scale, int64_t T, int64_t H, int64_t I,
                                                     int64_t E, int64_t top_k, uint16_t* y, void* workspace,
                                                     size_t workspace_bytes, void* stream,
                                                     const moe_w8a8_debug_t* dbg);

/* ---------------------------------------------------------------------------
 * SmoothQuant-folded activations, calibrated per expert ("W8A8 quantisation
 * of MiniMax-M3 on K100AI", section 2.2: part of the activations'
 * quantisation difficulty is moved onto the weights by a per-channel factor,
 * with statistics gathered per expert).  A factor s_e[h] > 0 per expert e and
 * hidden channel h multiplies the weights' input channel h and divides the
 * activation's channel h; the two cancel in exact arithmetic.
 *
 * moe_w8a8_quantize_weights_smoothed -- moe_w8a8_quantize_weights of the
 * rows w[r][k] * col_scale[k] (one binary32 multiply per element): call it
 * once per expert on its w13 rows [2I][H] with col_scale = s_e [H].  (w2 is
 * quantised as before: the factors act on GEMM1's input only.)
 *   col_scale  fp32 [K], device, 16-byte aligned
 * Errors: as moe_w8a8_quantize_weights; col_scale NULL -> INVALID_ARG.
 *
 * moe_w8a8_forward_smooth -- moe_w8a8_forward with the activation of each
 * (token, expert) slot taken as x[t][h] * rcp(s_e[h]) (rcp: the correctly
 * rounded binary32 reciprocal; one binary32 multiply) and quantised per slot
 * (amax over the slot's row, s = amax / 127), since the row now depends on the
 * expert.  The weights must have been folded with the same factors.
 *   smooth     fp32 [E][H], device, 16-byte aligned, every factor > 0 and
 *              finite (not checked)
 *   dbg        may be NULL; as moe_w8a8_forward_debug, with s_x[t] the scale
 *              of the token's first choice and q_x[t] its first slot's row
 * Errors: as moe_w8a8_forward; smooth NULL (T > 0) or misaligned ->
 * MOE_ERR_INVALID_ARG.  INT8 layer only.
 * ------------------------------------------------------------------------- */
MOE_W8A8_API moe_status_t moe_w8a8_quantize_weights_smoothed(const float* w, int64_t rows, int64_t K,
                                                             const float* col_scale, int8_t* w_q, float* w_scale,
                                                             void* stream);
MOE_W8A8_API moe_status_t moe_w8a8_forward_smooth(const uint16_t* x, const float* router_w,
                                                  const float* router_bias, const float* smooth,
                                                  const int8_t* w13_q, const float* w13_scale, const int8_t* w2_q,
                                                  const float* w2_scale, int64_t T, int64_t H, int64_t I, int64_t E,
                                                  int64_t top_k, uint16_t* y, void* workspace,
                                                  size_t workspace_bytes, void* stream, const moe_w8a8_debug_t* dbg);

/* ---------------------------------------------------------------------------
 * moe_w8a8_forward_host -- moe_w8a8_forward for activations that live in
 * host memory: x is copied in and y copied out inside the call, in token
 * chunks, so that the copies of one chunk overlap the layer's compute on
 * another.  The method's pages have no counterpart to it: it is the layer of
 * moe_w8a8_forward ("Tencent Hunyuan AI Infra on Hopper", section 1.3, and
 * "W8A8 quantisation of MiniMax-M3 on K100AI", section 2.1) applied to each
 * chunk of tokens, tokens being independent in the layer.
 *
 *   x_host      bf16 [T][H]  host memory, page-locked (cudaHostAlloc or
 *                            cudaHostRegister) for the copies to overlap
 *   y_host      bf16 [T][H]  host memory (output), page-locked likewise
 *   x_dev       bf16 [T][H]  device staging for x (caller-owned)
 *   y_dev       bf16 [T][H]  device staging for y (caller-owned)
 *   other arguments as moe_w8a8_forward; the workspace is sized for T
 *   copy_stream a second stream for the copies, or NULL (copies then go on
 *               `stream`, in order with the compute: nothing overlaps); with
 *               one chunk the copies go on `stream` in any case
 *   chunks      0: the library chooses (moe_w8a8_host_chunks); 1..16: that
 *               many chunks of near-equal token counts
 *
 * Measured on GB300 (prefill layer, T = 8192, H = 4096, 64 experts): the host
 * link moves ~200 GB/s each way, so x in and y out take about as long as the
 * layer; two chunks overlap them but make the two half-size layers cost 1.4x
 * the whole one, a net gain of 3 % (INT8) to 7 % (FP8); more chunks lose.
 *
 * Each chunk is a complete forward of its tokens: its result equals
 * moe_w8a8_forward on those tokens bit for bit, and with one chunk it equals
 * moe_w8a8_forward on the batch.  Over several chunks, the router's binary32
 * sums may associate differently than for the whole batch (the router's
 * partition of the hidden dimension depends on the token count), so a token
 * can differ from the whole-batch call only as two evaluations of the layer
 * within its stated accuracy can.  Every chunk re-reads the weights of the
 * experts its tokens touch.
 * Ordering: the copies wait for work queued on `stream` before the call (the
 * staging buffers are free), and work queued on `stream` after the call waits
 * for the last copy of y: synchronising `stream` makes y_host complete.
 * No host synchronisation.  Creates a few CUDA events once per host thread
 * (kept for the life of the process); allocates no memory.
 * Errors: as moe_w8a8_forward, checked before anything is queued, plus
 * MOE_ERR_INVALID_ARG for chunks outside 0..16 or a null/misaligned staging
 * or host pointer; MOE_ERR_CUDA for a failed copy, event or launch.
 * ------------------------------------------------------------------------- */
MOE_W8A8_API moe_status_t moe_w8a8_forward_host(const uint16_t* x_host, const float* router_w,
                                                const float* router_bias, const int8_t* w13_q,
                                                const float* w13_scale, const int8_t* w2_q, const float* w2_scale,
                                                int64_t T, int64_t H, int64_t I, int64_t E, int64_t top_k,
                                                uint16_t* y_host, uint16_t* x_dev, uint16_t* y_dev,
                                                void* workspace, size_t workspace_bytes, void* stream,
                                                void* copy_stream, int chunks);

/* moe_w8a8_forward_host for the FP8 (E4M3) layer of moe_w8a8_fp8_forward. */
MOE_W8A8_API moe_status_t moe_w8a8_fp8_forward_host(const uint16_t* x_host, const float* router_w,
                                                    const float* router_bias, const uint8_t* w13_q,
                                                    const float* w13_scale, const uint8_t* w2_q,
                                                    const float* w2_scale, int64_t T, int64_t H, int64_t I,
                                                    int64_t E, int64_t top_k, uint16_t* y_host, uint16_t* x_dev,
                                                    uint16_t* y_dev, void* workspace, size_t workspace_bytes,
                                                    void* stream, void* copy_stream, int chunks);

/* The number of chunks moe_w8a8_forward_host takes for chunks == 0: two when
 * T >= 2048 and one direction of the host link (about 200 GB/s on GB300)
 * moves x more slowly than HBM (about 6.6 TB/s) streams every expert's
 * weights once, i.e. when T * H * 2 * 32 > E * 3 * H * I bytes; else one.
 * 0 for T < 0. */
MOE_W8A8_API int moe_w8a8_host_chunks(int64_t T, int64_t H, int64_t I, int64_t E);

/* ---------------------------------------------------------------------------
 * moe_w8a8_device_error -- synchronise `stream`, then read and clear the
 * sticky device error word in the first bytes of `workspace`.  Returns
 * MOE_OK, MOE_ERR_DEVICE_TIMEOUT (a pipeline wait inside a kernel gave up;
 * the kernel released its resources and returned, its outputs are
 * undefined), MOE_ERR_DEVICE (an internal consistency check failed) or
 * MOE_ERR_CUDA (the synchronisation itself failed).
 * ------------------------------------------------------------------------- */
MOE_W8A8_API moe_status_t moe_w8a8_device_error(void* workspace, void* stream);

/* ---------------------------------------------------------------------------
 * moe_w8a8_set_wait_timeout_ns -- time limit of every spin-wait inside the
 * kernels launched after this call (process-wide; default 2e9 ns = 2 s).
 * A wait that runs out sets the device error word, abandons the kernel's
 * remaining work, drains the copies it has in flight and returns.  Returns
 * the previous limit.  0 restores the default.
 * ------------------------------------------------------------------------- */
MOE_W8A8_API uint64_t moe_w8a8_set_wait_timeout_ns(uint64_t ns);

/* ---------------------------------------------------------------------------
 * moe_w8a8_set_gemm_path -- test hook: force the kernel of every expert GEMM
 * and linear GEMM launched after this call (process-wide).  -1 (the default)
 * chooses by the average rows per group; 0, 1, 2 force the one-CTA
 * tensor-core kernel with 160-, 128- or 32-row tiles, 3 the CTA-pair
 * tensor-core kernel (the 160-row kernel where the channel blocks do not
 * pair up), 4 the CUDA-core dp4a kernel for groups of a few rows (the
 * automatic choice where its shape rule fails: K a multiple of 128 and at
 * most 28672, output channels a multiple of 16 for the gate/up GEMM and of
 * 64 otherwise).  Every path computes the same bits.  Returns the previous
 * setting, or -2 (and changes nothing) for a value outside [-1, 4].  The
 * FP8 layer has kernels of its own: while a path is forced, its entry points
 * return MOE_ERR_NOT_IMPLEMENTED and launch nothing.
 * ------------------------------------------------------------------------- */
MOE_W8A8_API int moe_w8a8_set_gemm_path(int path);

/* ---------------------------------------------------------------------------
 * moe_w8a8_set_profile_events -- measurement hook.  While set (on the calling
 * host thread), every moe_w8a8_forward records events[i] on its stream right
 * before its i-th kernel launch (0 router/top-k, 1 scan, 2 permute+quantise,
 * 3 GEMM1, 4 requantise, 5 GEMM2, 6 combine) and events[7] after the last,
 * and moe_w8a8_linear records events[0] (quantise), events[1] (GEMM) and
 * events[2] (end).  `events` holds `n` cudaEvent_t created by the caller
 * (n >= 8); NULL turns the hook off.  Returns MOE_ERR_INVALID_ARG if n < 8.
 * While set, the kernels are launched without programmatic dependent launch,
 * so that each event pair times one kernel alone.
 * ------------------------------------------------------------------------- */
MOE_W8A8_API moe_status_t moe_w8a8_set_profile_events(void* const* events, int n);

/* ---------------------------------------------------------------------------
 * moe_w8a8_launch_count -- measurement hook: the number of CUDA kernels the
 * library has launched (every entry point, every thread) since it was
 * loaded.  A caller reads it before and after a region to count the kernels
 * launched inside it.  Never fails.
 * ------------------------------------------------------------------------- */
MOE_W8A8_API uint64_t moe_w8a8_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_W8A8_H */

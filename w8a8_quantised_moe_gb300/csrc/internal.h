// internal.h -- declarations shared by the translation units of the library
// (host launchers of every kernel, the forward's workspace layout).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#ifdef __CUDACC__
#include <cuda_fp16.h>
#endif

namespace moe {

constexpr int kRouterTokens = 32;  // tokens per top-k CTA = tokens per routing chunk
constexpr int kRouterTargetCtas = 160;  // K slices of the router GEMM fill about this many CTAs
constexpr int kRouterMaxSlices = 8;     // at most this many K slices (partial logits per token)
constexpr int kRouterSmallT = 128;      // up to this many tokens the router runs on the CUDA cores
constexpr int kMaxExperts = 256;
constexpr int kMaxTopK = 8;
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;
// The process-wide limit of every in-kernel wait (moe_w8a8_set_wait_timeout_ns).
uint64_t current_timeout_ns();

// Bits of the sticky device error word (first int of a workspace).
constexpr int kErrTimeout = 1;  // a pipeline wait ran out of time
constexpr int kErrDevice = 2;   // a device-side consistency check failed

// Checked build (-DMOE_CHECKED=1): every index a kernel takes from data
// rather than from its launch shape (expert ids, slots, expert offsets,
// exact-path lists, gathered rows) is range-checked before its access; an
// index outside its range sets kErrDevice in the error word and the access
// is skipped (or the range clamped), where the normal build would read or
// write out of bounds.  Without the flag in_range() is the constant true and
// the checks compile away.
#ifndef MOE_CHECKED
#define MOE_CHECKED 0
#endif
constexpr bool kChecked = MOE_CHECKED != 0;

// Epilogue variants of the grouped GEMM.
enum class Epi : int {
    GateUp = 0,    // h = silu(g) * u, fp32 out (first expert GEMM)
    ScaleF32 = 1,  // (acc * s_act) * s_w, fp32 out (second expert GEMM)
    ScaleBF16 = 2  // (acc * s_act) * s_w, bf16 out (linear layer)
};

// Tile shapes of the grouped GEMM.
enum class GemmShape : int {
    Wide = 0,    // one CTA per tile, 160 activation rows: groups of a few hundred rows
    Mid = 1,     // one CTA per tile, 128 rows: about a hundred rows per group
    Narrow = 2,  // one CTA per tile, 32 rows: a few rows per group (decode)
    Pair = 3,    // CTA pairs, 256 weight rows x 192 activation rows per tile
    Skinny = 4   // CUDA-core dp4a, weights streamed once: a few rows per group (decode)
};

// Largest L1 norm of a quantised activation row for which the fp32
// tensor-core accumulation of int8 x int8 products is exact: every partial
// sum is then at most 128 * 2^17 = 2^24 in magnitude.
constexpr int kExactL1 = 1 << 17;

struct GemmArgs {
    const void* w;           // int8 weights [n_groups * w_rows_per_group][K]
    const void* act16;       // fp16 activation rows [total_rows][K] (exact int8 values)
    const int8_t* act8;      // int8 activation rows [total_rows][K] (Skinny only; act16 unused there)
    int K;                   // reduction length (multiple of 128)
    int n_cb;                // channel blocks per group
    int n_groups;            // groups (experts); 1 for the linear layer
    int total_rows;          // rows of the activation matrix
    const int32_t* offsets;  // [n_groups + 1] group row offsets, or nullptr: one group
    int w_rows_per_group;    // weight rows per group (2I, H or N)
    int up_offset;           // GateUp only: row offset of the up half (I)
    const float* w_scale;    // [n_groups * w_rows_per_group]
    const float* act_scale;  // [total_rows]
    void* out;               // fp32 or bf16 output
    int ld_out;              // output row length in elements
    int32_t* acc_out;        // optional raw accumulators [total_rows][w_rows_per_group]
    const int32_t* flags;    // [total_rows] nonzero: row above kExactL1, done by the exact path
    const int32_t* fb_list;  // rows above kExactL1 (any order)
    const int32_t* fb_count; // number of entries of fb_list
    int* error;              // sticky device error word
    uint64_t timeout_ns;
    int stall;               // test hook (MOE_INJECT=stall): the producer first waits on a barrier that
                             // nothing completes, so that the wait limit runs out
    unsigned int* sched;     // Skinny only, optional: two words, zero between launches, through which
                             // CTAs take work units in turn (nullptr: a fixed round-robin deal)
};

// The one-kernel layer for few tokens (fused.cu).  Pointers into the
// forward's workspace (FwdLayout) except x, Wr, bias, the weights (in g1, g2)
// and y.  q_tok: int8 codes [T][H] token-major; q_h: int8 [S][I]; g1 and g2
// as the multi-kernel forward fills them for the dp4a kernel, with g1.act8 =
// q_tok (rows gathered through slot_token).  bar, abort, exits: words of the
// workspace's error region that are zero between calls.
struct FusedArgs {
    const uint16_t* x;
    const float* Wr;
    const float* bias;
    int T, H, I, E, k, E_pad, KS, hs;
    float* P;
    int32_t *topk_ids;
    float* topk_w;
    int32_t *rank, *hist, *offsets, *counts;
    unsigned int* ticket;
    int32_t *slot_of, *slot_token;
    float *s_x, *s_slot;
    int8_t* q_tok;
    float *h, *s_h;
    int8_t* q_h;
    float* o;
    uint16_t* y;
    GemmArgs g1, g2;
    unsigned int* done1;  // [E] gate/up GEMM units finished per expert
    int* ready2;          // [E] nonzero once the expert's rows of h are requantised
    unsigned int* bar;
    int* abort;
    unsigned int* exits;
    int* error;
    uint64_t timeout_ns;
    int stall;  // test hook (MOE_INJECT=stall): CTA 0 skips one barrier arrival, every wait runs out
};
// Shapes the one-kernel layer takes: T <= kRouterSmallT, both GEMMs on the
// dp4a kernel's unit shapes, a row of x in one CTA's registers.
bool fused_supported(int64_t T, int64_t H, int64_t I, int64_t E, int64_t k);
cudaError_t launch_moe_fused(const FusedArgs& a, cudaStream_t st);

// Byte offsets, within the first 256 bytes of the workspace (the error
// region, zeroed once by the caller and left zero by every call), of the
// few-token router's ticket and of the one-kernel layer's barrier words.
constexpr size_t kTicketOffset = 128;
constexpr size_t kFusedCtlOffset = 192;
// the counter words of the dp4a GEMMs' unit scheduling (GemmArgs::sched;
// two per GEMM)
constexpr size_t kSchedOffset = 224;

// Launch plan of the router GEMM: experts padded to E_pad (a multiple of 16,
// or of 128 above 128), NB experts per CTA, the hidden dimension cut into KS
// slices of kb_per_slice 64-wide steps.
struct RouterPlan {
    int E_pad, NB, n_eb, KS, kb_per_slice;
    int hs;      // small router: rows of Wr per slice (KS slices)
    bool small;  // CUDA-core router (T <= kRouterSmallT): no weight split
};
RouterPlan router_plan(int64_t T, int64_t H, int64_t E);

// Forward workspace layout (byte offsets; every region 256-byte aligned).
struct FwdLayout {
    size_t err, counts, wsplit, logits, topk_ids, topk_w, rank, hist, offsets, slot_of, slot_token, s_x,
        s_slot, flag1, list1, flag2, list2, q_x16, h, s_h, q_h16, o, fctl, total;
};
FwdLayout fwd_layout(int64_t T, int64_t H, int64_t I, int64_t E, int64_t k);

struct LinLayout {
    size_t err, counts, s_x, flag, list, q_x16, total;
};
LinLayout lin_layout(int64_t M, int64_t N, int64_t K);

// ---- programmatic dependent launch ----
// A kernel launched with pdl = true may start while the previous kernel on
// the stream is still running: it runs its set-up (barrier init, tensor
// memory allocation) and then calls pdl_wait(), which returns once the
// previous grid has completed and its memory is visible, before its first
// global memory access.  Every kernel of the layer calls pdl_wait() first and
// pdl_trigger() right after it, so at most two grids overlap: the one
// finishing and the next one's set-up.  One exception: the one-CTA-per-row
// requantiser (few rows: decode) triggers before it waits, so that the down
// GEMM's CTAs take the SMs that the gate/up GEMM's last CTAs leave and
// prefetch their first weights there; each grid still waits for its
// predecessor's completion, and a dependent grid launches only once every
// CTA of its predecessor is running, so no grid can hold the SMs that an
// earlier one still needs.  The first kernel of each entry point is launched
// without PDL (it then serialises like a plain launch).  The dp4a GEMM reads
// the expert offsets and its weights before its wait (both complete before
// its predecessor started).
#ifdef __CUDACC__
// Checked build: true when lo <= v < hi, else records kErrDevice (when error
// is given) and returns false.  Always true in the normal build.
__device__ __forceinline__ bool in_range(long long v, long long lo, long long hi, int* error) {
    if (!kChecked || (v >= lo && v < hi)) return true;
    if (error != nullptr) atomicOr(error, kErrDevice);
    return false;
}

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Asynchronous 16-byte copy global -> shared (the LSU path, no registers),
// and the wait for every such copy this thread issued.
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                     static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst))),
                 "l"(gmem_src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}
// cp_async16 that writes 16 zero bytes instead when !valid (gmem_src is then
// not read); commit of the copies issued since the last commit, and the wait
// until at most N committed groups are still in flight.
__device__ __forceinline__ void cp_async16_zfill(void* smem_dst, const void* gmem_src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(
                     static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst))),
                 "l"(gmem_src), "r"(valid ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Quantisation code of v for the scale s = amax / 127 of its row:
// clamp(round_half_even(v / s), -128, 127) with v / s the correctly rounded
// binary32 quotient; s == 0 gives 0.  (Measured: replacing the division by a
// product with 1/s plus an exact fallback near the half-integers was slower
// in the quantisation kernels.)
__device__ __forceinline__ int quant_code_div(float v, float s) {
    if (s == 0.f) return 0;
    return min(127, max(-128, __float2int_rn(__fdiv_rn(v, s))));
}

// Eight codes (|q| <= 128) as exact fp16 values (four words, element 0 in the
// low half of word 0) or as int8 (two words, element 0 in the low byte).
__device__ __forceinline__ uint4 pack_codes_f16(const int (&q)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
        w[j] = (uint32_t)__half_as_ushort(__int2half_rn(q[2 * j])) |
               ((uint32_t)__half_as_ushort(__int2half_rn(q[2 * j + 1])) << 16);
    return make_uint4(w[0], w[1], w[2], w[3]);
}
__device__ __forceinline__ uint2 pack_codes_s8(const int (&q)[8]) {
    uint32_t w[2];
#pragma unroll
    for (int j = 0; j < 2; ++j)
        w[j] = (uint32_t)(uint8_t)q[4 * j] | ((uint32_t)(uint8_t)q[4 * j + 1] << 8) |
               ((uint32_t)(uint8_t)q[4 * j + 2] << 16) | ((uint32_t)(uint8_t)q[4 * j + 3] << 24);
    return make_uint2(w[0], w[1]);
}

// Warp reduction of N per-lane values down to STOP values per lane: each
// step exchanges half of the remaining values with the partner lane (lane ^ M)
// and keeps the half selected by that lane bit, so that 32 values cost 31
// shuffles instead of 160.  The order of the additions is fixed, so float
// sums are deterministic.  Afterwards lane l holds the sums of values
// [b, b + STOP) with b = (l / (32 / (N / STOP))) * STOP.
template <typename V, int N, int M, int STOP>
struct WarpButterfly {
    static __device__ __forceinline__ void run(V* v, int lane) {
        if constexpr (N > STOP) {
            const bool up = (lane & M) != 0;
#pragma unroll
            for (int i = 0; i < N / 2; ++i) {
                const V send = up ? v[i] : v[i + N / 2];
                const V keep = up ? v[i + N / 2] : v[i];
                v[i] = keep + __shfl_xor_sync(0xffffffffu, send, M);
            }
            WarpButterfly<V, N / 2, M / 2, STOP>::run(v, lane);
        } else {
#pragma unroll
            for (int m = M; m > 0; m >>= 1)
#pragma unroll
                for (int i = 0; i < STOP; ++i) v[i] += __shfl_xor_sync(0xffffffffu, v[i], m);
        }
    }
};
#endif

// Whether the layer's launches use programmatic dependent launch: on unless
// MOE_W8A8_NO_PDL is set in the environment, and off while per-kernel
// profiling events are set (events between kernels would time the overlap).
bool pdl_default();

// Kernels launched through launch_kernel since the library was loaded.
void count_launch();

// Host-side fault injection for tests of the error paths.  The environment
// variable MOE_INJECT (read at every call; a comma-separated list) names the
// faults to fake; none of them reaches the GPU:
//   ws_short     an entry point's workspace size check fails as if the
//                workspace were one byte short (MOE_ERR_WORKSPACE_TOO_SMALL)
//   bad_ptr      its pointer check fails as if a data pointer were null
//                (MOE_ERR_INVALID_ARG)
//   launch_fail  every kernel launch fails with cudaErrorLaunchFailure before
//                anything is queued (the entry point returns MOE_ERR_CUDA)
//   stall        every grouped GEMM launch starts with its producer waiting,
//                within the wait limit, on a barrier that nothing completes:
//                the limit runs out and the kernel takes its abort path (the
//                one fault that reaches the GPU; a test of the timeout path)
// kInjectBadSlot: after the quantiser, one slot index is overwritten with an
// out-of-range value; honoured only by the checked build, whose combine
// catches it (the normal build ignores it).
enum InjectFault : int { kInjectWsShort = 1, kInjectBadPtr = 2, kInjectLaunchFail = 4, kInjectStall = 8,
                         kInjectBadSlot = 16 };
bool injected(InjectFault f);

template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, bool pdl,
                          Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    if (injected(kInjectLaunchFail)) return cudaErrorLaunchFailure;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
    if (e == cudaSuccess) count_launch();
    return e;
}

// ---- launchers (return cudaSuccess or the launch error) ----
// pdl: launch with programmatic dependent launch (see above).
// Router: weight split, tensor-core logits (partials per K slice), top-k.
// The router's first kernel is launched without pdl; its later ones with pdl.
// For T <= kRouterSmallT (RouterPlan::small) the router's last kernel also
// computes the prefix sums of launch_scan (offsets, chunk bases in hist) and clears
// counts[0..1]; `ticket` is a zeroed workspace word that it leaves zeroed.
cudaError_t launch_router(const uint16_t* x, const float* Wr, const float* bias, int T, int H, int E, int k,
                          uint16_t* wsplit, float* logits, int32_t* topk_ids, float* topk_w, int32_t* rank,
                          int32_t* hist, int32_t* offsets, int32_t* counts, unsigned int* ticket, int* error,
                          uint64_t timeout_ns, cudaStream_t st, bool pdl);
cudaError_t launch_scan(int32_t* hist, int nchunk, int E, int32_t* offsets, int32_t* counts,
                        cudaStream_t st, bool pdl);
// Codes go to q16 (fp16 values, the tensor-core operand) and/or q8 (int8,
// the Skinny operand); either may be null.
cudaError_t launch_permute_quant(const uint16_t* x, const int32_t* topk_ids, const int32_t* rank,
                                 const int32_t* hist, int T, int H, int E, int k, int32_t* slot_of,
                                 int32_t* slot_token, float* s_x, float* s_slot, uint16_t* q16, int8_t* q8,
                                 int32_t* flags, int32_t* fb_list, int32_t* fb_count, int* error, cudaStream_t st,
                                 bool pdl);
// The same with SmoothQuant-folded activations per expert: each (token,
// choice) row is x[t] times the reciprocals of smooth[e] ([E][H]), quantised
// per slot; s_x[t] receives the scale of the token's first choice.  rcp:
// scratch of E * H floats for the reciprocals (two launches).
cudaError_t launch_permute_quant_smooth(const uint16_t* x, const float* smooth, float* rcp,
                                        const int32_t* topk_ids, const int32_t* rank, const int32_t* hist, int T,
                                        int H, int E, int k, int32_t* slot_of, int32_t* slot_token, float* s_x,
                                        float* s_slot, uint16_t* q16, int8_t* q8, int32_t* flags, int32_t* fb_list,
                                        int32_t* fb_count, int* error, cudaStream_t st, bool pdl);
cudaError_t launch_requant(const float* h, int S, int I, float* s_h, uint16_t* q16, int8_t* q8,
                           int32_t* flags, int32_t* fb_list, int32_t* fb_count, cudaStream_t st, bool pdl);
cudaError_t launch_combine(const float* o, const int32_t* slot_of, const float* topk_w, int T,
                           int H, int k, uint16_t* y, int* error, cudaStream_t st, bool pdl);
// col_scale (optional, [K]): the row quantised is w[r][k] * col_scale[k].
cudaError_t launch_quantize_weights(const float* w, int64_t rows, int K, int8_t* q, float* s,
                                    cudaStream_t st, const float* col_scale = nullptr);
// out[r][:] = the codes of q16[row_of[r * stride]][:] (row_of == nullptr:
// identity); src_rows bounds row_of's values (checked build).
cudaError_t launch_f16_rows_to_s8(const uint16_t* q16, const int32_t* row_of, int rows, int K,
                                  int row_stride_of, int src_rows, int8_t* q8, int* error, cudaStream_t st);
// out[r][:] = q8[row_of[r * stride]][:] (row_of == nullptr: identity).
cudaError_t launch_s8_rows_gather(const int8_t* q8, const int32_t* row_of, int rows, int K, int row_stride_of,
                                  int src_rows, int8_t* out, int* error, cudaStream_t st);
GemmShape choose_gemm_shape(long rows, long groups, long K);
// choose_gemm_shape unless a test forced a path (moe_w8a8_set_gemm_path);
// a forced Skinny falls back to the automatic choice where unsupported.
GemmShape pick_gemm_shape(long rows, long groups, long K, Epi epi, long w_rows_per_group, long up_offset);
cudaError_t launch_grouped_gemm(Epi epi, GemmShape shape, const GemmArgs& args, cudaStream_t st, bool pdl);
// CTA-pair kernel (gemm_pair.cu): needs an even number of channel blocks.
bool pair_gemm_supported(const GemmArgs& args);
cudaError_t launch_grouped_gemm_pair(Epi epi, const GemmArgs& args, cudaStream_t st, bool pdl);
// dp4a kernel (gemm_skinny.cu): needs act8, K a multiple of 128, and weight
// rows (Scale) or channels (GateUp) per group a multiple of 64 / 32.
bool skinny_gemm_supported(Epi epi, const GemmArgs& args);
bool skinny_shape_supported(Epi epi, long K, long w_rows_per_group, long up_offset);
cudaError_t launch_grouped_gemm_skinny(Epi epi, const GemmArgs& args, cudaStream_t st, bool pdl);

// FP8 (E4M3) variant (fp8.cu).  Codes are bytes; args.act8 carries the E4M3
// activation rows and args.w the E4M3 weights; GateUp and ScaleF32 only.
cudaError_t launch_quantize_weights_fp8(const float* w, int64_t rows, int K, uint8_t* q, float* s, cudaStream_t st);
cudaError_t launch_permute_quant_fp8(const uint16_t* x, const int32_t* topk_ids, const int32_t* rank,
                                     const int32_t* hist, int T, int H, int E, int k, int32_t* slot_of,
                                     int32_t* slot_token, float* s_x, float* s_slot, uint8_t* q8, int* error,
                                     cudaStream_t st, bool pdl);
cudaError_t launch_requant_fp8(const float* h, int S, int I, float* s_h, uint8_t* q8, cudaStream_t st, bool pdl);
cudaError_t launch_grouped_gemm_fp8(Epi epi, const GemmArgs& args, cudaStream_t st, bool pdl);

int num_sms();

// 2-D tiled tensor map (row-major, inner dimension contiguous).
bool make_tensor_map_2d(CUtensorMap* map, CUtensorMapDataType dt, int elem_bytes, const void* base,
                        uint64_t inner, uint64_t outer, uint32_t box_inner, uint32_t box_outer,
                        CUtensorMapSwizzle swz);
// 3-D tiled tensor map: dims[0] contiguous, dims[1] and dims[2] with the
// given byte strides (any order of strides).  One box of box[0] x box[1] x
// box[2] lands in shared memory as box[2] consecutive [box[1]][box[0]]
// tiles: one bulk copy where two 2-D boxes were needed.
bool make_tensor_map_3d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, const uint64_t (&dims)[3],
                        const uint64_t (&strides)[2], const uint32_t (&box)[3], CUtensorMapSwizzle swz);

}  // namespace moe

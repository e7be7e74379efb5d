// fused.cu -- the whole W8A8 MoE layer for few tokens (decode) as one
// persistent kernel: router, top-k and routing tables, per-token activation
// quantisation, the gate/up GEMM with the SiLU-times-up epilogue, the
// requantisation of its output, the down GEMM and the weighted combine run as
// phases of a single cooperative launch.
//
// "Tencent Hunyuan AI Infra on Hopper" (pnsm.cn), section 1.3, describes the
// fused MoE operator as one kernel that runs gate, top-k, the routing
// pre-processing, both expert GEMMs and the weighted aggregation in turn.
// Here the phases reuse the device bodies of the multi-kernel forward (the
// few-token router and the per-token quantiser of router_small.cuh, the dp4a
// work-unit loop of gemm_skinny.cuh) and the same arithmetic, so that every
// intermediate and the output equal that forward's bit for bit.  What differs
// from it: the activation codes are written once per token (not once per
// slot), next to the router, and the gate/up GEMM gathers its rows through the
// slot -> token map; the routing tables are built by every CTA in its own
// shared memory; and no kernel boundary separates the phases.
//
// Phases (CTA b of nblk, all CTAs resident: a cooperative launch):
//   A  router partial logits of K slice s (CTAs s < KS) and, on the next T
//      CTAs, the per-token quantisation of x (codes token-major)
//                                                        -- grid barrier 1
//   B  per token: slice sums, bias, top-k and softmax weights
//                                                        -- grid barrier 2
//   C  every CTA: the routing tables (shared memory); the gate/up GEMM (dp4a),
//      epilogue h = silu(gate) * up, units taken from a counter
//   D  the CTA that finishes an expert's last gate/up unit requantises the
//      expert's rows of h (s_h = amax / 127, int8 codes) and raises its flag
//   E  down GEMM (dp4a), o = (acc * s_h) * s_w; an expert's rows are staged
//      after its flag, so the down GEMM starts while the gate/up GEMM's last
//      units run                                         -- grid barrier 3
//   F  y[t] = bf16(sum_j w[t][j] * o[slot(t, j)]) in top-k order
// Every wait (the barriers, the experts' flags) is bounded by the library's
// wait limit; a CTA that runs out sets the timeout bit of the error word and
// an abort flag, after which every CTA skips the remaining phases and
// returns.  The last CTA to return clears the barrier words for the next call.
#include <mutex>

#include "gemm_common.cuh"
#include "gemm_skinny.cuh"
#include "router_small.cuh"

namespace moe {
namespace {

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Grid-wide barrier number n (1, 2, ...): every CTA arrives once per barrier
// on a counter that only grows during the launch, and waits until n * nblk
// arrivals.  Returns false (in every thread) when the wait gave up: another
// CTA aborted, or the limit ran out (then this CTA records the timeout and
// aborts the launch).  skip_arrival: the test hook's stall (MOE_INJECT=stall).
__device__ bool grid_barrier(const FusedArgs& a, unsigned n, bool skip_arrival = false) {
    __shared__ int ok_s;
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();  // this CTA's writes before the arrival
        if (!skip_arrival) atomicAdd(a.bar, 1u);
        const unsigned target = n * gridDim.x;
        const uint64_t t0 = global_timer_ns();
        int ok = 1;
        for (uint32_t i = 0;; ++i) {
            if (ld_acquire_u32(a.bar) >= target) break;
            if (*reinterpret_cast<volatile int*>(a.abort)) {
                ok = 0;
                break;
            }
            if ((i & 15u) == 15u && global_timer_ns() - t0 > a.timeout_ns) {
                atomicExch(a.abort, 1);
                atomicOr(a.error, kErrTimeout);
                ok = 0;
                break;
            }
            __nanosleep(32);
        }
        __threadfence();
        ok_s = ok;
    }
    __syncthreads();
    return ok_s != 0;
}

// After the top-k phase, in every CTA: the routing tables in shared memory
// (the slot of (token t, choice j) routed to expert e is offsets[e] plus the
// number of earlier tokens routed to e: the multi-kernel forward's order), so
// that no CTA waits for one CTA to build them.  offs_s [E + 1], map_s [S]
// (slot -> token), ssl_s [S] (slot -> activation scale), mask_s [chunks][E]
// (token bits of every 32-token chunk per expert).  CTA 0 also writes the
// global copies (offsets, slot_of, slot_token, s_slot) that the combine and
// the debug dumps read.
__device__ void build_tables(const FusedArgs& a, int* offs_s, int* map_s, float* ssl_s, uint32_t* mask_s) {
    __shared__ int32_t wsum[8];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int T = a.T, k = a.k, E = a.E, S = T * k;
    const int nchunk = (T + kRouterTokens - 1) / kRouterTokens;
    for (int i = tid; i < nchunk * E; i += blockDim.x) mask_s[i] = 0u;
    __syncthreads();
    for (int i = tid; i < S; i += blockDim.x) {
        const int t = i / k;
        const int e = __ldcg(a.topk_ids + i);
        if (in_range(e, 0, E, a.error)) atomicOr(&mask_s[(t / kRouterTokens) * E + e], 1u << (t % kRouterTokens));
    }
    __syncthreads();
    // exclusive prefix over the experts of their token counts (E <= 256 = blockDim)
    int32_t tot = 0;
    if (tid < E)
        for (int c = 0; c < nchunk; ++c) tot += __popc(mask_s[c * E + tid]);
    int32_t incl = tot;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int32_t o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    int32_t before = 0, all = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
        if (w < warp) before += wsum[w];
        all += wsum[w];
    }
    if (tid < E) offs_s[tid] = before + incl - tot;
    if (tid == 0) offs_s[E] = all;
    __syncthreads();
    for (int i = tid; i < S; i += blockDim.x) {
        const int t = i / k, c = t / kRouterTokens;
        const int e = __ldcg(a.topk_ids + i);
        int slot = -1;
        if (in_range(e, 0, E, a.error)) {
            slot = offs_s[e] + __popc(mask_s[c * E + e] & ((1u << (t % kRouterTokens)) - 1u));
            for (int cc = 0; cc < c; ++cc) slot += __popc(mask_s[cc * E + e]);
            if (!in_range(slot, 0, S, a.error)) slot = -1;
        }
        if (!kChecked || slot >= 0) {
            const float sx = __ldcg(a.s_x + t);
            map_s[slot] = t;
            ssl_s[slot] = sx;
            if (blockIdx.x == 0) {
                a.slot_token[slot] = t;
                a.s_slot[slot] = sx;
            }
        }
        if (blockIdx.x == 0) a.slot_of[i] = slot;
    }
    if (blockIdx.x == 0)
        for (int e = tid; e <= E; e += blockDim.x) a.offsets[e] = offs_s[e];
    __syncthreads();
}

// Slot row r of h: s_h[r] = amax / 127 and its int8 codes (one CTA; the
// arithmetic of the multi-kernel forward's requantiser).  The row is read
// twice (the second time from L2) so that few registers are live here: this
// runs inside the gate/up GEMM's loop, next to its weights in flight.
__device__ void requant_row(const FusedArgs& a, int r) {
    __shared__ float red_max[8];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int I = a.I;
    const float4* row = reinterpret_cast<const float4*>(a.h + (size_t)r * I);
    const int nv = I / 4;
    float amax = 0.f;
    for (int idx = tid; idx < nv; idx += blockDim.x) {
        const float4 v = __ldcg(row + idx);
        amax = fmaxf(fmaxf(fmaxf(amax, fabsf(v.x)), fmaxf(fabsf(v.y), fabsf(v.z))), fabsf(v.w));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    if (lane == 0) red_max[warp] = amax;
    __syncthreads();
    amax = red_max[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) amax = fmaxf(amax, red_max[i]);
    const float s = __fdiv_rn(amax, 127.0f);
    if (tid == 0) a.s_h[r] = s;
    for (int idx = tid; idx < nv; idx += blockDim.x) {
        const float4 v = __ldcg(row + idx);
        const int c0 = quant_code_div(v.x, s), c1 = quant_code_div(v.y, s), c2 = quant_code_div(v.z, s),
                  c3 = quant_code_div(v.w, s);
        reinterpret_cast<uint32_t*>(a.q_h + (size_t)r * I)[idx] =
            (uint32_t)(uint8_t)c0 | ((uint32_t)(uint8_t)c1 << 8) | ((uint32_t)(uint8_t)c2 << 16) |
            ((uint32_t)(uint8_t)c3 << 24);
    }
    __syncthreads();  // red_max is reused by the next row
}

// Hand-offs between the two GEMM phases, without a grid barrier: a CTA
// counts each gate/up unit it finishes on its expert's counter; the CTA that
// finishes an expert's last unit requantises that expert's rows of h (phase
// D of the multi-kernel forward) and raises its ready flag; a CTA waits for
// an expert's flag before it stages that expert's rows for the down GEMM.  A
// CTA moves to the down GEMM as soon as the gate/up units run out, so the
// down GEMM's first experts overlap the gate/up GEMM's last units.  The
// counter's result is read one unit after the increment (the warp does not
// wait for the atomic); the last increment's at the end.
__device__ void requant_expert(const FusedArgs& a, const int* offs_s, int e) {
    for (int r = offs_s[e]; r < offs_s[e + 1]; ++r) requant_row(a, r);
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();  // the expert's q_h and s_h before its flag
        atomicExch(a.ready2 + e, 1);
    }
}

struct FusedGateUpHook {
    static constexpr bool kWaits = false;
    static constexpr bool kCounts = true;
    const FusedArgs* a;
    const int* offs_s;
    int* req_s;  // two ints of shared memory, used in turn
    unsigned per_group;
    int pend_g = -1;  // thread 0: the expert of the increment in flight, and its result
    unsigned pend_old = 0;
    int ph = 0;
    __device__ __forceinline__ bool ready(int) { return true; }
    __device__ __forceinline__ void unit_end_pre() {
        if (threadIdx.x == 0) {
            req_s[ph] = (pend_g >= 0 && pend_old == per_group - 1u) ? pend_g : -1;
            pend_g = -1;
        }
    }
    __device__ __forceinline__ void unit_end_post(int g) {
        const int r = req_s[ph];
        ph ^= 1;
        if (r >= 0) requant_expert(*a, offs_s, r);
        if (threadIdx.x == 0) {
            __threadfence();  // this unit's h (every warp's, ordered by the barrier before)
            pend_old = atomicAdd(a->done1 + g, 1u);
            pend_g = g;
        }
    }
    __device__ __forceinline__ void end() {
        __syncthreads();
        unit_end_pre();
        __syncthreads();
        const int r = req_s[ph];
        ph ^= 1;
        if (r >= 0) requant_expert(*a, offs_s, r);
    }
};

struct FusedDownHook {
    static constexpr bool kWaits = true;
    static constexpr bool kCounts = false;
    const FusedArgs* a;
    // bounded wait for expert g's flag; false when the launch gave up
    __device__ __forceinline__ bool ready(int g) {
        const uint64_t t0 = global_timer_ns();
        for (uint32_t i = 0;; ++i) {
            if (ld_acquire_u32(reinterpret_cast<const unsigned*>(a->ready2 + g)) != 0u) return true;
            if (*reinterpret_cast<volatile int*>(a->abort)) return false;
            if ((i & 15u) == 15u && global_timer_ns() - t0 > a->timeout_ns) {
                atomicExch(a->abort, 1);
                atomicOr(a->error, kErrTimeout);
                return false;
            }
            __nanosleep(64);
        }
    }
    __device__ __forceinline__ void unit_end_pre() {}
    __device__ __forceinline__ void unit_end_post(int) {}
    __device__ __forceinline__ void end() {}
};

// Phase F, token t, part `part` of `nparts` of its columns: the weighted sum
// of its k slot rows of o in top-k order (the multi-kernel forward's combine).
__device__ void combine_part(const FusedArgs& a, int t, int part, int nparts) {
    __shared__ int32_t slot[kMaxTopK];
    __shared__ float w[kMaxTopK];
    const int k = a.k, H = a.H;
    if (threadIdx.x < k) {
        const int sl = __ldcg(a.slot_of + (size_t)t * k + threadIdx.x);
        slot[threadIdx.x] = in_range(sl, 0, (long long)a.T * k, part == 0 ? a.error : nullptr) ? sl : -1;
        w[threadIdx.x] = __ldcg(a.topk_w + (size_t)t * k + threadIdx.x);
    }
    __syncthreads();
    const int nv = H / 4;
    for (int i = part * 256 + threadIdx.x; i < nv; i += nparts * 256) {
        float4 v[kMaxTopK];
#pragma unroll
        for (int j = 0; j < kMaxTopK; ++j)
            if (j < k)
                v[j] = (!kChecked || slot[j] >= 0) ? __ldcg(reinterpret_cast<const float4*>(a.o + (size_t)slot[j] * H) + i)
                                                   : make_float4(0.f, 0.f, 0.f, 0.f);
        float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
        for (int j = 0; j < kMaxTopK; ++j) {
            if (j >= k) break;
            const float wj = w[j];
            a0 = __fadd_rn(a0, __fmul_rn(wj, v[j].x));
            a1 = __fadd_rn(a1, __fmul_rn(wj, v[j].y));
            a2 = __fadd_rn(a2, __fmul_rn(wj, v[j].z));
            a3 = __fadd_rn(a3, __fmul_rn(wj, v[j].w));
        }
        uint2 out;
        out.x = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(a0)) |
                ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(a1)) << 16);
        out.y = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(a2)) |
                ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(a3)) << 16);
        reinterpret_cast<uint2*>(a.y + (size_t)t * H)[i] = out;
    }
    __syncthreads();  // slot and w are reused by the next item of this CTA
}

// L2 prefetch, by thread 0 at the end of the gate/up GEMM (while the CTAs
// that finished first wait for the last), of the down-projection rows of
// unit bid of the down GEMM's unit table.  (Measured on the decode layer: the
// down GEMM phase 69.7 -> 68.0 us.  The same for the gate/up GEMM's first
// units during the routing phases made those phases 5 us longer, for 1.6 us
// gained in the GEMM: not done.)
__device__ void prefetch_gemm2(const FusedArgs& a, const int* offs_s, int bid) {
    const int per_group = a.H / kSkUnitScale;
    int u = bid;
    for (int g = 0; g < a.E; ++g) {
        if (offs_s[g + 1] == offs_s[g]) continue;
        if (u < per_group) {
            const int8_t* w = static_cast<const int8_t*>(a.g2.w) + ((size_t)g * a.H + (size_t)u * kSkUnitScale) * a.I;
            prefetch_l2_bulk(w, (uint32_t)((size_t)kSkUnitScale * a.I));
            return;
        }
        u -= per_group;
    }
}

// Every CTA calls this once, on every path out of the kernel; the last one
// clears the barrier words and the router's ticket for the next call (no CTA
// of this launch reads them any more).
__device__ void fused_exit(const FusedArgs& a) {
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        if (atomicAdd(a.exits, 1u) == gridDim.x - 1u) {
            *a.bar = 0u;
            *a.abort = 0;
            *a.ticket = 0u;
            __threadfence();
            *a.exits = 0u;
        }
    }
}

template <int EPT>
__global__ void __launch_bounds__(kSkThreads, 2) moe_fused_kernel(const FusedArgs a) {
    extern __shared__ __align__(16) float4 fused_smem[];  // router slice, then the GEMMs' activation rows
    __shared__ int unit_start[kMaxExperts + 1];
    __shared__ int row_start[kMaxExperts + 1];
    __shared__ int next_s[3];
    __shared__ int req_s[2];
    __shared__ int map_s[kRouterSmallT * kMaxTopK];    // slot -> token: the gate/up GEMM's row gather
    __shared__ float ssl_s[kRouterSmallT * kMaxTopK];  // slot -> activation scale
    __shared__ int offs_s[kMaxExperts + 1];            // expert slot offsets
    __shared__ uint32_t mask_s[kRFMaxChunks * kMaxExperts];
    const int bid = blockIdx.x, nblk = gridDim.x;
    const int S = a.T * a.k;

    // A: router partials | per-token quantisation
    if (bid == 0)
        for (int e = threadIdx.x; e < a.E; e += blockDim.x) {
            a.done1[e] = 0u;
            a.ready2[e] = 0;
        }
    for (int w = bid; w < a.KS + a.T; w += nblk) {
        if (w < a.KS) router_partial_body(a.x, a.Wr, a.T, a.H, a.E, a.E_pad, a.hs, a.P, fused_smem, w);
        else quant_token_body(a.x, a.H, w - a.KS, a.s_x, a.q_tok);
        __syncthreads();  // the slice's shared memory is reused by the next item
    }
    if (!grid_barrier(a, 1)) return fused_exit(a);

    // B: top-k per token
    for (int t = bid; t < a.T; t += nblk)
        router_finish_body<EPT, false>(a.P, a.KS, a.T, a.E, a.E_pad, a.bias, a.k, a.topk_ids, a.topk_w, a.rank,
                                       a.hist, a.offsets, a.counts, a.ticket, a.error, t, a.T);
    // the test hook stalls CTA 0 here: it never arrives, every wait runs out
    if (!grid_barrier(a, 2, a.stall != 0 && bid == 0)) return fused_exit(a);

    // C: the routing tables (every CTA), then the gate/up GEMM over the
    // slots, rows gathered from the token-major codes
    build_tables(a, offs_s, map_s, ssl_s, mask_s);
    GemmArgs g1 = a.g1;
    g1.offsets = offs_s;
    g1.act_scale = ssl_s;
    FusedGateUpHook up_hook{&a, offs_s, req_s, (unsigned)(a.I / kSkUnitGateUp)};
    skinny_run<(int)Epi::GateUp, kSkSrcGather>(g1, reinterpret_cast<int8_t*>(fused_smem), unit_start, row_start,
                                               next_s, bid, nblk, nullptr, a.T, map_s, up_hook);
    if (threadIdx.x == 0) prefetch_gemm2(a, offs_s, bid);

    // D + E: each expert's rows requantised by the CTA that finished its last
    // gate/up unit; the down GEMM, each expert after its flag
    GemmArgs g2 = a.g2;
    g2.offsets = offs_s;
    skinny_run<(int)Epi::ScaleF32, kSkSrcRows>(g2, reinterpret_cast<int8_t*>(fused_smem), unit_start, row_start,
                                               next_s, bid, nblk, nullptr, 0, nullptr, FusedDownHook{&a});
    if (!grid_barrier(a, 3)) return fused_exit(a);

    // F: combine, each token's columns in nparts parts
    const int blocks = (a.H / 4 + 255) / 256;
    int nparts = (nblk + a.T - 1) / a.T;
    if (nparts > blocks) nparts = blocks;
    for (int w = bid; w < a.T * nparts; w += nblk) combine_part(a, w / nparts, w % nparts, nparts);
    fused_exit(a);
}

size_t fused_smem_bytes(int64_t T, int64_t H, int64_t I, int64_t E) {
    const RouterPlan p = router_plan(T, H, E);
    const int64_t T64 = (T + kRPTile - 1) / kRPTile * kRPTile, E64 = (E + kRPTile - 1) / kRPTile * kRPTile;
    const int64_t router = (int64_t)p.hs * (T64 + E64) * (int64_t)sizeof(float);
    const int64_t g1 = skinny_smem_bytes((int)H), g2 = skinny_smem_bytes((int)I);
    const int64_t gemm = g1 > g2 ? g1 : g2;
    return (size_t)(router > gemm ? router : gemm);
}

template <int EPT>
cudaError_t launch_fused_impl(const FusedArgs& a, size_t smem, cudaStream_t st) {
    if (injected(kInjectLaunchFail)) return cudaErrorLaunchFailure;
    auto kern = moe_fused_kernel<EPT>;
    // the shared-memory attribute and the resident CTAs per SM, per
    // shared-memory size (queried once: host time here delays the launch)
    static std::mutex mu;
    static size_t smem_set = 0, occ_smem = 0;
    static int occ_cached = 0;
    int occ = 0;
    cudaError_t e = cudaSuccess;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (smem > smem_set) {
            e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return e;
            smem_set = smem;
        }
        if (occ_smem != smem || occ_cached == 0) {
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ_cached, kern, kSkThreads, smem);
            if (e != cudaSuccess) return e;
            occ_smem = smem;
        }
        occ = occ_cached;
    }
    if (occ < 1) return cudaErrorInvalidConfiguration;
    if (occ > 2) occ = 2;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(occ * num_sms()));
    cfg.blockDim = dim3(kSkThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;  // every CTA resident: the grid barriers need it
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, a);
    if (e == cudaSuccess) count_launch();
    return e;
}

}  // namespace

bool fused_supported(int64_t T, int64_t H, int64_t I, int64_t E, int64_t k) {
    if (T < 1 || T > kRouterSmallT || E > kMaxExperts || k > kMaxTopK) return false;
    if (H > 256 * 8 * kQtVec) return false;  // a row of x in one CTA's registers
    if (!skinny_shape_supported(Epi::GateUp, H, 2 * I, I) || !skinny_shape_supported(Epi::ScaleF32, I, H, 0))
        return false;
    return fused_smem_bytes(T, H, I, E) <= 200 * 1024;  // with the static shared memory, within 227 KB
}

cudaError_t launch_moe_fused(const FusedArgs& a, cudaStream_t st) {
    const size_t smem = fused_smem_bytes(a.T, a.H, a.I, a.E);
    if (a.E <= 32) return launch_fused_impl<1>(a, smem, st);
    if (a.E <= 64) return launch_fused_impl<2>(a, smem, st);
    if (a.E <= 128) return launch_fused_impl<4>(a, smem, st);
    return launch_fused_impl<8>(a, smem, st);
}

}  // namespace moe

// router.cu -- FP32-accurate router logits on the tensor cores, and top-k.
//
//   router_split_kernel  Wr fp32 [H][E] -> three bf16 matrices [3][E_pad][H]
//                        (K-major), hi = bf16(w), mid = bf16(w - hi),
//                        lo = bf16(w - hi - mid).  Each subtraction is exact and
//                        hi + mid + lo == w exactly (24 mantissa bits = 3 x 8).
//   router_gemm_kernel   partial logits P[ks][t][e] = sum over the ks-th slice
//                        of h of x[t][h] * (hi + mid + lo)[e][h]: three bf16 MMAs
//                        per K step into one fp32 accumulator.  x is bf16, so
//                        every product is exact in fp32 and the result is an
//                        fp32-accumulated dot product, like an FP32 GEMM.
//   router_partial_kernel  few tokens (decode): partial logits of every token
//                        over one slice of rows of the fp32 weights, fp32 FMAs
//                        on the CUDA cores (no split; ~128 CTAs for a tiny GEMM).
//   router_finish_kernel per token the slice sums, bias and top-k; the last
//                        CTA ranks the choices and computes the prefix sums.
//   topk_kernel          logits = sum_ks P[ks] (+ bias) in a fixed order, top-k
//                        with ties to the lower expert index, softmax over the
//                        selected logits, and per 32-token chunk the count of
//                        tokens per expert and each choice's rank in the chunk.
//
// Keeping the router at FP32 accuracy: "DeepSeek V4 950 FP8 inference on
// H100" (lpnh.cn), section 4.1.  Running the FP32-accurate router as bf16
// tensor-core GEMMs on a split of the FP32 weights (a high and a scaled low
// bf16 part there; three exact parts here): "Tencent Hunyuan AI Infra on
// Hopper" (pnsm.cn), section 1.2.  Gate -> top-k -> routing pre-processing:
// same page, section 1.3.
#include <cuda_bf16.h>

#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kRTM = 128;      // tokens per router tile (MMA M)
constexpr int kRBK = 64;       // K per stage
constexpr int kRThreads = 192; // producer, MMA, 4 epilogue warps

__device__ __forceinline__ uint16_t bf16_rn_bits(float v) { return __bfloat16_as_ushort(__float2bfloat16_rn(v)); }
__device__ __forceinline__ float bf16_bits_f(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

// 32x32 tiles through shared memory: coalesced reads of Wr rows, coalesced
// writes of the transposed bf16 rows.
__global__ void __launch_bounds__(256) router_split_kernel(const float* __restrict__ Wr, int H, int E, int E_pad,
                                                           uint16_t* __restrict__ out) {
    __shared__ float tile[32][33];
    const int h0 = blockIdx.x * 32, e0 = blockIdx.y * 32;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 8 rows per pass
    pdl_wait();
    pdl_trigger();
    for (int r = ty; r < 32; r += 8) {
        const int h = h0 + r, e = e0 + tx;
        tile[r][tx] = (h < H && e < E) ? Wr[(size_t)h * E + e] : 0.f;
    }
    __syncthreads();
    for (int r = ty; r < 32; r += 8) {
        const int e = e0 + r, h = h0 + tx;
        if (e >= E_pad || h >= H) continue;
        const float w = tile[tx][r];
        const uint16_t hi = bf16_rn_bits(w);
        const float r1 = __fsub_rn(w, bf16_bits_f(hi));
        const uint16_t mid = bf16_rn_bits(r1);
        const float r2 = __fsub_rn(r1, bf16_bits_f(mid));
        const uint16_t lo = bf16_rn_bits(r2);
        out[((size_t)0 * E_pad + e) * H + h] = hi;
        out[((size_t)1 * E_pad + e) * H + h] = mid;
        out[((size_t)2 * E_pad + e) * H + h] = lo;
    }
}

template <int NB, int NS>
struct RCfg {
    static constexpr int kStageA = kRTM * kRBK * 2;  // x tile
    static constexpr int kStageB = NB * kRBK * 2;    // one split of the W tile
    static constexpr int kStage = kStageA + 3 * kStageB;
    static constexpr int kOffBars = NS * kStage;
    static constexpr int kSmem = kOffBars + (2 * NS + 2) * 8 + 64 + 1024;
    static constexpr int kTmemAlloc = NB <= 32 ? 32 : NB <= 64 ? 64 : 128;
    static_assert(kStageB % 1024 == 0, "tiles keep 1024-byte alignment");
    static_assert(kSmem <= 232448, "shared memory budget");
};

// Grid: (token tiles, expert blocks of NB, K slices).  Writes partial logits
// P[ks][t][e] for its tokens, experts and slice.
template <int NB, int NS>
__global__ void __launch_bounds__(kRThreads, 1)
    router_gemm_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_w,
                       int T, int H, int E, int E_pad, int kb_per_slice, float* __restrict__ P, int* error,
                       uint64_t timeout_ns) {
    using C = RCfg<NB, NS>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kOffBars);
    uint64_t* empty = full + NS;
    uint64_t* acc_full = empty + NS;
    uint64_t* teardown = acc_full + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(teardown + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 2);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t0 = blockIdx.x * kRTM, e0 = blockIdx.y * NB;
    const int nkb = H / kRBK;
    const int kb0 = blockIdx.z * kb_per_slice, kb1 = min(nkb, kb0 + kb_per_slice);

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(teardown, 1);
        *abort_flag = 0;
        fence_barrier_init();
        tma_prefetch_desc(&tmap_x);
        tma_prefetch_desc(&tmap_w);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, C::kTmemAlloc);
        tmem_relinquish();
    }
    pdl_wait();  // the split weights of the previous kernel are visible from here
    pdl_trigger();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const WaitCtl ctl{abort_flag, error, timeout_ns, 0u};

    if (warp == 0) {
        // four boxes a stage (the x tile, the three weight parts); lanes 0-3
        // issue one each in the same warp instruction (a bulk tensor copy
        // costs its issuing thread ~200 cycles); lane 0 owns the waits
        if (lane < 4) {
            uint32_t it = 0;
            const CUtensorMap* map = lane == 0 ? &tmap_x : &tmap_w;
            const int row = lane == 0 ? t0 : (lane - 1) * E_pad + e0;
            const int off = lane == 0 ? 0 : C::kStageA + (lane - 1) * C::kStageB;
            for (int kb = kb0; kb < kb1; ++kb, ++it) {
                const uint32_t s = it % NS, ph = (it / NS) & 1u;
                int ok = 1;
                if (lane == 0) {
                    ok = mbar_wait(&empty[s], ph ^ 1u, ctl);
                    if (ok) mbar_arrive_expect_tx(&full[s], C::kStage);
                }
                if (!__shfl_sync(0xfu, ok, 0)) break;
                tma_load_2d(smem + s * C::kStage + off, map, &full[s], kb * kRBK, row);
            }
            if (lane == 0)
                for (uint32_t s = 0; s < (uint32_t)NS && s < it; ++s) {
                    const uint32_t last = it - 1 - ((it - 1 - s) % NS);
                    mbar_wait_drain(&full[s], (last / NS) & 1u);
                }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // bf16 A and B (format 1), fp32 D, M = 128, N = NB
            const uint32_t idesc = idesc_f16_f32(kRTM, NB) | (1u << 7) | (1u << 10);
            uint32_t it = 0;
            bool ok = true;
            for (int kb = kb0; kb < kb1; ++kb, ++it) {
                const uint32_t s = it % NS, ph = (it / NS) & 1u;
                if (!mbar_wait(&full[s], ph, ctl)) { ok = false; break; }
                tc_fence_after();
                const uint32_t a_base = smem_u32(smem + s * C::kStage);
#pragma unroll
                for (int ks = 0; ks < kRBK / 16; ++ks) {
                    const uint64_t adesc = smem_desc_sw128(a_base) + (uint64_t)(ks * 2);
#pragma unroll
                    for (int sp = 0; sp < 3; ++sp) {
                        const uint64_t bdesc =
                            smem_desc_sw128(a_base + C::kStageA + sp * C::kStageB) + (uint64_t)(ks * 2);
                        mma_f16_smem_a(tmem, adesc, bdesc, idesc, (kb != kb0 || ks != 0 || sp != 0) ? 1u : 0u);
                    }
                }
                mma_commit(&empty[s]);
            }
            if (ok) mma_commit(acc_full);
            mma_commit(teardown);
            mbar_wait_drain(teardown, 0);
        }
    } else {
        const int q = warp & 3;  // warps 2..5 cover TMEM lane quadrants 2, 3, 0, 1
        const int t = t0 + q * 32 + lane;
        if (kb1 > kb0 && mbar_wait(acc_full, 0, ctl)) {
            tc_fence_after();
#pragma unroll
            for (int c0 = 0; c0 < NB; c0 += 16) {
                uint32_t r[16];
                tmem_ld_16(tmem + ((uint32_t)(q * 32) << 16) + c0, r);
                tmem_wait_ld();
                if (t < T) {
                    float* dst = P + ((size_t)blockIdx.z * T + t) * E_pad + e0 + c0;
#pragma unroll
                    for (int i = 0; i < 16; i += 4)
                        *reinterpret_cast<float4*>(dst + i) = make_float4(
                            __uint_as_float(r[i]), __uint_as_float(r[i + 1]), __uint_as_float(r[i + 2]),
                            __uint_as_float(r[i + 3]));
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemAlloc);
    }
}

// Top-k of NT tokens' logits, one warp, the tokens' reductions interleaved:
// lane l holds the logits of experts l + 32 i (experts >= E are never taken).
// Ties go to the lower expert index; choice j of token r ends in lane j as
// my_e[r] and its softmax weight over the selected logits, my_w[r].
// A NaN logit (non-finite input, outside the layer's contract) ranks as
// -inf, so that every choice is still a valid expert index; the return value
// (the same in every lane) says whether the warp saw one, and the caller
// records it in the device error word.
template <int EPT, int NT>
__device__ __forceinline__ bool warp_topk(const float (&v_in)[NT][EPT], int E, int k, int lane, int (&my_e)[NT],
                                          float (&my_w)[NT]) {
    float v[NT][EPT];
    bool nan_seen = false;
#pragma unroll
    for (int r = 0; r < NT; ++r)
#pragma unroll
        for (int i = 0; i < EPT; ++i) {
            const float x = v_in[r][i];
            const bool nan = x != x;
            nan_seen |= nan && (lane + 32 * i) < E;
            v[r][i] = nan ? -INFINITY : x;
        }
    bool taken[NT][EPT];
    float sel0[NT], den[NT], my_v[NT];
#pragma unroll
    for (int r = 0; r < NT; ++r) {
#pragma unroll
        for (int i = 0; i < EPT; ++i) taken[r][i] = (lane + 32 * i) >= E;
        sel0[r] = 0.f;
        den[r] = 0.f;
        my_v[r] = 0.f;
        my_e[r] = 0;
    }
    for (int j = 0; j < k; ++j) {
        float bv[NT];
        int be[NT];
#pragma unroll
        for (int r = 0; r < NT; ++r) {
            bv[r] = -INFINITY;
            be[r] = 0x7fffffff;
#pragma unroll
            for (int i = 0; i < EPT; ++i) {
                const int e = lane + 32 * i;
                if (!taken[r][i] && (v[r][i] > bv[r] || (v[r][i] == bv[r] && e < be[r]))) {
                    bv[r] = v[r][i];
                    be[r] = e;
                }
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
#pragma unroll
            for (int r = 0; r < NT; ++r) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv[r], off);
                const int oe = __shfl_xor_sync(0xffffffffu, be[r], off);
                if (ov > bv[r] || (ov == bv[r] && oe < be[r])) {
                    bv[r] = ov;
                    be[r] = oe;
                }
            }
#pragma unroll
        for (int r = 0; r < NT; ++r) {
#pragma unroll
            for (int i = 0; i < EPT; ++i)
                if (lane + 32 * i == be[r]) taken[r][i] = true;
            if (j == 0) sel0[r] = bv[r];
            const float ex = expf(__fsub_rn(bv[r], sel0[r]));
            den[r] = __fadd_rn(den[r], ex);
            if (lane == j) {  // lane j keeps choice j
                my_v[r] = ex;
                my_e[r] = be[r];
            }
        }
    }
#pragma unroll
    for (int r = 0; r < NT; ++r) my_w[r] = __fdiv_rn(my_v[r], den[r]);
    return __any_sync(0xffffffffu, nan_seen);
}

// One 32-token chunk, by a whole CTA of 256 threads; `mask` is shared memory
// of 32 * EPT words.  The logits are read with ld.global.cg (from L2): when
// another CTA of this grid wrote them, no stale L1 line can be hit.
template <int EPT>
__device__ __forceinline__ void topk_chunk(const float* __restrict__ P, int KS, int T, int E, int E_pad,
                                           const float* __restrict__ bias, int k, int chunk,
                                           int32_t* __restrict__ topk_ids, float* __restrict__ topk_w,
                                           int32_t* __restrict__ rank, int32_t* __restrict__ hist, uint32_t* mask,
                                           int* __restrict__ error) {
    constexpr int EP = 32 * EPT;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int t0 = chunk * kRouterTokens;
    for (int i = tid; i < EP; i += 256) mask[i] = 0u;
    __syncthreads();
    // the logits of the warp's 4 tokens, loaded before any selection so that
    // the loads of all tokens are in flight together
    float vv[4][EPT];
    if (KS == 1) {
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int i = 0; i < EPT; ++i) {
                const int t = t0 + warp * 4 + r, e = lane + 32 * i;
                vv[r][i] = (t < T && e < E) ? __ldcg(P + (size_t)t * E_pad + e) : -INFINITY;
            }
    } else {
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int i = 0; i < EPT; ++i) {
                const int t = t0 + warp * 4 + r, e = lane + 32 * i;
                float part[kRouterMaxSlices];
#pragma unroll
                for (int ks = 0; ks < kRouterMaxSlices; ++ks)  // independent loads first
                    part[ks] = (ks < KS && t < T && e < E) ? __ldcg(P + ((size_t)ks * T + t) * E_pad + e) : 0.f;
                float acc = part[0];
#pragma unroll
                for (int ks = 1; ks < kRouterMaxSlices; ++ks)  // then the sum in slice order
                    if (ks < KS) acc = __fadd_rn(acc, part[ks]);
                vv[r][i] = (t < T && e < E) ? acc : -INFINITY;
            }
    }
    // the warp's 4 tokens selected together (their shuffle chains interleave)
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int i = 0; i < EPT; ++i) {
            const int e = lane + 32 * i;
            if (bias && e < E) vv[r][i] = __fadd_rn(vv[r][i], bias[e]);
        }
    int my_e[4];
    float my_w[4];
    if (warp_topk<EPT, 4>(vv, E, k, lane, my_e, my_w) && lane == 0) atomicOr(error, kErrDevice);
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int t = t0 + warp * 4 + r;
        if (t < T && lane < k) {
            topk_ids[(size_t)t * k + lane] = my_e[r];
            topk_w[(size_t)t * k + lane] = my_w[r];
            if (in_range(my_e[r], 0, E, error)) atomicOr(&mask[my_e[r]], 1u << (warp * 4 + r));
        }
    }
    __syncthreads();
    // chunk-local rank of each choice and the chunk's count per expert
    for (int i = tid; i < kRouterTokens * k; i += 256) {
        const int r = i / k, t = t0 + r;
        if (t < T) {
            const int e = topk_ids[(size_t)t * k + (i % k)];
            rank[(size_t)t * k + (i % k)] = in_range(e, 0, E, error) ? __popc(mask[e] & ((1u << r) - 1u)) : 0;
        }
    }
    for (int e = tid; e < E; e += 256) hist[(size_t)chunk * E + e] = __popc(mask[e]);
}

template <int EPT>
__global__ void __launch_bounds__(256) topk_kernel(const float* __restrict__ P, int KS, int T, int E, int E_pad,
                                                   const float* __restrict__ bias, int k,
                                                   int32_t* __restrict__ topk_ids, float* __restrict__ topk_w,
                                                   int32_t* __restrict__ rank, int32_t* __restrict__ hist,
                                                   int* __restrict__ error) {
    __shared__ uint32_t mask[32 * EPT];
    pdl_wait();
    pdl_trigger();
    topk_chunk<EPT>(P, KS, T, E, E_pad, bias, k, blockIdx.x, topk_ids, topk_w, rank, hist, mask, error);
}

// Few tokens (T <= kRouterSmallT): the router GEMM is far too small for the
// tensor cores to pay (one 128-token tile, a handful of CTAs, a weight split
// per call), so the CUDA cores compute the logits straight from the fp32
// weights, in two kernels.
//
// router_partial_kernel: CTA s owns rows [s*hs, (s+1)*hs) of Wr, about 128
// slices in all, and computes the partial logits of every token over them:
// P[s][t][e] = sum over its rows of x[t][h] * Wr[h][e], fp32 FMAs in row
// order.  Each SM thus reads only its own few KB of Wr and x, once (reading
// all of Wr for a block of tokens, as one kernel per token block must, made
// the loads the critical path: 192 KB per SM at one load round trip per 4 KB
// or so).  The slice is staged in shared memory (Wr rows with cp.async, x
// rows transposed to [h][t] fp32), then each thread accumulates a 4 x 4 block
// of (token, expert) sums per 64 x 64 output tile.
//
// router_finish_kernel: one CTA per token sums the slices in a fixed order
// (warp w sums its run of slices in order, then the 8 warp sums in order),
// adds the bias, and selects the top-k with its softmax weights.  The CTA that
// finishes last (an atomic ticket in the workspace, which it resets to zero
// for the next call) then builds the per-chunk expert masks of all tokens'
// choices, the ranks of each choice in its 32-token chunk, and the prefix
// sums that the scan kernel computes for larger T (expert offsets and the
// first slot of every (chunk, expert)), and clears the exact-path counters.
// Every CTA publishes its choices with a device-scope fence before taking its
// ticket, as in the classic threadfence reduction; nothing waits on another CTA.
constexpr int kRPTile = 64;         // output tile: 64 tokens x 64 experts, 4 x 4 per thread
constexpr int kRPTargetSlices = 128;
constexpr int kRPMaxLoads = 8;      // x vectors staged per thread (T <= 128, hs <= 128)
constexpr int kRFMaxChunks = kRouterSmallT / kRouterTokens;

__device__ __forceinline__ void cp_async4(void* smem_dst, const void* gmem_src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(
                     static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst))),
                 "l"(gmem_src)
                 : "memory");
}

__global__ void __launch_bounds__(256) router_partial_kernel(const uint16_t* __restrict__ x,
                                                             const float* __restrict__ Wr, int T, int H, int E,
                                                             int E_pad, int hs_max, float* __restrict__ P) {
    extern __shared__ float4 rp_smem[];
    const int T64 = (T + kRPTile - 1) / kRPTile * kRPTile;
    const int E64 = (E + kRPTile - 1) / kRPTile * kRPTile;
    float* xs = reinterpret_cast<float*>(rp_smem);  // [hs_max][T64]
    float* ws = xs + (size_t)hs_max * T64;           // [hs_max][E64]
    const int tid = threadIdx.x;
    const int s = blockIdx.x, h0 = s * hs_max, hs = min(hs_max, H - h0);
    pdl_wait();
    pdl_trigger();
    // Wr rows h0 .. h0 + hs (one contiguous block), columns padded with zeros to E64
    if (E % 4 == 0) {
        const int q = E / 4;
        for (int i = tid; i < hs * q; i += 256) {
            const int r = i / q, c = i - r * q;
            cp_async16(ws + (size_t)r * E64 + 4 * c, Wr + (size_t)(h0 + r) * E + 4 * c);
        }
    } else {
        for (int i = tid; i < hs * E; i += 256) {
            const int r = i / E, c = i - r * E;
            cp_async4(ws + (size_t)r * E64 + c, Wr + (size_t)(h0 + r) * E + c);
        }
    }
    for (int i = tid; i < hs * (E64 - E); i += 256) {
        const int r = i / (E64 - E);
        ws[(size_t)r * E64 + E + (i - r * (E64 - E))] = 0.f;
    }
    // x[t][h0 .. h0 + hs]: 8 bf16 per 16-byte load, every load in flight
    // before any store; stored transposed as fp32, tokens past T are zero
    const int hv = hs / 8;  // 16-byte vectors per token row
    uint4 v[kRPMaxLoads];
#pragma unroll
    for (int j = 0; j < kRPMaxLoads; ++j) {
        const int i = tid + 256 * j;
        const int t = i / hv, c = i - t * hv;
        v[j] = (t < T) ? __ldg(reinterpret_cast<const uint4*>(x + (size_t)t * H + h0) + c)
                       : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int j = 0; j < kRPMaxLoads; ++j) {
        const int i = tid + 256 * j;
        const int t = i / hv, c = i - t * hv;
        if (t < T64) {
            const uint32_t w4[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                xs[(size_t)(8 * c + 2 * m) * T64 + t] = __uint_as_float(w4[m] << 16);
                xs[(size_t)(8 * c + 2 * m + 1) * T64 + t] = __uint_as_float(w4[m] & 0xffff0000u);
            }
        }
    }
    cp_async_wait_all();
    __syncthreads();

    const int tx = tid & 15, ty = tid >> 4;
    float* out = P + (size_t)s * T * E_pad;
    for (int tt0 = 0; tt0 < T; tt0 += kRPTile)
        for (int te0 = 0; te0 < E; te0 += kRPTile) {
            float acc[4][4];
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int b = 0; b < 4; ++b) acc[a][b] = 0.f;
            const float* xp = xs + tt0 + 4 * ty;
            const float* wp = ws + te0 + 4 * tx;
#pragma unroll 8
            for (int h = 0; h < hs; ++h) {
                const float4 xv = *reinterpret_cast<const float4*>(xp + (size_t)h * T64);
                const float4 wv = *reinterpret_cast<const float4*>(wp + (size_t)h * E64);
                const float xa[4] = {xv.x, xv.y, xv.z, xv.w}, wa[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
                for (int a = 0; a < 4; ++a)
#pragma unroll
                    for (int b = 0; b < 4; ++b) acc[a][b] = fmaf(xa[a], wa[b], acc[a][b]);
            }
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                const int t = tt0 + 4 * ty + a;
                if (t >= T) continue;
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    const int e = te0 + 4 * tx + b;
                    if (e < E_pad) out[(size_t)t * E_pad + e] = acc[a][b];
                }
            }
        }
}

template <int EPT>
__global__ void __launch_bounds__(256) router_finish_kernel(const float* __restrict__ P, int KS, int T, int E,
                                                            int E_pad, const float* __restrict__ bias, int k,
                                                            int32_t* __restrict__ topk_ids,
                                                            float* __restrict__ topk_w, int32_t* __restrict__ rank,
                                                            int32_t* __restrict__ hist,
                                                            int32_t* __restrict__ offsets,
                                                            int32_t* __restrict__ counts,
                                                            unsigned int* __restrict__ ticket,
                                                            int* __restrict__ error) {
    constexpr int EP = 32 * EPT;
    __shared__ float part[8][EP];
    __shared__ uint32_t mask[kRFMaxChunks * kMaxExperts];
    __shared__ int32_t wsum[8];
    __shared__ int is_last;
    const int t = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    pdl_wait();
    pdl_trigger();
    // warp w: slices [w * per, (w + 1) * per) in order, kB slices' loads at a time
    constexpr int kB = EPT <= 2 ? 16 : 32 / EPT;
    const int per = (KS + 7) / 8;
    const int s0 = warp * per, s1 = min(KS, s0 + per);
    float acc[EPT];
#pragma unroll
    for (int i = 0; i < EPT; ++i) acc[i] = 0.f;
    for (int sb = s0; sb < s1; sb += kB) {
        float pv[kB][EPT];
#pragma unroll
        for (int u = 0; u < kB; ++u)
#pragma unroll
            for (int i = 0; i < EPT; ++i) {
                const int s = sb + u, e = lane + 32 * i;
                pv[u][i] = (s < s1 && e < E) ? __ldcg(P + ((size_t)s * T + t) * E_pad + e) : 0.f;
            }
#pragma unroll
        for (int u = 0; u < kB; ++u)
#pragma unroll
            for (int i = 0; i < EPT; ++i) acc[i] = __fadd_rn(acc[i], pv[u][i]);
    }
#pragma unroll
    for (int i = 0; i < EPT; ++i) part[warp][lane + 32 * i] = acc[i];
    __syncthreads();
    if (warp == 0) {
        float v[1][EPT];
#pragma unroll
        for (int i = 0; i < EPT; ++i) {
            const int e = lane + 32 * i;
            float l = part[0][e];
#pragma unroll
            for (int w = 1; w < 8; ++w) l = __fadd_rn(l, part[w][e]);
            if (bias && e < E) l = __fadd_rn(l, bias[e]);
            v[0][i] = e < E ? l : -INFINITY;
        }
        int my_e[1];
        float my_w[1];
        if (warp_topk<EPT, 1>(v, E, k, lane, my_e, my_w) && lane == 0) atomicOr(error, kErrDevice);
        if (lane < k) {
            topk_ids[(size_t)t * k + lane] = my_e[0];
            topk_w[(size_t)t * k + lane] = my_w[0];
        }
    }

    // ---- the last CTA: chunk masks, ranks, then the prefix sums
    __threadfence();  // this CTA's choices are visible device-wide before the ticket
    __syncthreads();
    if (tid == 0) is_last = atomicAdd(ticket, 1u) == gridDim.x - 1u;
    __syncthreads();
    if (!is_last) return;
    __threadfence();
    const int nchunk = (T + kRouterTokens - 1) / kRouterTokens;
    for (int i = tid; i < nchunk * E; i += 256) mask[i] = 0u;
    __syncthreads();
    for (int i = tid; i < T * k; i += 256) {
        const int tk = i / k;
        const int e = __ldcg(topk_ids + i);
        if (in_range(e, 0, E, error)) atomicOr(&mask[(tk / kRouterTokens) * E + e], 1u << (tk % kRouterTokens));
    }
    __syncthreads();
    for (int i = tid; i < T * k; i += 256) {
        const int tk = i / k;
        const int e = __ldcg(topk_ids + i);
        rank[i] = in_range(e, 0, E, error) ? __popc(mask[(tk / kRouterTokens) * E + e] & ((1u << (tk % kRouterTokens)) - 1u))
                                           : 0;
    }
    // per expert: first slot of each chunk relative to the expert, and its total
    int32_t tot = 0;
    if (tid < E) {
        for (int c = 0; c < nchunk; ++c) {
            hist[(size_t)c * E + tid] = tot;
            tot += __popc(mask[c * E + tid]);
        }
    }
    // exclusive prefix of the totals over the experts (E <= 256 = blockDim)
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
    const int32_t excl = before + incl - tot;
    if (tid < E) {
        for (int c = 0; c < nchunk; ++c) hist[(size_t)c * E + tid] += excl;
        offsets[tid] = excl;
    }
    if (tid == 0) {
        offsets[E] = all;
        counts[0] = 0;  // rows listed for the exact GEMM paths (GEMM1, GEMM2)
        counts[1] = 0;
        *ticket = 0u;   // ready for the next call
    }
}

// Thread layout: warp w owns tokens 4w..4w+3 of a 32-token chunk; lane l owns
// experts l + 32*i for i < EPT.

template <int NB, int NS>
cudaError_t launch_router_gemm(const uint16_t* x, const uint16_t* wsplit, int T, int H, int E, int E_pad,
                               int n_eb, int KS, int kb_per_slice, float* P, int* error, uint64_t timeout_ns,
                               cudaStream_t st, bool pdl) {
    using C = RCfg<NB, NS>;
    auto kern = router_gemm_kernel<NB, NS>;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [&] {
        attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    });
    if (attr_err != cudaSuccess) return attr_err;
    CUtensorMap tx, tw;
    if (!make_tensor_map_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, x, H, T, kRBK, kRTM,
                            CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    if (!make_tensor_map_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, wsplit, H, 3ull * E_pad, kRBK, NB,
                            CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    const dim3 grid((T + kRTM - 1) / kRTM, n_eb, KS);
    return launch_kernel(kern, grid, dim3(kRThreads), C::kSmem, st, pdl, tx, tw, T, H, E, E_pad, kb_per_slice, P,
                         error, timeout_ns);
}

cudaError_t launch_topk(const float* P, const RouterPlan& p, int T, int E, const float* bias, int k,
                        int32_t* topk_ids, float* topk_w, int32_t* rank, int32_t* hist, int* error, cudaStream_t st,
                        bool pdl) {
    const dim3 grid((T + kRouterTokens - 1) / kRouterTokens), block(256);
    if (E <= 32)
        return launch_kernel(topk_kernel<1>, grid, block, 0, st, pdl, P, p.KS, T, E, p.E_pad, bias, k, topk_ids,
                             topk_w, rank, hist, error);
    if (E <= 64)
        return launch_kernel(topk_kernel<2>, grid, block, 0, st, pdl, P, p.KS, T, E, p.E_pad, bias, k, topk_ids,
                             topk_w, rank, hist, error);
    if (E <= 128)
        return launch_kernel(topk_kernel<4>, grid, block, 0, st, pdl, P, p.KS, T, E, p.E_pad, bias, k, topk_ids,
                             topk_w, rank, hist, error);
    return launch_kernel(topk_kernel<8>, grid, block, 0, st, pdl, P, p.KS, T, E, p.E_pad, bias, k, topk_ids,
                         topk_w, rank, hist, error);
}

}  // namespace

RouterPlan router_plan(int64_t T, int64_t H, int64_t E) {
    RouterPlan p{};
    p.E_pad = E <= 128 ? (int)((E + 15) / 16 * 16) : (int)((E + 127) / 128 * 128);
    p.NB = p.E_pad <= 128 ? p.E_pad : 128;
    p.n_eb = (p.E_pad + p.NB - 1) / p.NB;
    p.small = T <= kRouterSmallT;
    if (p.small) {  // CUDA-core router: KS slices of hs rows of Wr (about kRPTargetSlices)
        const int64_t rows = (H + kRPTargetSlices - 1) / kRPTargetSlices;
        p.hs = (int)((rows + 7) / 8 * 8);
        p.KS = (int)((H + p.hs - 1) / p.hs);
        p.kb_per_slice = 0;
        return p;
    }
    const int nkb = (int)(H / kRBK);
    const long tiles = (long)((T + kRTM - 1) / kRTM) * p.n_eb;
    int ks = (int)(kRouterTargetCtas / (tiles > 0 ? tiles : 1));
    if (ks < 1) ks = 1;
    if (ks > kRouterMaxSlices) ks = kRouterMaxSlices;
    if (ks > nkb) ks = nkb;
    p.kb_per_slice = (nkb + ks - 1) / ks;
    p.KS = (nkb + p.kb_per_slice - 1) / p.kb_per_slice;
    return p;
}

cudaError_t launch_router(const uint16_t* x, const float* Wr, const float* bias, int T, int H, int E, int k,
                          uint16_t* wsplit, float* P, int32_t* topk_ids, float* topk_w, int32_t* rank,
                          int32_t* hist, int32_t* offsets, int32_t* counts, unsigned int* ticket, int* error,
                          uint64_t timeout_ns, cudaStream_t st, bool pdl) {
    const RouterPlan p = router_plan(T, H, E);
    cudaError_t e;
    if (p.small) {  // partial logits per slice of Wr; per token the sums and top-k; prefix sums
        const int T64 = (T + kRPTile - 1) / kRPTile * kRPTile, E64 = (E + kRPTile - 1) / kRPTile * kRPTile;
        const int smem = p.hs * (T64 + E64) * (int)sizeof(float);
        {
            static std::mutex mu;
            static int smem_set = 0;
            std::lock_guard<std::mutex> lock(mu);
            if (smem > smem_set) {
                e = cudaFuncSetAttribute(router_partial_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
                if (e != cudaSuccess) return e;
                smem_set = smem;
            }
        }
        e = launch_kernel(router_partial_kernel, dim3(p.KS), dim3(256), (size_t)smem, st, false, x, Wr, T, H, E,
                          p.E_pad, p.hs, P);
        if (e != cudaSuccess) return e;
        const dim3 grid(T), block(256);
        if (E <= 32)
            return launch_kernel(router_finish_kernel<1>, grid, block, 0, st, pdl, P, p.KS, T, E, p.E_pad, bias, k,
                                 topk_ids, topk_w, rank, hist, offsets, counts, ticket, error);
        if (E <= 64)
            return launch_kernel(router_finish_kernel<2>, grid, block, 0, st, pdl, P, p.KS, T, E, p.E_pad, bias, k,
                                 topk_ids, topk_w, rank, hist, offsets, counts, ticket, error);
        if (E <= 128)
            return launch_kernel(router_finish_kernel<4>, grid, block, 0, st, pdl, P, p.KS, T, E, p.E_pad, bias, k,
                                 topk_ids, topk_w, rank, hist, offsets, counts, ticket, error);
        return launch_kernel(router_finish_kernel<8>, grid, block, 0, st, pdl, P, p.KS, T, E, p.E_pad, bias, k,
                             topk_ids, topk_w, rank, hist, offsets, counts, ticket, error);
    }
    e = launch_kernel(router_split_kernel, dim3((H + 31) / 32, (p.E_pad + 31) / 32), dim3(256), 0, st, false, Wr, H,
                      E, p.E_pad, wsplit);
    if (e != cudaSuccess) return e;
    switch (p.NB) {
        case 16: e = launch_router_gemm<16, 6>(x, wsplit, T, H, E, p.E_pad, p.n_eb, p.KS, p.kb_per_slice, P, error, timeout_ns, st, pdl); break;
        case 32: e = launch_router_gemm<32, 6>(x, wsplit, T, H, E, p.E_pad, p.n_eb, p.KS, p.kb_per_slice, P, error, timeout_ns, st, pdl); break;
        case 48: e = launch_router_gemm<48, 5>(x, wsplit, T, H, E, p.E_pad, p.n_eb, p.KS, p.kb_per_slice, P, error, timeout_ns, st, pdl); break;
        case 64: e = launch_router_gemm<64, 5>(x, wsplit, T, H, E, p.E_pad, p.n_eb, p.KS, p.kb_per_slice, P, error, timeout_ns, st, pdl); break;
        case 80: e = launch_router_gemm<80, 4>(x, wsplit, T, H, E, p.E_pad, p.n_eb, p.KS, p.kb_per_slice, P, error, timeout_ns, st, pdl); break;
        case 96: e = launch_router_gemm<96, 4>(x, wsplit, T, H, E, p.E_pad, p.n_eb, p.KS, p.kb_per_slice, P, error, timeout_ns, st, pdl); break;
        case 112: e = launch_router_gemm<112, 3>(x, wsplit, T, H, E, p.E_pad, p.n_eb, p.KS, p.kb_per_slice, P, error, timeout_ns, st, pdl); break;
        default: e = launch_router_gemm<128, 3>(x, wsplit, T, H, E, p.E_pad, p.n_eb, p.KS, p.kb_per_slice, P, error, timeout_ns, st, pdl); break;
    }
    if (e != cudaSuccess) return e;
    return launch_topk(P, p, T, E, bias, k, topk_ids, topk_w, rank, hist, error, st, pdl);
}

}  // namespace moe

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
#include "router_small.cuh"

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

// The few-token router's kernels (router_small.cuh holds their bodies).
__global__ void __launch_bounds__(256) router_partial_kernel(const uint16_t* __restrict__ x,
                                                             const float* __restrict__ Wr, int T, int H, int E,
                                                             int E_pad, int hs_max, float* __restrict__ P) {
    extern __shared__ float4 rp_smem[];
    pdl_wait();
    pdl_trigger();
    router_partial_body(x, Wr, T, H, E, E_pad, hs_max, P, rp_smem, blockIdx.x);
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
    pdl_wait();
    pdl_trigger();
    router_finish_body<EPT>(P, KS, T, E, E_pad, bias, k, topk_ids, topk_w, rank, hist, offsets, counts, ticket,
                            error, blockIdx.x, gridDim.x);
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

// router_small.cuh -- the top-k selection, the few-token (CUDA-core) router
// and a per-token quantiser as device functions: used by router.cu's kernels
// and by the one-kernel layer (fused.cu), which must route and quantise
// exactly as the multi-kernel layer does.
#pragma once

#include <cuda_bf16.h>

#include "internal.h"

namespace moe {
namespace {

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

// Per-token dynamic quantisation of row t of x (bf16 [.][H]) by one CTA of
// 256 threads, the row held in registers (H <= 256 * 8 * kQtVec): s_x[t] =
// amax / 127 and the token's codes, written once (token-major) to q_tok
// [.][H].  The arithmetic of the per-slot quantisers of route.cu; the
// one-kernel layer runs it beside the router's partial logits, its gate/up
// GEMM gathering rows through the slot -> token map.
constexpr int kQtVec = 8;

__device__ __forceinline__ void quant_token_body(const uint16_t* __restrict__ x, int H, int t, float* __restrict__ s_x,
                                                 int8_t* __restrict__ q_tok) {
    __shared__ float red_max[8];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint4* row = reinterpret_cast<const uint4*>(x + (size_t)t * H);
    const int nv = H / 8;
    uint4 v[kQtVec];
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < kQtVec; ++i) {
        const int idx = tid + 256 * i;
        v[i] = idx < nv ? __ldg(row + idx) : make_uint4(0u, 0u, 0u, 0u);
        const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            amax = fmaxf(amax, fabsf(__uint_as_float((w[j] & 0xffffu) << 16)));
            amax = fmaxf(amax, fabsf(__uint_as_float(w[j] & 0xffff0000u)));
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    if (lane == 0) red_max[warp] = amax;
    __syncthreads();
    amax = red_max[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) amax = fmaxf(amax, red_max[i]);
    const float s = __fdiv_rn(amax, 127.0f);
    if (tid == 0) s_x[t] = s;
#pragma unroll
    for (int i = 0; i < kQtVec; ++i) {
        const int idx = tid + 256 * i;
        if (idx >= nv) break;
        const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
        int q[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            q[2 * j] = quant_code_div(__uint_as_float((w[j] & 0xffffu) << 16), s);
            q[2 * j + 1] = quant_code_div(__uint_as_float(w[j] & 0xffff0000u), s);
        }
        reinterpret_cast<uint2*>(q_tok + (size_t)t * H)[idx] = pack_codes_s8(q);
    }
    __syncthreads();  // red_max is reused by the CTA's next token
}

// The body of router_partial_kernel for slice s; rp_smem: the kernel's dynamic
// shared memory (router_plan's partial_smem bytes).
__device__ __forceinline__ void router_partial_body(const uint16_t* __restrict__ x, const float* __restrict__ Wr,
                                                    int T, int H, int E, int E_pad, int hs_max,
                                                    float* __restrict__ P, float4* rp_smem, int s) {
    const int T64 = (T + kRPTile - 1) / kRPTile * kRPTile;
    const int E64 = (E + kRPTile - 1) / kRPTile * kRPTile;
    float* xs = reinterpret_cast<float*>(rp_smem);  // [hs_max][T64]
    float* ws = xs + (size_t)hs_max * T64;           // [hs_max][E64]
    const int tid = threadIdx.x;
    const int h0 = s * hs_max, hs = min(hs_max, H - h0);
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

// The body of router_finish_kernel for token t of a grid of n_cta CTAs (one
// per token); the CTA that takes the last ticket builds the routing tables
// and returns true (every thread), the others return false.  TABLES = false:
// the token's choices only (no ticket, no tables; returns false).
template <int EPT, bool TABLES = true>
__device__ __forceinline__ bool router_finish_body(const float* __restrict__ P, int KS, int T, int E, int E_pad,
                                                   const float* __restrict__ bias, int k,
                                                   int32_t* __restrict__ topk_ids, float* __restrict__ topk_w,
                                                   int32_t* __restrict__ rank, int32_t* __restrict__ hist,
                                                   int32_t* __restrict__ offsets, int32_t* __restrict__ counts,
                                                   unsigned int* __restrict__ ticket, int* __restrict__ error, int t,
                                                   int n_cta) {
    constexpr int EP = 32 * EPT;
    __shared__ float part[8][EP];
    __shared__ uint32_t mask[kRFMaxChunks * kMaxExperts];
    __shared__ int32_t wsum[8];
    __shared__ int is_last;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
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

    if (!TABLES) {
        __syncthreads();  // part is reused by the CTA's next token
        return false;
    }
    // ---- the last CTA: chunk masks, ranks, then the prefix sums
    __threadfence();  // this CTA's choices are visible device-wide before the ticket
    __syncthreads();
    if (tid == 0) is_last = atomicAdd(ticket, 1u) == (unsigned)n_cta - 1u;
    __syncthreads();
    if (!is_last) return false;
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
    return true;
}

}  // namespace
}  // namespace moe

// route.cu -- routing and activation quantisation.
//
//   scan_kernel          expert offsets (exclusive prefix over experts) and the
//                        first slot of every (chunk, expert).
//   permute_quant_kernel slot of every (token, choice); per-token dynamic INT8
//                        quantisation of x, scattered into the token's slots
//                        (one to eight warps per token, by row length).
//   permute_quant_cta_kernel  the same with one CTA per token, the row held in
//                        registers: for few tokens (decode), where a warp per
//                        token leaves most of the GPU idle.
//   permute_quant_smooth_kernel  the same with SmoothQuant-folded activations
//                        per expert: one warp per (token, choice), a scale per slot.
//
// Routing pre-processing that reserves a contiguous slot range per expert:
// "Tencent Hunyuan AI Infra on Hopper" (pnsm.cn), section 1.3.  Per-token dynamic quantisation q = clamp(round(x/s)),
// s = amax/127: "W8A8 quantisation of MiniMax-M3 on K100AI" (mhpn.cn),
// section 2.1.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"

namespace moe {
namespace {

__device__ __forceinline__ float bf16_bits_to_float(uint32_t b) { return __uint_as_float(b << 16); }

// max |v| over 8 bf16 values (one 16-byte vector).
__device__ __forceinline__ float absmax8(const uint4 v) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float m = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        m = fmaxf(m, fabsf(bf16_bits_to_float(w[j] & 0xffffu)));
        m = fmaxf(m, fabsf(bf16_bits_to_float(w[j] >> 16)));
    }
    return m;
}

// Codes of 8 bf16 values (one 16-byte vector) and their L1 norm, added to l1.
__device__ __forceinline__ void quant8(const uint4 v, float s, int (&q)[8], int& l1) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        q[2 * j] = quant_code_div(bf16_bits_to_float(w[j] & 0xffffu), s);
        q[2 * j + 1] = quant_code_div(bf16_bits_to_float(w[j] >> 16), s);
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) l1 += abs(q[j]);
}

// One CTA.  hist [nchunk][E] holds per-chunk counts on entry and the first
// slot of every (chunk, expert) on exit; offsets[E+1] receives the exclusive
// prefix of the expert totals.  Thread (e, p) scans rows p*L..p*L+L-1 of
// column e; the parts are then combined.  The table is staged in shared
// memory when it fits.
constexpr int kScanThreads = 1024;
constexpr int kScanSmemInts = 40960;

__global__ void __launch_bounds__(kScanThreads) scan_kernel(int32_t* __restrict__ hist, int nchunk,
                                                            int E, int32_t* __restrict__ offsets,
                                                            int32_t* __restrict__ counts, int use_smem) {
    extern __shared__ int32_t tab_s[];
    __shared__ int32_t part_tot[kScanThreads];
    __shared__ int32_t total[kMaxExperts + 1];
    const int tid = threadIdx.x;
    const int n = nchunk * E;
    int32_t* tab = use_smem ? tab_s : hist;
    pdl_wait();
    pdl_trigger();
    if (tid < 2) counts[tid] = 0;  // rows listed for the exact GEMM path (GEMM1, GEMM2)
    if (use_smem) {
        for (int i = tid; i < n; i += kScanThreads) tab[i] = hist[i];
        __syncthreads();
    }
    int P = kScanThreads / E;  // parts per expert
    if (P > nchunk) P = nchunk;
    if (P < 1) P = 1;
    const int L = (nchunk + P - 1) / P;
    const int e = tid % E, p = tid / E;
    const bool active = (tid < E * P);
    int32_t run = 0;
    if (active) {
        const int r0 = p * L, r1 = min(nchunk, r0 + L);
        for (int r = r0; r < r1; ++r) {
            const int32_t v = tab[(size_t)r * E + e];
            tab[(size_t)r * E + e] = run;
            run += v;
        }
        part_tot[tid] = run;
    }
    __syncthreads();
    if (tid < E) {  // combine the parts of expert tid
        int32_t s = 0;
        for (int q = 0; q < P; ++q) {
            const int32_t v = part_tot[q * E + tid];
            part_tot[q * E + tid] = s;
            s += v;
        }
        total[tid] = s;
    }
    __syncthreads();
    if (tid == 0) {
        int32_t s = 0;
        for (int i = 0; i < E; ++i) {
            const int32_t v = total[i];
            total[i] = s;
            s += v;
        }
        total[E] = s;
    }
    __syncthreads();
    if (active) {
        const int r0 = p * L, r1 = min(nchunk, r0 + L);
        const int32_t add = total[e] + part_tot[tid];
        for (int r = r0; r < r1; ++r) tab[(size_t)r * E + e] += add;
    }
    for (int i = tid; i <= E; i += kScanThreads) offsets[i] = total[i];
    if (use_smem) {
        __syncthreads();
        for (int i = tid; i < n; i += kScanThreads) hist[i] = tab[i];
    }
}

// WPT warps per token (1, 2, 4 or 8), 8 warps per CTA.  With topk_ids ==
// nullptr the token's single "slot" is the token itself (the dense linear
// layer).  Besides the codes, every token gets the L1 norm of its code row;
// rows above kExactL1 are flagged in each of their slots and listed for the
// exact path of the GEMM.
// Each warp of a token takes every WPT-th 16-byte vector of the row; the row
// maximum and the L1 norm are combined through shared memory.  The amax pass
// and the code pass each read the row (the second mostly from cache).  Split
// rows keep more loads in flight per SM than one warp per token, whose single
// load in flight per lane left the dense linear layer's quantiser at a third
// of the HBM rate.  (Measured at T = 8192 with one warp per token: staging
// rows through shared memory with cp.async, 4 tokens per CTA, was slower: 53
// against 52 us.)  Registers are capped for 8 CTAs per SM (measured with one
// warp per token at T = 8192: 54 -> 51 us; unrolling the loops spills).
constexpr int kPqWarps = 8;

template <int WPT>
__global__ void __launch_bounds__(32 * kPqWarps, 8) permute_quant_kernel(
    const uint16_t* __restrict__ x, const int32_t* __restrict__ topk_ids,
    const int32_t* __restrict__ rank, const int32_t* __restrict__ base, int T, int H, int E, int k,
    int32_t* __restrict__ slot_of, int32_t* __restrict__ slot_token, float* __restrict__ s_x,
    float* __restrict__ s_slot, uint16_t* __restrict__ q16, int8_t* __restrict__ q8,
    int32_t* __restrict__ flags, int32_t* __restrict__ fb_list, int32_t* __restrict__ fb_count,
    int* __restrict__ error) {
    static_assert(WPT == 1 || WPT == 2 || WPT == 4 || WPT == 8, "warps per token");
    __shared__ float red_max[kPqWarps];
    __shared__ int red_l1[kPqWarps];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int sub = warp % WPT;  // this warp's share of the token's row
    const int t = blockIdx.x * (kPqWarps / WPT) + warp / WPT;
    pdl_wait();
    pdl_trigger();
    if (WPT == 1 && t >= T) return;
    const bool live = t < T;  // with WPT > 1 every warp reaches the block barriers
    int my_slot = t;  // -1: out of range (checked build), its writes skipped
    if (live && topk_ids != nullptr && lane < k) {
        const int e = topk_ids[(size_t)t * k + lane];
        my_slot = in_range(e, 0, E, error) ? base[(size_t)(t / kRouterTokens) * E + e] + rank[(size_t)t * k + lane]
                                           : -1;
        if (my_slot >= 0 && !in_range(my_slot, 0, (long long)T * k, error)) my_slot = -1;
        if (sub == 0) {
            slot_of[(size_t)t * k + lane] = my_slot;
            if (!kChecked || my_slot >= 0) slot_token[my_slot] = t;
        }
    }
    const int nk = (topk_ids != nullptr) ? k : 1;
    const uint4* row = reinterpret_cast<const uint4*>(x + (size_t)(live ? t : 0) * H);
    const int nv = live ? H / 8 : 0;  // 8 bf16 per 16-byte vector
    float amax = 0.f;
    for (int i = sub * 32 + lane; i < nv; i += 32 * WPT) amax = fmaxf(amax, absmax8(__ldg(row + i)));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    if (WPT > 1) {
        if (lane == 0) red_max[warp] = amax;
        __syncthreads();
        const int w0 = warp - sub;
#pragma unroll
        for (int w = 0; w < WPT; ++w) amax = fmaxf(amax, red_max[w0 + w]);
    }
    const float s = __fdiv_rn(amax, 127.0f);
    if (live && sub == 0) {
        if (lane == 0) s_x[t] = s;
        if (lane < nk && (!kChecked || my_slot >= 0)) s_slot[my_slot] = s;
    }
    int slots[kMaxTopK];  // slot j of the token is lane j's my_slot (taken before the lanes diverge)
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) slots[j] = __shfl_sync(0xffffffffu, my_slot, j);
    int l1 = 0;
    for (int i = sub * 32 + lane; i < nv; i += 32 * WPT) {
        int q[8];
        quant8(__ldg(row + i), s, q, l1);
        if (q16 != nullptr) {
            const uint4 ov = pack_codes_f16(q);
            for (int j = 0; j < nk; ++j)
                if (!kChecked || slots[j] >= 0) reinterpret_cast<uint4*>(q16 + (size_t)slots[j] * H)[i] = ov;
        }
        if (q8 != nullptr) {
            const uint2 ov8 = pack_codes_s8(q);
            for (int j = 0; j < nk; ++j)
                if (!kChecked || slots[j] >= 0) reinterpret_cast<uint2*>(q8 + (size_t)slots[j] * H)[i] = ov8;
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) l1 += __shfl_xor_sync(0xffffffffu, l1, off);
    if (WPT > 1) {
        if (lane == 0) red_l1[warp] = l1;
        __syncthreads();
        if (sub != 0) return;
        l1 = 0;
#pragma unroll
        for (int w = 0; w < WPT; ++w) l1 += red_l1[warp + w];
    }
    const int flagged = l1 > kExactL1 ? 1 : 0;
    if (live && lane < nk && (!kChecked || my_slot >= 0)) {
        flags[my_slot] = flagged;
        if (flagged) fb_list[atomicAdd(fb_count, 1)] = my_slot;
    }
}

// One CTA of 256 threads per token; the same outputs as permute_quant_kernel.
// H <= 16384, so a thread holds at most kPqVec 16-byte vectors of the row.
constexpr int kPqVec = 8;

__global__ void __launch_bounds__(256) permute_quant_cta_kernel(
    const uint16_t* __restrict__ x, const int32_t* __restrict__ topk_ids,
    const int32_t* __restrict__ rank, const int32_t* __restrict__ base, int T, int H, int E, int k,
    int32_t* __restrict__ slot_of, int32_t* __restrict__ slot_token, float* __restrict__ s_x,
    float* __restrict__ s_slot, uint16_t* __restrict__ q16, int8_t* __restrict__ q8,
    int32_t* __restrict__ flags, int32_t* __restrict__ fb_list, int32_t* __restrict__ fb_count,
    int* __restrict__ error) {
    __shared__ float red_max[8];
    __shared__ int red_l1[8];
    __shared__ int slots_s[kMaxTopK];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int t = blockIdx.x;
    pdl_wait();
    pdl_trigger();
    if (t >= T) return;
    const int nk = (topk_ids != nullptr) ? k : 1;
    if (tid < nk) {
        int my_slot = t;  // -1: out of range (checked build), its writes skipped
        if (topk_ids != nullptr) {
            const int e = topk_ids[(size_t)t * k + tid];
            my_slot = in_range(e, 0, E, error) ? base[(size_t)(t / kRouterTokens) * E + e] + rank[(size_t)t * k + tid]
                                               : -1;
            if (my_slot >= 0 && !in_range(my_slot, 0, (long long)T * k, error)) my_slot = -1;
            slot_of[(size_t)t * k + tid] = my_slot;
            if (!kChecked || my_slot >= 0) slot_token[my_slot] = t;
        }
        slots_s[tid] = my_slot;
    }
    const uint4* row = reinterpret_cast<const uint4*>(x + (size_t)t * H);
    const int nv = H / 8;  // 8 bf16 per 16-byte vector
    uint4 v[kPqVec];
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < kPqVec; ++i) {
        const int idx = tid + 256 * i;
        v[i] = idx < nv ? __ldg(row + idx) : make_uint4(0u, 0u, 0u, 0u);
        const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            amax = fmaxf(amax, fabsf(bf16_bits_to_float(w[j] & 0xffffu)));
            amax = fmaxf(amax, fabsf(bf16_bits_to_float(w[j] >> 16)));
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    if (lane == 0) red_max[warp] = amax;
    __syncthreads();  // also publishes slots_s
    amax = red_max[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) amax = fmaxf(amax, red_max[i]);
    const float s = __fdiv_rn(amax, 127.0f);
    if (tid == 0) s_x[t] = s;
    if (tid < nk && (!kChecked || slots_s[tid] >= 0)) s_slot[slots_s[tid]] = s;
    int l1 = 0;
#pragma unroll
    for (int i = 0; i < kPqVec; ++i) {
        const int idx = tid + 256 * i;
        if (idx >= nv) break;
        int q[8];
        quant8(v[i], s, q, l1);
        if (q16 != nullptr) {
            const uint4 ov = pack_codes_f16(q);
            for (int j = 0; j < nk; ++j)
                if (!kChecked || slots_s[j] >= 0) reinterpret_cast<uint4*>(q16 + (size_t)slots_s[j] * H)[idx] = ov;
        }
        if (q8 != nullptr) {
            const uint2 ov8 = pack_codes_s8(q);
            for (int j = 0; j < nk; ++j)
                if (!kChecked || slots_s[j] >= 0) reinterpret_cast<uint2*>(q8 + (size_t)slots_s[j] * H)[idx] = ov8;
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) l1 += __shfl_xor_sync(0xffffffffu, l1, off);
    if (lane == 0) red_l1[warp] = l1;
    __syncthreads();
    if (tid < nk) {
        int tot = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) tot += red_l1[i];
        const int flagged = tot > kExactL1 ? 1 : 0;
        if (!kChecked || slots_s[tid] >= 0) {
            flags[slots_s[tid]] = flagged;
            if (flagged) fb_list[atomicAdd(fb_count, 1)] = slots_s[tid];
        }
    }
}

// SmoothQuant-folded activations, per expert ("W8A8 quantisation of
// MiniMax-M3 on K100AI" (mhpn.cn), section 2.2: part of the activations'
// quantisation difficulty moves onto the weights through a per-channel
// factor, calibrated per expert).  The factor s_e[h] multiplies the weights'
// input channel h offline; here the activation is multiplied by its correctly
// rounded reciprocal.  A slot's row then depends on its expert, so one warp
// per (token, choice) quantises its own row with its own scale.
__device__ __forceinline__ void smooth8(const uint4 xv, const float4 r0, const float4 r1, float (&v)[8]) {
    const uint32_t w[4] = {xv.x, xv.y, xv.z, xv.w};
    const float r[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        v[2 * j] = __fmul_rn(bf16_bits_to_float(w[j] & 0xffffu), r[2 * j]);
        v[2 * j + 1] = __fmul_rn(bf16_bits_to_float(w[j] >> 16), r[2 * j + 1]);
    }
}

// rcp[i] = the correctly rounded reciprocal of smooth[i] (once per call,
// before the quantisers; n a multiple of 4).
__global__ void __launch_bounds__(256) smooth_rcp_kernel(const float* __restrict__ smooth, int64_t n4,
                                                         float* __restrict__ rcp) {
    pdl_wait();
    pdl_trigger();
    for (int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x; i < n4; i += (int64_t)gridDim.x * 256) {
        const float4 f = reinterpret_cast<const float4*>(smooth)[i];
        reinterpret_cast<float4*>(rcp)[i] = make_float4(__frcp_rn(f.x), __frcp_rn(f.y), __frcp_rn(f.z), __frcp_rn(f.w));
    }
}

__global__ void __launch_bounds__(256) permute_quant_smooth_kernel(
    const uint16_t* __restrict__ x, const float* __restrict__ rcp, const int32_t* __restrict__ topk_ids,
    const int32_t* __restrict__ rank, const int32_t* __restrict__ base, int T, int H, int E, int k,
    int32_t* __restrict__ slot_of, int32_t* __restrict__ slot_token, float* __restrict__ s_x,
    float* __restrict__ s_slot, uint16_t* __restrict__ q16, int8_t* __restrict__ q8, int32_t* __restrict__ flags,
    int32_t* __restrict__ fb_list, int32_t* __restrict__ fb_count, int* __restrict__ error) {
    const int lane = threadIdx.x & 31;
    const int64_t c = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);  // choice t * k + j
    pdl_wait();
    pdl_trigger();
    if (c >= (int64_t)T * k) return;
    const int t = (int)(c / k);
    const int e = topk_ids[c];
    if (!in_range(e, 0, E, error)) return;  // checked build: the choice is skipped
    const int slot = base[(size_t)(t / kRouterTokens) * E + e] + rank[c];
    if (!in_range(slot, 0, (long long)T * k, error)) return;
    if (lane == 0) {
        slot_of[c] = slot;
        slot_token[slot] = t;
    }
    const uint4* row = reinterpret_cast<const uint4*>(x + (size_t)t * H);
    const float4* fr = reinterpret_cast<const float4*>(rcp + (size_t)e * H);
    const int nv = H / 8;  // 8 bf16 per 16-byte vector
    float amax = 0.f;
    for (int i = lane; i < nv; i += 32) {
        float v[8];
        smooth8(__ldg(row + i), __ldg(fr + 2 * i), __ldg(fr + 2 * i + 1), v);
#pragma unroll
        for (int m = 0; m < 8; ++m) amax = fmaxf(amax, fabsf(v[m]));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    const float s = __fdiv_rn(amax, 127.0f);
    if (lane == 0) {
        s_slot[slot] = s;
        if (c - (int64_t)t * k == 0) s_x[t] = s;
    }
    int l1 = 0;
    for (int i = lane; i < nv; i += 32) {
        float v[8];
        smooth8(__ldg(row + i), __ldg(fr + 2 * i), __ldg(fr + 2 * i + 1), v);
        int q[8];
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            q[m] = quant_code_div(v[m], s);
            l1 += abs(q[m]);
        }
        if (q16 != nullptr) reinterpret_cast<uint4*>(q16 + (size_t)slot * H)[i] = pack_codes_f16(q);
        if (q8 != nullptr) reinterpret_cast<uint2*>(q8 + (size_t)slot * H)[i] = pack_codes_s8(q);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) l1 += __shfl_xor_sync(0xffffffffu, l1, off);
    if (lane == 0) {
        const int flagged = l1 > kExactL1 ? 1 : 0;
        flags[slot] = flagged;
        if (flagged) fb_list[atomicAdd(fb_count, 1)] = slot;
    }
}

// The same with one CTA of 256 threads per (token, choice) and the smoothed
// row in registers (H <= 256 * 8 * kSmVec): for few slots (decode).  It takes
// the factors themselves and forms each reciprocal where it is used, so that
// no table (and no extra launch) is needed for a few rows.
constexpr int kSmVec = 8;

__device__ __forceinline__ float4 rcp4(const float4 f) {
    return make_float4(__frcp_rn(f.x), __frcp_rn(f.y), __frcp_rn(f.z), __frcp_rn(f.w));
}

__global__ void __launch_bounds__(256) permute_quant_smooth_cta_kernel(
    const uint16_t* __restrict__ x, const float* __restrict__ smooth, const int32_t* __restrict__ topk_ids,
    const int32_t* __restrict__ rank, const int32_t* __restrict__ base, int T, int H, int E, int k,
    int32_t* __restrict__ slot_of, int32_t* __restrict__ slot_token, float* __restrict__ s_x,
    float* __restrict__ s_slot, uint16_t* __restrict__ q16, int8_t* __restrict__ q8, int32_t* __restrict__ flags,
    int32_t* __restrict__ fb_list, int32_t* __restrict__ fb_count, int* __restrict__ error) {
    __shared__ float red_max[8];
    __shared__ int red_l1[8];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t c = blockIdx.x;
    pdl_wait();
    pdl_trigger();
    if (c >= (int64_t)T * k) return;
    const int t = (int)(c / k);
    const int e = topk_ids[c];
    if (!in_range(e, 0, E, error)) return;  // checked build: the choice is skipped (CTA-uniform)
    const int slot = base[(size_t)(t / kRouterTokens) * E + e] + rank[c];
    if (!in_range(slot, 0, (long long)T * k, error)) return;
    if (tid == 0) {
        slot_of[c] = slot;
        slot_token[slot] = t;
    }
    const uint4* row = reinterpret_cast<const uint4*>(x + (size_t)t * H);
    const float4* fr = reinterpret_cast<const float4*>(smooth + (size_t)e * H);
    const int nv = H / 8;
    float v[kSmVec][8];
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < kSmVec; ++i) {
        const int idx = tid + 256 * i;
        if (idx < nv) {
            smooth8(__ldg(row + idx), rcp4(__ldg(fr + 2 * idx)), rcp4(__ldg(fr + 2 * idx + 1)), v[i]);
        } else {
#pragma unroll
            for (int m = 0; m < 8; ++m) v[i][m] = 0.f;
        }
#pragma unroll
        for (int m = 0; m < 8; ++m) amax = fmaxf(amax, fabsf(v[i][m]));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    if (lane == 0) red_max[warp] = amax;
    __syncthreads();
    amax = red_max[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) amax = fmaxf(amax, red_max[i]);
    const float s = __fdiv_rn(amax, 127.0f);
    if (tid == 0) {
        s_slot[slot] = s;
        if (c - (int64_t)t * k == 0) s_x[t] = s;
    }
    int l1 = 0;
#pragma unroll
    for (int i = 0; i < kSmVec; ++i) {
        const int idx = tid + 256 * i;
        if (idx >= nv) break;
        int q[8];
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            q[m] = quant_code_div(v[i][m], s);
            l1 += abs(q[m]);
        }
        if (q16 != nullptr) reinterpret_cast<uint4*>(q16 + (size_t)slot * H)[idx] = pack_codes_f16(q);
        if (q8 != nullptr) reinterpret_cast<uint2*>(q8 + (size_t)slot * H)[idx] = pack_codes_s8(q);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) l1 += __shfl_xor_sync(0xffffffffu, l1, off);
    if (lane == 0) red_l1[warp] = l1;
    __syncthreads();
    if (tid == 0) {
        int tot = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) tot += red_l1[i];
        const int flagged = tot > kExactL1 ? 1 : 0;
        flags[slot] = flagged;
        if (flagged) fb_list[atomicAdd(fb_count, 1)] = slot;
    }
}

}  // namespace

cudaError_t launch_scan(int32_t* hist, int nchunk, int E, int32_t* offsets, int32_t* counts,
                        cudaStream_t st, bool pdl) {
    const long n = (long)nchunk * E;
    const int use_smem = n <= kScanSmemInts ? 1 : 0;
    const size_t smem = use_smem ? (size_t)n * sizeof(int32_t) : 0;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t err = cudaFuncSetAttribute(scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               kScanSmemInts * (int)sizeof(int32_t));
        if (err != cudaSuccess) return err;
        attr_set = true;
    }
    return launch_kernel(scan_kernel, dim3(1), dim3(kScanThreads), smem, st, pdl, hist, nchunk, E, offsets, counts,
                         use_smem);
}

cudaError_t launch_permute_quant(const uint16_t* x, const int32_t* topk_ids, const int32_t* rank,
                                 const int32_t* hist, int T, int H, int E, int k, int32_t* slot_of,
                                 int32_t* slot_token, float* s_x, float* s_slot, uint16_t* q16, int8_t* q8,
                                 int32_t* flags, int32_t* fb_list, int32_t* fb_count, int* error, cudaStream_t st,
                                 bool pdl) {
    if (T == 0) return cudaSuccess;
    // few tokens: one CTA per token (measured at T = 8192: a warp per token
    // takes 52 us, a CTA per token 96 us; at T = 64, 8 us against 17 us)
#ifndef MOE_PQ_CTA_TOKENS_PER_SM
#define MOE_PQ_CTA_TOKENS_PER_SM 8
#endif
    if ((long)T <= (long)MOE_PQ_CTA_TOKENS_PER_SM * num_sms() && H <= 256 * 8 * kPqVec)
        return launch_kernel(permute_quant_cta_kernel, dim3(T), dim3(256), 0, st, pdl, x, topk_ids, rank, hist, T,
                             H, E, k, slot_of, slot_token, s_x, s_slot, q16, q8, flags, fb_list, fb_count, error);
    // warps per token: about four 16-byte vectors per lane (measured on the
    // three layer shapes, quantiser time in us for 1 / 2 / 4 / 8 warps per
    // token: H = 4096, T = 4096, one slot: 34.1 / 31.8 / 27.9 / 29.3;
    // H = 4096, T = 8192, top-2: 51.5 / 45.2 / 43.2 / 50.4; H = 7168,
    // T = 4096, top-8: 102.4 / 100.2 / 94.7 / 90.4)
#ifndef MOE_PQ_WPT
    const int per_lane4 = (H / 8 + 127) / 128;
    const int wpt = per_lane4 <= 1 ? 1 : per_lane4 <= 2 ? 2 : per_lane4 <= 4 ? 4 : 8;
#else
    const int wpt = MOE_PQ_WPT;
#endif
    const dim3 grid((unsigned)(((long)T * wpt + kPqWarps - 1) / kPqWarps)), block(32 * kPqWarps);
    if (wpt == 8)
        return launch_kernel(permute_quant_kernel<8>, grid, block, 0, st, pdl, x, topk_ids, rank, hist, T, H, E, k,
                             slot_of, slot_token, s_x, s_slot, q16, q8, flags, fb_list, fb_count, error);
    if (wpt == 4)
        return launch_kernel(permute_quant_kernel<4>, grid, block, 0, st, pdl, x, topk_ids, rank, hist, T, H, E, k,
                             slot_of, slot_token, s_x, s_slot, q16, q8, flags, fb_list, fb_count, error);
    if (wpt == 2)
        return launch_kernel(permute_quant_kernel<2>, grid, block, 0, st, pdl, x, topk_ids, rank, hist, T, H, E, k,
                             slot_of, slot_token, s_x, s_slot, q16, q8, flags, fb_list, fb_count, error);
    return launch_kernel(permute_quant_kernel<1>, grid, block, 0, st, pdl, x, topk_ids, rank, hist, T, H, E, k,
                         slot_of, slot_token, s_x, s_slot, q16, q8, flags, fb_list, fb_count, error);
}

cudaError_t launch_permute_quant_smooth(const uint16_t* x, const float* smooth, float* rcp,
                                        const int32_t* topk_ids, const int32_t* rank, const int32_t* hist, int T,
                                        int H, int E, int k, int32_t* slot_of, int32_t* slot_token, float* s_x,
                                        float* s_slot, uint16_t* q16, int8_t* q8, int32_t* flags, int32_t* fb_list,
                                        int32_t* fb_count, int* error, cudaStream_t st, bool pdl) {
    if (T == 0) return cudaSuccess;
    const int64_t n = (int64_t)T * k;
    // few slots: a CTA per slot (as the plain quantiser's threshold), reciprocals formed in place
    if (n <= (int64_t)MOE_PQ_CTA_TOKENS_PER_SM * num_sms() && H <= 256 * 8 * kSmVec)
        return launch_kernel(permute_quant_smooth_cta_kernel, dim3((unsigned)n), dim3(256), 0, st, pdl, x, smooth,
                             topk_ids, rank, hist, T, H, E, k, slot_of, slot_token, s_x, s_slot, q16, q8, flags,
                             fb_list, fb_count, error);
    // many slots: the reciprocal table once, then a warp per slot
    const int64_t n4 = (int64_t)E * H / 4;
    int64_t blocks = (n4 + 255) / 256;
    if (blocks > 4L * num_sms()) blocks = 4L * num_sms();
    cudaError_t e = launch_kernel(smooth_rcp_kernel, dim3((unsigned)blocks), dim3(256), 0, st, pdl, smooth, n4, rcp);
    if (e != cudaSuccess) return e;
    return launch_kernel(permute_quant_smooth_kernel, dim3((unsigned)((n + 7) / 8)), dim3(256), 0, st, pdl, x, rcp,
                         topk_ids, rank, hist, T, H, E, k, slot_of, slot_token, s_x, s_slot, q16, q8, flags,
                         fb_list, fb_count, error);
}

}  // namespace moe

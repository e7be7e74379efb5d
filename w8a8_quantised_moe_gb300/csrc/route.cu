// route.cu -- routing and activation quantisation.
//
//   router_topk_kernel   FP32 router logits, top-k with ties to the lower
//                        expert index, softmax over the selected logits, and
//                        per 32-token chunk: the count of tokens per expert and
//                        each choice's rank among the chunk's tokens of that
//                        expert.
//   scan_kernel          expert offsets (exclusive prefix over experts) and the
//                        first slot of every (chunk, expert).
//   permute_quant_kernel slot of every (token, choice); per-token dynamic INT8
//                        quantisation of x, scattered into the token's slots.
//
// Gate -> top-k -> routing pre-processing that reserves a contiguous slot
// range per expert: "Tencent Hunyuan AI Infra on Hopper" (pnsm.cn), section
// 1.3.  FP32 router: "DeepSeek V4 950 FP8 inference on H100" (lpnh.cn),
// section 4.1.  Per-token dynamic quantisation q = clamp(round(x/s)),
// s = amax/127: "W8A8 quantisation of MiniMax-M3 on K100AI" (mhpn.cn),
// section 2.1.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"

namespace moe {
namespace {

constexpr int RT = kRouterTokens;  // 32 tokens per CTA
constexpr int HK = 32;             // hidden channels per smem chunk

__device__ __forceinline__ float bf16_bits_to_float(uint32_t b) { return __uint_as_float(b << 16); }

// Thread layout: warp w owns tokens 4w..4w+3 of the chunk; lane l owns
// experts l + 32*i for i < EPT.  Each thread keeps 4 x EPT logits.
template <int EPT>
__global__ void __launch_bounds__(256) router_topk_kernel(const uint16_t* __restrict__ x,
                                                          const float* __restrict__ Wr,
                                                          const float* __restrict__ bias, int T,
                                                          int H, int E, int k,
                                                          int32_t* __restrict__ topk_ids,
                                                          float* __restrict__ topk_w,
                                                          int32_t* __restrict__ rank,
                                                          int32_t* __restrict__ hist) {
    constexpr int EP = 32 * EPT;  // padded expert count
    __shared__ __align__(16) float xsT[HK][RT];  // [h][token]
    __shared__ __align__(16) float ws[HK][EP];
    __shared__ uint32_t mask[EP];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int t0 = blockIdx.x * RT;

    float acc[4][EPT];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int i = 0; i < EPT; ++i) acc[r][i] = 0.f;
    for (int i = tid; i < EP; i += 256) mask[i] = 0u;

    for (int h0 = 0; h0 < H; h0 += HK) {
        {  // x chunk: 32 tokens x 32 channels; thread -> token tid/8, channels 4*(tid%8)..+3
            const int r = tid >> 3, c = (tid & 7) * 4, t = t0 + r;
            uint2 v = make_uint2(0u, 0u);
            if (t < T) v = *reinterpret_cast<const uint2*>(x + (size_t)t * H + h0 + c);
            xsT[c + 0][r] = bf16_bits_to_float(v.x & 0xffffu);
            xsT[c + 1][r] = bf16_bits_to_float(v.x >> 16);
            xsT[c + 2][r] = bf16_bits_to_float(v.y & 0xffffu);
            xsT[c + 3][r] = bf16_bits_to_float(v.y >> 16);
        }
        for (int i = tid; i < HK * EP; i += 256) {
            const int r = i / EP, e = i % EP;
            ws[r][e] = (e < E) ? Wr[(size_t)(h0 + r) * E + e] : 0.f;
        }
        __syncthreads();
#pragma unroll 8
        for (int hh = 0; hh < HK; ++hh) {
            const float4 xv = *reinterpret_cast<const float4*>(&xsT[hh][warp * 4]);
            const float xr[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
            for (int i = 0; i < EPT; ++i) {
                const float w = ws[hh][lane + 32 * i];
#pragma unroll
                for (int r = 0; r < 4; ++r) acc[r][i] = __fmaf_rn(xr[r], w, acc[r][i]);
            }
        }
        __syncthreads();
    }

    // top-k per token with warp-wide arg-max; ties go to the lower index
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int t = t0 + warp * 4 + r;
        float v[EPT];
#pragma unroll
        for (int i = 0; i < EPT; ++i) {
            const int e = lane + 32 * i;
            v[i] = (e < E) ? (bias ? __fadd_rn(acc[r][i], bias[e]) : acc[r][i]) : -INFINITY;
        }
        bool taken[EPT];
#pragma unroll
        for (int i = 0; i < EPT; ++i) taken[i] = (lane + 32 * i) >= E;
        float sel_v[kMaxTopK];
        int sel_e[kMaxTopK];
        for (int j = 0; j < k; ++j) {
            float bv = -INFINITY;
            int be = 0x7fffffff;
#pragma unroll
            for (int i = 0; i < EPT; ++i) {
                const int e = lane + 32 * i;
                if (!taken[i] && (v[i] > bv || (v[i] == bv && e < be))) {
                    bv = v[i];
                    be = e;
                }
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
                const int oe = __shfl_xor_sync(0xffffffffu, be, off);
                if (ov > bv || (ov == bv && oe < be)) {
                    bv = ov;
                    be = oe;
                }
            }
#pragma unroll
            for (int i = 0; i < EPT; ++i)
                if (lane + 32 * i == be) taken[i] = true;
            sel_v[j] = bv;
            sel_e[j] = be;
        }
        if (t < T && lane == 0) {
            float den = 0.f;
            float ex[kMaxTopK];
            for (int j = 0; j < k; ++j) {
                ex[j] = expf(__fsub_rn(sel_v[j], sel_v[0]));
                den = __fadd_rn(den, ex[j]);
            }
            for (int j = 0; j < k; ++j) {
                topk_ids[(size_t)t * k + j] = sel_e[j];
                topk_w[(size_t)t * k + j] = __fdiv_rn(ex[j], den);
                atomicOr(&mask[sel_e[j]], 1u << (warp * 4 + r));
            }
        }
    }
    __syncthreads();
    // chunk-local rank of each choice and the chunk's count per expert
    for (int i = tid; i < RT * k; i += 256) {
        const int r = i / k, t = t0 + r;
        if (t < T) {
            const int e = topk_ids[(size_t)t * k + (i % k)];
            rank[(size_t)t * k + (i % k)] = __popc(mask[e] & ((1u << r) - 1u));
        }
    }
    for (int e = tid; e < E; e += 256) hist[(size_t)blockIdx.x * E + e] = __popc(mask[e]);
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

// One warp per token.  With topk_ids == nullptr the token's single "slot" is
// the token itself (the dense linear layer).  Besides the codes, every token
// gets the L1 norm of its code row; rows above kExactL1 are flagged in each
// of their slots and listed for the exact path of the GEMM.
__global__ void __launch_bounds__(256) permute_quant_kernel(
    const uint16_t* __restrict__ x, const int32_t* __restrict__ topk_ids,
    const int32_t* __restrict__ rank, const int32_t* __restrict__ base, int T, int H, int E, int k,
    int32_t* __restrict__ slot_of, int32_t* __restrict__ slot_token, float* __restrict__ s_x,
    float* __restrict__ s_slot, uint16_t* __restrict__ q16, int32_t* __restrict__ flags,
    int32_t* __restrict__ fb_list, int32_t* __restrict__ fb_count) {
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (t >= T) return;
    int my_slot = t;
    if (topk_ids != nullptr && lane < k) {
        const int e = topk_ids[(size_t)t * k + lane];
        my_slot = base[(size_t)(t / kRouterTokens) * E + e] + rank[(size_t)t * k + lane];
        slot_of[(size_t)t * k + lane] = my_slot;
        slot_token[my_slot] = t;
    }
    const int nk = (topk_ids != nullptr) ? k : 1;
    const uint4* row = reinterpret_cast<const uint4*>(x + (size_t)t * H);
    const int nv = H / 8;  // 8 bf16 per 16-byte vector
    float amax = 0.f;
    for (int i = lane; i < nv; i += 32) {
        const uint4 v = __ldg(row + i);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            amax = fmaxf(amax, fabsf(bf16_bits_to_float(w[j] & 0xffffu)));
            amax = fmaxf(amax, fabsf(bf16_bits_to_float(w[j] >> 16)));
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    const float s = __fdiv_rn(amax, 127.0f);
    if (lane == 0) s_x[t] = s;
    int slots[kMaxTopK];
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) slots[j] = __shfl_sync(0xffffffffu, my_slot, j);
    if (lane < nk) s_slot[my_slot] = s;
    int l1 = 0;
    for (int i = lane; i < nv; i += 32) {
        const uint4 v = __ldg(row + i);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t out[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            int q0 = 0, q1 = 0;
            if (s != 0.f) {
                q0 = __float2int_rn(__fdiv_rn(bf16_bits_to_float(w[j] & 0xffffu), s));
                q1 = __float2int_rn(__fdiv_rn(bf16_bits_to_float(w[j] >> 16), s));
                q0 = min(127, max(-128, q0));
                q1 = min(127, max(-128, q1));
            }
            l1 += abs(q0) + abs(q1);
            out[j] = (uint32_t)__half_as_ushort(__int2half_rn(q0)) |
                     ((uint32_t)__half_as_ushort(__int2half_rn(q1)) << 16);
        }
        const uint4 ov = make_uint4(out[0], out[1], out[2], out[3]);
        for (int j = 0; j < nk; ++j) reinterpret_cast<uint4*>(q16 + (size_t)slots[j] * H)[i] = ov;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) l1 += __shfl_xor_sync(0xffffffffu, l1, off);
    const int flagged = l1 > kExactL1 ? 1 : 0;
    if (lane < nk) {
        flags[my_slot] = flagged;
        if (flagged) fb_list[atomicAdd(fb_count, 1)] = my_slot;
    }
}

}  // namespace

cudaError_t launch_router_topk(const uint16_t* x, const float* Wr, const float* bias, int T, int H,
                               int E, int k, int32_t* topk_ids, float* topk_w, int32_t* rank,
                               int32_t* hist, cudaStream_t st) {
    const int grid = (T + RT - 1) / RT;
    if (E <= 32)
        router_topk_kernel<1><<<grid, 256, 0, st>>>(x, Wr, bias, T, H, E, k, topk_ids, topk_w, rank, hist);
    else if (E <= 64)
        router_topk_kernel<2><<<grid, 256, 0, st>>>(x, Wr, bias, T, H, E, k, topk_ids, topk_w, rank, hist);
    else if (E <= 128)
        router_topk_kernel<4><<<grid, 256, 0, st>>>(x, Wr, bias, T, H, E, k, topk_ids, topk_w, rank, hist);
    else
        router_topk_kernel<8><<<grid, 256, 0, st>>>(x, Wr, bias, T, H, E, k, topk_ids, topk_w, rank, hist);
    return cudaGetLastError();
}

cudaError_t launch_scan(int32_t* hist, int nchunk, int E, int32_t* offsets, int32_t* counts,
                        cudaStream_t st) {
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
    scan_kernel<<<1, kScanThreads, smem, st>>>(hist, nchunk, E, offsets, counts, use_smem);
    return cudaGetLastError();
}

cudaError_t launch_permute_quant(const uint16_t* x, const int32_t* topk_ids, const int32_t* rank,
                                 const int32_t* hist, int T, int H, int E, int k, int32_t* slot_of,
                                 int32_t* slot_token, float* s_x, float* s_slot, uint16_t* q16,
                                 int32_t* flags, int32_t* fb_list, int32_t* fb_count, cudaStream_t st) {
    const int grid = (T + 7) / 8;
    permute_quant_kernel<<<grid, 256, 0, st>>>(x, topk_ids, rank, hist, T, H, E, k, slot_of, slot_token,
                                               s_x, s_slot, q16, flags, fb_list, fb_count);
    return cudaGetLastError();
}

}  // namespace moe

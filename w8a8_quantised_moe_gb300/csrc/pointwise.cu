// pointwise.cu -- row-wise kernels around the expert GEMMs.
//
//   requant_kernel          per slot row of h: s_h = amax/127,
//                           q_h = clamp(round(h/s_h)), written as exact fp16
//                           values (the tensor-core operand) and/or int8.
//   s8_rows_gather_kernel   copies int8 rows out by a row map (debug dumps).
//   combine_kernel          y[t] = bf16_rne(sum_j w[t][j] * o[slot(t, j)]).
//   quantize_weights_kernel per output channel: s = amax/127, q = round(w/s)
//                           (optionally of w times per-column smoothing factors).
//   f16_rows_to_s8_kernel   copies quantised rows out as int8 (debug dumps).
//
// Quantisation: "W8A8 quantisation of MiniMax-M3 on K100AI" (mhpn.cn),
// section 2.1; re-quantising the FP32 result for the next operator:
// "DeepSeek V4 950 FP8 inference on H100" (lpnh.cn), section 2.3; weighted
// combine at the end of the layer: "Tencent Hunyuan AI Infra on Hopper"
// (pnsm.cn), section 1.3.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"

namespace moe {
namespace {

__device__ __forceinline__ int quant_code(float v, float s) { return quant_code_div(v, s); }

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
    return v;
}

// One warp per row of h [S][I].  Like the activation quantiser it certifies
// every code row: rows whose L1 norm exceeds kExactL1 are flagged and listed
// for the exact path of the second GEMM.
// ROW_SMEM: rows of up to kRqSmemVec float4 pass through shared memory (each
// warp copies its row with cp.async, then reads it twice), so h is read from
// memory once; else the warp reads its row twice.  CTAs of kRqWarps warps.
// Measured at S = 16384, I = 1536: 33 us, against 37 us reading twice.
constexpr int kRqWarps = 4;
constexpr int kRqSmemVec = 512;  // I <= 2048

template <bool ROW_SMEM>
__global__ void __launch_bounds__(32 * kRqWarps) requant_kernel(const float* __restrict__ h, int S, int I,
                                                      float* __restrict__ s_h,
                                                      uint16_t* __restrict__ q16,
                                                      int8_t* __restrict__ q8,
                                                      int32_t* __restrict__ flags,
                                                      int32_t* __restrict__ fb_list,
                                                      int32_t* __restrict__ fb_count) {
    __shared__ float4 row_s[ROW_SMEM ? kRqWarps : 1][ROW_SMEM ? kRqSmemVec : 1];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int r = blockIdx.x * kRqWarps + warp;
    pdl_wait();
    pdl_trigger();
    if (r >= S) return;
    const float4* row = reinterpret_cast<const float4*>(h + (size_t)r * I);
    const int nv = I / 4;
    float4* rs = row_s[ROW_SMEM ? warp : 0];
    if constexpr (ROW_SMEM) {
        for (int i = lane; i < nv; i += 32) cp_async16(rs + i, row + i);  // the whole row in flight
        cp_async_wait_all();
        __syncwarp();
    }
    const float4* src = ROW_SMEM ? rs : row;
    float amax = 0.f;
    for (int i = lane; i < nv; i += 32) {
        const float4 v = src[i];
        amax = fmaxf(fmaxf(fmaxf(amax, fabsf(v.x)), fmaxf(fabsf(v.y), fabsf(v.z))), fabsf(v.w));
    }
    amax = warp_max(amax);
    const float s = __fdiv_rn(amax, 127.0f);
    if (lane == 0) s_h[r] = s;
    int l1 = 0;
    for (int i = lane; i < nv; i += 32) {
        const float4 v = src[i];
        const int a = quant_code(v.x, s), b = quant_code(v.y, s), c = quant_code(v.z, s), d = quant_code(v.w, s);
        l1 += abs(a) + abs(b) + abs(c) + abs(d);
        if (q16 != nullptr) {
            uint2 o;
            o.x = (uint32_t)__half_as_ushort(__int2half_rn(a)) |
                  ((uint32_t)__half_as_ushort(__int2half_rn(b)) << 16);
            o.y = (uint32_t)__half_as_ushort(__int2half_rn(c)) |
                  ((uint32_t)__half_as_ushort(__int2half_rn(d)) << 16);
            reinterpret_cast<uint2*>(q16 + (size_t)r * I)[i] = o;
        }
        if (q8 != nullptr) {
            const uint32_t packed = (uint32_t)(uint8_t)a | ((uint32_t)(uint8_t)b << 8) |
                                    ((uint32_t)(uint8_t)c << 16) | ((uint32_t)(uint8_t)d << 24);
            reinterpret_cast<uint32_t*>(q8 + (size_t)r * I)[i] = packed;
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) l1 += __shfl_xor_sync(0xffffffffu, l1, off);
    if (lane == 0) {
        const int flagged = l1 > kExactL1 ? 1 : 0;
        flags[r] = flagged;
        if (flagged) fb_list[atomicAdd(fb_count, 1)] = r;
    }
}

// One CTA of 256 threads per row of h, the row held in registers (I <= 256 *
// 4 * kRqVec): for few rows (decode), where a warp per row leaves most of the
// GPU idle.  The same outputs as requant_kernel.
constexpr int kRqVec = 8;

__global__ void __launch_bounds__(256) requant_cta_kernel(const float* __restrict__ h, int S, int I,
                                                          float* __restrict__ s_h, uint16_t* __restrict__ q16,
                                                          int8_t* __restrict__ q8, int32_t* __restrict__ flags,
                                                          int32_t* __restrict__ fb_list,
                                                          int32_t* __restrict__ fb_count) {
    __shared__ float red_max[8];
    __shared__ int red_l1[8];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int r = blockIdx.x;
    // the next kernel (the down GEMM) may launch before this one waits: its
    // CTAs then take the SMs that the gate/up GEMM's last CTAs leave, and
    // prefetch their first weights while those finish
    pdl_trigger();
    pdl_wait();
    if (r >= S) return;
    const float4* row = reinterpret_cast<const float4*>(h + (size_t)r * I);
    const int nv = I / 4;
    float4 v[kRqVec];
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < kRqVec; ++i) {
        const int idx = tid + 256 * i;
        v[i] = idx < nv ? row[idx] : make_float4(0.f, 0.f, 0.f, 0.f);
        amax = fmaxf(fmaxf(fmaxf(amax, fabsf(v[i].x)), fmaxf(fabsf(v[i].y), fabsf(v[i].z))), fabsf(v[i].w));
    }
    amax = warp_max(amax);
    if (lane == 0) red_max[warp] = amax;
    __syncthreads();
    amax = red_max[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) amax = fmaxf(amax, red_max[i]);
    const float s = __fdiv_rn(amax, 127.0f);
    if (tid == 0) s_h[r] = s;
    int l1 = 0;
#pragma unroll
    for (int i = 0; i < kRqVec; ++i) {
        const int idx = tid + 256 * i;
        if (idx >= nv) break;
        const int a = quant_code(v[i].x, s), b = quant_code(v[i].y, s), c = quant_code(v[i].z, s),
                  d = quant_code(v[i].w, s);
        l1 += abs(a) + abs(b) + abs(c) + abs(d);
        if (q16 != nullptr) {
            uint2 o;
            o.x = (uint32_t)__half_as_ushort(__int2half_rn(a)) |
                  ((uint32_t)__half_as_ushort(__int2half_rn(b)) << 16);
            o.y = (uint32_t)__half_as_ushort(__int2half_rn(c)) |
                  ((uint32_t)__half_as_ushort(__int2half_rn(d)) << 16);
            reinterpret_cast<uint2*>(q16 + (size_t)r * I)[idx] = o;
        }
        if (q8 != nullptr) {
            const uint32_t packed = (uint32_t)(uint8_t)a | ((uint32_t)(uint8_t)b << 8) |
                                    ((uint32_t)(uint8_t)c << 16) | ((uint32_t)(uint8_t)d << 24);
            reinterpret_cast<uint32_t*>(q8 + (size_t)r * I)[idx] = packed;
        }
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
        flags[r] = flagged;
        if (flagged) fb_list[atomicAdd(fb_count, 1)] = r;
    }
}

// Grid (tokens, column splits): a CTA of 256 threads covers every
// gridDim.y-th block of 256 float4 column groups of one token; each thread
// reads its k slot rows with independent loads.  Few tokens (decode) split
// each row over several CTAs to fill the GPU; many tokens use one CTA per
// token (measured: splitting then costs more than it gains).
template <int KMAX>  // k <= KMAX (register budget of the loads in flight)
__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ o,
                                                      const int32_t* __restrict__ slot_of,
                                                      const float* __restrict__ topk_w, int T,
                                                      int H, int k, uint16_t* __restrict__ y,
                                                      int* __restrict__ error) {
    const int t = blockIdx.x;
    pdl_wait();
    pdl_trigger();
    if (t >= T) return;
    __shared__ int32_t slot[kMaxTopK];
    __shared__ float w[kMaxTopK];
    if (threadIdx.x < k) {
        const int sl = slot_of[(size_t)t * k + threadIdx.x];
        // checked build: a slot out of range contributes nothing (-1)
        slot[threadIdx.x] = in_range(sl, 0, (long long)T * k, blockIdx.y == 0 ? error : nullptr) ? sl : -1;
        w[threadIdx.x] = topk_w[(size_t)t * k + threadIdx.x];
    }
    __syncthreads();
    const int nv = H / 4;
    for (int i = blockIdx.y * 256 + threadIdx.x; i < nv; i += gridDim.y * 256) {
        float4 v[KMAX];
#pragma unroll
        for (int j = 0; j < KMAX; ++j)  // independent loads first
            if (j < k)
                v[j] = (!kChecked || slot[j] >= 0) ? reinterpret_cast<const float4*>(o + (size_t)slot[j] * H)[i]
                                                   : make_float4(0.f, 0.f, 0.f, 0.f);
        float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
        for (int j = 0; j < KMAX; ++j) {  // then the sum in top-k order
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
        reinterpret_cast<uint2*>(y + (size_t)t * H)[i] = out;
    }
}

// One warp per weight row; grid-stride over rows.  With column factors cs
// (smoothing folded into the weights) the row quantised is w[r][k] * cs[k],
// one binary32 multiply per element.
template <bool CS>
__global__ void __launch_bounds__(256) quantize_weights_kernel(const float* __restrict__ w,
                                                               const float* __restrict__ cs, int64_t rows,
                                                               int K, int8_t* __restrict__ q,
                                                               float* __restrict__ s_out) {
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = (int64_t)gridDim.x * 8;
    auto ld4 = [&](const float* row, int i) {
        float4 v = reinterpret_cast<const float4*>(row)[i];
        if (CS) {
            const float4 c = reinterpret_cast<const float4*>(cs)[i];
            v = make_float4(__fmul_rn(v.x, c.x), __fmul_rn(v.y, c.y), __fmul_rn(v.z, c.z), __fmul_rn(v.w, c.w));
        }
        return v;
    };
    auto ld1 = [&](const float* row, int i) { return CS ? __fmul_rn(row[i], cs[i]) : row[i]; };
    for (int64_t r = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5); r < rows; r += nwarps) {
        const float* row = w + r * K;
        float amax = 0.f;
        if ((K & 3) == 0) {
            for (int i = lane; i < K / 4; i += 32) {
                const float4 v = ld4(row, i);
                amax = fmaxf(fmaxf(fmaxf(amax, fabsf(v.x)), fmaxf(fabsf(v.y), fabsf(v.z))), fabsf(v.w));
            }
        } else {
            for (int i = lane; i < K; i += 32) amax = fmaxf(amax, fabsf(ld1(row, i)));
        }
        amax = warp_max(amax);
        const float s = __fdiv_rn(amax, 127.0f);
        if (lane == 0) s_out[r] = s;
        int8_t* qr = q + r * K;
        if ((K & 3) == 0) {
            for (int i = lane; i < K / 4; i += 32) {
                const float4 v = ld4(row, i);
                const uint32_t packed = (uint32_t)(uint8_t)quant_code(v.x, s) |
                                        ((uint32_t)(uint8_t)quant_code(v.y, s) << 8) |
                                        ((uint32_t)(uint8_t)quant_code(v.z, s) << 16) |
                                        ((uint32_t)(uint8_t)quant_code(v.w, s) << 24);
                reinterpret_cast<uint32_t*>(qr)[i] = packed;
            }
        } else {
            for (int i = lane; i < K; i += 32) qr[i] = (int8_t)quant_code(ld1(row, i), s);
        }
    }
}

// q8[r][:] = int8(q16[row_of[r * stride]][:]) (row_of == nullptr: identity).
__global__ void f16_rows_to_s8_kernel(const uint16_t* __restrict__ q16, const int32_t* __restrict__ row_of,
                                      int rows, int K, int stride, int src_rows, int8_t* __restrict__ q8,
                                      int* __restrict__ error) {
    const int r = blockIdx.x;
    if (r >= rows) return;
    const int src = row_of ? row_of[(size_t)r * stride] : r;
    if (!in_range(src, 0, src_rows, threadIdx.x == 0 ? error : nullptr)) return;  // checked build
    for (int i = threadIdx.x; i < K; i += blockDim.x)
        q8[(size_t)r * K + i] = (int8_t)__half2int_rn(__ushort_as_half(q16[(size_t)src * K + i]));
}

__global__ void s8_rows_gather_kernel(const int8_t* __restrict__ q8, const int32_t* __restrict__ row_of, int rows,
                                      int K, int stride, int src_rows, int8_t* __restrict__ out,
                                      int* __restrict__ error) {
    const int r = blockIdx.x;
    if (r >= rows) return;
    const int src = row_of ? row_of[(size_t)r * stride] : r;
    if (!in_range(src, 0, src_rows, threadIdx.x == 0 ? error : nullptr)) return;  // checked build
    const uint4* s = reinterpret_cast<const uint4*>(q8 + (size_t)src * K);
    uint4* d = reinterpret_cast<uint4*>(out + (size_t)r * K);
    for (int i = threadIdx.x; i < K / 16; i += blockDim.x) d[i] = s[i];
}

}  // namespace

cudaError_t launch_s8_rows_gather(const int8_t* q8, const int32_t* row_of, int rows, int K, int row_stride_of,
                                  int src_rows, int8_t* out, int* error, cudaStream_t st) {
    if (rows == 0) return cudaSuccess;
    s8_rows_gather_kernel<<<rows, 256, 0, st>>>(q8, row_of, rows, K, row_stride_of, src_rows, out, error);
    return cudaGetLastError();
}

cudaError_t launch_requant(const float* h, int S, int I, float* s_h, uint16_t* q16, int8_t* q8,
                           int32_t* flags, int32_t* fb_list, int32_t* fb_count, cudaStream_t st, bool pdl) {
    if (S == 0) return cudaSuccess;
    // few rows: one CTA per row (measured at S = 16384: a warp per row takes
    // 37 us, a CTA per row 57 us; at S = 128 a CTA per row is faster)
#ifndef MOE_RQ_CTA_ROWS_PER_SM
#define MOE_RQ_CTA_ROWS_PER_SM 8
#endif
    if ((long)S <= (long)MOE_RQ_CTA_ROWS_PER_SM * num_sms() && I <= 256 * 4 * kRqVec)
        return launch_kernel(requant_cta_kernel, dim3(S), dim3(256), 0, st, pdl, h, S, I, s_h, q16, q8, flags,
                             fb_list, fb_count);
    const dim3 grid((S + kRqWarps - 1) / kRqWarps), block(32 * kRqWarps);
    if (I <= 4 * kRqSmemVec)
        return launch_kernel(requant_kernel<true>, grid, block, 0, st, pdl, h, S, I, s_h, q16, q8, flags, fb_list,
                             fb_count);
    return launch_kernel(requant_kernel<false>, grid, block, 0, st, pdl, h, S, I, s_h, q16, q8, flags, fb_list,
                         fb_count);
}

cudaError_t launch_combine(const float* o, const int32_t* slot_of, const float* topk_w, int T,
                           int H, int k, uint16_t* y, int* error, cudaStream_t st, bool pdl) {
    if (T == 0) return cudaSuccess;
    const int blocks = (H / 4 + 255) / 256;
    int split = (4 * num_sms() + T - 1) / T;
    if (split > blocks) split = blocks;
    if (split < 1) split = 1;
    const dim3 grid(T, split), block(256);
    if (k <= 2) return launch_kernel(combine_kernel<2>, grid, block, 0, st, pdl, o, slot_of, topk_w, T, H, k, y, error);
    if (k <= 4) return launch_kernel(combine_kernel<4>, grid, block, 0, st, pdl, o, slot_of, topk_w, T, H, k, y, error);
    return launch_kernel(combine_kernel<kMaxTopK>, grid, block, 0, st, pdl, o, slot_of, topk_w, T, H, k, y, error);
}

cudaError_t launch_quantize_weights(const float* w, int64_t rows, int K, int8_t* q, float* s,
                                    cudaStream_t st, const float* col_scale) {
    if (rows == 0) return cudaSuccess;
    int64_t blocks = (rows + 7) / 8;
    const int64_t cap = (int64_t)num_sms() * 16;
    if (blocks > cap) blocks = cap;
    if (col_scale)
        quantize_weights_kernel<true><<<(unsigned)blocks, 256, 0, st>>>(w, col_scale, rows, K, q, s);
    else
        quantize_weights_kernel<false><<<(unsigned)blocks, 256, 0, st>>>(w, nullptr, rows, K, q, s);
    return cudaGetLastError();
}

cudaError_t launch_f16_rows_to_s8(const uint16_t* q16, const int32_t* row_of, int rows, int K,
                                  int row_stride_of, int src_rows, int8_t* q8, int* error, cudaStream_t st) {
    if (rows == 0) return cudaSuccess;
    f16_rows_to_s8_kernel<<<rows, 256, 0, st>>>(q16, row_of, rows, K, row_stride_of, src_rows, q8, error);
    return cudaGetLastError();
}

}  // namespace moe

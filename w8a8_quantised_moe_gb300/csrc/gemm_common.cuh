// gemm_common.cuh -- device helpers shared by the grouped GEMM kernels
// (one CTA per tile in gemm.cu, CTA pairs in gemm_pair.cu): warp roles, the
// tile table, bounded warp-wide waits, the int8 -> fp16 conversion, the
// epilogue arithmetic and the exact CUDA-core path for rows whose L1 norm is
// above the exactness bound.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kThreads = 320;
constexpr int kTileM = 128;   // weight rows per tile
constexpr int kEpiWarp0 = 6;  // first epilogue warp


// Tile table of a launch: group g owns tiles [tile_start[g], tile_start[g+1]);
// inside a group, tile = cb * ntb + tb (token blocks fastest, so CTAs running
// at the same time share the weight tile).
struct Tiles {
    const int* tile_start;  // smem, [n_groups + 1]
    const int* row_start;   // smem, [n_groups + 1]
    int n_groups;
};

__device__ __forceinline__ int last_le(const int* a, int n, int v) {  // last i < n with a[i] <= v
    int lo = 0, hi = n - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (a[mid] <= v) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// Warp-uniform bounded wait: every lane polls, lane 0 owns the time limit.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const WaitCtl& ctl) {
    const int lane = threadIdx.x & 31;
    uint64_t t0 = 0;
    for (uint32_t i = 0;; ++i) {
        const bool ok = mbar_try_wait(bar, parity);
        if (__all_sync(0xffffffffu, ok)) return true;
        if ((i & 31u) == 31u) {
            int give_up = 0;
            if (lane == 0) {
                const uint64_t now = global_timer_ns();
                if (t0 == 0) t0 = now;
                if (*ctl.abort) {
                    give_up = 1;
                } else if (now - t0 > ctl.timeout_ns) {
                    give_up_timeout(ctl);
                    give_up = 1;
                }
            }
            if (__shfl_sync(0xffffffffu, give_up, 0)) return false;
        }
    }
}

// warp_wait on a barrier that the other CTA of a pair, or the pair's
// tensor-core commits, arrive on.
__device__ __forceinline__ bool warp_wait_cluster(uint64_t* bar, uint32_t parity, const WaitCtl& ctl) {
    const int lane = threadIdx.x & 31;
    uint64_t t0 = 0;
    for (uint32_t i = 0;; ++i) {
        const bool ok = mbar_try_wait_cluster(bar, parity);
        if (__all_sync(0xffffffffu, ok)) return true;
        if ((i & 31u) == 31u) {
            int give_up = 0;
            if (lane == 0) {
                const uint64_t now = global_timer_ns();
                if (t0 == 0) t0 = now;
                if (*ctl.abort) {
                    give_up = 1;
                } else if (now - t0 > ctl.timeout_ns) {
                    give_up_timeout(ctl);
                    give_up = 1;
                }
            }
            if (__shfl_sync(0xffffffffu, give_up, 0)) return false;
        }
    }
}

// Barrier of the four epilogue warps on an mbarrier of count 4 (bounded).
__device__ __forceinline__ bool epi_sync(uint64_t* bar, uint32_t& it, const WaitCtl& ctl) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
    const bool ok = warp_wait(bar, it & 1u, ctl);
    ++it;
    return ok;
}

// int8 x4 (one 32-bit word, element 0 in the low byte) -> two fp16x2 words
// (element 0 in the low half).  (q + 128) is placed in the mantissa of
// 1024.0h, giving 1024 + q + 128 exactly; subtracting 1152 leaves q.
__device__ __forceinline__ void s8x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
    const uint32_t u = w ^ 0x80808080u;
    uint32_t a = __byte_perm(u, 0x64646464u, 0x4140);
    uint32_t b = __byte_perm(u, 0x64646464u, 0x4342);
    const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
    __half2 ha = __hsub2(*reinterpret_cast<__half2*>(&a), bias);
    __half2 hb = __hsub2(*reinterpret_cast<__half2*>(&b), bias);
    lo = *reinterpret_cast<uint32_t*>(&ha);
    hi = *reinterpret_cast<uint32_t*>(&hb);
}

__device__ __forceinline__ void cvt_chunk(const uint4 w, uint32_t* v) {
    s8x4_to_f16x4(w.x, v[0], v[1]);
    s8x4_to_f16x4(w.y, v[2], v[3]);
    s8x4_to_f16x4(w.z, v[4], v[5]);
    s8x4_to_f16x4(w.w, v[6], v[7]);
}

__device__ __forceinline__ float silu_f32(float g) {
    return __fdiv_rn(g, __fadd_rn(1.0f, expf(-g)));
}

__device__ __forceinline__ float dequant(float acc, float s_act, float s_w) {
    return __fmul_rn(__fmul_rn(acc, s_act), s_w);
}

// Checked build: whether group g's rows [r0, r1) lie within [0, total)
// (records kErrDevice when not).  A kernel whose offsets fail it empties its
// whole tile (or unit) table, so that no tile reads or writes outside the
// rows, and reports the error.
__device__ __forceinline__ bool group_rows_ok(int r0, int r1, int total, int* error) {
    return in_range(r0, 0, (long long)r1 + 1, error) && in_range(r1, 0, (long long)total + 1, error);
}

// Exact CUDA-core path for the rows the certificate rejected: one warp per
// (row, output channel), int32 dot products over K, spread over every warp of
// the grid.
template <int EPI>
__device__ void fallback_rows(const GemmArgs& args, const int* row_start, int n_groups) {
    int n_fb = *args.fb_count;
    if (n_fb <= 0) return;
    if (!in_range(n_fb, 0, (long long)args.total_rows + 1, args.error)) n_fb = args.total_rows;
    const int lane = threadIdx.x & 31;
    const int per_row = (EPI == (int)Epi::GateUp) ? args.up_offset : args.w_rows_per_group;
    const long n_items = (long)n_fb * per_row;
    const int warps = (int)(blockDim.x >> 5);
    const int8_t* w = static_cast<const int8_t*>(args.w);
    const __half* act = static_cast<const __half*>(args.act16);
    for (long item = (long)blockIdx.x * warps + (threadIdx.x >> 5); item < n_items;
         item += (long)gridDim.x * warps) {
        const int row = args.fb_list[item / per_row];
        if (!in_range(row, 0, args.total_rows, args.error)) continue;  // checked build
        const int n = (int)(item % per_row);
        const int g = last_le(row_start, n_groups, row);
        const __half* a = act + (size_t)row * args.K;
        const int8_t* w0 = w + ((size_t)g * args.w_rows_per_group + n) * args.K;
        const int8_t* w1 = w0 + (size_t)args.up_offset * args.K;  // up row (GateUp only)
        int acc0 = 0, acc1 = 0;
        for (int k = lane * 8; k < args.K; k += 32 * 8) {
            const uint4 av = *reinterpret_cast<const uint4*>(a + k);
            const __half* ah = reinterpret_cast<const __half*>(&av);
            const uint2 wv0 = *reinterpret_cast<const uint2*>(w0 + k);
            const int8_t* wb0 = reinterpret_cast<const int8_t*>(&wv0);
            int q[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) q[i] = __half2int_rn(ah[i]);
#pragma unroll
            for (int i = 0; i < 8; ++i) acc0 += q[i] * (int)wb0[i];
            if (EPI == (int)Epi::GateUp) {
                const uint2 wv1 = *reinterpret_cast<const uint2*>(w1 + k);
                const int8_t* wb1 = reinterpret_cast<const int8_t*>(&wv1);
#pragma unroll
                for (int i = 0; i < 8; ++i) acc1 += q[i] * (int)wb1[i];
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            acc0 += __shfl_xor_sync(0xffffffffu, acc0, off);
            acc1 += __shfl_xor_sync(0xffffffffu, acc1, off);
        }
        if (lane != 0) continue;
        const float sa = args.act_scale[row];
        const float* sw = args.w_scale + (size_t)g * args.w_rows_per_group;
        if (EPI == (int)Epi::GateUp) {
            const float gv = dequant(__int2float_rn(acc0), sa, sw[n]);
            const float uv = dequant(__int2float_rn(acc1), sa, sw[args.up_offset + n]);
            static_cast<float*>(args.out)[(size_t)row * args.ld_out + n] = __fmul_rn(silu_f32(gv), uv);
            if (args.acc_out) {
                args.acc_out[(size_t)row * args.w_rows_per_group + n] = acc0;
                args.acc_out[(size_t)row * args.w_rows_per_group + args.up_offset + n] = acc1;
            }
        } else {
            const float v = dequant(__int2float_rn(acc0), sa, sw[n]);
            if (EPI == (int)Epi::ScaleF32)
                static_cast<float*>(args.out)[(size_t)row * args.ld_out + n] = v;
            else
                static_cast<__nv_bfloat16*>(args.out)[(size_t)row * args.ld_out + n] = __float2bfloat16_rn(v);
            if (args.acc_out) args.acc_out[(size_t)row * args.w_rows_per_group + n] = acc0;
        }
    }
}


}  // namespace
}  // namespace moe

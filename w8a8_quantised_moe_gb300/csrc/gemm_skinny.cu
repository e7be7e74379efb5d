// gemm_skinny.cu -- the grouped W8A8 GEMM for groups of a few activation
// rows (decode): exact int32 dot products on the CUDA cores (dp4a), with the
// same epilogues as the tensor-core kernels.
//
// With a handful of tokens per expert the expert GEMMs are weight streaming:
// each int8 weight byte is read once from HBM and meets only a few activation
// rows, so the tensor cores would idle while the converters of the
// tensor-core kernels sit on the critical path.  Here every warp streams four
// weight rows with coalesced 16-byte loads (512 contiguous bytes per row and
// step, several steps per row in flight), multiplies them against the
// group's activation rows staged once per work unit in shared memory, and
// reduces across the warp.  (Tried and measured slower: staging the weights
// through shared memory with TMA tensor boxes or 1-D bulk copies fed by one
// producer thread; that path delivered 10-16 bytes per clock per SM here.)
// int8 x int8 products summed in int32 are exact for any K the library accepts
// (K * 127 * 128 < 2^31), so no row needs the exact path of the tensor-core
// kernels.
//
// The grouped W8A8 GEMM with the scale outer product in its epilogue: "W8A8
// quantisation of MiniMax-M3 on K100AI" (mhpn.cn), section 2.1; decode as
// the bandwidth-bound regime of the expert GEMMs: "Tencent Hunyuan AI Infra
// on Hopper" (pnsm.cn), section 1.3.
#include <mutex>

#include "gemm_common.cuh"

namespace moe {
namespace {

constexpr int kSkThreads = 256;
constexpr int kSkWarps = kSkThreads / 32;
constexpr int kSkRows = 4;   // weight rows per warp item (GateUp: gate and up of two channels)
// Items per warp per work unit: measured on the decode layer, the gate/up
// GEMM (K = 4096) is fastest with one (117 against 121 us with two: finer
// units leave less of a tail), the down GEMM (K = 1536) with two (69.6 against
// 76.7 us: fewer units, less per-unit overhead).
constexpr int kSkItemsGateUp = 1;
constexpr int kSkItemsScale = 2;
constexpr int kSkChunk = 8;  // activation rows staged per pass
// weight rows (Scale) or channels (GateUp) of one work unit
constexpr int kSkUnitScale = kSkWarps * kSkItemsScale * kSkRows;        // weight rows per unit (64)
constexpr int kSkUnitGateUp = kSkWarps * kSkItemsGateUp * kSkRows / 2;  // gate/up channel pairs per unit (16)

__device__ __forceinline__ uint4 ld_stream16(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ int dot16(const uint4 w, const uint4 a, int acc) {
    acc = __dp4a((int)w.x, (int)a.x, acc);
    acc = __dp4a((int)w.y, (int)a.y, acc);
    acc = __dp4a((int)w.z, (int)a.z, acc);
    return __dp4a((int)w.w, (int)a.w, acc);
}

// One warp item: kSkRows weight rows x RC staged activation rows (rc valid),
// dot products over K, then the epilogue of the valid (row, channel) pairs.
// GateUp: rows are gate c, gate c+1, up c, up c+1 (c = first channel).
// Each batch issues NB 512-byte steps of every row before using any (NB * 2
// KB in flight per warp): measured on the down GEMM of the decode layer
// (K = 1536), 69.6 us against 76 us with two steps per batch.
template <int EPI, int RC, int NB = (RC <= 4 ? 4 : 2)>
__device__ __forceinline__ void skinny_item(const GemmArgs& args, const int8_t* __restrict__ act_s, int rc,
                                            int row0, int g, int first, int lane) {
    const int K = args.K;
    const int8_t* w = static_cast<const int8_t*>(args.w);
    const int8_t* wr[kSkRows];
    int wrow[kSkRows];  // weight row within the group
#pragma unroll
    for (int j = 0; j < kSkRows; ++j) {
        if (EPI == (int)Epi::GateUp) wrow[j] = (j >> 1) * args.up_offset + first + (j & 1);
        else wrow[j] = first + j;
        wr[j] = w + ((size_t)g * args.w_rows_per_group + wrow[j]) * K;
    }
    int acc[kSkRows][RC];
#pragma unroll
    for (int j = 0; j < kSkRows; ++j)
#pragma unroll
        for (int r = 0; r < RC; ++r) acc[j][r] = 0;

    for (int k0 = lane * 16; k0 < K; k0 += NB * 512) {
        uint4 wv[NB][kSkRows];
#pragma unroll
        for (int b = 0; b < NB; ++b) {  // every load of the batch first
            const int k = k0 + b * 512;
#pragma unroll
            for (int j = 0; j < kSkRows; ++j) wv[b][j] = k < K ? ld_stream16(wr[j] + k) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            const int k = k0 + b * 512;
            if (k < K) {
#pragma unroll
                for (int r = 0; r < RC; ++r) {
                    const uint4 a = *reinterpret_cast<const uint4*>(act_s + (size_t)r * K + k);
#pragma unroll
                    for (int j = 0; j < kSkRows; ++j) acc[j][r] = dot16(wv[b][j], a, acc[j][r]);
                }
            }
        }
    }

    const float* sw = args.w_scale + (size_t)g * args.w_rows_per_group;
    if (EPI == (int)Epi::GateUp) {
        // value (c, r, gate/up) at ((c * RC) + r) * 2 + gu: the reduction ends
        // with a channel's gate and up sums in the same lane
        constexpr int V = kSkRows * RC;
        int v[V];
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
            for (int r = 0; r < RC; ++r) {
                v[(c * RC + r) * 2 + 0] = acc[c][r];
                v[(c * RC + r) * 2 + 1] = acc[2 + c][r];
            }
        WarpButterfly<int, V, 16, 2>::run(v, lane);
        constexpr int kDup = 32 / (V / 2);
        const int p = lane / kDup;  // (c, r)
        const int c = p / RC, r = p % RC;
        if (lane % kDup == 0 && r < rc) {
            const int row = row0 + r;
            const int n = first + c;
            const float sa = args.act_scale[row];
            const float gv = dequant(__int2float_rn(v[0]), sa, sw[n]);
            const float uv = dequant(__int2float_rn(v[1]), sa, sw[args.up_offset + n]);
            static_cast<float*>(args.out)[(size_t)row * args.ld_out + n] = __fmul_rn(silu_f32(gv), uv);
            if (args.acc_out) {
                args.acc_out[(size_t)row * args.w_rows_per_group + n] = v[0];
                args.acc_out[(size_t)row * args.w_rows_per_group + args.up_offset + n] = v[1];
            }
        }
    } else {
        constexpr int V = kSkRows * RC;  // value (j, r) at j * RC + r
        int v[V];
#pragma unroll
        for (int j = 0; j < kSkRows; ++j)
#pragma unroll
            for (int r = 0; r < RC; ++r) v[j * RC + r] = acc[j][r];
        WarpButterfly<int, V, 16, 1>::run(v, lane);
        constexpr int kDup = 32 / V;
        const int p = lane / kDup;
        const int j = p / RC, r = p % RC;
        if (lane % kDup == 0 && r < rc) {
            const int row = row0 + r;
            const int n = first + j;
            const float val = dequant(__int2float_rn(v[0]), args.act_scale[row], sw[n]);
            if (EPI == (int)Epi::ScaleF32)
                static_cast<float*>(args.out)[(size_t)row * args.ld_out + n] = val;
            else
                static_cast<__nv_bfloat16*>(args.out)[(size_t)row * args.ld_out + n] = __float2bfloat16_rn(val);
            if (args.acc_out) args.acc_out[(size_t)row * args.w_rows_per_group + n] = v[0];
        }
    }
}

// Persistent grid over work units = (non-empty group, block of weight rows);
// per unit the group's activation rows pass through shared memory in chunks
// of kSkChunk rows (zero-padded to the kernel's chunk shape).
template <int EPI>
__global__ void __launch_bounds__(kSkThreads, 2) grouped_gemm_skinny_kernel(const GemmArgs args) {
    extern __shared__ __align__(16) int8_t act_s[];  // [kSkChunk][K]
    __shared__ int unit_start[kMaxExperts + 1];
    __shared__ int row_start[kMaxExperts + 1];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int G = args.n_groups;
    const int unit_rows = EPI == (int)Epi::GateUp ? kSkUnitGateUp : kSkUnitScale;
    const int per_group = (EPI == (int)Epi::GateUp ? args.up_offset : args.w_rows_per_group) / unit_rows;
    pdl_wait();  // the previous kernel's outputs (offsets, codes, scales) are visible from here
    pdl_trigger();

    if (warp == 0) {  // unit table: exclusive prefix of per_group over the non-empty groups
        int carry = 0;
        bool bad = false;  // checked build: an offset out of order or range
        for (int g0 = 0; g0 < G; g0 += 32) {
            const int g = g0 + lane;
            int r0 = 0, r1 = 0;
            if (g < G) {
                r0 = args.offsets ? args.offsets[g] : 0;
                r1 = args.offsets ? args.offsets[g + 1] : args.total_rows;
                if (!group_rows_ok(r0, r1, args.total_rows, args.error)) {
                    bad = true;
                    r0 = r1 = 0;
                }
                row_start[g] = r0;
            }
            const int v = (g < G && r1 > r0) ? per_group : 0;
            int incl = v;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int o = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += o;
            }
            if (g < G) unit_start[g] = carry + incl - v;
            carry += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) {
            unit_start[G] = carry;
            row_start[G] = args.offsets ? args.offsets[G] : args.total_rows;
        }
        if (kChecked && __any_sync(0xffffffffu, bad)) {  // an empty, consistent table: no unit runs
            for (int g = lane; g <= G; g += 32) {
                row_start[g] = 0;
                unit_start[g] = 0;
            }
        }
    }
    __syncthreads();
    const int total_units = unit_start[G];
    const int K = args.K;
    const int8_t* act = args.act8;

    // units dealt round-robin: the CTAs running at one time stream one window
    // of consecutive weight rows (measured faster than a contiguous range of
    // units per CTA)
    int staged_row0 = -1;  // first activation row in act_s (row ranges of groups are disjoint)
    for (int u = blockIdx.x; u < total_units; u += gridDim.x) {
        const int g = last_le(unit_start, G, u);
        const int unit = u - unit_start[g];
        const int r_begin = row_start[g], r_end = row_start[g + 1];
        for (int row0 = r_begin; row0 < r_end; row0 += kSkChunk) {
            const int rc = min(kSkChunk, r_end - row0);
            const int RC = rc <= 2 ? 2 : rc <= 4 ? 4 : 8;
            if (row0 != staged_row0) {
                // stage rows row0 .. row0 + rc, zeros up to RC
                __syncthreads();  // every warp is done with the previous rows
                const int n16 = RC * K / 16;
                const int valid16 = rc * K / 16;
                const uint4* src = reinterpret_cast<const uint4*>(act + (size_t)row0 * K);
                uint4* dst = reinterpret_cast<uint4*>(act_s);
                for (int i = threadIdx.x; i < n16; i += kSkThreads)
                    dst[i] = i < valid16 ? __ldg(src + i) : make_uint4(0, 0, 0, 0);
                __syncthreads();
                staged_row0 = row0;
            }
            constexpr int kItems = EPI == (int)Epi::GateUp ? kSkItemsGateUp : kSkItemsScale;
#pragma unroll 1
            for (int it = 0; it < kItems; ++it) {
                const int item = warp * kItems + it;
                const int first = EPI == (int)Epi::GateUp ? unit * kSkUnitGateUp + item * (kSkRows / 2)
                                                           : unit * kSkUnitScale + item * kSkRows;
                if (RC == 2) skinny_item<EPI, 2>(args, act_s, rc, row0, g, first, lane);
                else if (RC == 4) skinny_item<EPI, 4>(args, act_s, rc, row0, g, first, lane);
                else skinny_item<EPI, 8>(args, act_s, rc, row0, g, first, lane);
            }
        }
    }
}

template <int EPI>
cudaError_t launch_skinny_impl(const GemmArgs& args, cudaStream_t st, bool pdl) {
    auto kern = grouped_gemm_skinny_kernel<EPI>;
    const int smem = kSkChunk * args.K;
    static std::mutex mu;
    static int smem_set = 0;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (smem > smem_set) {
            const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
            if (e != cudaSuccess) return e;
            smem_set = smem;
        }
    }
    const int unit_rows = EPI == (int)Epi::GateUp ? kSkUnitGateUp : kSkUnitScale;
    const int per_group = (EPI == (int)Epi::GateUp ? args.up_offset : args.w_rows_per_group) / unit_rows;
    const long max_units = (long)per_group * args.n_groups;
    long grid = 2L * num_sms();
    if (max_units < grid) grid = max_units;
    if (grid < 1) grid = 1;
    return launch_kernel(kern, dim3((unsigned)grid), dim3(kSkThreads), (size_t)smem, st, pdl, args);
}

}  // namespace

bool skinny_shape_supported(Epi epi, long K, long w_rows_per_group, long up_offset) {
    if (K % 128 != 0 || K > 28672) return false;  // kSkChunk * K bytes of staging + the tables fit 227 KB
    if (epi == Epi::GateUp) return up_offset % kSkUnitGateUp == 0;
    return w_rows_per_group % kSkUnitScale == 0;
}

bool skinny_gemm_supported(Epi epi, const GemmArgs& args) {
    if (args.act8 == nullptr || args.n_groups > kMaxExperts) return false;
    return skinny_shape_supported(epi, args.K, args.w_rows_per_group, args.up_offset);
}

cudaError_t launch_grouped_gemm_skinny(Epi epi, const GemmArgs& args, cudaStream_t st, bool pdl) {
    if (!skinny_gemm_supported(epi, args)) return cudaErrorInvalidValue;
    switch (epi) {
        case Epi::GateUp: return launch_skinny_impl<0>(args, st, pdl);
        case Epi::ScaleF32: return launch_skinny_impl<1>(args, st, pdl);
        case Epi::ScaleBF16: return launch_skinny_impl<2>(args, st, pdl);
    }
    return cudaErrorInvalidValue;
}

}  // namespace moe

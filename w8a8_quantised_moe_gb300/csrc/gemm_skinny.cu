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
#include "gemm_skinny.cuh"

namespace moe {
namespace {

template <int EPI>
__global__ void __launch_bounds__(kSkThreads, 2) grouped_gemm_skinny_kernel(const GemmArgs args) {
    extern __shared__ __align__(16) int8_t act_s[];  // skinny_nbuf(K) x [kSkChunk][K]
    __shared__ int unit_start[kMaxExperts + 1];
    __shared__ int row_start[kMaxExperts + 1];
    __shared__ int next_s[3];
    skinny_run<EPI, kSkSrcRows, SkNoHook, true>(args, act_s, unit_start, row_start, next_s, blockIdx.x, gridDim.x);
}

template <int EPI>
cudaError_t launch_skinny_impl(const GemmArgs& args, cudaStream_t st, bool pdl) {
    auto kern = grouped_gemm_skinny_kernel<EPI>;
    const int smem = skinny_smem_bytes(args.K);
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

// peak_int8.cu -- contraction rates of this GPU for the exact int8 x int8 ->
// int32 product of the W8A8 layer, the denominators of its compute roofline.
//
// GB300 has no fast INT8 tensor path, so the library carries int8 values in
// fp16 through tcgen05.mma kind::f16 (every product and every partial sum of
// a 128-deep block is exact in the fp32 accumulator).  This program measures:
//   * tcgen05 kind::f16, one CTA, A and B in shared memory, M 128 x N 256;
//   * tcgen05 kind::f16, one CTA, A in tensor memory (as the library's GEMMs
//     hold the converted weights), M 128 x N 256;
//   * tcgen05 kind::f16 on CTA pairs, A in tensor memory, M 256 x N 192 and
//     N 256, issued eight MMAs per block as the pair GEMMs issue a K = 128
//     stage; once more with a commit after every block, as the GEMMs release
//     each shared-memory stage;
//   * tcgen05 kind::f8f6f4 (E4M3 x E4M3), one CTA, M 128 x N 256, the
//     FP8 layer's denominator;
//   * mma.sync m16n8k32 s8 x s8 -> s32, the legacy warp-level integer path.
// Each tensor-core case runs one issuing thread per CTA (or pair) that keeps
// its accumulator busy back to back, one CTA per SM; the issuing CTA times
// itself with clock64 from the first issue to the completion of the last MMA,
// and the whole grid is timed with CUDA events.  Every wait is bounded
// (2 s, then an error flag).  Prints one JSON line.
#include <cstdint>
#include <cstdio>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "csrc/ptx.cuh"

using namespace moe;

namespace {

constexpr int kSmemBytes = 160 * 1024;  // forces one CTA per SM
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kACol = 256;          // A operand columns in tensor memory (64 of them)

__device__ __forceinline__ uint16_t f16_bits_of_int(int v) { return __half_as_ushort(__int2half_rn(v)); }

__device__ bool wait_bounded(uint64_t* bar, uint32_t parity) {
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_timer_ns() - t0 > 2000000000ull) return false;
    return true;
}

__device__ __forceinline__ void mma_f8_smem_a(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                              uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// KIND 0: kind::f16 on int8-valued fp16; KIND 1: kind::f8f6f4 E4M3.
template <int KIND, bool A_TMEM, bool PAIR, int N, bool COMMIT_EACH>
__global__ void __launch_bounds__(128, 1) tc_rate(int blocks, long long* cycles, int* err) {
    extern __shared__ uint8_t raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    constexpr int kBRows = PAIR ? N / 2 : N;
    uint8_t* a_sm = sm;              // 128 rows x 128 B (A in shared memory only)
    uint8_t* b_sm = sm + 16384;      // kBRows x 128 B
    __shared__ uint64_t done_bar, stage_bar;
    __shared__ uint32_t tmem_slot;
    const int tid = threadIdx.x, warp = tid >> 5;
    const uint32_t rank = PAIR ? cluster_ctarank() : 0;

    for (int i = tid; i < (16384 + kBRows * 128) / 2; i += blockDim.x) {
        const int v = static_cast<int>((static_cast<uint32_t>(i) * 2654435761u) >> 9) % 128 - 64;
        reinterpret_cast<uint16_t*>(sm)[i] =
            KIND == 0 ? f16_bits_of_int(v) : static_cast<uint16_t>((v & 0x37) | ((v & 0x37) << 8));
    }
    if (tid == 0) {
        mbar_init(&done_bar, 1);
        mbar_init(&stage_bar, (1u << 20) - 1);  // never completes: takes the per-block commits
        fence_barrier_init();
    }
    if (warp == 0) {
        if (PAIR) {
            tmem_alloc_pair(&tmem_slot, kTmemCols);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(&tmem_slot, kTmemCols);
            tmem_relinquish();
        }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    if (PAIR) cluster_sync_all(); else __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    if (A_TMEM) {  // every warp fills its 32 lanes of the A columns
        uint32_t r[32];
        for (int c = 0; c < 64; c += 32) {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const int v = (tid * 7 + (c + j) * 13) % 128 - 64;
                r[j] = static_cast<uint32_t>(f16_bits_of_int(v)) * 0x10001u;
            }
            tmem_st_32(tmem + (static_cast<uint32_t>(warp * 32) << 16) + kACol + c, r);
        }
        tmem_wait_st();
    }
    tc_fence_before();
    if (PAIR) cluster_sync_all(); else __syncthreads();
    tc_fence_after();

    if (tid == 0 && rank == 0) {
        const uint32_t idesc = idesc_f16_f32(PAIR ? 256 : 128, N);
        const uint64_t ad = smem_desc_sw128(smem_u32(a_sm)), bd = smem_desc_sw128(smem_u32(b_sm));
        const long long c0 = clock64();
        for (int blk = 0; blk < blocks; ++blk) {
            if (PAIR) {
                mma8_f16_tmem_a_pair(tmem, tmem + kACol, bd, 0, idesc, blk ? 1u : 0u);
                if (COMMIT_EACH) mma_commit_pair(&stage_bar, 3);
            } else {
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t acc = (blk | ks) ? 1u : 0u;
                    const uint64_t bk = bd + static_cast<uint64_t>((ks & 3) * 2);
                    if (KIND == 1) mma_f8_smem_a(tmem, ad + static_cast<uint64_t>((ks & 3) * 2), bk, idesc, acc);
                    else if (A_TMEM) mma_f16_tmem_a(tmem, tmem + kACol + ks * 8, bk, idesc, acc);
                    else mma_f16_smem_a(tmem, ad + static_cast<uint64_t>((ks & 3) * 2), bk, idesc, acc);
                }
                if (COMMIT_EACH) mma_commit(&stage_bar);
            }
        }
        if (PAIR) mma_commit_pair(&done_bar, 3); else mma_commit(&done_bar);
        if (!wait_bounded(&done_bar, 0)) atomicOr(err, 1);
        cycles[blockIdx.x / (PAIR ? 2 : 1)] = clock64() - c0;
    }
    if (PAIR && tid == 0 && rank == 1 && !wait_bounded(&done_bar, 0)) atomicOr(err, 1);
    tc_fence_before();
    if (PAIR) cluster_sync_all(); else __syncthreads();
    tc_fence_after();
    if (warp == 0) {
        if (PAIR) tmem_dealloc_pair(tmem, kTmemCols); else tmem_dealloc(tmem, kTmemCols);
    }
}

// mma.sync m16n8k32 s8 x s8 -> s32, eight independent accumulator chains per warp
__global__ void __launch_bounds__(256) s8_rate(int iters, long long* cycles, int* sink) {
    uint32_t a[4], b[2];
    const uint32_t lane = threadIdx.x & 31;
#pragma unroll
    for (int i = 0; i < 4; ++i) a[i] = 0x01020304u * (lane + i + 1);
    b[0] = 0x05060708u * (lane + 3);
    b[1] = 0x0a0b0c0du * (lane + 5);
    int c[8][4] = {};
    const long long c0 = clock64();
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int j = 0; j < 8; ++j)
            asm volatile("mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                         "{%0,%1,%2,%3};"
                         : "+r"(c[j][0]), "+r"(c[j][1]), "+r"(c[j][2]), "+r"(c[j][3])
                         : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
    }
    const long long dt = clock64() - c0;
    int s = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) s += c[j][0] + c[j][1] + c[j][2] + c[j][3];
    if (s == 0x7fffffff) sink[0] = s;
    if (threadIdx.x == 0) cycles[blockIdx.x] = dt;
}

struct Result {
    double ops_per_clk_sm, tops, mhz;
};

template <typename Launch>
bool timed(Launch launch, int n_timers, double ops_total, double ops_per_timer_per_sm, long long* d_cyc,
           Result* out) {
    cudaEvent_t e0, e1;
    cudaEventCreate(&e0);
    cudaEventCreate(&e1);
    float ms = 0.f;
    for (int rep = 0; rep < 3; ++rep) {  // the last of three counts (warm clocks)
        cudaEventRecord(e0);
        if (launch() != cudaSuccess) return false;
        cudaEventRecord(e1);
        if (cudaEventSynchronize(e1) != cudaSuccess) return false;
        cudaEventElapsedTime(&ms, e0, e1);
    }
    static long long h[4096];
    if (cudaMemcpy(h, d_cyc, n_timers * sizeof(long long), cudaMemcpyDeviceToHost) != cudaSuccess) return false;
    long long mx = 1;
    for (int i = 0; i < n_timers; ++i) mx = h[i] > mx ? h[i] : mx;
    out->ops_per_clk_sm = ops_per_timer_per_sm / static_cast<double>(mx);
    out->tops = ops_total / (ms * 1e-3) / 1e12;
    out->mhz = static_cast<double>(mx) / (ms * 1e3);
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    return true;
}

template <int KIND, bool A_TMEM, bool PAIR, int N, bool COMMIT_EACH>
bool run_tc(int nsm, int blocks, long long* d_cyc, int* d_err, Result* out) {
    auto kern = tc_rate<KIND, A_TMEM, PAIR, N, COMMIT_EACH>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) != cudaSuccess)
        return false;
    const int grid = PAIR ? nsm & ~1 : nsm;
    auto launch = [=]() {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(grid);
        cfg.blockDim = dim3(128);
        cfg.dynamicSmemBytes = kSmemBytes;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = PAIR ? 2 : 1;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return cudaLaunchKernelEx(&cfg, kern, blocks, d_cyc, d_err);
    };
    const double k_per_mma = KIND == 0 ? 16 : 32;
    const double per_issuer = 2.0 * (PAIR ? 256 : 128) * N * k_per_mma * 8.0 * blocks;
    const int issuers = PAIR ? grid / 2 : grid;
    return timed(launch, issuers, per_issuer * issuers, per_issuer / (PAIR ? 2 : 1), d_cyc, out);
}

void print(const char* name, const Result& r, bool last) {
    printf("\"%s\": {\"ops_per_clk_per_sm\": %.0f, \"tops\": %.1f, \"sm_mhz\": %.0f}%s", name, r.ops_per_clk_sm,
           r.tops, r.mhz, last ? "" : ", ");
}

}  // namespace

int main() {
    int dev = 0, nsm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 2;
    cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    long long* d_cyc = nullptr;
    int* d_err = nullptr;
    if (cudaMalloc(&d_cyc, 4096 * sizeof(long long)) != cudaSuccess) return 2;
    if (cudaMalloc(&d_err, 4 * sizeof(int)) != cudaSuccess) return 2;
    cudaMemset(d_err, 0, 4 * sizeof(int));
    const int blocks = 4000;  // 32000 MMAs per issuer: a few milliseconds
    Result r[8];
    bool ok = run_tc<0, false, false, 256, false>(nsm, blocks, d_cyc, d_err, &r[0]) &&
              run_tc<0, true, false, 256, false>(nsm, blocks, d_cyc, d_err, &r[1]) &&
              run_tc<0, true, true, 192, false>(nsm, blocks, d_cyc, d_err, &r[2]) &&
              run_tc<0, true, true, 256, false>(nsm, blocks, d_cyc, d_err, &r[3]) &&
              run_tc<0, true, true, 192, true>(nsm, blocks, d_cyc, d_err, &r[4]) &&
              run_tc<1, false, false, 256, false>(nsm, blocks, d_cyc, d_err, &r[5]);
    if (!ok) {
        fprintf(stderr, "launch failed: %s\n", cudaGetErrorString(cudaGetLastError()));
        return 3;
    }
    const int s8_iters = 4000, s8_blocks = nsm * 4;  // four CTAs of eight warps per SM
    auto s8_launch = [=]() {
        s8_rate<<<s8_blocks, 256>>>(s8_iters, d_cyc, d_err + 2);
        return cudaGetLastError();
    };
    const double s8_per_cta = 2.0 * 16 * 8 * 32 * 8.0 * 8.0 * s8_iters;  // 8 warps x 8 chains
    if (!timed(s8_launch, s8_blocks, s8_per_cta * s8_blocks, s8_per_cta * 4, d_cyc, &r[6])) return 3;
    int h_err[4] = {};
    cudaMemcpy(h_err, d_err, sizeof(h_err), cudaMemcpyDeviceToHost);
    printf("{\"sms\": %d, \"wait_timeouts\": %d, ", nsm, h_err[0]);
    print("tcgen05_f16_int8_values_smem_a_m128_n256", r[0], false);
    print("tcgen05_f16_int8_values_tmem_a_m128_n256", r[1], false);
    print("tcgen05_f16_int8_values_pair_tmem_a_m256_n192", r[2], false);
    print("tcgen05_f16_int8_values_pair_tmem_a_m256_n256", r[3], false);
    print("tcgen05_f16_int8_values_pair_tmem_a_m256_n192_commit_per_block", r[4], false);
    print("tcgen05_e4m3_smem_a_m128_n256", r[5], false);
    print("mma_sync_s8_m16n8k32", r[6], true);
    printf("}\n");
    return h_err[0] ? 4 : 0;
}

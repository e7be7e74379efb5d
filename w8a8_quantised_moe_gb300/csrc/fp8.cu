// fp8.cu -- the FP8 (E4M3) variant of the layer: quantisers to E4M3 and the
// grouped FP8 GEMM on the tcgen05 tensor cores (kind::f8f6f4).
//
// "DeepSeek V4 950 FP8 inference on H100" (lpnh.cn): E4M3 weights and
// activations (section 2.1), FP8 operands with an FP32 accumulator whose
// result is re-quantised to FP8 for the next operator (2.3), per-channel
// weight scales and per-token dynamic activation scales (2.4), weight scales
// from the absolute maximum (3.1).  A row's scale is s = amax / 448 (the
// largest E4M3 magnitude) and its codes are the E4M3 values nearest to the
// binary32 quotients x / s, ties to even, saturated at 448
// (cvt.rn.satfinite.e4m3x2.f32).  Router, slots, SiLU gate and combine are
// the INT8 layer's kernels.
//
// GEMM.  E4M3 operands need no conversion on GB300: both the weight tile (A,
// 128 output channels x 128 K bytes) and the activation tile (B, N rows x 128
// K bytes) go from global memory to shared memory by TMA in the 128-byte
// swizzle, and one thread issues four K = 32 MMAs per stage reading both from
// shared memory, with D (fp32) in tensor memory.  The products of two E4M3
// values are exact; the tensor cores accumulate them in fp32.
//   warp 0      TMA producer
//   warp 1      TMEM allocator and MMA issuer
//   warps 2-5   epilogue (tcgen05.ld, scales, SiLU gate, outputs)
// Persistent grid, tiles dealt round-robin, accumulators double-buffered,
// every wait bounded (ptx.cuh); a timeout aborts the CTA cleanly.
#include <mutex>

#include "gemm_common.cuh"

namespace moe {
namespace {

constexpr float kE4m3Max = 448.0f;

// Two E4M3 codes (lo in the low byte) of two binary32 values: round to
// nearest even, saturate at +-448.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// Codes of four values of one row with scale s (s == 0: all codes 0).
__device__ __forceinline__ uint32_t e4m3_codes4(float a, float b, float c, float d, float s) {
    if (s == 0.f) return 0u;
    const uint32_t lo = e4m3x2(__fdiv_rn(a, s), __fdiv_rn(b, s));
    const uint32_t hi = e4m3x2(__fdiv_rn(c, s), __fdiv_rn(d, s));
    return lo | (hi << 16);
}

__device__ __forceinline__ float warp_max_f(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
    return v;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// One warp per weight row (fp32 [rows][K], K a multiple of 4); grid-stride.
__global__ void __launch_bounds__(256) quantize_weights_fp8_kernel(const float* __restrict__ w, int64_t rows, int K,
                                                                   uint8_t* __restrict__ q, float* __restrict__ s_out) {
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = (int64_t)gridDim.x * 8;
    for (int64_t r = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5); r < rows; r += nwarps) {
        const float4* row = reinterpret_cast<const float4*>(w + r * K);
        float amax = 0.f;
        for (int i = lane; i < K / 4; i += 32) {
            const float4 v = row[i];
            amax = fmaxf(fmaxf(fmaxf(amax, fabsf(v.x)), fmaxf(fabsf(v.y), fabsf(v.z))), fabsf(v.w));
        }
        amax = warp_max_f(amax);
        const float s = __fdiv_rn(amax, kE4m3Max);
        if (lane == 0) s_out[r] = s;
        uint32_t* qr = reinterpret_cast<uint32_t*>(q + r * K);
        for (int i = lane; i < K / 4; i += 32) {
            const float4 v = row[i];
            qr[i] = e4m3_codes4(v.x, v.y, v.z, v.w, s);
        }
    }
}

// One warp per token (bf16 [T][H]): slots of the token's k choices (as the
// INT8 quantiser computes them), s = amax / 448, E4M3 codes of the row
// written into each of its slot rows of q8 ([S][H] bytes).
__global__ void __launch_bounds__(256) permute_quant_fp8_kernel(
    const uint16_t* __restrict__ x, const int32_t* __restrict__ topk_ids, const int32_t* __restrict__ rank,
    const int32_t* __restrict__ base, int T, int H, int E, int k, int32_t* __restrict__ slot_of,
    int32_t* __restrict__ slot_token, float* __restrict__ s_x, float* __restrict__ s_slot,
    uint8_t* __restrict__ q8, int* __restrict__ error) {
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
    pdl_wait();
    pdl_trigger();
    if (t >= T) return;
    int my_slot = t;  // -1: out of range (checked build), its writes skipped
    if (lane < k) {
        const int e = topk_ids[(size_t)t * k + lane];
        my_slot = in_range(e, 0, E, error) ? base[(size_t)(t / kRouterTokens) * E + e] + rank[(size_t)t * k + lane]
                                           : -1;
        if (my_slot >= 0 && !in_range(my_slot, 0, (long long)T * k, error)) my_slot = -1;
        slot_of[(size_t)t * k + lane] = my_slot;
        if (!kChecked || my_slot >= 0) slot_token[my_slot] = t;
    }
    const uint4* row = reinterpret_cast<const uint4*>(x + (size_t)t * H);
    const int nv = H / 8;  // 8 bf16 per 16-byte vector
    float amax = 0.f;
    for (int i = lane; i < nv; i += 32) {
        const uint4 v = __ldg(row + i);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(w[j])), fabsf(bf16_hi(w[j]))));
    }
    amax = warp_max_f(amax);
    const float s = __fdiv_rn(amax, kE4m3Max);
    if (lane == 0) s_x[t] = s;
    if (lane < k && (!kChecked || my_slot >= 0)) s_slot[my_slot] = s;
    int slots[kMaxTopK];  // taken before the lanes' loop trip counts differ
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) slots[j] = __shfl_sync(0xffffffffu, my_slot, j);
    for (int i = lane; i < nv; i += 32) {
        const uint4 v = __ldg(row + i);
        const uint2 c = make_uint2(e4m3_codes4(bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y), s),
                                   e4m3_codes4(bf16_lo(v.z), bf16_hi(v.z), bf16_lo(v.w), bf16_hi(v.w), s));
        for (int j = 0; j < k; ++j)
            if (!kChecked || slots[j] >= 0) reinterpret_cast<uint2*>(q8 + (size_t)slots[j] * H)[i] = c;
    }
}

// One warp per slot row of h (fp32 [S][I]): s_h = amax / 448 and E4M3 codes.
__global__ void __launch_bounds__(256) requant_fp8_kernel(const float* __restrict__ h, int S, int I,
                                                          float* __restrict__ s_h, uint8_t* __restrict__ q8) {
    const int lane = threadIdx.x & 31;
    const int r = blockIdx.x * 8 + (threadIdx.x >> 5);
    pdl_wait();
    pdl_trigger();
    if (r >= S) return;
    const float4* row = reinterpret_cast<const float4*>(h + (size_t)r * I);
    float amax = 0.f;
    for (int i = lane; i < I / 4; i += 32) {
        const float4 v = row[i];
        amax = fmaxf(fmaxf(fmaxf(amax, fabsf(v.x)), fmaxf(fabsf(v.y), fabsf(v.z))), fabsf(v.w));
    }
    amax = warp_max_f(amax);
    const float s = __fdiv_rn(amax, kE4m3Max);
    if (lane == 0) s_h[r] = s;
    uint32_t* qr = reinterpret_cast<uint32_t*>(q8 + (size_t)r * I);
    for (int i = lane; i < I / 4; i += 32) {
        const float4 v = row[i];
        qr[i] = e4m3_codes4(v.x, v.y, v.z, v.w, s);
    }
}

// Few rows (decode): one CTA of 256 threads per token (or per row of h), the
// row held in registers, so that the whole GPU works on the few rows; the
// same outputs as the warp-per-row kernels above.  H <= 256 * 8 * kF8Vec
// (bf16 x) and I <= 256 * 4 * kF8Vec (fp32 h).
constexpr int kF8Vec = 8;

__device__ __forceinline__ float cta_max_f(float v, float* red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    v = warp_max_f(v);
    if (lane == 0) red[warp] = v;
    __syncthreads();
    v = red[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) v = fmaxf(v, red[i]);
    return v;
}

__global__ void __launch_bounds__(256) permute_quant_fp8_cta_kernel(
    const uint16_t* __restrict__ x, const int32_t* __restrict__ topk_ids, const int32_t* __restrict__ rank,
    const int32_t* __restrict__ base, int T, int H, int E, int k, int32_t* __restrict__ slot_of,
    int32_t* __restrict__ slot_token, float* __restrict__ s_x, float* __restrict__ s_slot,
    uint8_t* __restrict__ q8, int* __restrict__ error) {
    __shared__ float red[8];
    __shared__ int slots_s[kMaxTopK];
    const int tid = threadIdx.x;
    const int t = blockIdx.x;
    pdl_wait();
    pdl_trigger();
    if (t >= T) return;
    if (tid < k) {
        const int e = topk_ids[(size_t)t * k + tid];
        int my_slot = in_range(e, 0, E, error) ? base[(size_t)(t / kRouterTokens) * E + e] + rank[(size_t)t * k + tid]
                                               : -1;  // -1: out of range (checked build), its writes skipped
        if (my_slot >= 0 && !in_range(my_slot, 0, (long long)T * k, error)) my_slot = -1;
        slot_of[(size_t)t * k + tid] = my_slot;
        if (!kChecked || my_slot >= 0) slot_token[my_slot] = t;
        slots_s[tid] = my_slot;
    }
    const uint4* row = reinterpret_cast<const uint4*>(x + (size_t)t * H);
    const int nv = H / 8;  // 8 bf16 per 16-byte vector
    uint4 v[kF8Vec];
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < kF8Vec; ++i) {
        const int idx = tid + 256 * i;
        v[i] = idx < nv ? __ldg(row + idx) : make_uint4(0u, 0u, 0u, 0u);
        const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(w[j])), fabsf(bf16_hi(w[j]))));
    }
    amax = cta_max_f(amax, red);  // its barrier also publishes slots_s
    const float s = __fdiv_rn(amax, kE4m3Max);
    if (tid == 0) s_x[t] = s;
    if (tid < k && (!kChecked || slots_s[tid] >= 0)) s_slot[slots_s[tid]] = s;
#pragma unroll
    for (int i = 0; i < kF8Vec; ++i) {
        const int idx = tid + 256 * i;
        if (idx >= nv) break;
        const uint2 c = make_uint2(e4m3_codes4(bf16_lo(v[i].x), bf16_hi(v[i].x), bf16_lo(v[i].y), bf16_hi(v[i].y), s),
                                   e4m3_codes4(bf16_lo(v[i].z), bf16_hi(v[i].z), bf16_lo(v[i].w), bf16_hi(v[i].w), s));
        for (int j = 0; j < k; ++j)
            if (!kChecked || slots_s[j] >= 0) reinterpret_cast<uint2*>(q8 + (size_t)slots_s[j] * H)[idx] = c;
    }
}

__global__ void __launch_bounds__(256) requant_fp8_cta_kernel(const float* __restrict__ h, int S, int I,
                                                              float* __restrict__ s_h, uint8_t* __restrict__ q8) {
    __shared__ float red[8];
    const int tid = threadIdx.x;
    const int r = blockIdx.x;
    pdl_wait();
    pdl_trigger();
    if (r >= S) return;
    const float4* row = reinterpret_cast<const float4*>(h + (size_t)r * I);
    const int nv = I / 4;
    float4 v[kF8Vec];
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < kF8Vec; ++i) {
        const int idx = tid + 256 * i;
        v[i] = idx < nv ? row[idx] : make_float4(0.f, 0.f, 0.f, 0.f);
        amax = fmaxf(fmaxf(fmaxf(amax, fabsf(v[i].x)), fmaxf(fabsf(v[i].y), fabsf(v[i].z))), fabsf(v[i].w));
    }
    amax = cta_max_f(amax, red);
    const float s = __fdiv_rn(amax, kE4m3Max);
    if (tid == 0) s_h[r] = s;
    uint32_t* qr = reinterpret_cast<uint32_t*>(q8 + (size_t)r * I);
#pragma unroll
    for (int i = 0; i < kF8Vec; ++i) {
        const int idx = tid + 256 * i;
        if (idx >= nv) break;
        qr[idx] = e4m3_codes4(v[i].x, v[i].y, v[i].z, v[i].w, s);
    }
}

// One tcgen05 MMA, kind::f8f6f4, both operands from shared memory: D[M x N]
// (+)= A[M x 32] * B[N x 32]^T.  The instruction descriptor's operand format
// fields are 0 = E4M3 for this kind.
__device__ __forceinline__ void mma_f8_smem(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__host__ __device__ constexpr uint32_t idesc_e4m3_f32(uint32_t M, uint32_t N) {
    return (1u << 4)            // D format: f32
           | (0u << 7)          // A format: E4M3
           | (0u << 10)         // B format: E4M3
           | ((N >> 3) << 17)   // N / 8
           | ((M >> 4) << 24);  // M / 16
}

constexpr int kF8Threads = 192;  // producer, MMA, 4 epilogue warps
constexpr int kF8EpiWarp0 = 2;
constexpr int kF8BK = 128;       // K bytes (= elements) per stage

template <int BN_, int NS_>
struct F8Cfg {
    static constexpr int BN = BN_;  // activation rows per tile (MMA N, at most)
    static constexpr int NS = NS_;  // stages
    static constexpr int ND = 2;    // accumulator buffers
    static constexpr int kStageA = kTileM * kF8BK;  // [128 x 128] E4M3, two 64-row boxes
    static constexpr int kStageB = BN * kF8BK;      // [BN x 128] E4M3
    static constexpr int kStage = kStageA + kStageB;
    static constexpr int kTmemCols = ND * BN;
    static constexpr int kTmemAlloc = kTmemCols <= 128 ? 128 : kTmemCols <= 256 ? 256 : 512;
    static constexpr int kXchStride = 33;
    static constexpr int kXch = kTileM * kXchStride * 4;
    static constexpr int kOffXch = NS * kStage;
    static constexpr int kOffBars = kOffXch + kXch;
    static constexpr int kNumBars = 2 * NS + 2 * ND + 3;  // ..., teardown, epi_bar, stall_bar
    static constexpr int kOffTiles = kOffBars + kNumBars * 8;
    static constexpr int kOffRowInfo = kOffTiles + (kMaxExperts + 1) * 4 * 2;  // [2][BN] activation scales
    static constexpr int kOffMisc = kOffRowInfo + 2 * BN * 4;
    static constexpr int kSmem = kOffMisc + 64 + 1024;  // + alignment slack
    static_assert(kStageA % 1024 == 0 && kStageB % 1024 == 0, "stages keep 1024-byte alignment");
    static_assert(BN % 32 == 0 && BN <= 256, "tile width");
    static_assert(kTmemCols <= 512, "TMEM budget");
    static_assert(kSmem <= 232448, "shared memory budget");
};
// Wide tiles for groups of many rows; narrow tiles with a deep ring for a
// few rows per group (decode), where each stage is mostly a weight tile
// streamed from HBM and the depth of the ring sets the bytes in flight.
using F8Wide = F8Cfg<256, 4>;
using F8Narrow = F8Cfg<32, 10>;

template <int BN>
__device__ __forceinline__ void f8_decode_tile(const Tiles& t, int tile, int& g, int& cb, int& row0, int& nvalid) {
    g = last_le(t.tile_start, t.n_groups, tile);
    const int local = tile - t.tile_start[g];
    const int rows = t.row_start[g + 1] - t.row_start[g];
    const int ntb = (rows + BN - 1) / BN;
    cb = local / ntb;
    const int tb = local - cb * ntb;
    row0 = t.row_start[g] + tb * BN;
    nvalid = min(BN, t.row_start[g + 1] - row0);
}

// Activation boxes of 32, 64, 128 or BN rows: a tile loads the smallest that
// covers its valid rows (rows past the matrix read as zeros).
__device__ __forceinline__ int f8_box_index(int nvalid) {
    return nvalid <= 32 ? 0 : nvalid <= 64 ? 1 : nvalid <= 128 ? 2 : 3;
}
template <int BN>
__host__ __device__ constexpr int f8_box_rows(int i) {
    return i == 0 ? (BN < 32 ? BN : 32) : i == 1 ? (BN < 64 ? BN : 64) : i == 2 ? (BN < 128 ? BN : 128) : BN;
}

template <class C, int EPI>
__global__ void __launch_bounds__(kF8Threads, 1)
    grouped_gemm_fp8_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_b0,
                            const __grid_constant__ CUtensorMap tmap_b1, const __grid_constant__ CUtensorMap tmap_b2,
                            const __grid_constant__ CUtensorMap tmap_b3, const GemmArgs args) {
    constexpr int BN = C::BN, NS = C::NS, ND = C::ND;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBars);
    uint64_t* full = bars;                // [NS] both tiles of the stage landed
    uint64_t* empty = bars + NS;          // [NS] MMAs of the stage completed
    uint64_t* acc_full = bars + 2 * NS;   // [ND]
    uint64_t* acc_empty = acc_full + ND;  // [ND] 4 epilogue warps
    uint64_t* teardown = acc_empty + ND;
    uint64_t* epi_bar = teardown + 1;
    uint64_t* stall_bar = epi_bar + 1;  // test hook: nothing arrives on it
    int* tile_start = reinterpret_cast<int*>(smem + C::kOffTiles);
    int* row_start = tile_start + (kMaxExperts + 1);
    float* row_scale_s = reinterpret_cast<float*>(smem + C::kOffRowInfo);  // [2][BN]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 8);
    float* xch = reinterpret_cast<float*>(smem + C::kOffXch);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_groups = args.n_groups;
    const int nkb = args.K / kF8BK;  // K is a multiple of 128

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int d = 0; d < ND; ++d) {
            mbar_init(&acc_full[d], 1);
            mbar_init(&acc_empty[d], 4);
        }
        mbar_init(teardown, 1);
        mbar_init(epi_bar, 4);
        mbar_init(stall_bar, 1);
        *abort_flag = 0;
        fence_barrier_init();
        tma_prefetch_desc(&tmap_w);
        tma_prefetch_desc(&tmap_b0);
        tma_prefetch_desc(&tmap_b1);
        tma_prefetch_desc(&tmap_b2);
        tma_prefetch_desc(&tmap_b3);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, C::kTmemAlloc);
        tmem_relinquish();
    }
    pdl_wait();  // the previous kernel's outputs (offsets, codes, scales) are visible from here
    pdl_trigger();
    if (warp == 2) {  // tile table: tiles of group g = ceil(rows_g / BN) * n_cb
        int carry = 0;
        bool bad = false;  // checked build: an offset out of order or range
        for (int base = 0; base < n_groups; base += 32) {
            const int g = base + lane;
            int r0 = 0, r1 = 0;
            if (g < n_groups) {
                r0 = args.offsets ? args.offsets[g] : 0;
                r1 = args.offsets ? args.offsets[g + 1] : args.total_rows;
                if (!group_rows_ok(r0, r1, args.total_rows, args.error)) {
                    bad = true;
                    r0 = r1 = 0;
                }
                row_start[g] = r0;
                if (g == n_groups - 1) row_start[n_groups] = r1;
            }
            const int v = (g < n_groups) ? ((r1 - r0 + BN - 1) / BN) * args.n_cb : 0;
            int incl = v;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int o = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += o;
            }
            if (g < n_groups) tile_start[g] = carry + incl - v;
            carry += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) tile_start[n_groups] = carry;
        if (kChecked && __any_sync(0xffffffffu, bad)) {  // an empty, consistent table: no tile runs
            for (int g = lane; g <= n_groups; g += 32) {
                row_start[g] = 0;
                tile_start[g] = 0;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int total_tiles = tile_start[n_groups];
    const Tiles tiles{tile_start, row_start, n_groups};
    const WaitCtl ctl{abort_flag, args.error, args.timeout_ns, 0u};

    if (warp == 0) {
        // ---------------------------------------------------------- producer
        // three boxes a stage (weight rows 0-63 and 64-127, activation rows);
        // lanes 0-2 issue one each in the same warp instruction (a bulk
        // tensor copy costs its issuing thread ~200 cycles); lane 0 owns the
        // waits and the arrival
        if (lane < 3) {
            uint32_t it = 0;
            int ok = 1;
            if (lane == 0) ok = !args.stall || mbar_wait(stall_bar, 0, ctl);  // the test hook's wait runs out
            ok = __shfl_sync(0x7u, ok, 0);
            for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
                int g, cb, row0, nvalid;
                f8_decode_tile<BN>(tiles, tile, g, cb, row0, nvalid);
                int wrow0, wrow1;  // weight rows 0-63 and 64-127 of the tile
                if (EPI == (int)Epi::GateUp) {
                    wrow0 = g * args.w_rows_per_group + cb * 64;
                    wrow1 = wrow0 + args.up_offset;
                } else {
                    wrow0 = g * args.w_rows_per_group + cb * kTileM;
                    wrow1 = wrow0 + 64;
                }
                const int bi = f8_box_index(nvalid);
                const CUtensorMap* mb = bi == 0 ? &tmap_b0 : bi == 1 ? &tmap_b1 : bi == 2 ? &tmap_b2 : &tmap_b3;
                const uint32_t stage_bytes = (uint32_t)(C::kStageA + f8_box_rows<BN>(bi) * kF8BK);
                const CUtensorMap* map = lane == 2 ? mb : &tmap_w;
                const int row = lane == 0 ? wrow0 : lane == 1 ? wrow1 : row0;
                const int off = lane == 0 ? 0 : lane == 1 ? C::kStageA / 2 : C::kStageA;
                for (int kb = 0; kb < nkb; ++kb, ++it) {
                    const uint32_t s = it % NS, ph = (it / NS) & 1u;
                    if (lane == 0) {
                        ok = mbar_wait(&empty[s], ph ^ 1u, ctl);
                        if (ok) mbar_arrive_expect_tx(&full[s], stage_bytes);
                    }
                    ok = __shfl_sync(0x7u, ok, 0);
                    if (!ok) break;
                    tma_load_2d(smem + s * C::kStage + off, map, &full[s], kb * kF8BK, row);
                }
            }
            // drain: every fill issued must land before the CTA may exit
            if (lane == 0)
                for (uint32_t s = 0; s < (uint32_t)NS && s < it; ++s) {
                    const uint32_t last = it - 1 - ((it - 1 - s) % NS);
                    mbar_wait_drain(&full[s], (last / NS) & 1u);
                }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------ MMA issuer
        if (lane == 0) {
            uint32_t it = 0, tl = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x, ++tl) {
                int g, cb, row0, nvalid;
                f8_decode_tile<BN>(tiles, tile, g, cb, row0, nvalid);
                const uint32_t idesc = idesc_e4m3_f32(kTileM, (uint32_t)((nvalid + 15) & ~15));
                const uint32_t d = tl % ND;
                if (!mbar_wait(&acc_empty[d], ((tl / ND) & 1u) ^ 1u, ctl)) break;
                tc_fence_after();
                const uint32_t d_col = d * BN;
                for (int kb = 0; kb < nkb; ++kb, ++it) {
                    const uint32_t s = it % NS, ph = (it / NS) & 1u;
                    if (!mbar_wait(&full[s], ph, ctl)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t a_base = smem_u32(smem + s * C::kStage);
                    const uint32_t b_base = a_base + C::kStageA;
#pragma unroll
                    for (int ks = 0; ks < kF8BK / 32; ++ks)  // 32 bytes of K per MMA
                        mma_f8_smem(tmem + d_col, smem_desc_sw128(a_base) + (uint64_t)(ks * 2),
                                    smem_desc_sw128(b_base) + (uint64_t)(ks * 2), idesc,
                                    (kb != 0 || ks != 0) ? 1u : 0u);
                    mma_commit(&empty[s]);
                }
                if (!ok) break;
                mma_commit(&acc_full[d]);
            }
            mma_commit(teardown);
            mbar_wait_drain(teardown, 0);
        }
    } else {
        // --------------------------------------------------------- epilogue
        const int q = warp & 3;
        const int ew = warp - kF8EpiWarp0;  // 0..3
        const int row = q * 32 + lane;      // TMEM lane = weight row of the tile
        const uint32_t lane_addr = (uint32_t)(q * 32) << 16;
        uint32_t tl = 0, eit = 0;
        bool ok = true;
        for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x, ++tl) {
            int g, cb, row0, nvalid;
            f8_decode_tile<BN>(tiles, tile, g, cb, row0, nvalid);
            const uint32_t d = tl % ND;
            int wrow;  // this thread's weight row within the group
            if (EPI == (int)Epi::GateUp) wrow = (row >> 6) * args.up_offset + cb * 64 + (row & 63);
            else wrow = cb * kTileM + row;
            const float sw = __ldg(args.w_scale + (size_t)g * args.w_rows_per_group + wrow);
            // the tile's activation scales, staged while the MMAs run (buffer
            // tl & 1: its previous user, tile tl - 2, passed the last barrier)
            float* sa = row_scale_s + (tl & 1u) * BN;
            for (int j = ew * 32 + lane; j < BN; j += 128) sa[j] = j < nvalid ? __ldg(args.act_scale + row0 + j) : 0.f;
            if (!epi_sync(epi_bar, eit, ctl)) break;
            if (!warp_wait(&acc_full[d], (tl / ND) & 1u, ctl)) break;
            tc_fence_after();
            const uint32_t col0 = d * BN;
            const int nch = (nvalid + 31) / 32;
            for (int ch = 0; ch < nch; ++ch) {
                uint32_t r[32];
                tmem_ld_32(tmem + lane_addr + col0 + ch * 32, r);
                tmem_wait_ld();
                if (ch == nch - 1) {  // every column is in registers: release the accumulator
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&acc_empty[d]);
                }
                const int j0 = ch * 32;
                if (args.acc_out) {  // raw fp32 accumulators (their bit patterns)
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (j0 + j < nvalid)
                            args.acc_out[(size_t)(row0 + j0 + j) * args.w_rows_per_group + wrow] = (int32_t)r[j];
                }
                if (EPI == (int)Epi::GateUp) {
                    float* xrow = xch + row * C::kXchStride;
#pragma unroll
                    for (int j = 0; j < 32; ++j) xrow[j] = dequant(__uint_as_float(r[j]), sa[j0 + j], sw);
                    if (!epi_sync(epi_bar, eit, ctl)) { ok = false; break; }
                    // warp ew: tokens j0 + 8*ew .. +7; lanes: channels lane, lane + 32
                    float* out = static_cast<float*>(args.out);
#pragma unroll
                    for (int t = 0; t < 8; ++t) {
                        const int j = ew * 8 + t;
                        if (j0 + j < nvalid) {
                            const int rr = row0 + j0 + j;
#pragma unroll
                            for (int c2 = 0; c2 < 2; ++c2) {
                                const int c = lane + 32 * c2;
                                const float gv = xch[c * C::kXchStride + j];
                                const float uv = xch[(64 + c) * C::kXchStride + j];
                                out[(size_t)rr * args.ld_out + cb * 64 + c] = __fmul_rn(silu_f32(gv), uv);
                            }
                        }
                    }
                    if (!epi_sync(epi_bar, eit, ctl)) { ok = false; break; }
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        if (j0 + j < nvalid) {
                            const float v = dequant(__uint_as_float(r[j]), sa[j0 + j], sw);
                            static_cast<float*>(args.out)[(size_t)(row0 + j0 + j) * args.ld_out + wrow] = v;
                        }
                    }
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

template <class C, int EPI>
cudaError_t launch_fp8_impl(const GemmArgs& args, cudaStream_t st, bool pdl) {
    auto kern = grouped_gemm_fp8_kernel<C, EPI>;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [&] {
        attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    });
    if (attr_err != cudaSuccess) return attr_err;
    CUtensorMap tw, tb[4];
    const uint64_t w_rows = (uint64_t)args.n_groups * args.w_rows_per_group;
    if (!make_tensor_map_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, args.w, args.K, w_rows, kF8BK, 64,
                            CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    for (int i = 0; i < 4; ++i)
        if (!make_tensor_map_2d(&tb[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, args.act8, args.K,
                                (uint64_t)args.total_rows, kF8BK, f8_box_rows<C::BN>(i), CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
    const long max_tiles = ((long)(args.total_rows + C::BN - 1) / C::BN + args.n_groups) * args.n_cb;
    int grid = num_sms();
    if (max_tiles < grid) grid = (int)max_tiles;
    if (grid < 1) grid = 1;
    return launch_kernel(kern, dim3(grid), dim3(kF8Threads), C::kSmem, st, pdl, tw, tb[0], tb[1], tb[2], tb[3], args);
}

}  // namespace

cudaError_t launch_quantize_weights_fp8(const float* w, int64_t rows, int K, uint8_t* q, float* s, cudaStream_t st) {
    if (rows == 0) return cudaSuccess;
    int64_t blocks = (rows + 7) / 8;
    const int64_t cap = (int64_t)num_sms() * 16;
    if (blocks > cap) blocks = cap;
    return launch_kernel(quantize_weights_fp8_kernel, dim3((unsigned)blocks), dim3(256), 0, st, false, w, rows, K, q,
                         s);
}

cudaError_t launch_permute_quant_fp8(const uint16_t* x, const int32_t* topk_ids, const int32_t* rank,
                                     const int32_t* hist, int T, int H, int E, int k, int32_t* slot_of,
                                     int32_t* slot_token, float* s_x, float* s_slot, uint8_t* q8, int* error,
                                     cudaStream_t st, bool pdl) {
    if (T == 0) return cudaSuccess;
    if ((long)T <= 8L * num_sms() && H <= 256 * 8 * kF8Vec)  // few tokens: a CTA per token
        return launch_kernel(permute_quant_fp8_cta_kernel, dim3(T), dim3(256), 0, st, pdl, x, topk_ids, rank, hist,
                             T, H, E, k, slot_of, slot_token, s_x, s_slot, q8, error);
    return launch_kernel(permute_quant_fp8_kernel, dim3((T + 7) / 8), dim3(256), 0, st, pdl, x, topk_ids, rank, hist,
                         T, H, E, k, slot_of, slot_token, s_x, s_slot, q8, error);
}

cudaError_t launch_requant_fp8(const float* h, int S, int I, float* s_h, uint8_t* q8, cudaStream_t st, bool pdl) {
    if (S == 0) return cudaSuccess;
    if ((long)S <= 8L * num_sms() && I <= 256 * 4 * kF8Vec)  // few rows: a CTA per row
        return launch_kernel(requant_fp8_cta_kernel, dim3(S), dim3(256), 0, st, pdl, h, S, I, s_h, q8);
    return launch_kernel(requant_fp8_kernel, dim3((S + 7) / 8), dim3(256), 0, st, pdl, h, S, I, s_h, q8);
}

// The CTA-pair kernel (gemm_fp8_pair.cu).
bool fp8_pair_gemm_supported(const GemmArgs& args);
cudaError_t launch_grouped_gemm_fp8_pair(Epi epi, const GemmArgs& args, cudaStream_t st, bool pdl);

cudaError_t launch_grouped_gemm_fp8(Epi epi, const GemmArgs& args, cudaStream_t st, bool pdl) {
    if (args.total_rows == 0) return cudaSuccess;
    if (args.act8 == nullptr || args.K % kF8BK != 0) return cudaErrorInvalidValue;
    const bool narrow = (long)args.total_rows <= 32L * (args.n_groups > 0 ? args.n_groups : 1);
    // wide groups on CTA pairs when the channel blocks pair up (measured on the
    // prefill layer: see the pair kernel's notes)
    if (!narrow && fp8_pair_gemm_supported(args)) return launch_grouped_gemm_fp8_pair(epi, args, st, pdl);
    switch (epi) {
        case Epi::GateUp:
            return narrow ? launch_fp8_impl<F8Narrow, 0>(args, st, pdl) : launch_fp8_impl<F8Wide, 0>(args, st, pdl);
        case Epi::ScaleF32:
            return narrow ? launch_fp8_impl<F8Narrow, 1>(args, st, pdl) : launch_fp8_impl<F8Wide, 1>(args, st, pdl);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace moe

// gemm.cu -- exact INT8 grouped GEMM on the sm_103a tensor cores with a fused
// epilogue.
//
// For every group g (an expert, or the single weight matrix of the linear
// layer) and every row r of the group's contiguous row range:
//     acc[r][n] = sum_k act[r][k] * w[g][n][k]        (int8 x int8 -> int32)
// followed by the scale outer product (acc * s_act[r]) * s_w[g][n] in the
// epilogue ("W8A8 quantisation of MiniMax-M3 on K100AI" (mhpn.cn), section
// 2.1), and, for the first expert GEMM, h = silu(g) * u of the gate and up
// halves.
//
// GB300 has no INT8 tcgen05 MMA (kind::i8 does not exist on sm_103a), so the
// product runs on kind::f16: int8 values are exact in fp16, products of two
// of them (|p| <= 2^14) are exact in the fp32 accumulator, and every TMEM
// accumulation covers at most 1024 products, so every partial sum is an
// integer of magnitude <= 2^24 and therefore exact.  After each 1024-long K
// chunk the epilogue warps convert the fp32 accumulator to int32 and add it
// to a running int32 sum, which makes the whole GEMM exact for any int8 input
// and any K <= 131071.
//
// Operand roles ("swap AB"): A = 128 weight rows per tile, converted from
// int8 to fp16 by converter warps straight into tensor memory; B = a tile of
// BN activation rows, already fp16, loaded by TMA (128-byte swizzle) into
// shared memory; D = 128 x N fp32 accumulator in tensor memory, N = the
// tile's valid rows rounded up to 16.  Warp roles of a CTA (320 threads):
//   warp 0      TMA producer (int8 weight tile + fp16 activation tile)
//   warp 1      TMEM allocator and single-thread MMA issuer
//   warps 2-5   converters: int8 weight rows -> fp16 pairs -> tcgen05.st
//   warps 6-9   epilogue: tcgen05.ld, int32 chunk sums, scales, outputs
// The grid is persistent; tiles are dealt round-robin.  Every wait is
// bounded (see ptx.cuh); a timeout aborts the CTA cleanly.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kThreads = 320;
constexpr int kBK = 64;         // K elements per pipeline stage
constexpr int kChunkKB = 16;    // stages per exact accumulation chunk (1024 K)
constexpr int kNumA = 4;        // TMEM stages of the converted A operand
constexpr int kACols = kBK / 2; // TMEM columns of one A stage (two fp16 per column)
constexpr int kTileM = 128;     // weight rows per tile
constexpr int kStageA = kTileM * kBK;  // int8 bytes of one weight stage

template <int BN>
struct Cfg {
    static constexpr int kStageB = BN * kBK * 2;  // fp16 activation stage
    static constexpr int kStage = kStageA + kStageB;
    static constexpr int kStages = BN >= 128 ? 6 : 8;
    static constexpr int kXch = 64 * (BN + 1) * 4;  // gate/up exchange buffer
    static constexpr int kAccCols = BN;
    static constexpr int kTmemCols = kNumA * kACols + 2 * kAccCols;
    static constexpr int kTmemAlloc = kTmemCols <= 32 ? 32 : kTmemCols <= 64 ? 64 : kTmemCols <= 128 ? 128
                                      : kTmemCols <= 256 ? 256 : 512;
    // shared memory layout (offsets from a 1024-aligned base)
    static constexpr int kOffStages = 0;
    static constexpr int kOffXch = kStages * kStage;
    static constexpr int kOffBars = kOffXch + kXch;
    static constexpr int kNumBars = 2 * kStages + 2 * kNumA + 4 + 1 + 2;
    static constexpr int kOffTiles = kOffBars + kNumBars * 8;
    static constexpr int kOffMisc = kOffTiles + (kMaxExperts + 1) * 4 * 2;
    static constexpr int kSmem = kOffMisc + 64 + 1024;  // + alignment slack
    static_assert(kStageB % 1024 == 0, "B stage must keep 1024-byte alignment");
    static_assert(kTmemCols <= 512, "TMEM budget");
};

// Tile table of a launch: group g owns tiles [tile_start[g], tile_start[g+1]);
// inside a group, tile = cb * ntb + tb (token blocks fastest, so CTAs running
// at the same time share the weight tile).
struct Tiles {
    const int* tile_start;  // smem, [n_groups + 1]
    const int* row_start;   // smem, [n_groups + 1]
    int n_groups;
    int n_cb;
};

template <int BN>
__device__ __forceinline__ void decode_tile(const Tiles& t, int tile, int& g, int& cb, int& row0,
                                            int& nvalid) {
    int lo = 0, hi = t.n_groups - 1;
    while (lo < hi) {  // last g with tile_start[g] <= tile
        const int mid = (lo + hi + 1) >> 1;
        if (t.tile_start[mid] <= tile) lo = mid; else hi = mid - 1;
    }
    g = lo;
    const int local = tile - t.tile_start[g];
    const int rows = t.row_start[g + 1] - t.row_start[g];
    const int ntb = (rows + BN - 1) / BN;
    cb = local / ntb;
    const int tb = local - cb * ntb;
    row0 = t.row_start[g] + tb * BN;
    nvalid = min(BN, t.row_start[g + 1] - row0);
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
                    *ctl.abort = 1;
                    atomicOr(ctl.error, kErrTimeout);
                    give_up = 1;
                }
            }
            if (__shfl_sync(0xffffffffu, give_up, 0)) return false;
        }
    }
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

__device__ __forceinline__ float silu_f32(float g) {
    return __fdiv_rn(g, __fadd_rn(1.0f, expf(-g)));
}

template <int BN, int EPI>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmap_w,
                        const __grid_constant__ CUtensorMap tmap_b, const GemmArgs args) {
    using C = Cfg<BN>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBars);
    uint64_t* raw_full = bars;
    uint64_t* raw_empty = bars + C::kStages;
    uint64_t* a_full = bars + 2 * C::kStages;
    uint64_t* a_empty = a_full + kNumA;
    uint64_t* acc_full = a_empty + kNumA;
    uint64_t* acc_empty = acc_full + 2;
    uint64_t* teardown = acc_empty + 2;
    uint64_t* xch_full = teardown + 1;   // up-half warps -> gate-half warps
    uint64_t* xch_empty = teardown + 2;  // gate-half warps -> up-half warps
    int* tile_start = reinterpret_cast<int*>(smem + C::kOffTiles);
    int* row_start = tile_start + (kMaxExperts + 1);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 8);
    float* xch = reinterpret_cast<float*>(smem + C::kOffXch);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_groups = args.n_groups;
    const int nkb = args.K / kBK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&raw_full[s], 1);
            mbar_init(&raw_empty[s], 4 + 1);
        }
        for (int a = 0; a < kNumA; ++a) {
            mbar_init(&a_full[a], 4);
            mbar_init(&a_empty[a], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], 4);
        }
        mbar_init(teardown, 1);
        mbar_init(xch_full, 2);
        mbar_init(xch_empty, 2);
        *abort_flag = 0;
        fence_barrier_init();
        tma_prefetch_desc(&tmap_w);
        tma_prefetch_desc(&tmap_b);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, C::kTmemAlloc);
        tmem_relinquish();
    }
    if (warp == 2) {  // tile table: tiles of group g = ceil(rows_g / BN) * n_cb
        int carry = 0;
        for (int base = 0; base < n_groups; base += 32) {
            const int g = base + lane;
            int r0 = 0, r1 = 0;
            if (g < n_groups) {
                r0 = args.offsets ? args.offsets[g] : 0;
                r1 = args.offsets ? args.offsets[g + 1] : args.total_rows;
                row_start[g] = r0;
                if (g == n_groups - 1) row_start[n_groups] = r1;
            }
            int v = (g < n_groups) ? ((r1 - r0 + BN - 1) / BN) * args.n_cb : 0;
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
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int total_tiles = tile_start[n_groups];
    const Tiles tiles{tile_start, row_start, n_groups, args.n_cb};
    const WaitCtl ctl{abort_flag, args.error, args.timeout_ns};

    if (warp == 0) {
        // ---------------------------------------------------------- producer
        if (lane == 0) {
            uint32_t it = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
                int g, cb, row0, nvalid;
                decode_tile<BN>(tiles, tile, g, cb, row0, nvalid);
                int wrow0, wrow1;
                if (EPI == (int)Epi::GateUp) {
                    wrow0 = g * args.w_rows_per_group + cb * 64;
                    wrow1 = wrow0 + args.up_offset;
                } else {
                    wrow0 = g * args.w_rows_per_group + cb * kTileM;
                    wrow1 = wrow0 + 64;
                }
                for (int kb = 0; kb < nkb; ++kb, ++it) {
                    const uint32_t s = it % C::kStages, ph = (it / C::kStages) & 1u;
                    if (!mbar_wait(&raw_empty[s], ph ^ 1u, ctl)) { ok = false; break; }
                    uint8_t* st = smem + C::kOffStages + s * C::kStage;
                    mbar_arrive_expect_tx(&raw_full[s], C::kStage);
                    tma_load_2d(st, &tmap_w, &raw_full[s], kb * kBK, wrow0);
                    tma_load_2d(st + kStageA / 2, &tmap_w, &raw_full[s], kb * kBK, wrow1);
                    tma_load_2d(st + kStageA, &tmap_b, &raw_full[s], kb * kBK, row0);
                }
            }
            // drain: every fill issued must land before the CTA may exit
            for (uint32_t s = 0; s < (uint32_t)C::kStages && s < it; ++s) {
                const uint32_t last = it - 1 - ((it - 1 - s) % C::kStages);
                mbar_wait_drain(&raw_full[s], (last / C::kStages) & 1u);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------ MMA issuer
        if (lane == 0) {
            uint32_t it = 0, acc_it = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
                int g, cb, row0, nvalid;
                decode_tile<BN>(tiles, tile, g, cb, row0, nvalid);
                const uint32_t n_mma = (uint32_t)((nvalid + 15) & ~15);
                const uint32_t idesc = idesc_f16_f32(kTileM, n_mma);
                uint32_t d_col = 0;
                for (int kb = 0; kb < nkb; ++kb, ++it) {
                    if (kb % kChunkKB == 0) {
                        const uint32_t b = acc_it & 1u, ph = (acc_it >> 1) & 1u;
                        if (!mbar_wait(&acc_empty[b], ph ^ 1u, ctl)) { ok = false; break; }
                        d_col = (uint32_t)(kNumA * kACols) + b * (uint32_t)C::kAccCols;
                    }
                    const uint32_t s = it % C::kStages, ph = (it / C::kStages) & 1u;
                    const uint32_t a = it % kNumA, aph = (it / kNumA) & 1u;
                    if (!mbar_wait(&raw_full[s], ph, ctl)) { ok = false; break; }
                    if (!mbar_wait(&a_full[a], aph, ctl)) { ok = false; break; }
                    tc_fence_after();
                    const uint64_t bdesc = smem_desc_sw128(smem_u32(smem + C::kOffStages + s * C::kStage + kStageA));
#pragma unroll
                    for (int ks = 0; ks < kBK / 16; ++ks) {
                        mma_f16_tmem_a(tmem + d_col, tmem + a * kACols + ks * 8, bdesc + (uint64_t)(ks * 2), idesc,
                                       (kb % kChunkKB != 0 || ks != 0) ? 1u : 0u);
                    }
                    mma_commit(&raw_empty[s]);
                    mma_commit(&a_empty[a]);
                    if (kb % kChunkKB == kChunkKB - 1 || kb == nkb - 1) {
                        mma_commit(&acc_full[acc_it & 1u]);
                        ++acc_it;
                    }
                }
            }
            mma_commit(teardown);
            mbar_wait_drain(teardown, 0);
        }
    } else if (warp < 6) {
        // ------------------------------------------------------- converters
        const int q = warp & 3;
        const int row = q * 32 + lane;
        const uint32_t swz = (uint32_t)((row >> 1) & 3);
        uint32_t it = 0;
        bool ok = true;
        for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
            for (int kb = 0; kb < nkb; ++kb, ++it) {
                const uint32_t s = it % C::kStages, ph = (it / C::kStages) & 1u;
                const uint32_t a = it % kNumA, aph = (it / kNumA) & 1u;
                if (!warp_wait(&raw_full[s], ph, ctl)) { ok = false; break; }
                if (!warp_wait(&a_empty[a], aph ^ 1u, ctl)) { ok = false; break; }
                const uint8_t* src = smem + C::kOffStages + s * C::kStage + row * kBK;
                uint32_t v[32];
#pragma unroll
                for (int c = 0; c < 4; ++c) {  // 64-byte swizzle: chunk c sits at c ^ ((row >> 1) & 3)
                    const uint4 w = *reinterpret_cast<const uint4*>(src + ((c ^ swz) << 4));
                    s8x4_to_f16x4(w.x, v[c * 8 + 0], v[c * 8 + 1]);
                    s8x4_to_f16x4(w.y, v[c * 8 + 2], v[c * 8 + 3]);
                    s8x4_to_f16x4(w.z, v[c * 8 + 4], v[c * 8 + 5]);
                    s8x4_to_f16x4(w.w, v[c * 8 + 6], v[c * 8 + 7]);
                }
                tmem_st_32(tmem + ((uint32_t)(q * 32) << 16) + a * kACols, v);
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&a_full[a]);
                    mbar_arrive(&raw_empty[s]);
                }
            }
        }
    } else {
        // --------------------------------------------------------- epilogue
        const int q = warp & 3;
        const int row = q * 32 + lane;  // TMEM lane = weight row of the tile
        const uint32_t lane_addr = (uint32_t)(q * 32) << 16;
        uint32_t acc_it = 0, xch_it = 0;
        bool ok = true;
        const int nchunks = (nkb + kChunkKB - 1) / kChunkKB;
        for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
            int g, cb, row0, nvalid;
            decode_tile<BN>(tiles, tile, g, cb, row0, nvalid);
            int32_t sum[BN];
#pragma unroll
            for (int j = 0; j < BN; ++j) sum[j] = 0;
            for (int ch = 0; ch < nchunks; ++ch) {
                const uint32_t b = acc_it & 1u, ph = (acc_it >> 1) & 1u;
                if (!warp_wait(&acc_full[b], ph, ctl)) { ok = false; break; }
                tc_fence_after();
                const uint32_t col0 = (uint32_t)(kNumA * kACols) + b * (uint32_t)C::kAccCols;
#pragma unroll
                for (int cblk = 0; cblk < BN / 16; ++cblk) {
                    if (cblk * 16 < nvalid) {
                        uint32_t r[16];
                        tmem_ld_16(tmem + lane_addr + col0 + cblk * 16, r);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 16; ++i) sum[cblk * 16 + i] += __float2int_rn(__uint_as_float(r[i]));
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&acc_empty[b]);
                ++acc_it;
            }
            if (!ok) break;

            if (EPI == (int)Epi::GateUp) {
                const int half = row >> 6;  // 0: gate rows, 1: up rows
                const int c = row & 63;
                const int chan = cb * 64 + c;
                const int wrow = half * args.up_offset + chan;
                const float sw = args.w_scale[(size_t)g * args.w_rows_per_group + wrow];
                if (args.acc_out) {
#pragma unroll
                    for (int j = 0; j < BN; ++j)
                        if (j < nvalid) args.acc_out[(size_t)(row0 + j) * args.w_rows_per_group + wrow] = sum[j];
                }
                float* xrow = xch + c * (BN + 1);
                const uint32_t xph = xch_it & 1u;
                ++xch_it;
                if (half && !warp_wait(xch_empty, xph ^ 1u, ctl)) break;
#pragma unroll
                for (int j = 0; j < BN; ++j) {
                    if (j < nvalid) {
                        const float sa = __ldg(args.act_scale + row0 + j);
                        const float v = __fmul_rn(__fmul_rn(__int2float_rn(sum[j]), sa), sw);
                        if (half) xrow[j] = v; else sum[j] = __float_as_int(v);
                    }
                }
                if (half) {
                    __syncwarp();
                    if (lane == 0) mbar_arrive(xch_full);
                } else {
                    if (!warp_wait(xch_full, xph, ctl)) break;
                    float* out = reinterpret_cast<float*>(args.out);
#pragma unroll
                    for (int j = 0; j < BN; ++j) {
                        if (j < nvalid) {
                            const float gv = __int_as_float(sum[j]);
                            const float h = __fmul_rn(silu_f32(gv), xrow[j]);
                            out[(size_t)(row0 + j) * args.ld_out + chan] = h;
                        }
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(xch_empty);
                }
            } else {
                const int chan = cb * kTileM + row;
                const float sw = args.w_scale[(size_t)g * args.w_rows_per_group + chan];
                if (args.acc_out) {
#pragma unroll
                    for (int j = 0; j < BN; ++j)
                        if (j < nvalid) args.acc_out[(size_t)(row0 + j) * args.w_rows_per_group + chan] = sum[j];
                }
#pragma unroll
                for (int j = 0; j < BN; ++j) {
                    if (j < nvalid) {
                        const float sa = __ldg(args.act_scale + row0 + j);
                        const float v = __fmul_rn(__fmul_rn(__int2float_rn(sum[j]), sa), sw);
                        if (EPI == (int)Epi::ScaleF32) {
                            reinterpret_cast<float*>(args.out)[(size_t)(row0 + j) * args.ld_out + chan] = v;
                        } else {
                            reinterpret_cast<__nv_bfloat16*>(args.out)[(size_t)(row0 + j) * args.ld_out + chan] =
                                __float2bfloat16_rn(v);
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

// ------------------------------------------------------------------ host side

using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn get_encode_fn() {
    static EncodeFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeFn>(p);
    });
    return fn;
}

bool make_map_2d(CUtensorMap* map, CUtensorMapDataType dt, int elem_bytes, const void* base, uint64_t inner,
                 uint64_t outer, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swz) {
    EncodeFn enc = get_encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {inner * (uint64_t)elem_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BN, int EPI>
cudaError_t launch_impl(const GemmArgs& args, const void* w, const void* act16, cudaStream_t st) {
    using C = Cfg<BN>;
    auto kern = grouped_gemm_kernel<BN, EPI>;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [&] {
        attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    });
    if (attr_err != cudaSuccess) return attr_err;

    CUtensorMap tw, tb;
    const uint64_t w_rows = (uint64_t)args.n_groups * args.w_rows_per_group;
    if (!make_map_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, w, args.K, w_rows, kBK, 64,
                     CU_TENSOR_MAP_SWIZZLE_64B))
        return cudaErrorInvalidValue;
    if (!make_map_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, act16, args.K, (uint64_t)args.total_rows, kBK, BN,
                     CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;

    const long max_tiles = ((long)(args.total_rows + BN - 1) / BN + args.n_groups) * args.n_cb;
    int grid = num_sms();
    if (max_tiles < grid) grid = (int)max_tiles;
    if (grid < 1) grid = 1;
    kern<<<grid, kThreads, C::kSmem, st>>>(tw, tb, args);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_grouped_gemm(Epi epi, int bn, const GemmArgs& args, const void* w, const void* act16,
                                cudaStream_t st) {
    if (args.total_rows == 0) return cudaSuccess;
    switch (epi) {
        case Epi::GateUp:
            return bn == 128 ? launch_impl<128, 0>(args, w, act16, st) : launch_impl<32, 0>(args, w, act16, st);
        case Epi::ScaleF32:
            return bn == 128 ? launch_impl<128, 1>(args, w, act16, st) : launch_impl<32, 1>(args, w, act16, st);
        case Epi::ScaleBF16:
            return bn == 128 ? launch_impl<128, 2>(args, w, act16, st) : launch_impl<32, 2>(args, w, act16, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace moe

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
// Exactness.  GB300 has no INT8 tcgen05 MMA (kind::i8 does not exist on
// sm_103a), so the product runs on kind::f16: int8 values are exact in fp16
// and products of two of them (|p| <= 2^14) are exact in the fp32
// accumulator.  Every partial sum of a row r is bounded by
// 128 * sum_k |act[r][k]|, so when that L1 norm is at most 2^17 every
// partial sum is an integer of magnitude <= 2^24, exactly representable, and
// the fp32 accumulator holds the exact int32 result in any summation order.
// The quantisation kernels compute the L1 norm of every row and list the
// rows above the bound; this kernel skips them in its tensor-core epilogue
// and recomputes them after its tile loop with exact int32 dot products on
// the CUDA cores.  Typical activations stay far below the bound; the exact
// path only costs time on adversarial inputs.
//
// Operand roles ("swap AB"): A = 128 weight rows per tile, converted from
// int8 to fp16 by converter warps straight into tensor memory; B = a tile of
// BN activation rows, already fp16, loaded by TMA (128-byte swizzle) into
// shared memory; D = 128 x N fp32 accumulator in tensor memory, N = the
// tile's valid rows rounded up to 16.  One stage ring (NS stages of BK along
// K) carries both: the producer refills stage s after the MMAs that read it
// have completed, so the MMA thread waits once and commits once per stage.
// Warp roles of a CTA (320 threads):
//   warp 0      TMA producer (int8 weight tile + fp16 activation tile)
//   warp 1      TMEM allocator and single-thread MMA issuer
//   warps 2-5   converters: int8 weight rows -> fp16 pairs -> tcgen05.st
//   warps 6-9   epilogue: tcgen05.ld, scales, SiLU gate, outputs
// Shared-memory bandwidth (about 128 B/clk per SM, shared by TMA writes,
// tensor-core operand reads and LSU traffic) bounds this 1-SM MMA design:
// every stage moves the activation tile twice (TMA write, tensor-core read)
// and the int8 weight tile twice (TMA write, converter read).  So each tile
// loads only as many activation rows as it has valid rows (rounded up to a
// box of 32, 64, 128 or BN rows), and the accumulators are double-buffered
// so that the epilogue never holds up the MMAs.
// The grid is persistent; tiles are dealt round-robin.  Every wait is
// bounded (see ptx.cuh); a timeout aborts the CTA cleanly.
#include <cstdlib>
#include <mutex>

#include "gemm_common.cuh"

namespace moe {
namespace {

template <int BN_, int BK_, int NS_, int ND_>
struct Cfg {
    static constexpr int BN = BN_;  // activation rows per tile (MMA N)
    static constexpr int BK = BK_;  // K per stage
    static constexpr int NS = NS_;  // stages
    static constexpr int ND = ND_;  // accumulator buffers
    static constexpr int kStageA = kTileM * BK;  // int8 weights
    static constexpr int kStageB = BN * BK * 2;  // fp16 activations
    static constexpr int kStage = kStageA + kStageB;
    static constexpr int kACols = BK / 2;       // TMEM columns of one A stage
    static constexpr int kDCol0 = NS * kACols;  // first accumulator column
    static constexpr int kTmemCols = NS * kACols + ND * BN;
    static constexpr int kTmemAlloc = kTmemCols <= 32 ? 32 : kTmemCols <= 64 ? 64 : kTmemCols <= 128 ? 128
                                      : kTmemCols <= 256 ? 256 : 512;
    static constexpr int kXchStride = 33;
    static constexpr int kXch = kTileM * kXchStride * 4;  // gate/up exchange, 32 columns
    static constexpr int kOffXch = NS * kStage;
    static constexpr int kOffBars = kOffXch + kXch;
    static constexpr int kNumBars = 3 * NS + 2 * ND + 3;  // ..., teardown, epi_bar, stall_bar
    static constexpr int kOffTiles = kOffBars + kNumBars * 8;
    static constexpr int kOffRowInfo = kOffTiles + (kMaxExperts + 1) * 4 * 2;  // [2][BN] scales, [2][BN] flags
    static constexpr int kOffMisc = kOffRowInfo + 2 * BN * 4 * 2;
    static constexpr int kSmem = kOffMisc + 64 + 1024;  // + alignment slack
    static_assert(kStageB % 1024 == 0 && kStageA % 1024 == 0, "stages keep 1024-byte alignment");
    static_assert(kTmemCols <= 512, "TMEM budget");
    static_assert(BK == 64 || BK == 128 || BK == 256, "K per stage");
    // the int8 weight stage: one 64-byte-swizzled [128 x 64] tile for BK = 64,
    // else BK/128 sub-tiles of [128 x 128] with the 128-byte swizzle
    static constexpr int kSubA = BK == 64 ? kStageA : kTileM * 128;
    static constexpr int kNumSubA = BK == 64 ? 1 : BK / 128;
    static_assert(kSmem <= 232448, "shared memory budget");
};

// Each stage costs the MMA thread one wait and one commit, about 255 cycles
// that overlap the MMAs only by their ~45-cycle issue floor, so a stage
// takes max(MMA work, 45 * MMAs + 255) cycles: deep stages (many MMAs per
// wait) keep small tiles from paying the fixed cost many times.
#ifndef MOE_W_BN  // tile shapes: rows per tile, K per stage, stages, accumulators
#define MOE_W_BN 160
#define MOE_W_BK 128
#define MOE_W_NS 3
#define MOE_W_ND 2
#endif
#ifndef MOE_M_BN
#define MOE_M_BN 128
#define MOE_M_BK 128
#define MOE_M_NS 4
#define MOE_M_ND 2
#endif
#ifndef MOE_N_BN
#define MOE_N_BN 32
#define MOE_N_BK 256
#define MOE_N_NS 3
#define MOE_N_ND 2
#endif
using CfgWide = Cfg<MOE_W_BN, MOE_W_BK, MOE_W_NS, MOE_W_ND>;    // hundreds of rows per group
using CfgMid = Cfg<MOE_M_BN, MOE_M_BK, MOE_M_NS, MOE_M_ND>;     // about a hundred rows per group
using CfgNarrow = Cfg<MOE_N_BN, MOE_N_BK, MOE_N_NS, MOE_N_ND>;  // a few rows per group (decode)

template <int BN>
__device__ __forceinline__ void decode_tile(const Tiles& t, int tile, int& g, int& cb, int& row0,
                                            int& nvalid) {
    g = last_le(t.tile_start, t.n_groups, tile);
    const int local = tile - t.tile_start[g];
    const int rows = t.row_start[g + 1] - t.row_start[g];
    const int ntb = (rows + BN - 1) / BN;
    cb = local / ntb;
    const int tb = local - cb * ntb;
    row0 = t.row_start[g] + tb * BN;
    nvalid = min(BN, t.row_start[g + 1] - row0);
}

// Box heights of the activation tensor maps: a tile with nvalid rows loads
// the smallest box that covers them.
template <int BN>
__device__ __forceinline__ int box_index(int nvalid) {
    return nvalid <= 32 ? 0 : nvalid <= 64 ? 1 : nvalid <= 128 ? 2 : 3;
}
template <int BN>
__host__ __device__ constexpr int box_rows(int i) {
    return i == 0 ? (BN < 32 ? BN : 32) : i == 1 ? (BN < 64 ? BN : 64) : i == 2 ? (BN < 128 ? BN : 128) : BN;
}

template <class C, int EPI>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_b0,
                        const __grid_constant__ CUtensorMap tmap_b1, const __grid_constant__ CUtensorMap tmap_b2,
                        const __grid_constant__ CUtensorMap tmap_b3, const GemmArgs args) {
    constexpr int BN = C::BN, BK = C::BK, NS = C::NS, ND = C::ND;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBars);
    uint64_t* full = bars;                // [NS] TMA landed
    uint64_t* a_full = bars + NS;         // [NS] A stage converted into TMEM
    uint64_t* empty = bars + 2 * NS;      // [NS] MMAs of the stage completed
    uint64_t* acc_full = bars + 3 * NS;   // [ND]
    uint64_t* acc_empty = acc_full + ND;  // [ND]
    uint64_t* teardown = acc_empty + ND;
    uint64_t* epi_bar = teardown + 1;
    uint64_t* stall_bar = epi_bar + 1;  // test hook: nothing arrives on it
    int* tile_start = reinterpret_cast<int*>(smem + C::kOffTiles);
    int* row_start = tile_start + (kMaxExperts + 1);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 8);
    float* xch = reinterpret_cast<float*>(smem + C::kOffXch);
    float* row_scale_s = reinterpret_cast<float*>(smem + C::kOffRowInfo);       // [2][BN]
    int* row_flag_s = reinterpret_cast<int*>(smem + C::kOffRowInfo + 2 * BN * 4);  // [2][BN]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_groups = args.n_groups;
    const int nkb = (args.K + BK - 1) / BK;  // a partial last stage reads zeros past K (TMA fill)

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&a_full[s], 4);
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
        // A stage is 2 * kNumSubA weight boxes and BK / 64 activation boxes;
        // lane l issues box l, all in the same warp instruction (a bulk tensor
        // copy costs its issuing thread ~200 cycles).  Lane 0 owns the waits
        // and the arrival.
        constexpr int kBoxes = 2 * C::kNumSubA + BK / 64;
        static_assert(kBoxes <= 32, "boxes per stage");
        constexpr uint32_t kMask = kBoxes == 32 ? 0xffffffffu : ((1u << kBoxes) - 1u);
        if (lane < kBoxes) {
            uint32_t it = 0;
            int ok = 1;
            if (lane == 0) ok = !args.stall || mbar_wait(stall_bar, 0, ctl);  // the test hook's wait runs out
            ok = __shfl_sync(kMask, ok, 0);
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
                const int bi = box_index<BN>(nvalid);
                const CUtensorMap* mb = bi == 0 ? &tmap_b0 : bi == 1 ? &tmap_b1 : bi == 2 ? &tmap_b2 : &tmap_b3;
                const uint32_t stage_bytes = (uint32_t)(C::kStageA + box_rows<BN>(bi) * 128 * (BK / 64));
                // this lane's box: lanes [0, 2 * kNumSubA) rows 0-63 / 64-127 of weight
                // sub-tile l / 2; the rest the activation K halves
                const bool is_w = lane < 2 * C::kNumSubA;
                const int sa = lane >> 1, hh = lane - 2 * C::kNumSubA;
                const CUtensorMap* map = is_w ? &tmap_w : mb;
                const int row = is_w ? ((lane & 1) ? wrow1 : wrow0) : row0;
                const int off = is_w ? sa * C::kSubA + (lane & 1) * (C::kSubA / 2) : C::kStageA + hh * BN * 128;
                const int kx_off = is_w ? sa * (BK == 64 ? 64 : 128) : hh * 64;
                for (int kb = 0; kb < nkb; ++kb, ++it) {
                    const uint32_t s = it % NS, ph = (it / NS) & 1u;
                    if (lane == 0) {
                        ok = mbar_wait(&empty[s], ph ^ 1u, ctl);
                        if (ok) mbar_arrive_expect_tx(&full[s], stage_bytes);
                    }
                    ok = __shfl_sync(kMask, ok, 0);
                    if (!ok) break;
                    tma_load_2d(smem + s * C::kStage + off, map, &full[s], kb * BK + kx_off, row);
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
                decode_tile<BN>(tiles, tile, g, cb, row0, nvalid);
                const uint32_t idesc = idesc_f16_f32(kTileM, (uint32_t)((nvalid + 15) & ~15));
                const uint32_t d = tl % ND;
                if (!mbar_wait(&acc_empty[d], ((tl / ND) & 1u) ^ 1u, ctl)) break;
                tc_fence_after();
                const uint32_t d_col = (uint32_t)C::kDCol0 + d * BN;
                for (int kb = 0; kb < nkb; ++kb, ++it) {
                    const uint32_t s = it % NS, ph = (it / NS) & 1u;
                    // a_full implies full: the converters observed the TMA's
                    // completion before they converted this stage
                    if (!mbar_wait(&a_full[s], ph, ctl)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t b_base = smem_u32(smem + s * C::kStage + C::kStageA);
#pragma unroll
                    for (int ks = 0; ks < BK / 16; ++ks) {
                        const uint64_t bdesc =
                            smem_desc_sw128(b_base + (ks / 4) * BN * 128) + (uint64_t)((ks % 4) * 2);
                        mma_f16_tmem_a(tmem + d_col, tmem + s * C::kACols + ks * 8, bdesc, idesc,
                                       (kb != 0 || ks != 0) ? 1u : 0u);
                    }
                    mma_commit(&empty[s]);
                }
                if (!ok) break;
                mma_commit(&acc_full[d]);
            }
            mma_commit(teardown);
            mbar_wait_drain(teardown, 0);
        }
    } else if (warp < kEpiWarp0) {
        // ------------------------------------------------------- converters
        const int q = warp & 3;
        const int row = q * 32 + lane;
        uint32_t it = 0;
        bool ok = true;
        for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
            for (int kb = 0; kb < nkb; ++kb, ++it) {
                const uint32_t s = it % NS, ph = (it / NS) & 1u;
                // this fill was issued after the MMAs that last read TMEM stage
                // s completed, so full[s] also frees the TMEM stage
                if (!warp_wait(&full[s], ph, ctl)) { ok = false; break; }
                const uint8_t* src = smem + s * C::kStage + row * (BK == 64 ? 64 : 128);
                const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + s * C::kACols;
                if (BK == 64) {  // 64-byte swizzle: chunk c sits at c ^ ((row >> 1) & 3)
                    const uint32_t swz = (uint32_t)((row >> 1) & 3);
                    uint32_t v[32];
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        cvt_chunk(*reinterpret_cast<const uint4*>(src + ((c ^ swz) << 4)), v + c * 8);
                    tmem_st_32(taddr, v);
                } else {  // 128-byte swizzle: chunk c of a sub-tile row sits at c ^ (row & 7)
                    const uint32_t swz = (uint32_t)(row & 7);
#pragma unroll
                    for (int hh = 0; hh < BK / 64; ++hh) {  // 64 K per tcgen05.st
                        const uint8_t* sub = src + (hh >> 1) * C::kSubA;
                        uint32_t v[32];
#pragma unroll
                        for (int c = 0; c < 4; ++c)
                            cvt_chunk(*reinterpret_cast<const uint4*>(sub + ((((hh & 1) * 4 + c) ^ swz) << 4)),
                                      v + c * 8);
                        tmem_st_32(taddr + hh * 32, v);
                    }
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&a_full[s]);
            }
        }
    } else {
        // --------------------------------------------------------- epilogue
        const int q = warp & 3;
        const int ew = warp - kEpiWarp0;  // 0..3
        const int row = q * 32 + lane;    // TMEM lane = weight row of the tile
        const uint32_t lane_addr = (uint32_t)(q * 32) << 16;
        uint32_t tl = 0, eit = 0;
        bool ok = true;
        for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x, ++tl) {
            int g, cb, row0, nvalid;
            decode_tile<BN>(tiles, tile, g, cb, row0, nvalid);
            const uint32_t d = tl % ND;
            int wrow;  // this thread's weight row within the group
            if (EPI == (int)Epi::GateUp) wrow = (row >> 6) * args.up_offset + cb * 64 + (row & 63);
            else wrow = cb * kTileM + row;
            const float sw = __ldg(args.w_scale + (size_t)g * args.w_rows_per_group + wrow);
            // stage the tile's activation scales and exact-path flags in shared
            // memory while the MMAs run (buffer tl & 1: the previous user of it,
            // tile tl - 2, finished before the last epilogue barrier)
            float* sa = row_scale_s + (tl & 1u) * BN;
            int* fl = row_flag_s + (tl & 1u) * BN;
            for (int j = ew * 32 + lane; j < BN; j += 128) {
                const bool in = j < nvalid;
                sa[j] = in ? __ldg(args.act_scale + row0 + j) : 0.f;
                fl[j] = in ? __ldg(args.flags + row0 + j) : 1;
            }
            if (!epi_sync(epi_bar, eit, ctl)) break;
            if (!warp_wait(&acc_full[d], (tl / ND) & 1u, ctl)) break;
            tc_fence_after();
            const uint32_t col0 = (uint32_t)C::kDCol0 + d * BN;
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
                if (args.acc_out) {
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (fl[j0 + j] == 0)
                            args.acc_out[(size_t)(row0 + j0 + j) * args.w_rows_per_group + wrow] =
                                __float2int_rn(__uint_as_float(r[j]));
                }
                if (EPI == (int)Epi::GateUp) {
                    float* xrow = xch + row * C::kXchStride;
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        xrow[j] = dequant(__uint_as_float(r[j]), sa[j0 + j], sw);
                    }
                    if (!epi_sync(epi_bar, eit, ctl)) { ok = false; break; }
                    // warp ew: tokens j0 + 8*ew .. +7; lanes: channels lane, lane + 32
                    float* out = static_cast<float*>(args.out);
#pragma unroll
                    for (int t = 0; t < 8; ++t) {
                        const int j = ew * 8 + t;
                        const int rr = row0 + j0 + j;
                        if (fl[j0 + j] == 0) {
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
                        const int rr = row0 + j0 + j;
                        if (fl[j0 + j] == 0) {
                            const float v = dequant(__uint_as_float(r[j]), sa[j0 + j], sw);
                            if (EPI == (int)Epi::ScaleF32)
                                static_cast<float*>(args.out)[(size_t)rr * args.ld_out + wrow] = v;
                            else
                                static_cast<__nv_bfloat16*>(args.out)[(size_t)rr * args.ld_out + wrow] =
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
    if (!*abort_flag) fallback_rows<EPI>(args, row_start, n_groups);
}

// ------------------------------------------------------------------ host side

template <class C, int EPI>
cudaError_t launch_impl(const GemmArgs& args, cudaStream_t st, bool pdl) {
    auto kern = grouped_gemm_kernel<C, EPI>;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [&] {
        attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    });
    if (attr_err != cudaSuccess) return attr_err;

    CUtensorMap tw, tb[4];
    const uint64_t w_rows = (uint64_t)args.n_groups * args.w_rows_per_group;
    if (!make_tensor_map_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, args.w, args.K, w_rows, C::BK == 64 ? 64 : 128, 64,
                            C::BK == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    for (int i = 0; i < 4; ++i)
        if (!make_tensor_map_2d(&tb[i], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, args.act16, args.K,
                                (uint64_t)args.total_rows, 64, box_rows<C::BN>(i), CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;

    const long max_tiles = ((long)(args.total_rows + C::BN - 1) / C::BN + args.n_groups) * args.n_cb;
    int grid = num_sms();
    if (max_tiles < grid) grid = (int)max_tiles;
    if (grid < 1) grid = 1;
    return launch_kernel(kern, dim3(grid), dim3(kThreads), C::kSmem, st, pdl, tw, tb[0], tb[1], tb[2], tb[3], args);
}

template <int EPI>
cudaError_t launch_epi(GemmShape shape, const GemmArgs& args, cudaStream_t st, bool pdl) {
    switch (shape) {
        case GemmShape::Wide: return launch_impl<CfgWide, EPI>(args, st, pdl);
        case GemmShape::Mid: return launch_impl<CfgMid, EPI>(args, st, pdl);
        case GemmShape::Narrow: return launch_impl<CfgNarrow, EPI>(args, st, pdl);
        case GemmShape::Pair: break;    // dispatched by launch_grouped_gemm
        case GemmShape::Skinny: break;  // dispatched by launch_grouped_gemm
    }
    return cudaErrorInvalidValue;
}

}  // namespace

using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeFn get_encode_fn() {
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

bool make_tensor_map_2d(CUtensorMap* map, CUtensorMapDataType dt, int elem_bytes, const void* base, uint64_t inner,
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

bool make_tensor_map_3d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, const uint64_t (&dims)[3],
                        const uint64_t (&strides)[2], const uint32_t (&box)[3], CUtensorMapSwizzle swz) {
    EncodeFn enc = get_encode_fn();
    if (!enc) return false;
    const cuuint64_t d[3] = {dims[0], dims[1], dims[2]};
    const cuuint64_t st[2] = {strides[0], strides[1]};
    const cuuint32_t b[3] = {box[0], box[1], box[2]};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, dt, 3, const_cast<void*>(base), d, st, b, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

GemmShape choose_gemm_shape(long rows, long groups, long K) {
    (void)K;
    const long per_group = rows / (groups > 0 ? groups : 1);
#ifndef MOE_SKINNY_MAX_ROWS  // weight streaming: a few rows per group
#define MOE_SKINNY_MAX_ROWS 8
#endif
    if (per_group <= MOE_SKINNY_MAX_ROWS) return GemmShape::Skinny;
#ifndef MOE_PAIR_MIN_ROWS  // measured: CTA pairs win from about a hundred rows per group
#define MOE_PAIR_MIN_ROWS 96
#endif
    if (per_group >= MOE_PAIR_MIN_ROWS) return GemmShape::Pair;
    if (per_group >= 48) return GemmShape::Mid;
    return GemmShape::Narrow;
}

cudaError_t launch_grouped_gemm(Epi epi, GemmShape shape, const GemmArgs& args, cudaStream_t st, bool pdl) {
    if (args.total_rows == 0) return cudaSuccess;
    if (shape == GemmShape::Skinny) return launch_grouped_gemm_skinny(epi, args, st, pdl);
    if (shape == GemmShape::Pair) {
        if (pair_gemm_supported(args)) return launch_grouped_gemm_pair(epi, args, st, pdl);
        shape = GemmShape::Wide;
    }
    switch (epi) {
        case Epi::GateUp: return launch_epi<0>(shape, args, st, pdl);
        case Epi::ScaleF32: return launch_epi<1>(shape, args, st, pdl);
        case Epi::ScaleBF16: return launch_epi<2>(shape, args, st, pdl);
    }
    return cudaErrorInvalidValue;
}

}  // namespace moe

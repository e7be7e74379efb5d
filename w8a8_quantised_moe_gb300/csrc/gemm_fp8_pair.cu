// gemm_fp8_pair.cu -- the grouped FP8 (E4M3) GEMM on CTA pairs (tcgen05
// cta_group::2, kind::f8f6f4): the product and epilogues of the FP8 layer
// ("DeepSeek V4 950 FP8 inference on H100" (lpnh.cn), sections 2.1-2.4: E4M3
// operands, fp32 accumulation, per-token x per-channel scales applied to the
// result), for groups with enough rows to fill wide tiles.
//
// At the fp8 rate one CTA's 128 x 256 tile consumes its 16 KB weight stage and
// 32 KB activation stage in about 512 cycles: ~94 bytes per clock per SM, more
// than an SM takes in.  A cluster of two CTAs on neighbouring SMs computes one
// 256 x N tile instead:
//   A  256 weight rows = channel blocks 2p (even CTA) and 2p + 1 (odd CTA),
//      each CTA's 128 rows in its own shared memory;
//   B  N activation rows; rows [0, N/2) in the even CTA's shared memory,
//      [N/2, N) in the odd CTA's;
//   D  each CTA's tensor memory holds its 128 weight rows x N accumulators.
// The even CTA's MMA thread issues M = 256 MMAs that read both CTAs' operands,
// so each SM loads half of B per MMA column: 32 KB a stage for the same work.
//
// Roles per CTA (192 threads): warp 0 loads the stage (its weight rows and its
// half of the activation rows) by TMA; warp 1 allocates the pair's tensor
// memory and, in the even CTA, issues the MMAs, in the odd CTA relays each
// landed stage to the even CTA; warps 2-5 run the epilogue.
// Synchronisation (every wait bounded):
//   full[NS]       this CTA's stage landed (TMA transaction count)
//   pair_full[NS]  even CTA: the odd CTA's stage landed (its relay arrives)
//   empty[NS]      committed by the MMAs of the stage to both CTAs: free
//   acc_full[d]    committed to both CTAs: accumulator d complete
//   acc_empty[d]   even CTA, 8 arrivals (4 epilogue warps x 2 CTAs)
// Shared memory of the odd CTA is read by the even CTA's MMAs and both CTAs
// arrive on each other's barriers, so neither leaves before a final cluster
// barrier that every thread of both CTAs reaches on every path.
#include <mutex>

#include "gemm_common.cuh"

namespace moe {
namespace {

constexpr int kP8BK = 128;       // K bytes (= E4M3 elements) per stage
constexpr int kP8Threads = 192;  // TMA, MMA issuer / relay, 4 epilogue warps
constexpr int kP8Epi0 = 2;       // first epilogue warp
constexpr int kP8ND = 2;         // accumulator buffers

template <int BN_, int NS_>
struct P8Cfg {
    static constexpr int BN = BN_;        // activation rows per pair tile (MMA N, at most)
    static constexpr int NS = NS_;        // stages
    static constexpr int kHalf = BN / 2;  // activation rows per CTA
    static constexpr int kStageA = kTileM * kP8BK;  // [128 x 128] E4M3, two 64-row boxes
    static constexpr int kStageB = kHalf * kP8BK;   // [BN/2 x 128] E4M3
    static constexpr int kStage = kStageA + kStageB;
    static constexpr int kTmemCols = kP8ND * BN;
    static constexpr int kTmemAlloc = 512;  // a power of two; the pair takes all of it
    static constexpr int kXchStride = 33;
    static constexpr int kXch = kTileM * kXchStride * 4;  // GateUp: gate/up exchange
    static constexpr int kStoreBuf = 32 * kTileM * 4;     // ScaleF32: [32 rows][128 channels] staging
    static constexpr int kXchRegion = kXch > 2 * kStoreBuf ? kXch : 2 * kStoreBuf;
    static constexpr int kOffXch = NS * kStage;
    static constexpr int kOffBars = kOffXch + kXchRegion;
    static constexpr int kNumBars = 3 * NS + 2 * kP8ND + 3;  // ..., teardown, epi_bar, stall_bar
    static constexpr int kOffTiles = kOffBars + kNumBars * 8;
    static constexpr int kOffRowInfo = kOffTiles + (kMaxExperts + 1) * 4 * 2;  // [2][BN] activation scales
    static constexpr int kOffMisc = kOffRowInfo + 2 * BN * 4;
    static constexpr int kSmem = kOffMisc + 64 + 1024;
    static_assert(kStageA % 1024 == 0 && kStageB % 1024 == 0, "stages keep 1024-byte alignment");
    static_assert(BN % 32 == 0 && BN <= 256, "pair tile width");
    static_assert(kTmemCols <= kTmemAlloc, "TMEM budget");
    static_assert(kSmem <= 232448, "shared memory budget");
};
// Measured on the prefill layer (GEMM1 / GEMM2 us): 256-row tiles with 5
// stages 271 / 143; 4 stages 277 / 150; 192-row tiles with 6 stages 261 / 148;
// 128-row tiles with 7 stages 313 / 179.
#ifndef MOE_P8_NS
#define MOE_P8_NS 5
#endif
#ifndef MOE_P8_BN
#define MOE_P8_BN 256
#endif
using P8Wide = P8Cfg<MOE_P8_BN, MOE_P8_NS>;

// One tcgen05 MMA on the CTA pair, kind::f8f6f4, both operands from shared
// memory (each CTA's half at the same offset): D[256 x N] (+)= A * B^T, K = 32.
__device__ __forceinline__ void mma_f8_smem_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                                 uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Instruction descriptor of kind::f8f6f4 with E4M3 A and B (format 0), fp32 D.
__host__ __device__ constexpr uint32_t idesc_e4m3_pair(uint32_t M, uint32_t N) {
    return (1u << 4)            // D format: f32
           | (0u << 7)          // A format: E4M3
           | (0u << 10)         // B format: E4M3
           | ((N >> 3) << 17)   // N / 8
           | ((M >> 4) << 24);  // M / 16
}

// Pair tile -> group, channel-block pair, first row, valid rows (token blocks
// fastest inside a group).
template <int BN>
__device__ __forceinline__ void p8_decode_tile(const Tiles& t, int tile, int& g, int& cp, int& row0, int& nvalid) {
    g = last_le(t.tile_start, t.n_groups, tile);
    const int local = tile - t.tile_start[g];
    const int rows = t.row_start[g + 1] - t.row_start[g];
    const int ntb = (rows + BN - 1) / BN;
    cp = local / ntb;
    const int tb = local - cp * ntb;
    row0 = t.row_start[g] + tb * BN;
    nvalid = min(BN, t.row_start[g + 1] - row0);
}

// Box heights of the per-CTA activation maps: the smallest that covers a
// CTA's rows.
template <int HALF>
__host__ __device__ constexpr int p8_box_rows(int i) {
    return i == 0 ? (HALF < 16 ? HALF : 16) : i == 1 ? (HALF < 32 ? HALF : 32) : i == 2 ? (HALF < 64 ? HALF : 64)
                                                                                       : HALF;
}
__device__ __forceinline__ int p8_box_index(int h) { return h <= 16 ? 0 : h <= 32 ? 1 : h <= 64 ? 2 : 3; }

template <class C, int EPI>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kP8Threads, 1)
    grouped_gemm_fp8_pair_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_b0,
                                 const __grid_constant__ CUtensorMap tmap_b1,
                                 const __grid_constant__ CUtensorMap tmap_b2,
                                 const __grid_constant__ CUtensorMap tmap_b3,
                                 const __grid_constant__ CUtensorMap tmap_out, const GemmArgs args) {
    constexpr int BN = C::BN, NS = C::NS;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBars);
    uint64_t* full = bars;                    // [NS] this CTA's stage landed
    uint64_t* pair_full = full + NS;          // [NS] even CTA: the odd CTA's stage landed
    uint64_t* empty = pair_full + NS;         // [NS] the stage's MMAs completed (both CTAs)
    uint64_t* acc_full = empty + NS;          // [ND]
    uint64_t* acc_empty = acc_full + kP8ND;   // [ND], used in the even CTA
    uint64_t* teardown = acc_empty + kP8ND;
    uint64_t* epi_bar = teardown + 1;
    uint64_t* stall_bar = epi_bar + 1;  // test hook: nothing arrives on it
    int* tile_start = reinterpret_cast<int*>(smem + C::kOffTiles);
    int* row_start = tile_start + (kMaxExperts + 1);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 8);
    float* xch = reinterpret_cast<float*>(smem + C::kOffXch);
    float* row_scale_s = reinterpret_cast<float*>(smem + C::kOffRowInfo);  // [2][BN]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();  // 0: issues the MMAs
    const int cluster = blockIdx.x >> 1, n_clusters = gridDim.x >> 1;
    const int n_groups = args.n_groups;
    const int n_cp = args.n_cb >> 1;
    const int nkb = args.K / kP8BK;  // K is a multiple of 128

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&pair_full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int d = 0; d < kP8ND; ++d) {
            mbar_init(&acc_full[d], 1);
            mbar_init(&acc_empty[d], 8);
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
        if (EPI != (int)Epi::GateUp) tma_prefetch_desc(&tmap_out);
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_slot, C::kTmemAlloc);
        tmem_relinquish_pair();
    }
    pdl_wait();  // the previous kernel's outputs (offsets, codes, scales) are visible from here
    pdl_trigger();
    if (warp == 2) {  // tile table: pair tiles of group g = ceil(rows_g / BN) * n_cp
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
            const int v = (g < n_groups) ? ((r1 - r0 + BN - 1) / BN) * n_cp : 0;
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
    cluster_sync_all();  // both CTAs' barriers are initialised before anyone arrives remotely
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int total_tiles = tile_start[n_groups];
    const Tiles tiles{tile_start, row_start, n_groups};
    const WaitCtl ctl{abort_flag, args.error, args.timeout_ns,
                      cluster_addr(const_cast<const int*>(abort_flag), rank ^ 1u)};

    if (warp == 0) {
        // ------------------------------------------------ stage TMA (both CTAs)
        // A stage is three boxes (weight rows 0-63 and 64-127, activation
        // rows); lanes 0-2 issue one each in the same warp instruction, since
        // a bulk tensor copy costs its issuing thread ~200 cycles.  Lane 0
        // owns the waits and the arrival.
        if (lane < 3) {
            uint32_t it = 0;
            // the test hook stalls the even CTA only (the odd one is aborted through its peer flag)
            int ok = 1;
            if (lane == 0) ok = !(args.stall && rank == 0) || mbar_wait(stall_bar, 0, ctl);
            ok = __shfl_sync(0x7u, ok, 0);
            for (int tile = cluster; ok && tile < total_tiles; tile += n_clusters) {
                int g, cp, row0, nvalid;
                p8_decode_tile<BN>(tiles, tile, g, cp, row0, nvalid);
                const int cb = 2 * cp + (int)rank;
                int wrow0, wrow1;  // this CTA's weight rows 0-63 and 64-127
                if (EPI == (int)Epi::GateUp) {
                    wrow0 = g * args.w_rows_per_group + cb * 64;
                    wrow1 = wrow0 + args.up_offset;
                } else {
                    wrow0 = g * args.w_rows_per_group + cb * kTileM;
                    wrow1 = wrow0 + 64;
                }
                const int half = ((nvalid + 15) & ~15) >> 1;  // activation rows per CTA
                const int bi = p8_box_index(half);
                const CUtensorMap* mb = bi == 0 ? &tmap_b0 : bi == 1 ? &tmap_b1 : bi == 2 ? &tmap_b2 : &tmap_b3;
                const int brow = row0 + (int)rank * half;
                const uint32_t bytes = (uint32_t)(C::kStageA + p8_box_rows<C::kHalf>(bi) * kP8BK);
                // this lane's box: its tensor map, row and offset in the stage
                const CUtensorMap* map = lane == 2 ? mb : &tmap_w;
                const int row = lane == 0 ? wrow0 : lane == 1 ? wrow1 : brow;
                const int off = lane == 0 ? 0 : lane == 1 ? C::kStageA / 2 : C::kStageA;
                for (int kb = 0; kb < nkb; ++kb, ++it) {
                    const uint32_t s = it % NS, ph = (it / NS) & 1u;
                    // stage s is free once the MMAs of stage it - NS completed
                    if (lane == 0) {
                        ok = mbar_wait_cluster(&empty[s], ph ^ 1u, ctl);
                        if (ok) mbar_arrive_expect_tx(&full[s], bytes);
                    }
                    ok = __shfl_sync(0x7u, ok, 0);
                    if (!ok) break;
                    tma_load_2d(smem + s * C::kStage + off, map, &full[s], kb * kP8BK, row);
                }
            }
            // drain: every fill issued must land before the CTA may exit
            if (lane == 0)
                for (uint32_t s = 0; s < (uint32_t)NS && s < it; ++s) {
                    const uint32_t last = it - 1 - ((it - 1 - s) % NS);
                    mbar_wait_drain(&full[s], (last / NS) & 1u);
                }
        }
    } else if (warp == 1 && rank != 0) {
        // ------------------------------------------- relay (odd CTA)
        if (lane == 0) {
            const uint32_t pair_full_leader = cluster_addr(&pair_full[0], 0);
            uint32_t it = 0;
            bool ok = true;
            for (int tile = cluster; ok && tile < total_tiles; tile += n_clusters)
                for (int kb = 0; kb < nkb; ++kb, ++it) {
                    const uint32_t s = it % NS, ph = (it / NS) & 1u;
                    if (!mbar_wait(&full[s], ph, ctl)) { ok = false; break; }
                    mbar_arrive_cluster(pair_full_leader + s * 8);
                }
        }
    } else if (warp == 1) {
        // ------------------------------------------ MMA issuer (even CTA)
        if (lane == 0) {
            uint32_t it = 0, tl = 0;
            bool ok = true;
            for (int tile = cluster; ok && tile < total_tiles; tile += n_clusters, ++tl) {
                int g, cp, row0, nvalid;
                p8_decode_tile<BN>(tiles, tile, g, cp, row0, nvalid);
                const uint32_t idesc = idesc_e4m3_pair(2 * kTileM, (uint32_t)((nvalid + 15) & ~15));
                const uint32_t d = tl % kP8ND;
                if (!mbar_wait_cluster(&acc_empty[d], ((tl / kP8ND) & 1u) ^ 1u, ctl)) break;
                tc_fence_after();
                const uint32_t d_col = d * BN;
                for (int kb = 0; kb < nkb; ++kb, ++it) {
                    const uint32_t s = it % NS, ph = (it / NS) & 1u;
                    if (!mbar_wait(&full[s], ph, ctl)) { ok = false; break; }
                    if (!mbar_wait_cluster(&pair_full[s], ph, ctl)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t a_base = smem_u32(smem + s * C::kStage);
                    const uint32_t b_base = a_base + C::kStageA;
#pragma unroll
                    for (int ks = 0; ks < kP8BK / 32; ++ks)  // 32 bytes of K per MMA
                        mma_f8_smem_pair(tmem + d_col, smem_desc_sw128(a_base) + (uint64_t)(ks * 2),
                                         smem_desc_sw128(b_base) + (uint64_t)(ks * 2), idesc,
                                         (kb != 0 || ks != 0) ? 1u : 0u);
                    mma_commit_pair(&empty[s], 3);
                }
                if (!ok) break;
                mma_commit_pair(&acc_full[d], 3);
            }
            mma_commit_pair(teardown, 1);
            mbar_wait_drain(teardown, 0);
        }
    } else {
        // --------------------------------------------------------- epilogue
        const int q = warp & 3;
        const int ew = warp - kP8Epi0;  // 0..3
        const int row = q * 32 + lane;  // TMEM lane = weight row of this CTA's channel block
        const uint32_t lane_addr = (uint32_t)(q * 32) << 16;
        const uint32_t acc_empty_leader = cluster_addr(&acc_empty[0], 0);
        const bool store_issuer = (ew == 0 && lane == 0);
        uint32_t tl = 0, eit = 0, n_store = 0;
        bool ok = true;
        for (int tile = cluster; ok && tile < total_tiles; tile += n_clusters, ++tl) {
            int g, cp, row0, nvalid;
            p8_decode_tile<BN>(tiles, tile, g, cp, row0, nvalid);
            const int cb = 2 * cp + (int)rank;
            const uint32_t d = tl % kP8ND;
            int wrow;  // this thread's weight row within the group
            if (EPI == (int)Epi::GateUp) wrow = (row >> 6) * args.up_offset + cb * 64 + (row & 63);
            else wrow = cb * kTileM + row;
            const float sw = __ldg(args.w_scale + (size_t)g * args.w_rows_per_group + wrow);
            // the tile's activation scales, staged while the MMAs run (buffer
            // tl & 1: its previous user, tile tl - 2, passed the last barrier)
            float* sa = row_scale_s + (tl & 1u) * BN;
            for (int jj = ew * 32 + lane; jj < BN; jj += 128) sa[jj] = jj < nvalid ? __ldg(args.act_scale + row0 + jj) : 0.f;
            if (!epi_sync(epi_bar, eit, ctl)) break;
            if (!warp_wait_cluster(&acc_full[d], (tl / kP8ND) & 1u, ctl)) break;
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
                    if (lane == 0) mbar_arrive_cluster(acc_empty_leader + d * 8);
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
                } else if (j0 + 32 <= nvalid) {
                    // 32 valid rows: stage the [32 rows x 128 channels] block in
                    // shared memory and write it with one TMA store
                    uint8_t* buf = reinterpret_cast<uint8_t*>(xch) + (n_store & 1u) * C::kStoreBuf;
                    if (store_issuer) tma_store_wait_read<1>();  // the store that last read buf is done
                    if (!epi_sync(epi_bar, eit, ctl)) { ok = false; break; }
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        reinterpret_cast<float*>(buf)[j * kTileM + row] =
                            dequant(__uint_as_float(r[j]), sa[j0 + j], sw);
                    fence_proxy_async_smem();
                    if (!epi_sync(epi_bar, eit, ctl)) { ok = false; break; }
                    if (store_issuer) {
                        tma_store_2d(&tmap_out, buf, cb * kTileM, row0 + j0);
                        tma_store_commit();
                    }
                    ++n_store;
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

    if (EPI != (int)Epi::GateUp && warp == kP8Epi0 && lane == 0) tma_store_wait_all();
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // the pair's MMAs, TMA fills and remote arrivals are all done
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc_pair(tmem, C::kTmemAlloc);
    }
}

int max_fp8_pair_clusters(const void* kern, int smem) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(2 * (unsigned)num_sms(), 1, 1);
    cfg.blockDim = dim3(kP8Threads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n < 1) {
        cudaGetLastError();
        n = num_sms() / 2;
    }
    return n;
}

template <class C, int EPI>
cudaError_t launch_fp8_pair_impl(const GemmArgs& args, cudaStream_t st, bool pdl) {
    auto kern = grouped_gemm_fp8_pair_kernel<C, EPI>;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    static int clusters = 0;
    std::call_once(once, [&] {
        attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
        if (attr_err == cudaSuccess) clusters = max_fp8_pair_clusters(reinterpret_cast<const void*>(kern), C::kSmem);
    });
    if (attr_err != cudaSuccess) return attr_err;
    CUtensorMap tw, tb[4];
    const uint64_t w_rows = (uint64_t)args.n_groups * args.w_rows_per_group;
    if (!make_tensor_map_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, args.w, args.K, w_rows, kP8BK, 64,
                            CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    for (int i = 0; i < 4; ++i)
        if (!make_tensor_map_2d(&tb[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, args.act8, args.K,
                                (uint64_t)args.total_rows, kP8BK, p8_box_rows<C::kHalf>(i),
                                CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
    CUtensorMap tout = tw;  // unused by GateUp
    if (EPI == (int)Epi::ScaleF32 &&
        !make_tensor_map_2d(&tout, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, args.out, args.ld_out,
                            (uint64_t)args.total_rows, kTileM, 32, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    const long max_tiles = ((long)(args.total_rows + C::BN - 1) / C::BN + args.n_groups) * (args.n_cb / 2);
    long n = clusters;
    if (max_tiles < n) n = max_tiles;
    if (n < 1) n = 1;
    return launch_kernel(kern, dim3((unsigned)(2 * n)), dim3(kP8Threads), C::kSmem, st, pdl, tw, tb[0], tb[1], tb[2],
                         tb[3], tout, args);
}

}  // namespace

bool fp8_pair_gemm_supported(const GemmArgs& args) { return args.n_cb >= 2 && (args.n_cb & 1) == 0; }

cudaError_t launch_grouped_gemm_fp8_pair(Epi epi, const GemmArgs& args, cudaStream_t st, bool pdl) {
    if (args.total_rows == 0) return cudaSuccess;
    if (args.act8 == nullptr || args.K % kP8BK != 0 || !fp8_pair_gemm_supported(args)) return cudaErrorInvalidValue;
    switch (epi) {
        case Epi::GateUp: return launch_fp8_pair_impl<P8Wide, 0>(args, st, pdl);
        case Epi::ScaleF32: return launch_fp8_pair_impl<P8Wide, 1>(args, st, pdl);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace moe

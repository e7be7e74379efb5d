// gemm_pair.cu -- the exact INT8 grouped GEMM on CTA pairs (tcgen05
// cta_group::2): the same product and epilogues as gemm.cu ("W8A8
// quantisation of MiniMax-M3 on K100AI" (mhpn.cn), section 2.1; exactness
// certificate and exact CUDA-core path as described there), for groups with
// enough rows to fill wide tiles.
//
// A cluster of two CTAs on neighbouring SMs computes one 256 x N tile:
//   A  256 weight rows = channel blocks 2p (even CTA) and 2p + 1 (odd CTA);
//      each CTA converts its 128 int8 rows to fp16 in its own tensor memory.
//   B  N activation rows of one group (N = valid rows rounded up to 16);
//      rows [0, N/2) sit in the even CTA's shared memory, [N/2, N) in the odd
//      CTA's, each loaded by that CTA's TMA producer.
//   D  each CTA's tensor memory holds its 128 weight rows x N accumulators.
// The even CTA's MMA thread issues M = 256 MMAs that read both CTAs' operands.
// Against one CTA per tile this halves what each SM loads and keeps in
// shared memory per MMA column (one half of B instead of all of it), and
// every MMA instruction does twice the work for the same issue cost, which
// matters because the issuing thread shares its SM sub-partition with a
// converter and an epilogue warp.
//
// Roles per CTA (384 threads; 512 with a second converter group): warp 0
// loads the int8 weight rows (ring of NQ stages, deep: weights stream from HBM
// once), warp 10 loads this CTA's half of the activation rows (ring of NB
// stages: they are re-read from L2 by every channel-block pair), one bulk
// copy a stage each; warp 1 allocates TMEM and in the even CTA issues the
// MMAs with warp 11 (alternate stages); warps 2-5 convert (warps 12-15 too,
// each group half of every stage's K columns, for the scale epilogues);
// warps 6-9 run the epilogue.
// Synchronisation (every wait bounded; see ptx.cuh):
//   q_full/q_empty[NQ]  int8 stage landed / read by the converter warps
//   b_full[NB]          this CTA's activation half landed
//   done[NB]            committed by the even CTA's MMAs of a stage to both
//                       CTAs: its activation slot, and the A slot (it % NA) it
//                       read, are free again
//   a_ready[j]          even CTA, 8 arrivals per converter group (4 warps x 2 CTAs):
//                       tensor-memory A slot j holds the stage's weights in both
//                       CTAs.  Group 0's converters waited on their CTA's
//                       b_full first, so this also covers both halves of B.
//   acc_full[d]         per CTA, committed to both: accumulator d complete
//   acc_empty[d]        even CTA, 8 arrivals (4 epilogue warps x 2 CTAs)
// Shared memory of the odd CTA is read by the even CTA's MMAs, and both CTAs
// arrive on each other's barriers, so neither leaves before a final cluster
// barrier that every thread of both CTAs reaches on every path.
//
// The scale epilogues write a block of 32 rows x 128 channels through shared
// memory and one TMA store when all 32 rows are valid and none is on the
// exact path (measured: the second expert GEMM of the prefill workload drops
// from 0.28 to 0.20 ms, as per-element stores had kept the accumulators
// busy); other blocks, and GateUp, use per-element stores.
#include <mutex>

#include "gemm_common.cuh"

namespace moe {
namespace {

constexpr int kPairBK = 128;  // K per stage
#ifndef MOE_P_EARLY
#define MOE_P_EARLY 1
#endif
constexpr bool kEarlyTests = MOE_P_EARLY != 0;  // converters test the next barriers early
#ifndef MOE_P_READ_AHEAD
#define MOE_P_READ_AHEAD 1
#endif
constexpr bool kReadAhead = kEarlyTests && MOE_P_READ_AHEAD != 0;  // converters read the next stage early
#ifndef MOE_P_SLOT_LATE
#define MOE_P_SLOT_LATE 1
#endif
constexpr bool kSlotLate = MOE_P_SLOT_LATE != 0;  // the A-slot wait just before the first store

#ifndef MOE_P_ND
#define MOE_P_ND 2
#endif
constexpr int kPairND = MOE_P_ND;  // accumulator buffers

// MMA-issuing threads in the even CTA.  Measured: two beat one by 8-10% on
// the expert GEMMs.  At most two: an issuer may wait on a_ready[j] for stage
// i only while the phase of stage i - NA is complete (a parity wait cannot
// tell phases two apart).  With two issuers that holds for NA >= 2: an issuer
// has passed the wait of its previous stage, at most two stages back, or, on a
// tile's first stage, the tile_go barrier, which follows the other issuer's
// wait on stage i - 1.  A third issuer can be three stages past its previous
// wait, where two A slots no longer order it.
#ifndef MOE_P_ISSUERS
#define MOE_P_ISSUERS 2
#endif
constexpr int kIssuers = MOE_P_ISSUERS;
static_assert(kIssuers == 1 || kIssuers == 2, "one or two MMA issuers");
// Converter groups: each of the G groups of four warps (one per TMEM lane
// quadrant) converts 128 / G of the K columns of every stage, so that a
// stage's conversion takes less time.  Measured per-stage timestamps put a
// stage near 1100 cycles of which the conversion is ~250-400; the gain
// depends on the tile mix: with two groups the down GEMM of the prefill layer
// drops from 191 to 185 us and the 256-expert layer's gate/up GEMM from 2.00
// to 1.96 ms, while the prefill gate/up GEMM rises from 345 to 354 us.  So
// the gate/up GEMM runs one group, the scale epilogues two.
// + warp 10, the activation producer, warp 11, the second MMA issuer, and
// warps 12-15, the second converter group (if any)
constexpr int kPairBWarp = 10;
constexpr int kPairMma2Warp = 11;
constexpr int kPairConv1Warp0 = 12;
__host__ __device__ constexpr int pair_threads(int conv_groups) { return kThreads + 32 * kIssuers + 128 * (conv_groups - 1); }

template <int BN_, int NQ_, int NB_, int NA_, bool kStore_, int CONV_>
struct PairCfg {
    static constexpr int kConv = CONV_;                 // converter groups
    static constexpr int kThreadsPerCta = pair_threads(CONV_);
    static_assert(CONV_ == 1 || (CONV_ == 2 && kIssuers == 2 && kThreadsPerCta == 512), "warp layout");
    static constexpr int BN = BN_;        // activation rows per pair tile (MMA N, at most)
    static constexpr int NQ = NQ_;        // int8 weight stages (deep: weights stream from HBM)
    static constexpr int NB = NB_;        // activation stages
    static constexpr int NA = NA_;        // tensor-memory A slots (at most NB)
    static constexpr int kHalf = BN / 2;  // activation rows per CTA
    static constexpr int kQStage = kTileM * kPairBK;    // int8 weights, [128 x 128] 128-byte swizzle
    static constexpr int kSubB = kHalf * 128;           // one 64-wide K half of the fp16 rows
    static constexpr int kBStage = 2 * kSubB;
    static constexpr int kACols = kPairBK / 2;          // TMEM columns of one A slot
    static constexpr int kDCol0 = NA * kACols;          // first accumulator column
    static constexpr int kTmemCols = kDCol0 + kPairND * BN;
    static constexpr int kXchStride = 33;
    static constexpr int kXch = kTileM * kXchStride * 4;  // GateUp: gate/up exchange
    static constexpr int kStoreBuf = 32 * kTileM * 4;     // scale epilogues: [32 rows][128 channels] staging
    static constexpr int kOffQ = 0;
    static constexpr int kOffB = kOffQ + NQ * kQStage;
    static constexpr int kOffXch = kOffB + NB * kBStage;
    // GateUp exchanges g and u; the scale epilogues stage two TMA-store blocks
    static constexpr bool kStore = kStore_;
    static constexpr int kXchRegion = kStore ? (kXch > 2 * kStoreBuf ? kXch : 2 * kStoreBuf) : kXch;
    static constexpr int kOffBars = kOffXch + kXchRegion;
    // q_full, q_empty, b_full, done, a_ready, acc_full, acc_empty, tile_go,
    // one teardown barrier per issuer, epi_bar, stall_bar
    static constexpr int kNumBars = 2 * NQ + 2 * NB + NA + 3 * kPairND + kIssuers + 2;
    static constexpr int kOffTiles = kOffBars + kNumBars * 8;
    static constexpr int kOffRowInfo = kOffTiles + (kMaxExperts + 1) * 4 * 2;
    static constexpr int kOffMisc = kOffRowInfo + 2 * BN * 4 * 2;
    static constexpr int kSmem = kOffMisc + 64 + 1024;
    static_assert(kSubB % 1024 == 0 && kQStage % 1024 == 0, "stages keep 1024-byte alignment");
    static_assert(BN % 32 == 0 && BN <= 256, "pair tile width");
    static_assert(kTmemCols <= 512, "TMEM budget");
    // a converter learns that A slot (it % NA) is free from done[] of stage
    // it - NA, whose barrier cannot have moved on to a later phase when NB >= NA
    static_assert(NB >= NA, "activation ring and A slots");
    static_assert(NA >= kIssuers, "two issuers need two A slots");
    static_assert(kSmem <= 232448, "shared memory budget");
};

// Tensor memory holds the A slots and two accumulators (192-wide tiles with
// two A slots).  Weights and activations have separate rings (weights stream
// from HBM once, activations are re-read from L2 by every channel-block
// pair).  Measured: four activation stages matter (two or three are clearly
// slower).  The weight ring is as deep as shared memory allows: a weight
// stage lands ~3500 cycles after its TMA is issued, about three stages.
#ifndef MOE_P_BN  // pair tile width, A slots
#define MOE_P_BN 192
#define MOE_P_NA 2
#endif
#ifndef MOE_P_NB_GU  // activation stages: GateUp, scale epilogues
#define MOE_P_NB_GU 4
#define MOE_P_NB_SC 4
#endif
#ifndef MOE_P_NQ_GU  // int8 weight stages: GateUp (no store staging), scale epilogues
#define MOE_P_NQ_GU 6
#define MOE_P_NQ_SC 5
#endif
#ifndef MOE_P_CONV_GU  // converter groups: GateUp, scale epilogues
#define MOE_P_CONV_GU 1
#define MOE_P_CONV_SC 2
#endif
using CfgPairGU = PairCfg<MOE_P_BN, MOE_P_NQ_GU, MOE_P_NB_GU, MOE_P_NA, false, MOE_P_CONV_GU>;
using CfgPairSc = PairCfg<MOE_P_BN, MOE_P_NQ_SC, MOE_P_NB_SC, MOE_P_NA, true, MOE_P_CONV_SC>;

// Box heights of the per-CTA activation tensor maps: a CTA of a tile with
// half-width h loads the smallest box that covers h rows.
template <int HALF>
__host__ __device__ constexpr int pair_box_rows(int i) {
    return i == 0 ? (HALF < 16 ? HALF : 16) : i == 1 ? (HALF < 32 ? HALF : 32) : i == 2 ? (HALF < 64 ? HALF : 64)
                                                                                       : HALF;
}
__device__ __forceinline__ int pair_box_index(int h) { return h <= 16 ? 0 : h <= 32 ? 1 : h <= 64 ? 2 : 3; }

// Pair tile -> group, channel-block pair, first row, valid rows.  Inside a
// group, tile = cp * ntb + tb (token blocks fastest).
template <int BN>
__device__ __forceinline__ void decode_pair_tile(const Tiles& t, int tile, int& g, int& cp, int& row0,
                                                 int& nvalid) {
    g = last_le(t.tile_start, t.n_groups, tile);
    const int local = tile - t.tile_start[g];
    const int rows = t.row_start[g + 1] - t.row_start[g];
    const int ntb = (rows + BN - 1) / BN;
    cp = local / ntb;
    const int tb = local - cp * ntb;
    row0 = t.row_start[g] + tb * BN;
    nvalid = min(BN, t.row_start[g + 1] - row0);
}

template <class C, int EPI>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(C::kThreadsPerCta, 1)
    grouped_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_b0,
                             const __grid_constant__ CUtensorMap tmap_b1, const __grid_constant__ CUtensorMap tmap_b2,
                             const __grid_constant__ CUtensorMap tmap_b3, const __grid_constant__ CUtensorMap tmap_out,
                             const GemmArgs args) {
    constexpr int BN = C::BN, NQ = C::NQ, NB = C::NB;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBars);
    uint64_t* q_full = bars;                   // [NQ] int8 weight stage landed
    uint64_t* q_empty = q_full + NQ;           // [NQ] read by the 4 converter warps
    uint64_t* b_full = q_empty + NQ;           // [NB] activation half landed
    uint64_t* done = b_full + NB;              // [NB] MMAs of the stage done (both CTAs)
    uint64_t* a_ready = done + NB;             // [NA], used in the even CTA
    uint64_t* acc_full = a_ready + C::NA;    // [ND]
    uint64_t* acc_empty = acc_full + kPairND;  // [ND], used in the even CTA
    uint64_t* tile_go = acc_empty + kPairND;  // [ND], even CTA: the tile's overwriting MMAs are issued
    uint64_t* teardown = tile_go + kPairND;   // [kIssuers], one per issuer
    uint64_t* epi_bar = teardown + kIssuers;
    uint64_t* stall_bar = epi_bar + 1;  // the last barrier of the block; test hook: nothing arrives on it
    int* tile_start = reinterpret_cast<int*>(smem + C::kOffTiles);
    int* row_start = tile_start + (kMaxExperts + 1);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 8);
    float* xch = reinterpret_cast<float*>(smem + C::kOffXch);
    float* row_scale_s = reinterpret_cast<float*>(smem + C::kOffRowInfo);          // [2][BN]
    int* row_flag_s = reinterpret_cast<int*>(smem + C::kOffRowInfo + 2 * BN * 4);  // [2][BN]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();  // 0: issues the MMAs
    const int cluster = blockIdx.x >> 1, n_clusters = gridDim.x >> 1;
    const int n_groups = args.n_groups;
    const int n_cp = args.n_cb >> 1;
    const int nkb = (args.K + kPairBK - 1) / kPairBK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NQ; ++s) {
            mbar_init(&q_full[s], 1);
            mbar_init(&q_empty[s], 4 * C::kConv);
        }
        for (int s = 0; s < NB; ++s) {
            mbar_init(&b_full[s], 1);
            mbar_init(&done[s], 1);
        }
        for (int j = 0; j < C::NA; ++j) mbar_init(&a_ready[j], 8 * C::kConv);
        for (int d = 0; d < kPairND; ++d) {
            mbar_init(&acc_full[d], kIssuers);
            mbar_init(&tile_go[d], 1);
            mbar_init(&acc_empty[d], 8);
        }
        for (int r = 0; r < kIssuers; ++r) mbar_init(&teardown[r], 1);
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
        tmem_alloc_pair(tmem_slot, 512);
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

    if (warp == 0 || warp == kPairBWarp) {
        // ---------------------------------------- TMA producers (both CTAs)
        // warp 0 loads the int8 weight stages, warp 10 this CTA's half of the
        // activation rows, one bulk copy a stage each: a 3-D box holds the 64
        // gate and 64 up weight rows (GateUp) or a 2-D box the 128 consecutive
        // rows; the activation box holds both 64-wide K halves as two
        // [rows][128 B] sub-tiles rows * 128 bytes apart.
        const bool wprod = warp == 0;
        const uint32_t NR = wprod ? (uint32_t)NQ : (uint32_t)NB;  // ring depth
        if (lane == 0) {
            uint32_t it = 0;
            // the test hook stalls the even CTA's weight producer only: the odd CTA
            // learns of the abort through its peer abort flag
            bool ok = !(wprod && args.stall && rank == 0) || mbar_wait(stall_bar, 0, ctl);
            for (int tile = cluster; ok && tile < total_tiles; tile += n_clusters) {
                int g, cp, row0, nvalid;
                decode_pair_tile<BN>(tiles, tile, g, cp, row0, nvalid);
                const int cb = 2 * cp + (int)rank;
                const int wrow = g * args.w_rows_per_group + cb * (EPI == (int)Epi::GateUp ? 64 : kTileM);
                const int half = ((nvalid + 15) & ~15) >> 1;  // activation rows per CTA
                const int bi = pair_box_index(half);
                const CUtensorMap* mb = bi == 0 ? &tmap_b0 : bi == 1 ? &tmap_b1 : bi == 2 ? &tmap_b2 : &tmap_b3;
                const uint32_t bbytes = (uint32_t)(2 * pair_box_rows<C::kHalf>(bi) * 128);
                for (int kb = 0; kb < nkb; ++kb, ++it) {
                    const uint32_t s = it % NR, ph = (it / NR) & 1u;
                    if (wprod) {
                        if (!mbar_wait(&q_empty[s], ph ^ 1u, ctl)) { ok = false; break; }
                        uint8_t* st = smem + C::kOffQ + s * C::kQStage;
                        mbar_arrive_expect_tx(&q_full[s], (uint32_t)C::kQStage);
                        if (EPI == (int)Epi::GateUp) tma_load_3d(st, &tmap_w, &q_full[s], kb * kPairBK, wrow, 0);
                        else tma_load_2d(st, &tmap_w, &q_full[s], kb * kPairBK, wrow);
                    } else {
                        // slot s is free once the MMAs of stage it - NB completed
                        if (!mbar_wait_cluster(&done[s], ph ^ 1u, ctl)) { ok = false; break; }
                        uint8_t* st = smem + C::kOffB + s * C::kBStage;
                        mbar_arrive_expect_tx(&b_full[s], bbytes);
                        tma_load_3d(st, mb, &b_full[s], 0, row0 + (int)rank * half, 2 * kb);
                    }
                }
            }
            // drain: every fill issued must land before the CTA may exit
            for (uint32_t s = 0; s < NR && s < it; ++s) {
                const uint32_t last = it - 1 - ((it - 1 - s) % NR);
                mbar_wait_drain(wprod ? &q_full[s] : &b_full[s], (last / NR) & 1u);
            }
        }
    } else if (warp == 1 || (kIssuers == 2 && warp == kPairMma2Warp)) {
        // ------------------------------------------ MMA issuers (even CTA)
        // With two issuers, warp 1 issues the even K stages of every tile and
        // warp 11 (another SM sub-partition) the odd ones: each waits on its
        // own stages, so one's waits overlap the other's issue.  MMAs into one
        // accumulator may then run in either order (the sums are exact
        // integers), except that the tile's first, overwriting MMAs must come
        // first: warp 11 waits on tile_go[d], which warp 1 arrives on after
        // issuing them (tcgen05 fences order the two threads' MMAs).  Each
        // issuer commits its own stages and the tile (acc_full counts both).
        const int role = warp == 1 ? 0 : 1;
        if (lane == 0 && rank == 0) {
            uint32_t it = 0, tl = 0;
            bool ok = true;
            for (int tile = cluster; ok && tile < total_tiles; tile += n_clusters, ++tl) {
                int g, cp, row0, nvalid;
                decode_pair_tile<BN>(tiles, tile, g, cp, row0, nvalid);
                const uint32_t n_mma = (uint32_t)((nvalid + 15) & ~15);
                const uint32_t idesc = idesc_f16_f32(2 * kTileM, n_mma);
                // the second K half of B starts box-rows * 128 bytes into the stage
                const uint64_t b_sub16 =
                    (uint64_t)((pair_box_rows<C::kHalf>(pair_box_index((int)n_mma >> 1)) * 128) >> 4);
                const uint32_t d = tl % kPairND;
                if (role == 0) {
                    if (!mbar_wait_cluster(&acc_empty[d], ((tl / kPairND) & 1u) ^ 1u, ctl)) break;
                    tc_fence_after();
                } else if (nkb > role) {
                    if (!mbar_wait(&tile_go[d], (tl / kPairND) & 1u, ctl)) break;
                    tc_fence_after();
                }
                const uint32_t d_col = (uint32_t)C::kDCol0 + d * BN;
                for (int kb = role; kb < nkb; kb += kIssuers) {
                    const uint32_t itk = it + (uint32_t)kb;
                    const uint32_t s = itk % NB, j = itk % C::NA;
                    if (!mbar_wait_cluster(&a_ready[j], (itk / C::NA) & 1u, ctl)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t b_base = smem_u32(smem + C::kOffB + s * C::kBStage);
                    mma8_f16_tmem_a_pair(tmem + d_col, tmem + j * C::kACols, smem_desc_sw128(b_base), b_sub16, idesc,
                                         kb != 0 ? 1u : 0u);
                    if (kIssuers > 1 && kb == 0) {  // the overwriting MMAs are issued
                        tc_fence_before();
                        mbar_arrive(&tile_go[d]);
                    }
                    mma_commit_pair(&done[s], 3);
                }
                it += (uint32_t)nkb;
                if (!ok) break;
                mma_commit_pair(&acc_full[d], 3);
            }
            mma_commit_pair(&teardown[role], 1);
            mbar_wait_drain(&teardown[role], 0);
        }
    } else if ((warp >= 2 && warp < kEpiWarp0) ||
               (C::kConv == 2 && warp >= kPairConv1Warp0 && warp < kPairConv1Warp0 + 4)) {
        // ------------------------------------------------------- converters
        // Group cg (warps 2-5: 0; warps 12-15: 1) converts K columns
        // [cg * 128 / G, (cg + 1) * 128 / G) of every stage; warp w serves TMEM
        // lane quadrant w % 4.
        const int q = warp & 3;
        const int cg = (C::kConv == 2 && warp >= kPairConv1Warp0) ? 1 : 0;
        const int row = q * 32 + lane;
        const uint32_t a_ready_leader = cluster_addr(&a_ready[0], 0);
        uint32_t it = 0, qs = 0, qph = 0;  // the stage and its weight-ring slot and phase parity
        bool q_ready = false;              // the stage's weights were seen landed by the early test
        constexpr int kChunks = 8 / C::kConv;  // 16-byte chunks of its row this thread converts a stage
        uint4 raw[kChunks];                    // the stage's chunks, when read ahead at the previous stage
        bool have_raw = false;
        bool ok = true;
        for (int tile = cluster; ok && tile < total_tiles; tile += n_clusters) {
            for (int kb = 0; kb < nkb; ++kb, ++it) {
                const uint32_t bs = it % NB, j = it % C::NA;
                if (!q_ready && !warp_wait(&q_full[qs], qph, ctl)) { ok = false; break; }
                // A slot j is free once the MMAs of stage it - NA completed: tested
                // now, needed only at the first tensor-memory store below, so that
                // the test's latency overlaps the first half's conversion (the
                // same barrier and phase as a wait here; measured: prefill
                // 0.695 -> 0.681 ms, 256-expert layer 3.39 -> 3.28 ms, linear
                // 0.1153 -> 0.1099 ms)
                const uint32_t p = it - C::NA;
                const bool slot_free = it < (uint32_t)C::NA || (kSlotLate && mbar_test(&done[p % NB], (p / NB) & 1u));
                if (!kSlotLate && it >= (uint32_t)C::NA && !warp_wait_cluster(&done[p % NB], (p / NB) & 1u, ctl)) {
                    ok = false;
                    break;
                }
                // Early tests, answered while this stage converts: a satisfied
                // wait still costs its latency (measured ~120-140 cycles under
                // this kernel's load), so the next stage's weights and (group
                // 0) this stage's activations are tested now and their waits
                // skipped when already complete.  Neither phase can be behind
                // the one tested: this warp consumed the weight slot's previous
                // fill, and the activation slot's previous fill was waited
                // on by group 0 before its previous a_ready arrival.
                const uint32_t qs1 = qs + 1u == (uint32_t)NQ ? 0u : qs + 1u, qph1 = qs1 == 0u ? qph ^ 1u : qph;
                const bool q_next = kEarlyTests && mbar_test(&q_full[qs1], qph1);
                const bool b_now = kEarlyTests && cg == 0 && mbar_test(&b_full[bs], (it / NB) & 1u);
                const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + j * C::kACols;
                const uint32_t swz = (uint32_t)(row & 7);  // 128-byte swizzle: chunk c at c ^ (row & 7)
                if (!kReadAhead || !have_raw) {
                    const uint8_t* src = smem + C::kOffQ + qs * C::kQStage + row * 128;
#pragma unroll
                    for (int i = 0; i < kChunks; ++i)
                        raw[i] = *reinterpret_cast<const uint4*>(src + (((((i >> 2) + cg) * 4 + (i & 3)) ^ swz) << 4));
                }
#pragma unroll
                for (int h2 = 0; h2 < 2 / C::kConv; ++h2) {  // 64 K per tcgen05.st
                    const int hh = h2 + cg;
                    uint32_t v[32];
#pragma unroll
                    for (int c = 0; c < 4; ++c) cvt_chunk(raw[h2 * 4 + c], v + c * 8);
                    if (h2 == 0) {  // the slot's last readers are done before it is overwritten
                        if (kSlotLate && !__all_sync(0xffffffffu, slot_free) &&
                            !warp_wait_cluster(&done[p % NB], (p / NB) & 1u, ctl)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                    }
                    tmem_st_32(taddr + hh * 32, v);
                }
                if (!ok) break;
                // read the next stage's chunks now if its weights have landed:
                // their shared-memory latency then overlaps this stage's tail
                // (measured: 256-expert layer 3.47 -> 3.36 ms, linear 0.1195 ->
                // 0.1145 ms, prefill GEMM2 187 -> 182 us; GateUp +25 registers,
                // 165, no spills).  Its slot stays this warp's until the
                // q_empty arrival of the next stage.
                q_ready = __all_sync(0xffffffffu, q_next);
                have_raw = kReadAhead && q_ready;
                if (have_raw) {
                    const uint8_t* src1 = smem + C::kOffQ + qs1 * C::kQStage + row * 128;
#pragma unroll
                    for (int i = 0; i < kChunks; ++i)
                        raw[i] = *reinterpret_cast<const uint4*>(src1 + (((((i >> 2) + cg) * 4 + (i & 3)) ^ swz) << 4));
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&q_empty[qs]);  // the int8 stage has been read
                // the even CTA's MMAs read this CTA's half of B once the
                // arrival below is observed: group 0's arrival follows this
                // wait (placed after the conversion, so that activation latency
                // overlaps it), and a_ready completes only with group 0
                if (cg == 0 && !__all_sync(0xffffffffu, b_now) && !warp_wait(&b_full[bs], (it / NB) & 1u, ctl)) {
                    ok = false;
                    break;
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(a_ready_leader + j * 8);
                qs = qs1;
                qph = qph1;
            }
        }
    } else if (warp >= kEpiWarp0 && warp < kEpiWarp0 + 4) {
        // --------------------------------------------------------- epilogue
        const int q = warp & 3;
        const int ew = warp - kEpiWarp0;  // 0..3
        const int row = q * 32 + lane;    // TMEM lane = weight row of this CTA's channel block
        const uint32_t lane_addr = (uint32_t)(q * 32) << 16;
        const uint32_t acc_empty_leader = cluster_addr(&acc_empty[0], 0);
        const bool store_issuer = (ew == 0 && lane == 0);
        uint32_t tl = 0, eit = 0, n_store = 0;
        bool ok = true;
        for (int tile = cluster; ok && tile < total_tiles; tile += n_clusters, ++tl) {
            int g, cp, row0, nvalid;
            decode_pair_tile<BN>(tiles, tile, g, cp, row0, nvalid);
            const int cb = 2 * cp + (int)rank;
            const uint32_t d = tl % kPairND;
            int wrow;  // this thread's weight row within the group
            if (EPI == (int)Epi::GateUp) wrow = (row >> 6) * args.up_offset + cb * 64 + (row & 63);
            else wrow = cb * kTileM + row;
            const float sw = __ldg(args.w_scale + (size_t)g * args.w_rows_per_group + wrow);
            float* sa = row_scale_s + (tl & 1u) * BN;
            int* fl = row_flag_s + (tl & 1u) * BN;
            for (int jj = ew * 32 + lane; jj < BN; jj += 128) {
                const bool in = jj < nvalid;
                sa[jj] = in ? __ldg(args.act_scale + row0 + jj) : 0.f;
                fl[jj] = in ? __ldg(args.flags + row0 + jj) : 1;
            }
            if (!epi_sync(epi_bar, eit, ctl)) break;
            if (!warp_wait_cluster(&acc_full[d], (tl / kPairND) & 1u, ctl)) break;
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
                    if (lane == 0) mbar_arrive_cluster(acc_empty_leader + d * 8);
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
                    // per-element stores: measured, a TMA store of the h block
                    // does not pay here (this GEMM is not epilogue-bound)
                    float* xrow = xch + row * C::kXchStride;
#pragma unroll
                    for (int j = 0; j < 32; ++j) xrow[j] = dequant(__uint_as_float(r[j]), sa[j0 + j], sw);
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
                } else if (j0 + 32 <= nvalid && !__any_sync(0xffffffffu, fl[j0 + lane] != 0)) {
                    // 32 valid rows, none on the exact path (the same answer in
                    // all four warps): stage the [32 rows x 128 channels] block
                    // in shared memory and write it with one TMA store
                    uint8_t* buf = reinterpret_cast<uint8_t*>(xch) + (n_store & 1u) * C::kStoreBuf;
                    if (store_issuer) tma_store_wait_read<1>();  // the store that last read buf is done
                    if (!epi_sync(epi_bar, eit, ctl)) { ok = false; break; }
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float v = dequant(__uint_as_float(r[j]), sa[j0 + j], sw);
                        if (EPI == (int)Epi::ScaleF32)
                            reinterpret_cast<float*>(buf)[j * kTileM + row] = v;
                        else
                            reinterpret_cast<__nv_bfloat16*>(buf)[j * kTileM + row] = __float2bfloat16_rn(v);
                    }
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

    if (EPI != (int)Epi::GateUp && warp == kEpiWarp0 && lane == 0) tma_store_wait_all();
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // the pair's MMAs, TMA fills and remote arrivals are all done
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc_pair(tmem, 512);
    }
    if (!*abort_flag) fallback_rows<EPI>(args, row_start, n_groups);
}

int max_pair_clusters(const void* kern, int smem, int threads) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(2 * (unsigned)num_sms(), 1, 1);
    cfg.blockDim = dim3((unsigned)threads, 1, 1);
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
cudaError_t launch_pair_impl(const GemmArgs& args, cudaStream_t st, bool pdl) {
    auto kern = grouped_gemm_pair_kernel<C, EPI>;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    static int clusters = 0;
    std::call_once(once, [&] {
        attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
        if (attr_err == cudaSuccess) clusters = max_pair_clusters(reinterpret_cast<const void*>(kern), C::kSmem, C::kThreadsPerCta);
    });
    if (attr_err != cudaSuccess) return attr_err;

    CUtensorMap tw, tb[4];
    const uint64_t w_rows = (uint64_t)args.n_groups * args.w_rows_per_group;
    if (EPI == (int)Epi::GateUp) {
        // (k, row, half): half 1 is the up row up_offset rows below the gate row
        const uint64_t dims[3] = {(uint64_t)args.K, w_rows - (uint64_t)args.up_offset, 2};
        const uint64_t strides[2] = {(uint64_t)args.K, (uint64_t)args.up_offset * (uint64_t)args.K};
        const uint32_t box[3] = {128, 64, 2};
        if (!make_tensor_map_3d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, args.w, dims, strides, box,
                                CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
    } else if (!make_tensor_map_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, args.w, args.K, w_rows, 128, kTileM,
                                   CU_TENSOR_MAP_SWIZZLE_128B)) {
        return cudaErrorInvalidValue;
    }
    for (int i = 0; i < 4; ++i) {
        // (element within a 64-wide K chunk, row, K chunk)
        const uint64_t dims[3] = {64, (uint64_t)args.total_rows, (uint64_t)args.K / 64};
        const uint64_t strides[2] = {(uint64_t)args.K * 2, 128};
        const uint32_t box[3] = {64, (uint32_t)pair_box_rows<C::kHalf>(i), 2};
        if (!make_tensor_map_3d(&tb[i], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, args.act16, dims, strides, box,
                                CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
    }

    CUtensorMap tout = tw;  // unused by GateUp
    if (EPI == (int)Epi::ScaleF32 &&
        !make_tensor_map_2d(&tout, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, args.out, args.ld_out,
                            (uint64_t)args.total_rows, kTileM, 32, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    if (EPI == (int)Epi::ScaleBF16 &&
        !make_tensor_map_2d(&tout, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, args.out, args.ld_out,
                            (uint64_t)args.total_rows, kTileM, 32, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;

    const long max_tiles = ((long)(args.total_rows + C::BN - 1) / C::BN + args.n_groups) * (args.n_cb / 2);
    long n = clusters;
    if (max_tiles < n) n = max_tiles;
    if (n < 1) n = 1;
    return launch_kernel(kern, dim3((unsigned)(2 * n)), dim3(C::kThreadsPerCta), C::kSmem, st, pdl, tw, tb[0], tb[1],
                         tb[2], tb[3], tout, args);
}

}  // namespace

bool pair_gemm_supported(const GemmArgs& args) { return args.n_cb >= 2 && (args.n_cb & 1) == 0; }

cudaError_t launch_grouped_gemm_pair(Epi epi, const GemmArgs& args, cudaStream_t st, bool pdl) {
    if (args.total_rows == 0) return cudaSuccess;
    switch (epi) {
        case Epi::GateUp: return launch_pair_impl<CfgPairGU, 0>(args, st, pdl);
        case Epi::ScaleF32: return launch_pair_impl<CfgPairSc, 1>(args, st, pdl);
        case Epi::ScaleBF16: return launch_pair_impl<CfgPairSc, 2>(args, st, pdl);
    }
    return cudaErrorInvalidValue;
}

}  // namespace moe

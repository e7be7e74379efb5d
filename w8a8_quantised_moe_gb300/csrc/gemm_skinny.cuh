// gemm_skinny.cuh -- the dp4a grouped GEMM's work-unit loop as a device
// function: the body of grouped_gemm_skinny_kernel (gemm_skinny.cu) and of the
// GEMM phases of the fused decode kernel (fused.cu).  What it computes and
// why it is shaped so: gemm_skinny.cu.
#pragma once

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

// Where skinny_run's activation rows come from.
enum SkSrc : int {
    kSkSrcRows = 0,    // rows [total_rows][K] of act8
    kSkSrcGather = 1   // row r of the group table is row map[r] of act8
};

__host__ __device__ constexpr int skinny_smem_bytes(int K) { return kSkChunk * K; }

// Persistent grid over work units = (non-empty group, block of weight rows);
// per unit the group's activation rows pass through shared memory in chunks
// of kSkChunk rows (zero-padded to the kernel's chunk shape).  CTA `bid` of
// `nblk` starts with unit bid; its next units are bid + nblk, bid + 2 nblk,
// ... or, with args.sched, taken in turn from a counter (one taken a unit
// ahead, so the atomic's latency is hidden), which evens out CTAs whose units
// took longer.  act_s: skinny_smem_bytes(K) bytes; unit_start, row_start:
// kMaxExperts + 1 ints; next_s: two ints (shared memory: the unit taken from
// the counter reaches all threads through them, in turn).  The activation
// rows are read through L2 (coherent loads): they may have been written
// earlier in the same launch, before a grid-wide barrier.  kSkSrcGather:
// row_map [total_rows] gives each row's source row in act8 (map_rows rows),
// copied to map_s (total_rows ints of shared memory) first.
template <int EPI, int SRC = kSkSrcRows>
__device__ __forceinline__ void skinny_run(const GemmArgs& args, int8_t* act_s, int* unit_start, int* row_start,
                                           int* next_s, int bid, int nblk, const int32_t* row_map = nullptr,
                                           int map_rows = 0, int* map_s = nullptr) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int G = args.n_groups;
    const int unit_rows = EPI == (int)Epi::GateUp ? kSkUnitGateUp : kSkUnitScale;
    const int per_group = (EPI == (int)Epi::GateUp ? args.up_offset : args.w_rows_per_group) / unit_rows;
    const bool dyn = args.sched != nullptr;

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
    if (SRC == kSkSrcGather)
        for (int r = threadIdx.x; r < args.total_rows; r += kSkThreads) {
            const int m = row_map[r];
            map_s[r] = in_range(m, 0, map_rows, args.error) ? m : 0;
        }
    if (dyn && threadIdx.x == 0) next_s[0] = nblk + (int)atomicAdd(args.sched, 1u);  // used if bid has a unit
    __syncthreads();
    const int total_units = unit_start[G];
    const int K = args.K;
    const int8_t* act = args.act8;

    // un: the unit taken after u; grab: thread 0's request for the one after
    // un, in flight.  next_s slot ph is written next (a slot is rewritten only
    // after a barrier past its reads).
    int un = bid + nblk, ph = 1;
    unsigned grab = 0u;
    if (dyn) {
        un = bid < total_units ? next_s[0] : total_units;
        if (threadIdx.x == 0 && un < total_units) grab = nblk + atomicAdd(args.sched, 1u);
    }
    int staged_row0 = -1;  // first activation row in act_s (row ranges of groups are disjoint)
    for (int u = bid; u < total_units;) {
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
                uint4* dst = reinterpret_cast<uint4*>(act_s);
                if (SRC == kSkSrcGather) {
                    const int row16 = K / 16;
                    for (int i = threadIdx.x; i < n16; i += kSkThreads) {
                        const int r = i / row16;
                        dst[i] = r < rc ? __ldcg(reinterpret_cast<const uint4*>(act + (size_t)map_s[row0 + r] * K) +
                                                 (i - r * row16))
                                        : make_uint4(0, 0, 0, 0);
                    }
                } else {
                    const uint4* src = reinterpret_cast<const uint4*>(act + (size_t)row0 * K);
                    for (int i = threadIdx.x; i < n16; i += kSkThreads)
                        dst[i] = i < valid16 ? __ldcg(src + i) : make_uint4(0, 0, 0, 0);
                }
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
        // the next unit
        u = un;
        if (!dyn) {
            un += nblk;
        } else {
            if (threadIdx.x == 0) next_s[ph] = un < total_units ? (int)grab : total_units;
            __syncthreads();
            un = next_s[ph];
            ph ^= 1;
            if (threadIdx.x == 0 && un < total_units) grab = nblk + atomicAdd(args.sched, 1u);
        }
    }
    if (dyn) {  // the last CTA out leaves the counter words zero for the next launch
        __syncthreads();
        if (threadIdx.x == 0) {
            __threadfence();
            if (atomicAdd(args.sched + 1, 1u) == (unsigned)nblk - 1u) {
                args.sched[0] = 0u;
                args.sched[1] = 0u;
                __threadfence();
            }
        }
    }
}

}  // namespace
}  // namespace moe

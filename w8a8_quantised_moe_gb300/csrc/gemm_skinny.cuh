// gemm_skinny.cuh -- the dp4a grouped GEMM's work-unit loop as a device
// function: the body of grouped_gemm_skinny_kernel (gemm_skinny.cu) and of the
// GEMM phases of the one-kernel layer (fused.cu).  What it computes and why
// it is shaped so: gemm_skinny.cu.
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

// A warp item: kSkRows weight rows x RC staged activation rows (rc valid),
// dot products over K in batches of kSkNB 512-byte steps per row (every load
// of a batch issued before any is used), then the epilogue of the valid (row,
// channel) pairs.  GateUp: rows are gate c, gate c+1, up c, up c+1 (c = first
// channel).  The first batch of a warp's next item (in this step or the
// next) is issued before the current item's epilogue, so that it is in
// flight through the epilogue and the CTA's staging barrier.
constexpr int kSkNB = 4;

__device__ __forceinline__ int skinny_first(int EPI, int unit, int item) {
    return EPI == (int)Epi::GateUp ? unit * kSkUnitGateUp + item * (kSkRows / 2) : unit * kSkUnitScale + item * kSkRows;
}

template <int EPI>
__device__ __forceinline__ void skinny_load(uint4 (&wv)[kSkNB][kSkRows], const GemmArgs& args, int g, int first,
                                            int n, int lane) {
    const int K = args.K;
    const int8_t* w = static_cast<const int8_t*>(args.w) + (size_t)g * args.w_rows_per_group * K;
#pragma unroll
    for (int j = 0; j < kSkRows; ++j) {
        const int wrow = EPI == (int)Epi::GateUp ? (j >> 1) * args.up_offset + first + (j & 1) : first + j;
        const int8_t* wr = w + (size_t)wrow * K;
#pragma unroll
        for (int b = 0; b < kSkNB; ++b) {
            const int k = (n * kSkNB + b) * 512 + lane * 16;
            wv[b][j] = k < K ? ld_stream16(wr + k) : make_uint4(0u, 0u, 0u, 0u);
        }
    }
}

// acc[j][r] += batch n's products (int32: exact in any order).
template <int RC>
__device__ __forceinline__ void skinny_accum(const uint4 (&wv)[kSkNB][kSkRows], const int8_t* __restrict__ act_s,
                                             int K, int n, int lane, int (&acc)[kSkRows][RC]) {
#pragma unroll
    for (int b = 0; b < kSkNB; ++b) {
        const int k = (n * kSkNB + b) * 512 + lane * 16;
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

// The item's epilogue: reduction across the warp, then the valid (row,
// channel) outputs.
template <int EPI, int RC>
__device__ __forceinline__ void skinny_epilogue(const GemmArgs& args, int (&acc)[kSkRows][RC], int rc, int row0,
                                                int g, int first, int lane) {
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

// A step: unit u (group g, unit index within the group) and one chunk of up
// to kSkChunk of the group's activation rows, [row0, min(row0 + kSkChunk,
// r_end)).
struct SkStep {
    int g, unit, row0, r_end;
};

__host__ __device__ constexpr int skinny_items(int EPI) { return EPI == (int)Epi::GateUp ? kSkItemsGateUp : kSkItemsScale; }

// This warp's items of step `cur`; wv holds the first batch of the first
// item on entry and, on return, the first batch of `next`'s first item
// (when next_ok).
template <int EPI, int RC>
__device__ __forceinline__ void skinny_step(const GemmArgs& args, const int8_t* __restrict__ act_s,
                                            const SkStep& cur, const SkStep& next, bool next_ok, int nbat,
                                            uint4 (&wv)[kSkNB][kSkRows], int warp, int lane) {
    constexpr int kItems = skinny_items(EPI);
    const int rc = min(kSkChunk, cur.r_end - cur.row0);
#pragma unroll 1
    for (int it = 0; it < kItems; ++it) {
        const int first = skinny_first(EPI, cur.unit, warp * kItems + it);
        int acc[kSkRows][RC];
#pragma unroll
        for (int j = 0; j < kSkRows; ++j)
#pragma unroll
            for (int r = 0; r < RC; ++r) acc[j][r] = 0;
#pragma unroll 1
        for (int n = 0; n < nbat; ++n) {
            if (n > 0) skinny_load<EPI>(wv, args, cur.g, first, n, lane);
            skinny_accum<RC>(wv, act_s, args.K, n, lane, acc);
        }
        if (it + 1 < kItems) skinny_load<EPI>(wv, args, cur.g, skinny_first(EPI, cur.unit, warp * kItems + it + 1), 0, lane);
        else if (next_ok) skinny_load<EPI>(wv, args, next.g, skinny_first(EPI, next.unit, warp * kItems), 0, lane);
        skinny_epilogue<EPI, RC>(args, acc, rc, cur.row0, cur.g, first, lane);
    }
}

// Hooks through which the one-kernel layer hands work between its GEMMs
// inside skinny_run; SkNoHook: none (compiled away).
struct SkNoHook {
    static constexpr bool kWaits = false;   // ready() may wait
    static constexpr bool kCounts = false;  // unit_end_*() need a barrier at every unit's end
    // thread 0, before group g's rows are staged: false = give up (the CTA stops its units)
    __device__ __forceinline__ bool ready(int) { return true; }
    // thread 0, before the barrier that ends a unit
    __device__ __forceinline__ void unit_end_pre() {}
    // every thread, after it: the unit (of group g) is complete in every warp
    __device__ __forceinline__ void unit_end_post(int) {}
    // every thread, after the CTA's last unit
    __device__ __forceinline__ void end() {}
};

// Where skinny_run's activation rows come from.
enum SkSrc : int {
    kSkSrcRows = 0,    // rows [total_rows][K] of act8
    kSkSrcGather = 1   // row r of the group table is row map[r] of act8
};

__host__ __device__ constexpr int skinny_smem_bytes(int K) { return kSkChunk * K; }

// Copies rows row0 .. row0 + rc of the group table into act_s, zeros up to
// the step's row shape (coherent L2 loads: the rows may have been written
// earlier in the same launch, before a grid-wide barrier).
template <int SRC>
__device__ __forceinline__ void skinny_stage(int8_t* act_s, const int8_t* act, int K, int row0, int rc,
                                             const int* map_s) {
    const int RC = rc <= 2 ? 2 : rc <= 4 ? 4 : 8;
    const int n16 = RC * K / 16;
    uint4* dst = reinterpret_cast<uint4*>(act_s);
    if (SRC == kSkSrcGather) {
        const int row16 = K / 16;
        for (int i = threadIdx.x; i < n16; i += kSkThreads) {
            const int r = i / row16;
            dst[i] = r < rc ? __ldcg(reinterpret_cast<const uint4*>(act + (size_t)map_s[row0 + r] * K) + (i - r * row16))
                            : make_uint4(0, 0, 0, 0);
        }
    } else {
        const int valid16 = rc * K / 16;
        const uint4* src = reinterpret_cast<const uint4*>(act + (size_t)row0 * K);
        for (int i = threadIdx.x; i < n16; i += kSkThreads) dst[i] = i < valid16 ? __ldcg(src + i) : make_uint4(0, 0, 0, 0);
    }
}

// Persistent grid over work units = (non-empty group, block of weight rows);
// a step is one unit and one chunk of up to kSkChunk of its group's
// activation rows, staged in shared memory (zero-padded to the step's row
// shape).  CTA `bid` of `nblk` starts with unit bid; its next units are
// bid + nblk, bid + 2 nblk, ... or, with args.sched, taken in turn from a
// counter (one taken a unit ahead, so the atomic's latency is hidden), which
// evens out CTAs whose units took longer.  act_s: skinny_smem_bytes(K) bytes;
// unit_start, row_start: kMaxExperts + 1 ints; next_s: three ints (shared
// memory: the unit taken from the counter reaches all threads through the
// first two, in turn; the third carries a hook's give-up).  kSkSrcGather: row_map [total_rows] gives each row's source row
// in act8 (map_rows rows), copied to map_s (total_rows ints of shared memory)
// first; with row_map == nullptr, map_s already holds it.
// PDL (a separate kernel launched with programmatic dependent launch): the
// unit table is built, and thread 0 prefetches its first unit's weights into
// L2, before the wait for the previous kernel (the expert offsets and the
// weights were complete before that kernel started; the activation rows and
// scales are read only after the wait).
template <int EPI, int SRC = kSkSrcRows, class Hook = SkNoHook, bool PDL = false>
__device__ __forceinline__ void skinny_run(const GemmArgs& args, int8_t* act_s, int* unit_start, int* row_start,
                                           int* next_s, int bid, int nblk, const int32_t* row_map = nullptr,
                                           int map_rows = 0, int* map_s = nullptr, Hook hook = Hook()) {
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
    if (SRC == kSkSrcGather && row_map != nullptr)
        for (int r = threadIdx.x; r < args.total_rows; r += kSkThreads) {
            const int m = row_map[r];
            map_s[r] = in_range(m, 0, map_rows, args.error) ? m : 0;
        }
    __syncthreads();
    const int total_units = unit_start[G];
    if (PDL) {
        if (threadIdx.x == 0 && bid < total_units) {
            const int g = last_le(unit_start, G, bid);
            const int first = skinny_first(EPI, bid - unit_start[g], 0);
            const int8_t* w = static_cast<const int8_t*>(args.w) + ((size_t)g * args.w_rows_per_group + first) * args.K;
            if (EPI == (int)Epi::GateUp) {  // the unit's gate rows and its up rows
                prefetch_l2_bulk(w, (uint32_t)((size_t)kSkUnitGateUp * args.K));
                prefetch_l2_bulk(w + (size_t)args.up_offset * args.K, (uint32_t)((size_t)kSkUnitGateUp * args.K));
            } else {
                prefetch_l2_bulk(w, (uint32_t)((size_t)kSkUnitScale * args.K));
            }
        }
        pdl_wait();
        pdl_trigger();
    }
    if (dyn && threadIdx.x == 0) next_s[0] = nblk + (int)atomicAdd(args.sched, 1u);  // used if bid has a unit
    __syncthreads();
    const int K = args.K;
    const int8_t* act = args.act8;
    const int nbat = (K + kSkNB * 512 - 1) / (kSkNB * 512);
    auto step_of = [&](int u) {  // the first step of unit u
        SkStep st;
        st.g = last_le(unit_start, G, u);
        st.unit = u - unit_start[st.g];
        st.row0 = row_start[st.g];
        st.r_end = row_start[st.g + 1];
        return st;
    };

    // un: the unit taken after the current one; grab: thread 0's request for
    // the one after un, in flight.  next_s slot ph is written next (a slot is
    // rewritten only after a barrier past its reads).
    int un = bid + nblk, ph = 1;
    unsigned grab = 0u;
    if (dyn) {
        un = bid < total_units ? next_s[0] : total_units;
        if (threadIdx.x == 0 && un < total_units) grab = nblk + atomicAdd(args.sched, 1u);
    }
    if (bid >= total_units) un = total_units;
    SkStep cur{};
    uint4 wv[kSkNB][kSkRows];
    bool have = bid < total_units;
    if (have) {
        cur = step_of(bid);
        skinny_load<EPI>(wv, args, cur.g, skinny_first(EPI, cur.unit, warp * skinny_items(EPI)), 0, lane);
        if (Hook::kWaits) {
            if (threadIdx.x == 0) next_s[2] = hook.ready(cur.g) ? 0 : 1;
            __syncthreads();
            have = next_s[2] == 0;
        }
        if (have) skinny_stage<SRC>(act_s, act, K, cur.row0, min(kSkChunk, cur.r_end - cur.row0), map_s);
    }
    __syncthreads();
    while (have) {
        // the step after this one
        SkStep nxt = cur;
        const bool new_unit = cur.row0 + kSkChunk >= cur.r_end;
        bool next_ok = true;
        if (!new_unit) nxt.row0 = cur.row0 + kSkChunk;
        else if ((next_ok = un < total_units)) nxt = step_of(un);
        const int rc = min(kSkChunk, cur.r_end - cur.row0);
        if (rc <= 2) skinny_step<EPI, 2>(args, act_s, cur, nxt, next_ok, nbat, wv, warp, lane);
        else if (rc <= 4) skinny_step<EPI, 4>(args, act_s, cur, nxt, next_ok, nbat, wv, warp, lane);
        else skinny_step<EPI, 8>(args, act_s, cur, nxt, next_ok, nbat, wv, warp, lane);
        // the next step's rows, unless they are this step's (distinct groups
        // never share a first row); every warp's next batch is in flight
        const bool restage = next_ok && nxt.row0 != cur.row0;
        if (dyn && new_unit && threadIdx.x == 0) next_s[ph] = un < total_units ? (int)grab : total_units;
        if (new_unit) hook.unit_end_pre();
        if (Hook::kWaits && restage && threadIdx.x == 0) next_s[2] = hook.ready(nxt.g) ? 0 : 1;
        // every warp is done with act_s / next_s is set / a hook's word is set
        if (restage || (dyn && new_unit) || (Hook::kCounts && new_unit)) __syncthreads();
        if (new_unit) hook.unit_end_post(cur.g);
        if (Hook::kWaits && restage && next_s[2] != 0) break;  // every thread alike
        if (restage) {
            skinny_stage<SRC>(act_s, act, K, nxt.row0, min(kSkChunk, nxt.r_end - nxt.row0), map_s);
            __syncthreads();
        }
        if (new_unit) {
            if (!dyn) {
                un += nblk;
            } else {
                un = next_s[ph];
                ph ^= 1;
                if (threadIdx.x == 0 && un < total_units) grab = nblk + atomicAdd(args.sched, 1u);
            }
        }
        cur = nxt;
        have = next_ok;
    }
    hook.end();
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

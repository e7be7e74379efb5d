// api.cu -- the C ABI (include/moe_w8a8.h): argument checks, workspace
// layout and the launch sequence of the layer.
//
// Forward launch sequence on the caller's stream (no host synchronisation):
//   1 router           split of the router weights into three bf16 parts,
//                      tensor-core logits, top-k, weights, chunk counts/ranks
//                      (T <= 128: partial logits per slice of the fp32 weights
//                      on the CUDA cores, then per-token sums and top-k, whose
//                      last CTA also does step 2)
//   2 scan             expert offsets, first slot of every (chunk, expert)
//   3 permute_quant    slots; per-token quantisation scattered into slots
//   4 grouped GEMM 1   gate/up GEMM + scale outer product + SiLU(gate)*up -> h
//   5 requant          per-slot requantisation of h
//   6 grouped GEMM 2   down GEMM + scale outer product -> o
//   7 combine          weighted sum of each token's k slot rows -> y (bf16)
// The host-resident entry point runs this sequence once per token chunk,
// with the copies of x and y on a second stream.
#include <atomic>
#include <cstdlib>
#include <cstring>
#include <vector>

#include "moe_w8a8.h"
#include "internal.h"

namespace moe {

int num_sms() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) return 1;
    return n;
}

namespace {

std::atomic<uint64_t> g_timeout_ns{kDefaultTimeoutNs};
std::atomic<int> g_gemm_path{-1};  // -1: automatic choice of the GEMM kernel
thread_local cudaEvent_t const* t_events = nullptr;  // measurement hook

cudaError_t mark(int i, cudaStream_t st) {
    return t_events ? cudaEventRecord(t_events[i], st) : cudaSuccess;
}

bool pdl_env_off() {
    static const bool off = [] {
        const char* v = std::getenv("MOE_W8A8_NO_PDL");
        return v != nullptr && v[0] != '\0' && v[0] != '0';
    }();
    return off;
}

size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The dp4a GEMM's scheduling words in a workspace's error region (the GEMM
// leaves them zero).  Taken by the one-kernel layer, whose gate/up GEMM phase
// they shortened (decode layer: 122.5 -> 118.7 us); the separate dp4a
// kernels deal their units round-robin (measured: the decode layer 201.3 us
// round-robin, 203.4 us taking units from the counter).
unsigned int* sched_words(int* err) {
    return reinterpret_cast<unsigned int*>(reinterpret_cast<char*>(err) + kSchedOffset);
}

moe_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

bool moe_shape_ok(int64_t T, int64_t H, int64_t I, int64_t E, int64_t k) {
    if (T < 0 || T > (int64_t(1) << 20)) return false;
    if (H < 128 || H > 16384 || H % 128) return false;
    if (I < 128 || I > 16384 || I % 128) return false;
    if (E < 1 || E > kMaxExperts) return false;
    if (k < 1 || k > kMaxTopK || k > E) return false;
    return true;
}

}  // namespace

bool pdl_default() { return t_events == nullptr && !pdl_env_off(); }

uint64_t current_timeout_ns() { return g_timeout_ns.load(); }

bool injected(InjectFault f) {
    const char* v = std::getenv("MOE_INJECT");
    if (v == nullptr || v[0] == '\0') return false;
    const char* name = f == kInjectWsShort      ? "ws_short"
                       : f == kInjectBadPtr     ? "bad_ptr"
                       : f == kInjectLaunchFail ? "launch_fail"
                       : f == kInjectBadSlot    ? "bad_slot"
                                                : "stall";
    const size_t n = std::strlen(name);
    for (const char* p = v; *p != '\0';) {
        const char* end = std::strchr(p, ',');
        const size_t len = end ? (size_t)(end - p) : std::strlen(p);
        if (len == n && std::strncmp(p, name, n) == 0) return true;
        if (!end) break;
        p = end + 1;
    }
    return false;
}

namespace {
std::atomic<uint64_t> g_launches{0};
}
void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

GemmShape pick_gemm_shape(long rows, long groups, long K, Epi epi, long w_rows_per_group, long up_offset) {
    const int forced = g_gemm_path.load();
    if (forced >= 0 && forced <= (int)GemmShape::Skinny) {
        const GemmShape s = static_cast<GemmShape>(forced);
        if (s != GemmShape::Skinny || skinny_shape_supported(epi, K, w_rows_per_group, up_offset)) return s;
    }
    GemmShape s = choose_gemm_shape(rows, groups, K);
    if (s == GemmShape::Skinny && !skinny_shape_supported(epi, K, w_rows_per_group, up_offset))
        s = GemmShape::Narrow;
    return s;
}

FwdLayout fwd_layout(int64_t T, int64_t H, int64_t I, int64_t E, int64_t k) {
    FwdLayout L{};
    const int64_t S = T * k;
    const int64_t nchunk = (T + kRouterTokens - 1) / kRouterTokens;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off = align256(off + bytes);
        return at;
    };
    L.err = take(256);
    L.counts = take(2 * 4);
    const RouterPlan rp = router_plan(T, H, E);
    // the router's three-part bf16 weight split; once the router has run, the
    // smoothed layer keeps its reciprocal factors here (4 * E * H <= 6 * E_pad * H)
    L.wsplit = take((size_t)3 * rp.E_pad * H * 2);
    L.logits = take((size_t)rp.KS * T * rp.E_pad * 4);
    L.topk_ids = take(S * 4);
    L.topk_w = take(S * 4);
    L.rank = take(S * 4);
    L.hist = take(nchunk * E * 4);
    L.offsets = take((E + 1) * 4);
    L.slot_of = take(S * 4);
    L.slot_token = take(S * 4);
    L.s_x = take(T * 4);
    L.s_slot = take(S * 4);
    L.flag1 = take(S * 4);
    L.list1 = take(S * 4);
    L.flag2 = take(S * 4);
    L.list2 = take(S * 4);
    L.q_x16 = take(S * H * 2);
    L.h = take(S * I * 4);
    L.s_h = take(S * 4);
    L.q_h16 = take(S * I * 2);
    L.o = take(S * H * 4);
    L.fctl = take(2 * E * 4);  // the one-kernel layer's per-expert hand-off words
    L.total = off;
    return L;
}

LinLayout lin_layout(int64_t M, int64_t N, int64_t K) {
    (void)N;
    LinLayout L{};
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off = align256(off + bytes);
        return at;
    };
    L.err = take(256);
    L.counts = take(2 * 4);
    L.s_x = take(M * 4);
    L.flag = take(M * 4);
    L.list = take(M * 4);
    L.q_x16 = take(M * K * 2);
    L.total = off;
    return L;
}

}  // namespace moe

using namespace moe;

namespace {

template <typename T>
T* at(void* base, size_t off) {
    return reinterpret_cast<T*>(static_cast<char*>(base) + off);
}

moe_status_t forward_impl(const uint16_t* x, const float* router_w, const float* router_bias,
                          const int8_t* w13_q, const float* w13_scale, const int8_t* w2_q,
                          const float* w2_scale, int64_t T, int64_t H, int64_t I, int64_t E,
                          int64_t k, uint16_t* y, void* workspace, size_t workspace_bytes,
                          void* stream, const moe_w8a8_debug_t* dbg, bool fp8 = false,
                          const float* smooth = nullptr) {
    if (!moe_shape_ok(T, H, I, E, k)) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (T == 0) return MOE_OK;  // nothing is read or written
    if (smooth != nullptr && !aligned16(smooth)) return MOE_ERR_INVALID_ARG;
    const void* ptrs[] = {x, router_w, w13_q, w13_scale, w2_q, w2_scale, y, workspace};
    for (const void* p : ptrs)
        if (p == nullptr || !aligned16(p) || injected(kInjectBadPtr)) return MOE_ERR_INVALID_ARG;
    if (router_bias != nullptr && !aligned16(router_bias)) return MOE_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return MOE_ERR_INVALID_ARG;
    const FwdLayout L = fwd_layout(T, H, I, E, k);
    if (injected(kInjectWsShort) && workspace_bytes >= L.total) workspace_bytes = L.total - 1;
    if (workspace_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
    // the FP8 layer has its own GEMM kernels: a forced INT8 kernel choice
    // (moe_w8a8_set_gemm_path) cannot be honoured there
    if (fp8 && g_gemm_path.load() >= 0) return MOE_ERR_NOT_IMPLEMENTED;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int S = (int)(T * k);
    const int nchunk = (int)((T + kRouterTokens - 1) / kRouterTokens);
    int* err = at<int>(workspace, L.err);
    uint16_t* wsplit = at<uint16_t>(workspace, L.wsplit);
    float* logits = at<float>(workspace, L.logits);
    int32_t* topk_ids = at<int32_t>(workspace, L.topk_ids);
    float* topk_w = at<float>(workspace, L.topk_w);
    int32_t* rank = at<int32_t>(workspace, L.rank);
    int32_t* hist = at<int32_t>(workspace, L.hist);
    int32_t* offsets = at<int32_t>(workspace, L.offsets);
    int32_t* slot_of = at<int32_t>(workspace, L.slot_of);
    int32_t* slot_token = at<int32_t>(workspace, L.slot_token);
    float* s_x = at<float>(workspace, L.s_x);
    float* s_slot = at<float>(workspace, L.s_slot);
    int32_t* counts = at<int32_t>(workspace, L.counts);
    int32_t* flag1 = at<int32_t>(workspace, L.flag1);
    int32_t* list1 = at<int32_t>(workspace, L.list1);
    int32_t* flag2 = at<int32_t>(workspace, L.flag2);
    int32_t* list2 = at<int32_t>(workspace, L.list2);
    uint16_t* q_x16 = at<uint16_t>(workspace, L.q_x16);
    float* h = at<float>(workspace, L.h);
    float* s_h = at<float>(workspace, L.s_h);
    uint16_t* q_h16 = at<uint16_t>(workspace, L.q_h16);
    float* o = at<float>(workspace, L.o);
    const uint64_t timeout = g_timeout_ns.load();
    // GEMM kernels; the dp4a kernel reads int8 codes, which then take the
    // place of the fp16 ones in the same workspace regions
    const GemmShape shape1 = pick_gemm_shape(S, E, H, Epi::GateUp, 2 * I, I);
    const GemmShape shape2 = pick_gemm_shape(S, E, I, Epi::ScaleF32, H, 0);
    // 8-bit codes (int8 for the dp4a kernel, E4M3 for the FP8 layer) take the
    // place of the fp16 ones in the same workspace regions
    int8_t* q_x8 = (fp8 || shape1 == GemmShape::Skinny) ? reinterpret_cast<int8_t*>(q_x16) : nullptr;
    int8_t* q_h8 = (fp8 || shape2 == GemmShape::Skinny) ? reinterpret_cast<int8_t*>(q_h16) : nullptr;
    const bool pdl = pdl_default();  // every launch after the first

    cudaError_t e;
    if ((e = mark(0, st)) != cudaSuccess) return from_cuda(e);
    // the routing ticket of the small-batch router sits in the error region
    unsigned int* ticket = reinterpret_cast<unsigned int*>(reinterpret_cast<char*>(err) + kTicketOffset);
    e = launch_router(x, router_w, router_bias, (int)T, (int)H, (int)E, (int)k, wsplit, logits, topk_ids,
                      topk_w, rank, hist, offsets, counts, ticket, err, timeout, st, pdl);
    if (e != cudaSuccess) return from_cuda(e);
    if ((e = mark(1, st)) != cudaSuccess) return from_cuda(e);
    if (!router_plan(T, H, E).small) {  // else the router computed the prefix sums
        e = launch_scan(hist, nchunk, (int)E, offsets, counts, st, pdl);
        if (e != cudaSuccess) return from_cuda(e);
    }
    if ((e = mark(2, st)) != cudaSuccess) return from_cuda(e);
    if (fp8)
        e = launch_permute_quant_fp8(x, topk_ids, rank, hist, (int)T, (int)H, (int)E, (int)k, slot_of, slot_token,
                                     s_x, s_slot, reinterpret_cast<uint8_t*>(q_x8), err, st, pdl);
    else if (smooth)
        // the router's weight split is dead once the router has run: its region
        // (6 * E_pad * H >= 4 * E * H bytes) holds the smoothing reciprocals
        e = launch_permute_quant_smooth(x, smooth, reinterpret_cast<float*>(wsplit), topk_ids, rank, hist, (int)T,
                                        (int)H, (int)E, (int)k, slot_of, slot_token, s_x, s_slot,
                                        q_x8 ? nullptr : q_x16, q_x8, flag1, list1, counts + 0, err, st, pdl);
    else
        e = launch_permute_quant(x, topk_ids, rank, hist, (int)T, (int)H, (int)E, (int)k, slot_of, slot_token,
                                 s_x, s_slot, q_x8 ? nullptr : q_x16, q_x8, flag1, list1, counts + 0, err, st, pdl);
    if (e != cudaSuccess) return from_cuda(e);
    // test hook of the checked build: an out-of-range slot index for the
    // combine's checks to catch (0x7f7f7f7f; the normal build ignores it)
    if (kChecked && injected(kInjectBadSlot) && (e = cudaMemsetAsync(slot_of, 0x7f, 4, st)) != cudaSuccess)
        return from_cuda(e);

    GemmArgs g1{};
    g1.w = w13_q;
    g1.act16 = q_x16;
    g1.act8 = q_x8;
    g1.K = (int)H;
    g1.n_cb = (int)(I / 64);
    g1.n_groups = (int)E;
    g1.total_rows = S;
    g1.offsets = offsets;
    g1.w_rows_per_group = (int)(2 * I);
    g1.up_offset = (int)I;
    g1.w_scale = w13_scale;
    g1.act_scale = s_slot;
    g1.out = h;
    g1.ld_out = (int)I;
    g1.acc_out = dbg ? dbg->acc1 : nullptr;
    g1.flags = flag1;
    g1.fb_list = list1;
    g1.fb_count = counts + 0;
    g1.error = err;
    g1.timeout_ns = timeout;
    g1.stall = injected(kInjectStall) ? 1 : 0;
    if ((e = mark(3, st)) != cudaSuccess) return from_cuda(e);
    e = fp8 ? launch_grouped_gemm_fp8(Epi::GateUp, g1, st, pdl) : launch_grouped_gemm(Epi::GateUp, shape1, g1, st, pdl);
    if (e != cudaSuccess) return from_cuda(e);

    if ((e = mark(4, st)) != cudaSuccess) return from_cuda(e);
    if (fp8)
        e = launch_requant_fp8(h, S, (int)I, s_h, reinterpret_cast<uint8_t*>(q_h8), st, pdl);
    else if (q_h8)
        e = launch_requant(h, S, (int)I, s_h, nullptr, q_h8, flag2, list2, counts + 1, st, pdl);
    else
        e = launch_requant(h, S, (int)I, s_h, q_h16, dbg ? dbg->q_h : nullptr, flag2, list2, counts + 1, st, pdl);
    if (e != cudaSuccess) return from_cuda(e);

    GemmArgs g2{};
    g2.w = w2_q;
    g2.act16 = q_h16;
    g2.act8 = q_h8;
    g2.K = (int)I;
    g2.n_cb = (int)(H / 128);
    g2.n_groups = (int)E;
    g2.total_rows = S;
    g2.offsets = offsets;
    g2.w_rows_per_group = (int)H;
    g2.up_offset = 0;
    g2.w_scale = w2_scale;
    g2.act_scale = s_h;
    g2.out = o;
    g2.ld_out = (int)H;
    g2.acc_out = dbg ? dbg->acc2 : nullptr;
    g2.flags = flag2;
    g2.fb_list = list2;
    g2.fb_count = counts + 1;
    g2.error = err;
    g2.timeout_ns = timeout;
    g2.stall = g1.stall;
    if ((e = mark(5, st)) != cudaSuccess) return from_cuda(e);
    e = fp8 ? launch_grouped_gemm_fp8(Epi::ScaleF32, g2, st, pdl)
            : launch_grouped_gemm(Epi::ScaleF32, shape2, g2, st, pdl);
    if (e != cudaSuccess) return from_cuda(e);

    if ((e = mark(6, st)) != cudaSuccess) return from_cuda(e);
    e = launch_combine(o, slot_of, topk_w, (int)T, (int)H, (int)k, y, err, st, pdl);
    if (e != cudaSuccess) return from_cuda(e);
    if ((e = mark(7, st)) != cudaSuccess) return from_cuda(e);

    if (dbg) {
        auto cp = [&](void* dst, const void* src, size_t bytes) -> cudaError_t {
            if (!dst) return cudaSuccess;
            return cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToDevice, st);
        };
        const size_t Sb = (size_t)S * 4;
        if ((e = cp(dbg->topk_ids, topk_ids, Sb)) != cudaSuccess) return from_cuda(e);
        if ((e = cp(dbg->topk_w, topk_w, Sb)) != cudaSuccess) return from_cuda(e);
        if ((e = cp(dbg->offsets, offsets, (size_t)(E + 1) * 4)) != cudaSuccess) return from_cuda(e);
        if ((e = cp(dbg->slot_of, slot_of, Sb)) != cudaSuccess) return from_cuda(e);
        if ((e = cp(dbg->slot_token, slot_token, Sb)) != cudaSuccess) return from_cuda(e);
        if ((e = cp(dbg->s_x, s_x, (size_t)T * 4)) != cudaSuccess) return from_cuda(e);
        if ((e = cp(dbg->h, h, (size_t)S * I * 4)) != cudaSuccess) return from_cuda(e);
        if ((e = cp(dbg->s_h, s_h, Sb)) != cudaSuccess) return from_cuda(e);
        if ((e = cp(dbg->o, o, (size_t)S * H * 4)) != cudaSuccess) return from_cuda(e);
        if (q_h8 && (e = cp(dbg->q_h, q_h8, (size_t)S * I)) != cudaSuccess) return from_cuda(e);
        if ((e = cp(dbg->s_slot, s_slot, Sb)) != cudaSuccess) return from_cuda(e);
        if (dbg->q_slot) {  // every slot's row, in slot order
            e = q_x8 ? launch_s8_rows_gather(q_x8, nullptr, S, (int)H, 1, S, dbg->q_slot, err, st)
                     : launch_f16_rows_to_s8(q_x16, nullptr, S, (int)H, 1, S, dbg->q_slot, err, st);
            if (e != cudaSuccess) return from_cuda(e);
        }
        if (dbg->q_x) {
            // token t's quantised row sits in each of its slots; take the first
            e = q_x8 ? launch_s8_rows_gather(q_x8, slot_of, (int)T, (int)H, (int)k, S, dbg->q_x, err, st)
                     : launch_f16_rows_to_s8(q_x16, slot_of, (int)T, (int)H, (int)k, S, dbg->q_x, err, st);
            if (e != cudaSuccess) return from_cuda(e);
        }
    }
    return MOE_OK;
}

// The one-kernel layer (fused.cu) on the forward's workspace layout.
moe_status_t forward_fused_impl(const uint16_t* x, const float* router_w, const float* router_bias,
                                const int8_t* w13_q, const float* w13_scale, const int8_t* w2_q,
                                const float* w2_scale, int64_t T, int64_t H, int64_t I, int64_t E, int64_t k,
                                uint16_t* y, void* workspace, size_t workspace_bytes, void* stream,
                                const moe_w8a8_debug_t* dbg) {
    if (!moe_shape_ok(T, H, I, E, k)) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (T == 0) return MOE_OK;
    if (!fused_supported(T, H, I, E, k)) return MOE_ERR_UNSUPPORTED_SHAPE;
    const void* ptrs[] = {x, router_w, w13_q, w13_scale, w2_q, w2_scale, y, workspace};
    for (const void* p : ptrs)
        if (p == nullptr || !aligned16(p) || injected(kInjectBadPtr)) return MOE_ERR_INVALID_ARG;
    if (router_bias != nullptr && !aligned16(router_bias)) return MOE_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return MOE_ERR_INVALID_ARG;
    const FwdLayout L = fwd_layout(T, H, I, E, k);
    if (injected(kInjectWsShort) && workspace_bytes >= L.total) workspace_bytes = L.total - 1;
    if (workspace_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int S = (int)(T * k);
    const RouterPlan rp = router_plan(T, H, E);
    FusedArgs a{};
    a.x = x;
    a.Wr = router_w;
    a.bias = router_bias;
    a.T = (int)T;
    a.H = (int)H;
    a.I = (int)I;
    a.E = (int)E;
    a.k = (int)k;
    a.E_pad = rp.E_pad;
    a.KS = rp.KS;
    a.hs = rp.hs;
    a.P = at<float>(workspace, L.logits);
    a.topk_ids = at<int32_t>(workspace, L.topk_ids);
    a.topk_w = at<float>(workspace, L.topk_w);
    a.rank = at<int32_t>(workspace, L.rank);
    a.hist = at<int32_t>(workspace, L.hist);
    a.offsets = at<int32_t>(workspace, L.offsets);
    a.counts = at<int32_t>(workspace, L.counts);
    a.error = at<int>(workspace, L.err);
    a.ticket = reinterpret_cast<unsigned int*>(reinterpret_cast<char*>(a.error) + kTicketOffset);
    a.bar = reinterpret_cast<unsigned int*>(reinterpret_cast<char*>(a.error) + kFusedCtlOffset);
    a.abort = reinterpret_cast<int*>(reinterpret_cast<char*>(a.error) + kFusedCtlOffset + 4);
    a.exits = reinterpret_cast<unsigned int*>(reinterpret_cast<char*>(a.error) + kFusedCtlOffset + 8);
    a.slot_of = at<int32_t>(workspace, L.slot_of);
    a.slot_token = at<int32_t>(workspace, L.slot_token);
    a.s_x = at<float>(workspace, L.s_x);
    a.s_slot = at<float>(workspace, L.s_slot);
    a.q_tok = at<int8_t>(workspace, L.q_x16);  // T * H bytes of the S * H * 2
    a.h = at<float>(workspace, L.h);
    a.s_h = at<float>(workspace, L.s_h);
    a.q_h = at<int8_t>(workspace, L.q_h16);
    a.o = at<float>(workspace, L.o);
    a.y = y;
    a.timeout_ns = g_timeout_ns.load();
    a.stall = injected(kInjectStall) ? 1 : 0;

    GemmArgs& g1 = a.g1;
    g1.sched = sched_words(a.error);
    g1.w = w13_q;
    g1.act8 = a.q_tok;
    g1.K = (int)H;
    g1.n_groups = (int)E;
    g1.total_rows = S;
    g1.offsets = a.offsets;
    g1.w_rows_per_group = (int)(2 * I);
    g1.up_offset = (int)I;
    g1.w_scale = w13_scale;
    g1.act_scale = a.s_slot;
    g1.out = a.h;
    g1.ld_out = (int)I;
    g1.acc_out = dbg ? dbg->acc1 : nullptr;
    g1.error = a.error;
    g1.timeout_ns = a.timeout_ns;
    GemmArgs& g2 = a.g2;
    g2.sched = g1.sched + 2;
    a.done1 = at<unsigned int>(workspace, L.fctl);
    a.ready2 = at<int>(workspace, L.fctl + E * 4);
    g2.w = w2_q;
    g2.act8 = a.q_h;
    g2.K = (int)I;
    g2.n_groups = (int)E;
    g2.total_rows = S;
    g2.offsets = a.offsets;
    g2.w_rows_per_group = (int)H;
    g2.w_scale = w2_scale;
    g2.act_scale = a.s_h;
    g2.out = a.o;
    g2.ld_out = (int)H;
    g2.acc_out = dbg ? dbg->acc2 : nullptr;
    g2.error = a.error;
    g2.timeout_ns = a.timeout_ns;

    cudaError_t e;
    if ((e = mark(0, st)) != cudaSuccess) return from_cuda(e);
    if ((e = launch_moe_fused(a, st)) != cudaSuccess) return from_cuda(e);
    if ((e = mark(1, st)) != cudaSuccess) return from_cuda(e);

    if (dbg) {
        auto cp = [&](void* dst, const void* src, size_t bytes) -> cudaError_t {
            if (!dst) return cudaSuccess;
            return cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToDevice, st);
        };
        const size_t Sb = (size_t)S * 4;
        if ((e = cp(dbg->topk_ids, a.topk_ids, Sb)) != cudaSuccess) return from_cuda(e);
        if ((e = cp(dbg->topk_w, a.topk_w, Sb)) != cudaSuccess) return from_cuda(e);
        if ((e = cp(dbg->offsets, a.offsets, (size_t)(E + 1) * 4)) != cudaSuccess) return from_cuda(e);
        if ((e = cp(dbg->slot_of, a.slot_of, Sb)) != cudaSuccess) return from_cuda(e);
        if ((e = cp(dbg->slot_token, a.slot_token, Sb)) != cudaSuccess) return from_cuda(e);
        if ((e = cp(dbg->s_x, a.s_x, (size_t)T * 4)) != cudaSuccess) return from_cuda(e);
        if ((e = cp(dbg->q_x, a.q_tok, (size_t)T * H)) != cudaSuccess) return from_cuda(e);
        if ((e = cp(dbg->h, a.h, (size_t)S * I * 4)) != cudaSuccess) return from_cuda(e);
        if ((e = cp(dbg->s_h, a.s_h, Sb)) != cudaSuccess) return from_cuda(e);
        if ((e = cp(dbg->q_h, a.q_h, (size_t)S * I)) != cudaSuccess) return from_cuda(e);
        if ((e = cp(dbg->o, a.o, (size_t)S * H * 4)) != cudaSuccess) return from_cuda(e);
        if ((e = cp(dbg->s_slot, a.s_slot, Sb)) != cudaSuccess) return from_cuda(e);
        if (dbg->q_slot) {  // every slot's row: its token's codes
            e = launch_s8_rows_gather(a.q_tok, a.slot_token, S, (int)H, 1, (int)T, dbg->q_slot, a.error, st);
            if (e != cudaSuccess) return from_cuda(e);
        }
    }
    return MOE_OK;
}

// Host-resident activations: x copied in and y copied out in token chunks on
// a copy stream, overlapping the layer's compute on another chunk.  Tokens
// are independent in the layer, so each chunk is a whole forward of its own
// tokens (routing, expert GEMMs and combine over just those tokens).
// Splitting re-reads the touched experts' weights once per chunk, so two
// chunks are taken only where one direction of the host link moves x more
// slowly than HBM streams all the expert weights once (kLinkHbmRatio: about
// 200 GB/s per direction of the host link against about 6.6 TB/s of HBM).
constexpr double kLinkHbmRatio = 32.0;
constexpr int64_t kMinChunkTokens = 1024;
constexpr int kMaxChunks = 16;

int auto_chunks(int64_t T, int64_t H, int64_t I, int64_t E) {
    const double x_bytes = (double)T * (double)H * 2.0;
    const double w_bytes = (double)E * 3.0 * (double)H * (double)I;
    return (T >= 2 * kMinChunkTokens && x_bytes * kLinkHbmRatio > w_bytes) ? 2 : 1;
}

// One event pool per host thread, created on first use and kept for the
// life of the process (the only CUDA objects the library creates).
cudaEvent_t* event_pool(int n) {
    thread_local std::vector<cudaEvent_t> pool;
    while ((int)pool.size() < n) {
        cudaEvent_t ev;
        if (cudaEventCreateWithFlags(&ev, cudaEventDisableTiming) != cudaSuccess) return nullptr;
        pool.push_back(ev);
    }
    return pool.data();
}

moe_status_t forward_host_impl(const uint16_t* x_host, const float* router_w, const float* router_bias,
                               const int8_t* w13_q, const float* w13_scale, const int8_t* w2_q,
                               const float* w2_scale, int64_t T, int64_t H, int64_t I, int64_t E, int64_t k,
                               uint16_t* y_host, uint16_t* x_dev, uint16_t* y_dev, void* workspace,
                               size_t workspace_bytes, void* stream, void* copy_stream, int chunks, bool fp8) {
    if (!moe_shape_ok(T, H, I, E, k)) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (T == 0) return MOE_OK;
    const void* ptrs[] = {x_host, y_host, x_dev, y_dev, router_w, w13_q, w13_scale, w2_q, w2_scale, workspace};
    for (const void* p : ptrs)
        if (p == nullptr || !aligned16(p) || injected(kInjectBadPtr)) return MOE_ERR_INVALID_ARG;
    if (router_bias != nullptr && !aligned16(router_bias)) return MOE_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return MOE_ERR_INVALID_ARG;
    if (chunks < 0 || chunks > kMaxChunks) return MOE_ERR_INVALID_ARG;
    const size_t need = fwd_layout(T, H, I, E, k).total;
    if (injected(kInjectWsShort) && workspace_bytes >= need) workspace_bytes = need - 1;
    if (workspace_bytes < need) return MOE_ERR_WORKSPACE_TOO_SMALL;
    if (fp8 && g_gemm_path.load() >= 0) return MOE_ERR_NOT_IMPLEMENTED;
    int n = chunks == 0 ? auto_chunks(T, H, I, E) : chunks;
    if (n > T) n = (int)T;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    cudaStream_t ps = copy_stream ? static_cast<cudaStream_t>(copy_stream) : cs;
    const bool two = ps != cs && n > 1;
    if (!two) ps = cs;  // one chunk (or one stream): nothing to overlap, everything in order on `stream`
    cudaEvent_t* ev = two ? event_pool(2 * n + 2) : nullptr;  // start, in[n], out[n], done
    if (two && ev == nullptr) return MOE_ERR_CUDA;
    cudaError_t e;
    auto chunk = [&](int c, int64_t& t0, int64_t& tc) {
        t0 = T * c / n;
        tc = T * (c + 1) / n - t0;
    };
    if (two) {  // the staging buffers are free of earlier work on the compute stream
        if ((e = cudaEventRecord(ev[0], cs)) != cudaSuccess) return from_cuda(e);
        if ((e = cudaStreamWaitEvent(ps, ev[0], 0)) != cudaSuccess) return from_cuda(e);
    }
    for (int c = 0; c < n; ++c) {  // every input copy first: they run while earlier chunks compute
        int64_t t0, tc;
        chunk(c, t0, tc);
        const size_t off = (size_t)t0 * H, bytes = (size_t)tc * H * 2;
        if ((e = cudaMemcpyAsync(x_dev + off, x_host + off, bytes, cudaMemcpyHostToDevice, ps)) != cudaSuccess)
            return from_cuda(e);
        if (two && (e = cudaEventRecord(ev[1 + c], ps)) != cudaSuccess) return from_cuda(e);
    }
    for (int c = 0; c < n; ++c) {
        int64_t t0, tc;
        chunk(c, t0, tc);
        const size_t off = (size_t)t0 * H, bytes = (size_t)tc * H * 2;
        if (two && (e = cudaStreamWaitEvent(cs, ev[1 + c], 0)) != cudaSuccess) return from_cuda(e);
        const moe_status_t r = forward_impl(x_dev + off, router_w, router_bias, w13_q, w13_scale, w2_q, w2_scale,
                                            tc, H, I, E, k, y_dev + off, workspace, workspace_bytes, stream,
                                            nullptr, fp8);
        if (r != MOE_OK) return r;
        if (two) {
            if ((e = cudaEventRecord(ev[1 + n + c], cs)) != cudaSuccess) return from_cuda(e);
            if ((e = cudaStreamWaitEvent(ps, ev[1 + n + c], 0)) != cudaSuccess) return from_cuda(e);
        }
        if ((e = cudaMemcpyAsync(y_host + off, y_dev + off, bytes, cudaMemcpyDeviceToHost, ps)) != cudaSuccess)
            return from_cuda(e);
    }
    if (two) {  // work queued on the compute stream after this call sees y complete
        if ((e = cudaEventRecord(ev[1 + 2 * n], ps)) != cudaSuccess) return from_cuda(e);
        if ((e = cudaStreamWaitEvent(cs, ev[1 + 2 * n], 0)) != cudaSuccess) return from_cuda(e);
    }
    return MOE_OK;
}

}  // namespace

extern "C" {

const char* moe_w8a8_status_string(moe_status_t s) {
    switch (s) {
        case MOE_OK: return "MOE_OK";
        case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
        case MOE_ERR_UNSUPPORTED_SHAPE: return "MOE_ERR_UNSUPPORTED_SHAPE";
        case MOE_ERR_WORKSPACE_TOO_SMALL: return "MOE_ERR_WORKSPACE_TOO_SMALL";
        case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
        case MOE_ERR_DEVICE_TIMEOUT: return "MOE_ERR_DEVICE_TIMEOUT";
        case MOE_ERR_NOT_IMPLEMENTED: return "MOE_ERR_NOT_IMPLEMENTED";
        case MOE_ERR_DEVICE: return "MOE_ERR_DEVICE";
    }
    return "MOE_ERR_UNKNOWN";
}

int moe_w8a8_version(void) { return 100; }

uint64_t moe_w8a8_set_wait_timeout_ns(uint64_t ns) {
    return g_timeout_ns.exchange(ns == 0 ? kDefaultTimeoutNs : ns);
}

int moe_w8a8_set_gemm_path(int path) {
    if (path < -1 || path > (int)GemmShape::Skinny) return -2;
    return g_gemm_path.exchange(path);
}

moe_status_t moe_w8a8_fp8_quantize_weights(const float* w, int64_t rows, int64_t K, uint8_t* w_q, float* w_scale,
                                           void* stream) {
    if (rows < 0 || K < 4 || K > (int64_t(1) << 20) || K % 4 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (rows == 0) return MOE_OK;
    if (!w || !w_q || !w_scale || !aligned16(w) || !aligned16(w_q) || !aligned16(w_scale) ||
        injected(kInjectBadPtr))
        return MOE_ERR_INVALID_ARG;
    if (injected(kInjectLaunchFail)) return MOE_ERR_CUDA;
    return from_cuda(
        launch_quantize_weights_fp8(w, rows, (int)K, w_q, w_scale, static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_w8a8_fp8_forward(const uint16_t* x, const float* router_w, const float* router_bias,
                                  const uint8_t* w13_q, const float* w13_scale, const uint8_t* w2_q,
                                  const float* w2_scale, int64_t T, int64_t H, int64_t I, int64_t E, int64_t top_k,
                                  uint16_t* y, void* workspace, size_t workspace_bytes, void* stream) {
    return forward_impl(x, router_w, router_bias, reinterpret_cast<const int8_t*>(w13_q), w13_scale,
                        reinterpret_cast<const int8_t*>(w2_q), w2_scale, T, H, I, E, top_k, y, workspace,
                        workspace_bytes, stream, nullptr, true);
}

moe_status_t moe_w8a8_fp8_forward_debug(const uint16_t* x, const float* router_w, const float* router_bias,
                                        const uint8_t* w13_q, const float* w13_scale, const uint8_t* w2_q,
                                        const float* w2_scale, int64_t T, int64_t H, int64_t I, int64_t E,
                                        int64_t top_k, uint16_t* y, void* workspace, size_t workspace_bytes,
                                        void* stream, const moe_w8a8_debug_t* dbg) {
    return forward_impl(x, router_w, router_bias, reinterpret_cast<const int8_t*>(w13_q), w13_scale,
                        reinterpret_cast<const int8_t*>(w2_q), w2_scale, T, H, I, E, top_k, y, workspace,
                        workspace_bytes, stream, dbg, true);
}

moe_status_t moe_w8a8_quantize_weights(const float* w, int64_t rows, int64_t K, int8_t* w_q,
                                       float* w_scale, void* stream) {
    if (rows < 0 || K < 1 || K > (int64_t(1) << 20)) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (rows == 0) return MOE_OK;
    if (!w || !w_q || !w_scale || !aligned16(w) || !aligned16(w_q) || !aligned16(w_scale) ||
        injected(kInjectBadPtr))
        return MOE_ERR_INVALID_ARG;
    if (injected(kInjectLaunchFail)) return MOE_ERR_CUDA;
    return from_cuda(launch_quantize_weights(w, rows, (int)K, w_q, w_scale, static_cast<cudaStream_t>(stream)));
}

size_t moe_w8a8_workspace_size(int64_t T, int64_t H, int64_t I, int64_t E, int64_t top_k) {
    if (!moe_shape_ok(T, H, I, E, top_k)) return 0;
    return fwd_layout(T, H, I, E, top_k).total;
}

moe_status_t moe_w8a8_forward(const uint16_t* x, const float* router_w, const float* router_bias,
                              const int8_t* w13_q, const float* w13_scale, const int8_t* w2_q,
                              const float* w2_scale, int64_t T, int64_t H, int64_t I, int64_t E,
                              int64_t top_k, uint16_t* y, void* workspace, size_t workspace_bytes,
                              void* stream) {
    return forward_impl(x, router_w, router_bias, w13_q, w13_scale, w2_q, w2_scale, T, H, I, E, top_k, y,
                        workspace, workspace_bytes, stream, nullptr);
}

moe_status_t moe_w8a8_forward_host(const uint16_t* x_host, const float* router_w, const float* router_bias,
                                   const int8_t* w13_q, const float* w13_scale, const int8_t* w2_q,
                                   const float* w2_scale, int64_t T, int64_t H, int64_t I, int64_t E, int64_t top_k,
                                   uint16_t* y_host, uint16_t* x_dev, uint16_t* y_dev, void* workspace,
                                   size_t workspace_bytes, void* stream, void* copy_stream, int chunks) {
    return forward_host_impl(x_host, router_w, router_bias, w13_q, w13_scale, w2_q, w2_scale, T, H, I, E, top_k,
                             y_host, x_dev, y_dev, workspace, workspace_bytes, stream, copy_stream, chunks, false);
}

moe_status_t moe_w8a8_fp8_forward_host(const uint16_t* x_host, const float* router_w, const float* router_bias,
                                       const uint8_t* w13_q, const float* w13_scale, const uint8_t* w2_q,
                                       const float* w2_scale, int64_t T, int64_t H, int64_t I, int64_t E,
                                       int64_t top_k, uint16_t* y_host, uint16_t* x_dev, uint16_t* y_dev,
                                       void* workspace, size_t workspace_bytes, void* stream, void* copy_stream,
                                       int chunks) {
    return forward_host_impl(x_host, router_w, router_bias, reinterpret_cast<const int8_t*>(w13_q), w13_scale,
                             reinterpret_cast<const int8_t*>(w2_q), w2_scale, T, H, I, E, top_k, y_host, x_dev,
                             y_dev, workspace, workspace_bytes, stream, copy_stream, chunks, true);
}

int moe_w8a8_host_chunks(int64_t T, int64_t H, int64_t I, int64_t E) {
    if (T < 0) return 0;
    return T == 0 ? 1 : auto_chunks(T, H, I, E);
}

moe_status_t moe_w8a8_quantize_weights_smoothed(const float* w, int64_t rows, int64_t K, const float* col_scale,
                                                int8_t* w_q, float* w_scale, void* stream) {
    if (rows < 0 || K < 1 || K > (int64_t(1) << 20)) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (rows == 0) return MOE_OK;
    if (!w || !col_scale || !w_q || !w_scale || !aligned16(w) || !aligned16(col_scale) || !aligned16(w_q) ||
        !aligned16(w_scale) || injected(kInjectBadPtr))
        return MOE_ERR_INVALID_ARG;
    if (injected(kInjectLaunchFail)) return MOE_ERR_CUDA;
    return from_cuda(
        launch_quantize_weights(w, rows, (int)K, w_q, w_scale, static_cast<cudaStream_t>(stream), col_scale));
}

moe_status_t moe_w8a8_forward_smooth(const uint16_t* x, const float* router_w, const float* router_bias,
                                     const float* smooth, const int8_t* w13_q, const float* w13_scale,
                                     const int8_t* w2_q, const float* w2_scale, int64_t T, int64_t H, int64_t I,
                                     int64_t E, int64_t top_k, uint16_t* y, void* workspace, size_t workspace_bytes,
                                     void* stream, const moe_w8a8_debug_t* dbg) {
    if (T > 0 && smooth == nullptr) return MOE_ERR_INVALID_ARG;
    return forward_impl(x, router_w, router_bias, w13_q, w13_scale, w2_q, w2_scale, T, H, I, E, top_k, y,
                        workspace, workspace_bytes, stream, dbg, false, smooth);
}

moe_status_t moe_w8a8_forward_debug(const uint16_t* x, const float* router_w,
                                    const float* router_bias, const int8_t* w13_q,
                                    const float* w13_scale, const int8_t* w2_q,
                                    const float* w2_scale, int64_t T, int64_t H, int64_t I,
                                    int64_t E, int64_t top_k, uint16_t* y, void* workspace,
                                    size_t workspace_bytes, void* stream,
                                    const moe_w8a8_debug_t* dbg) {
    return forward_impl(x, router_w, router_bias, w13_q, w13_scale, w2_q, w2_scale, T, H, I, E, top_k, y,
                        workspace, workspace_bytes, stream, dbg);
}

int moe_w8a8_fused_supported(int64_t T, int64_t H, int64_t I, int64_t E, int64_t top_k) {
    return moe_shape_ok(T, H, I, E, top_k) && fused_supported(T, H, I, E, top_k) ? 1 : 0;
}

moe_status_t moe_w8a8_forward_fused(const uint16_t* x, const float* router_w, const float* router_bias,
                                    const int8_t* w13_q, const float* w13_scale, const int8_t* w2_q,
                                    const float* w2_scale, int64_t T, int64_t H, int64_t I, int64_t E,
                                    int64_t top_k, uint16_t* y, void* workspace, size_t workspace_bytes,
                                    void* stream, const moe_w8a8_debug_t* dbg) {
    return forward_fused_impl(x, router_w, router_bias, w13_q, w13_scale, w2_q, w2_scale, T, H, I, E, top_k, y,
                              workspace, workspace_bytes, stream, dbg);
}

size_t moe_w8a8_linear_workspace_size(int64_t M, int64_t N, int64_t K) {
    if (M < 0 || M > (int64_t(1) << 20) || N < 128 || N > 65536 || N % 128 || K < 128 || K > 65536 || K % 128)
        return 0;
    return lin_layout(M, N, K).total;
}

moe_status_t moe_w8a8_linear(const uint16_t* x, const int8_t* w_q, const float* w_scale, int64_t M,
                             int64_t N, int64_t K, uint16_t* y, void* workspace,
                             size_t workspace_bytes, void* stream) {
    const size_t need = moe_w8a8_linear_workspace_size(M, N, K);
    if (need == 0) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (M == 0) return MOE_OK;  // nothing is read or written
    const void* ptrs[] = {x, w_q, w_scale, y, workspace};
    for (const void* p : ptrs)
        if (p == nullptr || !aligned16(p) || injected(kInjectBadPtr)) return MOE_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return MOE_ERR_INVALID_ARG;
    if (injected(kInjectWsShort) && workspace_bytes >= need) workspace_bytes = need - 1;
    if (workspace_bytes < need) return MOE_ERR_WORKSPACE_TOO_SMALL;
    // a faked launch failure is reported before the first CUDA call (the memset)
    if (injected(kInjectLaunchFail)) return MOE_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const LinLayout L = lin_layout(M, N, K);
    float* s_x = at<float>(workspace, L.s_x);
    int32_t* counts = at<int32_t>(workspace, L.counts);
    int32_t* flag = at<int32_t>(workspace, L.flag);
    int32_t* list = at<int32_t>(workspace, L.list);
    uint16_t* q16 = at<uint16_t>(workspace, L.q_x16);
    const GemmShape shape = pick_gemm_shape(M, 1, K, Epi::ScaleBF16, N, 0);
    int8_t* q8 = shape == GemmShape::Skinny ? reinterpret_cast<int8_t*>(q16) : nullptr;
    cudaError_t e;
    if ((e = mark(0, st)) != cudaSuccess) return from_cuda(e);
    if ((e = cudaMemsetAsync(counts, 0, 2 * sizeof(int32_t), st)) != cudaSuccess) return from_cuda(e);
    // the quantiser follows a memset: a plain launch; the GEMM may overlap its tail
    e = launch_permute_quant(x, nullptr, nullptr, nullptr, (int)M, (int)K, 1, 1, nullptr, nullptr, s_x, s_x,
                             q8 ? nullptr : q16, q8, flag, list, counts, at<int>(workspace, L.err), st, false);
    if (e != cudaSuccess) return from_cuda(e);
    if ((e = mark(1, st)) != cudaSuccess) return from_cuda(e);
    GemmArgs g{};
    g.w = w_q;
    g.act16 = q16;
    g.act8 = q8;
    g.K = (int)K;
    g.n_cb = (int)(N / 128);
    g.n_groups = 1;
    g.total_rows = (int)M;
    g.offsets = nullptr;
    g.w_rows_per_group = (int)N;
    g.w_scale = w_scale;
    g.act_scale = s_x;
    g.out = y;
    g.ld_out = (int)N;
    g.acc_out = nullptr;
    g.flags = flag;
    g.fb_list = list;
    g.fb_count = counts;
    g.error = at<int>(workspace, L.err);
    g.timeout_ns = g_timeout_ns.load();
    g.stall = injected(kInjectStall) ? 1 : 0;
    if ((e = launch_grouped_gemm(Epi::ScaleBF16, shape, g, st, pdl_default())) != cudaSuccess)
        return from_cuda(e);
    return from_cuda(mark(2, st));
}

uint64_t moe_w8a8_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

moe_status_t moe_w8a8_set_profile_events(void* const* events, int n) {
    if (events == nullptr) {
        t_events = nullptr;
        return MOE_OK;
    }
    if (n < 8) return MOE_ERR_INVALID_ARG;
    t_events = reinterpret_cast<cudaEvent_t const*>(events);
    return MOE_OK;
}

moe_status_t moe_w8a8_device_error(void* workspace, void* stream) {
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return MOE_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
    int host = 0;
    if (cudaMemcpy(&host, workspace, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
    if (host != 0) {
        const int zero = 0;
        if (cudaMemcpy(workspace, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return MOE_ERR_CUDA;
    }
    if (host & kErrTimeout) return MOE_ERR_DEVICE_TIMEOUT;
    if (host & kErrDevice) return MOE_ERR_DEVICE;
    return MOE_OK;
}

}  // extern "C"

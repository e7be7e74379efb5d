// static_linear.cu -- the W8A8 linear layer with its scratch memory in a
// static device array instead of a caller-provided workspace.
//
// Some callers cannot allocate device memory when they call the layer: for
// example a plugin whose host framework hands it no allocator, or a serving
// loop that reserved all device memory for its own pool at start-up, where a
// fresh cudaMalloc would fail or fragment that pool (and would synchronise
// the device).  This entry point gives them the linear layer with no
// allocation at all: its scratch (the error word, exact-path counters,
// per-token scales and flags, and the quantised activation codes) is the
// file-scope array below, which every GPU that loads this library holds
// until the process exits.
#include <mutex>

#include "internal.h"
#include "moe_w8a8.h"

namespace {

constexpr size_t kStaticScratchBytes = size_t(8) << 20;  // 8 MiB per device
static __device__ __align__(256) unsigned char g_linear_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the current device's copy of the scratch array.  In host
// code the array's name is only a host-side stand-in, so the address is
// looked up once per device, with that device current, and cached.  The
// cached address belongs to the device's primary context: it stays valid
// until that context is destroyed (cudaDeviceReset), after which this entry
// point must not be called again in the process.
cudaError_t scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_linear_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

using namespace moe;

extern "C" moe_status_t moe_w8a8_linear_static(const uint16_t* x, const int8_t* w_q, const float* w_scale,
                                                int64_t M, int64_t N, int64_t K, uint16_t* y, void* stream) {
    if (M < 0 || M > (int64_t(1) << 20) || N < 128 || N > 65536 || N % 128 || K < 128 || K > 65536 || K % 128)
        return MOE_ERR_UNSUPPORTED_SHAPE;
    if (M == 0) return MOE_OK;  // nothing is read or written
    const LinLayout L = lin_layout(M, N, K);
    if (L.total > kStaticScratchBytes) return MOE_ERR_UNSUPPORTED_SHAPE;  // beyond the static scratch
    const void* ptrs[] = {x, w_q, w_scale, y};
    for (const void* p : ptrs)
        if (p == nullptr || !aligned16(p) || injected(kInjectBadPtr)) return MOE_ERR_INVALID_ARG;
    if (injected(kInjectLaunchFail)) return MOE_ERR_CUDA;  // faked before any CUDA call

    void* scratch = nullptr;
    cudaError_t e = scratch_address(&scratch);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    char* base = static_cast<char*>(scratch);
    int* err = reinterpret_cast<int*>(base + L.err);
    int32_t* counts = reinterpret_cast<int32_t*>(base + L.counts);
    float* s_x = reinterpret_cast<float*>(base + L.s_x);
    int32_t* flag = reinterpret_cast<int32_t*>(base + L.flag);
    int32_t* list = reinterpret_cast<int32_t*>(base + L.list);
    uint16_t* q16 = reinterpret_cast<uint16_t*>(base + L.q_x16);
    const GemmShape shape = pick_gemm_shape(M, 1, K, Epi::ScaleBF16, N, 0);
    int8_t* q8 = shape == GemmShape::Skinny ? reinterpret_cast<int8_t*>(q16) : nullptr;

    // the scratch keeps the previous call's contents: clear the exact-path
    // counters, which must start at zero.  The error word (zero when the
    // library is loaded) is sticky: moe_w8a8_linear_static_error reads and
    // clears it.
    if (cudaMemsetAsync(counts, 0, 2 * sizeof(int32_t), st) != cudaSuccess) return MOE_ERR_CUDA;
    e = launch_permute_quant(x, nullptr, nullptr, nullptr, (int)M, (int)K, 1, 1, nullptr, nullptr, s_x, s_x,
                             q8 ? nullptr : q16, q8, flag, list, counts, err, st, false);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
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
    g.error = err;
    g.timeout_ns = current_timeout_ns();
    g.stall = injected(kInjectStall) ? 1 : 0;
    e = launch_grouped_gemm(Epi::ScaleBF16, shape, g, st, false);
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

extern "C" moe_status_t moe_w8a8_linear_static_error(void* stream) {
    void* scratch = nullptr;
    if (scratch_address(&scratch) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return MOE_ERR_CUDA;
    int* err = reinterpret_cast<int*>(static_cast<char*>(scratch) + lin_layout(0, 0, 0).err);
    int host = 0;
    if (cudaMemcpy(&host, err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
    if (host != 0) {
        const int zero = 0;
        if (cudaMemcpy(err, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return MOE_ERR_CUDA;
    }
    if (host & kErrTimeout) return MOE_ERR_DEVICE_TIMEOUT;
    if (host & kErrDevice) return MOE_ERR_DEVICE;
    return MOE_OK;
}

// qs_noalloc.cu -- the whole layer without a caller-supplied workspace.
//
// Some callers cannot allocate device memory at all: a plugin or operator
// hosted by a framework that owns every device allocation and hands over only
// the input and output buffers, or a serving loop under a fixed memory budget
// where a cudaMalloc (and the device-wide synchronisation it can imply) is not
// allowed once the loop runs.  qs_moe_ffn_noalloc gives them the layer with its
// scratch kept in a fixed array inside this library instead: the caller passes
// inputs and outputs only.
//
// The scratch is the exchange area of the decode kernels (the one-kernel paths
// of qs_moe_ffn; the same one runs here for the same call): the 256-byte header
// (sticky status word and the counters of the persistent kernel), the counter
// region of the cluster kernel, the routing record (ids, weights), and the
// exchanged fp32 arrays -- logits [T x E], the shared expert's hs [T x S], the
// routed h [T*k x F] (persistent kernel), the per-entry down products
// [T*k x H] and the shared down products [T x H] (cluster kernel) -- the same
// regions a workspace holds.  The counters are never reset: every call adds a
// fixed amount to each of them, and a call's targets follow from its exit
// counter, read once the previous grid has completed.  So the array needs
// zeroing only once, at set-up.  It is one array shared by every call on a
// device and it keeps the last call's contents; calls that overlap on the GPU
// (different streams, no ordering between them) race on it.
#include "qs_common.cuh"
#include "qs_internal.h"

#include <mutex>

static constexpr size_t kNoAllocScratchBytes = 4u << 20;  // 4 MiB, held on every GPU that loads the library

// In host code this name is only a stand-in for the symbol; its device address
// comes from cudaGetSymbolAddress below, once per device.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

namespace {

constexpr int kMaxDev = 64;
std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDev] = {};

inline size_t up256(size_t v) { return (v + 255) / 256 * 256; }

// Exchange-area layout for T tokens: header, counters, routing record, exchanged fp32 regions.
qs::WsLayout noalloc_layout(const qs_moe_shape& s, int T) {
    qs::WsLayout L;
    size_t o = 0;
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o += up256(bytes);
        return at;
    };
    const size_t tk = (size_t)T * s.top_k;
    L.header = take(qs::kHeaderBytes);
    L.cx = take(qs::kCxBytes);
    L.ids = take(tk * 4);
    L.pw = take(tk * 4);
    L.xlog = take((size_t)T * s.n_experts * 4);
    L.xhs = take((size_t)T * (s.shared_ffn > 0 ? s.shared_ffn : 1) * 4);
    L.xh = take(tk * s.expert_ffn * 4);
    L.cpd = take(tk * s.hidden * 4);
    L.csdp = take((size_t)T * s.hidden * 4);
    L.total = o;
    return L;
}

// The current device's index, checked against the table below.
cudaError_t current_device(int* dev) {
    cudaError_t e = cudaGetDevice(dev);
    if (e != cudaSuccess) return e;
    return (*dev < 0 || *dev >= kMaxDev) ? cudaErrorInvalidDevice : cudaSuccess;
}

// Device address of the scratch array on the current device.  The first call on
// a device looks the address up and zeroes the array (so the status word, the
// exchange counters and the exit counter start at 0); later calls reuse it.
cudaError_t scratch_for_current_device(void** out, cudaStream_t st) {
    int dev = 0;
    cudaError_t e = current_device(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        e = cudaMemsetAsync(p, 0, kNoAllocScratchBytes, st);
        if (e != cudaSuccess) return e;
        e = cudaStreamSynchronize(st);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" int qs_moe_ffn_noalloc(const qs_moe_shape* shape, const void* x, const float* router_w,
                                  const float* router_bias, const qs_q2k_experts* experts,
                                  const qs_shared_expert* shared, float* out, int n_tokens, void* stream) {
    if (!shape || !x || !router_w || !out || !experts || !experts->blocks || n_tokens < 1) return QS_ERR_INVALID;
    if (qs_moe_workspace_bytes(shape, n_tokens) == 0) return QS_ERR_INVALID;  // shape checks of the ABI
    if (((uintptr_t)x & 15u) || ((uintptr_t)router_w & 15u) || ((uintptr_t)experts->blocks & 15u)) return QS_ERR_INVALID;
    const int64_t need = 84ll * (2ll * shape->expert_ffn * shape->hidden + (int64_t)shape->hidden * shape->expert_ffn) / 256;
    if (experts->expert_stride < need || experts->expert_stride % 16) return QS_ERR_INVALID;
    const bool has_shared = shape->shared_ffn > 0 && shared != nullptr;
    if (has_shared && (!shared->w_gate || !shared->w_up || !shared->w_down || !shared->w_gate_sig ||
                       ((uintptr_t)shared->w_gate & 15u) || ((uintptr_t)shared->w_up & 15u) ||
                       ((uintptr_t)shared->w_down & 15u) || ((uintptr_t)shared->w_gate_sig & 15u)))
        return QS_ERR_INVALID;
    qs_moe_shape eff = *shape;
    if (!has_shared) eff.shared_ffn = 0;
    // this entry point runs only the persistent decode kernel, whose exchange area must fit the array
    if (n_tokens > qs::kFusedMaxT) return QS_ERR_UNSUPPORTED;
    const qs::WsLayout L = noalloc_layout(eff, n_tokens);
    if (L.total > kNoAllocScratchBytes) return QS_ERR_WORKSPACE;
    // the kernel qs_moe_ffn would run for this call: one of the two one-kernel decode paths
    cudaError_t e;
    const bool cluster = qs::cluster_decode_supported(eff, n_tokens, &e);
    if (e != cudaSuccess) return qs::cuda_fail(e);
    if (!cluster && !qs::fused_decode_supported(eff, n_tokens, &e))
        return e == cudaSuccess ? QS_ERR_UNSUPPORTED : qs::cuda_fail(e);
    if (e != cudaSuccess) return qs::cuda_fail(e);
    void* scratch = nullptr;
    e = scratch_for_current_device(&scratch, (cudaStream_t)stream);
    if (e != cudaSuccess) return qs::cuda_fail(e);
    const uint8_t* blocks = static_cast<const uint8_t*>(experts->blocks);
    const uint16_t* wg = has_shared ? (const uint16_t*)shared->w_gate : nullptr;
    const uint16_t* wu = has_shared ? (const uint16_t*)shared->w_up : nullptr;
    const uint16_t* wd = has_shared ? (const uint16_t*)shared->w_down : nullptr;
    const uint16_t* wsig = has_shared ? (const uint16_t*)shared->w_gate_sig : nullptr;
    e = qs::launch_decode_kernel(eff, x, router_w, router_bias, blocks, experts->expert_stride, wg, wu, wd, wsig,
                                 n_tokens, out, scratch, L, (cudaStream_t)stream, false);
    if (e == cudaErrorNotSupported) return QS_ERR_UNSUPPORTED;
    return e == cudaSuccess ? QS_OK : qs::cuda_fail(e);
}

extern "C" int qs_noalloc_read_device_status(void* stream) {
    int dev = 0;
    cudaError_t e = current_device(&dev);
    if (e != cudaSuccess) return qs::cuda_fail(e);
    void* p = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_setup_mutex);
        p = g_scratch_ptr[dev];
    }
    e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return qs::cuda_fail(e);
    if (p == nullptr) return QS_OK;  // no call has run on this device
    uint32_t st = 0;
    e = cudaMemcpy(&st, p, sizeof(st), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return qs::cuda_fail(e);
    if (st != 0) {  // clear the status word only; the counters stay consistent across a time-out
        const uint32_t zero = 0;
        e = cudaMemcpy(p, &zero, sizeof(zero), cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return qs::cuda_fail(e);
    }
    return (int)st;
}

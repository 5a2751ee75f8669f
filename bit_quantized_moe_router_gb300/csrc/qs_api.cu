// qs_api.cu -- the C ABI of the Q2_K MoE-FFN library: argument checks,
// workspace layout and the order in which each entry point's kernels run.
#include "qs_common.cuh"
#include "qs_internal.h"

#include <algorithm>

namespace qs {

static thread_local int g_last_cuda_error = 0;

int cuda_fail(cudaError_t e) {
    g_last_cuda_error = (int)e;
    return QS_ERR_CUDA;
}

static inline size_t up256(size_t v) { return (v + 255) / 256 * 256; }
static inline bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

WsLayout ws_layout(const qs_moe_shape& s, int T) {
    WsLayout L;
    size_t o = 0;
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o += up256(bytes);
        return at;
    };
    const size_t E = (size_t)s.n_experts, k = (size_t)s.top_k, F = (size_t)s.expert_ffn, S = (size_t)s.shared_ffn;
    const size_t t = (size_t)std::max(T, 1);
    L.header = take(kHeaderBytes);
    L.logits = take(t * E * 4);
    L.ids = take(t * k * 4);
    L.pw = take(t * k * 4);
    L.counts = take(E * 4);
    L.offsets = take((E + 1) * 4);
    L.perm = take(t * k * 4);
    L.h = take(t * k * F * 4);
    L.hs = take(t * std::max<size_t>(S, 1) * 4);
    L.gate = take(t * 4);
    L.tickets = take((t + kRouteTok - 1) / kRouteTok * 4);
    const size_t tf = std::min<size_t>(t, kFusedMaxT);
    L.xlog = take(tf * E * 4);
    L.xhs = take(tf * std::max<size_t>(S, 1) * 4);
    L.xh = take(tf * k * F * 4);
    const size_t H = (size_t)s.hidden;
    const size_t tc = std::min<size_t>(t, kClusterMaxT);
    L.cx = take(kCxBytes);
    L.cpd = take(tc * k * H * 4);
    L.csdp = take(tc * H * 4);
    L.wr3 = take(3 * E * H * 2);
    L.lpart = take((size_t)kPrefillMaxKS * t * E * 4);
    L.xs = take(t * k * H * 2);
    L.cursor = take(E * 4);
    L.h16 = take(t * k * F * 2);
    L.hs16 = take(t * std::max<size_t>(S, 1) * 2);
    L.total = o;
    return L;
}

static bool shape_ok(const qs_moe_shape* s) {
    if (!s) return false;
    if (s->hidden <= 0 || s->hidden % 256 || s->hidden > 8192) return false;
    if (s->expert_ffn <= 0 || s->expert_ffn % 256 || s->expert_ffn > 8192) return false;
    if (s->shared_ffn < 0 || s->shared_ffn % 256 || s->shared_ffn > 65536) return false;
    if (s->n_experts < 1 || s->n_experts > 1024) return false;
    if (s->top_k < 1 || s->top_k > s->n_experts || s->top_k > 32) return false;
    if (s->x_dtype != QS_F32 && s->x_dtype != QS_BF16) return false;
    return true;
}

static bool experts_ok(const qs_moe_shape* s, const qs_q2k_experts* ex) {
    if (!ex || !ex->blocks || !aligned16(ex->blocks)) return false;
    const int64_t need = 84ll * (2ll * s->expert_ffn * s->hidden + (int64_t)s->hidden * s->expert_ffn) / 256;
    return ex->expert_stride >= need && ex->expert_stride % 16 == 0;
}

static bool shared_ok(const qs_moe_shape* s, const qs_shared_expert* sh) {
    if (s->shared_ffn == 0) return true;
    return sh && sh->w_gate && sh->w_up && sh->w_down && sh->w_gate_sig && aligned16(sh->w_gate) &&
           aligned16(sh->w_up) && aligned16(sh->w_down) && aligned16(sh->w_gate_sig);
}

template <class T>
static T* ws_at(void* ws, size_t off) {
    return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

// Which one-kernel decode path a call tries first.  Both give the layer within its tolerance.
// Measured side by side on one GB300 (35B-A3B layer, 1 to 8 tokens; H=4096 layer, 1 token),
// the persistent kernel -- whose 152 CTAs all take routed rows -- is the faster at every token
// count, so it goes first; the cluster kernel takes the calls the persistent kernel's plan
// does not.
static bool prefer_cluster(const qs_moe_shape& s, int T) {
    (void)s;
    (void)T;
    return false;
}

cudaError_t launch_decode_kernel(const qs_moe_shape& s, const void* x, const float* Wr, const float* bias,
                                 const uint8_t* experts, int64_t stride, const uint16_t* sg, const uint16_t* su,
                                 const uint16_t* sd, const uint16_t* ssig, int T, float* out, void* ws,
                                 const WsLayout& W, cudaStream_t st, bool x_host_mapped) {
    const bool cluster_first = prefer_cluster(s, T);
    for (int pass = 0; pass < 2; pass++) {
        const bool cluster = (pass == 0) == cluster_first;
        const cudaError_t e =
            cluster ? launch_cluster_decode(s, x, Wr, bias, experts, stride, sg, su, sd, ssig, T, out, ws, W, st,
                                            x_host_mapped)
                    : launch_fused_decode(s, x, Wr, bias, experts, stride, sg, su, sd, ssig, T, out, ws, W, st,
                                          x_host_mapped);
        if (e != cudaErrorNotSupported) return e;
    }
    return cudaErrorNotSupported;
}

}  // namespace qs

using namespace qs;

extern "C" {

const char* qs_status_string(int status) {
    switch (status) {
        case QS_OK: return "ok";
        case QS_ERR_INVALID: return "invalid argument";
        case QS_ERR_CUDA: return "CUDA error";
        case QS_ERR_TIMEOUT: return "device-side wait timed out";
        case QS_ERR_UNSUPPORTED: return "unsupported request";
        case QS_ERR_WORKSPACE: return "workspace missing or too small";
        default: return "unknown status";
    }
}

int qs_abi_version(void) { return QS_ABI_VERSION; }

int qs_last_cuda_error(void) { return g_last_cuda_error; }

size_t qs_moe_workspace_bytes(const qs_moe_shape* shape, int max_tokens) {
    if (!shape_ok(shape) || max_tokens < 1) return 0;
    return ws_layout(*shape, max_tokens).total;
}

// Host-buffer variant: the layer's workspace, then x's device copy, then out's device copy.
static size_t host_x_bytes(const qs_moe_shape& s, int T) {
    return (size_t)T * s.hidden * (s.x_dtype == QS_BF16 ? 2 : 4);
}

size_t qs_moe_host_workspace_bytes(const qs_moe_shape* shape, int max_tokens) {
    if (!shape_ok(shape) || max_tokens < 1) return 0;
    return ws_layout(*shape, max_tokens).total + up256(host_x_bytes(*shape, max_tokens)) +
           up256((size_t)max_tokens * shape->hidden * 4);
}

int qs_workspace_init(void* workspace, size_t workspace_bytes, void* stream) {
    if (!workspace || workspace_bytes < (size_t)kHeaderBytes || ((uintptr_t)workspace & 255u)) return QS_ERR_WORKSPACE;
    cudaError_t e = cudaMemsetAsync(workspace, 0, workspace_bytes, (cudaStream_t)stream);
    return e == cudaSuccess ? QS_OK : cuda_fail(e);
}

int qs_read_device_status(const void* workspace, void* stream) {
    if (!workspace) return QS_ERR_WORKSPACE;
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e);
    uint32_t st = 0;
    e = cudaMemcpy(&st, workspace, sizeof(st), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e);
    return (int)st;
}

static int check_ws(const qs_moe_shape* s, int T, void* ws, size_t bytes) {
    if (!ws || ((uintptr_t)ws & 255u)) return QS_ERR_WORKSPACE;
    if (bytes < ws_layout(*s, T).total) return QS_ERR_WORKSPACE;
    return QS_OK;
}

int qs_route_topk(const qs_moe_shape* shape, const void* x, const float* router_w, const float* router_bias,
                  int n_tokens, int32_t* topk_ids, float* topk_w, void* workspace, size_t workspace_bytes,
                  void* stream) {
    if (!shape_ok(shape) || !x || !router_w || !topk_ids || !topk_w || n_tokens < 1) return QS_ERR_INVALID;
    if (!aligned16(x) || !aligned16(router_w)) return QS_ERR_INVALID;
    if (int rc = check_ws(shape, n_tokens, workspace, workspace_bytes)) return rc;
    const WsLayout L = ws_layout(*shape, n_tokens);
    cudaError_t e = launch_route(*shape, x, router_w, router_bias, n_tokens, ws_at<float>(workspace, L.logits),
                                 topk_ids, topk_w, ws_at<uint32_t>(workspace, L.tickets), (cudaStream_t)stream);
    return e == cudaSuccess ? QS_OK : cuda_fail(e);
}

int qs_group_tokens(const qs_moe_shape* shape, const int32_t* topk_ids, int n_tokens, int32_t* counts,
                    int32_t* offsets, int32_t* perm, void* stream) {
    if (!shape_ok(shape) || !topk_ids || !counts || !offsets || !perm || n_tokens < 1) return QS_ERR_INVALID;
    if ((int64_t)n_tokens * shape->top_k > (1ll << 30)) return QS_ERR_INVALID;
    cudaError_t e = launch_group(shape->n_experts, shape->top_k, n_tokens, topk_ids, counts, offsets, perm,
                                 (cudaStream_t)stream);
    return e == cudaSuccess ? QS_OK : cuda_fail(e);
}

int qs_q2k_gemv_grouped(const qs_moe_shape* shape, const void* x, const qs_q2k_experts* experts,
                        const int32_t* offsets, const int32_t* perm, int n_tokens, float* h_out, void* stream) {
    if (!shape_ok(shape) || !x || !offsets || !perm || !h_out || n_tokens < 1) return QS_ERR_INVALID;
    if (!experts_ok(shape, experts)) return QS_ERR_INVALID;
    cudaError_t e = launch_gateup(*shape, x, static_cast<const uint8_t*>(experts->blocks), experts->expert_stride,
                                  offsets, perm, n_tokens, h_out, (cudaStream_t)stream);
    return e == cudaSuccess ? QS_OK : cuda_fail(e);
}

int qs_q2k_down_combine(const qs_moe_shape* shape, const qs_q2k_experts* experts, const float* h,
                        const int32_t* topk_ids, const float* topk_w, int n_tokens, float* out, int accumulate,
                        void* stream) {
    if (!shape_ok(shape) || !h || !topk_ids || !topk_w || !out || n_tokens < 1) return QS_ERR_INVALID;
    if (!experts_ok(shape, experts) || !aligned16(h)) return QS_ERR_INVALID;
    cudaError_t e = launch_down(*shape, static_cast<const uint8_t*>(experts->blocks), experts->expert_stride, h,
                                topk_ids, topk_w, shape->top_k, nullptr, nullptr, nullptr, n_tokens, out, accumulate,
                                (cudaStream_t)stream);
    return e == cudaSuccess ? QS_OK : cuda_fail(e);
}

int qs_shared_expert_ffn(const qs_moe_shape* shape, const void* x, const qs_shared_expert* shared, int n_tokens,
                         float* out, int accumulate, void* workspace, size_t workspace_bytes, void* stream) {
    if (!shape_ok(shape) || !x || !out || n_tokens < 1 || shape->shared_ffn == 0) return QS_ERR_INVALID;
    if (!aligned16(x) || !shared_ok(shape, shared)) return QS_ERR_INVALID;
    if (int rc = check_ws(shape, n_tokens, workspace, workspace_bytes)) return rc;
    const WsLayout L = ws_layout(*shape, n_tokens);
    cudaStream_t st = (cudaStream_t)stream;
    float* hs = ws_at<float>(workspace, L.hs);
    float* gate = ws_at<float>(workspace, L.gate);
    cudaError_t e = launch_shared_gateup(*shape, x, (const uint16_t*)shared->w_gate, (const uint16_t*)shared->w_up,
                                         (const uint16_t*)shared->w_gate_sig, n_tokens, hs, gate, st);
    if (e != cudaSuccess) return cuda_fail(e);
    e = launch_down(*shape, nullptr, 0, nullptr, nullptr, nullptr, 0, (const uint16_t*)shared->w_down, hs, gate,
                    n_tokens, out, accumulate, st);
    return e == cudaSuccess ? QS_OK : cuda_fail(e);
}

int qs_moe_ffn(const qs_moe_shape* shape, const void* x, const float* router_w, const float* router_bias,
               const qs_q2k_experts* experts, const qs_shared_expert* shared, float* out, int n_tokens,
               void* workspace, size_t workspace_bytes, void* stream) {
    if (!shape_ok(shape) || !x || !router_w || !out || n_tokens < 1) return QS_ERR_INVALID;
    if (!aligned16(x) || !aligned16(router_w) || !experts_ok(shape, experts)) return QS_ERR_INVALID;
    const bool has_shared = shape->shared_ffn > 0 && shared != nullptr;
    if (shape->shared_ffn > 0 && shared != nullptr && !shared_ok(shape, shared)) return QS_ERR_INVALID;
    if (int rc = check_ws(shape, n_tokens, workspace, workspace_bytes)) return rc;
    const WsLayout L = ws_layout(*shape, n_tokens);
    cudaStream_t st = (cudaStream_t)stream;
    const uint8_t* blocks = static_cast<const uint8_t*>(experts->blocks);
    float* hs = ws_at<float>(workspace, L.hs);
    float* gate = ws_at<float>(workspace, L.gate);
    int32_t* ids = ws_at<int32_t>(workspace, L.ids);
    float* pw = ws_at<float>(workspace, L.pw);
    cudaError_t e;
    {
        qs_moe_shape eff = *shape;
        if (!has_shared) eff.shared_ffn = 0;
        e = launch_decode_kernel(eff, x, router_w, router_bias, blocks, experts->expert_stride,
                                 has_shared ? (const uint16_t*)shared->w_gate : nullptr,
                                 has_shared ? (const uint16_t*)shared->w_up : nullptr,
                                 has_shared ? (const uint16_t*)shared->w_down : nullptr,
                                 has_shared ? (const uint16_t*)shared->w_gate_sig : nullptr, n_tokens, out, workspace, L,
                                 st, false);
        if (e == cudaSuccess) return QS_OK;
        if (e != cudaErrorNotSupported) return cuda_fail(e);
        e = launch_prefill(eff, x, router_w, router_bias, blocks, experts->expert_stride,
                           has_shared ? (const uint16_t*)shared->w_gate : nullptr,
                           has_shared ? (const uint16_t*)shared->w_up : nullptr,
                           has_shared ? (const uint16_t*)shared->w_down : nullptr,
                           has_shared ? (const uint16_t*)shared->w_gate_sig : nullptr, n_tokens, out, workspace, L, st);
        if (e == cudaSuccess) return QS_OK;
        if (e != cudaErrorNotSupported) return cuda_fail(e);
    }
    if (has_shared) {
        e = launch_shared_gateup(*shape, x, (const uint16_t*)shared->w_gate, (const uint16_t*)shared->w_up,
                                 (const uint16_t*)shared->w_gate_sig, n_tokens, hs, gate, st);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    e = launch_route(*shape, x, router_w, router_bias, n_tokens, ws_at<float>(workspace, L.logits), ids, pw,
                     ws_at<uint32_t>(workspace, L.tickets), st);
    if (e != cudaSuccess) return cuda_fail(e);
    e = launch_group(shape->n_experts, shape->top_k, n_tokens, ids, ws_at<int32_t>(workspace, L.counts),
                     ws_at<int32_t>(workspace, L.offsets), ws_at<int32_t>(workspace, L.perm), st);
    if (e != cudaSuccess) return cuda_fail(e);
    e = launch_gateup(*shape, x, blocks, experts->expert_stride, ws_at<int32_t>(workspace, L.offsets),
                      ws_at<int32_t>(workspace, L.perm), n_tokens, ws_at<float>(workspace, L.h), st);
    if (e != cudaSuccess) return cuda_fail(e);
    e = launch_down(*shape, blocks, experts->expert_stride, ws_at<float>(workspace, L.h), ids, pw, shape->top_k,
                    has_shared ? (const uint16_t*)shared->w_down : nullptr, hs, gate, n_tokens, out, 0, st);
    return e == cudaSuccess ? QS_OK : cuda_fail(e);
}

// Device address of pinned (page-locked, mapped) host memory, or nullptr for any other pointer.
static void* mapped_host(const void* p) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return nullptr;
    }
    return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

int qs_moe_ffn_cluster(const qs_moe_shape* shape, const void* x, const float* router_w, const float* router_bias,
                       const qs_q2k_experts* experts, const qs_shared_expert* shared, float* out, int n_tokens,
                       void* workspace, size_t workspace_bytes, void* stream) {
    if (!shape_ok(shape) || !x || !router_w || !out || n_tokens < 1) return QS_ERR_INVALID;
    if (!aligned16(x) || !aligned16(router_w) || !experts_ok(shape, experts)) return QS_ERR_INVALID;
    const bool has_shared = shape->shared_ffn > 0 && shared != nullptr;
    if (has_shared && !shared_ok(shape, shared)) return QS_ERR_INVALID;
    if (int rc = check_ws(shape, n_tokens, workspace, workspace_bytes)) return rc;
    qs_moe_shape eff = *shape;
    if (!has_shared) eff.shared_ffn = 0;
    const WsLayout L = ws_layout(*shape, n_tokens);
    const cudaError_t e = launch_cluster_decode(
        eff, x, router_w, router_bias, static_cast<const uint8_t*>(experts->blocks), experts->expert_stride,
        has_shared ? (const uint16_t*)shared->w_gate : nullptr, has_shared ? (const uint16_t*)shared->w_up : nullptr,
        has_shared ? (const uint16_t*)shared->w_down : nullptr,
        has_shared ? (const uint16_t*)shared->w_gate_sig : nullptr, n_tokens, out, workspace, L, (cudaStream_t)stream);
    if (e == cudaErrorNotSupported) return QS_ERR_UNSUPPORTED;
    return e == cudaSuccess ? QS_OK : cuda_fail(e);
}

int qs_moe_ffn_host(const qs_moe_shape* shape, const void* x_host, const float* router_w, const float* router_bias,
                    const qs_q2k_experts* experts, const qs_shared_expert* shared, float* out_host, int n_tokens,
                    void* workspace, size_t workspace_bytes, void* stream) {
    if (!shape_ok(shape) || !x_host || !out_host || n_tokens < 1) return QS_ERR_INVALID;
    if (!workspace || ((uintptr_t)workspace & 255u)) return QS_ERR_WORKSPACE;
    if (workspace_bytes < qs_moe_host_workspace_bytes(shape, n_tokens)) return QS_ERR_WORKSPACE;
    {
        // pinned x and out, a call a one-kernel decode path takes: it reads x and writes out
        // through their mapped addresses (no copies queued around it)
        void* xd = aligned16(x_host) ? mapped_host(x_host) : nullptr;
        void* od = xd && aligned16(out_host) ? mapped_host(out_host) : nullptr;
        const bool has_shared = shape->shared_ffn > 0 && shared != nullptr;
        if (od && router_w && aligned16(router_w) && experts_ok(shape, experts) &&
            (!has_shared || shared_ok(shape, shared))) {
            qs_moe_shape eff = *shape;
            if (!has_shared) eff.shared_ffn = 0;
            const WsLayout L = ws_layout(*shape, n_tokens);
            cudaError_t e = launch_decode_kernel(
                eff, xd, router_w, router_bias, static_cast<const uint8_t*>(experts->blocks), experts->expert_stride,
                has_shared ? (const uint16_t*)shared->w_gate : nullptr, has_shared ? (const uint16_t*)shared->w_up : nullptr,
                has_shared ? (const uint16_t*)shared->w_down : nullptr,
                has_shared ? (const uint16_t*)shared->w_gate_sig : nullptr, n_tokens, static_cast<float*>(od), workspace,
                L, (cudaStream_t)stream, true);
            if (e == cudaSuccess) return QS_OK;
            if (e != cudaErrorNotSupported) return cuda_fail(e);
        }
    }
    const size_t ws_bytes = ws_layout(*shape, n_tokens).total;
    const size_t xb = host_x_bytes(*shape, n_tokens);
    uint8_t* x_dev = static_cast<uint8_t*>(workspace) + ws_bytes;
    float* out_dev = reinterpret_cast<float*>(x_dev + up256(xb));
    cudaStream_t st = (cudaStream_t)stream;
    cudaError_t e = cudaMemcpyAsync(x_dev, x_host, xb, cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) return cuda_fail(e);
    const int rc = qs_moe_ffn(shape, x_dev, router_w, router_bias, experts, shared, out_dev, n_tokens, workspace,
                              ws_bytes, stream);
    if (rc != QS_OK) return rc;
    e = cudaMemcpyAsync(out_host, out_dev, (size_t)n_tokens * shape->hidden * 4, cudaMemcpyDeviceToHost, st);
    return e == cudaSuccess ? QS_OK : cuda_fail(e);
}

int qs_read_routing(const qs_moe_shape* shape, int n_tokens, const void* workspace, size_t workspace_bytes,
                    int32_t* ids_host, float* w_host, void* stream) {
    if (!shape_ok(shape) || n_tokens < 1 || !ids_host || !w_host) return QS_ERR_INVALID;
    if (int rc = check_ws(shape, n_tokens, const_cast<void*>(workspace), workspace_bytes)) return rc;
    const WsLayout L = ws_layout(*shape, n_tokens);
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e);
    const size_t n = (size_t)n_tokens * shape->top_k;
    const uint8_t* base = static_cast<const uint8_t*>(workspace);
    e = cudaMemcpy(ids_host, base + L.ids, n * sizeof(int32_t), cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaMemcpy(w_host, base + L.pw, n * sizeof(float), cudaMemcpyDeviceToHost);
    return e == cudaSuccess ? QS_OK : cuda_fail(e);
}

int qs_moe_ffn_launches(const qs_moe_shape* shape, int n_tokens, int has_shared) {
    if (!shape_ok(shape) || n_tokens < 1) return 0;
    qs_moe_shape eff = *shape;
    if (!has_shared) eff.shared_ffn = 0;
    cudaError_t e;
    if (cluster_decode_supported(eff, n_tokens, &e)) return 1;
    if (e != cudaSuccess) return -(int)e;
    if (fused_decode_supported(eff, n_tokens, &e)) return 1;
    if (e != cudaSuccess) return -(int)e;
    if (prefill_shape_ok(eff)) return prefill_launches();
    return eff.shared_ffn > 0 ? 5 : 4;
}

int qs_moe_ffn_q4k_launches(const qs_moe_shape* shape, int n_tokens, int has_shared) {
    if (!shape_ok(shape) || n_tokens < 1) return 0;
    qs_moe_shape eff = *shape;
    if (!has_shared) eff.shared_ffn = 0;
    cudaError_t e;
    if (fused_decode_supported(eff, n_tokens, &e)) return 1;
    if (e != cudaSuccess) return -(int)e;
    return eff.shared_ffn > 0 ? 6 : 4;
}

int qs_q2k_quantize(const float* w, int64_t n_rows, int64_t K, void* out, void* stream) {
    if (!w || !out || n_rows < 1 || K < 256 || K % 256 || !aligned16(w) || ((uintptr_t)out & 3u))
        return QS_ERR_INVALID;
    cudaError_t e = launch_quantize(w, n_rows * (K / 256), static_cast<uint8_t*>(out), (cudaStream_t)stream);
    return e == cudaSuccess ? QS_OK : cuda_fail(e);
}

int qs_moe_ffn_q4k(const qs_moe_shape* shape, const void* x, const float* router_w, const float* router_bias,
                   const qs_q4k_experts* experts, const qs_shared_expert* shared, float* out, int n_tokens,
                   void* workspace, size_t workspace_bytes, void* stream) {
    if (!shape_ok(shape) || !x || !router_w || !out || n_tokens < 1) return QS_ERR_INVALID;
    if (!aligned16(x) || !aligned16(router_w)) return QS_ERR_INVALID;
    if (!experts || !experts->blocks || !aligned16(experts->blocks)) return QS_ERR_INVALID;
    const int64_t need = 144ll * 3ll * shape->expert_ffn * shape->hidden / 256;
    if (experts->expert_stride < need || experts->expert_stride % 16) return QS_ERR_INVALID;
    const bool has_shared = shape->shared_ffn > 0 && shared != nullptr;
    if (has_shared && !shared_ok(shape, shared)) return QS_ERR_INVALID;
    if (q4k_down_smem(shape->top_k, shape->expert_ffn) > 200 * 1024) return QS_ERR_UNSUPPORTED;
    if (int rc = check_ws(shape, n_tokens, workspace, workspace_bytes)) return rc;
    const WsLayout L = ws_layout(*shape, n_tokens);
    cudaStream_t st = (cudaStream_t)stream;
    const uint8_t* blocks = static_cast<const uint8_t*>(experts->blocks);
    float* hs = ws_at<float>(workspace, L.hs);
    float* gate = ws_at<float>(workspace, L.gate);
    int32_t* ids = ws_at<int32_t>(workspace, L.ids);
    float* pw = ws_at<float>(workspace, L.pw);
    cudaError_t e;
    {  // one kernel (the persistent decode kernel with Q4_K routed rows) where it plans the call
        qs_moe_shape eff = *shape;
        if (!has_shared) eff.shared_ffn = 0;
        e = launch_fused_decode(eff, x, router_w, router_bias, blocks, experts->expert_stride,
                                has_shared ? (const uint16_t*)shared->w_gate : nullptr,
                                has_shared ? (const uint16_t*)shared->w_up : nullptr,
                                has_shared ? (const uint16_t*)shared->w_down : nullptr,
                                has_shared ? (const uint16_t*)shared->w_gate_sig : nullptr, n_tokens, out, workspace, L,
                                st, false, 1);
        if (e == cudaSuccess) return QS_OK;
        if (e != cudaErrorNotSupported) return cuda_fail(e);
    }
    if (has_shared) {
        e = launch_shared_gateup(*shape, x, (const uint16_t*)shared->w_gate, (const uint16_t*)shared->w_up,
                                 (const uint16_t*)shared->w_gate_sig, n_tokens, hs, gate, st);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    e = launch_route(*shape, x, router_w, router_bias, n_tokens, ws_at<float>(workspace, L.logits), ids, pw,
                     ws_at<uint32_t>(workspace, L.tickets), st);
    if (e != cudaSuccess) return cuda_fail(e);
    e = launch_group(shape->n_experts, shape->top_k, n_tokens, ids, ws_at<int32_t>(workspace, L.counts),
                     ws_at<int32_t>(workspace, L.offsets), ws_at<int32_t>(workspace, L.perm), st);
    if (e != cudaSuccess) return cuda_fail(e);
    e = launch_q4k_gateup(*shape, x, blocks, experts->expert_stride, ws_at<int32_t>(workspace, L.offsets),
                          ws_at<int32_t>(workspace, L.perm), n_tokens, ws_at<float>(workspace, L.h), st);
    if (e != cudaSuccess) return cuda_fail(e);
    e = launch_q4k_down(*shape, blocks, experts->expert_stride, ws_at<float>(workspace, L.h), ids, pw, n_tokens, out,
                        st);
    if (e != cudaSuccess) return cuda_fail(e);
    if (has_shared) {  // + gate * Wsd hs, added onto the routed rows
        e = launch_down(*shape, nullptr, 0, nullptr, nullptr, nullptr, 0, (const uint16_t*)shared->w_down, hs, gate,
                        n_tokens, out, 1, st);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    return QS_OK;
}

int qs_q4k_quantize(const float* w, int64_t n_rows, int64_t K, void* out, void* stream) {
    if (!w || !out || n_rows < 1 || K < 256 || K % 256 || !aligned16(w) || ((uintptr_t)out & 3u))
        return QS_ERR_INVALID;
    cudaError_t e = launch_q4k_quantize(w, n_rows * (K / 256), static_cast<uint8_t*>(out), (cudaStream_t)stream);
    return e == cudaSuccess ? QS_OK : cuda_fail(e);
}

int qs_steer_rows(float* out, const float* direction, float scale, int n_tokens, int hidden, void* stream) {
    if (!out || !direction || n_tokens < 1 || hidden < 4 || hidden % 4 || !aligned16(out) || !aligned16(direction))
        return QS_ERR_INVALID;
    if (scale == 0.0f) return QS_OK;
    cudaError_t e = launch_steer_rows(out, direction, scale, n_tokens, hidden, (cudaStream_t)stream);
    return e == cudaSuccess ? QS_OK : cuda_fail(e);
}

int qs_test_wait_timeout(void* workspace, size_t workspace_bytes, int limit_us, void* stream) {
    if (!workspace || workspace_bytes < (size_t)kHeaderBytes || ((uintptr_t)workspace & 255u) || limit_us < 1 ||
        limit_us > 1000000)
        return QS_ERR_INVALID;
    cudaError_t e = launch_test_wait(workspace, (uint64_t)limit_us * 1000ull, (cudaStream_t)stream);
    return e == cudaSuccess ? QS_OK : cuda_fail(e);
}

}  // extern "C"

// qs_internal.h -- host-side declarations shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "qs_moe.h"

namespace qs {

// Workspace regions (byte offsets from the workspace base; each 256-aligned).
struct WsLayout {
    size_t header = 0;
    size_t logits = 0;   // f32 [T x E]
    size_t ids = 0;      // i32 [T x k]
    size_t pw = 0;       // f32 [T x k]
    size_t counts = 0;   // i32 [E]
    size_t offsets = 0;  // i32 [E + 1]
    size_t perm = 0;     // i32 [T x k]
    size_t h = 0;        // f32 [T*k x F]
    size_t hs = 0;       // f32 [T x S]
    size_t gate = 0;     // f32 [T]
    size_t tickets = 0;  // u32 [ceil(T / kRouteTok)]
    // exchanged arrays of the persistent decode kernel (fp32; completion counters in the header)
    size_t xlog = 0;     // [Tf x E]
    size_t xhs = 0;      // [Tf x S]
    size_t xh = 0;       // [Tf*k x F]     (Tf = min(T, kFusedMaxT))
    // cluster decode kernel: its counters, per-entry routed down products, shared down products
    size_t cx = 0;       // kCxBytes of 64-bit counters, one per 32-byte sector
    size_t cpd = 0;      // f32 [Tc*k x H]  (Tc = min(T, kClusterMaxT))
    size_t csdp = 0;     // f32 [Tc x H]
    // tensor-core (prefill) path
    size_t wr3 = 0;      // bf16 [3 x E x H]  router weights as three bf16 planes
    size_t lpart = 0;    // f32 [kPrefillMaxKS x T x E] partial logits
    size_t xs = 0;       // fp16 [T*k x H] token rows in expert-sorted order
    size_t cursor = 0;   // i32 [E] fill pointers of the expert lists
    size_t h16 = 0;      // fp16 [T*k x F] (expert-sorted entries)
    size_t hs16 = 0;     // bf16 [T x S]
    size_t total = 0;
};

constexpr int kRouteTok = 8;    // tokens per router CTA chunk
constexpr int kFusedMaxT = 16;  // largest token count the persistent decode kernel takes
constexpr int kPrefillMaxKS = 4;  // largest split of H in the tensor-core router
constexpr int kClusterCtas = 8;   // CTAs per thread-block cluster of the cluster decode kernel
constexpr int kClusterMaxT = 8;   // largest token count the cluster decode kernel takes
constexpr int kCxBytes = 512;     // counter region of the cluster decode kernel

WsLayout ws_layout(const qs_moe_shape& s, int max_tokens);

// Record e as the calling thread's last CUDA failure (qs_last_cuda_error) and return QS_ERR_CUDA.
int cuda_fail(cudaError_t e);

// Decode-path launchers (qs_decode.cu).  All return the launch's cudaError_t.
cudaError_t launch_route(const qs_moe_shape& s, const void* x, const float* W, const float* bias, int T,
                         float* logits, int32_t* ids, float* pw, uint32_t* tickets, cudaStream_t st);
cudaError_t launch_group(int E, int k, int T, const int32_t* ids, int32_t* counts, int32_t* offsets, int32_t* perm,
                         cudaStream_t st);
cudaError_t launch_gateup(const qs_moe_shape& s, const void* x, const uint8_t* experts, int64_t stride,
                          const int32_t* offsets, const int32_t* perm, int T, float* h, cudaStream_t st);
cudaError_t launch_down(const qs_moe_shape& s, const uint8_t* experts, int64_t stride, const float* h,
                        const int32_t* ids, const float* pw, int n_slots, const uint16_t* sh_down,
                        const float* hs, const float* gate, int T, float* out, int accumulate, cudaStream_t st);
cudaError_t launch_shared_gateup(const qs_moe_shape& s, const void* x, const uint16_t* wg, const uint16_t* wu,
                                 const uint16_t* wsig, int T, float* hs, float* gate, cudaStream_t st);
cudaError_t launch_quantize(const float* w, int64_t n_blocks, uint8_t* out, cudaStream_t st);
cudaError_t launch_test_wait(void* ws, uint64_t limit_ns, cudaStream_t st);

// Q4_K routed experts (qs_q4k.cu): encoder, gate/up + SwiGLU into h, down + routing-weight
// combine into out (stored, not added).
cudaError_t launch_q4k_quantize(const float* w, int64_t n_blocks, uint8_t* out, cudaStream_t st);
cudaError_t launch_q4k_gateup(const qs_moe_shape& s, const void* x, const uint8_t* experts, int64_t stride,
                              const int32_t* offsets, const int32_t* perm, int T, float* h, cudaStream_t st);
cudaError_t launch_q4k_down(const qs_moe_shape& s, const uint8_t* experts, int64_t stride, const float* h,
                            const int32_t* ids, const float* pw, int T, float* out, cudaStream_t st);
size_t q4k_down_smem(int k, int F);

// Directional steering of output rows (qs_steer.cu): y <- y - scale * d * (d . y) per row.
cudaError_t launch_steer_rows(float* y, const float* d, float scale, int T, int H, cudaStream_t st);

// Persistent single-kernel decode path (qs_fused.cu).  cudaErrorNotSupported
// when the shape or token count is outside its plan; the caller then runs the
// per-step kernels.  sg == nullptr means no shared expert.  x_host_mapped: x and out are
// pinned host memory given by their device-mapped addresses (x read with plain loads).
cudaError_t launch_fused_decode(const qs_moe_shape& s, const void* x, const float* Wr, const float* bias,
                                const uint8_t* experts, int64_t stride, const uint16_t* sg, const uint16_t* su,
                                const uint16_t* sd, const uint16_t* ssig, int T, float* out, void* ws,
                                const WsLayout& W, cudaStream_t st, bool x_host_mapped = false,
                                int fmt = 0 /* 0: Q2_K, 1: Q4_K routed experts */);
bool fused_decode_supported(const qs_moe_shape& s, int T, cudaError_t* err);

// Decode path of thread-block clusters (qs_cluster.cu): one kernel; a cluster of
// kClusterCtas CTAs owns whole routed experts and shares h through distributed shared
// memory.  cudaErrorNotSupported when the shape or token count is outside its plan.
// x_host_mapped: x (and out) are pinned host memory given by their device-mapped
// addresses; the kernel reads x with plain loads instead of a bulk copy.
cudaError_t launch_cluster_decode(const qs_moe_shape& s, const void* x, const float* Wr, const float* bias,
                                  const uint8_t* experts, int64_t stride, const uint16_t* sg, const uint16_t* su,
                                  const uint16_t* sd, const uint16_t* ssig, int T, float* out, void* ws,
                                  const WsLayout& W, cudaStream_t st, bool x_host_mapped = false);
bool cluster_decode_supported(const qs_moe_shape& s, int T, cudaError_t* err);

// The one-kernel decode paths in qs_moe_ffn's order of preference for this token count
// (qs_api.cu): the first that takes the call is launched; cudaErrorNotSupported if neither.
cudaError_t launch_decode_kernel(const qs_moe_shape& s, const void* x, const float* Wr, const float* bias,
                                 const uint8_t* experts, int64_t stride, const uint16_t* sg, const uint16_t* su,
                                 const uint16_t* sd, const uint16_t* ssig, int T, float* out, void* ws,
                                 const WsLayout& W, cudaStream_t st, bool x_host_mapped);

// Tensor-core path for many tokens (qs_prefill.cu): prefill_launches() launches.  Needs bf16
// x and Q2_K row layouts it can stage (see prefill_shape_ok).
bool prefill_shape_ok(const qs_moe_shape& s);
int prefill_launches();
cudaError_t launch_prefill(const qs_moe_shape& s, const void* x, const float* Wr, const float* bias,
                           const uint8_t* experts, int64_t stride, const uint16_t* sg, const uint16_t* su,
                           const uint16_t* sd, const uint16_t* ssig, int T, float* out, void* ws, const WsLayout& W,
                           cudaStream_t st);

}  // namespace qs

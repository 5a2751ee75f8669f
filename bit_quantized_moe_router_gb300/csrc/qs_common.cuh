// qs_common.cuh -- device helpers shared by the kernels of the Q2_K MoE-FFN library.
//
// Inline PTX for sm_103a: mbarrier + bulk asynchronous copies (TMA engine, 1-D
// form) for staging weight rows in shared memory, acquire/release counters for
// the cross-CTA waits, and the 16x8-bit integer dot product (dp2a) the Q2_K
// GEMV is built on.  Every wait is bounded by the global timer and reports
// QS_ERR_TIMEOUT through the workspace status word instead of spinning forever.
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "qs_moe.h"

namespace qs {

constexpr int kBlockBytes = 84;     // one Q2_K block
constexpr int kBlockWeights = 256;  // weights per block
constexpr int kHeaderBytes = 256;   // workspace header (status + counters)
constexpr uint64_t kWaitNs = 200ull * 1000ull * 1000ull;  // 200 ms: any legitimate wait is microseconds

// Workspace header.  Counters live in separate 32-byte sectors.
struct WsHeader {
    uint32_t status;        // sticky qs_status of device-side failures (0 = ok)
    uint32_t where[7];      // first time-out of the tensor-core path: wait code, CTA, warp, counter
    uint32_t ctr[7][8];     // ctr[i][0] = counter i
};
static_assert(sizeof(WsHeader) <= kHeaderBytes, "header too large");

// Counters of the persistent decode kernel (CTAs that have published their logits, hs and
// h; CTAs that have left), never reset: every call adds gridDim to each, so a call finds its
// targets from the exit count.  And the counter of the wait test.
enum Counter { kCtrLogits = 0, kCtrHs = 1, kCtrExit = 2, kCtrTest = 3, kCtrH = 4 };

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void set_status(uint32_t* status, uint32_t code) {
    atomicCAS(status, 0u, code);
}

// ------------------------------------------------------------------ counters (gpu scope)

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void red_release_add(uint32_t* p, uint32_t v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t atom_acq_rel_add(uint32_t* p, uint32_t v) {
    uint32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

// Wait (one thread) until *p >= target; false (and status = TIMEOUT) after kWaitNs.
__device__ __forceinline__ bool wait_geq(const uint32_t* p, uint32_t target, uint32_t* status, uint64_t limit_ns = kWaitNs) {
    if (ld_acquire(p) >= target) return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        __nanosleep(32);
        if (ld_acquire(p) >= target) return true;
        if (global_timer_ns() - t0 > limit_ns) {
            set_status(status, QS_ERR_TIMEOUT);
            return false;
        }
    }
}

// ------------------------------------------------------------------ mbarrier + bulk copy

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// make mbarrier initialisation visible to the async (TMA) proxy
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

// plain arrival (release semantics at CTA scope)
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// As mbar_try_wait, but the thread may be suspended in hardware for up to
// `hint_ns` while the phase is incomplete; it resumes as soon as the phase
// completes, so a waiting warp costs (almost) no issue slots.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

// Bounded wait on an mbarrier phase.  Returns false after kWaitNs.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns = kWaitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (global_timer_ns() - t0 > limit_ns) return false;
    }
}

// Bulk copy global -> this CTA's shared memory; completion is counted on bar.
// dst, src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Hint: bring a span into L2 (16-byte aligned, multiple of 16 bytes).
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// ------------------------------------------------------------------ arithmetic

// d = c + a.lo16 * b.byte0 + a.hi16 * b.byte1   (a: two signed 16-bit, b: unsigned bytes)
__device__ __forceinline__ int dp2a_lo(int a, uint32_t b, int c) {
    int d;
    asm("dp2a.lo.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
// d = c + a.lo16 * b.byte2 + a.hi16 * b.byte3
__device__ __forceinline__ int dp2a_hi(int a, uint32_t b, int c) {
    int d;
    asm("dp2a.hi.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

__device__ __forceinline__ float silu(float z) { return z / (1.0f + expf(-z)); }
__device__ __forceinline__ float sigmoid(float z) { return 1.0f / (1.0f + expf(-z)); }

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ float load_x(const void* x, int x_dtype, size_t i) {
    if (x_dtype == QS_BF16) return bf16_lo(static_cast<const uint16_t*>(x)[i]);
    return static_cast<const float*>(x)[i];
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Block-wide max over all threads (blockDim multiple of 32, <= 1024); red: >= 32 floats of smem.
__device__ __forceinline__ float block_max(float v, float* red) {
    v = warp_max(v);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31, nw = blockDim.x >> 5;
    __syncthreads();
    if (l == 0) red[w] = v;
    __syncthreads();
    float r = (l < nw) ? red[l] : -INFINITY;
    r = warp_max(r);
    return r;
}

}  // namespace qs

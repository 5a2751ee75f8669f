// qs_warp.cuh -- warp-level helpers shared by the persistent decode kernels: relaxed and
// acquire/release accesses of exchanged data and counters at gpu scope, and the dense-row
// dot product of fp32 / bf16 rows held in shared or global memory.
#pragma once

#include "qs_common.cuh"

namespace qs {

__device__ __forceinline__ int vload(const int* p) { return *reinterpret_cast<const volatile int*>(p); }
__device__ __forceinline__ void vstore(int* p, int v) { *reinterpret_cast<volatile int*>(p) = v; }

// Relaxed gpu-scope loads of exchanged data: served by L2, never by a stale L1 line.
__device__ __forceinline__ float ld_relaxed_f32(const float* p) {
    float v;
    asm volatile("ld.relaxed.gpu.global.f32 %0, [%1];" : "=f"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ float4 ld_relaxed_f32x4(const float* p) {
    float4 v;
    asm volatile("ld.relaxed.gpu.global.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p)
                 : "memory");
    return v;
}

// 64-bit exchange counters (gpu scope).
__device__ __forceinline__ uint64_t ld_acquire_u64(const uint64_t* p) {
    uint64_t v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ uint64_t ld_relaxed_u64(const uint64_t* p) {
    uint64_t v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void red_release_add_u64(uint64_t* p, uint64_t v) {
    asm volatile("red.release.gpu.global.add.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ void red_relaxed_add_u64(uint64_t* p, uint64_t v) {
    asm volatile("red.relaxed.gpu.global.add.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// ------------------------------------------------------------------ dense rows

__device__ __forceinline__ void load8(const uint8_t* p, bool f32, float* v) {
    if (f32) {
        const float4 a = reinterpret_cast<const float4*>(p)[0];
        const float4 b = reinterpret_cast<const float4*>(p)[1];
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    } else {
        const uint4 w = *reinterpret_cast<const uint4*>(p);
        v[0] = bf16_lo(w.x); v[1] = bf16_hi(w.x);
        v[2] = bf16_lo(w.y); v[3] = bf16_hi(w.y);
        v[4] = bf16_lo(w.z); v[5] = bf16_hi(w.z);
        v[6] = bf16_lo(w.w); v[7] = bf16_hi(w.w);
    }
}

// One warp: dot products of one dense row (K elements, fp32 or bf16, shared or global memory)
// with T activation rows (fp32 or bf16, shared memory), lane-strided by 8 elements, then summed
// over the warp.  Every lane gets acc[t].
template <int MAXT>
__device__ __forceinline__ void warp_dense_row(const uint8_t* w, bool w_f32, int K, const uint8_t* act, bool a_f32,
                                               int T, float* acc) {
    const int lane = threadIdx.x & 31;
    const int wsz = w_f32 ? 4 : 2, asz = a_f32 ? 4 : 2;
#pragma unroll
    for (int t = 0; t < MAXT; t++) acc[t] = 0.0f;
#pragma unroll 4
    for (int i = lane * 8; i < K; i += 256) {  // unrolled: rows read from global memory keep loads in flight
        float wv[8];
        load8(w + (size_t)i * wsz, w_f32, wv);
#pragma unroll
        for (int t = 0; t < MAXT; t++) {
            if (t < T) {
                float av[8];
                load8(act + ((size_t)t * K + i) * asz, a_f32, av);
                float s = acc[t];
#pragma unroll
                for (int q = 0; q < 8; q++) s = fmaf(wv[q], av[q], s);
                acc[t] = s;
            }
        }
    }
#pragma unroll
    for (int t = 0; t < MAXT; t++)
        if (t < T) acc[t] = warp_sum(acc[t]);
}

// Two bf16 rows (a gate row and an up row) against the same activations in one pass: each row's
// sums are formed exactly as warp_dense_row forms them.
template <int MAXT>
__device__ __forceinline__ void warp_dense_rows2(const uint8_t* wa, const uint8_t* wb, int K, const uint8_t* act,
                                                 bool a_f32, int T, float* acc_a, float* acc_b) {
    const int lane = threadIdx.x & 31;
    const int asz = a_f32 ? 4 : 2;
#pragma unroll
    for (int t = 0; t < MAXT; t++) acc_a[t] = acc_b[t] = 0.0f;
#pragma unroll 2
    for (int i = lane * 8; i < K; i += 256) {
        float va[8], vb[8];
        load8(wa + (size_t)i * 2, false, va);
        load8(wb + (size_t)i * 2, false, vb);
#pragma unroll
        for (int t = 0; t < MAXT; t++) {
            if (t < T) {
                float av[8];
                load8(act + ((size_t)t * K + i) * asz, a_f32, av);
                float sa = acc_a[t], sb = acc_b[t];
#pragma unroll
                for (int q = 0; q < 8; q++) {
                    sa = fmaf(va[q], av[q], sa);
                    sb = fmaf(vb[q], av[q], sb);
                }
                acc_a[t] = sa;
                acc_b[t] = sb;
            }
        }
    }
#pragma unroll
    for (int t = 0; t < MAXT; t++) {
        if (t < T) {
            acc_a[t] = warp_sum(acc_a[t]);
            acc_b[t] = warp_sum(acc_b[t]);
        }
    }
}

// ------------------------------------------------------------------ routing (one warp per token)

// Order-preserving map of a logit to an unsigned key, + 1 so that 0 means "none" (the largest
// key, +inf's, is below 2^32 - 1).  -0 ranks as +0; a NaN ranks below every number.
__device__ __forceinline__ uint32_t topk_key(float x) {
    const float v = x == 0.0f ? 0.0f : x;
    const uint32_t b = __float_as_uint(v);
    return (v != v) ? 1u : ((b & 0x80000000u) ? ~b : (b | 0x80000000u)) + 1u;
}

// The logit back from its key (a NaN's key as -inf).
__device__ __forceinline__ float topk_logit(uint32_t key) {
    if (key <= 1u) return -INFINITY;
    const uint32_t o = key - 1u;
    return __uint_as_float((o & 0x80000000u) ? (o & 0x7fffffffu) : ~o);
}

// One selection round: the warp's largest key among the lanes' best untaken ones (one redux)
// and, among the lanes holding it, the lowest id (a second); marks it taken in its lane.
__device__ __forceinline__ void topk_round(uint32_t best, int bm, uint32_t& taken, int j, uint32_t& my_key,
                                           int& my_id) {
    const int lane = threadIdx.x & 31;
    const uint32_t gbest = __reduce_max_sync(0xffffffffu, best);
    const uint32_t cand = (best != 0u && best == gbest) ? (uint32_t)(lane + 32 * bm) : 0xffffffffu;
    const uint32_t gidx = __reduce_min_sync(0xffffffffu, cand);
    if (gidx != 0xffffffffu && (int)(gidx & 31u) == lane) taken |= 1u << (gidx >> 5);
    if (lane == j) {
        my_key = gbest;
        my_id = (int)gidx;
    }
}

// Softmax over the k selected logits (lane j < k holds the j-th, the largest in lane 0).
__device__ __forceinline__ float topk_softmax(uint32_t my_key, int k) {
    const int lane = threadIdx.x & 31;
    const float my_l = lane < k ? topk_logit(my_key) : -INFINITY;
    const float lmax = __shfl_sync(0xffffffffu, my_l, 0);
    const float ex = (lane < k) ? expf(my_l - lmax) : 0.0f;
    const float den = warp_sum(ex);
    return ex / den;
}

// Top-k of the E logits of one token (E <= 32 * MV, k <= 32), descending, ties to the lower id;
// softmax over the selected logits.  Lane j < k returns the j-th id and weight.  Lane l holds
// the keys of experts l + 32 m in registers.
template <int MV>
__device__ __forceinline__ void warp_topk(const float* l, int E, int k, int& id, float& w) {
    const int lane = threadIdx.x & 31;
    float lv[MV];
#pragma unroll
    for (int m = 0; m < MV; m++) {  // every load in flight before the first is used
        const int e = lane + 32 * m;
        lv[m] = e < E ? ld_relaxed_f32(l + e) : 0.0f;
    }
    uint32_t key[MV];
#pragma unroll
    for (int m = 0; m < MV; m++) key[m] = (lane + 32 * m < E) ? topk_key(lv[m]) : 0u;
    uint32_t taken = 0, my_key = 0;
    int my_id = 0;
    for (int j = 0; j < k; j++) {
        uint32_t best = 0;
        int bm = 0;
#pragma unroll
        for (int m = 0; m < MV; m++) {
            const bool better = !((taken >> m) & 1u) && key[m] > best;  // strict: lower m (lower id) wins ties
            best = better ? key[m] : best;
            bm = better ? m : bm;
        }
        topk_round(best, bm, taken, j, my_key, my_id);
    }
    id = my_id;
    w = topk_softmax(my_key, k);
}

// The same selection for E <= 1024 with few registers: every round re-reads the logits
// (L1/L2 hits after the first) instead of holding them.  Out of line: kept apart from the code of
// the common case.
static __device__ __noinline__ void warp_topk_stream(const float* l, int E, int k, int& id, float& w) {
    const int lane = threadIdx.x & 31;
    const int nm = (E + 31) >> 5;
    uint32_t taken = 0, my_key = 0;
    int my_id = 0;
    for (int j = 0; j < k; j++) {
        uint32_t best = 0;
        int bm = 0;
#pragma unroll 4
        for (int m = 0; m < nm; m++) {
            const int e = lane + 32 * m;
            const uint32_t key = e < E ? topk_key(ld_relaxed_f32(l + e)) : 0u;
            const bool better = !((taken >> m) & 1u) && key > best;
            best = better ? key : best;
            bm = better ? m : bm;
        }
        topk_round(best, bm, taken, j, my_key, my_id);
    }
    id = my_id;
    w = topk_softmax(my_key, k);
}

}  // namespace qs

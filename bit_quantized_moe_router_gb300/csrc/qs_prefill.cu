// qs_prefill.cu -- the layer for many tokens at once, on the fifth-generation tensor cores.
//
// "Prefill" of the MoE-FFN layer: the same computation as the decode path
// (router top-k + softmax, grouped Q2_K SwiGLU experts, weighted combine,
// sigmoid-gated bf16 shared expert), organised as per-expert GEMMs so the
// weights of an expert are read once for all the tokens routed to it.
//
//   pf_router_split     Wr (fp32) -> three bf16 planes with Wr = b1 + b2 + b3 exactly
//   pf_router_mma       partial logits  l = sum_p b_p . x  on tcgen05 (.kind::f16, bf16 A and B,
//                       fp32 accumulation; every product is exact), split along H
//   pf_topk             per token: sum of the partial logits (+ bias), top-k, softmax over the k,
//                       shared-expert gate sigmoid(w_sg . x), a count per chosen expert
//   pf_scan             expert offsets (exclusive scan of the counts)
//   pf_scatter          each (token, slot) entry claims a place in its expert's list; the token's
//                       row of x is copied there as fp16, so each expert's rows are contiguous
//   pf_expert<2>        gate+up: for each expert, h = silu(Wg x) * (Wu x) over its tokens (fp16 h);
//                       shared expert's gate/up over all tokens (bf16 hs)
//   pf_expert<1>        down: fp16 p * (Wd h) per (token, slot) entry (routed), and
//                       y[t] = sigmoid_gate[t] * Wsd hs[t] (shared)
//   pf_combine          y[t] += the token's k routed contributions, in slot order
// The expert counts are zeroed by a memset first.  No step uses atomics on
// floating-point data, so the result is the same from run to run.
//
// pf_expert is one persistent CTA per SM walking a list of work units
// (expert or shared, 128-row tile of the output features, up to 128 tokens).
// Its warps are specialised:
//   * a TMA thread streams the unit's raw weight bytes (Q2_K blocks or bf16
//     rows) into a ring of shared-memory slots, and the unit's token rows
//     (x, or h for the down projection) as 128B-swizzled B tiles into another;
//   * sixteen dequant warps turn raw Q2_K bytes into fp16 weights and write
//     them straight into tensor memory, which is the MMA's A operand (the
//     "TS" form: no shared-memory round trip for the dequantised weights);
//     the shared expert's bf16 tiles are the A operand as they land (SS form);
//   * one thread issues tcgen05.mma into a fp32 accumulator in tensor memory;
//   * four epilogue warps read the accumulator back (tcgen05.ld) and apply
//     SwiGLU or the routing weight, writing h, the fp16 partials or y.
// Every wait is bounded by the global timer; a time-out sets QS_ERR_TIMEOUT in
// the workspace status word and winds every role of the CTA down.
//
// Q2_K to fp16: a 16-weight sub-block has only four possible values,
// v_q = d*sc_lo*q - dmin*sc_hi (q = 0..3), computed once in fp32 and rounded
// to fp16; each pair of weights is then one byte-permute (prmt) out of that
// four-entry table, indexed by the two 2-bit codes.
#include "qs_common.cuh"
#include "qs_internal.h"
#include "qs_q2k.cuh"
#include "qs_tc.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>
#include <mutex>

namespace qs {
namespace {

constexpr int kNT = 128;                  // max tokens (B rows, MMA N) per unit
constexpr int kSlotBytes = 32768;         // one raw slot
constexpr int kMatStride = 16384;         // second matrix (up) inside a raw slot
constexpr int kBStageBytes = kNT * 128;   // B operand stage: 128 rows x 64 16-bit values
constexpr int kColBox = 112;              // bytes per row of a Q2_K column box (covers 84 + offset <= 12)
constexpr int kA0 = 256;                  // first TMEM column of the A stages
constexpr int kDeqWarps = 16;             // dequant warps of an expert kernel
constexpr int kWarpMma = kDeqWarps + 4;   // MMA issuer (+ TMEM allocation)
constexpr int kWarpRaw = kDeqWarps + 5;   // TMA of raw weights
constexpr int kWarpB = kDeqWarps + 6;     // TMA of B slices
constexpr int kExpertThreads = 32 * (kDeqWarps + 7);
constexpr int kRouterStages = 3;
constexpr int kRouterThreads = 192;
constexpr int kMaxKS = kPrefillMaxKS;     // router split of H
constexpr uint32_t kSleepNs = 20000;      // longest hardware suspension of a waiting thread per poll

enum RawMode : int { kRawColumn = 0, kRawTile = 1 };

// ------------------------------------------------------------------ small device helpers

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
    return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_u32(dst)),
        "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int x, int y, int z, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(
            smem_u32(dst)),
        "l"(map), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
        : "memory");
}
// x < 2^23 as a float, exactly: x in the mantissa of 2^23, minus 2^23 (no int-to-float conversion).
__device__ __forceinline__ float small_uint_to_float(uint32_t x) {
    return __uint_as_float(0x4B000000u | x) - 8388608.0f;
}

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
}

// Record the first time-out: status = QS_ERR_TIMEOUT and, beside it in the workspace
// header, which wait gave up (code), in which CTA and warp, at which counter.
__device__ __noinline__ void note_timeout(uint32_t* status, uint32_t code, uint32_t counter) {
    if (atomicCAS(status, 0u, (uint32_t)QS_ERR_TIMEOUT) == 0u) {
        status[1] = code;
        status[2] = blockIdx.x;
        status[3] = threadIdx.x >> 5;
        status[4] = counter;
        __threadfence();
    }
}

// Bounded wait on an mbarrier phase by lane 0 of the warp, result broadcast to
// the warp; on success every lane also observes the phase (acquire).  Returns
// false at once if the CTA is aborting, or after the time limit (then aborts).
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort, uint32_t* status,
                                          uint32_t code = 0, uint32_t counter = 0) {
    int ok = 1;
    if ((threadIdx.x & 31) == 0) {
        if (!mbar_try_wait(bar, parity)) {
            const uint64_t t0 = global_timer_ns();
            for (;;) {
                if (mbar_try_wait_sleep(bar, parity, kSleepNs)) break;
                if (*abort) {
                    ok = 0;
                    break;
                }
                if (global_timer_ns() - t0 > kWaitNs) {
                    *abort = 1;
                    note_timeout(status, code, counter);
                    ok = 0;
                    break;
                }
            }
        }
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (ok) (void)mbar_try_wait(bar, parity);
    return ok != 0;
}
// Bounded wait (lane 0 polls, result broadcast) until *tag == want.
__device__ __forceinline__ bool warp_wait_tag(const int* tag, int want, volatile int* abort, uint32_t* status,
                                              uint32_t code = 0) {
    int ok = 1;
    if ((threadIdx.x & 31) == 0) {
        const volatile int* t = tag;
        if (*t != want) {
            const uint64_t t0 = global_timer_ns();
            while (*t != want) {
                __nanosleep(64);
                if (*abort) {
                    ok = 0;
                    break;
                }
                if (global_timer_ns() - t0 > kWaitNs) {
                    *abort = 1;
                    note_timeout(status, code, (uint32_t)want);
                    ok = 0;
                    break;
                }
            }
        }
    }
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// Abort flag as one value for the whole warp (lane 0's reading).
__device__ __forceinline__ bool warp_aborted(volatile int* abort) {
    return __shfl_sync(0xffffffffu, *abort, 0) != 0;
}

// The same for a single thread.
__device__ __forceinline__ bool thread_wait(uint64_t* bar, uint32_t parity, volatile int* abort, uint32_t* status,
                                            uint32_t code = 0, uint32_t counter = 0) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        if (mbar_try_wait_sleep(bar, parity, kSleepNs)) return true;
        if (*abort) return false;
        if (global_timer_ns() - t0 > kWaitNs) {
            *abort = 1;
            note_timeout(status, code, counter);
            return false;
        }
    }
}

// ------------------------------------------------------------------ Q2_K -> fp16 for one 64-weight K slice

// w[0..20]: the 84-byte block as words (scales 0..3, qs 4..19, d | dmin << 16 in 20).
// K slice c (weights 64c .. 64c+63 of the block) uses scale bytes 4c..4c+3 (word c), code bytes
// 32(c>>1)..+31 (words 4+8(c>>1)..+7) and bit pairs j = 2(c&1) + jj, jj = 0, 1.  Half jj of the
// slice is weights 64c + 32jj .. +31 -> 16 packed fp16 pairs, lower K in the low half.  One code
// path serves every slice (the kernel stays small); a half keeps register pressure low.
__device__ __forceinline__ void dequant_half(uint32_t scw, const uint32_t (&qw)[8], int c, int jj, float d, float dm,
                                             uint32_t (&out)[16]) {
    const int sh = 4 * (c & 1) + 2 * jj;  // 2j
#pragma unroll
    for (int lh = 0; lh < 2; lh++) {
        const uint32_t sc = (scw >> (8 * (2 * jj + lh))) & 0xffu;
        const float a = d * small_uint_to_float(sc & 15u), m = dm * small_uint_to_float(sc >> 4);
        const uint32_t t0 = pack_h2(-m, a - m);
        const uint32_t t1 = pack_h2(fmaf(2.0f, a, -m), fmaf(3.0f, a, -m));
#pragma unroll
        for (int i = 0; i < 4; i++) {
            // bytes of q hold four weights' codes; byte b of sel selects table bytes (2q_b, 2q_b + 1):
            // one selector for four weights, its upper half for the last two
            const uint32_t q = (qw[4 * lh + i] >> sh) & 0x03030303u;
            const uint32_t sel = q * 34u + 0x10101010u;
            out[8 * lh + 2 * i] = __byte_perm(t0, t1, sel);
            out[8 * lh + 2 * i + 1] = __byte_perm(t0, t1, sel >> 16);
        }
    }
}

// ================================================================== router

// planes[p][e][h], Wr = planes[0] + planes[1] + planes[2] exactly (bf16 keeps 8 significant bits).
__global__ void __launch_bounds__(256) pf_router_split_kernel(const float* __restrict__ W, size_t n, uint16_t* planes) {
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        const float w = W[i];
        const __nv_bfloat16 b1 = __float2bfloat16_rn(w);
        const float r1 = w - __bfloat162float(b1);
        const __nv_bfloat16 b2 = __float2bfloat16_rn(r1);
        const float r2 = r1 - __bfloat162float(b2);
        const __nv_bfloat16 b3 = __float2bfloat16_rn(r2);
        planes[i] = __bfloat16_as_ushort(b1);
        planes[n + i] = __bfloat16_as_ushort(b2);
        planes[2 * n + i] = __bfloat16_as_ushort(b3);
    }
}

struct RouterParams {
    CUtensorMap map_w;  // bf16 [3][E][H], box 64 x 128 x 1, 128B swizzle
    CUtensorMap map_x;  // bf16 [T][H],    box 64 x 128,     128B swizzle
    float* lpart;       // [KS][T][E]
    int E, T, KBc;      // KBc: 64-wide K slices per split
    uint32_t* status;
};

struct RouterCtl {
    uint64_t full[kRouterStages], empty[kRouterStages], acc;
    uint32_t tmem;
    int abort;
};

// grid (ceil(E/128), ceil(T/128), KS); warp 0 TMA, warp 1 MMA (+TMEM), warps 2..5 epilogue.
__global__ void __launch_bounds__(kRouterThreads, 1) pf_router_mma_kernel(const __grid_constant__ RouterParams p) {
    extern __shared__ uint8_t rt_smem_raw[];
    uint8_t* sm = align1024(rt_smem_raw);
    constexpr int kStage = 4 * 16384;  // three A planes + B
    RouterCtl* ctl = reinterpret_cast<RouterCtl*>(sm + kRouterStages * kStage);
    volatile int* abort = &ctl->abort;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.x * 128, n0 = blockIdx.y * 128, ks = blockIdx.z;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kRouterStages; s++) {
            mbar_init(&ctl->full[s], 1);
            mbar_init(&ctl->empty[s], 1);
        }
        mbar_init(&ctl->acc, 1);
        ctl->abort = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(&ctl->tmem, 128);
        tc::tmem_relinquish();
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tbase = ctl->tmem;
    const int kb0 = ks * p.KBc;

    if (warp == 0) {
        if (lane == 0) {
            for (int i = 0; i < p.KBc; i++) {
                const int s = i % kRouterStages;
                if (i >= kRouterStages && !thread_wait(&ctl->empty[s], ((i / kRouterStages) - 1) & 1, abort, p.status, 12, i))
                    break;
                uint8_t* st = sm + s * kStage;
                mbar_arrive_expect_tx(&ctl->full[s], kStage);
                const int kx = (kb0 + i) * 64;
                for (int pl = 0; pl < 3; pl++) tma_load_3d(st + pl * 16384, &p.map_w, kx, m0, pl, &ctl->full[s]);
                tma_load_2d(st + 3 * 16384, &p.map_x, kx, n0, &ctl->full[s]);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t id = tc::idesc(tc::kBF16, 128, 128);
            bool ok = true;
            for (int i = 0; i < p.KBc && ok; i++) {
                const int s = i % kRouterStages;
                ok = thread_wait(&ctl->full[s], (i / kRouterStages) & 1, abort, p.status, 13, i);
                if (!ok) break;
                tc::fence_after();
                const uint32_t sa = smem_u32(sm + s * kStage);
                const uint64_t bd = tc::sdesc_sw128(sa + 3 * 16384);
                for (int pl = 0; pl < 3; pl++) {
                    const uint64_t ad = tc::sdesc_sw128(sa + pl * 16384);
#pragma unroll
                    for (int k16 = 0; k16 < 4; k16++)
                        tc::mma_ss_f16(tbase, ad + 2 * k16, bd + 2 * k16, id, (i | pl | k16) != 0);
                }
                tc::commit(&ctl->empty[s]);
            }
            tc::commit(&ctl->acc);  // also drains every MMA issued above
        }
    } else {
        const int q = warp & 3;
        const bool ok = warp_wait(&ctl->acc, 0, abort, p.status, 14);
        tc::fence_after();
        if (ok) {
            const int e = m0 + 32 * q + lane;
            for (int c0 = 0; c0 < 128; c0 += 16) {
                uint32_t r[16];
                tc::ld16(tc::taddr(tbase, 32 * q, c0), r);
                tc::wait_ld();
                if (e < p.E) {
#pragma unroll
                    for (int i = 0; i < 16; i++) {
                        const int t = n0 + c0 + i;
                        if (t < p.T) p.lpart[((size_t)ks * p.T + t) * p.E + e] = __uint_as_float(r[i]);
                    }
                }
            }
        }
    }
    tc::fence_before();
    __syncthreads();
    if (warp == 0 && lane == 0 && *abort) {
        // let copies still in flight land before the CTA's shared memory goes away
        for (int s = 0; s < kRouterStages; s++) (void)mbar_wait(&ctl->full[s], 0, 1000000ull);
    }
    if (warp == 1) {
        tc::fence_after();
        tc::tmem_dealloc(tbase, 128);
    }
}

// ================================================================== top-k, grouping, token rows

// One warp per token: logits = sum of the partials (+ bias), top-k, softmax over
// the k, the shared-expert gate sigmoid(w_sg . x), and one count per chosen
// expert (counts are zeroed before the launch).
__global__ void __launch_bounds__(256) pf_topk_kernel(const float* __restrict__ lpart, int KS,
                                                      const float* __restrict__ bias, int T, int E, int k, int H,
                                                      const uint16_t* __restrict__ x, const uint16_t* __restrict__ wsig,
                                                      float* logits, int32_t* ids, float* pw, float* gate_s,
                                                      int32_t* counts) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * 8 + warp;
    if (t >= T) return;
    float* lt = logits + (size_t)t * E;
    for (int e = lane; e < E; e += 32) {
        float l = 0.0f;
        for (int s = 0; s < KS; s++) l += lpart[((size_t)s * T + t) * E + e];
        if (bias) l += bias[e];
        lt[e] = l;
    }
    __syncwarp();
    topk_softmax_warp(lt, E, k, ids + (size_t)t * k, pw + (size_t)t * k);
    if (lane < k) atomicAdd(&counts[ids[(size_t)t * k + lane]], 1);  // lane j wrote id j itself
    if (wsig) {
        const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)t * H);
        const uint4* gr = reinterpret_cast<const uint4*>(wsig);
        float dot = 0.0f;
        for (int i = lane; i < H / 8; i += 32) {
            const uint4 v = xr[i], g = gr[i];
            const uint32_t vw[4] = {v.x, v.y, v.z, v.w}, gw[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
            for (int j = 0; j < 4; j++) {
                dot = fmaf(bf16_lo(vw[j]), bf16_lo(gw[j]), dot);
                dot = fmaf(bf16_hi(vw[j]), bf16_hi(gw[j]), dot);
            }
        }
        dot = warp_sum(dot);
        if (lane == 0) gate_s[t] = sigmoid(dot);
    }
}

// One block: offsets = exclusive scan of counts; cursor = offsets (the scatter's fill pointers).
__global__ void __launch_bounds__(1024) pf_scan_kernel(const int32_t* __restrict__ counts, int E, int32_t* offsets,
                                                       int32_t* cursor) {
    __shared__ int32_t wsum[32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = threadIdx.x;
    const int c = (e < E) ? counts[e] : 0;
    int s = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, s, o);
        if (lane >= o) s += v;
    }
    if (lane == 31) wsum[warp] = s;
    __syncthreads();
    if (warp == 0) {
        int w = (lane < (int)(blockDim.x >> 5)) ? wsum[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += v;
        }
        wsum[lane] = w;  // inclusive over warps
    }
    __syncthreads();
    const int excl = s - c + (warp > 0 ? wsum[warp - 1] : 0);
    if (e < E) {
        offsets[e] = excl;
        cursor[e] = excl;
    }
    if (e == E - 1) offsets[E] = excl + c;
}

// One warp per (token, slot) entry: claim its position in the expert's list
// (perm[pos] = t*k + slot) and copy the token's row of x, as fp16, to xs[pos].
// The order of entries inside one expert's list is arbitrary: every output of
// the expert GEMMs depends on its own entry only.
__global__ void __launch_bounds__(256) pf_scatter_kernel(const int32_t* __restrict__ ids, int n, int k, int H,
                                                         const uint16_t* __restrict__ x, int32_t* cursor,
                                                         int32_t* perm, uint16_t* xs) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int i = blockIdx.x * 8 + warp;
    if (i >= n) return;
    int pos = 0;
    if (lane == 0) {
        pos = atomicAdd(&cursor[ids[i]], 1);
        perm[pos] = i;
    }
    pos = __shfl_sync(0xffffffffu, pos, 0);
    const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)(i / k) * H);
    uint4* xo = reinterpret_cast<uint4*>(xs + (size_t)pos * H);
    for (int c = lane; c < H / 8; c += 32) {
        const uint4 v = xr[c];
        xo[c] = make_uint4(pack_h2(bf16_lo(v.x), bf16_hi(v.x)), pack_h2(bf16_lo(v.y), bf16_hi(v.y)),
                           pack_h2(bf16_lo(v.z), bf16_hi(v.z)), pack_h2(bf16_lo(v.w), bf16_hi(v.w)));
    }
}

// y[t] = (shared expert's row, already in y, or 0) + sum over the token's k slots, in slot order,
// of its fp16 routed contributions.  One thread per 8 consecutive outputs.
__global__ void __launch_bounds__(256) pf_combine_kernel(const uint16_t* __restrict__ yp, int T, int k, int H,
                                                         int has_shared, float* y) {
    const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;  // group of 8 outputs
    const size_t per_t = (size_t)H / 8;
    if (i >= (size_t)T * per_t) return;
    const size_t t = i / per_t, h0 = (i % per_t) * 8;
    float acc[8];
    float4* yo = reinterpret_cast<float4*>(y + t * H + h0);
    if (has_shared) {
        const float4 a = yo[0], b = yo[1];
        acc[0] = a.x; acc[1] = a.y; acc[2] = a.z; acc[3] = a.w;
        acc[4] = b.x; acc[5] = b.y; acc[6] = b.z; acc[7] = b.w;
    } else {
#pragma unroll
        for (int j = 0; j < 8; j++) acc[j] = 0.0f;
    }
    for (int s = 0; s < k; s++) {
        const uint4 v = *reinterpret_cast<const uint4*>(yp + (t * k + s) * H + h0);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; j++) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[j]));
            acc[2 * j] += f.x;
            acc[2 * j + 1] += f.y;
        }
    }
    yo[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    yo[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
}

// ================================================================== grouped expert GEMMs

constexpr int kNB = 6;  // B operand stages (shared memory, filled by TMA)
constexpr int kNRv = 3; // raw weight slots

struct ExpertParams {
    CUtensorMap map_q;   // routed Q2_K rows, column mode: u8 [E][rows][rowbytes], box 112 x 128 x 1
    CUtensorMap map_s0;  // shared bf16 matrix 0 (gate, or down): [rows][K], box 64 x 128, 128B swizzle
    CUtensorMap map_s1;  // shared bf16 matrix 1 (up)
    CUtensorMap map_br[3];  // B of routed units: xs [T*k][H] (gate/up) or h16 [T*k][F] (down), fp16,
                            // boxes of 64 x {128, 64, 32} rows
    CUtensorMap map_bs[3];  // B of shared units: x [T][H] (gate/up) or hs [T][S] (down), bf16, same boxes
    const uint8_t* experts;
    int64_t stride;      // bytes between experts
    int64_t q_off;       // byte offset of the first routed matrix inside an expert
    int q_rows_m1;       // row offset of routed matrix 1 (up) after matrix 0 (gate)
    int raw_mode;        // kRawColumn / kRawTile
    int rowbytes;        // routed row bytes = K/256 * 84
    int K, Ks;           // routed / shared contraction length
    int MT, MTs;         // 128-row output tiles of the routed / shared matrices
    int E, k, T, F, S, H;
    int n_sgroups;       // shared-expert token tiles (0 when there is no shared expert)
    int nt;              // token-tile height (MMA N limit)
    const int32_t* counts;
    const int32_t* offsets;
    const int32_t* perm;
    const float* pw;
    const float* gate_s;
    uint16_t* out_h;     // gate/up: h16 [T*k][F] (expert-sorted entries)
    uint16_t* out_hs;    // gate/up: hs  [T][S]
    uint16_t* yp;        // down: fp16 p * (Wd h) per (token, slot) entry [T*k][H]
    float* y;            // down: [T][H], the shared expert's contribution (stored, not added)
    uint32_t* status;
};

template <int NM>
struct ExpertCtl {
    static constexpr int NSA = (NM == 2) ? 4 : 8;  // A stages in tensor memory
    uint64_t afull[NSA], aempty[NSA];
    uint64_t bfull[kNB], bempty[kNB];
    uint64_t rawfull[kNRv], rawfree_d[kNRv], rawfree_m[kNRv];
    uint64_t accfull[2], accempty[2], drain;
    int raw_tag[kNRv];  // chunk number a raw slot is being filled with (set before the copy is issued)
    uint32_t tmem;
    int abort;
    int n_groups;
    int pad;
    int col_row[4][kNT];    // epilogue warp q: per accumulator column, its token (shared) or entry (routed)
    float col_scale[4][kNT];  // ... and the routing weight / shared gate
};

// Per-expert tables copied to shared memory at the start: unit-tile prefix, list offset, count.
struct ExpertTables {
    int* prefix;  // [E + 1]
    int* offs;    // [E]
    int* cnts;    // [E]
};

struct Unit {
    int shared;  // 1: shared-expert unit
    int e;       // expert (routed)
    int tok0;    // first token (shared) or first entry of the expert's list (routed)
    int n;       // valid B rows
    int mt;      // output row tile
    int brow;    // first B row: token (shared) or sorted entry (routed)
};

// Unit = (group g, output tile m).  Groups are token tiles: the shared expert's first, then each
// expert's.
__device__ __forceinline__ Unit make_unit(int g, int m, const ExpertParams& p, const ExpertTables& tb) {
    Unit U;
    U.mt = m;
    if (g < p.n_sgroups) {
        U.shared = 1;
        U.e = -1;
        U.tok0 = g * p.nt;
        U.n = min(p.nt, p.T - U.tok0);
        U.brow = U.tok0;
        return U;
    }
    const int gg = g - p.n_sgroups;
    int lo = 0, hi = p.E;  // largest e with prefix[e] <= gg
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (tb.prefix[mid] <= gg) lo = mid;
        else hi = mid;
    }
    U.shared = 0;
    U.e = lo;
    U.tok0 = (gg - tb.prefix[lo]) * p.nt;
    U.n = min(p.nt, tb.cnts[lo] - U.tok0);
    U.brow = tb.offs[lo] + U.tok0;
    return U;
}

// Iterate this CTA's units in order: body(U) for each; stop early when body returns false.
// Units (group-major) are dealt to CTAs one by one, for balance.
template <class Body>
__device__ __forceinline__ void for_units(const ExpertParams& p, const ExpertTables& tb, int n_groups, Body body) {
    const int n_su = p.n_sgroups * p.MTs, n_units = n_su + (n_groups - p.n_sgroups) * p.MT;
    for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
        const Unit U = (u < n_su) ? make_unit(u / p.MTs, u % p.MTs, p, tb)
                                  : make_unit(p.n_sgroups + (u - n_su) / p.MT, (u - n_su) % p.MT, p, tb);
        if (!body(U)) return;
    }
}

// Per-unit geometry shared by every role.
struct Geo {
    int KB;   // 64-wide K slices
    int nch;  // raw chunks
    int kpc;  // K slices per chunk
};
__device__ __forceinline__ Geo unit_geo(const Unit& U, const ExpertParams& p) {
    Geo g;
    if (U.shared) {
        g.KB = p.Ks / 64;
        g.nch = g.KB;
        g.kpc = 1;
    } else if (p.raw_mode == kRawColumn) {
        g.KB = p.K / 64;
        g.nch = p.K / 256;
        g.kpc = 4;
    } else {
        g.KB = p.K / 64;
        g.nch = 1;
        g.kpc = g.KB;
    }
    return g;
}

// NM = 2: gate+up (two weight matrices share the B operand); NM = 1: down.
// Warps 0..15 dequantise (routed units), 16..19 epilogue, 20 MMA (+TMEM), 21 TMA of raw weights,
// 22 TMA of B slices.
template <int NM>
__global__ void __launch_bounds__(kExpertThreads, 1) pf_expert_kernel(const __grid_constant__ ExpertParams p) {
    using Ctl = ExpertCtl<NM>;
    constexpr int NSA = Ctl::NSA;
    constexpr int NAB = (NM == 2) ? 1 : 2;           // accumulator buffers
    constexpr int kDeqPerSlice = (NM == 2) ? 8 : 4;  // dequant warps writing one A stage
    extern __shared__ uint8_t ex_smem_raw[];
    uint8_t* sm = align1024(ex_smem_raw);
    uint8_t* raw = sm;
    uint8_t* bst = sm + kNRv * kSlotBytes;
    Ctl* ctl = reinterpret_cast<Ctl*>(bst + kNB * kBStageBytes);
    ExpertTables tb;
    tb.prefix = reinterpret_cast<int*>(ctl + 1);
    tb.offs = tb.prefix + p.E + 1;
    tb.cnts = tb.offs + p.E;
    volatile int* abort = &ctl->abort;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NSA; s++) {
            mbar_init(&ctl->afull[s], kDeqPerSlice);
            mbar_init(&ctl->aempty[s], 1);
        }
        for (int s = 0; s < kNB; s++) {
            mbar_init(&ctl->bfull[s], 1);
            mbar_init(&ctl->bempty[s], 1);
        }
        for (int r = 0; r < kNRv; r++) {
            mbar_init(&ctl->rawfull[r], 1);
            mbar_init(&ctl->rawfree_d[r], kDeqWarps);
            mbar_init(&ctl->rawfree_m[r], 1);
        }
        for (int b = 0; b < 2; b++) {
            mbar_init(&ctl->accfull[b], 1);
            mbar_init(&ctl->accempty[b], 4);
        }
        mbar_init(&ctl->drain, 1);
        for (int r = 0; r < kNRv; r++) ctl->raw_tag[r] = -1;
        ctl->abort = 0;
        fence_barrier_init();
    }
    if (warp == kWarpMma) {
        tc::tmem_alloc(&ctl->tmem, 512);
        tc::tmem_relinquish();
    }
    for (int e = threadIdx.x; e < p.E; e += blockDim.x) {
        tb.offs[e] = p.offsets[e];
        tb.cnts[e] = p.counts[e];
    }
    if (warp == 0) {  // token tiles per expert: ceil(count / nt), exclusive prefix
        int carry = 0;
        for (int b = 0; b < p.E; b += 32) {
            const int e = b + lane;
            const int c = (e < p.E) ? (p.counts[e] + p.nt - 1) / p.nt : 0;
            int s = c;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, s, o);
                if (lane >= o) s += v;
            }
            if (e < p.E) tb.prefix[e] = carry + s - c;
            carry += __shfl_sync(0xffffffffu, s, 31);
        }
        if (lane == 0) {
            tb.prefix[p.E] = carry;
            ctl->n_groups = p.n_sgroups + carry;
        }
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tbase = ctl->tmem;
    const int n_groups = ctl->n_groups;

    if (warp < kDeqWarps) {
        // ---------------------------------------------------------- dequant warps: raw slot -> TMEM A stage
        // Warp w writes TMEM lane quarter q = w % 4 (rows 32q..32q+31) of matrix m (gate/up: bit 2
        // of w) for the K slices kb with kb % n_slice_groups == its group.
        const int q = warp & 3, r = 32 * q + lane;
        const int m = (NM == 2) ? ((warp >> 2) & 1) : 0;
        constexpr int kSliceGroups = (NM == 2) ? kDeqWarps / 8 : kDeqWarps / 4;
        const int grp = (NM == 2) ? (warp >> 3) : (warp >> 2);
        int G = 0, C = 0;
        int pend = -1;  // A stage whose tensor-memory store was issued but not yet signalled
        auto flush = [&]() {
            if (pend >= 0) {
                tc::wait_st();
                tc::fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&ctl->afull[pend]);
                pend = -1;
            }
        };
        for_units(p, tb, n_groups, [&](const Unit& U) -> bool {
            if (warp_aborted(abort)) return false;
            const Geo g = unit_geo(U, p);
            if (U.shared) {  // the MMA reads shared-expert tiles straight from the raw slots
                C += g.nch;
                return true;
            }
            const int nblk = (p.raw_mode == kRawColumn) ? 1 : p.K / 256;  // Q2_K blocks per row per chunk
            bool ok = true;
            for (int ch = 0; ch < g.nch && ok; ch++, C++) {
                const int slot = C % kNRv;
                // Shared-expert chunks in between are consumed by the MMA, not by these warps, so
                // they can be two fills ahead of the slot: wait for the slot to be tagged with this
                // chunk before the phase-parity wait, which cannot tell phases two apart.
                ok = warp_wait_tag(&ctl->raw_tag[slot], C, abort, p.status, 2) &&
                     warp_wait(&ctl->rawfull[slot], (C / kNRv) & 1, abort, p.status, 1, C);
                if (!ok) break;
                const uint8_t* sl = raw + slot * kSlotBytes + m * kMatStride;
#pragma unroll 1
                for (int blk = 0; blk < nblk && ok; blk++) {
                    uint32_t w[21];
                    if (p.raw_mode == kRawColumn) {
                        uint32_t win[24];
                        const uint8_t* row = sl + r * kColBox;
#pragma unroll
                        for (int c = 0; c < 6; c++) {
                            const uint4 x4 = *reinterpret_cast<const uint4*>(row + 16 * c);
                            win[4 * c] = x4.x;
                            win[4 * c + 1] = x4.y;
                            win[4 * c + 2] = x4.z;
                            win[4 * c + 3] = x4.w;
                        }
                        switch (((84 * ch) & 15) >> 2) {
#define QS_SEL(O) \
    case O:       \
        _Pragma("unroll") for (int i = 0; i < 21; i++) w[i] = win[i + O]; \
        break;
                            QS_SEL(0) QS_SEL(1) QS_SEL(2) QS_SEL(3)
#undef QS_SEL
                        }
                    } else {
                        const uint32_t* row = reinterpret_cast<const uint32_t*>(sl + (size_t)r * p.rowbytes + 84 * blk);
#pragma unroll
                        for (int i = 0; i < 21; i++) w[i] = row[i];
                    }
                    const float d = __half2float(__ushort_as_half((unsigned short)(w[20] & 0xffffu)));
                    const float dm = __half2float(__ushort_as_half((unsigned short)(w[20] >> 16)));
                    const int kb0 = (p.raw_mode == kRawColumn ? 4 * ch : 4 * blk);
#pragma unroll 1
                    for (int c = 0; c < 4 && ok; c++) {
                        const int kb = kb0 + c;
                        if (kb % kSliceGroups != grp) continue;
                        const uint32_t scw = (c == 0) ? w[0] : (c == 1) ? w[1] : (c == 2) ? w[2] : w[3];
                        uint32_t qw[8];
#pragma unroll
                        for (int i = 0; i < 8; i++) qw[i] = (c >= 2) ? w[12 + i] : w[4 + i];
                        uint32_t v[16];
                        dequant_half(scw, qw, c, 0, d, dm, v);
                        // signal the previous slice (its stores have overlapped this slice's
                        // dequantisation), wait for this slice's A stage, store this row's 32 columns
                        const int Gk = G + kb, s = Gk % NSA;
                        flush();
                        if (Gk >= NSA && !warp_wait(&ctl->aempty[s], ((Gk / NSA) - 1) & 1, abort, p.status, 3, Gk)) {
                            ok = false;
                            break;
                        }
                        tc::fence_after();
                        const uint32_t ta = tc::taddr(tbase, 32 * q, kA0 + s * 32 * NM + m * 32);
                        tc::st16(ta, v);
                        dequant_half(scw, qw, c, 1, d, dm, v);
                        tc::st16(ta + 16, v);
                        pend = s;
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&ctl->rawfree_d[slot]);
            }
            flush();  // before the next unit: the MMA must be able to finish this one
            G += g.KB;
            return ok;
        });
        flush();
    } else if (warp < kWarpMma) {
        // ---------------------------------------------------------- epilogue warps
        const int q = warp & 3, row = 32 * q + lane;
        int* crow = ctl->col_row[q];
        float* cscale = ctl->col_scale[q];
        int V = 0;
        for_units(p, tb, n_groups, [&](const Unit& U) -> bool {
            if (warp_aborted(abort)) return false;
            const int b = V % NAB;
            if (NM == 1) {  // column metadata of this unit, read back as broadcasts below
                for (int n = lane; n < U.n; n += 32) {
                    if (U.shared) {
                        crow[n] = U.tok0 + n;
                        cscale[n] = p.gate_s[U.tok0 + n];
                    } else {
                        const int ent = p.perm[U.brow + n];
                        crow[n] = ent;
                        cscale[n] = p.pw[ent];
                    }
                }
                __syncwarp();
            }
            if (!warp_wait(&ctl->accfull[b], (V / NAB) & 1, abort, p.status, 4, V)) return false;
            tc::fence_after();
            const int o = U.mt * 128 + row;  // output feature (gate/up: f; down: h)
            if (NM == 2) {
                uint16_t* dst = U.shared ? p.out_hs + (size_t)U.tok0 * p.S + o : p.out_h + (size_t)U.brow * p.F + o;
                const size_t ld = U.shared ? (size_t)p.S : (size_t)p.F;
#pragma unroll 1
                for (int c0 = 0; c0 < U.n; c0 += 16) {  // warp-uniform
                    uint32_t gv[16], uv[16];
                    tc::ld16(tc::taddr(tbase, 32 * q, c0), gv);
                    tc::ld16(tc::taddr(tbase, 32 * q, 128 + c0), uv);
                    tc::wait_ld();
#pragma unroll
                    for (int i = 0; i < 16; i++) {
                        if (c0 + i < U.n) {
                            const float gq = __uint_as_float(gv[i]);
                            const float hv = __fdividef(gq, 1.0f + __expf(-gq)) * __uint_as_float(uv[i]);
                            dst[(size_t)(c0 + i) * ld] = U.shared ? __bfloat16_as_ushort(__float2bfloat16_rn(hv))
                                                                  : __half_as_ushort(__float2half_rn(hv));
                        }
                    }
                }
            } else {
#pragma unroll 1
                for (int c0 = 0; c0 < U.n; c0 += 32) {  // warp-uniform
                    uint32_t av[32];
                    tc::ld32(tc::taddr(tbase, 32 * q, b * 128 + c0), av);
                    tc::wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; i++) {
                        if (c0 + i < U.n) {
                            const int rr = crow[c0 + i];  // token (shared) or entry (routed)
                            const float v = cscale[c0 + i] * __uint_as_float(av[i]);
                            if (U.shared) p.y[(size_t)rr * p.H + o] = v;
                            else p.yp[(size_t)rr * p.H + o] = __half_as_ushort(__float2half_rn(v));
                        }
                    }
                }
            }
            tc::fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl->accempty[b]);
            V++;
            return true;
        });
    } else if (warp == kWarpMma) {
        // ---------------------------------------------------------- MMA issuer
        // The whole warp runs the loop (its values are warp-uniform, so the MMA operands need no
        // per-instruction move into the uniform datapath); lane 0 issues the MMAs and commits.
        const uint32_t tmu = __shfl_sync(0xffffffffu, tbase, 0);
        const bool leader = lane == 0;
        int GA = 0, GB = 0, C = 0, V = 0;
        for_units(p, tb, n_groups, [&](const Unit& U) -> bool {
            if (warp_aborted(abort)) return false;
            const Geo g = unit_geo(U, p);
            const int b = V % NAB;
            if (V >= NAB && !warp_wait(&ctl->accempty[b], ((V / NAB) - 1) & 1, abort, p.status, 5, V)) return false;
            tc::fence_after();
            const int nmma = max(16, (U.n + 15) & ~15);
            const uint32_t id = tc::idesc(U.shared ? tc::kBF16 : tc::kF16, 128, nmma);
            for (int kb = 0; kb < g.KB; kb++) {
                const int sb = (GB + kb) % kNB;
                if (!warp_wait(&ctl->bfull[sb], ((GB + kb) / kNB) & 1, abort, p.status, 6, GB + kb)) return false;
                const uint64_t bd = tc::sdesc_sw128(smem_u32(bst + sb * kBStageBytes));
                if (U.shared) {
                    const int c = C + kb, slot = c % kNRv;
                    if (!warp_wait(&ctl->rawfull[slot], (c / kNRv) & 1, abort, p.status, 7, c)) return false;
                    tc::fence_after();
                    const uint32_t sa = smem_u32(raw + slot * kSlotBytes);
                    if (leader) {
#pragma unroll
                        for (int mq = 0; mq < NM; mq++) {
                            const uint32_t d = tmu + (NM == 2 ? mq * 128 : b * 128);
                            const uint64_t ad = tc::sdesc_sw128(sa + mq * kMatStride);
#pragma unroll
                            for (int k16 = 0; k16 < 4; k16++)
                                tc::mma_ss_f16(d, ad + 2 * k16, bd + 2 * k16, id, (kb | k16) != 0);
                        }
                        tc::commit(&ctl->rawfree_m[slot]);
                    }
                } else {
                    const int Gk = GA + kb, s = Gk % NSA;
                    if (!warp_wait(&ctl->afull[s], (Gk / NSA) & 1, abort, p.status, 8, Gk)) return false;
                    tc::fence_after();
                    if (leader) {
#pragma unroll
                        for (int mq = 0; mq < NM; mq++) {
                            const uint32_t d = tmu + (NM == 2 ? mq * 128 : b * 128);
                            const uint32_t a = tmu + kA0 + s * 32 * NM + mq * 32;
#pragma unroll
                            for (int k16 = 0; k16 < 4; k16++)
                                tc::mma_ts_f16(d, a + 8 * k16, bd + 2 * k16, id, (kb | k16) != 0);
                        }
                        tc::commit(&ctl->aempty[s]);
                    }
                }
                if (leader) tc::commit(&ctl->bempty[sb]);
                __syncwarp();
            }
            if (leader) tc::commit(&ctl->accfull[b]);
            __syncwarp();
            GB += g.KB;
            C += g.nch;
            if (!U.shared) GA += g.KB;
            V++;
            return true;
        });
        if (leader) {
            tc::commit(&ctl->drain);  // completes once every MMA issued above has
            (void)mbar_wait(&ctl->drain, 0);
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------- TMA: raw weights (warp 13), B slices (warp 14)
        const bool do_raw = (warp == kWarpRaw), do_b = (warp == kWarpB);
        if (lane == 0) {
            int C = 0, GB = 0;
            int used_d[kNRv] = {}, used_m[kNRv] = {}, last_use[kNRv];  // last consumer: 0 none, 1 dequant, 2 MMA
            for (int i = 0; i < kNRv; i++) last_use[i] = 0;
            for_units(p, tb, n_groups, [&](const Unit& U) -> bool {
                if (*abort) return false;
                const Geo g = unit_geo(U, p);
                const int row0 = U.mt * 128;
                for (int kb = 0; kb < g.KB; kb++) {
                    if (do_raw && kb % g.kpc == 0) {  // next raw chunk
                        const int ch = kb / g.kpc, slot = C % kNRv;
                        bool ok = true;
                        if (last_use[slot] == 1) {
                            ok = thread_wait(&ctl->rawfree_d[slot], used_d[slot] & 1, abort, p.status, 9, C);
                            used_d[slot]++;
                        } else if (last_use[slot] == 2) {
                            ok = thread_wait(&ctl->rawfree_m[slot], used_m[slot] & 1, abort, p.status, 10, C);
                            used_m[slot]++;
                        }
                        if (!ok) return false;
                        last_use[slot] = U.shared ? 2 : 1;
                        *reinterpret_cast<volatile int*>(&ctl->raw_tag[slot]) = C;
                        uint8_t* sl = raw + slot * kSlotBytes;
                        uint64_t* bar = &ctl->rawfull[slot];
                        if (U.shared) {
                            mbar_arrive_expect_tx(bar, NM * 16384);
                            tma_load_2d(sl, &p.map_s0, ch * 64, row0, bar);
                            if (NM == 2) tma_load_2d(sl + kMatStride, &p.map_s1, ch * 64, row0, bar);
                        } else if (p.raw_mode == kRawColumn) {
                            mbar_arrive_expect_tx(bar, NM * kColBox * 128);
                            const int x0 = (84 * ch) & ~15;
                            tma_load_3d(sl, &p.map_q, x0, row0, U.e, bar);
                            if (NM == 2) tma_load_3d(sl + kMatStride, &p.map_q, x0, p.q_rows_m1 + row0, U.e, bar);
                        } else {
                            const uint32_t bytes = 128u * (uint32_t)p.rowbytes;
                            mbar_arrive_expect_tx(bar, NM * bytes);
                            const uint8_t* src =
                                p.experts + (size_t)U.e * p.stride + p.q_off + (size_t)row0 * p.rowbytes;
                            bulk_g2s(sl, src, bytes, bar);
                            if (NM == 2) bulk_g2s(sl + kMatStride, src + (size_t)p.q_rows_m1 * p.rowbytes, bytes, bar);
                        }
                        C++;
                    }
                    // B slice: the unit's rows only (one 128-row box, or 64 and/or 32-row boxes),
                    // once the stage's previous slice is released.
                    if (!do_b) continue;
                    const int sb = GB % kNB;
                    if (GB >= kNB && !thread_wait(&ctl->bempty[sb], ((GB / kNB) - 1) & 1, abort, p.status, 11, GB))
                        return false;
                    const CUtensorMap* mp = U.shared ? p.map_bs : p.map_br;
                    uint8_t* bs = bst + sb * kBStageBytes;
                    const int r128 = U.n > 96 ? 128 : 0;
                    const int r64 = (r128 == 0 && U.n > 32) ? 64 : 0;
                    const int r32 = (r128 == 0 && U.n - r64 > 0) ? 32 : 0;
                    mbar_arrive_expect_tx(&ctl->bfull[sb], (uint32_t)(r128 + r64 + r32) * 128u);
                    if (r128) tma_load_2d(bs, &mp[0], kb * 64, U.brow, &ctl->bfull[sb]);
                    if (r64) tma_load_2d(bs, &mp[1], kb * 64, U.brow, &ctl->bfull[sb]);
                    if (r32) tma_load_2d(bs + r64 * 128, &mp[2], kb * 64, U.brow + r64, &ctl->bfull[sb]);
                    GB++;
                }
                return true;
            });
            if (*abort) {  // let issued copies land before the CTA exits
                for (int i = 1; do_raw && i <= kNRv && i <= C; i++) {
                    const int c = C - i;
                    (void)mbar_wait(&ctl->rawfull[c % kNRv], (c / kNRv) & 1, 1000000ull);
                }
                for (int i = 1; do_b && i <= kNB && i <= GB; i++) {
                    const int c = GB - i;
                    (void)mbar_wait(&ctl->bfull[c % kNB], (c / kNB) & 1, 1000000ull);
                }
            }
        }
    }

    tc::fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
        tc::fence_after();
        tc::tmem_dealloc(tbase, 512);
    }
}

// ================================================================== host side

using EncodeFn = PFN_cuTensorMapEncodeTiled_v12000;

EncodeFn get_encode() {
    static std::once_flag once;
    static EncodeFn fn = nullptr;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeFn>(f);
    });
    return fn;
}

bool encode(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* base, const uint64_t* dims,
            const uint64_t* strides, const uint32_t* box, CUtensorMapSwizzle sw) {
    EncodeFn fn = get_encode();
    if (!fn) return false;
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, dt, (cuuint32_t)rank, const_cast<void*>(base), reinterpret_cast<const cuuint64_t*>(dims),
              reinterpret_cast<const cuuint64_t*>(strides), reinterpret_cast<const cuuint32_t*>(box), es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D map over a row-major [rows][K] 16-bit matrix, box 64 x box_rows, 128-byte swizzle.
bool encode_rows16(CUtensorMap* m, CUtensorMapDataType dt, const void* base, int K, int64_t rows,
                   uint32_t box_rows = 128) {
    const uint64_t d[2] = {(uint64_t)K, (uint64_t)rows}, s[1] = {(uint64_t)K * 2};
    const uint32_t b[2] = {64, box_rows};
    return encode(m, dt, 2, base, d, s, b, CU_TENSOR_MAP_SWIZZLE_128B);
}
// The three B maps (box heights 128, 64, 32) of one operand.
bool encode_b(CUtensorMap* m3, CUtensorMapDataType dt, const void* base, int K, int64_t rows) {
    return encode_rows16(&m3[0], dt, base, K, rows, 128) && encode_rows16(&m3[1], dt, base, K, rows, 64) &&
           encode_rows16(&m3[2], dt, base, K, rows, 32);
}

// Raw-weight staging mode for a Q2_K matrix with contraction length K, or -1.
int raw_mode_for(int K, int nm) {
    const int rowbytes = K / 256 * 84;
    if (rowbytes % 16 == 0) return kRawColumn;
    if (128 * rowbytes <= (nm == 2 ? kMatStride : kSlotBytes)) return kRawTile;
    return -1;
}

struct PfFacts {
    int n_sm = 0;
    int smem_optin = 0;
    bool attr_set = false;
};

cudaError_t pf_facts(PfFacts** out) {
    static std::mutex mu;
    static PfFacts facts[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    PfFacts& f = facts[dev];
    if (f.n_sm == 0) {
        if ((e = cudaDeviceGetAttribute(&f.n_sm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
        if ((e = cudaDeviceGetAttribute(&f.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess)
            return e;
    }
    *out = &f;
    return cudaSuccess;
}

template <int NM>
size_t expert_smem(int E) {
    return 1024 + kNRv * kSlotBytes + kNB * kBStageBytes + sizeof(ExpertCtl<NM>) + 4 * (3 * E + 1);
}
size_t router_smem() { return 1024 + kRouterStages * 4 * 16384 + sizeof(RouterCtl); }

// Launch one expert kernel, one CTA per SM.
template <int NM>
cudaError_t launch_expert(ExpertParams& p, int n_sm, int E, cudaStream_t st) {
    pf_expert_kernel<NM><<<n_sm, kExpertThreads, expert_smem<NM>(E), st>>>(p);
    return cudaGetLastError();
}

int router_splits(int E, int T, int H, int n_sm) {
    const int tiles = ((E + 127) / 128) * ((T + 127) / 128);
    int ks = 1;
    while (ks < kMaxKS && tiles * ks * 2 <= n_sm && (H / 64) % (ks * 2) == 0) ks *= 2;
    return ks;
}

}  // namespace

bool prefill_shape_ok(const qs_moe_shape& s) {
    if (s.x_dtype != QS_BF16) return false;
    if (raw_mode_for(s.hidden, 2) < 0 || raw_mode_for(s.expert_ffn, 1) < 0) return false;
    if (s.shared_ffn % 128) return false;
    return true;
}

int prefill_launches() { return 8; }

cudaError_t launch_prefill(const qs_moe_shape& s, const void* x, const float* Wr, const float* bias,
                           const uint8_t* experts, int64_t stride, const uint16_t* sg, const uint16_t* su,
                           const uint16_t* sd, const uint16_t* ssig, int T, float* out, void* ws, const WsLayout& W,
                           cudaStream_t st) {
    if (!prefill_shape_ok(s)) return cudaErrorNotSupported;
    PfFacts* f = nullptr;
    cudaError_t e = pf_facts(&f);
    if (e != cudaSuccess) return e;
    const int H = s.hidden, E = s.n_experts, k = s.top_k, F = s.expert_ffn;
    const int S = (sg != nullptr) ? s.shared_ffn : 0;
    const int n = T * k;
    if ((size_t)f->smem_optin < expert_smem<2>(1024) || (size_t)f->smem_optin < expert_smem<1>(1024) ||
        (size_t)f->smem_optin < router_smem())
        return cudaErrorNotSupported;
    if (!get_encode()) return cudaErrorNotSupported;
    if (!f->attr_set) {
        if ((e = cudaFuncSetAttribute(pf_router_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)router_smem())) != cudaSuccess)
            return e;
        if ((e = cudaFuncSetAttribute(pf_expert_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)expert_smem<2>(1024))) != cudaSuccess)
            return e;
        if ((e = cudaFuncSetAttribute(pf_expert_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)expert_smem<1>(1024))) != cudaSuccess)
            return e;
        f->attr_set = true;
    }
    uint8_t* base = static_cast<uint8_t*>(ws);
    uint32_t* status = reinterpret_cast<uint32_t*>(base + W.header);
    uint16_t* wr3 = reinterpret_cast<uint16_t*>(base + W.wr3);
    float* lpart = reinterpret_cast<float*>(base + W.lpart);
    float* logits = reinterpret_cast<float*>(base + W.logits);
    int32_t* ids = reinterpret_cast<int32_t*>(base + W.ids);
    float* pw = reinterpret_cast<float*>(base + W.pw);
    int32_t* counts = reinterpret_cast<int32_t*>(base + W.counts);
    int32_t* offsets = reinterpret_cast<int32_t*>(base + W.offsets);
    int32_t* perm = reinterpret_cast<int32_t*>(base + W.perm);
    int32_t* cursor = reinterpret_cast<int32_t*>(base + W.cursor);
    uint16_t* xs = reinterpret_cast<uint16_t*>(base + W.xs);
    uint16_t* h16 = reinterpret_cast<uint16_t*>(base + W.h16);
    uint16_t* hs16 = reinterpret_cast<uint16_t*>(base + W.hs16);
    float* gate = reinterpret_cast<float*>(base + W.gate);

    // tensor maps (host-side encodings of the operands' shapes; no device work)
    RouterParams rp;
    {
        const uint64_t wd[3] = {(uint64_t)H, (uint64_t)E, 3}, ws_[2] = {(uint64_t)H * 2, (uint64_t)E * H * 2};
        const uint32_t wb[3] = {64, 128, 1};
        if (!encode(&rp.map_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, wr3, wd, ws_, wb, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !encode_rows16(&rp.map_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, H, T))
            return cudaErrorInvalidValue;
    }
    ExpertParams ep[2];
    for (int nm = 2; nm >= 1; nm--) {
        ExpertParams& p = ep[nm - 1];
        memset(&p, 0, sizeof(p));
        const int K = (nm == 2) ? H : F;
        const int rowbytes = K / 256 * 84;
        p.raw_mode = raw_mode_for(K, nm);
        p.rowbytes = rowbytes;
        p.experts = experts;
        p.stride = stride;
        p.q_off = (nm == 2) ? 0 : (int64_t)2 * F * (H / 256 * 84);
        p.q_rows_m1 = (nm == 2) ? F : 0;
        const int rows = (nm == 2) ? 2 * F : H;
        if (p.raw_mode == kRawColumn) {
            const uint64_t d[3] = {(uint64_t)rowbytes, (uint64_t)rows, (uint64_t)E};
            const uint64_t sd_[2] = {(uint64_t)rowbytes, (uint64_t)stride};
            const uint32_t b[3] = {kColBox, 128, 1};
            if (!encode(&p.map_q, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, experts + p.q_off, d, sd_, b,
                        CU_TENSOR_MAP_SWIZZLE_NONE))
                return cudaErrorInvalidValue;
        }
        if (!encode_b(p.map_br, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, nm == 2 ? xs : h16, K, n))
            return cudaErrorInvalidValue;
        p.K = K;
        p.MT = ((nm == 2) ? F : H) / 128;
        p.nt = kNT;
        p.E = E;
        p.k = k;
        p.T = T;
        p.F = F;
        p.S = S;
        p.H = H;
        if (S > 0) {
            p.Ks = (nm == 2) ? H : S;
            p.MTs = ((nm == 2) ? S : H) / 128;
            p.n_sgroups = (T + p.nt - 1) / p.nt;
            bool ok;
            if (nm == 2)
                ok = encode_rows16(&p.map_s0, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, sg, H, S) &&
                     encode_rows16(&p.map_s1, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, su, H, S) &&
                     encode_b(p.map_bs, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, H, T);
            else
                ok = encode_rows16(&p.map_s0, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, sd, S, H) &&
                     encode_b(p.map_bs, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, hs16, S, T);
            if (!ok) return cudaErrorInvalidValue;
        } else {
            p.Ks = 64;
            p.MTs = p.MT;
            p.n_sgroups = 0;
        }
        p.counts = counts;
        p.offsets = offsets;
        p.perm = perm;
        p.pw = pw;
        p.gate_s = gate;
        p.out_h = h16;
        p.out_hs = hs16;
        p.yp = xs;  // the expert-sorted x rows are dead once gate+up has run
        p.y = out;
        p.status = status;
    }

    // (0) zero the expert counts
    if ((e = cudaMemsetAsync(counts, 0, (size_t)E * sizeof(int32_t), st)) != cudaSuccess) return e;
    // (1) router planes, partial logits
    {
        const size_t nw = (size_t)E * H;
        const int blocks = (int)std::min<size_t>((nw + 255) / 256, (size_t)f->n_sm * 8);
        pf_router_split_kernel<<<blocks, 256, 0, st>>>(Wr, nw, wr3);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        const int KS = router_splits(E, T, H, f->n_sm);
        rp.lpart = lpart;
        rp.E = E;
        rp.T = T;
        rp.KBc = H / 64 / KS;
        rp.status = status;
        dim3 grid((E + 127) / 128, (T + 127) / 128, KS);
        pf_router_mma_kernel<<<grid, kRouterThreads, router_smem(), st>>>(rp);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        // (2) top-k, softmax, shared gate, expert counts
        pf_topk_kernel<<<(T + 7) / 8, 256, 0, st>>>(lpart, KS, bias, T, E, k, H, static_cast<const uint16_t*>(x), ssig,
                                                    logits, ids, pw, gate, counts);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    // (3) offsets, (4) entry positions + expert-sorted fp16 token rows
    pf_scan_kernel<<<1, 1024, 0, st>>>(counts, E, offsets, cursor);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    pf_scatter_kernel<<<(n + 7) / 8, 256, 0, st>>>(ids, n, k, H, static_cast<const uint16_t*>(x), cursor, perm, xs);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // (5) gate+up, (6) down
    if ((e = launch_expert<2>(ep[1], f->n_sm, E, st)) != cudaSuccess) return e;
    if ((e = launch_expert<1>(ep[0], f->n_sm, E, st)) != cudaSuccess) return e;
    // (7) y = shared + sum of the routed contributions
    const size_t groups = (size_t)T * H / 8;
    pf_combine_kernel<<<(unsigned)((groups + 255) / 256), 256, 0, st>>>(xs, T, k, H, S > 0, out);
    return cudaGetLastError();
}

}  // namespace qs

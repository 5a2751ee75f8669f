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
#include "qs_warp.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>
#include <mutex>

namespace qs {
namespace {

constexpr int kNT = 128;                  // max tokens per unit (MMA M: token rows)
constexpr int kWRows = 256;               // weight rows per unit (MMA N)
constexpr int kColBox = 112;              // bytes per row of a Q2_K column box (covers 84 + offset <= 12)
constexpr int kHalfSlot = 128 * kColBox;  // 128 rows of a column box
constexpr int kColSlot = 2 * kHalfSlot;   // raw slot of a column chunk: 256 rows of a column box
constexpr int kMaxSlot = 32768;           // largest raw slot: 128 whole rows of at most 256 bytes
constexpr int kABytes = kNT * 128;        // A stage: 128 token rows x 64 16-bit values (128-byte swizzle)
constexpr int kWBytes = kWRows * 128;     // W stage: 256 weight rows x 64 16-bit values (128-byte swizzle)
constexpr int kDeqWarps = 16;             // dequant warps of an expert kernel
constexpr int kWarpMma = kDeqWarps + 4;   // MMA issuer (+ TMEM allocation)
constexpr int kWarpRaw = kDeqWarps + 5;   // TMA of raw Q2_K weights and of the shared expert's W tiles
constexpr int kWarpA = kDeqWarps + 6;     // TMA of token rows (the A operand)
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

// `count` arrivals on an mbarrier at once.
__device__ __forceinline__ void mbar_arrive_count(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
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
// The same wait observed by lane 0 alone: the outcome reaches the warp through __syncwarp,
// which also orders the other lanes' later memory accesses after lane 0's acquire.  For
// warps whose lanes act on the phase only through lane 0 (the MMA issuer), or write what
// the phase released only after the barrier.
__device__ __forceinline__ bool lead_wait(uint64_t* bar, uint32_t parity, volatile int* abort, uint32_t* status,
                                          uint32_t code = 0, uint32_t counter = 0) {
    int ok = 1;
    if ((threadIdx.x & 31) == 0 && !mbar_try_wait(bar, parity)) {
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
    __syncwarp();
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
    int id;
    float w;
    if (E <= 256) warp_topk<8>(lt, E, k, id, w);  // each lane reads back the logits it stored
    else warp_topk_stream(lt, E, k, id, w);
    if (lane < k) {
        ids[(size_t)t * k + lane] = id;
        pw[(size_t)t * k + lane] = w;
        atomicAdd(&counts[id], 1);
    }
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

constexpr int kMaxNA = 6;  // A stages (token rows, filled by TMA): as many as shared memory holds
constexpr int kMaxNW = 3;  // W stages (dequantised weight rows, or the shared expert's bf16 rows by TMA)
constexpr int kMaxRv = 4;  // raw Q2_K slots: three column chunks, or four half-units of whole rows

struct ExpertParams {
    CUtensorMap map_q;   // routed Q2_K rows, column mode: u8 [E][rows][rowbytes], box 112 x 128 x 1
    CUtensorMap map_s0;  // shared bf16 matrix 0 (gate, or down): [rows][K], box 64 x 128, 128B swizzle
    CUtensorMap map_s1;  // shared bf16 matrix 1 (up)
    CUtensorMap map_br[3];  // A of routed units: xs [T*k][H] (gate/up) or h16 [T*k][F] (down), fp16,
                            // boxes of 64 x {128, 64, 32} rows
    CUtensorMap map_bs[3];  // A of shared units: x [T][H] (gate/up) or hs [T][S] (down), bf16, same boxes
    const uint8_t* experts;
    int64_t stride;      // bytes between experts
    int64_t q_off;       // byte offset of the first routed matrix inside an expert
    int q_rows_m1;       // row offset of routed matrix 1 (up) after matrix 0 (gate)
    int raw_mode;        // kRawColumn / kRawTile
    int rowbytes;        // routed row bytes = K/256 * 84
    int K, Ks;           // routed / shared contraction length
    int MT, MTs;         // output tiles of the routed / shared matrices (128 gate + 128 up rows, or 256 rows)
    int E, k, T, F, S, H;
    int n_sgroups;       // shared-expert token tiles (0 when there is no shared expert)
    int nt;              // token-tile height (MMA M)
    int na;              // A stages
    int slot;            // raw slot bytes (kColSlot, or 128 whole rows)
    int nrv;             // raw slots
    int nw;              // W stages
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

struct ExpertCtl {
    uint64_t afull[kMaxNA], aempty[kMaxNA];
    uint64_t wfull[kMaxNW], wempty[kMaxNW];
    uint64_t rawfull[kMaxRv], rawfree[kMaxRv];
    uint64_t accfull[2], accempty[2], drain;
    uint32_t tmem;
    int abort;
    int n_groups;
    int pad;
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
    int n;       // valid token rows
    int mt;      // output tile
    int brow;    // first token row: token (shared) or sorted entry (routed)
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
// Units (group-major) are dealt to CTAs one by one, for balance; a CTA's shared-expert units
// come before its routed ones.
template <class Body>
__device__ __forceinline__ void for_units(const ExpertParams& p, const ExpertTables& tb, int n_groups, Body body) {
    const int n_su = p.n_sgroups * p.MTs, n_units = n_su + (n_groups - p.n_sgroups) * p.MT;
    for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
        const Unit U = (u < n_su) ? make_unit(u / p.MTs, u % p.MTs, p, tb)
                                  : make_unit(p.n_sgroups + (u - n_su) / p.MT, (u - n_su) % p.MT, p, tb);
        if (!body(U)) return;
    }
}

// 64-wide K slices of a unit, and its raw Q2_K chunks: a column of blocks for all 256 weight
// rows (column mode), or 128 whole rows (tile mode: two chunks per unit); none for shared units.
__device__ __forceinline__ int unit_kb(const Unit& U, const ExpertParams& p) { return (U.shared ? p.Ks : p.K) / 64; }
__device__ __forceinline__ int unit_nch(const Unit& U, const ExpertParams& p) {
    return U.shared ? 0 : (p.raw_mode == kRawColumn ? p.K / 256 : 2);
}

// One thread's half row of a W stage: the 16 words (32 fp16 weights, K positions 32 jj .. 32 jj + 31
// of the slice) of weight row r, stored at their 128-byte-swizzled places.
__device__ __forceinline__ void store_w_half(uint8_t* wst, int r, int jj, const uint32_t (&v)[16]) {
    const uint32_t row = smem_u32(wst) + (uint32_t)r * 128u;
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const uint32_t a = row + ((uint32_t)((4 * jj + i) ^ (r & 7)) << 4);
        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(v[4 * i]), "r"(v[4 * i + 1]),
                     "r"(v[4 * i + 2]), "r"(v[4 * i + 3])
                     : "memory");
    }
}

// W stage of fill g and how many fills of that stage came before (NW is 2 or 3: divisions by
// constants).
__device__ __forceinline__ void w_stage(int g, int NW, int& s, int& fill) {
    if (NW == 2) {
        s = g & 1;
        fill = g >> 1;
    } else {
        s = g % 3;
        fill = g / 3;
    }
}

__device__ __forceinline__ uint4 lds128(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}

// NM = 2: gate+up (the unit's W rows are 128 gate rows, then the same 128 up rows);
// NM = 1: down (256 rows of one matrix).  D[token][weight row] accumulates in tensor memory
// (M = 128 token rows, N = 256 weight rows per MMA; two accumulator buffers).
// Warps 0..15 dequantise (routed units), 16..19 epilogue, 20 MMA (+TMEM), 21 TMA of raw weights
// and of the shared expert's W tiles, 22 TMA of token rows.
template <int NM>
__global__ void __launch_bounds__(kExpertThreads, 1) pf_expert_kernel(const __grid_constant__ ExpertParams p) {
    extern __shared__ uint8_t ex_smem_raw[];
    uint8_t* sm = align1024(ex_smem_raw);
    const int NA = p.na, SLOT = p.slot, NRV = p.nrv, NW = p.nw;
    uint8_t* ast = sm;                       // NA x kABytes
    uint8_t* wst = ast + NA * kABytes;       // NW x kWBytes
    uint8_t* raw = wst + NW * kWBytes;      // NRV x SLOT
    ExpertCtl* ctl = reinterpret_cast<ExpertCtl*>(raw + NRV * SLOT);
    ExpertTables tb;
    tb.prefix = reinterpret_cast<int*>(ctl + 1);
    tb.offs = tb.prefix + p.E + 1;
    tb.cnts = tb.offs + p.E;
    volatile int* abort = &ctl->abort;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NA; s++) {
            mbar_init(&ctl->afull[s], 1);
            mbar_init(&ctl->aempty[s], 1);
        }
        for (int s = 0; s < NW; s++) {
            mbar_init(&ctl->wfull[s], kDeqWarps / 2);
            mbar_init(&ctl->wempty[s], 1);
        }
        for (int r = 0; r < NRV; r++) {
            mbar_init(&ctl->rawfull[r], 1);
            mbar_init(&ctl->rawfree[r], kDeqWarps);
        }
        for (int b = 0; b < 2; b++) {
            mbar_init(&ctl->accfull[b], 1);
            mbar_init(&ctl->accempty[b], 4);
        }
        mbar_init(&ctl->drain, 1);
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
        // ---------------------------------------------------------- dequant warps: raw slot -> W stage
        // Thread: weight row r of the unit (gate/up: rows 0..127 gate, 128..255 up), both K halves
        // of the slices of its group's parity (warps 0..7 even slices, 8..15 odd).  A stage is full
        // once the eight warps of its group have stored their rows.
        const int r = 32 * (warp & 7) + lane, grp = warp >> 3;
        int GW = 0, C = 0;
        for_units(p, tb, n_groups, [&](const Unit& U) -> bool {
            if (warp_aborted(abort)) return false;
            const int KB = unit_kb(U, p);
            if (U.shared) {  // the raw-weight thread loads these W tiles
                GW += KB;
                return true;
            }
            // one 64-wide slice: weights of row r from the block words w[] -> W stage (GW + kb)
            auto slice = [&](int kb, int c, uint32_t scw, const uint32_t (&qw)[8], float d, float dm) -> bool {
                const int g = GW + kb;
                int s, fill;
                w_stage(g, NW, s, fill);
                uint32_t v[16];
                dequant_half(scw, qw, c, 0, d, dm, v);
                if (fill > 0 && !lead_wait(&ctl->wempty[s], (fill - 1) & 1, abort, p.status, 3, g)) return false;
                store_w_half(wst + s * kWBytes, r, 0, v);
                dequant_half(scw, qw, c, 1, d, dm, v);
                store_w_half(wst + s * kWBytes, r, 1, v);
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // generic stores -> MMA reads
                __syncwarp();
                if (lane == 0) mbar_arrive(&ctl->wfull[s]);
                return true;
            };
            if (p.raw_mode == kRawColumn) {
                const int nch = p.K / 256;
#pragma unroll 1
                for (int ch = 0; ch < nch; ch++, C++) {
                    const int slot = C % NRV;
                    if (!warp_wait(&ctl->rawfull[slot], (C / NRV) & 1, abort, p.status, 1, C)) return false;
                    // the block starts (84 ch) mod 16 bytes into the 112-byte row of the column box
                    const uint32_t row = smem_u32(raw + slot * SLOT) + (uint32_t)r * kColBox;
                    uint32_t win[24], w[21];
#pragma unroll
                    for (int i = 0; i < 6; i++) {
                        const uint4 x4 = lds128(row + 16 * i);
                        win[4 * i] = x4.x;
                        win[4 * i + 1] = x4.y;
                        win[4 * i + 2] = x4.z;
                        win[4 * i + 3] = x4.w;
                    }
                    switch (ch & 3) {
#define QS_SEL(O) \
    case O:       \
        _Pragma("unroll") for (int i = 0; i < 21; i++) w[i] = win[i + O]; \
        break;
                        QS_SEL(0) QS_SEL(1) QS_SEL(2) QS_SEL(3)
#undef QS_SEL
                    }
                    const float d = __half2float(__ushort_as_half((unsigned short)(w[20] & 0xffffu)));
                    const float dm = __half2float(__ushort_as_half((unsigned short)(w[20] >> 16)));
                    uint32_t q0[8], q1[8];
#pragma unroll
                    for (int i = 0; i < 8; i++) {
                        q0[i] = w[4 + i];
                        q1[i] = w[12 + i];
                    }
                    if (!slice(4 * ch + grp, grp, grp ? w[1] : w[0], q0, d, dm) ||
                        !slice(4 * ch + 2 + grp, 2 + grp, grp ? w[3] : w[2], q1, d, dm))
                        return false;
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&ctl->rawfree[slot]);
                }
            } else {
                // tile mode: chunk C holds rows 0..127, chunk C + 1 rows 128..255, each whole
                const int mine = C + (r >> 7), slot = mine % NRV;
                if (!warp_wait(&ctl->rawfull[C % NRV], (C / NRV) & 1, abort, p.status, 1, C) ||
                    !warp_wait(&ctl->rawfull[(C + 1) % NRV], ((C + 1) / NRV) & 1, abort, p.status, 1, C + 1))
                    return false;
                const uint32_t row = smem_u32(raw + slot * SLOT) + (uint32_t)(r & 127) * p.rowbytes;
#pragma unroll 1
                for (int kb = grp; kb < KB; kb += 2) {
                    const uint32_t blk = row + 84u * (uint32_t)(kb >> 2);
                    const int c = kb & 3;
                    uint32_t qw[8];
#pragma unroll
                    for (int i = 0; i < 8; i++) qw[i] = lds32(blk + 4u * (4 + 8 * (c >> 1) + i));
                    const uint32_t dd = lds32(blk + 80u);
                    const float d = __half2float(__ushort_as_half((unsigned short)(dd & 0xffffu)));
                    const float dm = __half2float(__ushort_as_half((unsigned short)(dd >> 16)));
                    if (!slice(kb, c, lds32(blk + 4u * c), qw, d, dm)) return false;
                }
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&ctl->rawfree[C % NRV]);
                    mbar_arrive(&ctl->rawfree[(C + 1) % NRV]);
                }
                C += 2;
            }
            GW += KB;
            return true;
        });
    } else if (warp < kWarpMma) {
        // ---------------------------------------------------------- epilogue warps
        // Thread: token row m = 32 q + lane of the unit (its accumulator lane).
        const int q = warp & 3, m = 32 * q + lane;
        int V = 0;
        for_units(p, tb, n_groups, [&](const Unit& U) -> bool {
            if (warp_aborted(abort)) return false;
            const int b = V & 1;
            const bool valid = m < U.n;
            // this row's destination and scale (read before the wait)
            int dst_row = 0;
            float scale = 1.0f;
            if (valid) {
                if (U.shared) {
                    dst_row = U.tok0 + m;
                    if (NM == 1) scale = p.gate_s[dst_row];
                } else if (NM == 2) {
                    dst_row = U.brow + m;
                } else {
                    dst_row = p.perm[U.brow + m];
                    scale = p.pw[dst_row];
                }
            }
            if (!warp_wait(&ctl->accfull[b], (V >> 1) & 1, abort, p.status, 4, V)) return false;
            tc::fence_after();
            const uint32_t tacc = tc::taddr(tbase, 32 * q, b * 256);
            if (NM == 2) {
                uint16_t* dst = U.shared ? p.out_hs + (size_t)dst_row * p.S + U.mt * 128
                                         : p.out_h + (size_t)dst_row * p.F + U.mt * 128;
#pragma unroll 1
                for (int j0 = 0; j0 < 128; j0 += 16) {
                    uint32_t gv[16], uv[16];
                    tc::ld16(tacc + j0, gv);
                    tc::ld16(tacc + 128 + j0, uv);
                    tc::wait_ld();
                    if (valid) {
                        uint32_t pk[8];
#pragma unroll
                        for (int i = 0; i < 8; i++) {
                            float hv[2];
#pragma unroll
                            for (int h = 0; h < 2; h++) {
                                const float gq = __uint_as_float(gv[2 * i + h]);
                                hv[h] = __fdividef(gq, 1.0f + __expf(-gq)) * __uint_as_float(uv[2 * i + h]);
                            }
                            if (U.shared) {
                                const __nv_bfloat162 t2 = __floats2bfloat162_rn(hv[0], hv[1]);
                                pk[i] = *reinterpret_cast<const uint32_t*>(&t2);
                            } else {
                                pk[i] = pack_h2(hv[0], hv[1]);
                            }
                        }
                        uint4* d4 = reinterpret_cast<uint4*>(dst + j0);
#pragma unroll
                        for (int i = 0; i < 2; i++) d4[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
                    }
                }
            } else {
#pragma unroll 1
                for (int j0 = 0; j0 < 256; j0 += 32) {
                    uint32_t av[32];
                    tc::ld32(tacc + j0, av);
                    tc::wait_ld();
                    if (valid) {
                        if (U.shared) {
                            float4* d4 = reinterpret_cast<float4*>(p.y + (size_t)dst_row * p.H + U.mt * 256 + j0);
#pragma unroll
                            for (int i = 0; i < 8; i++)
                                d4[i] = make_float4(scale * __uint_as_float(av[4 * i]), scale * __uint_as_float(av[4 * i + 1]),
                                                    scale * __uint_as_float(av[4 * i + 2]),
                                                    scale * __uint_as_float(av[4 * i + 3]));
                        } else {
                            uint32_t pk[16];
#pragma unroll
                            for (int i = 0; i < 16; i++)
                                pk[i] = pack_h2(scale * __uint_as_float(av[2 * i]), scale * __uint_as_float(av[2 * i + 1]));
                            uint4* d4 = reinterpret_cast<uint4*>(p.yp + (size_t)dst_row * p.H + U.mt * 256 + j0);
#pragma unroll
                            for (int i = 0; i < 4; i++)
                                d4[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
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
        // The whole warp runs the loop (its values are warp-uniform); lane 0 issues the MMAs and
        // the commits.  Per slice: four M = 128, N = 256, K = 16 MMAs into accumulator buffer V % 2.
        const uint32_t tmu = __shfl_sync(0xffffffffu, tbase, 0);
        const bool leader = lane == 0;
        int GA = 0, GW = 0, V = 0;
        int sa = 0, sw = 0;             // current A and W stages
        uint32_t pa = 0, pw = 0;        // ... and the parity of their fills
        for_units(p, tb, n_groups, [&](const Unit& U) -> bool {
            if (warp_aborted(abort)) return false;
            const int KB = unit_kb(U, p);
            const int b = V & 1;
            if (V >= 2 && !lead_wait(&ctl->accempty[b], ((V >> 1) - 1) & 1, abort, p.status, 5, V)) return false;
            tc::fence_after();
            const uint32_t id = tc::idesc(U.shared ? tc::kBF16 : tc::kF16, kNT, kWRows);
            const uint32_t d = tmu + b * 256;
            for (int kb = 0; kb < KB; kb++) {
                const int ga = GA + kb, gw = GW + kb;
                if (!lead_wait(&ctl->afull[sa], pa, abort, p.status, 6, ga)) return false;
                if (!lead_wait(&ctl->wfull[sw], pw, abort, p.status, 8, gw)) return false;
                tc::fence_after();
                if (leader) {
                    const uint64_t ad = tc::sdesc_sw128(smem_u32(ast + sa * kABytes));
                    const uint64_t bd = tc::sdesc_sw128(smem_u32(wst + sw * kWBytes));
#pragma unroll
                    for (int k16 = 0; k16 < 4; k16++) tc::mma_ss_f16(d, ad + 2 * k16, bd + 2 * k16, id, (kb | k16) != 0);
                    tc::commit(&ctl->aempty[sa]);
                    tc::commit(&ctl->wempty[sw]);
                }
                __syncwarp();
                if (++sa == NA) {  // next A and W stages and their phases
                    sa = 0;
                    pa ^= 1;
                }
                if (++sw == NW) {
                    sw = 0;
                    pw ^= 1;
                }
            }
            if (leader) tc::commit(&ctl->accfull[b]);
            __syncwarp();
            GA += KB;
            GW += KB;
            V++;
            return true;
        });
        if (leader) {
            tc::commit(&ctl->drain);  // completes once every MMA issued above has
            (void)mbar_wait(&ctl->drain, 0);
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------- TMA: raw weights + shared W tiles (warp 21),
        // token rows (warp 22)
        const bool do_raw = (warp == kWarpRaw), do_a = (warp == kWarpA);
        if (lane == 0) {
            int C = 0, GW = 0, GA = 0;
            int wt_last[kMaxNW];  // per W stage, the last fill this thread issued (-1: none)
            for (int i = 0; i < NW; i++) wt_last[i] = -1;
            for_units(p, tb, n_groups, [&](const Unit& U) -> bool {
                if (*abort) return false;
                const int KB = unit_kb(U, p);
                if (do_raw && U.shared) {
                    // the shared expert's bf16 rows are the W operand as they land: two 128-row boxes
                    for (int kb = 0; kb < KB; kb++) {
                        const int g = GW + kb;
                        int s, fill;
                        w_stage(g, NW, s, fill);
                        if (fill > 0 && !thread_wait(&ctl->wempty[s], (fill - 1) & 1, abort, p.status, 10, g))
                            return false;
                        uint8_t* w = wst + s * kWBytes;
                        uint64_t* bar = &ctl->wfull[s];
                        wt_last[s] = g;
                        mbar_arrive_expect_tx(bar, kWBytes);
                        mbar_arrive_count(bar, kDeqWarps / 2 - 1);
                        if (NM == 2) {
                            tma_load_2d(w, &p.map_s0, kb * 64, U.mt * 128, bar);
                            tma_load_2d(w + kWBytes / 2, &p.map_s1, kb * 64, U.mt * 128, bar);
                        } else {
                            tma_load_2d(w, &p.map_s0, kb * 64, U.mt * 256, bar);
                            tma_load_2d(w + kWBytes / 2, &p.map_s0, kb * 64, U.mt * 256 + 128, bar);
                        }
                    }
                } else if (do_raw) {
                    const int nch = unit_nch(U, p);
                    for (int ch = 0; ch < nch; ch++, C++) {
                        const int slot = C % NRV;
                        if (C >= NRV && !thread_wait(&ctl->rawfree[slot], ((C / NRV) - 1) & 1, abort, p.status, 9, C))
                            return false;
                        uint8_t* sl = raw + slot * SLOT;
                        uint64_t* bar = &ctl->rawfull[slot];
                        if (p.raw_mode == kRawColumn) {
                            const int x0 = (84 * ch) & ~15;
                            const int r0 = (NM == 2) ? U.mt * 128 : U.mt * 256;
                            const int r1 = (NM == 2) ? p.q_rows_m1 + U.mt * 128 : U.mt * 256 + 128;
                            mbar_arrive_expect_tx(bar, kColSlot);
                            tma_load_3d(sl, &p.map_q, x0, r0, U.e, bar);
                            tma_load_3d(sl + kHalfSlot, &p.map_q, x0, r1, U.e, bar);
                        } else {
                            const uint32_t bytes = 128u * (uint32_t)p.rowbytes;
                            const int row = (NM == 2) ? (ch == 0 ? 0 : p.q_rows_m1) + U.mt * 128 : U.mt * 256 + 128 * ch;
                            mbar_arrive_expect_tx(bar, bytes);
                            bulk_g2s(sl, p.experts + (size_t)U.e * p.stride + p.q_off + (size_t)row * p.rowbytes, bytes,
                                     bar);
                        }
                    }
                }
                GW += KB;
                if (do_a) {
                    // token rows: the unit's rows only (one 128-row box, or 64 and/or 32-row boxes)
                    const CUtensorMap* mp = U.shared ? p.map_bs : p.map_br;
                    const int r128 = U.n > 96 ? 128 : 0;
                    const int r64 = (r128 == 0 && U.n > 32) ? 64 : 0;
                    const int r32 = (r128 == 0 && U.n - r64 > 0) ? 32 : 0;
                    for (int kb = 0; kb < KB; kb++, GA++) {
                        const int s = GA % NA;
                        if (GA >= NA && !thread_wait(&ctl->aempty[s], ((GA / NA) - 1) & 1, abort, p.status, 11, GA))
                            return false;
                        uint8_t* as = ast + s * kABytes;
                        mbar_arrive_expect_tx(&ctl->afull[s], (uint32_t)(r128 + r64 + r32) * 128u);
                        if (r128) tma_load_2d(as, &mp[0], kb * 64, U.brow, &ctl->afull[s]);
                        if (r64) tma_load_2d(as, &mp[1], kb * 64, U.brow, &ctl->afull[s]);
                        if (r32) tma_load_2d(as + r64 * 128, &mp[2], kb * 64, U.brow + r64, &ctl->afull[s]);
                    }
                }
                return true;
            });
            if (*abort) {  // let issued copies land before the CTA exits
                for (int i = 1; do_raw && i <= NRV && i <= C; i++) {
                    const int c = C - i;
                    (void)mbar_wait(&ctl->rawfull[c % NRV], (c / NRV) & 1, 1000000ull);
                }
                for (int s = 0; do_raw && s < NW; s++)
                    if (wt_last[s] >= 0) (void)mbar_wait(&ctl->wfull[s], (wt_last[s] / NW) & 1, 1000000ull);
                for (int i = 1; do_a && i <= NA && i <= GA; i++) {
                    const int c = GA - i;
                    (void)mbar_wait(&ctl->afull[c % NA], (c / NA) & 1, 1000000ull);
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

// Raw-weight staging mode for a Q2_K matrix with contraction length K, or -1: column boxes of
// 112 bytes when rows are a multiple of 16 bytes, else 128 whole rows per raw slot.
int raw_mode_for(int K) {
    const int rowbytes = K / 256 * 84;
    if (rowbytes % 16 == 0) return kRawColumn;
    if (128 * rowbytes <= kMaxSlot) return kRawTile;
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

// Dynamic shared memory of an expert kernel with na A stages and raw slots of `slot` bytes.
size_t expert_smem(int E, int na, int slot, int nrv, int nw) {
    return 1024 + (size_t)na * kABytes + (size_t)nw * kWBytes + (size_t)nrv * slot + sizeof(ExpertCtl) +
           4 * (3 * (size_t)E + 1);
}
// Raw slot bytes for contraction length K (a column chunk, or 128 whole rows).
int slot_for(int K) {
    const int rowbytes = K / 256 * 84;
    return raw_mode_for(K) == kRawColumn ? kColSlot : 128 * rowbytes;
}
// A stages that fit beside the rest (0: the kernel does not fit at all).
struct StagePlan {
    int na, nw, nrv;  // A stages, W stages, raw slots (0: the kernel does not fit)
};
// Stages for contraction length K: three W stages, the raw slots (two column chunks, or four
// halves of whole-row units), and as many A stages (two at least) as fit beside them.  Of
// the plans measured at 2048 and 512 tokens of the 35B-A3B layer (W stages 2 or 3, column
// raw slots 2 or 3) this one was fastest.
StagePlan stages_for(int E, int K, size_t smem_optin) {
    StagePlan sp{kMaxNA, 3, raw_mode_for(K) == kRawColumn ? 2 : 4};
    while (sp.na >= 2 && expert_smem(E, sp.na, slot_for(K), sp.nrv, sp.nw) > smem_optin) sp.na--;
    if (sp.na < 2) sp.na = 0;
    return sp;
}
size_t router_smem() { return 1024 + kRouterStages * 4 * 16384 + sizeof(RouterCtl); }

// Launch one expert kernel, one CTA per SM.
template <int NM>
cudaError_t launch_expert(ExpertParams& p, int n_sm, int E, cudaStream_t st) {
    pf_expert_kernel<NM><<<n_sm, kExpertThreads, expert_smem(E, p.na, p.slot, p.nrv, p.nw), st>>>(p);
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
    if (raw_mode_for(s.hidden) < 0 || raw_mode_for(s.expert_ffn) < 0) return false;
    // units: 128 gate + 128 up rows (gate/up), 256 rows (down)
    if (s.expert_ffn % 128 || s.hidden % 256 || s.shared_ffn % 128) return false;
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
    const StagePlan sp2 = stages_for(E, H, (size_t)f->smem_optin);
    const StagePlan sp1 = stages_for(E, F, (size_t)f->smem_optin);
    if (sp2.na == 0 || sp1.na == 0 || (size_t)f->smem_optin < router_smem()) return cudaErrorNotSupported;
    if (!get_encode()) return cudaErrorNotSupported;
    if (!f->attr_set) {
        if ((e = cudaFuncSetAttribute(pf_router_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)router_smem())) != cudaSuccess)
            return e;
        if ((e = cudaFuncSetAttribute(pf_expert_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      f->smem_optin)) != cudaSuccess)
            return e;
        if ((e = cudaFuncSetAttribute(pf_expert_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      f->smem_optin)) != cudaSuccess)
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
        p.raw_mode = raw_mode_for(K);
        p.slot = slot_for(K);
        const StagePlan& sp = (nm == 2) ? sp2 : sp1;
        p.na = sp.na;
        p.nw = sp.nw;
        p.nrv = sp.nrv;
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
        p.MT = (nm == 2) ? F / 128 : H / 256;
        p.nt = kNT;
        p.E = E;
        p.k = k;
        p.T = T;
        p.F = F;
        p.S = S;
        p.H = H;
        if (S > 0) {
            p.Ks = (nm == 2) ? H : S;
            p.MTs = (nm == 2) ? S / 128 : H / 256;
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
